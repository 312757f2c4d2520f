"""Seeded synthetic inputs: activations with outlier channels and per-layer
orthogonal rotations.

This module only draws inputs.  It holds none of the hot path's arithmetic
(rotation, clipping, quantisation, attention); both the CUDA path and the CPU
oracle consume what it returns.

Rotations are input data to the library.  The K-side rotation follows the
OSCAR-RotationZoo card [File format]: R_K = R * H * P_br with R the
eigenvectors of the query covariance, H a head-dim Hadamard and P_br a
bit-reversal permutation; the V side uses a seeded QR-orthogonal matrix.  Exact
signed permutations are also offered: with them every rotated value is exact
in any precision, which makes whole-chain bit-exact checks possible.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# roles in the seed sequence
ROLE_CALIB, ROLE_Q, ROLE_K, ROLE_V, ROLE_RV, ROLE_CHANNELS, ROLE_PERM = range(7)


def rng_for(config_id: int, layer: int, role: int, extra: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([config_id, layer, role, extra]))


# --------------------------------------------------------------------------
# activations
# --------------------------------------------------------------------------
def outlier_channels(config_id: int, layer: int, head_dim: int, count: int | None = None):
    """Outlier channel indices: 2% of head_dim (at least 1), seeded per layer."""
    if count is None:
        count = max(1, int(round(0.02 * head_dim)))
    rng = rng_for(config_id, layer, ROLE_CHANNELS)
    return np.sort(rng.choice(head_dim, size=count, replace=False))


def activations(rng: np.random.Generator, shape, channels, kind: str = "t3", mag: float = 8.0):
    """N(0,1) float32 with heavy outlier channels on the last axis.

    kind 'scale': channels multiplied by ``mag``.
    kind 't3':    channels get ``mag`` * Student-t(3) added.
    """
    x = rng.standard_normal(size=shape, dtype=np.float32)
    ch = np.asarray(channels)
    if len(ch):
        if kind == "scale":
            x[..., ch] *= np.float32(mag)
        else:
            x[..., ch] += np.float32(mag) * rng.standard_t(3, size=x[..., ch].shape).astype(np.float32)
    return x


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bfloat16 value (ties to even), kept as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32)
    return r.view(np.float32).reshape(np.shape(x))


# --------------------------------------------------------------------------
# rotations
# --------------------------------------------------------------------------
def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (power of two), scaled by 1/sqrt(d)."""
    assert d & (d - 1) == 0
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h / math.sqrt(d)


def bit_reversal(d: int) -> np.ndarray:
    """Permutation matrix P with P[i, br(i)] = 1, br reversing log2(d) bits."""
    bits = int(math.log2(d))
    idx = np.array([int(format(i, f"0{bits}b")[::-1], 2) for i in range(d)])
    p = np.zeros((d, d))
    p[np.arange(d), idx] = 1.0
    return p


def eig_rotation(calib_q: np.ndarray) -> np.ndarray:
    """R_K = E H P_br in float64, E = eigenvectors of Sigma_Q = Q^T Q sorted by
    descending eigenvalue, each column's largest-magnitude entry made positive."""
    q = np.asarray(calib_q, np.float64)
    sigma = q.T @ q
    w, e = np.linalg.eigh(sigma)
    order = np.argsort(w)[::-1]
    e = e[:, order]
    piv = np.argmax(np.abs(e), axis=0)
    e = e * np.sign(e[piv, np.arange(e.shape[1])])
    d = e.shape[0]
    return e @ hadamard(d) @ bit_reversal(d)


def qr_rotation(rng: np.random.Generator, d: int) -> np.ndarray:
    a = rng.standard_normal((d, d))
    qm, rm = np.linalg.qr(a)
    return qm * np.sign(np.diag(rm))


def signed_permutation(rng: np.random.Generator, d: int) -> np.ndarray:
    perm = rng.permutation(d)
    sign = rng.choice(np.array([-1.0, 1.0]), size=d)
    p = np.zeros((d, d))
    p[np.arange(d), perm] = sign
    return p


# --------------------------------------------------------------------------
# named workloads
# --------------------------------------------------------------------------
@dataclass
class Workload:
    """Shapes and quantisation settings of one synthetic workload."""
    name: str
    config_id: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    context: int
    sink: int
    recent: int
    k_clip: float
    v_clip: float
    num_layers: int = 1
    absorb_v: bool = False
    in_fp32: bool = False
    act_kind: str = "t3"
    append_tokens: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    # Tiny single-layer decode: fp32 Q/K/V with channels 3, 17, 90 scaled x8.
    "tiny": Workload("tiny", 0, 1, 4, 1, 128, 1024, 64, 256, 0.96, 0.92,
                     in_fp32=True, act_kind="scale",
                     extra={"channels": [3, 17, 90], "calib_rows": 4096}),
    # Qwen3-4B-shaped attention layer, one decode step.
    "qwen3-4b-layer": Workload("qwen3-4b-layer", 1, 8, 32, 8, 128, 16384, 512, 2048, 0.96, 0.96),
    # Qwen3-8B-shaped decode over 36 layers, V rotation absorbed.
    "qwen3-8b-36L": Workload("qwen3-8b-36L", 2, 32, 32, 8, 128, 32768, 64, 256, 0.96, 0.92,
                             num_layers=36, absorb_v=True),
    # head_dim 512 decode.
    "hd512": Workload("hd512", 3, 4, 16, 8, 512, 65536, 512, 2048, 0.96, 0.96),
    # Qwen3-32B-shaped long context: phase 1 append of 8192 tokens, batch 4.
    "qwen3-32b-append": Workload("qwen3-32b-append", 4, 4, 64, 8, 128, 131072, 64, 256, 0.96, 0.92,
                                 append_tokens=8192),
    # Qwen3-32B-shaped long context: phase 2 decode, batch 1.
    "qwen3-32b-decode": Workload("qwen3-32b-decode", 4, 1, 64, 8, 128, 131072, 64, 256, 0.96, 0.92),
}


def rotations(w: Workload, layer: int, kind: str = "oscar"):
    """(R_K, R_V) float32 [D][D] for one layer.

    kind 'oscar': R_K from the eigenvectors of a seeded calibration set's
    Q^T Q times H times P_br; R_V seeded QR.  kind 'perm': exact signed
    permutations.  kind 'identity'.
    """
    d = w.head_dim
    if kind == "identity":
        e = np.eye(d, dtype=np.float32)
        return e, e.copy()
    if kind == "perm":
        return (signed_permutation(rng_for(w.config_id, layer, ROLE_PERM, 0), d).astype(np.float32),
                signed_permutation(rng_for(w.config_id, layer, ROLE_PERM, 1), d).astype(np.float32))
    ch = w.extra.get("channels")
    if ch is None:
        ch = outlier_channels(w.config_id, layer, d)
    calib = activations(rng_for(w.config_id, layer, ROLE_CALIB), (w.extra.get("calib_rows", 4096), d),
                        ch, kind=w.act_kind)
    rk = eig_rotation(calib).astype(np.float32)
    rv = qr_rotation(rng_for(w.config_id, layer, ROLE_RV), d).astype(np.float32)
    return rk, rv


def kv_rows(w: Workload, layer: int, n_tokens: int, batch: int | None = None, extra: int = 0):
    """(k, v) [B][n][Hkv][D] float32 (bf16-representable unless the workload is fp32)."""
    b = w.batch if batch is None else batch
    ch = w.extra.get("channels")
    if ch is None:
        ch = outlier_channels(w.config_id, layer, w.head_dim)
    shape = (b, n_tokens, w.num_kv_heads, w.head_dim)
    k = activations(rng_for(w.config_id, layer, ROLE_K, extra), shape, ch, kind=w.act_kind)
    v = activations(rng_for(w.config_id, layer, ROLE_V, extra), shape, ch, kind=w.act_kind)
    if not w.in_fp32:
        k, v = to_bf16_values(k), to_bf16_values(v)
    return k, v


def queries(w: Workload, layer: int, batch: int | None = None, extra: int = 0):
    """q [B][Hq][D] float32 (bf16-representable unless the workload is fp32)."""
    b = w.batch if batch is None else batch
    ch = w.extra.get("channels")
    if ch is None:
        ch = outlier_channels(w.config_id, layer, w.head_dim)
    q = activations(rng_for(w.config_id, layer, ROLE_Q, extra), (b, w.num_q_heads, w.head_dim), ch,
                    kind=w.act_kind)
    return q if w.in_fp32 else to_bf16_values(q)


# --------------------------------------------------------------------------
# device-side generation for large workloads (torch RNG on the GPU)
# --------------------------------------------------------------------------
def activations_torch(gen, shape, channels, kind: str = "t3", mag: float = 8.0, dtype=None, device="cuda"):
    """Same distribution as :func:`activations`, drawn with a seeded torch generator.

    Student-t(3) is drawn as z / sqrt(chi2_3 / 3) from four standard normals.
    """
    import torch

    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    ch = torch.as_tensor(np.asarray(channels), device=device, dtype=torch.long)
    if ch.numel():
        sub = list(shape[:-1]) + [ch.numel()]
        if kind == "scale":
            x[..., ch] *= mag
        else:
            z = torch.randn(sub, generator=gen, device=device)
            n = torch.randn([3] + sub, generator=gen, device=device)
            t3 = z / torch.sqrt((n * n).sum(0) / 3.0)
            x[..., ch] += mag * t3
    return x if dtype is None else x.to(dtype)
