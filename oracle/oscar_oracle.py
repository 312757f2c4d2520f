"""CPU oracle for the rotated INT2 KV cache: append (rotate, clip, group-128 INT2
quantise, BF16 sink/recent windows) and mixed INT2/BF16 decode attention.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline arm may import this module.  The product path (the
CUDA library and its Python binding) never calls it and shares no code with it.

It is deliberately plain: numpy, one pass, no blocking, no splits.  The codec is
computed in float32 with the operation order written below (numpy float32
element-wise ufuncs round every operation to nearest-even and never contract to
FMA); everything attention-side is float64.

Sources (titles of the pages describing OSCAR; section in brackets):

* OSCAR-LLAMACPP-Qwen3-4B-Thinking-2507-INT2-KV model card [Run]: per-row
  outlier clip before quantisation (clip ratio 0.96); first/last tokens kept
  high-precision (sink 512 / recent 2048); [Files] note: K and V are rotated
  by an orthogonal matrix after RoPE.
* OSCAR-LLAMACPP-Gemma-4-12B-it-INT2-KV card [Folders]: the rotation is applied
  to Q/K (and V); per-layer 512x512 rotations exist (head_dim 512).
* OSCAR-RotationZoo card [Available rotations]: G is the INT2 quant group size
  along head_dim (group128); [How to use]: K clip 0.96, V clip 0.92, V
  rotation absorbed, 64 prefix / 256 recent BF16 tokens, int2 KV dtype,
  quant group size 128; [File format]: one head_dim x head_dim rotation per
  layer, shared by the heads of the layer.
* hysenlabs article on FutureMLS-Lab/OSCAR [What OSCAR compresses]: bulk of the
  cache INT2, BF16 only for the first and the latest tokens; [How the offline rotation is
  fit]: the fit also yields clip limits applied ahead of rounding; fused
  mixed INT2+BF16 flash attention instead of dequantise-then-attend.

Readings taken where the pages are silent:

* quantiser: asymmetric per group of 128 along head_dim, scale=(max-min)/3,
  zero=min, both stored as IEEE fp16 (round-to-nearest-even);
* clip: t = ratio * max_j |r_j| over the whole rotated row (one token, one KV
  head, all head_dim channels), x = clamp(r, -t, t), before grouping;
* constant group (scale rounds to 0): every code is 0 and the value is zero;
* code = clamp(rint_half_even((x - zero) * (1 / scale)), 0, 3), with the
  reciprocal correctly rounded and no fused multiply-add;
* row-vector rotation k' = k R with R stored [D][D] row-major; Q uses R_K;
  the output is un-rotated once, o = o' R_V^T, unless the V rotation is
  absorbed by the caller;
* windows: sink = positions [0, S), ring = [max(S, T-W), T), INT2 = the rest;
  BF16 window copies hold BF16(RNE) of the same float32 rotated row;
* softmax scale 1/sqrt(D) unless given;
* data-free in-quant Hadamard (FLAG_HADAMARD): for a model with no calibrated
  rotation, K and V are rotated by the Sylvester Hadamard matrix of order 128
  (normalised by 1/sqrt(128)), block-diagonal over the head_dim groups, and Q
  and the output use that same matrix in place of R_K and R_V;
* K-only INT2 (FLAG_V_BF16): V is kept high precision, the BF16 of the
  float32 rotated row for every position in a [B][Hkv][capacity][D] region;
  K is stored as usual;
* Lloyd-Max levels (FLAG_LLOYD_MAX; hysenlabs article [Installing OSCAR and
  running a first Qwen3-8B calibration]: the SGLANG_LLOYD_MAX switch; [Where
  OSCAR loses]: LM_RATIO=1.16): the four levels of a group are
  zero + unit * (0, rho, rho + 1, 2 rho + 1), rho = LM_RATIO being the ratio of
  the outer to the inner gap between adjacent levels (the shape of the
  four-level Lloyd-Max quantiser of a Gaussian), spread over the group's
  min..max; rho is the printed 1.16 rounded to float32, the span 2 rho + 1 and
  the midpoints rho / 2, rho + 1/2 (both exact) and 3 rho / 2 + 1 (computed as
  span - rho / 2, one rounding) are float32; the code is the number of
  midpoints strictly below y: the nearest level, a tie going to the lower one;
* R_V calibration (RotationZoo [File format]: the V rotation comes from a
  covariance of the values weighted by scores): the printed V^T diag(K^T (Q^T Q) K) V read
  with K holding keys as columns, so each key row is weighted by its score
  energy w_t = k_t Q^T Q k_t^T; R_V = E H P_br as for R_K.

The byte layout written by :func:`append` is the one the C header documents
for the cache (regions, strides, code bit positions); it is implemented here
from that description, independently of the CUDA code.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

GROUP = 128
ALIGN = 256
NCAP_ROUND = 64

FLAG_ABSORB_V = 1
FLAG_IN_FP32 = 2
FLAG_OUT_FP32 = 4
FLAG_HADAMARD = 8
FLAG_V_BF16 = 16
FLAG_LLOYD_MAX = 32

# Lloyd-Max level ratio LM_RATIO = 1.16 as printed, rounded once to float32
LM_RATIO = float(np.float32(1.16))


def lloyd_max_thresholds():
    """(span, (m0, m1, m2)) of the Lloyd-Max codec as float32, each one
    IEEE round-to-nearest operation on rho = float32(LM_RATIO), in this order:
      span = 2 * rho + 1        (exact: 2 rho and 1 share the step of [2, 4))
      m0   = rho * 0.5          (exact)
      m1   = rho + 0.5          (exact: both are multiples of rho's step)
      m2   = span - m0          (the float32 nearest to 3 rho / 2 + 1)
    m0, m1, m2 are the midpoints between adjacent levels (0, rho, rho + 1, 2 rho + 1)."""
    rho = np.float32(LM_RATIO)
    span = np.float32(np.float32(2.0) * rho) + np.float32(1.0)
    m0 = np.float32(rho * np.float32(0.5))
    m1 = np.float32(rho + np.float32(0.5))
    m2 = np.float32(span - m0)
    return np.float32(span), (m0, m1, m2)


# --------------------------------------------------------------------------
# configuration and layout
# --------------------------------------------------------------------------
@dataclass
class Config:
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    sink: int
    recent: int
    capacity: int
    k_clip: float = 0.96
    v_clip: float = 0.92
    flags: int = 0
    group_size: int = GROUP

    @property
    def G(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _align(x: int) -> int:
    return (x + ALIGN - 1) // ALIGN * ALIGN


def layout(cfg: Config) -> dict:
    """Byte sizes of one layer's cache, per the header's documented formulas.

    Per layer: K role then V role (with FLAG_V_BF16 the V role is instead
    [B][Hkv][capacity][D] bf16, one row per position).  Per role: sink [B][Hkv][S][D] bf16, ring
    [B][Hkv][W][D] bf16, codes [B][Hkv][Ncap][D/4] u8, sz [B][Hkv][Ncap][D/128]
    x (fp16 scale, fp16 zero); Ncap = round_up(max(capacity - S, 0), 64); each
    region starts on a 256-byte boundary.
    """
    B, H, D, S, W = cfg.batch, cfg.num_kv_heads, cfg.head_dim, cfg.sink, cfg.recent
    ncap = -(-max(cfg.capacity - S, 0) // NCAP_ROUND) * NCAP_ROUND
    sink = _align(B * H * S * D * 2)
    ring = _align(B * H * W * D * 2)
    codes = _align(B * H * ncap * (D // 4))
    sz = _align(B * H * ncap * (D // GROUP) * 4)
    role = sink + ring + codes + sz
    # with FLAG_V_BF16 the V role is one BF16 row per position
    v_role = _align(B * H * cfg.capacity * D * 2) if cfg.flags & FLAG_V_BF16 else role
    return dict(ncap=ncap, sink_bytes=sink, ring_bytes=ring, codes_bytes=codes,
                sz_bytes=sz, role_bytes=role, v_role_bytes=v_role, layer_bytes=role + v_role,
                total_bytes=(role + v_role) * cfg.num_layers)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits.

    bf16 is the top half of a float32; rounding adds 0x7FFF plus the lowest kept
    bit before truncating, which is round-half-to-even on the dropped 16 bits.
    NaN stays a quiet NaN.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# rotation and codec
# --------------------------------------------------------------------------
def rotate_rows(x: np.ndarray, R: np.ndarray) -> np.ndarray:
    """r = x R (row vectors, R [D][D] row-major), exact float64 product rounded
    once to float32."""
    return (np.asarray(x, np.float64) @ np.asarray(R, np.float64)).astype(np.float32)


def hadamard_rotation(d: int) -> np.ndarray:
    """Rotation of the data-free in-quant Hadamard, float64 [d][d].

    The llama.cpp model card's environment table [Run] names an in-quant
    Hadamard that models with a baked rotation skip, and a base model without
    one falls back to data-free INT2 with it; the RotationZoo card's SGLang
    launch [How to use] sets its order to 128.  Read here as: block-diagonal over the d / 128 groups, each
    block the Sylvester Hadamard matrix of order 128, H[i][k] =
    (-1)^popcount(i & k), divided by sqrt(128) so that it is orthogonal.
    """
    n = GROUP
    blk = np.empty((n, n), dtype=np.float64)
    for i in range(n):
        for k in range(n):
            blk[i, k] = -1.0 if bin(i & k).count("1") % 2 else 1.0
    blk /= math.sqrt(n)
    R = np.zeros((d, d), dtype=np.float64)
    for j in range(d // n):
        R[j * n:(j + 1) * n, j * n:(j + 1) * n] = blk
    return R


def sylvester_hadamard(n: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order n (a power of two) divided by sqrt(n),
    float64: H[i][k] = (-1)^popcount(i & k) / sqrt(n)."""
    i = np.arange(n)
    bits = np.bitwise_and.outer(i, i)
    par = np.zeros_like(bits)
    while bits.any():
        par ^= bits & 1
        bits >>= 1
    return np.where(par == 1, -1.0, 1.0) / math.sqrt(n)


def bit_reversal_index(n: int) -> np.ndarray:
    """br[i] = i with its log2(n) bits reversed."""
    b = int(round(math.log2(n)))
    return np.array([int(format(i, f"0{b}b")[::-1], 2) if b else 0 for i in range(n)])


def rotation_from_covariance(sigma: np.ndarray) -> np.ndarray:
    """R = E H P_br for a symmetric positive semi-definite covariance, float64 [D][D].

    E = the eigenvectors of sigma by descending eigenvalue (ties by index), each
    column signed so that its largest-magnitude entry (the first, on ties) is
    positive; H = sylvester_hadamard(D); P_br[i, br(i)] = 1, so column j of R
    is column br(j) of E H.  The eigen-solver is the library one (numpy eigh).
    """
    sigma = np.asarray(sigma, np.float64)
    d = sigma.shape[0]
    w, e = np.linalg.eigh(sigma)
    order = np.argsort(-w, kind="stable")
    e = e[:, order]
    piv = np.argmax(np.abs(e), axis=0)
    e = e * np.where(e[piv, np.arange(d)] < 0, -1.0, 1.0)
    eh = e @ sylvester_hadamard(d)
    return eh[:, bit_reversal_index(d)]


def calibrate_rk(calib_q: np.ndarray) -> np.ndarray:
    """K-side rotation fitted to a calibration set of query rows, float64 [D][D].

    OSCAR-RotationZoo card [File format]: R_K = R H P_br, R the eigenvectors of
    the query covariance, H a head-dim Hadamard, P_br the eigenvalue-sorted
    bit-reversal permutation; hysenlabs article [How the offline rotation is
    fit]: Q activations are captured offline and the rotation derived from
    their covariance.  Read as: Sigma = Q^T Q (float64 over the rows), then
    rotation_from_covariance(Sigma).
    """
    q = np.asarray(calib_q, np.float64)
    return rotation_from_covariance(q.T @ q)


def score_energy(calib_q: np.ndarray, calib_k: np.ndarray) -> np.ndarray:
    """w_t = k_t (Q^T Q) k_t^T for every key row: the sum over the calibration
    queries of the squared logit q_n . k_t, float64 [n_kv]."""
    q = np.asarray(calib_q, np.float64)
    k = np.asarray(calib_k, np.float64)
    sigma_q = q.T @ q
    return np.sum((k @ sigma_q) * k, axis=1)


def calibrate_rv(calib_q: np.ndarray, calib_k: np.ndarray, calib_v: np.ndarray) -> np.ndarray:
    """V-side rotation fitted to the value covariance weighted by score energy, float64 [D][D].

    OSCAR-RotationZoo card [File format]: the V rotation file is built on
    Sigma_V = V^T diag(K^T (Q^T Q) K) V, with the same R H P_br construction as
    the K side.  The printed product composes when K holds the keys as columns
    (D x n_kv) and Q and V hold rows: K^T Q^T Q K = S^T S with S = Q K the
    logits of every calibration query against every key, whose diagonal is each
    key's score energy w_t (score_energy).  Read as: Sigma_V = sum_t w_t v_t^T v_t
    over the key/value rows of one layer (row t of calib_k and of calib_v are
    the same token and KV head), then rotation_from_covariance(Sigma_V).
    """
    v = np.asarray(calib_v, np.float64)
    w = score_energy(calib_q, calib_k)
    return rotation_from_covariance((v * w[:, None]).T @ v)


def rotations_of(cfg: "Config", R_K, R_V):
    """(R_K, R_V) a call uses: the given matrices, or the in-quant Hadamard for
    both when cfg.flags has FLAG_HADAMARD (the given ones are then ignored)."""
    if cfg.flags & FLAG_HADAMARD:
        H = hadamard_rotation(cfg.head_dim)
        return H, H
    return R_K, R_V


def lloyd_max_levels(rho: float = LM_RATIO) -> np.ndarray:
    """The four Lloyd-Max levels in units of the group's step: 0, rho, rho+1, 2rho+1.

    Adjacent gaps are rho, 1, rho: the outer gaps are rho times the inner one,
    as in the four-level Lloyd-Max quantiser of a Gaussian (levels +-0.4528,
    +-1.510 standard deviations, outer/inner gap 1.167)."""
    return np.array([0.0, rho, rho + 1.0, 2.0 * rho + 1.0], dtype=np.float64)


def quantize_rows(r: np.ndarray, ratio: float, lloyd_max: bool = False):
    """Clip then group-128 asymmetric INT2 quantisation of float32 rows.

    r: [N, D] float32 rotated rows.  Returns (codes [N, D] uint8 in 0..3,
    scale [N, D/128] float16, zero [N, D/128] float16).

    Steps, each a float32 round-to-nearest operation:
      a = max_j |r_j| ; t = ratio * a ; x = min(max(r, -t), t)
      per group: mn = min x, mx = max x ; s32 = (mx - mn) / span
      scale = fp16(s32) ; zero = fp16(mn)
      scale == 0      -> code 0
      otherwise inv = 1 / scale ; y = (x - zero) * inv
    Uniform levels (span 3): code = clamp(rint(y), 0, 3).
    Lloyd-Max levels (span 2 rho + 1, levels lloyd_max_levels(), float32
    span and midpoints from lloyd_max_thresholds()): code = the number of
    midpoints between adjacent levels that lie strictly below y.
    A non-finite scale or zero also yields code 0.
    """
    r = np.ascontiguousarray(r, dtype=np.float32)
    n, d = r.shape
    ng = d // GROUP
    a = np.max(np.abs(r), axis=1)
    t = (np.float32(ratio) * a).astype(np.float32)
    x = np.minimum(np.maximum(r, -t[:, None]), t[:, None])
    xg = x.reshape(n, ng, GROUP)
    mn = xg.min(axis=2)
    mx = xg.max(axis=2)
    lm_span, lm_mids = lloyd_max_thresholds()
    span = lm_span if lloyd_max else np.float32(3.0)
    s32 = ((mx - mn) / span).astype(np.float32)
    with np.errstate(over="ignore"):
        scale = s32.astype(np.float16)
        zero = mn.astype(np.float16)
    sf = scale.astype(np.float32)
    zf = zero.astype(np.float32)
    ok = (sf != 0) & np.isfinite(sf) & np.isfinite(zf)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        inv = np.where(ok, np.float32(1.0) / np.where(ok, sf, np.float32(1.0)), np.float32(0.0))
        inv = inv.astype(np.float32)
        y = ((xg - zf[:, :, None]).astype(np.float32) * inv[:, :, None]).astype(np.float32)
        if lloyd_max:
            q = sum((y > m).astype(np.float64) for m in lm_mids)
        else:
            q = np.rint(y)
    q = np.where(ok[:, :, None], q, 0.0)
    codes = np.clip(q, 0, 3).astype(np.uint8).reshape(n, d)
    return codes, scale, zero


def dequantize_rows(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray, lloyd_max: bool = False) -> np.ndarray:
    """x_hat = zero + scale * level(code), exact in float64 (fp16 inputs);
    level(c) = c, or lloyd_max_levels()[c] with Lloyd-Max levels."""
    n, d = codes.shape
    s = scale.astype(np.float64).repeat(GROUP, axis=1)
    z = zero.astype(np.float64).repeat(GROUP, axis=1)
    lev = lloyd_max_levels()[codes] if lloyd_max else codes.astype(np.float64)
    return z + s * lev


# --------------------------------------------------------------------------
# physical code packing (the header's bit layout)
# --------------------------------------------------------------------------
def pack_codes(codes: np.ndarray, role: int) -> np.ndarray:
    """Pack [N, D] codes (0..3) into [N, D/4] bytes.

    A row is D/16 little-endian 32-bit words; word w, bit b holds the code of
    one dim.  With j the 128-dim group:
      K (role 0): word j*8 + 2*c + i (c 0..3, i 0..1); for p in 0..7 with
        kk = 4*i + p//2 and h = p%2: bit 2p <- dim 128j + 16kk + 2c + 8h,
        bit 16+2p <- that dim + 1.
      V (role 1): word j*8 + g (g 0..7); bit 2n (n 0..15) <- dim 128j + 8n + g.
    """
    n, d = codes.shape
    words = np.zeros((n, d // 16), dtype=np.uint32)
    for dim, word, bit in _bit_map(d, role):
        words[:, word] |= codes[:, dim].astype(np.uint32) << np.uint32(bit)
    return words.view(np.uint8).reshape(n, d // 4)


def unpack_codes(packed: np.ndarray, d: int, role: int) -> np.ndarray:
    n = packed.shape[0]
    words = np.ascontiguousarray(packed, dtype=np.uint8).reshape(n, d // 4).view(np.uint32)
    codes = np.zeros((n, d), dtype=np.uint8)
    for dim, word, bit in _bit_map(d, role):
        codes[:, dim] = (words[:, word] >> np.uint32(bit)) & np.uint32(3)
    return codes


def _bit_map(d: int, role: int):
    """(dim, word, bit) triples for every dim of a row."""
    out = []
    for j in range(d // GROUP):
        if role == 0:
            for c in range(4):
                for i in range(2):
                    for p in range(8):
                        kk = 4 * i + p // 2
                        h = p % 2
                        dim = GROUP * j + 16 * kk + 2 * c + 8 * h
                        word = j * 8 + 2 * c + i
                        out.append((dim, word, 2 * p))
                        out.append((dim + 1, word, 16 + 2 * p))
        else:
            for g in range(8):
                for n in range(16):
                    out.append((GROUP * j + 8 * n + g, j * 8 + g, 2 * n))
    return out


# --------------------------------------------------------------------------
# cache views
# --------------------------------------------------------------------------
class CacheView:
    """numpy views of one (layer, role) of a cache byte buffer."""

    def __init__(self, cfg: Config, buf: np.ndarray, layer: int, role: int):
        lay = layout(cfg)
        B, H, D, S, W = cfg.batch, cfg.num_kv_heads, cfg.head_dim, cfg.sink, cfg.recent
        base = layer * lay["layer_bytes"] + role * lay["role_bytes"]
        ncap = lay["ncap"]
        o = base
        self.full = None
        if role == 1 and cfg.flags & FLAG_V_BF16:
            cap = cfg.capacity
            self.full = buf[o:o + B * H * cap * D * 2].view(np.uint16).reshape(B, H, cap, D)
            self.sink = self.ring = self.codes = self.sz = None
            return
        self.sink = buf[o:o + B * H * S * D * 2].view(np.uint16).reshape(B, H, S, D)
        o += lay["sink_bytes"]
        self.ring = buf[o:o + B * H * W * D * 2].view(np.uint16).reshape(B, H, W, D)
        o += lay["ring_bytes"]
        self.codes = buf[o:o + B * H * ncap * D // 4].reshape(B, H, ncap, D // 4)
        o += lay["codes_bytes"]
        self.sz = buf[o:o + B * H * ncap * (D // GROUP) * 4].view(np.float16).reshape(
            B, H, ncap, D // GROUP, 2)


def new_cache(cfg: Config) -> np.ndarray:
    return np.zeros(layout(cfg)["total_bytes"], dtype=np.uint8)


# --------------------------------------------------------------------------
# append
# --------------------------------------------------------------------------
def append(cfg: Config, cache: np.ndarray, layer: int, k_new: np.ndarray, v_new: np.ndarray,
           start_pos, R_K: np.ndarray, R_V: np.ndarray, return_rot: bool = False):
    """Write n new tokens per sequence at positions start_pos[b] .. +n-1.

    k_new, v_new: [B][n][Hkv][D] float (bf16 values as float32, or float32).
    R_K, R_V: [D][D] rotations of this layer (ignored with FLAG_HADAMARD,
    which rotates both by :func:`hadamard_rotation`).  Every position p >= S gets its
    INT2 row; p < S also goes to the BF16 sink; p >= start_pos[b] + n - W also
    goes to the BF16 ring slot p mod W.  With FLAG_V_BF16 the V row of every
    position goes to the V role's BF16 row p instead.  Positions outside
    [0, capacity) are not stored.
    """
    B, n, H, D = k_new.shape
    S, W, cap = cfg.sink, cfg.recent, cfg.capacity
    R_K, R_V = rotations_of(cfg, R_K, R_V)
    rots = []
    for role, (x, R, ratio) in enumerate(((k_new, R_K, cfg.k_clip), (v_new, R_V, cfg.v_clip))):
        view = CacheView(cfg, cache, layer, role)
        r = rotate_rows(np.asarray(x, np.float32).reshape(-1, D), R).reshape(B, n, H, D)
        rots.append(r)
        codes, scale, zero = quantize_rows(r.reshape(-1, D), ratio, bool(cfg.flags & FLAG_LLOYD_MAX))
        packed = pack_codes(codes, role).reshape(B, n, H, D // 4)
        scale = scale.reshape(B, n, H, -1)
        zero = zero.reshape(B, n, H, -1)
        rb = f32_to_bf16_bits(r.reshape(-1, D)).reshape(B, n, H, D)
        for b in range(B):
            newlen = int(start_pos[b]) + n
            for t in range(n):
                p = int(start_pos[b]) + t
                if p < 0 or p >= cap:
                    continue  # outside the cache: not stored
                if view.full is not None:
                    view.full[b, :, p, :] = rb[b, t]  # V kept BF16 at every position
                    continue
                if p < S:
                    view.sink[b, :, p, :] = rb[b, t]
                else:
                    view.codes[b, :, p - S, :] = packed[b, t]
                    view.sz[b, :, p - S, :, 0] = scale[b, t]
                    view.sz[b, :, p - S, :, 1] = zero[b, t]
                if W > 0 and p >= newlen - W:
                    view.ring[b, :, p % W, :] = rb[b, t]
    if return_rot:
        return rots[0], rots[1]
    return None


# --------------------------------------------------------------------------
# decode
# --------------------------------------------------------------------------
def regions(T: int, S: int, W: int):
    """(n_sink, Tq, n_int2, n_ring): sink [0, n_sink), INT2 [S, Tq), ring [Tq, T)."""
    if T <= S:
        return T, T, 0, 0
    tq = max(S, T - W)
    return S, tq, tq - S, T - tq


def dequant_history(cfg: Config, cache: np.ndarray, layer: int, role: int, b: int, h: int, T: int):
    """[T, D] float64 values the decode attends to for one (b, kv head)."""
    view = CacheView(cfg, cache, layer, role)
    if view.full is not None:
        return bf16_bits_to_f32(view.full[b, h, :T]).astype(np.float64)
    D, S, W = cfg.head_dim, cfg.sink, cfg.recent
    n_sink, tq, n_int, n_ring = regions(T, S, W)
    out = np.zeros((T, D), dtype=np.float64)
    if n_sink:
        out[:n_sink] = bf16_bits_to_f32(view.sink[b, h, :n_sink])
    if n_int:
        codes = unpack_codes(view.codes[b, h, :n_int], D, role)
        sc = view.sz[b, h, :n_int, :, 0]
        ze = view.sz[b, h, :n_int, :, 1]
        out[S:tq] = dequantize_rows(codes, sc, ze, bool(cfg.flags & FLAG_LLOYD_MAX))
    for p in range(tq, T):
        out[p] = bf16_bits_to_f32(view.ring[b, h, p % W])
    return out


def decode(cfg: Config, cache: np.ndarray, layer: int, q: np.ndarray, seq_lens, R_K: np.ndarray,
           R_V: np.ndarray, sm_scale: float = 0.0, absorb_v: bool = False):
    """One decode step of attention over the mixed cache, float64.

    q: [B][Hq][D] (bf16 values as float).  Query head i reads KV head i // G.
    Returns (out [B][Hq][D] float64, lse [B][Hq] float64 natural log).
    """
    B, Hq, D = q.shape
    G = cfg.G
    scale = sm_scale if sm_scale > 0 else 1.0 / math.sqrt(D)
    R_K, R_V = rotations_of(cfg, R_K, R_V)
    RK = np.asarray(R_K, np.float64)
    RV = np.asarray(R_V, np.float64)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    for b in range(B):
        T = int(seq_lens[b])
        for h in range(cfg.num_kv_heads):
            K = dequant_history(cfg, cache, layer, 0, b, h, T)
            V = dequant_history(cfg, cache, layer, 1, b, h, T)
            for i in range(h * G, (h + 1) * G):
                qr = np.asarray(q[b, i], np.float64) @ RK
                s = scale * (K @ qr)
                m = s.max()
                e = np.exp(s - m)
                l = e.sum()
                o_rot = (e @ V) / l
                out[b, i] = o_rot if absorb_v else o_rot @ RV.T
                lse[b, i] = m + math.log(l)
    return out, lse
