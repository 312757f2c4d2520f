"""GPU parity over seeded random configurations of the whole path.

Each case draws, from its seed alone: head_dim, the GQA shape (G = 1..8),
batch, sink and ring sizes, the mode flags (absorbed V, V kept BF16, Lloyd-Max
levels, float32 inputs), how the rows are appended (one to three kv_append
calls of different sizes, a start offset per sequence), the decode lengths
(empty sequences, lengths inside the BF16 windows, full lengths), the split
count, the layer of a multi-layer cache, the softmax scale, the workspace size
(one to five partial slots or the default) and the length hint.  The
rotations are exact signed permutations, so every rotated value, and hence the
cache, is exact on both sides:

  * the GPU cache after the kv_append calls equals the oracle's byte for byte;
  * attn_decode of those bytes agrees with the oracle's decode within the
    tolerances of the decode tests (float32 output max-abs <= 5e-3, rel-L2
    <= 2e-4; lse within 1e-4 + 1e-5 |lse|), and its bf16 output is the float32
    output rounded to nearest (see _compare);
  * decode_step (one more append of 1..6 tokens fused with the decode) leaves
    the oracle's cache bytes, agrees with the oracle's append + decode within
    the same tolerances, and gives the same output and lse bits as kv_append
    followed by attn_decode (it streams the blocks the append leaves alone
    before the append completes, so a block read too early would show).

The in-quant Hadamard is not an exact rotation in float32, so its cases decode
the oracle's cache bytes on both sides instead (the Hadamard tests check its
append on the GPU's own rotated rows).

OSCAR_SWEEP_SEEDS=a-b runs every test of this file over seeds a to b - 1
instead of the committed ones, e.g. for a long stress run."""
import os

import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S
from oracle import oscar_oracle as O
from tests.gpu_helpers import (assert_same_decode, bf16_round64, dev, dev_i32, dev_rot, gpu_append, gpu_decode, kcfg,
                               new_cache, rel_l2, workspace_bytes)

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs CUDA")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_kv_cache_append_gb300 import build
    build.build()


def draw(seed: int, hadamard: bool = False) -> dict:
    """One random configuration, a pure function of the seed."""
    r = np.random.default_rng(seed)
    D = int(r.choice([128, 128, 128, 256, 512]))
    G = int(r.choice([1, 2, 4, 8]))
    Hkv = int(r.choice([1, 2, 4])) if D == 128 else int(r.choice([1, 2]))
    B = int(r.integers(1, 5))
    S_ = int(r.choice([0, 8, 16, 64]))
    W = int(r.choice([16, 64, 256])) if S_ == 0 else int(r.choice([0, 16, 64, 256]))
    flags = K.FLAG_HADAMARD if hadamard else 0
    for f, p in ((K.FLAG_ABSORB_V, 0.3), (K.FLAG_V_BF16, 0.25), (K.FLAG_LLOYD_MAX, 0.25), (K.FLAG_IN_FP32, 0.3)):
        if r.random() < p:
            flags |= f
    total = int(r.integers(1, 2500 if D == 128 else 1200))  # rows appended per sequence
    nch = int(r.integers(1, 4))
    cuts = sorted(set(int(x) for x in r.integers(1, total, nch - 1))) if total > 1 else []
    chunks = [b - a for a, b in zip([0] + cuts, cuts + [total])]
    offs = [int(x) for x in r.integers(0, 40, B)]
    n_step = int(r.integers(1, 7))
    cap = max(offs) + total + n_step + int(r.integers(0, 50))
    lens = []
    for b in range(B):
        end = offs[b] + total
        kind = r.integers(0, 4)
        lens.append(0 if kind == 0 else (int(r.integers(1, end + 1)) if kind == 1 else end))
    splits = int(r.choice([0, 0, 0, 1, 3, 9]))
    layers = int(r.integers(1, 4))
    layer = int(r.integers(0, layers))
    sm_scale = float(r.uniform(0.02, 0.2)) if r.random() < 0.3 else 0.0
    slots = int(r.integers(1, 6)) if r.random() < 0.25 else 0  # a workspace of this many partial slots
    if slots:
        splits = min(splits, slots)
    hint = int(r.choice([0, cap, max(1, cap // 3)]))
    return dict(D=D, Hq=G * Hkv, Hkv=Hkv, B=B, S=S_, W=W, flags=flags, chunks=chunks, offs=offs, cap=cap,
                lens=lens, splits=splits, n_step=n_step, layers=layers, layer=layer, sm_scale=sm_scale,
                slots=slots, hint=hint, seed=seed)


def _rows(rng, shape, ch, fp32):
    x = S.activations(rng, shape, ch)
    return x if fp32 else S.to_bf16_values(x)


def _oracle_decode(c, cache, q, lens, RK, RV, absorb, layer=0, sm_scale=0.0):
    """The oracle's decode; an empty sequence has its defined output (zeros,
    lse = -inf), which the oracle does not evaluate."""
    ref, ref_lse = O.decode(c, cache, layer, q, [max(1, t) for t in lens], RK, RV, sm_scale=sm_scale,
                            absorb_v=absorb)
    for b, t in enumerate(lens):
        if t == 0:
            ref[b] = 0.0
            ref_lse[b] = -np.inf
    return ref, ref_lse


def _compare(c, ref, ref_lse, o16, o32, lse, lse32, what):
    """The float32 output against the oracle within the decode tests'
    tolerances.  The bf16 output is the same float32 result rounded to nearest
    (one computation, two stores): it must equal that rounding bit for bit, and
    so lies within the bf16 unit roundoff (2^-8 relative per element: 8
    significant bits, rounding to nearest) plus the float32 tolerance of the
    oracle.  (Comparing it with the oracle rounded to
    bf16 instead fails where an output sits on a bf16 rounding tie: a
    dequantized INT2 value has fp16 precision, so one-hot attention puts about
    one output in eight exactly on a tie, where float32 noise decides the
    rounding direction.)"""
    r32 = rel_l2(o32, ref)
    m32 = float(np.abs(o32 - ref).max()) if ref.size else 0.0
    assert m32 <= 5e-3 and r32 <= 2e-4, f"{what}: fp32 max-abs {m32} rel-L2 {r32}"
    same = o16 == bf16_round64(o32)
    assert same.all(), f"{what}: bf16 output differs from the rounded float32 output at {np.argwhere(~same)[:4].tolist()}"
    r16 = rel_l2(o16, ref)
    assert r16 <= 2.0 ** -8 + 2e-4, f"{what}: bf16 rel-L2 {r16}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: empty sequences differ"
    dl = float(np.max(np.abs(lse[fin] - ref_lse[fin]) - 1e-5 * np.abs(ref_lse[fin]))) if fin.any() else 0.0
    assert dl <= 1e-4, f"{what}: lse {dl}"
    assert np.array_equal(lse, lse32), f"{what}: lse depends on the output type"


def _seeds(default):
    """The committed seeds, or those of OSCAR_SWEEP_SEEDS ("a-b": seeds a to
    b - 1, every test of this file) for a longer stress run."""
    spec = os.environ.get("OSCAR_SWEEP_SEEDS", "")
    if spec:
        a, b = (int(x) for x in spec.split("-"))
        return list(range(a, b))
    return list(default)


SEEDS = _seeds(range(48))


def _config(p):
    return O.Config(p["layers"], p["B"], p["Hq"], p["Hkv"], p["D"], p["S"], p["W"], p["cap"], 0.96, 0.92,
                    flags=p["flags"])


def _gpu_decode(c, p, cache, q, lens, RK, RV, out_fp32):
    ws = workspace_bytes(c, p["slots"]) if p["slots"] else None
    return gpu_decode(c, cache, p["layer"], q, lens, RK, RV, sm_scale=p["sm_scale"], num_splits=p["splits"],
                      hint=p["hint"], out_fp32=out_fp32, ws_bytes=ws)


@pytest.mark.parametrize("seed", SEEDS)
def test_sweep_chain(seed):
    p = draw(seed)
    D, B, Hq, Hkv, L = p["D"], p["B"], p["Hq"], p["Hkv"], p["layer"]
    c = _config(p)
    fp32 = bool(p["flags"] & K.FLAG_IN_FP32)
    absorb = bool(p["flags"] & K.FLAG_ABSORB_V)
    rng = np.random.default_rng(1000 + seed)
    RK = S.signed_permutation(rng, D).astype(np.float32)
    RV = S.signed_permutation(rng, D).astype(np.float32)
    ch = rng.choice(D, max(1, round(0.02 * D)), replace=False)

    # appends: the same rows through the oracle and the GPU
    ocache, gcache = O.new_cache(c), new_cache(c)
    pos = list(p["offs"])
    for n in p["chunks"]:
        k, v = _rows(rng, (B, n, Hkv, D), ch, fp32), _rows(rng, (B, n, Hkv, D), ch, fp32)
        O.append(c, ocache, L, k, v, pos, RK, RV)
        gpu_append(c, gcache, L, k, v, pos, RK, RV)
        pos = [x + n for x in pos]
    got = gcache.cpu().numpy()
    diff = np.nonzero(got != ocache)[0]
    assert diff.size == 0, f"{p}: {diff.size} cache bytes differ, first at {diff[:8]}"

    # decode of those bytes
    q = _rows(rng, (B, Hq, D), ch, fp32)
    ref, ref_lse = _oracle_decode(c, ocache, q, p["lens"], RK, RV, absorb, L, p["sm_scale"])
    o16, lse = _gpu_decode(c, p, gcache, q, p["lens"], RK, RV, False)
    o32, lse32 = _gpu_decode(c, p, gcache, q, p["lens"], RK, RV, True)
    _compare(c, ref, ref_lse, o16, o32, lse, lse32, f"attn_decode {p}")

    # decode_step: n_step more rows at each sequence's end, then the decode of
    # the new lengths, in one call
    n = p["n_step"]
    k, v = _rows(rng, (B, n, Hkv, D), ch, fp32), _rows(rng, (B, n, Hkv, D), ch, fp32)
    q = _rows(rng, (B, Hq, D), ch, fp32)
    lens = [x + n for x in pos]
    O.append(c, ocache, L, k, v, pos, RK, RV)
    ref, ref_lse = _oracle_decode(c, ocache, q, lens, RK, RV, absorb, L, p["sm_scale"])
    kc = kcfg(c)
    lay = K.layout_query(kc)
    dt = torch.float32 if fp32 else torch.bfloat16
    outs = []
    for out_fp32 in (False, True):
        kc.flags = (c.flags & ~K.FLAG_OUT_FP32) | (K.FLAG_OUT_FP32 if out_fp32 else 0)
        res = []
        for fused in (True, False):
            gc = gcache.clone()
            out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                             device="cuda")
            lse_t = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
            ws = torch.empty(workspace_bytes(c, p["slots"]) if p["slots"] else lay["decode_workspace_bytes"],
                             dtype=torch.uint8, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            new_rows = (dev(k, dt), dev(v, dt), dev_i32(pos))
            dec = dict(lse=lse_t, seq_len_hint=p["hint"], sm_scale=p["sm_scale"], num_splits=p["splits"], status=st)
            if fused:
                K.decode_step(kc, gc, L, *new_rows, dev(q, dt), dev_i32(lens), dev_rot(RK), dev_rot(RV), out, ws, **dec)
            else:
                K.kv_append(kc, gc, L, *new_rows, dev_rot(RK), dev_rot(RV), status=st)
                K.attn_decode(kc, gc, L, dev(q, dt), dev_i32(lens), dev_rot(RK), dev_rot(RV), out, ws, **dec)
            torch.cuda.synchronize()
            assert int(st.item()) == 0, f"{'decode_step' if fused else 'append + decode'} status {int(st.item())}"
            diff = np.nonzero(gc.cpu().numpy() != ocache)[0]
            assert diff.size == 0, f"{p}: fused {fused}: {diff.size} cache bytes differ, first at {diff[:8]}"
            res.append((out.float().cpu().numpy(), lse_t.cpu().numpy()))
        # the fused call streams blocks the append leaves alone before it completes:
        # it must read exactly what the sequential calls read
        (of, lf), (os_, ls) = res
        assert_same_decode(of, os_, lf, ls)
        outs.append((of.astype(np.float64), lf.astype(np.float64)))
    (o16, lse), (o32, lse32) = outs
    _compare(c, ref, ref_lse, o16, o32, lse, lse32, f"decode_step {p}")


@pytest.mark.parametrize("seed", _seeds(range(100, 112)))
def test_sweep_hadamard_decode(seed):
    p = draw(seed, hadamard=True)
    D, B, Hq, Hkv, L = p["D"], p["B"], p["Hq"], p["Hkv"], p["layer"]
    c = _config(p)
    fp32 = bool(p["flags"] & K.FLAG_IN_FP32)
    rng = np.random.default_rng(1000 + seed)
    ch = rng.choice(D, max(1, round(0.02 * D)), replace=False)
    cache = O.new_cache(c)
    pos = list(p["offs"])
    for n in p["chunks"]:
        k, v = _rows(rng, (B, n, Hkv, D), ch, fp32), _rows(rng, (B, n, Hkv, D), ch, fp32)
        O.append(c, cache, L, k, v, pos, None, None)
        pos = [x + n for x in pos]
    q = _rows(rng, (B, Hq, D), ch, fp32)
    ref, ref_lse = _oracle_decode(c, cache, q, p["lens"], None, None, bool(p["flags"] & K.FLAG_ABSORB_V), L,
                                  p["sm_scale"])
    gc = torch.from_numpy(cache).cuda()
    o16, lse = _gpu_decode(c, p, gc, q, p["lens"], None, None, False)
    o32, lse32 = _gpu_decode(c, p, gc, q, p["lens"], None, None, True)
    _compare(c, ref, ref_lse, o16, o32, lse, lse32, f"attn_decode {p}")


def draw_append(seed: int) -> dict:
    """One random append configuration (general rotations), a pure function of
    the seed: call sizes on both sides of the 1024-rows-per-role switch between
    the row-parallel (or sliced) and the tiled (or tensor-core) kernels."""
    r = np.random.default_rng(seed)
    D = int(r.choice([128, 128, 256, 512]))
    Hkv = int(r.choice([1, 2, 4, 8])) if D == 128 else int(r.choice([1, 2, 4]))
    B = int(r.integers(1, 5))
    S_ = int(r.choice([0, 8, 16, 64]))
    W = int(r.choice([0, 16, 64, 256])) if S_ > 0 else int(r.choice([16, 64, 256]))
    flags = 0
    for f, p in ((K.FLAG_IN_FP32, 0.4), (K.FLAG_LLOYD_MAX, 0.2), (K.FLAG_V_BF16, 0.2), (K.FLAG_HADAMARD, 0.2)):
        if r.random() < p:
            flags |= f
    chunks = []
    for _ in range(int(r.integers(1, 4))):
        if r.random() < 0.5:
            chunks.append(int(r.integers(1, max(2, 1024 // (B * Hkv)) + 1)))  # <= 1024 rows per role
        else:
            chunks.append(int(r.integers(1024 // (B * Hkv) + 1, 4200 // (B * Hkv) + 2)))
    offs = [int(x) for x in r.integers(0, 70, B)]
    cap = max(offs) + sum(chunks) + int(r.integers(0, 40))
    return dict(D=D, Hkv=Hkv, B=B, S=S_, W=W, flags=flags, chunks=chunks, offs=offs, cap=cap, seed=seed)


@pytest.mark.parametrize("seed", _seeds(range(200, 224)))
def test_sweep_append_codec_on_gpu_rows(seed):
    """General rotations (calibrated R_K, random orthogonal R_V, or the in-quant
    Hadamard).  The GPU's float32 rotation is checked against the float64
    product with the error bounds of a D-term float32 dot product: every
    element within gamma_D = D u (u = 2^-24) times sum_i |x_i R_ij| (the
    worst case of any summation order), and the root-mean-square error within
    2 sqrt(D) u times the root mean square of those sums (rounding errors that
    add as a random walk; a product in bf16 arithmetic would exceed it by four
    orders of magnitude).  The
    rows are not correctly rounded, so the codec is checked on the GPU's own
    rows: the oracle quantises the rows each call exports through
    debug_rot_out (identity rotation, no Hadamard) and the two caches must
    match byte for byte."""
    p = draw_append(seed)
    D, B, Hkv = p["D"], p["B"], p["Hkv"]
    had = bool(p["flags"] & K.FLAG_HADAMARD)
    c = O.Config(1, B, Hkv, Hkv, D, p["S"], p["W"], p["cap"], 0.96, 0.92, flags=p["flags"])
    plain = O.Config(1, B, Hkv, Hkv, D, p["S"], p["W"], p["cap"], 0.96, 0.92,
                     flags=p["flags"] & (K.FLAG_LLOYD_MAX | K.FLAG_V_BF16))
    fp32 = bool(p["flags"] & K.FLAG_IN_FP32)
    rng = np.random.default_rng(2000 + seed)
    ch = rng.choice(D, max(1, round(0.02 * D)), replace=False)
    if had:
        RK = RV = None
        Rk64 = Rv64 = O.hadamard_rotation(D)
    else:
        RK = S.eig_rotation(S.activations(rng, (2048, D), ch)).astype(np.float32)
        RV = S.qr_rotation(rng, D).astype(np.float32)
        Rk64, Rv64 = RK.astype(np.float64), RV.astype(np.float64)
    eye = np.eye(D, dtype=np.float32)
    ocache, gcache = O.new_cache(plain), new_cache(c)
    pos = list(p["offs"])
    for n in p["chunks"]:
        k, v = _rows(rng, (B, n, Hkv, D), ch, fp32), _rows(rng, (B, n, Hkv, D), ch, fp32)
        rot = gpu_append(c, gcache, 0, k, v, pos, RK, RV, want_rot=True).cpu().numpy()
        u = 2.0 ** -24
        for role, (x, R) in enumerate(((k, Rk64), (v, Rv64))):
            exact = x.astype(np.float64) @ R
            terms = np.abs(x.astype(np.float64)) @ np.abs(R)
            err = np.abs(rot[:, :, :, role] - exact)
            worst = float(np.max(err - D * u * terms))
            assert worst <= 1e-30, f"{p}: role {role} rotation error beyond gamma_D: {worst}"
            rms, rms_terms = float(np.sqrt(np.mean(err ** 2))), float(np.sqrt(np.mean(terms ** 2)))
            assert rms <= 2 * np.sqrt(D) * u * rms_terms, f"{p}: role {role} rotation rms error {rms} ({rms_terms})"
        O.append(plain, ocache, 0, rot[:, :, :, 0], rot[:, :, :, 1], pos, eye, eye)
        pos = [x + n for x in pos]
    got = gcache.cpu().numpy()
    diff = np.nonzero(got != ocache)[0]
    assert diff.size == 0, f"{p}: {diff.size} cache bytes differ, first at {diff[:8]}"
