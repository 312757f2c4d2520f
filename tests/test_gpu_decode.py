"""GPU parity: attn_decode against the oracle on identical cache bytes.

The oracle builds the cache (its own append) from seeded inputs; the same bytes
are uploaded and decoded on the GPU.  Tolerances (BF16 output compared with the
oracle's float64 result rounded to BF16; float32 output with the float64 result):
  rel-L2(bf16 out, bf16(oracle)) <= 1e-3
  max |fp32 out - oracle| <= 5e-3 and rel-L2 <= 2e-4
  |lse - oracle| <= 1e-4 + 1e-5 |oracle| (natural log; the scores of these
  heavy-tailed workloads reach ~1e2 and mma.sync accumulates in float32)."""
import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S
from oracle import oscar_oracle as O
from tests.gpu_helpers import bf16_round64, gpu_decode, rel_l2, workspace_bytes

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs CUDA")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_kv_cache_append_gb300 import build
    build.build()


def _build(c, seq_lens, seed, rot="oscar", act="t3", layer=0):
    D = c.head_dim
    rng = np.random.default_rng(seed)
    if rot == "oscar":
        calib = S.activations(rng, (2048, D), rng.choice(D, 3, replace=False), kind=act)
        RK = S.eig_rotation(calib).astype(np.float32)
        RV = S.qr_rotation(rng, D).astype(np.float32)
    elif rot == "identity":
        RK = RV = np.eye(D, dtype=np.float32)
    else:
        RK = S.qr_rotation(rng, D).astype(np.float32)
        RV = S.qr_rotation(rng, D).astype(np.float32)
    ch = rng.choice(D, max(1, round(0.02 * D)), replace=False)
    T = max(seq_lens)
    fp32 = bool(c.flags & K.FLAG_IN_FP32)
    k = S.activations(rng, (c.batch, T, c.num_kv_heads, D), ch, kind=act)
    v = S.activations(rng, (c.batch, T, c.num_kv_heads, D), ch, kind=act)
    q = S.activations(rng, (c.batch, c.num_q_heads, D), ch, kind=act)
    if not fp32:
        k, v, q = S.to_bf16_values(k), S.to_bf16_values(v), S.to_bf16_values(q)
    cache = O.new_cache(c)
    O.append(c, cache, layer, k, v, [0] * c.batch, RK, RV)
    return cache, q, RK, RV


def _check(c, cache, q, seq_lens, RK, RV, layer=0, num_splits=0, sm_scale=0.0, tol_fp32=2e-4):
    absorb = bool(c.flags & K.FLAG_ABSORB_V)
    ref, ref_lse = O.decode(c, cache, layer, q, seq_lens, RK, RV, sm_scale=sm_scale, absorb_v=absorb)
    gc = torch.from_numpy(cache).cuda()
    o16, lse = gpu_decode(c, gc, layer, q, seq_lens, RK, RV, sm_scale=sm_scale, num_splits=num_splits,
                          out_fp32=False)
    o32, lse32 = gpu_decode(c, gc, layer, q, seq_lens, RK, RV, sm_scale=sm_scale, num_splits=num_splits,
                            out_fp32=True)
    r16 = rel_l2(o16, bf16_round64(ref))
    r32 = rel_l2(o32, ref)
    m32 = float(np.abs(o32 - ref).max())
    dl = float(np.max(np.abs(lse - ref_lse) - 1e-5 * np.abs(ref_lse)))
    assert r16 <= 1e-3, f"bf16 rel-L2 {r16}"
    assert m32 <= 5e-3 and r32 <= tol_fp32, f"fp32 max-abs {m32} rel-L2 {r32}"
    assert dl <= 1e-4, f"lse {dl}"
    assert np.array_equal(lse, lse32)
    return r16, r32, m32


DEC_CASES = [
    # D, B, Hq, Hkv, S, W, seq_lens, flags
    (128, 1, 4, 1, 64, 256, [1024], 0),
    (128, 2, 8, 2, 16, 32, [700, 333], 0),                 # ragged
    (128, 2, 4, 2, 64, 256, [200, 64], 0),                 # S+W >= T: all BF16
    (128, 1, 8, 8, 512, 0, [2000], 0),                     # W = 0, G = 1
    (128, 2, 16, 2, 0, 100, [1500, 900], 0),               # S = 0, G = 8
    (128, 3, 6, 3, 20, 40, [30, 19, 1], 0),                # T <= S, T = 1
    (128, 1, 16, 8, 64, 256, [4000], K.FLAG_ABSORB_V),     # G = 2, absorbed V
    (256, 2, 8, 2, 32, 64, [900, 513], 0),
    (512, 1, 4, 2, 512, 256, [2300], 0),
    (512, 2, 16, 2, 8, 8, [333, 1000], 0),                 # D = 512, G = 8
]


@pytest.mark.parametrize("case", DEC_CASES)
def test_decode_parity(case):
    D, B, Hq, Hkv, S_, W, lens, flags = case
    c = O.Config(1, B, Hq, Hkv, D, S_, W, max(lens) + 37, 0.96, 0.92, flags=flags)
    cache, q, RK, RV = _build(c, lens, seed=D * 7 + B + Hq)
    _check(c, cache, q, lens, RK, RV)


def test_decode_tiny_fp32_inputs():
    w = S.WORKLOADS["tiny"]
    c = O.Config(1, 1, 4, 1, 128, 64, 256, 1024, 0.96, 0.92, flags=K.FLAG_IN_FP32)
    RK, RV = S.rotations(w, 0)
    k, v = S.kv_rows(w, 0, 1024)
    q = S.queries(w, 0)
    cache = O.new_cache(c)
    O.append(c, cache, 0, k, v, [0], RK, RV)
    _check(c, cache, q, [1024], RK, RV)


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_decode_split_counts_agree(splits):
    c = O.Config(1, 2, 8, 2, 128, 64, 128, 3000, 0.96, 0.92)
    lens = [2900, 1700]
    cache, q, RK, RV = _build(c, lens, seed=11)
    _check(c, cache, q, lens, RK, RV, num_splits=splits)


def test_decode_custom_scale_and_layer():
    c = O.Config(3, 1, 4, 2, 128, 16, 16, 400, 0.96, 0.92)
    cache, q, RK, RV = _build(c, [390], seed=12, layer=2)
    _check(c, cache, q, [390], RK, RV, layer=2, sm_scale=0.05)


def test_decode_constant_v_gives_constant():
    # Every V row is the same lattice row (values -1.5, -0.5, 0.5, 1.5 -> zero -1.5,
    # scale 1, codes 0..3, exact in INT2 and in BF16), V clip 1, R_V = I: the
    # output of every head is that row.
    D = 128
    c = O.Config(1, 1, 4, 1, D, 8, 8, 600, 0.96, 1.0)
    rng = np.random.default_rng(13)
    T = 500
    row = (-1.5 + (np.arange(D) % 4)).astype(np.float32)
    k = S.to_bf16_values(rng.standard_normal((1, T, 1, D)).astype(np.float32))
    v = np.broadcast_to(row, (1, T, 1, D)).copy()
    I = np.eye(D, dtype=np.float32)
    cache = O.new_cache(c)
    O.append(c, cache, 0, k, v, [0], I, I)
    q = S.to_bf16_values(rng.standard_normal((1, 4, D)).astype(np.float32))
    gc = torch.from_numpy(cache).cuda()
    o32, _ = gpu_decode(c, gc, 0, q, [T], I, I, out_fp32=True)
    ref, _ = O.decode(c, cache, 0, q, [T], I, I)
    assert np.abs(ref - row.astype(np.float64)).max() < 1e-12
    assert np.abs(o32 - row.astype(np.float64)).max() < 1e-5


def test_decode_empty_sequence_status():
    c = O.Config(1, 2, 4, 1, 128, 4, 4, 64)
    cache, q, RK, RV = _build(c, [10, 10], seed=14)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o32, lse = gpu_decode(c, torch.from_numpy(cache).cuda(), 0, q, [10, 0], RK, RV, out_fp32=True, status=st)
    assert int(st.item()) & K.DEV_EMPTY
    assert np.all(o32[1] == 0) and np.all(np.isneginf(lse[1]))
    ref, _ = O.decode(c, cache, 0, q[:1], [10], RK, RV)
    assert np.abs(o32[0] - ref[0]).max() < 5e-3


def _check_rows(c, cache, q, lens, RK, RV, **kw):
    """Decode with the given lengths; non-empty sequences against the oracle,
    empty ones against their defined output (zeros, lse = -inf, EMPTY flag)."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gc = torch.from_numpy(cache).cuda()
    o32, lse = gpu_decode(c, gc, 0, q, lens, RK, RV, out_fp32=True, status=st, **kw)
    ref, ref_lse = O.decode(c, cache, 0, q, [max(1, t) for t in lens], RK, RV)
    for b, t in enumerate(lens):
        if t == 0:
            assert np.all(o32[b] == 0) and np.all(np.isneginf(lse[b]))
            continue
        assert np.abs(o32[b] - ref[b]).max() <= 5e-3 and rel_l2(o32[b], ref[b]) <= 2e-4, b
        assert np.max(np.abs(lse[b] - ref_lse[b]) - 1e-5 * np.abs(ref_lse[b])) <= 1e-4, b
    assert bool(int(st.item()) & K.DEV_EMPTY) == (0 in lens)


def test_decode_ragged_batch_with_empty_and_full_sequences():
    # the work of all sequences is cut into equal slices: slices cross sequence
    # boundaries, skip empty sequences and cover one at full capacity
    cap = 1500
    c = O.Config(1, 6, 16, 4, 128, 16, 64, cap)
    lens = [0, 1, 300, cap, 17, 0]
    cache, q, RK, RV = _build(c, [cap], seed=31)
    _check_rows(c, cache, q, lens, RK, RV)


@pytest.mark.parametrize("slots", [1, 2, 3, 5])
def test_decode_small_workspace(slots):
    # fewer than 3 partial slots: slices are cut on unit boundaries; from 3 up
    # no unit may be shared by more CTAs than there are slots
    c = O.Config(1, 3, 8, 2, 128, 8, 32, 900)
    lens = [900, 0, 257]
    cache, q, RK, RV = _build(c, [900], seed=32 + slots)
    _check_rows(c, cache, q, lens, RK, RV, ws_bytes=workspace_bytes(c, slots))


def test_decode_many_units_per_cta():
    """Thousands of short sequences: each CTA's slice spans more units than one
    segment table holds, so the table is rebuilt in windows.  The cache is
    built on the GPU; the automatic decomposition is compared with one CTA per
    split (num_splits = 1) and sampled sequences with the oracle."""
    B, Hq, Hkv, D, S_, W, cap = 16384, 8, 2, 128, 4, 8, 40
    c = O.Config(1, B, Hq, Hkv, D, S_, W, cap)
    kc = K.KVConfig(1, B, Hq, Hkv, D, S_, W, cap, 0.96, 0.92)
    lay = K.layout_query(kc)
    cache = torch.zeros(lay["total_bytes"], dtype=torch.uint8, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(33)
    ch = np.array([3, 77])
    k = S.activations_torch(gen, (B, cap, Hkv, D), ch, dtype=torch.bfloat16)
    v = S.activations_torch(gen, (B, cap, Hkv, D), ch, dtype=torch.bfloat16)
    q = S.activations_torch(gen, (B, Hq, D), ch, dtype=torch.bfloat16)
    rng = np.random.default_rng(33)
    RK = S.qr_rotation(rng, D).astype(np.float32)
    RV = S.qr_rotation(rng, D).astype(np.float32)
    rk, rv = torch.from_numpy(RK).cuda(), torch.from_numpy(RV).cuda()
    K.kv_append(kc, cache, 0, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"), rk, rv)
    lens = rng.integers(0, cap + 1, B).astype(np.int32)
    lens[:4] = [0, 1, cap, 23]
    seq = torch.from_numpy(lens).cuda()
    outs = []
    for ns in (0, 1):
        out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        ws = torch.empty(lay["decode_workspace_bytes"], dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        kc2 = K.KVConfig(1, B, Hq, Hkv, D, S_, W, cap, 0.96, 0.92, K.FLAG_OUT_FP32)
        K.attn_decode(kc2, cache, 0, q, seq, rk, rv, out, ws, lse=lse, seq_len_hint=cap, num_splits=ns, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == K.DEV_EMPTY
        outs.append((out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)))
    # the two decompositions sum in different orders: each must be within the
    # decode tolerance of the oracle, so they are compared with that tolerance
    (o0, l0), (o1, l1) = outs
    assert np.abs(o0 - o1).max() <= 5e-3 and rel_l2(o0, o1) <= 2e-4
    fin = np.isfinite(l1)
    assert np.array_equal(np.isfinite(l0), fin)
    assert np.max(np.abs(l0[fin] - l1[fin]) - 1e-5 * np.abs(l1[fin])) <= 1e-4
    assert np.all(o0[lens == 0] == 0)
    for b in [1, 2, 3, int(np.argmax(lens))]:
        oc = O.Config(1, 1, Hq, Hkv, D, S_, W, cap)
        ocache = O.new_cache(oc)
        O.append(oc, ocache, 0, k[b:b + 1].float().cpu().numpy(), v[b:b + 1].float().cpu().numpy(), [0], RK, RV)
        ref, ref_lse = O.decode(oc, ocache, 0, q[b:b + 1].float().cpu().numpy(), [int(lens[b])], RK, RV)
        assert np.abs(o0[b] - ref[0]).max() <= 5e-3 and rel_l2(o0[b], ref[0]) <= 2e-4, b
        assert np.max(np.abs(l0[b] - ref_lse[0]) - 1e-5 * np.abs(ref_lse[0])) <= 1e-4, b


@pytest.mark.parametrize("D,flags", [(128, 0), (128, K.FLAG_ABSORB_V), (256, 0), (512, 0), (512, K.FLAG_ABSORB_V)])
@pytest.mark.parametrize("splits", [4, 16])
def test_decode_merge_paths(D, flags, splits):
    # With num_splits = n every (sequence, KV head) is shared by n CTAs whose
    # last merges the n partials; at head_dim 256 / 512 with V un-rotated it
    # leaves o' in workspace slot 0 and unrot_kernel applies R_V^T.  The result
    # must meet the oracle, and the kernel count must say whether unrot ran.
    c = O.Config(1, 2, 8, 2, D, 16, 64, 2600, 0.96, 0.92, flags=flags)
    lens = [2500, 1300]
    cache, q, RK, RV = _build(c, lens, seed=D + splits + flags)
    _check(c, cache, q, lens, RK, RV, num_splits=splits)
    from tests.gpu_helpers import kcfg
    assert K.decode_kernels(kcfg(c)) == 2 + (D >= 256 and not flags & K.FLAG_ABSORB_V)


@pytest.mark.parametrize("splits", [0, 4, 16])
def test_decode_g8_few_units(splits):
    # G = 8 with few (sequence, KV head) units: the merging CTA leaves o' in
    # slot 0 and unrot_kernel applies R_V^T (three kernels)
    c = O.Config(1, 1, 32, 4, 128, 16, 64, 3000, 0.96, 0.92)
    lens = [2900]
    cache, q, RK, RV = _build(c, lens, seed=80 + splits)
    _check(c, cache, q, lens, RK, RV, num_splits=splits)
    from tests.gpu_helpers import kcfg
    assert K.decode_kernels(kcfg(c)) == 3
