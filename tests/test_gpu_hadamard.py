"""GPU parity of the data-free in-quant Hadamard (FLAG_HADAMARD).

Append: the GPU's rotated rows (its debug output) are within 2e-6 of the
float64 product with the oracle's block-diagonal Hadamard, and the cache bytes
equal, bit for bit, what the oracle's codec writes for those same float32 rows
(appended to an oracle cache with R = I, which leaves them unchanged).  Decode:
outputs against the oracle on identical cache bytes, with the tolerances of the
calibrated-rotation decode tests.  decode_step with the flag agrees with
kv_append followed by attn_decode (assert_same_decode; the output transform
here is the warp Hadamard, the same in every merging CTA).  No rotation matrix
is passed anywhere."""
import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S
from oracle import oscar_oracle as O
from tests.gpu_helpers import assert_same_decode, bf16_round64, gpu_append, gpu_decode, new_cache, rel_l2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs CUDA")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_kv_cache_append_gb300 import build
    build.build()


def _inputs(seed, B, n, H, D, fp32=False):
    rng = np.random.default_rng(seed)
    ch = rng.choice(D, size=max(1, D // 50), replace=False)
    k = S.activations(rng, (B, n, H, D), ch)
    v = S.activations(rng, (B, n, H, D), ch)
    if not fp32:
        k, v = S.to_bf16_values(k), S.to_bf16_values(v)
    return k, v


APPEND_CASES = [
    # D, B, Hkv, S, W, cap, chunks (n per call), start offsets per sequence;
    # rows per call <= 512 and > 512 reach both row-parallel variants
    (128, 2, 2, 16, 32, 256, [40, 1, 7, 64], [0, 3]),
    (128, 2, 4, 16, 64, 400, [100, 1, 50], [0, 2]),
    (128, 1, 8, 4, 8, 2100, [1500, 3], [0]),
    (256, 2, 2, 5, 9, 200, [33, 17, 2], [1, 0]),
    (512, 2, 2, 8, 16, 160, [50, 31, 1], [0, 7]),
]


@pytest.mark.parametrize("case", APPEND_CASES)
@pytest.mark.parametrize("fp32", [False, True])
def test_hadamard_append(case, fp32):
    D, B, H, S_, W, cap, chunks, offs = case
    c = O.Config(1, B, 2 * H, H, D, S_, W, cap, 0.96, 0.92,
                 flags=K.FLAG_HADAMARD | (K.FLAG_IN_FP32 if fp32 else 0))
    plain = O.Config(1, B, 2 * H, H, D, S_, W, cap, 0.96, 0.92)
    Hm = O.hadamard_rotation(D)
    eye = np.eye(D, dtype=np.float32)
    ocache, gcache = O.new_cache(plain), new_cache(c)
    pos = list(offs)
    for i, n in enumerate(chunks):
        k, v = _inputs(300 + i, B, n, H, D, fp32)
        rot = gpu_append(c, gcache, 0, k, v, pos, None, None, want_rot=True).cpu().numpy()
        for role, x in enumerate((k, v)):
            exact = x.astype(np.float64) @ Hm
            assert np.abs(rot[:, :, :, role] - exact).max() <= 2e-6 * np.abs(exact).max()
        O.append(plain, ocache, 0, rot[:, :, :, 0], rot[:, :, :, 1], pos, eye, eye)
        pos = [p + n for p in pos]
    got = gcache.cpu().numpy()
    diff = np.nonzero(got != ocache)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


DEC_CASES = [
    # D, B, Hq, Hkv, S, W, seq_lens, extra flags
    (128, 1, 4, 1, 64, 256, [1024], 0),
    (128, 2, 8, 2, 16, 32, [700, 333], 0),                 # ragged
    (128, 2, 16, 2, 0, 100, [1500, 900], 0),               # S = 0, G = 8
    (128, 2, 4, 2, 64, 256, [200, 64], 0),                 # S + W >= T: all BF16
    (128, 1, 16, 8, 64, 256, [3000], K.FLAG_ABSORB_V),     # G = 2, output in the Hadamard basis
    (128, 2, 8, 2, 32, 64, [800, 257], K.FLAG_IN_FP32),    # float32 q, k, v: qrot transforms float32 rows
    (256, 2, 8, 2, 8, 16, [400, 150], 0),
    (512, 1, 4, 2, 16, 64, [600], 0),
]


@pytest.mark.parametrize("case", DEC_CASES)
def test_hadamard_decode(case):
    D, B, Hq, Hkv, S_, W, seq_lens, extra = case
    c = O.Config(1, B, Hq, Hkv, D, S_, W, max(seq_lens), 0.96, 0.92, flags=K.FLAG_HADAMARD | extra)
    rng = np.random.default_rng(D + B + Hq)
    ch = rng.choice(D, max(1, round(0.02 * D)), replace=False)
    T = max(seq_lens)
    k = S.activations(rng, (B, T, Hkv, D), ch)
    v = S.activations(rng, (B, T, Hkv, D), ch)
    q = S.activations(rng, (B, Hq, D), ch)
    if not extra & K.FLAG_IN_FP32:
        k, v, q = S.to_bf16_values(k), S.to_bf16_values(v), S.to_bf16_values(q)
    cache = O.new_cache(c)
    O.append(c, cache, 0, k, v, [0] * B, None, None)
    ref, ref_lse = O.decode(c, cache, 0, q, seq_lens, None, None, absorb_v=bool(extra & K.FLAG_ABSORB_V))
    gc = torch.from_numpy(cache).cuda()
    o16, lse = gpu_decode(c, gc, 0, q, seq_lens, None, None, out_fp32=False)
    o32, lse32 = gpu_decode(c, gc, 0, q, seq_lens, None, None, out_fp32=True)
    r16, r32 = rel_l2(o16, bf16_round64(ref)), rel_l2(o32, ref)
    m32 = float(np.abs(o32 - ref).max())
    dl = float(np.max(np.abs(lse - ref_lse) - 1e-5 * np.abs(ref_lse)))
    assert r16 <= 1e-3, f"bf16 rel-L2 {r16}"
    assert m32 <= 5e-3 and r32 <= 2e-4, f"fp32 max-abs {m32} rel-L2 {r32}"
    assert dl <= 1e-4, f"lse {dl}"
    assert np.array_equal(lse, lse32)


@pytest.mark.parametrize("case", [(128, 2, 32, 8, 64, 256, 4096, [4000, 777], 1),
                                  (256, 2, 8, 4, 16, 32, 700, [650, 90], 3)])
def test_hadamard_decode_step_equals_append_then_decode(case):
    D, B, Hq, Hkv, S_, W, cap, pre, n = case
    kc = K.KVConfig(1, B, Hq, Hkv, D, S_, W, cap, 0.96, 0.92, K.FLAG_OUT_FP32 | K.FLAG_HADAMARD)
    lay = K.layout_query(kc)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2000 + D + n)
    ch = np.array([5, 77])
    rand = lambda shape: S.activations_torch(gen, shape, ch, dtype=torch.bfloat16)
    cache = torch.zeros(lay["total_bytes"], dtype=torch.uint8, device="cuda")
    T0 = max(pre)
    K.kv_append(kc, cache, 0, rand((B, T0, Hkv, D)), rand((B, T0, Hkv, D)),
                torch.zeros(B, dtype=torch.int32, device="cuda"), None, None)
    k_new, v_new, q = rand((B, n, Hkv, D)), rand((B, n, Hkv, D)), rand((B, Hq, D))
    start = torch.tensor(pre, dtype=torch.int32, device="cuda")
    seq = start + n
    results = []
    for fused in (False, True):
        c = cache.clone()
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
        ws = torch.empty(lay["decode_workspace_bytes"], dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            K.decode_step(kc, c, 0, k_new, v_new, start, q, seq, None, None, out, ws, lse=lse, seq_len_hint=cap,
                          status=st)
        else:
            K.kv_append(kc, c, 0, k_new, v_new, start, None, None, status=st)
            K.attn_decode(kc, c, 0, q, seq, None, None, out, ws, lse=lse, seq_len_hint=cap, status=st)
        torch.cuda.synchronize()
        results.append((c.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy(), int(st.item())))
    (c0, o0, l0, s0), (c1, o1, l1, s1) = results
    assert s0 == s1 == 0
    assert np.array_equal(c0, c1)
    assert np.isfinite(o0).all()
    assert_same_decode(o0, o1, l0, l1)


@pytest.mark.parametrize("D", [128, 512])
@pytest.mark.parametrize("splits", [4, 16])
def test_hadamard_decode_merge_paths(D, splits):
    # the last CTA's merge applies H whether 4 or 16 CTAs share a unit
    B, Hq, Hkv, T = 2, 8, 2, 1900
    c = O.Config(1, B, Hq, Hkv, D, 16, 64, T, 0.96, 0.92, flags=K.FLAG_HADAMARD)
    rng = np.random.default_rng(D + splits)
    ch = rng.choice(D, max(1, round(0.02 * D)), replace=False)
    k = S.to_bf16_values(S.activations(rng, (B, T, Hkv, D), ch))
    v = S.to_bf16_values(S.activations(rng, (B, T, Hkv, D), ch))
    q = S.to_bf16_values(S.activations(rng, (B, Hq, D), ch))
    lens = [T, 1100]
    cache = O.new_cache(c)
    O.append(c, cache, 0, k, v, [0] * B, None, None)
    ref, ref_lse = O.decode(c, cache, 0, q, lens, None, None)
    gc = torch.from_numpy(cache).cuda()
    o32, lse32 = gpu_decode(c, gc, 0, q, lens, None, None, out_fp32=True, num_splits=splits)
    r32, m32 = rel_l2(o32, ref), float(np.abs(o32 - ref).max())
    dl = float(np.max(np.abs(lse32 - ref_lse) - 1e-5 * np.abs(ref_lse)))
    assert m32 <= 5e-3 and r32 <= 2e-4, f"fp32 max-abs {m32} rel-L2 {r32}"
    assert dl <= 1e-4, f"lse {dl}"
