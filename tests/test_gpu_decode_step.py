"""decode_step (append + decode in one call) against kv_append followed by
attn_decode: the same kernels on the same data, so outputs, lse, cache bytes and
status words must be identical bit for bit, whatever blocks the fused call
streams before the append completes and whichever CTA merges a unit
(assert_same_decode).  Cases cover one and several new tokens,
ring wrap, appends longer than the ring, new positions inside the sink, G = 8
and D = 256.  The oracle agreement of the sequential calls is covered by the
decode and append parity tests."""
import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S
from tests.gpu_helpers import assert_same_decode

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs CUDA")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_kv_cache_append_gb300 import build
    build.build()


CASES = [
    # D, B, Hq, Hkv, S, W, cap, prefilled lengths, n_new
    (128, 3, 16, 4, 16, 64, 1200, [500, 63, 1000], 1),
    (128, 2, 32, 8, 64, 256, 4096, [4000, 777], 5),
    (128, 2, 8, 2, 8, 16, 600, [100, 300], 40),       # append longer than the ring
    (128, 3, 8, 2, 32, 64, 400, [3, 31, 200], 2),     # new positions inside the sink
    (128, 1, 64, 8, 64, 256, 3000, [2500], 1),        # G = 8
    (256, 2, 8, 4, 16, 32, 700, [650, 90], 3),        # D = 256
]


def _rand(gen, shape, ch):
    return S.activations_torch(gen, shape, ch, dtype=torch.bfloat16)


@pytest.mark.parametrize("case", CASES)
def test_decode_step_equals_append_then_decode(case):
    D, B, Hq, Hkv, S_, W, cap, pre, n = case
    kc = K.KVConfig(1, B, Hq, Hkv, D, S_, W, cap, 0.96, 0.92, K.FLAG_OUT_FP32)
    lay = K.layout_query(kc)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + D + n)
    ch = np.array([5, 77])
    rng = np.random.default_rng(D + n)
    rk = torch.from_numpy(S.qr_rotation(rng, D).astype(np.float32)).cuda()
    rv = torch.from_numpy(S.qr_rotation(rng, D).astype(np.float32)).cuda()
    cache = torch.zeros(lay["total_bytes"], dtype=torch.uint8, device="cuda")
    T0 = max(pre)
    K.kv_append(kc, cache, 0, _rand(gen, (B, T0, Hkv, D), ch), _rand(gen, (B, T0, Hkv, D), ch),
                torch.zeros(B, dtype=torch.int32, device="cuda"), rk, rv)
    k_new, v_new = _rand(gen, (B, n, Hkv, D), ch), _rand(gen, (B, n, Hkv, D), ch)
    q = _rand(gen, (B, Hq, D), ch)
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
            K.decode_step(kc, c, 0, k_new, v_new, start, q, seq, rk, rv, out, ws, lse=lse, seq_len_hint=cap,
                          status=st)
        else:
            K.kv_append(kc, c, 0, k_new, v_new, start, rk, rv, status=st)
            K.attn_decode(kc, c, 0, q, seq, rk, rv, out, ws, lse=lse, seq_len_hint=cap, status=st)
        torch.cuda.synchronize()
        results.append((c.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy(), int(st.item())))
    (c0, o0, l0, s0), (c1, o1, l1, s1) = results
    assert s0 == s1 == 0
    assert np.array_equal(c0, c1)
    assert np.isfinite(o0).all()
    assert_same_decode(o0, o1, l0, l1)
