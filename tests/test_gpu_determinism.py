"""Repeated attn_decode calls on the same inputs: outputs and lse identical bit
for bit (assert_same_decode), although the CTA that merges a unit's partial
results (the last of the unit's CTAs to finish) changes from call to call.
Each case shares every unit among several CTAs and reaches both sources of R_V
at the merge: rows prefetched into shared memory (head_dim 128, a merging CTA
with no copy in flight) and rows read through L2; the un-rotation does the same
arithmetic in the same order from either."""
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


@pytest.mark.parametrize("case", [(128, 2, 32, 8, 64, 256, 4001, 0),
                                  (128, 2, 32, 8, 64, 256, 4001, K.FLAG_V_BF16),
                                  (128, 1, 64, 8, 64, 256, 8000, 0),
                                  (256, 2, 16, 4, 16, 64, 3000, 0)])
def test_repeated_decodes_are_bit_identical(case):
    D, B, Hq, Hkv, S_, W, T, extra = case
    kc = K.KVConfig(1, B, Hq, Hkv, D, S_, W, T, 0.96, 0.92, K.FLAG_OUT_FP32 | extra)
    lay = K.layout_query(kc)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5000 + D + Hq)
    ch = np.array([3, 70])
    rand = lambda shape: S.activations_torch(gen, shape, ch, dtype=torch.bfloat16)
    rng = np.random.default_rng(D + T)
    rk = torch.from_numpy(S.qr_rotation(rng, D).astype(np.float32)).cuda()
    rv = torch.from_numpy(S.qr_rotation(rng, D).astype(np.float32)).cuda()
    cache = torch.zeros(lay["total_bytes"], dtype=torch.uint8, device="cuda")
    K.kv_append(kc, cache, 0, rand((B, T, Hkv, D)), rand((B, T, Hkv, D)),
                torch.zeros(B, dtype=torch.int32, device="cuda"), rk, rv)
    q = rand((B, Hq, D))
    seq = torch.tensor([T] + [T - 777] * (B - 1), dtype=torch.int32, device="cuda")
    ws = torch.empty(lay["decode_workspace_bytes"], dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(24):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
        K.attn_decode(kc, cache, 0, q, seq, rk, rv, out, ws, lse=lse, seq_len_hint=T, status=st)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o0, l0 = outs[0][0].cpu().numpy(), outs[0][1].cpu().numpy()
    assert np.isfinite(o0).all()
    for o, l in outs[1:]:
        assert_same_decode(o0, o.cpu().numpy(), l0, l.cpu().numpy())
