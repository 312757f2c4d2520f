"""attn_decode_static: the decode entry point for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).

Checked through the C ABI: two calls in a row give the same output and lse as
attn_decode with a caller-provided workspace, within the decode tolerances used
elsewhere; a configuration whose smallest decode needs more scratch than the
array holds is rejected before anything is launched.  This file is collected
last so that a failure here does not hide the other tests' results."""
import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S
from oracle import oscar_oracle as O
from tests.gpu_helpers import kcfg, rel_l2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs CUDA")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_kv_cache_append_gb300 import build
    build.build()


def test_static_scratch_matches_workspace_entry_point_twice():
    D, B, Hq, Hkv, S_, W = 128, 3, 16, 4, 64, 128
    lens = [2500, 1900, 777]
    c = O.Config(1, B, Hq, Hkv, D, S_, W, 2600, 0.96, 0.92, flags=K.FLAG_OUT_FP32)
    rng = np.random.default_rng(21)
    ch = rng.choice(D, 3, replace=False)
    RK = S.qr_rotation(rng, D).astype(np.float32)
    RV = S.qr_rotation(rng, D).astype(np.float32)
    k = S.to_bf16_values(S.activations(rng, (B, max(lens), Hkv, D), ch))
    v = S.to_bf16_values(S.activations(rng, (B, max(lens), Hkv, D), ch))
    q = S.to_bf16_values(S.activations(rng, (B, Hq, D), ch))
    ocache = O.new_cache(c)
    O.append(c, ocache, 0, k, v, [0] * B, RK, RV)

    kc = kcfg(c)
    cache = torch.from_numpy(ocache).cuda()
    qt = torch.from_numpy(q).to(torch.bfloat16).cuda()
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    rk, rv = torch.from_numpy(RK).cuda(), torch.from_numpy(RV).cuda()
    lay = K.layout_query(kc)
    ws = torch.empty(lay["decode_workspace_bytes"], dtype=torch.uint8, device="cuda")
    ref = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    ref_lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    K.attn_decode(kc, cache, 0, qt, seq, rk, rv, ref, ws, lse=ref_lse, seq_len_hint=max(lens))
    torch.cuda.synchronize()
    ref_np, ref_lse_np = ref.cpu().numpy().astype(np.float64), ref_lse.cpu().numpy().astype(np.float64)

    for _ in range(2):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = K.attn_decode_static(kc, cache, 0, qt, seq, rk, rv, out, lse=lse, seq_len_hint=max(lens), status=st)
        torch.cuda.synchronize()
        assert rc == 0 and int(st.item()) == 0
        o = out.cpu().numpy().astype(np.float64)
        l = lse.cpu().numpy().astype(np.float64)
        assert np.isfinite(o).all() and np.isfinite(l).all()
        assert rel_l2(o, ref_np) <= 2e-4 and np.abs(o - ref_np).max() <= 5e-3
        assert np.max(np.abs(l - ref_lse_np) - 1e-5 * np.abs(ref_lse_np)) <= 1e-4


def test_static_scratch_rejects_oversized_decode():
    import ctypes
    # B * Hq = 65536 heads of D = 128: one split alone needs > 64 MiB of scratch.
    # Every pointer is NULL: the size check comes first, so a regression in it
    # fails on the host instead of launching on buffers that do not exist.
    kc = K.KVConfig(1, 1024, 64, 8, 128, 0, 0, 64)
    assert K.STATIC_SCRATCH_BYTES == 16 << 20
    rc = K.lib().attn_decode_static(ctypes.byref(kc.c()), None, 0, None, None, 0, None, None, 0.0, 0, None, None,
                                    None, None)
    assert rc == -3
    # an explicit split count that does not fit is rejected too; the buffers
    # are the sizes this configuration needs, so a regression that launched
    # anyway would still stay inside them
    kc = K.KVConfig(1, 64, 32, 8, 128, 0, 0, 64)
    lay = K.layout_query(kc)
    cache = torch.zeros(lay["total_bytes"], dtype=torch.uint8, device="cuda")
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    seq = torch.full((64,), 64, dtype=torch.int32, device="cuda")
    eye = torch.eye(128, dtype=torch.float32, device="cuda")
    rc = K.attn_decode_static(kc, cache, 0, q, seq, eye, eye, out, num_splits=64, check=False)
    assert rc == -3
