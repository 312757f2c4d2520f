"""The split kernel's bounded waits: when a barrier wait runs out the kernel
flags OSCAR_DEV_TIMEOUT, returns, and the context stays usable.

The wait is made to run out without faulting or hanging anything: a test hook
shortens the bound to 1 ms and has CTA 0's first copy expect 16 bytes more than
its copies deliver, so that barrier never completes while every copy lands.
The call must return with the status bit set; with the hook cleared, the next
decode on the same stream is correct and its status clean."""
import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S
from oracle import oscar_oracle as O
from tests.gpu_helpers import gpu_decode, rel_l2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs CUDA")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_kv_cache_append_gb300 import build
    build.build()


@pytest.mark.parametrize("D,Hq,Hkv,lens", [(128, 8, 2, [900, 400]), (512, 4, 2, [700, 300])])
def test_wait_timeout_sets_status_and_context_stays_usable(D, Hq, Hkv, lens):
    B = len(lens)
    c = O.Config(1, B, Hq, Hkv, D, 16, 32, max(lens) + 5, 0.96, 0.92, flags=K.FLAG_OUT_FP32)
    rng = np.random.default_rng(D + 3)
    RK = S.qr_rotation(rng, D).astype(np.float32)
    RV = S.qr_rotation(rng, D).astype(np.float32)
    ch = rng.choice(D, 3, replace=False)
    k = S.to_bf16_values(S.activations(rng, (B, max(lens), Hkv, D), ch))
    v = S.to_bf16_values(S.activations(rng, (B, max(lens), Hkv, D), ch))
    q = S.to_bf16_values(S.activations(rng, (B, Hq, D), ch))
    ocache = O.new_cache(c)
    O.append(c, ocache, 0, k, v, [0] * B, RK, RV)
    gcache = torch.from_numpy(ocache).cuda()

    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    K.set_wait_test(1_000_000, 16)
    try:
        gpu_decode(c, gcache, 0, q, lens, RK, RV, status=st)  # returns: the waits are bounded
    finally:
        K.set_wait_test(0, 0)
    assert int(st.item()) & K.DEV_TIMEOUT

    st.zero_()
    ref, _ = O.decode(c, ocache, 0, q, lens, RK, RV)
    out, _ = gpu_decode(c, gcache, 0, q, lens, RK, RV, status=st)
    assert int(st.item()) == 0
    assert rel_l2(out, ref) <= 2e-4 and np.abs(out - ref).max() <= 5e-3


def test_wait_test_hook_rejects_bad_values():
    with pytest.raises(K.OscarError):
        K.set_wait_test(20_000_000_000, 0)
    with pytest.raises(K.OscarError):
        K.set_wait_test(0, -1)
    K.set_wait_test(0, 0)
