"""GPU parity: kv_append against the oracle.

With exact rotations (signed permutations) every rotated value is exact on both
sides, so the whole cache must match byte for byte.  With calibrated rotations
the GPU's float32 rotated rows may differ from the correctly rounded product in
the last bit, so the oracle quantises the GPU's own rows (exported through
debug_rot_out) and the cache must again match byte for byte."""
import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S
from oracle import oscar_oracle as O
from tests.gpu_helpers import gpu_append, new_cache

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


CASES = [
    # D, B, Hkv, S, W, cap, chunks (n per call), start offsets per sequence
    (128, 2, 2, 16, 32, 256, [40, 1, 7, 64], [0, 3]),
    (128, 3, 1, 0, 0, 130, [65, 65], [0, 0, 1]),
    (128, 1, 4, 10, 4, 64, [3, 3, 3, 20], [0]),        # S > W: positions in both windows
    (128, 2, 8, 64, 256, 1024, [600, 1], [0, 100]),
    (256, 2, 2, 5, 9, 200, [33, 17, 2], [1, 0]),
    (512, 2, 2, 8, 16, 160, [50, 31, 1], [0, 7]),
    # row counts per call chosen to reach every append kernel: <= 512 rows and
    # 513..1024 rows (row-parallel kernel, 4 and 8 rows per CTA), > 1024 rows
    # (tiled kernels: tensor cores at D = 128 with bf16 input, CUDA cores otherwise)
    (128, 2, 4, 16, 64, 400, [100, 1, 50], [0, 2]),
    (256, 2, 4, 8, 32, 720, [600, 100], [0, 5]),
    (512, 1, 4, 4, 8, 460, [300, 150], [3]),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("fp32", [False, True])
def test_append_exact_chain_bitwise(case, fp32):
    D, B, H, S_, W, cap, chunks, offs = case
    c = O.Config(2, B, H * 2, H, D, S_, W, cap, 0.96, 0.92, flags=K.FLAG_IN_FP32 if fp32 else 0)
    rng = np.random.default_rng(D + B)
    RK = S.signed_permutation(rng, D).astype(np.float32)
    RV = S.signed_permutation(rng, D).astype(np.float32)
    ocache = O.new_cache(c)
    gcache = new_cache(c)
    pos = list(offs)
    for i, n in enumerate(chunks):
        k, v = _inputs(100 + i, B, n, H, D, fp32)
        O.append(c, ocache, 1, k, v, pos, RK, RV)
        gpu_append(c, gcache, 1, k, v, pos, RK, RV)
        pos = [p + n for p in pos]
    got = gcache.cpu().numpy()
    diff = np.nonzero(got != ocache)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


@pytest.mark.parametrize("fp32", [False, True])
def test_append_calibrated_rotation_codec_exact_on_gpu_rows(fp32):
    """Calibrated rotations: the GPU's float32 rotation (tensor cores with R
    split into three bf16 pieces at head_dim 128 with bf16 rows, fp32 FMAs
    otherwise) is within 2e-6 of the float64 product but not correctly rounded,
    so the codec is checked on the GPU's own rows: the oracle quantises the rows
    the append exports through debug_rot_out (identity rotation in its own
    append) and the two caches must match byte for byte (codes, scale/zero,
    BF16 sink and ring).  Calls of more than 1024 rows per role take the tiled
    kernels (tensor cores with bf16 input), small ones the row-parallel kernel."""
    w = S.WORKLOADS["qwen3-4b-layer"]
    D, B, H, S_, W, cap = 128, 2, 8, 64, 128, 512
    flags = K.FLAG_IN_FP32 if fp32 else 0
    c = O.Config(1, B, 32, H, D, S_, W, cap, 0.96, 0.92, flags=flags)
    plain = O.Config(1, B, 32, H, D, S_, W, cap, 0.96, 0.92)
    RK, RV = S.rotations(w, 0)
    eye = np.eye(D, dtype=np.float32)
    ocache, gcache = O.new_cache(plain), new_cache(c)
    pos = [0, 5]
    for i, n in enumerate([300, 1, 40, 120]):  # 4800 rows, then 16, 640 and 1920 rows per role
        k, v = _inputs(900 + i, B, n, H, D, fp32)
        rot = gpu_append(c, gcache, 0, k, v, pos, RK, RV, want_rot=True).cpu().numpy()
        for role, (x, R) in enumerate(((k, RK), (v, RV))):
            exact = x.astype(np.float64) @ R.astype(np.float64)
            assert np.abs(rot[:, :, :, role] - exact).max() <= 2e-6 * np.abs(exact).max()
        O.append(plain, ocache, 0, rot[:, :, :, 0], rot[:, :, :, 1], pos, eye, eye)
        pos = [p + n for p in pos]
    got = gcache.cpu().numpy()
    diff = np.nonzero(got != ocache)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


def test_append_over_capacity_sets_status_and_skips():
    D, B, H = 128, 2, 1
    c = O.Config(1, B, 1, H, D, 4, 4, 20)
    k, v = _inputs(5, B, 8, H, D)
    I = np.eye(D, dtype=np.float32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gcache = new_cache(c)
    gpu_append(c, gcache, 0, k, v, [0, 16], I, I, status=st)     # b=1 writes positions 16..23
    assert int(st.item()) & K.DEV_OVER_CAPACITY
    # rows inside capacity match an oracle run of the first four tokens (the
    # oracle writes 0..3 for b=0 and 16..19 for b=1; the GPU also wrote 4..7
    # for b=0, so compare only what both wrote)
    ocache = O.new_cache(c)
    O.append(c, ocache, 0, k[:, :4], v[:, :4], [0, 16], I, I)
    g = gcache.cpu().numpy()
    gv, ov = O.CacheView(c, g, 0, 0), O.CacheView(c, ocache, 0, 0)
    assert np.array_equal(gv.sink[0], ov.sink[0])
    assert np.array_equal(gv.codes[1, 0, 12:16], ov.codes[1, 0, 12:16])


def test_append_nonfinite_sets_status():
    D = 128
    c = O.Config(1, 1, 1, 1, D, 0, 0, 8)
    k, v = _inputs(6, 1, 2, 1, D)
    k[0, 1, 0, 3] = np.inf
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_append(c, new_cache(c), 0, k, v, [0], np.eye(D, dtype=np.float32), np.eye(D, dtype=np.float32), status=st)
    assert int(st.item()) & K.DEV_NONFINITE
