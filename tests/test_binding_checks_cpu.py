"""The Python binding refuses, before any call reaches the library, tensors whose
dtype, shape or size does not match what the kernels read or write through
them (a wrong one would make a kernel read or write past the buffer's end).
CPU only: the checks run before the device pointers are taken."""
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K

CFG = K.KVConfig(1, 2, 8, 2, 128, 4, 8, 64)


def _decode_args(**over):
    B, Hq, D = CFG.batch, CFG.num_q_heads, CFG.head_dim
    lay = K.layout_query(CFG)
    args = dict(cfg=CFG, cache=torch.zeros(lay["total_bytes"], dtype=torch.uint8), layer=0,
                q=torch.zeros(B, Hq, D, dtype=torch.bfloat16), seq_lens=torch.zeros(B, dtype=torch.int32),
                R_K=torch.zeros(D, D), R_V=torch.zeros(D, D), out=torch.zeros(B, Hq, D, dtype=torch.bfloat16),
                workspace=torch.zeros(256, dtype=torch.uint8), lse=torch.zeros(B, Hq))
    args.update(over)
    return args


def _append_args(**over):
    B, H, D = CFG.batch, CFG.num_kv_heads, CFG.head_dim
    lay = K.layout_query(CFG)
    args = dict(cfg=CFG, cache=torch.zeros(lay["total_bytes"], dtype=torch.uint8), layer=0,
                k_new=torch.zeros(B, 3, H, D, dtype=torch.bfloat16), v_new=torch.zeros(B, 3, H, D, dtype=torch.bfloat16),
                start_pos=torch.zeros(B, dtype=torch.int32), R_K=torch.zeros(D, D), R_V=torch.zeros(D, D))
    args.update(over)
    return args


def test_valid_arguments_reach_the_device_check():
    # every check passes; the first refusal is that the tensors are on the host
    with pytest.raises(ValueError, match="CUDA tensor"):
        K.attn_decode(**_decode_args())
    with pytest.raises(ValueError, match="CUDA tensor"):
        K.kv_append(**_append_args())


@pytest.mark.parametrize("over", [
    dict(q=torch.zeros(2, 8, 128, dtype=torch.float32)),          # fp32 q without OSCAR_FLAG_IN_FP32
    dict(q=torch.zeros(2, 4, 128, dtype=torch.bfloat16)),         # wrong number of query heads
    dict(out=torch.zeros(2, 8, 64, dtype=torch.bfloat16)),        # output too small
    dict(out=torch.zeros(2, 8, 128, dtype=torch.float32)),        # fp32 out without OSCAR_FLAG_OUT_FP32
    dict(lse=torch.zeros(2, 4)),                                  # lse too small
    dict(seq_lens=torch.zeros(2, dtype=torch.int64)),
    dict(seq_lens=torch.zeros(3, dtype=torch.int32)),
    dict(R_K=torch.zeros(64, 64)),                                 # rotation too small
    dict(R_V=torch.zeros(128, 128, dtype=torch.bfloat16)),
    dict(cache=torch.zeros(1024, dtype=torch.uint8)),             # cache smaller than the layout
    dict(workspace=torch.zeros(256, dtype=torch.float32)),
])
def test_decode_refuses_mismatched_tensors(over):
    with pytest.raises(ValueError, match="oscar_kv"):
        K.attn_decode(**_decode_args(**over))


@pytest.mark.parametrize("over", [
    dict(k_new=torch.zeros(2, 3, 2, 128, dtype=torch.float32)),   # fp32 rows without OSCAR_FLAG_IN_FP32
    dict(v_new=torch.zeros(2, 4, 2, 128, dtype=torch.bfloat16)),  # V and K disagree on n_new
    dict(k_new=torch.zeros(2, 3, 1, 128, dtype=torch.bfloat16), v_new=torch.zeros(2, 3, 1, 128, dtype=torch.bfloat16)),
    dict(start_pos=torch.zeros(1, dtype=torch.int32)),
    dict(R_K=torch.zeros(128, 127)),
    dict(cache=torch.zeros(10, dtype=torch.uint8)),
])
def test_append_refuses_mismatched_tensors(over):
    with pytest.raises(ValueError, match="oscar_kv"):
        K.kv_append(**_append_args(**over))


def test_append_debug_rows_must_hold_every_rotated_row():
    with pytest.raises(ValueError, match="debug_rot"):
        K.kv_append(**_append_args(), debug_rot=torch.zeros(2, 3, 2, 128))


def test_calibration_refuses_mismatched_tensors():
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="oscar_kv"):
        K.calibrate_rk(torch.zeros(10, 128, dtype=torch.bfloat16), torch.zeros(128, 128), ws)
    with pytest.raises(ValueError, match="oscar_kv"):
        K.calibrate_rk(torch.zeros(10, 128), torch.zeros(64, 64), ws)
    with pytest.raises(ValueError):
        K.calibrate_rv(torch.zeros(10, 128), torch.zeros(5, 128), torch.zeros(6, 128), torch.zeros(128, 128), ws)
    with pytest.raises(ValueError, match="oscar_kv"):
        K.calibrate_rv(torch.zeros(10, 128), torch.zeros(5, 128), torch.zeros(5, 128),
                       torch.zeros(128, 128, dtype=torch.float64), ws)


def test_decode_kernel_count():
    # query rotation + split attention, and the un-rotation kernel only at
    # head_dim 256 / 512 with V neither absorbed nor Hadamard-rotated
    assert K.decode_kernels(K.KVConfig(1, 2, 8, 2, 128, 4, 8, 64)) == 2
    assert K.decode_kernels(K.KVConfig(1, 2, 8, 2, 256, 4, 8, 64)) == 3
    assert K.decode_kernels(K.KVConfig(1, 2, 8, 2, 512, 4, 8, 64)) == 3
    assert K.decode_kernels(K.KVConfig(1, 2, 8, 2, 512, 4, 8, 64, flags=K.FLAG_ABSORB_V)) == 2
    assert K.decode_kernels(K.KVConfig(1, 2, 8, 2, 512, 4, 8, 64, flags=K.FLAG_HADAMARD)) == 2
    # head_dim 128: only with G > 4 and at most 16 (sequence, KV head) pairs
    assert K.decode_kernels(K.KVConfig(1, 1, 64, 8, 128, 4, 8, 64)) == 3
    assert K.decode_kernels(K.KVConfig(1, 4, 64, 8, 128, 4, 8, 64)) == 2
    assert K.decode_kernels(K.KVConfig(1, 1, 64, 8, 128, 4, 8, 64, flags=K.FLAG_ABSORB_V)) == 2
    with pytest.raises(K.OscarError):
        K.decode_kernels(K.KVConfig(1, 2, 8, 3, 128, 4, 8, 64))  # 8 query heads over 3 KV heads
