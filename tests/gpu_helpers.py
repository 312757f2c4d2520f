"""Helpers for GPU parity tests: upload seeded inputs, call the C-ABI through the
binding, download results.  Expected values always come from the oracle."""
import numpy as np
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from oracle import oscar_oracle as O


def kcfg(c: O.Config) -> K.KVConfig:
    return K.KVConfig(c.num_layers, c.batch, c.num_q_heads, c.num_kv_heads, c.head_dim, c.sink, c.recent,
                      c.capacity, c.k_clip, c.v_clip, c.flags)


def dev(x, dtype=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype).cuda()


def dev_i32(x):
    return torch.tensor(np.asarray(x, dtype=np.int32), dtype=torch.int32, device="cuda")


def dev_rot(R):
    """A rotation matrix on the device as float32, or None (in-quant Hadamard)."""
    return None if R is None else dev(R, torch.float32)


def new_cache(c: O.Config):
    return torch.zeros(O.layout(c)["total_bytes"], dtype=torch.uint8, device="cuda")


def gpu_append(c: O.Config, cache, layer, k, v, start_pos, RK, RV, want_rot=False, status=None):
    fp32 = bool(c.flags & K.FLAG_IN_FP32)
    dt = torch.float32 if fp32 else torch.bfloat16
    kt, vt = dev(k, dt), dev(v, dt)
    B, n, H, D = k.shape
    rot = torch.empty((B, n, H, 2, D), dtype=torch.float32, device="cuda") if want_rot else None
    K.kv_append(kcfg(c), cache, layer, kt, vt, dev_i32(start_pos), dev_rot(RK), dev_rot(RV),
                debug_rot=rot, status=status)
    torch.cuda.synchronize()
    return rot


def workspace_bytes(c: O.Config, slots: int) -> int:
    """attn_decode workspace with `slots` partial slots per query head (the
    formula documented with kv_layout_query)."""
    a = lambda x: (x + 255) // 256 * 256
    bq, units, Dg = c.batch * c.num_q_heads, c.batch * c.num_kv_heads, c.head_dim // 128
    nqt = 2 if c.num_q_heads // c.num_kv_heads > 4 else 1
    return (a(units * Dg * nqt * 2048) + a(units * Dg * nqt * 4096) + 2 * a(bq * Dg * 4)
            + a(bq * slots * c.head_dim * 4) + a(bq * slots * 8) + a(units * 4))


def gpu_decode(c: O.Config, cache, layer, q, seq_lens, RK, RV, sm_scale=0.0, num_splits=0, hint=0,
               status=None, out_fp32=None, ws_bytes=None):
    kc = kcfg(c)
    if out_fp32 is not None:
        kc.flags = (kc.flags & ~K.FLAG_OUT_FP32) | (K.FLAG_OUT_FP32 if out_fp32 else 0)
    lay = K.layout_query(kc)
    fp32_in = bool(c.flags & K.FLAG_IN_FP32)
    qt = dev(q, torch.float32 if fp32_in else torch.bfloat16)
    B, Hq, D = q.shape
    out = torch.empty((B, Hq, D), dtype=torch.float32 if kc.flags & K.FLAG_OUT_FP32 else torch.bfloat16,
                      device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ws = torch.empty(ws_bytes or lay["decode_workspace_bytes"], dtype=torch.uint8, device="cuda")
    K.attn_decode(kc, cache, layer, qt, dev_i32(seq_lens), dev_rot(RK), dev_rot(RV), out,
                  ws, lse=lse, seq_len_hint=hint, sm_scale=sm_scale, num_splits=num_splits, status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def bf16_round64(x):
    return O.bf16_bits_to_f32(O.f32_to_bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


def rel_l2(a, b):
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-30))


def assert_same_decode(o0, o1, l0, l1):
    """Two decodes of the same cache bytes and query must agree bit for bit,
    outputs and lse: the scores, the softmax, the merge of the partial results
    (slots in a fixed order) and the V un-rotation (one loop whose arithmetic
    and order do not depend on where the merging CTA reads R_V from) are one
    fixed computation, whichever CTA merges a unit.  A read of stale cache data
    changes the scores, hence both."""
    o0 = np.asarray(o0, np.float32)
    o1 = np.asarray(o1, np.float32)
    diff = np.argwhere(o0.view(np.uint32) != o1.view(np.uint32))
    assert diff.size == 0, (f"outputs differ at {len(diff)} entries, first (b, head, channel) {diff[:8].tolist()}, "
                            f"max |diff| {np.abs(o0.astype(np.float64) - o1).max():.3e}")
    l0 = np.asarray(l0, np.float32)
    l1 = np.asarray(l1, np.float32)
    assert np.array_equal(l0.view(np.uint32), l1.view(np.uint32)), f"lse max |diff| {np.abs(l0 - l1).max():.3e}"
