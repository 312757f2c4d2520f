"""Full-size parity: every workload at its real shape, in the launch
configuration bench.py times (automatic split count, seq_len_hint = context).

Inputs are drawn on the GPU with a seeded torch generator.  The GPU builds the
whole cache with kv_append and decodes all sequences; the oracle rebuilds the
cache of sampled (sequence, KV head) pairs from the same inputs (copied to the
host) and decodes them.  Two tests run the bench's decode_step instead (the
cache filled to T - 1 tokens, the call appending the last one and decoding).  With exact rotations (signed permutations) the GPU
cache must equal the oracle's bit for bit on the sampled pairs, and the decode
outputs must agree within the decode tolerances.  One test also runs the
calibrated rotations: there the oracle quantises the GPU's own float32 rotated
rows (the append's debug output), the cache bytes must again match and the
decode meets the same tolerances."""
import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S
from oracle import oscar_oracle as O
from tests.gpu_helpers import bf16_round64, rel_l2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs CUDA")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_kv_cache_append_gb300 import build
    build.build()


def _fill(w, cfg, cache, layer, RK, RV, T, seed, upto=None, rot_pairs=()):
    """Draw T tokens per sequence and GPU-append the first `upto` (all by default);
    returns the bf16 K and V inputs kept on the device.  For every (b, h) in
    rot_pairs the GPU's own float32 rotated K and V rows (the append's
    debug_rot_out) are collected into rot_pairs[(b, h)] = [T][2][D]."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    ch = S.outlier_channels(w.config_id, layer, w.head_dim)
    shape = (w.batch, T, w.num_kv_heads, w.head_dim)
    k = S.activations_torch(gen, shape, ch, dtype=torch.bfloat16)
    v = S.activations_torch(gen, shape, ch, dtype=torch.bfloat16)
    chunk = max(1, (1 << 26) // (w.batch * w.num_kv_heads * w.head_dim))
    upto = T if upto is None else upto
    rows = {bh: np.zeros((upto, 2, w.head_dim), np.float32) for bh in rot_pairs}
    for p in range(0, upto, chunk):
        n = min(chunk, upto - p)
        dbg = (torch.empty((w.batch, n, w.num_kv_heads, 2, w.head_dim), dtype=torch.float32, device="cuda")
               if rot_pairs else None)
        K.kv_append(cfg, cache, layer, k[:, p:p + n].contiguous(), v[:, p:p + n].contiguous(),
                    torch.full((w.batch,), p, dtype=torch.int32, device="cuda"), RK, RV, debug_rot=dbg)
        for (b, h), r in rows.items():
            r[p:p + n] = dbg[b, :, h].cpu().numpy()
    if isinstance(rot_pairs, dict):
        rot_pairs.update(rows)
    q = S.activations_torch(gen, (w.batch, w.num_q_heads, w.head_dim), ch, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    return k, v, q


def _oracle_pair(w, k, v, q, b, h, T, RK, RV, gpu_rows=None):
    """Oracle cache + decode for one (sequence b, KV head h) from the device inputs.
    With gpu_rows ([T][2][D], the GPU's own float32 rotated rows) the oracle
    quantises those rows (identity rotation in its append) instead of rotating
    the inputs itself; the decode still rotates q by R_K and un-rotates by R_V."""
    G = w.num_q_heads // w.num_kv_heads
    c = O.Config(1, 1, G, 1, w.head_dim, w.sink, w.recent, T, w.k_clip, w.v_clip)
    qq = q[b:b + 1, h * G:(h + 1) * G].float().cpu().numpy()
    cache = O.new_cache(c)
    if gpu_rows is None:
        kk = k[b:b + 1, :, h:h + 1].float().cpu().numpy()
        vv = v[b:b + 1, :, h:h + 1].float().cpu().numpy()
        O.append(c, cache, 0, kk, vv, [0], RK, RV)
    else:
        eye = np.eye(w.head_dim, dtype=np.float32)
        O.append(c, cache, 0, gpu_rows[None, :, None, 0], gpu_rows[None, :, None, 1], [0], eye, eye)
    out, lse = O.decode(c, cache, 0, qq, [T], RK, RV, absorb_v=w.absorb_v)
    return c, cache, out[0], lse[0]


def _compare_cache_pair(w, gcache_np, ocfg, ocache, cfg_full, layer, b, h):
    """Bytes of one (b, h) in every region must match."""
    full = O.Config(cfg_full.num_layers, cfg_full.batch, cfg_full.num_q_heads, cfg_full.num_kv_heads,
                    cfg_full.head_dim, cfg_full.sink, cfg_full.recent, cfg_full.capacity)
    for role in (0, 1):
        gv = O.CacheView(full, gcache_np, layer, role)
        ov = O.CacheView(ocfg, ocache, 0, role)
        n = ov.codes.shape[2]
        assert np.array_equal(gv.sink[b, h], ov.sink[0, 0])
        assert np.array_equal(gv.ring[b, h], ov.ring[0, 0])
        assert np.array_equal(gv.codes[b, h, :n], ov.codes[0, 0])
        assert np.array_equal(gv.sz[b, h, :n].view(np.uint16), ov.sz[0, 0].view(np.uint16))


def _decode_all(w, cfg, cache, layer, q, T, RK, RV, out_fp32, step_kv=None):
    """attn_decode over T tokens, or with step_kv = (k, v) of the last token the
    bench's decode_step: append that token at T - 1, then decode (re-appending
    the same token writes the same bytes, so it may run twice)."""
    kc = K.KVConfig(**{**cfg.__dict__})
    kc.flags = (kc.flags & ~K.FLAG_OUT_FP32) | (K.FLAG_OUT_FP32 if out_fp32 else 0)
    lay = K.layout_query(kc)
    out = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else torch.bfloat16, device="cuda")
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ws = torch.empty(lay["decode_workspace_bytes"], dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    seq = torch.full((w.batch,), T, dtype=torch.int32, device="cuda")
    if step_kv is None:
        K.attn_decode(kc, cache, layer, q, seq, RK, RV, out, ws, lse=lse, seq_len_hint=T, status=st)
    else:
        K.decode_step(kc, cache, layer, step_kv[0], step_kv[1], seq - 1, q, seq, RK, RV, out, ws, lse=lse,
                      seq_len_hint=T, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _run(wname, samples, layers=(0,), rot="perm", T=None, fused=False):
    w = S.WORKLOADS[wname]
    T = T or w.context
    flags = K.FLAG_ABSORB_V if w.absorb_v else 0
    L = max(layers) + 1
    cfg = K.KVConfig(L, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.sink, w.recent, w.context,
                     w.k_clip, w.v_clip, flags)
    lay = K.layout_query(cfg)
    cache = torch.zeros(lay["total_bytes"], dtype=torch.uint8, device="cuda")
    G = w.num_q_heads // w.num_kv_heads
    for layer in layers:
        RKn, RVn = S.rotations(w, layer, kind=rot)
        RK, RV = torch.from_numpy(RKn).cuda(), torch.from_numpy(RVn).cuda()
        # calibrated rotations: the GPU's float32 rotation need not be correctly
        # rounded, so the oracle quantises the GPU's own rotated rows
        rows = {} if rot == "oscar" else ()
        if rot == "oscar":
            rows.update({bh: None for bh in samples})
        k, v, q = _fill(w, cfg, cache, layer, RK, RV, T, seed=4242 + layer, upto=T - 1 if fused else T,
                        rot_pairs=rows)
        if rot == "oscar":
            for bh in samples:  # the GPU rotation is within 2e-6 of the float64 product
                kk = k[bh[0], :T, bh[1]].float().cpu().numpy().astype(np.float64)
                exact = kk @ RKn.astype(np.float64)
                assert np.abs(rows[bh][:, 0] - exact).max() <= 2e-6 * np.abs(exact).max()
        step_kv = (k[:, T - 1:T].contiguous(), v[:, T - 1:T].contiguous()) if fused else None
        o16, _ = _decode_all(w, cfg, cache, layer, q, T, RK, RV, out_fp32=False, step_kv=step_kv)
        o32, l32 = _decode_all(w, cfg, cache, layer, q, T, RK, RV, out_fp32=True, step_kv=step_kv)
        gnp = cache.cpu().numpy()
        for b, h in samples:
            ocfg, ocache, ref, ref_lse = _oracle_pair(w, k, v, q, b, h, T, RKn, RVn,
                                                      gpu_rows=rows[(b, h)] if rot == "oscar" else None)
            _compare_cache_pair(w, gnp, ocfg, ocache, cfg, layer, b, h)
            sl = slice(h * G, (h + 1) * G)
            r16 = rel_l2(o16[b, sl], bf16_round64(ref))
            r32 = rel_l2(o32[b, sl], ref)
            m32 = float(np.abs(o32[b, sl] - ref).max())
            dl = float(np.max(np.abs(l32[b, sl] - ref_lse) - 1e-5 * np.abs(ref_lse)))
            assert r16 <= 1e-3, (wname, layer, b, h, r16)
            assert m32 <= 5e-3 and r32 <= 2e-4, (wname, layer, b, h, m32, r32)
            assert dl <= 1e-4, (wname, layer, b, h, dl)


def test_full_qwen3_4b_layer():
    _run("qwen3-4b-layer", samples=[(0, 0), (3, 5), (7, 7)])


def test_full_qwen3_4b_layer_decode_step():
    # the bench's step: the cache holds T - 1 tokens, decode_step appends the
    # last one and decodes over T
    _run("qwen3-4b-layer", samples=[(0, 0), (4, 2), (7, 7)], fused=True)


def test_full_qwen3_32b_decode_step():
    _run("qwen3-32b-decode", samples=[(0, 0), (0, 7)], fused=True)


def test_full_qwen3_4b_layer_calibrated_rotations():
    # calibrated R (tensor-core append at this size): the cache bytes of the
    # sampled pairs equal the oracle's quantisation of the GPU's own rotated
    # rows, and the decode meets the usual tolerances against that cache
    _run("qwen3-4b-layer", samples=[(1, 2), (6, 5)], rot="oscar")


def test_full_qwen3_32b_decode():
    _run("qwen3-32b-decode", samples=[(0, 0), (0, 6)])


def test_full_hd512():
    _run("hd512", samples=[(0, 0), (3, 7)])


def test_full_qwen3_8b_two_layers():
    # two of the 36 layers at full batch and context (each layer is an independent launch)
    _run("qwen3-8b-36L", samples=[(0, 0), (31, 7)], layers=(0, 35))


def test_full_qwen3_32b_append_positions():
    """Phase-1 append: 8192 new tokens per sequence at positions 122880..131071."""
    w = S.WORKLOADS["qwen3-32b-append"]
    D, H, n, T = w.head_dim, w.num_kv_heads, w.append_tokens, w.context
    cfg = K.KVConfig(1, w.batch, w.num_q_heads, H, D, w.sink, w.recent, T, w.k_clip, w.v_clip)
    lay = K.layout_query(cfg)
    cache = torch.zeros(lay["total_bytes"], dtype=torch.uint8, device="cuda")
    RKn, RVn = S.rotations(w, 0, kind="perm")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    ch = S.outlier_channels(w.config_id, 0, D)
    k = S.activations_torch(gen, (w.batch, n, H, D), ch, dtype=torch.bfloat16)
    v = S.activations_torch(gen, (w.batch, n, H, D), ch, dtype=torch.bfloat16)
    start = T - n
    K.kv_append(cfg, cache, 0, k, v, torch.full((w.batch,), start, dtype=torch.int32, device="cuda"),
                torch.from_numpy(RKn).cuda(), torch.from_numpy(RVn).cuda())
    torch.cuda.synchronize()
    g = cache.cpu().numpy()
    full = O.Config(1, w.batch, w.num_q_heads, H, D, w.sink, w.recent, T)
    for b, h in [(0, 0), (3, 7)]:
        oc = O.Config(1, 1, 1, 1, D, w.sink, w.recent, T)
        ocache = O.new_cache(oc)
        O.append(oc, ocache, 0, k[b:b + 1, :, h:h + 1].float().cpu().numpy(),
                 v[b:b + 1, :, h:h + 1].float().cpu().numpy(), [start], RKn, RVn)
        for role in (0, 1):
            gv, ov = O.CacheView(full, g, 0, role), O.CacheView(oc, ocache, 0, role)
            r0 = start - w.sink
            assert np.array_equal(gv.codes[b, h, r0:r0 + n], ov.codes[0, 0, r0:r0 + n])
            assert np.array_equal(gv.sz[b, h, r0:r0 + n].view(np.uint16), ov.sz[0, 0, r0:r0 + n].view(np.uint16))
            assert np.array_equal(gv.ring[b, h], ov.ring[0, 0])
