"""C-ABI library: loads, exports every declared symbol, host-only layout
arithmetic and argument validation.  No GPU compute is launched here."""
import ctypes
import os
import re

import pytest

from int2_kv_cache_append_gb300 import oscar_kv as K
from oracle import oscar_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from int2_kv_cache_append_gb300 import build
    build.build()
    return K.lib()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "oscar_kv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^int\s+(\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    decl = _declared_symbols()
    assert decl == sorted(K.EXPORTS)
    for name in decl:
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


@pytest.mark.parametrize("shape", [
    (1, 1, 4, 1, 128, 64, 256, 1024), (2, 3, 8, 2, 256, 5, 7, 100), (36, 32, 32, 8, 128, 64, 256, 32768),
    (1, 4, 16, 8, 512, 512, 2048, 65536), (1, 2, 2, 2, 128, 0, 0, 1), (1, 1, 8, 1, 128, 300, 0, 200)])
@pytest.mark.parametrize("flags", [0, K.FLAG_V_BF16, K.FLAG_LLOYD_MAX, K.FLAG_LLOYD_MAX | K.FLAG_V_BF16])
def test_layout_matches_oracle(lib, shape, flags):
    L, B, Hq, Hkv, D, S, W, cap = shape
    got = K.layout_query(K.KVConfig(L, B, Hq, Hkv, D, S, W, cap, flags=flags))
    exp = O.layout(O.Config(L, B, Hq, Hkv, D, S, W, cap, flags=flags))
    for key in ("ncap", "sink_bytes", "ring_bytes", "codes_bytes", "sz_bytes", "role_bytes", "v_role_bytes",
                "layer_bytes", "total_bytes"):
        assert got[key] == exp[key], key
    assert got["max_splits"] == K.MAX_SPLITS
    # documented workspace formula
    a = lambda x: (x + 255) // 256 * 256
    bq, units, Dg = B * Hq, B * Hkv, D // 128
    nqt = 2 if Hq // Hkv > 4 else 1
    ws = (a(units * Dg * nqt * 2048) + a(units * Dg * nqt * 4096) + 2 * a(bq * Dg * 4) + a(bq * 64 * D * 4)
          + a(bq * 64 * 8) + a(units * 4))
    assert got["decode_workspace_bytes"] == ws


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 64, -5), ("head_dim", 192, -5), ("group_size", 64, -5), ("num_q_heads", 6, -1),
    ("num_q_heads", 72, -5), ("k_clip", 0.0, -1), ("v_clip", 1.5, -1), ("sink", -1, -1), ("recent", -3, -1),
    ("capacity", 0, -1), ("batch", 0, -1), ("flags", 64, -1)])
def test_layout_rejects_bad_config(lib, field, value, code):
    cfg = K.KVConfig(1, 2, 8, 4 if field == "num_q_heads" and value == 6 else 8, 128, 4, 8, 64)
    if field == "num_q_heads" and value == 72:
        cfg.num_kv_heads = 8
    setattr(cfg, field, value)
    out = K._Layout()
    assert lib.kv_layout_query(ctypes.byref(cfg.c()), ctypes.byref(out)) == code


def test_entry_points_validate_before_launch(lib):
    cfg = K.KVConfig(1, 1, 4, 1, 128, 4, 8, 64)
    c = cfg.c()
    P = ctypes.c_void_p
    big = P(1 << 20)  # never dereferenced: every call below fails validation first
    # null cache
    assert lib.kv_append(ctypes.byref(c), None, 0, big, big, big, 1, big, big, None, None, None) == -1
    # layer out of range
    assert lib.kv_append(ctypes.byref(c), big, 1, big, big, big, 1, big, big, None, None, None) == -1
    # misaligned cache
    assert lib.kv_append(ctypes.byref(c), P((1 << 20) + 16), 0, big, big, big, 1, big, big, None, None, None) == -1
    # n_new beyond capacity
    assert lib.kv_append(ctypes.byref(c), big, 0, big, big, big, 65, big, big, None, None, None) == -2
    # decode: too many splits, hint beyond capacity, workspace too small for one split
    assert lib.attn_decode(ctypes.byref(c), big, 0, big, big, 0, big, big, 0.0, 65, big, None, big, 1 << 30,
                           None, None) == -1
    assert lib.attn_decode(ctypes.byref(c), big, 0, big, big, 65, big, big, 0.0, 1, big, None, big, 1 << 30,
                           None, None) == -2
    assert lib.attn_decode(ctypes.byref(c), big, 0, big, big, 0, big, big, 0.0, 1, big, None, big, 16, None,
                           None) == -3
    # decode_step validates both halves before launching anything
    assert lib.decode_step(ctypes.byref(c), None, 0, big, big, big, 1, big, big, 0, big, big, 0.0, 0, big, None,
                           big, 1 << 30, None, None) == -1
    assert lib.decode_step(ctypes.byref(c), big, 0, big, big, big, 65, big, big, 0, big, big, 0.0, 0, big, None,
                           big, 1 << 30, None, None) == -2
    assert lib.decode_step(ctypes.byref(c), big, 0, big, big, big, 1, big, big, 0, big, big, 0.0, 0, big, None,
                           big, 16, None, None) == -3
    # bad config passes through the same validation
    bad = K.KVConfig(1, 1, 4, 1, 96, 4, 8, 64).c()
    assert lib.attn_decode(ctypes.byref(bad), big, 0, big, big, 0, big, big, 0.0, 1, big, None, big, 1 << 30,
                           None, None) == -5


def test_hadamard_flag_makes_rotations_optional(lib):
    P = ctypes.c_void_p
    big = P(1 << 20)  # never dereferenced: every call below stops in validation
    plain = K.KVConfig(1, 1, 4, 1, 128, 4, 8, 64).c()
    had = K.KVConfig(1, 1, 4, 1, 128, 4, 8, 64, flags=K.FLAG_HADAMARD).c()
    out = K._Layout()
    assert lib.kv_layout_query(ctypes.byref(had), ctypes.byref(out)) == 0
    # without the flag a NULL rotation is an invalid argument ...
    assert lib.kv_append(ctypes.byref(plain), big, 0, big, big, big, 65, None, big, None, None, None) == -1
    assert lib.attn_decode(ctypes.byref(plain), big, 0, big, big, 0, big, None, 0.0, 1, big, None, big, 16,
                           None, None) == -1
    # ... with it the NULLs pass and validation goes on to the next check
    assert lib.kv_append(ctypes.byref(had), big, 0, big, big, big, 65, None, None, None, None, None) == -2
    assert lib.attn_decode(ctypes.byref(had), big, 0, big, big, 0, None, None, 0.0, 1, big, None, big, 16,
                           None, None) == -3
    assert lib.decode_step(ctypes.byref(had), big, 0, big, big, big, 1, big, big, 0, None, None, 0.0, 0, big,
                           None, big, 16, None, None) == -3


def test_calibrate_entry_points_validate_before_launch(lib):
    P = ctypes.c_void_p
    big = P(1 << 20)  # never dereferenced: every call below stops in validation
    n = ctypes.c_uint64(0)
    assert lib.oscar_calibrate_workspace_query(96, ctypes.byref(n)) == -5
    assert lib.oscar_calibrate_workspace_query(128, None) == -1
    for d in (128, 256, 512):
        assert lib.oscar_calibrate_workspace_query(d, ctypes.byref(n)) == 0
        assert n.value == 3 * (-(-d * d * 8 // 256) * 256) + (-(-d * 8 // 256) * 256) + 256
    f = lib.oscar_calibrate_rk
    f.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, P, ctypes.c_uint64, P, P]
    assert f(big, 1000, 96, big, big, 1 << 30, None, None) == -5          # head_dim
    assert f(None, 1000, 128, big, big, 1 << 30, None, None) == -1        # null rows
    assert f(big, 0, 128, big, big, 1 << 30, None, None) == -1            # no rows
    assert f(big, 65535 * 4096 + 1, 128, big, big, 1 << 30, None, None) == -1  # more row chunks than grid z
    assert f(P((1 << 20) + 4), 1000, 128, big, big, 1 << 30, None, None) == -1  # misaligned
    assert f(big, 1000, 128, big, big, 1000, None, None) == -3            # workspace too small


def test_calibrate_rv_entry_points_validate_before_launch(lib):
    P = ctypes.c_void_p
    big = P(1 << 20)  # never dereferenced: every call below stops in validation
    n = ctypes.c_uint64(0)
    q = lib.oscar_calibrate_rv_workspace_query
    q.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint64)]
    assert q(96, 100, ctypes.byref(n)) == -5
    assert q(128, 0, ctypes.byref(n)) == -1
    assert q(128, 100, None) == -1
    a = lambda x: -(-x // 256) * 256
    for d in (128, 256, 512):
        for rows in (1, 1000, 160000):
            assert q(d, rows, ctypes.byref(n)) == 0
            # the R_K workspace followed by one float64 weight per key row
            assert n.value == 3 * a(d * d * 8) + a(d * 8) + 256 + a(rows * 8)
    f = lib.oscar_calibrate_rv
    f.argtypes = [P, ctypes.c_int64, P, P, ctypes.c_int64, ctypes.c_int32, P, P, ctypes.c_uint64, P, P]
    ok = dict(q=big, nq=1000, k=big, v=big, nkv=500, d=128, r=big, ws=big, wsb=1 << 30)
    call = lambda **kw: f(*({**ok, **kw}.values()), None, None)
    assert call(d=96) == -5                                   # head_dim
    for name in ("q", "k", "v", "r", "ws"):
        assert call(**{name: None}) == -1                     # null pointer
    assert call(nq=0) == -1 and call(nkv=0) == -1             # no rows
    assert call(nkv=65535 * 4096 + 1) == -1 and call(nq=65535 * 4096 + 1) == -1  # grid z holds 65535 chunks
    assert call(k=P((1 << 20) + 4)) == -1                     # misaligned
    assert call(ws=P((1 << 20) + 128)) == -1                  # workspace not 256-aligned
    assert call(wsb=3 * a(128 * 128 * 8) + a(128 * 8) + 256) == -3   # no room for the weights


def test_binding_refuses_host_tensors(lib):
    # the kernels would dereference a host address on the GPU: refused before the call
    import torch
    with pytest.raises(ValueError, match="CUDA tensor"):
        K._ptr(torch.zeros(4))
    assert K._ptr(None) is None
    cfg = K.KVConfig(1, 1, 4, 1, 128, 4, 8, 64)
    with pytest.raises(ValueError):
        K.kv_append(cfg, torch.zeros(64, dtype=torch.uint8), 0, torch.zeros(1, 1, 1, 128), torch.zeros(1, 1, 1, 128),
                    torch.zeros(1, dtype=torch.int32), torch.eye(128), torch.eye(128))
