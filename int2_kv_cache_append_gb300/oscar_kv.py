"""Thin ctypes binding of liboscar_kv.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module converts
torch tensors to pointers and checks return codes.  It raises if the library
has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liboscar_kv.so")

GROUP = 128
MAX_SPLITS = 64
FLAG_ABSORB_V = 1
FLAG_IN_FP32 = 2
FLAG_OUT_FP32 = 4
FLAG_HADAMARD = 8  # rotate by the in-quant Hadamard; R_K / R_V may be None
FLAG_V_BF16 = 16  # K-only INT2: V kept BF16 at every position
FLAG_LLOYD_MAX = 32  # INT2 codes index Lloyd-Max levels (0, rho, rho + 1, 2 rho + 1), rho = 1.16 (float32)

DEV_OVER_CAPACITY = 1
DEV_NONFINITE = 2
DEV_FP16_RANGE = 4
DEV_TIMEOUT = 8
DEV_EMPTY = 16

STATUS_NAMES = {0: "OK", -1: "INVALID", -2: "CAPACITY", -3: "WORKSPACE", -4: "LAUNCH", -5: "UNSUPPORTED"}

# every symbol include/oscar_kv.h declares
EXPORTS = ("kv_layout_query", "kv_append", "attn_decode", "decode_step", "attn_decode_static",
           "oscar_kv_set_profile_events", "oscar_kv_set_wait_test", "oscar_kv_decode_kernels",
           "oscar_calibrate_workspace_query",
           "oscar_calibrate_rk",
           "oscar_calibrate_rv_workspace_query", "oscar_calibrate_rv")
STATIC_SCRATCH_BYTES = 16 << 20


class OscarError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({STATUS_NAMES.get(code, '?')})")
        self.code = code


class _Config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("sink", ctypes.c_int32), ("recent", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("k_clip", ctypes.c_float), ("v_clip", ctypes.c_float), ("flags", ctypes.c_uint32)]


class _Layout(ctypes.Structure):
    _fields_ = [("ncap", ctypes.c_uint64), ("sink_bytes", ctypes.c_uint64), ("ring_bytes", ctypes.c_uint64),
                ("codes_bytes", ctypes.c_uint64), ("sz_bytes", ctypes.c_uint64), ("role_bytes", ctypes.c_uint64),
                ("layer_bytes", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64),
                ("decode_workspace_bytes", ctypes.c_uint64), ("max_splits", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("v_role_bytes", ctypes.c_uint64)]


@dataclass
class KVConfig:
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    sink: int
    recent: int
    capacity: int
    k_clip: float = 0.96
    v_clip: float = 0.92
    flags: int = 0
    group_size: int = GROUP

    def c(self) -> _Config:
        return _Config(self.num_layers, self.batch, self.num_q_heads, self.num_kv_heads, self.head_dim,
                       self.group_size, self.sink, self.recent, self.capacity, self.k_clip, self.v_clip,
                       self.flags)


_lib = None


def lib():
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with int2_kv_cache_append_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        L.kv_layout_query.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Layout)]
        L.kv_layout_query.restype = ctypes.c_int
        L.kv_append.argtypes = [ctypes.POINTER(_Config), P, ctypes.c_int32, P, P, P, ctypes.c_int32, P, P, P, P, P]
        L.kv_append.restype = ctypes.c_int
        L.attn_decode.argtypes = [ctypes.POINTER(_Config), P, ctypes.c_int32, P, P, ctypes.c_int32, P, P,
                                  ctypes.c_float, ctypes.c_int32, P, P, P, ctypes.c_uint64, P, P]
        L.attn_decode.restype = ctypes.c_int
        L.attn_decode_static.argtypes = [ctypes.POINTER(_Config), P, ctypes.c_int32, P, P, ctypes.c_int32, P, P,
                                         ctypes.c_float, ctypes.c_int32, P, P, P, P]
        L.attn_decode_static.restype = ctypes.c_int
        L.decode_step.argtypes = [ctypes.POINTER(_Config), P, ctypes.c_int32, P, P, P, ctypes.c_int32, P, P,
                                  ctypes.c_int32, P, P, ctypes.c_float, ctypes.c_int32, P, P, P, ctypes.c_uint64, P, P]
        L.decode_step.restype = ctypes.c_int
        L.oscar_kv_set_profile_events.argtypes = [P, P]
        L.oscar_kv_set_profile_events.restype = ctypes.c_int
        L.oscar_kv_set_wait_test.argtypes = [ctypes.c_uint64, ctypes.c_int32]
        L.oscar_kv_set_wait_test.restype = ctypes.c_int
        L.oscar_kv_decode_kernels.argtypes = [ctypes.POINTER(_Config)]
        L.oscar_kv_decode_kernels.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(t):
    """Device address of a tensor argument (None -> NULL).  The library's kernels
    read it as a dense array in device memory, so a host tensor or a strided view
    is refused here instead of reaching the GPU."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"oscar_kv: expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError("oscar_kv: expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _check(t, name: str, dtypes, shape=None, min_bytes=None, optional: bool = False):
    """Refuse, before anything reaches the GPU, a tensor whose dtype, shape or
    size does not match what the library will read or write through it."""
    if t is None:
        if optional:
            return
        raise ValueError(f"oscar_kv: {name} is required")
    if t.dtype not in dtypes:
        raise ValueError(f"oscar_kv: {name} must be {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"oscar_kv: {name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if min_bytes is not None and t.numel() * t.element_size() < min_bytes:
        raise ValueError(f"oscar_kv: {name} holds {t.numel() * t.element_size()} bytes, needs {min_bytes}")


def _dt():
    import torch
    return torch


def _check_cache(cfg: "KVConfig", cache):
    torch = _dt()
    _check(cache, "cache", (torch.uint8,), min_bytes=layout_query(cfg)["total_bytes"])


def _check_rot(cfg: "KVConfig", R, name: str):
    torch = _dt()
    # with the in-quant Hadamard the matrices are not read (None allowed)
    _check(R, name, (torch.float32,), min_bytes=cfg.head_dim * cfg.head_dim * 4,
           optional=bool(cfg.flags & FLAG_HADAMARD))


def _in_dtypes(cfg: "KVConfig"):
    torch = _dt()
    return (torch.float32,) if cfg.flags & FLAG_IN_FP32 else (torch.bfloat16,)


def _check_decode_io(cfg: "KVConfig", q, seq_lens, out, lse, status):
    torch = _dt()
    B, Hq, D = cfg.batch, cfg.num_q_heads, cfg.head_dim
    _check(q, "q", _in_dtypes(cfg), shape=(B, Hq, D))
    _check(seq_lens, "seq_lens", (torch.int32,), shape=(B,))
    _check(out, "out", (torch.float32,) if cfg.flags & FLAG_OUT_FP32 else (torch.bfloat16,), shape=(B, Hq, D))
    _check(lse, "lse", (torch.float32,), min_bytes=B * Hq * 4, optional=True)
    _check(status, "status", (torch.int32,), min_bytes=4, optional=True)


def _check_append_io(cfg: "KVConfig", k_new, v_new, start_pos, debug_rot, status):
    torch = _dt()
    B, H, D = cfg.batch, cfg.num_kv_heads, cfg.head_dim
    if k_new is None or k_new.dim() != 4:
        raise ValueError("oscar_kv: k_new must be [batch][n_new][num_kv_heads][head_dim]")
    n = int(k_new.shape[1])
    _check(k_new, "k_new", _in_dtypes(cfg), shape=(B, n, H, D))
    _check(v_new, "v_new", _in_dtypes(cfg), shape=(B, n, H, D))
    _check(start_pos, "start_pos", (torch.int32,), shape=(B,))
    _check(debug_rot, "debug_rot", (torch.float32,), min_bytes=B * n * H * 2 * D * 4, optional=True)
    _check(status, "status", (torch.int32,), min_bytes=4, optional=True)


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def layout_query(cfg: KVConfig) -> dict:
    out = _Layout()
    rc = lib().kv_layout_query(ctypes.byref(cfg.c()), ctypes.byref(out))
    if rc != 0:
        raise OscarError("kv_layout_query", rc)
    return {name: getattr(out, name) for name, _ in _Layout._fields_}


def kv_append(cfg: KVConfig, cache, layer: int, k_new, v_new, start_pos, R_K, R_V, debug_rot=None,
              status=None, stream=None, check: bool = True) -> int:
    _check_append_io(cfg, k_new, v_new, start_pos, debug_rot, status)
    _check_cache(cfg, cache)
    _check_rot(cfg, R_K, "R_K")
    _check_rot(cfg, R_V, "R_V")
    rc = lib().kv_append(ctypes.byref(cfg.c()), _ptr(cache), layer, _ptr(k_new), _ptr(v_new), _ptr(start_pos),
                         int(k_new.shape[1]), _ptr(R_K), _ptr(R_V), _ptr(debug_rot), _ptr(status), _stream(stream))
    if check and rc != 0:
        raise OscarError("kv_append", rc)
    return rc


def attn_decode(cfg: KVConfig, cache, layer: int, q, seq_lens, R_K, R_V, out, workspace, lse=None,
                seq_len_hint: int = 0, sm_scale: float = 0.0, num_splits: int = 0, status=None, stream=None,
                check: bool = True) -> int:
    _check_decode_io(cfg, q, seq_lens, out, lse, status)
    _check_cache(cfg, cache)
    _check_rot(cfg, R_K, "R_K")
    _check_rot(cfg, R_V, "R_V")
    _check(workspace, "workspace", (_dt().uint8,))
    rc = lib().attn_decode(ctypes.byref(cfg.c()), _ptr(cache), layer, _ptr(q), _ptr(seq_lens), int(seq_len_hint),
                           _ptr(R_K), _ptr(R_V), float(sm_scale), int(num_splits), _ptr(out), _ptr(lse),
                           _ptr(workspace), int(workspace.numel() * workspace.element_size()), _ptr(status),
                           _stream(stream))
    if check and rc != 0:
        raise OscarError("attn_decode", rc)
    return rc


def decode_step(cfg: KVConfig, cache, layer: int, k_new, v_new, start_pos, q, seq_lens, R_K, R_V, out, workspace,
                lse=None, seq_len_hint: int = 0, sm_scale: float = 0.0, num_splits: int = 0, status=None,
                stream=None, check: bool = True) -> int:
    """kv_append of k_new/v_new ([B][n][Hkv][D]) at start_pos, then attn_decode, in one call."""
    _check_append_io(cfg, k_new, v_new, start_pos, None, status)
    _check_decode_io(cfg, q, seq_lens, out, lse, status)
    _check_cache(cfg, cache)
    _check_rot(cfg, R_K, "R_K")
    _check_rot(cfg, R_V, "R_V")
    _check(workspace, "workspace", (_dt().uint8,))
    n_new = int(k_new.shape[1])
    rc = lib().decode_step(ctypes.byref(cfg.c()), _ptr(cache), layer, _ptr(k_new), _ptr(v_new), _ptr(start_pos),
                           n_new, _ptr(q), _ptr(seq_lens), int(seq_len_hint), _ptr(R_K), _ptr(R_V), float(sm_scale),
                           int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace),
                           int(workspace.numel() * workspace.element_size()), _ptr(status), _stream(stream))
    if check and rc != 0:
        raise OscarError("decode_step", rc)
    return rc


def attn_decode_static(cfg: KVConfig, cache, layer: int, q, seq_lens, R_K, R_V, out, lse=None,
                       seq_len_hint: int = 0, sm_scale: float = 0.0, num_splits: int = 0, status=None, stream=None,
                       check: bool = True) -> int:
    """attn_decode with the library's fixed scratch array (no workspace argument)."""
    _check_decode_io(cfg, q, seq_lens, out, lse, status)
    _check_cache(cfg, cache)
    _check_rot(cfg, R_K, "R_K")
    _check_rot(cfg, R_V, "R_V")
    rc = lib().attn_decode_static(ctypes.byref(cfg.c()), _ptr(cache), layer, _ptr(q), _ptr(seq_lens),
                                  int(seq_len_hint), _ptr(R_K), _ptr(R_V), float(sm_scale), int(num_splits),
                                  _ptr(out), _ptr(lse), _ptr(status), _stream(stream))
    if check and rc != 0:
        raise OscarError("attn_decode_static", rc)
    return rc


def set_profile_events(start=None, stop=None) -> None:
    """Record torch.cuda.Event pair around the split kernel of later attn_decode calls (None, None stops)."""
    lib().oscar_kv_set_profile_events(None if start is None else ctypes.c_void_p(start.cuda_event),
                                      None if stop is None else ctypes.c_void_p(stop.cuda_event))


def decode_kernels(cfg: KVConfig) -> int:
    """Kernels one attn_decode call launches (see oscar_kv_decode_kernels)."""
    rc = lib().oscar_kv_decode_kernels(ctypes.byref(cfg.c()))
    if rc < 0:
        raise OscarError("oscar_kv_decode_kernels", rc)
    return rc


def set_wait_test(wait_ns: int = 0, extra_bytes: int = 0) -> None:
    """Timeout-path test hook (see oscar_kv_set_wait_test); (0, 0) restores normal operation."""
    rc = lib().oscar_kv_set_wait_test(int(wait_ns), int(extra_bytes))
    if rc != 0:
        raise OscarError("oscar_kv_set_wait_test", rc)


def _calib_fns():
    L = lib()
    if not getattr(L, "_calib_ready", False):
        L.oscar_calibrate_workspace_query.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_uint64)]
        L.oscar_calibrate_workspace_query.restype = ctypes.c_int
        L.oscar_calibrate_rk.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
        L.oscar_calibrate_rk.restype = ctypes.c_int
        L.oscar_calibrate_rv_workspace_query.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint64)]
        L.oscar_calibrate_rv_workspace_query.restype = ctypes.c_int
        L.oscar_calibrate_rv.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
        L.oscar_calibrate_rv.restype = ctypes.c_int
        L._calib_ready = True
    return L


def calibrate_workspace_bytes(head_dim: int) -> int:
    n = ctypes.c_uint64(0)
    rc = _calib_fns().oscar_calibrate_workspace_query(int(head_dim), ctypes.byref(n))
    if rc != 0:
        raise OscarError("oscar_calibrate_workspace_query", rc)
    return int(n.value)


def calibrate_rk(q, R_out, workspace, status=None, stream=None, check: bool = True) -> int:
    """R_K fitted to the float32 query rows q [n][D] (see oscar_calibrate_rk); writes R_out [D][D]."""
    torch = _dt()
    if q is None or q.dim() != 2:
        raise ValueError("oscar_kv: q must be [n_rows][head_dim] float32")
    n, d = int(q.shape[0]), int(q.shape[1])
    _check(q, "q", (torch.float32,))
    _check(R_out, "R_out", (torch.float32,), shape=(d, d))
    _check(workspace, "workspace", (torch.uint8,))
    _check(status, "status", (torch.int32,), min_bytes=4, optional=True)
    rc = _calib_fns().oscar_calibrate_rk(_ptr(q), n, d, _ptr(R_out), _ptr(workspace),
                                         int(workspace.numel() * workspace.element_size()), _ptr(status),
                                         _stream(stream))
    if check and rc != 0:
        raise OscarError("oscar_calibrate_rk", rc)
    return rc


def calibrate_rv_workspace_bytes(head_dim: int, n_kv_rows: int) -> int:
    n = ctypes.c_uint64(0)
    rc = _calib_fns().oscar_calibrate_rv_workspace_query(int(head_dim), int(n_kv_rows), ctypes.byref(n))
    if rc != 0:
        raise OscarError("oscar_calibrate_rv_workspace_query", rc)
    return int(n.value)


def calibrate_rv(q, k, v, R_out, workspace, status=None, stream=None, check: bool = True) -> int:
    """R_V fitted to the score-weighted covariance of the float32 value rows v [n][D],
    each weighted by k_t q^T q k_t^T (see oscar_calibrate_rv); writes R_out [D][D]."""
    torch = _dt()
    if q is None or q.dim() != 2 or k is None or k.dim() != 2:
        raise ValueError("oscar_kv: q and k must be [n_rows][head_dim] float32")
    nq, d = int(q.shape[0]), int(q.shape[1])
    nkv = int(k.shape[0])
    if v is None or tuple(k.shape) != tuple(v.shape) or int(k.shape[1]) != d:
        raise ValueError("k and v must both be [n_kv][head_dim] with the head_dim of q")
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, name, (torch.float32,))
    _check(R_out, "R_out", (torch.float32,), shape=(d, d))
    _check(workspace, "workspace", (torch.uint8,))
    _check(status, "status", (torch.int32,), min_bytes=4, optional=True)
    rc = _calib_fns().oscar_calibrate_rv(_ptr(q), nq, _ptr(k), _ptr(v), nkv, d, _ptr(R_out), _ptr(workspace),
                                         int(workspace.numel() * workspace.element_size()), _ptr(status),
                                         _stream(stream))
    if check and rc != 0:
        raise OscarError("oscar_calibrate_rv", rc)
    return rc
