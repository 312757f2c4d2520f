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
           "oscar_kv_set_profile_events", "oscar_calibrate_workspace_query", "oscar_calibrate_rk",
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
    rc = lib().kv_append(ctypes.byref(cfg.c()), _ptr(cache), layer, _ptr(k_new), _ptr(v_new), _ptr(start_pos),
                         int(k_new.shape[1]), _ptr(R_K), _ptr(R_V), _ptr(debug_rot), _ptr(status), _stream(stream))
    if check and rc != 0:
        raise OscarError("kv_append", rc)
    return rc


def attn_decode(cfg: KVConfig, cache, layer: int, q, seq_lens, R_K, R_V, out, workspace, lse=None,
                seq_len_hint: int = 0, sm_scale: float = 0.0, num_splits: int = 0, status=None, stream=None,
                check: bool = True) -> int:
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
    n, d = int(q.shape[0]), int(q.shape[1])
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
    nq, d = int(q.shape[0]), int(q.shape[1])
    nkv = int(k.shape[0])
    if tuple(k.shape) != tuple(v.shape) or int(k.shape[1]) != d:
        raise ValueError("k and v must both be [n_kv][head_dim] with the head_dim of q")
    rc = _calib_fns().oscar_calibrate_rv(_ptr(q), nq, _ptr(k), _ptr(v), nkv, d, _ptr(R_out), _ptr(workspace),
                                         int(workspace.numel() * workspace.element_size()), _ptr(status),
                                         _stream(stream))
    if check and rc != 0:
        raise OscarError("oscar_calibrate_rv", rc)
    return rc
