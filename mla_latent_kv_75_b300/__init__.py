"""Python binding of libmla.so: Multi-head Latent Attention over a latent KV cache on B300.

A thin ctypes layer: every function has the name and argument order of the C entry point
declared in ``include/mla.h`` and only marshals arguments (torch tensors become device
pointers, the current torch stream becomes the cudaStream_t). All arithmetic runs in the
library's CUDA kernels. There is no CPU fallback: importing this package fails if the
library has not been built (``python mla_latent_kv_75_b300/build.py``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libmla.so is not built; run `python mla_latent_kv_75_b300/build.py` "
                      "(the CUDA library is required, there is no fallback)")

_lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------------------- ABI types
MLA_F32 = 0
MLA_BF16 = 1

STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CAPACITY",
          4: "MLA_ERR_MISALIGNED", 5: "MLA_ERR_CUDA", 6: "MLA_ERR_TIMEOUT",
          7: "MLA_ERR_WORKSPACE", 8: "MLA_ERR_LENGTH"}


class MlaDims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("n_h", ctypes.c_int32), ("d_hc", ctypes.c_int32),
                ("d_hr", ctypes.c_int32), ("d_c", ctypes.c_int32), ("d_cq", ctypes.c_int32),
                ("rope_base", ctypes.c_float), ("scale", ctypes.c_float),
                ("dtype", ctypes.c_int32)]


class MlaWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("W_DQ", "W_UQ", "W_QR", "W_DKV", "W_KR", "W_UK", "W_UV")]


class MlaCache(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_void_p), ("seq_base", ctypes.c_void_p),
                ("capacity", ctypes.c_int64)]


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (%s)" % (where, STATUS.get(status, status),
                                          mla_status_string(status)))


_P = ctypes.c_void_p
_I = ctypes.c_int32
_PD, _PW, _PC = ctypes.POINTER(MlaDims), ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaCache)
_SZ = ctypes.POINTER(ctypes.c_size_t)

_SIGS = {
    "mla_append_cache": [_PD, _PW, _P, _P, _P, _I, _PC, _P],
    "mla_project_q_workspace_size": [_PD, _I, _SZ],
    "mla_project_q": [_PD, _PW, _P, _P, _I, _P, ctypes.c_size_t, _P, _P, _P],
    "mla_decode_workspace_size": [_PD, _I, _I, _SZ],
    "mla_decode_absorbed": [_PD, _PW, _P, _P, _PC, _P, _I, _I, _P, ctypes.c_size_t, _P, _P],
    "mla_prefill_workspace_size": [_PD, _I, _I, _I, _SZ],
    "mla_prefill": [_PD, _PW, _P, _P, _I, _I, _I, _PC, _P, ctypes.c_size_t, _P, _P],
    "mla_decode_absorbed_static": [_PD, _PW, _P, _P, _PC, _P, _I, _I, _P, _P],
    "mla_project_q_absorbed": [_PD, _PW, _P, _P, _I, _P, ctypes.c_size_t, _P, _P, _P],
    "mla_decode_absorbed_latent": [_PD, _PW, _P, _P, _PC, _P, _I, _I, _P, ctypes.c_size_t, _P,
                                   _P],
    "mla_decode_step_workspace_size": [_PD, _I, _I, _SZ],
    "mla_output_projection_workspace_size": [_PD, _I, _SZ],
    "mla_merge_query_absorption": [_PD, _P, _P, _P, _P],
    "mla_project_q_premerged": [_PD, _PW, _P, _P, _P, _I, _P, ctypes.c_size_t, _P, _P, _P],
    "mla_output_projection": [_PD, _P, _P, _I, _P, ctypes.c_size_t, _P, _P],
    "mla_decode_step": [_PD, _PW, _P, _P, _PC, _P, _I, _I, _P, ctypes.c_size_t, _P, _P],
    "mla_select_topk": [_P, ctypes.c_int64, _P, _I, _I, _I, _P, _P, _P],
    "mla_decode_sparse_workspace_size": [_PD, _I, _I, _SZ],
    "mla_decode_absorbed_sparse": [_PD, _PW, _P, _P, _PC, _P, _I, _I, _P, ctypes.c_int64, _I, _P,
                                   ctypes.c_size_t, _P, _P],
    "mla_get_device_status": [_P],
    "mla_fast_path": [_PD],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int32
_lib.mla_debug_arm_wait_timeout.argtypes = [ctypes.c_int64]
_lib.mla_debug_arm_wait_timeout.restype = ctypes.c_int32
_lib.mla_status_string.argtypes = [ctypes.c_int32]
_lib.mla_status_string.restype = ctypes.c_char_p
_lib.mla_trace_arm.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int32),
                               ctypes.c_int32]
_lib.mla_trace_arm.restype = ctypes.c_int32
_lib.mla_trace_disarm.argtypes = []
_lib.mla_trace_disarm.restype = ctypes.c_int32
_lib.mla_kernel_name.argtypes = [ctypes.c_int32]
_lib.mla_kernel_name.restype = ctypes.c_char_p


# ----------------------------------------------------------------------------- marshalling
def _ptr(x) -> Optional[int]:
    """Device pointer of a torch tensor (or pass an int / None through)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MLAError(status, where)


def make_dims(d: int, n_h: int, d_hc: int, d_hr: int, d_c: int, d_cq: int,
              dtype: int = MLA_BF16, rope_base: float = 10000.0, scale: float = 0.0) -> MlaDims:
    return MlaDims(d, n_h, d_hc, d_hr, d_c, d_cq, rope_base, scale, dtype)


def make_weights(W: Dict[str, object]) -> MlaWeights:
    return MlaWeights(*[_ptr(W.get(n)) for n in
                        ("W_DQ", "W_UQ", "W_QR", "W_DKV", "W_KR", "W_UK", "W_UV")])


def make_cache(rows, seq_base, capacity: Optional[int] = None) -> MlaCache:
    if capacity is None:
        capacity = rows.shape[0]
    return MlaCache(_ptr(rows), _ptr(seq_base), int(capacity))


# ----------------------------------------------------------------------------- entry points
def mla_status_string(status: int) -> str:
    return _lib.mla_status_string(int(status)).decode()


def mla_fast_path(dims: MlaDims) -> int:
    return int(_lib.mla_fast_path(ctypes.byref(dims)))


def mla_append_cache(dims, weights, h, seq_idx, pos, n, cache, stream=None) -> None:
    _check(_lib.mla_append_cache(ctypes.byref(dims), ctypes.byref(weights), _ptr(h),
                                 _ptr(seq_idx), _ptr(pos), int(n), ctypes.byref(cache),
                                 _stream(stream)), "mla_append_cache")


def mla_project_q_workspace_size(dims, n) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.mla_project_q_workspace_size(ctypes.byref(dims), int(n), ctypes.byref(out)),
           "mla_project_q_workspace_size")
    return out.value


def mla_project_q(dims, weights, h, pos, n, ws, ws_bytes, q_c, q_r, stream=None) -> None:
    _check(_lib.mla_project_q(ctypes.byref(dims), ctypes.byref(weights), _ptr(h), _ptr(pos),
                              int(n), _ptr(ws), int(ws_bytes), _ptr(q_c), _ptr(q_r),
                              _stream(stream)), "mla_project_q")


def mla_decode_workspace_size(dims, B, max_len) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.mla_decode_workspace_size(ctypes.byref(dims), int(B), int(max_len),
                                          ctypes.byref(out)), "mla_decode_workspace_size")
    return out.value


def mla_decode_absorbed(dims, weights, q_c, q_r, cache, seq_len, B, max_len, ws, ws_bytes, o,
                        stream=None) -> None:
    _check(_lib.mla_decode_absorbed(ctypes.byref(dims), ctypes.byref(weights), _ptr(q_c),
                                    _ptr(q_r), ctypes.byref(cache), _ptr(seq_len), int(B),
                                    int(max_len), _ptr(ws), int(ws_bytes), _ptr(o),
                                    _stream(stream)), "mla_decode_absorbed")


def mla_project_q_absorbed(dims, weights, h, pos, n, ws, ws_bytes, q_t, q_r, stream=None) -> None:
    _check(_lib.mla_project_q_absorbed(ctypes.byref(dims), ctypes.byref(weights), _ptr(h),
                                       _ptr(pos), int(n), _ptr(ws), int(ws_bytes), _ptr(q_t),
                                       _ptr(q_r), _stream(stream)), "mla_project_q_absorbed")


def mla_decode_absorbed_latent(dims, weights, q_t, q_r, cache, seq_len, B, max_len, ws, ws_bytes,
                               o, stream=None) -> None:
    _check(_lib.mla_decode_absorbed_latent(ctypes.byref(dims), ctypes.byref(weights), _ptr(q_t),
                                           _ptr(q_r), ctypes.byref(cache), _ptr(seq_len),
                                           int(B), int(max_len), _ptr(ws), int(ws_bytes),
                                           _ptr(o), _stream(stream)), "mla_decode_absorbed_latent")


def mla_decode_step_workspace_size(dims, B, max_len) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.mla_decode_step_workspace_size(ctypes.byref(dims), int(B), int(max_len),
                                               ctypes.byref(out)), "mla_decode_step_workspace_size")
    return out.value


def mla_decode_step(dims, weights, h, pos, cache, seq_len, B, max_len, ws, ws_bytes, o,
                    stream=None) -> None:
    _check(_lib.mla_decode_step(ctypes.byref(dims), ctypes.byref(weights), _ptr(h), _ptr(pos),
                                ctypes.byref(cache), _ptr(seq_len), int(B), int(max_len),
                                _ptr(ws), int(ws_bytes), _ptr(o), _stream(stream)),
           "mla_decode_step")


def mla_merge_query_absorption(dims, W_UQ, W_UK, W_UQK, stream=None) -> None:
    _check(_lib.mla_merge_query_absorption(ctypes.byref(dims), _ptr(W_UQ), _ptr(W_UK),
                                           _ptr(W_UQK), _stream(stream)),
           "mla_merge_query_absorption")


def mla_project_q_premerged(dims, weights, W_UQK, h, pos, n, ws, ws_bytes, q_t, q_r,
                            stream=None) -> None:
    _check(_lib.mla_project_q_premerged(ctypes.byref(dims), ctypes.byref(weights), _ptr(W_UQK),
                                        _ptr(h), _ptr(pos), int(n), _ptr(ws), int(ws_bytes),
                                        _ptr(q_t), _ptr(q_r), _stream(stream)),
           "mla_project_q_premerged")


def mla_output_projection_workspace_size(dims, n) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.mla_output_projection_workspace_size(ctypes.byref(dims), int(n),
                                                     ctypes.byref(out)),
           "mla_output_projection_workspace_size")
    return out.value


def mla_output_projection(dims, W_O, o, n, ws, ws_bytes, u, stream=None) -> None:
    _check(_lib.mla_output_projection(ctypes.byref(dims), _ptr(W_O), _ptr(o), int(n), _ptr(ws),
                                      int(ws_bytes), _ptr(u), _stream(stream)),
           "mla_output_projection")


def mla_select_topk(scores, score_stride, seq_len, B, max_len, k, sel_pos, sel_count,
                    stream=None) -> None:
    _check(_lib.mla_select_topk(_ptr(scores), int(score_stride), _ptr(seq_len), int(B),
                                int(max_len), int(k), _ptr(sel_pos), _ptr(sel_count),
                                _stream(stream)), "mla_select_topk")


def mla_decode_sparse_workspace_size(dims, B, k) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.mla_decode_sparse_workspace_size(ctypes.byref(dims), int(B), int(k),
                                                 ctypes.byref(out)),
           "mla_decode_sparse_workspace_size")
    return out.value


def mla_decode_absorbed_sparse(dims, weights, q_c, q_r, cache, seq_len, B, max_len, scores,
                               score_stride, k, ws, ws_bytes, o, stream=None) -> None:
    _check(_lib.mla_decode_absorbed_sparse(ctypes.byref(dims), ctypes.byref(weights), _ptr(q_c),
                                           _ptr(q_r), ctypes.byref(cache), _ptr(seq_len),
                                           int(B), int(max_len), _ptr(scores),
                                           int(score_stride), int(k), _ptr(ws), int(ws_bytes),
                                           _ptr(o), _stream(stream)),
           "mla_decode_absorbed_sparse")


MLA_STATIC_WS_BYTES = 32 << 20


def mla_decode_absorbed_static(dims, weights, q_c, q_r, cache, seq_len, B, max_len, o,
                               stream=None) -> None:
    """mla_decode_absorbed with the library's built-in scratch array instead of a caller
    workspace (for callers that cannot allocate device memory)."""
    _check(_lib.mla_decode_absorbed_static(ctypes.byref(dims), ctypes.byref(weights), _ptr(q_c),
                                           _ptr(q_r), ctypes.byref(cache), _ptr(seq_len),
                                           int(B), int(max_len), _ptr(o), _stream(stream)),
           "mla_decode_absorbed_static")


def mla_prefill_workspace_size(dims, n_tok, B, max_T) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.mla_prefill_workspace_size(ctypes.byref(dims), int(n_tok), int(B), int(max_T),
                                           ctypes.byref(out)), "mla_prefill_workspace_size")
    return out.value


def mla_prefill(dims, weights, h, cu_seqlens, B, n_tok, max_T, cache, ws, ws_bytes, o,
                stream=None) -> None:
    _check(_lib.mla_prefill(ctypes.byref(dims), ctypes.byref(weights), _ptr(h),
                            _ptr(cu_seqlens), int(B), int(n_tok), int(max_T),
                            ctypes.byref(cache), _ptr(ws), int(ws_bytes), _ptr(o),
                            _stream(stream)), "mla_prefill")


def mla_debug_arm_wait_timeout(limit_ns: int) -> None:
    """Make the next decode attention launch's bounded wait run out after limit_ns (test hook)."""
    _check(_lib.mla_debug_arm_wait_timeout(int(limit_ns)), "mla_debug_arm_wait_timeout")


def mla_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(_lib.mla_get_device_status(_stream(stream)))


def mla_kernel_name(kernel_id: int) -> str:
    return _lib.mla_kernel_name(int(kernel_id)).decode()


class KernelTrace:
    """Records a CUDA event pair around each of the next ``capacity`` kernel launches the
    library makes (mla_trace_arm / mla_trace_disarm); ``launches()`` then gives
    (kernel name, milliseconds) per launch."""

    def __init__(self, capacity: int):
        import torch
        self.capacity = capacity
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.events:  # materialise the cudaEvent_t handles
            e.record()
        torch.cuda.synchronize()
        self._handles = (ctypes.c_void_p * (2 * capacity))(*[e.cuda_event for e in self.events])
        self._ids = (ctypes.c_int32 * capacity)()
        self.count = 0

    def __enter__(self):
        _check(_lib.mla_trace_arm(self._handles, self._ids, self.capacity), "mla_trace_arm")
        return self

    def __exit__(self, *exc):
        self.count = int(_lib.mla_trace_disarm())
        return False

    def launches(self):
        """Call after synchronising the device."""
        return [(mla_kernel_name(self._ids[k]),
                 self.events[2 * k].elapsed_time(self.events[2 * k + 1]))
                for k in range(self.count)]


def raw_status(fn_name: str, *args) -> int:
    """Call an entry point with raw ctypes arguments and return its status code (tests)."""
    return int(getattr(_lib, fn_name)(*args))


def lib() -> ctypes.CDLL:
    return _lib
