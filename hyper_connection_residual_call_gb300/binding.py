"""Thin Python binding of the C ABI in ``include/ts_hc.h`` (ctypes).

Two layers, both argument marshalling only -- every step of the computation
runs in the library's CUDA kernels:

* ``ts_hc_*``: the C entry points under their own names, taking raw device
  pointers (ints), a ``TsWeight`` struct and a CUDA stream handle; they return
  the ``ts_status`` code.
* ``hc_call`` / ``hc_inject_call`` / ``hc_mixer`` / ``hc_inject_add`` /
  ``hc_replicate_entry`` / ``hc_stack``: the same calls for torch CUDA
  tensors. They allocate outputs/workspace with torch when not given, pass
  the current torch stream, and raise ``HCError`` on any error status.

There is no fallback: if the library is not built or cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

from .build import LIB_PATH

TS_OK, TS_ERR_INVALID_ARG, TS_ERR_UNSUPPORTED, TS_ERR_CUDA, TS_ERR_WORKSPACE, TS_ERR_TIMEOUT = range(6)
TS_W_BF16, TS_W_INT4_AFFINE = 0, 1
RMS_EPS = 1e-6  # families/qwen4/mod.rs, RMS_EPS

EXPORTS = ("ts_hc_workspace_bytes", "ts_hc_workspace_layout", "ts_hc_call", "ts_hc_inject_add",
           "ts_hc_mixer", "ts_hc_call_debug", "ts_hc_inject_call", "ts_hc_entry_call", "ts_hc_exit_logits",
           "ts_hc_replicate_entry", "ts_hc_ple_workspace_bytes", "ts_hc_ple_workspace_layout", "ts_hc_ple",
           "ts_hc_last_error",
           "ts_hc_device_status", "ts_hc_call_noalloc", "ts_hc_stack_workspace_bytes", "ts_hc_stack",
           "ts_hc_stack_ple_workspace_bytes", "ts_hc_stack_ple", "ts_hc_selftest_timeout")
TS_HC_STATIC_SCRATCH_BYTES = 64 * 1024 * 1024  # include/ts_hc.h


class HCError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"ts_hc status {status}: {message}")
        self.status = status


class TsWeight(ctypes.Structure):
    _fields_ = [
        ("type", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("data", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("biases", ctypes.c_void_p),
    ]


class TsHcModule(ctypes.Structure):
    """``ts_hc_module``: one hyper-connection module's hc_norm weight and linears."""
    _fields_ = [
        ("hc_norm_w", ctypes.c_void_p),
        ("down", TsWeight),
        ("up", TsWeight),
        ("inject", TsWeight),
    ]


class TsHcPleModule(ctypes.Structure):
    """``ts_hc_ple_module``: a stack's PLE tensors."""
    _fields_ = [
        ("table", ctypes.c_void_p),
        ("n_rows", ctypes.c_long),
        ("key_proj", ctypes.c_void_p),
        ("value_proj", ctypes.c_void_p),
        ("norm_key_w", ctypes.c_void_p),
        ("norm_query_w", ctypes.c_void_p),
        ("norm_conv_w", ctypes.c_void_p),
        ("conv_w", ctypes.c_void_p),
    ]


# ts_hc_sublayer_fn: (user, layer, which, t0, M, mixed, &out, stream) -> ts_status
SUBLAYER_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p)

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load ``libts_hc.so`` (once). Raises if it is missing: there is no fallback."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library {p} is not built; run hyper_connection_residual_call_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i, l, sz, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_size_t, ctypes.c_float
        wp = ctypes.POINTER(TsWeight)
        lib.ts_hc_workspace_bytes.argtypes = [i, i, i, i]
        lib.ts_hc_workspace_bytes.restype = sz
        lib.ts_hc_workspace_layout.argtypes = [i, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
        lib.ts_hc_workspace_layout.restype = i
        lib.ts_hc_call.argtypes = [vp, vp, wp, wp, wp, vp, vp, l, i, i, i, i, f, vp, sz, vp]
        lib.ts_hc_call.restype = i
        lib.ts_hc_mixer.argtypes = [vp, vp, wp, wp, vp, i, i, i, i, f, vp, sz, vp]
        lib.ts_hc_mixer.restype = i
        lib.ts_hc_call_debug.argtypes = [vp, vp, wp, wp, wp, vp, vp, l, i, i, i, i, f, vp, sz, vp, vp]
        lib.ts_hc_call_debug.restype = i
        lib.ts_hc_inject_add.argtypes = [vp, vp, vp, l, i, i, i, vp]
        lib.ts_hc_inject_add.restype = i
        lib.ts_hc_inject_call.argtypes = [vp, vp, vp, l, vp, wp, wp, wp, vp, vp, l, i, i, i, i, f, vp, sz, vp]
        lib.ts_hc_inject_call.restype = i
        lib.ts_hc_entry_call.argtypes = [vp, vp, vp, wp, wp, wp, vp, vp, l, i, i, i, i, f, vp, sz, vp]
        lib.ts_hc_entry_call.restype = i
        lib.ts_hc_exit_logits.argtypes = [vp, vp, vp, l, vp, wp, wp, vp, i, vp, vp, i, i, i, i, f, vp, sz, vp]
        lib.ts_hc_exit_logits.restype = i
        lib.ts_hc_ple_workspace_bytes.argtypes = [i, i, i]
        lib.ts_hc_ple_workspace_bytes.restype = sz
        lib.ts_hc_ple_workspace_layout.argtypes = [i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz), ctypes.POINTER(sz)]
        lib.ts_hc_ple_workspace_layout.restype = i
        lib.ts_hc_ple.argtypes = [vp, vp, vp, l, vp, vp, vp, vp, vp, vp, vp, i, i, i, f, vp, sz, vp]
        lib.ts_hc_ple.restype = i
        lib.ts_hc_call_noalloc.argtypes = [vp, vp, wp, wp, wp, vp, vp, l, i, i, i, i, f, vp]
        lib.ts_hc_call_noalloc.restype = i
        lib.ts_hc_replicate_entry.argtypes = [vp, vp, i, i, i, vp]
        lib.ts_hc_replicate_entry.restype = i
        mp = ctypes.POINTER(TsHcModule)
        lib.ts_hc_stack_workspace_bytes.argtypes = [i, i, i, i]
        lib.ts_hc_stack_workspace_bytes.restype = sz
        lib.ts_hc_stack.argtypes = [vp, i, mp, mp, i, mp, SUBLAYER_FN, vp, vp, i, i, i, i, f, vp, sz, vp]
        lib.ts_hc_stack.restype = i
        lib.ts_hc_stack_ple_workspace_bytes.argtypes = [i, i, i, i]
        lib.ts_hc_stack_ple_workspace_bytes.restype = sz
        lib.ts_hc_stack_ple.argtypes = [vp, i, mp, mp, i, mp, ctypes.POINTER(TsHcPleModule), vp, vp, SUBLAYER_FN,
                                        vp, vp, i, i, i, i, f, vp, sz, vp]
        lib.ts_hc_stack_ple.restype = i
        lib.ts_hc_selftest_timeout.argtypes = [vp]
        lib.ts_hc_selftest_timeout.restype = i
        lib.ts_hc_last_error.argtypes = []
        lib.ts_hc_last_error.restype = ctypes.c_char_p
        lib.ts_hc_device_status.argtypes = [vp, ctypes.POINTER(i)]
        lib.ts_hc_device_status.restype = i
        if path is None:
            _lib = lib
        return lib


# ------------------------------------------------------------- C names

def ts_hc_workspace_bytes(M: int, H: int, C: int, lowrank: int) -> int:
    return library().ts_hc_workspace_bytes(M, H, C, lowrank)


def ts_hc_workspace_layout(M: int, H: int, C: int, lowrank: int) -> Tuple[int, int]:
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    st = library().ts_hc_workspace_layout(M, H, C, lowrank, ctypes.byref(a), ctypes.byref(b))
    _check(st)
    return a.value, b.value


def ts_hc_call(raw, hc_norm_w, down, up, inject, mixed, inject_w, inject_stride, M, H, C, lowrank,
               eps, workspace, workspace_bytes, stream) -> int:
    return library().ts_hc_call(raw, hc_norm_w, _wref(down), _wref(up), _wref(inject), mixed, inject_w,
                                inject_stride, M, H, C, lowrank, eps, workspace, workspace_bytes, stream)


def ts_hc_mixer(raw, hc_norm_w, down, up, mixed, M, H, C, lowrank, eps, workspace, workspace_bytes,
                stream) -> int:
    return library().ts_hc_mixer(raw, hc_norm_w, _wref(down), _wref(up), mixed, M, H, C, lowrank, eps,
                                 workspace, workspace_bytes, stream)


def ts_hc_call_debug(raw, hc_norm_w, down, up, inject, mixed, inject_w, inject_stride, M, H, C, lowrank,
                     eps, workspace, workspace_bytes, w_out, stream) -> int:
    """ts_hc_call (ts_hc_mixer when ``inject`` is None) that also writes w = sigmoid(up(act))."""
    return library().ts_hc_call_debug(raw, hc_norm_w, _wref(down), _wref(up), _wref(inject), mixed, inject_w,
                                      inject_stride, M, H, C, lowrank, eps, workspace, workspace_bytes, w_out,
                                      stream)


def ts_hc_inject_add(raw, out, inject_w, inject_stride, M, H, C, stream) -> int:
    return library().ts_hc_inject_add(raw, out, inject_w, inject_stride, M, H, C, stream)


def ts_hc_inject_call(raw, out, prev_inject_w, prev_inject_stride, hc_norm_w, down, up, inject, mixed,
                      inject_w, inject_stride, M, H, C, lowrank, eps, workspace, workspace_bytes,
                      stream) -> int:
    return library().ts_hc_inject_call(raw, out, prev_inject_w, prev_inject_stride, hc_norm_w, _wref(down),
                                       _wref(up), _wref(inject), mixed, inject_w, inject_stride, M, H, C,
                                       lowrank, eps, workspace, workspace_bytes, stream)


def ts_hc_entry_call(emb, raw, hc_norm_w, down, up, inject, mixed, inject_w, inject_stride, M, H, C, lowrank,
                     eps, workspace, workspace_bytes, stream) -> int:
    """Entry replication fused into the first call: raw = repeat(emb, C), then the call on it."""
    return library().ts_hc_entry_call(emb, raw, hc_norm_w, _wref(down), _wref(up), _wref(inject), mixed, inject_w,
                                      inject_stride, M, H, C, lowrank, eps, workspace, workspace_bytes, stream)


def ts_hc_exit_logits(raw, out, prev_inject_w, prev_inject_stride, hc_norm_w, down, up, lm_head, V, mixed, logits,
                      M, H, C, lowrank, eps, workspace, workspace_bytes, stream) -> int:
    """The exit: (inject-add,) hyper_connection_mixer, then lm_head into fp32 logits."""
    return library().ts_hc_exit_logits(raw, out, prev_inject_w, prev_inject_stride, hc_norm_w, _wref(down), _wref(up),
                                       lm_head, V, mixed, logits, M, H, C, lowrank, eps, workspace, workspace_bytes,
                                       stream)


def ts_hc_ple_workspace_bytes(M: int, H: int, C: int) -> int:
    return library().ts_hc_ple_workspace_bytes(M, H, C)


def ts_hc_ple_workspace_layout(M: int, H: int, C: int) -> Tuple[int, int, int]:
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(library().ts_hc_ple_workspace_layout(M, H, C, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def ts_hc_ple(hidden, rows, table, n_rows, key_proj, value_proj, norm_key_w, norm_query_w, norm_conv_w, conv_w,
              conv_state, M, H, C, eps, workspace, workspace_bytes, stream) -> int:
    """The PLE gate added to the wide residual (in place), for M consecutive tokens."""
    return library().ts_hc_ple(hidden, rows, table, n_rows, key_proj, value_proj, norm_key_w, norm_query_w,
                               norm_conv_w, conv_w, conv_state, M, H, C, eps, workspace, workspace_bytes, stream)


def ts_hc_call_noalloc(raw, hc_norm_w, down, up, inject, mixed, inject_w, inject_stride, M, H, C, lowrank,
                       eps, stream) -> int:
    """ts_hc_call with its scratch in the library's own device array (no workspace argument),
    for callers that cannot allocate device memory."""
    return library().ts_hc_call_noalloc(raw, hc_norm_w, _wref(down), _wref(up), _wref(inject), mixed,
                                        inject_w, inject_stride, M, H, C, lowrank, eps, stream)


def ts_hc_replicate_entry(emb, raw, M, H, C, stream) -> int:
    return library().ts_hc_replicate_entry(emb, raw, M, H, C, stream)


def ts_hc_stack_workspace_bytes(max_chunk: int, H: int, C: int, lowrank: int) -> int:
    return library().ts_hc_stack_workspace_bytes(max_chunk, H, C, lowrank)


def ts_hc_stack(emb, T, attn, mlp, n_layers, final_mixer, sublayer, user, mixed_out, max_chunk, H, C, lowrank,
                eps, workspace, workspace_bytes, stream) -> int:
    """``attn`` / ``mlp``: ctypes arrays of ``TsHcModule`` (or None); ``final_mixer``: a
    ``TsHcModule`` (or None); ``sublayer``: a ``SUBLAYER_FN`` (or None)."""
    return library().ts_hc_stack(emb, T, attn, mlp, n_layers, _wref(final_mixer),
                                 sublayer if sublayer is not None else SUBLAYER_FN(), user, mixed_out,
                                 max_chunk, H, C, lowrank, eps, workspace, workspace_bytes, stream)


def ts_hc_stack_ple_workspace_bytes(max_chunk: int, H: int, C: int, lowrank: int) -> int:
    return library().ts_hc_stack_ple_workspace_bytes(max_chunk, H, C, lowrank)


def ts_hc_stack_ple(emb, T, attn, mlp, n_layers, final_mixer, ple, ple_rows, ple_conv_state, sublayer, user,
                    mixed_out, max_chunk, H, C, lowrank, eps, workspace, workspace_bytes, stream) -> int:
    """As ``ts_hc_stack``, with ``ple`` a ``TsHcPleModule`` (or None) and the row ids and
    conv state as device pointers."""
    return library().ts_hc_stack_ple(emb, T, attn, mlp, n_layers, _wref(final_mixer),
                                     None if ple is None else ctypes.byref(ple), ple_rows, ple_conv_state,
                                     sublayer if sublayer is not None else SUBLAYER_FN(), user, mixed_out,
                                     max_chunk, H, C, lowrank, eps, workspace, workspace_bytes, stream)


def ts_hc_selftest_timeout(stream) -> int:
    """Launches the failure-path self-test (a bounded wait that must give up)."""
    return library().ts_hc_selftest_timeout(stream)


def ts_hc_last_error() -> str:
    return library().ts_hc_last_error().decode()


def ts_hc_device_status(stream) -> Tuple[int, int]:
    v = ctypes.c_int()
    st = library().ts_hc_device_status(stream, ctypes.byref(v))
    return st, v.value


def _wref(w: Optional[TsWeight]):
    return None if w is None else ctypes.byref(w)


def _check(st: int) -> None:
    if st != TS_OK:
        raise HCError(st, ts_hc_last_error())


# ------------------------------------------------------------- torch layer

def _torch():
    import torch
    return torch


def _stream_handle(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def weight_struct(w) -> TsWeight:
    """A ``TsWeight`` for a weight with attributes kind, data, scale, bias, group
    (tensors already on the device)."""
    s = TsWeight()
    if w.kind == "bf16":
        s.type, s.group = TS_W_BF16, 0
        s.data = w.data.data_ptr()
    elif w.kind == "int4":
        s.type, s.group = TS_W_INT4_AFFINE, int(w.group)
        s.data, s.scales, s.biases = w.data.data_ptr(), w.scale.data_ptr(), w.bias.data_ptr()
    else:
        raise ValueError(f"unknown weight kind {w.kind!r}")
    return s


def _need(t, name, dtype, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise HCError(TS_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise HCError(TS_ERR_INVALID_ARG, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise HCError(TS_ERR_INVALID_ARG, f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise HCError(TS_ERR_INVALID_ARG, f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def workspace(M: int, H: int, C: int, L: int, device=None):
    torch = _torch()
    n = max(ts_hc_workspace_bytes(M, H, C, L), 256)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def hc_call(raw, weights, *, H: int, C: int, mixed=None, inject_w=None, inject_stride: Optional[int] = None,
            eps: float = RMS_EPS, ws=None, stream=None):
    """attn_hc / mlp_hc on raw [M, C*H] bf16 with ``weights`` (g, down, up, inject).

    Returns (mixed [M, H] bf16, inject_w fp32). With a caller-given ``inject_w``
    buffer and ``inject_stride``, token t's gates land at element t*inject_stride.
    """
    torch = _torch()
    M = raw.shape[0]
    L = weights.down.rows
    _need(raw, "raw", torch.bfloat16, (M, C * H))
    _need(weights.g, "hc_norm_w", torch.bfloat16, (C * H,))
    if mixed is None:
        mixed = torch.empty((M, H), dtype=torch.bfloat16, device=raw.device)
    _need(mixed, "mixed", torch.bfloat16, (M, H))
    if inject_w is None:
        inject_stride = C
        inject_w = torch.empty((max(M, 1), C), dtype=torch.float32, device=raw.device)
    if inject_stride is None:
        raise HCError(TS_ERR_INVALID_ARG, "inject_stride is required with a caller-given inject_w")
    if ws is None:
        ws = workspace(M, H, C, L, raw.device)
    st = ts_hc_call(raw.data_ptr(), weights.g.data_ptr(), weight_struct(weights.down),
                    weight_struct(weights.up), weight_struct(weights.inject), mixed.data_ptr(),
                    inject_w.data_ptr(), inject_stride, M, H, C, L, eps, ws.data_ptr(),
                    ws.numel() * ws.element_size(), _stream_handle(stream))
    _check(st)
    return mixed, inject_w


def hc_mixer(raw, weights, *, H: int, C: int, mixed=None, eps: float = RMS_EPS, ws=None, stream=None):
    """The final hyper_connection_mixer on raw [M, C*H] bf16; returns mixed [M, H] bf16."""
    torch = _torch()
    M = raw.shape[0]
    L = weights.down.rows
    _need(raw, "raw", torch.bfloat16, (M, C * H))
    _need(weights.g, "hc_norm_w", torch.bfloat16, (C * H,))
    if mixed is None:
        mixed = torch.empty((M, H), dtype=torch.bfloat16, device=raw.device)
    _need(mixed, "mixed", torch.bfloat16, (M, H))
    if ws is None:
        ws = workspace(M, H, C, L, raw.device)
    st = ts_hc_mixer(raw.data_ptr(), weights.g.data_ptr(), weight_struct(weights.down),
                     weight_struct(weights.up), mixed.data_ptr(), M, H, C, L, eps, ws.data_ptr(),
                     ws.numel() * ws.element_size(), _stream_handle(stream))
    _check(st)
    return mixed


def hc_call_debug(raw, weights, *, H: int, C: int, mixed=None, inject_w=None, inject_stride: Optional[int] = None,
                  eps: float = RMS_EPS, ws=None, w_out=None, stream=None):
    """``hc_call`` (or the mixer when ``weights.inject`` is None) through ``ts_hc_call_debug``.

    Returns (mixed, inject_w or None, w) with w = sigmoid(up(act)) fp32 [M, C*H].
    """
    torch = _torch()
    M = raw.shape[0]
    L = weights.down.rows
    _need(raw, "raw", torch.bfloat16, (M, C * H))
    _need(weights.g, "hc_norm_w", torch.bfloat16, (C * H,))
    if mixed is None:
        mixed = torch.empty((M, H), dtype=torch.bfloat16, device=raw.device)
    _need(mixed, "mixed", torch.bfloat16, (M, H))
    has_inject = weights.inject is not None
    if has_inject and inject_w is None:
        inject_stride = C
        inject_w = torch.empty((max(M, 1), C), dtype=torch.float32, device=raw.device)
    if has_inject and inject_stride is None:
        raise HCError(TS_ERR_INVALID_ARG, "inject_stride is required with a caller-given inject_w")
    if w_out is None:
        w_out = torch.empty((max(M, 1), C * H), dtype=torch.float32, device=raw.device)
    _need(w_out, "w_out", torch.float32)
    if ws is None:
        ws = workspace(M, H, C, L, raw.device)
    st = ts_hc_call_debug(raw.data_ptr(), weights.g.data_ptr(), weight_struct(weights.down),
                          weight_struct(weights.up), weight_struct(weights.inject) if has_inject else None,
                          mixed.data_ptr(), inject_w.data_ptr() if has_inject else None, inject_stride or 0, M, H,
                          C, L, eps, ws.data_ptr(), ws.numel() * ws.element_size(), w_out.data_ptr(),
                          _stream_handle(stream))
    _check(st)
    return mixed, (inject_w if has_inject else None), w_out[:M]


def hc_inject_add(raw, out, inject_w, *, H: int, C: int, inject_stride: Optional[int] = None, stream=None):
    """raw[m, c*H+h] += out[m, h] * inject_w[m*stride + c], in place; returns raw."""
    torch = _torch()
    M = raw.shape[0]
    _need(raw, "raw", torch.bfloat16, (M, C * H))
    _need(out, "out", torch.bfloat16, (M, H))
    if not inject_w.is_cuda or inject_w.dtype != torch.float32:
        raise HCError(TS_ERR_INVALID_ARG, "inject_w must be a CUDA float32 tensor")
    st = ts_hc_inject_add(raw.data_ptr(), out.data_ptr(), inject_w.data_ptr(),
                          C if inject_stride is None else inject_stride, M, H, C, _stream_handle(stream))
    _check(st)
    return raw


def hc_inject_call(raw, out, prev_inject_w, weights, *, H: int, C: int, prev_inject_stride: Optional[int] = None,
                   mixed=None, inject_w=None, inject_stride: Optional[int] = None, eps: float = RMS_EPS,
                   ws=None, stream=None):
    """The previous sublayer's inject-add fused into the next call: raw += out * prev gates
    (in place), then attn_hc / mlp_hc on it -- or the exit mixer when weights.inject is None.
    Returns (mixed, inject_w); inject_w is None for the mixer."""
    torch = _torch()
    M = raw.shape[0]
    L = weights.down.rows
    _need(raw, "raw", torch.bfloat16, (M, C * H))
    _need(out, "out", torch.bfloat16, (M, H))
    _need(weights.g, "hc_norm_w", torch.bfloat16, (C * H,))
    if not prev_inject_w.is_cuda or prev_inject_w.dtype != torch.float32:
        raise HCError(TS_ERR_INVALID_ARG, "prev_inject_w must be a CUDA float32 tensor")
    if mixed is None:
        mixed = torch.empty((M, H), dtype=torch.bfloat16, device=raw.device)
    _need(mixed, "mixed", torch.bfloat16, (M, H))
    has_inject = weights.inject is not None
    if has_inject and inject_w is None:
        inject_stride = C
        inject_w = torch.empty((max(M, 1), C), dtype=torch.float32, device=raw.device)
    if has_inject and inject_stride is None:
        raise HCError(TS_ERR_INVALID_ARG, "inject_stride is required with a caller-given inject_w")
    if ws is None:
        ws = workspace(M, H, C, L, raw.device)
    st = ts_hc_inject_call(raw.data_ptr(), out.data_ptr(), prev_inject_w.data_ptr(),
                           C if prev_inject_stride is None else prev_inject_stride, weights.g.data_ptr(),
                           weight_struct(weights.down), weight_struct(weights.up),
                           weight_struct(weights.inject) if has_inject else None, mixed.data_ptr(),
                           inject_w.data_ptr() if has_inject else None, inject_stride or 0, M, H, C, L, eps,
                           ws.data_ptr(), ws.numel() * ws.element_size(), _stream_handle(stream))
    _check(st)
    return mixed, (inject_w if has_inject else None)


def hc_entry_call(emb, weights, *, C: int, raw=None, mixed=None, inject_w=None, inject_stride: Optional[int] = None,
                  eps: float = RMS_EPS, ws=None, stream=None):
    """The entry replication fused into the first call: raw [M, C*H] = emb [M, H] repeated C
    times (written), then attn_hc on it -- or the mixer when weights.inject is None.
    Returns (raw, mixed, inject_w or None)."""
    torch = _torch()
    M, H = emb.shape
    L = weights.down.rows
    _need(emb, "emb", torch.bfloat16, (M, H))
    _need(weights.g, "hc_norm_w", torch.bfloat16, (C * H,))
    if raw is None:
        raw = torch.empty((M, C * H), dtype=torch.bfloat16, device=emb.device)
    _need(raw, "raw", torch.bfloat16, (M, C * H))
    if mixed is None:
        mixed = torch.empty((M, H), dtype=torch.bfloat16, device=emb.device)
    _need(mixed, "mixed", torch.bfloat16, (M, H))
    has_inject = weights.inject is not None
    if has_inject and inject_w is None:
        inject_stride = C
        inject_w = torch.empty((max(M, 1), C), dtype=torch.float32, device=emb.device)
    if has_inject and inject_stride is None:
        raise HCError(TS_ERR_INVALID_ARG, "inject_stride is required with a caller-given inject_w")
    if ws is None:
        ws = workspace(M, H, C, L, emb.device)
    st = ts_hc_entry_call(emb.data_ptr(), raw.data_ptr(), weights.g.data_ptr(), weight_struct(weights.down),
                          weight_struct(weights.up), weight_struct(weights.inject) if has_inject else None,
                          mixed.data_ptr(), inject_w.data_ptr() if has_inject else None, inject_stride or 0, M, H, C,
                          L, eps, ws.data_ptr(), ws.numel() * ws.element_size(), _stream_handle(stream))
    _check(st)
    return raw, mixed, (inject_w if has_inject else None)


def hc_exit_logits(raw, weights, lm_head, *, H: int, C: int, out=None, prev_inject_w=None,
                   prev_inject_stride: Optional[int] = None, mixed=None, logits=None, eps: float = RMS_EPS, ws=None,
                   stream=None):
    """The decoder's exit: with ``out`` given, raw += out * prev gates (in place) first; then the
    mixer (``weights``: g, down, up) and lm_head [V, H] bf16. Returns (mixed [M, H] bf16,
    logits [M, V] fp32)."""
    torch = _torch()
    M = raw.shape[0]
    L = weights.down.rows
    V = lm_head.shape[0]
    _need(raw, "raw", torch.bfloat16, (M, C * H))
    _need(weights.g, "hc_norm_w", torch.bfloat16, (C * H,))
    _need(lm_head, "lm_head", torch.bfloat16, (V, H))
    if mixed is None:
        mixed = torch.empty((M, H), dtype=torch.bfloat16, device=raw.device)
    _need(mixed, "mixed", torch.bfloat16, (M, H))
    if logits is None:
        logits = torch.empty((M, V), dtype=torch.float32, device=raw.device)
    _need(logits, "logits", torch.float32, (M, V))
    if out is not None:
        _need(out, "out", torch.bfloat16, (M, H))
        if prev_inject_w is None or not prev_inject_w.is_cuda or prev_inject_w.dtype != torch.float32:
            raise HCError(TS_ERR_INVALID_ARG, "prev_inject_w must be a CUDA float32 tensor with out")
    if ws is None:
        ws = workspace(M, H, C, L, raw.device)
    st = ts_hc_exit_logits(raw.data_ptr(), out.data_ptr() if out is not None else None,
                           prev_inject_w.data_ptr() if out is not None else None,
                           (C if prev_inject_stride is None else prev_inject_stride) if out is not None else 0,
                           weights.g.data_ptr(), weight_struct(weights.down), weight_struct(weights.up),
                           lm_head.data_ptr(), V, mixed.data_ptr(), logits.data_ptr(), M, H, C, L, eps, ws.data_ptr(),
                           ws.numel() * ws.element_size(), _stream_handle(stream))
    _check(st)
    return mixed, logits


def hc_ple(hidden, rows, weights, conv_state, *, C: int, eps: float = RMS_EPS, ws=None, stream=None):
    """The PLE gate on hidden [M, C*H] bf16 (in place) for M consecutive tokens of one
    sequence. ``rows`` int32 [M, 16] table row ids; ``weights`` has table, key_proj,
    value_proj, norm_key, norm_query, norm_conv, conv_w; ``conv_state`` fp32 [9, C*H]
    (updated). Returns (hidden, the workspace)."""
    torch = _torch()
    M = hidden.shape[0]
    H = weights.value_proj.shape[0]
    W = C * H
    _need(hidden, "hidden", torch.bfloat16, (M, W))
    _need(rows, "rows", torch.int32, (M, 16))
    _need(weights.table, "table", torch.bfloat16)
    _need(weights.key_proj, "key_proj", torch.bfloat16, (W, H))
    _need(weights.value_proj, "value_proj", torch.bfloat16, (H, H))
    for name in ("norm_key", "norm_query", "norm_conv"):
        _need(getattr(weights, name), name, torch.bfloat16, (W,))
    _need(weights.conv_w, "conv_w", torch.bfloat16, (W, 4))
    _need(conv_state, "conv_state", torch.float32, (9, W))
    if ws is None:
        ws = torch.empty(max(ts_hc_ple_workspace_bytes(M, H, C), 256), dtype=torch.uint8, device=hidden.device)
    st = ts_hc_ple(hidden.data_ptr(), rows.data_ptr(), weights.table.data_ptr(), weights.table.shape[0],
                   weights.key_proj.data_ptr(), weights.value_proj.data_ptr(), weights.norm_key.data_ptr(),
                   weights.norm_query.data_ptr(), weights.norm_conv.data_ptr(), weights.conv_w.data_ptr(),
                   conv_state.data_ptr(), M, H, C, eps, ws.data_ptr(), ws.numel() * ws.element_size(),
                   _stream_handle(stream))
    _check(st)
    return hidden, ws


def hc_replicate_entry(emb, *, C: int, raw=None, stream=None):
    """raw [M, C*H] bf16 with every stream equal to emb [M, H] (repeat, not pad)."""
    torch = _torch()
    M, H = emb.shape
    _need(emb, "emb", torch.bfloat16, (M, H))
    if raw is None:
        raw = torch.empty((M, C * H), dtype=torch.bfloat16, device=emb.device)
    _need(raw, "raw", torch.bfloat16, (M, C * H))
    _check(ts_hc_replicate_entry(emb.data_ptr(), raw.data_ptr(), M, H, C, _stream_handle(stream)))
    return raw


def device_status(stream=None) -> int:
    st, v = ts_hc_device_status(_stream_handle(stream))
    _check(st)
    return v


def module_struct(w) -> TsHcModule:
    """A ``TsHcModule`` for weights with attributes g, down, up, inject (inject may be None)."""
    m = TsHcModule()
    m.hc_norm_w = w.g.data_ptr()
    m.down, m.up = weight_struct(w.down), weight_struct(w.up)
    if w.inject is not None:
        m.inject = weight_struct(w.inject)
    return m


def stack_workspace(max_chunk: int, H: int, C: int, L: int, device=None, with_ple: bool = False):
    torch = _torch()
    n = (ts_hc_stack_ple_workspace_bytes if with_ple else ts_hc_stack_workspace_bytes)(max_chunk, H, C, L)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def ple_module_struct(w) -> TsHcPleModule:
    """A ``TsHcPleModule`` for PLE weights with attributes table, key_proj, value_proj,
    norm_key, norm_query, norm_conv, conv_w."""
    m = TsHcPleModule()
    m.table = w.table.data_ptr()
    m.n_rows = w.table.shape[0]
    m.key_proj, m.value_proj = w.key_proj.data_ptr(), w.value_proj.data_ptr()
    m.norm_key_w, m.norm_query_w = w.norm_key.data_ptr(), w.norm_query.data_ptr()
    m.norm_conv_w, m.conv_w = w.norm_conv.data_ptr(), w.conv_w.data_ptr()
    return m


def hc_stack(emb, layers, final, sublayer, *, C: int, max_chunk: Optional[int] = None, mixed_out=None,
             eps: float = RMS_EPS, ws=None, stream=None, ple=None, ple_rows=None, ple_state=None):
    """The decoder stack's hyper-connection path on T tokens through ``ts_hc_stack``
    (``ts_hc_stack_ple`` when ``ple`` is given).

    ``emb`` [T, H] bf16; ``layers``: a sequence of (attn, mlp) weights (g, down, up,
    inject); ``final``: the exit mixer's weights. ``sublayer(layer, which, t0, mixed)``
    gets the call's output ``mixed`` ([M, H] bf16, a view into the workspace) and
    returns the sublayer output, a CUDA bf16 tensor [M, H] that it may compute on the
    current stream; the driver injects it with the call's gates. ``ple``: PLE weights
    (table, key_proj, value_proj, norm_key, norm_query, norm_conv, conv_w) applied
    before layer 1's attn_hc, with ``ple_rows`` int32 [T, 16] and ``ple_state`` fp32
    [9, C*H] (updated). Returns (mixed_out [T, H], the last chunk's residual
    [M, C*H] -- a view into ``ws``).
    """
    torch = _torch()
    T, H = emb.shape
    L = final.down.rows
    _need(emb, "emb", torch.bfloat16, (T, H))
    max_chunk = max(T, 1) if max_chunk is None else max_chunk
    if mixed_out is None:
        mixed_out = torch.empty((T, H), dtype=torch.bfloat16, device=emb.device)
    _need(mixed_out, "mixed_out", torch.bfloat16, (T, H))
    if ple is not None:
        _need(ple_rows, "ple_rows", torch.int32, (T, 16))
        _need(ple_state, "ple_state", torch.float32, (9, C * H))
    if ws is None:
        ws = stack_workspace(max_chunk, H, C, L, emb.device, with_ple=ple is not None)
    n = len(layers)
    attn = (TsHcModule * max(n, 1))(*[module_struct(a) for a, _ in layers])
    mlp = (TsHcModule * max(n, 1))(*[module_struct(m) for _, m in layers])
    fin = module_struct(final)
    keep, errors = [], []
    base = ws.data_ptr()

    def trampoline(user, layer, which, t0, M, mixed_ptr, out_pp, stream_h):
        try:
            off = mixed_ptr - base
            mixed = ws[off:off + 2 * M * H].view(torch.bfloat16).view(M, H)
            out = sublayer(layer, which, t0, mixed)
            _need(out, "sublayer output", torch.bfloat16, (M, H))
            if stream is not None:  # the caching allocator must not hand it out before the driver's stream used it
                out.record_stream(stream)
            keep.append(out)
            out_pp[0] = out.data_ptr()
            return TS_OK
        except Exception as e:  # reported after the C call returns
            errors.append(e)
            return TS_ERR_INVALID_ARG

    fn = SUBLAYER_FN(trampoline)
    if ple is None:
        st = ts_hc_stack(emb.data_ptr(), T, attn, mlp, n, fin, fn, None, mixed_out.data_ptr(), max_chunk, H, C,
                         L, eps, base, ws.numel() * ws.element_size(), _stream_handle(stream))
    else:
        st = ts_hc_stack_ple(emb.data_ptr(), T, attn, mlp, n, fin, ple_module_struct(ple), ple_rows.data_ptr(),
                             ple_state.data_ptr(), fn, None, mixed_out.data_ptr(), max_chunk, H, C, L, eps, base,
                             ws.numel() * ws.element_size(), _stream_handle(stream))
    if errors:
        raise errors[0]
    _check(st)
    M_last = T - (max(T, 1) - 1) // max_chunk * max_chunk if T else 0
    raw_last = ws[:2 * M_last * C * H].view(torch.bfloat16).view(M_last, C * H)
    return mixed_out, raw_last
