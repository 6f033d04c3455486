"""Python binding of liboases.so, the GB300 library for the Oases TP block.

Argument marshalling only: every step of the block runs in the library's CUDA
kernels.  Functions carry the C names (``oases_block_fwd`` ...) and take torch
tensors (device or host), raw integer pointers, or None.  Streams are
``torch.cuda.Stream`` objects, raw ``cudaStream_t`` integers or None (the
legacy default stream).  A non-OK status raises ``OasesError``.

The library must be built (``build_library()``); importing this module does not
build it, and every call fails loudly if the shared object is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

from .build import LIB, build as build_library

_lib = None

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA", 5: "TIMEOUT",
          6: "INJECTED"}
KIND = {"ffn": 0, "attn": 1, "layer": 2}
DTYPE = {"f32": 0, "bf16": 1, "mxfp8": 2}
RECOMPUTE = {"none": 0, "full": 1, "fine": 2, "selective": 3}
REDUCE = {"fused": 0, "separate": 1}
EVENTS = ["F", "R", "B", "C(F)", "C(R)", "C(B)", "Sync"]
OPS = ["ln", "f", "col", "row", "g", "attn"]
PARAM_NAMES = ("ln1_g", "ln1_b", "wqkv", "bqkv", "wo", "bo",
               "ln2_g", "ln2_b", "w1", "b1", "w2", "b2")


class OasesError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(what)


class BlockDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kind", "dtype", "batch", "seq", "hidden", "ffn", "heads", "w", "sub_batches",
                 "pre_ln", "residual", "causal", "recompute", "reduce")] + [("ln_eps", ctypes.c_float)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_NAMES]


class Grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_NAMES]


def lib():
    """The loaded shared library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError("liboases.so is not built (run tensor_model_transformer_tp_gb300"
                               ".build.build()); there is no fallback path")
        L = ctypes.CDLL(LIB)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        dp, wp, gp = ctypes.POINTER(BlockDesc), ctypes.POINTER(Weights), ctypes.POINTER(Grads)
        L.oases_workspace_bytes.argtypes = [dp, i32]
        L.oases_workspace_bytes.restype = sz
        L.oases_block_fwd.argtypes = [dp, wp, vp, vp, vp, sz, vp, vp]
        L.oases_block_fwd.restype = i32
        L.oases_block_recompute_bwd.argtypes = [dp, wp, vp, vp, vp, gp, vp, sz, vp, vp]
        L.oases_block_recompute_bwd.restype = i32
        L.oases_stack_step.argtypes = [dp, i32, wp, vp, vp, vp, vp, gp, vp, sz, vp, vp]
        L.oases_stack_step.restype = i32
        L.oases_status_str.argtypes = [i32]
        L.oases_status_str.restype = ctypes.c_char_p
        L.oases_last_error.restype = ctypes.c_char_p
        L.oases_version.restype = ctypes.c_char_p
        L.oases_schedule_trace.argtypes = [dp, i32, i32, ctypes.POINTER(ctypes.c_int32), i32]
        L.oases_schedule_trace.restype = i32
        L.oases_last_launch_count.restype = i32
        L.oases_check_device.argtypes = [vp]
        L.oases_check_device.restype = i32
        L.oases_shutdown.argtypes = []
        L.oases_shutdown.restype = i32
        _lib = L
    return _lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr() if t.numel() > 0 else None
    if hasattr(t, "ctypes"):  # numpy
        return t.ctypes.data if t.size > 0 else None
    raise TypeError("expected a tensor, an array, an int pointer or None, got %r" % type(t))


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int) -> None:
    if st != 0:
        L = lib()
        raise OasesError(st, "%s: %s %s" % (STATUS.get(st, st), L.oases_status_str(st).decode(),
                                            L.oases_last_error().decode()))


def make_desc(kind: str, dtype: str, batch: int, seq: int, hidden: int, ffn: int = 0,
              heads: int = 0, w: int = 1, sub_batches: int = 2, pre_ln: bool = True,
              residual: bool = True, causal: bool = True, recompute: str = "fine",
              eps: float = 1e-5, reduce: str = "fused") -> BlockDesc:
    return BlockDesc(KIND[kind], DTYPE[dtype], batch, seq, hidden, ffn, heads, w, sub_batches,
                     int(pre_ln), int(residual), int(causal), RECOMPUTE[recompute], REDUCE[reduce],
                     eps)


def desc_from_shape(shape, recompute: str = "fine", sub_batches: Optional[int] = None,
                    reduce: str = "fused") -> BlockDesc:
    """BlockDesc from any object with the BlockShape attributes."""
    return make_desc(shape.kind, shape.dtype, shape.batch, shape.seq, shape.hidden, shape.ffn,
                     shape.heads, shape.w,
                     shape.sub_batches if sub_batches is None else sub_batches,
                     shape.pre_ln, shape.residual, shape.causal, recompute, shape.eps, reduce)


def weights_struct(params: Dict) -> Weights:
    return Weights(*[_ptr(params.get(n)) for n in PARAM_NAMES])


def grads_struct(grads: Dict) -> Grads:
    return Grads(*[_ptr(grads.get(n)) for n in PARAM_NAMES])


def oases_workspace_bytes(desc: BlockDesc, n_layers: int = 1) -> int:
    return int(lib().oases_workspace_bytes(ctypes.byref(desc), n_layers))


def oases_block_fwd(desc, weights, x, y, workspace, ws_bytes=None, s0=None, s1=None) -> None:
    w = weights if isinstance(weights, Weights) else weights_struct(weights)
    nb = ws_bytes if ws_bytes is not None else _nbytes(workspace)
    _check(lib().oases_block_fwd(ctypes.byref(desc), ctypes.byref(w), _ptr(x), _ptr(y),
                                 _ptr(workspace), nb, _stream(s0), _stream(s1)))


def oases_block_recompute_bwd(desc, weights, x_saved, dy, dx, grads, workspace, ws_bytes=None,
                              s0=None, s1=None) -> None:
    w = weights if isinstance(weights, Weights) else weights_struct(weights)
    g = grads if isinstance(grads, Grads) else grads_struct(grads)
    nb = ws_bytes if ws_bytes is not None else _nbytes(workspace)
    _check(lib().oases_block_recompute_bwd(ctypes.byref(desc), ctypes.byref(w), _ptr(x_saved),
                                           _ptr(dy), _ptr(dx), ctypes.byref(g), _ptr(workspace),
                                           nb, _stream(s0), _stream(s1)))


def oases_stack_step(desc, per_layer: Sequence, x, g, y, dx, per_layer_grads: Sequence,
                     workspace, ws_bytes=None, s0=None, s1=None) -> None:
    n = len(per_layer)
    W = (Weights * n)(*[p if isinstance(p, Weights) else weights_struct(p) for p in per_layer])
    G = (Grads * n)(*[p if isinstance(p, Grads) else grads_struct(p) for p in per_layer_grads])
    nb = ws_bytes if ws_bytes is not None else _nbytes(workspace)
    _check(lib().oases_stack_step(ctypes.byref(desc), n, W, _ptr(x), _ptr(g), _ptr(y), _ptr(dx),
                                  G, _ptr(workspace), nb, _stream(s0), _stream(s1)))


def oases_schedule_trace(desc, n_layers: int, phase: int) -> List[tuple]:
    L = lib()
    n = L.oases_schedule_trace(ctypes.byref(desc), n_layers, phase, None, 0)
    if n < 0:
        raise OasesError(1, "invalid descriptor")
    buf = (ctypes.c_int32 * max(n, 1))()
    L.oases_schedule_trace(ctypes.byref(desc), n_layers, phase, buf, n)
    return [(EVENTS[e & 0xF], OPS[(e >> 4) & 0xF], e >> 16, (e >> 8) & 0xFF) for e in buf[:n]]


def oases_last_launch_count() -> int:
    return int(lib().oases_last_launch_count())


def oases_check_device(stream=None) -> None:
    _check(lib().oases_check_device(_stream(stream)))


def oases_shutdown() -> None:
    """Release the library's cached host-side state (copy streams, this
    thread's events, tensor-map cache); later calls make it again."""
    _check(lib().oases_shutdown())


def oases_status_str(st: int) -> str:
    return lib().oases_status_str(st).decode()


def oases_version() -> str:
    return lib().oases_version().decode()


def _nbytes(t) -> int:
    if t is None:
        return 0
    if hasattr(t, "numel"):
        return t.numel() * t.element_size()
    if hasattr(t, "nbytes"):
        return int(t.nbytes)
    raise TypeError("pass ws_bytes with a raw workspace pointer")


__all__ = ["BlockDesc", "Weights", "Grads", "OasesError", "build_library", "lib", "make_desc",
           "desc_from_shape", "weights_struct", "grads_struct", "oases_workspace_bytes",
           "oases_block_fwd", "oases_block_recompute_bwd", "oases_stack_step",
           "oases_schedule_trace", "oases_last_launch_count", "oases_check_device", "oases_shutdown",
           "oases_status_str", "oases_version", "PARAM_NAMES"]
