"""Python binding of the slmoe C ABI (``include/slmoe.h``): argument marshalling only.

Every step of the layer runs in the CUDA kernels of ``libslmoe.so``; this module turns
torch tensors into device pointers and ctypes structs, calls the C entry points with the
same names, and raises ``SlmoeError`` on a non-zero return code.  There is no fallback:
if the library is missing the import of an entry point fails loudly.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = ["SlmoeError", "Config", "Weights", "WorkspaceLayout", "load", "build", "config",
           "weights", "slmoe_workspace_size", "slmoe_workspace_layout_get", "slmoe_route",
           "slmoe_route_noalloc", "slmoe_topk", "slmoe_mxfp4_quantize", "slmoe_mxfp8_quantize", "slmoe_topk_workspace_size", "slmoe_wait_abort_check",
           "slmoe_qb_histogram", "slmoe_qb_update", "slmoe_signsgd_update",
           "slmoe_forward", "slmoe_backward", "slmoe_backward_workspace_size", "slmoe_backward_layout_get",
           "backward_views", "Grads", "grads",
           "slmoe_device_sm_count", "workspace_views", "slmoe_last_error",
           "slmoe_set_stage_events", "slmoe_launch_count", "F32", "BF16", "MXFP4", "LIB_PATH"]

F32, BF16, MXFP4 = 0, 1, 2
LIB_PATH = _build.LIB


class SlmoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"slmoe error {code}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("d_latent", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("I", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("I_shared", ctypes.c_int32), ("nbins", ctypes.c_int32),
                ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("dtype", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("W_r", "W_in", "W13", "W2", "gamma", "W_out", "W13_s", "W2_s", "W13_scale", "W2_scale")]


class Grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("dW_r", "dW_in", "dW13", "dW2", "dgamma", "dW_out", "dW13_s", "dW2_s")]


class BackwardLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("dz", "dye", "dg", "gu", "dgu", "dx_lat", "gu_s", "dgu_s", "total")]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("scores", "topk_idx", "topk_w", "counts", "offsets", "perm", "slot_pos", "x_lat",
                 "h", "y_e", "z", "h_s", "status", "total")]


_lib = None


def build(force=False):
    return _build.build(force=force)


def load():
    """The loaded ``libslmoe.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with latent_space_experts_gb300.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    CP, WP = ctypes.POINTER(Config), ctypes.POINTER(Weights)
    sig = {
        "slmoe_workspace_size": (SZ, [CP]),
        "slmoe_workspace_layout_get": (ctypes.c_int, [CP, ctypes.POINTER(WorkspaceLayout)]),
        "slmoe_last_error": (ctypes.c_char_p, []),
        "slmoe_device_sm_count": (ctypes.c_int, []),
        "slmoe_route": (ctypes.c_int, [CP, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "slmoe_route_noalloc": (ctypes.c_int, [CP, P, P, P, P, P, P, P, P, P, P, P, P, P, P]),
        "slmoe_topk_workspace_size": (SZ, [I32, I32, I32]),
        "slmoe_topk": (ctypes.c_int, [P, P, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P]),
        "slmoe_wait_abort_check": (ctypes.c_int, [P, ctypes.c_uint64, P]),
        "slmoe_mxfp4_quantize": (ctypes.c_int, [P, I64, I32, P, P, P]),
        "slmoe_mxfp8_quantize": (ctypes.c_int, [P, I64, I32, P, P, P]),
        "slmoe_qb_histogram": (ctypes.c_int, [P, I64, I32, I32, P, P, P]),
        "slmoe_qb_update": (ctypes.c_int, [P, I32, I32, I32, P, P, P]),
        "slmoe_signsgd_update": (ctypes.c_int, [P, I32, ctypes.c_float, P, P]),
        "slmoe_forward": (ctypes.c_int, [CP, P, WP, P, P, P, P, P, P, P, SZ, P]),
        "slmoe_backward_workspace_size": (SZ, [CP]),
        "slmoe_backward_layout_get": (ctypes.c_int, [CP, ctypes.POINTER(BackwardLayout)]),
        "slmoe_backward": (ctypes.c_int, [CP, P, WP, P, P, ctypes.POINTER(Grads), ctypes.c_int, P, SZ, P, P,
                                          SZ, P]),
        "slmoe_set_stage_events": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
        "slmoe_launch_count": (ctypes.c_longlong, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("slmoe entry points take CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("slmoe entry points take contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc):
    if rc != 0:
        raise SlmoeError(rc, load().slmoe_last_error().decode())


def config(shape, T=None, dtype=None) -> Config:
    """A Config from a ``synthetic.LayerShape``-like object (T and the layer type overridable)."""
    if dtype is None:
        dtype = BF16 if shape.dtype == "bf16" else F32
    return Config(T=shape.T if T is None else T, d=shape.d, d_latent=shape.d_latent, E=shape.E,
                  k=shape.k, I=shape.I, n_shared=shape.n_shared, I_shared=shape.I_shared,
                  nbins=shape.nbins, beta1=shape.beta1, beta2=shape.beta2, eps=shape.eps,
                  dtype=dtype)


def weights(inp: dict) -> Weights:
    """A Weights struct from a dict of CUDA tensors; for the MXFP4 layer type the dict holds the
    packed codes as W13 / W2 and their scales as W13_scale / W2_scale."""
    return Weights(*[_ptr(inp.get(n)) for n in ("W_r", "W_in", "W13", "W2", "gamma", "W_out",
                                                 "W13_s", "W2_s", "W13_scale", "W2_scale")])


def grads(g: dict) -> Grads:
    """A Grads struct from a dict of fp32 CUDA tensors named as its fields."""
    return Grads(*[_ptr(g[n]) for n in ("dW_r", "dW_in", "dW13", "dW2", "dgamma", "dW_out", "dW13_s", "dW2_s")])


def slmoe_last_error() -> str:
    return load().slmoe_last_error().decode()


_event_array = None


def slmoe_set_stage_events(events):
    """Hand the library torch.cuda.Event objects (recorded once, so that they exist) to be
    recorded after each stage of slmoe_forward on this thread; None turns it off."""
    global _event_array
    if not events:
        _event_array = None
        return load().slmoe_set_stage_events(None, 0)
    _event_array = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return load().slmoe_set_stage_events(_event_array, len(events))


def slmoe_launch_count() -> int:
    return load().slmoe_launch_count()


def slmoe_device_sm_count() -> int:
    return load().slmoe_device_sm_count()


def slmoe_workspace_size(cfg: Config) -> int:
    n = load().slmoe_workspace_size(ctypes.byref(cfg))
    if n == 0:
        raise SlmoeError(-1, load().slmoe_last_error().decode())
    return n


def slmoe_workspace_layout_get(cfg: Config) -> dict:
    out = WorkspaceLayout()
    _check(load().slmoe_workspace_layout_get(ctypes.byref(cfg), ctypes.byref(out)))
    return {n: getattr(out, n) for n, _ in WorkspaceLayout._fields_}


def workspace_views(cfg: Config, ws):
    """torch views of the intermediates inside a workspace tensor (uint8, on the device)."""
    import torch
    L = slmoe_workspace_layout_get(cfg)
    act = torch.float32 if cfg.dtype == F32 else torch.bfloat16
    T, k, E = cfg.T, cfg.k, cfg.E

    def view(name, dtype, shape, at=0):
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[L[name] + at:L[name] + at + nbytes].view(dtype).view(*shape)

    if cfg.dtype == MXFP4:   # x_lat and h as MXFP8: codes, then their block scales
        dl, I = cfg.d_latent, cfg.I
        lat = dict(x_lat=view("x_lat", torch.uint8, (T, dl)),
                   x_lat_scales=view("x_lat", torch.uint8, (T, dl // 32), at=T * dl),
                   h=view("h", torch.uint8, (T * k, I)),
                   h_scales=view("h", torch.uint8, (T * k, I // 32), at=T * k * I))
    else:
        lat = dict(x_lat=view("x_lat", act, (T, cfg.d_latent)), h=view("h", act, (T * k, cfg.I)))

    return dict(scores=view("scores", torch.float32, (T, E)),
                topk_idx=view("topk_idx", torch.int32, (T, k)),
                topk_w=view("topk_w", torch.float32, (T, k)),
                counts=view("counts", torch.int32, (E,)),
                offsets=view("offsets", torch.int32, (E + 1,)),
                perm=view("perm", torch.int32, (T * k,)),
                slot_pos=view("slot_pos", torch.int32, (T, k)),
                **lat,
                y_e=view("y_e", act, (T * k, cfg.d_latent)),
                z=view("z", act, (T, cfg.d_latent)),
                h_s=view("h_s", act, (T, cfg.n_shared * cfg.I_shared)),
                status=view("status", torch.int32, (4,)))


def slmoe_route(cfg, x, W_r, bias, logit_offset, topk_idx, topk_w, scores, counts, offsets, perm,
                slot_pos, hist, status, workspace, stream=None):
    _check(load().slmoe_route(ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(bias), _ptr(logit_offset),
                              _ptr(topk_idx), _ptr(topk_w), _ptr(scores), _ptr(counts), _ptr(offsets),
                              _ptr(perm), _ptr(slot_pos), _ptr(hist), _ptr(status), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)))


def slmoe_route_noalloc(cfg, x, W_r, bias, logit_offset, topk_idx, topk_w, scores, counts, offsets,
                        perm, slot_pos, hist, status, stream=None):
    """slmoe_route with the library's fixed per-device scratch instead of a workspace: for
    callers that cannot hand out device memory per call.  Calls that may overlap on one
    device race on that scratch; the first call on a device sets it up."""
    _check(load().slmoe_route_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(bias),
                                      _ptr(logit_offset), _ptr(topk_idx), _ptr(topk_w), _ptr(scores),
                                      _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(slot_pos),
                                      _ptr(hist), _ptr(status), _stream(stream)))


def slmoe_topk_workspace_size(T, E, k) -> int:
    n = load().slmoe_topk_workspace_size(T, E, k)
    if n == 0:
        raise SlmoeError(-1, load().slmoe_last_error().decode())
    return n


def slmoe_topk(scores, bias, T, E, k, topk_idx, topk_w, counts, offsets, perm, slot_pos, status,
               workspace, stream=None):
    _check(load().slmoe_topk(_ptr(scores), _ptr(bias), T, E, k, _ptr(topk_idx), _ptr(topk_w),
                             _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(slot_pos), _ptr(status),
                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream(stream)))


def slmoe_mxfp4_quantize(W, rows, K, packed, scales, stream=None):
    _check(load().slmoe_mxfp4_quantize(_ptr(W), rows, K, _ptr(packed), _ptr(scales), _stream(stream)))


def slmoe_mxfp8_quantize(X, rows, K, codes, scales, stream=None):
    _check(load().slmoe_mxfp8_quantize(_ptr(X), rows, K, _ptr(codes), _ptr(scales), _stream(stream)))


def slmoe_wait_abort_check(status, wait_limit_ns, stream=None):
    _check(load().slmoe_wait_abort_check(_ptr(status), int(wait_limit_ns), _stream(stream)))


def slmoe_qb_histogram(scores, T, E, nbins, hist, status=None, stream=None):
    _check(load().slmoe_qb_histogram(_ptr(scores), T, E, nbins, _ptr(hist), _ptr(status),
                                     _stream(stream)))


def slmoe_qb_update(hist, E, nbins, k, q_out, bias, stream=None):
    _check(load().slmoe_qb_update(_ptr(hist), E, nbins, k, _ptr(q_out), _ptr(bias), _stream(stream)))


def slmoe_signsgd_update(counts, E, step, bias, stream=None):
    _check(load().slmoe_signsgd_update(_ptr(counts), E, float(step), _ptr(bias), _stream(stream)))


def slmoe_forward(cfg, x, w: Weights, bias, logit_offset, y, topk_idx_out, hist, status, workspace,
                  stream=None):
    _check(load().slmoe_forward(ctypes.byref(cfg), _ptr(x), ctypes.byref(w), _ptr(bias),
                                _ptr(logit_offset), _ptr(y), _ptr(topk_idx_out), _ptr(hist),
                                _ptr(status), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)))


def slmoe_backward_workspace_size(cfg: Config) -> int:
    n = load().slmoe_backward_workspace_size(ctypes.byref(cfg))
    if n == 0:
        raise SlmoeError(-1, load().slmoe_last_error().decode())
    return n


def slmoe_backward(cfg, x, w: Weights, dy, dx, g: Grads, accumulate, fwd_workspace, status, workspace,
                   stream=None):
    _check(load().slmoe_backward(ctypes.byref(cfg), _ptr(x), ctypes.byref(w), _ptr(dy), _ptr(dx),
                                 ctypes.byref(g), int(accumulate), _ptr(fwd_workspace),
                                 fwd_workspace.numel() * fwd_workspace.element_size(), _ptr(status),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)))


def slmoe_backward_layout_get(cfg: Config) -> dict:
    out = BackwardLayout()
    _check(load().slmoe_backward_layout_get(ctypes.byref(cfg), ctypes.byref(out)))
    return {n: getattr(out, n) for n, _ in BackwardLayout._fields_}


def backward_views(cfg: Config, ws):
    """torch views of the backward's intermediates inside its workspace (uint8, on the device)."""
    import torch
    L = slmoe_backward_layout_get(cfg)
    T, k, dl, I, Is = cfg.T, cfg.k, cfg.d_latent, cfg.I, cfg.I_shared

    def view(name, dtype, shape):
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[L[name]:L[name] + nbytes].view(dtype).view(*shape)

    bf = torch.bfloat16
    return dict(dz=view("dz", torch.float32, (T, dl)), dye=view("dye", bf, (T * k, dl)),
                dg=view("dg", torch.float32, (T, k)), gu=view("gu", torch.float32, (T * k, 2 * I)),
                dgu=view("dgu", bf, (T * k, 2 * I)), dx_lat=view("dx_lat", bf, (T, dl)),
                gu_s=view("gu_s", torch.float32, (T, 2 * Is)), dgu_s=view("dgu_s", bf, (T, 2 * Is)))
