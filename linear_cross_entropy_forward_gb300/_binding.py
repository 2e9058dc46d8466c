"""ctypes binding of libflce.so (include/flce.h).

Argument marshalling only: tensors become raw device pointers plus sizes and
the current CUDA stream; every step of the computation runs in the library's
kernels.  If the library has not been built, or the device is not a GB300
(sm_103), the calls raise -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .workloads import IGNORE_INDEX, RED_NONE, reduction_code

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libflce.so")

FLCE_OK = 0
_ERR_NAMES = {1: "BAD_ARG", 2: "BAD_SHAPE", 3: "ALIGN", 4: "WS_TOO_SMALL", 5: "LABEL",
              6: "TIMEOUT", 7: "CUDA", 8: "DEVICE", 9: "SCRATCH_LIMIT", 10: "BOUNDS"}


class FlceError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"flce error {code} ({_ERR_NAMES.get(code, '?')}): {msg}")
        self.code = code


class FlceParams(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("H", ctypes.c_int64), ("V", ctypes.c_int64),
                ("ignore_index", ctypes.c_int64), ("reduction", ctypes.c_int32),
                ("zloss_coef", ctypes.c_float), ("softcap", ctypes.c_float),
                ("validate", ctypes.c_int32), ("chunk_v", ctypes.c_int64),
                ("weight_layout", ctypes.c_int32), ("label_smoothing", ctypes.c_float),
                ("class_weight", ctypes.c_void_p), ("v_offset", ctypes.c_int64),
                ("v_total", ctypes.c_int64), ("chunk_n", ctypes.c_int64),
                ("dhidden_fp32", ctypes.c_int32)]


WEIGHT_HV, WEIGHT_VH = 0, 1


def layout_code(layout) -> int:
    """'hv' (weight [H,V], the default) or 'vh' (weight [V,H], nn.Linear) -> ABI code."""
    if layout in (WEIGHT_HV, "hv"):
        return WEIGHT_HV
    if layout in (WEIGHT_VH, "vh"):
        return WEIGHT_VH
    raise ValueError(f"weight_layout must be 'hv' or 'vh', got {layout!r}")


_lib = None
_lock = threading.Lock()

EXPORTED = ("flce_workspace_size", "flce_forward", "flce_backward", "flce_status",
            "flce_kernel_launches", "flce_strerror", "flce_version", "flce_forward_noalloc",
            "flce_shard_stats", "flce_combine_shards", "flce_forward_backward",
            "flce_scale_bf16", "flce_selftest_wait_timeout", "flce_plan_tiles",
            "flce_check_params")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libflce.so (once) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = _open(path)
        return _lib


def use_library(path: str) -> ctypes.CDLL:
    """Route every later call of this module through the library at `path` (the same
    C ABI, e.g. libflce_debug.so, the build with in-kernel bounds checks); returns the
    library used until now (None if none was loaded), to hand back later."""
    global _lib
    with _lock:
        prev = _lib
        _lib = _open(path)
        return prev


def restore_library(lib) -> None:
    """Undo use_library: route calls through `lib` again (None: load on next use)."""
    global _lib
    with _lock:
        _lib = lib


def _open(path: str) -> ctypes.CDLL:
    """dlopen one build of the library and declare its signatures."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m linear_cross_entropy_forward_gb300.build`")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(FlceParams)
    vp = ctypes.c_void_p
    lib.flce_check_params.argtypes = [P]
    lib.flce_check_params.restype = ctypes.c_int
    lib.flce_workspace_size.argtypes = [P, ctypes.c_int]
    lib.flce_workspace_size.restype = ctypes.c_size_t
    lib.flce_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.flce_forward.restype = ctypes.c_int
    lib.flce_backward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                  vp]
    lib.flce_backward.restype = ctypes.c_int
    lib.flce_status.argtypes = [vp, vp]
    lib.flce_status.restype = ctypes.c_int
    lib.flce_strerror.argtypes = [ctypes.c_int]
    lib.flce_strerror.restype = ctypes.c_char_p
    lib.flce_shard_stats.argtypes = [P, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.flce_shard_stats.restype = ctypes.c_int
    lib.flce_combine_shards.argtypes = [P, vp, ctypes.c_int32, vp, vp, vp, vp, vp, vp,
                                        ctypes.c_size_t, vp]
    lib.flce_combine_shards.restype = ctypes.c_int
    lib.flce_kernel_launches.argtypes = [P, ctypes.c_int]
    lib.flce_kernel_launches.restype = ctypes.c_int
    lib.flce_forward_backward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                          ctypes.c_size_t, vp]
    lib.flce_forward_backward.restype = ctypes.c_int
    lib.flce_scale_bf16.argtypes = [vp, ctypes.c_int64, vp, vp]
    lib.flce_scale_bf16.restype = ctypes.c_int
    lib.flce_selftest_wait_timeout.argtypes = [vp, ctypes.c_size_t, ctypes.c_uint64, vp]
    lib.flce_selftest_wait_timeout.restype = ctypes.c_int
    i32 = ctypes.c_int32
    lib.flce_plan_tiles.argtypes = [i32, i32, i32, ctypes.c_int64, i32, i32, i32,
                                    ctypes.POINTER(i32)]
    lib.flce_plan_tiles.restype = ctypes.c_int
    lib.flce_version.argtypes = []
    lib.flce_version.restype = ctypes.c_int
    return lib


def _check(code: int):
    if code != FLCE_OK:
        raise FlceError(code, load_library().flce_strerror(code).decode())


def make_params(N, H, V, reduction="mean", ignore_index=IGNORE_INDEX, zloss_coef=0.0,
                softcap=0.0, validate=False, chunk_v=0, weight_layout="hv",
                label_smoothing=0.0, class_weight=None, v_offset=0, v_total=0,
                chunk_n=0, dhidden_fp32=False) -> FlceParams:
    """class_weight: a CUDA fp32 [V] tensor (kept alive by the caller) or None.
    v_offset / v_total: this weight is columns [v_offset, v_offset + V) of a vocabulary
    of v_total entries (0: the whole vocabulary).  chunk_n: token chunk of
    flce_forward_backward (multiple of 512, 0 = auto).  dhidden_fp32: the backward
    writes dhidden as fp32 (unrounded) instead of bf16."""
    cw = class_weight.data_ptr() if class_weight is not None else None
    return FlceParams(int(N), int(H), int(V), int(ignore_index), reduction_code(reduction),
                      float(zloss_coef), float(softcap), 1 if validate else 0, int(chunk_v),
                      layout_code(weight_layout), float(label_smoothing), cw, int(v_offset),
                      int(v_total), int(chunk_n), 1 if dhidden_fp32 else 0)


def _dims(hidden, weight, weight_layout):
    N, H = hidden.shape
    V = weight.shape[1] if layout_code(weight_layout) == WEIGHT_HV else weight.shape[0]
    wshape = (H, V) if layout_code(weight_layout) == WEIGHT_HV else (V, H)
    return N, H, V, wshape


def workspace_size(params: FlceParams, phase: int) -> int:
    lib = load_library()
    _check(lib.flce_check_params(ctypes.byref(params)))
    n = lib.flce_workspace_size(ctypes.byref(params), phase)
    if n == 0:
        raise FlceError(1, f"no workspace phase {phase}")
    return int(n)


def plan_tiles(m_tiles, n_tiles, raster, panel_bytes, a_hint=0, b_hint=0, pairs=76):
    """The GEMM schedule the library plans (host arithmetic, no GPU needed):
    (group, a_hint, b_hint); see flce_plan_tiles in flce.h."""
    out = (ctypes.c_int32 * 3)()
    _check(load_library().flce_plan_tiles(m_tiles, n_tiles, raster, panel_bytes, a_hint,
                                          b_hint, pairs, out))
    return tuple(out)


def kernel_launches(params: FlceParams, phase: int) -> int:
    """Kernels one forward (phase 0) / backward (phase 1) call enqueues."""
    return int(load_library().flce_kernel_launches(ctypes.byref(params), phase))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t, name, dtype, shape, device=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the other tensors on {device}")


def _on_current_device(t):
    """The library launches on the current CUDA device: the tensors must live there."""
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensors are on {t.device} but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()} (use torch.cuda.device)")
    return t.device


def _need_out(out, names_shapes_dtypes, device):
    if len(out) != len(names_shapes_dtypes):
        raise ValueError(f"out must hold {len(names_shapes_dtypes)} tensors")
    for t, (name, shape, dtype) in zip(out, names_shapes_dtypes):
        _need(t, name, dtype, shape, device)
    return out


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _workspace(params, phase, device, workspace):
    """The caller's workspace (checked), or a new one when none is given."""
    need = workspace_size(params, phase)
    if workspace is None:
        return torch.empty(need, dtype=torch.uint8, device=device)
    if not isinstance(workspace, torch.Tensor) or workspace.dtype != torch.uint8 \
            or not workspace.is_contiguous() or workspace.device != device:
        raise TypeError(f"workspace must be a contiguous uint8 tensor on {device}")
    if workspace.numel() < need:
        # never a silent allocation behind a caller that passes its own memory
        raise ValueError(f"workspace holds {workspace.numel()} bytes; this call needs {need} "
                         f"(workspace_size(params, {phase}))")
    return workspace


def flce_forward(hidden, weight, labels, reduction="mean", ignore_index=IGNORE_INDEX,
                 zloss_coef=0.0, softcap=0.0, validate=False, workspace=None, stream=None,
                 out=None, weight_layout="hv", label_smoothing=0.0, class_weight=None):
    """Forward pass through the C ABI.

    Returns (loss, entropy, lse, ez): loss/entropy are [N] for reduction 'none'
    and [1] otherwise; lse/ez are the per-row [N] statistics saved for backward.
    weight is [H,V] (weight_layout 'hv') or [V,H] ('vh', nn.Linear).  label_smoothing
    and class_weight (CUDA fp32 [V]) follow torch's cross_entropy definitions.
    """
    lib = load_library()
    N, H, V, wshape = _dims(hidden, weight, weight_layout)
    _need(hidden, "hidden", torch.bfloat16, (N, H))
    dev = _on_current_device(hidden)
    _need(weight, "weight", torch.bfloat16, wshape, dev)
    _need(labels, "labels", torch.int64, (N,), dev)
    if class_weight is not None:
        _need(class_weight, "class_weight", torch.float32, (V,), dev)
    p = make_params(N, H, V, reduction, ignore_index, zloss_coef, softcap, validate,
                    weight_layout=weight_layout, label_smoothing=label_smoothing,
                    class_weight=class_weight)
    n_out = N if p.reduction == RED_NONE else 1
    if out is None:
        loss = torch.empty(n_out, dtype=torch.float32, device=dev)
        ent = torch.empty(n_out, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        ez = torch.empty(N, dtype=torch.float32, device=dev)
    else:
        f32 = torch.float32
        loss, ent, lse, ez = _need_out(out, [("loss", (n_out,), f32), ("entropy", (n_out,), f32),
                                             ("lse", (N,), f32), ("ez", (N,), f32)], dev)
    ws = _workspace(p, 0, dev, workspace)
    _check(lib.flce_forward(ctypes.byref(p), _ptr(hidden), _ptr(weight), _ptr(labels),
                            _ptr(loss), _ptr(ent), _ptr(lse), _ptr(ez), _ptr(ws), ws.numel(),
                            _stream(stream)))
    return loss, ent, lse, ez


def flce_backward(hidden, weight, labels, lse, ez, g_loss, g_entropy, reduction="mean",
                  ignore_index=IGNORE_INDEX, zloss_coef=0.0, softcap=0.0, validate=False,
                  chunk_v=0, workspace=None, stream=None, out=None, weight_layout="hv",
                  label_smoothing=0.0, class_weight=None, v_offset=0, v_total=0,
                  dhidden_fp32=False):
    """Backward pass through the C ABI; returns (dhidden [N,H] bf16 -- fp32 with
    dhidden_fp32 --, dweight bf16 shaped like weight).

    g_loss / g_entropy: fp32 [N] for reduction 'none', [1] otherwise, or None (zero).
    With a vocabulary shard (v_total > 0) dweight is the shard's and dhidden is the
    shard's term of the sum over shards.
    """
    lib = load_library()
    N, H, V, wshape = _dims(hidden, weight, weight_layout)
    _need(hidden, "hidden", torch.bfloat16, (N, H))
    dev = _on_current_device(hidden)
    _need(weight, "weight", torch.bfloat16, wshape, dev)
    _need(labels, "labels", torch.int64, (N,), dev)
    _need(lse, "lse", torch.float32, (N,), dev)
    _need(ez, "ez", torch.float32, (N,), dev)
    if class_weight is not None:
        _need(class_weight, "class_weight", torch.float32, (V,), dev)
    p = make_params(N, H, V, reduction, ignore_index, zloss_coef, softcap, validate, chunk_v,
                    weight_layout, label_smoothing, class_weight, v_offset, v_total,
                    dhidden_fp32=dhidden_fp32)
    n_g = N if p.reduction == RED_NONE else 1
    if g_loss is not None:
        _need(g_loss, "g_loss", torch.float32, (n_g,), dev)
    if g_entropy is not None:
        _need(g_entropy, "g_entropy", torch.float32, (n_g,), dev)
    dh_dtype = torch.float32 if dhidden_fp32 else torch.bfloat16
    if out is None:
        dh = torch.empty(N, H, dtype=dh_dtype, device=dev)
        dw = torch.empty(wshape, dtype=torch.bfloat16, device=dev)
    else:
        dh, dw = _need_out(out, [("dhidden", (N, H), dh_dtype),
                                 ("dweight", wshape, torch.bfloat16)], dev)
    ws = _workspace(p, 1, dev, workspace)
    _check(lib.flce_backward(ctypes.byref(p), _ptr(hidden), _ptr(weight), _ptr(labels),
                             _ptr(lse), _ptr(ez), _ptr(g_loss), _ptr(g_entropy), _ptr(dh),
                             _ptr(dw), _ptr(ws), ws.numel(), _stream(stream)))
    return dh, dw


def flce_forward_backward(hidden, weight, labels, g_loss, g_entropy, reduction="mean",
                          ignore_index=IGNORE_INDEX, zloss_coef=0.0, softcap=0.0,
                          validate=False, chunk_n=0, workspace=None, stream=None, out=None,
                          weight_layout="hv", label_smoothing=0.0, class_weight=None,
                          dhidden_fp32=False):
    """Forward and backward in one call (the upstream gradients known up front).

    g_loss / g_entropy: fp32 [N] for reduction 'none', [1] otherwise, or None (zero).
    Returns (loss, entropy, lse, ez, dhidden, dweight) -- what flce_forward followed by
    flce_backward returns -- at 6*N*H*V flops instead of 8*N*H*V.  dhidden is fp32
    with dhidden_fp32.
    """
    lib = load_library()
    N, H, V, wshape = _dims(hidden, weight, weight_layout)
    _need(hidden, "hidden", torch.bfloat16, (N, H))
    dev = _on_current_device(hidden)
    _need(weight, "weight", torch.bfloat16, wshape, dev)
    _need(labels, "labels", torch.int64, (N,), dev)
    if class_weight is not None:
        _need(class_weight, "class_weight", torch.float32, (V,), dev)
    p = make_params(N, H, V, reduction, ignore_index, zloss_coef, softcap, validate,
                    weight_layout=weight_layout, label_smoothing=label_smoothing,
                    class_weight=class_weight, chunk_n=chunk_n, dhidden_fp32=dhidden_fp32)
    n_g = N if p.reduction == RED_NONE else 1
    dh_dtype = torch.float32 if dhidden_fp32 else torch.bfloat16
    if g_loss is not None:
        _need(g_loss, "g_loss", torch.float32, (n_g,), dev)
    if g_entropy is not None:
        _need(g_entropy, "g_entropy", torch.float32, (n_g,), dev)
    if out is None:
        loss = torch.empty(n_g, dtype=torch.float32, device=dev)
        ent = torch.empty(n_g, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        ez = torch.empty(N, dtype=torch.float32, device=dev)
        dh = torch.empty(N, H, dtype=dh_dtype, device=dev)
        dw = torch.empty(wshape, dtype=torch.bfloat16, device=dev)
    else:
        f32, bf = torch.float32, torch.bfloat16
        loss, ent, lse, ez, dh, dw = _need_out(
            out, [("loss", (n_g,), f32), ("entropy", (n_g,), f32), ("lse", (N,), f32),
                  ("ez", (N,), f32), ("dhidden", (N, H), dh_dtype),
                  ("dweight", wshape, bf)], dev)
    ws = _workspace(p, 3, dev, workspace)
    _check(lib.flce_forward_backward(ctypes.byref(p), _ptr(hidden), _ptr(weight), _ptr(labels),
                                     _ptr(g_loss), _ptr(g_entropy), _ptr(loss), _ptr(ent),
                                     _ptr(lse), _ptr(ez), _ptr(dh), _ptr(dw), _ptr(ws),
                                     ws.numel(), _stream(stream)))
    return loss, ent, lse, ez, dh, dw


def flce_scale_bf16(x, g, stream=None):
    """x *= g[0] in place (x: contiguous CUDA bf16, g: CUDA fp32 [1]); a no-op on the
    device when g is exactly 1."""
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.bfloat16 \
            or not x.is_contiguous():
        raise TypeError("x must be a contiguous CUDA bf16 tensor")
    dev = _on_current_device(x)
    _need(g, "g", torch.float32, (1,), dev)
    _check(load_library().flce_scale_bf16(_ptr(x), x.numel(), _ptr(g), _stream(stream)))
    return x


def flce_shard_stats(hidden, weight, labels, v_offset, v_total, softcap=0.0,
                     ignore_index=IGNORE_INDEX, weight_layout="hv", validate=False,
                     workspace=None, stream=None, out=None):
    """Statistics [4, N] fp32 of one vocabulary shard (columns [v_offset, v_offset + V)
    of v_total); see flce.h for their meaning."""
    lib = load_library()
    N, H, V, wshape = _dims(hidden, weight, weight_layout)
    _need(hidden, "hidden", torch.bfloat16, (N, H))
    dev = _on_current_device(hidden)
    _need(weight, "weight", torch.bfloat16, wshape, dev)
    _need(labels, "labels", torch.int64, (N,), dev)
    p = make_params(N, H, V, "none", ignore_index, 0.0, softcap, validate,
                    weight_layout=weight_layout, v_offset=v_offset, v_total=v_total)
    if out is not None:
        _need(out, "out", torch.float32, (4, N), dev)
    stats = out if out is not None else torch.empty(4, N, dtype=torch.float32, device=dev)
    ws = _workspace(p, 0, dev, workspace)
    _check(lib.flce_shard_stats(ctypes.byref(p), _ptr(hidden), _ptr(weight), _ptr(labels),
                                _ptr(stats), _ptr(ws), ws.numel(), _stream(stream)))
    return stats


def flce_combine_shards(stats, labels, v_total, reduction="mean", ignore_index=IGNORE_INDEX,
                        zloss_coef=0.0, H=8, validate=False, workspace=None, stream=None):
    """Merge [P, 4, N] shard statistics into (loss, entropy, lse, ez) for the whole
    vocabulary of v_total entries."""
    lib = load_library()
    P, four, N = stats.shape
    _need(stats, "stats", torch.float32, (P, 4, N))
    dev = _on_current_device(stats)
    _need(labels, "labels", torch.int64, (N,), dev)
    # No weight is read here: the parameters describe the whole vocabulary as one
    # shard, in the [V,H] layout, which puts no alignment rule on its size.
    p = make_params(N, H, v_total, reduction, ignore_index, zloss_coef, 0.0, validate,
                    weight_layout=WEIGHT_VH, v_offset=0, v_total=v_total)
    n_out = N if p.reduction == RED_NONE else 1
    loss = torch.empty(n_out, dtype=torch.float32, device=dev)
    ent = torch.empty(n_out, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    ez = torch.empty(N, dtype=torch.float32, device=dev)
    ws = _workspace(p, 2, dev, workspace)
    _check(lib.flce_combine_shards(ctypes.byref(p), _ptr(stats), P, _ptr(labels), _ptr(loss),
                                   _ptr(ent), _ptr(lse), _ptr(ez), _ptr(ws), ws.numel(),
                                   _stream(stream)))
    return loss, ent, lse, ez


def selftest_wait_timeout(limit_ns=20_000_000, stream=None) -> int:
    """Run the bounded-wait self-test (a wait that nothing satisfies, given up after
    limit_ns) and return the status flce_status then reads (FLCE_ERR_TIMEOUT = 6)."""
    lib = load_library()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    _check(lib.flce_selftest_wait_timeout(_ptr(ws), ws.numel(), int(limit_ns), _stream(stream)))
    return flce_status(ws, stream)


def flce_status(workspace, stream=None) -> int:
    """Device-side status of the last call that used `workspace` (synchronises)."""
    return int(load_library().flce_status(_ptr(workspace), _stream(stream)))


class _LinearCrossEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight, labels, reduction, ignore_index, zloss_coef, softcap,
                weight_layout, label_smoothing, class_weight):
        loss, ent, lse, ez = flce_forward(hidden, weight, labels, reduction, ignore_index,
                                          zloss_coef, softcap, weight_layout=weight_layout,
                                          label_smoothing=label_smoothing,
                                          class_weight=class_weight)
        ctx.save_for_backward(hidden, weight, labels, lse, ez)
        ctx.cfg = (reduction, ignore_index, zloss_coef, softcap, weight_layout,
                   label_smoothing, class_weight)
        if reduction_code(reduction) != RED_NONE:
            loss, ent = loss[0], ent[0]
        return loss, ent

    @staticmethod
    def backward(ctx, g_loss, g_ent):
        hidden, weight, labels, lse, ez = ctx.saved_tensors
        (reduction, ignore_index, zloss_coef, softcap, weight_layout, label_smoothing,
         class_weight) = ctx.cfg
        n_g = hidden.shape[0] if reduction_code(reduction) == RED_NONE else 1

        def prep(g):
            if g is None:
                return None
            return g.detach().reshape(n_g).to(torch.float32).contiguous()

        dh, dw = flce_backward(hidden, weight, labels, lse, ez, prep(g_loss), prep(g_ent),
                               reduction, ignore_index, zloss_coef, softcap,
                               weight_layout=weight_layout, label_smoothing=label_smoothing,
                               class_weight=class_weight)
        return dh, dw, None, None, None, None, None, None, None, None


class _LinearCrossEntropyGradInForward(torch.autograd.Function):
    """The gradients of loss + entropy_coef * entropy are computed in the forward
    (flce_forward_backward with g_loss = 1) and scaled by the loss's upstream
    gradient in the backward; the entropy output carries no gradient of its own."""

    @staticmethod
    def forward(ctx, hidden, weight, labels, reduction, ignore_index, zloss_coef, softcap,
                weight_layout, label_smoothing, class_weight, entropy_coef):
        if reduction_code(reduction) == RED_NONE:
            raise ValueError("grad_in_forward needs reduction 'mean' or 'sum'")
        dev = hidden.device
        one = torch.ones(1, dtype=torch.float32, device=dev)
        ce = torch.full((1,), float(entropy_coef), dtype=torch.float32, device=dev)
        loss, ent, _, _, dh, dw = flce_forward_backward(
            hidden, weight, labels, one, ce, reduction, ignore_index, zloss_coef, softcap,
            weight_layout=weight_layout, label_smoothing=label_smoothing,
            class_weight=class_weight)
        ctx.save_for_backward(dh, dw)
        ctx.mark_non_differentiable(ent)
        return loss[0], ent[0]

    @staticmethod
    def backward(ctx, g_loss, g_ent):
        dh, dw = ctx.saved_tensors
        if g_loss is None:
            return (None,) * 11
        g = g_loss.detach().reshape(1).to(torch.float32).contiguous()
        flce_scale_bf16(dh, g)
        flce_scale_bf16(dw, g)
        return dh, dw, None, None, None, None, None, None, None, None, None


def linear_cross_entropy(hidden, weight, labels, reduction="mean", ignore_index=IGNORE_INDEX,
                         zloss_coef=0.0, softcap=0.0, weight_layout="hv", label_smoothing=0.0,
                         class_weight=None, grad_in_forward=False, entropy_coef=0.0):
    """loss, entropy = linear_cross_entropy(hidden, weight, labels, reduction)

    The call of verl PR #462 ("API"): hidden [N,H] bf16, weight [H,V] bf16,
    labels [N] int64.  `loss` is the cross-entropy (+ z-loss); the page's
    log-probability is -loss when z-loss is off.  Differentiable w.r.t. hidden
    and weight.  weight_layout='vh' takes an nn.Linear-style weight [V,H];
    label_smoothing and class_weight (fp32 [V], not differentiated) follow torch's
    cross_entropy.

    grad_in_forward=True (reduction 'mean' or 'sum'; Liger-Kernel PR #551's
    gradient in forward): the forward also computes the gradients of
    loss + entropy_coef * entropy, with no recompute in the backward, which only
    scales them by the loss's upstream gradient.  The entropy output is then not
    differentiable: its weight in the objective is entropy_coef.
    """
    if grad_in_forward:
        return _LinearCrossEntropyGradInForward.apply(
            hidden, weight, labels, reduction, ignore_index, zloss_coef, softcap, weight_layout,
            label_smoothing, class_weight, entropy_coef)
    return _LinearCrossEntropy.apply(hidden, weight, labels, reduction, ignore_index,
                                     zloss_coef, softcap, weight_layout, label_smoothing,
                                     class_weight)
