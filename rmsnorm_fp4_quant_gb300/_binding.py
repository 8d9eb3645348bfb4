"""ctypes binding of libfp4q.so: argument marshalling only, no computation."""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional, Tuple

from .build import DEBUG_LIBPATH, LIBPATH

FP4_DT_BF16, FP4_DT_FP16 = 0, 1
FP4_NVFP4, FP4_MXFP4, FP4_E4M3_B32 = 0, 1, 2
FP4_SF_ROWMAJOR, FP4_SF_SWIZZLED, FP4_SF_BOTH = 0, 1, 2
FP4_OK, FP4_ERR_INVALID_ARG, FP4_ERR_UNSUPPORTED_SHAPE, FP4_ERR_MISALIGNED = 0, 1, 2, 3
FP4_ERR_CUDA, FP4_ERR_TIMEOUT = 4, 5
FP4_EPI_BF16, FP4_EPI_GELU_BF16, FP4_EPI_GELU_NVFP4 = 0, 1, 2

_FORMATS = {"nvfp4": FP4_NVFP4, "mxfp4": FP4_MXFP4, "e4m3b32": FP4_E4M3_B32}
_LAYOUTS = {"rowmajor": FP4_SF_ROWMAJOR, "swizzled": FP4_SF_SWIZZLED, "both": FP4_SF_BOTH}
_BLOCK = {FP4_NVFP4: 16, FP4_MXFP4: 32, FP4_E4M3_B32: 32}

_lib = None
_debug_lib = None
_override = None     # the library the calls below go to inside `using_library`


class Fp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = f"{where}: {fp4_status_string(status)} (status {status})"
        if status == 4:
            msg += f", cudaError {fp4_last_cuda_error()}"
        super().__init__(msg)
        self.status = status


def lib_path() -> str:
    return LIBPATH


def lib() -> ctypes.CDLL:
    """Loads libfp4q.so (once) and returns it (or the library selected with
    `using_library`).  Raises if it has not been built."""
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        _lib = _open(LIBPATH, "python -m rmsnorm_fp4_quant_gb300.build")
    return _lib


def debug_lib() -> ctypes.CDLL:
    """Loads libfp4q_debug.so, the build with bounds checks and the fault
    injector (include/fp4q.h, "Debug build").  Raises if it has not been built."""
    global _debug_lib
    if _debug_lib is None:
        _debug_lib = _open(DEBUG_LIBPATH, "python -m rmsnorm_fp4_quant_gb300.build --debug")
    return _debug_lib


@contextlib.contextmanager
def using_library(L: ctypes.CDLL):
    """Inside the block every call of this module goes to `L` (e.g. debug_lib())."""
    global _override
    old = _override
    _override = L
    try:
        yield L
    finally:
        _override = old


def _open(path: str, how: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `{how}` (needs nvcc)")
    L = ctypes.CDLL(path)
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.fp4_add_rmsnorm_quant.argtypes = [vp, vp, vp, ctypes.c_float, i64, i64, ci, ci, ci,
                                        vp, vp, vp, vp]
    L.fp4_add_rmsnorm_quant.restype = ci
    L.fp4_add_rmsnorm_quant_gs.argtypes = [vp, vp, vp, vp, ctypes.c_float, i64, i64, ci, ci, ci,
                                           vp, vp, vp, vp]
    L.fp4_add_rmsnorm_quant_gs.restype = ci
    L.fp4_add_rmsnorm_quant_ex.argtypes = [vp, i64, vp, i64, vp, vp, ctypes.c_float, i64, i64,
                                           ci, ci, ci, vp, vp, vp, vp, vp, ci, vp]
    L.fp4_add_rmsnorm_quant_ex.restype = ci
    L.fp4_quantize.argtypes = [vp, vp, i64, i64, ci, ci, ci, vp, vp, vp, ci, vp]
    L.fp4_quantize.restype = ci
    L.fp4_dequant.argtypes = [vp, vp, i64, i64, ci, ci, vp, vp]
    L.fp4_dequant.restype = ci
    L.fp4_sf_size_bytes.argtypes = [i64, i64, ci, ci]
    L.fp4_sf_size_bytes.restype = i64
    L.fp4_status_string.argtypes = [ci]
    L.fp4_status_string.restype = ctypes.c_char_p
    L.fp4_last_cuda_error.argtypes = []
    L.fp4_last_cuda_error.restype = ci
    L.fp4_launch_shape.argtypes = [i64, i64, ci, ci, ci, ctypes.POINTER(ctypes.c_int64)]
    L.fp4_launch_shape.restype = ci
    L.fp4_gemm_nvfp4_bf16.argtypes = [vp, vp, vp, vp, ctypes.c_float, vp, vp, i64, i64, i64,
                                      vp, ci, ci, vp]
    L.fp4_gemm_nvfp4_bf16.restype = ci
    L.fp4_gemm_mxfp4_bf16.argtypes = L.fp4_gemm_nvfp4_bf16.argtypes
    L.fp4_gemm_mxfp4_bf16.restype = ci
    L.fp4_gemm_nvfp4_gelu_bf16.argtypes = [vp, vp, vp, vp, ctypes.c_float, vp, i64, i64, i64,
                                           vp, ci, ci, vp]
    L.fp4_gemm_nvfp4_gelu_bf16.restype = ci
    L.fp4_gemm_nvfp4_gelu_nvfp4.argtypes = [vp, vp, vp, vp, ctypes.c_float, vp, i64, i64, i64,
                                            vp, vp, ci, ci, vp]
    L.fp4_gemm_nvfp4_gelu_nvfp4.restype = ci
    L.fp4_gemm_variant.argtypes = [i64, i64, i64, ci, ci, ci]
    L.fp4_gemm_variant.restype = ci
    L.fp4_gemm_ex.argtypes = [vp, vp, vp, vp, ci, ci, ctypes.c_float, vp, vp, i64, i64, i64,
                              vp, vp, vp, ci, ci, vp, vp]
    L.fp4_gemm_ex.restype = ci
    L.fp4_read_device_status.argtypes = [vp, vp]
    L.fp4_read_device_status.restype = ci
    L.fp4_debug_build.argtypes = []
    L.fp4_debug_build.restype = ci
    L.fp4_debug_configure.argtypes = [i64, i64, ci, ci, ci, vp]
    L.fp4_debug_configure.restype = ci
    return L


# ---------------------------------------------------------------------------
# Same names as the C ABI; raw integer addresses and a raw stream handle.
# ---------------------------------------------------------------------------
def fp4_add_rmsnorm_quant(input_ptr: int, residual_ptr: int, weight_ptr: int, eps: float,
                          M: int, H: int, dtype: int, fmt: int, sf_layout: int,
                          out_packed_ptr: int, out_sf_ptr: int, out_sf_rowmajor_ptr: int,
                          stream: int) -> int:
    return lib().fp4_add_rmsnorm_quant(input_ptr, residual_ptr, weight_ptr, eps, M, H, dtype,
                                       fmt, sf_layout, out_packed_ptr, out_sf_ptr,
                                       out_sf_rowmajor_ptr or None, stream or None)


def fp4_add_rmsnorm_quant_gs(input_ptr: int, residual_ptr: int, weight_ptr: int,
                             global_scale_ptr: int, eps: float, M: int, H: int, dtype: int,
                             fmt: int, sf_layout: int, out_packed_ptr: int, out_sf_ptr: int,
                             out_sf_rowmajor_ptr: int, stream: int) -> int:
    return lib().fp4_add_rmsnorm_quant_gs(input_ptr, residual_ptr, weight_ptr,
                                          global_scale_ptr or None, eps, M, H, dtype, fmt,
                                          sf_layout, out_packed_ptr, out_sf_ptr,
                                          out_sf_rowmajor_ptr or None, stream or None)


def fp4_add_rmsnorm_quant_ex(input_ptr: int, input_row_stride: int, residual_ptr: int,
                             residual_row_stride: int, weight_ptr: int, global_scale_ptr: int,
                             eps: float, M: int, H: int, dtype: int, fmt: int, sf_layout: int,
                             out_packed_ptr: int, out_sf_ptr: int, out_sf_rowmajor_ptr: int,
                             out_y_ptr: int, status_ptr: int, pdl: int, stream: int) -> int:
    return lib().fp4_add_rmsnorm_quant_ex(input_ptr, input_row_stride, residual_ptr,
                                          residual_row_stride, weight_ptr, global_scale_ptr or None,
                                          eps, M, H, dtype, fmt, sf_layout, out_packed_ptr,
                                          out_sf_ptr, out_sf_rowmajor_ptr or None,
                                          out_y_ptr or None, status_ptr or None, pdl,
                                          stream or None)


def fp4_quantize(input_ptr: int, global_scale_ptr: int, M: int, H: int, dtype: int, fmt: int,
                 sf_layout: int, out_packed_ptr: int, out_sf_ptr: int, out_sf_rowmajor_ptr: int,
                 pdl: int, stream: int) -> int:
    return lib().fp4_quantize(input_ptr, global_scale_ptr or None, M, H, dtype, fmt, sf_layout,
                              out_packed_ptr, out_sf_ptr, out_sf_rowmajor_ptr or None, pdl,
                              stream or None)


def fp4_dequant(packed_ptr: int, sf_ptr: int, M: int, H: int, fmt: int, sf_layout: int,
                out_ptr: int, stream: int) -> int:
    return lib().fp4_dequant(packed_ptr, sf_ptr, M, H, fmt, sf_layout, out_ptr, stream or None)


def fp4_gemm_nvfp4_bf16(a_packed_ptr: int, b_packed_ptr: int, sfa_ptr: int, sfb_ptr: int,
                        alpha: float, bias_ptr: int, residual_ptr: int, M: int, N: int, K: int,
                        out_ptr: int, variant: int, pdl: int, stream: int) -> int:
    return lib().fp4_gemm_nvfp4_bf16(a_packed_ptr, b_packed_ptr, sfa_ptr, sfb_ptr, alpha,
                                     bias_ptr or None, residual_ptr or None, M, N, K, out_ptr,
                                     variant, pdl, stream or None)


def fp4_gemm_mxfp4_bf16(a_packed_ptr: int, b_packed_ptr: int, sfa_ptr: int, sfb_ptr: int,
                        alpha: float, bias_ptr: int, residual_ptr: int, M: int, N: int, K: int,
                        out_ptr: int, variant: int, pdl: int, stream: int) -> int:
    return lib().fp4_gemm_mxfp4_bf16(a_packed_ptr, b_packed_ptr, sfa_ptr, sfb_ptr, alpha,
                                     bias_ptr or None, residual_ptr or None, M, N, K, out_ptr,
                                     variant, pdl, stream or None)


def fp4_gemm_nvfp4_gelu_bf16(a_packed_ptr: int, b_packed_ptr: int, sfa_ptr: int, sfb_ptr: int,
                             alpha: float, bias_ptr: int, M: int, N: int, K: int, out_ptr: int,
                             variant: int, pdl: int, stream: int) -> int:
    return lib().fp4_gemm_nvfp4_gelu_bf16(a_packed_ptr, b_packed_ptr, sfa_ptr, sfb_ptr, alpha,
                                          bias_ptr or None, M, N, K, out_ptr, variant, pdl,
                                          stream or None)


def fp4_gemm_nvfp4_gelu_nvfp4(a_packed_ptr: int, b_packed_ptr: int, sfa_ptr: int, sfb_ptr: int,
                              alpha: float, bias_ptr: int, M: int, N: int, K: int,
                              out_packed_ptr: int, out_sf_ptr: int, variant: int, pdl: int,
                              stream: int) -> int:
    return lib().fp4_gemm_nvfp4_gelu_nvfp4(a_packed_ptr, b_packed_ptr, sfa_ptr, sfb_ptr, alpha,
                                           bias_ptr or None, M, N, K, out_packed_ptr,
                                           out_sf_ptr, variant, pdl, stream or None)


def fp4_gemm_ex(a_packed_ptr: int, b_packed_ptr: int, sfa_ptr: int, sfb_ptr: int, fmt: int,
                epilogue: int, alpha: float, bias_ptr: int, residual_ptr: int, M: int, N: int,
                K: int, out_ptr: int, out_packed_ptr: int, out_sf_ptr: int, variant: int,
                pdl: int, status_ptr: int, stream: int) -> int:
    return lib().fp4_gemm_ex(a_packed_ptr, b_packed_ptr, sfa_ptr, sfb_ptr, fmt, epilogue, alpha,
                             bias_ptr or None, residual_ptr or None, M, N, K, out_ptr or None,
                             out_packed_ptr or None, out_sf_ptr or None, variant, pdl,
                             status_ptr or None, stream or None)


def fp4_read_device_status(status_ptr: int, stream: int) -> int:
    return lib().fp4_read_device_status(status_ptr or None, stream or None)


def fp4_debug_build() -> int:
    return lib().fp4_debug_build()


def fp4_debug_configure(wait_limit_cycles: int, shrink_bytes: int, drop_kernel: int,
                        drop_cta: int, drop_iter: int, violations_ptr: int) -> int:
    return lib().fp4_debug_configure(wait_limit_cycles, shrink_bytes, drop_kernel, drop_cta,
                                     drop_iter, violations_ptr or None)


def fp4_sf_size_bytes(M: int, H: int, fmt: int, layout: int) -> int:
    return lib().fp4_sf_size_bytes(M, H, fmt, layout)


def fp4_status_string(status: int) -> str:
    return lib().fp4_status_string(status).decode()


def fp4_last_cuda_error() -> int:
    return lib().fp4_last_cuda_error()


_SHAPE_KEYS = ("kernel", "chunks_per_thread", "threads_per_slice", "slices_per_cta",
               "cluster", "stages", "threads_per_cta", "ctas")


def fp4_launch_shape(M: int, H: int, dtype: int, fmt: int, sf_layout: int) -> dict:
    """The launch fp4_add_rmsnorm_quant would make on the current device."""
    out = (ctypes.c_int64 * 8)()
    st = lib().fp4_launch_shape(M, H, dtype, fmt, sf_layout, out)
    if st != 0:
        raise Fp4Error(st, "fp4_launch_shape")
    d = dict(zip(_SHAPE_KEYS, list(out)))
    d["kernel"] = "fused_tma_kernel" if d["kernel"] == 0 else "fused_direct_kernel"
    return d


# GEMM schedules by `variant` number: (kernel, output tile width)
_GEMM_SCHEDULES = {0: ("gemm_nvfp4_kernel", 128), 1: ("gemm_nvfp4_kernel", 256),
                   2: ("gemm_nvfp4_persistent_kernel", 128),
                   3: ("gemm_nvfp4_persistent_kernel", 256), 4: ("gemm_nvfp4_kernel", 128)}


def fp4_gemm_variant(M: int, N: int, K: int, fmt: int = 0, fp4_out: bool = False,
                     variant: int = -1) -> dict:
    """The schedule the GEMM entry points would run for an M x N x K product
    on the current device: {"variant", "kernel", "tile_n", "split_k"}."""
    v = lib().fp4_gemm_variant(M, N, K, fmt, 1 if fp4_out else 0, variant)
    if v < 0:
        raise ValueError("the GEMM rejects these sizes or this variant")
    kernel, tile_n = _GEMM_SCHEDULES[v]
    return {"variant": v, "kernel": kernel, "tile_n": tile_n, "split_k": v == 4}


# ---------------------------------------------------------------------------
# torch-tensor convenience layer (allocation and stream lookup only)
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _check_cuda(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return FP4_DT_BF16
    if t.dtype == torch.float16:
        return FP4_DT_FP16
    raise ValueError("dtype must be bfloat16 or float16")


def _gs_ptr(global_scale) -> int:
    if global_scale is None:
        return 0
    torch = _torch()
    _check_cuda(global_scale, "global_scale")
    if global_scale.dtype != torch.float32 or global_scale.numel() != 1:
        raise ValueError("global_scale must be a CUDA float32 tensor with one element")
    return global_scale.data_ptr()


def _outputs(lead, M, H, f, lay, dev, out_packed, out_sf, out_sf_rowmajor):
    torch = _torch()
    if out_packed is None:
        out_packed = torch.empty(*lead, H // 2, dtype=torch.uint8, device=dev)
    nb = H // _BLOCK[f]
    if out_sf is None:
        if lay == FP4_SF_ROWMAJOR:
            out_sf = torch.empty(*lead, nb, dtype=torch.uint8, device=dev)
        else:
            out_sf = torch.empty(max(fp4_sf_size_bytes(M, H, f, lay), 0), dtype=torch.uint8,
                                 device=dev)
    if lay == FP4_SF_BOTH and out_sf_rowmajor is None:
        out_sf_rowmajor = torch.empty(*lead, nb, dtype=torch.uint8, device=dev)
    for name, t in (("out_packed", out_packed), ("out_sf", out_sf)):
        _check_cuda(t, name)
    return out_packed, out_sf, out_sf_rowmajor


def _row_stride(t, name) -> int:
    """Elements between rows: dense tensors, or 2-D views with unit column stride
    (e.g. a column slice of a wider matrix)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.is_contiguous():
        return t.shape[-1]
    if t.dim() == 2 and t.stride(1) == 1:
        return t.stride(0)
    raise ValueError(f"{name} must be contiguous or a 2-D view with unit column stride")


def _status_ptr(status) -> int:
    if status is None:
        return 0
    torch = _torch()
    _check_cuda(status, "status")
    if status.dtype != torch.int32 or status.numel() != 1:
        raise ValueError("status must be a CUDA int32 tensor with one element")
    return status.data_ptr()


def read_device_status(status, stream=None) -> int:
    """Synchronises the stream and returns the device status word as a status
    code (FP4_OK or FP4_ERR_TIMEOUT)."""
    st = fp4_read_device_status(_status_ptr(status), _stream_handle(stream))
    if st not in (FP4_OK, FP4_ERR_TIMEOUT):
        raise Fp4Error(st, "fp4_read_device_status")
    return st


def add_rmsnorm_fp4quant(input, residual, weight, eps: float = 1e-6, fmt: str = "nvfp4",
                         sf_layout: str = "rowmajor", out_packed=None, out_sf=None,
                         out_sf_rowmajor=None, global_scale=None, return_y: bool = False,
                         out_y=None, status=None, pdl: bool = False, stream=None) -> Tuple:
    """residual += input (in place); returns (packed, sf) or, for
    sf_layout="both", (packed, sf_tiled, sf_rowmajor), with y (the normalised,
    weighted rows in the input dtype) appended when return_y is set or out_y
    given.  ``input`` may be 2-D (M, H), a 2-D view with a row stride, or 3-D
    (B, S, H); packed has the same leading shape with H/2 bytes.  Scale buffers
    are uint8: row-major (M, H/b), tiled flat.  ``global_scale``: optional CUDA
    float32 tensor of one element (E4M3 formats).  ``status``: optional CUDA
    int32 tensor of one element that receives FP4_ERR_TIMEOUT if a kernel
    gave up on a bounded wait (never cleared by the call).  ``pdl``: launch as
    a programmatic dependent of the previous kernel on the stream."""
    xs = _row_stride(input, "input")
    rs = _row_stride(residual, "residual")
    _check_cuda(weight, "weight")
    if input.shape != residual.shape or input.dtype != residual.dtype:
        raise ValueError("input and residual must have the same shape and dtype")
    if weight.dtype != input.dtype or weight.dim() != 1 or weight.shape[0] != input.shape[-1]:
        raise ValueError("weight must be (H,) with the input's dtype")
    torch = _torch()
    dt = _dtype_code(input)
    f = _FORMATS[fmt]
    lay = _LAYOUTS[sf_layout]
    H = input.shape[-1]
    lead = tuple(input.shape[:-1])
    M = 1
    for d in lead:
        M *= d
    out_packed, out_sf, out_sf_rowmajor = _outputs(lead, M, H, f, lay, input.device, out_packed,
                                                   out_sf, out_sf_rowmajor)
    if return_y and out_y is None:
        out_y = torch.empty(*lead, H, dtype=input.dtype, device=input.device)
    if out_y is not None:
        _check_cuda(out_y, "out_y")
    st = fp4_add_rmsnorm_quant_ex(input.data_ptr(), xs, residual.data_ptr(), rs, weight.data_ptr(),
                                  _gs_ptr(global_scale), float(eps), M, H, dt, f, lay,
                                  out_packed.data_ptr(), out_sf.data_ptr(),
                                  out_sf_rowmajor.data_ptr() if out_sf_rowmajor is not None else 0,
                                  out_y.data_ptr() if out_y is not None else 0,
                                  _status_ptr(status), 1 if pdl else 0, _stream_handle(stream))
    if st != 0:
        raise Fp4Error(st, "fp4_add_rmsnorm_quant")
    outs = (out_packed, out_sf, out_sf_rowmajor) if lay == FP4_SF_BOTH else (out_packed, out_sf)
    return outs + (out_y,) if out_y is not None else outs


def quantize_fp4(x, fmt: str = "nvfp4", sf_layout: str = "swizzled", global_scale=None,
                 out_packed=None, out_sf=None, out_sf_rowmajor=None, pdl: bool = False,
                 stream=None) -> Tuple:
    """Block-quantize x (M, H) or (B, S, H) itself (no add, no norm); returns
    (packed, sf) or (packed, sf_tiled, sf_rowmajor) for sf_layout="both".
    ``pdl``: launch as a programmatic dependent of the previous kernel."""
    _check_cuda(x, "x")
    dt = _dtype_code(x)
    f = _FORMATS[fmt]
    lay = _LAYOUTS[sf_layout]
    H = x.shape[-1]
    lead = tuple(x.shape[:-1])
    M = 1
    for d in lead:
        M *= d
    out_packed, out_sf, out_sf_rowmajor = _outputs(lead, M, H, f, lay, x.device, out_packed,
                                                   out_sf, out_sf_rowmajor)
    st = fp4_quantize(x.data_ptr(), _gs_ptr(global_scale), M, H, dt, f, lay,
                      out_packed.data_ptr(), out_sf.data_ptr(),
                      out_sf_rowmajor.data_ptr() if out_sf_rowmajor is not None else 0,
                      1 if pdl else 0, _stream_handle(stream))
    if st != 0:
        raise Fp4Error(st, "fp4_quantize")
    if lay == FP4_SF_BOTH:
        return out_packed, out_sf, out_sf_rowmajor
    return out_packed, out_sf


def dequant(packed, sf, M: int, H: int, fmt: str = "nvfp4", sf_layout: str = "rowmajor",
            out=None, stream=None):
    """fp32 (M, H) = E2M1 value of each code times its block scale."""
    torch = _torch()
    _check_cuda(packed, "packed")
    _check_cuda(sf, "sf")
    if out is None:
        out = torch.empty(M, H, dtype=torch.float32, device=packed.device)
    st = fp4_dequant(packed.data_ptr(), sf.data_ptr(), M, H, _FORMATS[fmt], _LAYOUTS[sf_layout],
                     out.data_ptr(), _stream_handle(stream))
    if st != 0:
        raise Fp4Error(st, "fp4_dequant")
    return out


def _pdl_mode(pdl) -> int:
    """False / True -> 0 / 1; an int is passed on as given (2: static weights)."""
    return int(pdl) if not isinstance(pdl, bool) else (1 if pdl else 0)


def gemm_nvfp4_bf16(a_packed, b_packed, sfa, sfb, alpha: float = 1.0, bias=None, residual=None,
                    out=None, variant: int = -1, pdl=False, stream=None, fmt="nvfp4",
                    status=None):
    """bf16 (M, N) = alpha * deq(A) @ deq(B)^T (+ bias) (+ residual) from packed
    NVFP4 operands (M, K/2) and (N, K/2) and their tiled scale buffers.
    fmt "mxfp4" takes MXFP4 operands (UE8M0 scale per 32 codes) instead.
    variant: -1 automatic (see fp4_gemm_variant), 0 / 1 = one CTA per 128x128 /
    128x256 output tile, 2 / 3 = persistent CTAs over 128x128 / 128x256 tiles
    (automatic for many tiles), 4 = 128x128 tiles with the K loop split over a
    cluster (automatic for few output tiles and long K).  pdl: False / True (0 /
    1), or 2 when the kernel before this one writes neither b_packed nor sfb
    (B's first copies then start before the dependency wait).  status: optional
    CUDA int32 tensor of one element that receives FP4_ERR_TIMEOUT if a kernel
    gave up on a bounded wait (fp4_gemm_ex)."""
    torch = _torch()
    for name, t in (("a_packed", a_packed), ("b_packed", b_packed), ("sfa", sfa), ("sfb", sfb)):
        _check_cuda(t, name)
        if t.dtype != torch.uint8:
            raise ValueError(f"{name} must be uint8")
    M, K = a_packed.shape[0], 2 * a_packed.shape[-1]
    N = b_packed.shape[0]
    if b_packed.shape[-1] * 2 != K:
        raise ValueError("a_packed and b_packed disagree on K")
    for name, t in (("bias", bias), ("residual", residual)):
        if t is not None:
            _check_cuda(t, name)
            if t.dtype != torch.bfloat16:
                raise ValueError(f"{name} must be bfloat16")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=a_packed.device)
    _check_cuda(out, "out")
    if fmt not in ("nvfp4", "mxfp4"):
        raise ValueError("fmt must be 'nvfp4' or 'mxfp4'")
    if status is None:
        call = fp4_gemm_nvfp4_bf16 if fmt == "nvfp4" else fp4_gemm_mxfp4_bf16
        st = call(a_packed.data_ptr(), b_packed.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                  float(alpha), bias.data_ptr() if bias is not None else 0,
                  residual.data_ptr() if residual is not None else 0, M, N, K, out.data_ptr(),
                  int(variant), _pdl_mode(pdl), _stream_handle(stream))
    else:
        st = fp4_gemm_ex(a_packed.data_ptr(), b_packed.data_ptr(), sfa.data_ptr(),
                         sfb.data_ptr(), _FORMATS[fmt], FP4_EPI_BF16, float(alpha),
                         bias.data_ptr() if bias is not None else 0,
                         residual.data_ptr() if residual is not None else 0, M, N, K,
                         out.data_ptr(), 0, 0, int(variant), _pdl_mode(pdl),
                         _status_ptr(status), _stream_handle(stream))
    if st != 0:
        raise Fp4Error(st, f"fp4_gemm_{fmt}_bf16")
    return out


def gemm_nvfp4_gelu(a_packed, b_packed, sfa, sfb, alpha: float = 1.0, bias=None,
                    out_format: str = "bf16", variant: int = -1, pdl: bool = False, stream=None):
    """GELU(alpha * deq(A) @ deq(B)^T + bias) from NVFP4 operands; out_format
    "bf16" returns a (M, N) bf16 tensor, "nvfp4" returns (packed (M, N/2),
    tiled scales) ready to be the next GEMM's A operand."""
    torch = _torch()
    for name, t in (("a_packed", a_packed), ("b_packed", b_packed), ("sfa", sfa), ("sfb", sfb)):
        _check_cuda(t, name)
    if bias is not None:
        _check_cuda(bias, "bias")
        if bias.dtype != torch.bfloat16:
            raise ValueError("bias must be bfloat16")
    M, K, N = a_packed.shape[0], 2 * a_packed.shape[-1], b_packed.shape[0]
    bp = bias.data_ptr() if bias is not None else 0
    dev = a_packed.device
    if out_format == "bf16":
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        st = fp4_gemm_nvfp4_gelu_bf16(a_packed.data_ptr(), b_packed.data_ptr(), sfa.data_ptr(),
                                      sfb.data_ptr(), float(alpha), bp, M, N, K, out.data_ptr(),
                                      int(variant), _pdl_mode(pdl), _stream_handle(stream))
        if st != 0:
            raise Fp4Error(st, "fp4_gemm_nvfp4_gelu_bf16")
        return out
    if out_format != "nvfp4":
        raise ValueError("out_format must be 'bf16' or 'nvfp4'")
    packed = torch.empty(M, N // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(max(1, fp4_sf_size_bytes(M, N, FP4_NVFP4, FP4_SF_SWIZZLED)), dtype=torch.uint8,
                     device=dev)
    st = fp4_gemm_nvfp4_gelu_nvfp4(a_packed.data_ptr(), b_packed.data_ptr(), sfa.data_ptr(),
                                   sfb.data_ptr(), float(alpha), bp, M, N, K, packed.data_ptr(),
                                   sf.data_ptr(), int(variant), _pdl_mode(pdl),
                                   _stream_handle(stream))
    if st != 0:
        raise Fp4Error(st, "fp4_gemm_nvfp4_gelu_nvfp4")
    return packed, sf
