"""Thin ctypes binding of libmbw.so (include/mbw.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libmbw.so. PyTorch supplies device memory and the current stream.
If the library is missing the calls raise; there is no fallback path.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmbw.so")

MBW_OK = 0
OP_GEMV_BF16 = 1
OP_GEMV_INT4_G64 = 2
OP_GEMV_INT4_AWQ_G128 = 3
OP_GEMM_SKINNY_BF16 = 4
OP_GEMV_INT8_PC = 5
FUSE_NORM = 0x100
FUSE_GLU = 0x200
FUSE_RESIDUAL = 0x400
REPACKED = 0x800

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_ST = ctypes.c_int

_lock = threading.Lock()
_lib = None


class MbwFusion(ctypes.Structure):
    """struct mbw_fusion of include/mbw.h."""
    _fields_ = [("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float), ("residual", ctypes.c_void_p),
                ("up_weights", ctypes.c_void_p), ("up_scales", ctypes.c_void_p), ("up_zeros", ctypes.c_void_p)]

# name -> (argtypes, restype)
SIGNATURES = {
    "gemv_bf16": ([_P, _P, _P, _I64, _I64, _P, _SZ, _P], _ST),
    "gemv_int4_g64": ([_P, _P, _P, _P, _I64, _I64, _P, _SZ, _P], _ST),
    "gemv_int4_awq_g128": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _ST),
    "gemv_int4_awq_g128_repacked": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _ST),
    "mbw_repack_int4": ([_P, _P, _I64, _I64, _P], _ST),
    "gemm_skinny_bf16": ([_P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _ST),
    "gemv_int8_pc": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _ST),
    "mbw_quantize_int8_pc": ([_P, _P, _P, _I64, _I64, _P], _ST),
    "gemv_fused": ([ctypes.c_int, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.POINTER(MbwFusion), _P, _SZ, _P], _ST),
    "gemv_fused_awq_g128": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(MbwFusion), _P, _SZ,
                             _P], _ST),
    "mbw_workspace_bytes": ([ctypes.c_int, _I64, _I64, _I64], _SZ),
    "mbw_dequant_int4_g64": ([_P, _P, _P, _I64, _I64, _P], _ST),
    "mbw_dequant_int4_awq_g128": ([_P, _P, _P, _P, _I64, _I64, _P], _ST),
    "mbw_set_output_fp32": ([ctypes.c_int], _ST),
    "mbw_autotune": ([ctypes.c_int, _I64, _I64, _I64, _P], _ST),
    "mbw_plan_candidates": ([ctypes.c_int, _I64, _I64, _I64], ctypes.c_int),
    "mbw_plan_select": ([ctypes.c_int, _I64, _I64, _I64, ctypes.c_int], _ST),
    "mbw_plan_index": ([ctypes.c_int, _I64, _I64, _I64], ctypes.c_int),
    "mbw_plan_describe": ([ctypes.c_int, _I64, _I64, _I64, ctypes.c_char_p, _SZ], _ST),
    "mbw_check_device_error": ([], _ST),
    "mbw_selftest_wait_expiry": ([_I64, _P], _ST),
    "mbw_inject_launch_failures": ([ctypes.c_int], _ST),
    "mbw_launch_count": ([], ctypes.c_uint64),
    "mbw_status_string": ([_ST], ctypes.c_char_p),
    "mbw_last_error": ([], ctypes.c_char_p),
}


class MbwError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn} failed: status {status} ({detail})")
        self.status = status
        self.detail = detail


def lib() -> ctypes.CDLL:
    """The loaded libmbw.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                       "`python -m memory_bound_weight_gb300.build`")
                L = ctypes.CDLL(LIB_PATH)
                for name, (args, res) in SIGNATURES.items():
                    f = getattr(L, name)
                    f.argtypes = args
                    f.restype = res
                _lib = L
    return _lib


def check(fn: str, status: int) -> None:
    if status != MBW_OK:
        L = lib()
        name = L.mbw_status_string(status).decode()
        detail = L.mbw_last_error().decode()
        raise MbwError(fn, status, f"{name}: {detail}")


def _torch():
    import torch

    return torch


def _stream_ptr(device) -> int:
    torch = _torch()
    return torch.cuda.current_stream(device).cuda_stream


def _need(t, name, dtype, ndim):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _common_device(*ts):
    """The one device all given tensors (None skipped) are on."""
    devs = {t.device for t in ts if t is not None}
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one device, got {sorted(str(d) for d in devs)}")
    return devs.pop()


def _on_current_device(*ts):
    """All tensors on one CUDA device, the current one: the library plans and
    launches on the current device, and a kernel given another device's memory
    would fault."""
    torch = _torch()
    d = _common_device(*ts)
    cur = torch.cuda.current_device()
    if d.index != cur:
        raise ValueError(f"tensors are on {d} but the current CUDA device is cuda:{cur} (torch.cuda.set_device)")
    return d


def _need_shape(t, name, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


_tls = threading.local()


def _out_dtype():
    torch = _torch()
    return torch.float32 if getattr(_tls, "fp32", False) else torch.bfloat16


@contextlib.contextmanager
def output_fp32():
    """Within this block, calls on this thread write the fp32 accumulator (test hook)."""
    check("mbw_set_output_fp32", lib().mbw_set_output_fp32(1))
    _tls.fp32 = True
    try:
        yield
    finally:
        lib().mbw_set_output_fp32(0)
        _tls.fp32 = False


def _alloc_out(shape, like, out):
    torch = _torch()
    dt = _out_dtype()
    if out is None:
        return torch.empty(shape, dtype=dt, device=like.device)
    _need(out, "out", dt, len(shape))
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out must have shape {tuple(shape)}")
    return out


def _ws(workspace):
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


# ----------------------------------------------------------------- calls ----
def gemv_bf16(W, x, out=None, workspace=None):
    """y = W . x; W bf16 (N, K), x bf16 (K,) -> y (N,)."""
    torch = _torch()
    _need(W, "W", torch.bfloat16, 2)
    _need(x, "x", torch.bfloat16, 1)
    N, K = W.shape
    if x.shape[0] != K:
        raise ValueError("x must have length K")
    y = _alloc_out((N,), W, out)
    _on_current_device(W, x, y, workspace)
    wp, wn = _ws(workspace)
    check("gemv_bf16", lib().gemv_bf16(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, wp, wn,
                                       _stream_ptr(W.device)))
    return y


def gemv_int4_g64(Wq, scales, x, out=None, workspace=None):
    """y = W . x; Wq uint8 (N, K/2), scales fp16 (N, K/64), x bf16 (K,) -> y (N,)."""
    torch = _torch()
    _need(Wq, "Wq", torch.uint8, 2)
    _need(scales, "scales", torch.float16, 2)
    _need(x, "x", torch.bfloat16, 1)
    N = Wq.shape[0]
    K = x.shape[0]
    if Wq.shape[1] * 2 != K or tuple(scales.shape) != (N, K // 64):
        raise ValueError("shapes: Wq (N, K/2), scales (N, K/64), x (K,)")
    y = _alloc_out((N,), Wq, out)
    _on_current_device(Wq, scales, x, y, workspace)
    wp, wn = _ws(workspace)
    check("gemv_int4_g64", lib().gemv_int4_g64(Wq.data_ptr(), scales.data_ptr(), x.data_ptr(), y.data_ptr(),
                                               N, K, wp, wn, _stream_ptr(Wq.device)))
    return y


def gemv_int4_awq_g128(Wq, scales, zeros, X, out=None, workspace=None, repacked=False):
    """Y = X . W^T; Wq uint8 (N, K/2), scales fp16 (N, G), zeros uint8 (N, ceil(G/2)),
    X bf16 (M, K) or (K,) -> Y (M, N) or (N,). `repacked`: Wq is in the layout of
    repack_int4 (calls gemv_int4_awq_g128_repacked)."""
    torch = _torch()
    vec = X.dim() == 1
    X2 = X.unsqueeze(0) if vec else X
    _need(Wq, "Wq", torch.uint8, 2)
    _need(scales, "scales", torch.float16, 2)
    _need(zeros, "zeros", torch.uint8, 2)
    _need(X2, "X", torch.bfloat16, 2)
    M, K = X2.shape
    N = Wq.shape[0]
    G = K // 128
    if Wq.shape[1] * 2 != K or tuple(scales.shape) != (N, G) or tuple(zeros.shape) != (N, (G + 1) // 2):
        raise ValueError("shapes: Wq (N, K/2), scales (N, K/128), zeros (N, ceil(K/256)), X (M, K)")
    Y = _alloc_out((M, N), Wq, None if out is None else (out.unsqueeze(0) if vec else out))
    _on_current_device(Wq, scales, zeros, X2, Y, workspace)
    wp, wn = _ws(workspace)
    name = "gemv_int4_awq_g128_repacked" if repacked else "gemv_int4_awq_g128"
    check(name, getattr(lib(), name)(
        Wq.data_ptr(), scales.data_ptr(), zeros.data_ptr(), X2.data_ptr(), Y.data_ptr(), M, N, K, wp, wn,
        _stream_ptr(Wq.device)))
    return Y[0] if vec else Y


def repack_int4(Wq, out=None):
    """Canonical INT4 codes uint8 (N, K/2) -> the load-time repacked layout (a new
    tensor, or `out`, which may be Wq itself)."""
    torch = _torch()
    _need(Wq, "Wq", torch.uint8, 2)
    N, half = Wq.shape
    Wr = torch.empty_like(Wq) if out is None else out
    if Wr.shape != Wq.shape or Wr.dtype != torch.uint8 or not Wr.is_contiguous():
        raise ValueError("out must be a contiguous uint8 tensor of Wq's shape")
    _on_current_device(Wq, Wr)
    check("mbw_repack_int4", lib().mbw_repack_int4(Wq.data_ptr(), Wr.data_ptr(), N, 2 * half, _stream_ptr(Wq.device)))
    return Wr


def gemm_skinny_bf16(X, W, out=None, workspace=None):
    """Y = X . W^T; X bf16 (M, K), W bf16 (N, K) -> Y (M, N)."""
    torch = _torch()
    _need(X, "X", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("W must be (N, K)")
    Y = _alloc_out((M, N), W, out)
    _on_current_device(X, W, Y, workspace)
    wp, wn = _ws(workspace)
    check("gemm_skinny_bf16", lib().gemm_skinny_bf16(X.data_ptr(), W.data_ptr(), Y.data_ptr(), M, N, K, wp, wn,
                                                     _stream_ptr(W.device)))
    return Y


def gemv_int8_pc(Wq, scales, X, out=None, workspace=None):
    """Y = X . W^T; Wq int8 (N, K), scales fp32 (N,), X bf16 (M, K) or (K,) -> Y (M, N) or (N,)."""
    torch = _torch()
    vec = X.dim() == 1
    X2 = X.unsqueeze(0) if vec else X
    _need(Wq, "Wq", torch.int8, 2)
    _need(scales, "scales", torch.float32, 1)
    _need(X2, "X", torch.bfloat16, 2)
    M, K = X2.shape
    N = Wq.shape[0]
    if Wq.shape[1] != K or scales.shape[0] != N:
        raise ValueError("shapes: Wq (N, K), scales (N,), X (M, K)")
    Y = _alloc_out((M, N), Wq, None if out is None else (out.unsqueeze(0) if vec else out))
    _on_current_device(Wq, scales, X2, Y, workspace)
    wp, wn = _ws(workspace)
    check("gemv_int8_pc", lib().gemv_int8_pc(Wq.data_ptr(), scales.data_ptr(), X2.data_ptr(), Y.data_ptr(), M, N, K,
                                             wp, wn, _stream_ptr(Wq.device)))
    return Y[0] if vec else Y


def gemv_fused(op, W, scales, X, out=None, norm_weight=None, norm_eps=1e-6, residual=None, up_weights=None,
               up_scales=None, workspace=None):
    """One GEMV of format `op` (OP_GEMV_BF16 / _INT4_G64 / _INT8_PC) with optional fusions:
    RMSNorm prologue (norm_weight bf16 (K,)), gated SiLU epilogue (up_weights / up_scales, same
    layout as W / scales), residual add (residual bf16 shaped like the output; may be `out`).
    X bf16 (M, K) or (K,) -> Y (M, N) or (N,)."""
    torch = _torch()
    vec = X.dim() == 1
    X2 = X.unsqueeze(0) if vec else X
    _need(X2, "X", torch.bfloat16, 2)
    M, K = X2.shape
    N = W.shape[0]
    wdt, sdt, kdiv = {OP_GEMV_BF16: (torch.bfloat16, None, 1), OP_GEMV_INT4_G64: (torch.uint8, torch.float16, 2),
                      OP_GEMV_INT8_PC: (torch.int8, torch.float32, 1)}[op]
    _need(W, "W", wdt, 2)
    if W.shape[1] * kdiv != K:
        raise ValueError("W does not match K")
    sshape = None if sdt is None else ((N, K // 64) if op == OP_GEMV_INT4_G64 else (N,))
    if sdt is not None:
        _need(scales, "scales", sdt, len(sshape))
        _need_shape(scales, "scales", sshape)
    f = MbwFusion()
    if norm_weight is not None:
        _need(norm_weight, "norm_weight", torch.bfloat16, 1)
        if norm_weight.shape[0] != K:
            raise ValueError("norm_weight must have length K")
        f.norm_weight = norm_weight.data_ptr()
        f.norm_eps = float(norm_eps)
    if up_weights is not None:
        _need(up_weights, "up_weights", wdt, 2)
        if tuple(up_weights.shape) != tuple(W.shape):
            raise ValueError("up_weights must have W's shape")
        f.up_weights = up_weights.data_ptr()
        if sdt is not None:
            _need(up_scales, "up_scales", sdt, len(sshape))
            _need_shape(up_scales, "up_scales", sshape)
            f.up_scales = up_scales.data_ptr()
    Y = _alloc_out((M, N), X2, None if out is None else (out.unsqueeze(0) if vec else out))
    if residual is not None:
        r2 = residual.unsqueeze(0) if residual.dim() == 1 else residual
        _need(r2, "residual", torch.bfloat16, 2)
        if tuple(r2.shape) != (M, N):
            raise ValueError("residual must be shaped like the output")
        f.residual = r2.data_ptr()
    _on_current_device(W, scales if sdt is not None else None, X2, Y, norm_weight, residual, up_weights,
                       up_scales if (up_weights is not None and sdt is not None) else None, workspace)
    wp, wn = _ws(workspace)
    check("gemv_fused", lib().gemv_fused(op, W.data_ptr(), None if scales is None else scales.data_ptr(),
                                         X2.data_ptr(), Y.data_ptr(), M, N, K, ctypes.byref(f), wp, wn,
                                         _stream_ptr(X2.device)))
    return Y[0] if vec else Y


def gemv_fused_awq_g128(Wq, scales, zeros, X, out=None, norm_weight=None, norm_eps=1e-6, residual=None,
                        up_weights=None, up_scales=None, up_zeros=None, repacked=False, workspace=None):
    """gemv_int4_awq_g128 (Wq uint8 (N, K/2), scales fp16 (N, K/128), zeros uint8 (N, (K/128+1)/2); codes
    canonical or, with repacked=True, from repack_int4) with optional fusions: RMSNorm prologue
    (norm_weight bf16 (K,)), gated SiLU epilogue (up_weights / up_scales / up_zeros, same layouts),
    residual add (bf16 shaped like the output; may be `out`). X bf16 (M, K) or (K,) -> Y (M, N) or (N,)."""
    torch = _torch()
    vec = X.dim() == 1
    X2 = X.unsqueeze(0) if vec else X
    _need(X2, "X", torch.bfloat16, 2)
    M, K = X2.shape
    _need(Wq, "Wq", torch.uint8, 2)
    N = Wq.shape[0]
    if Wq.shape[1] * 2 != K:
        raise ValueError("Wq does not match K")
    G = K // 128
    _need(scales, "scales", torch.float16, 2)
    _need_shape(scales, "scales", (N, G))
    _need(zeros, "zeros", torch.uint8, 2)
    _need_shape(zeros, "zeros", (N, (G + 1) // 2))
    f = MbwFusion()
    if norm_weight is not None:
        _need(norm_weight, "norm_weight", torch.bfloat16, 1)
        if norm_weight.shape[0] != K:
            raise ValueError("norm_weight must have length K")
        f.norm_weight = norm_weight.data_ptr()
        f.norm_eps = float(norm_eps)
    if up_weights is not None:
        _need(up_weights, "up_weights", torch.uint8, 2)
        if tuple(up_weights.shape) != tuple(Wq.shape):
            raise ValueError("up_weights must have Wq's shape")
        _need(up_scales, "up_scales", torch.float16, 2)
        _need_shape(up_scales, "up_scales", (N, G))
        _need(up_zeros, "up_zeros", torch.uint8, 2)
        _need_shape(up_zeros, "up_zeros", (N, (G + 1) // 2))
        f.up_weights, f.up_scales, f.up_zeros = up_weights.data_ptr(), up_scales.data_ptr(), up_zeros.data_ptr()
    Y = _alloc_out((M, N), X2, None if out is None else (out.unsqueeze(0) if vec else out))
    if residual is not None:
        r2 = residual.unsqueeze(0) if residual.dim() == 1 else residual
        _need(r2, "residual", torch.bfloat16, 2)
        if tuple(r2.shape) != (M, N):
            raise ValueError("residual must be shaped like the output")
        f.residual = r2.data_ptr()
    _on_current_device(Wq, scales, zeros, X2, Y, norm_weight, residual, up_weights, up_scales, up_zeros, workspace)
    wp, wn = _ws(workspace)
    check("gemv_fused_awq_g128", lib().gemv_fused_awq_g128(Wq.data_ptr(), scales.data_ptr(), zeros.data_ptr(),
                                                           X2.data_ptr(), Y.data_ptr(), M, N, K, int(bool(repacked)),
                                                           ctypes.byref(f), wp, wn, _stream_ptr(X2.device)))
    return Y[0] if vec else Y


def quantize_int8_pc(W):
    """BF16 W (N, K) -> (Wq int8 (N, K), scales fp32 (N,)), scale = max|w| / 127 per row."""
    torch = _torch()
    _need(W, "W", torch.bfloat16, 2)
    N, K = W.shape
    _on_current_device(W)
    Wq = torch.empty((N, K), dtype=torch.int8, device=W.device)
    sc = torch.empty((N,), dtype=torch.float32, device=W.device)
    check("mbw_quantize_int8_pc", lib().mbw_quantize_int8_pc(W.data_ptr(), Wq.data_ptr(), sc.data_ptr(), N, K,
                                                             _stream_ptr(W.device)))
    return Wq, sc


def dequant_int4_g64(Wq, scales):
    torch = _torch()
    _need(Wq, "Wq", torch.uint8, 2)
    _need(scales, "scales", torch.float16, 2)
    N, K = Wq.shape[0], Wq.shape[1] * 2
    _need_shape(scales, "scales", (N, K // 64))
    _on_current_device(Wq, scales)
    out = torch.empty((N, K), dtype=torch.float32, device=Wq.device)
    check("mbw_dequant_int4_g64", lib().mbw_dequant_int4_g64(Wq.data_ptr(), scales.data_ptr(), out.data_ptr(),
                                                             N, K, _stream_ptr(Wq.device)))
    return out


def dequant_int4_awq_g128(Wq, scales, zeros):
    torch = _torch()
    _need(Wq, "Wq", torch.uint8, 2)
    _need(scales, "scales", torch.float16, 2)
    _need(zeros, "zeros", torch.uint8, 2)
    N, K = Wq.shape[0], Wq.shape[1] * 2
    G = K // 128
    _need_shape(scales, "scales", (N, G))
    _need_shape(zeros, "zeros", (N, (G + 1) // 2))
    _on_current_device(Wq, scales, zeros)
    out = torch.empty((N, K), dtype=torch.float32, device=Wq.device)
    check("mbw_dequant_int4_awq_g128", lib().mbw_dequant_int4_awq_g128(
        Wq.data_ptr(), scales.data_ptr(), zeros.data_ptr(), out.data_ptr(), N, K, _stream_ptr(Wq.device)))
    return out


def autotune(op: int, M: int, N: int, K: int) -> None:
    torch = _torch()
    check("mbw_autotune", lib().mbw_autotune(op, M, N, K, torch.cuda.current_stream().cuda_stream))


def plan_describe(op: int, M: int, N: int, K: int) -> str:
    buf = ctypes.create_string_buffer(256)
    check("mbw_plan_describe", lib().mbw_plan_describe(op, M, N, K, buf, 256))
    return buf.value.decode()


def plan_candidates(op: int, M: int, N: int, K: int) -> int:
    return int(lib().mbw_plan_candidates(op, M, N, K))


def plan_select(op: int, M: int, N: int, K: int, index: int) -> None:
    check("mbw_plan_select", lib().mbw_plan_select(op, M, N, K, index))


def plan_index(op: int, M: int, N: int, K: int) -> int:
    return int(lib().mbw_plan_index(op, M, N, K))


def workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return int(lib().mbw_workspace_bytes(op, M, N, K))


def launch_count() -> int:
    return int(lib().mbw_launch_count())


def check_device_error() -> None:
    check("mbw_check_device_error", lib().mbw_check_device_error())


def inject_launch_failures(count: int) -> None:
    """The next `count` launching calls on this thread raise MbwError with
    MBW_ERR_CUDA and launch nothing (host-side fault injection; 0 turns it off)."""
    check("mbw_inject_launch_failures", lib().mbw_inject_launch_failures(int(count)))


def selftest_wait_expiry(tries: int) -> None:
    """Launch, on the current stream, the two one-thread kernels whose bounded
    waits expire after `tries` rounds; the next check_device_error() raises
    MbwError with MBW_ERR_DEVICE_TIMEOUT."""
    check("mbw_selftest_wait_expiry", lib().mbw_selftest_wait_expiry(int(tries), _stream_ptr(None)))
