"""Device-side fills for the seeded synthetic inputs of ``inputs.py``.

The multi-GB decode-step workloads are generated in place on the GPU by
libmbw_inputs.so, which evaluates the same counter-based generator as the
numpy code in ``inputs.py`` (so the oracle can regenerate any sampled row on
the host, bit for bit). No GEMV arithmetic lives here.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import inputs as gen

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libmbw_inputs.so")
_lock = threading.Lock()
_lib = None
_tables = {}


def _L():
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(_LIB_PATH):
                    raise RuntimeError(f"{_LIB_PATH} missing: run `python -m memory_bound_weight_gb300.build`")
                L = ctypes.CDLL(_LIB_PATH)
                P, I64, U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
                L.mbw_gen_bf16_table.argtypes = [P, I64, I64, U64, P, P]
                L.mbw_gen_bytes.argtypes = [P, I64, I64, U64, P]
                L.mbw_gen_f16_scales.argtypes = [P, I64, I64, U64, P]
                L.mbw_gen_i8_table.argtypes = [P, I64, I64, U64, P, P]
                L.mbw_gen_f32_uniform.argtypes = [P, I64, I64, U64, ctypes.c_float, ctypes.c_float, P]
                for f in (L.mbw_gen_bf16_table, L.mbw_gen_bytes, L.mbw_gen_f16_scales, L.mbw_gen_i8_table,
                          L.mbw_gen_f32_uniform):
                    f.restype = ctypes.c_int
                _lib = L
    return _lib


def _stream(dev):
    import torch

    return torch.cuda.current_stream(dev).cuda_stream


def _table(sigma, dev):
    import torch

    key = (float(sigma), str(dev))
    if key not in _tables:
        t = gen.normal_table(sigma).view("int16")
        _tables[key] = torch.from_numpy(t.copy()).to(dev)
    return _tables[key]


def _i8_table(sigma, dev):
    import torch

    key = ("i8", float(sigma), str(dev))
    if key not in _tables:
        _tables[key] = torch.from_numpy(gen.int8_table(sigma).copy()).to(dev)
    return _tables[key]


def _ok(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what}: CUDA error {rc}")


def bf16_normal_(t, seed: int, stream: int, sigma: float, start: int = 0):
    """Fill a contiguous bf16 CUDA tensor with elements start.. of the bf16 normal stream."""
    tab = _table(sigma, t.device)
    _ok(_L().mbw_gen_bf16_table(t.data_ptr(), t.numel(), start, gen.stream_key(seed, stream), tab.data_ptr(),
                                _stream(t.device)), "mbw_gen_bf16_table")
    return t


def bytes_(t, seed: int, stream: int, start: int = 0):
    _ok(_L().mbw_gen_bytes(t.data_ptr(), t.numel() * t.element_size(), start, gen.stream_key(seed, stream),
                           _stream(t.device)), "mbw_gen_bytes")
    return t


def f16_scales_(t, seed: int, stream: int, start: int = 0):
    _ok(_L().mbw_gen_f16_scales(t.data_ptr(), t.numel(), start, gen.stream_key(seed, stream), _stream(t.device)),
        "mbw_gen_f16_scales")
    return t


# ---------------------------------------------------------------- tensors ----
def bf16_weights(seed: int, mi: int, N: int, K: int, device="cuda"):
    import torch

    t = torch.empty((N, K), dtype=torch.bfloat16, device=device)
    return bf16_normal_(t, seed, gen.stream_id(mi, gen.KIND_W), gen.W_SIGMA)


def bf16_activations(seed: int, mi: int, M: int, K: int, device="cuda"):
    import torch

    t = torch.empty((M, K), dtype=torch.bfloat16, device=device)
    return bf16_normal_(t, seed, gen.stream_id(mi, gen.KIND_X), gen.X_SIGMA)


def int4_codes(seed: int, mi: int, N: int, K: int, device="cuda"):
    import torch

    t = torch.empty((N, K // 2), dtype=torch.uint8, device=device)
    return bytes_(t, seed, gen.stream_id(mi, gen.KIND_W))


def f16_group_scales(seed: int, mi: int, N: int, groups: int, device="cuda"):
    import torch

    t = torch.empty((N, groups), dtype=torch.float16, device=device)
    return f16_scales_(t, seed, gen.stream_id(mi, gen.KIND_SCALES))


def u4_zero_points(seed: int, mi: int, N: int, groups: int, device="cuda"):
    import torch

    if groups % 2:
        raise ValueError("device fill of zero points needs an even group count")
    t = torch.empty((N, groups // 2), dtype=torch.uint8, device=device)
    return bytes_(t, seed, gen.stream_id(mi, gen.KIND_ZEROS))


def int8_codes(seed: int, mi: int, N: int, K: int, device="cuda"):
    import torch

    t = torch.empty((N, K), dtype=torch.int8, device=device)
    tab = _i8_table(gen.I8_SIGMA, t.device)
    _ok(_L().mbw_gen_i8_table(t.data_ptr(), t.numel(), 0, gen.stream_key(seed, gen.stream_id(mi, gen.KIND_W)),
                              tab.data_ptr(), _stream(t.device)), "mbw_gen_i8_table")
    return t


def f32_row_scales(seed: int, mi: int, N: int, device="cuda"):
    import torch

    t = torch.empty((N,), dtype=torch.float32, device=device)
    _ok(_L().mbw_gen_f32_uniform(t.data_ptr(), N, 0, gen.stream_key(seed, gen.stream_id(mi, gen.KIND_SCALES)),
                                 float(gen.I8_SCALE_LO), float(gen.I8_SCALE_SPAN), _stream(t.device)),
        "mbw_gen_f32_uniform")
    return t
