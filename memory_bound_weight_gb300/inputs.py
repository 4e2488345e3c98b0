"""Seeded synthetic inputs shared by the GPU path's tests/bench and the oracle.

This module holds no GEMV arithmetic. It only turns (seed, stream, index) into
bits, so that the CUDA kernels and the fp64 CPU oracle see bit-identical
inputs. The pages measure on trained checkpoints (Qwen2.5-7B, TinyLlama-1.1B);
none is available here, so these tensors stand in for their shapes and value
ranges only.

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the constants of Vigna's public splitmix64.c).
Element i of stream (seed, stream) is the (i+1)-th output of a splitmix64
sequence whose state starts at key(seed, stream). It is counter based, so any
element can be regenerated on its own (the oracle regenerates sampled rows of
the multi-GB workloads this way), and the device fill kernels in
``csrc/gen_inputs.cu`` evaluate the same function.

Value maps (one hash = 64 bits):
  * bf16 ~ N(0, sigma^2): 4 values per hash, 16 bits each (low half first),
    each an index into a 65,536-entry table of normal quantiles rounded to bf16
    (table entry j = bf16_rne(fp32(sigma * Phi^-1((j + 0.5) / 65536)))). Using a
    table keeps host and device free of transcendental-function mismatches.
  * packed uint4 codes / zero points: 8 bytes per hash, little-endian, each
    byte two independent uniform nibbles.
  * fp16 ~ U(0.001, 0.01): 1 value per hash from its top 24 bits u:
    fp16_rne(((fp32(u) * 2^-24) * 0.009f) + 0.001f), every fp32 step rounded
    separately (no fused multiply-add).
  * int8 codes in [-127, 127], shaped like a per-channel quantized Gaussian
    row: 4 values per hash, 16 bits each, each an index into a 65,536-entry
    table (entry j = clip(rint(32 * Phi^-1((j + 0.5) / 65536)), -127, 127)),
    so codes spread over about +-4 sigma and a few saturate at +-127.
  * fp32 ~ U(0.0002, 0.001) (per-channel INT8 scales, about max|w| / 127 for
    N(0, 0.02^2) rows): 1 value per hash, ((fp32(u) * 2^-24) * 0.0008f) +
    0.0002f, each fp32 step rounded separately.
"""
from __future__ import annotations

import functools

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor kinds; the stream id of tensor `kind` of matrix `mi` is mi * 16 + kind
KIND_W = 1
KIND_X = 2
KIND_SCALES = 3
KIND_ZEROS = 4

W_SIGMA = 0.02
X_SIGMA = 1.0
SCALE_LO = 0.001
SCALE_SPAN = 0.009
I8_SIGMA = 32.0
I8_SCALE_LO = np.float32(0.0002)
I8_SCALE_SPAN = np.float32(0.0008)


def stream_id(matrix_index: int, kind: int) -> int:
    return int(matrix_index) * 16 + int(kind)


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> int:
    """Starting state of a stream: mix64(seed * golden + stream * c) mod 2^64."""
    s = (int(seed) * int(GOLDEN) + int(stream) * int(_STREAM_MUL)) & 0xFFFFFFFFFFFFFFFF
    return int(_mix64(np.array([s], dtype=np.uint64))[0])


def hashes(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the stream, as uint64."""
    key = np.uint64(stream_key(seed, stream))
    i = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = key + (i + np.uint64(1)) * GOLDEN
    return _mix64(z)


def _f32_to_bf16_rne(f: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    nan = (b & 0x7FFFFFFF) > 0x7F800000
    r = ((b + (np.uint32(0x7FFF) + ((b >> 16) & 1))) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


@functools.lru_cache(maxsize=8)
def normal_table(sigma: float) -> np.ndarray:
    """65,536 bf16 bit patterns: quantiles (j+0.5)/65536 of N(0, sigma^2)."""
    from scipy.special import ndtri

    p = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    v = (sigma * ndtri(p)).astype(np.float32)
    t = _f32_to_bf16_rne(v)
    t.setflags(write=False)
    return t


@functools.lru_cache(maxsize=4)
def int8_table(sigma: float) -> np.ndarray:
    """65,536 int8 codes: quantiles (j+0.5)/65536 of N(0, sigma^2), rounded, clipped to +-127."""
    from scipy.special import ndtri

    p = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    t = np.clip(np.rint(sigma * ndtri(p)), -127, 127).astype(np.int8)
    t.setflags(write=False)
    return t


def _table_indices(seed: int, stream: int, n: int, start: int) -> np.ndarray:
    h0 = start // 4
    h1 = (start + n + 3) // 4
    h = hashes(seed, stream, h0, h1 - h0)
    idx = h.view(np.uint16).reshape(-1)  # little-endian: low 16 bits first
    off = start - 4 * h0
    return idx[off:off + n]


def int8_normal(seed: int, stream: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    """n int8 codes from the quantile table, elements start .. start+n-1."""
    if n == 0:
        return np.zeros(0, dtype=np.int8)
    return int8_table(sigma)[_table_indices(seed, stream, n, start)]


def f32_uniform(seed: int, stream: int, n: int, lo: np.float32, span: np.float32, start: int = 0) -> np.ndarray:
    """n fp32 ~ U(lo, lo + span): ((fp32(u) * 2^-24) * span) + lo, u = top 24 bits of a hash."""
    if n == 0:
        return np.zeros(0, dtype=np.float32)
    u = (hashes(seed, stream, start, n) >> np.uint64(40)).astype(np.float32)
    s = u * np.float32(2.0 ** -24)
    s = s * np.float32(span)
    return s + np.float32(lo)


def bf16_normal(seed: int, stream: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    """n bf16 bit patterns (uint16) ~ N(0, sigma^2), elements start .. start+n-1."""
    if n == 0:
        return np.zeros(0, dtype=np.uint16)
    return normal_table(sigma)[_table_indices(seed, stream, n, start)]


def random_bytes(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n uniform bytes (uint8), bytes start .. start+n-1 of the stream."""
    if n == 0:
        return np.zeros(0, dtype=np.uint8)
    h0 = start // 8
    h1 = (start + n + 7) // 8
    b = hashes(seed, stream, h0, h1 - h0).view(np.uint8)
    off = start - 8 * h0
    return b[off:off + n].copy()


def f16_uniform_scales(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n fp16 bit patterns (uint16) ~ U(0.001, 0.01)."""
    if n == 0:
        return np.zeros(0, dtype=np.uint16)
    u = (hashes(seed, stream, start, n) >> np.uint64(40)).astype(np.float32)
    s = u * np.float32(2.0 ** -24)
    s = s * np.float32(SCALE_SPAN)
    s = s + np.float32(SCALE_LO)
    return s.astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------- tensors ----
def bf16_weights(seed: int, mi: int, N: int, K: int, row0: int = 0, rows: int | None = None) -> np.ndarray:
    """BF16 weight rows [row0, row0+rows) of matrix mi, shape (rows, K), uint16."""
    rows = N - row0 if rows is None else rows
    return bf16_normal(seed, stream_id(mi, KIND_W), rows * K, W_SIGMA, start=row0 * K).reshape(rows, K)


def bf16_activations(seed: int, mi: int, M: int, K: int) -> np.ndarray:
    """x (M=1) or X (M, K) ~ N(0, 1), uint16 bf16 bits."""
    return bf16_normal(seed, stream_id(mi, KIND_X), M * K, X_SIGMA).reshape(M, K)


def int4_codes(seed: int, mi: int, N: int, K: int, row0: int = 0, rows: int | None = None) -> np.ndarray:
    """Packed uint4 codes, shape (rows, K//2) uint8; low nibble = even k."""
    rows = N - row0 if rows is None else rows
    rb = K // 2
    return random_bytes(seed, stream_id(mi, KIND_W), rows * rb, start=row0 * rb).reshape(rows, rb)


def f16_group_scales(seed: int, mi: int, N: int, groups: int, row0: int = 0, rows: int | None = None) -> np.ndarray:
    """fp16 scales, shape (rows, groups) uint16."""
    rows = N - row0 if rows is None else rows
    return f16_uniform_scales(seed, stream_id(mi, KIND_SCALES), rows * groups, start=row0 * groups).reshape(rows, groups)


def u4_zero_points(seed: int, mi: int, N: int, groups: int, row0: int = 0, rows: int | None = None) -> np.ndarray:
    """Packed uint4 zero points, shape (rows, ceil(groups/2)) uint8; low nibble = even group."""
    rows = N - row0 if rows is None else rows
    zb = (groups + 1) // 2
    z = random_bytes(seed, stream_id(mi, KIND_ZEROS), rows * zb, start=row0 * zb).reshape(rows, zb)
    if groups % 2:  # the unused high nibble of the last byte is kept zero
        z[:, -1] &= 0x0F
    return z


def int8_codes(seed: int, mi: int, N: int, K: int, row0: int = 0, rows: int | None = None) -> np.ndarray:
    """Symmetric INT8 codes, shape (rows, K) int8, values in [-127, 127]."""
    rows = N - row0 if rows is None else rows
    return int8_normal(seed, stream_id(mi, KIND_W), rows * K, I8_SIGMA, start=row0 * K).reshape(rows, K)


def f32_row_scales(seed: int, mi: int, N: int, row0: int = 0, rows: int | None = None) -> np.ndarray:
    """Per-output-channel fp32 scales, shape (rows,)."""
    rows = N - row0 if rows is None else rows
    return f32_uniform(seed, stream_id(mi, KIND_SCALES), rows, I8_SCALE_LO, I8_SCALE_SPAN, start=row0)
