"""Matrix shapes of the decode workloads and their algorithmic byte counts.

Byte accounting follows the pages' ceiling arithmetic: a decode step reads
every weight matrix once, so tokens/s <= bandwidth / bytes of weights per
token (tinyinfer, "How I Built an LLM Inference Engine From Scratch in CUDA",
TL;DR; llm-rs vs vLLM, sec. 2). Only the matrices streamed by the GEMVs are
counted (the embedding table is gathered one row per token).

Per GEMV the algorithmic bytes are weights + group scales (+ zero points)
+ the activation vector(s) x; the output y is reported alongside.
"""
from __future__ import annotations

from dataclasses import dataclass

FMT_BF16 = "bf16"
FMT_INT4_G64 = "int4_g64"
FMT_INT4_AWQ_G128 = "int4_awq_g128"
FMT_INT8_PC = "int8_pc"

# Fusion bits of a call (the MBW_FUSE_* values of include/mbw.h).
FUSE_NORM = 0x100      # RMSNorm prologue: reads a bf16 [K] norm weight
FUSE_GLU = 0x200       # gated SiLU epilogue: streams a second (up) matrix of the same shape
FUSE_RESIDUAL = 0x400  # residual add: reads a bf16 [M][N] residual


@dataclass(frozen=True)
class Mat:
    name: str
    N: int  # output rows
    K: int  # reduction length
    fuse: int = 0  # FUSE_* bits of the call that streams it


def bits_per_weight(code_bits: int, group: int, scale_bits: int, zero_bits: int) -> float:
    """Storage bits per weight of a grouped format: code + (scale + zero) / group."""
    return code_bits + (scale_bits + zero_bits) / group


def weight_bytes(fmt: str, N: int, K: int) -> int:
    """Bytes of one stored weight matrix in the layout the library takes."""
    if fmt == FMT_BF16:
        return 2 * N * K
    if fmt == FMT_INT4_G64:
        return N * K // 2 + 2 * N * (K // 64)
    if fmt == FMT_INT4_AWQ_G128:
        G = K // 128
        return N * K // 2 + 2 * N * G + N * ((G + 1) // 2)
    if fmt == FMT_INT8_PC:
        return N * K + 4 * N
    raise ValueError(fmt)


def bytes_alg(fmt: str, M: int, N: int, K: int) -> int:
    """Algorithmic bytes of one call: weights (+ scales, zeros) + M activation rows (bf16)."""
    return weight_bytes(fmt, N, K) + 2 * M * K


def call_weight_bytes(fmt: str, m: Mat) -> int:
    """Weight bytes one call streams (both matrices of a gated call)."""
    return weight_bytes(fmt, m.N, m.K) * (2 if m.fuse & FUSE_GLU else 1)


def call_bytes(fmt: str, M: int, m: Mat) -> int:
    """Algorithmic bytes of one call with its fusions: weights, x, and the
    norm weight and residual it reads."""
    b = call_weight_bytes(fmt, m) + 2 * M * m.K
    if m.fuse & FUSE_NORM:
        b += 2 * m.K
    if m.fuse & FUSE_RESIDUAL:
        b += 2 * M * m.N
    return b


def call_flops(M: int, m: Mat) -> int:
    return flops(M, m.N, m.K) * (2 if m.fuse & FUSE_GLU else 1)


def out_bytes(M: int, N: int) -> int:
    return 2 * M * N


def flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


# ---------------------------------------------------------------- models ----
# TinyLlama-1.1B: hidden 2048, MLP 5632, 22 layers, 32 query heads, 4 KV heads
# of 64 dims, vocabulary 32000 (the model of tinyinfer's measurements).
TINYLLAMA_LAYER = (
    Mat("q", 2048, 2048), Mat("k", 256, 2048), Mat("v", 256, 2048), Mat("o", 2048, 2048),
    Mat("gate", 5632, 2048), Mat("up", 5632, 2048), Mat("down", 2048, 5632),
)
TINYLLAMA_LAYERS = 22
TINYLLAMA_HEAD = Mat("lm_head", 32000, 2048)
# The same layer with the projections that share an input concatenated along
# the output rows, as an engine launches them (tinyinfer, "fused
# projections"): [Wq; Wk; Wv] and [Wgate; Wup] each become one GEMV. The
# bytes streamed are unchanged; the dependent launches per layer drop from 7 to 4.
TINYLLAMA_LAYER_FUSED = (
    Mat("qkv", 2048 + 256 + 256, 2048), Mat("o", 2048, 2048), Mat("gate_up", 2 * 5632, 2048),
    Mat("down", 2048, 5632),
)

# The fused-projection layer with the small ops of the layer folded into its
# GEMVs (NEXT-1, NEXT-4): the attention RMSNorm into q/k/v, the residual adds
# into o and down, and the MLP RMSNorm plus SwiGLU into the gate/up call, which
# streams gate and up (5632 rows each) and writes silu(gate) * up. The head
# takes the final RMSNorm. Same weights and launches as the fused layer.
TINYLLAMA_LAYER_FUSEDOPS = (
    Mat("qkv", 2048 + 256 + 256, 2048, FUSE_NORM), Mat("o", 2048, 2048, FUSE_RESIDUAL),
    Mat("gate_up", 5632, 2048, FUSE_NORM | FUSE_GLU), Mat("down", 2048, 5632, FUSE_RESIDUAL),
)
TINYLLAMA_HEAD_NORM = Mat("lm_head", 32000, 2048, FUSE_NORM)

# Qwen2.5-7B: hidden 3584, MLP 18944, 28 layers, 28 query heads and 4 KV heads
# of 128 dims (Q, K, V concatenated to 4608 rows), vocabulary 152064
# (the model of llm-rs's single-stream measurements).
QWEN25_7B_LAYER = (
    Mat("qkv", 4608, 3584), Mat("o", 3584, 3584), Mat("gate", 18944, 3584),
    Mat("up", 18944, 3584), Mat("down", 3584, 18944),
)
QWEN25_7B_LAYERS = 28
QWEN25_7B_HEAD = Mat("lm_head", 152064, 3584)
# The same layer with gate and up, which read the same x, stored as one
# [Wgate; Wup] matrix of 37888 rows and streamed by one GEMV (tinyinfer's
# fused projections): the same weights in 113 calls instead of 141.
QWEN25_7B_LAYER_FUSED = (
    Mat("qkv", 4608, 3584), Mat("o", 3584, 3584), Mat("gate_up", 2 * 18944, 3584), Mat("down", 3584, 18944),
)
# The same layer with the small ops folded into its GEMVs (NEXT-1, NEXT-4 on
# the AWQ path): the attention RMSNorm into q/k/v, the residual adds into o and
# down, the MLP RMSNorm and SwiGLU into one gate/up call (gate and up streamed
# together, 18944 output rows); the head takes the final RMSNorm.
QWEN25_7B_LAYER_FUSEDOPS = (
    Mat("qkv", 4608, 3584, FUSE_NORM), Mat("o", 3584, 3584, FUSE_RESIDUAL),
    Mat("gate_up", 18944, 3584, FUSE_NORM | FUSE_GLU), Mat("down", 3584, 18944, FUSE_RESIDUAL),
)
QWEN25_7B_HEAD_NORM = Mat("lm_head", 152064, 3584, FUSE_NORM)

# Qwen3-4B: hidden 2560, MLP 9728, 36 layers, 32 query heads and 8 KV heads
# of 128 dims, vocabulary 151936 (the model of TileInfer's INT8 measurements:
# every linear layer and the lm_head in INT8, about 4 GB per token). The
# projections that share an input are concatenated: [Wq; Wk; Wv] = 6144 rows,
# [Wgate; Wup] = 19456 rows.
QWEN3_4B_LAYER_FUSED = (
    Mat("qkv", 4096 + 1024 + 1024, 2560), Mat("o", 2560, 4096), Mat("gate_up", 2 * 9728, 2560),
    Mat("down", 2560, 9728),
)
QWEN3_4B_LAYERS = 36
QWEN3_4B_HEAD = Mat("lm_head", 151936, 2560)

# The four TinyLlama-shaped INT4 matrices of tinyinfer's per-matrix bandwidth table.
TINYLLAMA_TABLE_SHAPES = (
    Mat("q/o", 2048, 2048), Mat("gate/up", 5632, 2048), Mat("down", 2048, 5632),
    Mat("lm_head", 32000, 2048),
)

SKINNY_M = (1, 8, 16, 32, 64, 128, 256)
SKINNY_SHAPES = (Mat("gate/up", 18944, 3584), Mat("down", 3584, 18944))
AWQ_M = (1, 16, 64)


def decode_step(layer, layers: int, head: Mat) -> list[Mat]:
    """Every matrix one decode token streams, in execution order."""
    mats = []
    for li in range(layers):
        for m in layer:
            mats.append(Mat(f"L{li}.{m.name}", m.N, m.K, m.fuse))
    mats.append(head)
    return mats


def tinyllama_step(fused: bool = False, fusedops: bool = False) -> list[Mat]:
    if fusedops:
        return decode_step(TINYLLAMA_LAYER_FUSEDOPS, TINYLLAMA_LAYERS, TINYLLAMA_HEAD_NORM)
    layer = TINYLLAMA_LAYER_FUSED if fused else TINYLLAMA_LAYER
    return decode_step(layer, TINYLLAMA_LAYERS, TINYLLAMA_HEAD)


def qwen25_7b_step(fusedops: bool = False, fused: bool = False) -> list[Mat]:
    if fusedops:
        return decode_step(QWEN25_7B_LAYER_FUSEDOPS, QWEN25_7B_LAYERS, QWEN25_7B_HEAD_NORM)
    return decode_step(QWEN25_7B_LAYER_FUSED if fused else QWEN25_7B_LAYER, QWEN25_7B_LAYERS, QWEN25_7B_HEAD)


def qwen3_4b_step() -> list[Mat]:
    return decode_step(QWEN3_4B_LAYER_FUSED, QWEN3_4B_LAYERS, QWEN3_4B_HEAD)


def step_weight_bytes(mats, fmt: str, head_fmt: str | None = None) -> int:
    total = 0
    for m in mats:
        f = head_fmt if (head_fmt is not None and m.name == "lm_head") else fmt
        total += call_weight_bytes(f, m)
    return total


def step_bytes_alg(mats, fmt: str, M: int = 1, head_fmt: str | None = None) -> int:
    return step_weight_bytes(mats, fmt, head_fmt) + sum(call_bytes(fmt, M, m) - call_weight_bytes(fmt, m)
                                                          for m in mats)


def step_params(mats) -> int:
    return sum(m.N * m.K for m in mats)
