"""Byte accounting pinned to the figures the pages print (CPU only).

The roofline denominators and the bench's bytes-per-step come from
memory_bound_weight_gb300.workloads; these checks tie it to the pages.
"""
import pytest

from memory_bound_weight_gb300 import workloads as wl


def test_tinyllama_fp16_and_int4_bytes_and_ceilings():
    # tinyinfer, TL;DR: TinyLlama-1.1B reads 2.07 GB per token in 16-bit floats
    # (ceiling ~81 tok/s at 168 GB/s) and 0.55 GB with 4-bit codes plus one fp16
    # scale per 64 weights (ceiling ~305 tok/s).
    mats = wl.tinyllama_step()
    fp16 = 2 * wl.step_params(mats)
    int4 = wl.step_weight_bytes(mats, wl.FMT_INT4_G64)
    assert round(fp16 / 1e9, 2) == 2.07
    assert round(int4 / 1e9, 2) == 0.55
    assert int(168e9 / fp16) == 81
    assert int(168e9 / int4) == 305


def test_tinyinfer_decode_fraction_of_ceiling():
    # tinyinfer, version table: 235.2 tok/s is 77% of the ceiling; 200.7 is 66%; 212.3 is 69%.
    int4 = wl.step_weight_bytes(wl.tinyllama_step(), wl.FMT_INT4_G64)
    for toks, pct in ((235.2, 77), (200.7, 66), (212.3, 69)):
        assert round(100 * toks * int4 / 168e9) == pct


def test_bits_per_weight_table():
    # llm-rs vs vLLM, sec. 6 format table: AWQ 4 + 32/128 = 4.25 (fp16 scale + zero per
    # 128); llm-rs 4-bit 4 + 64/32 = 6 (f32 scale + offset per 32). tinyinfer: 4 bits plus
    # one fp16 scale per 64 weights = 4.25.
    assert wl.bits_per_weight(4, 128, 16, 16) == 4.25
    assert wl.bits_per_weight(4, 32, 32, 32) == 6.0
    assert wl.bits_per_weight(4, 64, 16, 0) == 4.25
    # the stored layouts of this library
    assert wl.weight_bytes(wl.FMT_INT4_G64, 64, 6400) * 8 / (64 * 6400) == 4.25
    assert wl.weight_bytes(wl.FMT_INT4_AWQ_G128, 64, 256 * 25) * 8 / (64 * 6400) == 4 + 20 / 128


def test_qwen_awq_floor_about_6ms():
    # llm-rs vs vLLM, sec. 6: 7B AWQ with a BF16 output layer has a ~6 ms floor at 768 GB/s,
    # and the output layer alone is about 1 GB.
    mats = wl.qwen25_7b_step()
    b = wl.step_weight_bytes(mats, wl.FMT_INT4_AWQ_G128, head_fmt=wl.FMT_BF16)
    assert 5.5e-3 < b / 768e9 < 6.5e-3
    head = wl.weight_bytes(wl.FMT_BF16, wl.QWEN25_7B_HEAD.N, wl.QWEN25_7B_HEAD.K)
    assert round(head / 1e9) == 1


def test_qwen_bf16_floor():
    # llm-rs vs vLLM, sec. 2: ~15 GB in BF16, 15 GB / 768 GB/s = 19.6 ms; the
    # matrices alone are 14.14 GB (the rest is the embedding table).
    mats = wl.qwen25_7b_step()
    b = wl.step_weight_bytes(mats, wl.FMT_BF16)
    assert 14.0e9 < b < 15.0e9
    assert round(15e9 / 768e9 * 1e3, 1) == 19.5 or round(15e9 / 768e9 * 1e3, 1) == 19.6
    assert len(mats) == 141


def test_config_shapes():
    assert [(m.N, m.K) for m in wl.TINYLLAMA_TABLE_SHAPES] == [(2048, 2048), (5632, 2048), (2048, 5632), (32000, 2048)]
    assert wl.bytes_alg(wl.FMT_BF16, 1, 2048, 2048) == 2048 * 2048 * 2 + 4096
    assert wl.bytes_alg(wl.FMT_INT4_G64, 1, 2048, 2048) == 2_232_320
    assert wl.bytes_alg(wl.FMT_INT4_G64, 1, 32000, 2048) == 34_820_096


def test_fused_tinyllama_step_streams_the_same_weights():
    # concatenating q/k/v and gate/up changes the launches, not the bytes
    a, b = wl.tinyllama_step(), wl.tinyllama_step(fused=True)
    assert len(a) == 155 and len(b) == 89
    for fmt in (wl.FMT_BF16, wl.FMT_INT4_G64, wl.FMT_INT4_AWQ_G128):
        assert wl.step_weight_bytes(a, fmt) == wl.step_weight_bytes(b, fmt)
    assert wl.step_params(a) == wl.step_params(b)


def test_qwen3_4b_int8_step_is_about_4_gb():
    """TileInfer, 'Pushing further with cheating: INT8 quantization': INT8
    weights halve the Qwen3-4B step from ~8 GB of BF16 weights to ~4 GB."""
    mats = wl.qwen3_4b_step()
    assert len(mats) == 4 * 36 + 1
    b8 = wl.step_weight_bytes(mats, wl.FMT_INT8_PC)
    b16 = wl.step_weight_bytes(mats, wl.FMT_BF16)
    assert 3.9e9 < b8 < 4.1e9 and 7.9e9 < b16 < 8.1e9
    # the per-channel scales add 4 bytes per output row
    assert b8 - sum(m.N * m.K for m in mats) == 4 * sum(m.N for m in mats)
    assert abs(b8 / b16 - 0.5) < 1e-3


def test_fused_qwen_awq_step_streams_the_same_weights():
    """The AWQ step with the small ops fused streams the same weight bytes in 113 calls instead of 141 (gate and up
    in one gated call per layer); the fusions add only the norm weights and the residuals read."""
    plain, fused = wl.qwen25_7b_step(), wl.qwen25_7b_step(fusedops=True)
    fmt = wl.FMT_INT4_AWQ_G128
    assert len(plain) == 141 and len(fused) == 113
    assert wl.step_weight_bytes(plain, fmt) == wl.step_weight_bytes(fused, fmt)
    extra = wl.step_bytes_alg(fused, fmt) - wl.step_bytes_alg(plain, fmt)
    norms = 28 * 2 * 3584 * 2 + 3584 * 2          # q/k/v and gate/up norm weights per layer, the head's
    residuals = 28 * 2 * 3584 * 2                   # o and down
    x_saved = 28 * 3584 * 2                         # up no longer reads its own x
    assert extra == norms + residuals - x_saved


def test_fused_qwen_bf16_step_streams_the_same_weights():
    """Gate and up stored as one [Wgate; Wup] matrix: the same weight bytes and
    parameters in 113 GEMVs instead of 141."""
    plain, fused = wl.qwen25_7b_step(), wl.qwen25_7b_step(fused=True)
    assert len(plain) == 141 and len(fused) == 113
    assert wl.step_weight_bytes(plain, wl.FMT_BF16) == wl.step_weight_bytes(fused, wl.FMT_BF16)
    assert wl.step_params(plain) == wl.step_params(fused)
    assert sum(m.N for m in fused if m.name.endswith("gate_up")) == 28 * 2 * 18944
