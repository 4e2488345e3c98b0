"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=[p.__name__ for p in oracle_pins.PINS])
def test_pin(orc, pin):
    pin(orc)


def test_fixture_is_hand_worked_not_generated():
    """The golden dequant table is read as text; it carries its citation header."""
    import os

    path = os.path.join(oracle_pins.GOLDEN, "int4_dequant_hand.txt")
    head = open(path).read(2000)
    assert "tinyinfer" in head and "llm-rs vs vLLM" in head
    assert len(oracle_pins.load_dequant_fixture()) >= 30


def test_int8_fixture_is_hand_worked():
    """The INT8 table is read as text and carries its citation header."""
    import os

    head = open(os.path.join(oracle_pins.GOLDEN, "int8_pc_hand.txt")).read(1500)
    assert "TileInfer" in head and "INT8 quantization" in head
    gemv, quant = oracle_pins.load_int8_fixture()
    assert len(gemv) >= 5 and len(quant) >= 4


def test_fusion_fixture_is_hand_worked():
    import os

    head = open(os.path.join(oracle_pins.GOLDEN, "fusion_hand.txt")).read(1200)
    assert "llm-rs vs vLLM" in head and "yalm" in head and "TileInfer" in head
    norm, glu, res = oracle_pins.load_fusion_fixture()
    assert len(norm) >= 5 and len(glu) >= 5 and len(res) >= 3


def test_results_do_not_depend_on_the_thread_count(orc):
    """The row loops run in parallel, but each row is summed in one thread
    in order, so 1 and 4 threads give the same bits."""
    import numpy as np

    from memory_bound_weight_gb300 import inputs as gen

    N, K, M = 37, 512, 3
    W = gen.bf16_weights(40, 0, N, K)
    X = gen.bf16_activations(40, 1, M, K)
    c, s64 = gen.int4_codes(40, 2, N, K), gen.f16_group_scales(40, 3, N, K // 64)
    s128, z = gen.f16_group_scales(40, 4, N, K // 128), gen.u4_zero_points(40, 5, N, K // 128)
    q8, s8 = gen.int8_codes(40, 6, N, K), gen.f32_row_scales(40, 7, N)
    G = gen.bf16_activations(40, 8, 1, K)[0]

    def run():
        out = []
        for r in (orc.gemm_bf16(W, X), orc.gemm_int4_g64(c, s64, X), orc.gemm_int4_awq_g128(c, s128, z, X),
                  orc.gemm_int4_awq_g128(orc.repack_int4(c), s128, z, X, repacked=True),
                  orc.gemm_int8_pc(q8, s8, X), orc.quantize_int8_pc(W)):
            out.extend(r)
        out += [orc.rmsnorm_bf16(X, G, 1e-6), orc.dequant_int4_g64(c, s64, N, K),
                orc.dequant_int4_awq_g128(c, s128, z, N, K)]
        return out

    n = orc.num_threads()
    try:
        orc.set_num_threads(4)
        many = run()
        orc.set_num_threads(1)
        one = run()
    finally:
        orc.set_num_threads(n)
    assert len(many) == len(one) == 15
    for a, b in zip(many, one):
        assert a.dtype == b.dtype and np.array_equal(a.view(np.uint8), b.view(np.uint8))
