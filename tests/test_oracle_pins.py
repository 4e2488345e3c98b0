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
