"""Degenerate sizes and output guard bands for every entry point that takes a
batch (GPU).

K = 0 is the empty sum (outputs set to zero); N = 0 or M = 0 launches
nothing. Ragged shapes on the tensor-core paths (partial 128-row tiles,
partial batch tiles, a CTA pair whose second tile lies past N, batches past
256 that the library runs in slices) must not write outside Y: a sentinel band before and after Y stays untouched, and Y matches
the oracle.
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_parity, dev_bf16, dev_f16, dev_u8
from memory_bound_weight_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - the marker keeps these off CPU runs
    pytest.skip("needs a GPU", allow_module_level=True)

import memory_bound_weight_gb300 as mbw  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def u8(shape):
    return torch.empty(shape, dtype=torch.uint8, device="cuda")


def f16(shape):
    return torch.empty(shape, dtype=torch.float16, device="cuda")


def b16(shape):
    return torch.zeros(shape, dtype=torch.bfloat16, device="cuda")


@pytest.mark.parametrize("repacked", [False, True])
@pytest.mark.parametrize("M", [1, 3, 20])
def test_awq_degenerate_sizes(M, repacked):
    # K = 0: Y is the empty sum
    N = 9
    y = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
    mbw.gemv_int4_awq_g128(u8((N, 0)), f16((N, 0)), u8((N, 0)), b16((M, 0)), out=y, repacked=repacked)
    assert torch.count_nonzero(y).item() == 0
    # N = 0 and M = 0 launch nothing
    before = mbw.launch_count()
    out = mbw.gemv_int4_awq_g128(u8((0, 64)), f16((0, 1)), u8((0, 1)), b16((M, 128)), repacked=repacked)
    assert out.numel() == 0
    out = mbw.gemv_int4_awq_g128(u8((N, 64)), f16((N, 1)), u8((N, 1)), b16((0, 128)), repacked=repacked)
    assert out.numel() == 0
    assert mbw.launch_count() == before


def test_skinny_and_repack_degenerate_sizes():
    N = 11
    y = torch.full((20, N), 5.0, dtype=torch.bfloat16, device="cuda")
    mbw.gemm_skinny_bf16(b16((20, 0)), b16((N, 0)), out=y)
    assert torch.count_nonzero(y).item() == 0
    before = mbw.launch_count()
    assert mbw.gemm_skinny_bf16(b16((0, 64)), b16((N, 64))).numel() == 0
    assert mbw.gemm_skinny_bf16(b16((20, 64)), b16((0, 64))).numel() == 0
    assert mbw.repack_int4(u8((0, 32))).numel() == 0
    assert mbw.repack_int4(u8((4, 0))).numel() == 0
    assert mbw.launch_count() == before


def guarded(M, N):
    """Y (M, N) inside a buffer with 64 sentinel elements on each side."""
    buf = torch.full((M * N + 128,), -7.0, dtype=torch.bfloat16, device="cuda")
    return buf, buf[64:64 + M * N].view(M, N)


def bands_intact(buf, M, N):
    return bool(torch.all(buf[:64] == -7.0)) and bool(torch.all(buf[64 + M * N:] == -7.0))


@pytest.mark.parametrize("M,N,K", [(20, 130, 384), (16, 1, 128), (64, 257, 1024), (100, 129, 256), (300, 130, 256)])
def test_awq_tensor_core_guard_bands(orc, M, N, K):
    G = K // 128
    c, s, z = gen.int4_codes(1800 + N, 0, N, K), gen.f16_group_scales(1800 + N, 0, N, G), gen.u4_zero_points(1800 + N, 0, N, G)
    X = gen.bf16_activations(1800 + N, 0, M, K)
    Y, A = orc.gemm_int4_awq_g128(c, s, z, X)
    for repacked in (False, True):
        cd = mbw.repack_int4(dev_u8(c)) if repacked else dev_u8(c)
        op = mbw.OP_GEMV_INT4_AWQ_G128 | (mbw.REPACKED if repacked else 0)
        for i in range(mbw.plan_candidates(op, M, N, K)):
            mbw.plan_select(op, M, N, K, i)
            buf, y = guarded(M, N)
            mbw.gemv_int4_awq_g128(cd, dev_f16(s), dev_u8(z), dev_bf16(X), out=y, repacked=repacked)
            desc = mbw.plan_describe(op, M, N, K)
            assert bands_intact(buf, M, N), desc
            assert_parity(y, Y, A, f"awq guard {M}x{N}x{K} {desc}")


@pytest.mark.parametrize("M,N,K", [(130, 300, 512), (256, 129, 256), (9, 200, 192), (200, 1, 64),
                                   (300, 200, 256), (520, 130, 128)])  # batches past 256: 2 and 3 slices
def test_skinny_tensor_core_guard_bands(orc, M, N, K):
    W = gen.bf16_weights(1900 + N, 0, N, K)
    X = gen.bf16_activations(1900 + N, 0, M, K)
    Y, A = orc.gemm_bf16(W, X)
    Wd, Xd = dev_bf16(W), dev_bf16(X)
    for i in range(mbw.plan_candidates(mbw.OP_GEMM_SKINNY_BF16, M, N, K)):
        mbw.plan_select(mbw.OP_GEMM_SKINNY_BF16, M, N, K, i)
        desc = mbw.plan_describe(mbw.OP_GEMM_SKINNY_BF16, M, N, K)
        if not desc.startswith("tcgen05"):
            continue
        buf, y = guarded(M, N)
        mbw.gemm_skinny_bf16(Xd, Wd, out=y)
        assert bands_intact(buf, M, N), desc
        assert_parity(y, Y, A, f"skinny guard {M}x{N}x{K} {desc}")
