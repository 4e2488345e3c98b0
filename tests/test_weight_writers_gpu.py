"""A load-time weight writer followed by a GEMV on the same stream, with no
host synchronization in between.

The GEMV kernels stream their weights before they wait for the kernel in
front of them (programmatic dependent launch). The library's weight writers
(the INT8 quantizer, TileInfer "Pushing further with cheating: INT8
quantization"; the INT4 repack, llm-rs vs vLLM sec. 6 on Marlin's load-time
reorder) end with a plainly ordered empty kernel, so the GEMV behind them must
read the weights they wrote. Each round first refills the weight buffers with
other contents, so a GEMV that read ahead of the writer would return a product
of the stale weights and fail the comparison with the oracle.
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
from memory_bound_weight_gb300 import _binding  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def test_quantize_then_int8_gemv_without_sync(orc):
    N, K = 6144, 2560
    W = gen.bf16_weights(1501, 0, N, K)
    X = gen.bf16_activations(1501, 1, 1, K)
    q_ref, s_ref = orc.quantize_int8_pc(W)
    Y, A = orc.gemm_int8_pc(q_ref, s_ref, X)
    Wd, xd = dev_bf16(W), dev_bf16(X[0])
    stale_q = torch.from_numpy(gen.int8_codes(1501, 2, N, K)).cuda()
    stale_s = torch.from_numpy(gen.f32_row_scales(1501, 3, N)).cuda()
    Wq = torch.empty_like(stale_q)
    sc = torch.empty_like(stale_s)
    stream = torch.cuda.current_stream().cuda_stream
    for plan in range(min(3, mbw.plan_candidates(mbw.OP_GEMV_INT8_PC, 1, N, K))):
        mbw.plan_select(mbw.OP_GEMV_INT8_PC, 1, N, K, plan)
        Wq.copy_(stale_q)
        sc.copy_(stale_s)
        _binding.check("mbw_quantize_int8_pc", _binding.lib().mbw_quantize_int8_pc(
            Wd.data_ptr(), Wq.data_ptr(), sc.data_ptr(), N, K, stream))
        y = mbw.gemv_int8_pc(Wq, sc, xd)  # same stream, no synchronization
        assert_parity(y, Y[0], A[0], f"quantize -> gemv_int8_pc ({mbw.plan_describe(mbw.OP_GEMV_INT8_PC, 1, N, K)})")
    assert np.array_equal(Wq.cpu().numpy(), q_ref) and np.array_equal(sc.cpu().numpy(), s_ref)


@pytest.mark.parametrize("M", [1, 16])
def test_repack_in_place_then_awq_gemv_without_sync(orc, M):
    N, K = 4608, 3584
    G = K // 128
    c = gen.int4_codes(1502, 0, N, K)
    s = gen.f16_group_scales(1502, 0, N, G)
    z = gen.u4_zero_points(1502, 0, N, G)
    X = gen.bf16_activations(1502, 1, M, K)
    Y, A = orc.gemm_int4_awq_g128(c, s, z, X)
    cd = dev_u8(c)
    sd, zd, Xd = dev_f16(s), dev_u8(z), dev_bf16(X)
    buf = torch.empty_like(cd)
    op = mbw.OP_GEMV_INT4_AWQ_G128 | mbw.REPACKED
    for plan in range(min(3, mbw.plan_candidates(op, M, N, K))):
        mbw.plan_select(op, M, N, K, plan)
        buf.copy_(cd)  # canonical codes: stale for the repacked product
        mbw.repack_int4(buf, out=buf)  # in place
        Yd = mbw.gemv_int4_awq_g128(buf, sd, zd, Xd, repacked=True)  # same stream, no synchronization
        assert_parity(Yd, Y, A, f"repack -> awq repacked M={M} ({mbw.plan_describe(op, M, N, K)})")
