"""The failure path of the kernels' bounded waits, on the GPU without a fault.

Every mbarrier wait in the bulk-copy GEMV and tcgen05 GEMM kernels gives up
after a fixed number of try_wait rounds, sets a device flag and leaves its
loop; the host reads the flag as MBW_ERR_DEVICE_TIMEOUT. Here two one-thread
kernels (one per family) wait on an mbarrier that nothing arrives at, with a
small round limit, so the wait runs out. The test checks the reported status,
that reading clears it, and that the context still computes correct results.
"""
import pytest

import oracle
from gpu_util import assert_parity, dev_bf16, dev_f16, dev_u8
from memory_bound_weight_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - the marker keeps these off CPU runs
    pytest.skip("needs a GPU", allow_module_level=True)

import memory_bound_weight_gb300 as mbw  # noqa: E402

MBW_ERR_DEVICE_TIMEOUT = 7


def test_expired_wait_is_reported_then_cleared():
    mbw.check_device_error()  # nothing left over from earlier launches
    before = mbw.launch_count()
    mbw.selftest_wait_expiry(4096)
    assert mbw.launch_count() == before + 2
    with pytest.raises(mbw.MbwError) as e:
        mbw.check_device_error()
    assert e.value.status == MBW_ERR_DEVICE_TIMEOUT
    mbw.check_device_error()  # read once, cleared


def test_expiry_time_grows_with_the_round_limit():
    # the wait really spins its rounds: 16x the rounds takes clearly longer
    ms = {}
    for tries in (1 << 10, 1 << 14):
        mbw.selftest_wait_expiry(tries)  # warm
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mbw.selftest_wait_expiry(tries)
        e1.record()
        torch.cuda.synchronize()
        ms[tries] = e0.elapsed_time(e1)
        with pytest.raises(mbw.MbwError):
            mbw.check_device_error()
    assert ms[1 << 14] > 4 * ms[1 << 10], ms


def test_context_still_computes_after_an_expired_wait():
    mbw.selftest_wait_expiry(256)
    with pytest.raises(mbw.MbwError):
        mbw.check_device_error()
    orc = oracle.load()
    # AWQ batch 16 (tcgen05 GEMM) and BF16 batch 1 after the expiry
    M, N, K = 16, 300, 512
    c, s, z = gen.int4_codes(2100, 0, N, K), gen.f16_group_scales(2100, 0, N, K // 128), gen.u4_zero_points(2100, 0, N, K // 128)
    X = gen.bf16_activations(2100, 0, M, K)
    Y, A = orc.gemm_int4_awq_g128(c, s, z, X)
    y = mbw.gemv_int4_awq_g128(dev_u8(c), dev_f16(s), dev_u8(z), dev_bf16(X))
    assert_parity(y, Y, A, "awq after expiry")
    W = gen.bf16_weights(2101, 0, N, K)
    x = gen.bf16_activations(2101, 0, 1, K)
    Yb, Ab = orc.gemm_bf16(W, x)
    Wd, xd = dev_bf16(W), dev_bf16(x[0])
    for i in range(mbw.plan_candidates(mbw.OP_GEMV_BF16, 1, N, K)):  # the bulk-copy plans among them
        mbw.plan_select(mbw.OP_GEMV_BF16, 1, N, K, i)
        yb = mbw.gemv_bf16(Wd, xd)
        assert_parity(yb, Yb[0], Ab[0], f"bf16 after expiry {mbw.plan_describe(mbw.OP_GEMV_BF16, 1, N, K)}")
    mbw.check_device_error()
