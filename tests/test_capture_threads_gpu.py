"""Two conventions of the C ABI on the GPU: calls are capturable into CUDA
graphs even for a shape never planned (the default plan is taken, no tuning
happens, and mbw_autotune refuses a capturing stream), and calls from several
host threads on their own streams are safe (the plan cache is shared under a
lock) and give the same results as one thread."""
import threading

import pytest

import oracle
from gpu_util import assert_parity, dev_bf16, dev_f16, dev_u8, host_bits16
from memory_bound_weight_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - the marker keeps these off CPU runs
    pytest.skip("needs a GPU", allow_module_level=True)

import memory_bound_weight_gb300 as mbw  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def test_unplanned_shapes_capture_into_a_graph(orc):
    # shapes no other test plans: the first call of each happens inside the capture
    N1, K1 = 1111, 1536
    W = gen.bf16_weights(2200, 0, N1, K1)
    x = gen.bf16_activations(2200, 0, 1, K1)
    Yb, Ab = orc.gemm_bf16(W, x)
    M2, N2, K2 = 24, 515, 640
    c, s, z = gen.int4_codes(2201, 0, N2, K2), gen.f16_group_scales(2201, 0, N2, K2 // 128), \
        gen.u4_zero_points(2201, 0, N2, K2 // 128)
    X = gen.bf16_activations(2201, 0, M2, K2)
    Ya, Aa = orc.gemm_int4_awq_g128(c, s, z, X)
    Wd, xd, cd, sd, zd, Xd = dev_bf16(W), dev_bf16(x[0]), dev_u8(c), dev_f16(s), dev_u8(z), dev_bf16(X)
    yb = torch.empty((N1,), dtype=torch.bfloat16, device="cuda")
    ya = torch.empty((M2, N2), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=st):
        mbw.gemv_bf16(Wd, xd, out=yb)
        mbw.gemv_int4_awq_g128(cd, sd, zd, Xd, out=ya)
        with pytest.raises(mbw.MbwError) as e:
            mbw.autotune(mbw.OP_GEMV_BF16, 1, N1, K1)  # refused while capturing
        assert e.value.status == 1
    yb.zero_()
    ya.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_parity(yb, Yb[0], Ab[0], f"captured bf16 {mbw.plan_describe(mbw.OP_GEMV_BF16, 1, N1, K1)}")
    assert_parity(ya, Ya, Aa, f"captured awq {mbw.plan_describe(mbw.OP_GEMV_INT4_AWQ_G128, M2, N2, K2)}")


def test_calls_from_two_threads_match_one_thread(orc):
    cases = []
    for t, (N, K) in enumerate(((1234, 2048), (777, 4096))):
        c, s = gen.int4_codes(2300 + t, 0, N, K), gen.f16_group_scales(2300 + t, 0, N, K // 64)
        x = gen.bf16_activations(2300 + t, 0, 1, K)
        Y, A = orc.gemm_int4_g64(c, s, x)
        cases.append((dev_u8(c), dev_f16(s), dev_bf16(x[0]), Y[0], A[0]))
    outs = [[], []]
    errors = []

    def worker(t):
        try:
            cd, sd, xd = cases[t][:3]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                ys = [mbw.gemv_int4_g64(cd, sd, xd) for _ in range(50)]
            stream.synchronize()
            outs[t] = [host_bits16(y) for y in ys]
        except Exception as ex:  # reported below, on the main thread
            errors.append(ex)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    # the threads made the first calls of both shapes; now one thread
    ref = [host_bits16(mbw.gemv_int4_g64(cd, sd, xd)) for cd, sd, xd, _, _ in cases]
    for t, (cd, sd, xd, Y, A) in enumerate(cases):
        assert len(outs[t]) == 50
        assert all((o == ref[t]).all() for o in outs[t]), f"thread {t}: results differ from one thread"
        assert_parity(mbw.gemv_int4_g64(cd, sd, xd), Y, A, f"int4 {t}")
