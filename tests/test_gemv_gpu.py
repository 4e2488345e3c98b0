"""GPU parity of the weight-streaming GEMV kernels against the fp64 oracle.

Every call goes through the C ABI (libmbw.so via the ctypes binding). Small
shapes span several CTA tiles and a ragged tail and run every candidate plan
(each kernel instantiation x split-K factor); full-size shapes run the plans
the benchmark uses and compare every row (or sampled rows where the oracle
would take too long).
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_parity, dev_bf16, dev_f16, dev_u8, host_bits16, host_f64
from memory_bound_weight_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - the marker keeps these off CPU runs
    pytest.skip("needs a GPU", allow_module_level=True)

import memory_bound_weight_gb300 as mbw  # noqa: E402
from memory_bound_weight_gb300 import inputs_gpu  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def bf16_case(seed, N, K, M=1):
    W = gen.bf16_weights(seed, 0, N, K)
    X = gen.bf16_activations(seed, 0, M, K)
    return W, X


def g64_case(seed, N, K):
    return gen.int4_codes(seed, 0, N, K), gen.f16_group_scales(seed, 0, N, K // 64), gen.bf16_activations(seed, 0, 1, K)


def awq_case(seed, N, K, M):
    G = K // 128
    return (gen.int4_codes(seed, 0, N, K), gen.f16_group_scales(seed, 0, N, G), gen.u4_zero_points(seed, 0, N, G),
            gen.bf16_activations(seed, 0, M, K))


def each_plan(op, M, N, K):
    n = mbw.plan_candidates(op, M, N, K)
    assert n >= 1
    for i in range(n):
        mbw.plan_select(op, M, N, K, i)
        yield i, mbw.plan_describe(op, M, N, K)


# ------------------------------------------------------------ small shapes ----
@pytest.mark.parametrize("N,K", [(1, 8), (7, 64), (33, 200), (257, 1032), (1000, 2048), (96, 5632), (2501, 1040)])
def test_bf16_all_plans(orc, N, K):
    W, X = bf16_case(100 + N, N, K)
    Y, A = orc.gemm_bf16(W, X)
    Wd, xd = dev_bf16(W), dev_bf16(X[0])
    for i, desc in each_plan(mbw.OP_GEMV_BF16, 1, N, K):
        y = mbw.gemv_bf16(Wd, xd)
        assert_parity(y, Y[0], A[0], f"bf16 {N}x{K} plan {desc}")


@pytest.mark.parametrize("N,K", [(1, 64), (5, 128), (37, 320), (300, 2048), (130, 5632), (64, 18944)])
def test_int4_g64_all_plans(orc, N, K):
    c, s, X = g64_case(200 + N, N, K)
    Y, A = orc.gemm_int4_g64(c, s, X)
    cd, sd, xd = dev_u8(c), dev_f16(s), dev_bf16(X[0])
    for i, desc in each_plan(mbw.OP_GEMV_INT4_G64, 1, N, K):
        y = mbw.gemv_int4_g64(cd, sd, xd)
        assert_parity(y, Y[0], A[0], f"g64 {N}x{K} plan {desc}")


@pytest.mark.parametrize("N,K,M", [(3, 128, 1), (45, 384, 1), (129, 1024, 3), (64, 256, 8), (33, 640, 9),
                                   (70, 3584, 2), (17, 18944, 1), (40, 512, 5), (300, 5632, 2), (2501, 3584, 1),
                                   (77, 18944, 4)])
def test_int4_awq_all_plans(orc, N, K, M):
    c, s, z, X = awq_case(300 + N, N, K, M)
    Y, A = orc.gemm_int4_awq_g128(c, s, z, X)
    cd, sd, zd, Xd = dev_u8(c), dev_f16(s), dev_u8(z), dev_bf16(X)
    for i, desc in each_plan(mbw.OP_GEMV_INT4_AWQ_G128, M, N, K):
        y = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)
        assert_parity(y, Y, A, f"awq {M}x{N}x{K} plan {desc}")


@pytest.mark.parametrize("M,N,K", [(1, 77, 512), (2, 64, 256), (3, 130, 1024), (4, 33, 2048), (5, 40, 128),
                                   (8, 257, 3584), (9, 64, 512), (16, 96, 1024)])
def test_skinny_bf16_all_plans(orc, M, N, K):
    W, X = bf16_case(400 + M, N, K, M)
    Y, A = orc.gemm_bf16(W, X)
    Wd, Xd = dev_bf16(W), dev_bf16(X)
    for i, desc in each_plan(mbw.OP_GEMM_SKINNY_BF16, M, N, K):
        y = mbw.gemm_skinny_bf16(Xd, Wd)
        assert_parity(y, Y, A, f"skinny {M}x{N}x{K} plan {desc}")


# --------------------------------------------------- exactness and invariants ----
def test_dequant_bit_exact(orc):
    for N, K in ((37, 320), (256, 2048)):
        c, s, _ = g64_case(500 + N, N, K)
        got = mbw.dequant_int4_g64(dev_u8(c), dev_f16(s)).cpu().numpy().astype(np.float64)
        assert np.array_equal(got, orc.dequant_int4_g64(c, s, N, K))
    for N, K in ((45, 384), (100, 3584)):
        c, s, z, _ = awq_case(500 + N, N, K, 1)
        got = mbw.dequant_int4_awq_g128(dev_u8(c), dev_f16(s), dev_u8(z)).cpu().numpy().astype(np.float64)
        assert np.array_equal(got, orc.dequant_int4_awq_g128(c, s, z, N, K))


@pytest.mark.parametrize("fmt", ["bf16", "g64", "awq"])
def test_one_hot_x_gives_the_exact_column(orc, fmt):
    """x = e_k: with fp32 output the GEMV returns column k of the weights
    exactly, on every plan -- the in-kernel unpack and dequant are bit-exact."""
    N, K = 200, 1024
    if fmt == "bf16":
        W, _ = bf16_case(601, N, K)
        deq = np.array([[orc.bf16_to_double(int(b)) for b in row] for row in W[:, [0, 1, 63, 64, 127, 128, 511, 1023]]])
        deq_full = np.zeros((N, K))
        deq_full[:, [0, 1, 63, 64, 127, 128, 511, 1023]] = deq
        deq = deq_full
        Wd = dev_bf16(W)
    elif fmt == "g64":
        c, s, _ = g64_case(602, N, K)
        deq = orc.dequant_int4_g64(c, s, N, K)
        cd, sd = dev_u8(c), dev_f16(s)
    else:
        c, s, z, _ = awq_case(603, N, K, 1)
        deq = orc.dequant_int4_awq_g128(c, s, z, N, K)
        cd, sd, zd = dev_u8(c), dev_f16(s), dev_u8(z)
    op = {"bf16": mbw.OP_GEMV_BF16, "g64": mbw.OP_GEMV_INT4_G64, "awq": mbw.OP_GEMV_INT4_AWQ_G128}[fmt]
    xs = {}
    for k in (0, 1, 63, 64, 127, 128, 511, 1023):
        e = np.zeros(K, dtype=np.uint16)
        e[k] = 0x3F80  # 1.0
        xs[k] = dev_bf16(e)
    for _, desc in each_plan(op, 1, N, K):  # every family and instantiation
        for k, xd in xs.items():
            with mbw.output_fp32():
                if fmt == "bf16":
                    y = mbw.gemv_bf16(Wd, xd)
                elif fmt == "g64":
                    y = mbw.gemv_int4_g64(cd, sd, xd)
                else:
                    y = mbw.gemv_int4_awq_g128(cd, sd, zd, xd)
            assert np.array_equal(host_f64(y), deq[:, k]), (fmt, k, desc)


def test_power_of_two_scaling_and_determinism():
    """On every plan: a repeated call returns the same bits (fixed-order sums,
    no atomics), and scaling x by a power of two scales the fp32 output
    exactly."""
    N, K = 3000, 2048
    c, s, X = g64_case(700, N, K)
    cd, sd = dev_u8(c), dev_f16(s)
    x = dev_bf16(X[0])
    x2 = (x.float() * 4.0).to(torch.bfloat16)
    for _, desc in each_plan(mbw.OP_GEMV_INT4_G64, 1, N, K):
        with mbw.output_fp32():
            y1 = mbw.gemv_int4_g64(cd, sd, x)
            y1b = mbw.gemv_int4_g64(cd, sd, x)
            y2 = mbw.gemv_int4_g64(cd, sd, x2)
        assert torch.equal(y1, y1b), desc
        assert torch.equal(y2, y1 * 4.0), desc
    W, Xb = bf16_case(701, N, K)
    Wd = dev_bf16(W)
    xb = dev_bf16(Xb[0])
    xh = (xb.float() * 0.5).to(torch.bfloat16)
    for _, desc in each_plan(mbw.OP_GEMV_BF16, 1, N, K):
        with mbw.output_fp32():
            a = mbw.gemv_bf16(Wd, xb)
            b = mbw.gemv_bf16(Wd, xb)
            h = mbw.gemv_bf16(Wd, xh)
        assert torch.equal(a, b), desc
        assert torch.equal(h, a * 0.5), desc


def test_zero_weights_give_exact_zero():
    """Codes equal to the zero point are zero weights: every plan returns an
    exact zero (n - z enters the products exactly, so nothing is left over
    from cancellation)."""
    N, K = 513, 2048
    codes = torch.full((N, K // 2), 0x88, dtype=torch.uint8, device="cuda")  # q = 8 -> w = 0
    scales = torch.full((N, K // 64), 1.0, dtype=torch.float16, device="cuda")
    x = dev_bf16(gen.bf16_activations(7, 0, 1, K)[0])
    for _, desc in each_plan(mbw.OP_GEMV_INT4_G64, 1, N, K):
        with mbw.output_fp32():
            y = mbw.gemv_int4_g64(codes, scales, x)
        assert torch.count_nonzero(y).item() == 0, desc
    # AWQ: every code equal to its group's zero point (5), canonical and repacked codes
    G = K // 128
    codes = torch.full((N, K // 2), 0x55, dtype=torch.uint8, device="cuda")
    zeros = torch.full((N, (G + 1) // 2), 0x55, dtype=torch.uint8, device="cuda")
    scales = torch.full((N, G), 3.0, dtype=torch.float16, device="cuda")
    for M in (1, 4, 16):
        X = dev_bf16(gen.bf16_activations(8, 0, M, K))
        for rp in (False, True):
            op = mbw.OP_GEMV_INT4_AWQ_G128 | (mbw.REPACKED if rp else 0)
            for _, desc in each_plan(op, M, N, K):
                with mbw.output_fp32():
                    y = mbw.gemv_int4_awq_g128(codes, scales, zeros, X, repacked=rp)
                assert torch.count_nonzero(y).item() == 0, desc


def test_edge_cases_and_canaries(orc):
    # K = 0: the empty sum
    y = torch.full((5,), 7.0, dtype=torch.bfloat16, device="cuda")
    Wz = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    xz = torch.empty((0,), dtype=torch.bfloat16, device="cuda")
    mbw.gemv_bf16(Wz, xz, out=y)
    assert torch.count_nonzero(y).item() == 0
    # N = 0: no-op
    out = mbw.gemv_bf16(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros(64, dtype=torch.bfloat16, device="cuda"))
    assert out.numel() == 0
    # guard bands around y stay untouched for ragged N
    for N in (1, 7, 2049):
        K = 512
        W, X = bf16_case(800 + N, N, K)
        Y, A = orc.gemm_bf16(W, X)
        buf = torch.full((N + 64,), -3.0, dtype=torch.bfloat16, device="cuda")
        y = buf[32:32 + N]
        mbw.gemv_bf16(dev_bf16(W), dev_bf16(X[0]), out=y)
        assert torch.all(buf[:32] == -3.0) and torch.all(buf[32 + N:] == -3.0)
        assert_parity(y, Y[0], A[0], f"canary N={N}")


def test_device_generator_matches_host():
    N, K = 300, 3584
    W = inputs_gpu.bf16_weights(0, 5, N, K)
    assert np.array_equal(host_bits16(W), gen.bf16_weights(0, 5, N, K))
    c = inputs_gpu.int4_codes(0, 5, N, K)
    assert np.array_equal(c.cpu().numpy(), gen.int4_codes(0, 5, N, K))
    s = inputs_gpu.f16_group_scales(0, 5, N, K // 128)
    assert np.array_equal(host_bits16(s), gen.f16_group_scales(0, 5, N, K // 128))
    z = inputs_gpu.u4_zero_points(0, 5, N, K // 128)
    assert np.array_equal(z.cpu().numpy(), gen.u4_zero_points(0, 5, N, K // 128))
    # a row range in the middle of a stream
    W2 = gen.bf16_weights(0, 5, N, K, row0=123, rows=7)
    assert np.array_equal(host_bits16(W[123:130]), W2)


# ------------------------------------------------------------- full sizes ----
def test_tinyllama_int4_shapes_full_rows(orc):
    """The four TinyLlama-shaped INT4 g64 matrices and the 256-row K/V shape,
    every row, with the autotuned plans the benchmark uses."""
    for mi, (N, K) in enumerate([(2048, 2048), (5632, 2048), (2048, 5632), (32000, 2048), (256, 2048)]):
        mbw.autotune(mbw.OP_GEMV_INT4_G64, 1, N, K)
        cd = inputs_gpu.int4_codes(0, mi, N, K)
        sd = inputs_gpu.f16_group_scales(0, mi, N, K // 64)
        xd = inputs_gpu.bf16_activations(0, mi, 1, K)[0]
        y = mbw.gemv_int4_g64(cd, sd, xd)
        Y, A = orc.gemm_int4_g64(cd.cpu().numpy(), host_bits16(sd), host_bits16(xd)[None, :])
        assert_parity(y, Y[0], A[0], f"g64 {N}x{K} ({mbw.plan_describe(mbw.OP_GEMV_INT4_G64, 1, N, K)})")


def test_bf16_2048_full(orc):
    W, X = bf16_case(0, 2048, 2048)
    mbw.autotune(mbw.OP_GEMV_BF16, 1, 2048, 2048)
    y = mbw.gemv_bf16(dev_bf16(W), dev_bf16(X[0]))
    Y, A = orc.gemm_bf16(W, X)
    assert_parity(y, Y[0], A[0], "bf16 2048x2048")


@pytest.mark.parametrize("N,K", [(4608, 3584), (3584, 18944), (152064, 3584)])
def test_qwen_shapes_sampled_rows(orc, N, K):
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(N - 8, N),
                                     np.random.default_rng(N).integers(0, N, 112)]))
    Wd = inputs_gpu.bf16_weights(0, 1, N, K)
    xd = inputs_gpu.bf16_activations(0, 1, 1, K)[0]
    y = mbw.gemv_bf16(Wd, xd)
    Wr = np.stack([gen.bf16_weights(0, 1, N, K, row0=int(r), rows=1)[0] for r in rows])
    Y, A = orc.gemm_bf16(Wr, host_bits16(xd)[None, :])
    assert_parity(y[torch.from_numpy(rows).cuda()], Y[0], A[0], f"bf16 {N}x{K} sampled")
    del Wd
    # the same shape in AWQ form, batch 1 and 16
    G = K // 128
    cd = inputs_gpu.int4_codes(0, 2, N, K)
    sd = inputs_gpu.f16_group_scales(0, 2, N, G)
    zd = inputs_gpu.u4_zero_points(0, 2, N, G)
    cr = np.stack([gen.int4_codes(0, 2, N, K, row0=int(r), rows=1)[0] for r in rows])
    sr = np.stack([gen.f16_group_scales(0, 2, N, G, row0=int(r), rows=1)[0] for r in rows])
    zr = np.stack([gen.u4_zero_points(0, 2, N, G, row0=int(r), rows=1)[0] for r in rows])
    for M in (1, 16):
        Xd = inputs_gpu.bf16_activations(0, 3, M, K)
        Yd = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)
        Y, A = orc.gemm_int4_awq_g128(cr, sr, zr, host_bits16(Xd))
        assert_parity(Yd[:, torch.from_numpy(rows).cuda()], Y, A, f"awq M={M} {N}x{K} sampled")


# -------------------------------------------------- tensor-core skinny GEMM ----
@pytest.mark.parametrize("M,N,K", [(16, 128, 64), (16, 300, 256), (32, 257, 512), (48, 128, 1032), (64, 640, 3584),
                                   (100, 200, 192), (128, 130, 128), (256, 384, 1024), (300, 129, 256)])
def test_skinny_tcgen05_all_plans(orc, M, N, K):
    W, X = bf16_case(900 + M, N, K, M)
    Y, A = orc.gemm_bf16(W, X)
    Wd, Xd = dev_bf16(W), dev_bf16(X)
    seen_tc = False
    for i, desc in each_plan(mbw.OP_GEMM_SKINNY_BF16, M, N, K):
        seen_tc |= desc.startswith("tcgen05")
        y = mbw.gemm_skinny_bf16(Xd, Wd)
        assert_parity(y, Y, A, f"skinny {M}x{N}x{K} plan {desc}")
    assert seen_tc


@pytest.mark.parametrize("M,N,K", [(256, 640, 3584), (128, 300, 2048), (200, 1000, 4096), (256, 128, 18944),
                                   (129, 257, 1024)])
def test_skinny_tcgen05_cta_pair_plans(orc, M, N, K):
    """The CTA-pair kernel (cta_group::2 MMAs across two SMs): every pair plan,
    including split-K clusters of up to 4 pairs, an odd number of 128-row tiles
    (the last pair's second CTA reads rows past N) and partial batch tiles."""
    W, X = bf16_case(960 + M + N, N, K, M)
    Y, A = orc.gemm_bf16(W, X)
    Wd, Xd = dev_bf16(W), dev_bf16(X)
    seen = 0
    for i, desc in each_plan(mbw.OP_GEMM_SKINNY_BF16, M, N, K):
        if "cta pair" not in desc:
            continue
        seen += 1
        y = mbw.gemm_skinny_bf16(Xd, Wd)
        assert_parity(y, Y, A, f"skinny pair {M}x{N}x{K} plan {desc}")
        with mbw.output_fp32():
            y1 = mbw.gemm_skinny_bf16(Xd, Wd)
            y2 = mbw.gemm_skinny_bf16(Xd, Wd)
        assert torch.equal(y1, y2), desc
    assert seen >= 4


@pytest.mark.parametrize("N,K", [(18944, 3584), (3584, 18944)])
def test_skinny_cta_pair_config_shapes_sampled_rows(orc, N, K):
    """Every CTA-pair plan at the Qwen2.5-7B MLP shapes, batch 256, sampled rows."""
    M = 256
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(N - 8, N),
                                     np.random.default_rng(N + 5).integers(0, N, 48)]))
    Wd = inputs_gpu.bf16_weights(0, 9, N, K)
    Xd = inputs_gpu.bf16_activations(0, 10, M, K)
    Wr = np.stack([gen.bf16_weights(0, 9, N, K, row0=int(r), rows=1)[0] for r in rows])
    Yr, Ar = orc.gemm_bf16(Wr, host_bits16(Xd))
    sel = torch.from_numpy(rows).cuda()
    seen = 0
    for i, desc in each_plan(mbw.OP_GEMM_SKINNY_BF16, M, N, K):
        if "cta pair" not in desc:
            continue
        seen += 1
        Y = mbw.gemm_skinny_bf16(Xd, Wd)
        assert_parity(Y[:, sel], Yr, Ar, f"skinny pair M={M} {N}x{K} plan {desc}")
    assert seen >= 4


def test_skinny_tcgen05_deterministic_and_scaling():
    M, N, K = 64, 1024, 2048
    W, X = bf16_case(950, N, K, M)
    Wd, Xd = dev_bf16(W), dev_bf16(X)
    with mbw.output_fp32():
        y1 = mbw.gemm_skinny_bf16(Xd, Wd)
        y2 = mbw.gemm_skinny_bf16(Xd, Wd)
        y4 = mbw.gemm_skinny_bf16((Xd.float() * 4).to(torch.bfloat16), Wd)
    assert torch.equal(y1, y2)
    assert torch.equal(y4, y1 * 4)
    assert mbw.plan_describe(mbw.OP_GEMM_SKINNY_BF16, M, N, K).startswith("tcgen05")


@pytest.mark.parametrize("M", [16, 64, 256])
@pytest.mark.parametrize("N,K", [(18944, 3584), (3584, 18944)])
def test_skinny_config_shapes_sampled_rows(orc, M, N, K):
    """The Qwen2.5-7B MLP shapes at the skinny batch sizes, default plan, every
    batch row of 96 sampled weight rows against the oracle."""
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(N - 8, N),
                                     np.random.default_rng(N + M).integers(0, N, 80)]))
    Wd = inputs_gpu.bf16_weights(0, 7, N, K)
    Xd = inputs_gpu.bf16_activations(0, 8, M, K)
    Y = mbw.gemm_skinny_bf16(Xd, Wd)
    Wr = np.stack([gen.bf16_weights(0, 7, N, K, row0=int(r), rows=1)[0] for r in rows])
    Yr, Ar = orc.gemm_bf16(Wr, host_bits16(Xd))
    assert_parity(Y[:, torch.from_numpy(rows).cuda()], Yr, Ar, f"skinny M={M} {N}x{K} sampled")


@pytest.mark.parametrize("N,K", [(2560, 2048), (11264, 2048), (2048, 5632), (5632, 2048)])
def test_int4_g64_every_plan_at_step_shapes(orc, N, K):
    """Every candidate plan (all families, instantiations, splits, CTAs per SM)
    at the fused and named TinyLlama shapes, on sampled rows: the register-
    and shared-memory-staged latency kernels own up to six items per warp
    only at these sizes."""
    rows = np.unique(np.concatenate([np.arange(0, 16), np.arange(N - 16, N),
                                     np.random.default_rng(N + K).integers(0, N, 64)]))
    cd = inputs_gpu.int4_codes(0, 3, N, K)
    sd = inputs_gpu.f16_group_scales(0, 3, N, K // 64)
    xd = inputs_gpu.bf16_activations(0, 4, 1, K)
    c = np.stack([gen.int4_codes(0, 3, N, K, row0=int(r), rows=1)[0] for r in rows])
    s = np.stack([gen.f16_group_scales(0, 3, N, K // 64, row0=int(r), rows=1)[0] for r in rows])
    Y, A = orc.gemm_int4_g64(c, s, host_bits16(xd))
    sel = torch.from_numpy(rows).cuda()
    for i, desc in each_plan(mbw.OP_GEMV_INT4_G64, 1, N, K):
        y = mbw.gemv_int4_g64(cd, sd, xd[0])
        assert_parity(y[sel], Y[0], A[0], f"g64 {N}x{K} plan {desc}")


# ------------------------------------------ AWQ batched tensor-core path ----
@pytest.mark.parametrize("N,K,M", [(130, 256, 16), (128, 384, 5), (300, 1024, 33), (64, 3584, 64),
                                   (257, 512, 100), (40, 1280, 17), (200, 640, 130)])
def test_int4_awq_batched_all_plans(orc, N, K, M):
    c, s, z, X = awq_case(800 + M, N, K, M)
    Y, A = orc.gemm_int4_awq_g128(c, s, z, X)
    cd, sd, zd, Xd = dev_u8(c), dev_f16(s), dev_u8(z), dev_bf16(X)
    seen_tc = False
    for i, desc in each_plan(mbw.OP_GEMV_INT4_AWQ_G128, M, N, K):
        seen_tc |= desc.startswith("tcgen05")
        y = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)
        assert_parity(y, Y, A, f"awq {M}x{N}x{K} plan {desc}")
    assert seen_tc


def test_int4_awq_batched_one_hot_rows_exact(orc):
    """Batch row m = e_{k_m}: with fp32 output every tensor-core plan (tcgen05
    and the batched mma.sync family) returns column k_m of the dequantized
    weights exactly (exact unpack, exact products, the group scale applied in
    fp32 to a single nonzero term)."""
    N, K, M = 200, 1024, 24
    c, s, z, _ = awq_case(811, N, K, 1)
    deq = orc.dequant_int4_awq_g128(c, s, z, N, K)
    ks = [(37 * m + 5) % K for m in range(M)]
    X = np.zeros((M, K), dtype=np.uint16)
    for m, k in enumerate(ks):
        X[m, k] = 0x3F80
    cd, sd, zd, Xd = dev_u8(c), dev_f16(s), dev_u8(z), dev_bf16(X)
    for i, desc in each_plan(mbw.OP_GEMV_INT4_AWQ_G128, M, N, K):
        if not desc.startswith(("tcgen05", "awq_mma")):
            continue
        with mbw.output_fp32():
            y = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)
        got = host_f64(y)
        for m, k in enumerate(ks):
            assert np.array_equal(got[m], deq[:, k]), (desc, m, k)


@pytest.mark.parametrize("M", [16, 64])
@pytest.mark.parametrize("N,K", [(18944, 3584), (3584, 18944)])
def test_int4_awq_batched_config_shapes_sampled_rows(orc, M, N, K):
    G = K // 128
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(N - 8, N),
                                     np.random.default_rng(N + M).integers(0, N, 48)]))
    cd = inputs_gpu.int4_codes(0, 21, N, K)
    sd = inputs_gpu.f16_group_scales(0, 21, N, G)
    zd = inputs_gpu.u4_zero_points(0, 21, N, G)
    Xd = inputs_gpu.bf16_activations(0, 22, M, K)
    Y = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)
    assert mbw.plan_describe(mbw.OP_GEMV_INT4_AWQ_G128, M, N, K).startswith(("tcgen05", "awq_mma"))
    c = np.stack([gen.int4_codes(0, 21, N, K, row0=int(r), rows=1)[0] for r in rows])
    s = np.stack([gen.f16_group_scales(0, 21, N, G, row0=int(r), rows=1)[0] for r in rows])
    z = np.stack([gen.u4_zero_points(0, 21, N, G, row0=int(r), rows=1)[0] for r in rows])
    Yr, Ar = orc.gemm_int4_awq_g128(c, s, z, host_bits16(Xd))
    assert_parity(Y[:, torch.from_numpy(rows).cuda()], Yr, Ar, f"awq M={M} {N}x{K} sampled")


def test_weights_at_a_32_byte_offset_every_plan(orc):
    """The weight pointer only has to be 32-byte aligned: every plan of every
    format runs on weights that start 32 bytes into a larger allocation."""
    N, K = 300, 1024
    W, X = bf16_case(1201, N, K)
    big = torch.empty(N * K + 64, dtype=torch.bfloat16, device="cuda")
    Wd = big[16:16 + N * K].view(N, K)
    Wd.copy_(dev_bf16(W))
    assert Wd.data_ptr() % 64 == 32
    Y, A = orc.gemm_bf16(W, X)
    for _, desc in each_plan(mbw.OP_GEMV_BF16, 1, N, K):
        assert_parity(mbw.gemv_bf16(Wd, dev_bf16(X[0])), Y[0], A[0], f"bf16 offset plan {desc}")

    c, s, X1 = g64_case(1202, N, K)
    bigc = torch.empty(N * K // 2 + 64, dtype=torch.uint8, device="cuda")
    cd = bigc[32:32 + N * K // 2].view(N, K // 2)
    cd.copy_(dev_u8(c))
    Y, A = orc.gemm_int4_g64(c, s, X1)
    for _, desc in each_plan(mbw.OP_GEMV_INT4_G64, 1, N, K):
        assert_parity(mbw.gemv_int4_g64(cd, dev_f16(s), dev_bf16(X1[0])), Y[0], A[0], f"g64 offset plan {desc}")

    q = gen.int8_codes(1203, 0, N, K)
    sq = gen.f32_row_scales(1203, 0, N)
    bigq = torch.empty(N * K + 64, dtype=torch.int8, device="cuda")
    qd = bigq[32:32 + N * K].view(N, K)
    qd.copy_(torch.from_numpy(q).cuda())
    Y, A = orc.gemm_int8_pc(q, sq, X)
    for _, desc in each_plan(mbw.OP_GEMV_INT8_PC, 1, N, K):
        assert_parity(mbw.gemv_int8_pc(qd, torch.from_numpy(sq).cuda(), dev_bf16(X[0])), Y[0], A[0],
                      f"int8 offset plan {desc}")
    # 16 bytes is not enough
    with pytest.raises(mbw.MbwError):
        mbw.gemv_int8_pc(bigq[16:16 + N * K].view(N, K), torch.from_numpy(sq).cuda(), dev_bf16(X[0]))


# ------------------------------------ every plan at the Qwen2.5-7B BF16 shapes ----
@pytest.mark.parametrize("N,K", [(4608, 3584), (3584, 3584), (18944, 3584), (3584, 18944), (152064, 3584)])
def test_bf16_every_plan_at_qwen_step_shapes(orc, N, K):
    """Every candidate plan of the batch-1 BF16 GEMV (each family,
    instantiation, split-K factor and CTAs per SM), then the autotuned plan,
    at the shapes of the Qwen2.5-7B decode step; every row against the
    oracle. The weights come from the device generator (bit-identical to the
    host one, test_device_generator_matches_host) and are read back for the
    oracle."""
    op = mbw.OP_GEMV_BF16
    Wd = inputs_gpu.bf16_weights(0, 11, N, K)
    xd = inputs_gpu.bf16_activations(0, 12, 1, K)[0]
    Y, A = orc.gemm_bf16(host_bits16(Wd).reshape(N, K), host_bits16(xd)[None, :])
    for i, desc in each_plan(op, 1, N, K):
        assert_parity(mbw.gemv_bf16(Wd, xd), Y[0], A[0], f"bf16 {N}x{K} plan {i}: {desc}")
    mbw.autotune(op, 1, N, K)
    assert 0 <= mbw.plan_index(op, 1, N, K) < mbw.plan_candidates(op, 1, N, K)
    assert_parity(mbw.gemv_bf16(Wd, xd), Y[0], A[0], f"bf16 {N}x{K} autotuned: {mbw.plan_describe(op, 1, N, K)}")


@pytest.mark.parametrize("M", [8, 32, 128])
@pytest.mark.parametrize("N,K", [(18944, 3584), (3584, 18944)])
def test_skinny_every_plan_at_qwen_mlp_shapes(orc, M, N, K):
    """Every candidate plan of the skinny BF16 GEMM, then the autotuned plan,
    at the Qwen2.5-7B MLP shapes and batches 8, 32 and 128: every batch row of
    112 sampled weight rows (the first and last 16 and 80 at random)."""
    op = mbw.OP_GEMM_SKINNY_BF16
    rows = np.unique(np.concatenate([np.arange(0, 16), np.arange(N - 16, N),
                                     np.random.default_rng(N + 7 * M).integers(0, N, 80)]))
    Wd = inputs_gpu.bf16_weights(0, 13, N, K)
    Xd = inputs_gpu.bf16_activations(0, 14, M, K)
    Wr = np.stack([gen.bf16_weights(0, 13, N, K, row0=int(r), rows=1)[0] for r in rows])
    Yr, Ar = orc.gemm_bf16(Wr, host_bits16(Xd))
    sel = torch.from_numpy(rows).cuda()
    for i, desc in each_plan(op, M, N, K):
        Y = mbw.gemm_skinny_bf16(Xd, Wd)
        assert_parity(Y[:, sel], Yr, Ar, f"skinny M={M} {N}x{K} plan {i}: {desc}")
    mbw.autotune(op, M, N, K)
    Y = mbw.gemm_skinny_bf16(Xd, Wd)
    assert_parity(Y[:, sel], Yr, Ar, f"skinny M={M} {N}x{K} autotuned: {mbw.plan_describe(op, M, N, K)}")
