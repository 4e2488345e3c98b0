"""GPU parity of the symmetric per-channel INT8 GEMV and quantizer against the
fp64 oracle (TileInfer, "Pushing further with cheating: INT8 quantization").

Every call goes through the C ABI. Small shapes span several CTA tiles and a
ragged tail and run every candidate plan; the Qwen3-4B decode shapes run every
plan on sampled rows. The unpack is checked exactly on every byte value, the
scale application exactly against fp32 rounding of s * q, and the device
quantizer bit for bit against the oracle's.
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_parity, dev_bf16, host_bits16, host_f64
from memory_bound_weight_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - the marker keeps these off CPU runs
    pytest.skip("needs a GPU", allow_module_level=True)

import memory_bound_weight_gb300 as mbw  # noqa: E402
from memory_bound_weight_gb300 import inputs_gpu  # noqa: E402

OP = mbw.OP_GEMV_INT8_PC


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def dev_i8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int8)).cuda()


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def int8_case(seed, N, K, M):
    return gen.int8_codes(seed, 0, N, K), gen.f32_row_scales(seed, 0, N), gen.bf16_activations(seed, 0, M, K)


def each_plan(M, N, K):
    n = mbw.plan_candidates(OP, M, N, K)
    assert n >= 1
    for i in range(n):
        mbw.plan_select(OP, M, N, K, i)
        yield i, mbw.plan_describe(OP, M, N, K)


@pytest.mark.parametrize("N,K,M", [(1, 128, 1), (7, 256, 1), (33, 640, 1), (257, 1024, 2), (1000, 2560, 1),
                                   (96, 9728, 1), (130, 4096, 4), (64, 2560, 8), (45, 384, 9), (17, 12800, 3),
                                   (300, 2048, 5)])
def test_int8_all_plans(orc, N, K, M):
    q, s, X = int8_case(900 + N + M, N, K, M)
    Y, A = orc.gemm_int8_pc(q, s, X)
    qd, sd, Xd = dev_i8(q), dev_f32(s), dev_bf16(X)
    families = set()
    for i, desc in each_plan(M, N, K):
        families.add(desc.split()[0])
        y = mbw.gemv_int8_pc(qd, sd, Xd)
        assert_parity(y, Y, A, f"int8 {M}x{N}x{K} plan {desc}")
        with mbw.output_fp32():
            y32 = mbw.gemv_int8_pc(qd, sd, Xd)
        # fp32 output: only accumulation rounding is left, far inside the bound
        err = np.abs(host_f64(y32) - Y)
        assert np.all(err <= 1e-4 * A + 1e-7), (desc, float(err.max()))
    if K // 128 >= 4:  # the streaming family needs a super-block per warp
        assert "mma2" in families


@pytest.mark.parametrize("N,K,M", [(40, 256, 12), (257, 1024, 16), (130, 2560, 17), (300, 1280, 33), (64, 640, 64),
                                   (33, 9728, 40), (520, 512, 100), (16, 128, 9)])
def test_int8_batched_every_plan(orc, N, K, M):
    """Batches above 8: every plan, the batched mma.sync family (one launch
    per 16 .. 64 rows, every weight read once per launch) among them, against
    the oracle; fp32 output leaves only accumulation rounding."""
    q, s, X = int8_case(1300 + N + M, N, K, M)
    Y, A = orc.gemm_int8_pc(q, s, X)
    qd, sd, Xd = dev_i8(q), dev_f32(s), dev_bf16(X)
    families = set()
    for i, desc in each_plan(M, N, K):
        families.add(desc.split()[0])
        assert_parity(mbw.gemv_int8_pc(qd, sd, Xd), Y, A, f"int8 {M}x{N}x{K} plan {desc}")
        with mbw.output_fp32():
            y32 = mbw.gemv_int8_pc(qd, sd, Xd)
        err = np.abs(host_f64(y32) - Y)
        assert np.all(err <= 1e-4 * A + 1e-7), (desc, float(err.max()))
    assert "int8_mma" in families


def test_int8_batched_deterministic_and_default_plan(orc):
    """The built-in plan of a batch above 8 is the batched family; two calls
    give bitwise the same output."""
    N, K, M = 1000, 2560, 24
    q, s, X = int8_case(1400, N, K, M)
    qd, sd, Xd = dev_i8(q), dev_f32(s), dev_bf16(X)
    assert mbw.plan_describe(OP, M, N, K).startswith("int8_mma")
    y1, y2 = mbw.gemv_int8_pc(qd, sd, Xd), mbw.gemv_int8_pc(qd, sd, Xd)
    assert torch.equal(y1, y2)
    Y, A = orc.gemm_int8_pc(q, s, X)
    assert_parity(y1, Y, A, "int8 M=24 default plan")


@pytest.mark.parametrize("M", [16, 64])
@pytest.mark.parametrize("N,K", [(6144, 2560), (19456, 2560), (2560, 9728)])
def test_int8_batched_every_plan_at_qwen3_4b_shapes(orc, N, K, M):
    """Every plan at batch 16 and 64 on the Qwen3-4B shapes, then the autotuned
    plan; sampled rows, every batch row."""
    rows = np.unique(np.concatenate([np.arange(0, 16), np.arange(N - 16, N),
                                     np.random.default_rng(N + K + M).integers(0, N, 48)]))
    qd = inputs_gpu.int8_codes(0, 60, N, K)
    sd = inputs_gpu.f32_row_scales(0, 60, N)
    Xd = inputs_gpu.bf16_activations(0, 61, M, K)
    q = np.stack([gen.int8_codes(0, 60, N, K, row0=int(r), rows=1)[0] for r in rows])
    s = np.concatenate([gen.f32_row_scales(0, 60, N, row0=int(r), rows=1) for r in rows])
    Y, A = orc.gemm_int8_pc(q, s, host_bits16(Xd))
    sel = torch.from_numpy(rows).cuda()
    for _, desc in each_plan(M, N, K):
        assert_parity(mbw.gemv_int8_pc(qd, sd, Xd)[:, sel], Y, A, f"int8 M={M} {N}x{K} plan {desc}")
    mbw.autotune(OP, M, N, K)
    assert_parity(mbw.gemv_int8_pc(qd, sd, Xd)[:, sel], Y, A, f"int8 M={M} {N}x{K} autotuned")


def test_int8_every_byte_value_exact(orc):
    """Codes q[i][k] = ((i + k) mod 256) - 128 cover all 256 byte values in
    every column; x = one-hot rows, scale 1: with fp32 output each batch row
    returns one column of codes exactly (the unpack is exact, including the
    out-of-format -128)."""
    N, K, M = 256, 512, 8
    i = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    q = (((i + k) % 256) - 128).astype(np.int8)
    s = np.ones(N, dtype=np.float32)
    ks = [0, 1, 2, 3, 127, 128, 300, 511]
    X = np.zeros((M, K), dtype=np.uint16)
    for m, kk in enumerate(ks):
        X[m, kk] = 0x3F80
    qd, sd, Xd = dev_i8(q), dev_f32(s), dev_bf16(X)
    for _, desc in each_plan(M, N, K):
        with mbw.output_fp32():
            y = host_f64(mbw.gemv_int8_pc(qd, sd, Xd))
        for m, kk in enumerate(ks):
            assert np.array_equal(y[m], q[:, kk].astype(np.float64)), (desc, m, kk)


def test_int8_scale_applied_once_exactly(orc):
    """One-hot x: y_i = fp32(s_i * q_ik), the fp32 rounding of the exact
    product the oracle returns (one nonzero product, one scale multiply)."""
    N, K = 300, 1024
    q, s, _ = int8_case(931, N, K, 1)
    deq = s.astype(np.float64)[:, None] * q.astype(np.float64)
    ks = [5, 64, 700, 1023]
    X = np.zeros((len(ks), K), dtype=np.uint16)
    for m, kk in enumerate(ks):
        X[m, kk] = 0x3F80
    qd, sd, Xd = dev_i8(q), dev_f32(s), dev_bf16(X)
    for _, desc in each_plan(len(ks), N, K):
        with mbw.output_fp32():
            y = mbw.gemv_int8_pc(qd, sd, Xd).cpu().numpy()
        for m, kk in enumerate(ks):
            assert np.array_equal(y[m], deq[:, kk].astype(np.float32)), (desc, m, kk)


def test_int8_deterministic_scaling_and_edges(orc):
    N, K = 2560, 4096
    qd = inputs_gpu.int8_codes(3, 40, N, K)
    sd = inputs_gpu.f32_row_scales(3, 40, N)
    xd = inputs_gpu.bf16_activations(3, 41, 1, K)
    with mbw.output_fp32():
        y1 = mbw.gemv_int8_pc(qd, sd, xd[0])
        y2 = mbw.gemv_int8_pc(qd, sd, xd[0])
        assert torch.equal(y1, y2)
        # x * 2^-4 is exact in bf16 and scales every partial sum exactly
        y3 = mbw.gemv_int8_pc(qd, sd, (xd[0].float() * 2.0 ** -4).to(torch.bfloat16))
        assert torch.equal(y3, y1 * 2.0 ** -4)
        # scales * 2 doubles the output exactly
        y4 = mbw.gemv_int8_pc(qd, sd * 2.0, xd[0])
        assert torch.equal(y4, y1 * 2.0)
    # K == 0 writes zeros; N == 0 and M == 0 launch nothing
    y = torch.full((5,), 7.0, dtype=torch.bfloat16, device="cuda")
    mbw.gemv_int8_pc(torch.empty((5, 0), dtype=torch.int8, device="cuda"), torch.ones(5, device="cuda"),
                     torch.empty((0,), dtype=torch.bfloat16, device="cuda"), out=y)
    assert torch.count_nonzero(y.float()) == 0
    before = mbw.launch_count()
    mbw.gemv_int8_pc(torch.empty((0, 128), dtype=torch.int8, device="cuda"), torch.ones(0, device="cuda"),
                     torch.zeros((128,), dtype=torch.bfloat16, device="cuda"))
    assert mbw.launch_count() == before
    with pytest.raises(mbw.MbwError):
        mbw.gemv_int8_pc(dev_i8(np.zeros((4, 192), dtype=np.int8)), torch.ones(4, device="cuda"),
                         torch.zeros((192,), dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("N,K", [(6144, 2560), (2560, 4096), (19456, 2560), (2560, 9728)])
def test_int8_every_plan_at_qwen3_4b_shapes(orc, N, K):
    """Every candidate plan at the Qwen3-4B decode shapes, on sampled rows
    (first and last tiles plus random rows)."""
    rows = np.unique(np.concatenate([np.arange(0, 16), np.arange(N - 16, N),
                                     np.random.default_rng(N + K).integers(0, N, 64)]))
    qd = inputs_gpu.int8_codes(0, 50, N, K)
    sd = inputs_gpu.f32_row_scales(0, 50, N)
    xd = inputs_gpu.bf16_activations(0, 51, 1, K)
    q = np.stack([gen.int8_codes(0, 50, N, K, row0=int(r), rows=1)[0] for r in rows])
    s = np.concatenate([gen.f32_row_scales(0, 50, N, row0=int(r), rows=1) for r in rows])
    Y, A = orc.gemm_int8_pc(q, s, host_bits16(xd))
    sel = torch.from_numpy(rows).cuda()
    families = set()
    for _, desc in each_plan(1, N, K):
        families.add(desc.split()[0])
        y = mbw.gemv_int8_pc(qd, sd, xd[0])
        assert_parity(y[sel], Y[0], A[0], f"int8 {N}x{K} plan {desc}")
    assert {"mma2", "bulk"} <= families  # the register-ring and the bulk-fed streaming kernels both ran


def test_int8_lm_head_sampled_rows(orc):
    N, K = 151936, 2560
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(N - 8, N),
                                     np.random.default_rng(7).integers(0, N, 48)]))
    qd = inputs_gpu.int8_codes(0, 52, N, K)
    sd = inputs_gpu.f32_row_scales(0, 52, N)
    xd = inputs_gpu.bf16_activations(0, 53, 1, K)
    y = mbw.gemv_int8_pc(qd, sd, xd[0])
    q = np.stack([gen.int8_codes(0, 52, N, K, row0=int(r), rows=1)[0] for r in rows])
    s = np.concatenate([gen.f32_row_scales(0, 52, N, row0=int(r), rows=1) for r in rows])
    Y, A = orc.gemm_int8_pc(q, s, host_bits16(xd))
    assert_parity(y[torch.from_numpy(rows).cuda()], Y[0], A[0], "int8 lm_head sampled")


def test_device_int8_generators_match_host():
    q = inputs_gpu.int8_codes(5, 7, 33, 640).cpu().numpy()
    assert np.array_equal(q, gen.int8_codes(5, 7, 33, 640))
    s = inputs_gpu.f32_row_scales(5, 7, 1001).cpu().numpy()
    assert np.array_equal(s.view(np.uint32), gen.f32_row_scales(5, 7, 1001).view(np.uint32))


# ------------------------------------------------------------- quantizer ----
@pytest.mark.parametrize("N,K", [(37, 300), (256, 2560), (5, 1), (64, 9728)])
def test_quantizer_bit_exact(orc, N, K):
    W = gen.bf16_weights(960 + K, 0, N, K)
    W[0] = 0                              # an all-zero row
    if N > 2:
        W[1] = W[1] & 0x807F              # tiny (subnormal) values
        W[2, K // 2] = 0xC2FE             # a negative maximum
    qr, sr = orc.quantize_int8_pc(W)
    qd, sd = mbw.quantize_int8_pc(dev_bf16(W))
    assert np.array_equal(sd.cpu().numpy().view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(qd.cpu().numpy(), qr)


def test_quantize_then_gemv(orc):
    """The load-time step and the decode GEMV together: quantize BF16 weights
    on the device, run the GEMV, compare with the oracle on the oracle's own
    quantization of the same weights."""
    N, K = 1000, 2560
    W = gen.bf16_weights(971, 0, N, K)
    X = gen.bf16_activations(971, 0, 2, K)
    qr, sr = orc.quantize_int8_pc(W)
    Y, A = orc.gemm_int8_pc(qr, sr, X)
    qd, sd = mbw.quantize_int8_pc(dev_bf16(W))
    y = mbw.gemv_int8_pc(qd, sd, dev_bf16(X))
    assert_parity(y, Y, A, "quantize + gemv")
