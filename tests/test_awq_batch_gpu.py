"""GPU parity of the batched AWQ-style INT4 kernel on mma.sync (plans
"awq_mma": batches of 5 .. 64 rows per launch, weights streamed once) against
the fp64 oracle (llm-rs vs vLLM, sec. 6 format table: 4-bit codes, fp16 scale
and zero point per 128 weights; sec. 3: batching).

Every call goes through the C ABI. Ragged shapes span several 16-row tiles and
a ragged last tile, 1 .. 8-rank split-K clusters (including ranks whose warps
get no super-block) and batches that need padding or several 32-row slices.
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

OP = mbw.OP_GEMV_INT4_AWQ_G128


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def awq_case(seed, N, K, M):
    G = K // 128
    return (gen.int4_codes(seed, 0, N, K), gen.f16_group_scales(seed, 0, N, G), gen.u4_zero_points(seed, 0, N, G),
            gen.bf16_activations(seed, 0, M, K))


def awqb_plans(op, M, N, K):
    """(index, description) of every batched mma.sync plan of the shape; each selected in turn."""
    n = mbw.plan_candidates(op, M, N, K)
    out = []
    for i in range(n):
        mbw.plan_select(op, M, N, K, i)
        d = mbw.plan_describe(op, M, N, K)
        if d.startswith("awq_mma"):
            out.append((i, d))
    return out


@pytest.mark.parametrize("N,K,M", [(40, 256, 5), (130, 512, 8), (257, 768, 9), (33, 1024, 16), (200, 1280, 17),
                                   (64, 2048, 31), (129, 512, 32), (300, 1024, 33), (17, 3584, 64),
                                   (70, 768, 65), (100, 512, 130)])
@pytest.mark.parametrize("repacked", [False, True])
def test_awq_batch_every_plan_ragged(orc, N, K, M, repacked):
    c, s, z, X = awq_case(1800 + N + M, N, K, M)
    Y, A = orc.gemm_int4_awq_g128(c, s, z, X)
    cd = mbw.repack_int4(dev_u8(c)) if repacked else dev_u8(c)
    sd, zd, Xd = dev_f16(s), dev_u8(z), dev_bf16(X)
    op = OP | (mbw.REPACKED if repacked else 0)
    plans = awqb_plans(op, M, N, K)
    assert plans, "no batched mma.sync plan"
    for i, desc in plans:
        mbw.plan_select(op, M, N, K, i)
        # Y inside a buffer with sentinels on both sides
        buf = torch.full((M * N + 128,), -7.0, dtype=torch.bfloat16, device="cuda")
        y = buf[64:64 + M * N].view(M, N)
        mbw.gemv_int4_awq_g128(cd, sd, zd, Xd, out=y, repacked=repacked)
        assert_parity(y, Y, A, f"awq_mma {M}x{N}x{K} rp={repacked} plan {i}: {desc}")
        assert torch.all(buf[:64] == -7.0) and torch.all(buf[64 + M * N:] == -7.0), desc


@pytest.mark.parametrize("M", [8, 16, 40])
def test_awq_batch_one_hot_rows_exact(orc, M):
    """Batch row m = e_{k_m}, fp32 output: every batched mma.sync plan returns
    column k_m of the dequantized weights exactly."""
    N, K = 200, 1024
    c, s, z, _ = awq_case(1811, N, K, 1)
    deq = orc.dequant_int4_awq_g128(c, s, z, N, K)
    ks = [(37 * m + 5) % K for m in range(M)]
    X = np.zeros((M, K), dtype=np.uint16)
    for m, k in enumerate(ks):
        X[m, k] = 0x3F80
    cd, sd, zd, Xd = dev_u8(c), dev_f16(s), dev_u8(z), dev_bf16(X)
    for i, desc in awqb_plans(OP, M, N, K):
        mbw.plan_select(OP, M, N, K, i)
        with mbw.output_fp32():
            got = host_f64(mbw.gemv_int4_awq_g128(cd, sd, zd, Xd))
        for m, k in enumerate(ks):
            assert np.array_equal(got[m], deq[:, k]), (desc, m, k)


def test_awq_batch_deterministic_and_scaling():
    N, K, M = 1000, 2048, 16
    c, s, z, X = awq_case(1821, N, K, M)
    cd, sd, zd, Xd = dev_u8(c), dev_f16(s), dev_u8(z), dev_bf16(X)
    for i, desc in awqb_plans(OP, M, N, K):
        mbw.plan_select(OP, M, N, K, i)
        with mbw.output_fp32():
            y1 = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)
            y2 = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)
            y4 = mbw.gemv_int4_awq_g128(cd, sd, zd, (Xd.float() * 4).to(torch.bfloat16))
        assert torch.equal(y1, y2), desc
        assert torch.equal(y4, y1 * 4), desc


@pytest.mark.parametrize("M", [16, 33, 64])
@pytest.mark.parametrize("N,K", [(18944, 3584), (3584, 18944), (4608, 3584)])
def test_awq_batch_every_plan_at_qwen_shapes(orc, N, K, M):
    """Every batched mma.sync plan at Qwen2.5-7B shapes (canonical codes),
    every batch row of 96 sampled weight rows, then the autotuned plan."""
    G = K // 128
    rows = np.unique(np.concatenate([np.arange(0, 16), np.arange(N - 16, N),
                                     np.random.default_rng(N + 11 * M).integers(0, N, 64)]))
    cd = inputs_gpu.int4_codes(0, 70, N, K)
    sd = inputs_gpu.f16_group_scales(0, 70, N, G)
    zd = inputs_gpu.u4_zero_points(0, 70, N, G)
    Xd = inputs_gpu.bf16_activations(0, 71, M, K)
    cr = np.stack([gen.int4_codes(0, 70, N, K, row0=int(r), rows=1)[0] for r in rows])
    sr = np.stack([gen.f16_group_scales(0, 70, N, G, row0=int(r), rows=1)[0] for r in rows])
    zr = np.stack([gen.u4_zero_points(0, 70, N, G, row0=int(r), rows=1)[0] for r in rows])
    Yr, Ar = orc.gemm_int4_awq_g128(cr, sr, zr, host_bits16(Xd))
    sel = torch.from_numpy(rows).cuda()
    plans = awqb_plans(OP, M, N, K)
    assert plans
    for i, desc in plans:
        mbw.plan_select(OP, M, N, K, i)
        Y = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)
        assert_parity(Y[:, sel], Yr, Ar, f"awq_mma M={M} {N}x{K} plan {i}: {desc}")
    mbw.autotune(OP, M, N, K)
    Y = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)
    assert_parity(Y[:, sel], Yr, Ar, f"awq M={M} {N}x{K} autotuned: {mbw.plan_describe(OP, M, N, K)}")


def test_batches_sharing_a_plan_key():
    """Batches 9 .. 16 share one plan-cache entry (16 columns): a plan chosen at
    M = 16 serves M = 9 and 12 as well."""
    N, K = 300, 1024
    c, s, z, X = awq_case(1831, N, K, 16)
    o = oracle.load()
    cd, sd, zd = dev_u8(c), dev_f16(s), dev_u8(z)
    i, desc = awqb_plans(OP, 16, N, K)[0]
    mbw.plan_select(OP, 16, N, K, i)
    for M in (16, 9, 12):
        Y, A = o.gemm_int4_awq_g128(c, s, z, X[:M])
        assert mbw.plan_describe(OP, M, N, K) == desc
        assert_parity(mbw.gemv_int4_awq_g128(cd, sd, zd, dev_bf16(X[:M])), Y, A, f"M={M} {desc}")
