"""Large and tall matrices on the GPU, every plan against the fp64 oracle.

* Weights past 2^32 bytes, in every format: a 32-bit byte offset anywhere in
  a kernel's addressing would read the wrong rows past the boundary.
* Tall matrices at batch widths whose per-tile partial sums do not fit one
  wave's share of rows in shared memory (INT8 at batch 8, repacked AWQ codes
  at batch 4): the launch then takes more CTAs, in several waves, instead of
  refusing the shape.

Every candidate plan runs; the rows compared are the first and last ones, the
rows on both sides of the first one that starts past 2^32 bytes, and 40 at
random, each for every batch row. The weights come from the device generator,
bit-identical to the host generator
(test_gemv_gpu.py::test_device_generator_matches_host); the oracle gets the
sampled rows from the host generator.
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_parity, host_bits16
from memory_bound_weight_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - the marker keeps these off CPU runs
    pytest.skip("needs a GPU", allow_module_level=True)

import memory_bound_weight_gb300 as mbw  # noqa: E402
from memory_bound_weight_gb300 import inputs_gpu  # noqa: E402

SEED = 2027
GIB4 = 1 << 32


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def sample_rows(N, rowbytes):
    """First and last rows, the rows around the first one that starts past
    2^32 bytes (when the matrix reaches it) and 40 at random."""
    b = GIB4 // rowbytes
    parts = [np.arange(0, 4), np.arange(N - 4, N), np.random.default_rng(N).integers(0, N, 40)]
    if b < N:
        parts.append(np.arange(max(0, b - 4), min(N, b + 5)))
    return np.unique(np.concatenate(parts))


def each_plan(op, M, N, K):
    n = mbw.plan_candidates(op, M, N, K)
    assert n >= 1, (op, M, N, K)
    for i in range(n):
        mbw.plan_select(op, M, N, K, i)
        yield i, mbw.plan_describe(op, M, N, K)


def stack_rows(fn, rows):
    return np.stack([fn(int(r)) for r in rows])


def test_bf16_past_4_gib(orc):
    N, K = 270000, 8192  # 4.42 GB; rows from 262144 on start past 2^32 bytes
    rows = sample_rows(N, 2 * K)
    assert rows.max() * 2 * K >= GIB4
    sel = torch.from_numpy(rows).cuda()
    Wd = inputs_gpu.bf16_weights(SEED, 0, N, K)
    Wr = stack_rows(lambda r: gen.bf16_weights(SEED, 0, N, K, row0=r, rows=1)[0], rows)
    for M in (1, 16, 256):
        Xd = inputs_gpu.bf16_activations(SEED, M, M, K)
        Y, A = orc.gemm_bf16(Wr, host_bits16(Xd))
        if M == 1:
            for i, desc in each_plan(mbw.OP_GEMV_BF16, 1, N, K):
                assert_parity(mbw.gemv_bf16(Wd, Xd[0])[sel], Y[0], A[0], f"bf16 {N}x{K} plan {i}: {desc}")
        else:
            for i, desc in each_plan(mbw.OP_GEMM_SKINNY_BF16, M, N, K):
                assert_parity(mbw.gemm_skinny_bf16(Xd, Wd)[:, sel], Y, A, f"skinny M={M} {N}x{K} plan {i}: {desc}")


def test_int4_g64_past_4_gib(orc):
    N, K = 540000, 16384  # 4.42 GB of codes; rows from 524288 on start past 2^32 bytes
    rows = sample_rows(N, K // 2)
    assert rows.max() * (K // 2) >= GIB4
    sel = torch.from_numpy(rows).cuda()
    cd = inputs_gpu.int4_codes(SEED, 2, N, K)
    sd = inputs_gpu.f16_group_scales(SEED, 2, N, K // 64)
    xd = inputs_gpu.bf16_activations(SEED, 2, 1, K)
    cr = stack_rows(lambda r: gen.int4_codes(SEED, 2, N, K, row0=r, rows=1)[0], rows)
    sr = stack_rows(lambda r: gen.f16_group_scales(SEED, 2, N, K // 64, row0=r, rows=1)[0], rows)
    Y, A = orc.gemm_int4_g64(cr, sr, host_bits16(xd))
    for i, desc in each_plan(mbw.OP_GEMV_INT4_G64, 1, N, K):
        assert_parity(mbw.gemv_int4_g64(cd, sd, xd[0])[sel], Y[0], A[0], f"g64 {N}x{K} plan {i}: {desc}")


def test_int4_awq_past_4_gib(orc):
    """Canonical codes at batch 1, 16 and 64, then the same codes repacked in
    place at batch 1 and 16."""
    N, K = 540000, 16384
    G = K // 128
    rows = sample_rows(N, K // 2)
    sel = torch.from_numpy(rows).cuda()
    cd = inputs_gpu.int4_codes(SEED, 3, N, K)
    sd = inputs_gpu.f16_group_scales(SEED, 3, N, G)
    zd = inputs_gpu.u4_zero_points(SEED, 3, N, G)
    cr = stack_rows(lambda r: gen.int4_codes(SEED, 3, N, K, row0=r, rows=1)[0], rows)
    sr = stack_rows(lambda r: gen.f16_group_scales(SEED, 3, N, G, row0=r, rows=1)[0], rows)
    zr = stack_rows(lambda r: gen.u4_zero_points(SEED, 3, N, G, row0=r, rows=1)[0], rows)
    ref = {}
    for M in (1, 16, 64):
        Xd = inputs_gpu.bf16_activations(SEED, 30 + M, M, K)
        ref[M] = (Xd,) + tuple(orc.gemm_int4_awq_g128(cr, sr, zr, host_bits16(Xd)))
    op = mbw.OP_GEMV_INT4_AWQ_G128
    for M in (1, 16, 64):
        Xd, Y, A = ref[M]
        for i, desc in each_plan(op, M, N, K):
            assert_parity(mbw.gemv_int4_awq_g128(cd, sd, zd, Xd)[:, sel], Y, A, f"awq M={M} {N}x{K} plan {i}: {desc}")
    mbw.repack_int4(cd, out=cd)
    for M in (1, 16):
        Xd, Y, A = ref[M]
        for i, desc in each_plan(op | mbw.REPACKED, M, N, K):
            got = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd, repacked=True)[:, sel]
            assert_parity(got, Y, A, f"awq repacked M={M} {N}x{K} plan {i}: {desc}")


def test_int4_awq_repacked_batch_4_on_a_million_rows(orc):
    """Batch 4 on 1,000,000 rows of repacked codes: one wave's per-tile
    partials do not fit, so every plan here runs in several waves."""
    N, K, M = 1000000, 1024, 4
    G = K // 128
    rows = sample_rows(N, K // 2)
    sel = torch.from_numpy(rows).cuda()
    cd = inputs_gpu.int4_codes(SEED, 4, N, K)
    sd = inputs_gpu.f16_group_scales(SEED, 4, N, G)
    zd = inputs_gpu.u4_zero_points(SEED, 4, N, G)
    Xd = inputs_gpu.bf16_activations(SEED, 4, M, K)
    cr = stack_rows(lambda r: gen.int4_codes(SEED, 4, N, K, row0=r, rows=1)[0], rows)
    sr = stack_rows(lambda r: gen.f16_group_scales(SEED, 4, N, G, row0=r, rows=1)[0], rows)
    zr = stack_rows(lambda r: gen.u4_zero_points(SEED, 4, N, G, row0=r, rows=1)[0], rows)
    Y, A = orc.gemm_int4_awq_g128(cr, sr, zr, host_bits16(Xd))
    mbw.repack_int4(cd, out=cd)
    op = mbw.OP_GEMV_INT4_AWQ_G128 | mbw.REPACKED
    for i, desc in each_plan(op, M, N, K):
        got = mbw.gemv_int4_awq_g128(cd, sd, zd, Xd, repacked=True)[:, sel]
        assert_parity(got, Y, A, f"awq repacked M=4 {N}x{K} plan {i}: {desc}")


def test_int8_past_4_gib_and_tall_batches(orc):
    """Batch 1 and 8 on 4.42 GB of INT8 codes (batch 8 only in several waves),
    then batch 20 (slices of 8) on the tuned plan."""
    N, K = 270000, 16384
    rows = sample_rows(N, K)
    assert rows.max() * K >= GIB4
    sel = torch.from_numpy(rows).cuda()
    qd = inputs_gpu.int8_codes(SEED, 5, N, K)
    sd = inputs_gpu.f32_row_scales(SEED, 5, N)
    qr = stack_rows(lambda r: gen.int8_codes(SEED, 5, N, K, row0=r, rows=1)[0], rows)
    sr = np.concatenate([gen.f32_row_scales(SEED, 5, N, row0=int(r), rows=1) for r in rows])
    op = mbw.OP_GEMV_INT8_PC
    for M in (1, 8):
        Xd = inputs_gpu.bf16_activations(SEED, 50 + M, M, K)
        Y, A = orc.gemm_int8_pc(qr, sr, host_bits16(Xd))
        for i, desc in each_plan(op, M, N, K):
            assert_parity(mbw.gemv_int8_pc(qd, sd, Xd)[:, sel], Y, A, f"int8 M={M} {N}x{K} plan {i}: {desc}")
    Xd = inputs_gpu.bf16_activations(SEED, 70, 20, K)
    Y, A = orc.gemm_int8_pc(qr, sr, host_bits16(Xd))
    mbw.autotune(op, 8, N, K)
    assert_parity(mbw.gemv_int8_pc(qd, sd, Xd)[:, sel], Y, A, f"int8 M=20 {N}x{K} autotuned")


def test_rows_too_long_for_any_gemv_plan(orc):
    """K = 2^20 at batch 1: no GEMV kernel can stage x, so the call is refused
    with MBW_ERR_UNSUPPORTED before any launch and the context stays usable;
    the skinny GEMM from batch 5 on streams X through its ring and computes
    the same rows at batch 8 (every plan)."""
    N, K = 16, 1 << 20
    W, X = gen.bf16_weights(SEED, 6, N, K), gen.bf16_activations(SEED, 6, 8, K)
    Wd = torch.from_numpy(W.view(np.int16)).view(torch.bfloat16).cuda()
    Xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
    assert mbw.plan_candidates(mbw.OP_GEMV_BF16, 1, N, K) == 0
    with pytest.raises(mbw.MbwError) as err:
        mbw.gemv_bf16(Wd, Xd[0])
    assert err.value.status == 5
    Y, A = orc.gemm_bf16(W, X)
    for i, desc in each_plan(mbw.OP_GEMM_SKINNY_BF16, 8, N, K):
        assert_parity(mbw.gemm_skinny_bf16(Xd, Wd), Y, A, f"skinny M=8 {N}x{K} plan {i}: {desc}")
