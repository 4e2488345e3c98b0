"""GPU parity of the load-time INT4 repack and of the AWQ-style GEMV over
repacked codes (llm-rs vs vLLM, sec. 6 and sec. 7: 4-bit weights reordered
once at load time so the unpack hands the multiply its operands in order).

Every call goes through the C ABI. The device repack is compared byte for byte
with the oracle's; the repacked GEMV runs every candidate plan on small
ragged shapes across the batch range (the streaming tensor-core kernels at
M <= 4, the tcgen05 kernel above) and against the oracle on sampled rows at
the Qwen2.5-7B shapes, with the canonical call's tolerance.
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

OP = mbw.OP_GEMV_INT4_AWQ_G128 | mbw.REPACKED


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def awq_case(seed, N, K, M):
    G = K // 128
    return (gen.int4_codes(seed, 0, N, K), gen.f16_group_scales(seed, 0, N, G), gen.u4_zero_points(seed, 0, N, G),
            gen.bf16_activations(seed, 0, M, K))


@pytest.mark.parametrize("N,K", [(1, 8), (3, 24), (7, 128), (33, 640), (257, 3584), (5, 18944)])
def test_repack_bit_exact(orc, N, K):
    c = gen.int4_codes(1500 + N, 0, N, K)
    want = orc.repack_int4(c)
    cd = dev_u8(c)
    got = mbw.repack_int4(cd)
    assert np.array_equal(got.cpu().numpy(), want)
    # in place, and three applications give the codes back
    r = cd.clone()
    for _ in range(3):
        mbw.repack_int4(r, out=r)
    assert torch.equal(r, cd)


def test_repack_every_word_pattern_of_one_nibble(orc):
    """Each of the 8 slots x 16 values alone in a word, in every word of a row."""
    rows = []
    for j in range(8):
        for v in range(16):
            q = np.zeros((1, 64), dtype=np.uint8)
            q[0, j::8] = v
            rows.append(q)
    q = np.concatenate(rows)
    c = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(mbw.repack_int4(dev_u8(c)).cpu().numpy(), orc.repack_int4(c))


def each_plan(M, N, K):
    n = mbw.plan_candidates(OP, M, N, K)
    assert n >= 1
    for i in range(n):
        mbw.plan_select(OP, M, N, K, i)
        yield i, mbw.plan_describe(OP, M, N, K)


@pytest.mark.parametrize("N,K,M", [(3, 128, 1), (45, 384, 1), (129, 1024, 3), (17, 18944, 1), (70, 3584, 2),
                                   (40, 512, 4), (128, 384, 5), (64, 256, 8), (130, 256, 16), (40, 1280, 17),
                                   (300, 1024, 33), (64, 3584, 64), (257, 512, 100)])
def test_repacked_awq_all_plans(orc, N, K, M):
    c, s, z, X = awq_case(1600 + N + M, N, K, M)
    Y, A = orc.gemm_int4_awq_g128(c, s, z, X)
    # the oracle's product over the oracle's repack is the canonical product
    Yr, Ar = orc.gemm_int4_awq_g128(orc.repack_int4(c), s, z, X, repacked=True)
    assert np.array_equal(Y, Yr) and np.array_equal(A, Ar)
    rd = mbw.repack_int4(dev_u8(c))
    sd, zd, Xd = dev_f16(s), dev_u8(z), dev_bf16(X)
    kinds = set()
    for i, desc in each_plan(M, N, K):
        kinds.add(desc.split()[0])
        y = mbw.gemv_int4_awq_g128(rd, sd, zd, Xd, repacked=True)
        assert_parity(y, Y, A, f"repacked awq {M}x{N}x{K} plan {desc}")
    assert "simt" not in kinds
    assert ("tcgen05" in kinds) == (M > 4)


def test_repacked_one_hot_rows_exact(orc):
    """Batch row m = e_{k_m}, fp32 output: every plan returns column k_m of the
    dequantized weights exactly (the unpack and the pairing of codes with x
    are exact; one nonzero product per output)."""
    N, K = 200, 1024
    c, s, z, _ = awq_case(1700, N, K, 1)
    deq = orc.dequant_int4_awq_g128(c, s, z, N, K)
    ks = [0, 1, 2, 3, 5, 7, 8, 127, 128, 513, 1000, 1023] + list(range(16, 36))
    for M in (4, 32):
        X = np.zeros((M, K), dtype=np.uint16)
        for m in range(M):
            X[m, ks[m % len(ks)]] = 0x3F80
        rd = mbw.repack_int4(dev_u8(c))
        sd, zd, Xd = dev_f16(s), dev_u8(z), dev_bf16(X)
        for _, desc in each_plan(M, N, K):
            with mbw.output_fp32():
                y = host_f64(mbw.gemv_int4_awq_g128(rd, sd, zd, Xd, repacked=True))
            for m in range(M):
                assert np.array_equal(y[m], deq[:, ks[m % len(ks)]]), (desc, m)


@pytest.mark.parametrize("N,K", [(18944, 3584), (3584, 18944)])
def test_repacked_qwen_shapes_sampled_rows(orc, N, K):
    """The Qwen2.5-7B MLP shapes at batch 1, 16 and 64, every plan, sampled rows."""
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(N - 8, N),
                                     np.random.default_rng(N + 3).integers(0, N, 64)]))
    G = K // 128
    cd = inputs_gpu.int4_codes(0, 60, N, K)
    sd = inputs_gpu.f16_group_scales(0, 60, N, G)
    zd = inputs_gpu.u4_zero_points(0, 60, N, G)
    rd = mbw.repack_int4(cd)
    del cd
    cr = np.stack([gen.int4_codes(0, 60, N, K, row0=int(r), rows=1)[0] for r in rows])
    sr = np.stack([gen.f16_group_scales(0, 60, N, G, row0=int(r), rows=1)[0] for r in rows])
    zr = np.stack([gen.u4_zero_points(0, 60, N, G, row0=int(r), rows=1)[0] for r in rows])
    sel = torch.from_numpy(rows).cuda()
    for M in (1, 16, 64):
        Xd = inputs_gpu.bf16_activations(0, 61, M, K)
        Y, A = orc.gemm_int4_awq_g128(cr, sr, zr, host_bits16(Xd))
        for _, desc in each_plan(M, N, K):
            y = mbw.gemv_int4_awq_g128(rd, sd, zd, Xd, repacked=True)
            assert_parity(y[:, sel], Y, A, f"repacked awq M={M} {N}x{K} plan {desc}")
