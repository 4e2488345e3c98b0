"""GPU parity of the fused GEMV calls (gemv_fused) against the fp64 oracle.

The fusions follow the pages: an RMSNorm prologue folded into the projection
(llm-rs vs vLLM, "norms folded into the projections"), the gated SiLU product
silu(W1.x) * (W3.x) and the residual add in the GEMV epilogue (yalm, sec. 3.3;
TileInfer: SwiGLU in the GEMV epilogue). Every combination runs every
candidate plan (mma2 and latency families) on ragged shapes of each format.

Tolerance (fused_tol.py, from the arithmetic and oracle-only data): the stated
bar 2e-3 * sum_k |w_ik xn_k| + 1e-5 on the product, plus one bf16 spacing of
|w_ik| for each activation element the oracle marks as lying within the
kernels' fp32 error bound of a bf16 rounding boundary; the gated product
propagates its two fp32 row sums through silu(a) * b; stores add their bf16
rounding.
"""
import numpy as np
import pytest

import oracle
from fused_tol import fused_reference, near_tie_gap
from gpu_util import dev_bf16, dev_f16, dev_u8, host_f64
from memory_bound_weight_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - the marker keeps these off CPU runs
    pytest.skip("needs a GPU", allow_module_level=True)

import memory_bound_weight_gb300 as mbw  # noqa: E402

COMBOS = {"norm": (1, 0, 0), "glu": (0, 1, 0), "res": (0, 0, 1), "norm+glu": (1, 1, 0), "norm+res": (1, 0, 1),
          "glu+res": (0, 1, 1), "all": (1, 1, 1)}
SHAPES = [("bf16", 33, 512, 1), ("bf16", 130, 1024, 3), ("g64", 45, 512, 1), ("g64", 300, 2048, 1),
          ("i8", 77, 640, 1), ("i8", 257, 2560, 2)]
OPS = {"bf16": mbw.OP_GEMV_BF16, "g64": mbw.OP_GEMV_INT4_G64, "i8": mbw.OP_GEMV_INT8_PC}
EPS = 1e-5


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def weights(fmt, seed, mi, N, K):
    """Host arrays and device tensors of one weight matrix."""
    if fmt == "bf16":
        W = gen.bf16_weights(seed, mi, N, K)
        return (W, None), (dev_bf16(W), None)
    if fmt == "g64":
        c, s = gen.int4_codes(seed, mi, N, K), gen.f16_group_scales(seed, mi, N, K // 64)
        return (c, s), (dev_u8(c), dev_f16(s))
    q, s = gen.int8_codes(seed, mi, N, K), gen.f32_row_scales(seed, mi, N)
    return (q, s), (torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())


def reference(orc, fmt, w, wu, X, g, R):
    """Oracle value and tolerance of the fused output."""
    v, tol, _ = fused_reference(orc, fmt, w, wu, X, g, R, EPS)
    return v, tol


def check(y, v, tol, what):
    got = host_f64(y).reshape(v.shape)
    bad = np.abs(got - v) > tol
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; first {i}: got {got[i]!r} "
                             f"want {v[i]!r} tol {tol[i]!r}")


def fused_op(op, norm, glu, res):
    return op | (mbw.FUSE_NORM if norm else 0) | (mbw.FUSE_GLU if glu else 0) | (mbw.FUSE_RESIDUAL if res else 0)


@pytest.mark.parametrize("combo", sorted(COMBOS))
@pytest.mark.parametrize("fmt,N,K,M", SHAPES, ids=[f"{s[0]}-{s[1]}x{s[2]}-M{s[3]}" for s in SHAPES])
def test_fused_every_plan(orc, fmt, N, K, M, combo):
    norm, glu, res = COMBOS[combo]
    seed = 1300 + N + K
    w, wd = weights(fmt, seed, 0, N, K)
    wu, wud = weights(fmt, seed, 1, N, K) if glu else ((None, None), (None, None))
    X = gen.bf16_activations(seed, 2, M, K)
    g = gen.bf16_activations(seed, 3, 1, K)[0] if norm else None
    R = gen.bf16_activations(seed, 4, M, N) if res else None
    v, tol = reference(orc, fmt, w, wu if glu else None, X, g, R)
    Xd = dev_bf16(X)
    gd = dev_bf16(g) if norm else None
    Rd = dev_bf16(R) if res else None
    op = fused_op(OPS[fmt], norm, glu, res)
    n = mbw.plan_candidates(op, M, N, K)
    assert n >= 1
    for i in range(n):
        mbw.plan_select(op, M, N, K, i)
        desc = mbw.plan_describe(op, M, N, K)
        y = mbw.gemv_fused(OPS[fmt], wd[0], wd[1], Xd, norm_weight=gd, norm_eps=EPS, residual=Rd,
                           up_weights=wud[0], up_scales=wud[1])
        check(y, v, tol, f"{fmt} {combo} {M}x{N}x{K} plan {desc}")


def test_rmsnorm_prologue_matches_the_oracle_bf16(orc):
    """W = identity (BF16), fp32 output: y is the kernel's own normalised bf16
    x. It equals the oracle's RMSNorm except where the fp32 factor rounds to
    the other bf16 neighbour: at most one ulp, rarely, and only on elements
    the oracle marks as near a rounding boundary."""
    K = 1024
    X = gen.bf16_activations(1401, 0, 4, K)
    g = gen.bf16_activations(1401, 1, 1, K)[0]
    ref = orc.rmsnorm_bf16(X, g, EPS)
    gap = near_tie_gap(orc, X, g, EPS)
    eye = torch.eye(K, dtype=torch.bfloat16, device="cuda")
    op = fused_op(mbw.OP_GEMV_BF16, 1, 0, 0)
    for i in range(mbw.plan_candidates(op, 4, K, K)):
        mbw.plan_select(op, 4, K, K, i)
        with mbw.output_fp32():
            y = mbw.gemv_fused(mbw.OP_GEMV_BF16, eye, None, dev_bf16(X), norm_weight=dev_bf16(g), norm_eps=EPS)
        got = y.to(torch.bfloat16).cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(host_f64(y), host_f64(y.to(torch.bfloat16)))  # y is a bf16 value
        diff = np.abs(got.astype(np.int32) - ref.astype(np.int32))
        assert diff.max() <= 1 and (diff > 0).mean() < 0.01, (mbw.plan_describe(op, 4, K, K), int((diff > 0).sum()))
        # and only where the oracle's fp64 value lies within the fp32 error bound of a rounding boundary
        assert np.all(gap[diff > 0] > 0), (mbw.plan_describe(op, 4, K, K), int(((diff > 0) & (gap == 0)).sum()))


def test_residual_in_place_and_determinism(orc):
    N, K, M = 2560, 2048, 2
    w, wd = weights("i8", 1411, 0, N, K)
    X = gen.bf16_activations(1411, 2, M, K)
    R = gen.bf16_activations(1411, 4, M, N)
    v, tol = reference(orc, "i8", w, None, X, None, R)
    Y = dev_bf16(R).clone()
    mbw.gemv_fused(mbw.OP_GEMV_INT8_PC, wd[0], wd[1], dev_bf16(X), out=Y, residual=Y)  # y += W.x in place
    check(Y, v, tol, "in-place residual")
    # the same call twice gives bitwise the same result
    a = mbw.gemv_fused(mbw.OP_GEMV_INT8_PC, wd[0], wd[1], dev_bf16(X), residual=dev_bf16(R))
    b = mbw.gemv_fused(mbw.OP_GEMV_INT8_PC, wd[0], wd[1], dev_bf16(X), residual=dev_bf16(R))
    assert torch.equal(a, b)


def test_fused_tinyllama_shapes_sampled_rows(orc):
    """The TinyLlama decode step's fused calls: q/k/v with the attention
    RMSNorm, gate/up (5632 + 5632 rows) with the MLP RMSNorm and SwiGLU, down
    and o with the residual add; every row compared."""
    K = 2048
    X = gen.bf16_activations(1421, 0, 1, K)
    g = gen.bf16_activations(1421, 1, 1, K)[0]
    cases = [("qkv", 2560, 2048, (1, 0, 0)), ("gate_up", 5632, 2048, (1, 1, 0)), ("o", 2048, 2048, (0, 0, 1)),
             ("down", 2048, 5632, (0, 0, 1))]
    for name, N, Kc, (norm, glu, res) in cases:
        Xc = X if Kc == K else gen.bf16_activations(1421, 5, 1, Kc)
        w, wd = weights("g64", 1421, 10, N, Kc)
        wu, wud = weights("g64", 1421, 11, N, Kc) if glu else ((None, None), (None, None))
        R = gen.bf16_activations(1421, 6, 1, N) if res else None
        v, tol = reference(orc, "g64", w, wu if glu else None, Xc, g if norm else None, R)
        mbw.autotune(fused_op(mbw.OP_GEMV_INT4_G64, norm, glu, res), 1, N, Kc)
        y = mbw.gemv_fused(mbw.OP_GEMV_INT4_G64, wd[0], wd[1], dev_bf16(Xc[0]),
                           norm_weight=dev_bf16(g) if norm else None, norm_eps=EPS,
                           residual=dev_bf16(R[0]) if res else None, up_weights=wud[0], up_scales=wud[1])
        check(y, v[0], tol[0], f"tinyllama {name}")


@pytest.mark.parametrize("combo", ["norm", "norm+glu"])
@pytest.mark.parametrize("fmt", ["bf16", "g64", "i8"])
def test_fused_norm_same_sign_every_plan(orc, fmt, combo):
    """Weights, activations and norm weight all positive, fp32 output: every
    term of every row sum is positive, so |y| = sum_k |w_ik xn_k| and the
    tolerance is below 0.25% of |y| (asserted). A norm factor 0.3% off would
    scale every output by 1.003 and fail (test_fused_tolerance.py plants
    exactly that in the oracle's activation)."""
    norm, glu, res = COMBOS[combo]
    N, K, M = 300, 2048, 1
    seed = 1700 + len(fmt)
    (w, wd) = positive_weights(fmt, seed, 0, N, K)
    (wu, wud) = positive_weights(fmt, seed, 1, N, K) if glu else (None, (None, None))
    X = gen.bf16_activations(seed, 2, M, K) & np.uint16(0x7FFF)
    g = gen.bf16_activations(seed, 3, 1, K)[0] & np.uint16(0x7FFF)
    v, tol, allow = fused_reference(orc, fmt, w, wu, X, g, None, EPS, out_fp32=True)
    assert np.all(v > 0) and np.max((tol - 1e-5) / v) < 2.5e-3 and allow.max() < 5e-4
    Xd, gd = dev_bf16(X), dev_bf16(g)
    op = fused_op(OPS[fmt], norm, glu, res)
    for i in range(mbw.plan_candidates(op, M, N, K)):
        mbw.plan_select(op, M, N, K, i)
        with mbw.output_fp32():
            y = mbw.gemv_fused(OPS[fmt], wd[0], wd[1], Xd, norm_weight=gd, norm_eps=EPS, up_weights=wud[0],
                               up_scales=wud[1])
        check(y, v, tol, f"same-sign {fmt} {combo} plan {mbw.plan_describe(op, M, N, K)}")


def positive_weights(fmt, seed, mi, N, K):
    """A weight matrix with every dequantized weight >= 0: bf16 sign bits
    cleared, INT4 codes >= 8 (w = (q - 8) s), INT8 codes |q|."""
    if fmt == "bf16":
        W = gen.bf16_weights(seed, mi, N, K) & np.uint16(0x7FFF)
        return (W, None), (dev_bf16(W), None)
    if fmt == "g64":
        c = gen.int4_codes(seed, mi, N, K) | np.uint8(0x88)
        s = gen.f16_group_scales(seed, mi, N, K // 64)
        return (c, s), (dev_u8(c), dev_f16(s))
    q = np.abs(gen.int8_codes(seed, mi, N, K).astype(np.int16)).astype(np.int8)
    s = gen.f32_row_scales(seed, mi, N)
    return (q, s), (torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())


# ------------------------------------------------ AWQ-style INT4 (group 128) ----
def awq_weights(seed, mi, N, K, repacked):
    G = K // 128
    c = gen.int4_codes(seed, mi, N, K)
    s, z = gen.f16_group_scales(seed, mi, N, G), gen.u4_zero_points(seed, mi, N, G)
    cd = mbw.repack_int4(dev_u8(c)) if repacked else dev_u8(c)
    return (c, s, z), (cd, dev_f16(s), dev_u8(z))


AWQ_SHAPES = [(45, 1024, 1), (300, 2048, 1), (130, 1280, 3), (77, 1024, 4), (40, 2048, 9)]


def test_fused_awq_needs_a_super_block_per_warp():
    """The fused AWQ calls run on the streaming tensor-core kernel, whose
    smallest instantiation has 4 warps along K, each needing a 256-k
    super-block: below K = 1024 a fused call is refused as unsupported (a
    plain call still runs)."""
    N, K = 40, 512
    _, wd = awq_weights(1971, 0, N, K, False)
    x = dev_bf16(gen.bf16_activations(1971, 2, 1, K)[0])
    g = dev_bf16(gen.bf16_activations(1971, 3, 1, K)[0])
    with pytest.raises(mbw.MbwError) as e:
        mbw.gemv_fused_awq_g128(wd[0], wd[1], wd[2], x, norm_weight=g)
    assert e.value.status == 5  # MBW_ERR_UNSUPPORTED
    assert mbw.gemv_fused_awq_g128(wd[0], wd[1], wd[2], x).shape == (N,)


@pytest.mark.parametrize("repacked", [False, True])
@pytest.mark.parametrize("combo", sorted(COMBOS))
@pytest.mark.parametrize("N,K,M", AWQ_SHAPES, ids=[f"{n}x{k}-M{m}" for n, k, m in AWQ_SHAPES])
def test_fused_awq_every_plan(orc, N, K, M, combo, repacked):
    """gemv_fused_awq_g128, every fusion combination, every plan (the streaming
    tensor-core kernel; batches above 4 in slices of 4), canonical and repacked
    codes, against the oracle under the fused tolerance."""
    norm, glu, res = COMBOS[combo]
    seed = 1900 + N + K
    w, wd = awq_weights(seed, 0, N, K, repacked)
    wu, wud = awq_weights(seed, 1, N, K, repacked) if glu else (None, (None, None, None))
    X = gen.bf16_activations(seed, 2, M, K)
    g = gen.bf16_activations(seed, 3, 1, K)[0] if norm else None
    R = gen.bf16_activations(seed, 4, M, N) if res else None
    v, tol, _ = fused_reference(orc, "awq", w, wu, X, g, R, EPS)
    Xd = dev_bf16(X)
    gd = dev_bf16(g) if norm else None
    Rd = dev_bf16(R) if res else None
    op = fused_op(mbw.OP_GEMV_INT4_AWQ_G128, norm, glu, res) | (mbw.REPACKED if repacked else 0)
    n = mbw.plan_candidates(op, M, N, K)
    assert n >= 1
    for i in range(n):
        mbw.plan_select(op, M, N, K, i)
        desc = mbw.plan_describe(op, M, N, K)
        y = mbw.gemv_fused_awq_g128(wd[0], wd[1], wd[2], Xd, norm_weight=gd, norm_eps=EPS, residual=Rd,
                                    up_weights=wud[0], up_scales=wud[1], up_zeros=wud[2], repacked=repacked)
        check(y, v, tol, f"awq {combo} rp={repacked} {M}x{N}x{K} plan {desc}")


def test_fused_awq_same_sign_norm(orc):
    """Same-sign AWQ data (codes >= 8 > zero points, so every dequantized
    weight is > 0), fp32 output: the tolerance is below 0.25% of |y| and every
    plan meets it, so a 0.3% norm-factor error would fail."""
    N, K = 300, 2048
    G = K // 128
    c = gen.int4_codes(1951, 0, N, K) | np.uint8(0x88)  # codes 8 .. 15
    s = gen.f16_group_scales(1951, 0, N, G)
    z = gen.u4_zero_points(1951, 0, N, G) & np.uint8(0x77)  # zero points 0 .. 7
    X = gen.bf16_activations(1951, 2, 1, K) & np.uint16(0x7FFF)
    g = gen.bf16_activations(1951, 3, 1, K)[0] & np.uint16(0x7FFF)
    v, tol, allow = fused_reference(orc, "awq", (c, s, z), None, X, g, None, EPS, out_fp32=True)
    assert np.all(v > 0) and np.max((tol - 1e-5) / v) < 2.5e-3 and allow.max() < 5e-4
    op = fused_op(mbw.OP_GEMV_INT4_AWQ_G128, 1, 0, 0)
    for i in range(mbw.plan_candidates(op, 1, N, K)):
        mbw.plan_select(op, 1, N, K, i)
        with mbw.output_fp32():
            y = mbw.gemv_fused_awq_g128(dev_u8(c), dev_f16(s), dev_u8(z), dev_bf16(X[0]), norm_weight=dev_bf16(g),
                                        norm_eps=EPS)
        check(y, v[0], tol[0], f"same-sign awq plan {mbw.plan_describe(op, 1, N, K)}")


def test_fused_awq_qwen_shapes_sampled_rows(orc):
    """The Qwen2.5-7B decode layer's fused AWQ calls at batch 1 on the
    autotuned plans, codes repacked at load time: q/k/v with the RMSNorm,
    gate/up (18944 + 18944 rows) with the RMSNorm and SwiGLU, o and down with
    the residual add; sampled rows."""
    K0 = 3584
    X = gen.bf16_activations(1961, 0, 1, K0)
    g = gen.bf16_activations(1961, 1, 1, K0)[0]
    cases = [("qkv", 4608, K0, (1, 0, 0)), ("gate_up", 18944, K0, (1, 1, 0)), ("o", 3584, K0, (0, 0, 1)),
             ("down", 3584, 18944, (0, 0, 1))]
    for name, N, K, (norm, glu, res) in cases:
        Xc = X if K == K0 else gen.bf16_activations(1961, 5, 1, K)
        rows = np.unique(np.concatenate([np.arange(0, 16), np.arange(N - 16, N),
                                         np.random.default_rng(N + K).integers(0, N, 48)]))
        w, wd = awq_weights(1961, 10, N, K, True)
        wu, wud = awq_weights(1961, 11, N, K, True) if glu else (None, (None, None, None))
        R = gen.bf16_activations(1961, 6, 1, N) if res else None
        wr = tuple(a[rows] for a in w)
        wur = tuple(a[rows] for a in wu) if glu else None
        v, tol, _ = fused_reference(orc, "awq", wr, wur, Xc, g if norm else None, R[:, rows] if res else None, EPS)
        op = fused_op(mbw.OP_GEMV_INT4_AWQ_G128, norm, glu, res) | mbw.REPACKED
        mbw.autotune(op, 1, N, K)
        y = mbw.gemv_fused_awq_g128(wd[0], wd[1], wd[2], dev_bf16(Xc[0]), norm_weight=dev_bf16(g) if norm else None,
                                    norm_eps=EPS, residual=dev_bf16(R[0]) if res else None, up_weights=wud[0],
                                    up_scales=wud[1], up_zeros=wud[2], repacked=True)
        check(y[torch.from_numpy(rows).cuda()], v[0], tol[0], f"qwen awq {name} ({mbw.plan_describe(op, 1, N, K)})")
