"""Expected values and tolerances of the fused GEMV calls, from the fp64
oracle and from the arithmetic alone (no kernel output enters them).

The fusions follow the pages: the RMSNorm prologue folded into the projection
(llm-rs vs vLLM, "Decode: from ~35% to ~70% of the ceiling": norms folded into
the projections), the gated product silu(W.x) * (U.x) and the residual add in
the GEMV epilogue (yalm, sec. 3.3 fusion; TileInfer, SwiGLU in the GEMV
epilogue).

The normalised activation. The kernels form v' = fl(fl(x * r') * g) with
r' = 1 / sqrtf(sum_k x_k^2 / K + eps) in fp32: the squares of bf16 values are
exact in fp32, their sum (any order, all terms positive) is within
gamma_{K-1} = (K-1) u / (1 - (K-1) u) of the exact sum (u = 2^-24); the
division by K, the fp32 eps, the addition, the square root, the reciprocal and
the two products each add at most u. The square root halves the relative error
of its argument, so |v' / v - 1| <= delta(K) = ((K - 1) / 2 + 6) u, plus second-
order terms (covered by a 0.1% margin). The kernel's bf16 activation can
therefore differ from the oracle's bf16(v) only where v lies within
delta(K) |v| of a bf16 rounding boundary (a midpoint between two neighbours),
and there by one bf16 spacing. `near_tie_gap` marks those elements from the
oracle's fp64 v alone.

The tolerance of a fused output (A = sum_k |w_ik xn_k| over the oracle's bf16
activation, T = the marked elements of the row's activation):
  * plain product, with or without the prologue: the stated bar
    2e-3 A + 1e-5, plus allow = sum_{k in T} |w_ik| * spacing_k;
  * residual add: + 2^-8 |R| for the bf16 store of W.x + R;
  * gated product: each fp32 row sum within e = 1e-4 A + allow of the oracle's,
    propagated through silu(a) * b as 1.1 |b| e_a + |silu(a)| e_b + 1.1 e_a e_b
    (|silu'| <= 1.1), then 2^-8 |v| + 1e-5 for the bf16 store.
"""
import numpy as np

from oracle_pins import np_bf16_to_f64, np_round_bf16  # noqa: F401  (np_round_bf16: re-exported)

U32 = 2.0 ** -24
REL_TOL = 2e-3
ABS_TOL = 1e-5
SUM_REL = 1e-4  # fp32 row-sum error of the gated product's two sums


def norm_delta(K: int) -> float:
    """Relative error bound of the kernels' fp32 normalised value before its bf16 rounding."""
    return ((K - 1) / 2.0 + 6.0) * U32 * 1.001


def near_tie_gap(orc, X, g, eps):
    """(M, K): the bf16 spacing at the oracle's normalised value v where v is
    within delta(K) |v| (plus the fp64 oracle's own rounding) of a bf16
    rounding boundary, else 0."""
    V = np.atleast_2d(orc.rmsnorm_f64(X, g, eps))
    K = V.shape[1]
    a = np.abs(V)
    _, e = np.frexp(a)
    sp = np.ldexp(1.0, np.maximum(e - 8, -133))
    mid = np.floor(a / sp) * sp + sp / 2.0
    near = np.abs(a - mid) <= (norm_delta(K) + 8 * 2.0 ** -53) * a
    return np.where(near & (a > 0), sp, 0.0)


def abs_weights(orc, fmt, w):
    """|dequantized W| (N, K) in float64 for fmt in bf16 / g64 / i8 / awq (w = (codes, scales, zeros))."""
    if fmt == "bf16":
        return np.abs(np_bf16_to_f64(w[0]))
    if fmt == "g64":
        N, K = w[0].shape[0], w[0].shape[1] * 2
        return np.abs(orc.dequant_int4_g64(w[0], w[1], N, K))
    if fmt == "awq":
        N, K = w[0].shape[0], w[0].shape[1] * 2
        return np.abs(orc.dequant_int4_awq_g128(w[0], w[1], w[2], N, K))
    return np.abs(w[0].astype(np.float64)) * np.abs(w[1].astype(np.float64))[:, None]


def ogemm(orc, fmt, w, X):
    if fmt == "bf16":
        return orc.gemm_bf16(w[0], X)
    if fmt == "g64":
        return orc.gemm_int4_g64(w[0], w[1], X)
    if fmt == "awq":
        return orc.gemm_int4_awq_g128(w[0], w[1], w[2], X)
    return orc.gemm_int8_pc(w[0], w[1], X)


def fused_reference(orc, fmt, w, wu, X, g, R, eps, out_fp32=False):
    """(oracle value, tolerance, allow / A of the gate product) of a fused
    output; wu (up weights), g (norm weight) and R (residual) may be None.
    out_fp32: the kernel writes its fp32 result (the test hook), so the bf16
    store terms are left out."""
    store = 0.0 if out_fp32 else 2.0 ** -8
    Xn = orc.rmsnorm_bf16(X, g, eps) if g is not None else X
    gap = near_tie_gap(orc, X, g, eps) if g is not None else None

    def product(ww):
        y, a = ogemm(orc, fmt, ww, Xn)
        allow = (abs_weights(orc, fmt, ww) @ gap.T).T if gap is not None else np.zeros_like(y)
        return y, a, allow

    yg, ag, allow_g = product(w)
    if wu is not None:
        yu, au, allow_u = product(wu)
        e_g = SUM_REL * ag + allow_g
        e_u = SUM_REL * au + allow_u
        v = orc.swiglu(yg, yu)
        sg = np.abs(orc.swiglu(yg, np.ones_like(yg)))
        err = 1.1 * np.abs(yu) * e_g + sg * e_u + 1.1 * e_g * e_u
        if R is not None:
            v = orc.add_residual(v, R)
        tol = err + store * np.abs(v) + ABS_TOL
    else:
        v = yg
        tol = REL_TOL * ag + allow_g + ABS_TOL
        if R is not None:
            v = orc.add_residual(v, R)
            tol = tol + store * np.abs(np_bf16_to_f64(R))
    return v, tol, allow_g / np.maximum(ag, 1e-300)
