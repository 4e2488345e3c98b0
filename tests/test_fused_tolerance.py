"""The fused-call tolerance on the CPU: its near-tie marking against an fp32
emulation of the kernels' RMSNorm arithmetic, and a planted norm-factor error
(in the oracle's activation) that it must catch."""
import numpy as np
import pytest

import oracle
from fused_tol import fused_reference, near_tie_gap, norm_delta
from oracle_pins import np_bf16_to_f64, np_round_bf16
from memory_bound_weight_gb300 import inputs as gen

EPS = 1e-5


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    v = np.random.default_rng(3).standard_normal(200000).astype(np.float32) * 3.0
    v[:4] = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -130]  # ties to even, a subnormal
    want = torch.from_numpy(v).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(np_round_bf16(v.astype(np.float64)), want)


def emulate_norm_fp32(X, g, eps, order):
    """bf16 activation as an fp32 kernel forms it: sum of squares in fp32 in
    the given order, / K, + eps, sqrtf, reciprocal, x * r * g, RNE to bf16."""
    Xf = np_bf16_to_f64(X).astype(np.float32)
    gf = np_bf16_to_f64(g).astype(np.float32)
    M, K = Xf.shape
    out = np.empty((M, K))
    for m in range(M):
        sq = Xf[m] * Xf[m]
        if order == "sequential":
            s = np.float32(0)
            for t in sq:
                s = np.float32(s + t)
        elif order == "reversed":
            s = np.float32(0)
            for t in sq[::-1]:
                s = np.float32(s + t)
        else:  # strided per "thread", then a tree over the partials
            part = sq.reshape(-1, 32).sum(axis=0, dtype=np.float32)
            while part.size > 1:
                part = (part[0::2] + part[1::2]).astype(np.float32)
            s = part[0]
        r = np.float32(1.0) / np.sqrt(np.float32(s / np.float32(K) + np.float32(eps)))
        out[m] = np_round_bf16(((Xf[m] * r).astype(np.float32) * gf).astype(np.float32).astype(np.float64))
    return out


@pytest.mark.parametrize("K", [512, 2048, 5632])
def test_every_fp32_rounding_flip_is_marked(orc, K):
    X = gen.bf16_activations(1601, K, 6, K)
    g = gen.bf16_activations(1601, K + 1, 1, K)[0]
    ref = np_bf16_to_f64(orc.rmsnorm_bf16(X, g, EPS))
    gap = near_tie_gap(orc, X, g, EPS)
    assert (gap > 0).mean() < 0.1  # a few percent: delta(K) is 1.6e-5 (K = 512) .. 1.7e-4 (K = 5632)
    for order in ("sequential", "reversed", "tree"):
        got = emulate_norm_fp32(X, g, EPS, order)
        diff = got != ref
        assert np.all(gap[diff] > 0), (order, int(diff.sum()), int((diff & (gap == 0)).sum()))
        assert np.all(np.abs(got - ref)[diff] <= gap[diff])


def test_delta_grows_with_k():
    assert norm_delta(2048) < norm_delta(18944) < 2e-3
    assert norm_delta(2048) == pytest.approx((2047 / 2 + 6) * 2.0 ** -24, rel=2e-3)


def positive_case(seed, N, K):
    """BF16 weights, activations and norm weight with their sign bits cleared:
    every term of every row sum is positive."""
    W = gen.bf16_weights(seed, 0, N, K) & np.uint16(0x7FFF)
    X = gen.bf16_activations(seed, 1, 1, K) & np.uint16(0x7FFF)
    g = gen.bf16_activations(seed, 2, 1, K)[0] & np.uint16(0x7FFF)
    return W, X, g


def test_a_norm_factor_off_by_three_tenths_of_a_percent_fails(orc):
    """Same-sign data, fp32 output (as the same-sign GPU test runs): the
    tolerance stays under 0.25% of |y|, and an activation normalised with a
    factor 0.3% too large (planted in the oracle's own activation) fails on
    almost every output; the correct activation passes."""
    N, K = 300, 2048
    W, X, g = positive_case(1611, N, K)
    v, tol, allow = fused_reference(orc, "bf16", (W, None), None, X, g, None, EPS, out_fp32=True)
    assert np.all(v > 0) and np.max((tol - 1e-5) / v) < 2.5e-3 and allow.max() < 5e-4
    V = orc.rmsnorm_f64(X, g, EPS)
    for factor, want_fail in ((1.003, True), (1.0, False), (0.997, True)):
        xn = np_round_bf16(V * factor)
        bits = (xn.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        y, _ = orc.gemm_bf16(W, bits)
        bad = np.abs(y - v) > tol
        if want_fail:
            assert bad.mean() > 0.95, (factor, bad.mean())
        else:
            assert not bad.any()


@pytest.mark.parametrize("fmt", ["bf16", "g64", "i8"])
def test_same_sign_gated_tolerance_is_tight(orc, fmt):
    """The same-sign GPU case of the gated product: its tolerance is below
    0.25% of the output, so a 0.3% error in the activation (which scales both
    row sums, and the output by at least as much) fails it."""
    N, K = 300, 2048
    W, X, g = positive_case(1621, N, K)
    if fmt == "bf16":
        w, wu = (W, None), (gen.bf16_weights(1621, 5, N, K) & np.uint16(0x7FFF), None)
    elif fmt == "g64":
        w = (gen.int4_codes(1621, 0, N, K) | np.uint8(0x88), gen.f16_group_scales(1621, 0, N, K // 64))
        wu = (gen.int4_codes(1621, 1, N, K) | np.uint8(0x88), gen.f16_group_scales(1621, 1, N, K // 64))
    else:
        w = (np.abs(gen.int8_codes(1621, 0, N, K).astype(np.int16)).astype(np.int8), gen.f32_row_scales(1621, 0, N))
        wu = (np.abs(gen.int8_codes(1621, 1, N, K).astype(np.int16)).astype(np.int8), gen.f32_row_scales(1621, 1, N))
    v, tol, _ = fused_reference(orc, fmt, w, wu, X, g, None, EPS, out_fp32=True)
    assert np.all(v > 0) and np.max((tol - 1e-5) / v) < 2.5e-3
