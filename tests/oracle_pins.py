"""Checks that pin the fp64 oracle to facts outside itself.

Each pin is a function taking a loaded ``oracle.Oracle`` and raising
AssertionError on failure. They are run against the real oracle
(test_oracle_pins.py) and against copies of oracle.c with planted mistakes
(test_oracle_mutants.py), which every plausible mistake must fail.

What each pin compares with:
  * number formats: numpy's float16 and torch's bfloat16 conversions (library
    routines), exhaustively over all 65,536 bit patterns;
  * dequant: hand-worked values in tests/golden/int4_dequant_hand.txt and an
    independent vectorised numpy unpack;
  * products: exact rational arithmetic (fractions.Fraction) on tiny shapes,
    and numpy's fp64 matmul of the numpy dequant;
  * invariants: power-of-two scaling, identity / one-hot weights, one-hot x,
    consistent permutation of k, batch = separate calls, linearity on
    disjoint supports;
  * load-time INT4 repack: hand-worked words and one-hot products in
    tests/golden/int4_repack_hand.txt, the permutation's order (three
    applications are the identity), and equality with the canonical product;
  * INT8 per-channel: hand-worked values in tests/golden/int8_pc_hand.txt
    (GEMV and quantizer, including ties and a non-dyadic scale), exact
    rational products, numpy's matmul, scale linearity, and the quantizer's
    properties stated on the page (largest entry on +-127, every entry
    within half a scale).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

from memory_bound_weight_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------ helpers ----
def np_bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """bfloat16 bits -> float64 through numpy's binary32 decoder."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def np_f16_to_f64(h: np.ndarray) -> np.ndarray:
    return np.asarray(h, dtype=np.uint16).view(np.float16).astype(np.float64)


def np_unpack_codes(codes: np.ndarray) -> np.ndarray:
    """(N, K/2) packed bytes -> (N, K) codes, low nibble first."""
    lo = codes & 0x0F
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1).astype(np.int64)


def np_pack_codes(q: np.ndarray) -> np.ndarray:
    q = np.asarray(q, dtype=np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def np_dequant_g64(codes, scales) -> np.ndarray:
    q = np_unpack_codes(codes)
    s = np.repeat(np_f16_to_f64(scales), 64, axis=1)
    return (q - 8) * s


def np_dequant_awq(codes, scales, zeros, K) -> np.ndarray:
    G = K // 128
    q = np_unpack_codes(codes)
    z = np_unpack_codes(zeros)[:, :G]
    s = np_f16_to_f64(scales)
    return (q - np.repeat(z, 128, axis=1)) * np.repeat(s, 128, axis=1)


def f64_to_bf16_exact(v: np.ndarray) -> np.ndarray:
    """bf16 bits of values known to be exactly representable in bf16."""
    f = np.asarray(v, dtype=np.float32)
    assert np.array_equal(f.astype(np.float64), np.asarray(v, dtype=np.float64))
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


def np_round_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even, computed
    exactly in float64 (8 significant bits; spacing 2^-133 below 2^-126).
    Returns float64. Finite inputs inside the bf16 range only."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, e = np.frexp(a)  # a = f * 2^e, f in [0.5, 1)
    spacing = np.ldexp(1.0, np.maximum(e - 8, -133))
    return np.sign(v) * np.rint(a / spacing) * spacing


def sum_bound(K: int, yabs: np.ndarray) -> np.ndarray:
    """Bound on the rounding error of a K-term fp64 sum with sum |terms| = yabs."""
    return K * 2.0 ** -53 * yabs + 1e-300


def small_bf16_case(seed, N, K, M=1):
    W = gen.bf16_weights(seed, 0, N, K)
    X = gen.bf16_activations(seed, 0, M, K)
    return W, X


def small_g64_case(seed, N, K, M=1):
    c = gen.int4_codes(seed, 0, N, K)
    s = gen.f16_group_scales(seed, 0, N, K // 64)
    X = gen.bf16_activations(seed, 0, M, K)
    return c, s, X


def small_awq_case(seed, N, K, M=1):
    G = K // 128
    c = gen.int4_codes(seed, 0, N, K)
    s = gen.f16_group_scales(seed, 0, N, G)
    z = gen.u4_zero_points(seed, 0, N, G)
    X = gen.bf16_activations(seed, 0, M, K)
    return c, s, z, X


def small_int8_case(seed, N, K, M=1):
    q = gen.int8_codes(seed, 0, N, K)
    s = gen.f32_row_scales(seed, 0, N)
    X = gen.bf16_activations(seed, 0, M, K)
    return q, s, X


def np_dequant_int8(q, s) -> np.ndarray:
    return np.asarray(s, dtype=np.float32).astype(np.float64)[:, None] * np.asarray(q, dtype=np.int8).astype(np.float64)


def load_int8_fixture():
    gemv, quant = [], []
    with open(os.path.join(GOLDEN, "int8_pc_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "gemv":
                _, N, K, codes, scales, x, row, expect = parts
                gemv.append(dict(N=int(N), K=int(K), codes=[int(v) for v in codes.split(",")],
                                 scales=[int(v, 16) for v in scales.split(",")],
                                 x=[int(v, 16) for v in x.split(",")], row=int(row), expect=Fraction(expect)))
            else:
                _, K, w, scale, codes = parts
                quant.append(dict(K=int(K), w=[int(v, 16) for v in w.split(",")], scale=int(scale, 16),
                                  codes=[int(v) for v in codes.split(",")]))
    return gemv, quant


def load_fusion_fixture():
    norm, glu, res = [], [], []
    with open(os.path.join(GOLDEN, "fusion_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            p = line.split()
            if p[0] == "rmsnorm":
                norm.append(dict(K=int(p[1]), eps=float(p[2]), x=[int(v, 16) for v in p[3].split(",")],
                                 g=[int(v, 16) for v in p[4].split(",")], expect=[int(v, 16) for v in p[5].split(",")]))
            elif p[0] == "swiglu":
                glu.append((float(p[1]), float(p[2]), float(p[3])))
            else:
                res.append((float(p[1]), int(p[2], 16), float(p[3])))
    return norm, glu, res


# --------------------------------------------------------------- pins ----
def pin_f16_decoder_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint16)
    ref = np_f16_to_f64(bits)
    got = np.array([o.f16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_bf16_decoder_exhaustive(o):
    import torch

    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([o.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_bf16_rounding(o):
    """double -> bf16 RNE equals torch's float32 -> bfloat16 on float32 inputs,
    including exact ties and subnormals."""
    import torch

    rng = np.random.default_rng(7)
    f = rng.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    ties = ((rng.integers(0, 0x7F00, 500).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    sub = (rng.integers(1, 2 ** 23, 500).astype(np.uint32)).view(np.float32)
    big = np.array([3.3e38, -3.3e38, 1.0, -0.0, 0.0, 2.0 ** -130], dtype=np.float32)
    allf = np.concatenate([f, ties, sub, big])
    ref = torch.from_numpy(allf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([o.double_to_bf16(float(v)) for v in allf], dtype=np.uint16)
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:5]


def _parse_hex_list(spec: str) -> list[int]:
    """'9F*32,00*2' -> bytes; '1D1F,2000' -> words."""
    out = []
    for part in spec.split(","):
        if "*" in part:
            v, n = part.split("*")
            out += [int(v, 16)] * int(n)
        else:
            out.append(int(part, 16))
    return out


def load_dequant_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "int4_dequant_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            fmt, N, K, codes, scales, zeros, i, k, expect = line.split()
            rows.append(dict(fmt=fmt, N=int(N), K=int(K), codes=_parse_hex_list(codes),
                             scales=_parse_hex_list(scales),
                             zeros=None if zeros == "-" else _parse_hex_list(zeros),
                             i=int(i), k=int(k), expect=Fraction(expect)))
    return rows


def pin_dequant_hand_worked(o):
    cases = load_dequant_fixture()
    assert len(cases) >= 20
    for c in cases:
        N, K = c["N"], c["K"]
        codes = np.array(c["codes"], dtype=np.uint8).reshape(N, K // 2)
        if c["fmt"] == "g64":
            scales = np.array(c["scales"], dtype=np.uint16).reshape(N, K // 64)
            w = o.dequant_int4_g64(codes, scales, N, K)
        else:
            G = K // 128
            scales = np.array(c["scales"], dtype=np.uint16).reshape(N, G)
            zeros = np.array(c["zeros"], dtype=np.uint8).reshape(N, (G + 1) // 2)
            w = o.dequant_int4_awq_g128(codes, scales, zeros, N, K)
        got = Fraction(float(w[c["i"], c["k"]]))
        assert got == c["expect"], (c, got)


def pin_dequant_vs_numpy(o):
    for seed, N, K in ((1, 5, 128), (2, 3, 320), (3, 7, 64)):
        c, s, _ = small_g64_case(seed, N, K)
        assert np.array_equal(o.dequant_int4_g64(c, s, N, K), np_dequant_g64(c, s))
    for seed, N, K in ((4, 5, 256), (5, 3, 384), (6, 2, 128)):
        c, s, z, _ = small_awq_case(seed, N, K)
        assert np.array_equal(o.dequant_int4_awq_g128(c, s, z, N, K), np_dequant_awq(c, s, z, K))


def _exact_check(y, yabs, Wf, Xf):
    """Wf (N, K) and Xf (M, K) float64 arrays whose products are exact."""
    M, K = Xf.shape
    N = Wf.shape[0]
    for m in range(M):
        for i in range(N):
            terms = [Fraction(float(Wf[i, k])) * Fraction(float(Xf[m, k])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            exact_abs = sum((abs(t) for t in terms), Fraction(0))
            bound = Fraction(K) * Fraction(2) ** -53 * exact_abs
            assert abs(Fraction(float(y[m, i])) - exact) <= bound, (m, i)
            assert abs(Fraction(float(yabs[m, i])) - exact_abs) <= bound, (m, i)


def pin_bruteforce_exact(o):
    for seed, N, K, M in ((11, 3, 64, 1), (12, 2, 128, 2), (13, 4, 256, 1)):
        W, X = small_bf16_case(seed, N, K, M)
        y, ya = o.gemm_bf16(W, X)
        _exact_check(y, ya, np_bf16_to_f64(W), np_bf16_to_f64(X))
        c, s, X = small_g64_case(seed, N, K, M)
        y, ya = o.gemm_int4_g64(c, s, X)
        _exact_check(y, ya, np_dequant_g64(c, s), np_bf16_to_f64(X))
        if K % 128 == 0:
            c, s, z, X = small_awq_case(seed, N, K, M)
            y, ya = o.gemm_int4_awq_g128(c, s, z, X)
            _exact_check(y, ya, np_dequant_awq(c, s, z, K), np_bf16_to_f64(X))


def pin_vs_numpy_matmul(o):
    for seed, N, K, M in ((21, 37, 320, 1), (22, 9, 1024, 3), (23, 64, 128, 1)):
        W, X = small_bf16_case(seed, N, K, M)
        y, ya = o.gemm_bf16(W, X)
        Wf, Xf = np_bf16_to_f64(W), np_bf16_to_f64(X)
        assert np.all(np.abs(y - Xf @ Wf.T) <= 2 * sum_bound(K, ya))
        assert np.all(np.abs(ya - np.abs(Xf) @ np.abs(Wf).T) <= 2 * sum_bound(K, ya))
        c, s, X = small_g64_case(seed, N, K, M)
        y, ya = o.gemm_int4_g64(c, s, X)
        Wd, Xf = np_dequant_g64(c, s), np_bf16_to_f64(X)
        assert np.all(np.abs(y - Xf @ Wd.T) <= 2 * sum_bound(K, ya))
        assert np.all(np.abs(ya - np.abs(Xf) @ np.abs(Wd).T) <= 2 * sum_bound(K, ya))
        if K % 128 == 0:
            c, s, z, X = small_awq_case(seed, N, K, M)
            y, ya = o.gemm_int4_awq_g128(c, s, z, X)
            Wd = np_dequant_awq(c, s, z, K)
            assert np.all(np.abs(y - Xf @ Wd.T) <= 2 * sum_bound(K, ya))


def pin_power_of_two_scaling(o):
    """y(2^j x) == 2^j y(x) exactly: scaling x by a power of two scales every
    product and partial sum exactly."""
    N, K = 6, 256
    W, X = small_bf16_case(31, N, K, 2)
    c, s, _ = small_g64_case(31, N, K)
    c2, s2, z2, _ = small_awq_case(31, N, K)
    for j in (1, -3, 5):
        Xj = f64_to_bf16_exact(np_bf16_to_f64(X) * 2.0 ** j)
        y, _ = o.gemm_bf16(W, X)
        yj, _ = o.gemm_bf16(W, Xj)
        assert np.array_equal(yj, y * 2.0 ** j)
        y, _ = o.gemm_int4_g64(c, s, X)
        yj, _ = o.gemm_int4_g64(c, s, Xj)
        assert np.array_equal(yj, y * 2.0 ** j)
        y, _ = o.gemm_int4_awq_g128(c2, s2, z2, X)
        yj, _ = o.gemm_int4_awq_g128(c2, s2, z2, Xj)
        assert np.array_equal(yj, y * 2.0 ** j)


def pin_identity_and_one_hot(o):
    K = 128
    _, X = small_bf16_case(41, 1, K, 1)
    xf = np_bf16_to_f64(X)[0]
    # bf16 identity
    eye = f64_to_bf16_exact(np.eye(K))
    y, ya = o.gemm_bf16(eye, X)
    assert np.array_equal(y[0], xf) and np.array_equal(ya[0], np.abs(xf))
    # INT4 g64 identity: q = 9 on the diagonal, 8 elsewhere, scale 1.0
    q = np.full((K, K), 8, dtype=np.uint8)
    np.fill_diagonal(q, 9)
    ones = np.full((K, K // 64), 0x3C00, dtype=np.uint16)
    y, _ = o.gemm_int4_g64(np_pack_codes(q), ones, X)
    assert np.array_equal(y[0], xf)
    # AWQ identity: zero point 3, q = 4 on the diagonal, 3 elsewhere, scale 1.0
    q = np.full((K, K), 3, dtype=np.uint8)
    np.fill_diagonal(q, 4)
    zeros = np.full((K, 1), 0x03, dtype=np.uint8)
    ones = np.full((K, 1), 0x3C00, dtype=np.uint16)
    y, _ = o.gemm_int4_awq_g128(np_pack_codes(q), ones, zeros, X)
    assert np.array_equal(y[0], xf)
    # one-hot rows at a permutation of columns: y_i = x_{c_i}
    N = 40
    cols = np.random.default_rng(3).permutation(K)[:N]
    Wh = np.zeros((N, K))
    Wh[np.arange(N), cols] = 1.0
    y, _ = o.gemm_bf16(f64_to_bf16_exact(Wh), X)
    assert np.array_equal(y[0], xf[cols])
    # one-hot x = e_k: y = column k of the dequantized weights
    Nn = 9
    c, s, _ = small_g64_case(42, Nn, K)
    cw, sw, zw, _ = small_awq_case(42, Nn, K)
    Wb, _ = small_bf16_case(42, Nn, K)
    deq = o.dequant_int4_g64(c, s, Nn, K)
    deqa = o.dequant_int4_awq_g128(cw, sw, zw, Nn, K)
    for k in (0, 1, 63, 64, 127):
        e = np.zeros((1, K))
        e[0, k] = 1.0
        eb = f64_to_bf16_exact(e)
        assert np.array_equal(o.gemm_int4_g64(c, s, eb)[0][0], deq[:, k])
        assert np.array_equal(o.gemm_int4_awq_g128(cw, sw, zw, eb)[0][0], deqa[:, k])
        assert np.array_equal(o.gemm_bf16(Wb, eb)[0][0], np_bf16_to_f64(Wb)[:, k])


def pin_permutation_invariance(o):
    """Permuting k the same way in W and x changes only the summation order."""
    N, K = 5, 256
    rng = np.random.default_rng(51)
    W, X = small_bf16_case(51, N, K)
    p = rng.permutation(K)
    y, ya = o.gemm_bf16(W, X)
    yp, _ = o.gemm_bf16(np.ascontiguousarray(W[:, p]), np.ascontiguousarray(X[:, p]))
    assert np.all(np.abs(y - yp) <= 2 * sum_bound(K, ya))
    # INT4: permute whole groups (with their scales) and codes within each group
    c, s, _ = small_g64_case(51, N, K)
    q = np_unpack_codes(c)
    gp = rng.permutation(K // 64)
    within = rng.permutation(64)
    kp = (gp[:, None] * 64 + within[None, :]).reshape(-1)
    y, ya = o.gemm_int4_g64(c, s, X)
    yp, _ = o.gemm_int4_g64(np_pack_codes(q[:, kp]), np.ascontiguousarray(s[:, gp]), np.ascontiguousarray(X[:, kp]))
    assert np.all(np.abs(y - yp) <= 2 * sum_bound(K, ya))


def pin_batch_equals_separate(o):
    N, K, M = 7, 256, 4
    W, X = small_bf16_case(61, N, K, M)
    c, s, _ = small_g64_case(61, N, K)
    c2, s2, z2, _ = small_awq_case(61, N, K)
    Yb, _ = o.gemm_bf16(W, X)
    Yg, _ = o.gemm_int4_g64(c, s, X)
    Ya, _ = o.gemm_int4_awq_g128(c2, s2, z2, X)
    for m in range(M):
        xm = X[m:m + 1]
        assert np.array_equal(Yb[m], o.gemm_bf16(W, xm)[0][0])
        assert np.array_equal(Yg[m], o.gemm_int4_g64(c, s, xm)[0][0])
        assert np.array_equal(Ya[m], o.gemm_int4_awq_g128(c2, s2, z2, xm)[0][0])


def pin_linearity_disjoint(o):
    """x1 on even k, x2 on odd k: x1 + x2 is exact, so y(x1+x2) = y(x1) + y(x2)
    up to fp64 summation rounding."""
    N, K = 6, 384
    W, X = small_bf16_case(71, N, K)
    c, s, z, _ = small_awq_case(71, N, K)
    x1 = X.copy()
    x1[:, 1::2] = 0
    x2 = X.copy()
    x2[:, 0::2] = 0
    for f in (lambda x: o.gemm_bf16(W, x), lambda x: o.gemm_int4_awq_g128(c, s, z, x)):
        y, ya = f(X)
        y1, _ = f(x1)
        y2, _ = f(x2)
        assert np.all(np.abs(y - (y1 + y2)) <= 3 * sum_bound(K, ya))


def pin_yabs_bounds(o):
    """|y| <= yabs always; yabs is the sum of |w x| (pinned to numpy above)."""
    W, X = small_bf16_case(81, 20, 512, 2)
    y, ya = o.gemm_bf16(W, X)
    assert np.all(np.abs(y) <= ya) and np.all(ya > 0)


def pin_int8_hand_worked(o):
    gemv, quant = load_int8_fixture()
    assert len(gemv) >= 5 and len(quant) >= 4
    for c in gemv:
        q = np.array(c["codes"], dtype=np.int8).reshape(c["N"], c["K"])
        s = np.array(c["scales"], dtype=np.uint32).view(np.float32)
        x = np.array(c["x"], dtype=np.uint16).reshape(1, c["K"])
        y, _ = o.gemm_int8_pc(q, s, x)
        assert Fraction(float(y[0, c["row"]])) == c["expect"], (c, y)
    for c in quant:
        w = np.array(c["w"], dtype=np.uint16).reshape(1, c["K"])
        q, s = o.quantize_int8_pc(w)
        assert int(s.view(np.uint32)[0]) == c["scale"], (c, hex(int(s.view(np.uint32)[0])))
        assert q[0].tolist() == c["codes"], (c, q)


def pin_int8_exact_and_numpy(o):
    for seed, N, K, M in ((91, 3, 64, 1), (92, 2, 128, 2), (93, 5, 48, 1)):
        q, s, X = small_int8_case(seed, N, K, M)
        y, ya = o.gemm_int8_pc(q, s, X)
        _exact_check(y, ya, np_dequant_int8(q, s), np_bf16_to_f64(X))
    for seed, N, K, M in ((94, 37, 640, 1), (95, 9, 1024, 3)):
        q, s, X = small_int8_case(seed, N, K, M)
        y, ya = o.gemm_int8_pc(q, s, X)
        Wd, Xf = np_dequant_int8(q, s), np_bf16_to_f64(X)
        assert np.all(np.abs(y - Xf @ Wd.T) <= 2 * sum_bound(K, ya))
        assert np.all(np.abs(ya - np.abs(Xf) @ np.abs(Wd).T) <= 2 * sum_bound(K, ya))


def pin_int8_invariants(o):
    N, K, M = 7, 256, 3
    q, s, X = small_int8_case(101, N, K, M)
    y, ya = o.gemm_int8_pc(q, s, X)
    # a row's scale scales only that row's output (x2 is exact in fp32 and fp64)
    s2 = s.copy()
    s2[3] = s2[3] * np.float32(2.0)
    y2, _ = o.gemm_int8_pc(q, s2, X)
    assert np.array_equal(y2[:, 3], 2.0 * y[:, 3])
    assert np.array_equal(np.delete(y2, 3, axis=1), np.delete(y, 3, axis=1))
    # negating the codes negates the output
    yn, _ = o.gemm_int8_pc(-q, s, X)
    assert np.array_equal(yn, -y)
    # one-hot x = e_k picks column k of the dequantized weights
    for k in (0, 1, 127, 255):
        e = np.zeros((1, K))
        e[0, k] = 1.0
        ye, _ = o.gemm_int8_pc(q, s, f64_to_bf16_exact(e))
        assert np.array_equal(ye[0], np_dequant_int8(q, s)[:, k])
    # identity codes with scale 1: y = x
    eye = np.eye(K, dtype=np.int8)
    yi, _ = o.gemm_int8_pc(eye, np.ones(K, dtype=np.float32), X[:1])
    assert np.array_equal(yi[0], np_bf16_to_f64(X[0]))
    # the batch equals separate calls
    for m in range(M):
        assert np.array_equal(y[m], o.gemm_int8_pc(q, s, X[m:m + 1])[0][0])
    # power-of-two scaling of x
    Xj = f64_to_bf16_exact(np_bf16_to_f64(X) * 2.0 ** -3)
    assert np.array_equal(o.gemm_int8_pc(q, s, Xj)[0], y * 2.0 ** -3)
    assert np.all(np.abs(y) <= ya)


def pin_int8_quantizer_properties(o):
    """The page's rule: the largest entry of a row lands on +-127 and every
    entry is within half a scale of scale * code (up to the fp32 quotient)."""
    N, K = 12, 300
    W = gen.bf16_weights(111, 0, N, K)
    W[5] = 0          # an all-zero row
    W[6, :] = W[6, :] & 0x807F  # tiny (subnormal) bf16 values
    W[7, 17] = 0xC2FE  # a negative maximum, -127
    q, s = o.quantize_int8_pc(W)
    Wf = np_bf16_to_f64(W)
    for i in range(N):
        amax = float(np.max(np.abs(Wf[i])))
        if amax == 0.0:
            assert s[i] == 0 and not q[i].any()
            continue
        si = Fraction(float(s[i]))
        # s is amax / 127 correctly rounded to fp32 (half an ulp; fixed ulp 2^-149 below 2^-126)
        half_ulp = max(si * Fraction(2) ** -24, Fraction(2) ** -150)
        assert abs(si * 127 - Fraction(amax)) <= 127 * half_ulp
        j = int(np.argmax(np.abs(Wf[i])))
        assert int(q[i, j]) == (127 if Wf[i, j] > 0 else -127), (i, j, q[i, j])
        assert np.all(np.abs(q[i].astype(np.int64)) <= 127)
        for k in range(K):
            t = Fraction(float(Wf[i, k])) / si
            assert abs(t - int(q[i, k])) <= Fraction(1, 2) + Fraction(1, 2 ** 16), (i, k)
            if Wf[i, k] == 0:
                assert q[i, k] == 0


def pin_fusions_hand_worked(o):
    norm, glu, res = load_fusion_fixture()
    assert len(norm) >= 5 and len(glu) >= 5 and len(res) >= 3
    for c in norm:
        got = o.rmsnorm_bf16(np.array([c["x"]], dtype=np.uint16), np.array(c["g"], dtype=np.uint16), c["eps"])
        assert got[0].tolist() == c["expect"], (c, [hex(v) for v in got[0]])
    out = o.swiglu(np.array([a for a, _, _ in glu]), np.array([b for _, b, _ in glu]))
    for (a, b, e), v in zip(glu, out):
        assert abs(v - e) <= 1e-15 * max(1.0, abs(e)), (a, b, v, e)
    out = o.add_residual(np.array([y for y, _, _ in res]), np.array([r for _, r, _ in res], dtype=np.uint16))
    assert out.tolist() == [e for _, _, e in res]


def pin_rmsnorm_invariants(o):
    K = 640
    X = gen.bf16_activations(131, 0, 3, K)
    G = gen.bf16_weights(131, 1, 1, K)[0]
    ones = np.full(K, 0x3F80, dtype=np.uint16)
    xn = o.rmsnorm_bf16(X, G, 0.0)
    # scale invariance without eps: x * 2^j has the same norm-scaled values exactly
    for j in (-3, 4):
        Xj = f64_to_bf16_exact(np_bf16_to_f64(X) * 2.0 ** j)
        assert np.array_equal(o.rmsnorm_bf16(Xj, G, 0.0), xn)
    # g * 2 doubles every output exactly; -x negates it
    G2 = f64_to_bf16_exact(np_bf16_to_f64(G) * 2.0)
    assert np.array_equal(np_bf16_to_f64(o.rmsnorm_bf16(X, G2, 0.0)), 2.0 * np_bf16_to_f64(xn))
    Xneg = X ^ np.uint16(0x8000)
    assert np.array_equal(np_bf16_to_f64(o.rmsnorm_bf16(Xneg, G, 0.0)), -np_bf16_to_f64(xn))
    # unit weight: the normalised row has mean square 1 (up to bf16 rounding)
    u = np_bf16_to_f64(o.rmsnorm_bf16(X, ones, 0.0))
    assert np.all(np.abs(np.mean(u * u, axis=1) - 1.0) < 2.0 ** -7)
    # a large eps shrinks the outputs toward zero
    big = np_bf16_to_f64(o.rmsnorm_bf16(X, ones, 1e6))
    assert np.all(np.abs(big) <= np.abs(np_bf16_to_f64(X)) / 990.0)  # 1/sqrt(1e6 + ~1), then bf16 rounding
    # batch rows are independent
    for m in range(3):
        assert np.array_equal(o.rmsnorm_bf16(X[m], G, 1e-6), o.rmsnorm_bf16(X, G, 1e-6)[m])


def pin_rmsnorm_f64(o):
    """The unrounded normalised activation: a worked case, an independent
    50-digit decimal evaluation of x * g / sqrt(mean(x^2) + eps), the unit
    mean square with g = 1, and its bf16 rounding equal to rmsnorm_bf16."""
    import decimal

    # x = (3, 4), g = 1, eps = 0: mean(x^2) = 12.5, so v = (3, 4) / sqrt(12.5)
    v = o.rmsnorm_f64(np.array([0x4040, 0x4080], dtype=np.uint16), np.array([0x3F80, 0x3F80], dtype=np.uint16), 0.0)
    assert abs(v[0] - 0.848528137423857) <= 1e-15 and abs(v[1] - 1.131370849898476) <= 1e-15, v
    K = 96
    X = gen.bf16_activations(133, 0, 3, K)
    G = gen.bf16_weights(133, 1, 1, K)[0]
    eps = 1e-5
    V = o.rmsnorm_f64(X, G, eps)
    ctx = decimal.Context(prec=50)
    Xf, Gf = np_bf16_to_f64(X), np_bf16_to_f64(G)
    for m in range(3):
        ss = sum((ctx.multiply(decimal.Decimal(float(x)), decimal.Decimal(float(x))) for x in Xf[m]),
                 decimal.Decimal(0))
        root = ctx.sqrt(ctx.add(ctx.divide(ss, decimal.Decimal(K)), decimal.Decimal(eps)))
        for k in range(K):
            want = float(ctx.divide(ctx.multiply(decimal.Decimal(float(Xf[m, k])), decimal.Decimal(float(Gf[k]))),
                                    root))
            assert abs(V[m, k] - want) <= 4 * 2.0 ** -52 * abs(want), (m, k, V[m, k], want)
    ones = np.full(K, 0x3F80, dtype=np.uint16)
    U = o.rmsnorm_f64(X, ones, 0.0)
    assert np.all(np.abs(np.mean(U * U, axis=1) - 1.0) < 1e-13)
    assert np.array_equal(np_round_bf16(V), np_bf16_to_f64(o.rmsnorm_bf16(X, G, eps)))


def pin_swiglu_identities(o):
    a = np.random.default_rng(5).standard_normal(2000) * 6.0
    ones = np.ones_like(a)
    s = o.swiglu(a, ones)
    # silu(a) - silu(-a) = a, and silu(a) = a (1 + tanh(a / 2)) / 2 (another closed form)
    assert np.all(np.abs(s - o.swiglu(-a, ones) - a) <= 1e-14 * (1 + np.abs(a)))
    assert np.all(np.abs(s - a * (1.0 + np.tanh(a / 2.0)) / 2.0) <= 1e-14 * (1 + np.abs(a)))
    # linear in the up operand
    b = np.random.default_rng(6).standard_normal(2000)
    assert np.allclose(o.swiglu(a, b), s * b, rtol=0, atol=1e-13)


def load_repack_fixture():
    rep, dots = [], []
    with open(os.path.join(GOLDEN, "int4_repack_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "repack":
                rep.append((_parse_hex_list(parts[1]), _parse_hex_list(parts[2])))
            else:
                _, codes, scale, zb, k, expect = parts
                dots.append(dict(codes=_parse_hex_list(codes), scale=int(scale, 16), zeros=int(zb, 16), k=int(k),
                                 expect=Fraction(expect)))
    return rep, dots


def pin_repack_hand_worked(o):
    """Hand-worked repacked words, and one-hot products over repacked codes
    (tests/golden/int4_repack_hand.txt)."""
    rep, dots = load_repack_fixture()
    assert len(rep) >= 6 and len(dots) >= 8
    for canon, packed in rep:
        c = np.array(canon, dtype=np.uint8).reshape(1, -1)
        got = o.repack_int4(c)
        assert got.tolist() == [packed], (canon, [hex(v) for v in got[0]])
    for d in dots:
        K = 128
        codes = np.array(d["codes"], dtype=np.uint8).reshape(1, K // 2)
        X = np.zeros((1, K), dtype=np.uint16)
        X[0, d["k"]] = 0x3F80
        Y, _ = o.gemm_int4_awq_g128(codes, np.array([[d["scale"]]], dtype=np.uint16),
                                    np.array([[d["zeros"]]], dtype=np.uint8), X, repacked=True)
        assert Fraction(float(Y[0, 0])) == d["expect"], (d, Y[0, 0])


def pin_repack_permutation(o):
    """The repack is a fixed permutation of the 8 nibbles of a word with cycles
    (0)(7)(1 4 2)(3 5 6): applied three times it is the identity, twice it is
    the inverse; it maps the nibble-count histogram of every row onto itself;
    and the product over repacked codes equals the product over the canonical
    ones (the canonical product is pinned above), bit for bit."""
    rng = np.random.default_rng(41)
    c = rng.integers(0, 256, size=(7, 192), dtype=np.uint8)
    r1 = o.repack_int4(c)
    r3 = o.repack_int4(o.repack_int4(r1))
    assert np.array_equal(r3, c)
    assert not np.array_equal(r1, c)
    assert np.array_equal(np.sort(np_unpack_codes(r1), axis=1), np.sort(np_unpack_codes(c), axis=1))
    # bytes 4w .. 4w+3 hold exactly the codes of k = 8w .. 8w+7
    q, qr = np_unpack_codes(c), np_unpack_codes(r1)
    for w in range(q.shape[1] // 8):
        assert np.array_equal(np.sort(q[:, 8 * w:8 * w + 8], axis=1), np.sort(qr[:, 8 * w:8 * w + 8], axis=1))
    for seed, N, K, M in ((42, 5, 256, 2), (43, 3, 384, 1)):
        cc, s, z, X = small_awq_case(seed, N, K, M)
        Y0, A0 = o.gemm_int4_awq_g128(cc, s, z, X)
        Y1, A1 = o.gemm_int4_awq_g128(o.repack_int4(cc), s, z, X, repacked=True)
        assert np.array_equal(Y0, Y1) and np.array_equal(A0, A1)


PINS = [
    pin_f16_decoder_exhaustive,
    pin_bf16_decoder_exhaustive,
    pin_bf16_rounding,
    pin_dequant_hand_worked,
    pin_dequant_vs_numpy,
    pin_bruteforce_exact,
    pin_vs_numpy_matmul,
    pin_power_of_two_scaling,
    pin_identity_and_one_hot,
    pin_permutation_invariance,
    pin_batch_equals_separate,
    pin_linearity_disjoint,
    pin_yabs_bounds,
    pin_int8_hand_worked,
    pin_int8_exact_and_numpy,
    pin_int8_invariants,
    pin_int8_quantizer_properties,
    pin_fusions_hand_worked,
    pin_rmsnorm_invariants,
    pin_rmsnorm_f64,
    pin_swiglu_identities,
    pin_repack_hand_worked,
    pin_repack_permutation,
]


def run_all(o) -> dict:
    """{pin name: None if it passed, else the failure text}."""
    out = {}
    for p in PINS:
        try:
            p(o)
            out[p.__name__] = None
        except Exception as e:  # noqa: BLE001 - a crash counts as a failed pin
            out[p.__name__] = f"{type(e).__name__}: {e}"[:300]
    return out
