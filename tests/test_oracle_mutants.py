"""Planted mistakes in the oracle must fail at least one pin.

Each case copies oracle/oracle.c to a temporary directory, plants one plausible
mistake (a swapped nibble, a wrong group or row stride, a dropped term, a sign,
a transposed index, a wrong exponent bias ...), compiles it, and runs the pin
suite against it. A mutant that passes every pin would mean the pins cannot
see that kind of mistake. The real oracle is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text to find, replacement, which occurrence (1-based))
MUTANTS = [
    ("nibble_order", "(k % 2 == 0) ? (b & 0x0F) : (b >> 4)", "(k % 2 == 0) ? (b >> 4) : (b & 0x0F)", 1),
    ("g64_zero_point", "(double)(q - 8) * s", "(double)(q - 7) * s", 1),
    ("g64_group_index", "scales[i * (K / 64) + k / 64]", "scales[i * (K / 64) + k / 128]", 1),
    ("g64_scale_row_stride", "scales[i * (K / 64) + k / 64]", "scales[i * (K / 128) + k / 64]", 1),
    ("code_row_stride", "codes[i * (K / 2) + k / 2]", "codes[i * (K / 4) + k / 2]", 1),
    ("awq_zero_nibble_order", "(g % 2 == 0) ? (zb & 0x0F) : (zb >> 4)", "(g % 2 == 0) ? (zb >> 4) : (zb & 0x0F)", 1),
    ("awq_zero_stride", "int64_t zstride = (G + 1) / 2;", "int64_t zstride = G / 2;", 1),
    ("awq_sign", "(double)(q - z) * s", "(double)(z - q) * s", 1),
    ("awq_group_boundary_off_by_one", "int64_t g = k / 128;", "int64_t g = (k + 1) / 128 < G ? (k + 1) / 128 : G - 1;", 1),
    ("f16_exponent_bias", "ldexp(1024.0 + (double)f, e - 25)", "ldexp(1024.0 + (double)f, e - 24)", 1),
    ("f16_subnormal", "ldexp((double)f, -24)", "ldexp((double)f, -25)", 1),
    ("f16_implicit_bit", "ldexp(1024.0 + (double)f, e - 25)", "ldexp((double)f, e - 25)", 1),
    ("bf16_exponent_bias", "ldexp(128.0 + (double)f, e - 134)", "ldexp(128.0 + (double)f, e - 133)", 1),
    ("bf16_subnormal", "ldexp((double)f, -133)", "ldexp((double)f, -132)", 1),
    ("rne_ties_to_odd", "fmod(fl, 2.0) != 0.0", "fmod(fl, 2.0) == 0.0", 1),
    ("bf16_dropped_last_term", "for (int64_t k = 0; k < K; k++) {", "for (int64_t k = 0; k < K - 1; k++) {", 1),
    ("g64_dropped_last_term", "for (int64_t k = 0; k < K; k++) {", "for (int64_t k = 0; k < K - 1; k++) {", 2),
    ("awq_dropped_first_term", "for (int64_t k = 0; k < K; k++) {", "for (int64_t k = 1; k < K; k++) {", 3),
    ("g64_reversed_x", "X[m * K + k]", "X[m * K + (K - 1 - k)]", 2),
    ("bf16_reversed_w", "W[i * K + k]", "W[i * K + (K - 1 - k)]", 1),
    ("yabs_signed", "aabs += fabs(w * x);", "aabs += w * x;", 1),
    ("awq_acc_sign", "acc += w * x;", "acc -= w * x;", 3),
    ("output_transposed", "Y[m * N + i] = acc;", "Y[i * M + m] = acc;", 1),
    ("batch_row_of_x", "X[m * K + k]", "X[0 * K + k]", 1),
    ("int8_scale_of_row_0", "(double)S[i] * (double)Q[i * K + k]", "(double)S[0] * (double)Q[i * K + k]", 1),
    ("int8_scale_dropped", "(double)S[i] * (double)Q[i * K + k]", "(double)Q[i * K + k]", 1),
    ("int8_codes_unsigned", "(double)S[i] * (double)Q[i * K + k]", "(double)S[i] * (double)(uint8_t)Q[i * K + k]", 1),
    ("int8_code_row_stride", "(double)S[i] * (double)Q[i * K + k]", "(double)S[i] * (double)Q[i * (K - 1) + k]", 1),
    ("int8_dropped_last_term", "for (int64_t k = 0; k < K; k++) {", "for (int64_t k = 0; k < K - 1; k++) {", 4),
    ("int8_acc_sign", "acc += w * x;", "acc -= w * x;", 4),
    ("quant_divisor_128", "amax / 127.0f", "amax / 128.0f", 1),
    ("quant_ties_away", "rintf(t)", "roundf(t)", 1),
    ("quant_truncate", "rintf(t)", "truncf(t)", 1),
    ("quant_signed_max", "(float)fabs(oracle_bf16_to_double(W[i * K + k]))", "(float)oracle_bf16_to_double(W[i * K + k])", 1),
    ("rmsnorm_mean_over_k_minus_1", "ss / (double)K + eps", "ss / (double)(K - 1) + eps", 1),
    ("rmsnorm_eps_dropped", "ss / (double)K + eps", "ss / (double)K", 1),
    ("rmsnorm_no_sqrt", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / (ss / (double)K + eps)", 1),
    ("rmsnorm_weight_dropped", "x * inv * g", "x * inv", 1),
    ("rmsnorm_abs_sum", "ss += x * x;", "ss += fabs(x);", 1),
    ("swiglu_exp_sign", "exp(-A[i])", "exp(A[i])", 1),
    ("swiglu_gate_up_swapped", "A[i] / (1.0 + exp(-A[i])) * B[i]", "B[i] / (1.0 + exp(-B[i])) * A[i]", 1),
    ("residual_subtracted", "Y[i] + oracle_bf16_to_double(R[i])", "Y[i] - oracle_bf16_to_double(R[i])", 1),
    ("quant_first_entry_skipped", "for (int64_t k = 0; k < K; k++) {", "for (int64_t k = 1; k < K; k++) {", 5),
    ("repack_inverse_permutation", "return j / 2 + 4 * (j % 2);", "return (j % 4) * 2 + j / 4;", 1),
    ("repack_nibble_halves_swapped", "(t % 2 == 0 ? q : q << 4)", "(t % 2 == 0 ? q << 4 : q)", 1),
    ("repacked_decode_nibble_order", "(t % 2 == 0) ? (b & 0x0F) : (b >> 4)", "(t % 2 == 0) ? (b >> 4) : (b & 0x0F)", 1),
    ("repacked_decode_word_stride", "(k / 8) * 4 + t / 2]", "(k / 8) * 8 + t / 2]", 1),
    ("repacked_gemm_reads_canonical", "dequant_awq_any(codes, scales, zeros, K, i, k, repacked)",
     "dequant_awq_any(codes, scales, zeros, K, i, k, 0)", 1),
]


def _plant(src: str, find: str, repl: str, nth: int) -> str:
    pos = -1
    for _ in range(nth):
        pos = src.find(find, pos + 1)
        assert pos >= 0, f"mutation anchor not found: {find!r} #{nth}"
    return src[:pos] + repl + src[pos + len(find):]


@pytest.mark.parametrize("name,find,repl,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, find, repl, nth):
    with open(SRC) as f:
        src = f.read()
    mutated = _plant(src, find, repl, nth)
    assert mutated != src
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(mutated)
    lib = oracle.build(str(path), str(tmp_path / f"liboracle_{name}.so"))
    o = oracle.load(lib)
    for pin in oracle_pins.PINS:
        try:
            pin(o)
        except Exception:  # noqa: BLE001 - any failure means the pin saw the mistake
            return
    pytest.fail(f"mutant {name} passed every pin")
