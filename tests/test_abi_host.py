"""Host-side checks of the C ABI (no GPU needed, no compute call is made).

The library must load, export every function include/mbw.h declares, and
reject bad arguments with a status before it touches CUDA.
"""
import ctypes
import os
import re

import pytest

from memory_bound_weight_gb300 import _binding as B
from memory_bound_weight_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mbw.h")


@pytest.fixture(scope="module")
def L():
    mbuild.build()
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s*\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("gemv_bf16", "gemv_int4_g64", "gemv_int4_awq_g128", "gemm_skinny_bf16"):
        assert n in names
    assert len(names) >= 16


def test_every_declared_symbol_is_exported(L):
    raw = ctypes.CDLL(B.LIB_PATH)
    for n in declared_functions():
        assert hasattr(raw, n), n


def test_binding_covers_the_header(L):
    assert sorted(B.SIGNATURES) == declared_functions()


def test_input_generator_library_is_separate(L):
    gen = ctypes.CDLL(os.path.join(os.path.dirname(B.LIB_PATH), "libmbw_inputs.so"))
    for n in ("mbw_gen_bf16_table", "mbw_gen_bytes", "mbw_gen_f16_scales"):
        assert hasattr(gen, n)
    raw = ctypes.CDLL(B.LIB_PATH)
    assert not hasattr(raw, "mbw_gen_bytes")


def test_status_strings(L):
    for code, name in [(0, "MBW_OK"), (1, "MBW_ERR_INVALID_ARG"), (2, "MBW_ERR_MISALIGNED"),
                       (3, "MBW_ERR_BAD_SHAPE"), (4, "MBW_ERR_WORKSPACE_TOO_SMALL"), (5, "MBW_ERR_UNSUPPORTED"),
                       (6, "MBW_ERR_CUDA"), (7, "MBW_ERR_DEVICE_TIMEOUT")]:
        assert L.mbw_status_string(code).decode() == name


def _fusion(norm=None, eps=1e-6, res=None, up=None, ups=None):
    f = B.MbwFusion()
    f.norm_weight, f.norm_eps, f.residual, f.up_weights, f.up_scales = norm, eps, res, up, ups
    return ctypes.byref(f)


A16 = 0x10000  # fake, 16-byte aligned addresses: never dereferenced on these paths
A16b = 0x20000
A16c = 0x30000


@pytest.mark.parametrize("call,expect", [
    (lambda L: L.gemv_bf16(A16, A16b, A16c, -1, 64, None, 0, None), 1),
    (lambda L: L.gemv_bf16(A16, A16b, A16c, 8, 60, None, 0, None), 3),
    (lambda L: L.gemv_bf16(A16 + 2, A16b, A16c, 8, 64, None, 0, None), 2),
    (lambda L: L.gemv_bf16(A16, A16b + 8, A16c, 8, 64, None, 0, None), 2),
    (lambda L: L.gemv_bf16(None, A16b, A16c, 8, 64, None, 0, None), 1),
    (lambda L: L.gemv_bf16(A16, A16b, A16c, 1 << 31, 64, None, 0, None), 3),
    (lambda L: L.gemv_bf16(A16, A16b, A16c, (1 << 31) - (1 << 16) + 1, 64, None, 0, None), 3),  # above MBW_MAX_DIM
    (lambda L: L.gemm_skinny_bf16(A16, A16b, A16c, (1 << 31) - (1 << 16) + 1, 8, 16, None, 0, None), 3),
    (lambda L: L.gemv_bf16(None, None, None, 0, 64, None, 0, None), 0),  # N == 0: no-op
    (lambda L: L.gemv_int4_g64(A16, A16b, A16c, A16c, 8, 96, None, 0, None), 3),
    (lambda L: L.gemv_int4_g64(A16, A16b + 1, A16c, A16c, 8, 128, None, 0, None), 2),
    (lambda L: L.gemv_int4_g64(A16, None, A16c, A16c, 8, 128, None, 0, None), 1),
    (lambda L: L.gemv_int4_awq_g128(A16, A16b, A16c, A16c, A16, 1, 8, 192, None, 0, None), 3),
    (lambda L: L.gemv_int4_awq_g128(A16, A16b, None, A16c, A16, 1, 8, 256, None, 0, None), 1),
    (lambda L: L.gemv_int4_awq_g128(A16, A16b, A16c, A16c, A16, 0, 8, 256, None, 0, None), 0),
    (lambda L: L.gemv_int4_awq_g128(A16, A16b, A16c, A16c, A16, -2, 8, 256, None, 0, None), 1),
    (lambda L: L.gemm_skinny_bf16(A16, A16b, A16c, 4, 8, 12, None, 0, None), 3),
    (lambda L: L.gemm_skinny_bf16(A16, A16b, A16c + 4, 4, 8, 16, None, 0, None), 2),
    (lambda L: L.gemm_skinny_bf16(A16, A16b, A16c, 0, 8, 16, None, 0, None), 0),
    (lambda L: L.gemv_bf16(A16 + 16, A16b, A16c, 8, 64, None, 0, None), 2),  # weights need 32 bytes
    (lambda L: L.gemv_int4_g64(A16 + 16, A16b, A16c, A16c, 8, 128, None, 0, None), 2),
    (lambda L: L.gemv_int4_awq_g128(A16 + 16, A16b, A16c, A16c, A16, 1, 8, 256, None, 0, None), 2),
    (lambda L: L.gemm_skinny_bf16(A16, A16b + 16, A16c, 4, 8, 16, None, 0, None), 2),
    (lambda L: L.gemv_int8_pc(A16 + 16, A16b, A16c, A16, 1, 8, 256, None, 0, None), 2),
    (lambda L: L.gemv_int8_pc(A16, A16b, A16c, A16, 1, 8, 192, None, 0, None), 3),
    (lambda L: L.gemv_fused(3, A16, A16b, A16c, A16, 1, 8, 256, None, None, 0, None), 1),  # AWQ: no fused path
    (lambda L: L.gemv_fused(1, A16, None, A16c, A16, 1, 8, 0, None, None, 0, None), 3),     # K = 0
    (lambda L: L.gemv_fused(2, A16, A16b, A16c, A16, 2, 8, 256, None, None, 0, None), 3),   # g64 takes M = 1
    (lambda L: L.gemv_fused(5, A16 + 16, A16b, A16c, A16, 1, 8, 256, None, None, 0, None), 2),
    (lambda L: L.gemv_fused(5, A16, None, A16c, A16, 1, 8, 256, None, None, 0, None), 1),
    (lambda L: L.gemv_fused(1, A16, None, A16c, A16, 1, 8, 256, _fusion(norm=A16b + 8), None, 0, None), 2),
    (lambda L: L.gemv_fused(1, A16, None, A16c, A16, 1, 8, 256, _fusion(norm=A16b, eps=-1.0), None, 0, None), 1),
    (lambda L: L.gemv_fused(5, A16, A16b, A16c, A16, 1, 8, 256, _fusion(up=A16c), None, 0, None), 1),  # no up_scales
    (lambda L: L.gemv_fused(5, A16, A16b, A16c, A16, 1, 8, 256, _fusion(up=A16c + 16, ups=A16b), None, 0, None), 2),
    (lambda L: L.gemv_fused(1, A16, None, A16c, A16, 1, 8, 96, _fusion(res=A16b), None, 0, None), 3),  # fused BF16: K % 64
    (lambda L: L.gemv_int8_pc(A16, A16b + 2, A16c, A16, 1, 8, 256, None, 0, None), 2),
    (lambda L: L.gemv_int8_pc(A16 + 8, A16b, A16c, A16, 1, 8, 256, None, 0, None), 2),
    (lambda L: L.gemv_int8_pc(A16, None, A16c, A16, 1, 8, 256, None, 0, None), 1),
    (lambda L: L.gemv_int8_pc(A16, A16b, A16c, A16, 0, 8, 256, None, 0, None), 0),
    (lambda L: L.gemv_int8_pc(A16, A16b, A16c, A16, 1, -8, 256, None, 0, None), 1),
    (lambda L: L.mbw_quantize_int8_pc(A16, A16b, None, 8, 64, None), 1),
    (lambda L: L.mbw_quantize_int8_pc(A16 + 1, A16b, A16c, 8, 64, None), 2),
    (lambda L: L.mbw_quantize_int8_pc(A16, A16b, A16c + 2, 8, 64, None), 2),
    (lambda L: L.mbw_quantize_int8_pc(A16, A16b, A16c, 0, 64, None), 0),
    (lambda L: L.mbw_dequant_int4_g64(A16, A16b, A16c, 4, 100, None), 3),
    (lambda L: L.mbw_dequant_int4_awq_g128(A16, A16b, None, A16c, 4, 128, None), 1),
    (lambda L: L.mbw_repack_int4(A16, A16b, 8, 60, None), 3),   # K % 8
    (lambda L: L.mbw_repack_int4(None, A16b, 8, 64, None), 1),
    (lambda L: L.mbw_repack_int4(A16 + 2, A16b, 8, 64, None), 2),
    (lambda L: L.mbw_repack_int4(A16, A16b + 1, 8, 64, None), 2),
    (lambda L: L.mbw_repack_int4(A16, A16b, 0, 64, None), 0),
    (lambda L: L.mbw_repack_int4(A16, A16b, 8, -64, None), 1),
    (lambda L: L.gemv_int4_awq_g128_repacked(A16 + 16, A16b, A16c, A16c, A16, 1, 8, 256, None, 0, None), 2),
    (lambda L: L.gemv_int4_awq_g128_repacked(A16, A16b, A16c, A16c, A16, 1, 8, 192, None, 0, None), 3),
    (lambda L: L.gemv_int4_awq_g128_repacked(A16, A16b, None, A16c, A16, 1, 8, 256, None, 0, None), 1),
    (lambda L: L.gemv_int4_awq_g128_repacked(A16, A16b, A16c, A16c, A16, 0, 8, 256, None, 0, None), 0),
    # no kernel fits: x of one CTA's k-range, split over the largest cluster, exceeds shared memory
    (lambda L: L.gemv_bf16(A16, A16b, A16c, 16, 1 << 20, None, 0, None), 5),
    (lambda L: L.gemv_int8_pc(A16, A16b, A16c, A16, 8, 16, 1 << 17, None, 0, None), 5),
    (lambda L: L.gemv_int4_awq_g128(A16, A16b, A16c, A16c, A16, 64, 16, 1 << 18, None, 0, None), 5),
    (lambda L: L.mbw_set_output_fp32(2), 1),
    (lambda L: L.mbw_plan_select(9, 1, 8, 64, 0), 1),
    (lambda L: L.mbw_autotune(9, 1, 8, 64, None), 1),
    (lambda L: L.mbw_selftest_wait_expiry(0, None), 1),              # tries below 1
    (lambda L: L.mbw_selftest_wait_expiry((1 << 18) + 1, None), 1),  # above the kernels' own limit
])
def test_argument_errors_without_cuda(L, call, expect):
    assert call(L) == expect
    if expect != 0:
        assert L.mbw_last_error().decode() != ""


def test_planner_host_logic(L):
    # candidate enumeration and plan description run on the host
    for op, M, N, K in [(1, 1, 2048, 2048), (2, 1, 2048, 5632), (3, 16, 3584, 18944), (4, 8, 18944, 3584),
                        (5, 1, 9728, 2560), (5, 8, 2560, 9728)]:
        n = L.mbw_plan_candidates(op, M, N, K)
        assert n >= 1
        buf = ctypes.create_string_buffer(256)
        assert L.mbw_plan_describe(op, M, N, K, buf, 256) == 0
        assert b"split_k=" in buf.value
    assert L.mbw_plan_candidates(2, 1, 8, 96) == 0  # K not a multiple of 64
    assert L.mbw_plan_candidates(7, 1, 8, 64) == 0
    assert L.mbw_plan_candidates(5, 1, 8, 192) == 0  # INT8: K not a multiple of 128
    assert L.mbw_plan_candidates(1, 1, (1 << 31) - (1 << 16) + 1, 64) == 0  # N above MBW_MAX_DIM
    assert L.mbw_plan_candidates(1, 1, (1 << 31) - (1 << 16), 64) >= 1  # N at MBW_MAX_DIM
    # fused ops: only the mma2 and latency families, described with their fusions
    for op in (1 | 0x100, 2 | 0x300, 5 | 0x700):
        n = L.mbw_plan_candidates(op, 1, 2048, 2048)
        assert 1 <= n < L.mbw_plan_candidates(op & 0xFF, 1, 2048, 2048) or (op & 0xFF) == 5
        for i in range(n):
            assert L.mbw_plan_select(op, 1, 2048, 2048, i) == 0
            assert L.mbw_plan_describe(op, 1, 2048, 2048, buf, 256) == 0
            assert buf.value.split()[0] in (b"mma2", b"lat") and b"+" in buf.value
    # fused AWQ (canonical or repacked codes): the streaming tensor-core kernel, 4 batch rows per launch
    for op in (3 | 0x100, 3 | 0x700, 3 | 0x800 | 0x300):
        for M in (1, 9):
            n = L.mbw_plan_candidates(op, M, 2048, 2048)
            assert n >= 1
            for i in range(n):
                assert L.mbw_plan_select(op, M, 2048, 2048, i) == 0
                assert L.mbw_plan_describe(op, M, 2048, 2048, buf, 256) == 0
                assert buf.value.startswith(b"mma2") and b"+" in buf.value
                assert buf.value.endswith(b" codes=repacked") == bool(op & 0x800)
    assert L.mbw_plan_candidates(4 | 0x100, 8, 2048, 2048) == 0  # no fused skinny GEMM
    assert L.mbw_plan_candidates(5 | 0x1000, 1, 2048, 2048) == 0  # unknown flag bit
    # repacked INT4 codes (AWQ only): the tensor-core families, never the SIMT ones
    assert L.mbw_plan_candidates(5 | 0x800, 1, 2048, 2048) == 0
    assert L.mbw_plan_candidates(2 | 0x800, 1, 2048, 2048) == 0
    for M, N, K in ((1, 3584, 18944), (3, 4608, 3584), (16, 18944, 3584), (64, 3584, 3584)):
        n = L.mbw_plan_candidates(3 | 0x800, M, N, K)
        assert 1 <= n < L.mbw_plan_candidates(3, M, N, K)
        kinds = set()
        for i in range(n):
            assert L.mbw_plan_select(3 | 0x800, M, N, K, i) == 0
            assert L.mbw_plan_describe(3 | 0x800, M, N, K, buf, 256) == 0
            assert buf.value.endswith(b" codes=repacked")
            kinds.add(buf.value.split()[0])
        assert b"simt" not in kinds
        assert (b"tcgen05" in kinds) == (M > 4)
    # BF16 SIMT with 32-byte lane loads needs K % 16 == 0; its persistent form
    # needs batch 1, no split, and at least one row group per warp of the grid
    def simt_descs(M, N, K):
        out = []
        for i in range(L.mbw_plan_candidates(1, M, N, K)):
            assert L.mbw_plan_select(1, M, N, K, i) == 0
            assert L.mbw_plan_describe(1, M, N, K, buf, 256) == 0
            if buf.value.startswith(b"simt"):
                out.append(buf.value)
        return out
    big = simt_descs(1, 18944, 3584)
    assert any(b"chunk_bytes=32" in d and b"persistent" not in d for d in big)
    pers = [d for d in big if b"persistent" in d]
    assert pers and all(b"split_k=1 " in d for d in pers)
    assert {int(d.split(b"ctas_per_sm=")[1]) for d in pers} == set(range(1, 9))
    assert not any(b"chunk_bytes=32" in d for d in simt_descs(1, 18944, 1032))  # K % 16 == 8
    assert not any(b"persistent" in d for d in simt_descs(1, 300, 3584))  # fewer rows than warps
    assert not any(b"chunk_bytes=32" in d for d in simt_descs(2, 18944, 3584))  # batch 2

    # BF16 row stream: batch 1 only, x (2K bytes) at most 64 KB, no split
    def kinds(M, N, K):
        out = set()
        for i in range(L.mbw_plan_candidates(1, M, N, K)):
            assert L.mbw_plan_select(1, M, N, K, i) == 0
            assert L.mbw_plan_describe(1, M, N, K, buf, 256) == 0
            out.add(buf.value.split()[0])
            if buf.value.startswith(b"rows"):
                assert b"split_k=1" in buf.value
        return out
    assert b"rows" in kinds(1, 18944, 3584) and b"rows" in kinds(1, 3584, 18944) and b"rows" in kinds(1, 1, 8)
    assert b"rows" not in kinds(2, 18944, 3584) and b"rows" not in kinds(1, 64, 32776)

    # bulk-fed INT4: group-64 (batch 1), AWQ up to batch 4, whole super-blocks, no fusions
    def int4_kinds(op, M, N, K):
        out = set()
        for i in range(L.mbw_plan_candidates(op, M, N, K)):
            assert L.mbw_plan_select(op, M, N, K, i) == 0
            assert L.mbw_plan_describe(op, M, N, K, buf, 256) == 0
            out.add(buf.value.split()[0])
        return out
    assert b"bulk" in int4_kinds(2, 1, 11264, 2048) and b"bulk" in int4_kinds(2, 1, 32000, 2048)
    assert b"bulk" in int4_kinds(3, 4, 18944, 3584) and b"bulk" in int4_kinds(3 | 0x800, 1, 3584, 18944)
    assert b"bulk" not in int4_kinds(3, 1, 64, 384) and b"bulk" not in int4_kinds(3 | 0x100, 1, 2048, 2048)
    buf = ctypes.create_string_buffer(256)
    assert L.mbw_plan_describe(5, 1, 9728, 2560, buf, 256) == 0 and b"int8_pc" in buf.value
    assert L.mbw_workspace_bytes(1, 1, 2048, 2048) == 0
    # a shape no kernel fits has no candidate and describes its plan as none
    assert L.mbw_plan_candidates(1, 1, 16, 1 << 20) == 0 and L.mbw_plan_index(1, 1, 16, 1 << 20) == -1
    assert L.mbw_plan_describe(1, 1, 16, 1 << 20, buf, 256) == 0 and buf.value.startswith(b"none")
    # the skinny GEMM streams X through the tensor-core ring: any K from batch 5 on
    assert L.mbw_plan_candidates(4, 8, 16, 1 << 24) >= 1


def test_tall_matrices_have_a_plan_at_every_batch(L):
    """The tensor-core GEMV families keep one partial sum per 16-row tile a CTA
    owns in shared memory; past one wave's share of rows that fits, a launch
    takes more CTAs (several waves) instead of refusing the shape. So every
    call shape the header accepts has at least one plan, up to a few million
    rows and K = 65536 (INT8 at batch 8 and the repacked AWQ codes at batch 4
    had none on tall matrices before)."""
    cases = [(1, (1, 2, 4, 8)), (2, (1,)), (3, (1, 2, 3, 4, 5, 8, 16, 64, 256)), (3 | 0x800, (1, 4, 16, 64)),
             (4, (5, 8, 16, 64, 256)), (5, (1, 2, 3, 4, 5, 8, 16, 64))]
    for op, Ms in cases:
        for K in (1024, 4096, 16384, 65536):
            for N in (16, 4096, 300000, 1000000, 4000000):
                for M in Ms:
                    assert L.mbw_plan_candidates(op, M, N, K) >= 1, (op, M, N, K)
    # an INT8 batch of 8 on 300,000 rows: the tensor-core families run, in several waves
    buf = ctypes.create_string_buffer(256)
    kinds = set()
    for i in range(L.mbw_plan_candidates(5, 8, 300000, 4096)):
        assert L.mbw_plan_select(5, 8, 300000, 4096, i) == 0
        assert L.mbw_plan_describe(5, 8, 300000, 4096, buf, 256) == 0
        kinds.add(buf.value.split()[0])
    assert b"mma2" in kinds


def test_int8_batches_above_8_plan_the_batched_family(L):
    """INT8 calls above 8 rows get the batched mma.sync family (one launch per
    16, 32 or 64 rows) as built-in plan and among the candidates, next to the
    sliced GEMVs; at 8 rows and below it is never a candidate."""
    buf = ctypes.create_string_buffer(256)
    cases = ((9, 16), (16, 16), (17, 32), (32, 32), (33, 64), (64, 64), (200, 64))
    for M, cols in cases:  # the built-in plans first (selecting a candidate replaces the plan of the batch's key)
        assert L.mbw_plan_describe(5, M, 19456, 2560, buf, 256) == 0
        assert buf.value.startswith(b"int8_mma fmt=int8_pc batch_cols=%d " % cols), (M, buf.value)
    for M, _ in cases:
        kinds = set()
        for i in range(L.mbw_plan_candidates(5, M, 19456, 2560)):
            assert L.mbw_plan_select(5, M, 19456, 2560, i) == 0
            assert L.mbw_plan_describe(5, M, 19456, 2560, buf, 256) == 0
            kinds.add(buf.value.split()[0])
        assert b"int8_mma" in kinds and b"mma2" in kinds
    for M in (1, 4, 8):
        for i in range(L.mbw_plan_candidates(5, M, 19456, 2560)):
            assert L.mbw_plan_select(5, M, 19456, 2560, i) == 0
            assert L.mbw_plan_describe(5, M, 19456, 2560, buf, 256) == 0
            assert not buf.value.startswith(b"int8_mma")
    # fused INT8 calls stay on the GEMV families with fusion hooks
    for i in range(L.mbw_plan_candidates(5 | 0x100, 16, 2048, 2048)):
        assert L.mbw_plan_select(5 | 0x100, 16, 2048, 2048, i) == 0
        assert L.mbw_plan_describe(5 | 0x100, 16, 2048, 2048, buf, 256) == 0
        assert buf.value.split()[0] in (b"mma2", b"lat")


def test_output_hook_is_thread_local(L):
    import threading

    assert L.mbw_set_output_fp32(1) == 0
    seen = []

    def other():
        # a fresh thread starts with bf16 output; setting it there does not leak back
        seen.append(L.mbw_set_output_fp32(0))

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert seen == [0]
    assert L.mbw_set_output_fp32(0) == 0


def _gpu_present():
    try:
        import torch

        return torch.cuda.is_available()
    except ImportError:  # pragma: no cover
        return False


@pytest.mark.skipif(_gpu_present(), reason="valid-looking fake addresses must never reach a real GPU")
def test_injected_launch_failures(L):
    """Host-side fault injection: every launching call, given arguments that pass
    its checks, fails with MBW_ERR_CUDA at its launch and launches nothing."""
    calls = {
        "gemv_bf16": lambda: L.gemv_bf16(A16, A16b, A16c, 8, 64, None, 0, None),
        "gemv_int4_g64": lambda: L.gemv_int4_g64(A16, A16b, A16c, A16c, 8, 128, None, 0, None),
        "gemv_int4_awq_g128": lambda: L.gemv_int4_awq_g128(A16, A16b, A16c, A16c, A16, 1, 8, 256, None, 0, None),
        "gemv_int4_awq_g128_repacked":
            lambda: L.gemv_int4_awq_g128_repacked(A16, A16b, A16c, A16c, A16, 20, 8, 256, None, 0, None),
        "gemm_skinny_bf16": lambda: L.gemm_skinny_bf16(A16, A16b, A16c, 4, 8, 16, None, 0, None),
        "gemv_int8_pc": lambda: L.gemv_int8_pc(A16, A16b, A16c, A16, 1, 8, 256, None, 0, None),
        "gemv_fused": lambda: L.gemv_fused(1, A16, None, A16c, A16, 1, 8, 256, _fusion(norm=A16b), None, 0, None),
        "mbw_repack_int4": lambda: L.mbw_repack_int4(A16, A16b, 8, 64, None),
        "mbw_quantize_int8_pc": lambda: L.mbw_quantize_int8_pc(A16, A16b, A16c, 8, 64, None),
        "mbw_dequant_int4_g64": lambda: L.mbw_dequant_int4_g64(A16, A16b, A16c, 4, 128, None),
        "mbw_dequant_int4_awq_g128": lambda: L.mbw_dequant_int4_awq_g128(A16, A16b, A16c, A16c, 4, 128, None),
    }
    assert L.mbw_inject_launch_failures(-1) == 1
    n0 = L.mbw_launch_count()
    try:
        for name, call in calls.items():
            assert L.mbw_inject_launch_failures(1) == 0
            assert call() == 6, name
            assert "injected launch failure" in L.mbw_last_error().decode(), name
        # a call stopped by its argument checks does not use up an injection
        assert L.mbw_inject_launch_failures(1) == 0
        assert L.gemv_bf16(A16, A16b, A16c, 8, 60, None, 0, None) == 3
        assert calls["gemv_bf16"]() == 6
    finally:
        L.mbw_inject_launch_failures(0)
    assert L.mbw_launch_count() == n0
