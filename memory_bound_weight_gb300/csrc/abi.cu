// abi.cu -- the extern "C" entry points of libmbw.so (declared in mbw.h):
// argument checks on the host, plan lookup, launch, status reporting.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <cstring>
#include <string>

#include "internal.h"
#include "mbw.h"

namespace mbw {

static thread_local std::string g_last_error;
static thread_local int g_out_f32 = 0;
static thread_local uint64_t g_launches = 0;
static thread_local int g_injected_failures = 0;  // mbw_inject_launch_failures

void set_last_error(const std::string& msg) { g_last_error = msg; }
void count_launch() { ++g_launches; }

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

static mbw_status fail(mbw_status st, const std::string& msg) {
    g_last_error = msg;
    return st;
}

static mbw_status cuda_fail(cudaError_t e, const char* where) {
    g_last_error = std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return MBW_ERR_CUDA;
}

static bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// The test hook's failure, taken at the point where a call would launch.
static bool take_injected_failure(const char* where) {
    if (g_injected_failures <= 0) return false;
    --g_injected_failures;
    g_last_error = std::string(where) + ": injected launch failure (mbw_inject_launch_failures)";
    return true;
}

// Common size checks. Returns MBW_OK, or an error with the detail set.
static mbw_status check_sizes(const char* fn, int64_t M, int64_t N, int64_t K, int64_t kunit) {
    if (M < 0 || N < 0 || K < 0) return fail(MBW_ERR_INVALID_ARG, std::string(fn) + ": negative size");
    if (N > MBW_MAX_DIM || K > MBW_MAX_DIM || M > MBW_MAX_DIM)
        return fail(MBW_ERR_BAD_SHAPE, std::string(fn) + ": N, K and M must be at most MBW_MAX_DIM (2^31 - 2^16)");
    if (K % kunit != 0)
        return fail(MBW_ERR_BAD_SHAPE, std::string(fn) + ": K must be a multiple of " + std::to_string(kunit));
    return MBW_OK;
}

static mbw_status zero_output(void* y, int64_t M, int64_t N, cudaStream_t s) {
    const size_t bytes = (size_t)M * (size_t)N * (g_out_f32 ? 4 : 2);
    cudaError_t e = cudaMemsetAsync(y, 0, bytes, s);
    return e == cudaSuccess ? MBW_OK : cuda_fail(e, "cudaMemsetAsync");
}

// Run a CUDA-core streaming GEMV over M activation rows, in slices of the
// planned kernel's batch width.
// `op` may carry MBW_FUSE_* bits; `fz` then holds the fusion pointers.
static mbw_status run_simt(int fmt, int op, const uint8_t* W, const uint16_t* scales, const uint8_t* zeros,
                           const uint16_t* X, void* Y, int64_t M, int64_t N, int64_t K, cudaStream_t s,
                           const float* rscale = nullptr, const mbw_fusion* fz = nullptr) {
    if (take_injected_failure("GEMV launch")) return MBW_ERR_CUDA;
    const Plan p = plan_lookup(op, M, N, K, s);
    if (p.kind == PLAN_NONE)
        return fail(MBW_ERR_UNSUPPORTED, "no kernel fits this shape: the x of one CTA's k-range (split over the "
                                         "largest cluster) does not fit shared memory; see mbw_plan_candidates");
    const int width = plan_batch_width(fmt, p);
    GemvArgs a{};
    a.W = W;
    a.scales = scales;
    a.zeros = zeros;
    a.N = (int)N;
    a.K = (int)K;
    a.chunks = (int)(fmt == FMT_BF16 ? K / 8 : fmt == FMT_I8 ? K / 16 : K / 32);
    a.split_chunks = (a.chunks + p.split - 1) / p.split;
    a.groups = (int)(fmt == FMT_G64 ? K / 64 : fmt == FMT_AWQ ? K / 128 : 0);
    a.zstride = (a.groups + 1) / 2;
    a.out_f32 = g_out_f32;
    a.rscale = rscale;
    a.x_natural = (op & MBW_REPACKED) ? 1 : 0;
    if (fz) {
        a.norm_w = static_cast<const uint16_t*>(fz->norm_weight);
        a.norm_eps = fz->norm_eps;
        if (fz->up_weights) {
            a.glu = 1;
            a.W2 = static_cast<const uint8_t*>(fz->up_weights);
            a.scales2 = static_cast<const uint16_t*>(fz->up_scales);
            a.rscale2 = static_cast<const float*>(fz->up_scales);
            if (fmt == FMT_AWQ) a.zeros2 = static_cast<const uint8_t*>(fz->up_zeros);
        }
    }
    const size_t ybytes = g_out_f32 ? 4 : 2;
    for (int64_t m0 = 0; m0 < M; m0 += width) {
        a.x = X + m0 * K;
        a.y = static_cast<char*>(Y) + (size_t)m0 * (size_t)N * ybytes;
        if (fz && fz->residual) a.residual = static_cast<const uint16_t*>(fz->residual) + (size_t)m0 * (size_t)N;
        a.M = (int)((M - m0) < width ? (M - m0) : width);
        cudaError_t e = launch_plan(fmt, p, a, s);
        if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    }
    return MBW_OK;
}

// AWQ-style INT4 call (`op` may carry MBW_REPACKED): checks, then the planned launch.
static mbw_status awq_call(const char* fn, int op, const uint8_t* Wq, const void* scales, const uint8_t* zeros,
                           const void* X, void* Y, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    mbw_status st = check_sizes(fn, M, N, K, 128);
    if (st != MBW_OK) return st;
    if (N == 0 || M == 0) return MBW_OK;
    if (!Y || (K > 0 && (!Wq || !scales || !zeros || !X)))
        return fail(MBW_ERR_INVALID_ARG, std::string(fn) + ": NULL pointer");
    if (!aligned(Wq, 32) || !aligned(X, 16) || !aligned(Y, 16) || !aligned(scales, 2))
        return fail(MBW_ERR_MISALIGNED,
                    std::string(fn) + ": Wq must be 32-byte aligned, X and Y 16-byte, scales 2-byte");
    if (K == 0) return zero_output(Y, M, N, stream);
    return run_simt(FMT_AWQ, op, Wq, (const uint16_t*)scales, zeros, (const uint16_t*)X, Y, M, N, K, stream);
}

}  // namespace mbw

using namespace mbw;

extern "C" {

mbw_status gemv_bf16(const void* W, const void* x, void* y, int64_t N, int64_t K, void* workspace,
                     size_t ws_bytes, mbw_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    mbw_status st = check_sizes("gemv_bf16", 1, N, K, 8);
    if (st != MBW_OK) return st;
    if (N == 0) return MBW_OK;
    if (!y || (K > 0 && (!W || !x))) return fail(MBW_ERR_INVALID_ARG, "gemv_bf16: NULL pointer");
    if (!aligned(W, 32) || !aligned(x, 16) || !aligned(y, 16))
        return fail(MBW_ERR_MISALIGNED, "gemv_bf16: W must be 32-byte aligned, x and y 16-byte");
    if (K == 0) return zero_output(y, 1, N, (cudaStream_t)stream);
    return run_simt(FMT_BF16, MBW_OP_GEMV_BF16, (const uint8_t*)W, nullptr, nullptr, (const uint16_t*)x, y, 1, N,
                    K, (cudaStream_t)stream);
}

mbw_status gemv_int4_g64(const uint8_t* Wq, const void* scales, const void* x, void* y, int64_t N, int64_t K,
                         void* workspace, size_t ws_bytes, mbw_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    mbw_status st = check_sizes("gemv_int4_g64", 1, N, K, 64);
    if (st != MBW_OK) return st;
    if (N == 0) return MBW_OK;
    if (!y || (K > 0 && (!Wq || !scales || !x))) return fail(MBW_ERR_INVALID_ARG, "gemv_int4_g64: NULL pointer");
    if (!aligned(Wq, 32) || !aligned(x, 16) || !aligned(y, 16) || !aligned(scales, 2))
        return fail(MBW_ERR_MISALIGNED, "gemv_int4_g64: Wq must be 32-byte aligned, x and y 16-byte, scales 2-byte");
    if (K == 0) return zero_output(y, 1, N, (cudaStream_t)stream);
    return run_simt(FMT_G64, MBW_OP_GEMV_INT4_G64, Wq, (const uint16_t*)scales, nullptr, (const uint16_t*)x, y, 1,
                    N, K, (cudaStream_t)stream);
}

mbw_status gemv_int4_awq_g128(const uint8_t* Wq, const void* scales, const uint8_t* zeros, const void* X, void* Y,
                              int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                              mbw_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    return awq_call("gemv_int4_awq_g128", MBW_OP_GEMV_INT4_AWQ_G128, Wq, scales, zeros, X, Y, M, N, K,
                    (cudaStream_t)stream);
}

mbw_status gemv_int4_awq_g128_repacked(const uint8_t* Wr, const void* scales, const uint8_t* zeros, const void* X,
                                       void* Y, int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                                       mbw_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    return awq_call("gemv_int4_awq_g128_repacked", MBW_OP_GEMV_INT4_AWQ_G128 | MBW_REPACKED, Wr, scales, zeros, X,
                    Y, M, N, K, (cudaStream_t)stream);
}

mbw_status mbw_repack_int4(const uint8_t* Wq, uint8_t* Wr, int64_t N, int64_t K, mbw_stream_t stream) {
    mbw_status st = check_sizes("mbw_repack_int4", 1, N, K, 8);
    if (st != MBW_OK) return st;
    if (N == 0 || K == 0) return MBW_OK;
    if (!Wq || !Wr) return fail(MBW_ERR_INVALID_ARG, "mbw_repack_int4: NULL pointer");
    if (!aligned(Wq, 4) || !aligned(Wr, 4))
        return fail(MBW_ERR_MISALIGNED, "mbw_repack_int4: Wq and Wr must be 4-byte aligned");
    if (take_injected_failure("repack launch")) return MBW_ERR_CUDA;
    cudaError_t e = launch_repack_int4(Wq, Wr, N, K, (cudaStream_t)stream);
    return e == cudaSuccess ? MBW_OK : cuda_fail(e, "repack launch");
}

mbw_status gemv_int8_pc(const int8_t* Wq, const float* scales, const void* X, void* Y, int64_t M, int64_t N,
                        int64_t K, void* workspace, size_t ws_bytes, mbw_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    mbw_status st = check_sizes("gemv_int8_pc", M, N, K, 128);
    if (st != MBW_OK) return st;
    if (N == 0 || M == 0) return MBW_OK;
    if (!Y || (K > 0 && (!Wq || !scales || !X))) return fail(MBW_ERR_INVALID_ARG, "gemv_int8_pc: NULL pointer");
    if (!aligned(Wq, 32) || !aligned(X, 16) || !aligned(Y, 16) || !aligned(scales, 4))
        return fail(MBW_ERR_MISALIGNED, "gemv_int8_pc: Wq must be 32-byte aligned, X and Y 16-byte, scales 4-byte");
    if (K == 0) return zero_output(Y, M, N, (cudaStream_t)stream);
    return run_simt(FMT_I8, MBW_OP_GEMV_INT8_PC, (const uint8_t*)Wq, nullptr, nullptr, (const uint16_t*)X, Y, M, N,
                    K, (cudaStream_t)stream, scales);
}

mbw_status mbw_quantize_int8_pc(const void* W, int8_t* Wq, float* scales, int64_t N, int64_t K,
                                mbw_stream_t stream) {
    mbw_status st = check_sizes("mbw_quantize_int8_pc", 1, N, K, 1);
    if (st != MBW_OK) return st;
    if (N == 0) return MBW_OK;
    if (!scales || (K > 0 && (!W || !Wq))) return fail(MBW_ERR_INVALID_ARG, "mbw_quantize_int8_pc: NULL pointer");
    if (!aligned(W, 2) || !aligned(scales, 4))
        return fail(MBW_ERR_MISALIGNED, "mbw_quantize_int8_pc: W must be 2-byte aligned, scales 4-byte");
    if (take_injected_failure("quantize launch")) return MBW_ERR_CUDA;
    cudaError_t e = launch_quantize_int8_pc((const uint16_t*)W, Wq, scales, N, K, (cudaStream_t)stream);
    return e == cudaSuccess ? MBW_OK : cuda_fail(e, "quantize launch");
}

mbw_status gemv_fused(int op, const void* W, const void* scales, const void* X, void* Y, int64_t M, int64_t N,
                      int64_t K, const mbw_fusion* fusion, void* workspace, size_t ws_bytes, mbw_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    int fmt;
    switch (op) {
        case MBW_OP_GEMV_BF16: fmt = FMT_BF16; break;
        case MBW_OP_GEMV_INT4_G64: fmt = FMT_G64; break;
        case MBW_OP_GEMV_INT8_PC: fmt = FMT_I8; break;
        default: return fail(MBW_ERR_INVALID_ARG, "gemv_fused: op must be MBW_OP_GEMV_BF16, _INT4_G64 or _INT8_PC");
    }
    const int64_t kmul = (fmt == FMT_BF16) ? 8 : (fmt == FMT_G64) ? 64 : 128;
    mbw_status st = check_sizes("gemv_fused", M, N, K, kmul);
    if (st != MBW_OK) return st;
    if (N == 0 || M == 0) return MBW_OK;
    if (K == 0) return fail(MBW_ERR_BAD_SHAPE, "gemv_fused: K must be positive");
    if (fmt == FMT_G64 && M != 1) return fail(MBW_ERR_BAD_SHAPE, "gemv_fused: INT4 g64 takes M = 1");
    if (!W || !X || !Y || (fmt != FMT_BF16 && !scales)) return fail(MBW_ERR_INVALID_ARG, "gemv_fused: NULL pointer");
    const size_t salign = (fmt == FMT_I8) ? 4 : 2;
    if (!aligned(W, 32) || !aligned(X, 16) || !aligned(Y, 16) || (scales && !aligned(scales, salign)))
        return fail(MBW_ERR_MISALIGNED, "gemv_fused: W must be 32-byte aligned, X and Y 16-byte, scales 2 or 4 bytes");
    int fop = op;
    if (fusion) {
        if (fusion->norm_weight) {
            if (!aligned(fusion->norm_weight, 16))
                return fail(MBW_ERR_MISALIGNED, "gemv_fused: norm_weight must be 16-byte aligned");
            if (!(fusion->norm_eps >= 0.0f)) return fail(MBW_ERR_INVALID_ARG, "gemv_fused: norm_eps must be >= 0");
            fop |= MBW_FUSE_NORM;
        }
        if (fusion->up_weights) {
            if (!aligned(fusion->up_weights, 32))
                return fail(MBW_ERR_MISALIGNED, "gemv_fused: up_weights must be 32-byte aligned");
            if (fmt != FMT_BF16 && (!fusion->up_scales || !aligned(fusion->up_scales, salign)))
                return fail(MBW_ERR_INVALID_ARG, "gemv_fused: up_scales missing or misaligned");
            fop |= MBW_FUSE_GLU;
        }
        if (fusion->residual) {
            if (!aligned(fusion->residual, 2))
                return fail(MBW_ERR_MISALIGNED, "gemv_fused: residual must be 2-byte aligned");
            fop |= MBW_FUSE_RESIDUAL;
        }
    }
    if (fmt == FMT_G64 || fmt == FMT_I8) {
        if (fmt == FMT_G64 && K % 256 != 0 && (fop & MBW_FUSE_MASK))
            return fail(MBW_ERR_BAD_SHAPE, "gemv_fused: fused INT4 g64 needs K % 256 == 0");
    } else if ((fop & MBW_FUSE_MASK) && K % 64 != 0) {
        return fail(MBW_ERR_BAD_SHAPE, "gemv_fused: fused BF16 needs K % 64 == 0");
    }
    if (mbw_plan_candidates(fop, M, N, K) == 0)
        return fail(MBW_ERR_UNSUPPORTED, "gemv_fused: no kernel for this shape and fusion");
    return run_simt(fmt, fop, (const uint8_t*)W, (const uint16_t*)scales, nullptr, (const uint16_t*)X, Y, M, N, K,
                    (cudaStream_t)stream, fmt == FMT_I8 ? (const float*)scales : nullptr,
                    (fop & MBW_FUSE_MASK) ? fusion : nullptr);
}

mbw_status gemv_fused_awq_g128(const uint8_t* Wq, const void* scales, const uint8_t* zeros, const void* X, void* Y,
                               int64_t M, int64_t N, int64_t K, int repacked, const mbw_fusion* fusion,
                               void* workspace, size_t ws_bytes, mbw_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    if (repacked != 0 && repacked != 1) return fail(MBW_ERR_INVALID_ARG, "gemv_fused_awq_g128: repacked must be 0 or 1");
    const int op = MBW_OP_GEMV_INT4_AWQ_G128 | (repacked ? MBW_REPACKED : 0);
    int fop = op;
    if (fusion) {
        if (fusion->norm_weight) {
            if (!aligned(fusion->norm_weight, 16))
                return fail(MBW_ERR_MISALIGNED, "gemv_fused_awq_g128: norm_weight must be 16-byte aligned");
            if (!(fusion->norm_eps >= 0.0f))
                return fail(MBW_ERR_INVALID_ARG, "gemv_fused_awq_g128: norm_eps must be >= 0");
            fop |= MBW_FUSE_NORM;
        }
        if (fusion->up_weights) {
            if (!aligned(fusion->up_weights, 32))
                return fail(MBW_ERR_MISALIGNED, "gemv_fused_awq_g128: up_weights must be 32-byte aligned");
            if (!fusion->up_scales || !aligned(fusion->up_scales, 2) || !fusion->up_zeros)
                return fail(MBW_ERR_INVALID_ARG, "gemv_fused_awq_g128: up_scales or up_zeros missing or misaligned");
            fop |= MBW_FUSE_GLU;
        }
        if (fusion->residual) {
            if (!aligned(fusion->residual, 2))
                return fail(MBW_ERR_MISALIGNED, "gemv_fused_awq_g128: residual must be 2-byte aligned");
            fop |= MBW_FUSE_RESIDUAL;
        }
    }
    if (!(fop & MBW_FUSE_MASK))
        return awq_call("gemv_fused_awq_g128", op, Wq, scales, zeros, X, Y, M, N, K, (cudaStream_t)stream);
    mbw_status st = check_sizes("gemv_fused_awq_g128", M, N, K, 256);
    if (st != MBW_OK) return st;
    if (N == 0 || M == 0) return MBW_OK;
    if (K == 0) return fail(MBW_ERR_BAD_SHAPE, "gemv_fused_awq_g128: K must be positive");
    if (!Wq || !scales || !zeros || !X || !Y) return fail(MBW_ERR_INVALID_ARG, "gemv_fused_awq_g128: NULL pointer");
    if (!aligned(Wq, 32) || !aligned(X, 16) || !aligned(Y, 16) || !aligned(scales, 2))
        return fail(MBW_ERR_MISALIGNED,
                    "gemv_fused_awq_g128: Wq must be 32-byte aligned, X and Y 16-byte, scales 2-byte");
    if (mbw_plan_candidates(fop, M, N, K) == 0)
        return fail(MBW_ERR_UNSUPPORTED, "gemv_fused_awq_g128: no kernel for this shape and fusion");
    return run_simt(FMT_AWQ, fop, Wq, (const uint16_t*)scales, zeros, (const uint16_t*)X, Y, M, N, K,
                    (cudaStream_t)stream, nullptr, fusion);
}

mbw_status gemm_skinny_bf16(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K,
                            void* workspace, size_t ws_bytes, mbw_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    mbw_status st = check_sizes("gemm_skinny_bf16", M, N, K, 8);
    if (st != MBW_OK) return st;
    if (N == 0 || M == 0) return MBW_OK;
    if (!Y || (K > 0 && (!W || !X))) return fail(MBW_ERR_INVALID_ARG, "gemm_skinny_bf16: NULL pointer");
    if (!aligned(W, 32) || !aligned(X, 16) || !aligned(Y, 16))
        return fail(MBW_ERR_MISALIGNED, "gemm_skinny_bf16: W must be 32-byte aligned, X and Y 16-byte");
    if (K == 0) return zero_output(Y, M, N, (cudaStream_t)stream);
    return run_simt(FMT_BF16, MBW_OP_GEMM_SKINNY_BF16, (const uint8_t*)W, nullptr, nullptr, (const uint16_t*)X, Y,
                    M, N, K, (cudaStream_t)stream);
}

size_t mbw_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
    (void)op;
    (void)M;
    (void)N;
    (void)K;
    return 0;
}

mbw_status mbw_dequant_int4_g64(const uint8_t* Wq, const void* scales, float* out, int64_t N, int64_t K,
                                mbw_stream_t stream) {
    mbw_status st = check_sizes("mbw_dequant_int4_g64", 1, N, K, 64);
    if (st != MBW_OK) return st;
    if (N == 0 || K == 0) return MBW_OK;
    if (!Wq || !scales || !out) return fail(MBW_ERR_INVALID_ARG, "mbw_dequant_int4_g64: NULL pointer");
    if (!aligned(scales, 2) || !aligned(out, 4)) return fail(MBW_ERR_MISALIGNED, "mbw_dequant_int4_g64: alignment");
    if (take_injected_failure("dequant launch")) return MBW_ERR_CUDA;
    cudaError_t e = launch_dequant(FMT_G64, Wq, (const uint16_t*)scales, nullptr, out, N, K, (cudaStream_t)stream);
    return e == cudaSuccess ? MBW_OK : cuda_fail(e, "dequant launch");
}

mbw_status mbw_dequant_int4_awq_g128(const uint8_t* Wq, const void* scales, const uint8_t* zeros, float* out,
                                     int64_t N, int64_t K, mbw_stream_t stream) {
    mbw_status st = check_sizes("mbw_dequant_int4_awq_g128", 1, N, K, 128);
    if (st != MBW_OK) return st;
    if (N == 0 || K == 0) return MBW_OK;
    if (!Wq || !scales || !zeros || !out)
        return fail(MBW_ERR_INVALID_ARG, "mbw_dequant_int4_awq_g128: NULL pointer");
    if (!aligned(scales, 2) || !aligned(out, 4))
        return fail(MBW_ERR_MISALIGNED, "mbw_dequant_int4_awq_g128: alignment");
    if (take_injected_failure("dequant launch")) return MBW_ERR_CUDA;
    cudaError_t e = launch_dequant(FMT_AWQ, Wq, (const uint16_t*)scales, zeros, out, N, K, (cudaStream_t)stream);
    return e == cudaSuccess ? MBW_OK : cuda_fail(e, "dequant launch");
}

mbw_status mbw_set_output_fp32(int enable) {
    if (enable != 0 && enable != 1) return fail(MBW_ERR_INVALID_ARG, "mbw_set_output_fp32: 0 or 1");
    g_out_f32 = enable;
    return MBW_OK;
}

mbw_status mbw_check_device_error(void) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    const int f = tma_take_fault();
    const int f2 = tc_take_fault();
    if (f < 0 || f2 < 0) return cuda_fail(cudaGetLastError(), "reading the device fault flag");
    if (f || f2) return fail(MBW_ERR_DEVICE_TIMEOUT, "a bounded wait inside a kernel expired");
    return MBW_OK;
}

mbw_status mbw_selftest_wait_expiry(int64_t tries, mbw_stream_t stream) {
    if (tries < 1 || tries > MBW_WAIT_LIMIT)
        return fail(MBW_ERR_INVALID_ARG, "mbw_selftest_wait_expiry: tries must be in [1, MBW_WAIT_LIMIT]");
    cudaError_t e = launch_tma_wait_expiry((long long)tries, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "wait-expiry launch");
    e = launch_tc_wait_expiry((long long)tries, (cudaStream_t)stream);
    return e == cudaSuccess ? MBW_OK : cuda_fail(e, "wait-expiry launch");
}

mbw_status mbw_inject_launch_failures(int count) {
    if (count < 0) return fail(MBW_ERR_INVALID_ARG, "mbw_inject_launch_failures: count must be >= 0");
    g_injected_failures = count;
    return MBW_OK;
}

uint64_t mbw_launch_count(void) { return g_launches; }

const char* mbw_status_string(mbw_status s) {
    switch (s) {
        case MBW_OK: return "MBW_OK";
        case MBW_ERR_INVALID_ARG: return "MBW_ERR_INVALID_ARG";
        case MBW_ERR_MISALIGNED: return "MBW_ERR_MISALIGNED";
        case MBW_ERR_BAD_SHAPE: return "MBW_ERR_BAD_SHAPE";
        case MBW_ERR_WORKSPACE_TOO_SMALL: return "MBW_ERR_WORKSPACE_TOO_SMALL";
        case MBW_ERR_UNSUPPORTED: return "MBW_ERR_UNSUPPORTED";
        case MBW_ERR_CUDA: return "MBW_ERR_CUDA";
        case MBW_ERR_DEVICE_TIMEOUT: return "MBW_ERR_DEVICE_TIMEOUT";
        default: return "MBW_ERR_UNKNOWN";
    }
}

const char* mbw_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
