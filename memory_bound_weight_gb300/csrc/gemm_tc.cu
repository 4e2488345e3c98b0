// gemm_tc.cu -- skinny-batch Y = X . W^T on the sm_103a tensor cores
// (tcgen05 MMA with a TMEM accumulator, operands staged by TMA).
//
// Batching raises the arithmetic intensity to ~M FLOP per weight byte (llm-rs
// vs vLLM, sec. 3 "Batching moves decode from memory toward math"); at GB300's
// ridge (~286 FLOP/B) every M <= 256 is still bound by the weight stream or
// close to it, so the kernel must stream W at HBM rate while the tensor pipe
// keeps up. Layout ("swap AB"): the 128 weight rows of a tile are the MMA's M
// side (A = W tile, K-major), the batch is the MMA's N side (B = X tile,
// K-major), so Y^T[128 x n] accumulates in TMEM (lane = weight row, column =
// batch row).
//
// CTA = 6 warps: warp 0 issues TMA loads (one elected thread), warp 1 owns
// TMEM and issues tcgen05.mma (one elected thread), warps 2..5 are the
// epilogue (TMEM -> registers -> bf16 -> global, coalesced along weight rows).
// Stages of 64 k (128-byte rows, 128-byte swizzle) flow through a ring of
// mbarriers: full[s] completes when both TMA loads of stage s landed;
// empty[s] completes when the MMAs that read stage s are done (tcgen05.commit).
// Short, wide shapes split K over a thread-block cluster; each rank writes its
// fp32 partial tile to its shared memory and the ranks sum slices of the tile
// through distributed shared memory, in rank order (deterministic).
// Every mbarrier wait is bounded: on expiry the kernel records a fault flag,
// makes sure no MMA is still writing TMEM, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cooperative_groups.h>

#include "device.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace mbw {

__device__ int g_tc_fault;
static constexpr long long kTcSpin = 1ll << 22;

struct TcArgs {
    void* y;
    int M, N, K;
    int m0;        // first batch row of this launch
    int kstages;   // 64-k stages per cluster rank
    int out_f32;
    const void* xpf;   // the launch's X rows, prefetched into L2 before the wait
    size_t xpf_bytes;
};

__device__ __forceinline__ uint32_t tc_smem(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool tc_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(tc_smem(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity) {
    for (long long i = 0; i < kTcSpin; ++i)
        if (tc_try_wait(bar, parity)) return true;
    atomicExch(&g_tc_fault, 1);
    return false;
}

__device__ __forceinline__ void tc_tma_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(tc_smem(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(tc_smem(bar))
        : "memory");
}

// K-major operand tile with 128-byte rows (64 bf16) in 128-byte-swizzled
// 8-row atoms of 1024 bytes: leading offset unused, stride offset 1024.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;               // leading byte offset (ignored for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;     // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;               // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;               // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16, A = B = bf16, D = f32, both K-major.
__host__ __device__ constexpr uint32_t tc_idesc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

template <int NT>  // batch tile (MMA N): 16 .. 256, multiple of 16
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX,
                   const TcArgs a, const int S, const int D) {
    constexpr int TMEM_COLS = NT <= 32 ? 32 : NT <= 64 ? 64 : NT <= 128 ? 128 : 256;
    constexpr uint32_t A_BYTES = 128 * 128;   // 128 rows x 64 bf16
    constexpr uint32_t B_BYTES = NT * 128;    // NT rows x 64 bf16
    constexpr uint32_t STAGE = A_BYTES + B_BYTES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    pdl_launch_dependents();
    prefetch_l2_grid_share(a.xpf, a.xpf_bytes);

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / S;
    const int row0 = tile * 128;
    const int KS = (a.K + 63) / 64;
    const int ks0 = rank * a.kstages;
    const int nks = max(0, min(KS, ks0 + a.kstages) - ks0);

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)D * STAGE);
    uint64_t* empty = full + D;
    uint64_t* accum = empty + D;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < D; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(&full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(&empty[s])));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(accum)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_smem(tmem_slot)),
                     "n"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer ----
        if (lane == 0) {
            // W tiles do not depend on the previous kernel: fill the whole
            // ring with them first, then wait, then add the X tiles (X may be
            // the previous kernel's output).
            const int npre = min(D, nks);
            for (int i = 0; i < npre; ++i) {
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem(&full[i])),
                             "r"(STAGE)
                             : "memory");
                tc_tma_2d(smem + (size_t)i * STAGE, &mapW, (ks0 + i) * 64, row0, &full[i]);
            }
            pdl_wait();
            for (int i = 0; i < npre; ++i)
                tc_tma_2d(smem + (size_t)i * STAGE + A_BYTES, &mapX, (ks0 + i) * 64, a.m0, &full[i]);
            for (int i = npre; i < nks; ++i) {
                const int s = i % D;
                if (!tc_wait(&empty[s], ((i / D) - 1) & 1)) break;
                uint8_t* st = smem + (size_t)s * STAGE;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem(&full[s])),
                             "r"(STAGE)
                             : "memory");
                const int kc = (ks0 + i) * 64;
                tc_tma_2d(st, &mapW, kc, row0, &full[s]);
                tc_tma_2d(st + A_BYTES, &mapX, kc, a.m0, &full[s]);
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------- MMA issuer ----
        if (lane == 0) {
            bool ok = true;
            const uint32_t idesc = tc_idesc(128, NT);
            for (int i = 0; i < nks; ++i) {
                const int s = i % D;
                if (ok) ok = tc_wait(&full[s], (i / D) & 1);
                if (ok) {
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t sa = tc_smem(smem + (size_t)s * STAGE);
                    const uint64_t da = tc_desc(sa), db = tc_desc(sa + A_BYTES);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
                        // advance 16 k (32 bytes) inside the swizzle atom: +2 in the address field
                        asm volatile(
                            "{\n\t.reg .pred p;\n\t"
                            "setp.ne.b32 p, %4, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                            "l"(da + 2 * k), "l"(db + 2 * k), "r"(idesc), "r"(acc)
                            : "memory");
                    }
                }
                // release the stage once these MMAs have read it (also on error, so the producer can finish)
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 tc_smem(&empty[s]))
                             : "memory");
            }
            // accumulator complete (or, after an error, no MMA left in flight)
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             tc_smem(accum))
                         : "memory");
        }
    } else {
        // ----------------------------------------------------- epilogue ----
        const bool ok = tc_wait(accum, 0);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const int lrow = quarter * 32 + lane;
        float* part = reinterpret_cast<float*>(smem);  // [NT][128] fp32 partials (ring reused)
#pragma unroll 1
        for (int c = 0; c < NT; c += 16) {
            uint32_t v[16];
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c;
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                "[%16];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                  "=r"(v[15])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float f = (ok && nks > 0) ? __uint_as_float(v[j]) : 0.f;
                const int m = c + j;
                if (S == 1) {
                    if (a.m0 + m < a.M && row0 + lrow < a.N)
                        store_out(a.y, (int64_t)(a.m0 + m) * a.N + row0 + lrow, f, a.out_f32);
                } else {
                    part[m * 128 + lrow] = f;
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();

    if (S > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        float* part = reinterpret_cast<float*>(smem);
        const int total = NT * 128;
        const int lo = rank * total / S, hi = (rank + 1) * total / S;
        for (int e = lo + (int)threadIdx.x; e < hi; e += 192) {
            const int m = e / 128, r = e % 128;
            float v = 0.f;
            for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(part + e, s);
            if (a.m0 + m < a.M && row0 + r < a.N) store_out(a.y, (int64_t)(a.m0 + m) * a.N + row0 + r, v, a.out_f32);
        }
        cluster.sync();
    }
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(TMEM_COLS));
    }
}

// ------------------------------------------------------------ host side ----
// The tensor-map encoder lives in the driver; it is looked up through the
// runtime at first use, so libmbw.so has no link-time dependency on libcuda.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

static bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                      uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_batch_tile(int64_t M) {
    const int64_t m = M > 256 ? 256 : M;
    int n = (int)((m + 15) / 16 * 16);
    if (n < 16) n = 16;
    // instantiated tiles
    if (n <= 16) return 16;
    if (n <= 32) return 32;
    if (n <= 64) return 64;
    if (n <= 128) return 128;
    return 256;
}

// Ring depth for a shared-memory budget: ring 0 = deep (one CTA per SM),
// ring 1 = about 100 KB, so that the next launch's CTA fits beside this one
// and streams its first W tiles while this one finishes.
static int tc_stages(int nt, int ring) {
    const size_t stage = 128 * 128 + (size_t)nt * 128;
    int d = (int)(((ring == 0 ? 180 : 96) * 1024) / stage);
    if (d > 8) d = 8;
    if (d < 2) d = 2;
    return d;
}

size_t tc_smem_bytes(int nt, int D, int split) {
    const size_t stage = 128 * 128 + (size_t)nt * 128;
    size_t ring = (size_t)D * stage;
    const size_t part = (size_t)nt * 128 * 4;
    if (split > 1 && part > ring) ring = part;
    return 1024 + ring + (size_t)(2 * D + 1) * 8 + 16;
}

template <int NT>
static cudaError_t launch_nt(const CUtensorMap& mw, const CUtensorMap& mx, const TcArgs& a, int split, int ring,
                             int tiles, cudaStream_t s) {
    const int D = tc_stages(NT, ring);
    const size_t smem = tc_smem_bytes(NT, D, split);
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * split), 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (split > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)split;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    count_launch();
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<NT>, mw, mx, a, split, D);
}

// Y[M][N] = X[M][K] . W[N][K]^T, bf16, in batch slices of up to 256 rows.
cudaError_t launch_gemm_tc(const uint16_t* X, const uint16_t* W, void* Y, int64_t M, int64_t N, int64_t K, int split,
                           int ring, int out_f32, cudaStream_t s) {
    const int nt = tc_batch_tile(M);
    CUtensorMap mw, mx;
    if (!encode_2d(&mw, W, (uint64_t)K, (uint64_t)N, 64, 128)) return cudaErrorInvalidValue;
    if (!encode_2d(&mx, X, (uint64_t)K, (uint64_t)M, 64, (uint32_t)nt)) return cudaErrorInvalidValue;
    const int tiles = (int)((N + 127) / 128);
    const int KS = (int)((K + 63) / 64);
    if (split < 1) split = 1;
    if (split > KS) split = KS;
    TcArgs a;
    a.y = Y;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.kstages = (KS + split - 1) / split;
    a.out_f32 = out_f32;
    for (int64_t m0 = 0; m0 < M; m0 += 256) {
        a.m0 = (int)m0;
        a.xpf = X + m0 * K;
        a.xpf_bytes = (size_t)((M - m0 < 256) ? (M - m0) : 256) * (size_t)K * 2;
        cudaError_t e;
        switch (nt) {
            case 16: e = launch_nt<16>(mw, mx, a, split, ring, tiles, s); break;
            case 32: e = launch_nt<32>(mw, mx, a, split, ring, tiles, s); break;
            case 64: e = launch_nt<64>(mw, mx, a, split, ring, tiles, s); break;
            case 128: e = launch_nt<128>(mw, mx, a, split, ring, tiles, s); break;
            default: e = launch_nt<256>(mw, mx, a, split, ring, tiles, s); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int tc_take_fault() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_fault, sizeof(int)) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_tc_fault, &z, sizeof(int));
    return v;
}

}  // namespace mbw
