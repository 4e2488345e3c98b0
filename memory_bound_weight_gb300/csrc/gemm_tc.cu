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
// CTA = 6 warps: warp 0 issues TMA loads and warp 1 owns TMEM and issues
// tcgen05.mma (each runs its loop on the whole warp and issues from one
// elected lane), warps 2..5 are the
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
static constexpr long long kTcSpin = MBW_WAIT_LIMIT;

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

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, long long limit = kTcSpin) {
    for (long long i = 0; i < limit; ++i)
        if (tc_try_wait(bar, parity)) return true;
    atomicExch(&g_tc_fault, 1);
    return false;
}

// The roles that issue tcgen05.mma and TMA copies run their loops on the
// whole warp and issue from one elected lane. With a lone active lane (the
// rest of the warp parked at a barrier) tcgen05.mma issues ~3x slower, and
// every later wait of that lane stalls until the MMAs in flight drain.
__device__ __forceinline__ bool tc_elect() {
    uint32_t e;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
    return e != 0;
}

// a bounded wait with one outcome for the whole warp
__device__ __forceinline__ bool tc_wait_warp(uint64_t* bar, uint32_t parity) {
    return __all_sync(0xFFFFFFFFu, tc_wait(bar, parity));
}

// After a producer's slot wait gave up at stage `stop` (< n), wait (bounded,
// whole warp) for the bulk copies of the stages it issued that may still be in
// flight: the last D before `stop`, whose slots are not reused. Then no copy
// lands in shared memory after the ring is reused or the CTA exits.
__device__ __forceinline__ void tc_drain_issued(uint64_t* full, int stop, int n, int D) {
    if (stop >= n) return;
    for (int j = max(0, stop - D); j < stop; ++j) tc_wait_warp(&full[j % D], (j / D) & 1);
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

// INT4 helpers of the AWQ path: the nibbles at bits 0-3 and 16-19 of v as the
// bf16 pair (128 + n_lo, 128 + n_hi); an exact bf16x2 subtract; the x chunk
// permutation (0,4) (1,5) (2,6) (3,7) that matches the unpack's k order.
__device__ __forceinline__ uint32_t tc_nib(uint32_t v) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(0x000F000Fu), "r"(0x43004300u));
    return r;
}
__device__ __forceinline__ uint32_t tc_sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint4 tc_perm(uint4 v) {
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    return o;
}

// NT: batch tile (MMA N), 16 .. 256, multiple of 16. C: independent TMEM
// accumulators the k-steps rotate over -- consecutive MMAs into one
// accumulator wait for each other, so a single chain runs at the MMA latency
// instead of the tensor pipe's rate; the epilogue adds the C partial sums.
// BPS: 64-k boxes per ring stage: two boxes per stage mean one wait and one
// commit per 8 MMAs; a one-box stage keeps more stages in a small ring.
template <int NT, int C, int BPS>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX,
                   const TcArgs a, const int S, const int D) {
    constexpr int NTP = NT <= 32 ? 32 : NT <= 64 ? 64 : NT <= 128 ? 128 : 256;  // columns per accumulator
    constexpr int TMEM_COLS = NTP * C;
    static_assert(TMEM_COLS <= 512, "");
    constexpr uint32_t A_BYTES = 128 * 128;   // 128 rows x 64 bf16 (one box)
    constexpr uint32_t B_BYTES = NT * 128;    // NT rows x 64 bf16 (one box)
    constexpr uint32_t STAGE = BPS * (A_BYTES + B_BYTES);  // W boxes, then X boxes
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    pdl_launch_dependents();
    prefetch_l2_grid_share(a.xpf, a.xpf_bytes);

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / S;
    const int row0 = tile * 128;
    const int KS = (a.K + 64 * BPS - 1) / (64 * BPS);  // stages (boxes past K read zeros)
    const int ks0 = rank * a.kstages;
    const int nks = max(0, min(KS, ks0 + a.kstages) - ks0);

    // barriers after the ring and after the split-K partial tile that reuses it
    // (a commit may still land on a ring barrier while the epilogue writes partials)
    const size_t ring_bytes = max((size_t)D * STAGE, S > 1 ? (size_t)NT * 128 * 4 : (size_t)0);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ring_bytes);
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
        const bool leader = tc_elect();
        // W tiles do not depend on the previous kernel: fill the whole
        // ring with them first, then wait, then add the X tiles (X may be
        // the previous kernel's output).
        const int npre = min(D, nks);
        if (leader)
            for (int i = 0; i < npre; ++i) {
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem(&full[i])),
                             "r"(STAGE)
                             : "memory");
                for (int bb = 0; bb < BPS; ++bb)
                    tc_tma_2d(smem + (size_t)i * STAGE + bb * A_BYTES, &mapW, ((ks0 + i) * BPS + bb) * 64, row0,
                              &full[i]);
            }
        __syncwarp();
        pdl_wait();
        if (leader)
            for (int i = 0; i < npre; ++i)
                for (int bb = 0; bb < BPS; ++bb)
                    tc_tma_2d(smem + (size_t)i * STAGE + BPS * A_BYTES + bb * B_BYTES, &mapX,
                              ((ks0 + i) * BPS + bb) * 64, a.m0, &full[i]);
        __syncwarp();
        int i = npre;
        for (; i < nks; ++i) {
            const int s = i % D;
            if (!tc_wait_warp(&empty[s], ((i / D) - 1) & 1)) break;
            uint8_t* st = smem + (size_t)s * STAGE;
            if (leader) {
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem(&full[s])),
                             "r"(STAGE)
                             : "memory");
                for (int bb = 0; bb < BPS; ++bb) {
                    const int kc = ((ks0 + i) * BPS + bb) * 64;
                    tc_tma_2d(st + bb * A_BYTES, &mapW, kc, row0, &full[s]);
                    tc_tma_2d(st + BPS * A_BYTES + bb * B_BYTES, &mapX, kc, a.m0, &full[s]);
                }
            }
            __syncwarp();
        }
        tc_drain_issued(full, i, nks, D);
        if (S > 1) asm volatile("bar.arrive 1, 160;" ::: "memory");  // the ring may now hold the partials
    } else if (warp == 1) {
        // --------------------------------------------------- MMA issuer ----
        {
            const bool leader = tc_elect();
            bool ok = true;
            const uint32_t idesc = tc_idesc(128, NT);
            for (int i = 0; i < nks; ++i) {
                const int s = i % D;
                if (ok) ok = tc_wait_warp(&full[s], (i / D) & 1);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (ok && leader) {
                    const uint32_t sa = tc_smem(smem + (size_t)s * STAGE);
#pragma unroll
                    for (int bb = 0; bb < BPS; ++bb) {
                        const uint64_t da = tc_desc(sa + bb * A_BYTES), db = tc_desc(sa + BPS * A_BYTES + bb * B_BYTES);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int t = (i * BPS + bb) * 4 + k;  // k-step; accumulator t % C
                            const uint32_t acc = (t >= C) ? 1u : 0u;
                            // advance 16 k (32 bytes) inside the swizzle atom: +2 in the address field
                            asm volatile(
                                "{\n\t.reg .pred p;\n\t"
                                "setp.ne.b32 p, %4, 0;\n\t"
                                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
                                    tmem + (uint32_t)((t % C) * NTP)),
                                "l"(da + 2 * k), "l"(db + 2 * k), "r"(idesc), "r"(acc)
                                : "memory");
                        }
                    }
                }
                // release the stage once these MMAs have read it (also on error, so the producer can finish)
                if (leader)
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     tc_smem(&empty[s]))
                                 : "memory");
                __syncwarp();
            }
            // accumulator complete (or, after an error, no MMA left in flight)
            if (leader)
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 tc_smem(accum))
                             : "memory");
            __syncwarp();
        }
    } else {
        // ----------------------------------------------------- epilogue ----
        const bool ok = tc_wait(accum, 0);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // split-K: the partials reuse the ring, which the producer may still be
        // draining after a failed wait; it arrives here once no copy is in flight
        if (S > 1) asm volatile("bar.sync 1, 160;" ::: "memory");
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const int lrow = quarter * 32 + lane;
        float* part = reinterpret_cast<float*>(smem);  // [NT][128] fp32 partials (ring reused)
#pragma unroll 1
        for (int c = 0; c < NT; c += 16) {
            float fs[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) fs[j] = 0.f;
            // all C accumulators of this 16-column block, then one wait (a wait
            // per load would put a TMEM round trip per accumulator on the epilogue)
            uint32_t v[C][16];
#pragma unroll
            for (int ch = 0; ch < C; ++ch) {
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ch * NTP + c);
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                    "[%16];"
                    : "=r"(v[ch][0]), "=r"(v[ch][1]), "=r"(v[ch][2]), "=r"(v[ch][3]), "=r"(v[ch][4]), "=r"(v[ch][5]),
                      "=r"(v[ch][6]), "=r"(v[ch][7]), "=r"(v[ch][8]), "=r"(v[ch][9]), "=r"(v[ch][10]),
                      "=r"(v[ch][11]), "=r"(v[ch][12]), "=r"(v[ch][13]), "=r"(v[ch][14]), "=r"(v[ch][15])
                    : "r"(taddr));
            }
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int ch = 0; ch < C; ++ch) {
                // an accumulator no k-step reached holds no data
                if (ch < nks * 4 * BPS) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) fs[j] += __uint_as_float(v[ch][j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float f = (ok && nks > 0) ? fs[j] : 0.f;
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

// ----------------------------------------------------------------------------
// CTA-pair variant for batch tiles of 128 and 256 (tcgen05.mma cta_group::2:
// M = 256 across the two SMs of a pair). Each CTA of the pair stages its own
// 128 weight rows and its half of the batch tile's X rows; the even CTA
// issues one MMA for the pair, which reads A (W) from each CTA's own shared
// memory and B (X) split by batch halves, and leaves each CTA's 128 rows x NT
// outputs in that CTA's TMEM. At large batch X is two thirds of a one-CTA
// stage; halving it fits more stages of the weight stream in the ring and
// halves the X traffic out of L2.
// Cluster rank r: member r & 1 of the pair, split-K rank r >> 1 (clusters of
// 2 S CTAs). Both CTAs' loads of a stage complete on the even CTA's full
// barrier; the even CTA's commits release both CTAs' ring slots and
// accumulators (multicast). Every wait is bounded.
__device__ __forceinline__ uint32_t tc_cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void tc_cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int NT, int C, int BPS>
__global__ void __launch_bounds__(192, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX,
                    const TcArgs a, const int S, const int D) {
    constexpr int NH = NT / 2;  // X rows this CTA stages
    constexpr int NTP = NT <= 128 ? 128 : 256;
    constexpr int TMEM_COLS = NTP * C;
    static_assert(TMEM_COLS <= 512 && (NT == 128 || NT == 256), "");
    constexpr uint32_t A_BYTES = 128 * 128;  // 128 rows x 64 bf16 (one box)
    constexpr uint32_t B_BYTES = NH * 128;   // NH rows x 64 bf16 (one box)
    constexpr uint32_t STAGE = BPS * (A_BYTES + B_BYTES);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    pdl_launch_dependents();
    prefetch_l2_grid_share(a.xpf, a.xpf_bytes);

    const uint32_t crank = tc_cluster_rank();
    const int member = (int)(crank & 1u), krank = (int)(crank >> 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x / (2 * S)) * 256 + member * 128;
    const int KS = (a.K + 64 * BPS - 1) / (64 * BPS);
    const int ks0 = krank * a.kstages;
    const int nks = max(0, min(KS, ks0 + a.kstages) - ks0);
    const uint16_t pair_mask = (uint16_t)(3u << (2 * krank));

    // barriers after the ring and after the split-K partial tile that reuses it
    const size_t ring_bytes = max((size_t)D * STAGE, S > 1 ? (size_t)NT * 128 * 4 : (size_t)0);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ring_bytes);  // the even CTA's count both halves
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
        // one warp of each CTA of the pair, collectively
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_smem(tmem_slot)),
                     "n"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    // the peer's barriers exist before any remote arrive or multicast commit reaches them
    tc_cluster_sync_all();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer ----
        // Both CTAs' loads complete on the even CTA's full barriers (the
        // .cta_group::2 form may name the peer's barrier); the even CTA
        // expects the bytes of both halves of a stage.
        const bool leader = tc_elect();
        const int xrow = a.m0 + member * NH;
        const int npre = min(D, nks);
        uint32_t fbar0;  // full[0] of the even CTA
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(fbar0) : "r"(tc_smem(full)), "r"(crank & ~1u));
        auto tma2 = [&](void* dst, const CUtensorMap* map, int c0, int c1, int s) {
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, "
                "{%2, %3}], [%4];" ::"r"(tc_smem(dst)),
                "l"(map), "r"(c0), "r"(c1), "r"(fbar0 + 8u * s)
                : "memory");
        };
        if (leader)
            for (int i = 0; i < npre; ++i) {
                if (member == 0)
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem(&full[i])),
                                 "r"(2 * STAGE)
                                 : "memory");
                for (int bb = 0; bb < BPS; ++bb)
                    tma2(smem + (size_t)i * STAGE + bb * A_BYTES, &mapW, ((ks0 + i) * BPS + bb) * 64, row0, i);
            }
        __syncwarp();
        pdl_wait();
        if (leader)
            for (int i = 0; i < npre; ++i)
                for (int bb = 0; bb < BPS; ++bb)
                    tma2(smem + (size_t)i * STAGE + BPS * A_BYTES + bb * B_BYTES, &mapX, ((ks0 + i) * BPS + bb) * 64,
                         xrow, i);
        __syncwarp();
        int i = npre;
        for (; i < nks; ++i) {
            const int s = i % D;
            if (!tc_wait_warp(&empty[s], ((i / D) - 1) & 1)) break;
            uint8_t* st = smem + (size_t)s * STAGE;
            if (leader) {
                if (member == 0)
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem(&full[s])),
                                 "r"(2 * STAGE)
                                 : "memory");
                for (int bb = 0; bb < BPS; ++bb) {
                    const int kc = ((ks0 + i) * BPS + bb) * 64;
                    tma2(st + bb * A_BYTES, &mapW, kc, row0, s);
                    tma2(st + BPS * A_BYTES + bb * B_BYTES, &mapX, kc, xrow, s);
                }
            }
            __syncwarp();
        }
        // both CTAs' copies complete on the even CTA's barriers, so the even CTA
        // drains for the pair; the cluster barrier at the end keeps the odd CTA
        // resident until it has
        if (member == 0) tc_drain_issued(full, i, nks, D);
        if (S > 1) asm volatile("bar.arrive 1, 160;" ::: "memory");  // the ring may now hold the partials
    } else if (warp == 1) {
        // ----------------------------------------- MMA issuer (even CTA) ----
        const bool leader = tc_elect();
        if (member == 0) {
            bool ok = true;
            const uint32_t idesc = tc_idesc(256, NT);
            for (int i = 0; i < nks; ++i) {
                const int s = i % D;
                if (ok) ok = tc_wait_warp(&full[s], (i / D) & 1);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (ok && leader) {
                    const uint32_t sa = tc_smem(smem + (size_t)s * STAGE);
#pragma unroll
                    for (int bb = 0; bb < BPS; ++bb) {
                        const uint64_t da = tc_desc(sa + bb * A_BYTES), db = tc_desc(sa + BPS * A_BYTES + bb * B_BYTES);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int t = (i * BPS + bb) * 4 + k;  // k-step; accumulator t % C
                            asm volatile(
                                "{\n\t.reg .pred p;\n\t"
                                "setp.ne.b32 p, %4, 0;\n\t"
                                "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
                                    tmem + (uint32_t)((t % C) * NTP)),
                                "l"(da + 2 * k), "l"(db + 2 * k), "r"(idesc), "r"((t >= C) ? 1u : 0u)
                                : "memory");
                        }
                    }
                }
                // release the stage in both CTAs once these MMAs have read it (also on error)
                if (leader)
                    asm volatile(
                        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
                        "[%0], %1;" ::"r"(tc_smem(&empty[s])),
                        "h"(pair_mask)
                        : "memory");
                __syncwarp();
            }
            if (leader)
                asm volatile(
                    "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
                    "[%0], %1;" ::"r"(tc_smem(accum)),
                    "h"(pair_mask)
                    : "memory");
            __syncwarp();
        }
    } else {
        // ----------------------------------------------------- epilogue ----
        const bool ok = tc_wait(accum, 0);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // split-K: the partials reuse the ring, which the producer may still be
        // draining after a failed wait; it arrives here once no copy is in flight
        if (S > 1) asm volatile("bar.sync 1, 160;" ::: "memory");
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const int lrow = quarter * 32 + lane;
        float* part = reinterpret_cast<float*>(smem);  // [NT][128] fp32 partials (ring reused)
#pragma unroll 1
        for (int c = 0; c < NT; c += 16) {
            float fs[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) fs[j] = 0.f;
            uint32_t v[C][16];
#pragma unroll
            for (int ch = 0; ch < C; ++ch) {
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ch * NTP + c);
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                    "[%16];"
                    : "=r"(v[ch][0]), "=r"(v[ch][1]), "=r"(v[ch][2]), "=r"(v[ch][3]), "=r"(v[ch][4]), "=r"(v[ch][5]),
                      "=r"(v[ch][6]), "=r"(v[ch][7]), "=r"(v[ch][8]), "=r"(v[ch][9]), "=r"(v[ch][10]),
                      "=r"(v[ch][11]), "=r"(v[ch][12]), "=r"(v[ch][13]), "=r"(v[ch][14]), "=r"(v[ch][15])
                    : "r"(taddr));
            }
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int ch = 0; ch < C; ++ch) {
                if (ch < nks * 4 * BPS) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) fs[j] += __uint_as_float(v[ch][j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float f = (ok && nks > 0) ? fs[j] : 0.f;
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
        // the split-K ranks of this CTA's rows are cluster ranks 2 kr + member
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        float* part = reinterpret_cast<float*>(smem);
        const int total = NT * 128;
        const int lo = krank * total / S, hi = (krank + 1) * total / S;
        for (int e = lo + (int)threadIdx.x; e < hi; e += 192) {
            const int m = e / 128, r = e % 128;
            float v = 0.f;
            for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(part + e, 2 * s + member);
            if (a.m0 + m < a.M && row0 + r < a.N) store_out(a.y, (int64_t)(a.m0 + m) * a.N + row0 + r, v, a.out_f32);
        }
        cluster.sync();
    } else {
        // both CTAs are done with the pair's TMEM before it is released
        tc_cluster_sync_all();
    }
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(TMEM_COLS));
    }
}

// ----------------------------------------------------------------------------
// AWQ-style INT4 (group 128, uint4 zero point, fp16 scale) batched GEMM.
//
// Every group of 128 k has its own scale per weight row, so the scale cannot
// ride inside one exact tensor-core accumulation over K, and folding it into
// bf16 weights would round them. Here each 128-k stage is one group, and four
// roles run concurrently, decoupled by mbarriers:
//   * warp 0 (one elected lane) streams the packed codes (128 rows x 64 bytes) and
//     the X tile (two 64-k halves, 128-byte swizzle) with TMA into a deep ring
//     (the codes are the HBM stream; the ring holds no converted operand);
//   * the next UW warps (one thread per weight row and k-part) unpack their row's
//     codes to exact bf16 (q - z) and store them with tcgen05.st into one of
//     two A operands held in TMEM (lane = weight row; column c of a 16-k step
//     = the bf16 pair of k 2c, 2c+1 -- measured), so the 4x wider converted
//     operand never touches shared memory; they also permute the X tile's
//     16-byte chunks in place to the same k order (pairs (0,4) (1,5) (2,6)
//     (3,7), the order the nibble unpack produces; codes in the load-time
//     repacked layout unpack in natural k order and X is used as loaded);
//     the products are exact and the tensor core adds in fp32;
//   * warp 1 (one elected lane) issues the stage's MMAs (A from TMEM, X from
//     shared memory) into the groups' TMEM accumulators;
//   * the last 4 warps (one thread per weight row) read each accumulator back,
//     multiply by the row's fp32 group scale and accumulate in registers.
// The MMA issuer is the serial role: it does one commit per stage (stage
// done, waited on by both the unpack and the read-back warps) and, when there
// are as many accumulators as A operands, one wait (A ready): the unpack
// warps then check that the accumulator is free, in parallel. With fewer
// accumulators that check stays with the MMA issuer, so the unpack warps can
// still run NA groups ahead. The unpack warps wait for a ring slot once per
// slot.
// A cluster splits K for short, wide shapes (partials summed through
// distributed shared memory in rank order). Every wait is bounded; on expiry
// the kernel records the fault flag and skips the remaining work.
struct TcAwqArgs {
    const uint16_t* scales;  // fp16 [N][G]
    const uint8_t* zeros;    // uint4 [N][zstride], low nibble = even group
    void* y;
    int M, N, K, G, zstride;
    int m0;       // first batch row of this launch
    int kstages;  // groups per cluster rank
    int out_f32;
    const void* xpf;  // the launch's X rows, prefetched into L2 before the wait
    size_t xpf_bytes;
    int x_natural;    // codes in the repacked layout: X is used as loaded
};

// A ring slot holds GS groups: the codes of 128 rows x GS*64 bytes as GS/2
// TMA boxes of 128-byte rows in 128-byte-swizzled atoms (a thread per row
// then reads its row without bank conflicts), and the X tile of each group
// (two 64-k halves).
template <int NT>
struct TcAwqLayout {
    static constexpr int GS = 4;                      // groups per ring slot
    static constexpr uint32_t X_HALF = NT * 128;      // NT rows x 64 bf16 (SW128 atoms)
    static constexpr uint32_t X_GROUP = 2 * X_HALF;
    static constexpr uint32_t Q_ROW = GS * 64;        // code bytes of one row per slot
    static constexpr uint32_t Q_BOX = 128 * 128;      // one box: 128 rows x 2 groups
    static constexpr uint32_t OFF_Q = GS * X_GROUP;   // inside a ring slot
    static constexpr uint32_t SLOT = OFF_Q + 128 * Q_ROW;
    static constexpr uint32_t TX = 128 * Q_ROW + GS * X_GROUP;  // bytes TMA delivers per slot
    // The roles hand over GP groups per stage: one wait, commit and arrive
    // per stage. Each group keeps its own accumulators (its scale differs).
    static constexpr int GP = 2;                      // groups per stage
    static constexpr int NA = 4;                      // TMEM A operands (groups)
    static constexpr int A_COLS = 64;                 // TMEM columns of one 128-k A operand
    static constexpr int D_COL0 = NA * A_COLS;        // accumulators follow the A operands
    // a group's 8 MMAs rotate over C independent accumulators (one chain of
    // dependent MMAs runs at the MMA latency; the stage's two groups are two
    // chains more); NB groups' accumulators in flight
    static constexpr int C = (NT == 64) ? 1 : 2;
    static constexpr int NB = 4;
    static constexpr int NAS = NA / GP, NBS = NB / GP;  // stages in flight
    static_assert(NA % GP == 0 && NB % GP == 0 && GS % GP == 0, "");
    static constexpr int TMEM_COLS = 512;
    static_assert(D_COL0 + NB * C * NT <= TMEM_COLS, "");
    // Unpack warps: 4 row quarters x KH k-parts of a group. The unpack is
    // latency-bound with two of these warps per scheduler; at batch tile 16
    // the kernel's registers leave room for four.
    static constexpr int UW = (NT == 16) ? 16 : 8;
    static constexpr int KH = UW / 4;
    static constexpr int NWD = 16 / KH;  // 32-bit code words per lane and group (8 or 4)
    static constexpr int THREADS = 32 * (2 + UW + 4);
};

template <int NT>  // batch tile: 16, 32 or 64
__global__ void __launch_bounds__(TcAwqLayout<NT>::THREADS, 1)
    gemm_tc_awq_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapX,
                       const TcAwqArgs a, const int S, const int D) {
    using L = TcAwqLayout<NT>;
    constexpr int NB = L::NB;
    constexpr int TMEM_COLS = L::TMEM_COLS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    pdl_launch_dependents();
    prefetch_l2_grid_share(a.xpf, a.xpf_bytes);

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / S;
    const int row0 = tile * 128;
    const int ks0 = rank * a.kstages;
    const int nks = max(0, min(a.G, ks0 + a.kstages) - ks0);

    constexpr int GS = L::GS, GP = L::GP, NAS = L::NAS, NBS = L::NBS;
    const int nst = (nks + GP - 1) / GP;  // stages of GP groups
    uint8_t* ring = smem;
    uint64_t* qfull = reinterpret_cast<uint64_t*>(ring + (size_t)D * L::SLOT);
    uint64_t* empty = qfull + D;
    uint64_t* aready = empty + D;   // [NAS]: stage p's A operands are in TMEM (p % NAS)
    uint64_t* mdone = aready + NAS;  // [NAS]: stage p's MMAs are done: frees its A operands, fills its accumulators
    uint64_t* dempty = mdone + NAS;  // [NBS]: stage p's accumulators have been read back (p % NBS)
    uint64_t* done = dempty + NBS;
    static_assert(NBS <= NAS, "a stage's accumulators are reused no sooner than its A operands");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    // this CTA's scales (fp16) and zero points (one byte each) of its rows and
    // groups, loaded once: a per-group global load would put an L2 round trip
    // on every group's critical path
    uint16_t* s_tab = reinterpret_cast<uint16_t*>(done + 2);               // [kstages][128]
    uint8_t* z_tab = reinterpret_cast<uint8_t*>(s_tab + 128 * a.kstages);  // [kstages][128]

    if (threadIdx.x == 0) {
        for (int s = 0; s < D; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(&qfull[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(&empty[s])));
        }
        for (int b = 0; b < NAS; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(tc_smem(&aready[b])), "n"(L::UW));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(&mdone[b])));
        }
        for (int b = 0; b < NBS; ++b)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(tc_smem(&dempty[b])));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(done)));
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

    if (warp == 0 && lane == 0) {
        // start the code stream before anything else (codes do not depend on the previous kernel)
        const int npre = min(D, (nks + GS - 1) / GS);
        for (int j = 0; j < npre; ++j) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem(&qfull[j])), "r"(L::TX)
                         : "memory");
            for (int q = 0; q < GS / 2; ++q)
                tc_tma_2d(ring + (size_t)j * L::SLOT + L::OFF_Q + q * L::Q_BOX, &mapQ, (ks0 + j * GS + 2 * q) * 64,
                          row0, &qfull[j]);
        }
    }
    // The CTA's scale and zero tables, [group][row], loaded by all threads at
    // once (a per-group load, or a per-thread loop of dependent load/store
    // pairs, puts an L2 round trip on every group of the critical path).
    for (int e = threadIdx.x; e < nks * 128; e += L::THREADS) {
        const int i = e >> 7, rr = e & 127;
        const size_t row = (size_t)min(row0 + rr, a.N - 1);
        s_tab[i * 128 + rr] = ld_ro_u16(a.scales + row * a.G + ks0 + i);
        const uint32_t zb = ld_ro_u8(a.zeros + row * a.zstride + ((ks0 + i) >> 1));
        z_tab[i * 128 + rr] = (uint8_t)(((ks0 + i) & 1) ? (zb >> 4) : (zb & 0xF));
    }
    __syncthreads();

    float acc[NT];  // epilogue warps: this row's outputs for the launch's batch columns
#pragma unroll
    for (int c = 0; c < NT; ++c) acc[c] = 0.f;
    bool ok = true;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer ----
        const bool leader = tc_elect();
        // a slot = GS groups; codes do not depend on the previous kernel:
        // fill the ring with them first, then wait, then add the X tiles
        const int nslots = (nks + GS - 1) / GS;
        const int npre = min(D, nslots);  // slots whose codes are already on the way (issued above)
        auto load_x = [&](uint8_t* st, int j, uint64_t* bar) {
            for (int g = 0; g < GS; ++g) {
                const int kc = (ks0 + j * GS + g) * 128;
                tc_tma_2d(st + g * L::X_GROUP, &mapX, kc, a.m0, bar);
                tc_tma_2d(st + g * L::X_GROUP + L::X_HALF, &mapX, kc + 64, a.m0, bar);
            }
        };
        pdl_wait();
        if (leader)
            for (int j = 0; j < npre; ++j) load_x(ring + (size_t)j * L::SLOT, j, &qfull[j]);
        __syncwarp();
        int j = npre;
        for (; j < nslots; ++j) {
            const int s = j % D;
            if (!tc_wait_warp(&empty[s], ((j / D) - 1) & 1)) break;
            uint8_t* st = ring + (size_t)s * L::SLOT;
            if (leader) {
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem(&qfull[s])),
                             "r"(L::TX)
                             : "memory");
                for (int q = 0; q < GS / 2; ++q)
                    tc_tma_2d(st + L::OFF_Q + q * L::Q_BOX, &mapQ, (ks0 + j * GS + 2 * q) * 64, row0, &qfull[s]);
                load_x(st, j, &qfull[s]);
            }
            __syncwarp();
        }
        tc_drain_issued(qfull, j, nslots, D);  // before the __syncthreads after which the ring holds partials
    } else if (warp == 1) {
        // --------------------------------------------------- MMA issuer ----
        {
            const bool leader = tc_elect();
            const uint32_t idesc = tc_idesc(128, NT);
            for (int p = 0; p < nst; ++p) {
                const int pa = p % NAS, pb = p % NBS;
                if (ok) ok = tc_wait_warp(&aready[pa], (p / NAS) & 1);
                // accumulators free; with NBS == NAS the unpack warps checked them before aready
                if (NBS < NAS && ok && p >= NBS) ok = tc_wait_warp(&dempty[pb], ((p / NBS) - 1) & 1);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (ok && leader) {
#pragma unroll
                    for (int gg = 0; gg < GP; ++gg) {
                        const int i = p * GP + gg;
                        if (i >= nks) break;
                        const int j = i / GS, s = j % D, g = i - j * GS;
                        const uint32_t ta = tmem + (uint32_t)((pa * GP + gg) * L::A_COLS);
                        const uint32_t dcol = (uint32_t)(L::D_COL0 + (pb * GP + gg) * L::C * NT);
                        const uint32_t sx = tc_smem(ring + (size_t)s * L::SLOT + g * L::X_GROUP);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint64_t db = tc_desc(sx + h * L::X_HALF);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int kk = h * 4 + k;  // k-step of the group; accumulator kk % C
                                const uint32_t accf = (kk >= L::C) ? 1u : 0u;
                                // A: 8 TMEM columns per 16 k; X: +32 bytes per 16 k inside the swizzle atom
                                asm volatile(
                                    "{\n\t.reg .pred p;\n\t"
                                    "setp.ne.b32 p, %4, 0;\n\t"
                                    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
                                        tmem + dcol + (uint32_t)((kk % L::C) * NT)),
                                    "r"(ta + (uint32_t)(kk * 8)), "l"(db + 2 * k), "r"(idesc), "r"(accf)
                                    : "memory");
                            }
                        }
                    }
                }
                if (leader) {
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     tc_smem(&mdone[pa]))
                                 : "memory");
                    // ring slot free once the stage holding its last group is done
                    const int il = min(nks, (p + 1) * GP) - 1, jl = il / GS;
                    if (il - jl * GS == GS - 1 || il == nks - 1)
                        asm volatile(
                            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                tc_smem(&empty[jl % D]))
                            : "memory");
                }
                __syncwarp();
            }
            // every MMA issued above has completed before TMEM is released
            if (leader)
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 tc_smem(done))
                             : "memory");
            __syncwarp();
            tc_wait_warp(done, 0);
        }
    } else if (warp < 2 + L::UW) {
        // ------------------------------------------------------ unpack ----
        constexpr int NWD = L::NWD;
        const int cw = warp - 2;            // 0 .. UW-1
        const int h = cw >> 2;              // k-part of the group this warp unpacks
        const int quarter = warp & 3;       // TMEM lanes 32*quarter .. +31 (the warp's accessible quarter)
        const int r = quarter * 32 + lane;  // weight row of the tile
        for (int p = 0; p < nst; ++p) {
            const int pa = p % NAS, pb = p % NBS;
            const int i0 = p * GP, j = i0 / GS, s = j % D;
            if (i0 % GS == 0) ok = __all_sync(0xFFFFFFFFu, ok && tc_wait(&qfull[s], (j / D) & 1));  // once per slot
            if (NBS == NAS) {
                // accumulators free (stage p - NBS read back, which also means its MMAs, the users of
                // these A operands, are done): checked here, in parallel, for the MMA thread
                if (p >= NBS) ok = __all_sync(0xFFFFFFFFu, ok && tc_wait(&dempty[pb], ((p / NBS) - 1) & 1));
            } else if (p >= NAS) {
                // A operands free: stage p - NAS's MMAs are done
                ok = __all_sync(0xFFFFFFFFu, ok && tc_wait(&mdone[pa], ((p / NAS) - 1) & 1));
            }
            // all lanes take part in the (warp-collective) TMEM stores
            uint8_t* st = ring + (size_t)s * L::SLOT;
#pragma unroll
            for (int gg = 0; gg < GP; ++gg) {
                const int i = i0 + gg;
                if (i >= nks) break;
                const int g = i - j * GS;
                const uint32_t zc = z_tab[i * 128 + r];
                uint32_t av[4 * NWD];
                {
                    // row r of box g/2; 16-byte chunk c of the row sits at chunk c ^ (r & 7)
                    const uint8_t* qrow = st + L::OFF_Q + (g >> 1) * L::Q_BOX + r * 128;
                    const int c0 = (g & 1) * 4 + h * (NWD / 4);
                    uint32_t wv[NWD];
#pragma unroll
                    for (int ch = 0; ch < NWD / 4; ++ch) {
                        uint4 q = make_uint4(0, 0, 0, 0);
                        if (ok) q = *reinterpret_cast<const uint4*>(qrow + (((c0 + ch) ^ (r & 7)) << 4));
                        wv[4 * ch + 0] = q.x;
                        wv[4 * ch + 1] = q.y;
                        wv[4 * ch + 2] = q.z;
                        wv[4 * ch + 3] = q.w;
                    }
                    const uint32_t zz = (0x4300u | zc) * 0x00010001u;
#pragma unroll
                    for (int c = 0; c < NWD; ++c) {
                        av[4 * c + 0] = tc_sub(tc_nib(wv[c]), zz);
                        av[4 * c + 1] = tc_sub(tc_nib(wv[c] >> 4), zz);
                        av[4 * c + 2] = tc_sub(tc_nib(wv[c] >> 8), zz);
                        av[4 * c + 3] = tc_sub(tc_nib(wv[c] >> 12), zz);
                    }
                }
                const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) +
                                    (uint32_t)((pa * GP + gg) * L::A_COLS + h * 4 * NWD);
                if constexpr (NWD == 8) {
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
                        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(ta),
                        "r"(av[0]), "r"(av[1]), "r"(av[2]), "r"(av[3]), "r"(av[4]), "r"(av[5]), "r"(av[6]),
                        "r"(av[7]), "r"(av[8]), "r"(av[9]), "r"(av[10]), "r"(av[11]), "r"(av[12]), "r"(av[13]),
                        "r"(av[14]), "r"(av[15]), "r"(av[16]), "r"(av[17]), "r"(av[18]), "r"(av[19]), "r"(av[20]),
                        "r"(av[21]), "r"(av[22]), "r"(av[23]), "r"(av[24]), "r"(av[25]), "r"(av[26]), "r"(av[27]),
                        "r"(av[28]), "r"(av[29]), "r"(av[30]), "r"(av[31])
                        : "memory");
                } else {
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
                        "%15,%16};" ::"r"(ta),
                        "r"(av[0]), "r"(av[1]), "r"(av[2]), "r"(av[3]), "r"(av[4]), "r"(av[5]), "r"(av[6]),
                        "r"(av[7]), "r"(av[8]), "r"(av[9]), "r"(av[10]), "r"(av[11]), "r"(av[12]), "r"(av[13]),
                        "r"(av[14]), "r"(av[15])
                        : "memory");
                }
                if (ok && !a.x_natural) {
                    uint4* xs = reinterpret_cast<uint4*>(st + g * L::X_GROUP);
                    for (int c = cw * 32 + lane; c < NT * 16; c += L::UW * 32) xs[c] = tc_perm(xs[c]);
                }
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem(&aready[pa])) : "memory");
        }
    } else {
        // ---------------------------------------------------- read back ----
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
        const int r = quarter * 32 + lane;     // weight row of the tile
        for (int p = 0; p < nst; ++p) {
            const int pa = p % NAS, pb = p % NBS;
            ok = __all_sync(0xFFFFFFFFu, ok && tc_wait(&mdone[pa], (p / NAS) & 1));
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
            for (int gg = 0; gg < GP; ++gg) {
                const int i = p * GP + gg;
                if (i >= nks) break;
                const float sc = f16_bits_to_f32(s_tab[i * 128 + r]);
                // Issue the TMEM loads of up to 64 columns (all C accumulators of CB
                // 8-column blocks) before one wait: a wait after every load puts a
                // TMEM round trip per block on this role's per-group time.
                constexpr int CB = (64 / (8 * L::C)) < (NT / 8) ? (64 / (8 * L::C)) : (NT / 8);
#pragma unroll
                for (int cc0 = 0; cc0 < NT; cc0 += 8 * CB) {
                    uint32_t v[CB][L::C][8];
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb)
#pragma unroll
                        for (int ch = 0; ch < L::C; ++ch) {
                            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) +
                                                   (uint32_t)(L::D_COL0 + ((pb * GP + gg) * L::C + ch) * NT + cc0 + 8 * cb);
                            asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                                         : "=r"(v[cb][ch][0]), "=r"(v[cb][ch][1]), "=r"(v[cb][ch][2]), "=r"(v[cb][ch][3]),
                                           "=r"(v[cb][ch][4]), "=r"(v[cb][ch][5]), "=r"(v[cb][ch][6]), "=r"(v[cb][ch][7])
                                         : "r"(taddr));
                        }
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb)
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            float gsum = 0.f;
#pragma unroll
                            for (int ch = 0; ch < L::C; ++ch) gsum += __uint_as_float(v[cb][ch][jj]);
                            // the group's partial sum, scaled once by the row's group scale
                            acc[cc0 + 8 * cb + jj] = fmaf(sc, gsum, acc[cc0 + 8 * cb + jj]);
                        }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem(&dempty[pb])) : "memory");
        }
        if (S == 1) {
            // rows are the fast index of the stores: a warp writes 32 consecutive outputs per batch row
#pragma unroll
            for (int c = 0; c < NT; ++c) {
                const int m = a.m0 + c;
                if (m < a.M && row0 + r < a.N) store_out(a.y, (int64_t)m * a.N + row0 + r, ok ? acc[c] : 0.f, a.out_f32);
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();

    if (S > 1) {
        // every accumulator has been read back and every MMA is done: the ring is free for the partials
        float* part = reinterpret_cast<float*>(smem);  // [NT][128]
        if (warp >= 2 + L::UW) {
            const int r = (warp & 3) * 32 + lane;
#pragma unroll
            for (int c = 0; c < NT; ++c) part[c * 128 + r] = ok ? acc[c] : 0.f;
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int total = NT * 128;
        const int lo = rank * total / S, hi = (rank + 1) * total / S;
        for (int e = lo + (int)threadIdx.x; e < hi; e += L::THREADS) {
            const int m = e / 128, rr = e % 128;
            float v = 0.f;
            for (int s2 = 0; s2 < S; ++s2) v += *cluster.map_shared_rank(part + e, s2);
            if (a.m0 + m < a.M && row0 + rr < a.N)
                store_out(a.y, (int64_t)(a.m0 + m) * a.N + row0 + rr, v, a.out_f32);
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

static bool encode_2d_typed(CUtensorMap* map, CUtensorMapDataType dt, uint32_t esize, const void* base,
                            uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                            CUtensorMapSwizzle swz) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * esize};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [outer][inner] operand, 128-byte swizzle
static bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                      uint32_t box_outer) {
    return encode_2d_typed(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, box_inner, box_outer,
                           CU_TENSOR_MAP_SWIZZLE_128B);
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
static int tc_stages(int nt, int ring, int bps) {
    const size_t stage = (128 * 128 + (size_t)nt * 128) * bps;
    int d = (int)(((ring == 0 ? 200 : 96) * 1024) / stage);
    if (d > 8) d = 8;
    if (d < 2) d = 2;
    return d;
}

size_t tc_smem_bytes(int nt, int D, int split, int bps) {
    const size_t stage = (128 * 128 + (size_t)nt * 128) * bps;
    size_t ring = (size_t)D * stage;
    const size_t part = (size_t)nt * 128 * 4;
    if (split > 1 && part > ring) ring = part;
    return 1024 + ring + (size_t)(2 * D + 1) * 8 + 16;
}

// CTA-pair kernel: a CTA stages 128 W rows and nt/2 X rows per box.
static int tc2_stages(int nt, int ring, int bps) {
    const size_t stage = (128 * 128 + (size_t)(nt / 2) * 128) * bps;
    int d = (int)(((ring == 0 ? 200 : 96) * 1024) / stage);
    if (d > 8) d = 8;
    if (d < 2) d = 2;
    return d;
}

static size_t tc2_smem_bytes(int nt, int D, int split, int bps) {
    const size_t stage = (128 * 128 + (size_t)(nt / 2) * 128) * bps;
    size_t ring = (size_t)D * stage;
    const size_t part = (size_t)nt * 128 * 4;
    if (split > 1 && part > ring) ring = part;
    return 1024 + ring + (size_t)(2 * D + 1) * 8 + 16;
}

template <int NT, int C, int BPS>
static cudaError_t launch_nt2(const CUtensorMap& mw, const CUtensorMap& mx, const TcArgs& a, int split, int ring,
                              int tiles, cudaStream_t s) {
    const int D = tc2_stages(NT, ring, BPS);
    const size_t smem = tc2_smem_bytes(NT, D, split, BPS);
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc2_kernel<NT, C, BPS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((tiles + 1) / 2 * 2 * split), 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = (unsigned)(2 * split);
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    count_launch();
    return cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<NT, C, BPS>, mw, mx, a, split, D);
}

template <int NT, int C, int BPS>
static cudaError_t launch_nt(const CUtensorMap& mw, const CUtensorMap& mx, const TcArgs& a, int split, int ring,
                             int tiles, cudaStream_t s) {
    const int D = tc_stages(NT, ring, BPS);
    const size_t smem = tc_smem_bytes(NT, D, split, BPS);
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel<NT, C, BPS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<NT, C, BPS>, mw, mx, a, split, D);
}

// Y[M][N] = X[M][K] . W[N][K]^T, bf16, in batch slices of up to 256 rows.
// cfg bit 0: ring (0 deep, 1 co-resident); bit 1: two 64-k boxes per stage;
// bit 2: CTA pairs (batch tiles 128 and 256, split_k <= 4).
cudaError_t launch_gemm_tc(const uint16_t* X, const uint16_t* W, void* Y, int64_t M, int64_t N, int64_t K, int split,
                           int cfg_, int out_f32, cudaStream_t s) {
    const int ring = cfg_ & 1, bps = (cfg_ & 2) ? 2 : 1, pair = (cfg_ & 4) ? 1 : 0;
    const int nt = tc_batch_tile(M);
    if (pair && (nt < 128 || split > 4)) return cudaErrorInvalidValue;
    CUtensorMap mw, mx;
    if (!encode_2d(&mw, W, (uint64_t)K, (uint64_t)N, 64, 128)) return cudaErrorInvalidValue;
    if (!encode_2d(&mx, X, (uint64_t)K, (uint64_t)M, 64, (uint32_t)(pair ? nt / 2 : nt))) return cudaErrorInvalidValue;
    const int tiles = (int)((N + 127) / 128);
    const int KS = (int)((K + 64 * bps - 1) / (64 * bps));
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
        // accumulator chains: all of TMEM with one CTA per SM (deep ring),
        // half of it when the next launch's CTA shares the SM
#define MBW_TC(NT_, C0, C1)                                                                              \
    e = ring == 0 ? (bps == 2 ? launch_nt<NT_, C0, 2>(mw, mx, a, split, ring, tiles, s)                  \
                              : launch_nt<NT_, C0, 1>(mw, mx, a, split, ring, tiles, s))                 \
                  : (bps == 2 ? launch_nt<NT_, C1, 2>(mw, mx, a, split, ring, tiles, s)                  \
                              : launch_nt<NT_, C1, 1>(mw, mx, a, split, ring, tiles, s))
#define MBW_TC2(NT_, C0, C1)                                                                             \
    e = ring == 0 ? (bps == 2 ? launch_nt2<NT_, C0, 2>(mw, mx, a, split, ring, tiles, s)                 \
                              : launch_nt2<NT_, C0, 1>(mw, mx, a, split, ring, tiles, s))                \
                  : (bps == 2 ? launch_nt2<NT_, C1, 2>(mw, mx, a, split, ring, tiles, s)                 \
                              : launch_nt2<NT_, C1, 1>(mw, mx, a, split, ring, tiles, s))
        if (pair) {
            if (nt == 128)
                MBW_TC2(128, 4, 2);
            else
                MBW_TC2(256, 2, 1);
        } else {
            switch (nt) {
                case 16: MBW_TC(16, 4, 4); break;
                case 32: MBW_TC(32, 4, 4); break;
                case 64: MBW_TC(64, 4, 2); break;
                case 128: MBW_TC(128, 4, 2); break;
                default: MBW_TC(256, 2, 1); break;
            }
        }
#undef MBW_TC2
#undef MBW_TC
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// AWQ batch tile for a call of M rows (a launch covers up to 64 of them).
int tc_awq_batch_tile(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : 64; }

// bytes after the ring: barriers, TMEM slot, then the scale and zero tables
template <int NT>
static size_t tc_awq_tail_bytes(int kstages) {
    using L = TcAwqLayout<NT>;
    return (size_t)(2 * 8 + 2 * L::NA + 2 * L::NB + 2) * 8 + (size_t)128 * kstages * 3 + 16;
}

template <int NT>
static int tc_awq_stages(int kstages) {  // ring slots (of GS groups each); 0 if the tables leave no room
    const size_t budget = 210 * 1024;
    const size_t tail = tc_awq_tail_bytes<NT>(kstages);
    if (tail + 2 * TcAwqLayout<NT>::SLOT > budget) return 0;
    int d = (int)((budget - tail) / TcAwqLayout<NT>::SLOT);
    return d > 8 ? 8 : d;
}

// Whether a K split leaves room for the per-CTA scale and zero tables.
bool tc_awq_fits(int64_t M, int64_t K, int split) {
    const int G = (int)(K / 128);
    const int gs = TcAwqLayout<16>::GS;
    if (split < 1) split = 1;
    const int kst = ((G + split - 1) / split + gs - 1) / gs * gs;
    const int nt = tc_awq_batch_tile(M);
    return (nt == 16 ? tc_awq_stages<16>(kst) : nt == 32 ? tc_awq_stages<32>(kst) : tc_awq_stages<64>(kst)) >= 2;
}

template <int NT>
static cudaError_t launch_awq_nt(const CUtensorMap& mq, const CUtensorMap& mx, const TcAwqArgs& a, int split,
                                 int tiles, cudaStream_t s) {
    const int D = tc_awq_stages<NT>(a.kstages);
    if (D < 2) return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)D * TcAwqLayout<NT>::SLOT + tc_awq_tail_bytes<NT>(a.kstages);
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_awq_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * split), 1, 1);
    cfg.blockDim = dim3(TcAwqLayout<NT>::THREADS, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, gemm_tc_awq_kernel<NT>, mq, mx, a, split, D);
}

// Y[M][N] = X[M][K] . dequant(W)^T for AWQ-style INT4 weights, in batch
// slices of up to 64 rows; K split over a cluster of `split` CTAs.
cudaError_t launch_gemm_tc_awq(const uint8_t* Q, const uint16_t* scales, const uint8_t* zeros, const uint16_t* X,
                               void* Y, int64_t M, int64_t N, int64_t K, int split, int out_f32, int x_natural,
                               cudaStream_t s) {
    const int nt = tc_awq_batch_tile(M);
    CUtensorMap mq, mx;
    if (!encode_2d_typed(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Q, (uint64_t)(K / 2), (uint64_t)N, 128, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!encode_2d(&mx, X, (uint64_t)K, (uint64_t)M, 64, (uint32_t)nt)) return cudaErrorInvalidValue;
    const int tiles = (int)((N + 127) / 128);
    const int G = (int)(K / 128);
    if (split < 1) split = 1;
    if (split > G) split = G;
    TcAwqArgs a;
    a.scales = scales;
    a.zeros = zeros;
    a.y = Y;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.G = G;
    a.zstride = (G + 1) / 2;
    // whole ring slots per cluster rank (only the last rank may end inside one)
    const int gs = TcAwqLayout<16>::GS;
    a.kstages = ((G + split - 1) / split + gs - 1) / gs * gs;
    a.out_f32 = out_f32;
    a.x_natural = x_natural;
    for (int64_t m0 = 0; m0 < M; m0 += 64) {
        a.m0 = (int)m0;
        a.xpf = X + m0 * K;
        a.xpf_bytes = (size_t)((M - m0 < 64) ? (M - m0) : 64) * (size_t)K * 2;
        cudaError_t e;
        switch (nt) {
            case 16: e = launch_awq_nt<16>(mq, mx, a, split, tiles, s); break;
            case 32: e = launch_awq_nt<32>(mq, mx, a, split, tiles, s); break;
            default: e = launch_awq_nt<64>(mq, mx, a, split, tiles, s); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// The expiry path of the bounded wait, run on purpose: one thread waits on an
// mbarrier that expects one arrival that never comes. The wait gives up after
// `tries` rounds and raises the fault flag exactly as a stalled pipeline would;
// the kernel touches nothing outside its own shared memory.
__global__ void tc_wait_expiry_kernel(long long tries) {
    __shared__ __align__(8) uint64_t bar;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    (void)tc_wait(&bar, 0, tries);
}

cudaError_t launch_tc_wait_expiry(long long tries, cudaStream_t s) {
    tc_wait_expiry_kernel<<<1, 1, 0, s>>>(tries);
    count_launch();
    return cudaGetLastError();
}

int tc_take_fault() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_fault, sizeof(int)) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_tc_fault, &z, sizeof(int));
    return v;
}

}  // namespace mbw
