// gemv_tma.cu -- weight-streaming GEMV for sm_103a fed by the bulk-copy
// (TMA) engine.
//
// Same arithmetic as gemv_mma.cu (bf16 nibble pairs, exact subtract,
// mma.sync.m16n8k16 with fp32 accumulation, batch in the n columns), but the
// weights reach the SM through a shared-memory ring filled by one producer
// thread with cp.async.bulk: the consumer warps spend no issue slots on
// address arithmetic, predicates or load bookkeeping, and the ring depth, not
// the register file, sets how many bytes are in flight.
//
//   * CTA = 1 producer warp + W consumer warps. CTA row-group c of G owns the
//     contiguous 16-row tile range [c*T/G, (c+1)*T/G); a cluster of S CTAs
//     splits the k-range.
//   * A ring stage holds one tile (16 rows) x W 64-byte blocks of each row
//     (consumer warp w takes block w). Rows sit at a stride of 64*W + 64 bytes
//     so that the two rows each 8-lane phase of a 16-byte-per-lane load
//     touches fall in disjoint banks. The producer issues one bulk copy per
//     row per stage (16-byte aligned, 16-byte multiple) and arms the stage's full barrier
//     with the byte count; consumers arrive on the stage's empty barrier.
//   * Programmatic dependent launch: the producer never waits for the
//     previous grid (it only reads weights), so the ring fills while the
//     previous kernel finishes; consumers wait before staging x.
//   * Group scales (and AWQ zero points) are small: each consumer lane loads
//     its own, two stages ahead. Producer and consumers walk the (tile,
//     chunk) sequence with counters (no division in the loops).
//   * Every mbarrier wait is bounded. On expiry the kernel records the fault in
//     a device flag (read by mbw_check_device_error), the producer waits
//     (bounded) for the copies it issued, and all threads leave normally.
//
// Per-tile partial sums go to shared memory and are summed over warps (and
// over cluster ranks through distributed shared memory) once, in a fixed
// order: deterministic, no global scratch.
#include <cooperative_groups.h>

#include <algorithm>

#include "device.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace mbw {

__device__ int g_tma_fault;  // set by a bounded wait that expired

static constexpr long long kSpinLimit = MBW_WAIT_LIMIT;  // try_wait rounds before giving up

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait; returns false (and records the fault) if the phase never completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit = kSpinLimit) {
    for (long long i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicExch(&g_tma_fault, 1);
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t nibs(uint32_t v) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(0x000F000Fu), "r"(0x43004300u));
    return r;
}

__device__ __forceinline__ uint32_t bsub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint4 pair_perm(uint4 v) {
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    return o;
}

// Shared-memory layout (bytes), identical on host and device.
struct TmaSmem {
    int BK, xwords, ntmax, rowstride;
    size_t ring_off, stage_bytes, x_off, red_off, bar_off, total;
};

__host__ __device__ inline TmaSmem tma_smem_layout(int fmt, int64_t K, int N, int M, int W, int D, int S, int G) {
    TmaSmem L;
    L.BK = (fmt == FMT_BF16) ? 32 : 128;
    const int64_t KB = (K + L.BK - 1) / L.BK;
    const int64_t BS = (KB + S - 1) / S;  // blocks per cluster rank
    L.xwords = (int)(BS * (L.BK / 8));
    const int T = (N + 15) / 16;
    L.ntmax = (T + G - 1) / G;
    L.rowstride = 64 * W + 64;  // rows g and g+1 land 16 banks apart
    L.ring_off = 0;
    L.stage_bytes = (size_t)16 * L.rowstride;
    L.x_off = L.ring_off + (size_t)D * L.stage_bytes;
    const size_t x_bytes = ((size_t)M * L.xwords + L.BK / 8) * 16;  // + one block of zero words
    const size_t fin_bytes = (size_t)L.ntmax * 16 * M * 4;
    L.red_off = L.x_off + ((x_bytes > fin_bytes ? x_bytes : fin_bytes) + 15) / 16 * 16;
    const size_t red_bytes = (size_t)L.ntmax * W * 16 * M * 4;
    L.bar_off = (L.red_off + red_bytes + 15) / 16 * 16;
    L.total = L.bar_off + (size_t)2 * D * 8;
    return L;
}

template <int FMT, int W, int D>
__global__ void __launch_bounds__((W + 1) * 32)
    gemv_tma_kernel(const GemvArgs a, const int S) {
    constexpr int BK = (FMT == FMT_BF16) ? 32 : 128;
    constexpr int XW = BK / 8;
    extern __shared__ __align__(128) uint8_t smem[];

    pdl_launch_dependents();

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x / S;
    const int cgid = blockIdx.x / S;
    const int T = (a.N + 15) / 16;
    const int t0 = (int)(((long long)T * cgid) / G);
    const int nt = (int)(((long long)T * (cgid + 1)) / G) - t0;
    const int mb = a.M;
    const TmaSmem L = tma_smem_layout(FMT, a.K, a.N, mb, W, D, S, G);

    const int KB = a.K / BK;  // the plan guarantees K % BK == 0
    const int BS = (KB + S - 1) / S;
    const int cb0 = rank * BS;                       // first block of this CTA's k-range
    const int ncb = max(0, min(KB, cb0 + BS) - cb0);  // blocks in the k-range
    const int nchunk = (ncb + W - 1) / W;            // stages per tile
    const int nstage = nt * nchunk;
    const size_t rowbytes = (FMT == FMT_BF16) ? (size_t)a.K * 2 : (size_t)a.K / 2;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    uint64_t* empty = full + D;
    if (threadIdx.x == 0) {
        for (int s = 0; s < D; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == W) {
        // ------------------------------------------------------ producer ----
        if (lane == 0 && nstage > 0) {
            uint64_t policy;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
            bool ok = true;
            int s = 0, ph = 0;  // ring slot and its use count parity
            int tl = 0, c = 0;  // tile and chunk of the stage being issued
            int i = 0;
            for (; i < nstage && ok; ++i) {
                if (i >= D) ok = mbar_wait(&empty[s], ph ^ 1);
                if (!ok) break;
                const int row0 = (t0 + tl) * 16;
                const int nrows = min(16, a.N - row0);
                const int blk = cb0 + c * W;
                const uint32_t want = (uint32_t)min(W, cb0 + ncb - blk) * 64;
                mbar_expect_tx(&full[s], want * (uint32_t)nrows);
                uint8_t* st = smem + L.ring_off + (size_t)s * L.stage_bytes;
                const uint8_t* src = a.W + (size_t)row0 * rowbytes + (size_t)blk * 64;
                for (int r = 0; r < nrows; ++r)
                    bulk_g2s(st + (size_t)r * L.rowstride, src + (size_t)r * rowbytes, want, &full[s], policy);
                if (++s == D) {
                    s = 0;
                    ph ^= 1;
                }
                if (++c == nchunk) {
                    c = 0;
                    ++tl;
                }
            }
            if (!ok) {
                // drain: wait (bounded) for the copies that may still be in flight,
                // stages i - D .. i - 1 (every earlier slot was released, so its copy landed)
                for (int j = max(0, i - D); j < i; ++j) mbar_wait(&full[j % D], (j / D) & 1);
            }
        }
    } else {
        // ----------------------------------------------------- consumers ----
        const int g = lane >> 2, q = lane & 3;
        pdl_wait();
        // stage x for the CTA's k-range (+ zero words), consumer warps only
        uint4* xs = reinterpret_cast<uint4*>(smem + L.x_off);
        const int cwords = ncb * XW;
        for (int i = threadIdx.x; i < mb * L.xwords + XW; i += W * 32) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (i < mb * L.xwords) {
                const int m = i / L.xwords;
                const int wi = i - m * L.xwords;
                if (wi < cwords) v = ld_ro16(a.x + (size_t)m * a.K + (size_t)cb0 * BK + (size_t)wi * 8);
                if (FMT != FMT_BF16 && !a.x_natural) v = pair_perm(v);
            }
            xs[i] = v;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(W * 32) : "memory");

        bool xon;
        int xm;
        if (FMT == FMT_G64) {
            xm = g >> 1;
            xon = (xm < mb) && ((g & 1) == (q >> 1));
        } else {
            xm = g;
            xon = xm < mb;
        }
        // x word of (chunk c, lane): xbase + c * xcstep; lanes without x read zeros
        const uint4* xbase = xon ? xs + (size_t)xm * L.xwords + (size_t)warp * XW : xs + (size_t)mb * L.xwords;
        const int xcstep = xon ? W * XW : 0;
        float* red = reinterpret_cast<float*>(smem + L.red_off);
        const int rs = L.rowstride;
        const uint8_t* ring = smem + L.ring_off + warp * 64 + q * 16;

        // scale cursor: rows g, g+8 of (tile st, chunk sc), this warp's block
        int stt = 0, sch = 0;
        auto scale_words = [&](uint32_t& o0, uint32_t& o1) {
            o0 = o1 = 0;
            if (FMT == FMT_BF16) return;
            const int b = cb0 + sch * W + warp;
            if (stt < nt && b < cb0 + ncb) {
                const int r0 = min((t0 + stt) * 16 + g, a.N - 1);
                const int r1 = min((t0 + stt) * 16 + g + 8, a.N - 1);
                if (FMT == FMT_G64) {
                    const uint16_t* p0 = a.scales + (size_t)r0 * a.groups + 2 * b;
                    const uint16_t* p1 = a.scales + (size_t)r1 * a.groups + 2 * b;
                    o0 = (uint32_t)ld_ro_u16(p0) | ((uint32_t)ld_ro_u16(p0 + 1) << 16);
                    o1 = (uint32_t)ld_ro_u16(p1) | ((uint32_t)ld_ro_u16(p1 + 1) << 16);
                } else {
                    const uint32_t sh = (b & 1) * 4;
                    o0 = (uint32_t)ld_ro_u16(a.scales + (size_t)r0 * a.groups + b) |
                         ((((uint32_t)ld_ro_u8(a.zeros + (size_t)r0 * a.zstride + (b >> 1))) >> sh & 0xF) << 16);
                    o1 = (uint32_t)ld_ro_u16(a.scales + (size_t)r1 * a.groups + b) |
                         ((((uint32_t)ld_ro_u8(a.zeros + (size_t)r1 * a.zstride + (b >> 1))) >> sh & 0xF) << 16);
                }
            }
            if (++sch == nchunk) {
                sch = 0;
                ++stt;
            }
        };
        // scales two stages ahead: (sa0, sa1) for stage i, (sb0, sb1) for i + 1
        uint32_t sa0, sa1, sb0, sb1;
        scale_words(sa0, sa1);
        scale_words(sb0, sb1);

        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        float acc2[4] = {0.f, 0.f, 0.f, 0.f};
        bool ok = true;
        int s = 0, ph = 0, c = 0, tl = 0;
        for (int i = 0; i < nstage; ++i) {
            uint32_t sn0, sn1;
            scale_words(sn0, sn1);  // stage i + 2
            if (ok) ok = mbar_wait(&full[s], ph);
            const int b = cb0 + c * W + warp;
            if (ok && b < cb0 + ncb) {
                const uint8_t* st = ring + (size_t)s * L.stage_bytes;
                const uint4 w0 = *reinterpret_cast<const uint4*>(st + g * rs);
                const uint4 w1 = *reinterpret_cast<const uint4*>(st + (g + 8) * rs);
                const uint4* xp = xbase + (size_t)c * xcstep;
                if (FMT == FMT_BF16) {
                    const uint4 xv = xp[q];
                    mma_16816(acc, w0.x, w1.x, w0.y, w1.y, xv.x, xv.y);
                    mma_16816(acc2, w0.z, w1.z, w0.w, w1.w, xv.z, xv.w);
                } else {
                    const uint32_t zz0 = (0x4300u | ((FMT == FMT_G64) ? 8u : (sa0 >> 16))) * 0x00010001u;
                    const uint32_t zz1 = (0x4300u | ((FMT == FMT_G64) ? 8u : (sa1 >> 16))) * 0x00010001u;
                    float d0[4] = {0.f, 0.f, 0.f, 0.f};
                    float d1[4] = {0.f, 0.f, 0.f, 0.f};
                    const uint32_t wa[4] = {w0.x, w0.y, w0.z, w0.w};
                    const uint32_t wb[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint4 xv = xp[4 * q + jj];
                        mma_16816(d0, bsub(nibs(wa[jj]), zz0), bsub(nibs(wb[jj]), zz1), bsub(nibs(wa[jj] >> 4), zz0),
                                  bsub(nibs(wb[jj] >> 4), zz1), xv.x, xv.y);
                        mma_16816(d1, bsub(nibs(wa[jj] >> 8), zz0), bsub(nibs(wb[jj] >> 8), zz1),
                                  bsub(nibs(wa[jj] >> 12), zz0), bsub(nibs(wb[jj] >> 12), zz1), xv.z, xv.w);
                    }
                    if (FMT == FMT_G64) {
                        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&sa0));
                        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&sa1));
                        acc[0] = fmaf(f0.x, d0[0] + d1[0], acc[0]);
                        acc[0] = fmaf(f0.y, d0[1] + d1[1], acc[0]);
                        acc[2] = fmaf(f1.x, d0[2] + d1[2], acc[2]);
                        acc[2] = fmaf(f1.y, d0[3] + d1[3], acc[2]);
                    } else {
                        const float f0 = f16_bits_to_f32(sa0 & 0xFFFF), f1 = f16_bits_to_f32(sa1 & 0xFFFF);
                        acc[0] = fmaf(f0, d0[0] + d1[0], acc[0]);
                        acc[1] = fmaf(f0, d0[1] + d1[1], acc[1]);
                        acc[2] = fmaf(f1, d0[2] + d1[2], acc[2]);
                        acc[3] = fmaf(f1, d0[3] + d1[3], acc[3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            sa0 = sb0;
            sa1 = sb1;
            sb0 = sn0;
            sb1 = sn1;
            if (++s == D) {
                s = 0;
                ph ^= 1;
            }
            if (++c == nchunk) {
                c = 0;
                float* rp = red + ((size_t)(tl * W + warp) * 16) * mb;
                if (FMT == FMT_BF16) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[k] += acc2[k];
                }
                if (FMT == FMT_G64) {
                    if (q < mb) {
                        rp[g * mb + q] = acc[0];
                        rp[(g + 8) * mb + q] = acc[2];
                    }
                } else {
                    if (2 * q < mb) {
                        rp[g * mb + 2 * q] = acc[0];
                        rp[(g + 8) * mb + 2 * q] = acc[2];
                    }
                    if (2 * q + 1 < mb) {
                        rp[g * mb + 2 * q + 1] = acc[1];
                        rp[(g + 8) * mb + 2 * q + 1] = acc[3];
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] = acc2[k] = 0.f;
                ++tl;
            }
        }
        if (nchunk == 0) {
            for (int t = 0; t < nt; ++t) {
                float* rp = red + ((size_t)(t * W + warp) * 16) * mb;
                for (int k = lane; k < 16 * mb; k += 32) rp[k] = 0.f;
            }
        }
    }
    __syncthreads();

    // Sum over the consumer warps in warp order: fin[tile][row][m] (in the x area).
    float* red = reinterpret_cast<float*>(smem + L.red_off);
    float* fin = reinterpret_cast<float*>(smem + L.x_off);
    const int nthr = (W + 1) * 32;
    const int nout = nt * 16 * mb;
    for (int i = threadIdx.x; i < nout; i += nthr) {
        const int t = i / (16 * mb);
        const int rm = i - t * 16 * mb;
        float v = 0.f;
        for (int w = 0; w < W; ++w) v += red[((size_t)(t * W + w) * 16) * mb + rm];
        fin[i] = v;
    }
    const int row0 = t0 * 16;
    if (S == 1) {
        __syncthreads();
        for (int i = threadIdx.x; i < nout; i += nthr) {
            const int m = i / (nt * 16), lr = i - m * nt * 16;
            if (row0 + lr < a.N) store_out(a.y, (int64_t)m * a.N + row0 + lr, fin[lr * mb + m], a.out_f32);
        }
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int R = nt * 16;
    const int lo = rank * R / S, hi = (rank + 1) * R / S;
    const int span = hi - lo;
    for (int i = threadIdx.x; i < span * mb; i += nthr) {
        const int m = i / span, lr = lo + (i - m * span);
        float v = 0.f;
        for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(fin + lr * mb + m, s);
        if (row0 + lr < a.N) store_out(a.y, (int64_t)m * a.N + row0 + lr, v, a.out_f32);
    }
    cluster.sync();
}

// ------------------------------------------------------------- tables ----
using TmaFn = void (*)(const GemvArgs, const int);
struct TmaEntry {
    TmaConfig cfg;
    TmaFn fn;
};
#define MBW_T(F, W, D) \
    { {W, D}, gemv_tma_kernel<F, W, D> }

static const TmaEntry kTmaBf16[] = {MBW_T(FMT_BF16, 4, 8), MBW_T(FMT_BF16, 8, 4), MBW_T(FMT_BF16, 8, 8)};
static const TmaEntry kTmaG64[] = {MBW_T(FMT_G64, 4, 8), MBW_T(FMT_G64, 8, 4), MBW_T(FMT_G64, 8, 8)};
static const TmaEntry kTmaAwq[] = {MBW_T(FMT_AWQ, 4, 8), MBW_T(FMT_AWQ, 8, 4), MBW_T(FMT_AWQ, 8, 8)};
#undef MBW_T

static const TmaEntry* tma_table(int fmt, int* n) {
    switch (fmt) {
        case FMT_BF16:
            *n = (int)(sizeof(kTmaBf16) / sizeof(kTmaBf16[0]));
            return kTmaBf16;
        case FMT_G64:
            *n = (int)(sizeof(kTmaG64) / sizeof(kTmaG64[0]));
            return kTmaG64;
        case FMT_AWQ:
            *n = (int)(sizeof(kTmaAwq) / sizeof(kTmaAwq[0]));
            return kTmaAwq;
        default:
            *n = 0;
            return nullptr;
    }
}

int tma_num_configs(int fmt) {
    int n;
    tma_table(fmt, &n);
    return n;
}

TmaConfig tma_config(int fmt, int idx) {
    int n;
    return tma_table(fmt, &n)[idx].cfg;
}

static int tma_groups(int fmt, const TmaConfig& c, int64_t N, int64_t K, int M, int split, int occ) {
    return fitted_row_groups(N, split, occ, kSmemFit, [&](int G) {
        return tma_smem_layout(fmt, K, (int)N, M, c.warps, c.depth, split, G).total;
    });
}

size_t tma_smem_bytes(int fmt, const TmaConfig& c, int64_t N, int64_t K, int M, int split, int occ) {
    return tma_smem_layout(fmt, K, (int)N, M, c.warps, c.depth, split, tma_groups(fmt, c, N, K, M, split, occ)).total;
}

cudaError_t launch_gemv_tma(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s) {
    int n;
    const TmaEntry* t = tma_table(fmt, &n);
    if (p.cfg < 0 || p.cfg >= n || a.M < 1 || a.M > mma_max_batch(fmt)) return cudaErrorInvalidValue;
    const TmaEntry& e = t[p.cfg];
    const int G = tma_groups(fmt, e.cfg, a.N, a.K, a.M, p.split, p.occ);
    const size_t smem = tma_smem_bytes(fmt, e.cfg, a.N, a.K, a.M, p.split, p.occ);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(G * p.split), 1, 1);
    cfg.blockDim = dim3((unsigned)((e.cfg.warps + 1) * 32), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.split > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)p.split;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    count_launch();
    return cudaLaunchKernelEx(&cfg, e.fn, a, p.split);
}

// ---------------------------------------------------------- row stream ----
// BF16 weights at batch 1, fed by per-warp bulk-copy rings over whole rows.
// y[i] = sum_k W[i][k] x[k], every weight read once (llm-rs vs vLLM, sec. 2:
// single-request decode is a weight stream; the kernel's job is to keep HBM
// busy, which on this GPU means keeping ~100 KB or more in flight per SM).
//
// CTA c of G owns the rows [N c / G, N (c + 1) / G); with row-major weights
// those rows are one contiguous byte range, cut into stages of SEG bytes (the
// last one shorter). Stage s belongs to warp s % W, whose lane 0 copies it with
// one cp.async.bulk into one of the warp's D ring slots and refills the slot as
// soon as the warp has read it. Each SM thus keeps about W * D * SEG bytes in
// flight with a few large copies, the ring rather than the register file
// setting the depth, and the weights stream as long contiguous runs (the
// pattern a plain linear read sweeps at full HBM rate).
//
// Rows are 16-byte multiples, so a stage holds whole 16-byte chunks of one or
// more rows: the warp sums each row piece over its lanes (fp32) and stores the
// piece's partial in shared memory; after the stream, row i's pieces (stages
// floor(2K i / SEG) .. floor((2K (i + 1) - 1) / SEG), at most ceil(2K / SEG) + 1
// of them) are summed in stage order: deterministic, no global scratch.
//
// x is staged once per CTA as bf16 and widened at use (each 16-byte chunk of a
// row meets the matching 16 bytes of x). PDL: every warp issues its first D
// copies before waiting for the previous grid. Every wait is bounded; on
// expiry the warp stops consuming, raises the fault flag, and lane 0 waits
// (bounded) for the copies it still has in flight before the CTA exits.
struct RowsSmem {
    int P;        // partial slots per row
    int rows_max; // rows of the largest CTA share
    size_t ring_off, bar_off, x_off, part_off, total;
};

__host__ __device__ inline RowsSmem rows_smem_layout(int64_t K, int64_t N, int G, int W, int D, int SEG) {
    RowsSmem L;
    const int64_t rb = 2 * K;
    L.P = (int)((rb + SEG - 1) / SEG) + 1;
    L.rows_max = (int)((N + G - 1) / G);
    L.ring_off = 0;
    L.bar_off = (size_t)W * D * SEG;
    L.x_off = (L.bar_off + (size_t)W * D * 8 + 127) / 128 * 128;
    L.part_off = (L.x_off + (size_t)rb + 15) / 16 * 16;
    L.total = L.part_off + (size_t)L.rows_max * L.P * sizeof(float);
    return L;
}

template <int W, int D, int SEG>
__global__ void __launch_bounds__(W * 32, 2) gemv_rows_bf16_kernel(const GemvArgs a, const int G) {
    extern __shared__ __align__(128) uint8_t smem[];
    const RowsSmem L = rows_smem_layout(a.K, a.N, G, W, D, SEG);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    const uint8_t* xs = smem + L.x_off;
    float* part = reinterpret_cast<float*>(smem + L.part_off);

    pdl_launch_dependents();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rb = 2 * (int)a.K;  // bytes per row
    const int r0 = (int)((int64_t)a.N * blockIdx.x / G);
    const int r1 = (int)((int64_t)a.N * (blockIdx.x + 1) / G);
    const int64_t nbytes = (int64_t)(r1 - r0) * rb;
    const int nst = (int)((nbytes + SEG - 1) / SEG);
    const uint8_t* src = a.W + (size_t)r0 * (size_t)rb;
    uint64_t* wfull = full + warp * D;
    uint8_t* wring = smem + L.ring_off + (size_t)warp * D * SEG;

    uint64_t policy = 0;
    if (lane == 0) {
        for (int j = 0; j < D; ++j) mbar_init(&wfull[j], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    }
    // lane 0: the warp's j-th stage (stage warp + j W) into slot j % D
    auto issue = [&](int j) {
        const int st = warp + j * W;
        if (st >= nst) return;
        const int64_t off = (int64_t)st * SEG;
        const uint32_t len = (uint32_t)min((int64_t)SEG, nbytes - off);
        uint64_t* bar = &wfull[j % D];
        mbar_expect_tx(bar, len);
        bulk_g2s(wring + (size_t)(j % D) * SEG, src + off, len, bar, policy);
    };
    if (lane == 0)
        for (int j = 0; j < D; ++j) issue(j);
    __syncwarp();

    prefetch_l2_grid_share(a.x, (size_t)rb);
    pdl_wait();
    for (int i = threadIdx.x; i < rb / 16; i += W * 32)
        reinterpret_cast<uint4*>(smem + L.x_off)[i] = ld_ro16(a.x + (size_t)i * 8);
    __syncthreads();

    bool ok = true;
    int j = 0;
    for (; warp + j * W < nst; ++j) {
        const int st = warp + j * W;
        ok = __all_sync(0xffffffffu, mbar_wait(&wfull[j % D], (j / D) & 1));
        if (!ok) break;
        const int64_t b0 = (int64_t)st * SEG;
        const int64_t b1 = min(b0 + SEG, nbytes);
        const uint8_t* stage = wring + (size_t)(j % D) * SEG;
        int i = (int)(b0 / rb);  // CTA-local row of the stage's first byte
        int64_t rs = (int64_t)i * rb;
        while (rs < b1) {
            const int p0 = (int)(max(b0, rs) - b0);  // piece in stage bytes
            const int p1 = (int)(min(b1, rs + rb) - b0);
            const uint8_t* xp = xs + (b0 - rs);      // x byte for stage byte o: xp + o
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
            for (int o = p0 + lane * 16; o < p1; o += 512) {
                const uint4 w = *reinterpret_cast<const uint4*>(stage + o);
                const uint4 xv = *reinterpret_cast<const uint4*>(xp + o);
                acc0 = fmaf(bf16lo_to_f32(w.x), bf16lo_to_f32(xv.x), acc0);
                acc1 = fmaf(bf16hi_to_f32(w.x), bf16hi_to_f32(xv.x), acc1);
                acc0 = fmaf(bf16lo_to_f32(w.y), bf16lo_to_f32(xv.y), acc0);
                acc1 = fmaf(bf16hi_to_f32(w.y), bf16hi_to_f32(xv.y), acc1);
                acc0 = fmaf(bf16lo_to_f32(w.z), bf16lo_to_f32(xv.z), acc0);
                acc1 = fmaf(bf16hi_to_f32(w.z), bf16hi_to_f32(xv.z), acc1);
                acc0 = fmaf(bf16lo_to_f32(w.w), bf16lo_to_f32(xv.w), acc0);
                acc1 = fmaf(bf16hi_to_f32(w.w), bf16hi_to_f32(xv.w), acc1);
            }
            const float v = warp_sum(acc0 + acc1);
            if (lane == 0) part[i * L.P + (st - (int)(rs / SEG))] = v;
            ++i;
            rs += rb;
        }
        __syncwarp();  // every lane has read the slot
        if (lane == 0) issue(j + D);
    }
    if (!ok && lane == 0) {
        // drain: the copies issued and not yet waited for, stages j .. j + D - 1
        for (int jj = j; jj < j + D && warp + jj * W < nst; ++jj) mbar_wait(&wfull[jj % D], (jj / D) & 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < r1 - r0; i += W * 32) {
        const int64_t rs = (int64_t)i * rb;
        const int f = (int)(rs / SEG), l = (int)((rs + rb - 1) / SEG);
        float v = 0.f;
        for (int st = f; st <= l; ++st) v += part[i * L.P + (st - f)];
        store_out(a.y, r0 + i, v, a.out_f32);
    }
}

struct RowsEntry {
    RowsConfig cfg;
    TmaFn fn;
};
#define MBW_R(W, D, SEG) \
    { {W, D, SEG}, gemv_rows_bf16_kernel<W, D, SEG> }
static const RowsEntry kRows[] = {
    MBW_R(8, 3, 8192), MBW_R(8, 2, 8192), MBW_R(4, 6, 8192), MBW_R(4, 4, 8192), MBW_R(4, 3, 16384),
    MBW_R(16, 2, 4096), MBW_R(8, 4, 4096), MBW_R(8, 2, 4096), MBW_R(4, 4, 4096), MBW_R(12, 2, 8192),
    MBW_R(8, 3, 4096), MBW_R(4, 3, 8192), MBW_R(12, 2, 4096), MBW_R(8, 2, 6144), MBW_R(16, 2, 3072),
    MBW_R(4, 2, 8192), MBW_R(8, 1, 8192),
};
#undef MBW_R

int rows_num_configs() { return (int)(sizeof(kRows) / sizeof(kRows[0])); }

RowsConfig rows_config(int idx) { return kRows[idx].cfg; }

int rows_ctas(int64_t N, int occ) { return (int)std::min<int64_t>(N, (int64_t)device_sm_count() * occ); }

size_t rows_smem_bytes(const RowsConfig& c, int64_t N, int64_t K, int occ) {
    return rows_smem_layout(K, N, rows_ctas(N, occ), c.warps, c.depth, c.seg).total;
}

cudaError_t launch_gemv_rows(const Plan& p, const GemvArgs& a, cudaStream_t s) {
    if (p.cfg < 0 || p.cfg >= rows_num_configs() || a.M != 1 || p.split != 1 || p.occ < 1 || a.N < 1)
        return cudaErrorInvalidValue;
    const RowsEntry& e = kRows[p.cfg];
    const int G = rows_ctas(a.N, p.occ);
    const size_t smem = rows_smem_bytes(e.cfg, a.N, a.K, p.occ);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G, 1, 1);
    cfg.blockDim = dim3((unsigned)(e.cfg.warps * 32), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    count_launch();
    return cudaLaunchKernelEx(&cfg, e.fn, a, G);
}

// -------------------------------------------- bulk-fed INT4 / INT8 GEMV ----
// y[m][i] = sum_g s[i][g] sum_{k in g} (q[i][k] - z[i][g]) x[m][k] (tinyinfer,
// INT4 group-64 with z = 8; llm-rs vs vLLM sec. 6, the AWQ-style group-128
// layout with a zero point per group).
// INT4 codes (group-64, or AWQ-style group-128 with zero points) at batch
// 1 .. 4, with the arithmetic of the "mma2" kernels (gemv_mma.cu: each lane
// takes 32 bytes of rows g and g+8 per 128-byte super-block; n - z enters the
// MMA exactly as a bf16 pair), but fed like the row stream above: one producer
// lane copies, per stage, the 16 rows of a tile over a chunk of the CTA's
// k-range, one cp.async.bulk per row, into a ring of D stages shared by the W
// consumer warps. A register ring holds a few KB per warp; this ring holds up
// to ~170 KB per SM, issued by one thread, so the consumers spend no issue
// slots on load addresses and the stream keeps enough bytes in flight.
//
// INT8 (symmetric, one fp32 scale per output channel; TileInfer, "Pushing
// further with cheating: INT8 quantization") runs through the same ring: a
// 128-byte super-block of a row is 128 codes (128 k), a lane's 32 bytes of rows
// g and g+8 become exact bf16 pairs (i8_pairs), column n of the MMA is batch
// row n (up to 8), and the row's scale multiplies its finished sum in the store.
//
//   * stage i = (tile i / nch, chunk i % nch): rows at a stride of KC * 128 + 16
//     bytes (rows g and g + 1 then fall in different bank groups for the
//     16-byte fragment reads); consumer warp w takes super-blocks
//     w BSC .. w BSC + BSC - 1 of the chunk;
//   * full[s] (expect-tx) and empty[s] (one arrival per consumer warp); the
//     producer never waits for the previous grid, the consumers wait before
//     staging x;
//   * group scales and zero points are loaded per lane from global memory
//     one stage ahead (a few bytes per super-block);
//   * x sits in shared memory with each 8-word quarter of a super-block at
//     word 10 q (the four quarters' lanes reading word w hit four different
//     bank groups; lanes without a batch column read zero words 1 .. 8);
//   * per-tile partials are summed over warps (and cluster ranks, through
//     distributed shared memory) once, in a fixed order.
struct QbulkSmem {
    int KR;         // super-blocks per cluster rank
    int rowstride;  // bytes between rows of a stage
    int xwords;     // 16-byte x words per batch row (the rank's k-range), as laid out: 40 per super-block
    int ntmax;      // most tiles any CTA owns
    size_t stage_bytes, x_off, red_off, bar_off, total;
};

__host__ __device__ inline QbulkSmem qbulk_smem_layout(int fmt, int64_t K, int64_t N, int M, int W, int D, int BSC, int S,
                                                   int G) {
    QbulkSmem L;
    const int KB = (int)(K / (fmt == FMT_I8 ? 128 : 256));  // 128-byte super-blocks per row
    const int xp = (fmt == FMT_I8) ? 20 : 40;                // x words per super-block, as laid out
    L.KR = (KB + S - 1) / S;
    L.rowstride = W * BSC * 128 + 16;
    L.stage_bytes = (size_t)16 * L.rowstride;
    L.xwords = L.KR * xp;
    const int T = (int)((N + 15) / 16);
    L.ntmax = (T + G - 1) / G;
    L.x_off = (size_t)D * L.stage_bytes;
    const size_t x_bytes = ((size_t)M * L.xwords + xp) * 16;  // + one super-block of zero words
    const size_t fin_bytes = (size_t)L.ntmax * 16 * M * 4;    // the per-row sums, over x after the stream
    L.red_off = L.x_off + ((x_bytes > fin_bytes ? x_bytes : fin_bytes) + 15) / 16 * 16;
    L.bar_off = (L.red_off + (size_t)L.ntmax * W * 16 * M * 4 + 7) / 8 * 8;
    L.total = L.bar_off + (size_t)2 * D * 8;
    return L;
}

template <int FMT, int W, int D, int BSC>
__global__ void __launch_bounds__((W + 1) * 32, 1) gemv_qbulk_kernel(const GemvArgs a, const int S) {
    constexpr bool I8 = (FMT == FMT_I8);
    constexpr int BK = I8 ? 128 : 256;  // k per 128-byte row super-block
    constexpr int XW = BK / 8;          // 16-byte x words per super-block (logical)
    constexpr int XP = I8 ? 20 : 40;    // as laid out: each lane quarter's words at QW q
    constexpr int QW = I8 ? 5 : 10;
    constexpr int KC = W * BSC;         // super-blocks per stage
    extern __shared__ __align__(128) uint8_t smem[];

    pdl_launch_dependents();

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int G = gridDim.x / S;
    const int cgid = blockIdx.x / S;
    const int T = (a.N + 15) / 16;
    const int t0 = (int)(((long long)T * cgid) / G);
    const int nt = (int)(((long long)T * (cgid + 1)) / G) - t0;
    const int mb = a.M;
    const QbulkSmem L = qbulk_smem_layout(FMT, a.K, a.N, mb, W, D, BSC, S, G);
    const int KB = (int)(a.K / BK);
    const int kb0 = rank * L.KR;                        // the rank's first super-block
    const int krb = max(0, min(KB, kb0 + L.KR) - kb0);  // and its count
    const int nch = (krb + KC - 1) / KC;                // stages per tile
    const int nst = nt * nch;
    const size_t rowbytes = I8 ? (size_t)a.K : (size_t)a.K / 2;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    uint64_t* empty = full + D;
    if (threadIdx.x == 0) {
        for (int s = 0; s < D; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == W) {
        // -------------------------------------------------------- producer ----
        if (lane == 0 && nst > 0) {
            // the CTA's rows' scales (and zero points) into L2 first: the consumers load them per lane, a few
            // stages ahead, and would otherwise wait on DRAM for each (both ranges are contiguous)
            auto prefetch_l2 = [](const void* base, size_t bytes) {
                // whole 16-byte units inside [base, base + bytes) only: nothing outside the buffer is touched
                const uintptr_t b0 = (reinterpret_cast<uintptr_t>(base) + 15) & ~uintptr_t(15);
                const uintptr_t b1 = (reinterpret_cast<uintptr_t>(base) + bytes) & ~uintptr_t(15);
                for (uintptr_t p = b0; p < b1; p += 65536) {
                    const uint32_t n = (uint32_t)min((uintptr_t)65536, b1 - p);
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(n) : "memory");
                }
            };
            const int rlo = t0 * 16, rhi = min(a.N, (t0 + nt) * 16);
            if (I8)
                prefetch_l2(a.rscale + rlo, (size_t)(rhi - rlo) * 4);
            else
                prefetch_l2(a.scales + (size_t)rlo * a.groups, (size_t)(rhi - rlo) * a.groups * 2);
            if (FMT == FMT_AWQ) prefetch_l2(a.zeros + (size_t)rlo * a.zstride, (size_t)(rhi - rlo) * a.zstride);
            uint64_t policy;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
            bool ok = true;
            int tl = 0, ch = 0, i = 0;
            for (; i < nst; ++i) {
                const int slot = i % D;
                if (i >= D) ok = mbar_wait(&empty[slot], ((i / D) - 1) & 1);
                if (!ok) break;
                const int c0 = ch * KC;
                const uint32_t bytes = (uint32_t)min(KC, krb - c0) * 128;
                mbar_expect_tx(&full[slot], bytes * 16);
                uint8_t* st = smem + (size_t)slot * L.stage_bytes;
                const int row0 = (t0 + tl) * 16;
                const uint8_t* src = a.W + (size_t)(kb0 + c0) * 128;
                for (int r = 0; r < 16; ++r)
                    bulk_g2s(st + (size_t)r * L.rowstride, src + (size_t)min(row0 + r, a.N - 1) * rowbytes, bytes,
                             &full[slot], policy);
                if (++ch == nch) {
                    ch = 0;
                    ++tl;
                }
            }
            if (!ok) {
                // drain: the stages issued last may still be landing (earlier slots were released)
                for (int j = max(0, i - D); j < i; ++j) mbar_wait(&full[j % D], (j / D) & 1);
            }
        }
        __syncwarp();  // the whole warp reaches the block-wide barriers below together
    } else {
        // ------------------------------------------------------- consumers ----
        pdl_wait();
        uint4* xs = reinterpret_cast<uint4*>(smem + L.x_off);
        const int cwords = krb * XW;
        const int lxw = L.KR * XW;  // logical x words per batch row
        const int nxw = mb * lxw;
        for (int i0 = 0; i0 < nxw + XP; i0 += W * 32) {
            const int i = i0 + threadIdx.x;
            uint4 v = make_uint4(0, 0, 0, 0);
            int m = mb, wi = i - nxw;  // the zero block
            if (i < nxw) {
                m = i / lxw;
                wi = i - m * lxw;
                if (wi < cwords) v = ld_ro16(a.x + (size_t)m * a.K + (size_t)kb0 * BK + (size_t)wi * 8);
                if (I8)
                    v = perm_i8(v);
                else if (!a.x_natural)
                    v = pair_perm(v);
            }
            if (i < nxw + XP) {
                // logical word XW b + (XW / 4) q + w of a batch row sits at XP b + QW q + w
                const int pw = (i < nxw) ? (wi / XW) * XP + ((wi % XW) / (XW / 4)) * QW + wi % (XW / 4) : wi;
                xs[(size_t)m * L.xwords + pw] = v;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(W * 32) : "memory");

        // B fragment of this lane (column n = g): group-64 n = 4m + j, AWQ n = 2m + j, INT8 n = m
        int xm;
        bool xon;
        if (FMT == FMT_G64) {
            xm = g >> 2;
            xon = (xm < mb) && ((g & 3) == q);
        } else if (FMT == FMT_AWQ) {
            xm = g >> 1;
            xon = (xm < mb) && ((g & 1) == (q >> 1));
        } else {
            xm = g;
            xon = xm < mb;
        }
        const uint4* xrow = xon ? xs + (size_t)xm * L.xwords + QW * q : xs + (size_t)mb * L.xwords + 1;
        const int xstep = xon ? XP : 0;
        float* red = reinterpret_cast<float*>(smem + L.red_off);
        const uint16_t* sc = a.scales;

        // scales and zero points of this warp's super-blocks of stage (tl, ch), for rows g and g+8
        auto load_sc = [&](int tl, int ch, uint32_t (&s0)[BSC], uint32_t (&s1)[BSC], uint32_t (&zb)[BSC]) {
            const int row0 = (t0 + tl) * 16;
            const int r0 = min(row0 + g, a.N - 1), r1 = min(row0 + g + 8, a.N - 1);
            const int cb = ch * KC + warp * BSC;
#pragma unroll
            for (int j = 0; j < BSC; ++j) {
                const int gb = kb0 + min(cb + j, krb - 1);
                if (I8) {
                    s0[j] = s1[j] = zb[j] = 0;  // INT8: one scale per row, applied in the store
                } else if (FMT == FMT_G64) {
                    const uint16_t* p0 = sc + (size_t)r0 * a.groups + (size_t)gb * 4 + 2 * (q & 1);
                    const uint16_t* p1 = sc + (size_t)r1 * a.groups + (size_t)gb * 4 + 2 * (q & 1);
                    s0[j] = (uint32_t)ld_ro_u16(p0) | ((uint32_t)ld_ro_u16(p0 + 1) << 16);
                    s1[j] = (uint32_t)ld_ro_u16(p1) | ((uint32_t)ld_ro_u16(p1 + 1) << 16);
                    zb[j] = 0;
                } else {
                    const uint16_t* p0 = sc + (size_t)r0 * a.groups + (size_t)gb * 2;
                    const uint16_t* p1 = sc + (size_t)r1 * a.groups + (size_t)gb * 2;
                    s0[j] = (uint32_t)ld_ro_u16(p0) | ((uint32_t)ld_ro_u16(p0 + 1) << 16);
                    s1[j] = (uint32_t)ld_ro_u16(p1) | ((uint32_t)ld_ro_u16(p1 + 1) << 16);
                    zb[j] = (uint32_t)ld_ro_u8(a.zeros + (size_t)r0 * a.zstride + gb) |
                            ((uint32_t)ld_ro_u8(a.zeros + (size_t)r1 * a.zstride + gb) << 8);
                }
            }
        };
        // two stages ahead: stage i + 1 in n*, stage i + 2 in m*
        uint32_t ns0[BSC], ns1[BSC], nzb[BSC], ms0[BSC], ms1[BSC], mzb[BSC];
        if (nst > 0) load_sc(0, 0, ns0, ns1, nzb);
        if (nst > 1) load_sc(nch > 1 ? 0 : 1, nch > 1 ? 1 : 0, ms0, ms1, mzb);

        bool ok = true;
        int i = 0;
        for (int tl = 0; tl < nt && ok; ++tl) {
            float acc0 = 0.f, acc2 = 0.f;
            float c8[4] = {0.f, 0.f, 0.f, 0.f}, e8[4] = {0.f, 0.f, 0.f, 0.f};  // INT8: rows g, g+8 x columns 2q, 2q+1
            for (int ch = 0; ch < nch; ++ch, ++i) {
                const int slot = i % D;
                const int cb = ch * KC + warp * BSC;  // rank-local super-block of j = 0
                uint32_t s0[BSC], s1[BSC], zb[BSC];
#pragma unroll
                for (int j = 0; j < BSC; ++j) {
                    s0[j] = ns0[j];
                    s1[j] = ns1[j];
                    zb[j] = nzb[j];
                    ns0[j] = ms0[j];
                    ns1[j] = ms1[j];
                    nzb[j] = mzb[j];
                }
                if (i + 2 < nst) {  // stage i + 2: (tl, ch + 2) or into the next tile
                    int t2 = tl, c2 = ch + 2;
                    while (c2 >= nch) {
                        c2 -= nch;
                        ++t2;
                    }
                    load_sc(t2, c2, ms0, ms1, mzb);
                }
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full[slot], (i / D) & 1));
                if (!ok) break;
                const uint8_t* st = smem + (size_t)slot * L.stage_bytes + (size_t)g * L.rowstride +
                                    (size_t)(warp * BSC) * 128 + q * 32;
#pragma unroll
                for (int j = 0; j < BSC; ++j) {
                    if (cb + j < krb) {
                        const uint8_t* p = st + j * 128;
                        const uint4 a0 = *reinterpret_cast<const uint4*>(p);
                        const uint4 a1 = *reinterpret_cast<const uint4*>(p + 16);
                        const uint4 c0 = *reinterpret_cast<const uint4*>(p + 8 * L.rowstride);
                        const uint4 c1 = *reinterpret_cast<const uint4*>(p + 8 * L.rowstride + 16);
                        const uint4* xp = xrow + (size_t)(cb + j) * xstep;
                        if (I8) {
                            // word w of rows g and g+8: codes (0,2) and (1,3) as exact bf16 pairs, one MMA
                            // per word; x is in the matching pair order (perm_i8), 4 words per lane
                            const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                            const uint32_t wb[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                            for (int w = 0; w < 8; w += 2) {
                                const uint4 xv = xp[w >> 1];
                                uint32_t p0, p1, p2, p3;
                                i8_pairs(wa[w], p0, p2);
                                i8_pairs(wb[w], p1, p3);
                                mma_16816(c8, p0, p1, p2, p3, xv.x, xv.y);
                                i8_pairs(wa[w + 1], p0, p2);
                                i8_pairs(wb[w + 1], p1, p3);
                                mma_16816(e8, p0, p1, p2, p3, xv.z, xv.w);
                            }
                            continue;
                        }
                        // n - z as exact bf16 pairs (128 + n minus 128 + z; AWQ: this lane's group
                        // is q >> 1, low or high nibble of the zero byte; group-64: z = 8)
                        uint32_t zz0, zz1;
                        if (FMT == FMT_G64) {
                            zz0 = zz1 = 0x43084308u;
                        } else {
                            const uint32_t sh = (q >> 1) * 4;
                            zz0 = (0x4300u | ((zb[j] >> sh) & 0xF)) * 0x00010001u;
                            zz1 = (0x4300u | ((zb[j] >> (8 + sh)) & 0xF)) * 0x00010001u;
                        }
                        // four accumulator sets: chains of 4 dependent MMAs instead of 8
                        float d0[4] = {0.f, 0.f, 0.f, 0.f};
                        float d1[4] = {0.f, 0.f, 0.f, 0.f};
                        float e0[4] = {0.f, 0.f, 0.f, 0.f};
                        float e1[4] = {0.f, 0.f, 0.f, 0.f};
                        const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                        const uint32_t wb[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                        for (int w = 0; w < 8; w += 2) {
                            const uint4 xv = xp[w], xu = xp[w + 1];
                            mma_16816(d0, bsub(nibs(wa[w]), zz0), bsub(nibs(wb[w]), zz1), bsub(nibs(wa[w] >> 4), zz0),
                                      bsub(nibs(wb[w] >> 4), zz1), xv.x, xv.y);
                            mma_16816(d1, bsub(nibs(wa[w] >> 8), zz0), bsub(nibs(wb[w] >> 8), zz1),
                                      bsub(nibs(wa[w] >> 12), zz0), bsub(nibs(wb[w] >> 12), zz1), xv.z, xv.w);
                            mma_16816(e0, bsub(nibs(wa[w + 1]), zz0), bsub(nibs(wb[w + 1]), zz1),
                                      bsub(nibs(wa[w + 1] >> 4), zz0), bsub(nibs(wb[w + 1] >> 4), zz1), xu.x, xu.y);
                            mma_16816(e1, bsub(nibs(wa[w + 1] >> 8), zz0), bsub(nibs(wb[w + 1] >> 8), zz1),
                                      bsub(nibs(wa[w + 1] >> 12), zz0), bsub(nibs(wb[w + 1] >> 12), zz1), xu.z, xu.w);
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            d0[e] += e0[e];
                            d1[e] += e1[e];
                        }
                        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&s0[j]));
                        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&s1[j]));
                        acc0 = fmaf(f0.x, d0[0] + d1[0], acc0);
                        acc0 = fmaf(f0.y, d0[1] + d1[1], acc0);
                        acc2 = fmaf(f1.x, d0[2] + d1[2], acc2);
                        acc2 = fmaf(f1.y, d0[3] + d1[3], acc2);
                    }
                }
                __syncwarp();  // every lane has read the stage
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
            if (!ok) break;
            float* rp = red + ((size_t)(tl * W + warp) * 16) * mb;
            if (I8) {
                if (2 * q < mb) {
                    rp[g * mb + 2 * q] = c8[0] + e8[0];
                    rp[(g + 8) * mb + 2 * q] = c8[2] + e8[2];
                }
                if (2 * q + 1 < mb) {
                    rp[g * mb + 2 * q + 1] = c8[1] + e8[1];
                    rp[(g + 8) * mb + 2 * q + 1] = c8[3] + e8[3];
                }
            } else if (FMT == FMT_G64) {
                // lanes q and q^1 hold the other two groups of the same batch
                const float v0 = acc0 + __shfl_xor_sync(0xFFFFFFFFu, acc0, 1);
                const float v2 = acc2 + __shfl_xor_sync(0xFFFFFFFFu, acc2, 1);
                const int m = q >> 1;
                if ((q & 1) == 0 && m < mb) {
                    rp[g * mb + m] = v0;
                    rp[(g + 8) * mb + m] = v2;
                }
            } else if (q < mb) {
                rp[g * mb + q] = acc0;
                rp[(g + 8) * mb + q] = acc2;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(W * 32) : "memory");
        float* fin = reinterpret_cast<float*>(smem + L.x_off);  // [tile row][m]: sums over the warps
        for (int k = threadIdx.x; k < nt * 16 * mb; k += W * 32) {
            const int t = k / (16 * mb);
            const int rm = k - t * 16 * mb;
            float v = 0.f;
            for (int w = 0; w < W; ++w) v += red[((size_t)(t * W + w) * 16) * mb + rm];
            fin[k] = v;
        }
    }
    float* fin = reinterpret_cast<float*>(smem + L.x_off);
    if (S == 1) {
        __syncthreads();
        for (int k = threadIdx.x; k < nt * 16 * mb; k += (W + 1) * 32) {
            const int m = k / (nt * 16), o = k - m * nt * 16;
            const int row = t0 * 16 + o;
            if (row < a.N) {
                float v = fin[o * mb + m];
                if (I8) v *= __ldg(a.rscale + row);
                store_out(a.y, (int64_t)m * a.N + row, v, a.out_f32);
            }
        }
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    // rank s writes rows [s Ro / S, (s + 1) Ro / S) of the CTA group's Ro rows, every batch row
    const int Ro = nt * 16;
    const int lo = rank * Ro / S, hi = (rank + 1) * Ro / S;
    const int span = hi - lo;
    for (int k = threadIdx.x; k < span * mb; k += (W + 1) * 32) {
        const int m = k / span, o = lo + (k - m * span);
        float v = 0.f;
        for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(fin + o * mb + m, s);
        const int row = t0 * 16 + o;
        if (row < a.N) {
            if (I8) v *= __ldg(a.rscale + row);
            store_out(a.y, (int64_t)m * a.N + row, v, a.out_f32);
        }
    }
    cluster.sync();
}

struct QbulkEntry {
    QbulkConfig cfg;
    TmaFn fn;
};
#define MBW_B(F, W, D, B) \
    { {W, D, B}, gemv_qbulk_kernel<F, W, D, B> }
static const QbulkEntry kQbulkG64[] = {MBW_B(FMT_G64, 8, 4, 1),  MBW_B(FMT_G64, 8, 6, 1),  MBW_B(FMT_G64, 4, 6, 2),
                                   MBW_B(FMT_G64, 7, 6, 2),  MBW_B(FMT_G64, 8, 4, 2),  MBW_B(FMT_G64, 4, 4, 2),
                                   MBW_B(FMT_G64, 14, 6, 1), MBW_B(FMT_G64, 16, 5, 1), MBW_B(FMT_G64, 11, 4, 2)};
static const QbulkEntry kQbulkAwq[] = {MBW_B(FMT_AWQ, 8, 4, 1),  MBW_B(FMT_AWQ, 8, 6, 1),  MBW_B(FMT_AWQ, 4, 6, 2),
                                   MBW_B(FMT_AWQ, 7, 6, 2),  MBW_B(FMT_AWQ, 8, 4, 2),  MBW_B(FMT_AWQ, 4, 4, 2),
                                   MBW_B(FMT_AWQ, 14, 6, 1), MBW_B(FMT_AWQ, 16, 5, 1), MBW_B(FMT_AWQ, 11, 4, 2)};

static const QbulkEntry kQbulkI8[] = {MBW_B(FMT_I8, 10, 4, 2), MBW_B(FMT_I8, 5, 6, 4),  MBW_B(FMT_I8, 8, 6, 1),
                                    MBW_B(FMT_I8, 16, 5, 1), MBW_B(FMT_I8, 16, 3, 2), MBW_B(FMT_I8, 4, 6, 2),
                                    MBW_B(FMT_I8, 8, 4, 2)};
#undef MBW_B

static const QbulkEntry* qbulk_table(int fmt, int* n) {
    if (fmt == FMT_G64) {
        *n = (int)(sizeof(kQbulkG64) / sizeof(kQbulkG64[0]));
        return kQbulkG64;
    }
    if (fmt == FMT_AWQ) {
        *n = (int)(sizeof(kQbulkAwq) / sizeof(kQbulkAwq[0]));
        return kQbulkAwq;
    }
    if (fmt == FMT_I8) {
        *n = (int)(sizeof(kQbulkI8) / sizeof(kQbulkI8[0]));
        return kQbulkI8;
    }
    *n = 0;
    return nullptr;
}

int qbulk_num_configs(int fmt) {
    int n;
    qbulk_table(fmt, &n);
    return n;
}

QbulkConfig qbulk_config(int fmt, int idx) {
    int n;
    return qbulk_table(fmt, &n)[idx].cfg;
}

// (occ CTAs of this kernel share an SM's 227 KB)
static int qbulk_groups(int fmt, const QbulkConfig& c, int64_t N, int64_t K, int M, int split, int occ) {
    return fitted_row_groups(N, split, occ, (size_t)227 * 1024 / occ, [&](int G) {
        return qbulk_smem_layout(fmt, K, N, M, c.warps, c.depth, c.bsc, split, G).total;
    });
}

size_t qbulk_smem_bytes(int fmt, const QbulkConfig& c, int64_t N, int64_t K, int M, int split, int occ) {
    return qbulk_smem_layout(fmt, K, N, M, c.warps, c.depth, c.bsc, split, qbulk_groups(fmt, c, N, K, M, split, occ))
        .total;
}

cudaError_t launch_gemv_qbulk(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s) {
    int n;
    const QbulkEntry* t = qbulk_table(fmt, &n);
    if (!t || p.cfg < 0 || p.cfg >= n || a.M < 1 || a.M > mma2_max_batch(fmt) || a.K % (fmt == FMT_I8 ? 128 : 256) != 0 ||
        a.glu)
        return cudaErrorInvalidValue;
    const QbulkEntry& e = t[p.cfg];
    const int G = qbulk_groups(fmt, e.cfg, a.N, a.K, a.M, p.split, p.occ);
    const size_t smem = qbulk_smem_bytes(fmt, e.cfg, a.N, a.K, a.M, p.split, p.occ);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(G * p.split), 1, 1);
    cfg.blockDim = dim3((unsigned)((e.cfg.warps + 1) * 32), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.split > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)p.split;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    count_launch();
    return cudaLaunchKernelEx(&cfg, e.fn, a, p.split);
}

// The expiry path of the bounded wait, run on purpose: one thread waits on an
// mbarrier whose single expected arrival never comes, gives up after `tries`
// rounds and raises the fault flag; nothing outside its shared memory is touched.
__global__ void tma_wait_expiry_kernel(long long tries) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    (void)mbar_wait(&bar, 0, tries);
}

cudaError_t launch_tma_wait_expiry(long long tries, cudaStream_t s) {
    tma_wait_expiry_kernel<<<1, 1, 0, s>>>(tries);
    count_launch();
    return cudaGetLastError();
}

// Read and clear the fault flag of the bounded waits (host side).
int tma_take_fault() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_tma_fault, sizeof(int)) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_tma_fault, &z, sizeof(int));
    return v;
}

}  // namespace mbw
