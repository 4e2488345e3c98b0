// gemv_mma.cu -- weight-streaming GEMV for sm_103a with the tensor core as the
// multiply-add unit.
//
// Y[m][i] = sum_k X[m][k] * w(i, k) for BF16, INT4 group-64 and AWQ-style INT4
// group-128 weights and a small batch M (1..8; 1..4 for group-64).
//
// Why mma here: at batch 1 every weight is used for one multiply-add (llm-rs
// vs vLLM, sec. 2), so the kernel must retire ~41 INT4 weights per SM clock to
// keep up with HBM on GB300 -- about 3 issue slots per weight. Unpacking a
// nibble and doing the fp32 multiply-add on the CUDA cores costs ~4. Here the
// CUDA cores only turn codes into bf16 pairs (one LOP3 per two codes, one
// exact bf16 subtract), and mma.sync.m16n8k16 retires the multiply-adds with
// fp32 accumulation, taking its A operand straight from the registers the
// weight stream was loaded into. The batch rides in the MMA's n = 8 columns.
// (tcgen05 would need the operand staged through shared memory and a TMEM
// round trip per group; the batched skinny GEMM uses it where M >= 16.)
//
// Work decomposition:
//   * warp task = 16*R16 weight rows x one k-slice; lane (g = lane/4,
//     q = lane%4) loads 16 bytes of rows g and g+8 per 64-byte block of each
//     row, i.e. the 4 lanes of a quad read 64 contiguous bytes of a row;
//   * CTA = (W / WK) row tiles x WK k-slices; a cluster of S CTAs splits K
//     further. Partial sums are reduced in shared memory across the CTA's
//     k-slices and through distributed shared memory across the cluster, in a
//     fixed order (deterministic, no global scratch, no spin waits);
//   * every lane keeps U blocks of weights in flight (register double
//     buffer); with programmatic dependent launch the first U blocks are
//     requested before the kernel waits for the previous grid, and x is read
//     only after that wait;
//   * x (the CTA's k-range) is staged once per CTA in shared memory, in the
//     order the B fragments need it.
//
// Exactness: a code n in a bf16 pair is built as 0x4300 | n = 128 + n, and
// 128 + n - (128 + z) = n - z is exact in bf16; products (n - z) * x are exact
// and the tensor core accumulates in fp32. The group scale multiplies the
// group's fp32 partial sum. BF16 weights go to the tensor core unchanged.
#include <cooperative_groups.h>

#include "device.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace mbw {

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (v & 0x000F000F) | 0x43004300: the two nibbles at bits 0-3 and 16-19 as
// bf16 values 128 + n.
__device__ __forceinline__ uint32_t nib_pair(uint32_t v) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(0x000F000Fu), "r"(0x43004300u));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// x staging: 8 bf16 x[8w..8w+7] -> pairs (0,4) (1,5) (2,6) (3,7), the order in
// which the INT4 A fragments pair their nibbles.
__device__ __forceinline__ uint4 perm_pairs(uint4 v) {
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);  // x0 | x4 << 16
    o.y = __byte_perm(v.x, v.z, 0x7632);  // x1 | x5 << 16
    o.z = __byte_perm(v.y, v.w, 0x5410);  // x2 | x6 << 16
    o.w = __byte_perm(v.y, v.w, 0x7632);  // x3 | x7 << 16
    return o;
}

template <int FMT>
struct MmaTraits;
template <>
struct MmaTraits<FMT_BF16> {
    static constexpr int BK = 32;  // k per 64-byte row block
};
template <>
struct MmaTraits<FMT_G64> {
    static constexpr int BK = 128;
};
template <>
struct MmaTraits<FMT_AWQ> {
    static constexpr int BK = 128;
};

template <int FMT, int W, int R16, int U>
__global__ void __launch_bounds__(W * 32)
    gemv_mma_kernel(const GemvArgs a, const int S, const int WK) {
    constexpr int BK = MmaTraits<FMT>::BK;
    constexpr int WPB = (FMT == FMT_BF16) ? 1 : 4;  // 16-byte x words per quad lane per block
    extern __shared__ uint4 smem_u4[];

    pdl_launch_dependents();

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int wr = warp / WK, wk = warp - wr * WK;
    const int KB = (a.K + BK - 1) / BK;
    const int TS = S * WK;
    const int BS = (KB + TS - 1) / TS;
    const int b0 = (rank * WK + wk) * BS;
    const int b1 = min(KB, b0 + BS);
    const int nblk = max(0, b1 - b0);
    const int iters = (nblk + U - 1) / U;
    const int cb0 = rank * WK * BS;  // first block of this CTA's k-range
    const int cnb = max(0, min(KB, cb0 + WK * BS) - cb0);
    const int rows_cta = (W / WK) * 16 * R16;
    const int tile_row = (blockIdx.x / S) * rows_cta + wr * 16 * R16;
    const size_t rowbytes = (FMT == FMT_BF16) ? (size_t)a.K * 2 : (size_t)a.K / 2;

    int rowc[R16][2];
    const uint8_t* wp[R16][2];
#pragma unroll
    for (int r = 0; r < R16; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            rowc[r][h] = min(tile_row + 16 * r + g + 8 * h, a.N - 1);
            wp[r][h] = a.W + (size_t)rowc[r][h] * rowbytes + q * 16;
        }

    uint4 cur[U][R16][2];
    uint32_t scur[U][R16][2];  // g64: two fp16 scales; AWQ: fp16 scale | zero << 16

    auto load = [&](uint4 (&buf)[U][R16][2], uint32_t (&sb)[U][R16][2], int it) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + it * U + u;
            const bool ok = (b < b1) && ((b * BK + (q + 1) * (BK / 4)) <= a.K);
#pragma unroll
            for (int r = 0; r < R16; ++r)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    buf[u][r][h] = ok ? ld_stream16(wp[r][h] + (size_t)b * 64) : make_uint4(0, 0, 0, 0);
                    if (FMT == FMT_G64) {
                        const int gi = 2 * b;
                        const uint16_t* sp = a.scales + (size_t)rowc[r][h] * a.groups + gi;
                        const uint32_t s0 = (b < b1) ? ld_ro_u16(sp) : 0;
                        const uint32_t s1 = (b < b1 && gi + 1 < a.groups) ? ld_ro_u16(sp + 1) : 0;
                        sb[u][r][h] = s0 | (s1 << 16);
                    } else if (FMT == FMT_AWQ) {
                        const uint32_t s = (b < b1) ? ld_ro_u16(a.scales + (size_t)rowc[r][h] * a.groups + b) : 0;
                        const uint32_t zb =
                            (b < b1) ? ld_ro_u8(a.zeros + (size_t)rowc[r][h] * a.zstride + (b >> 1)) : 0;
                        const uint32_t z = (b & 1) ? (zb >> 4) : (zb & 0xF);
                        sb[u][r][h] = s | (z << 16);
                    }
                }
        }
    };

    if (iters > 0) load(cur, scur, 0);

    pdl_wait();

    // Stage x for blocks [cb0, cb0 + cnb) of every batch row:
    // xs[m][(b - cb0) * (BK / 8) + word] (16-byte words of 8 k; INT4 pairs permuted).
    const int mb = a.M;
    const int xwords = cnb * (BK / 8);
    for (int i = threadIdx.x; i < mb * xwords; i += W * 32) {
        const int m = i / xwords;
        const int wi = i - m * xwords;
        const int k = cb0 * BK + wi * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (k < a.K) v = ld_ro16(a.x + (size_t)m * a.K + k);
        smem_u4[i] = (FMT == FMT_BF16) ? v : perm_pairs(v);
    }
    __syncthreads();

    // B-fragment source of this lane: column n = g.
    int xm;
    bool xon;
    if (FMT == FMT_G64) {
        xm = g >> 1;
        xon = (xm < mb) && ((g & 1) == (q >> 1));
    } else {
        xm = g;
        xon = xm < mb;
    }
    const uint4* xrow = smem_u4 + (size_t)(xon ? xm : 0) * xwords;

    float acc[R16][4];
#pragma unroll
    for (int r = 0; r < R16; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[r][i] = 0.f;

    for (int it = 0; it < iters; ++it) {
        uint4 nxt[U][R16][2];
        uint32_t snxt[U][R16][2];
        if (it + 1 < iters) load(nxt, snxt, it + 1);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + it * U + u;
            if (b < b1) {
                const int lb = b - cb0;
                if (FMT == FMT_BF16) {
                    const uint4 xv = xon ? xrow[lb * 4 + q] : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int r = 0; r < R16; ++r) {
                        const uint4 wg = cur[u][r][0], wg8 = cur[u][r][1];
                        mma_bf16_16816(acc[r], wg.x, wg8.x, wg.y, wg8.y, xv.x, xv.y);
                        mma_bf16_16816(acc[r], wg.z, wg8.z, wg.w, wg8.w, xv.z, xv.w);
                    }
                } else {
                    uint4 xv[WPB];
#pragma unroll
                    for (int j = 0; j < WPB; ++j) xv[j] = xon ? xrow[lb * 16 + 4 * q + j] : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int r = 0; r < R16; ++r) {
                        uint32_t zz[2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t z = (FMT == FMT_G64) ? 8u : (scur[u][r][h] >> 16);
                            zz[h] = (0x4300u | z) * 0x00010001u;  // (128 + z, 128 + z)
                        }
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        const uint32_t* wg = &cur[u][r][0].x;
                        const uint32_t* wg8 = &cur[u][r][1].x;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const int sh = 8 * hh;
                                const uint32_t a0 = bf16x2_sub(nib_pair(wg[j] >> sh), zz[0]);
                                const uint32_t a2 = bf16x2_sub(nib_pair(wg[j] >> (sh + 4)), zz[0]);
                                const uint32_t a1 = bf16x2_sub(nib_pair(wg8[j] >> sh), zz[1]);
                                const uint32_t a3 = bf16x2_sub(nib_pair(wg8[j] >> (sh + 4)), zz[1]);
                                const uint32_t bb0 = hh ? xv[j].z : xv[j].x;
                                const uint32_t bb1 = hh ? xv[j].w : xv[j].y;
                                mma_bf16_16816(d, a0, a1, a2, a3, bb0, bb1);
                            }
                        }
                        if (FMT == FMT_G64) {
                            // columns 2m (even group) and 2m + 1 (odd group) of batch m = q
                            const uint32_t sg = scur[u][r][0], sg8 = scur[u][r][1];
                            acc[r][0] = fmaf(f16_bits_to_f32(sg & 0xFFFF), d[0], acc[r][0]);
                            acc[r][0] = fmaf(f16_bits_to_f32(sg >> 16), d[1], acc[r][0]);
                            acc[r][2] = fmaf(f16_bits_to_f32(sg8 & 0xFFFF), d[2], acc[r][2]);
                            acc[r][2] = fmaf(f16_bits_to_f32(sg8 >> 16), d[3], acc[r][2]);
                        } else {
                            const float sg = f16_bits_to_f32(scur[u][r][0] & 0xFFFF);
                            const float sg8 = f16_bits_to_f32(scur[u][r][1] & 0xFFFF);
                            acc[r][0] = fmaf(sg, d[0], acc[r][0]);
                            acc[r][1] = fmaf(sg, d[1], acc[r][1]);
                            acc[r][2] = fmaf(sg8, d[2], acc[r][2]);
                            acc[r][3] = fmaf(sg8, d[3], acc[r][3]);
                        }
                    }
                }
            }
        }
        if (it + 1 < iters) {
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < R16; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        cur[u][r][h] = nxt[u][r][h];
                        scur[u][r][h] = snxt[u][r][h];
                    }
        }
    }

    // Partial sums -> red[row_in_cta][k-slice][m] (8 batch columns), then a
    // fixed-order sum over the CTA's k-slices and the cluster's ranks.
    __syncthreads();  // x staging area is reused
    float* red = reinterpret_cast<float*>(smem_u4);
#pragma unroll
    for (int r = 0; r < R16; ++r) {
        const int lr0 = wr * 16 * R16 + 16 * r + g;
        if (FMT == FMT_G64) {
            red[(lr0 * WK + wk) * 8 + q] = acc[r][0];
            red[((lr0 + 8) * WK + wk) * 8 + q] = acc[r][2];
            // columns 4..7 are never used for group-64 (batch <= 4)
        } else {
            red[(lr0 * WK + wk) * 8 + 2 * q] = acc[r][0];
            red[(lr0 * WK + wk) * 8 + 2 * q + 1] = acc[r][1];
            red[((lr0 + 8) * WK + wk) * 8 + 2 * q] = acc[r][2];
            red[((lr0 + 8) * WK + wk) * 8 + 2 * q + 1] = acc[r][3];
        }
    }
    __syncthreads();
    const int nout = rows_cta * mb;
    float* fin = red + rows_cta * WK * 8;  // per-CTA sums [row][m]
    for (int t = threadIdx.x; t < nout; t += W * 32) {
        const int lr = t / mb, m = t - lr * mb;
        float v = 0.f;
        for (int k = 0; k < WK; ++k) v += red[(lr * WK + k) * 8 + m];
        fin[t] = v;
    }
    const int row_base = (blockIdx.x / S) * rows_cta;
    if (S == 1) {
        __syncthreads();
        for (int t = threadIdx.x; t < nout; t += W * 32) {
            const int m = t / rows_cta, lr = t - m * rows_cta;
            if (row_base + lr < a.N) store_out(a.y, (int64_t)m * a.N + row_base + lr, fin[lr * mb + m], a.out_f32);
        }
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    // rank s writes the rows [s * rows_cta / S, (s + 1) * rows_cta / S) of every batch row
    const int lo = rank * rows_cta / S, hi = (rank + 1) * rows_cta / S;
    const int span = hi - lo;
    for (int t = threadIdx.x; t < span * mb; t += W * 32) {
        const int m = t / span, lr = lo + (t - m * span);
        float v = 0.f;
        for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(fin + lr * mb + m, s);
        if (row_base + lr < a.N) store_out(a.y, (int64_t)m * a.N + row_base + lr, v, a.out_f32);
    }
    cluster.sync();
}

// ------------------------------------------------------------- tables ----
using MmaFn = void (*)(const GemvArgs, const int, const int);
struct MmaEntry {
    MmaConfig cfg;
    MmaFn fn;
};
#define MBW_M(F, W, R, U) \
    { {W, R, U}, gemv_mma_kernel<F, W, R, U> }

static const MmaEntry kMmaBf16[] = {
    MBW_M(FMT_BF16, 4, 1, 4), MBW_M(FMT_BF16, 4, 2, 4), MBW_M(FMT_BF16, 8, 1, 4), MBW_M(FMT_BF16, 8, 2, 2),
    MBW_M(FMT_BF16, 8, 1, 8),
};
static const MmaEntry kMmaG64[] = {
    MBW_M(FMT_G64, 4, 1, 2), MBW_M(FMT_G64, 4, 2, 2), MBW_M(FMT_G64, 8, 1, 2), MBW_M(FMT_G64, 8, 2, 1),
    MBW_M(FMT_G64, 8, 1, 4), MBW_M(FMT_G64, 4, 1, 4),
};
static const MmaEntry kMmaAwq[] = {
    MBW_M(FMT_AWQ, 4, 1, 2), MBW_M(FMT_AWQ, 4, 2, 2), MBW_M(FMT_AWQ, 8, 1, 2), MBW_M(FMT_AWQ, 8, 2, 1),
    MBW_M(FMT_AWQ, 8, 1, 4), MBW_M(FMT_AWQ, 4, 1, 4),
};
#undef MBW_M

static const MmaEntry* mma_table(int fmt, int* n) {
    switch (fmt) {
        case FMT_BF16:
            *n = (int)(sizeof(kMmaBf16) / sizeof(kMmaBf16[0]));
            return kMmaBf16;
        case FMT_G64:
            *n = (int)(sizeof(kMmaG64) / sizeof(kMmaG64[0]));
            return kMmaG64;
        default:
            *n = (int)(sizeof(kMmaAwq) / sizeof(kMmaAwq[0]));
            return kMmaAwq;
    }
}

int mma_num_configs(int fmt) {
    int n;
    mma_table(fmt, &n);
    return n;
}

MmaConfig mma_config(int fmt, int idx) {
    int n;
    return mma_table(fmt, &n)[idx].cfg;
}

int mma_max_batch(int fmt) { return fmt == FMT_G64 ? 4 : 8; }

size_t mma_smem_bytes(int fmt, const MmaConfig& c, int64_t K, int M, int split, int wk) {
    const int BK = (fmt == FMT_BF16) ? 32 : 128;
    const int64_t KB = (K + BK - 1) / BK;
    const int64_t TS = (int64_t)split * wk;
    const int64_t BS = (KB + TS - 1) / TS;
    const size_t xs = (size_t)M * (size_t)(wk * BS) * (BK / 8) * 16;
    const int rows_cta = (c.warps / wk) * 16 * c.r16;
    const size_t red = (size_t)rows_cta * wk * 8 * 4 + (size_t)rows_cta * 8 * 4;
    return xs > red ? xs : red;
}

cudaError_t launch_gemv_mma(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s) {
    int n;
    const MmaEntry* t = mma_table(fmt, &n);
    if (p.cfg < 0 || p.cfg >= n) return cudaErrorInvalidValue;
    const MmaEntry& e = t[p.cfg];
    if (e.cfg.warps % p.wk != 0) return cudaErrorInvalidValue;
    const int rows_cta = (e.cfg.warps / p.wk) * 16 * e.cfg.r16;
    const int groups = (a.N + rows_cta - 1) / rows_cta;
    const size_t smem = mma_smem_bytes(fmt, e.cfg, a.K, a.M, p.split, p.wk);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(groups * p.split), 1, 1);
    cfg.blockDim = dim3((unsigned)(e.cfg.warps * 32), 1, 1);
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
    return cudaLaunchKernelEx(&cfg, e.fn, a, p.split, p.wk);
}

}  // namespace mbw
