// gemv_mma.cu -- weight-streaming GEMV for sm_103a with the tensor core as the
// multiply-add unit.
//
// Y[m][i] = sum_k X[m][k] * w(i, k) for BF16, INT4 group-64 and AWQ-style INT4
// group-128 weights and a small batch M (1..8; 1..4 for group-64).
//
// Why mma here: at batch 1 every weight is used for one multiply-add (llm-rs
// vs vLLM, sec. 2), so at GB300's HBM rate the kernel must retire ~41 INT4
// weights per SM clock -- about 3 issue slots per weight. Unpacking a nibble
// and doing the fp32 multiply-add on the CUDA cores costs ~4 (measured: the
// CUDA-core kernel saturates its integer pipe at a third of HBM bandwidth).
// Here the CUDA cores only turn codes into bf16 pairs (one LOP3 per two codes
// and one exact bf16 subtract), and mma.sync.m16n8k16 retires the multiply-
// adds with fp32 accumulation, taking its A operand straight from the
// registers the weight stream was loaded into. The batch rides in the MMA's
// n = 8 columns. (tcgen05 would need the operand staged through shared memory
// and a TMEM round trip per scale group; the batched skinny GEMM uses it.)
//
// Work decomposition (balanced and persistent):
//   * the weight rows are cut into 16-row tiles; CTA row-group c of G owns
//     the contiguous tile range [c*T/G, (c+1)*T/G), so no SM gets more than
//     one tile more than another;
//   * inside a CTA every warp owns one k-slice of every tile (K split W ways,
//     and S ways more across a thread-block cluster for short, wide shapes);
//     lane (g = lane/4, q = lane%4) loads 16 bytes of rows g and g+8 per
//     64-byte row block, so a quad reads 64 contiguous bytes of a row;
//   * a warp walks its (tile, block) sequence through a U-deep register ring:
//     consume slot u, refill it with the block U steps ahead, so loads keep
//     flowing across tile boundaries; per-tile partial sums go to shared
//     memory and are summed over warps (and cluster ranks, through
//     distributed shared memory) once, in a fixed order: deterministic, no
//     global scratch, no spin waits;
//   * programmatic dependent launch: the ring is filled before the kernel
//     waits for the previous grid; x is staged (once per CTA, in the order the
//     B fragments want it) only after that wait.
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

// (v & 0x000F000F) | 0x43004300: the nibbles at bits 0-3 and 16-19 as the
// bf16 pair (128 + n_lo, 128 + n_hi).
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

// Shared memory layout of one launch (bytes): x words (later reused for the
// per-CTA sums) at 0, per-warp partial sums at red_off.
struct MmaSmem {
    int xwords;  // 16-byte x words per batch row
    int ntmax;   // most tiles any CTA owns
    size_t x_bytes, red_off, red_bytes, total;
};

__host__ __device__ inline MmaSmem mma_smem_layout(int BK, int64_t K, int N, int M, int W, int S, int G) {
    MmaSmem L;
    const int64_t KB = (K + BK - 1) / BK;
    const int64_t BS = (KB + (int64_t)S * W - 1) / ((int64_t)S * W);
    L.xwords = (int)(W * BS * (BK / 8));
    const int T = (N + 15) / 16;
    L.ntmax = (T + G - 1) / G;
    L.x_bytes = (size_t)M * L.xwords * 16;
    const size_t fin_bytes = (size_t)L.ntmax * 16 * M * 4;
    L.red_off = ((L.x_bytes > fin_bytes ? L.x_bytes : fin_bytes) + 15) / 16 * 16;
    L.red_bytes = (size_t)L.ntmax * W * 16 * M * 4;
    L.total = L.red_off + L.red_bytes;
    return L;
}

template <int FMT, int W, int U>
__global__ void __launch_bounds__(W * 32)
    gemv_mma_kernel(const GemvArgs a, const int S) {
    constexpr int BK = MmaTraits<FMT>::BK;
    extern __shared__ uint4 smem_u4[];

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
    const MmaSmem L = mma_smem_layout(BK, a.K, a.N, mb, W, S, G);

    const int KB = (a.K + BK - 1) / BK;
    const int BS = (KB + S * W - 1) / (S * W);
    const int cb0 = rank * W * BS;                  // first block of this CTA's k-range
    const int b0 = cb0 + warp * BS;                 // this warp's k-slice
    const int nb = max(0, min(KB, b0 + BS) - b0);
    const int total = nt * nb;                      // (tile, block) steps of this warp
    const size_t rowbytes = (FMT == FMT_BF16) ? (size_t)a.K * 2 : (size_t)a.K / 2;
    const bool scale32 = (FMT == FMT_G64) && ((a.groups & 1) == 0) && ((((uintptr_t)a.scales) & 3) == 0);

    // ring of U slots: codes of rows g and g+8, and their scale words
    uint4 ring[U][2];
    uint32_t sring[U][2];

    // load the next step (tile t0 + ltile, block b0 + lblk) into slot u;
    // steps are loaded strictly in order
    int ltile = 0, lblk = 0;
    auto load = [&](int u) {
        const int b = b0 + lblk;
        const int rbase = (t0 + ltile) * 16 + g;
        if (++lblk == nb) {
            lblk = 0;
            ++ltile;
        }
        const bool kin = (b * BK + (q + 1) * (BK / 4)) <= a.K;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = min(rbase + 8 * h, a.N - 1);
            ring[u][h] = kin ? ld_stream16(a.W + (size_t)row * rowbytes + (size_t)b * 64 + q * 16)
                             : make_uint4(0, 0, 0, 0);
            if (FMT == FMT_G64) {
                const uint16_t* sp = a.scales + (size_t)row * a.groups + 2 * b;
                if (scale32) {
                    sring[u][h] = __ldg(reinterpret_cast<const unsigned int*>(sp));
                } else {
                    const uint32_t s1 = (2 * b + 1 < a.groups) ? ld_ro_u16(sp + 1) : 0u;
                    sring[u][h] = (uint32_t)ld_ro_u16(sp) | (s1 << 16);
                }
            } else if (FMT == FMT_AWQ) {
                const uint32_t s = ld_ro_u16(a.scales + (size_t)row * a.groups + b);
                const uint32_t zb = ld_ro_u8(a.zeros + (size_t)row * a.zstride + (b >> 1));
                sring[u][h] = s | (((b & 1) ? (zb >> 4) : (zb & 0xF)) << 16);
            }
        }
    };

#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < total) load(u);

    // x is produced by the previous kernel in the stream: wait for it only now.
    pdl_wait();

    // Stage x for the CTA's k-range: xs[m][w] = 16-byte word w (8 k) of batch
    // row m, INT4 pairs permuted.
    const int cwords = max(0, min(KB, cb0 + W * BS) - cb0) * (BK / 8);
    for (int i = threadIdx.x; i < mb * L.xwords; i += W * 32) {
        const int m = i / L.xwords;
        const int wi = i - m * L.xwords;
        const int k = cb0 * BK + wi * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (wi < cwords && k < a.K) v = ld_ro16(a.x + (size_t)m * a.K + k);
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
    const uint4* xw = smem_u4 + (size_t)(xon ? xm : 0) * L.xwords + (size_t)(b0 - cb0) * (BK / 8);
    float* red = reinterpret_cast<float*>(reinterpret_cast<char*>(smem_u4) + L.red_off);

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int ct = 0, cb = 0;  // tile and block (within the k-slice) of the step being consumed

    for (int j0 = 0; j0 < total; j0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u;
            if (j < total) {
                const uint4 wg = ring[u][0], wg8 = ring[u][1];
                const uint32_t sg = sring[u][0], sg8 = sring[u][1];
                if (j + U < total) load(u);
                if (FMT == FMT_BF16) {
                    const uint4 xv = xon ? xw[cb * 4 + q] : make_uint4(0, 0, 0, 0);
                    mma_bf16_16816(acc, wg.x, wg8.x, wg.y, wg8.y, xv.x, xv.y);
                    mma_bf16_16816(acc, wg.z, wg8.z, wg.w, wg8.w, xv.z, xv.w);
                } else {
                    const uint32_t zg = (FMT == FMT_G64) ? 8u : (sg >> 16);
                    const uint32_t zg8 = (FMT == FMT_G64) ? 8u : (sg8 >> 16);
                    const uint32_t zz0 = (0x4300u | zg) * 0x00010001u;  // (128 + z, 128 + z)
                    const uint32_t zz1 = (0x4300u | zg8) * 0x00010001u;
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    const uint32_t wa[4] = {wg.x, wg.y, wg.z, wg.w};
                    const uint32_t wb[4] = {wg8.x, wg8.y, wg8.z, wg8.w};
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint4 xv = xon ? xw[cb * 16 + 4 * q + jj] : make_uint4(0, 0, 0, 0);
                        const uint32_t a4 = wa[jj] >> 4, b4 = wb[jj] >> 4;
                        const uint32_t a8 = wa[jj] >> 8, b8 = wb[jj] >> 8;
                        const uint32_t a12 = wa[jj] >> 12, b12 = wb[jj] >> 12;
                        mma_bf16_16816(d, bf16x2_sub(nib_pair(wa[jj]), zz0), bf16x2_sub(nib_pair(wb[jj]), zz1),
                                       bf16x2_sub(nib_pair(a4), zz0), bf16x2_sub(nib_pair(b4), zz1), xv.x, xv.y);
                        mma_bf16_16816(d, bf16x2_sub(nib_pair(a8), zz0), bf16x2_sub(nib_pair(b8), zz1),
                                       bf16x2_sub(nib_pair(a12), zz0), bf16x2_sub(nib_pair(b12), zz1), xv.z,
                                       xv.w);
                    }
                    if (FMT == FMT_G64) {
                        // columns 2m (even group) and 2m + 1 (odd group) of batch m = q
                        acc[0] = fmaf(f16_bits_to_f32(sg & 0xFFFF), d[0], acc[0]);
                        acc[0] = fmaf(f16_bits_to_f32(sg >> 16), d[1], acc[0]);
                        acc[2] = fmaf(f16_bits_to_f32(sg8 & 0xFFFF), d[2], acc[2]);
                        acc[2] = fmaf(f16_bits_to_f32(sg8 >> 16), d[3], acc[2]);
                    } else {
                        const float s0 = f16_bits_to_f32(sg & 0xFFFF), s1 = f16_bits_to_f32(sg8 & 0xFFFF);
                        acc[0] = fmaf(s0, d[0], acc[0]);
                        acc[1] = fmaf(s0, d[1], acc[1]);
                        acc[2] = fmaf(s1, d[2], acc[2]);
                        acc[3] = fmaf(s1, d[3], acc[3]);
                    }
                }
                if (++cb == nb) {
                    // tile done: its partials -> red[tile][warp][row][m]
                    float* rp = red + ((size_t)(ct * W + warp) * 16) * mb;
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
                    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                    cb = 0;
                    ++ct;
                }
            }
        }
    }
    if (nb == 0) {
        // a warp whose k-slice is empty still contributes zeros for every tile
        for (int t = 0; t < nt; ++t) {
            float* rp = red + ((size_t)(t * W + warp) * 16) * mb;
            for (int i = lane; i < 16 * mb; i += 32) rp[i] = 0.f;
        }
    }
    __syncthreads();

    // Sum over warps in warp order: fin[tile][row][m] (reuses the x area,
    // which is no longer read).
    float* fin = reinterpret_cast<float*>(smem_u4);
    const int nout = nt * 16 * mb;
    for (int i = threadIdx.x; i < nout; i += W * 32) {
        const int t = i / (16 * mb);
        const int rm = i - t * 16 * mb;
        float v = 0.f;
        for (int w = 0; w < W; ++w) v += red[((size_t)(t * W + w) * 16) * mb + rm];
        fin[i] = v;
    }
    const int row0 = t0 * 16;
    if (S == 1) {
        __syncthreads();
        for (int i = threadIdx.x; i < nout; i += W * 32) {
            const int m = i / (nt * 16), lr = i - m * nt * 16;
            if (row0 + lr < a.N) store_out(a.y, (int64_t)m * a.N + row0 + lr, fin[lr * mb + m], a.out_f32);
        }
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    // rank s writes rows [s * R / S, (s + 1) * R / S) of the CTA's R rows, for every batch row
    const int R = nt * 16;
    const int lo = rank * R / S, hi = (rank + 1) * R / S;
    const int span = hi - lo;
    for (int i = threadIdx.x; i < span * mb; i += W * 32) {
        const int m = i / span, lr = lo + (i - m * span);
        float v = 0.f;
        for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(fin + lr * mb + m, s);
        if (row0 + lr < a.N) store_out(a.y, (int64_t)m * a.N + row0 + lr, v, a.out_f32);
    }
    cluster.sync();
}

// ------------------------------------------------------------- tables ----
using MmaFn = void (*)(const GemvArgs, const int);
struct MmaEntry {
    MmaConfig cfg;
    MmaFn fn;
};
#define MBW_M(F, W, U) \
    { {W, U}, gemv_mma_kernel<F, W, U> }

static const MmaEntry kMmaBf16[] = {
    MBW_M(FMT_BF16, 4, 4), MBW_M(FMT_BF16, 4, 8), MBW_M(FMT_BF16, 8, 4), MBW_M(FMT_BF16, 8, 8),
};
static const MmaEntry kMmaG64[] = {
    MBW_M(FMT_G64, 4, 2), MBW_M(FMT_G64, 4, 4), MBW_M(FMT_G64, 8, 2), MBW_M(FMT_G64, 8, 4),
};
static const MmaEntry kMmaAwq[] = {
    MBW_M(FMT_AWQ, 4, 2), MBW_M(FMT_AWQ, 4, 4), MBW_M(FMT_AWQ, 8, 2), MBW_M(FMT_AWQ, 8, 4),
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

// CTA row-groups of a launch: `occ` CTAs per SM in total, at most one per
// 16-row tile, a multiple of the cluster size.
int mma_row_groups(int64_t N, int split, int occ) {
    const int sms = device_sm_count();
    const int64_t T = (N + 15) / 16;
    int64_t G = ((int64_t)sms * occ) / split;
    if (G > T) G = T;
    if (G < 1) G = 1;
    return (int)G;
}

size_t mma_smem_bytes(int fmt, const MmaConfig& c, int64_t N, int64_t K, int M, int split, int occ) {
    const int BK = (fmt == FMT_BF16) ? 32 : 128;
    const int G = mma_row_groups(N, split, occ);
    return mma_smem_layout(BK, K, (int)N, M, c.warps, split, G).total;
}

cudaError_t launch_gemv_mma(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s) {
    int n;
    const MmaEntry* t = mma_table(fmt, &n);
    if (p.cfg < 0 || p.cfg >= n || a.M < 1 || a.M > mma_max_batch(fmt)) return cudaErrorInvalidValue;
    const MmaEntry& e = t[p.cfg];
    const int G = mma_row_groups(a.N, p.split, p.occ);
    const size_t smem = mma_smem_bytes(fmt, e.cfg, a.N, a.K, a.M, p.split, p.occ);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(G * p.split), 1, 1);
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
    return cudaLaunchKernelEx(&cfg, e.fn, a, p.split);
}

}  // namespace mbw
