// gemv_mma.cu -- weight-streaming GEMV for sm_103a with the tensor core as the
// multiply-add unit.
//
// Y[m][i] = sum_k X[m][k] * w(i, k) for BF16, INT4 group-64, AWQ-style INT4
// group-128 and symmetric per-channel INT8 weights (the last in the "mma2"
// family only) and a small batch M (1..8; 1..4 for group-64).
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
//     flowing across tile boundaries; load pointers advance by one block and
//     are rebuilt only at tile changes, and K is a whole number of blocks, so
//     the loop carries no per-block predicates; per-tile partial sums go to shared
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
    int xwords;  // 16-byte x words per batch row (as laid out in shared memory)
    int ntmax;   // most tiles any CTA owns
    size_t x_bytes, red_off, red_bytes, total;
};

// xpad: x words per block as laid out (0: BK / 8, packed). The "mma2" INT4 and
// INT8 kernels pad: each lane quarter's words start at word 10 q (INT4, 8 words
// per quarter) or 5 q (INT8, 4 words), so that the four quarters' lanes reading
// their word w hit four different bank groups.
__host__ __device__ inline MmaSmem mma_smem_layout(int BK, int64_t K, int N, int M, int W, int S, int G, int glu = 0,
                                                   int xpad = 0) {
    MmaSmem L;
    const int64_t KB = (K + BK - 1) / BK;
    const int64_t BS = (KB + (int64_t)S * W - 1) / ((int64_t)S * W);
    const int xpb = xpad ? xpad : BK / 8;
    L.xwords = (int)(W * BS * xpb);
    const int T = (N + 15) / 16;
    L.ntmax = (T + G - 1) / G * (glu ? 2 : 1);  // logical tiles (gate/up pairs under the gated epilogue)
    L.x_bytes = ((size_t)M * L.xwords + xpb) * 16;  // + one block of zero words
    const size_t fin_bytes = (size_t)L.ntmax * 16 * M * 4;
    L.red_off = ((L.x_bytes > fin_bytes ? L.x_bytes : fin_bytes) + 15) / 16 * 16;
    L.red_bytes = (size_t)L.ntmax * W * 16 * M * 4;
    L.total = L.red_off + L.red_bytes;
    return L;
}

template <int FMT, int W, int U>
__global__ void __launch_bounds__(W * 32, 16 / W)
    gemv_mma_kernel(const GemvArgs a, const int S) {
    constexpr int BK = MmaTraits<FMT>::BK;
    constexpr int XW = BK / 8;                      // 16-byte x words per row block
    constexpr int SPB = (FMT == FMT_G64) ? 2 : 1;   // scale entries per row block
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

    const int KB = a.K / BK;  // the plan guarantees K % BK == 0
    const int BS = (KB + S * W - 1) / (S * W);
    const int cb0 = rank * W * BS;  // first block of this CTA's k-range
    const int b0 = cb0 + warp * BS;  // this warp's k-slice
    const int nb = max(0, min(KB, b0 + BS) - b0);
    const int total = nt * nb;  // (tile, block) steps of this warp
    const size_t rowbytes = (FMT == FMT_BF16) ? (size_t)a.K * 2 : (size_t)a.K / 2;

    // Load cursor: pointers into rows g and g+8 of the tile being loaded.
    // They advance by one block per load and are rebuilt only at tile changes.
    int lt = 0, lb = 0;
    const uint8_t* wp0 = nullptr;
    const uint8_t* wp1 = nullptr;
    const uint16_t* sp0 = nullptr;
    const uint16_t* sp1 = nullptr;
    const uint8_t* zp0 = nullptr;
    const uint8_t* zp1 = nullptr;
    auto set_rows = [&](int t) {
        const int r0 = min((t0 + t) * 16 + g, a.N - 1);
        const int r1 = min((t0 + t) * 16 + g + 8, a.N - 1);
        wp0 = a.W + (size_t)r0 * rowbytes + (size_t)b0 * 64 + q * 16;
        wp1 = a.W + (size_t)r1 * rowbytes + (size_t)b0 * 64 + q * 16;
        if (FMT != FMT_BF16) {
            sp0 = a.scales + (size_t)r0 * a.groups + (size_t)b0 * SPB;
            sp1 = a.scales + (size_t)r1 * a.groups + (size_t)b0 * SPB;
        }
        if (FMT == FMT_AWQ) {
            zp0 = a.zeros + (size_t)r0 * a.zstride;
            zp1 = a.zeros + (size_t)r1 * a.zstride;
        }
    };
    if (nt > 0) set_rows(0);

    uint4 rw[U][2];      // codes / weights of rows g and g+8
    uint32_t rsc[U][2];  // g64: two fp16 scales; AWQ: fp16 scale | zero << 16

    auto load = [&](int u) {
        rw[u][0] = ld_stream16(wp0);
        rw[u][1] = ld_stream16(wp1);
        if (FMT == FMT_G64) {
            rsc[u][0] = (uint32_t)ld_ro_u16(sp0) | ((uint32_t)ld_ro_u16(sp0 + 1) << 16);
            rsc[u][1] = (uint32_t)ld_ro_u16(sp1) | ((uint32_t)ld_ro_u16(sp1 + 1) << 16);
        } else if (FMT == FMT_AWQ) {
            const int b = b0 + lb;
            const uint32_t sh = (b & 1) * 4;
            rsc[u][0] = (uint32_t)ld_ro_u16(sp0) | ((((uint32_t)ld_ro_u8(zp0 + (b >> 1))) >> sh & 0xF) << 16);
            rsc[u][1] = (uint32_t)ld_ro_u16(sp1) | ((((uint32_t)ld_ro_u8(zp1 + (b >> 1))) >> sh & 0xF) << 16);
        }
        wp0 += 64;
        wp1 += 64;
        sp0 += SPB;
        sp1 += SPB;
        if (++lb == nb) {
            lb = 0;
            if (++lt < nt) set_rows(lt);
        }
    };

#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < total) load(u);

    // x is produced by the previous kernel in the stream: wait for it only now.
    prefetch_l2_grid_share(a.x, (size_t)a.M * a.K * 2);
    pdl_wait();

    // Stage x for the CTA's k-range: xs[m][w] = 16-byte word w (8 k) of batch
    // row m (INT4: pairs permuted), followed by XW zero words for lanes that
    // carry no x.
    uint4* xs = smem_u4;
    const int cwords = max(0, min(KB, cb0 + W * BS) - cb0) * XW;
    for (int i = threadIdx.x; i < mb * L.xwords + XW; i += W * 32) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (i < mb * L.xwords) {
            const int m = i / L.xwords;
            const int wi = i - m * L.xwords;
            if (wi < cwords) v = ld_ro16(a.x + (size_t)m * a.K + (size_t)cb0 * BK + (size_t)wi * 8);
            if (FMT != FMT_BF16 && !a.x_natural) v = perm_pairs(v);
        }
        xs[i] = v;
    }
    __syncthreads();

    // B-fragment source of this lane: column n = g (batch g; group-64: batch
    // g/2, group parity g%2 matching the lane's quad half).
    bool xon;
    int xm;
    if (FMT == FMT_G64) {
        xm = g >> 1;
        xon = (xm < mb) && ((g & 1) == (q >> 1));
    } else {
        xm = g;
        xon = xm < mb;
    }
    const uint4* xbase = xon ? xs + (size_t)xm * L.xwords + (size_t)(b0 - cb0) * XW : xs + (size_t)mb * L.xwords;
    const int xstep = xon ? XW : 0;
    const uint4* xp = xbase;
    float* red = reinterpret_cast<float*>(reinterpret_cast<char*>(smem_u4) + L.red_off);

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc2[4] = {0.f, 0.f, 0.f, 0.f};  // second chain (BF16)
    int cb = 0, ct = 0;

    for (int j0 = 0; j0 < total; j0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (j0 + u < total) {
                const uint4 w0 = rw[u][0], w1 = rw[u][1];
                const uint32_t s0 = rsc[u][0], s1 = rsc[u][1];
                if (j0 + u + U < total) load(u);
                if (FMT == FMT_BF16) {
                    const uint4 xv = xp[q];
                    mma_bf16_16816(acc, w0.x, w1.x, w0.y, w1.y, xv.x, xv.y);
                    mma_bf16_16816(acc2, w0.z, w1.z, w0.w, w1.w, xv.z, xv.w);
                } else {
                    const uint32_t zz0 = (0x4300u | ((FMT == FMT_G64) ? 8u : (s0 >> 16))) * 0x00010001u;
                    const uint32_t zz1 = (0x4300u | ((FMT == FMT_G64) ? 8u : (s1 >> 16))) * 0x00010001u;
                    float d0[4] = {0.f, 0.f, 0.f, 0.f};
                    float d1[4] = {0.f, 0.f, 0.f, 0.f};
                    const uint32_t wa[4] = {w0.x, w0.y, w0.z, w0.w};
                    const uint32_t wb[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint4 xv = xp[4 * q + jj];
                        mma_bf16_16816(d0, bf16x2_sub(nib_pair(wa[jj]), zz0), bf16x2_sub(nib_pair(wb[jj]), zz1),
                                       bf16x2_sub(nib_pair(wa[jj] >> 4), zz0), bf16x2_sub(nib_pair(wb[jj] >> 4), zz1),
                                       xv.x, xv.y);
                        mma_bf16_16816(d1, bf16x2_sub(nib_pair(wa[jj] >> 8), zz0),
                                       bf16x2_sub(nib_pair(wb[jj] >> 8), zz1), bf16x2_sub(nib_pair(wa[jj] >> 12), zz0),
                                       bf16x2_sub(nib_pair(wb[jj] >> 12), zz1), xv.z, xv.w);
                    }
                    if (FMT == FMT_G64) {
                        // columns 2m (even group) and 2m + 1 (odd group) of batch m = q
                        const float2 sg = __half22float2(*reinterpret_cast<const __half2*>(&s0));
                        const float2 sg8 = __half22float2(*reinterpret_cast<const __half2*>(&s1));
                        acc[0] = fmaf(sg.x, d0[0] + d1[0], acc[0]);
                        acc[0] = fmaf(sg.y, d0[1] + d1[1], acc[0]);
                        acc[2] = fmaf(sg8.x, d0[2] + d1[2], acc[2]);
                        acc[2] = fmaf(sg8.y, d0[3] + d1[3], acc[2]);
                    } else {
                        const float sa = f16_bits_to_f32(s0 & 0xFFFF), sb = f16_bits_to_f32(s1 & 0xFFFF);
                        acc[0] = fmaf(sa, d0[0] + d1[0], acc[0]);
                        acc[1] = fmaf(sa, d0[1] + d1[1], acc[1]);
                        acc[2] = fmaf(sb, d0[2] + d1[2], acc[2]);
                        acc[3] = fmaf(sb, d0[3] + d1[3], acc[3]);
                    }
                }
                xp += xstep;
                if (++cb == nb) {
                    // tile done: its partials -> red[tile][warp][row][m]
                    float* rp = red + ((size_t)(ct * W + warp) * 16) * mb;
                    if (FMT == FMT_BF16) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[i] += acc2[i];
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
                    for (int i = 0; i < 4; ++i) acc[i] = acc2[i] = 0.f;
                    cb = 0;
                    ++ct;
                    xp = xbase;
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

    // Sum over warps in warp order: fin[tile][row][m] (reuses the x area).
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

// ----------------------------------------------------------------------------
// "mma2": 32 bytes of each of rows g and g+8 per lane per 128-byte super-block.
//
// A lane's 32 bytes of a row are 64 INT4 codes = exactly one group-64 scale
// group (or half an AWQ group-128 group, or 16 BF16 weights). The 4 lanes of a
// quad cover 4 groups; the B fragment routes column n = 4m + j only the x of
// quad lane j (group j) of batch m, so each MMA keeps the 4 groups apart in 4
// columns and a lane needs only the 2 scales of its own columns. Compared to
// 16-byte chunks this halves the load, scale and epilogue instructions per
// weight; the nibble arithmetic (3 shifts + 4 LOP3 + 4 bf16 subtracts per 8
// codes) is unchanged.
//   group-64 : column n = 4m + j, batch M <= 2; lane (g,q) holds groups
//              2(q&1), 2(q&1)+1 of batch q>>1; lanes q and q^1 are summed at
//              the end of a tile.
//   AWQ      : column n = 2m + j, j = group within the super-block, M <= 4;
//              lane (g,q) holds both groups of batch q.
//   BF16     : column n = m (M <= 8); lane q's 16 weights feed 4 MMAs.
//   INT8     : column n = m (M <= 8); a lane's 32 bytes of a row are 32
//              codes, 8 MMAs per super-block (one per 32-bit word of rows g
//              and g+8); every code of a row shares the row's fp32 scale,
//              which multiplies the row's finished sum in the store (TileInfer,
//              "Pushing further with cheating: INT8 quantization").
// FZ: 1 in the twin instantiated for fused calls (RMSNorm prologue, gated
// and residual epilogues); 0 compiles the fusions out.
template <int FMT, int W, int U, int ASYNC, int FZ>
__global__ void __launch_bounds__(W * 32, 16 / W)
    gemv_mma2_kernel(const GemvArgs a, const int S) {
    constexpr int BK = (FMT == FMT_BF16) ? 64 : (FMT == FMT_I8) ? 128 : 256;  // k per 128-byte row super-block
    constexpr int XW = BK / 8;                                              // 16-byte x words per super-block
    extern __shared__ uint4 smem_u4[];

    pdl_launch_dependents();

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int G = gridDim.x / S;
    const int cgid = blockIdx.x / S;
    int t0, nt;  // the CTA's logical tiles (gate/up pairs under the gated epilogue)
    cta_tile_range<FZ>(a, G, cgid, t0, nt);
    const int mb = a.M;
    constexpr int XPAD = (FMT == FMT_G64 || FMT == FMT_AWQ) ? 40 : (FMT == FMT_I8) ? 20 : 0;
    const MmaSmem L = mma_smem_layout(BK, a.K, a.N, mb, W, S, G, gated<FZ>(a) ? 1 : 0, XPAD);

    const int KB = a.K / BK;  // the plan guarantees K % BK == 0
    const int BS = (KB + S * W - 1) / (S * W);
    const int cb0 = rank * W * BS;
    const int b0 = cb0 + warp * BS;
    const int nb = max(0, min(KB, b0 + BS) - b0);
    const int total = nt * nb;
    const size_t rowbytes = (FMT == FMT_BF16) ? (size_t)a.K * 2 : (FMT == FMT_I8) ? (size_t)a.K : (size_t)a.K / 2;

    // load cursor (rows g, g+8 of the tile being loaded)
    int lb = 0, lt = 0;
    const uint8_t* wp0 = nullptr;
    const uint8_t* wp1 = nullptr;
    const uint16_t* sp0 = nullptr;
    const uint16_t* sp1 = nullptr;
    const uint8_t* zp0 = nullptr;
    const uint8_t* zp1 = nullptr;
    const uint8_t* ap[4] = {nullptr, nullptr, nullptr, nullptr};  // ASYNC: sources of this lane's 4 copies
    auto set_rows = [&](int t) {
        const int tl = t0 + t;
        const uint8_t* Wt = tile_weights<FZ>(a, tl);
        const uint16_t* St = tile_scales<FZ>(a, tl);
        const int trow = tile_row0<FZ>(a, tl);
        const int r0 = min(trow + g, a.N - 1);
        const int r1 = min(trow + g + 8, a.N - 1);
        if (ASYNC) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                ap[j] = Wt + (size_t)min(trow + ring_copy_row(lane, j), a.N - 1) * rowbytes + (size_t)b0 * 128 +
                        ring_copy_byte(lane);
        } else {
            wp0 = Wt + (size_t)r0 * rowbytes + (size_t)b0 * 128 + q * 32;
            wp1 = Wt + (size_t)r1 * rowbytes + (size_t)b0 * 128 + q * 32;
        }
        if (FMT == FMT_G64) {
            sp0 = St + (size_t)r0 * a.groups + (size_t)b0 * 4 + 2 * (q & 1);
            sp1 = St + (size_t)r1 * a.groups + (size_t)b0 * 4 + 2 * (q & 1);
        } else if (FMT == FMT_AWQ) {
            sp0 = St + (size_t)r0 * a.groups + (size_t)b0 * 2;
            sp1 = St + (size_t)r1 * a.groups + (size_t)b0 * 2;
            const uint8_t* Zt = (gated<FZ>(a) && (tl & 1)) ? a.zeros2 : a.zeros;  // up or gate tile
            zp0 = Zt + (size_t)r0 * a.zstride + b0;
            zp1 = Zt + (size_t)r1 * a.zstride + b0;
        }
    };
    if (nt > 0) set_rows(0);

    uint4 rw[U][4];      // [u][0..1] row g (32 bytes), [u][2..3] row g+8 (register ring)
    // cp.async ring (ASYNC): slot u of this warp is one ring slot of 2 KB
    // (device.cuh: fragment lane L's chunk c at c * 512 + L * 16, filled by
    // sector-complete copies).
    // INT8: the fp32 scales of the CTA's rows, read before the wait (they are weights)
    float* rsc = reinterpret_cast<float*>(reinterpret_cast<char*>(smem_u4) + L.total);
    constexpr bool ZF = (FMT == FMT_G64 || FMT == FMT_AWQ);  // INT4
    constexpr int XP = XPAD ? XPAD : XW;                      // physical x words per super-block
    const int lxw = L.xwords / XP * XW;                       // logical x words per batch row
    const size_t sc_bytes = (FMT == FMT_I8) ? (size_t)L.ntmax * 16 * 4 : 0;
    uint8_t* abase = reinterpret_cast<uint8_t*>(smem_u4) + (L.total + sc_bytes + 127) / 128 * 128 +
                     (size_t)warp * U * 4 * 512;
    const uint8_t* aring = abase + lane * 16;
    uint32_t rs[U][2];   // group-64: 2 fp16 scales per row; AWQ: 2 fp16 scales per row
    uint32_t rz[U];      // AWQ: zero-point byte of rows g (bits 0-7) and g+8 (bits 8-15)

    auto load = [&](int u) {
        if (ASYNC) {
            uint8_t* d = abase + (size_t)u * 4 * 512;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                cp_async16(d + ring_copy_dst(lane, j), ap[j]);
                ap[j] += 128;
            }
        } else {
            const u32x8 v0 = ld_stream32(wp0);  // one 256-bit load per row: whole sectors
            const u32x8 v1 = ld_stream32(wp1);
            rw[u][0] = make_uint4(v0.v[0], v0.v[1], v0.v[2], v0.v[3]);
            rw[u][1] = make_uint4(v0.v[4], v0.v[5], v0.v[6], v0.v[7]);
            rw[u][2] = make_uint4(v1.v[0], v1.v[1], v1.v[2], v1.v[3]);
            rw[u][3] = make_uint4(v1.v[4], v1.v[5], v1.v[6], v1.v[7]);
        }
        if (FMT == FMT_G64 || FMT == FMT_AWQ) {
            rs[u][0] = (uint32_t)ld_ro_u16(sp0) | ((uint32_t)ld_ro_u16(sp0 + 1) << 16);
            rs[u][1] = (uint32_t)ld_ro_u16(sp1) | ((uint32_t)ld_ro_u16(sp1 + 1) << 16);
        }
        if (FMT == FMT_AWQ) rz[u] = (uint32_t)ld_ro_u8(zp0) | ((uint32_t)ld_ro_u8(zp1) << 8);
        wp0 += 128;
        wp1 += 128;
        sp0 += (FMT == FMT_G64) ? 4 : 2;
        sp1 += (FMT == FMT_G64) ? 4 : 2;
        zp0 += 1;
        zp1 += 1;
        if (++lb == nb) {
            lb = 0;
            if (++lt < nt) set_rows(lt);
        }
    };

#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (u < total) load(u);
        if (ASYNC) cp_async_commit();  // one group per step, empty past the end
    }

    if (FMT == FMT_I8)
        for (int i = threadIdx.x; i < nt * 16; i += W * 32) {
            const int tl = t0 + (i >> 4);
            rsc[i] = __ldg(tile_rscale<FZ>(a, tl) + min(tile_row0<FZ>(a, tl) + (i & 15), a.N - 1));
        }

    prefetch_l2_grid_share(a.x, (size_t)a.M * a.K * 2);
    pdl_wait();

    // RMSNorm prologue: factor per batch row into the (still unused) partial-sum area
    float* nscr = reinterpret_cast<float*>(reinterpret_cast<char*>(smem_u4) + L.red_off);
    if (FZ && a.norm_w) norm_factors(a, nscr, W * 32);

    uint4* xs = smem_u4;
    const int cwords = max(0, min(KB, cb0 + W * BS) - cb0) * XW;
    const int nxw = mb * lxw;  // logical words
    for (int i0 = 0; i0 < nxw + XP; i0 += W * 32) {
        const int i = i0 + threadIdx.x;
        uint4 v = make_uint4(0, 0, 0, 0);
        int m = mb, wi = i - nxw;  // the zero block
        if (i < nxw) {
            m = i / lxw;
            wi = i - m * lxw;
            if (wi < cwords) {
                v = ld_ro16(a.x + (size_t)m * a.K + (size_t)cb0 * BK + (size_t)wi * 8);
                if (FZ && a.norm_w) v = norm_word(v, nscr[W * mb + m], a.norm_w + (size_t)cb0 * BK + (size_t)wi * 8);
            }
            if (FMT == FMT_I8)
                v = perm_i8(v);
            else if (FMT != FMT_BF16 && !a.x_natural)
                v = perm_pairs(v);
        }
        if (i < nxw + XP) {
            // logical word 32 b + 8 q + w of a batch row sits at 40 b + 10 q + w (INT4), word
            // 16 b + 4 q + w at 20 b + 5 q + w (INT8); the zero block (m = mb) is written as it is
            const int pw = (i >= nxw) ? wi
                           : ZF       ? (wi >> 5) * 40 + ((wi & 31) >> 3) * 10 + (wi & 7)
                           : (FMT == FMT_I8) ? (wi >> 4) * 20 + ((wi & 15) >> 2) * 5 + (wi & 3)
                                             : wi;
            xs[(size_t)m * L.xwords + pw] = v;
        }
    }
    __syncthreads();

    // B fragment of this lane: column n = g
    bool xon;
    int xm;
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
    // lane's x words of a super-block: INT4 words 8q .. 8q+7, INT8 4q .. 4q+3, BF16 2q, 2q+1
    const int xoff = (FMT == FMT_BF16) ? 2 * q : (FMT == FMT_I8) ? 4 * q : 8 * q;
    // (INT4: the quarter at 10 q, INT8 at 5 q; the lanes without a column read zero
    // words from 1 on, a bank group apart from the quarters' reads)
    const int xq = ZF ? 10 * q : (FMT == FMT_I8) ? 5 * q : xoff;
    const uint4* xbase = xon ? xs + (size_t)xm * L.xwords + (size_t)(b0 - cb0) * XP + xq
                             : xs + (size_t)mb * L.xwords + (XPAD ? 1 : 0);
    const int xstep = xon ? XP : 0;
    const uint4* xp = xbase;
    float* red = reinterpret_cast<float*>(reinterpret_cast<char*>(smem_u4) + L.red_off);

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc2[4] = {0.f, 0.f, 0.f, 0.f};
    int cb = 0, ct = 0;

    for (int j0 = 0; j0 < total; j0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (j0 + u < total) {
                uint4 a0, a1, c0, c1;
                if (ASYNC) {
                    cp_async_wait<U - 1>();  // this lane's copies of step j0 + u have landed
                    __syncwarp();            // and so have the other lanes'
                    const uint8_t* d = aring + (size_t)u * 4 * 512;
                    a0 = *reinterpret_cast<const uint4*>(d);
                    a1 = *reinterpret_cast<const uint4*>(d + 512);
                    c0 = *reinterpret_cast<const uint4*>(d + 1024);
                    c1 = *reinterpret_cast<const uint4*>(d + 1536);
                } else {
                    a0 = rw[u][0];
                    a1 = rw[u][1];
                    c0 = rw[u][2];
                    c1 = rw[u][3];
                }
                const uint32_t s0 = rs[u][0], s1 = rs[u][1];
                const uint32_t zb = (FMT == FMT_AWQ) ? rz[u] : 0u;
                if (!ASYNC && j0 + u + U < total) load(u);
                if (FMT == FMT_BF16) {
                    const uint4 x0 = xp[0], x1 = xp[1];
                    mma_bf16_16816(acc, a0.x, c0.x, a0.y, c0.y, x0.x, x0.y);
                    mma_bf16_16816(acc2, a0.z, c0.z, a0.w, c0.w, x0.z, x0.w);
                    mma_bf16_16816(acc, a1.x, c1.x, a1.y, c1.y, x1.x, x1.y);
                    mma_bf16_16816(acc2, a1.z, c1.z, a1.w, c1.w, x1.z, x1.w);
                } else if (FMT == FMT_I8) {
                    const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    const uint32_t wb[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        uint32_t p0, p1, p2, p3;
                        i8_pairs(wa[w], p0, p2);
                        i8_pairs(wb[w], p1, p3);
                        const uint4 xv = xp[w >> 1];
                        if (w & 1)
                            mma_bf16_16816(acc2, p0, p1, p2, p3, xv.z, xv.w);
                        else
                            mma_bf16_16816(acc, p0, p1, p2, p3, xv.x, xv.y);
                    }
                } else {
                    // codes n -> bf16 128 + n (exact), minus the bf16 128 + z (exact): n - z enters the MMA
                    uint32_t zz0, zz1;
                    if (FMT == FMT_G64) {
                        zz0 = zz1 = 0x43084308u;
                    } else {
                        const uint32_t sh = (q >> 1) * 4;  // this lane's group: low or high nibble
                        zz0 = (0x4300u | ((zb >> sh) & 0xF)) * 0x00010001u;
                        zz1 = (0x4300u | ((zb >> (8 + sh)) & 0xF)) * 0x00010001u;
                    }
                    float d0[4] = {0.f, 0.f, 0.f, 0.f};
                    float d1[4] = {0.f, 0.f, 0.f, 0.f};
                    const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    const uint32_t wb[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const uint4 xv = xp[w];
                        mma_bf16_16816(d0, bf16x2_sub(nib_pair(wa[w]), zz0), bf16x2_sub(nib_pair(wb[w]), zz1),
                                       bf16x2_sub(nib_pair(wa[w] >> 4), zz0), bf16x2_sub(nib_pair(wb[w] >> 4), zz1),
                                       xv.x, xv.y);
                        mma_bf16_16816(d1, bf16x2_sub(nib_pair(wa[w] >> 8), zz0), bf16x2_sub(nib_pair(wb[w] >> 8), zz1),
                                       bf16x2_sub(nib_pair(wa[w] >> 12), zz0),
                                       bf16x2_sub(nib_pair(wb[w] >> 12), zz1), xv.z, xv.w);
                    }
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&s0));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&s1));
                    // columns 2q, 2q+1: AWQ groups 0, 1 of batch q; group-64 groups 2(q&1), 2(q&1)+1 of batch q>>1
                    acc[0] = fmaf(f0.x, d0[0] + d1[0], acc[0]);
                    acc[0] = fmaf(f0.y, d0[1] + d1[1], acc[0]);
                    acc[2] = fmaf(f1.x, d0[2] + d1[2], acc[2]);
                    acc[2] = fmaf(f1.y, d0[3] + d1[3], acc[2]);
                }
                if (ASYNC) {
                    __syncwarp();  // every lane has read slot u before it is refilled
                    if (j0 + u + U < total) load(u);
                    cp_async_commit();
                }
                xp += xstep;
                if (++cb == nb) {
                    float* rp = red + ((size_t)(ct * W + warp) * 16) * mb;
                    if (FMT == FMT_BF16 || FMT == FMT_I8) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[i] += acc2[i];
                        if (2 * q < mb) {
                            rp[g * mb + 2 * q] = acc[0];
                            rp[(g + 8) * mb + 2 * q] = acc[2];
                        }
                        if (2 * q + 1 < mb) {
                            rp[g * mb + 2 * q + 1] = acc[1];
                            rp[(g + 8) * mb + 2 * q + 1] = acc[3];
                        }
                    } else if (FMT == FMT_G64) {
                        // lanes q and q^1 hold the other two groups of the same batch
                        const float v0 = acc[0] + __shfl_xor_sync(0xFFFFFFFFu, acc[0], 1);
                        const float v2 = acc[2] + __shfl_xor_sync(0xFFFFFFFFu, acc[2], 1);
                        const int m = q >> 1;
                        if ((q & 1) == 0 && m < mb) {
                            rp[g * mb + m] = v0;
                            rp[(g + 8) * mb + m] = v2;
                        }
                    } else {
                        if (q < mb) {
                            rp[g * mb + q] = acc[0];
                            rp[(g + 8) * mb + q] = acc[2];
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = acc2[i] = 0.f;
                    cb = 0;
                    ++ct;
                    xp = xbase;
                }
            }
        }
    }
    if (nb == 0) {
        for (int t = 0; t < nt; ++t) {
            float* rp = red + ((size_t)(t * W + warp) * 16) * mb;
            for (int i = lane; i < 16 * mb; i += 32) rp[i] = 0.f;
        }
    }
    __syncthreads();

    float* fin = reinterpret_cast<float*>(smem_u4);  // [lr][m]: sums over the CTA's warps
    const int nout = nt * 16 * mb;
    for (int i = threadIdx.x; i < nout; i += W * 32) {
        const int t = i / (16 * mb);
        const int rm = i - t * 16 * mb;
        float v = 0.f;
        for (int w = 0; w < W; ++w) v += red[((size_t)(t * W + w) * 16) * mb + rm];
        fin[i] = v;
    }
    // output row o of the CTA; under the gated epilogue it pairs gate row
    // gate_row(o) with up row gate_row(o) + 16 (local logical rows)
    const int nto = gated<FZ>(a) ? nt / 2 : nt;
    const int orow0 = (gated<FZ>(a) ? t0 / 2 : t0) * 16;
    auto gate_row = [&](int o) { return gated<FZ>(a) ? (o >> 4) * 32 + (o & 15) : o; };
    if (S == 1) {
        __syncthreads();
        for (int i = threadIdx.x; i < nto * 16 * mb; i += W * 32) {
            const int m = i / (nto * 16), o = i - m * nto * 16;
            if (orow0 + o >= a.N) continue;
            const int lr = gate_row(o);
            float v = fin[lr * mb + m], v2 = 0.f;
            if (FMT == FMT_I8) v *= rsc[lr];
            if (gated<FZ>(a)) {
                v2 = fin[(lr + 16) * mb + m];
                if (FMT == FMT_I8) v2 *= rsc[lr + 16];
            }
            store_fused<FZ>(a, m, orow0 + o, v, v2);
        }
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    // rank s writes output rows [s * Ro / S, (s + 1) * Ro / S) of the CTA group's Ro rows, every batch row
    const int Ro = nto * 16;
    const int lo = rank * Ro / S, hi = (rank + 1) * Ro / S;
    const int span = hi - lo;
    for (int i = threadIdx.x; i < span * mb; i += W * 32) {
        const int m = i / span, o = lo + (i - m * span);
        const int lr = gate_row(o);
        float v = 0.f, v2 = 0.f;
        for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(fin + lr * mb + m, s);
        if (FMT == FMT_I8) v *= rsc[lr];
        if (gated<FZ>(a)) {
            for (int s = 0; s < S; ++s) v2 += *cluster.map_shared_rank(fin + (lr + 16) * mb + m, s);
            if (FMT == FMT_I8) v2 *= rsc[lr + 16];
        }
        if (orow0 + o < a.N) store_fused<FZ>(a, m, orow0 + o, v, v2);
    }
    cluster.sync();
}

// ------------------------------------------------------------- tables ----
using MmaFn = void (*)(const GemvArgs, const int);
struct MmaEntry {
    MmaConfig cfg;
    MmaFn fn;   // plain calls
    MmaFn fnf;  // fused calls (mma2 FZ = 1 twin; null where the format has no fused path)
};
#define MBW_M(F, W, U) \
    { {W, U, 0}, gemv_mma_kernel<F, W, U>, nullptr }

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

#define MBW_M2(F, W, U, A) \
    { {W, U, A}, gemv_mma2_kernel<F, W, U, A, 0>, gemv_mma2_kernel<F, W, U, A, 1> }
static const MmaEntry kMma2Bf16[] = {MBW_M2(FMT_BF16, 8, 2, 0), MBW_M2(FMT_BF16, 8, 4, 0), MBW_M2(FMT_BF16, 4, 4, 0),
                                     MBW_M2(FMT_BF16, 8, 4, 1), MBW_M2(FMT_BF16, 8, 6, 1)};
static const MmaEntry kMma2G64[] = {MBW_M2(FMT_G64, 8, 2, 0), MBW_M2(FMT_G64, 8, 3, 0), MBW_M2(FMT_G64, 4, 2, 0),
                                    MBW_M2(FMT_G64, 4, 3, 0), MBW_M2(FMT_G64, 8, 4, 1), MBW_M2(FMT_G64, 8, 6, 1),
                                    MBW_M2(FMT_G64, 4, 6, 1)};
static const MmaEntry kMma2Awq[] = {MBW_M2(FMT_AWQ, 8, 2, 0), MBW_M2(FMT_AWQ, 8, 3, 0), MBW_M2(FMT_AWQ, 4, 2, 0),
                                    MBW_M2(FMT_AWQ, 8, 4, 1), MBW_M2(FMT_AWQ, 8, 6, 1)};
static const MmaEntry kMma2I8[] = {MBW_M2(FMT_I8, 8, 2, 0), MBW_M2(FMT_I8, 8, 3, 0), MBW_M2(FMT_I8, 4, 3, 0),
                                   MBW_M2(FMT_I8, 8, 4, 1), MBW_M2(FMT_I8, 8, 6, 1), MBW_M2(FMT_I8, 4, 8, 1)};
#undef MBW_M2

static const MmaEntry* mma2_table(int fmt, int* n) {
    switch (fmt) {
        case FMT_BF16:
            *n = (int)(sizeof(kMma2Bf16) / sizeof(kMma2Bf16[0]));
            return kMma2Bf16;
        case FMT_G64:
            *n = (int)(sizeof(kMma2G64) / sizeof(kMma2G64[0]));
            return kMma2G64;
        case FMT_AWQ:
            *n = (int)(sizeof(kMma2Awq) / sizeof(kMma2Awq[0]));
            return kMma2Awq;
        case FMT_I8:
            *n = (int)(sizeof(kMma2I8) / sizeof(kMma2I8[0]));
            return kMma2I8;
        default:
            *n = 0;
            return nullptr;
    }
}

int mma2_num_configs(int fmt) {
    int n;
    mma2_table(fmt, &n);
    return n;
}

MmaConfig mma2_config(int fmt, int idx) {
    int n;
    return mma2_table(fmt, &n)[idx].cfg;
}

int mma2_max_batch(int fmt) { return fmt == FMT_G64 ? 2 : fmt == FMT_AWQ ? 4 : 8; }
int mma2_block_k(int fmt) { return fmt == FMT_BF16 ? 64 : fmt == FMT_I8 ? 128 : 256; }

static size_t mma2_layout_bytes(int fmt, const MmaConfig& c, int64_t N, int64_t K, int M, int split, int G, int glu) {
    const int xpad = (fmt == FMT_G64 || fmt == FMT_AWQ) ? 40 : (fmt == FMT_I8) ? 20 : 0;
    const MmaSmem L = mma_smem_layout(mma2_block_k(fmt), K, (int)N, M, c.warps, split, G, glu, xpad);
    const size_t base = L.total + (fmt == FMT_I8 ? (size_t)L.ntmax * 16 * 4 : 0);  // + INT8 row scales
    if (!c.async) return base;
    return (base + 127) / 128 * 128 + (size_t)c.warps * c.u * 4 * 512;
}

static int mma2_groups(int fmt, const MmaConfig& c, int64_t N, int64_t K, int M, int split, int occ, int glu) {
    return fitted_row_groups(N, split, occ, kSmemFit,
                             [&](int G) { return mma2_layout_bytes(fmt, c, N, K, M, split, G, glu); });
}

size_t mma2_smem_bytes(int fmt, const MmaConfig& c, int64_t N, int64_t K, int M, int split, int occ, int glu) {
    return mma2_layout_bytes(fmt, c, N, K, M, split, mma2_groups(fmt, c, N, K, M, split, occ, glu), glu);
}

cudaError_t launch_gemv_mma2(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s) {
    // a gated launch reads the up matrix's codes, scales (not BF16) and zero points (AWQ)
    if (a.glu && (!a.W2 || (fmt != FMT_BF16 && !a.scales2) || (fmt == FMT_AWQ && !a.zeros2)))
        return cudaErrorInvalidValue;
    int n;
    const MmaEntry* t = mma2_table(fmt, &n);
    if (t == nullptr || p.cfg < 0 || p.cfg >= n || a.M < 1 || a.M > mma2_max_batch(fmt)) return cudaErrorInvalidValue;
    const MmaEntry& e = t[p.cfg];
    const MmaFn fn = gemv_fused_args(a) ? e.fnf : e.fn;
    if (fn == nullptr) return cudaErrorInvalidValue;
    const int G = mma2_groups(fmt, e.cfg, a.N, a.K, a.M, p.split, p.occ, a.glu);
    const size_t smem = mma2_layout_bytes(fmt, e.cfg, a.N, a.K, a.M, p.split, G, a.glu);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
    return cudaLaunchKernelEx(&cfg, fn, a, p.split);
}

static const MmaEntry* mma_table(int fmt, int* n) {
    switch (fmt) {
        case FMT_BF16:
            *n = (int)(sizeof(kMmaBf16) / sizeof(kMmaBf16[0]));
            return kMmaBf16;
        case FMT_G64:
            *n = (int)(sizeof(kMmaG64) / sizeof(kMmaG64[0]));
            return kMmaG64;
        case FMT_AWQ:
            *n = (int)(sizeof(kMmaAwq) / sizeof(kMmaAwq[0]));
            return kMmaAwq;
        default:
            *n = 0;
            return nullptr;
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

static int mma_groups(int fmt, const MmaConfig& c, int64_t N, int64_t K, int M, int split, int occ) {
    const int BK = (fmt == FMT_BF16) ? 32 : 128;
    return fitted_row_groups(N, split, occ, kSmemFit,
                             [&](int G) { return mma_smem_layout(BK, K, (int)N, M, c.warps, split, G).total; });
}

size_t mma_smem_bytes(int fmt, const MmaConfig& c, int64_t N, int64_t K, int M, int split, int occ) {
    const int BK = (fmt == FMT_BF16) ? 32 : 128;
    return mma_smem_layout(BK, K, (int)N, M, c.warps, split, mma_groups(fmt, c, N, K, M, split, occ)).total;
}

cudaError_t launch_gemv_mma(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s) {
    int n;
    const MmaEntry* t = mma_table(fmt, &n);
    if (p.cfg < 0 || p.cfg >= n || a.M < 1 || a.M > mma_max_batch(fmt)) return cudaErrorInvalidValue;
    const MmaEntry& e = t[p.cfg];
    const int G = mma_groups(fmt, e.cfg, a.N, a.K, a.M, p.split, p.occ);
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
