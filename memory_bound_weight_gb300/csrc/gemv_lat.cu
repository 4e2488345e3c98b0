// gemv_lat.cu -- latency-oriented GEMV for the small matrices of a decode
// chain (batch 1..8), INT4 group-64, symmetric per-channel INT8 and BF16.
//
// In a decode step every GEMV waits for the one before it (its x is the
// previous kernel's output), so a small matrix costs the chain's release
// latency plus everything its kernel does AFTER griddepcontrol.wait, not
// its bytes over the HBM rate. Measured on GB300 with per-CTA timestamps, a
// streaming kernel spent ~0.6 us staging x through shared memory, ~1 us in
// its unpack/MMA loop and ~0.5 us in a two-barrier reduction after the wait,
// for a 2 MB matrix whose weights had arrived long before. This family moves
// all of that off the dependent path it can:
//   * every weight item a warp owns (16 rows x one 128-byte row super-block,
//     as in the "mma2" layout: 32 bytes of rows g and g+8 per lane) is loaded
//     into registers before the wait, so the next launch streams its whole
//     share while the previous one finishes;
//   * the first NPRE items are also unpacked to bf16 MMA fragments before the
//     wait (INT4), the rest right after it while the x loads are in flight;
//   * x is read straight into the B-fragment registers of the lanes that
//     carry it (no shared-memory staging, no barrier);
//   * one __syncthreads, then each output sums its warps' partials in a fixed
//     order and stores (cluster ranks add theirs through distributed shared
//     memory when K is split over a cluster).
// The number of items a warp may own is a template constant (NI): plans
// whose shape needs more are not offered, and the streaming families take
// those shapes.
//
// Arithmetic is that of the mma2 family: codes become exact bf16 (128 + n) -
// (128 + 8) pairs, products with bf16 x are exact, the tensor core
// accumulates in fp32 and the group scale multiplies each group's fp32
// partial. INT8 codes become exact bf16 pairs the same way and the row's
// fp32 scale multiplies the row's finished sum. BF16 weights go to the
// tensor core unchanged.
#include <cooperative_groups.h>

#include <algorithm>

#include "device.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace mbw {

namespace {

__device__ __forceinline__ void lat_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the nibbles at bits 0-3 and 16-19 of v as the bf16 pair (128 + n_lo, 128 + n_hi)
__device__ __forceinline__ uint32_t lat_nib(uint32_t v) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(0x000F000Fu), "r"(0x43004300u));
    return r;
}

__device__ __forceinline__ uint32_t lat_sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// 8 bf16 x[8w..8w+7] -> pairs (0,4) (1,5) (2,6) (3,7), the order in which the
// INT4 fragments pair their nibbles.
__device__ __forceinline__ uint4 lat_perm(uint4 v) {
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    return o;
}

// INT8 fragments of one item for one lane: word w of rows g and g+8 -> the A
// registers of the one MMA of word w (codes 0, 2 | 1, 3 of the word).
__device__ __forceinline__ void lat_unpack_i8(const u32x8& ra, const u32x8& rb, uint32_t (&A)[8][8]) {
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        i8_pairs(ra.v[w], A[w][0], A[w][2]);
        i8_pairs(rb.v[w], A[w][1], A[w][3]);
    }
}

// INT4 fragments of one item for one lane: word w of rows g (wa) and g+8 (wb)
// -> the A registers of the two MMAs of word w, (q - 8) exact in bf16.
__device__ __forceinline__ void lat_unpack(const u32x8& ra, const u32x8& rb, uint32_t (&A)[8][8]) {
    const uint32_t z = 0x43084308u;  // (128 + 8, 128 + 8)
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t wa = ra.v[w], wb = rb.v[w];
        A[w][0] = lat_sub(lat_nib(wa), z);
        A[w][1] = lat_sub(lat_nib(wb), z);
        A[w][2] = lat_sub(lat_nib(wa >> 4), z);
        A[w][3] = lat_sub(lat_nib(wb >> 4), z);
        A[w][4] = lat_sub(lat_nib(wa >> 8), z);
        A[w][5] = lat_sub(lat_nib(wb >> 8), z);
        A[w][6] = lat_sub(lat_nib(wa >> 12), z);
        A[w][7] = lat_sub(lat_nib(wb >> 12), z);
    }
}

}  // namespace

// Shared memory: per-warp partials [ntmax][WK][16][M], per-CTA sums
// [ntmax][16][M] (read by the other ranks of a split-K cluster), then one
// x slot per warp: 72 words (64 + 8 pad words of 16 bytes) per super-block
// of the warp's k-slice (xsb = min(NI, k-slice length)); then the INT8 row
// scales of the CTA ([ntmax][16] fp32, `scf` floats, 0 for other formats);
// then the RMSNorm prologue's scratch ((16 + 1) x 8 floats, its own area: warps
// write their partials while others may still read the factors); then, for the
// staged variants, the item ring (W x NI x 2 KB).
constexpr int kLatNormFloats = (16 + 1) * 8;
__host__ __device__ inline size_t lat_red_floats(int ntmax, int WK, int M) {
    return ((size_t)ntmax * (WK + 1) * 16 * M + 3) / 4 * 4;  // 16-byte aligned end
}
__host__ __device__ inline size_t lat_sc_floats(int fmt, int ntmax) { return fmt == FMT_I8 ? (size_t)ntmax * 16 : 0; }
__host__ __device__ inline size_t lat_norm_off(int ntmax, int W, int WK, int M, int xsb, size_t scf) {
    return lat_red_floats(ntmax, WK, M) + (size_t)W * 72 * 4 * xsb + scf;
}
// (`fz`: the instantiation is the fused one, which alone has the norm area)
__host__ __device__ inline size_t lat_smem_floats(int ntmax, int W, int WK, int M, int xsb, size_t scf, int fz) {
    return lat_norm_off(ntmax, W, WK, M, xsb, scf) + (fz ? kLatNormFloats : 0);
}
__host__ __device__ inline size_t lat_ring_off(int ntmax, int W, int WK, int M, int xsb, size_t scf, int fz) {
    return (lat_smem_floats(ntmax, W, WK, M, xsb, scf, fz) * 4 + 127) / 128 * 128;
}

// W warps = WK along K x WT along the CTA's row tiles. Warp (wk, wt) owns
// super-blocks [b0, b0 + nb) of tiles wt, wt + WT, ... of the CTA's range.
// NI: most items a warp may own. NPRE: items unpacked before the wait.
// STG: items past NPRE wait in a shared-memory ring (cp.async). LEAN: the
// INT4 unpack and MMAs stream one 32-bit word at a time from the ring, with
// x read from the slot per word, so a warp needs few registers and 16 warps
// fit beside the next launch.
// FZ: 1 in the twin instantiated for fused calls (RMSNorm prologue, gated
// and residual epilogues); 0 compiles the fusions out.
template <int FMT, int W, int WT, int NI, int NPRE, int STG, int LEAN, int FZ>
__global__ void __launch_bounds__(W * 32, (16 / W) > 2 ? (16 / W) : 2)
    gemv_lat_kernel(const GemvArgs a, const int S) {
    static_assert(FMT == FMT_G64 || FMT == FMT_BF16 || FMT == FMT_I8, "INT4 group-64, INT8 and BF16 only");
    static_assert(FMT != FMT_BF16 || NPRE == 0, "BF16 needs no unpack");
    static_assert(FMT == FMT_G64 || LEAN == 0, "the lean path is INT4 only");
    static_assert(NPRE <= NI, "");
    static_assert(!LEAN || (STG && NPRE == 0), "the lean path reads staged items");
    static_assert(W % WT == 0, "");
    constexpr int WK = W / WT;
    constexpr int BK = (FMT == FMT_BF16) ? 64 : (FMT == FMT_I8) ? 128 : 256;  // k per 128-byte row super-block
    extern __shared__ float lat_smem[];

    pdl_launch_dependents();

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wk = warp % WK, wt = warp / WK;
    const int g = lane >> 2, q = lane & 3;
    const int G = gridDim.x / S;
    const int cgid = blockIdx.x / S;
    int t0, nt;  // the CTA's logical tiles (gate/up pairs under the gated epilogue)
    cta_tile_range<FZ>(a, G, cgid, t0, nt);
    const int ntmax = ((a.N + 15) / 16 + G - 1) / G * (gated<FZ>(a) ? 2 : 1);
    const int mb = a.M;
    const int KB = a.K / BK;  // the plan guarantees K % BK == 0
    const int BS = (KB + S * WK - 1) / (S * WK);
    const int b0 = rank * WK * BS + wk * BS;  // this warp's k-slice of super-blocks
    const int nb = max(0, min(KB, b0 + BS) - b0);
    const int ntw = (nt > wt) ? (nt - wt + WT - 1) / WT : 0;  // tiles of this warp
    const int total = ntw * nb;  // items of this warp; the plan guarantees total <= NI
    const size_t rowbytes = (FMT == FMT_BF16) ? (size_t)a.K * 2 : (FMT == FMT_I8) ? (size_t)a.K : (size_t)a.K / 2;
    const int xsb = min(NI, BS);  // x super-blocks per warp slot
    const size_t scf = lat_sc_floats(FMT, ntmax);

    // ---------------------------------------------- before the wait ----
    // Items live in registers (STG = 0), or -- past the first NPRE, which are
    // unpacked early -- in a per-warp shared-memory ring filled with cp.async
    // (STG = 1): one 2 KB ring slot per item (device.cuh: fragment lane L's
    // chunk c at c * 512 + L * 16, filled by sector-complete copies).
    u32x8 ra[NI], rb[NI];  // 32 bytes of rows g and g+8 per register-held item
    uint32_t rs[NI][2];    // group-64: the 2 fp16 scales of this lane's columns, rows g and g+8
    uint8_t* ringw = reinterpret_cast<uint8_t*>(lat_smem) + lat_ring_off(ntmax, W, WK, mb, xsb, scf, FZ) +
                     (size_t)warp * NI * 2048;
    uint8_t* ring = ringw + lane * 16;
#pragma unroll
    for (int j = 0; j < NI; ++j) {
        if (j < total) {
            const int tt = j / nb;
            const int b = b0 + (j - tt * nb);
            const int tile = t0 + wt + tt * WT;
            const uint8_t* Wt = tile_weights<FZ>(a, tile);
            const int trow = tile_row0<FZ>(a, tile);
            const int r0 = min(trow + g, a.N - 1);
            const int r1 = min(trow + g + 8, a.N - 1);
            const uint8_t* p0 = Wt + (size_t)r0 * rowbytes + (size_t)b * 128 + q * 32;
            const uint8_t* p1 = Wt + (size_t)r1 * rowbytes + (size_t)b * 128 + q * 32;
            if (!STG || j < NPRE) {
                ra[j] = ld_stream32(p0);
                rb[j] = ld_stream32(p1);
            } else {
                uint8_t* d = ringw + (size_t)j * 2048;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    cp_async16(d + ring_copy_dst(lane, c),
                               Wt + (size_t)min(trow + ring_copy_row(lane, c), a.N - 1) * rowbytes +
                                   (size_t)b * 128 + ring_copy_byte(lane));
            }
            if (FMT == FMT_G64) {
                const uint16_t* st = tile_scales<FZ>(a, tile);
                const uint16_t* s0 = st + (size_t)r0 * a.groups + (size_t)b * 4 + 2 * (q & 1);
                const uint16_t* s1 = st + (size_t)r1 * a.groups + (size_t)b * 4 + 2 * (q & 1);
                rs[j][0] = (uint32_t)ld_ro_u16(s0) | ((uint32_t)ld_ro_u16(s0 + 1) << 16);
                rs[j][1] = (uint32_t)ld_ro_u16(s1) | ((uint32_t)ld_ro_u16(s1 + 1) << 16);
            }
        }
    }
    if (STG) cp_async_commit();
    uint32_t A[NPRE > 0 ? NPRE : 1][8][8];
#pragma unroll
    for (int j = 0; j < NPRE; ++j) {
        if (j < total) {
            if (FMT == FMT_I8)
                lat_unpack_i8(ra[j], rb[j], A[j]);
            else
                lat_unpack(ra[j], rb[j], A[j]);
        }
    }
    // INT8: the fp32 scales of the CTA's rows (weights: read before the wait)
    float* rsc = lat_smem + lat_red_floats(ntmax, WK, mb) + (size_t)W * 72 * 4 * xsb;
    if (FMT == FMT_I8)
        for (int i = threadIdx.x; i < nt * 16; i += W * 32) {
            const int tl = t0 + (i >> 4);
            rsc[i] = __ldg(tile_rscale<FZ>(a, tl) + min(tile_row0<FZ>(a, tl) + (i & 15), a.N - 1));
        }

    // Addresses of the x words this lane reads after the wait: word i of the
    // warp's x (super-block i / (M * words per row), batch row, word) is
    // read by lane i % 32. At batch 1 word i is simply x + b0 * BK + 8 i.
    constexpr int XWSB = BK / 8;  // 16-byte x words per batch row per super-block
    constexpr int XLD = 2 * NI;   // most x loads per lane (M * XWSB <= 64 per super-block)
    const int sbw = mb * XWSB;    // words per super-block
    const int nxw = nb * sbw;     // words this warp reads
    auto x_addr = [&](int r) -> const uint16_t* {
        const int wi = lane + 32 * r;
        const int sb = wi / sbw, rem = wi - sb * sbw;
        const int m = rem / XWSB, w = rem - m * XWSB;
        return a.x + (size_t)m * a.K + (size_t)(b0 + sb) * BK + w * 8;
    };
    // the lean variant keeps its registers for after the wait and derives
    // these there (batch > 1 only)
    const uint16_t* xsrc[LEAN ? 1 : XLD];
    if (!LEAN && mb > 1) {
#pragma unroll
        for (int r = 0; r < XLD; ++r) xsrc[LEAN ? 0 : r] = (lane + 32 * r < nxw) ? x_addr(r) : nullptr;
    }
    const uint16_t* xlin = a.x + (size_t)b0 * BK + lane * 8;

    prefetch_l2_grid_share(a.x, (size_t)a.M * a.K * 2);
    // x is produced by the previous kernel in the stream: wait for it only now.
    pdl_wait();

    // ----------------------------------------------- after the wait ----
    // B fragment of this lane: column n = g.
    //   group-64: n = 4m + j carries batch m, group j of the super-block; lane
    //             (g, q) supplies it only when j == q (x words 8q .. 8q+7);
    //   BF16:     n = m; x words 2q, 2q+1 of the super-block;
    //   INT8:     n = m; x words 4q .. 4q+3 of the super-block.
    int xm;
    bool xon;
    if (FMT == FMT_G64) {
        xm = g >> 2;
        xon = (xm < mb) && ((g & 3) == q);
    } else {
        xm = g;
        xon = xm < mb;
    }
    constexpr int XWL = (FMT == FMT_G64) ? 8 : (FMT == FMT_I8) ? 4 : 2;  // x words per B-fragment lane per super-block
    // The warp reads all the x it needs in one round of 16-byte loads and
    // hands each B-fragment lane its words through a per-warp shared-memory
    // slot (one pad word per 8 keeps those reads conflict-free). Loading per
    // item, a lane issuing eight loads itself, or eight rounds of shuffles
    // each cost more latency.
    uint4* xslot = reinterpret_cast<uint4*>(lat_smem + lat_red_floats(ntmax, WK, mb)) + (size_t)warp * (72 * xsb);
    // RMSNorm prologue: the CTA's factor per batch row
    float* nscr = lat_smem + lat_norm_off(ntmax, W, WK, mb, xsb, scf);
    if (FZ && a.norm_w) norm_factors(a, nscr, W * 32);
    {
        uint4 v[XLD];
#pragma unroll
        for (int r = 0; r < XLD; ++r) {
            v[r] = make_uint4(0, 0, 0, 0);
            if (lane + 32 * r < nxw)
                v[r] = ld_ro16(mb == 1 ? xlin + 256 * r : LEAN ? x_addr(r) : xsrc[LEAN ? 0 : r]);
        }
#pragma unroll
        for (int r = 0; r < XLD; ++r) {
            const int wi = lane + 32 * r;
            if (FZ && wi < nxw && a.norm_w) {
                const int sb = wi / sbw, rem = wi - sb * sbw;
                const int m = rem / XWSB, w = rem - m * XWSB;
                v[r] = norm_word(v[r], nscr[W * mb + m], a.norm_w + (size_t)(b0 + sb) * BK + w * 8);
            }
            if (wi < nxw)
                xslot[wi + (wi >> 3)] = (FMT == FMT_G64) ? lat_perm(v[r]) : (FMT == FMT_I8) ? perm_i8(v[r]) : v[r];
        }
    }
    __syncwarp();
    // slot index of this lane's first x word of super-block sb of its k-slice
    auto xword0 = [&](int sb) {
        return sb * sbw + ((FMT == FMT_G64) ? (min(xm, 1) * 32 + 8 * q) : (FMT == FMT_I8) ? (g * 16 + 4 * q) : (g * 8 + 2 * q));
    };
    uint4 xv[LEAN ? 1 : XWL];
    auto load_x = [&](int sb) {
#pragma unroll
        for (int w = 0; w < XWL; ++w) {
            const int wi = xword0(sb) + w;
            xv[w] = xon ? xslot[wi + (wi >> 3)] : make_uint4(0, 0, 0, 0);
        }
    };
    if (!LEAN && total > 0) load_x(0);
    if (STG) {
        cp_async_wait<0>();  // this lane's copies have landed
        __syncwarp();        // and so have the other lanes'
    }

    float* red = lat_smem;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc2[4] = {0.f, 0.f, 0.f, 0.f};  // BF16: second MMA chain
#pragma unroll
    for (int j = 0; j < NI; ++j) {
        if (j < total) {
            const int tt = j / nb;
            const int bi = j - tt * nb;
            if (LEAN) {
                // stream the item from the ring one 32-bit word at a time
                const uint8_t* d = ring + (size_t)j * 2048;
                const int x0 = xword0(bi);
                float dd[4][4] = {};
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint4 ca = *reinterpret_cast<const uint4*>(d + c * 512);
                    const uint4 cb = *reinterpret_cast<const uint4*>(d + 1024 + c * 512);
                    const uint32_t wa4[4] = {ca.x, ca.y, ca.z, ca.w};
                    const uint32_t wb4[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int w = 4 * c + u;
                        uint4 x4 = make_uint4(0, 0, 0, 0);
                        if (xon) x4 = xslot[x0 + w + ((x0 + w) >> 3)];
                        const uint32_t wa = wa4[u], wb = wb4[u];
                        const uint32_t z = 0x43084308u;
                        lat_mma(dd[(w & 1) * 2], lat_sub(lat_nib(wa), z), lat_sub(lat_nib(wb), z),
                                lat_sub(lat_nib(wa >> 4), z), lat_sub(lat_nib(wb >> 4), z), x4.x, x4.y);
                        lat_mma(dd[(w & 1) * 2 + 1], lat_sub(lat_nib(wa >> 8), z), lat_sub(lat_nib(wb >> 8), z),
                                lat_sub(lat_nib(wa >> 12), z), lat_sub(lat_nib(wb >> 12), z), x4.z, x4.w);
                    }
                }
                float ds[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) ds[i] = (dd[0][i] + dd[1][i]) + (dd[2][i] + dd[3][i]);
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&rs[j][0]));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&rs[j][1]));
                acc[0] = fmaf(f0.x, ds[0], acc[0]);
                acc[0] = fmaf(f0.y, ds[1], acc[0]);
                acc[2] = fmaf(f1.x, ds[2], acc[2]);
                acc[2] = fmaf(f1.y, ds[3], acc[2]);
            } else {
                if (j > 0 && nb > 1) load_x(bi);
                if (STG && j >= NPRE) {
                    const uint8_t* d = ring + (size_t)j * 2048;
                    const uint4 c0 = *reinterpret_cast<const uint4*>(d);
                    const uint4 c1 = *reinterpret_cast<const uint4*>(d + 512);
                    const uint4 c2 = *reinterpret_cast<const uint4*>(d + 1024);
                    const uint4 c3 = *reinterpret_cast<const uint4*>(d + 1536);
                    ra[j] = u32x8{{c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w}};
                    rb[j] = u32x8{{c2.x, c2.y, c2.z, c2.w, c3.x, c3.y, c3.z, c3.w}};
                }
                if (FMT == FMT_G64) {
                    uint32_t Aj[8][8];
                    if (j < NPRE) {
#pragma unroll
                        for (int w = 0; w < 8; ++w)
#pragma unroll
                            for (int i = 0; i < 8; ++i) Aj[w][i] = A[j < NPRE ? j : 0][w][i];
                    } else {
                        lat_unpack(ra[j], rb[j], Aj);
                    }
                    // four independent accumulator chains of four MMAs each
                    float d[4][4] = {};
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        lat_mma(d[(w & 1) * 2], Aj[w][0], Aj[w][1], Aj[w][2], Aj[w][3], xv[w].x, xv[w].y);
                        lat_mma(d[(w & 1) * 2 + 1], Aj[w][4], Aj[w][5], Aj[w][6], Aj[w][7], xv[w].z, xv[w].w);
                    }
                    float ds[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) ds[i] = (d[0][i] + d[1][i]) + (d[2][i] + d[3][i]);
                    // columns 2q, 2q+1 = groups 2(q&1), 2(q&1)+1 of batch q>>1
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&rs[j][0]));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&rs[j][1]));
                    acc[0] = fmaf(f0.x, ds[0], acc[0]);
                    acc[0] = fmaf(f0.y, ds[1], acc[0]);
                    acc[2] = fmaf(f1.x, ds[2], acc[2]);
                    acc[2] = fmaf(f1.y, ds[3], acc[2]);
                } else if (FMT == FMT_I8) {
                    uint32_t Aj[8][8];
                    if (j < NPRE) {
#pragma unroll
                        for (int w = 0; w < 8; ++w)
#pragma unroll
                            for (int i = 0; i < 4; ++i) Aj[w][i] = A[j < NPRE ? j : 0][w][i];
                    } else {
                        lat_unpack_i8(ra[j], rb[j], Aj);
                    }
                    // four independent accumulator chains of two MMAs each
                    float d[4][4] = {};
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const uint4 x4 = xv[w >> 1];
                        lat_mma(d[w & 3], Aj[w][0], Aj[w][1], Aj[w][2], Aj[w][3], (w & 1) ? x4.z : x4.x,
                                (w & 1) ? x4.w : x4.y);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] += (d[0][i] + d[1][i]) + (d[2][i] + d[3][i]);
                } else {
                    const u32x8& wa = ra[j];
                    const u32x8& wb = rb[j];
                    lat_mma(acc, wa.v[0], wb.v[0], wa.v[1], wb.v[1], xv[0].x, xv[0].y);
                    lat_mma(acc2, wa.v[2], wb.v[2], wa.v[3], wb.v[3], xv[0].z, xv[0].w);
                    lat_mma(acc, wa.v[4], wb.v[4], wa.v[5], wb.v[5], xv[1].x, xv[1].y);
                    lat_mma(acc2, wa.v[6], wb.v[6], wa.v[7], wb.v[7], xv[1].z, xv[1].w);
                }
            }
            if (bi == nb - 1) {
                // end of this warp's k-slice of its tile: per-warp partials
                const int t = wt + tt * WT;
                float* rp = red + ((size_t)(t * WK + wk) * 16) * mb;
                if (FMT == FMT_G64) {
                    const float v0 = acc[0] + __shfl_xor_sync(0xFFFFFFFFu, acc[0], 1);
                    const float v2 = acc[2] + __shfl_xor_sync(0xFFFFFFFFu, acc[2], 1);
                    const int m = q >> 1;
                    if ((q & 1) == 0 && m < mb) {
                        rp[g * mb + m] = v0;
                        rp[(g + 8) * mb + m] = v2;
                    }
                } else {
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
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = acc2[i] = 0.f;
            }
        }
    }
    if (nb == 0) {
        // an empty k-slice still contributes zeros for each of its tiles
        for (int t = wt; t < nt; t += WT) {
            float* rp = red + ((size_t)(t * WK + wk) * 16) * mb;
            for (int i = lane; i < 16 * mb; i += 32) rp[i] = 0.f;
        }
    }
    __syncthreads();

    // each output: the sum over the K-warps in order. Local logical row lr
    // (tile lr / 16) of batch row m; under the gated epilogue output row o
    // pairs gate row gate_row(o) with up row gate_row(o) + 16.
    const int nto = gated<FZ>(a) ? nt / 2 : nt;
    const int orow0 = (gated<FZ>(a) ? t0 / 2 : t0) * 16;
    auto gate_row = [&](int o) { return gated<FZ>(a) ? (o >> 4) * 32 + (o & 15) : o; };
    auto wsum = [&](int lr, int m) -> float {
        const float* rp = red + ((size_t)(lr >> 4) * WK * 16 + (lr & 15)) * mb + m;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < WK; ++w) v += rp[(size_t)w * 16 * mb];
        return v;
    };
    if (S == 1) {
        for (int i = threadIdx.x; i < nto * 16 * mb; i += W * 32) {
            const int o = (mb == 1) ? i : i / mb;
            const int m = (mb == 1) ? 0 : i - o * mb;
            if (orow0 + o >= a.N) continue;
            const int lr = gate_row(o);
            float v = wsum(lr, m), v2 = 0.f;
            if (FMT == FMT_I8) v *= rsc[lr];
            if (gated<FZ>(a)) {
                v2 = wsum(lr + 16, m);
                if (FMT == FMT_I8) v2 *= rsc[lr + 16];
            }
            store_fused<FZ>(a, m, orow0 + o, v, v2);
        }
        return;
    }
    float* fin = red + (size_t)ntmax * WK * 16 * mb;  // [lr][m]: this rank's sums
    for (int i = threadIdx.x; i < nt * 16 * mb; i += W * 32) fin[i] = wsum(i / mb, i - (i / mb) * mb);
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    // rank s writes output rows [s * Ro / S, (s + 1) * Ro / S) of the CTA group's Ro rows
    const int Ro = nto * 16;
    const int lo = rank * Ro / S, hi = (rank + 1) * Ro / S;
    const int span = hi - lo;
    for (int i = threadIdx.x; i < span * mb; i += W * 32) {
        const int o = lo + i / mb;
        const int m = i - (i / mb) * mb;
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
namespace {
using LatFn = void (*)(const GemvArgs, const int);
struct LatEntry {
    LatConfig cfg;
    LatFn fn;   // plain calls
    LatFn fnf;  // fused calls (the FZ = 1 twin)
};
#define MBW_L(F, W, WT, NI, NP, ST, LN) \
    { {W, WT, NI, NP, ST, LN}, gemv_lat_kernel<F, W, WT, NI, NP, ST, LN, 0>, gemv_lat_kernel<F, W, WT, NI, NP, ST, LN, 1> }
const LatEntry kLatG64[] = {
    MBW_L(FMT_G64, 8, 1, 1, 1, 0, 0), MBW_L(FMT_G64, 8, 1, 1, 0, 0, 0), MBW_L(FMT_G64, 8, 1, 2, 0, 0, 0),
    MBW_L(FMT_G64, 8, 1, 3, 0, 0, 0), MBW_L(FMT_G64, 4, 1, 1, 1, 0, 0), MBW_L(FMT_G64, 8, 1, 2, 1, 1, 0),
    MBW_L(FMT_G64, 8, 1, 4, 1, 1, 0), MBW_L(FMT_G64, 8, 1, 6, 0, 1, 0), MBW_L(FMT_G64, 16, 2, 2, 0, 1, 1),
    MBW_L(FMT_G64, 16, 2, 3, 0, 1, 1), MBW_L(FMT_G64, 16, 1, 2, 0, 1, 1), MBW_L(FMT_G64, 8, 1, 3, 0, 1, 1),
    MBW_L(FMT_G64, 8, 1, 5, 0, 1, 1)};
const LatEntry kLatI8[] = {MBW_L(FMT_I8, 8, 1, 1, 1, 0, 0), MBW_L(FMT_I8, 8, 1, 2, 1, 0, 0), MBW_L(FMT_I8, 8, 1, 2, 0, 0, 0),
                           MBW_L(FMT_I8, 8, 1, 3, 0, 0, 0), MBW_L(FMT_I8, 8, 1, 4, 0, 1, 0), MBW_L(FMT_I8, 8, 1, 6, 0, 1, 0),
                           MBW_L(FMT_I8, 16, 1, 2, 0, 0, 0), MBW_L(FMT_I8, 4, 1, 2, 1, 0, 0)};
const LatEntry kLatBf16[] = {MBW_L(FMT_BF16, 8, 1, 2, 0, 0, 0), MBW_L(FMT_BF16, 8, 1, 4, 0, 0, 0),
                             MBW_L(FMT_BF16, 4, 1, 4, 0, 0, 0), MBW_L(FMT_BF16, 16, 1, 2, 0, 0, 0),
                             MBW_L(FMT_BF16, 16, 2, 2, 0, 0, 0), MBW_L(FMT_BF16, 8, 1, 4, 0, 1, 0),
                             MBW_L(FMT_BF16, 8, 1, 6, 0, 1, 0)};
#undef MBW_L

const LatEntry* lat_table(int fmt, int* n) {
    if (fmt == FMT_G64) {
        *n = (int)(sizeof(kLatG64) / sizeof(kLatG64[0]));
        return kLatG64;
    }
    if (fmt == FMT_BF16) {
        *n = (int)(sizeof(kLatBf16) / sizeof(kLatBf16[0]));
        return kLatBf16;
    }
    if (fmt == FMT_I8) {
        *n = (int)(sizeof(kLatI8) / sizeof(kLatI8[0]));
        return kLatI8;
    }
    *n = 0;
    return nullptr;
}
}  // namespace

int lat_num_configs(int fmt) {
    int n;
    lat_table(fmt, &n);
    return n;
}

LatConfig lat_config(int fmt, int idx) {
    int n;
    return lat_table(fmt, &n)[idx].cfg;
}

// the per-warp x slot holds 64 words per super-block: M * (x words per row per super-block) <= 64
int lat_max_batch(int fmt) { return fmt == FMT_G64 ? 2 : fmt == FMT_I8 ? 4 : 8; }
int lat_block_k(int fmt) { return fmt == FMT_BF16 ? 64 : fmt == FMT_I8 ? 128 : 256; }

// Most items any warp owns under this split (0 if the shape does not fit the family).
int lat_items_per_warp(int fmt, const LatConfig& c, int64_t N, int64_t K, int split, int occ, int glu) {
    const int BK = lat_block_k(fmt);
    if (K % BK != 0) return 0;
    const int WK = c.warps / c.wt;
    const int64_t KB = K / BK;
    const int64_t BS = (KB + (int64_t)split * WK - 1) / ((int64_t)split * WK);
    if ((int64_t)(split - 1) * WK * BS >= KB) return 0;  // a cluster rank without k-range
    const int G = mma_row_groups(N, split, occ);
    const int64_t T = (N + 15) / 16;
    const int64_t ntmax = (T + G - 1) / G * (glu ? 2 : 1);
    return (int)((ntmax + c.wt - 1) / c.wt * BS);
}

size_t lat_smem_bytes(int fmt, const LatConfig& c, int64_t N, int64_t K, int M, int split, int occ, int glu, int fz) {
    const int G = mma_row_groups(N, split, occ);
    const int64_t T = (N + 15) / 16;
    const int ntmax = (int)((T + G - 1) / G) * (glu ? 2 : 1);
    const int WK = c.warps / c.wt;
    const int64_t KB = K / lat_block_k(fmt);
    const int64_t BS = (KB + (int64_t)split * WK - 1) / ((int64_t)split * WK);
    const int xsb = (int)std::min<int64_t>(c.ni, BS);
    const size_t scf = lat_sc_floats(fmt, ntmax);
    if (c.staged) return lat_ring_off(ntmax, c.warps, WK, M, xsb, scf, fz) + (size_t)c.warps * c.ni * 2048;
    return lat_smem_floats(ntmax, c.warps, WK, M, xsb, scf, fz) * sizeof(float);
}

cudaError_t launch_gemv_lat(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s) {
    // a gated launch reads the up matrix's codes, scales (not BF16) and zero points (AWQ)
    if (a.glu && (!a.W2 || (fmt != FMT_BF16 && !a.scales2) || (fmt == FMT_AWQ && !a.zeros2)))
        return cudaErrorInvalidValue;
    int n;
    const LatEntry* t = lat_table(fmt, &n);
    if (t == nullptr || p.cfg < 0 || p.cfg >= n || a.M < 1 || a.M > lat_max_batch(fmt)) return cudaErrorInvalidValue;
    const LatEntry& e = t[p.cfg];
    const int items = lat_items_per_warp(fmt, e.cfg, a.N, a.K, p.split, p.occ, a.glu);
    if (items < 1 || items > e.cfg.ni) return cudaErrorInvalidValue;
    const int G = mma_row_groups(a.N, p.split, p.occ);
    const int fz = gemv_fused_args(a);
    const size_t smem = lat_smem_bytes(fmt, e.cfg, a.N, a.K, a.M, p.split, p.occ, a.glu, fz);
    const LatFn fn = fz ? e.fnf : e.fn;
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

}  // namespace mbw
