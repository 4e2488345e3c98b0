// gemv_awq_batch.cu -- AWQ-style INT4 (group 128) product for a batch of
// 5 .. 64 activation rows, and the symmetric INT8 one for 9 .. 64, on the
// mma.sync tensor-core path, every weight read once per launch.
//
// Y[m][i] = sum_g s[i][g] * sum_{k in g} (q[i][k] - z[i][g]) * X[m][k]
// (llm-rs vs vLLM, sec. 6 format table: 4-bit codes with an fp16 scale and a
// zero point per 128 weights; sec. 3: batching moves decode from memory toward
// math: the weights are streamed once for all M rows).
//
// Why this family next to the tcgen05 one: at batch 16 the tensor work per
// weight byte is small enough for mma.sync, and the unpacked codes go from the
// registers they were loaded into straight to the MMA's A operand -- no store
// of the converted operand to shared or tensor memory and no per-group hand-
// over between unpack, MMA and read-back roles.
//
// Mapping (swap-AB: weight rows on the MMA's M side, the batch on its N side,
// 8 batch rows per n-block, NB n-blocks):
//   * weight rows are cut into 16-row tiles; CTA row-group c of G owns the
//     contiguous tile range [c*T/G, (c+1)*T/G);
//   * K is cut into super-blocks of 256 (two groups); cluster rank r of S owns
//     super-blocks [KB*r/S, KB*(r+1)/S) and splits them evenly over its warps
//     (a warp may get none when the rank has fewer super-blocks than warps);
//     each warp walks (tile, super-block) through a U-deep register ring;
//   * lane (g = lane/4, q = lane%4) loads, for rows g and g+8 of the tile, 16
//     bytes of the first group (bytes 16q .. 16q+15 of the 128-byte row block)
//     and 16 bytes of the second (bytes 64+16q ..): so a quad's 4 words w of
//     one group hold 32 consecutive codes each lane, and every MMA -- one code
//     word of each quad lane, two MMAs per word -- sums within one group, whose
//     fp32 partial is then scaled by that group's scale;
//   * X (the CTA's k-range, all batch rows, zero rows past M) is staged in
//     shared memory after the programmatic-dependent-launch wait, in the k
//     order of the code nibbles, with lane q's 16-byte words of a group
//     transposed (word w of lane q at 4w + q) and a row pitch of 4 (mod 8)
//     16-byte chunks, so that each 8-lane phase of a B-fragment load hits 8
//     distinct bank groups;
//   * at the end of each tile the warps' fp32 partials go to one of two
//     shared-memory slots, one barrier, and all threads sum them over warps in
//     warp order and store (or keep them for the cluster's DSMEM sum in rank
//     order): deterministic, no global scratch.
//
// Exactness: a code n in a bf16 pair is 0x4300 | n = 128 + n; subtracting the
// bf16 pair 128 + z gives n - z exactly; (n - z) * x is exact in fp32 and the
// tensor core accumulates in fp32; the group scale multiplies the group's fp32
// sum once.
//
// Symmetric INT8 with one fp32 scale per output channel (TileInfer, "Pushing
// further with cheating: INT8 quantization") runs through the same skeleton
// at batches above the INT8 GEMVs' 8 rows: a 128-byte super-block of a row is
// 128 codes (128 k), the lane's 16-byte chunks of rows g and g+8 become exact
// bf16 pairs (i8_pairs: codes 0, 2 and 1, 3 of each word), X is staged with
// the matching pair permutation (perm_i8) at an odd row pitch, the MMAs
// accumulate over the warp's whole k-range, and the row's scale multiplies the
// finished sum once in the store.
#include <cooperative_groups.h>

#include <algorithm>

#include "device.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace mbw {

namespace {

__device__ __forceinline__ void awqb_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// nibbles at bits 0-3 and 16-19 of v minus the zero point, as a bf16 pair:
// ((v & 0x000F000F) | 0x43004300) - (128 + z, 128 + z)
__device__ __forceinline__ uint32_t awqb_pair(uint32_t v, uint32_t zz) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(0x000F000Fu), "r"(0x43004300u));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(zz));
    return r;
}

// 8 bf16 x[8w..8w+7] -> pairs (0,4) (1,5) (2,6) (3,7): the order in which the
// canonical codes' nibble pairs come out of awqb_pair (slots t and t + 4).
__device__ __forceinline__ uint4 awqb_perm(uint4 v) {
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    return o;
}

}  // namespace

// Shared memory of one launch: staged X [Mp][pitch] 16-byte chunks, then the
// warps' per-tile partials [ntmax][WK][16][Mp] fp32 (when WK > 1 or S > 1),
// then (WK > 1 and S > 1) the CTA's tile sums [ntmax][16][Mp] fp32 for the
// cluster's sum; with the shared-memory ring (async) also the warps' rings
// [W][U][4][32][16 B] and the CTA's scale [ntmax][16][2 kbr] fp16 and zero-point
// [ntmax][16][kbr] byte tables.
struct AwqbSmem {
    int pitch;  // 16-byte chunks per staged X row
    int ntmax;  // most tiles any CTA owns
    int kbr;    // most super-blocks any cluster rank owns
    size_t red_off, fin_off, ring_off, stab_off, ztab_off, total;
};

__host__ __device__ inline AwqbSmem awqb_smem_layout(int fmt, int64_t K, int64_t N, int Mp, int W, int WK, int U,
                                                     int async, int S, int G) {
    AwqbSmem L;
    const bool i8 = fmt == FMT_I8;
    const int KB = (int)(K / (i8 ? 128 : 256));
    L.kbr = (KB + S - 1) / S;
    // INT8: 16 chunks per super-block and an odd pitch (each 8-lane phase of a
    // B-fragment read then covers 8 bank groups)
    L.pitch = i8 ? L.kbr * 16 + 1 : L.kbr * 32 + 4;
    const int64_t T = (N + 15) / 16;
    L.ntmax = (int)((T + G - 1) / G);
    L.red_off = (size_t)Mp * L.pitch * 16;
    const size_t red = (WK > 1 || S > 1) ? (size_t)L.ntmax * WK * 16 * Mp * 4 : 0;
    L.fin_off = L.red_off + red;
    L.ring_off = L.fin_off + ((WK > 1 && S > 1) ? (size_t)L.ntmax * 16 * Mp * 4 : 0);
    const bool tabs = async && !i8;  // AWQ scale and zero-point tables
    L.stab_off = L.ring_off + (async ? (size_t)W * U * 2048 : 0);
    L.ztab_off = L.stab_off + (tabs ? (size_t)L.ntmax * 16 * 2 * L.kbr * 2 : 0);
    L.total = L.ztab_off + (tabs ? ((size_t)L.ntmax * 16 * L.kbr + 15) / 16 * 16 : 0);
    return L;
}

// W = WT x WK warps: warp (wt, wk) owns the CTA's tiles wt, wt + WT, ... and
// k-slice wk of WK of the CTA's super-blocks.
// EARLY: 1 = a ring slot is copied out and refilled before its super-block is
// computed (U super-blocks of loads in flight during the compute, 19 more
// registers), 0 = refilled after (U - 1 in flight).
// ASYNC: 1 = the ring is in shared memory, filled by each lane's own 16-byte
// cp.async copies (a quad's four copies of a row's group are one 64-byte run:
// whole sectors), U slots deep per warp, refilled after its super-block is
// computed; scales and zero points come from per-CTA tables loaded once.
template <int FMT, int NB, int WT, int WK, int U, int MINB, int EARLY, int ASYNC>
__global__ void __launch_bounds__(WT * WK * 32, MINB) gemv_awq_batch_kernel(const GemvArgs a, const int S) {
    constexpr bool I8 = (FMT == FMT_I8);
    constexpr int BKS = I8 ? 128 : 256;  // k per 128-byte row super-block
    constexpr int W = WT * WK;
    constexpr int MP = 8 * NB;  // batch rows of the launch, padded
    extern __shared__ uint4 smem_u4[];

    pdl_launch_dependents();

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wt = warp % WT, wk = warp / WT;
    const int g = lane >> 2, q = lane & 3;
    const int G = gridDim.x / S;
    const int cgid = blockIdx.x / S;
    const int T = (a.N + 15) / 16;
    const int t0 = (int)(((long long)T * cgid) / G);
    const int nt = (int)(((long long)T * (cgid + 1)) / G) - t0;
    const AwqbSmem L = awqb_smem_layout(FMT, a.K, a.N, MP, W, WK, U, ASYNC, S, G);

    // super-blocks of this cluster rank, then of this warp's k-slice (may be none)
    const int KB = a.K / BKS;
    const int kb0 = (int)(((long long)KB * rank) / S);
    const int nkb = (int)(((long long)KB * (rank + 1)) / S) - kb0;
    const int wb0 = kb0 + (nkb * wk) / WK;
    const int nbw = kb0 + (nkb * (wk + 1)) / WK - wb0;
    const int ntw = (nt > wt) ? (nt - wt + WT - 1) / WT : 0;  // tiles of this warp
    const int total = ntw * nbw;
    const size_t rowbytes = I8 ? (size_t)a.K : (size_t)a.K / 2;

    // load cursor: rows g and g + 8 of the tile being loaded, as 32-bit offsets
    // from the matrix (code bytes, scale and zero-point entries; the launch
    // requires N * K / 2 < 2^32)
    int lb = 0, lt = 0;
    uint32_t wo0 = 0, wo1 = 0, so0 = 0, so1 = 0, zo0 = 0, zo1 = 0;
    auto set_rows = [&](int i) {
        const int trow = (t0 + wt + i * WT) * 16;
        const uint32_t r0 = (uint32_t)min(trow + g, a.N - 1);
        const uint32_t r1 = (uint32_t)min(trow + g + 8, a.N - 1);
        wo0 = r0 * (uint32_t)rowbytes + (uint32_t)wb0 * 128u + (uint32_t)q * 16u;
        wo1 = r1 * (uint32_t)rowbytes + (uint32_t)wb0 * 128u + (uint32_t)q * 16u;
        so0 = r0 * (uint32_t)a.groups + (uint32_t)wb0 * 2u;
        so1 = r1 * (uint32_t)a.groups + (uint32_t)wb0 * 2u;
        zo0 = r0 * (uint32_t)a.zstride + (uint32_t)wb0;
        zo1 = r1 * (uint32_t)a.zstride + (uint32_t)wb0;
    };
    if (total > 0) set_rows(0);

    uint4 rc[U][4];    // [u][0] row g group 0, [1] row g group 1, [2] row g+8 group 0, [3] row g+8 group 1
    uint32_t rs[U][2];  // fp16 scales of groups 0 | 1 << 16: row g, row g+8
    uint32_t rz[U];     // zero-point byte of row g (bits 0-7) and row g+8 (bits 8-15)
    // async ring of this warp: slot u, chunk c (the rc[u][c] order) of lane L at (u * 4 + c) * 512 + L * 16
    uint8_t* aring = reinterpret_cast<uint8_t*>(smem_u4) + L.ring_off + (size_t)warp * U * 2048 + lane * 16;
    auto load = [&](int u) {
        if (ASYNC) {
            cp_async16(aring + (size_t)(u * 4 + 0) * 512, a.W + wo0);
            cp_async16(aring + (size_t)(u * 4 + 1) * 512, a.W + wo0 + 64);
            cp_async16(aring + (size_t)(u * 4 + 2) * 512, a.W + wo1);
            cp_async16(aring + (size_t)(u * 4 + 3) * 512, a.W + wo1 + 64);
            wo0 += 128;
            wo1 += 128;
            if (++lb == nbw) {
                lb = 0;
                if (++lt < ntw) set_rows(lt);
            }
            return;
        }
        rc[u][0] = ld_stream16(a.W + wo0);
        rc[u][1] = ld_stream16(a.W + wo0 + 64);
        rc[u][2] = ld_stream16(a.W + wo1);
        rc[u][3] = ld_stream16(a.W + wo1 + 64);
        if (!I8) {
            rs[u][0] = (uint32_t)ld_ro_u16(a.scales + so0) | ((uint32_t)ld_ro_u16(a.scales + so0 + 1) << 16);
            rs[u][1] = (uint32_t)ld_ro_u16(a.scales + so1) | ((uint32_t)ld_ro_u16(a.scales + so1 + 1) << 16);
            rz[u] = (uint32_t)ld_ro_u8(a.zeros + zo0) | ((uint32_t)ld_ro_u8(a.zeros + zo1) << 8);
        }
        wo0 += 128;
        wo1 += 128;
        so0 += 2;
        so1 += 2;
        zo0 += 1;
        zo1 += 1;
        if (++lb == nbw) {
            lb = 0;
            if (++lt < ntw) set_rows(lt);
        }
    };
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (u < total) load(u);
        if (ASYNC) cp_async_commit();  // one group per step, empty past the end
    }
    uint16_t* stab = reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(smem_u4) + L.stab_off);
    uint8_t* ztab = reinterpret_cast<uint8_t*>(smem_u4) + L.ztab_off;
    if (ASYNC && !I8) {
        // the CTA's scales (2 per super-block) and zero-point bytes (1 per
        // super-block) of its rows and this rank's super-blocks; weights-side
        // data, read before the wait
        for (int i = threadIdx.x; i < nt * 16 * nkb; i += W * 32) {
            const int tr = i / nkb, sbl = i - tr * nkb;
            const int row = min((t0 + tr / 16) * 16 + (tr & 15), a.N - 1);
            const size_t gi = (size_t)row * a.groups + (size_t)(kb0 + sbl) * 2;
            stab[((size_t)tr * L.kbr + sbl) * 2] = ld_ro_u16(a.scales + gi);
            stab[((size_t)tr * L.kbr + sbl) * 2 + 1] = ld_ro_u16(a.scales + gi + 1);
            ztab[(size_t)tr * L.kbr + sbl] = ld_ro_u8(a.zeros + (size_t)row * a.zstride + kb0 + sbl);
        }
    }

    prefetch_l2_grid_share(a.x, (size_t)a.M * a.K * 2);
    pdl_wait();

    // Stage X[:, kb0*BKS .. (kb0 + nkb)*BKS) for MP rows (zeros past M).
    // AWQ: logical chunk c of a super-block = 16 h + 4 q' + w' goes to 16 h + 4 w' + q'.
    // INT8: chunks in order, each 8-x chunk as the pairs (0,2) (1,3) (4,6) (5,7).
    uint4* xs = smem_u4;
    const int cpr = nkb * (BKS / 8);  // chunks per row
    for (int i = threadIdx.x; i < MP * cpr; i += W * 32) {
        const int m = i / cpr, c = i - m * cpr;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (m < a.M) {
            v = ld_ro16(a.x + (size_t)m * a.K + (size_t)kb0 * BKS + (size_t)c * 8);
            if (I8)
                v = perm_i8(v);
            else if (!a.x_natural)
                v = awqb_perm(v);
        }
        int phys = c;
        if (!I8) {
            const int c32 = c & 31;
            phys = (c & ~31) | (c32 & 16) | ((c32 & 3) << 2) | ((c32 >> 2) & 3);
        }
        xs[(size_t)m * L.pitch + phys] = v;
    }
    __syncthreads();

    float* red = reinterpret_cast<float*>(reinterpret_cast<char*>(smem_u4) + L.red_off);
    float* fin = reinterpret_cast<float*>(reinterpret_cast<char*>(smem_u4) + ((WK > 1) ? L.fin_off : L.red_off));
    // B fragments of this lane: batch row 8 nb + g; AWQ: chunk 4 w' + q of each
    // group; INT8: chunks 2q, 2q + 1 of each 64-byte half of the super-block
    const uint4* xl = I8 ? xs + (size_t)g * L.pitch + 2 * q + (size_t)(wb0 - kb0) * 16
                         : xs + (size_t)g * L.pitch + q + (size_t)(wb0 - kb0) * 32;

    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
    float acc1[1][4] = {{0.f, 0.f, 0.f, 0.f}};  // INT8 at one n-block: a second accumulator chain
    int j = 0, lt2 = 0;
    for (int s0 = 0; s0 < total; s0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (s0 + u < total) {
                const uint4* xb = xl + j * (BKS / 8);
                uint4 cw[4];
                uint32_t cs[2], cz;
                if (ASYNC) {
                    cp_async_wait<U - 1>();  // this lane's copies of the step have landed
#pragma unroll
                    for (int e = 0; e < 4; ++e) cw[e] = *reinterpret_cast<const uint4*>(aring + (size_t)(u * 4 + e) * 512);
                    cs[0] = cs[1] = cz = 0;
                    if (!I8) {
                        const int tr = (wt + lt2 * WT) * 16, sbl = wb0 - kb0 + j;
                        cs[0] = *reinterpret_cast<const uint32_t*>(stab + ((size_t)(tr + g) * L.kbr + sbl) * 2);
                        cs[1] = *reinterpret_cast<const uint32_t*>(stab + ((size_t)(tr + g + 8) * L.kbr + sbl) * 2);
                        cz = (uint32_t)ztab[(size_t)(tr + g) * L.kbr + sbl] |
                             ((uint32_t)ztab[(size_t)(tr + g + 8) * L.kbr + sbl] << 8);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) cw[e] = rc[u][e];
                    cs[0] = I8 ? 0u : rs[u][0];
                    cs[1] = I8 ? 0u : rs[u][1];
                    cz = I8 ? 0u : rz[u];
                    if (EARLY && s0 + u + U < total) load(u);
                }
                if (I8) {
                    // word w of a lane's 16-byte chunk holds codes k0 .. k0 + 3: its pairs (0,2), (1,3)
                    // meet the x pairs of the chunk's half (w & 1) of staged chunk 2q + (w >> 1)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t wa[4] = {cw[h].x, cw[h].y, cw[h].z, cw[h].w};
                        const uint32_t wb[4] = {cw[2 + h].x, cw[2 + h].y, cw[2 + h].z, cw[2 + h].w};
#pragma unroll
                        for (int wp = 0; wp < 2; ++wp) {
                            uint32_t a02[2], a13[2], b02[2], b13[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                i8_pairs(wa[2 * wp + e], a02[e], a13[e]);
                                i8_pairs(wb[2 * wp + e], b02[e], b13[e]);
                            }
#pragma unroll
                            for (int nb = 0; nb < NB; ++nb) {
                                const uint4 xv = xb[(size_t)nb * 8 * L.pitch + h * 8 + wp];
                                awqb_mma(acc[nb], a02[0], b02[0], a13[0], b13[0], xv.x, xv.y);
                                awqb_mma(NB == 1 ? acc1[0] : acc[nb], a02[1], b02[1], a13[1], b13[1], xv.z, xv.w);
                            }
                        }
                    }
                }
#pragma unroll
                for (int h = 0; h < 2 && !I8; ++h) {
                    const uint32_t zb = cz;
                    const uint32_t zz0 = (0x4300u | ((zb >> (4 * h)) & 0xF)) * 0x00010001u;
                    const uint32_t zz1 = (0x4300u | ((zb >> (8 + 4 * h)) & 0xF)) * 0x00010001u;
                    const uint32_t wa[4] = {cw[h].x, cw[h].y, cw[h].z, cw[h].w};
                    const uint32_t wb[4] = {cw[2 + h].x, cw[2 + h].y, cw[2 + h].z, cw[2 + h].w};
                    // accumulator chains: one per n-block, and at one n-block two
                    // (nibble slots 0/1 and 2/3), so that dependent MMAs interleave
                    constexpr int NH = (NB == 1) ? 2 : 1;
                    float dl[NB][4], dh[NB][4];
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                        for (int e = 0; e < 4; ++e) dl[nb][e] = dh[nb][e] = 0.f;
                    float (&dx)[NB][4] = (NH == 2) ? dh : dl;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t l0 = awqb_pair(wa[w], zz0), l1 = awqb_pair(wb[w], zz1);
                        const uint32_t l2 = awqb_pair(wa[w] >> 4, zz0), l3 = awqb_pair(wb[w] >> 4, zz1);
                        const uint32_t h0 = awqb_pair(wa[w] >> 8, zz0), h1 = awqb_pair(wb[w] >> 8, zz1);
                        const uint32_t h2 = awqb_pair(wa[w] >> 12, zz0), h3 = awqb_pair(wb[w] >> 12, zz1);
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb) {
                            const uint4 xv = xb[(size_t)nb * 8 * L.pitch + h * 16 + 4 * w];
                            awqb_mma(dl[nb], l0, l1, l2, l3, xv.x, xv.y);
                            awqb_mma(dx[nb], h0, h1, h2, h3, xv.z, xv.w);
                        }
                    }
                    const uint32_t sg = cs[0], sg8 = cs[1];
                    const float f0 = __half2float(__ushort_as_half((unsigned short)(h ? (sg >> 16) : (sg & 0xFFFF))));
                    const float f1 = __half2float(__ushort_as_half((unsigned short)(h ? (sg8 >> 16) : (sg8 & 0xFFFF))));
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        if (NH == 2)
#pragma unroll
                            for (int e = 0; e < 4; ++e) dl[nb][e] += dh[nb][e];
                        acc[nb][0] = fmaf(f0, dl[nb][0], acc[nb][0]);
                        acc[nb][1] = fmaf(f0, dl[nb][1], acc[nb][1]);
                        acc[nb][2] = fmaf(f1, dl[nb][2], acc[nb][2]);
                        acc[nb][3] = fmaf(f1, dl[nb][3], acc[nb][3]);
                    }
                }
                // the slot is consumed (its values have fed the MMAs): refill it U super-blocks ahead
                if ((ASYNC || !EARLY) && s0 + u + U < total) load(u);
                if (ASYNC) cp_async_commit();
                if (++j == nbw) {
                    // this warp's k-slice of tile t done: store it (one k-slice, no
                    // cluster) or keep the partial for the sums after the loop
                    const int t = wt + lt2 * WT;
                    const int row0 = (t0 + t) * 16;
                    if (I8 && NB == 1) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc[0][e] += acc1[0][e];
                            acc1[0][e] = 0.f;
                        }
                    }
                    // INT8: the row scales of rows g and g + 8 (applied once, to the finished sum)
                    float sg = 1.f, sg8 = 1.f;
                    if (I8 && WK == 1 && S == 1) {
                        sg = __ldg(a.rscale + min(row0 + g, a.N - 1));
                        sg8 = __ldg(a.rscale + min(row0 + g + 8, a.N - 1));
                    }
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        const int m = 8 * nb + 2 * q;
                        if (WK == 1 && S == 1) {
                            if (m < a.M) {
                                if (row0 + g < a.N)
                                    store_out(a.y, (int64_t)m * a.N + row0 + g, acc[nb][0] * sg, a.out_f32);
                                if (row0 + g + 8 < a.N)
                                    store_out(a.y, (int64_t)m * a.N + row0 + g + 8, acc[nb][2] * sg8, a.out_f32);
                            }
                            if (m + 1 < a.M) {
                                if (row0 + g < a.N)
                                    store_out(a.y, (int64_t)(m + 1) * a.N + row0 + g, acc[nb][1] * sg, a.out_f32);
                                if (row0 + g + 8 < a.N)
                                    store_out(a.y, (int64_t)(m + 1) * a.N + row0 + g + 8, acc[nb][3] * sg8,
                                              a.out_f32);
                            }
                        } else {
                            float* rp = red + ((size_t)(t * WK + wk) * 16) * MP;
                            rp[g * MP + m] = acc[nb][0];
                            rp[g * MP + m + 1] = acc[nb][1];
                            rp[(g + 8) * MP + m] = acc[nb][2];
                            rp[(g + 8) * MP + m + 1] = acc[nb][3];
                        }
                        acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
                    }
                    j = 0;
                    ++lt2;
                }
            }
        }
    }
    if (WK == 1 && S == 1) return;
    if (nbw == 0) {
        // a warp without super-blocks contributes zero partials for its tiles
        for (int i = 0; i < ntw; ++i) {
            float* rp = red + ((size_t)((wt + i * WT) * WK + wk) * 16) * MP;
            for (int e = lane; e < 16 * MP; e += 32) rp[e] = 0.f;
        }
    }
    __syncthreads();
    if (WK > 1) {
        // sum the k-slices of every tile in slice order: store, or keep for the cluster
        for (int i = threadIdx.x; i < nt * 16 * a.M; i += W * 32) {
            const int t = i / (16 * a.M), rm = i - t * 16 * a.M;
            const int m = rm >> 4, r = rm & 15;
            float v = 0.f;
#pragma unroll
            for (int k2 = 0; k2 < WK; ++k2) v += red[((size_t)(t * WK + k2) * 16 + r) * MP + m];
            const int row = (t0 + t) * 16 + r;
            if (S == 1) {
                if (row < a.N) store_out(a.y, (int64_t)m * a.N + row, I8 ? v * __ldg(a.rscale + row) : v, a.out_f32);
            } else {
                fin[((size_t)t * 16 + r) * MP + m] = v;
            }
        }
        if (S == 1) return;
    }

    // split K: rank s sums rows [s * R / S, (s + 1) * R / S) of the CTA group's R
    // rows over the cluster's ranks, in rank order, and stores them
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int R = nt * 16;
    const int lo = rank * R / S, hi = (rank + 1) * R / S;
    const int span = hi - lo;
    for (int i = threadIdx.x; i < span * a.M; i += W * 32) {
        const int m = i / span, lr = lo + (i - m * span);
        float v = 0.f;
        for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(fin + (size_t)lr * MP + m, s);
        const int row = t0 * 16 + lr;
        if (row < a.N) store_out(a.y, (int64_t)m * a.N + row, I8 ? v * __ldg(a.rscale + row) : v, a.out_f32);
    }
    cluster.sync();
}

// ------------------------------------------------------------- tables ----
using AwqbFn = void (*)(const GemvArgs, const int);
struct AwqbEntry {
    AwqbConfig cfg;
    AwqbFn fn;
};
// WT x WK warps; MINB: CTAs per SM the instantiation is register-bounded for
// (128 registers per thread at 16 warps per SM; up to 255 with fewer);
// EARLY: refill before the compute; ASYNC: shared-memory ring (see the kernel)
#define MBW_AB(F, NB, WT, WK, U, MINB, EARLY, ASYNC) \
    { {NB, WT, WK, U, MINB, EARLY, ASYNC, F}, gemv_awq_batch_kernel<F, NB, WT, WK, U, MINB, EARLY, ASYNC> }
static const AwqbEntry kAwqb[] = {
    MBW_AB(FMT_AWQ, 1, 8, 1, 3, 2, 0, 0), MBW_AB(FMT_AWQ, 1, 8, 2, 3, 1, 0, 0), MBW_AB(FMT_AWQ, 1, 8, 2, 2, 1, 1, 0),
    MBW_AB(FMT_AWQ, 1, 8, 1, 5, 1, 1, 0), MBW_AB(FMT_AWQ, 1, 8, 2, 4, 1, 0, 1), MBW_AB(FMT_AWQ, 1, 8, 1, 6, 2, 0, 1),
    MBW_AB(FMT_AWQ, 2, 8, 2, 2, 1, 0, 0), MBW_AB(FMT_AWQ, 2, 8, 2, 2, 1, 1, 0), MBW_AB(FMT_AWQ, 2, 8, 1, 4, 1, 1, 0),
    MBW_AB(FMT_AWQ, 2, 8, 1, 6, 1, 0, 0), MBW_AB(FMT_AWQ, 2, 4, 2, 4, 1, 1, 0), MBW_AB(FMT_AWQ, 2, 8, 2, 4, 1, 0, 1),
    MBW_AB(FMT_AWQ, 2, 8, 2, 6, 1, 0, 1), MBW_AB(FMT_AWQ, 2, 8, 1, 8, 2, 0, 1), MBW_AB(FMT_AWQ, 4, 8, 1, 2, 1, 0, 0),
    MBW_AB(FMT_AWQ, 4, 8, 1, 3, 1, 1, 0), MBW_AB(FMT_AWQ, 4, 4, 2, 3, 1, 1, 0), MBW_AB(FMT_AWQ, 4, 8, 2, 4, 1, 0, 1),
    MBW_AB(FMT_AWQ, 4, 8, 1, 6, 1, 0, 1), MBW_AB(FMT_AWQ, 8, 8, 1, 2, 1, 0, 0), MBW_AB(FMT_AWQ, 8, 8, 1, 4, 1, 0, 1),
    // INT8 at batches above 8 (9 .. 64 rows per launch)
    MBW_AB(FMT_I8, 2, 8, 1, 4, 1, 0, 0), MBW_AB(FMT_I8, 2, 8, 2, 2, 1, 1, 0), MBW_AB(FMT_I8, 2, 8, 2, 4, 1, 0, 1),
    MBW_AB(FMT_I8, 2, 8, 1, 6, 2, 0, 1), MBW_AB(FMT_I8, 4, 8, 1, 3, 1, 0, 0), MBW_AB(FMT_I8, 4, 8, 2, 2, 1, 1, 0),
    MBW_AB(FMT_I8, 4, 8, 2, 4, 1, 0, 1), MBW_AB(FMT_I8, 8, 8, 1, 2, 1, 0, 0), MBW_AB(FMT_I8, 8, 8, 1, 4, 1, 0, 1),
    MBW_AB(FMT_I8, 8, 4, 2, 3, 1, 0, 1),
};
#undef MBW_AB

int awqb_num_configs() { return (int)(sizeof(kAwqb) / sizeof(kAwqb[0])); }
AwqbConfig awqb_config(int idx) { return kAwqb[idx].cfg; }

// CTA row-groups: one wave of occ CTAs per SM, or more groups (several waves)
// where the per-tile partials and tables of one wave's share do not fit the
// planner's limit (at most 227 KB over the occ CTAs of an SM).
int awqb_row_groups(const AwqbConfig& c, int64_t N, int64_t K, int split, int occ) {
    const size_t limit = std::min(kSmemFit, (size_t)227 * 1024 / occ);
    return fitted_row_groups(N, split, occ, limit, [&](int G) {
        return awqb_smem_layout(c.fmt, K, N, 8 * c.nb, c.wt * c.wk, c.wk, c.u, c.async, split, G).total;
    });
}

size_t awqb_smem_bytes(const AwqbConfig& c, int64_t N, int64_t K, int split, int occ) {
    const int G = awqb_row_groups(c, N, K, split, occ);
    return awqb_smem_layout(c.fmt, K, N, 8 * c.nb, c.wt * c.wk, c.wk, c.u, c.async, split, G).total;
}

cudaError_t launch_gemv_awq_batch(const Plan& p, const GemvArgs& a, cudaStream_t s) {
    if (p.cfg < 0 || p.cfg >= awqb_num_configs()) return cudaErrorInvalidValue;
    const AwqbEntry& e = kAwqb[p.cfg];
    const bool i8 = e.cfg.fmt == FMT_I8;
    if (a.M < 1 || a.M > 8 * e.cfg.nb || a.K % (i8 ? 128 : 256) != 0) return cudaErrorInvalidValue;
    if (i8 && !a.rscale) return cudaErrorInvalidValue;
    const uint64_t rowbytes = i8 ? (uint64_t)a.K : (uint64_t)(a.K / 2);
    if ((uint64_t)a.N * rowbytes > 0xFFFFFFFFull) return cudaErrorInvalidValue;  // 32-bit offsets
    const int G = awqb_row_groups(e.cfg, a.N, a.K, p.split, p.occ);
    const size_t smem = awqb_smem_bytes(e.cfg, a.N, a.K, p.split, p.occ);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(G * p.split), 1, 1);
    cfg.blockDim = dim3((unsigned)(e.cfg.wt * e.cfg.wk * 32), 1, 1);
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
