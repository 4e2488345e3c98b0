// gemv_simt.cu -- CUDA-core weight-streaming GEMV for sm_103a.
//
// y[m][i] = sum_k x[m][k] * w(i, k) for BF16, INT4 group-64 and AWQ-style INT4
// group-128 weights; one call reads every weight once (llm-rs vs vLLM, sec. 2:
// "the job is streaming weights").
//
// Mapping (prior art: the pages' warp-per-row matvec -- yalm sec. 3.1, llm-rs
// "Going down a level: SIMT kernels" -- and tinyinfer's R rows per warp, where
// each lane issues R independent 16-byte loads per step):
//   * a warp owns R consecutive rows; its 32 lanes read consecutive 16-byte
//     chunks of each row, so one warp-wide load covers 512 contiguous bytes of
//     a row; every lane keeps R x U chunks in flight (register double buffer);
//   * the CTA's WARPS warps own WARPS x R rows; x (the CTA's k-slice) is staged
//     once in shared memory as fp32, laid out plane-major so that lane-strided
//     reads are bank-conflict free, and shared by all rows of the CTA;
//   * short, wide matrices split K over a thread-block cluster of S CTAs; each
//     CTA reduces its rows over its k-slice and rank 0 sums the S partials in
//     rank order through distributed shared memory (deterministic, no global
//     scratch, no spin waits: barrier.cluster co-schedules the cluster);
//   * programmatic dependent launch: the kernel lets the next kernel launch at
//     once, issues its first batch of weight (and scale) loads, and only then
//     waits for the previous grid before it reads x.
//
// INT4 unpack is exact: a code n becomes the float 2^23 + n by OR-ing it into
// the mantissa of 2^23, and subtracting 2^23 + z (z = 8, or the AWQ zero point)
// leaves n - z exactly. The group scale multiplies the group's fp32 partial sum,
// so no dequantized weight is ever rounded.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>

#include "device.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace mbw {

template <int FMT>
struct Traits;
template <>
struct Traits<FMT_BF16> {
    static constexpr int CW = 8;  // weights per 16-byte chunk
};
template <>
struct Traits<FMT_G64> {
    static constexpr int CW = 32;
};
template <>
struct Traits<FMT_AWQ> {
    static constexpr int CW = 32;
};

template <int FMT, int WARPS, int R, int U, int MB>
__global__ void __launch_bounds__(WARPS * 32, 16 / WARPS)
    gemv_simt_kernel(const GemvArgs a, const int S) {
    constexpr int CW = Traits<FMT>::CW;
    constexpr int PL = CW / 4;  // float4 planes per chunk
    extern __shared__ float4 smem[];

    pdl_launch_dependents();

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int rowblock = blockIdx.x / S;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c0 = rank * a.split_chunks;
    const int c1 = min(a.chunks, c0 + a.split_chunks);
    const int nc = max(c1 - c0, 0);
    const int iters = (nc + 32 * U - 1) / (32 * U);

    const int row_base = rowblock * (WARPS * R) + warp * R;
    const uint8_t* wrow[R];
    int rowc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        rowc[r] = min(row_base + r, a.N - 1);
        wrow[r] = a.W + (size_t)rowc[r] * (size_t)a.chunks * 16;
    }

    uint4 cur[R][U];
    uint16_t scur[R][U];
    uint8_t zcur[R][U];

    auto load = [&](uint4 (&buf)[R][U], uint16_t (&sb)[R][U], uint8_t (&zb)[R][U], int it) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + it * 32 * U + u * 32 + lane;
            const bool ok = c < c1;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                buf[r][u] = ok ? ld_stream16(wrow[r] + (size_t)c * 16) : make_uint4(0, 0, 0, 0);
                if (FMT == FMT_G64) {
                    sb[r][u] = ok ? ld_ro_u16(a.scales + (size_t)rowc[r] * a.groups + (c >> 1)) : 0;
                } else if (FMT == FMT_AWQ) {
                    const int g = c >> 2;
                    sb[r][u] = ok ? ld_ro_u16(a.scales + (size_t)rowc[r] * a.groups + g) : 0;
                    zb[r][u] = ok ? ld_ro_u8(a.zeros + (size_t)rowc[r] * a.zstride + (g >> 1)) : 0;
                }
            }
        }
    };

    if (iters > 0) load(cur, scur, zcur, 0);

    // x is produced by the previous kernel in the stream: wait for it only now.
    prefetch_l2_grid_share(a.x, (size_t)a.M * a.K * 2);
    pdl_wait();

    // Stage this CTA's k-slice of x as fp32, plane-major:
    // smem[(m * PL + p) * nc + lc] = x[m][(c0 + lc) * CW + 4p .. +4].
    {
        const int per_m = nc * CW / 8;  // 16-byte pieces of x per activation row
        for (int i = threadIdx.x; i < MB * per_m; i += WARPS * 32) {
            const int m = i / per_m;
            const int j = i - m * per_m;
            const int kl = j * 8;
            const int lc = kl / CW;
            const int p0 = (kl % CW) / 4;
            const uint4 v = (m < a.M) ? ld_ro16(a.x + (size_t)m * a.K + (size_t)c0 * CW + kl)
                                      : make_uint4(0, 0, 0, 0);
            smem[(m * PL + p0) * nc + lc] =
                make_float4(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x), bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
            smem[(m * PL + p0 + 1) * nc + lc] =
                make_float4(bf16lo_to_f32(v.z), bf16hi_to_f32(v.z), bf16lo_to_f32(v.w), bf16hi_to_f32(v.w));
        }
    }
    __syncthreads();

    float acc[R][MB];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[r][m] = 0.f;

    for (int it = 0; it < iters; ++it) {
        uint4 nxt[R][U];
        uint16_t snxt[R][U];
        uint8_t znxt[R][U];
        if (it + 1 < iters) load(nxt, snxt, znxt, it + 1);

#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + it * 32 * U + u * 32 + lane;
            if (c < c1) {
                const int lc = c - c0;
                if (FMT == FMT_BF16) {
#pragma unroll
                    for (int m = 0; m < MB; ++m) {
                        const float4 xa = smem[(m * PL + 0) * nc + lc];
                        const float4 xb = smem[(m * PL + 1) * nc + lc];
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint4 w = cur[r][u];
                            float s = acc[r][m];
                            s = fmaf(bf16lo_to_f32(w.x), xa.x, s);
                            s = fmaf(bf16hi_to_f32(w.x), xa.y, s);
                            s = fmaf(bf16lo_to_f32(w.y), xa.z, s);
                            s = fmaf(bf16hi_to_f32(w.y), xa.w, s);
                            s = fmaf(bf16lo_to_f32(w.z), xb.x, s);
                            s = fmaf(bf16hi_to_f32(w.z), xb.y, s);
                            s = fmaf(bf16lo_to_f32(w.w), xb.z, s);
                            s = fmaf(bf16hi_to_f32(w.w), xb.w, s);
                            acc[r][m] = s;
                        }
                    }
                } else {
                    float zf[R], sc[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        sc[r] = f16_bits_to_f32(scur[r][u]);
                        if (FMT == FMT_G64) {
                            zf[r] = 8388616.0f;  // 2^23 + 8
                        } else {
                            const int g = c >> 2;
                            const uint32_t z = (g & 1) ? (zcur[r][u] >> 4) : (zcur[r][u] & 0xF);
                            zf[r] = __uint_as_float(0x4B000000u | z);  // 2^23 + z
                        }
                    }
#pragma unroll
                    for (int m = 0; m < MB; ++m) {
                        float part[R];
#pragma unroll
                        for (int r = 0; r < R; ++r) part[r] = 0.f;
#pragma unroll
                        for (int p = 0; p < PL; ++p) {
                            const float4 xv = smem[(m * PL + p) * nc + lc];
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const uint4 w4 = cur[r][u];
                                const uint32_t w = (p < 2) ? w4.x : (p < 4) ? w4.y : (p < 6) ? w4.z : w4.w;
                                const int sh = (p & 1) * 16;  // nibbles 0-3 or 4-7 of the word
                                float t = part[r];
                                t = fmaf(code_minus((w >> (sh + 0)) & 0xF, zf[r]), xv.x, t);
                                t = fmaf(code_minus((w >> (sh + 4)) & 0xF, zf[r]), xv.y, t);
                                t = fmaf(code_minus((w >> (sh + 8)) & 0xF, zf[r]), xv.z, t);
                                t = fmaf(code_minus((w >> (sh + 12)) & 0xF, zf[r]), xv.w, t);
                                part[r] = t;
                            }
                        }
#pragma unroll
                        for (int r = 0; r < R; ++r) acc[r][m] = fmaf(sc[r], part[r], acc[r][m]);
                    }
                }
            }
        }
        if (it + 1 < iters) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    cur[r][u] = nxt[r][u];
                    scur[r][u] = snxt[r][u];
                    zcur[r][u] = znxt[r][u];
                }
        }
    }

#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[r][m] = warp_sum(acc[r][m]);

    if (S == 1) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MB; ++m)
                if (lane == ((r * MB + m) & 31) && row_base + r < a.N && m < a.M)
                    store_out(a.y, (int64_t)m * a.N + row_base + r, acc[r][m], a.out_f32);
        return;
    }

    // Split-K: partials of this CTA's rows -> shared memory, then rank 0 sums
    // the S partials in rank order through distributed shared memory.
    const size_t xs_floats = (size_t)MB * PL * a.split_chunks * 4;
    float* red = reinterpret_cast<float*>(smem) + xs_floats;
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MB; ++m) red[(warp * R + r) * MB + m] = acc[r][m];
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (rank == 0) {
        for (int t = threadIdx.x; t < WARPS * R * MB; t += WARPS * 32) {
            float v = 0.f;
            for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(red + t, s);
            const int row = rowblock * (WARPS * R) + t / MB;
            const int m = t % MB;
            if (row < a.N && m < a.M) store_out(a.y, (int64_t)m * a.N + row, v, a.out_f32);
        }
    }
    cluster.sync();
}

// BF16 at batch 1 with 32-byte lane loads: a lane reads 16 weights of a row per
// load (ld.global v8), so one warp instruction covers 1 KB of the row, twice
// the run of the 16-byte kernel above; the matrix is then read as long
// contiguous runs, which the DRAM serves at nearly the rate of a linear sweep
// (measured on 18944 x 3584 BF16: 512-byte runs per row cost ~2.5 us more per
// launch than a grid-stride read, 1 KB runs ~0.5 us). Same row ownership, x
// staging (fp32, plane-major, 4 planes per chunk), double buffer, reduction and
// split-K cluster sum as above; chunk = 32 bytes, K % 16 == 0.
template <int WARPS, int R, int U>
__global__ void __launch_bounds__(WARPS * 32, 16 / WARPS) gemv_simt_bf16w_kernel(const GemvArgs a, const int S) {
    constexpr int PL = 4;  // float4 planes per 32-byte chunk (16 weights)
    extern __shared__ float4 smem[];

    pdl_launch_dependents();

    const int rank = (S > 1) ? (int)cg::this_cluster().block_rank() : 0;
    const int rowblock = blockIdx.x / S;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunks = a.chunks / 2;  // 32-byte chunks per row (a.chunks counts 16-byte ones)
    const int split = (chunks + S - 1) / S;
    const int c0 = rank * split;
    const int c1 = min(chunks, c0 + split);
    const int nc = max(c1 - c0, 0);
    const int iters = (nc + 32 * U - 1) / (32 * U);

    const int row_base = rowblock * (WARPS * R) + warp * R;
    const uint8_t* wrow[R];
#pragma unroll
    for (int r = 0; r < R; ++r) wrow[r] = a.W + (size_t)min(row_base + r, a.N - 1) * (size_t)chunks * 32;

    u32x8 cur[R][U];
    auto load = [&](u32x8 (&buf)[R][U], int it) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + it * 32 * U + u * 32 + lane;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (c < c1) {
                    buf[r][u] = ld_stream32(wrow[r] + (size_t)c * 32);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) buf[r][u].v[e] = 0;
                }
            }
        }
    };
    if (iters > 0) load(cur, 0);

    prefetch_l2_grid_share(a.x, (size_t)a.K * 2);
    pdl_wait();

    // x of this CTA's k-slice as fp32: smem[p * nc + lc] = x[(c0 + lc) * 16 + 4p .. +4]
    for (int i = threadIdx.x; i < nc * 2; i += WARPS * 32) {
        const int lc = i >> 1, p0 = (i & 1) * 2;
        const uint4 v = ld_ro16(a.x + (size_t)(c0 + lc) * 16 + (size_t)p0 * 4);
        smem[p0 * nc + lc] = make_float4(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x), bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
        smem[(p0 + 1) * nc + lc] =
            make_float4(bf16lo_to_f32(v.z), bf16hi_to_f32(v.z), bf16lo_to_f32(v.w), bf16hi_to_f32(v.w));
    }
    __syncthreads();

    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;

    for (int it = 0; it < iters; ++it) {
        u32x8 nxt[R][U];
        if (it + 1 < iters) load(nxt, it + 1);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + it * 32 * U + u * 32 + lane;
            if (c < c1) {
                const int lc = c - c0;
#pragma unroll
                for (int p = 0; p < PL; ++p) {
                    const float4 xv = smem[p * nc + lc];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t w0 = cur[r][u].v[2 * p], w1 = cur[r][u].v[2 * p + 1];
                        float t = acc[r];
                        t = fmaf(bf16lo_to_f32(w0), xv.x, t);
                        t = fmaf(bf16hi_to_f32(w0), xv.y, t);
                        t = fmaf(bf16lo_to_f32(w1), xv.z, t);
                        t = fmaf(bf16hi_to_f32(w1), xv.w, t);
                        acc[r] = t;
                    }
                }
            }
        }
        if (it + 1 < iters) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int u = 0; u < U; ++u) cur[r][u] = nxt[r][u];
        }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = warp_sum(acc[r]);

    if (S == 1) {
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (lane == (r & 31) && row_base + r < a.N) store_out(a.y, row_base + r, acc[r], a.out_f32);
        return;
    }

    // split K: partials of this CTA's rows -> shared memory, then rank 0 sums the
    // S partials in rank order through distributed shared memory
    float* red = reinterpret_cast<float*>(smem) + (size_t)PL * split * 4;
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) red[warp * R + r] = acc[r];
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (rank == 0) {
        for (int t = threadIdx.x; t < WARPS * R; t += WARPS * 32) {
            float v = 0.f;
            for (int s = 0; s < S; ++s) v += *cluster.map_shared_rank(red + t, s);
            const int row = rowblock * (WARPS * R) + t;
            if (row < a.N) store_out(a.y, row, v, a.out_f32);
        }
    }
    cluster.sync();
}

// Persistent form of the 32-byte kernel (batch 1, no split): a grid of
// `occ` CTAs per SM, each staging the whole of x once; warp w of the grid takes
// the R-row groups w, w + TW, w + 2 TW, ... (TW = warps in the grid), and its
// register double buffer runs across group boundaries, so a warp's next rows
// are in flight while it finishes the current ones. A non-persistent grid
// instead restarts cold in every CTA of its second wave (x staged again, one
// chunk per row in flight until the staging ends).
template <int WARPS, int R, int U>
__global__ void __launch_bounds__(WARPS * 32, 16 / WARPS) gemv_simt_bf16p_kernel(const GemvArgs a, const int) {
    constexpr int PL = 4;
    extern __shared__ float4 smem[];

    pdl_launch_dependents();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunks = a.chunks / 2;
    const int iters = (chunks + 32 * U - 1) / (32 * U);
    const int ngroups = (a.N + R - 1) / R;
    const int TW = gridDim.x * WARPS;
    int g = blockIdx.x * WARPS + warp;
    int it = 0;

    auto load = [&](u32x8 (&buf)[R][U], int grp, int itn) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* wr = a.W + (size_t)min(grp * R + r, a.N - 1) * (size_t)chunks * 32;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = itn * 32 * U + u * 32 + lane;
                if (c < chunks) {
                    buf[r][u] = ld_stream32(wr + (size_t)c * 32);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) buf[r][u].v[e] = 0;
                }
            }
        }
    };
    u32x8 cur[R][U];
    if (g < ngroups) load(cur, g, 0);

    prefetch_l2_grid_share(a.x, (size_t)a.K * 2);
    pdl_wait();

    // the whole of x as fp32: smem[p * chunks + c] = x[c * 16 + 4p .. +4]
    for (int i = threadIdx.x; i < chunks * 2; i += WARPS * 32) {
        const int c = i >> 1, p0 = (i & 1) * 2;
        const uint4 v = ld_ro16(a.x + (size_t)c * 16 + (size_t)p0 * 4);
        smem[p0 * chunks + c] = make_float4(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x), bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
        smem[(p0 + 1) * chunks + c] =
            make_float4(bf16lo_to_f32(v.z), bf16hi_to_f32(v.z), bf16lo_to_f32(v.w), bf16hi_to_f32(v.w));
    }
    __syncthreads();

    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;

    while (g < ngroups) {
        int ng = g, nit = it + 1;
        if (nit == iters) {
            nit = 0;
            ng = g + TW;
        }
        u32x8 nxt[R][U];
        if (ng < ngroups) load(nxt, ng, nit);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = it * 32 * U + u * 32 + lane;
            if (c < chunks) {
#pragma unroll
                for (int p = 0; p < PL; ++p) {
                    const float4 xv = smem[p * chunks + c];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t w0 = cur[r][u].v[2 * p], w1 = cur[r][u].v[2 * p + 1];
                        float t = acc[r];
                        t = fmaf(bf16lo_to_f32(w0), xv.x, t);
                        t = fmaf(bf16hi_to_f32(w0), xv.y, t);
                        t = fmaf(bf16lo_to_f32(w1), xv.z, t);
                        t = fmaf(bf16hi_to_f32(w1), xv.w, t);
                        acc[r] = t;
                    }
                }
            }
        }
        if (nit == 0) {  // the group's last chunks: reduce over the warp and store its rows
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float v = warp_sum(acc[r]);
                if (lane == (r & 31) && g * R + r < a.N) store_out(a.y, g * R + r, v, a.out_f32);
                acc[r] = 0.f;
            }
        }
        if (ng < ngroups) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int u = 0; u < U; ++u) cur[r][u] = nxt[r][u];
        }
        g = ng;
        it = nit;
    }
}

// ------------------------------------------------------------- tables ----
using KernFn = void (*)(const GemvArgs, const int);
struct Entry {
    SimtConfig cfg;
    KernFn fn;
};
#define MBW_E(F, W, R, U, MB) \
    { {W, R, U, MB, 16}, gemv_simt_kernel<F, W, R, U, MB> }
#define MBW_EW(W, R, U) \
    { {W, R, U, 1, 32}, gemv_simt_bf16w_kernel<W, R, U> }
#define MBW_EP(W, R, U) \
    { {W, R, U, 1, 32, 1}, gemv_simt_bf16p_kernel<W, R, U> }

static const Entry kBf16[] = {
    MBW_E(FMT_BF16, 4, 1, 4, 1), MBW_E(FMT_BF16, 4, 2, 4, 1), MBW_E(FMT_BF16, 8, 1, 8, 1),
    MBW_E(FMT_BF16, 4, 4, 2, 1), MBW_E(FMT_BF16, 8, 2, 2, 1), MBW_E(FMT_BF16, 8, 1, 4, 1),
    MBW_E(FMT_BF16, 4, 2, 2, 2), MBW_E(FMT_BF16, 4, 2, 2, 4), MBW_E(FMT_BF16, 4, 1, 2, 8),
    MBW_EW(4, 2, 2), MBW_EW(4, 4, 1), MBW_EW(4, 1, 4), MBW_EW(8, 2, 2), MBW_EW(8, 1, 4),
    MBW_EW(8, 1, 2),  MBW_EP(4, 4, 1), MBW_EP(4, 2, 2), MBW_EP(4, 2, 1), MBW_EP(8, 2, 1), MBW_EP(8, 1, 2),
    MBW_EP(4, 1, 2),
};
static const Entry kG64[] = {
    MBW_E(FMT_G64, 4, 1, 2, 1), MBW_E(FMT_G64, 4, 2, 2, 1), MBW_E(FMT_G64, 4, 4, 1, 1),
    MBW_E(FMT_G64, 8, 2, 2, 1), MBW_E(FMT_G64, 8, 1, 4, 1), MBW_E(FMT_G64, 8, 2, 1, 1),
};
static const Entry kAwq[] = {
    MBW_E(FMT_AWQ, 4, 1, 2, 1), MBW_E(FMT_AWQ, 4, 2, 2, 1), MBW_E(FMT_AWQ, 4, 4, 1, 1),
    MBW_E(FMT_AWQ, 8, 2, 2, 1), MBW_E(FMT_AWQ, 8, 1, 4, 1), MBW_E(FMT_AWQ, 4, 2, 1, 2),
    MBW_E(FMT_AWQ, 4, 2, 1, 4), MBW_E(FMT_AWQ, 4, 1, 1, 8),
};
#undef MBW_E
#undef MBW_EW
#undef MBW_EP

static const Entry* table(int fmt, int* n) {
    switch (fmt) {
        case FMT_BF16:
            *n = (int)(sizeof(kBf16) / sizeof(kBf16[0]));
            return kBf16;
        case FMT_G64:
            *n = (int)(sizeof(kG64) / sizeof(kG64[0]));
            return kG64;
        case FMT_AWQ:
            *n = (int)(sizeof(kAwq) / sizeof(kAwq[0]));
            return kAwq;
        default:
            *n = 0;
            return nullptr;
    }
}

int simt_num_configs(int fmt) {
    int n;
    table(fmt, &n);
    return n;
}

SimtConfig simt_config(int fmt, int idx) {
    int n;
    const Entry* t = table(fmt, &n);
    return t[idx].cfg;
}

size_t simt_smem_bytes(int fmt, const SimtConfig& c, const GemvArgs& a, int split) {
    if (c.persist) return (size_t)(a.chunks / 2) * 16 * sizeof(float);  // the whole of x, fp32
    if (c.cb == 32) {  // BF16, 32-byte chunks of 16 weights: the x slice of the widest rank, then the partials
        const size_t split32 = (size_t)(a.chunks / 2 + split - 1) / split;
        return split32 * 16 * sizeof(float) + ((split > 1) ? (size_t)c.warps * c.r * sizeof(float) : 0);
    }
    const int cw = (fmt == FMT_BF16) ? 8 : 32;
    const size_t xs = (size_t)c.mb * a.split_chunks * cw * sizeof(float);
    const size_t red = (split > 1) ? (size_t)c.warps * c.r * c.mb * sizeof(float) : 0;
    return xs + red;
}

cudaError_t launch_gemv_simt(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s) {
    int n;
    const Entry* t = table(fmt, &n);
    if (p.cfg < 0 || p.cfg >= n) return cudaErrorInvalidValue;
    const Entry& e = t[p.cfg];
    const int rows_per_cta = e.cfg.warps * e.cfg.r;
    int rowblocks = (a.N + rows_per_cta - 1) / rows_per_cta;
    if (e.cfg.persist) {
        if (p.split != 1 || p.occ < 1) return cudaErrorInvalidValue;
        rowblocks = std::min(rowblocks, device_sm_count() * p.occ);
    }
    const size_t smem = simt_smem_bytes(fmt, e.cfg, a, p.split);

    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rowblocks * p.split), 1, 1);
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

// -------------------------------------------------------------- dequant ----
// out[i][k] = (q - z) * s in fp32; exact (4-bit integer times an fp16 value).
__global__ void dequant_int4_kernel(const uint8_t* __restrict__ Wq, const uint16_t* __restrict__ scales,
                                    const uint8_t* __restrict__ zeros, float* __restrict__ out, int64_t N,
                                    int64_t K, int group, int awq) {
    const int64_t nbytes = N * (K / 2);
    const int64_t G = K / group;
    const int64_t zstride = (G + 1) / 2;
    for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nbytes;
         b += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = b / (K / 2);
        const int64_t k = (b - i * (K / 2)) * 2;
        const int64_t g = k / group;
        const float s = f16_bits_to_f32(scales[i * G + g]);
        uint32_t z = 8;
        if (awq) {
            const uint8_t zb = zeros[i * zstride + g / 2];
            z = (g & 1) ? (zb >> 4) : (zb & 0xF);
        }
        const float zf = __uint_as_float(0x4B000000u | z);
        const uint8_t byte = Wq[b];
        out[i * K + k] = code_minus(byte & 0xF, zf) * s;
        out[i * K + k + 1] = code_minus(byte >> 4, zf) * s;
    }
}

cudaError_t launch_dequant(int fmt, const uint8_t* Wq, const uint16_t* scales, const uint8_t* zeros, float* out,
                           int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nbytes = N * (K / 2);
    const int threads = 256;
    int64_t blocks = (nbytes + threads - 1) / threads;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    count_launch();
    dequant_int4_kernel<<<(unsigned)blocks, threads, 0, s>>>(Wq, scales, zeros, out, N, K,
                                                              fmt == FMT_G64 ? 64 : 128, fmt == FMT_AWQ);
    return cudaGetLastError();
}

}  // namespace mbw
