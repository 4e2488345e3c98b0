// device.cuh -- small sm_103a device helpers shared by the libmbw kernels:
// streaming 16/32-byte weight loads, programmatic dependent launch controls,
// warp reductions and the number formats the kernels read.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.h"

namespace mbw {

// ---------------------------------------------------------------- loads ----
// Weights are read exactly once per call: bypass L1 and mark the lines
// evict-first in L2 so they do not push out x, scales and the next kernel's
// prefetched tiles.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

struct u32x8 {
    uint32_t v[8];
};

// 32-byte load (sm_100+ 256-bit ld.global), evict-first in L2.
__device__ __forceinline__ u32x8 ld_stream32(const void* p) {
    u32x8 r;
    asm volatile(
        "ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]), "=r"(r.v[5]),
          "=r"(r.v[6]), "=r"(r.v[7])
        : "l"(p));
    return r;
}

// Read-only data reused across warps (x, scales): normal caching.
__device__ __forceinline__ uint4 ld_ro16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint16_t ld_ro_u16(const void* p) {
    uint16_t r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint8_t ld_ro_u8(const void* p) {
    uint16_t r;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(r) : "l"(p));
    return (uint8_t)r;
}

// 16-byte asynchronous global -> shared copy (L2 only), grouped per thread.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------- programmatic dependent launch ----
// The next kernel in the stream may start its prologue (weight prefetch) once
// every CTA of this grid has issued launch_dependents.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Block until the previous grid in the stream has completed and its memory is
// visible. A no-op when the kernel was launched without the PDL attribute.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Bring [base, base + bytes) into L2, the whole grid sharing the work (one
// prefetch per 128-byte line, at most a few per thread). Issued before
// pdl_wait() for the activations: L2 is the device's point of coherence, so
// if the previous grid is still writing those bytes its stores update the
// lines this brings in, and the reads after the wait hit L2 instead of DRAM.
__device__ __forceinline__ void prefetch_l2_grid_share(const void* base, size_t bytes) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    const uintptr_t a0 = b & ~uintptr_t(127);
    const size_t lines = (b + bytes - a0 + 127) / 128;
    const size_t nthr = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < lines; i += nthr) {
        uintptr_t p = a0 + i * 128;
        if (p < b) p = b;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
}

// Shared-memory ring slots of 16 rows x 128 bytes (one row super-block of a
// 16-row tile). Fragment lane L = 4g + q uses bytes 32q .. 32q+31 of rows g
// and g+8; its 16-byte chunk c (0, 1: row g; 2, 3: row g+8) sits at
// c * 512 + L * 16, so its reads are conflict-free. The copies are
// sector-complete instead: copy instruction j (0..3) moves rows 4j .. 4j+3
// whole, lane l taking 16-byte chunk l % 8 of row 4j + l / 8, so each 32-byte
// DRAM sector is requested once (two 16-byte copies per lane of its own 32
// bytes split every sector over two requests). A lane then reads chunks other
// lanes copied: __syncwarp after the copies have landed, and before a slot is
// refilled.
__device__ __forceinline__ uint32_t ring_copy_dst(int lane, int j) {
    const int r = 4 * j + (lane >> 3), cc = lane & 7;
    return (uint32_t)(((r >> 3) * 2 + (cc & 1)) * 512 + (4 * (r & 7) + (cc >> 1)) * 16);
}
// Source row (within the tile) and byte offset (within the super-block) of copy j of `lane`.
__device__ __forceinline__ int ring_copy_row(int lane, int j) { return 4 * j + (lane >> 3); }
__device__ __forceinline__ int ring_copy_byte(int lane) { return (lane & 7) * 16; }

// ------------------------------------------------------------- formats ----
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// Exact float of a 4-bit code n (0..15) minus an integer offset `zf` given as
// 2^23 + z: 2^23 + n is exact in fp32, and so is the difference n - z.
__device__ __forceinline__ float code_minus(uint32_t n, float zf) {
    return __uint_as_float(0x4B000000u | n) - zf;
}

// Symmetric INT8 codes (TileInfer, "Pushing further with cheating: INT8
// quantization") as exact bf16 pairs for the tensor core. A two's-complement
// byte b is q = (b & 0x7F) - 128 * (b >> 7), so the bf16 pair
// (0x4300 | (b & 0x7F)) = 128 + (b & 0x7F) minus (0x4300 | (b & 0x80)) = 128
// or 256 is q exactly: two LOP3 and one bf16 subtract per two codes. Bytes 0
// and 2 of v become p02, bytes 1 and 3 become p13 (the x operand is permuted
// to match).
__device__ __forceinline__ void i8_pairs(uint32_t v, uint32_t& p02, uint32_t& p13) {
    const uint32_t u = v >> 8;
    uint32_t a, b, c, d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a) : "r"(v), "r"(0x007F007Fu), "r"(0x43004300u));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(b) : "r"(v), "r"(0x00800080u), "r"(0x43004300u));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(c) : "r"(u), "r"(0x007F007Fu), "r"(0x43004300u));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(u), "r"(0x00800080u), "r"(0x43004300u));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(p02) : "r"(a), "r"(b));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(p13) : "r"(c), "r"(d));
}

// 8 bf16 x[8w..8w+7] -> pairs (0,2) (1,3) (4,6) (5,7): the order of the INT8
// pairs above (word u of the codes multiplies x pairs 2u' and 2u'+1 of its 8-x word).
__device__ __forceinline__ uint4 perm_i8(uint4 v) {
    uint4 o;
    o.x = __byte_perm(v.x, v.y, 0x5410);  // x0 | x2 << 16
    o.y = __byte_perm(v.x, v.y, 0x7632);  // x1 | x3 << 16
    o.z = __byte_perm(v.z, v.w, 0x5410);  // x4 | x6 << 16
    o.w = __byte_perm(v.z, v.w, 0x7632);  // x5 | x7 << 16
    return o;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ void store_out(void* y, int64_t idx, float v, int out_f32) {
    if (out_f32)
        static_cast<float*>(y)[idx] = v;
    else
        static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

// ------------------------------------------------------------- fusions ----
// The helpers below take FZ = 1 in the kernels instantiated for fused calls;
// with FZ = 0 every fusion branch compiles away.
//
// Which matrix and physical 16-row tile a logical tile t reads: under the
// gated epilogue logical tiles alternate between W (gate) and W2 (up).
template <int FZ>
__device__ __forceinline__ bool gated(const GemvArgs& a) { return FZ && a.glu; }
template <int FZ>
__device__ __forceinline__ const uint8_t* tile_weights(const GemvArgs& a, int t) {
    return (gated<FZ>(a) && (t & 1)) ? a.W2 : a.W;
}
template <int FZ>
__device__ __forceinline__ int tile_row0(const GemvArgs& a, int t) { return (gated<FZ>(a) ? (t >> 1) : t) * 16; }
template <int FZ>
__device__ __forceinline__ const uint16_t* tile_scales(const GemvArgs& a, int t) {
    return (gated<FZ>(a) && (t & 1)) ? a.scales2 : a.scales;
}
template <int FZ>
__device__ __forceinline__ const float* tile_rscale(const GemvArgs& a, int t) {
    return (gated<FZ>(a) && (t & 1)) ? a.rscale2 : a.rscale;
}

// The CTA's logical tile range [t0, t0 + nt) of row-group `cg` of `G`: whole
// output tiles, and whole gate/up pairs under the gated epilogue.
template <int FZ>
__device__ __forceinline__ void cta_tile_range(const GemvArgs& a, int G, int cg, int& t0, int& nt) {
    const int T = (a.N + 15) / 16;
    const int f = gated<FZ>(a) ? 2 : 1;
    const int p0 = (int)(((long long)T * cg) / G);
    const int p1 = (int)(((long long)T * (cg + 1)) / G);
    t0 = p0 * f;
    nt = (p1 - p0) * f;
}

// RMSNorm prologue (llm-rs vs vLLM, "norms folded into the projections"):
// 1 / sqrt(mean_k x[m][k]^2 + eps) for every batch row m, summed by the whole
// CTA in a fixed order (deterministic). `scratch` needs (warps + 1) * M
// floats; the factor of row m is left in scratch[warps * M + m]. Contains two
// __syncthreads: every thread of the CTA must call it.
__device__ __forceinline__ void norm_factors(const GemvArgs& a, float* scratch, int nthreads) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = nthreads >> 5;
    const int words = a.K / 8;
    for (int m = 0; m < a.M; ++m) {
        float s = 0.f;
        for (int i = threadIdx.x; i < words; i += nthreads) {
            const uint4 v = ld_ro16(a.x + (size_t)m * a.K + (size_t)i * 8);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = bf16lo_to_f32(w[j]), hi = bf16hi_to_f32(w[j]);
                s = fmaf(lo, lo, s);
                s = fmaf(hi, hi, s);
            }
        }
        s = warp_sum(s);
        if (lane == 0) scratch[m * nw + warp] = s;
    }
    __syncthreads();
    if (threadIdx.x < a.M) {
        float t = 0.f;
        for (int w = 0; w < nw; ++w) t += scratch[threadIdx.x * nw + w];
        scratch[nw * a.M + threadIdx.x] = 1.0f / sqrtf(t / (float)a.K + a.norm_eps);
    }
    __syncthreads();
}

// x word (8 bf16 at k .. k+7 of batch row m) -> bf16(x * r * g), rounded to nearest even.
__device__ __forceinline__ uint4 norm_word(uint4 v, float r, const uint16_t* g) {
    const uint4 gv = ld_ro16(g);
    const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float lo = bf16lo_to_f32(xw[j]) * r * bf16lo_to_f32(gw[j]);
        const float hi = bf16hi_to_f32(xw[j]) * r * bf16hi_to_f32(gw[j]);
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float silu_f32(float v) { return v / (1.0f + expf(-v)); }

// Store output (m, row) of a finished row sum (INT8 scales already applied):
// v is the sum of W's row, v2 that of W2's row under the gated epilogue;
// SwiGLU (yalm sec. 3.3, TileInfer: SwiGLU in the GEMV epilogue), then the
// residual add (yalm: fused matmul + add_residuals), then the bf16 store.
template <int FZ>
__device__ __forceinline__ void store_fused(const GemvArgs& a, int m, int row, float v, float v2) {
    if (gated<FZ>(a)) v = silu_f32(v) * v2;
    const int64_t idx = (int64_t)m * a.N + row;
    if (FZ && a.residual) v += bf16lo_to_f32(a.residual[idx]);
    store_out(a.y, idx, v, a.out_f32);
}

}  // namespace mbw
