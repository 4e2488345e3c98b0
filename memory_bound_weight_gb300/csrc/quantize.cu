// quantize.cu -- load-time weight transforms.
//
// Quantizer of BF16 weights to symmetric INT8 with
// one fp32 scale per output channel (TileInfer, "Pushing further with
// cheating: INT8 quantization": codes in [-127, 127], scale = max|w| / 127,
// every entry rounded to the nearest multiple of the scale).
//
// Decisions in fp32, as stored: s = max|w| / 127 with IEEE division, the
// quotient w / s with IEEE division, rounded to the nearest integer with ties
// to even (rintf); an all-zero row gets s = 0 and codes 0. Weights must be
// finite. One CTA per row (grid-stride over rows), two passes over the row:
// the max, then the codes (the second pass reads the row from L1/L2).
#include <cuda_bf16.h>

#include "device.cuh"
#include "internal.h"

namespace mbw {

namespace {

constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads) quantize_int8_pc_kernel(const uint16_t* __restrict__ W,
                                                                         int8_t* __restrict__ Q,
                                                                         float* __restrict__ S, int64_t N,
                                                                         int64_t K) {
    __shared__ float wmax[kQuantThreads / 32];
    for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
        const uint16_t* w = W + row * K;
        float m = 0.f;
        for (int64_t k = threadIdx.x; k < K; k += kQuantThreads) m = fmaxf(m, fabsf(bf16lo_to_f32(w[k])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
        __syncthreads();
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < kQuantThreads / 32; ++i) amax = fmaxf(amax, wmax[i]);
        const float s = __fdiv_rn(amax, 127.0f);
        if (threadIdx.x == 0) S[row] = s;
        int8_t* q = Q + row * K;
        for (int64_t k = threadIdx.x; k < K; k += kQuantThreads) {
            float r = 0.f;
            if (s != 0.f) r = fminf(fmaxf(rintf(__fdiv_rn(bf16lo_to_f32(w[k]), s)), -127.f), 127.f);
            q[k] = (int8_t)(int)r;
        }
        __syncthreads();  // wmax is rewritten for the next row
    }
}

// Load-time INT4 repack (llm-rs vs vLLM, sec. 6 on Marlin: 4-bit weights
// reordered once at load time so the unpack hands the multiply its operands
// directly). In each 32-bit word of 8 codes (k = 8w + j in nibble slot j) the
// even-k nibbles move to slots 0-3 and the odd-k nibbles to slots 4-7, each in
// k order; the unpack's masks (bits 0-3 with 16-19, then 4-7 with 20-23, ...)
// then give the pairs (k0, k1), (k2, k3), ... in order.
__device__ __forceinline__ uint32_t repack_word(uint32_t v) {
    uint32_t e = v & 0x0F0F0F0Fu, o = (v >> 4) & 0x0F0F0F0Fu;  // even / odd k, one per byte
    e = (e | (e >> 4)) & 0x00FF00FFu;
    o = (o | (o >> 4)) & 0x00FF00FFu;
    e = (e | (e >> 8)) & 0x0000FFFFu;
    o = (o | (o >> 8)) & 0x0000FFFFu;
    return e | (o << 16);
}

// One word per thread and step; in place is fine (each word is read before
// the same thread writes it).
__global__ void repack_int4_kernel(const uint32_t* in, uint32_t* out, int64_t nwords) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nwords;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = repack_word(in[i]);
}

// Launched after each weight writer above, without the programmatic-
// serialization attribute, so it starts only once the writer has completed
// and its stores are visible. The library's GEMVs read weights before their
// griddepcontrol.wait and may start early relative to the kernel in front of
// them; with this kernel in between, that kernel wrote nothing they read.
__global__ void weights_written_fence_kernel() {}

cudaError_t launch_weights_fence(cudaStream_t s) {
    count_launch();
    weights_written_fence_kernel<<<1, 32, 0, s>>>();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_repack_int4(const uint8_t* Wq, uint8_t* Wr, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nwords = N * (K / 8);
    if (nwords <= 0) return cudaSuccess;
    const int64_t blocks = (nwords + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    count_launch();
    repack_int4_kernel<<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, s>>>(
        reinterpret_cast<const uint32_t*>(Wq), reinterpret_cast<uint32_t*>(Wr), nwords);
    const cudaError_t e = cudaGetLastError();
    return e != cudaSuccess ? e : launch_weights_fence(s);
}

cudaError_t launch_quantize_int8_pc(const uint16_t* W, int8_t* Wq, float* scales, int64_t N, int64_t K,
                                    cudaStream_t s) {
    if (N <= 0) return cudaSuccess;
    const int64_t grid = N < (int64_t)device_sm_count() * 8 ? N : (int64_t)device_sm_count() * 8;
    count_launch();
    quantize_int8_pc_kernel<<<(unsigned)grid, kQuantThreads, 0, s>>>(W, Wq, scales, N, K);
    const cudaError_t e = cudaGetLastError();
    return e != cudaSuccess ? e : launch_weights_fence(s);
}

}  // namespace mbw
