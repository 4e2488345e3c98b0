// quantize.cu -- load-time quantizer of BF16 weights to symmetric INT8 with
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

}  // namespace

cudaError_t launch_quantize_int8_pc(const uint16_t* W, int8_t* Wq, float* scales, int64_t N, int64_t K,
                                    cudaStream_t s) {
    if (N <= 0) return cudaSuccess;
    const int64_t grid = N < (int64_t)device_sm_count() * 8 ? N : (int64_t)device_sm_count() * 8;
    count_launch();
    quantize_int8_pc_kernel<<<(unsigned)grid, kQuantThreads, 0, s>>>(W, Wq, scales, N, K);
    return cudaGetLastError();
}

}  // namespace mbw
