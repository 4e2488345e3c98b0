// gen_inputs.cu -- device evaluation of the seeded synthetic-input generators
// (libmbw_inputs.so; not part of libmbw.so and holds no GEMV arithmetic).
//
// Same definition as memory_bound_weight_gb300/inputs.py: element i of a
// stream is the (i+1)-th output of a splitmix64 sequence started at `key`
// (Steele, Lea & Flood, OOPSLA 2014; constants of Vigna's splitmix64.c):
//   z = key + (i + 1) * 0x9E3779B97F4A7C15
//   z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
//   z = (z ^ (z >> 27)) * 0x94D049BB133111EB
//   h = z ^ (z >> 31)
// The host computes `key`; these kernels fill multi-GB tensors in place so
// that the oracle can regenerate any sampled row on the host bit for bit.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t splitmix_at(uint64_t key, uint64_t i) {
    uint64_t z = key + (i + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// bf16 from a 65,536-entry quantile table, 4 values per hash (low 16 bits first).
__global__ void gen_table16(uint16_t* __restrict__ out, int64_t n, int64_t start, uint64_t key,
                            const uint16_t* __restrict__ table) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n; j += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = start + j;
        const uint64_t h = splitmix_at(key, (uint64_t)(e >> 2));
        out[j] = table[(h >> (16 * (e & 3))) & 0xFFFF];
    }
}

// uniform bytes, 8 per hash, little-endian.
__global__ void gen_bytes(uint8_t* __restrict__ out, int64_t n, int64_t start, uint64_t key) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n; j += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = start + j;
        const uint64_t h = splitmix_at(key, (uint64_t)(e >> 3));
        out[j] = (uint8_t)(h >> (8 * (e & 7)));
    }
}

// fp16 ~ U(0.001, 0.01): fp16_rne(((fp32(u) * 2^-24) * 0.009f) + 0.001f), u = top 24 bits.
__global__ void gen_scales(uint16_t* __restrict__ out, int64_t n, int64_t start, uint64_t key) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n; j += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t h = splitmix_at(key, (uint64_t)(start + j));
        const float u = __uint2float_rn((unsigned)(h >> 40));
        float s = __fmul_rn(u, 5.9604644775390625e-08f);  // 2^-24
        s = __fmul_rn(s, 0.009f);
        s = __fadd_rn(s, 0.001f);
        out[j] = __half_as_ushort(__float2half_rn(s));
    }
}

// int8 from a 65,536-entry code table, 4 values per hash (low 16 bits first).
__global__ void gen_table8(int8_t* __restrict__ out, int64_t n, int64_t start, uint64_t key,
                           const int8_t* __restrict__ table) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n; j += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = start + j;
        const uint64_t h = splitmix_at(key, (uint64_t)(e >> 2));
        out[j] = table[(h >> (16 * (e & 3))) & 0xFFFF];
    }
}

// fp32 ~ U(lo, lo + span): ((fp32(u) * 2^-24) * span) + lo, u = top 24 bits.
__global__ void gen_f32_uniform(float* __restrict__ out, int64_t n, int64_t start, uint64_t key, float lo,
                                float span) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n; j += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t h = splitmix_at(key, (uint64_t)(start + j));
        const float u = __uint2float_rn((unsigned)(h >> 40));
        float s = __fmul_rn(u, 5.9604644775390625e-08f);  // 2^-24
        s = __fmul_rn(s, span);
        out[j] = __fadd_rn(s, lo);
    }
}

int grid_for(int64_t n) {
    int64_t b = (n + 255) / 256;
    if (b > 152 * 32) b = 152 * 32;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace

extern "C" int mbw_gen_bf16_table(void* out, int64_t n, int64_t start, uint64_t key, const void* table,
                                  cudaStream_t s) {
    if (n <= 0) return 0;
    gen_table16<<<grid_for(n), 256, 0, s>>>((uint16_t*)out, n, start, key, (const uint16_t*)table);
    return (int)cudaGetLastError();
}

extern "C" int mbw_gen_bytes(void* out, int64_t n, int64_t start, uint64_t key, cudaStream_t s) {
    if (n <= 0) return 0;
    gen_bytes<<<grid_for(n), 256, 0, s>>>((uint8_t*)out, n, start, key);
    return (int)cudaGetLastError();
}

extern "C" int mbw_gen_f16_scales(void* out, int64_t n, int64_t start, uint64_t key, cudaStream_t s) {
    if (n <= 0) return 0;
    gen_scales<<<grid_for(n), 256, 0, s>>>((uint16_t*)out, n, start, key);
    return (int)cudaGetLastError();
}

extern "C" int mbw_gen_i8_table(void* out, int64_t n, int64_t start, uint64_t key, const void* table,
                                cudaStream_t s) {
    if (n <= 0) return 0;
    gen_table8<<<grid_for(n), 256, 0, s>>>((int8_t*)out, n, start, key, (const int8_t*)table);
    return (int)cudaGetLastError();
}

extern "C" int mbw_gen_f32_uniform(void* out, int64_t n, int64_t start, uint64_t key, float lo, float span,
                                   cudaStream_t s) {
    if (n <= 0) return 0;
    gen_f32_uniform<<<grid_for(n), 256, 0, s>>>((float*)out, n, start, key, lo, span);
    return (int)cudaGetLastError();
}
