// S3 and weight packing: the NVFP4 block quantiser Q over whole tensors.
//
// Activations (bf16 x [T][H]) get one dynamic tensor scale per call,
// s = max|x| / 2688; weight matrices get one tensor scale each.  Two passes:
// a max-magnitude reduction (atomicMax on the fp32 bit pattern, which orders
// like the value for non-negative floats), then one thread per 16-element
// block running quant_block16.  Both passes stream the tensor with 16-byte
// loads; the second writes 8 code bytes and 1 scale byte per block.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16x2_absmax(uint32_t v) {
    return fmaxf(fabsf(bf16_to_f32(v & 0xFFFFu)), fabsf(bf16_to_f32(v >> 16)));
}

__device__ __forceinline__ void block_atomic_max(float v, uint32_t* target) {
    __shared__ float red[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        v = threadIdx.x < kThreads / 32 ? red[threadIdx.x] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (threadIdx.x == 0 && v > 0.0f) atomicMax(target, __float_as_uint(v));
    }
}

__global__ void __launch_bounds__(kThreads) k_amax_bf16(const uint4* __restrict__ x, size_t n16,
                                                        uint32_t* __restrict__ amax) {
    float m = 0.0f;
    for (size_t i = blockIdx.x * (size_t)kThreads + threadIdx.x; i < n16;
         i += (size_t)gridDim.x * kThreads) {
        const uint4 v = __ldg(x + i);
        m = fmaxf(m, fmaxf(fmaxf(bf16x2_absmax(v.x), bf16x2_absmax(v.y)),
                           fmaxf(bf16x2_absmax(v.z), bf16x2_absmax(v.w))));
    }
    block_atomic_max(m, amax);
}

__global__ void __launch_bounds__(kThreads) k_quant_bf16(const uint4* __restrict__ x, size_t nblocks,
                                                         const uint32_t* __restrict__ amax,
                                                         uint2* __restrict__ codes,
                                                         uint8_t* __restrict__ scales,
                                                         float* __restrict__ sx_out) {
    const float s = tensor_scale_from_amax_bits(*amax);
    const size_t b = blockIdx.x * (size_t)kThreads + threadIdx.x;
    if (b == 0) *sx_out = s;
    if (b >= nblocks) return;
    const uint4 v0 = __ldg(x + 2 * b), v1 = __ldg(x + 2 * b + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[kBlock];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = bf16_to_f32(w[i] & 0xFFFFu);
        f[2 * i + 1] = bf16_to_f32(w[i] >> 16);
    }
    uint2 c;
    const uint32_t S = quant_block16(f, s, c);
    codes[b] = c;
    scales[b] = (uint8_t)S;
}

__global__ void __launch_bounds__(kThreads) k_amax_f32_mats(const float4* __restrict__ w,
                                                            size_t per_mat4,
                                                            uint32_t* __restrict__ amax) {
    const int m = blockIdx.y;
    const float4* base = w + (size_t)m * per_mat4;
    float a = 0.0f;
    for (size_t i = blockIdx.x * (size_t)kThreads + threadIdx.x; i < per_mat4;
         i += (size_t)gridDim.x * kThreads) {
        const float4 v = __ldg(base + i);
        a = fmaxf(a, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    block_atomic_max(a, amax + m);
}

__global__ void __launch_bounds__(kThreads) k_quant_f32_mats(const float4* __restrict__ w,
                                                             size_t blocks_per_mat, int M,
                                                             const uint32_t* __restrict__ amax,
                                                             uint2* __restrict__ codes,
                                                             uint8_t* __restrict__ scales) {
    const size_t b = blockIdx.x * (size_t)kThreads + threadIdx.x;
    if (b >= blocks_per_mat * (size_t)M) return;
    const size_t m = b / blocks_per_mat;
    const float s = tensor_scale_from_amax_bits(amax[m]);
    float f[kBlock];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 v = __ldg(w + 4 * b + i);
        f[4 * i] = v.x;
        f[4 * i + 1] = v.y;
        f[4 * i + 2] = v.z;
        f[4 * i + 3] = v.w;
    }
    uint2 c;
    const uint32_t S = quant_block16(f, s, c);
    codes[b] = c;
    scales[b] = (uint8_t)S;
}

__global__ void k_finish_tensor_scales(uint32_t* __restrict__ amax_then_scale, int M) {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m < M) {
        const float s = tensor_scale_from_amax_bits(amax_then_scale[m]);
        amax_then_scale[m] = __float_as_uint(s);
    }
}

int reduction_grid(size_t work16) {
    size_t g = (work16 + kThreads - 1) / kThreads;
    return (int)(g < 4 * 152 ? (g == 0 ? 1 : g) : 4 * 152);
}

}  // namespace

cudaError_t launch_quant_act(const uint16_t* x, int T, int H, uint8_t* codes, uint8_t* scales,
                             float* sx, uint32_t* amax, cudaStream_t st) {
    const size_t n = (size_t)T * H;
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    if (n > 0) {
        k_amax_bf16<<<reduction_grid(n / 8), kThreads, 0, st>>>(
            reinterpret_cast<const uint4*>(x), n / 8, amax);
        count_launches(1);
    }
    return launch_quant_act_given_amax(x, T, H, codes, scales, sx, amax, st);
}

cudaError_t launch_quant_act_given_amax(const uint16_t* x, int T, int H, uint8_t* codes,
                                        uint8_t* scales, float* sx, const uint32_t* amax,
                                        cudaStream_t st) {
    const size_t nblocks = (size_t)T * H / kBlock;
    const size_t grid = nblocks == 0 ? 1 : (nblocks + kThreads - 1) / kThreads;
    k_quant_bf16<<<(unsigned)grid, kThreads, 0, st>>>(reinterpret_cast<const uint4*>(x), nblocks,
                                                      amax, reinterpret_cast<uint2*>(codes),
                                                      scales, sx);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_quant_weights(const float* w, int M, int rows, int cols, uint8_t* codes,
                                 uint8_t* scales, float* ts, cudaStream_t st) {
    uint32_t* amax = reinterpret_cast<uint32_t*>(ts);
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t) * (size_t)M, st);
    if (e != cudaSuccess) return e;
    const size_t per_mat = (size_t)rows * cols;
    dim3 g1(reduction_grid(per_mat / 4 / 4) > 64 ? 64 : reduction_grid(per_mat / 4 / 4), M);
    k_amax_f32_mats<<<g1, kThreads, 0, st>>>(reinterpret_cast<const float4*>(w), per_mat / 4,
                                              amax);
    const size_t blocks_per_mat = per_mat / kBlock;
    const size_t total = blocks_per_mat * (size_t)M;
    k_quant_f32_mats<<<(unsigned)((total + kThreads - 1) / kThreads), kThreads, 0, st>>>(
        reinterpret_cast<const float4*>(w), blocks_per_mat, M, amax,
        reinterpret_cast<uint2*>(codes), scales);
    k_finish_tensor_scales<<<(M + 255) / 256, 256, 0, st>>>(amax, M);
    count_launches(3);
    return cudaGetLastError();
}

}  // namespace moe
