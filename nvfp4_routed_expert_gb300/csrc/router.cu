// S1 + S2: router logits, top-k and the renormalised softmax weights.
//
// Logits: one warp per expert row of Wr (fp32 [E][H], read once per token
// tile with 16-byte loads), a tile of up to 8 tokens of bf16 x staged in
// shared memory; fp32 accumulation, fixed reduction order.
// Top-k: one warp per token; k rounds of a warp arg-max on (logit desc,
// expert index asc), so exact ties go to the lower index; weights
// w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0) over the k picks.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kTokTile = 8;
constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32) k_router_logits(
    const uint16_t* __restrict__ x, const float* __restrict__ Wr, const float* __restrict__ bias,
    int T, int H, int E, float* __restrict__ logits) {
    extern __shared__ uint32_t xs[];  // [kTokTile][H/2] bf16 pairs
    const int t0 = blockIdx.y * kTokTile;
    const int nt = min(kTokTile, T - t0);
    const int hw = H / 2;
    for (int i = threadIdx.x; i < kTokTile * hw; i += blockDim.x) {
        const int t = i / hw;
        xs[i] = t < nt ? reinterpret_cast<const uint32_t*>(x + (size_t)(t0 + t) * H)[i % hw] : 0u;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kWarps + warp;
    if (e >= E) return;
    const float4* wr = reinterpret_cast<const float4*>(Wr + (size_t)e * H);
    float acc[kTokTile];
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) acc[t] = 0.0f;
#pragma unroll 4
    for (int c = lane; c < H / 4; c += 32) {
        const float4 w = __ldg(wr + c);
#pragma unroll
        for (int t = 0; t < kTokTile; ++t) {
            const uint2 p = *reinterpret_cast<const uint2*>(&xs[t * hw + 2 * c]);
            acc[t] = fmaf(w.x, bf16_to_f32(p.x & 0xFFFFu), acc[t]);
            acc[t] = fmaf(w.y, bf16_to_f32(p.x >> 16), acc[t]);
            acc[t] = fmaf(w.z, bf16_to_f32(p.y & 0xFFFFu), acc[t]);
            acc[t] = fmaf(w.w, bf16_to_f32(p.y >> 16), acc[t]);
        }
    }
    const float b = bias ? bias[e] : 0.0f;
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0 && t < nt) logits[(size_t)(t0 + t) * E + e] = v + b;
    }
}

// One warp per token.  E <= 1024 so every lane holds at most 32 logits.
__global__ void k_topk(const float* __restrict__ logits, int T, int E, int k,
                       int32_t* __restrict__ idx, float* __restrict__ w) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= T) return;
    const float* row = logits + (size_t)warp * E;
    const int per_lane = (E + 31) / 32;
    float v[32];
    uint32_t taken = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int e = lane + 32 * j;
        if (j < per_lane && e < E) {
            v[j] = row[e];
        } else {
            v[j] = -FLT_MAX;
            taken |= 1u << j;
        }
    }
    int my_e = 0;
    float my_v = 0.0f;
    for (int r = 0; r < k; ++r) {
        float bv = -FLT_MAX;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (!((taken >> j) & 1u) && (v[j] > bv || be == 0x7FFFFFFF)) {
                bv = v[j];
                be = lane + 32 * j;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == r) {
            my_e = be;
            my_v = bv;
        }
    }
    const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
    const float z = lane < k ? expf(my_v - v0) : 0.0f;
    const float sum = warp_sum(z);
    if (lane < k) {
        idx[(size_t)warp * k + lane] = my_e;
        w[(size_t)warp * k + lane] = __fdiv_rn(z, sum);
    }
}

}  // namespace

cudaError_t launch_router(const uint16_t* x, const float* Wr, const float* bias, int T,
                          const Shape& s, float* logits, int32_t* idx, float* w, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const size_t smem = (size_t)kTokTile * s.H * sizeof(uint16_t);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(k_router_logits, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             128 * 1024);
        attr_set = true;
    }
    dim3 grid((s.E + kWarps - 1) / kWarps, (T + kTokTile - 1) / kTokTile);
    k_router_logits<<<grid, kWarps * 32, smem, st>>>(x, Wr, bias, T, s.H, s.E, logits);
    count_launches(1);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_topk(logits, T, s, idx, w, st);
}

cudaError_t launch_topk(const float* logits, int T, const Shape& s, int32_t* idx, float* w,
                        cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int warps_per_block = 8;
    k_topk<<<(T + warps_per_block - 1) / warps_per_block, warps_per_block * 32, 0, st>>>(
        logits, T, s.E, s.k, idx, w);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
