// S1 + S2: router logits, top-k and the renormalised softmax weights.
//
// Logits: one warp per expert row of Wr (fp32 [E][H], read once per token
// tile with 16-byte loads), a tile of up to 8 tokens of bf16 x staged in
// shared memory; fp32 accumulation, fixed reduction order.
// Top-k: one warp per token; k rounds of a warp arg-max on (logit desc,
// expert index asc), so exact ties go to the lower index; weights
// w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0) over the k picks.  With the
// route-tail skip (keep < k) a pick of rank >= keep whose expert is not marked
// resident is dropped: expert -1, weight 0, the others renormalised over the
// kept picks.

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kMaxDevices = 64;
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

// Order-preserving unsigned key of a float (larger float, larger key; -0 and
// +0 both map to +0's key, so they tie like the floats do).
__device__ __forceinline__ uint32_t f32_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_f32(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr int kTopkWarps = 8;   // warps (tokens) per block of k_topk

// One warp per token; lane l holds the logits of experts l + 32 j (j < PL,
// PL * 32 >= E) as keys (0: no expert).  The order is value descending, ties
// to the lower index.
//
// Threshold pass: tau = the k-th largest of the 32 lane maxima (a bitonic
// sort of the maxima across the warp).  The k lanes with the largest maxima
// hold k keys >= tau, so every top-k key is >= tau; the keys >= tau (about k
// of them for continuous logits) are gathered in shared memory, one per lane,
// and each one's rank is the number of candidates ahead of it (larger key, or
// equal key and lower index) -- 32 shuffles.  With more than 32 candidates
// (many equal logits) the round pass below runs instead.
//
// Round pass: each lane keeps its own best (largest key, lowest j) and a mask
// of its taken slots; each of the k rounds takes the warp's largest key and,
// among the lanes holding it, the lowest expert index (two warp reductions);
// only the winning lane rescans its slots.
template <int PL>
__global__ void __launch_bounds__(kTopkWarps * 32) k_topk(const float* __restrict__ logits, int T, int E, int k,
                                                          int keep, const uint8_t* __restrict__ resident,
                                                          int32_t* __restrict__ idx, float* __restrict__ w) {
    __shared__ uint2 cand[kTopkWarps][32];   // (key, expert) of the candidates, then of the picks by rank
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int wib = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= T) return;
    const float* row = logits + (size_t)warp * E;
    uint32_t key[PL];
#pragma unroll
    for (int j = 0; j < PL; ++j) {
        const int e = lane + 32 * j;
        key[j] = e < E ? f32_key(row[e]) : 0u;
    }
    int my_e = 0;
    uint32_t my_k = 0;
    // ---- threshold pass
    uint32_t lm = 0;
#pragma unroll
    for (int j = 0; j < PL; ++j) lm = max(lm, key[j]);
    uint32_t v = lm;   // bitonic sort of the lane maxima, descending in lane order
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool desc = (lane & size) == 0;
            const bool keep_max = ((lane & stride) == 0) == desc;
            v = keep_max ? max(v, o) : min(v, o);
        }
    }
    const uint32_t tau = __shfl_sync(0xffffffffu, v, k - 1);
    int nc = 0;
#pragma unroll
    for (int j = 0; j < PL; ++j) nc += key[j] >= tau ? 1 : 0;
    int incl = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const int n_cand = __shfl_sync(0xffffffffu, incl, 31);
    if (n_cand <= 32) {
        int pos = incl - nc;
#pragma unroll
        for (int j = 0; j < PL; ++j) {
            if (key[j] >= tau) cand[wib][pos++] = make_uint2(key[j], (uint32_t)(lane + 32 * j));
        }
        __syncwarp();
        const uint2 c = lane < n_cand ? cand[wib][lane] : make_uint2(0u, 0xFFFFFFFFu);
        int rank = 0;
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const uint32_t tk = __shfl_sync(0xffffffffu, c.x, t);
            const uint32_t te = __shfl_sync(0xffffffffu, c.y, t);
            rank += (tk > c.x || (tk == c.x && te < c.y)) ? 1 : 0;
        }
        __syncwarp();
        if (lane < n_cand && rank < k) cand[wib][rank] = c;
        __syncwarp();
        if (lane < k) {
            const uint2 pick = cand[wib][lane];
            my_k = pick.x;
            my_e = (int)pick.y;
        }
    } else {
    // ---- round pass
    uint32_t bk = 0;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < PL; ++j) {
        if (key[j] > bk) {
            bk = key[j];
            bj = j;
        }
    }
    uint32_t taken = 0;
    for (int r = 0; r < k; ++r) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t e = __reduce_min_sync(0xffffffffu, bk == m ? (uint32_t)(lane + 32 * bj) : 0xFFFFFFFFu);
        if (lane == r) {
            my_e = (int)e;
            my_k = m;
        }
        if ((int)(e & 31u) == lane) {
            taken |= 1u << (e >> 5);
            bk = 0;
            bj = 0;
#pragma unroll
            for (int j = 0; j < PL; ++j) {
                if (!((taken >> j) & 1u) && key[j] > bk) {
                    bk = key[j];
                    bj = j;
                }
            }
        }
    }
    }
    const float my_v = key_f32(my_k);
    const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
    const bool kept = lane < k && (lane < keep || (resident && resident[my_e] != 0));
    const float z = kept ? expf(my_v - v0) : 0.0f;
    const float sum = warp_sum(z);
    if (lane < k) {
        idx[(size_t)warp * k + lane] = kept ? my_e : -1;
        w[(size_t)warp * k + lane] = kept ? __fdiv_rn(z, sum) : 0.0f;
    }
}

}  // namespace

cudaError_t launch_router(const uint16_t* x, const float* Wr, const float* bias, int T,
                          const Shape& s, float* logits, int32_t* idx, float* w, cudaStream_t st,
                          int keep, const uint8_t* resident) {
    if (T == 0) return cudaSuccess;
    const size_t smem = (size_t)kTokTile * s.H * sizeof(uint16_t);
    // the x tile needs more than the default 48 KB above hidden 3072: raise the
    // limit once per device (the attribute is per device), under a lock
    static std::mutex mu;
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t ae = cudaGetDevice(&dev);
    if (ae != cudaSuccess) return ae;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            ae = cudaFuncSetAttribute(k_router_logits, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      128 * 1024);
            if (ae != cudaSuccess) return ae;
            attr_set[dev] = true;
        }
    }
    dim3 grid((s.E + kWarps - 1) / kWarps, (T + kTokTile - 1) / kTokTile);
    k_router_logits<<<grid, kWarps * 32, smem, st>>>(x, Wr, bias, T, s.H, s.E, logits);
    count_launches(1);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_topk(logits, T, s, idx, w, st, keep, resident);
}

cudaError_t launch_topk(const float* logits, int T, const Shape& s, int32_t* idx, float* w,
                        cudaStream_t st, int keep, const uint8_t* resident) {
    if (keep < 1 || keep > s.k) keep = s.k;
    if (T == 0) return cudaSuccess;
    const int warps_per_block = kTopkWarps;
    const unsigned grid = (unsigned)((T + warps_per_block - 1) / warps_per_block);
    const int per_lane = (s.E + 31) / 32;
    if (per_lane <= 1)
        k_topk<1><<<grid, warps_per_block * 32, 0, st>>>(logits, T, s.E, s.k, keep, resident, idx, w);
    else if (per_lane <= 2)
        k_topk<2><<<grid, warps_per_block * 32, 0, st>>>(logits, T, s.E, s.k, keep, resident, idx, w);
    else if (per_lane <= 4)
        k_topk<4><<<grid, warps_per_block * 32, 0, st>>>(logits, T, s.E, s.k, keep, resident, idx, w);
    else if (per_lane <= 8)
        k_topk<8><<<grid, warps_per_block * 32, 0, st>>>(logits, T, s.E, s.k, keep, resident, idx, w);
    else if (per_lane <= 16)
        k_topk<16><<<grid, warps_per_block * 32, 0, st>>>(logits, T, s.E, s.k, keep, resident, idx, w);
    else
        k_topk<32><<<grid, warps_per_block * 32, 0, st>>>(logits, T, s.E, s.k, keep, resident, idx, w);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
