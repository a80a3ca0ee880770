// S5 and S6 as grouped GEMV on CUDA cores (every decode batch).
//
// S5 (k_gateup): one CTA per (active expert, 16-feature block).  For each pair
// routed to the expert (expert-grouped order), the pair's activation row is
// expanded once into shared memory as signed int8 (value * 2) plus the fp32
// block scales; 16 half-warps then each stream one gate row and one up row
// of the expert with 16-byte loads and form exact integer block sums
// (dp4a), combined in fp32.  h = silu(g) * u for the 16 features is one NVFP4
// block, quantised by 16 lanes with the static tensor scale s_h and written
// to row r of hq/hs.
//
// S6 (k_down): one CTA per (token, 16 output rows).  For each slot j in order
// the pair's h_hat row is expanded into shared memory, 16 half-warps each
// stream one row of the expert's down matrix, and the weighted result is
// accumulated in slot order (deterministic), then y (fp32) and the optional
// bf16 residual sum are written.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRowsPerCta = 16;   // half-warps per CTA
constexpr int kThreads = 256;

// Expand one NVFP4 row (K elements) into shared memory:
//   sx8[seg*8 + i]  int8x4 words of value*2 (elements 4i .. 4i+3 of the segment)
//   ssc[b]          fp32 block scales
__device__ __forceinline__ void stage_row(const uint8_t* __restrict__ codes,
                                          const uint8_t* __restrict__ scales, int K,
                                          uint32_t* sx8, float* ssc) {
    const int nseg = K / 32;
    for (int seg = threadIdx.x; seg < nseg; seg += blockDim.x) {
        const uint4 c = __ldg(reinterpret_cast<const uint4*>(codes) + seg);
        XSeg xs;
        load_xseg(c, xs);
        uint4* dst = reinterpret_cast<uint4*>(sx8 + seg * 8);
        dst[0] = make_uint4(xs.v[0], xs.v[1], xs.v[2], xs.v[3]);
        dst[1] = make_uint4(xs.v[4], xs.v[5], xs.v[6], xs.v[7]);
    }
    for (int b = threadIdx.x; b < K / 16; b += blockDim.x) ssc[b] = e4m3_to_f32(scales[b]);
}

__device__ __forceinline__ void read_xseg(const uint32_t* sx8, int seg, XSeg& x) {
    const uint4* src = reinterpret_cast<const uint4*>(sx8 + seg * 8);
    const uint4 a = src[0], b = src[1];
    x.v[0] = a.x; x.v[1] = a.y; x.v[2] = a.z; x.v[3] = a.w;
    x.v[4] = b.x; x.v[5] = b.y; x.v[6] = b.z; x.v[7] = b.w;
}

__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// E2M1 nibble of one value (RNE on |v|, saturating, sign copied).
__device__ __forceinline__ uint32_t e2m1_one(float v) {
    float t[8] = {v, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    return e2m1x8_rn_satfinite(t) & 0xFu;
}

__global__ void __launch_bounds__(kThreads) k_gateup(
    int H, int I, int k, const uint8_t* __restrict__ g_codes, const uint8_t* __restrict__ g_scales,
    const float* __restrict__ g_ts, const uint8_t* __restrict__ u_codes,
    const uint8_t* __restrict__ u_scales, const float* __restrict__ u_ts, float h_scale,
    const uint32_t* __restrict__ scal, const float* __restrict__ sx,
    const int32_t* __restrict__ active, const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm,
    const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xsc, uint8_t* __restrict__ hq,
    uint8_t* __restrict__ hs) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* sx8 = reinterpret_cast<uint32_t*>(smem);                 // H/32 * 8 words
    float* ssc = reinterpret_cast<float*>(smem + (size_t)H);           // H/16 floats
    __shared__ float hbuf[kRowsPerCta];

    if (blockIdx.y >= scal[kScalActive]) return;
    const int e = active[blockIdx.y];
    const int r0 = offsets[e], r1 = offsets[e + 1];
    const int f0 = blockIdx.x * kRowsPerCta;
    const int rs = threadIdx.x >> 4;          // half-warp = feature slot
    const int hl = threadIdx.x & 15;
    const int f = f0 + rs;
    const size_t row_bytes = (size_t)H / 2;
    const uint8_t* gc = g_codes + ((size_t)e * I + f) * row_bytes;
    const uint8_t* uc = u_codes + ((size_t)e * I + f) * row_bytes;
    const uint8_t* gs = g_scales + ((size_t)e * I + f) * (H / 16);
    const uint8_t* us = u_scales + ((size_t)e * I + f) * (H / 16);
    const float x_s = *sx;
    const float gscale = __fmul_rn(__fmul_rn(g_ts[e], x_s), 0.25f);
    const float uscale = __fmul_rn(__fmul_rn(u_ts[e], x_s), 0.25f);
    const int nseg = H / 32;

    for (int r = r0; r < r1; ++r) {
        const int t = perm[r] / k;
        __syncthreads();  // previous pair's staging and hbuf are consumed
        stage_row(xq + (size_t)t * (H / 2), xsc + (size_t)t * (H / 16), H, sx8, ssc);
        __syncthreads();
        float ga = 0.0f, ua = 0.0f;
#pragma unroll 4
        for (int seg = hl; seg < nseg; seg += 16) {
            const uint4 wg = __ldg(reinterpret_cast<const uint4*>(gc) + seg);
            const uint4 wu = __ldg(reinterpret_cast<const uint4*>(uc) + seg);
            const uint32_t sg = __ldg(reinterpret_cast<const uint16_t*>(gs) + seg);
            const uint32_t su = __ldg(reinterpret_cast<const uint16_t*>(us) + seg);
            XSeg x;
            read_xseg(sx8, seg, x);
            const float2 xsc2 = make_float2(ssc[2 * seg], ssc[2 * seg + 1]);
            ga += dot_seg32(wg, sg, x, xsc2);
            ua += dot_seg32(wu, su, x, xsc2);
        }
        ga = half_warp_sum(ga);
        ua = half_warp_sum(ua);
        if (hl == 0) {
            const float g = __fmul_rn(ga, gscale);
            const float u = __fmul_rn(ua, uscale);
            hbuf[rs] = __fmul_rn(silu(g), u);
        }
        __syncthreads();
        if (threadIdx.x < 16) {
            // Q on the 16-feature block with the static scale s_h
            const float v = hbuf[threadIdx.x];
            float a = fabsf(v);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0x0000ffffu, a, o, 16));
            const float q = __fdiv_rn(a, __fmul_rn(6.0f, h_scale));
            const uint32_t S = e4m3_rn_satfinite(q);
            uint32_t c = 0;
            if (S != 0) c = e2m1_one(__fdiv_rn(v, __fmul_rn(e4m3_to_f32(S), h_scale)));
            const uint32_t hi = __shfl_down_sync(0x0000ffffu, c, 1, 16);
            const size_t hrow = (size_t)r * (I / 2) + f0 / 2;
            if ((threadIdx.x & 1) == 0) hq[hrow + threadIdx.x / 2] = (uint8_t)(c | (hi << 4));
            if (threadIdx.x == 0) hs[(size_t)r * (I / 16) + f0 / 16] = (uint8_t)S;
        }
    }
}

__global__ void __launch_bounds__(kThreads) k_down(
    int H, int I, int k, const uint8_t* __restrict__ d_codes, const uint8_t* __restrict__ d_scales,
    const float* __restrict__ d_ts, float h_scale, const int32_t* __restrict__ idx,
    const float* __restrict__ wts, const int32_t* __restrict__ inv,
    const uint8_t* __restrict__ hq, const uint8_t* __restrict__ hsc,
    const uint16_t* __restrict__ residual, float* __restrict__ y, uint16_t* __restrict__ x_next) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* sx8 = reinterpret_cast<uint32_t*>(smem);                 // I/32 * 8 words
    float* ssc = reinterpret_cast<float*>(smem + (size_t)I);           // I/16 floats

    const int t = blockIdx.x;
    const int rs = threadIdx.x >> 4, hl = threadIdx.x & 15;
    const int row = blockIdx.y * kRowsPerCta + rs;
    const int nseg = I / 32;
    const size_t row_bytes = (size_t)I / 2;
    float yacc = 0.0f;
    for (int j = 0; j < k; ++j) {
        const int p = t * k + j;
        const int e = idx[p];
        const int r = inv[p];
        if (e < 0) continue;   // dropped by the route-tail skip (the same for the whole CTA)
        __syncthreads();
        stage_row(hq + (size_t)r * row_bytes, hsc + (size_t)r * (I / 16), I, sx8, ssc);
        __syncthreads();
        const uint8_t* dc = d_codes + ((size_t)e * H + row) * row_bytes;
        const uint8_t* ds = d_scales + ((size_t)e * H + row) * (I / 16);
        float acc = 0.0f;
#pragma unroll 4
        for (int seg = hl; seg < nseg; seg += 16) {
            const uint4 wd = __ldg(reinterpret_cast<const uint4*>(dc) + seg);
            const uint32_t sd = __ldg(reinterpret_cast<const uint16_t*>(ds) + seg);
            XSeg x;
            read_xseg(sx8, seg, x);
            acc += dot_seg32(wd, sd, x, make_float2(ssc[2 * seg], ssc[2 * seg + 1]));
        }
        acc = half_warp_sum(acc);
        const float o = __fmul_rn(acc, __fmul_rn(__fmul_rn(d_ts[e], h_scale), 0.25f));
        yacc = fmaf(wts[p], o, yacc);
    }
    if (hl == 0) {
        const size_t off = (size_t)t * H + row;
        y[off] = yacc;
        if (x_next) x_next[off] = f32_to_bf16_rn(bf16_to_f32(residual[off]) + yacc);
    }
}

}  // namespace

cudaError_t launch_gateup(const Shape& s, int T, const ExpertWeights& gate,
                          const ExpertWeights& up, float h_scale, const Workspace& ws,
                          cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int P = T * s.k;
    const int ny = P < s.E ? P : s.E;
    const size_t smem = (size_t)s.H + (size_t)s.H / 16 * sizeof(float);
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(k_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(s.I / kRowsPerCta, ny);
    k_gateup<<<grid, kThreads, smem, st>>>(s.H, s.I, s.k, gate.codes, gate.scales, gate.ts,
                                           up.codes, up.scales, up.ts, h_scale, ws.scal, ws.sx, ws.active,
                                           ws.offsets, ws.perm, ws.xq, ws.xs, ws.hq, ws.hs);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_down(const Shape& s, int T, const ExpertWeights& down, float h_scale,
                        const Workspace& ws, const uint16_t* residual, float* y,
                        uint16_t* x_next, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const size_t smem = (size_t)s.I + (size_t)s.I / 16 * sizeof(float);
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(k_down, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(T, s.H / kRowsPerCta);
    k_down<<<grid, kThreads, smem, st>>>(s.H, s.I, s.k, down.codes, down.scales, down.ts, h_scale,
                                         ws.idx, ws.w, ws.inv, ws.hq, ws.hs, residual, y, x_next);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
