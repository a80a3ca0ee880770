// Decode path: one persistent, cooperatively launched kernel that runs S1..S6
// for up to 8 tokens through a whole stack of layers (one layer for
// moe_forward, up to 64 for moe_stack_forward).
//
// Decode is bound by memory bandwidth (capy-flash v0.7.1, "Why it matters"),
// and at one token a layer moves only ~22 MB, so the kernel keeps every SM
// resident for the whole stack and separates the phases of a layer with grid
// barriers instead of kernel launches:
//
//   R  router logits of the CTA's experts (rows of Wr, prefetched to L2 one
//      layer ahead)                                              -> barrier
//   T  in every CTA, redundantly: top-k + softmax of the <= 8 tokens, the
//      expert-grouped permutation of the <= 128 pairs, and the NVFP4 form of
//      x expanded to int8 in shared memory; then L2 prefetch of this CTA's
//      share of the layer's down rows and the next layer's router rows
//   G  gate/up items (routed expert x 16 features), each item's 32 weight
//      rows streamed HBM -> shared memory by bulk copies through an mbarrier
//      ring; SwiGLU and requantisation of h; h written to global -> barrier
//   D  down items (16 output rows x routed expert) through the same ring;
//      per-pair outputs combined in slot order, residual added  -> barrier
//
// All grid barriers and mbarrier waits are bounded (see sync.cuh).
#include <cfloat>

#include "common.cuh"
#include "decode.h"
#include "kernels.h"
#include "sync.cuh"

namespace moe {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;   // 16: one feature / output row per warp
constexpr int kRows = 16;
constexpr int kMaxSlots = 16;
constexpr int kMaxCand = 2048;          // top-k candidates of all tokens

constexpr int kBarD = kMaxSlots;          // first mbarrier of the down ring
constexpr int kBarX = 2 * kMaxSlots;      // x staging

struct Smem {
    uint64_t bar[2 * kMaxSlots + 1];   // gate/up ring, down ring, x staging
    int32_t idx[kDecodeMaxPairs];  // [t][j]
    float w[kDecodeMaxPairs];
    int32_t perm[kDecodeMaxPairs];
    int32_t inv[kDecodeMaxPairs];
    int32_t pe[kDecodeMaxPairs];   // expert of each expert-grouped position
    int32_t act_e[kDecodeMaxPairs];
    int32_t act_off[kDecodeMaxPairs + 1];
    int32_t n_act;
    uint32_t flag;
    float sx;
    uint32_t pending;              // bit s: ring slot s has a copy in flight
    uint32_t redu[kWarps];
    float red[kWarps][kDecodeMaxTokens];
    float hbuf[kMaxSlots][kDecodeMaxTokens][kRows];
    float obuf[kDecodeMaxPairs][kRows];
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Phase stamp (layer 0 only) by thread 0 of the first and the last CTA.
constexpr int kStamps = 16;
__device__ __forceinline__ void stamp(const DecodeParams& p, int l, int slot) {
    if (p.phase_ns && l == 0 && threadIdx.x == 0) {
        if (blockIdx.x == 0) p.phase_ns[slot] = globaltimer_ns();
        if (blockIdx.x == gridDim.x - 1) p.phase_ns[kStamps + slot] = globaltimer_ns();
    }
}

__device__ __forceinline__ uint32_t e2m1_one(float v) {
    float t[8] = {v, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    return e2m1x8_rn_satfinite(t) & 0xFu;
}

// fp32 -> uint32 key with the same order (finite values); 0 is below every key
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void read_seg8(const uint32_t* src, XSeg& x) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
    const uint4 a = s[0], b = s[1];
    x.v[0] = a.x; x.v[1] = a.y; x.v[2] = a.z; x.v[3] = a.w;
    x.v[4] = b.x; x.v[5] = b.y; x.v[6] = b.z; x.v[7] = b.w;
}

// Wait for every ring slot that still has a copy in flight (bounded), so that
// no bulk copy lands in shared memory after the CTA has exited.
__device__ void drain(Smem& sm, uint32_t phase_bits, uint32_t* err) {
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2 * kMaxSlots; ++s) {
            if ((sm.pending >> s) & 1u) {
                if (!mbar_wait(&sm.bar[s], (phase_bits >> s) & 1u)) atomicOr(err, kDevErrTimeout);
            }
        }
        sm.pending = 0;
    }
    __syncthreads();
}

// Wait for ring slots [s0, s0 + n); false (after draining) on timeout.
__device__ __forceinline__ bool wait_slots(Smem& sm, int s0, int n, uint32_t& phase_bits,
                                           uint32_t* err) {
    for (int i = 0; i < n; ++i) {
        const int s = s0 + i;
        if (!mbar_wait(&sm.bar[s], (phase_bits >> s) & 1u)) {
            atomicOr(err, kDevErrTimeout);
            drain(sm, phase_bits, err);
            return false;
        }
        phase_bits ^= 1u << s;
    }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1) k_decode(const __grid_constant__ DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    uint8_t* region_a = smem_raw + p.region_a_off;   // x_hat / h_hat as int8 + fp32 block scales
    uint8_t* region_b = smem_raw + p.region_b_off;   // x staging + top-k candidates, then the ring
    const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int T = p.T, H = p.H, E = p.E, k = p.k, I = p.I, P = T * k;
    const int nseg_h = H / 32, nseg_i = I / 32;
    const int kc = k < 32 ? k : 32;                 // candidates per 32-logit chunk
    const int nchunk_e = (E + 31) / 32;
    const int ncand = nchunk_e * kc;                // candidates per token

    if (tid == 0) {
        for (int s = 0; s <= 2 * kMaxSlots; ++s) mbar_init(&sm.bar[s], 1);
        fence_mbar_init();
        sm.pending = 0;
    }
    __syncthreads();
    uint32_t phase_bits = 0;      // parity of the next phase of each ring slot
    uint32_t xphase = 0;          // parity of the x-staging barrier
    uint32_t nbar = 0;            // grid barriers passed

    for (int l = 0; l < p.L; ++l) {
        const DecodeLayer& Ly = p.layer[l];
        const uint16_t* x_cur = l == 0 ? p.x_in : ((l - 1) & 1 ? p.xbuf1 : p.xbuf0);
        const uint16_t* res = l == 0 ? p.residual0 : x_cur;
        uint16_t* x_nxt = l == p.L - 1 ? p.x_out : (l & 1 ? p.xbuf1 : p.xbuf0);
        uint16_t* xs_bf16 = reinterpret_cast<uint16_t*>(region_b);
        float* cand_v = reinterpret_cast<float*>(region_b + (((size_t)T * H * 2 + 15) & ~(size_t)15));
        int32_t* cand_i = reinterpret_cast<int32_t*>(cand_v + (size_t)T * ncand);

        // ---------------------------------------------------------------- R
        stamp(p, l, 0);
        if (tid == 0) {
            const uint32_t bytes = (uint32_t)(T * H * 2);
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sm.bar[kBarX], bytes);
            bulk_load(xs_bf16, x_cur, bytes, &sm.bar[kBarX]);
        }
        if (!mbar_wait(&sm.bar[kBarX], xphase)) {
            atomicOr(p.err, kDevErrTimeout);
            return;  // nothing else in flight
        }
        xphase ^= 1u;
        stamp(p, l, 1);
        {
            // 4 experts per pass, 4 warps per expert, each warp a quarter of H
            const int g = warp >> 2, q = warp & 3, hq = H / 4;
            for (int e0 = c; e0 < E; e0 += 4 * G) {
                const int e = e0 + g * G;
                float acc[kDecodeMaxTokens];
#pragma unroll
                for (int t = 0; t < kDecodeMaxTokens; ++t) acc[t] = 0.0f;
                if (e < E) {
                    const float* wr = Ly.wr + (size_t)e * H + (size_t)q * hq;
                    for (int h = lane * 4; h < hq; h += 128) {
                        const float4 w4 = __ldg(reinterpret_cast<const float4*>(wr + h));
#pragma unroll
                        for (int t = 0; t < kDecodeMaxTokens; ++t) {
                            if (t < T) {
                                const uint2 xp = *reinterpret_cast<const uint2*>(
                                    xs_bf16 + (size_t)t * H + (size_t)q * hq + h);
                                acc[t] = fmaf(w4.x, bf16_to_f32(xp.x & 0xFFFFu), acc[t]);
                                acc[t] = fmaf(w4.y, bf16_to_f32(xp.x >> 16), acc[t]);
                                acc[t] = fmaf(w4.z, bf16_to_f32(xp.y & 0xFFFFu), acc[t]);
                                acc[t] = fmaf(w4.w, bf16_to_f32(xp.y >> 16), acc[t]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < kDecodeMaxTokens; ++t) {
                    if (t < T) {
                        const float v = warp_sum(acc[t]);
                        if (lane == 0) sm.red[warp][t] = v;
                    }
                }
                __syncthreads();
                if (tid < 4 * T) {
                    const int gg = tid / T, t = tid % T;
                    const int ee = e0 + gg * G;
                    if (ee < E) {
                        const float sum = ((sm.red[4 * gg][t] + sm.red[4 * gg + 1][t]) +
                                           sm.red[4 * gg + 2][t]) + sm.red[4 * gg + 3][t];
                        p.logits[(size_t)t * E + ee] = sum + (Ly.bias ? Ly.bias[ee] : 0.0f);
                    }
                }
                __syncthreads();
            }
        }
        stamp(p, l, 2);
        if (!grid_barrier(p.bar, nbar++, p.err, &sm.flag)) return;
        stamp(p, l, 3);

        // ---------------------------------------------------------------- T
        // stage 1: each 32-logit chunk's own top-kc (warp arg-max by redux)
        for (int task = warp; task < T * nchunk_e; task += kWarps) {
            const int t = task / nchunk_e, ch = task % nchunk_e, e = ch * 32 + lane;
            const float v = e < E ? __ldcg(p.logits + (size_t)t * E + e) : 0.0f;
            uint32_t key = e < E ? order_key(v) : 0u;
            for (int r = 0; r < kc; ++r) {
                const uint32_t mx = __reduce_max_sync(0xffffffffu, key);
                const uint32_t win = __reduce_min_sync(0xffffffffu, key == mx ? (uint32_t)e : 0xFFFFFFFFu);
                const int slot = t * ncand + ch * kc + r;
                if ((uint32_t)e == win) {
                    cand_v[slot] = mx != 0u ? v : -FLT_MAX;
                    cand_i[slot] = mx != 0u ? e : 0x7FFFFFFF;
                    key = 0u;
                }
            }
        }
        __syncthreads();
        stamp(p, l, 4);
        // stage 2: k-way merge of the chunks' sorted candidate lists, one warp
        // per token, one lane per list; stage 3: softmax over the picks
        if (warp < T) {
            const int t = warp;
            const float* cv = cand_v + (size_t)t * ncand + (size_t)lane * kc;
            const int32_t* ci = cand_i + (size_t)t * ncand + (size_t)lane * kc;
            int head = 0;
            float hv = 0.0f;
            int hi = 0x7FFFFFFF;
            if (lane < nchunk_e) {
                hv = cv[0];
                hi = ci[0];
            }
            uint32_t key = hi != 0x7FFFFFFF ? order_key(hv) : 0u;
            int my_e = 0;
            float my_v = 0.0f;
            for (int r = 0; r < k; ++r) {
                const uint32_t mx = __reduce_max_sync(0xffffffffu, key);
                const uint32_t win = __reduce_min_sync(0xffffffffu, key == mx ? (uint32_t)hi : 0xFFFFFFFFu);
                const uint32_t wl = __ballot_sync(0xffffffffu, key == mx && (uint32_t)hi == win);
                const int src = __ffs(wl) - 1;
                const float wv = __shfl_sync(0xffffffffu, hv, src);
                if (lane == r) {
                    my_e = (int)win;
                    my_v = wv;
                }
                if (lane == src) {
                    ++head;
                    if (head < kc) {
                        hv = cv[head];
                        hi = ci[head];
                        key = hi != 0x7FFFFFFF ? order_key(hv) : 0u;
                    } else {
                        key = 0u;
                        hi = 0x7FFFFFFF;
                    }
                }
            }
            const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
            const float z = lane < k ? expf(my_v - v0) : 0.0f;
            const float sum = warp_sum(z);
            if (lane < k) {
                sm.idx[t * k + lane] = my_e;
                sm.w[t * k + lane] = __fdiv_rn(z, sum);
            }
        }
        __syncthreads();
        if (tid < P) {  // rank of pair tid in (expert, pair id) order
            const int e = sm.idx[tid];
            int rank = 0;
            for (int qq = 0; qq < P; ++qq) {
                const int eq = sm.idx[qq];
                rank += (eq < e) || (eq == e && qq < tid);
            }
            sm.perm[rank] = tid;
            sm.inv[tid] = rank;
            sm.pe[rank] = e;
        }
        stamp(p, l, 5);
        // max |x| over the call (non-negative floats order like their bits)
        uint32_t am_bits = 0;
        for (int i = tid; i < T * H / 2; i += kThreads) {
            const uint32_t two = reinterpret_cast<const uint32_t*>(xs_bf16)[i];
            am_bits = max(am_bits, max(__float_as_uint(fabsf(bf16_to_f32(two & 0xFFFFu))),
                                       __float_as_uint(fabsf(bf16_to_f32(two >> 16)))));
        }
        am_bits = __reduce_max_sync(0xffffffffu, am_bits);
        if (lane == 0) sm.redu[warp] = am_bits;
        __syncthreads();
        if (warp == 0) {  // tensor scale; active-expert list
            const uint32_t a = __reduce_max_sync(0xffffffffu, lane < kWarps ? sm.redu[lane] : 0u);
            if (lane == 0) sm.sx = tensor_scale_from_amax_bits(a);
            int base = 0;
            for (int r0 = 0; r0 < P; r0 += 32) {
                const int r = r0 + lane;
                const bool first = r < P && (r == 0 || sm.pe[r] != sm.pe[r - 1]);
                const uint32_t m = __ballot_sync(0xffffffffu, first);
                if (first) {
                    const int a_ = base + __popc(m & lt_mask);
                    sm.act_e[a_] = sm.pe[r];
                    sm.act_off[a_] = r;
                }
                base += __popc(m);
            }
            if (lane == 0) {
                sm.act_off[base] = P;
                sm.n_act = base;
            }
        }
        __syncthreads();
        stamp(p, l, 6);
        const float s_x = sm.sx;
        // NVFP4 form of x, one thread per 4 elements: int8 (value*2) + fp32 block scales
        uint32_t* xs8 = reinterpret_cast<uint32_t*>(region_a);                  // [T][H/4] words
        float* xsc = reinterpret_cast<float*>(region_a + (size_t)T * H);       // [T][H/16]
        for (int gi = tid; gi < T * H / 4; gi += kThreads) {
            const int t = gi / (H / 4), e4 = gi % (H / 4);
            const uint2 xp = reinterpret_cast<const uint2*>(xs_bf16)[gi];
            const float f[4] = {bf16_to_f32(xp.x & 0xFFFFu), bf16_to_f32(xp.x >> 16),
                                bf16_to_f32(xp.y & 0xFFFFu), bf16_to_f32(xp.y >> 16)};
            float am = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
            const uint32_t amask = __activemask();
            am = fmaxf(am, __shfl_xor_sync(amask, am, 1));
            am = fmaxf(am, __shfl_xor_sync(amask, am, 2));
            const uint32_t S = e4m3_rn_satfinite(__fdiv_rn(am, __fmul_rn(6.0f, s_x)));
            uint32_t nib = 0;
            if (S != 0) {
                const float m = __fmul_rn(e4m3_to_f32(S), s_x);
                float tq[8] = {__fdiv_rn(f[0], m), __fdiv_rn(f[1], m), __fdiv_rn(f[2], m),
                               __fdiv_rn(f[3], m), 0.f, 0.f, 0.f, 0.f};
                nib = e2m1x8_rn_satfinite(tq) & 0xFFFFu;
            }
            xs8[gi] = nib4_to_s8(nib);
            if ((e4 & 3) == 0) xsc[t * (H / 16) + e4 / 4] = e4m3_to_f32(S);
            if (c == 0) {  // the call's NVFP4 activations, for inspection
                reinterpret_cast<uint16_t*>(p.xq)[gi] = (uint16_t)nib;
                if ((e4 & 3) == 0) p.xs[t * (H / 16) + e4 / 4] = (uint8_t)S;
            }
        }
        if (c == 0) {  // routing results, for inspection
            if (tid == 0) *p.sx = s_x;
            if (tid < P) {
                p.idx[tid] = sm.idx[tid];
                p.w[tid] = sm.w[tid];
                p.perm[tid] = sm.perm[tid];
                p.inv[tid] = sm.inv[tid];
            }
            for (int e = tid; e <= E; e += kThreads) {
                int below = 0, at = 0;
                for (int qq = 0; qq < P; ++qq) {
                    below += sm.idx[qq] < e;
                    at += sm.idx[qq] == e;
                }
                if (e < E) p.counts[e] = at;
                p.offsets[e] = below;
            }
        }
        __syncthreads();
        stamp(p, l, 7);
        const int n_act = sm.n_act;
        // down ring: waves of up to slots_d/2 routed experts of one 16-row chunk
        const int d_nchunk = H / kRows;
        const int d_my_chunks = c < d_nchunk ? (d_nchunk - 1 - c) / G + 1 : 0;
        const uint32_t dcodes = (uint32_t)(kRows * I / 2), dscales = (uint32_t)(kRows * I / 16);
        const uint32_t d_slot_bytes = dcodes + dscales;
        const int dW = min(n_act, p.slots_d / 2);
        const int d_wpc = (n_act + dW - 1) / dW;
        const int d_waves = d_my_chunks * d_wpc;
        uint8_t* d_ring = region_b + p.d_off;
        auto issue_d_wave = [&](int v) {
            const int ch = c + (v / d_wpc) * G, a0 = (v % d_wpc) * dW, nw = min(dW, n_act - a0);
            for (int i = 0; i < nw; ++i) {
                const int s = (v & 1) * dW + i, e = sm.act_e[a0 + i];
                const size_t row0 = (size_t)e * H + (size_t)ch * kRows;
                uint8_t* dst = d_ring + (size_t)s * d_slot_bytes;
                mbar_arrive_expect_tx(&sm.bar[kBarD + s], d_slot_bytes);
                bulk_load(dst, Ly.dc + row0 * (I / 2), dcodes, &sm.bar[kBarD + s]);
                bulk_load(dst + dcodes, Ly.ds + row0 * (I / 16), dscales, &sm.bar[kBarD + s]);
                sm.pending |= 1u << (kBarD + s);
            }
        };
        // L2 prefetch: this CTA's down rows of the routed experts, next layer's router rows
        {
            const int nchunk = H / kRows;
            const int my_chunks = c < nchunk ? (nchunk - 1 - c) / G + 1 : 0;
            for (int i = tid; i < my_chunks * n_act; i += kThreads) {
                const int ch = c + (i / n_act) * G, e = sm.act_e[i % n_act];
                const size_t row0 = (size_t)e * H + (size_t)ch * kRows;
                prefetch_l2(Ly.dc + row0 * (I / 2), (uint32_t)(kRows * I / 2));
                prefetch_l2(Ly.ds + row0 * (I / 16), (uint32_t)(kRows * I / 16));
            }
            if (l + 1 < p.L) {
                const float* wr_next = p.layer[l + 1].wr;
                for (int e = c + tid * G; e < E; e += kThreads * G)
                    prefetch_l2(wr_next + (size_t)e * H, (uint32_t)(H * 4));
            }
        }
        stamp(p, l, 8);

        // ---------------------------------------------------------------- G
        {
            const int nfb = I / kRows;
            const int n_items = n_act * nfb;
            const int my_items = c < n_items ? (n_items - 1 - c) / G + 1 : 0;
            const uint32_t half_codes = (uint32_t)(kRows * H / 2), half_scales = (uint32_t)(kRows * H / 16);
            const uint32_t slot_bytes = 2 * (half_codes + half_scales);
            const int S = p.slots_g;
            const int W = my_items <= S ? my_items : S / 2;     // items per wave
            const int n_waves = W > 0 ? (my_items + W - 1) / W : 0;
            auto slot_of = [&](int m) { return W == my_items ? m : ((m / W) & 1) * W + m % W; };
            auto issue = [&](int m) {
                const int it = c + m * G, a = it / nfb, fb = it % nfb, s = slot_of(m);
                const int e = sm.act_e[a];
                const size_t row0 = (size_t)e * I + (size_t)fb * kRows;
                uint8_t* dst = region_b + (size_t)s * slot_bytes;
                mbar_arrive_expect_tx(&sm.bar[s], slot_bytes);
                bulk_load(dst, Ly.gc + row0 * (H / 2), half_codes, &sm.bar[s]);
                bulk_load(dst + half_codes, Ly.gs + row0 * (H / 16), half_scales, &sm.bar[s]);
                bulk_load(dst + half_codes + half_scales, Ly.uc + row0 * (H / 2), half_codes, &sm.bar[s]);
                bulk_load(dst + 2 * half_codes + half_scales, Ly.us + row0 * (H / 16), half_scales,
                          &sm.bar[s]);
                sm.pending |= 1u << s;
            };
            if (tid == 0) {
                fence_proxy_async_smem();
                for (int m = 0; m < my_items && m < 2 * W; ++m) issue(m);
                if (p.d_early)  // the down rows land in their own slots while gate/up runs
                    for (int v = 0; v < d_waves && v < 2; ++v) issue_d_wave(v);
            }
            for (int v = 0; v < n_waves; ++v) {
                const int m0 = v * W, nw = min(W, my_items - m0);
                if (!wait_slots(sm, slot_of(m0), nw, phase_bits, p.err)) return;
                if (v == 0) stamp(p, l, 9);
                // every item of the wave: warp = feature, lanes split H
                for (int i = 0; i < nw; ++i) {
                    const int it = c + (m0 + i) * G, a = it / nfb;
                    const int e = sm.act_e[a], r0 = sm.act_off[a], r1 = sm.act_off[a + 1];
                    const uint8_t* slot = region_b + (size_t)slot_of(m0 + i) * slot_bytes;
                    const uint8_t* grow = slot + (size_t)warp * (H / 2);
                    const uint8_t* gsc = slot + half_codes + (size_t)warp * (H / 16);
                    const uint8_t* urow = slot + half_codes + half_scales + (size_t)warp * (H / 2);
                    const uint8_t* usc = slot + 2 * half_codes + half_scales + (size_t)warp * (H / 16);
                    const float gs = __fmul_rn(__fmul_rn(Ly.gts[e], s_x), 0.25f);
                    const float us = __fmul_rn(__fmul_rn(Ly.uts[e], s_x), 0.25f);
                    for (int r = r0; r < r1; ++r) {
                        const int t = sm.perm[r] / k;
                        float ga = 0.0f, ua = 0.0f;
                        for (int seg = lane; seg < nseg_h; seg += 32) {
                            XSeg x;
                            read_seg8(xs8 + (size_t)t * (H / 4) + seg * 8, x);
                            const float2 xs2 = *reinterpret_cast<const float2*>(xsc + t * (H / 16) + 2 * seg);
                            const uint4 wg = *reinterpret_cast<const uint4*>(grow + seg * 16);
                            const uint4 wu = *reinterpret_cast<const uint4*>(urow + seg * 16);
                            const uint32_t sg = *reinterpret_cast<const uint16_t*>(gsc + seg * 2);
                            const uint32_t su = *reinterpret_cast<const uint16_t*>(usc + seg * 2);
                            ga += dot_seg32(wg, sg, x, xs2);
                            ua += dot_seg32(wu, su, x, xs2);
                        }
                        ga = warp_sum(ga);
                        ua = warp_sum(ua);
                        if (lane == 0)
                            sm.hbuf[i][r - r0][warp] = __fmul_rn(silu(__fmul_rn(ga, gs)), __fmul_rn(ua, us));
                    }
                }
                __syncthreads();  // wave consumed, hbuf complete
                if (tid == 0) {
                    for (int i = 0; i < nw; ++i) sm.pending &= ~(1u << slot_of(m0 + i));
                    fence_proxy_async_smem();
                    for (int m = m0 + 2 * W; m < min(my_items, m0 + 3 * W); ++m) issue(m);
                }
                // Q on each 16-feature block: one half-warp per (item, pair) task,
                // tasks numbered across the wave's items; the loop base is
                // warp-uniform so both halves run every shuffle
                const int half = lane >> 4, hl = lane & 15;
                int n_tasks = 0;
                for (int i = 0; i < nw; ++i) {
                    const int a = (c + (m0 + i) * G) / nfb;
                    n_tasks += sm.act_off[a + 1] - sm.act_off[a];
                }
                for (int base = 2 * warp; base < n_tasks; base += 2 * kWarps) {
                    const int tq = base + half;
                    const bool valid = tq < n_tasks;
                    int i = 0, pr = tq, a = 0, fb = 0, r0 = 0;
                    if (valid) {
                        for (;; ++i) {
                            const int it = c + (m0 + i) * G;
                            a = it / nfb;
                            fb = it % nfb;
                            r0 = sm.act_off[a];
                            const int np = sm.act_off[a + 1] - r0;
                            if (pr < np) break;
                            pr -= np;
                        }
                    }
                    const float hv = valid ? sm.hbuf[i][pr][hl] : 0.0f;
                    float am = fabsf(hv);
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
                    const float q = __fdiv_rn(am, __fmul_rn(6.0f, p.h_scale));
                    const uint32_t Sh = e4m3_rn_satfinite(q);
                    uint32_t code = 0;
                    if (Sh != 0) code = e2m1_one(__fdiv_rn(hv, __fmul_rn(e4m3_to_f32(Sh), p.h_scale)));
                    const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
                    if (valid) {
                        const int r = r0 + pr;
                        if ((hl & 1) == 0)
                            p.hq[(size_t)r * (I / 2) + fb * 8 + hl / 2] = (uint8_t)(code | (hi << 4));
                        if (hl == 0) p.hs[(size_t)r * (I / 16) + fb] = (uint8_t)Sh;
                    }
                }
                __syncthreads();  // hbuf read before the next wave overwrites it
            }
        }
        stamp(p, l, 10);
        if (!grid_barrier(p.bar, nbar++, p.err, &sm.flag)) return;
        stamp(p, l, 11);

        // ---------------------------------------------------------------- D
        {
            uint32_t* hs8 = reinterpret_cast<uint32_t*>(region_a);                 // [P][I/4] words
            float* hsc = reinterpret_cast<float*>(region_a + (size_t)P * I);      // [P][I/16]
            for (int i = tid; i < P * nseg_i; i += kThreads) {
                const uint4 cw = __ldcg(reinterpret_cast<const uint4*>(p.hq) + i);
                XSeg x;
                load_xseg(cw, x);
                uint4* d = reinterpret_cast<uint4*>(hs8 + (size_t)i * 8);
                d[0] = make_uint4(x.v[0], x.v[1], x.v[2], x.v[3]);
                d[1] = make_uint4(x.v[4], x.v[5], x.v[6], x.v[7]);
            }
            for (int i = tid; i < P * (I / 16); i += kThreads) hsc[i] = e4m3_to_f32(__ldcg(p.hs + i));
            __syncthreads();
            stamp(p, l, 12);
            if (!p.d_early && tid == 0) {
                fence_proxy_async_smem();
                for (int v = 0; v < d_waves && v < 2; ++v) issue_d_wave(v);
            }
            const float os_h = p.h_scale;
            const int half = lane >> 4, hl = lane & 15;
            for (int v = 0; v < d_waves; ++v) {
                const int ch = c + (v / d_wpc) * G, a0 = (v % d_wpc) * dW, nw = min(dW, n_act - a0);
                if (!wait_slots(sm, kBarD + (v & 1) * dW, nw, phase_bits, p.err)) return;
                if (v == 0) stamp(p, l, 13);
                for (int i = 0; i < nw; ++i) {  // warp = output row; half-warps = two pairs
                    const int a = a0 + i, e = sm.act_e[a], r0 = sm.act_off[a], r1 = sm.act_off[a + 1];
                    const uint8_t* slot = d_ring + (size_t)((v & 1) * dW + i) * d_slot_bytes;
                    const uint8_t* drow = slot + (size_t)warp * (I / 2);
                    const uint8_t* dsc = slot + dcodes + (size_t)warp * (I / 16);
                    const float os = __fmul_rn(__fmul_rn(Ly.dts[e], os_h), 0.25f);
                    for (int r = r0; r < r1; r += 2) {
                        const int rr = r + half;
                        float acc = 0.0f;
                        if (rr < r1) {
                            for (int seg = hl; seg < nseg_i; seg += 16) {
                                XSeg x;
                                read_seg8(hs8 + (size_t)rr * (I / 4) + seg * 8, x);
                                const float2 hs2 = *reinterpret_cast<const float2*>(hsc + rr * (I / 16) + 2 * seg);
                                const uint4 wd = *reinterpret_cast<const uint4*>(drow + seg * 16);
                                const uint32_t sd = *reinterpret_cast<const uint16_t*>(dsc + seg * 2);
                                acc += dot_seg32(wd, sd, x, hs2);
                            }
                        }
#pragma unroll
                        for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                        if (hl == 0 && rr < r1) sm.obuf[rr][warp] = __fmul_rn(acc, os);
                    }
                }
                __syncthreads();  // wave consumed
                if (tid == 0) {
                    for (int i = 0; i < nw; ++i) sm.pending &= ~(1u << (kBarD + (v & 1) * dW + i));
                    fence_proxy_async_smem();
                    if (v + 2 < d_waves) issue_d_wave(v + 2);
                }
                if (v % d_wpc == d_wpc - 1) {  // chunk complete: combine in slot order, residual
                    if (tid < T * kRows) {
                        const int t = tid / kRows, w = tid % kRows;
                        float y = 0.0f;
                        for (int j = 0; j < k; ++j)
                            y = fmaf(sm.w[t * k + j], sm.obuf[sm.inv[t * k + j]][w], y);
                        const size_t off = (size_t)t * H + (size_t)ch * kRows + w;
                        if (Ly.y) Ly.y[off] = y;
                        if (x_nxt) x_nxt[off] = f32_to_bf16_rn(bf16_to_f32(__ldcg(res + off)) + y);
                    }
                    __syncthreads();  // obuf read before the next chunk writes it
                }
            }
        }
        stamp(p, l, 14);
        if (!grid_barrier(p.bar, nbar++, p.err, &sm.flag)) return;
        stamp(p, l, 15);
    }
}

}  // namespace

bool decode_supported(const Shape& s, int T) {
    if (T < 1 || T > kDecodeMaxTokens || T * s.k > kDecodeMaxPairs) return false;
    if (s.H > 4096 || s.I > 2048 || s.E > 1024) return false;
    return decode_smem_plan(s, T).ok;
}

DecodeSmemPlan decode_smem_plan(const Shape& s, int T) {
    DecodeSmemPlan pl{};
    const size_t head = (sizeof(Smem) + 1023) / 1024 * 1024;
    const size_t P = (size_t)T * s.k;
    const size_t a_x = (size_t)T * s.H + (size_t)T * (s.H / 16) * 4;
    const size_t a_h = P * s.I + P * (s.I / 16) * 4;
    const size_t a = ((a_x > a_h ? a_x : a_h) + 1023) / 1024 * 1024;
    const size_t total = kDecodeSmemBytes;
    if (head + a >= total) return pl;
    const size_t b = total - head - a;
    const size_t slot_g = 2 * ((size_t)kRows * s.H / 2 + (size_t)kRows * s.H / 16);
    const size_t slot_d = (size_t)kRows * s.I / 2 + (size_t)kRows * s.I / 16;
    const size_t kc = s.k < 32 ? s.k : 32;
    const size_t cand = (size_t)T * ((s.E + 31) / 32) * kc;
    const size_t stage = (((size_t)T * s.H * 2 + 15) & ~(size_t)15) + cand * 8;
    if (stage > b || cand > kMaxCand) return pl;
    // early down ring: a full 16-slot down ring after the gate/up slots, if
    // at least 3 gate/up slots remain and the ring clears the x staging area
    const size_t d_ring = (size_t)kMaxSlots * slot_d;
    size_t sg = 0, sd = 0, d_off = 0;
    int early = 0;
    if (b > d_ring && (b - d_ring) / slot_g >= 3 && (b - d_ring) >= stage) {
        early = 1;
        d_off = ((b - d_ring) / 16) * 16;
        sg = d_off / slot_g;
        sd = kMaxSlots;
    } else {
        sg = b / slot_g;
        sd = b / slot_d;
    }
    if (sg > kMaxSlots) sg = kMaxSlots;
    if (sd > kMaxSlots) sd = kMaxSlots;
    if (sg < 2 || sd < 2) return pl;
    pl.ok = true;
    pl.region_a_off = (uint32_t)head;
    pl.region_b_off = (uint32_t)(head + a);
    pl.slots_g = (int)sg;
    pl.slots_d = (int)(sd & ~(size_t)1);
    pl.d_off = (uint32_t)d_off;
    pl.d_early = early;
    pl.bytes = total;
    return pl;
}

cudaError_t launch_decode(const DecodeParams& prm, cudaStream_t st) {
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(k_decode, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kDecodeSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(prm.bar, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kDecodeSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_decode, prm);
    count_launches(1);
    return e;
}

}  // namespace moe
