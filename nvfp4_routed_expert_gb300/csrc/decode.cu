// Decode path: one persistent, cooperatively launched kernel that runs S1..S6
// for up to 8 tokens through a whole stack of layers (one layer for
// moe_forward, up to 64 for moe_stack_forward).
//
// Decode is bound by memory bandwidth (capy-flash v0.7.1, "Why it matters"):
// at one token a layer moves ~22 MB, a few microseconds of HBM time, so what
// decides the speed is how little latency sits between the HBM streams.  The
// kernel keeps every SM resident for the whole stack and hands data between
// CTAs through tagged words instead of grid barriers: every exchanged value
// travels in a 64-bit word whose top 16 bits are a tag naming the layer that
// wrote it, so a reader polls the data itself and needs one L2 round trip,
// not a barrier followed by a read.  Per layer:
//
//   R  x of the layer (tagged words of the previous layer, or the input);
//      router logits of the CTA's experts from router rows already in shared
//      memory (loaded by bulk copy during the previous layer) -> tagged logits;
//      the next layer's router rows start loading (after G instead, when the
//      gate/up slots need their space)
//   Q  in every CTA, redundantly: the NVFP4 form of x, held as f16 values
//   T  all logits (tagged words); in every CTA: top-k + softmax, the
//      expert-grouped permutation, the active-expert list; the CTA's share of
//      the routed experts' gate/up AND down rows starts streaming from HBM into
//      shared-memory slots at once
//   G  gate/up items (routed expert x 16 features) as their rows land; SwiGLU
//      and requantisation of h -> tagged h words
//   D  all h (tagged words); down rows of the CTA's output rows for every
//      routed expert (already in shared memory, or streaming through the
//      freed gate/up slots); per-pair outputs combined in slot order, residual
//      added -> tagged x of the next layer (or the stack's output)
//
// Every phase runs once per layer, so the kernel's code is fetched once per
// layer too: rare paths are kept out of line (a probe that added 64 KB of
// straight-line code to each layer cost 10 us per layer).
//
// Every wait (mbarrier or tagged word) is bounded: a wait that runs out sets
// the status word, the CTA waits (bounded) for its own copies in flight and
// returns, and the other CTAs see the status word and return too.
#include <cfloat>

#include "common.cuh"
#include "decode.h"
#include "kernels.h"
#include "sync.cuh"

namespace moe {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;   // 16: one feature / output row per warp
constexpr int kRows = 16;               // features per gate/up item = one NVFP4 block of h
constexpr int kMaxSlotsG = 8;
constexpr int kMaxSlotsD = 32;
constexpr int kMaxSlotsDArea = 16;
constexpr int kMaxWrRows = 8;
constexpr int kMaxDRows = 64;
constexpr int kMaxTopK = 16;            // largest top-k the fused kernel takes

constexpr int kBarG = 0;
constexpr int kBarD = kMaxSlotsG;
constexpr int kBarX = kBarD + kMaxSlotsD;
constexpr int kBarWr = kBarX + 1;
constexpr int kNumBars = kBarWr + 1;
static_assert(kNumBars <= 64, "phase and pending masks are 64-bit");

constexpr uint32_t kPollLimit = 1u << 20;   // polls of one batch of tagged words (~1 s)

// tagged words in flight per thread: enough for one round trip at the decode
// shapes, few enough to keep the code small at one token
template <int T>
__host__ __device__ constexpr int poll_batch() { return T == 1 ? 2 : T <= 2 ? 4 : T <= 4 ? 8 : 16; }

struct Head {
    uint64_t bar[kNumBars];
    int32_t idx[kDecodeMaxPairs];      // [t][j]
    uint32_t selk[kDecodeMaxPairs];    // order keys of the picks
    float w[kDecodeMaxPairs];
    uint32_t gmax[kDecodeMaxTokens][kWarps];   // per token, the largest key of each warp's experts
    uint32_t tau[kDecodeMaxTokens];
    int32_t ccount[kDecodeMaxTokens];
    int32_t perm[kDecodeMaxPairs];
    int32_t inv[kDecodeMaxPairs];
    int32_t pe[kDecodeMaxPairs];       // expert of each expert-grouped position
    int32_t act_e[kDecodeMaxPairs];
    int32_t act_off[kDecodeMaxPairs + 1];
    float act_gs[kDecodeMaxPairs];     // gate / up / down output scales per active expert
    float act_us[kDecodeMaxPairs];
    float act_ds[kDecodeMaxPairs];
    float bias[kMaxWrRows];
    int32_t pair_unit[kDecodeMaxPairs];   // active-expert index of each expert-grouped position
    int32_t pair_tok[kDecodeMaxPairs];    // token of each expert-grouped position
    uint32_t pair_slot[kDecodeMaxPairs];  // shared-memory offset of the down slot of each position's unit
    int32_t it_a[kMaxSlotsG];             // items of the current gate/up wave: active expert,
    int32_t it_fb[kMaxSlotsG];            // feature block, first position, offset of the slot
    int32_t it_r0[kMaxSlotsG];
    uint32_t it_slot[kMaxSlotsG];
    int16_t wt_i[kMaxSlotsG * kDecodeMaxTokens];   // (item, pair) tasks of a gate/up wave
    int16_t wt_r[kMaxSlotsG * kDecodeMaxTokens];
    int32_t n_wt;
    int32_t n_act;
    int32_t n_pos;                     // pairs computed (all T * k unless the route-tail skip dropped some)
    uint8_t resident[1024];            // route-tail skip: experts never skipped
    float sx;
    uint64_t pending;                  // bit b: mbarrier b has a copy in flight
    uint32_t redu[kWarps];
    float red[kWarps][kDecodeMaxTokens];
    float hbuf[kMaxSlotsG][kDecodeMaxTokens][kRows];
    uint16_t res[kDecodeMaxTokens][kMaxDRows];
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

__device__ __forceinline__ uint64_t ld_relaxed_b64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Publish a tagged exchange word.  The tag grows each time a word is reused
// (two layers later, the tag of that layer), so a max-reduction at L2 writes it
// like a store; unlike a store it is performed in L2 at once rather than
// lingering in the SM (plain stores were measured to reach the other SMs
// microseconds late, and a fence after them costs the writer a round trip).
__device__ __forceinline__ void publish_b64(uint64_t* p, uint64_t v) {
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Tagged exchange word: the layer tag in the top 16 bits, up to 48 bits of payload.
constexpr int kTagShift = 48;
__device__ __forceinline__ uint64_t tagged(uint32_t tag, uint64_t payload) {
    return ((uint64_t)tag << kTagShift) | payload;
}
__device__ __forceinline__ uint32_t tag_of(uint64_t w) { return (uint32_t)(w >> kTagShift); }



__device__ __forceinline__ void prefetch_line_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t e2m1_one(float v) {
    float t[8] = {v, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    return e2m1x8_rn_satfinite(t) & 0xFu;
}

// fp32 -> uint32 key with the same order (finite values; -0 and +0 get the
// same key, as they compare equal); 0 is below every key
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sum each of eight per-lane values over the 16 lanes of a half-warp, by
// halving: at xor distance 8 a lane keeps four of the values (adding its
// partner's), at 4 two, at 2 one, at 1 that one.  8 shuffles instead of 32;
// the total of value q ends in the lanes whose bits 3, 2, 1 spell q.
__device__ __forceinline__ float half_warp_sum8(const float* v, int hl) {
    float a[4], b[2];
    const bool s3 = (hl & 8) != 0, s2 = (hl & 4) != 0, s1 = (hl & 2) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        a[i] = (s3 ? v[4 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, s3 ? v[i] : v[4 + i], 8);
#pragma unroll
    for (int i = 0; i < 2; ++i)
        b[i] = (s2 ? a[2 + i] : a[i]) + __shfl_xor_sync(0xffffffffu, s2 ? a[i] : a[2 + i], 4);
    float c = (s1 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, s1 ? b[0] : b[1], 2);
    return c + __shfl_xor_sync(0xffffffffu, c, 1);
}

// The same over a whole warp (xor distances 16, 8, 4 halving, then 2 and 1):
// the total of value q ends in the lanes whose bits 4, 3, 2 spell q.  The
// additions pair the same partial sums as a plain butterfly per value, so the
// totals are the same floats.
__device__ __forceinline__ float warp_sum8(const float* v, int lane) {
    float a[4], b[2];
    const bool s4 = (lane & 16) != 0, s3 = (lane & 8) != 0, s2 = (lane & 4) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        a[i] = (s4 ? v[4 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, s4 ? v[i] : v[4 + i], 16);
#pragma unroll
    for (int i = 0; i < 2; ++i)
        b[i] = (s3 ? a[2 + i] : a[i]) + __shfl_xor_sync(0xffffffffu, s3 ? a[i] : a[2 + i], 8);
    float c = (s2 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, s2 ? b[0] : b[1], 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    return c + __shfl_xor_sync(0xffffffffu, c, 1);
}

// Activations are stored as f16x2 words of their E2M1 values, split in four
// quarters: words 4j .. 4j+3 of every 32-element segment (its elements
// 8j .. 8j+7) in quarter j, `quarter` words after quarter j - 1, so that lanes
// reading consecutive segments read consecutive 16-byte words (no shared-memory
// bank conflicts).
__device__ __forceinline__ void read_seg16h(const uint32_t* p, size_t quarter, uint32_t* x) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(p + (size_t)j * quarter);
        x[4 * j] = v.x;
        x[4 * j + 1] = v.y;
        x[4 * j + 2] = v.z;
        x[4 * j + 3] = v.w;
    }
}

// Wait until the n tagged words at src all carry `tag` and hand each payload
// to consume(i, payload).  Every thread of the CTA calls it; the result is the
// same in all of them (false: the wait ran out or another CTA failed).
template <int kBatch, class F>
__device__ __forceinline__ bool poll_tagged(const uint64_t* src, int n, uint32_t tag,
                                            uint32_t* err, F&& consume) {
    bool ok = true;
#pragma unroll 1
    for (int base = 0; base < n; base += kThreads * kBatch) {
        uint64_t v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = base + j * kThreads + (int)threadIdx.x;
            v[j] = (ok && i < n) ? ld_relaxed_b64(src + i) : tagged(tag, 0ull);
        }
#pragma unroll 1
        for (uint32_t spin = 0; ok; ++spin) {
            bool all = true;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) all &= tag_of(v[j]) == tag;
            if (all) break;
            if (spin >= kPollLimit) {
                atomicOr(err, kDevErrTimeout);
                ok = false;
                break;
            }
            if ((spin & 63u) == 63u && ld_relaxed_gpu(err) != 0) {
                ok = false;
                break;
            }
            if (spin > 16) __nanosleep(32);
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = base + j * kThreads + (int)threadIdx.x;
                if (i < n && tag_of(v[j]) != tag) v[j] = ld_relaxed_b64(src + i);
            }
        }
        if (ok) {
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = base + j * kThreads + (int)threadIdx.x;
                if (i < n) consume(i, v[j]);
            }
        }
    }
    return __syncthreads_and(ok ? 1 : 0) != 0;
}

// Wait (bounded) for every mbarrier that still has a copy in flight, so that
// no bulk copy lands in shared memory after the CTA has exited.
__device__ __noinline__ void drain(Head& hd, uint64_t phase_bits, uint32_t* err) {
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int b = 0; b < kNumBars; ++b) {
            if ((hd.pending >> b) & 1ull) {
                if (!mbar_wait(&hd.bar[b], (uint32_t)(phase_bits >> b) & 1u)) atomicOr(err, kDevErrTimeout);
            }
        }
        hd.pending = 0;
    }
    __syncthreads();
}

// Bulk copies of one gate/up item (16 gate rows and 16 up rows of an expert,
// codes and scales) into a slot, completing on `bar`.
__device__ __forceinline__ void issue_item(uint64_t* bar, uint8_t* dst, const uint8_t* gc,
                                        const uint8_t* gs, const uint8_t* uc, const uint8_t* us,
                                        size_t row0, int H, bool arm = true) {
    const uint32_t codes = (uint32_t)(kRows * H / 2), scales = (uint32_t)(kRows * H / 16);
    if (arm) mbar_arrive_expect_tx(bar, 2 * (codes + scales));
    bulk_load(dst, gc + row0 * (H / 2), codes, bar);
    bulk_load(dst + codes, gs + row0 * (H / 16), scales, bar);
    bulk_load(dst + codes + scales, uc + row0 * (H / 2), codes, bar);
    bulk_load(dst + 2 * codes + scales, us + row0 * (H / 16), scales, bar);
}

// Bulk copies of `rows` down rows (codes, then scales) into a slot.
__device__ __forceinline__ void issue_unit(uint64_t* bar, uint8_t* dst, const uint8_t* dc,
                                        const uint8_t* ds, size_t row0, int rows, int I,
                                        bool arm = true) {
    const uint32_t codes = (uint32_t)(rows * I / 2), scales = (uint32_t)(rows * I / 16);
    if (arm) mbar_arrive_expect_tx(bar, codes + scales);
    bulk_load(dst, dc + row0 * (I / 2), codes, bar);
    bulk_load(dst + codes, ds + row0 * (I / 16), scales, bar);
}

// Bulk copies of the router rows c, c + G, ... (n of them) into wr_s.
__device__ __noinline__ void issue_router_rows(uint64_t* bar, float* wr_s, const float* wr, int c,
                                               int G, int n, int H) {
    mbar_arrive_expect_tx(bar, (uint32_t)(n * H * 4));
#pragma unroll 1
    for (int j = 0; j < n; ++j)
        bulk_load(wr_s + (size_t)j * H, wr + (size_t)(c + j * G) * H, (uint32_t)(H * 4), bar);
}

template <int T>
__global__ void __launch_bounds__(kThreads, 1) k_decode(const __grid_constant__ DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Head& hd = *reinterpret_cast<Head*>(smem_raw);
    const DecodeSmemPlan& pl = p.plan;
    float* wr_s = reinterpret_cast<float*>(smem_raw + pl.wr_off);
    uint8_t* area_a = smem_raw + pl.a_off;
    uint8_t* ring = smem_raw + pl.ring_off;
    uint8_t* gslots = smem_raw + pl.g_off;   // gate/up slot s at gslots + s * sg
    const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int H = p.H, E = p.E, k = p.k, I = p.I, P = T * k;
    const int nseg_h = H / 32, nseg_i = I / 32, nb_i = I / 16, nfb = I / kRows;

    // static split of the router rows and of the output rows of the down step
    const int n_my_e = c < E ? (E - 1 - c) / G + 1 : 0;
    const int npr = H / 2, q_pr = npr / G, rem_pr = npr % G;
    const int my_pairs = q_pr + (c < rem_pr ? 1 : 0);
    const int d_r0 = 2 * (c * q_pr + min(c, rem_pr));
    const int d_nrows = 2 * my_pairs;
    const int d_rows = pl.d_rows;

    // tagged exchange words: logits [2][T][E], h [2][P][I/16][2], x [2][T][H/2]
    const size_t tl_words = (size_t)T * E, th_words = (size_t)P * nb_i * 2,
                 tx_words = (size_t)T * (H / 2);
    uint64_t* tag_l = p.tags;
    uint64_t* tag_h = tag_l + 2 * tl_words;
    uint64_t* tag_x = tag_h + 2 * th_words;

    // ring scratch of the T step: logits and the top-k candidate lists
    // (keys and expert indices, up to E per token)
    float* lg = reinterpret_cast<float*>(ring);                                       // [T][E]
    uint32_t* cand_k = reinterpret_cast<uint32_t*>(lg + (((size_t)T * E + 3) & ~(size_t)3));  // [T][E]
    int32_t* cand_i = reinterpret_cast<int32_t*>(cand_k + (size_t)T * E);           // [T][E]
    // area a: x as int8 + block scales + the bf16 staging of x; later h
    uint32_t* xh = reinterpret_cast<uint32_t*>(area_a);                        // [4][T * H/32][4] f16x2
    float* xsc = reinterpret_cast<float*>(area_a + (size_t)T * H * 2);        // [T][H/16]
    uint16_t* xs_bf16 = reinterpret_cast<uint16_t*>(area_a + (size_t)T * H * 2 + (size_t)T * (H / 16) * 4);  // [T][H]
    uint32_t* hh = reinterpret_cast<uint32_t*>(area_a);                        // [4][P * I/32][4] f16x2
    float* hsc = reinterpret_cast<float*>(area_a + (size_t)P * I * 2);        // [P][I/16]
    float* obuf = hsc + (size_t)P * nb_i;                                      // [P][d_rows]

    // slot sizes
    const uint32_t g_codes = (uint32_t)(kRows * H / 2), g_scales = (uint32_t)(kRows * H / 16);
    const uint32_t sg = 2 * (g_codes + g_scales);
    const uint32_t d_codes = (uint32_t)(d_nrows * I / 2);
    const uint32_t sd = (uint32_t)(d_rows * (I / 2 + I / 16));
    auto d_slot_ptr = [&](int s) {
        return s < pl.slots_d ? smem_raw + pl.d_area_off + (size_t)s * sd
                              : ring + (size_t)(s - pl.slots_d) * sd;   // freed gate/up area
    };

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) mbar_init(&hd.bar[b], 1);
        fence_mbar_init();
        hd.pending = 0;
    }
    __syncthreads();
    uint64_t ph = 0;   // thread 0: parity of the next phase of each mbarrier

    // Thread 0 waits for the n mbarriers bar0 + (first + i) % mod and keeps the
    // phase bits; the CTA barrier hands the outcome to the other threads and
    // orders their reads of the landed data after the wait.  (Bookkeeping that
    // every thread repeats costs 16 warps' worth of issue slots, so it is done
    // once.)  On a timeout the CTA drains its copies and the caller returns.
    auto wait_bars = [&](int bar0, int first, int n, int mod) -> bool {
        bool ok = true;
        if (tid == 0) {
            int sl = first % mod;
#pragma unroll 1
            for (int i = 0; i < n && ok; ++i) {
                const int b = bar0 + sl;
                ok = mbar_wait(&hd.bar[b], (uint32_t)(ph >> b) & 1u);
                if (ok) {
                    ph ^= 1ull << b;
                    hd.pending &= ~(1ull << b);
                }
                if (++sl == mod) sl = 0;
            }
            if (!ok) atomicOr(p.err, kDevErrTimeout);
        }
        if (!__syncthreads_and(ok ? 1 : 0)) {
            drain(hd, ph, p.err);
            return false;
        }
        return true;
    };
    // thread 0 only: router rows of layer l2 -> wr_s
    auto issue_wr = [&](int l2) {
        issue_router_rows(&hd.bar[kBarWr], wr_s, p.layer[l2].wr, c, G, n_my_e, H);
        hd.pending |= 1ull << kBarWr;
    };

    if (tid == 0) issue_wr(0);

#pragma unroll 1
    for (int l = 0; l < p.L; ++l) {
        const DecodeLayer& Ly = p.layer[l];
        const uint32_t tag = (uint32_t)l + 1;        // tag of the words this layer writes
        const int buf = l & 1;
        const bool last = l == p.L - 1;
        const int keep = Ly.keep < k ? Ly.keep : k;   // route-tail skip: ranks always computed
        stamp(p, l, 0);
        if (keep < k) {
            for (int e = tid; e < E; e += kThreads) hd.resident[e] = Ly.resident ? Ly.resident[e] : 0;
        }

        // ------------------------------------------------------------------ R
        // loads whose latency hides behind the wait for x
        const float bias_r = (tid < n_my_e && Ly.bias) ? __ldg(Ly.bias + c + tid * G) : 0.0f;
        uint16_t res_r = 0;
        if (l == 0 && p.residual0 && tid < T * d_nrows)
            res_r = p.residual0[(size_t)(tid / d_nrows) * H + d_r0 + tid % d_nrows];
        if (l == 0) {
            if (tid == 0) {
                const uint32_t bytes = (uint32_t)(T * H * 2);
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&hd.bar[kBarX], bytes);
                bulk_load(xs_bf16, p.x_in, bytes, &hd.bar[kBarX]);
                hd.pending |= 1ull << kBarX;
            }
            if (!wait_bars(kBarX, 0, 1, 1)) return;
        } else {
            uint32_t* xw = reinterpret_cast<uint32_t*>(xs_bf16);
            if (!poll_tagged<poll_batch<T>()>(tag_x + (size_t)((l - 1) & 1) * tx_words, (int)tx_words,
                                              tag - 1, p.err, [&](int i, uint64_t v) { xw[i] = (uint32_t)v; })) {
                drain(hd, ph, p.err);
                return;
            }
        }
        if (tid < n_my_e) hd.bias[tid] = bias_r;
        if (tid < T * d_nrows) {
            const int t = tid / d_nrows, j = tid % d_nrows;
            hd.res[t][j] = l == 0 ? res_r : xs_bf16[(size_t)t * H + d_r0 + j];
        }
        stamp(p, l, 1);
        // (the wait ends in a CTA barrier, which also publishes bias and res)
        if (!wait_bars(kBarWr, 0, 1, 1)) return;
        {
            // 4 experts per pass, 4 warps per expert, each warp a quarter of H
            const int g = warp >> 2, qq = warp & 3, hq4 = H / 4;
#pragma unroll 1
            for (int j0 = 0; j0 < n_my_e; j0 += 4) {
                const int j = j0 + g;
                float acc[T];
#pragma unroll
                for (int t = 0; t < T; ++t) acc[t] = 0.0f;
                if (j < n_my_e) {
                    const float* wr = wr_s + (size_t)j * H + (size_t)qq * hq4;
                    const uint16_t* xr = xs_bf16 + (size_t)qq * hq4;
#pragma unroll 1
                    for (int h = lane * 4; h < hq4; h += 128) {
                        const float4 w4 = *reinterpret_cast<const float4*>(wr + h);
#pragma unroll
                        for (int t = 0; t < T; ++t) {
                            const uint2 xp = *reinterpret_cast<const uint2*>(xr + (size_t)t * H + h);
                            acc[t] = fmaf(w4.x, bf16_to_f32(xp.x & 0xFFFFu), acc[t]);
                            acc[t] = fmaf(w4.y, bf16_to_f32(xp.x >> 16), acc[t]);
                            acc[t] = fmaf(w4.z, bf16_to_f32(xp.y & 0xFFFFu), acc[t]);
                            acc[t] = fmaf(w4.w, bf16_to_f32(xp.y >> 16), acc[t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const float v = warp_sum(acc[t]);
                    if (lane == 0) hd.red[warp][t] = v;
                }
                __syncthreads();
                if (tid < 4 * T) {
                    const int gg = tid / T, t = tid % T, jj = j0 + gg;
                    if (jj < n_my_e) {
                        const int e = c + jj * G;
                        const float sum = ((hd.red[4 * gg][t] + hd.red[4 * gg + 1][t]) + hd.red[4 * gg + 2][t]) +
                                          hd.red[4 * gg + 3][t];
                        const float v = sum + hd.bias[jj];
                        publish_b64(tag_l + (size_t)buf * tl_words + (size_t)t * E + e,
                                    tagged(tag, __float_as_uint(v)));
                        if (p.debug) p.logits[(size_t)t * E + e] = v;
                    }
                }
                if (j0 + 4 < n_my_e) __syncthreads();   // hd.red is reused by the next pass
            }
        }
        // the router rows are consumed: the next layer's start streaming now, so
        // that they have landed before this layer's h exchange (stores of the
        // exchange queue behind reads still in flight)
        if (!last && tid == 0 && !pl.g_over_wr) {
            fence_proxy_async_smem();
            issue_wr(l + 1);
        }
        stamp(p, l, 2);

        // ------------------------------------------------------------------ Q
        // (while the other CTAs are still finishing their logits)
        // the tensor scale of x from max |x| over the call (non-negative
        // floats order like their bits)
        auto x_scale = [&]() -> float {
            uint32_t am_bits = 0;
#pragma unroll 1
            for (int i = tid; i < T * H / 2; i += kThreads) {
                const uint32_t two = reinterpret_cast<const uint32_t*>(xs_bf16)[i];
                am_bits = max(am_bits, max(__float_as_uint(fabsf(bf16_to_f32(two & 0xFFFFu))),
                                           __float_as_uint(fabsf(bf16_to_f32(two >> 16)))));
            }
            am_bits = __reduce_max_sync(0xffffffffu, am_bits);
            if (lane == 0) hd.redu[warp] = am_bits;
            __syncthreads();
            // every warp reduces the 16 warp maxima itself (no second barrier)
            return tensor_scale_from_amax_bits(__reduce_max_sync(0xffffffffu, lane < kWarps ? hd.redu[lane] : 0u));
        };
        // one thread per 4 elements: E2M1 codes as f16 values + fp32 block
        // scales.  At one token, when the gate/up slots leave the x staging
        // alone, this runs after the weight copies are issued, where it hides
        // behind their latency instead of standing between the router step and
        // the logits; otherwise (the slots cover the staging) it runs here.
        // (Only the one-token kernel carries the second call site: a copy of
        // the loop per layer costs instruction fetch at eight tokens.)
        const bool late_q = T == 1 && !pl.g_over_wr;
        float s_x = late_q ? 0.0f : x_scale();
        auto quantize_x = [&]() {
#pragma unroll 1
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
                {   // four codes -> two f16x2 words: quarter (gi & 7) / 2 of segment gi / 8
                    uint32_t* d = xh + (size_t)((gi & 7) >> 1) * (T * H / 8) + (size_t)(gi >> 3) * 4 + (gi & 1) * 2;
                    *reinterpret_cast<uint2*>(d) = make_uint2(e2m1x2_to_f16x2(nib & 0xFFu), e2m1x2_to_f16x2(nib >> 8));
                }
                if ((e4 & 3) == 0) xsc[t * (H / 16) + e4 / 4] = e4m3_to_f32(S);
                if (p.debug && c == 0) {  // the call's NVFP4 activations, for inspection
                    reinterpret_cast<uint16_t*>(p.xq)[gi] = (uint16_t)nib;
                    if ((e4 & 3) == 0) p.xs[t * (H / 16) + e4 / 4] = (uint8_t)S;
                }
            }
        };
        if (!late_q) {
            quantize_x();
            if (p.debug && c == 0 && tid == 0) *p.sx = s_x;
        }

        stamp(p, l, 3);

        // ------------------------------------------------------------------ T
        if (!poll_tagged<poll_batch<T>()>(tag_l + (size_t)buf * tl_words, (int)tl_words, tag, p.err,
                                          [&](int i, uint64_t v) { reinterpret_cast<uint32_t*>(lg)[i] = (uint32_t)v; })) {
            drain(hd, ph, p.err);
            return;
        }
        stamp(p, l, 4);
        // Top-k of each token's E logits (value descending, ties to the lower
        // expert index), without sorting them:
        //  1. each warp takes the largest key of its experts (expert e lives in
        //     warp (e mod 512) / 32), per token;
        //  2. tau = the k-th largest of those warp maxima: k logits are >= tau,
        //     so every logit of the top k is too (with fewer than k warps holding
        //     experts, tau = 0 keeps every logit);
        //  3. the logits >= tau (a few times k of them) go to a candidate list;
        //  4. each candidate's rank among the candidates is its slot.
        // The result does not depend on the order of the candidate list.
        if (tid < T) hd.ccount[tid] = 0;
        {
            constexpr int kPer = (1024 + kThreads - 1) / kThreads;   // experts per thread (E <= 1024)
#pragma unroll
            for (int t = 0; t < T; ++t) {
                uint32_t m = 0;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int e = tid + i * kThreads;
                    if (e < E) m = max(m, order_key(lg[(size_t)t * E + e]));
                }
                m = __reduce_max_sync(0xffffffffu, m);
                if (lane == 0) hd.gmax[t][warp] = m;
            }
        }
        __syncthreads();
        stamp(p, l, 12);
        uint32_t tau1 = 0;   // one token: every warp's own copy of tau
        if (T == 1 || warp < T) {
            // the k-th largest of the (up to) 16 warp maxima: lane j < 16 holds
            // maximum j; its rank takes 16 independent shuffles (no chain of
            // dependent shared-memory loads)
            const int t = T == 1 ? 0 : warp;
            const int ng = E >= kThreads ? kWarps : (E + 31) / 32;   // warps holding experts
            const uint32_t g = lane < ng ? hd.gmax[t][lane] : 0u;
            int r0 = 0, r1 = 0;
#pragma unroll
            for (int j = 0; j < kWarps; j += 2) {
                const uint32_t g0 = __shfl_sync(0xffffffffu, g, j), g1 = __shfl_sync(0xffffffffu, g, j + 1);
                r0 += j < ng && (g0 > g || (g0 == g && j < lane));
                r1 += j + 1 < ng && (g1 > g || (g1 == g && j + 1 < lane));
            }
            const int rank = r0 + r1;
            if (T == 1) {
                const uint32_t m = __ballot_sync(0xffffffffu, lane < ng && rank == k - 1);
                tau1 = ng < k ? 0u : __shfl_sync(0xffffffffu, g, __ffs(m) - 1);
            } else if (ng < k) {
                if (lane == 0) hd.tau[t] = 0u;
            } else if (lane < ng && rank == k - 1) {
                hd.tau[t] = g;
            }
        }
        if (T > 1) __syncthreads();
        {
            constexpr int kPer = (1024 + kThreads - 1) / kThreads;
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const uint32_t tau = T == 1 ? tau1 : hd.tau[t];
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int e = tid + i * kThreads;
                    if (e < E) {
                        const uint32_t key = order_key(lg[(size_t)t * E + e]);
                        if (key >= tau && key != 0u) {
                            const int pos = atomicAdd(&hd.ccount[t], 1);
                            cand_k[(size_t)t * E + pos] = key;
                            cand_i[(size_t)t * E + pos] = e;
                        }
                    }
                }
            }
            __syncthreads();
            // warp t ranks the candidates of token t: up to 32 at a time, one per
            // lane, each lane's rank by independent shuffles; more candidates
            // (rare) take a loop over the list
            if (warp < T) {
                const int t = warp;
                const int nc = hd.ccount[t];
                const uint32_t* ck = cand_k + (size_t)t * E;
                const int32_t* ci = cand_i + (size_t)t * E;
                if (nc <= 32) {
                    const uint32_t key = lane < nc ? ck[lane] : 0u;
                    const int e = lane < nc ? ci[lane] : 0x7FFFFFFF;
                    int r0 = 0, r1 = 0;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const uint32_t k0 = __shfl_sync(0xffffffffu, key, j), k1 = __shfl_sync(0xffffffffu, key, j + 1);
                        const int e0 = __shfl_sync(0xffffffffu, e, j), e1 = __shfl_sync(0xffffffffu, e, j + 1);
                        r0 += k0 > key || (k0 == key && e0 < e);
                        r1 += k1 > key || (k1 == key && e1 < e);
                    }
                    const int rank = r0 + r1;
                    if (lane < nc && rank < k) {
                        hd.idx[t * k + rank] = e;
                        hd.selk[t * k + rank] = key;
                    }
                } else {
#pragma unroll 1
                    for (int c0 = lane; c0 < nc; c0 += 32) {
                        const uint32_t key = ck[c0];
                        const int e = ci[c0];
                        int r0 = 0, r1 = 0;
#pragma unroll 1
                        for (int j = 0; j + 1 < nc; j += 2) {
                            const uint32_t k0 = ck[j], k1 = ck[j + 1];
                            r0 += k0 > key || (k0 == key && ci[j] < e);
                            r1 += k1 > key || (k1 == key && ci[j + 1] < e);
                        }
                        if (nc & 1) r0 += ck[nc - 1] > key || (ck[nc - 1] == key && ci[nc - 1] < e);
                        const int rank = r0 + r1;
                        if (rank < k) {
                            hd.idx[t * k + rank] = e;
                            hd.selk[t * k + rank] = key;
                        }
                    }
                }
            }
        }
        __syncwarp();   // warp t ranked token t and takes its softmax next
        stamp(p, l, 13);
        // renormalised softmax over the kept picks, one warp per token; with the
        // route-tail skip a pick of rank >= keep whose expert is not resident is
        // dropped (expert -1, weight 0)
        if (warp < T) {
            const int t = warp;
            const uint32_t kk = lane < k ? hd.selk[t * k + lane] : 0u;
            const uint32_t u = (kk & 0x80000000u) ? (kk & 0x7FFFFFFFu) : ~kk;   // key -> value
            const float v = __uint_as_float(u);
            const float v0 = __shfl_sync(0xffffffffu, v, 0);
            const int e = lane < k ? hd.idx[t * k + lane] : 0;
            const bool kept = lane < k && (lane < keep || hd.resident[e] != 0);
            const float z = kept ? expf(v - v0) : 0.0f;
            const float sum = warp_sum(z);
            if (lane < k) {
                hd.w[t * k + lane] = kept ? __fdiv_rn(z, sum) : 0.0f;
                if (!kept) hd.idx[t * k + lane] = -1;
            }
            if (T == 1) {
                // one token: its kept picks are distinct experts, so a pick's
                // position is the number of kept picks with a lower expert
                // (independent shuffles); the active experts are the positions
                const int ke = kept ? e : 0x7FFFFFFF;
                int q0 = 0, q1 = 0;
#pragma unroll
                for (int j = 0; j < kMaxTopK; j += 2) {
                    q0 += __shfl_sync(0xffffffffu, ke, j) < ke;
                    q1 += __shfl_sync(0xffffffffu, ke, j + 1) < ke;
                }
                const int pos = q0 + q1;
                const int np1 = __popc(__ballot_sync(0xffffffffu, kept));
                if (kept) {
                    hd.perm[pos] = lane;
                    hd.inv[lane] = pos;
                    hd.pe[pos] = e;
                    hd.pair_tok[pos] = 0;
                    hd.act_e[pos] = e;
                    hd.act_off[pos] = pos;
                    hd.pair_unit[pos] = pos;
                } else if (lane < k) {
                    hd.inv[lane] = -1;
                }
                if (lane == 0) {
                    hd.act_off[np1] = np1;
                    hd.n_act = np1;
                    hd.n_pos = np1;
                }
            }
        }
        __syncthreads();
        int n_pos;
        if (T == 1) {
            n_pos = hd.n_pos;
        } else {
        int live = 0;
        if (tid < P) {  // rank of pair tid among the kept pairs in (expert, pair id) order
            const int e = hd.idx[tid];
            live = e >= 0;
            int rank = 0;
#pragma unroll 8
            for (int qq = 0; qq < P; ++qq) {
                const int eq = hd.idx[qq];
                rank += eq >= 0 && ((eq < e) || (eq == e && qq < tid));
            }
            if (live) {
                hd.perm[rank] = tid;
                hd.inv[tid] = rank;
                hd.pe[rank] = e;
                hd.pair_tok[rank] = tid / k;
            } else {
                hd.inv[tid] = -1;
            }
        }
        n_pos = __syncthreads_count(live);
        if (warp == 0) {  // active-expert list
            int base = 0;
#pragma unroll 1
            for (int r0 = 0; r0 < n_pos; r0 += 32) {
                const int r = r0 + lane;
                const bool first = r < n_pos && (r == 0 || hd.pe[r] != hd.pe[r - 1]);
                const uint32_t m = __ballot_sync(0xffffffffu, first);
                if (first) {
                    const int a_ = base + __popc(m & lt_mask);
                    hd.act_e[a_] = hd.pe[r];
                    hd.act_off[a_] = r;
                }
                if (r < n_pos) hd.pair_unit[r] = base + __popc(m & (lt_mask | (1u << lane))) - 1;
                base += __popc(m);
            }
            if (lane == 0) {
                hd.act_off[base] = n_pos;
                hd.n_act = base;
            }
        }
        __syncthreads();
        }
        stamp(p, l, 14);
        const int n_act = hd.n_act;
        const int n_items = n_act * nfb;
        // items go to CTAs in reverse order, so that the CTAs with an extra item
        // are the ones with one router row fewer
        const int cg = G - 1 - c;
        const int my_items = cg < n_items ? (n_items - 1 - cg) / G + 1 : 0;
        const int n_units = d_nrows > 0 ? n_act : 0;
        const int S_G = pl.slots_g;
        const int S_D0 = pl.slots_d;
        const int S_D = pl.slots_d_total;
        if (tid < n_pos) hd.pair_slot[tid] = (uint32_t)(d_slot_ptr(hd.pair_unit[tid] % S_D) - smem_raw);
        // thread 0: gate/up items [m_begin, m_end) of this CTA, item m into slot m % S_G
        auto issue_g = [&](int m_begin, int m_end) {
#pragma unroll 1
            for (int m = m_begin; m < m_end; ++m) {
                const int it = cg + m * G, a = it / nfb, fb = it % nfb, s = m % S_G;
                issue_item(&hd.bar[kBarG + s], gslots + (size_t)s * sg, Ly.gc, Ly.gs, Ly.uc, Ly.us,
                           (size_t)hd.act_e[a] * I + (size_t)fb * kRows, H);
                hd.pending |= 1ull << (kBarG + s);
            }
        };
        // warp 0 (all lanes): down rows [d_r0, d_r0 + d_nrows) of active experts
        // [u_begin, u_end), expert u into slot u % S_D, one lane per expert
        // (one thread issuing a wave's copies one after the other took
        // microseconds at eight tokens)
        auto issue_d_warp = [&](int u_begin, int u_end) {
            fence_proxy_async_smem();
            uint32_t mlo = 0, mhi = 0;   // pending bits of the barriers armed here
#pragma unroll 1
            for (int u = u_begin + lane; u < u_end; u += 32) {
                const int s = u % S_D, b = kBarD + s;
                issue_unit(&hd.bar[b], d_slot_ptr(s), Ly.dc, Ly.ds, (size_t)hd.act_e[u] * H + d_r0, d_nrows, I);
                if (b < 32) mlo |= 1u << b;
                else mhi |= 1u << (b - 32);
            }
            mlo = __reduce_or_sync(0xffffffffu, mlo);
            mhi = __reduce_or_sync(0xffffffffu, mhi);
            if (lane == 0) hd.pending |= ((uint64_t)mhi << 32) | mlo;
        };
        // When all of the CTA's gate/up items (down units) fit in the slots at
        // once, their copies complete on one mbarrier armed with the total, so
        // one wait covers them all.
        const bool batch_g = my_items <= S_G, batch_d = n_units <= S_D0;
        if (warp == 0) {
            // the candidates and x staging are dead: the weight streams start,
            // one lane per gate/up item here, one lane per down unit in warp 1
            fence_proxy_async_smem();
            const int ni = min(my_items, S_G);
            if (batch_g && lane == 0 && ni > 0) mbar_arrive_expect_tx(&hd.bar[kBarG], (uint32_t)ni * sg);
            __syncwarp();
            if (lane < ni) {
                const int it = cg + lane * G, a = it / nfb, fb = it % nfb;
                issue_item(&hd.bar[kBarG + (batch_g ? 0 : lane)], gslots + (size_t)lane * sg, Ly.gc, Ly.gs,
                           Ly.uc, Ly.us, (size_t)hd.act_e[a] * I + (size_t)fb * kRows, H, !batch_g);
            }
            __syncwarp();
            if (lane == 0 && ni > 0)
                atomicOr(reinterpret_cast<unsigned long long*>(&hd.pending),
                         batch_g ? 1ull << kBarG : (((1ull << ni) - 1ull) << kBarG));
            stamp(p, l, 15);
        }
        // warp 1: the down rows of the active experts, one lane per unit.  At
        // one token they are issued once the gate/up rows have landed, so that
        // they do not share the HBM stream the gate/up wait depends on (the
        // down step is ≥ 3 us away); otherwise here.
        auto issue_down_first = [&]() {
            fence_proxy_async_smem();
            const int nu = min(n_units, S_D0);
            if (batch_d && lane == 0 && nu > 0)
                mbar_arrive_expect_tx(&hd.bar[kBarD], (uint32_t)nu * (uint32_t)(d_nrows * (I / 2 + I / 16)));
            __syncwarp();
            if (lane < nu)
                issue_unit(&hd.bar[kBarD + (batch_d ? 0 : lane)], d_slot_ptr(lane), Ly.dc, Ly.ds,
                           (size_t)hd.act_e[lane] * H + d_r0, d_nrows, I, !batch_d);
            __syncwarp();
            if (lane == 0 && nu > 0)
                atomicOr(reinterpret_cast<unsigned long long*>(&hd.pending),
                         batch_d ? 1ull << kBarD : (((1ull << nu) - 1ull) << kBarD));
        };
        const bool late_d = T == 1 && my_items > 0;
        if (warp == 1 && !late_d) issue_down_first();
        if (!last && tid >= 32 && tid < 32 + 4 * 32) {  // next layer's small arrays -> L2
            const DecodeLayer& Ln = p.layer[l + 1];
            const int which = (tid - 32) / 32, line = (tid - 32) % 32;
            const float* arr = which == 0 ? Ln.bias : which == 1 ? Ln.gts : which == 2 ? Ln.uts : Ln.dts;
            if (arr && line * 32 < E) prefetch_line_l2(arr + line * 32);
        }
        if constexpr (T == 1) {
            if (late_q) {   // the scale and the codes of x, behind the copies' latency
                s_x = x_scale();
                quantize_x();
                if (p.debug && c == 0 && tid == 0) *p.sx = s_x;
            }
        }
        if (tid >= kThreads - n_act) {  // output scales of the active experts (last warps)
            const int a = tid - (kThreads - n_act), e = hd.act_e[a];
            hd.act_gs[a] = __fmul_rn(__fmul_rn(__ldg(Ly.gts + e), s_x), 0.25f);
            hd.act_us[a] = __fmul_rn(__fmul_rn(__ldg(Ly.uts + e), s_x), 0.25f);
            hd.act_ds[a] = __fmul_rn(__fmul_rn(__ldg(Ly.dts + e), p.h_scale), 0.25f);
        }
        // the first gate/up wait ends in a CTA barrier that publishes the
        // above; a CTA without gate/up items needs its own
        if (my_items == 0) __syncthreads();
        stamp(p, l, 5);

        // ------------------------------------------------------------------ G
        {
            const int W = my_items <= S_G ? my_items : (S_G / 2 > 0 ? S_G / 2 : 1);
            const int half = lane >> 4, hl = lane & 15;
            // warp 0: the items of the wave from m0 (nw of them), one lane each
            // (active expert, feature block, first position, slot), and the
            // wave's (item, pair) task list
            auto build_wave = [&](int m0, int nw) {
                if (warp == 0) {
                    int np = 0, r0 = 0;
                    if (lane < nw) {
                        const int it = cg + (m0 + lane) * G, a = it / nfb;
                        r0 = hd.act_off[a];
                        np = hd.act_off[a + 1] - r0;
                        hd.it_a[lane] = a;
                        hd.it_fb[lane] = it - a * nfb;
                        hd.it_r0[lane] = r0;
                        hd.it_slot[lane] = (uint32_t)((m0 + lane) % S_G) * sg;
                    }
                    int incl = np;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int v = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += v;
                    }
                    for (int j = 0; j < np; ++j) {
                        hd.wt_i[incl - np + j] = (int16_t)lane;
                        hd.wt_r[incl - np + j] = (int16_t)(r0 + j);
                    }
                    if (lane == 31) hd.n_wt = incl;
                }
            };
            if (my_items > 0) build_wave(0, min(W, my_items));
#pragma unroll 1
            for (int m0 = 0; m0 < my_items; m0 += W) {
                const int nw = min(W, my_items - m0);
                // the wait ends in a CTA barrier, which also publishes the task list
                if (!(batch_g ? wait_bars(kBarG, 0, 1, 1) : wait_bars(kBarG, m0, nw, S_G))) return;
                if (m0 == 0) stamp(p, l, 6);
                if constexpr (T == 1) {
                    if (m0 == 0 && warp == 1 && late_d) issue_down_first();
                }
                const int n_wt = hd.n_wt;
                // warp f computes feature f of every task, up to four tasks at a
                // time (independent dot products in flight), lanes split H
                {
                    const int f = warp;
#pragma unroll 1
                    for (int t0 = 0; t0 < n_wt; t0 += 4) {
                        float ga[4], ua[4];
                        int tok[4];
                        const uint8_t* wrow[4];
                        const int nq = min(4, n_wt - t0);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int tq = min(t0 + q, n_wt - 1);
                            tok[q] = T == 1 ? 0 : hd.pair_tok[hd.wt_r[tq]];   // one token: x loads shared
                            wrow[q] = gslots + hd.it_slot[hd.wt_i[tq]];
                            ga[q] = 0.0f;
                            ua[q] = 0.0f;
                        }
#pragma unroll 1
                        for (int seg = lane; seg < nseg_h; seg += 32) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                if (q >= nq) break;   // warp-uniform
                                uint32_t x[16];
                                read_seg16h(xh + ((size_t)tok[q] * (H / 32) + seg) * 4, (size_t)T * H / 8, x);
                                const float2 xs2 = *reinterpret_cast<const float2*>(xsc + tok[q] * (H / 16) + 2 * seg);
                                const uint8_t* sl = wrow[q];
                                const uint4 wg = *reinterpret_cast<const uint4*>(sl + (size_t)f * (H / 2) + seg * 16);
                                const uint4 wu = *reinterpret_cast<const uint4*>(sl + g_codes + g_scales + (size_t)f * (H / 2) + seg * 16);
                                const uint32_t sgw = *reinterpret_cast<const uint16_t*>(sl + g_codes + (size_t)f * (H / 16) + seg * 2);
                                const uint32_t suw = *reinterpret_cast<const uint16_t*>(sl + 2 * g_codes + g_scales + (size_t)f * (H / 16) + seg * 2);
                                ga[q] += dot_seg32_h(wg, sgw, x, xs2);
                                ua[q] += dot_seg32_h(wu, suw, x, xs2);
                            }
                        }
                        float v8[8];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            v8[q] = ga[q];
                            v8[4 + q] = ua[q];
                        }
                        // gate sum of task q in lane 8 (q >> 1) + 4 (q & 1), up sum 16 lanes on
                        const float tot = warp_sum8(v8, lane);
                        const int src = 8 * ((lane & 3) >> 1) + 4 * (lane & 1);
                        const float gq = __shfl_sync(0xffffffffu, tot, src);
                        const float uq = __shfl_sync(0xffffffffu, tot, src + 16);
                        if (lane < nq) {
                            const float g = gq, u = uq;
                            const int tq = t0 + lane, i = hd.wt_i[tq], a = hd.it_a[i];
                            hd.hbuf[i][hd.wt_r[tq] - hd.it_r0[i]][f] =
                                __fmul_rn(silu(__fmul_rn(g, hd.act_gs[a])), __fmul_rn(u, hd.act_us[a]));
                        }
                    }
                }
                __syncthreads();  // wave consumed, hbuf complete
                if (tid == 0 && m0 + S_G < my_items) {
                    fence_proxy_async_smem();
                    issue_g(m0 + S_G, min(my_items, m0 + nw + S_G));
                }
                // Q on each 16-feature block: one half-warp per (item, pair)
                // task; the loop base is warp-uniform so both halves run every shuffle
#pragma unroll 1
                for (int base = 2 * warp; base < n_wt; base += 2 * kWarps) {
                    const int tq = base + half;
                    const bool valid = tq < n_wt;
                    const int i = valid ? hd.wt_i[tq] : 0;
                    const int r = valid ? hd.wt_r[tq] : hd.it_r0[0];
                    const int fb = hd.it_fb[i], pr = r - hd.it_r0[i];
                    const float hv = valid ? hd.hbuf[i][pr][hl] : 0.0f;
                    float am = fabsf(hv);
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
                    const uint32_t Sh = e4m3_rn_satfinite(__fdiv_rn(am, __fmul_rn(6.0f, p.h_scale)));
                    uint32_t code = 0;
                    if (Sh != 0) code = e2m1_one(__fdiv_rn(hv, __fmul_rn(e4m3_to_f32(Sh), p.h_scale)));
                    // lanes 0-7 of the half gather codes 0-7, lanes 8-15 codes 8-15
                    uint32_t wv = code << (4 * (hl & 7));
                    wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
                    wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
                    wv |= __shfl_xor_sync(0xffffffffu, wv, 4);
                    const uint32_t whi = __shfl_down_sync(0xffffffffu, wv, 8);   // codes 8-15 to lane 0 of the half
                    if (valid && hl == 0) {
                        // the block's 16 codes and scale as two tagged words:
                        // codes 0-11 | codes 12-15, scale
                        const uint64_t codes = (uint64_t)wv | ((uint64_t)whi << 32);
                        uint64_t* th = tag_h + (size_t)buf * th_words + ((size_t)r * nb_i + fb) * 2;
                        publish_b64(th, tagged(tag, codes & 0xFFFFFFFFFFFFull));
                        publish_b64(th + 1, tagged(tag, (codes >> 48) | ((uint64_t)Sh << 16)));
                        if (p.debug) {
                            *reinterpret_cast<uint2*>(p.hq + (size_t)r * (I / 2) + fb * 8) = make_uint2(wv, whi);
                            p.hs[(size_t)r * nb_i + fb] = (uint8_t)Sh;
                        }
                    }
                }
                if (m0 + W < my_items) {
                    __syncthreads();  // hbuf and the task list read before the next wave's
                    build_wave(m0 + W, min(W, my_items - m0 - W));
                }
            }
        }
        // the gate/up area is free: down rows beyond the down area stream into it
        if (warp == 0 && n_units > S_D0) issue_d_warp(S_D0, min(n_units, S_D));
        if (tid == 0 && !last && pl.g_over_wr) {   // the router rows were gate/up slots
            fence_proxy_async_smem();
            issue_wr(l + 1);
        }
        if (p.debug && c == 0) {  // routing results, for inspection: a CTA with the fewest items,
                           // after its gate/up work, while it would wait for h anyway
            if (tid < P) {
                p.idx[tid] = hd.idx[tid];
                p.w[tid] = hd.w[tid];
                if (tid < n_pos) p.perm[tid] = hd.perm[tid];
                p.inv[tid] = hd.inv[tid];
            }
#pragma unroll 1
            for (int e = tid; e <= E; e += kThreads) {
                int below = 0, at = 0;
#pragma unroll 8
                for (int qq = 0; qq < P; ++qq) {
                    const int eq = hd.idx[qq];
                    below += eq >= 0 && eq < e;
                    at += eq == e;
                }
                if (e < E) p.counts[e] = at;
                p.offsets[e] = below;
            }
        }
        stamp(p, l, 7);

        // ------------------------------------------------------------------ D
        if (n_units > 0) {
            // h of every pair -> int8 + block scales in area a
            if (!poll_tagged<poll_batch<T>()>(tag_h + (size_t)buf * th_words, n_pos * nb_i * 2, tag, p.err,
                                              [&](int i, uint64_t v) {
                                                  // block blk = r * I/16 + b: quarters 2 (b & 1)
                                                  // and 2 (b & 1) + 1 of segment blk / 2
                                                  const int blk = i >> 1;
                                                  uint32_t* d = hh + (size_t)((blk & 1) * 2) * (P * I / 8) + (size_t)(blk >> 1) * 4;
                                                  uint32_t* d1 = d + (size_t)P * I / 8;
                                                  if ((i & 1) == 0) {        // codes 0-11
                                                      uint32_t f[4];
                                                      e2m1x8_to_f16x2x4((uint32_t)v, f);
                                                      *reinterpret_cast<uint4*>(d) = make_uint4(f[0], f[1], f[2], f[3]);
                                                      *reinterpret_cast<uint2*>(d1) =
                                                          make_uint2(e2m1x2_to_f16x2((uint32_t)(v >> 32) & 0xFFu),
                                                                     e2m1x2_to_f16x2((uint32_t)(v >> 40) & 0xFFu));
                                                  } else {                   // codes 12-15, scale
                                                      *reinterpret_cast<uint2*>(d1 + 2) =
                                                          make_uint2(e2m1x2_to_f16x2((uint32_t)v & 0xFFu),
                                                                     e2m1x2_to_f16x2((uint32_t)(v >> 8) & 0xFFu));
                                                      hsc[blk] = e4m3_to_f32((uint32_t)(v >> 16) & 0xFFu);
                                                  }
                                              })) {
                drain(hd, ph, p.err);
                return;
            }
            stamp(p, l, 8);
            const int W = n_units <= S_D ? n_units : S_D / 2;
            const int half = lane >> 4, hl = lane & 15;
#pragma unroll 1
            for (int u0 = 0; u0 < n_units; u0 += W) {
                const int nw = min(W, n_units - u0);
                if (!(batch_d ? wait_bars(kBarD, 0, 1, 1) : wait_bars(kBarD, u0, nw, S_D))) return;
                if (u0 == 0) stamp(p, l, 9);
                // the wave's pairs are the expert-grouped positions [rb0, rb1); warp =
                // output row, half-warps take pairs, up to eight pairs each in flight
                const int rb0 = hd.act_off[u0], rb1 = hd.act_off[u0 + nw];
#pragma unroll 1
                for (int row = warp; row < d_nrows; row += kWarps) {
#pragma unroll 1
                    for (int rb = rb0; rb < rb1; rb += 16) {
                        float acc[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int r = rb + 2 * q + half;
                            acc[q] = 0.0f;
                            if (r < rb1) {
                                const uint8_t* slot = smem_raw + hd.pair_slot[r];
                                const uint8_t* drow = slot + (size_t)row * (I / 2);
                                const uint8_t* dsc = slot + d_codes + (size_t)row * (I / 16);
#pragma unroll 1
                                for (int seg = hl; seg < nseg_i; seg += 16) {
                                    uint32_t x[16];
                                    read_seg16h(hh + ((size_t)r * (I / 32) + seg) * 4, (size_t)P * I / 8, x);
                                    const float2 hs2 = *reinterpret_cast<const float2*>(hsc + r * nb_i + 2 * seg);
                                    const uint4 wd = *reinterpret_cast<const uint4*>(drow + seg * 16);
                                    const uint32_t sdw = *reinterpret_cast<const uint16_t*>(dsc + seg * 2);
                                    acc[q] += dot_seg32_h(wd, sdw, x, hs2);
                                }
                            }
                        }
                        const float tot = half_warp_sum8(acc, hl);
                        if ((hl & 1) == 0) {   // lanes 2q and 2q + 1 hold pair q's total
                            const int r = rb + 2 * (hl >> 1) + half;
                            if (r < rb1) obuf[(size_t)r * d_rows + row] = __fmul_rn(tot, hd.act_ds[hd.pair_unit[r]]);
                        }
                    }
                }
                __syncthreads();  // wave consumed
                if (warp == 0 && u0 + S_D < n_units) issue_d_warp(u0 + S_D, min(n_units, u0 + nw + S_D));
            }
            stamp(p, l, 10);
            // combine in slot order, residual; tagged x of the next layer or the output
#pragma unroll 1
            for (int i = tid; i < T * my_pairs; i += kThreads) {
                const int t = i / my_pairs, pp = i % my_pairs, j0 = 2 * pp;
                // slot order; a pick the route-tail skip dropped has no position.
                // All loads first, then the chain of FMAs.
                int pos[kMaxTopK];
                float wj[kMaxTopK];
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j) {
                    pos[j] = j < k ? hd.inv[t * k + j] : -1;
                    wj[j] = j < k ? hd.w[t * k + j] : 0.0f;
                }
                float2 o[kMaxTopK];
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    o[j] = pos[j] >= 0 ? *reinterpret_cast<const float2*>(obuf + (size_t)pos[j] * d_rows + j0)
                                       : make_float2(0.f, 0.f);
                float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j) {
                    if (pos[j] >= 0) {
                        y0 = fmaf(wj[j], o[j].x, y0);
                        y1 = fmaf(wj[j], o[j].y, y1);
                    }
                }
                const size_t off = (size_t)t * H + d_r0 + j0;
                if (Ly.y) *reinterpret_cast<float2*>(Ly.y + off) = make_float2(y0, y1);
                if (l > 0 || p.residual0) {
                    const uint32_t b0 = f32_to_bf16_rn(bf16_to_f32(hd.res[t][j0]) + y0);
                    const uint32_t b1 = f32_to_bf16_rn(bf16_to_f32(hd.res[t][j0 + 1]) + y1);
                    const uint32_t word = b0 | (b1 << 16);
                    if (!last) {
                        publish_b64(tag_x + (size_t)buf * tx_words + (size_t)t * (H / 2) + d_r0 / 2 + pp,
                                    tagged(tag, word));
                    }
                    else if (p.x_out)
                        *reinterpret_cast<uint32_t*>(p.x_out + off) = word;
                }
            }
            __syncthreads();  // obuf and res read before the next layer reuses them
        }
        stamp(p, l, 11);
    }
}

// Self-test of the bounded waits: the same tagged-word poll the decode kernel
// uses, on words that nothing writes, then the same mbarrier wait on a barrier
// that nothing arrives on.  Each must run out and report kDevErrTimeout
// (err[0]: the poll, err[1]: the mbarrier); nothing is left in flight.
__global__ void __launch_bounds__(kThreads, 1) k_selftest_waits(const uint64_t* words, int n,
                                                                 uint32_t* err) {
    __shared__ uint64_t bar;
    poll_tagged<2>(words, n, 1u, err, [](int, uint64_t) {});
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0)) atomicOr(err + 1, kDevErrTimeout);
    }
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int sm_count() {
    static int cached_dev = -1, cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev != cached_dev) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached = n;
        cached_dev = dev;
    }
    return cached;
}

template <int T>
cudaError_t launch_t(const DecodeParams& prm, cudaStream_t st) {
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(k_decode<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kDecodeSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sm_count());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kDecodeSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_decode<T>, prm);
    count_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_selftest_waits(const uint64_t* words, int n, uint32_t* err, cudaStream_t st) {
    k_selftest_waits<<<1, kThreads, 0, st>>>(words, n, err);
    count_launches(1);
    return cudaGetLastError();
}

size_t decode_tag_bytes(const Shape& s, int T) {
    const size_t P = (size_t)T * s.k;
    return 2 * ((size_t)T * s.E + P * (s.I / 16) * 2 + (size_t)T * (s.H / 2)) * sizeof(uint64_t);
}

DecodeSmemPlan decode_smem_plan(const Shape& s, int T, int grid) {
    DecodeSmemPlan pl{};
    if (grid < 1 || T < 1 || T > kDecodeMaxTokens) return pl;
    const size_t P = (size_t)T * s.k;
    const size_t head = align_up(sizeof(Head), 1024);
    pl.wr_rows = (s.E + grid - 1) / grid;
    const int npr = s.H / 2;
    pl.d_rows = 2 * ((npr + grid - 1) / grid);
    if (pl.wr_rows > kMaxWrRows || pl.d_rows > kMaxDRows) return pl;
    const size_t wr = align_up((size_t)pl.wr_rows * s.H * 4, 1024);
    const size_t a_x = (size_t)T * s.H * 2 + (size_t)T * (s.H / 16) * 4 + (size_t)T * s.H * 2;
    const size_t a_h = P * s.I * 2 + P * (s.I / 16) * 4 + P * pl.d_rows * 4;
    const size_t a = align_up(a_x > a_h ? a_x : a_h, 1024);
    if (head + wr + a >= kDecodeSmemBytes) return pl;
    const size_t ring = kDecodeSmemBytes - head - wr - a;
    // T step scratch: logits [T][E] and the candidate keys and indices [T][E] each
    const size_t scratch = align_up((size_t)T * s.E, 4) * 4 + (size_t)T * s.E * 8;
    if (scratch > ring || s.E > 1024) return pl;
    const size_t sg = 2 * ((size_t)kRows * s.H / 2 + (size_t)kRows * s.H / 16);
    const size_t sd = (size_t)pl.d_rows * (s.I / 2 + s.I / 16);
    const size_t units_max = P < (size_t)s.E ? P : (size_t)s.E;
    const size_t items_max = (units_max * (s.I / kRows) + grid - 1) / grid;
    const size_t min_d = units_max < 4 ? units_max : 4;
    // layout: head | area a | router rows | ring.  Gate/up slots start at the
    // ring; when the CTA has more items than fit there, they start instead at
    // the bf16 staging of x in area a (dead once x is quantised) and run over
    // the router rows (whose next layer's copies then wait for gate/up to end).
    const size_t a_off = head, wr_off = head + a, ring_off = head + a + wr;
    const size_t end = kDecodeSmemBytes;
    const size_t x_live = (size_t)T * s.H * 2 + (size_t)T * (s.H / 16) * 4;   // f16 x + scales
    if (end - ring_off < sg + min_d * sd) return pl;
    auto slots_in = [&](size_t from) {
        size_t n = (end - min_d * sd - from) / sg;
        if (n > items_max) n = items_max;
        if (n > (size_t)kMaxSlotsG) n = kMaxSlotsG;
        return n;
    };
    size_t g_off = ring_off;
    size_t n_g = slots_in(ring_off);
    bool over = false;
    const size_t g_ext = align_up(a_off + x_live, 128);
    if (n_g < items_max && slots_in(g_ext) > n_g) {
        g_off = g_ext;
        n_g = slots_in(g_ext);
        over = true;
    }
    if (n_g < 1) return pl;
    // down slots after the gate/up slots, never below the ring (area a holds h
    // and the router rows the next layer's copies while the down step runs)
    size_t d_area_off = align_up(g_off + n_g * sg, 128);
    if (d_area_off < ring_off) d_area_off = ring_off;
    size_t n_d = (end - d_area_off) / sd;
    if (n_d > units_max) n_d = units_max;
    if (n_d > (size_t)kMaxSlotsDArea) n_d = kMaxSlotsDArea;
    if (n_d < 1) return pl;
    // once gate/up is done, more down slots in the ring below the down area
    size_t n_d_total = n_d + (d_area_off - ring_off) / sd;
    if (n_d_total > (size_t)kMaxSlotsD) n_d_total = kMaxSlotsD;
    pl.ok = true;
    pl.a_off = (uint32_t)a_off;
    pl.wr_off = (uint32_t)wr_off;
    pl.ring_off = (uint32_t)ring_off;
    pl.g_off = (uint32_t)g_off;
    pl.d_area_off = (uint32_t)d_area_off;
    pl.g_over_wr = over;
    pl.slots_g = (int)n_g;
    pl.slots_d = (int)n_d;
    pl.slots_d_total = (int)n_d_total;
    pl.bytes = kDecodeSmemBytes;
    return pl;
}

bool decode_supported(const Shape& s, int T) {
    if (T < 1 || T > kDecodeMaxTokens || T * s.k > kDecodeMaxPairs) return false;
    if (s.E > 1024 || s.k > 16 || s.I % 128 != 0 || s.H % 64 != 0) return false;
    return decode_smem_plan(s, T, sm_count()).ok;
}

cudaError_t launch_decode(DecodeParams& prm, cudaStream_t st) {
    const Shape s{prm.H, prm.E, prm.k, prm.I};
    if (prm.L < 1 || prm.L > kDecodeMaxLayers) return cudaErrorInvalidValue;
    if (prm.L > 1 && !prm.residual0) return cudaErrorInvalidValue;  // layers > 0 need x
    prm.plan = decode_smem_plan(s, prm.T, sm_count());
    if (!prm.plan.ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(prm.tags, 0, decode_tag_bytes(s, prm.T), st);
    if (e != cudaSuccess) return e;
    switch (prm.T) {
        case 1: return launch_t<1>(prm, st);
        case 2: return launch_t<2>(prm, st);
        case 3: return launch_t<3>(prm, st);
        case 4: return launch_t<4>(prm, st);
        case 5: return launch_t<5>(prm, st);
        case 6: return launch_t<6>(prm, st);
        case 7: return launch_t<7>(prm, st);
        case 8: return launch_t<8>(prm, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
