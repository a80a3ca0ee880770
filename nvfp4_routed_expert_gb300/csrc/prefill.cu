// Prefill path (more than 8 tokens): S5 and S6 as block-scaled FP4 grouped
// GEMMs on the tensor cores (tcgen05.mma kind::mxf4nvf4, scale_vec::4X: one
// E4M3 scale per 16 elements, fp32 accumulators in tensor memory).
//
// The grouped GEMM is the one dense contraction of the layer: every expert e
// multiplies the rows routed to it (m_e of them, expert-grouped order from S4)
// by its weights.  Work items are (128-row M-tile of one expert, N-tile); the
// tile list is built on the device from the expert offsets.
//
//   gate/up  A = x_hat rows gathered by token        [128 x H]   (NVFP4)
//            B = [128 gate rows ; 128 up rows] of e   [256 x H]   (NVFP4)
//            epilogue: h = silu(g) * u, Q(h; s_h) -> hq/hs rows (expert order)
//   down     A = h_hat rows (contiguous, expert order) [128 x I]
//            B = 256 down rows of e                    [256 x I]
//            epilogue: w_pair * o as fp16 partials per pair
//   combine  y[t] = sum_j partial[inv(t, j)] in slot order (+ residual)
//
// One persistent CTA per SM, warp-specialised:
//   warps 0-3   producers: TMA tiles into 128B-swizzled shared-memory stages
//               (thread 0), plus, in gate/up, the A rows gathered by token
//               with cp.async (eight lanes per 128-byte row); block scales
//               come as 2 KB tiles in a lane-major layout (below)
//   warps 4-11  epilogue: tcgen05.ld of the accumulator (lane = tile row)
//   warps 12-15 block scales: once a stage has landed, warp 12 + j writes
//               its scales from shared memory into lane quarter j of the
//               stage's scale columns (tcgen05.st)
//   warp 16     MMA issue (one thread), tcgen05.commit to mbarriers
//
// Tiled block-scale layout: for every 128 rows (group g) and every 256
// elements of K (stage kb) one 2048-byte chunk at ((g * K/256) + kb) * 2048:
// four k-steps of 512 bytes, each [32 lanes i][4 row quarters j][4 bytes],
// the 4 bytes being the scales of row 128 g + 32 j + i for the k-step's 64
// elements.  Lane i's 16 bytes of a k-step are the four scale columns the
// block-scaled MMA reads in lane i of every lane quarter (row 32 j + i in
// column j), so each scale warp stores them with one 16-byte shared load per
// k-step.  Weight scales are tiled once when the layer is created; the gate/up
// epilogue writes h's scales tiled per M-tile for the down GEMM; gate/up
// gathers x's scales into the layout with 4-byte cp.async copies.
//
// Every wait is bounded; a wait that runs out records the error, makes the
// other roles leave their loops, and the CTA frees its tensor memory after
// its last MMA has completed.
#include "common.cuh"
#include "kernels.h"
#include "prefill.h"
#include "sync.cuh"

namespace moe {

namespace {

constexpr int kStages = 4;
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kStageK = 256;                        // elements of K per stage (128 bytes per row)
constexpr int kABytes = kTileM * kStageK / 2;       // 16 KB
constexpr int kBBytes = kTileN * kStageK / 2;       // 32 KB
constexpr int kSfABytes = kTileM * 16;              // 2 KB: 16 scale bytes per row per stage
constexpr int kSfBBytes = kTileN * 16;              // 4 KB
constexpr int kSfChunk = 2048;                      // one 128-row group, one stage, tiled
constexpr int kStageBytes = kABytes + kBBytes + kSfABytes + kSfBBytes;
constexpr int kProducers = 128, kEpilogue = 256;   // epilogue: two warps per lane quarter
constexpr int kSfWarp0 = 4 + kEpilogue / 32;       // four scale warps, one per lane quarter
constexpr int kMmaWarp = kSfWarp0 + 4;
constexpr int kThreads = 32 * (kMmaWarp + 1);
static_assert(kSfWarp0 % 4 == 0, "scale warp j must own lane quarter j");
// tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kTileN;               // fp32 accumulator 128 lanes x 256
constexpr uint32_t kSfColsPerStage = 48;            // SFA 4 k-steps x 4 + SFB 4 x 8
constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024;
// The down GEMM (two k-stages per tile) runs with three stages and uses the
// fourth stage's space to stage its fp16 output: 4 KB per epilogue warp.
constexpr int kDownStages = 3;
constexpr int kStageOutBytes = 32 * 128;            // 32 rows x 64 fp16, 128-byte swizzled
static_assert(kDownStages * kStageBytes + 8 * kStageOutBytes <= kStages * kStageBytes, "down staging");

struct alignas(8) Bars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t sf_full[kStages];  // the stage's scales are in tensor memory (FP4 modes)
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t mma_done;
    uint32_t tmem_base;
    volatile uint32_t abort;
};

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;                 // leading offset (not used for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                 // descriptor version
    d |= (uint64_t)2 << 61;                 // 128-byte swizzle
    return d;
}

// E2M1 x E2M1, fp32 accumulate, UE4M3 scales, M = 128, N = 256, K-major A and B
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kTileN >> 3) << 17) |
                            ((uint32_t)(kTileM >> 4) << 24);
// BF16 x BF16 -> fp32 (kind::f16), M = 128, N = 256, K-major A and B
constexpr uint32_t kIdescBf16 = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(kTileN >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);

__device__ __forceinline__ void mma_fp4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t sfa,
                                        uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::
            "r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdescBf16), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 / 32 consecutive columns of this warp's 32 lanes from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 32 consecutive columns of this warp's 32 lanes; tmem_wait_ld makes them usable
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars& b, uint32_t* err) {
    for (uint32_t i = 0; i < kMbarSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && b.abort) return false;
        if (i > 1024) __nanosleep(64);
    }
    atomicOr(err, kDevErrTimeout);
    b.abort = 1;
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive on the phase and arm it with `bytes` of expected transactions.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size a multiple of
// 16), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// TMA tile load of the tensor map's box at (x, y) into shared memory,
// completing on `bar` (x in elements, a multiple of 16 bytes).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// TMA tile store of the tensor map's box at (x, y) from shared memory (x in
// elements, a multiple of 16 bytes; the box must lie inside the tensor), as
// one bulk group of this thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// 16-byte asynchronous copy global -> shared (zero fill when !valid); the
// thread's copies are tracked by cp_async_arrive.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

// Arrive on `bar` once all of this thread's earlier cp.async copies have landed
// (the arrival is one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One block of 16 h features of one row from its gate and up accumulators:
// h = silu(g f0) * (u f1) and its Q with the static scale s (the scale code is
// returned, the 16 nibbles written to codes).  The epilogue's arithmetic is
// kept short: silu takes an approximate reciprocal of 1 + e^-z, with e^-z
// computed as 2^(-z log2 e) by the approximate base-2 exponential (the
// exponent capped at e^80, where silu is below 1e-33 either way; relative
// error of e^-z about (2 + |z|) 2^-24, the |z| part from rounding z log2 e,
// and at most that in silu), and f1 is applied to
// the block maximum and folded into the one per-block factor the elements are
// multiplied by, instead of a division per element.  Each quotient is within a
// few ulp of the correctly rounded evaluation, so a code can differ from it
// only for a value at a rounding boundary.
__device__ __forceinline__ uint32_t swiglu_quant16(const uint32_t* g, const uint32_t* u, float f0, float f1,
                                                   float s, uint2& codes) {
    float h[16];
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float z = __fmul_rn(__uint_as_float(g[i]), f0);
        float e;   // e^-z = 2^(-z log2 e), on the MUFU
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(__fmul_rn(fminf(-z, 80.0f), 1.4426950408889634f)));
        const float d = 1.0f + e;
        float y;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(d));
        h[i] = __fmul_rn(__fmul_rn(z, y), __uint_as_float(u[i]));
        a = fmaxf(a, fabsf(h[i]));
    }
    const uint32_t S = e4m3_rn_satfinite(__fdiv_rn(__fmul_rn(a, f1), __fmul_rn(6.0f, s)));
    if (S == 0) {
        codes = make_uint2(0u, 0u);
        return 0u;
    }
    const float c = __fdiv_rn(f1, __fmul_rn(e4m3_to_f32(S), s));
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = __fmul_rn(h[i], c);
    codes.x = e2m1x8_rn_satfinite(t);
    codes.y = e2m1x8_rn_satfinite(t + 8);
    return S;
}

template <GemmMode kMode>
__global__ void __launch_bounds__(kThreads, 1) k_grouped_gemm(const __grid_constant__ GemmParams p) {
    constexpr bool kGateUp = kMode == GemmMode::kGateUp;
    constexpr bool kRouter = kMode == GemmMode::kRouter;
    constexpr bool kDown = kMode == GemmMode::kDown;
    constexpr int nst = kMode == GemmMode::kDown ? kDownStages : kStages;   // pipeline stages
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ Bars bars;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = p.K;                              // contraction length (H or I)
    // stages of 128 bytes per row: 256 FP4 elements, or 64 bf16 elements for
    // the router, whose K loop runs over Wr's hi part and then its lo part
    const int kstages = kRouter ? 2 * (K / 64) : K / kStageK;
    const int n_tiles_n = kRouter ? (p.E + kTileN - 1) / kTileN
                                  : p.N_total / (kGateUp ? kTileN / 2 : kTileN);
    const uint32_t n_mtiles = kRouter ? (uint32_t)((p.T + kTileM - 1) / kTileM) : *p.n_mtiles;
    const uint32_t n_work = n_mtiles * (uint32_t)n_tiles_n;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            // thread 0 arrives once per stage (arming the TMA and bulk bytes);
            // in gate/up every producer also arrives, asynchronously, when
            // its gathered A row and scales have landed
            mbar_init(&bars.full[s], kGateUp ? kProducers + 1 : 1);
            mbar_init(&bars.empty[s], 1);
            mbar_init(&bars.sf_full[s], 128);
        }
        mbar_init(&bars.acc_full, 1);
        mbar_init(&bars.acc_empty, kEpilogue);
        mbar_init(&bars.mma_done, 1);
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp < 4) {
        // ------------------------------------------------------------ producers
        // Thread 0 issues the TMA tiles and bulk scale copies; in gate/up every
        // producer thread also takes part in gathering the A rows by token.
        if (kGateUp || tid == 0) {
            uint32_t it = 0;
            const int kbs = K / kStageK;                // stages of one tile (FP4 modes)
            for (uint32_t w = blockIdx.x; w < n_work && !bars.abort; w += gridDim.x) {
                const int nt = (int)(w % n_tiles_n);
                const uint32_t mt = w / n_tiles_n;
                int e = 0, row0, rows;
                if (kRouter) {
                    row0 = (int)mt * kTileM;
                    rows = min(kTileM, p.T - row0);
                } else {
                    const int4 m = p.mtiles[mt];       // (expert, row0, rows, -)
                    e = m.x;
                    row0 = m.y;
                    rows = m.z;
                }
                // gate/up gathers A by token: thread tid copies 16-byte chunk tid % 8
                // of rows 16 j + tid / 8 (8 lanes per 128-byte row), and the 16
                // scale bytes of the stage (4 k-steps) of row tid
                int tok_c[8], tok_s = -1;
                if (kGateUp) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int r = 16 * j + (tid >> 3);
                        tok_c[j] = r < rows ? p.perm[row0 + r] / p.k : -1;
                    }
                    tok_s = tid < rows ? p.perm[row0 + tid] / p.k : -1;
                }
                // first B row of the tile in the tensor maps (a multiple of 128)
                const int b_row0 = kRouter ? nt * kTileN
                                           : e * p.N_total + nt * (kGateUp ? kTileN / 2 : kTileN);
                const size_t b_grp = (size_t)(b_row0 / 128);
                for (int kb = 0; kb < kstages; ++kb, ++it) {
                    const int s = (int)(it % nst);
                    const uint32_t round = it / nst;
                    if (round > 0 && !wait_or_abort(&bars.empty[s], (round - 1) & 1u, bars, p.err)) break;
                    uint8_t* sA = smem + (size_t)s * kStageBytes;
                    uint8_t* sB = sA + kABytes;
                    uint8_t* sSA = sB + kBBytes;
                    uint8_t* sSB = sSA + kSfABytes;
                    // 128 bytes of K per row per stage; the router's second half
                    // re-reads x against Wr's lo part
                    const bool lo_half = kRouter && kb >= kstages / 2;
                    const int kbyte = (kRouter ? (kb % (kstages / 2)) : kb) * 128;
                    if (tid == 0) {
                        if (kGateUp) {
                            mbar_arrive_expect_tx(&bars.full[s], (uint32_t)(kBBytes + kSfBBytes));
                            tma_load_2d(sB, &p.tm_b, kbyte, b_row0, &bars.full[s]);                 // 128 gate rows
                            tma_load_2d(sB + kBBytes / 2, &p.tm_b2, kbyte, b_row0, &bars.full[s]);  // 128 up rows
                            bulk_load(sSB, p.b_sf_tiled + (b_grp * kbs + kb) * kSfChunk, kSfChunk, &bars.full[s]);
                            bulk_load(sSB + kSfChunk, p.b2_sf_tiled + (b_grp * kbs + kb) * kSfChunk, kSfChunk,
                                      &bars.full[s]);
                        } else if (kRouter) {
                            mbar_arrive_expect_tx(&bars.full[s], (uint32_t)(kABytes + kBBytes));
                            tma_load_2d(sB, lo_half ? &p.tm_b2 : &p.tm_b, kbyte / 2, b_row0, &bars.full[s]);
                            tma_load_2d(sA, &p.tm_a, kbyte / 2, row0, &bars.full[s]);
                        } else {
                            mbar_arrive_expect_tx(&bars.full[s], (uint32_t)(kABytes + kBBytes + kSfABytes + kSfBBytes));
                            tma_load_2d(sB, &p.tm_b, kbyte, b_row0, &bars.full[s]);                 // 256 down rows
                            tma_load_2d(sA, &p.tm_a, kbyte, row0, &bars.full[s]);                   // 128 h rows
                            bulk_load(sSA, p.a_sf_tiled + ((size_t)mt * kbs + kb) * kSfChunk, kSfChunk,
                                      &bars.full[s]);
                            bulk_load(sSB, p.b_sf_tiled + (b_grp * kbs + kb) * kSfChunk, kSfChunk, &bars.full[s]);
                            bulk_load(sSB + kSfChunk, p.b_sf_tiled + ((b_grp + 1) * kbs + kb) * kSfChunk, kSfChunk,
                                      &bars.full[s]);
                        }
                    }
                    if (kGateUp) {
                        // A rows gathered by token: 16-byte chunk tid % 8 of rows
                        // 16 j + tid / 8 into the 128-byte swizzled layout, and row
                        // tid's 16 scale bytes as row tid of a row-major [128][16]
                        // block (one line per copy; the scale warps tile them);
                        // zeros past the tile's rows
                        const int c = tid & 7;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int r = 16 * j + (tid >> 3);
                            const int t = tok_c[j] < 0 ? 0 : tok_c[j];
                            cp_async16(sA + r * 128 + ((c ^ (r & 7)) << 4),
                                       p.a_codes + (size_t)t * (K / 2) + kbyte + c * 16, tok_c[j] >= 0);
                        }
                        cp_async16(sSA + tid * 16, p.a_scales + (size_t)(tok_s < 0 ? 0 : tok_s) * (K / 16) + kb * 16,
                                   tok_s >= 0);
                        cp_async_arrive(&bars.full[s]);
                    }
                }
            }
            // nothing of this thread may land after the CTA exits: its own copies,
            // and (thread 0, after an abort) the tiles of the stages it armed
            asm volatile("cp.async.wait_all;" ::: "memory");
            if (tid == 0 && bars.abort) {
                for (uint32_t i = it > (uint32_t)nst ? it - nst : 0; i < it; ++i)
                    mbar_wait(&bars.full[i % nst], (i / nst) & 1u, 1u << 20);
            }
        }
    } else if (warp < kSfWarp0) {
        // ------------------------------------------------------------- epilogue
        // warps 4-11: warp w reads lane quarter w % 4 (tile rows 32q .. 32q+31);
        // the two warps of a quarter split the tile's columns (hsel)
        const int q = warp & 3;
        const int hsel = (warp - 4) >> 2;
        const int row = 32 * q + lane;          // tile row = tensor-memory lane
        // down: a tile's M-tile entry is loaded two tiles ahead and its row
        // weight and weight tensor scale one tile ahead, so that the short
        // wait for its accumulator does not also wait on that chain of loads
        int4 dm_cur = make_int4(0, 0, 0, 0), dm_nxt = make_int4(0, 0, 0, 0);
        float dw_cur = 0.0f, dts_cur = 0.0f;
        if (kDown) {
            const uint32_t w0 = blockIdx.x, w1 = w0 + gridDim.x;
            if (w0 < n_work) {
                dm_cur = p.mtiles[w0 / n_tiles_n];
                dw_cur = row < dm_cur.z ? p.pair_w_perm[dm_cur.y + row] : 0.0f;
                dts_cur = p.b_tensor_scale[dm_cur.x];
            }
            if (w1 < n_work) dm_nxt = p.mtiles[w1 / n_tiles_n];
        }
        uint32_t tile = 0;
        for (uint32_t w = blockIdx.x; w < n_work && !bars.abort; w += gridDim.x, ++tile) {
            const int nt = (int)(w % n_tiles_n);
            const uint32_t mt = w / n_tiles_n;
            int e = 0, row0, rows;
            float dw_nxt = 0.0f, dts_nxt = 0.0f;
            int4 dm_nn = make_int4(0, 0, 0, 0);
            if (kRouter) {
                row0 = (int)mt * kTileM;
                rows = min(kTileM, p.T - row0);
            } else if (kDown) {
                e = dm_cur.x;
                row0 = dm_cur.y;
                rows = dm_cur.z;
                const uint32_t w1 = w + gridDim.x, w2 = w1 + gridDim.x;
                if (w1 < n_work) {
                    dw_nxt = row < dm_nxt.z ? p.pair_w_perm[dm_nxt.y + row] : 0.0f;
                    dts_nxt = p.b_tensor_scale[dm_nxt.x];
                }
                if (w2 < n_work) dm_nn = p.mtiles[w2 / n_tiles_n];
            } else {
                const int4 m = p.mtiles[mt];
                e = m.x;
                row0 = m.y;
                rows = m.z;
            }
            const bool valid = row < rows;
            const size_t r = (size_t)row0 + row;
            // this tile's scalar factors, loaded before the wait so their latency hides behind it
            float f0 = 0.0f, f1 = 0.0f;
            if (kGateUp) {
                f0 = __fmul_rn(p.a_tensor_scale[0], p.b_tensor_scale[e]);
                f1 = __fmul_rn(p.a_tensor_scale[0], p.b2_tensor_scale[e]);
            } else if (kDown) {
                f0 = valid ? __fmul_rn(dw_cur, __fmul_rn(p.h_scale, dts_cur)) : 0.0f;
            }
            if (!wait_or_abort(&bars.acc_full, tile & 1u, bars, p.err)) break;
            tc_fence_after();
            const uint32_t acc = tmem + ((uint32_t)(32 * q) << 16);
            if (kRouter) {
                // each 32 x 16 block goes through shared memory (the stages'
                // scale areas, unused by the router: 17-float rows, no bank
                // conflicts on the row-wise writes) so that a warp store covers
                // two 64-byte row segments instead of 32 rows
                float* tb = reinterpret_cast<float*>(smem + (size_t)((warp - 4) >> 1) * kStageBytes + kABytes +
                                                     kBBytes) + ((warp - 4) & 1) * (32 * 17);
                const int cc = lane & 15, rh = lane >> 4;
                for (int c0 = hsel * (kTileN / 2); c0 < (hsel + 1) * (kTileN / 2); c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(acc + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int e = nt * kTileN + c0 + 16 * hf + cc;
                        const float b = (p.bias && e < p.E) ? p.bias[e] : 0.0f;
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 16; ++i) tb[lane * 17 + i] = __uint_as_float(v[16 * hf + i]);
                        __syncwarp();
#pragma unroll
                        for (int m = 0; m < 16; ++m) {
                            const int rr = 2 * m + rh;   // row within the warp's 32
                            if (32 * q + rr < rows && e < p.E)
                                p.logits[((size_t)row0 + 32 * q + rr) * p.E + e] = tb[rr * 17 + cc] + b;
                        }
                    }
                }
            } else if (kGateUp) {
                // blocks b = 2 hsel, 2 hsel + 1 and 2 hsel + 4, 2 hsel + 5: two blocks per load pair,
                // stored together
                for (int bp = 0; bp < 2; ++bp) {
                    const int b0 = 2 * hsel + 4 * bp;
                    uint32_t g[32], u[32];
                    tmem_ld32(acc + 16 * b0, g);
                    tmem_ld32(acc + kTileN / 2 + 16 * b0, u);
                    tmem_wait_ld();
                    uint2 c0, c1;
                    const uint32_t S0 = swiglu_quant16(g, u, f0, f1, p.h_scale, c0);
                    const uint32_t S1 = swiglu_quant16(g + 16, u + 16, f0, f1, p.h_scale, c1);
                    const uint16_t S01 = (uint16_t)(S0 | (S1 << 8));
                    const int fb = nt * (kTileN / 32) + b0;      // first of the two blocks (even)
                    if (valid) {
                        *reinterpret_cast<uint4*>(p.out_codes + r * (p.N_total / 2) + fb * 8) =
                            make_uint4(c0.x, c0.y, c1.x, c1.y);
                        *reinterpret_cast<uint16_t*>(p.out_scales + r * (p.N_total / 16) + fb) = S01;
                    }
                    // the down GEMM's A scales, tiled per M-tile (rows past the
                    // tile's end hold the scale of a zero row: 0); blocks fb and
                    // fb + 1 are neighbours there too
                    *reinterpret_cast<uint16_t*>(p.out_sf_tiled +
                                                 ((size_t)mt * (p.N_total / kStageK) + (fb >> 4)) * kSfChunk +
                                                 ((fb >> 2) & 3) * 512 + lane * 16 + q * 4 + (fb & 3)) = S01;
                }
            } else {
                // 64 columns at a time: scale, convert to fp16, stage the warp's
                // 32 x 64 block in shared memory (128-byte rows, 16-byte chunks
                // swizzled by row: the TMA's 128-byte swizzle), then one lane
                // stores it with a TMA tile store, which runs on while the warp
                // goes on; a quarter with rows past the M-tile's end (whose
                // neighbours in the partials belong to the next M-tile) is
                // written row by row instead
                uint8_t* buf = smem + (size_t)kDownStages * kStageBytes + (size_t)(warp - 4) * kStageOutBytes;
                const bool whole = 32 * q + 32 <= rows;
                bool over = false;   // a partial that fp16 would turn into infinity
                for (int c0 = hsel * (kTileN / 2); c0 < (hsel + 1) * (kTileN / 2); c0 += 64) {
                    uint32_t o[64];
                    tmem_ld32(acc + c0, o);
                    tmem_ld32(acc + c0 + 32, o + 32);
                    tmem_wait_ld();
                    // the previous store has read the staging buffer
                    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        __half2 hv[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float v0 = __fmul_rn(__uint_as_float(o[8 * c + 2 * i]), f0);
                            const float v1 = __fmul_rn(__uint_as_float(o[8 * c + 2 * i + 1]), f0);
                            over |= fmaxf(fabsf(v0), fabsf(v1)) >= 65520.0f;
                            hv[i] = __floats2half2_rn(v0, v1);
                        }
                        *reinterpret_cast<uint4*>(buf + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                            *reinterpret_cast<uint4*>(&hv[0]);
                    }
                    if (whole) {
                        fence_proxy_async_smem();   // the staged block, to the TMA
                        __syncwarp();
                        if (lane == 0) tma_store_2d(&p.tm_out, nt * kTileN + c0, row0 + 32 * q, buf);
                    } else {
                        __syncwarp();
                        const int c = lane & 7;
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            const int rr = 4 * it + (lane >> 3);        // row within the warp's 32
                            const uint4 v = *reinterpret_cast<const uint4*>(buf + rr * 128 + ((c ^ (rr & 7)) << 4));
                            if (32 * q + rr < rows) {
                                const size_t gr = (size_t)row0 + 32 * q + rr;
                                *reinterpret_cast<uint4*>(p.partial + gr * p.N_total + (size_t)nt * kTileN + c0 + 8 * c) = v;
                            }
                        }
                        __syncwarp();
                    }
                }
                // rows past the tile's end hold f0 = 0, so only stored rows count
                if (__any_sync(0xffffffffu, over) && lane == 0) atomicOr(p.err, kDevErrOverflow);
            }
            tc_fence_before();
            mbar_arrive(&bars.acc_empty);
            if (kDown) {
                dm_cur = dm_nxt;
                dw_cur = dw_nxt;
                dts_cur = dts_nxt;
                dm_nxt = dm_nn;
            }
        }
        // down: this warp's tile stores have completed before the CTA exits
        if (!kRouter && !kGateUp && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    } else if (warp < kMmaWarp) {
        // ---------------------------------------------------------- scale warps
        // warp 12 + j (lane quarter j): for every stage, once its tiles have
        // landed, lane i loads its 16 bytes of each k-step of the A and B
        // scale tiles and stores them as the stage's 48 scale columns
        // (A: 4 per k-step; B: 4 per k-step for rows 0-127, then 4 for 128-255);
        // word c of lane i's 16 bytes of a k-step is row 32 c + i.  Gate/up's
        // A scales arrive row-major (row r's 4 k-steps at 16 r): lane i loads
        // rows i, 32 + i, 64 + i, 96 + i and takes word ks of each.
        if (!kRouter) {
            const int q = warp & 3;
            uint32_t it = 0;
            for (uint32_t w = blockIdx.x; w < n_work && !bars.abort; w += gridDim.x) {
                bool ok = true;
                for (int kb = 0; kb < kstages; ++kb, ++it) {
                    const int s = (int)(it % nst);
                    if (!wait_or_abort(&bars.full[s], (it / nst) & 1u, bars, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint8_t* sSA = smem + (size_t)s * kStageBytes + kABytes + kBBytes;
                    const uint8_t* sSB = sSA + kSfABytes;
                    uint32_t a[16], b[32];
                    if (kGateUp) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 vr = *reinterpret_cast<const uint4*>(sSA + (32 * c + lane) * 16);
                            a[c] = vr.x, a[4 + c] = vr.y, a[8 + c] = vr.z, a[12 + c] = vr.w;
                        }
                    }
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint4 v0 = *reinterpret_cast<const uint4*>(sSB + ks * 512 + lane * 16);
                        const uint4 v1 = *reinterpret_cast<const uint4*>(sSB + kSfChunk + ks * 512 + lane * 16);
                        if (!kGateUp) {
                            const uint4 va = *reinterpret_cast<const uint4*>(sSA + ks * 512 + lane * 16);
                            a[4 * ks] = va.x, a[4 * ks + 1] = va.y, a[4 * ks + 2] = va.z, a[4 * ks + 3] = va.w;
                        }
                        b[8 * ks] = v0.x, b[8 * ks + 1] = v0.y, b[8 * ks + 2] = v0.z, b[8 * ks + 3] = v0.w;
                        b[8 * ks + 4] = v1.x, b[8 * ks + 5] = v1.y, b[8 * ks + 6] = v1.z, b[8 * ks + 7] = v1.w;
                    }
                    const uint32_t sf = tmem + ((uint32_t)(32 * q) << 16) + kAccCols + (uint32_t)s * kSfColsPerStage;
                    tmem_st16(sf, a);
                    tmem_st32(sf + 16, b);
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    tc_fence_before();
                    mbar_arrive(&bars.sf_full[s]);
                }
                if (!ok) break;
            }
        } else {
            // router: S3's max |x| from the x tiles as they pass (each element
            // once: the first N-tile's hi half), then the stage goes to the
            // MMA thread.  Thread i of the 128 reads 16-byte chunks i, i + 128,
            // ... of the 16 KB tile (the order does not matter to a maximum);
            // bf16 magnitudes compare as their bit patterns, NaN counted as 0
            // (as fmaxf ignores it).
            const int sub = tid - 32 * kSfWarp0;
            uint32_t mx = 0;   // two bf16 magnitudes, packed
            uint32_t it = 0;
            for (uint32_t w = blockIdx.x; w < n_work && !bars.abort; w += gridDim.x) {
                const bool scan = p.amax != nullptr && (int)(w % n_tiles_n) == 0;
                bool ok = true;
                for (int kb = 0; kb < kstages; ++kb, ++it) {
                    const int s = (int)(it % nst);
                    if (!wait_or_abort(&bars.full[s], (it / nst) & 1u, bars, p.err)) {
                        ok = false;
                        break;
                    }
                    if (scan && kb < kstages / 2) {
                        const uint4* a = reinterpret_cast<const uint4*>(smem + (size_t)s * kStageBytes);
#pragma unroll
                        for (int i = 0; i < kABytes / 16 / 128; ++i) {
                            const uint4 v = a[sub + 128 * i];
                            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t m = wv[j] & 0x7FFF7FFFu;
                                mx = __vmaxu2(mx, m & ~__vcmpgtu2(m, 0x7F807F80u));
                            }
                        }
                    }
                    mbar_arrive(&bars.sf_full[s]);
                }
                if (!ok) break;
            }
            uint32_t m16 = max(mx & 0xFFFFu, mx >> 16);
            m16 = __reduce_max_sync(0xffffffffu, m16);
            if (lane == 0 && m16 != 0) atomicMax(p.amax, m16 << 16);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA
        uint32_t it = 0, tile = 0;
        if (lane == 0) {
            for (uint32_t w = blockIdx.x; w < n_work && !bars.abort; w += gridDim.x, ++tile) {
                if (tile > 0 && !wait_or_abort(&bars.acc_empty, (tile - 1) & 1u, bars, p.err)) break;
                tc_fence_after();
                bool ok = true;
                for (int kb = 0; kb < kstages; ++kb, ++it) {
                    const int s = (int)(it % nst);
                    // wait for the scale warps (who waited for the tiles): FP4
                    // modes for the scales in tensor memory, the router for the
                    // max |x| pass over the x tile
                    if (!wait_or_abort(&bars.sf_full[s], (it / nst) & 1u, bars, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (kGateUp) fence_proxy_async_smem();   // A rows came by cp.async
                    const uint32_t a0 = smem_u32(smem + (size_t)s * kStageBytes);
                    const uint32_t b0 = a0 + kABytes;
                    const uint32_t sf = tmem + kAccCols + (uint32_t)s * kSfColsPerStage;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {   // 4 MMAs of 32 bytes of K per 128-byte row
                        const uint32_t accumulate = (kb > 0 || ks > 0) ? 1u : 0u;
                        if (kRouter)
                            mma_bf16(tmem, desc_sw128(a0 + ks * 32), desc_sw128(b0 + ks * 32), accumulate);
                        else
                            mma_fp4(tmem, desc_sw128(a0 + ks * 32), desc_sw128(b0 + ks * 32), sf + 4 * ks,
                                    sf + 16 + 8 * ks, accumulate);
                    }
                    mma_commit(&bars.empty[s]);   // frees the stage once these MMAs are done
                }
                if (!ok) break;
                mma_commit(&bars.acc_full);
            }
            // every MMA issued has completed before tensor memory is released
            mma_commit(&bars.mma_done);
            if (!mbar_wait(&bars.mma_done, 0)) atomicOr(p.err, kDevErrTimeout);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// Expert-major list of 128-row M-tiles: (expert, first row, rows).
__global__ void __launch_bounds__(1024) k_build_mtiles(const int32_t* __restrict__ offsets, int E,
                                                       int4* __restrict__ mtiles,
                                                       uint32_t* __restrict__ n_mtiles) {
    __shared__ int warp_tot[32];
    __shared__ int total;
    const int e = threadIdx.x, lane = e & 31, wp = e >> 5;
    const int cnt = e < E ? offsets[e + 1] - offsets[e] : 0;
    const int nt = (cnt + kTileM - 1) / kTileM;
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[wp] = incl;
    __syncthreads();
    if (wp == 0) {
        const int t = warp_tot[lane];
        int ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += v;
        }
        warp_tot[lane] = ti - t;
        if (lane == 31) total = ti;
    }
    __syncthreads();
    const int base = incl - nt + warp_tot[wp];
    for (int i = 0; i < nt; ++i) {
        const int r0 = i * kTileM;
        const int rows = cnt - r0 < kTileM ? cnt - r0 : kTileM;
        mtiles[base + i] = make_int4(e, offsets[e] + r0, rows, 0);
    }
    if (e == 0) *n_mtiles = (uint32_t)total;
}

// y[t] = sum_j partial[inv[t*k + j]] in slot order (+ residual); fp16 partials, fp32 sums.
__global__ void __launch_bounds__(256) k_combine(const __half* __restrict__ partial,
                                                 const int32_t* __restrict__ inv, int T, int k, int H,
                                                 const uint16_t* __restrict__ residual,
                                                 float* __restrict__ y, uint16_t* __restrict__ x_next) {
    const size_t n8 = (size_t)T * (H / 8);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8;
         i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / (H / 8)), c = (int)(i % (H / 8));
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const int r = inv[(size_t)t * k + j];
            if (r < 0) continue;   // dropped by the route-tail skip
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(partial + (size_t)r * H) + c);
            const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __half22float2(h2[q]);
                acc[2 * q] += f.x;
                acc[2 * q + 1] += f.y;
            }
        }
        float4* yo = reinterpret_cast<float4*>(y + (size_t)t * H) + 2 * c;
        yo[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        yo[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        if (x_next) {
            const uint4 rv = __ldg(reinterpret_cast<const uint4*>(residual + (size_t)t * H) + c);
            const uint32_t w[4] = {rv.x, rv.y, rv.z, rv.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t lo = f32_to_bf16_rn(bf16_to_f32(w[q] & 0xFFFFu) + acc[2 * q]);
                const uint32_t hi = f32_to_bf16_rn(bf16_to_f32(w[q] >> 16) + acc[2 * q + 1]);
                o[q] = lo | (hi << 16);
            }
            reinterpret_cast<uint4*>(x_next + (size_t)t * H)[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// cuTensorMapEncodeTiled, reached through the runtime (no link against the driver library)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static const EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return EncodeTiledFn(nullptr);
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

// 2-D tensor map over `rows` rows of `inner` elements (row pitch row_bytes),
// box {box_inner, box_rows}, 128-byte swizzle, zero fill outside the tensor.
bool map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
            uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
    const EncodeTiledFn fn = encoder();
    if (!fn || !base) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm(GemmMode mode, const GemmParams& prm, cudaStream_t st) {
    static int configured = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured != dev) {
        e = cudaFuncSetAttribute(k_grouped_gemm<GemmMode::kGateUp>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_grouped_gemm<GemmMode::kDown>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_grouped_gemm<GemmMode::kRouter>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = dev;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    switch (mode) {
        case GemmMode::kGateUp:
            k_grouped_gemm<GemmMode::kGateUp><<<sms, kThreads, kSmemBytes, st>>>(prm);
            break;
        case GemmMode::kDown:
            k_grouped_gemm<GemmMode::kDown><<<sms, kThreads, kSmemBytes, st>>>(prm);
            break;
        case GemmMode::kRouter:
            k_grouped_gemm<GemmMode::kRouter><<<sms, kThreads, kSmemBytes, st>>>(prm);
            break;
    }
    count_launches(1);
    return cudaGetLastError();
}

// Split fp32 Wr into bf16 hi = RN(w) and lo = RN(w - hi): hi + lo carries ~16
// significant bits of each weight.
__global__ void k_router_split(const float* __restrict__ Wr, size_t n, uint16_t* __restrict__ hi,
                               uint16_t* __restrict__ lo) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const float w = Wr[i];
        const uint16_t h = f32_to_bf16_rn(w);
        hi[i] = h;
        lo[i] = f32_to_bf16_rn(w - bf16_to_f32(h));
    }
}

// Weight scales [rows][K/16] -> the tiled block-scale layout (one byte per
// thread; runs once per matrix when a layer is created).
__global__ void k_tile_scales(const uint8_t* __restrict__ src, size_t rows, int K, uint8_t* __restrict__ dst) {
    const int kbs = K / kStageK;
    const size_t n = rows * (size_t)(K / 16);
    for (size_t o = blockIdx.x * (size_t)blockDim.x + threadIdx.x; o < n; o += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(o & 3), j = (int)((o >> 2) & 3), i = (int)((o >> 4) & 31), ks = (int)((o >> 9) & 3);
        const size_t chunk = o >> 11;
        const int kb = (int)(chunk % kbs);
        const size_t row = (chunk / kbs) * 128 + 32 * j + i;
        dst[o] = src[row * (size_t)(K / 16) + kb * 16 + ks * 4 + c];
    }
}

}  // namespace

size_t tiled_scale_bytes(size_t rows, int K) { return rows * (size_t)(K / 16); }

cudaError_t launch_tile_scales(const uint8_t* scales, size_t rows, int K, uint8_t* tiled, cudaStream_t st) {
    if (rows % 128 || K % kStageK) return cudaErrorInvalidValue;
    const size_t n = tiled_scale_bytes(rows, K);
    const size_t grid = (n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192;
    k_tile_scales<<<(unsigned)grid, 256, 0, st>>>(scales, rows, K, tiled);
    count_launches(1);
    return cudaGetLastError();
}

size_t router_split_bytes(const Shape& s) { return (size_t)2 * s.E * s.H * sizeof(uint16_t); }

bool router_tc_supported(const Shape& s) { return s.H % 64 == 0; }

cudaError_t launch_router_split(const float* Wr, int E, int H, uint16_t* hi, uint16_t* lo,
                                cudaStream_t st) {
    const size_t n = (size_t)E * H;
    k_router_split<<<(unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0, st>>>(
        Wr, n, hi, lo);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_router_tc(const uint16_t* x, const uint16_t* w_hi, const uint16_t* w_lo,
                             const float* bias, int T, const Shape& s, float* logits,
                             uint32_t* amax, uint32_t* err, cudaStream_t st) {
    GemmParams r{};
    r.K = s.H;
    r.T = T;
    r.E = s.E;
    r.x_bf16 = x;
    r.w_hi = w_hi;
    r.w_lo = w_lo;
    r.bias = bias;
    r.logits = logits;
    r.amax = amax;
    r.err = err;
    const uint64_t H = (uint64_t)s.H;
    if (!map_2d(&r.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT16, w_hi, H, (uint64_t)s.E, H * 2, 64, kTileN) ||
        !map_2d(&r.tm_b2, CU_TENSOR_MAP_DATA_TYPE_UINT16, w_lo, H, (uint64_t)s.E, H * 2, 64, kTileN) ||
        !map_2d(&r.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, H, (uint64_t)T, H * 2, 64, kTileM))
        return cudaErrorInvalidValue;
    return launch_gemm(GemmMode::kRouter, r, st);
}

bool prefill_supported(const Shape& s) {
    return s.H % kStageK == 0 && s.I % kStageK == 0 && s.I % (kTileN / 2) == 0 &&
           s.H % kTileN == 0;
}

cudaError_t launch_prefill_gateup(const Shape& s, const ExpertWeights& gate, const ExpertWeights& up,
                                  float h_scale, const Workspace& ws, uint32_t* err, cudaStream_t st) {
    k_build_mtiles<<<1, 1024, 0, st>>>(ws.offsets, s.E, ws.mtiles, ws.scal + kScalMTiles);
    count_launches(1);
    GemmParams g{};
    g.K = s.H;
    g.N_total = s.I;
    g.k = s.k;
    g.h_scale = h_scale;
    g.mtiles = ws.mtiles;
    g.n_mtiles = ws.scal + kScalMTiles;
    g.perm = ws.perm;
    g.a_codes = ws.xq;
    g.a_scales = ws.xs;
    g.a_tensor_scale = ws.sx;
    g.b_sf_tiled = gate.sf_tiled;
    g.b_tensor_scale = gate.ts;
    g.b2_sf_tiled = up.sf_tiled;
    g.b2_tensor_scale = up.ts;
    g.out_codes = ws.hq;
    g.out_scales = ws.hs;
    g.out_sf_tiled = ws.hs_tiled;
    g.err = err;
    if (!gate.sf_tiled || !up.sf_tiled || !ws.hs_tiled) return cudaErrorInvalidValue;
    const uint64_t row_b = (uint64_t)s.H / 2, rows = (uint64_t)s.E * s.I;
    if (!map_2d(&g.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, gate.codes, row_b, rows, row_b, 128, kTileN / 2) ||
        !map_2d(&g.tm_b2, CU_TENSOR_MAP_DATA_TYPE_UINT8, up.codes, row_b, rows, row_b, 128, kTileN / 2))
        return cudaErrorInvalidValue;
    return launch_gemm(GemmMode::kGateUp, g, st);
}

cudaError_t launch_prefill_down(const Shape& s, int T, const ExpertWeights& down, float h_scale,
                                const Workspace& ws, const uint16_t* residual, float* y,
                                uint16_t* x_next, uint32_t* err, cudaStream_t st) {
    GemmParams d{};
    d.K = s.I;
    d.N_total = s.H;
    d.k = s.k;
    d.h_scale = h_scale;
    d.mtiles = ws.mtiles;
    d.n_mtiles = ws.scal + kScalMTiles;
    d.perm = ws.perm;
    d.a_sf_tiled = ws.hs_tiled;
    d.b_sf_tiled = down.sf_tiled;
    d.b_tensor_scale = down.ts;
    if (!down.sf_tiled || !ws.hs_tiled) return cudaErrorInvalidValue;
    d.pair_w_perm = ws.wperm;
    if (!ws.wperm) return cudaErrorInvalidValue;
    d.partial = ws.partial;
    d.err = err;
    const uint64_t row_b = (uint64_t)s.I / 2;
    if (!map_2d(&d.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, down.codes, row_b, (uint64_t)s.E * s.H, row_b, 128,
                kTileN) ||
        !map_2d(&d.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, ws.hq, row_b, (uint64_t)T * s.k, row_b, 128, kTileM) ||
        !map_2d(&d.tm_out, CU_TENSOR_MAP_DATA_TYPE_UINT16, ws.partial, (uint64_t)s.H, (uint64_t)T * s.k,
                (uint64_t)s.H * 2, 64, 32))
        return cudaErrorInvalidValue;
    cudaError_t e = launch_gemm(GemmMode::kDown, d, st);
    if (e != cudaSuccess) return e;
    const size_t n8 = (size_t)T * (s.H / 8);
    size_t grid = (n8 + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    k_combine<<<(unsigned)grid, 256, 0, st>>>(ws.partial, ws.inv, T, s.k, s.H, residual, y, x_next);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
