// Internal launchers of the NVFP4 MoE layer kernels (not part of the C ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace moe {

// Shape of one layer as the kernels see it.
struct Shape {
    int H, E, k, I;
};

// Scratch regions carved from the caller's workspace (see workspace_layout).
struct Workspace {
    uint32_t* scal;        // [64] scalars: kScalAmax, kScalSx, ...
    float* logits;         // [Tm][E]
    int32_t* idx;          // [Tm][k]
    float* w;              // [Tm][k]
    int32_t* counts;       // [E]
    int32_t* offsets;      // [E+1]
    int32_t* active;       // [E] experts with at least one pair, ascending
    int32_t* chunk_cnt;    // [nchunks][E] per-chunk histograms, then chunk bases
    int32_t* group_cnt;    // [ngroups][E] sums over groups of kPermGroup chunks, then group
                           // bases (only when nchunks > kPermGroupMin)
    int32_t* perm;         // [Pm]
    int32_t* inv;          // [Pm]
    uint8_t* xq;           // [Tm][H/2]
    uint8_t* xs;           // [Tm][H/16]
    float* sx;             // fp32 tensor scale of x (points into scal by default)
    uint8_t* hq;           // [Pm][I/2]
    uint8_t* hs;           // [Pm][I/16]
    uint16_t* xbuf0;       // [min(Tm,8)][H] bf16 activations between stacked layers
    uint16_t* xbuf1;
    uint64_t* tags;        // tagged exchange words of the fused decode kernel
    int4* mtiles;          // [Pm/128 + E + 1] M-tiles of the tensor-core GEMMs (prefill)
    uint8_t* hs_tiled;     // [Pm/128 + E + 1][I/16 * 128] hs tiled per M-tile (prefill)
    __half* partial;       // [Pm][H] weighted fp16 outputs per pair (prefill)
    float* wperm;          // [Pm] router weight of each expert-grouped position (prefill)
    size_t bytes;
};

constexpr int kScalAmax = 0;     // fp32 bits of max|x| (atomicMax target)
constexpr int kScalSx = 1;       // fp32 tensor scale of x
constexpr int kScalActive = 2;   // number of active experts
constexpr int kScalMTiles = 4;   // number of M-tiles of the tensor-core GEMMs
constexpr int kScalCount = 64;

constexpr int kPermChunk = 1024;  // pairs per permutation chunk
// Above kPermGroupMin chunks the per-expert scan over the chunks runs in two
// levels: sums over groups of kPermGroup chunks, the scan over the groups,
// then each group's chunks from its base.
constexpr int kPermGroup = 16;
constexpr int kPermGroupMin = 64;
__host__ __device__ constexpr int perm_groups(int nchunks) {
    return nchunks > kPermGroupMin ? (nchunks + kPermGroup - 1) / kPermGroup : 0;
}

// with_prefill: include the regions only the tensor-core prefill path uses
// (the M-tile list and the fp16 partial outputs); with_decode: the tagged
// exchange words of the fused decode kernel
Workspace workspace_layout(const Shape& s, int max_tokens, void* base, bool with_prefill,
                           bool with_decode = false);

// Calls with more tokens than this go through the tensor-core prefill path.
constexpr int kPrefillMinTokens = 9;

// Adds n to the process-wide count of kernels launched by this library.
void count_launches(int n);

// S3: quantise bf16 x [T][H]; writes codes/scales and *sx (device).
cudaError_t launch_quant_act(const uint16_t* x, int T, int H, uint8_t* codes, uint8_t* scales,
                             float* sx, uint32_t* amax_scratch, cudaStream_t st);
// S3 when max |x| is already in *amax (fp32 bits): the quantiser pass alone.
cudaError_t launch_quant_act_given_amax(const uint16_t* x, int T, int H, uint8_t* codes,
                                        uint8_t* scales, float* sx, const uint32_t* amax,
                                        cudaStream_t st);

// Weight quantiser: fp32 [M][rows][cols] with a per-matrix tensor scale.
cudaError_t launch_quant_weights(const float* w, int M, int rows, int cols, uint8_t* codes,
                                 uint8_t* scales, float* ts, cudaStream_t st);

// S1 + S2: logits [T][E] and top-k indices / weights.  keep < k turns on the
// route-tail skip (resident: per-expert mask [E] of experts never skipped, or
// null): dropped picks get expert -1 and weight 0.
cudaError_t launch_router(const uint16_t* x, const float* Wr, const float* bias, int T,
                          const Shape& s, float* logits, int32_t* idx, float* w, cudaStream_t st,
                          int keep, const uint8_t* resident);
// S2 alone, on logits already in memory.
cudaError_t launch_topk(const float* logits, int T, const Shape& s, int32_t* idx, float* w,
                        cudaStream_t st, int keep, const uint8_t* resident);

// S4: counts, offsets, active list, perm, inv.
cudaError_t launch_permute(const int32_t* idx, int T, const Shape& s, const Workspace& ws,
                           cudaStream_t st);

// S5: gate/up GEMV, SwiGLU and requantisation of h for every pair.
struct ExpertWeights {
    const uint8_t* codes;
    const uint8_t* scales;
    const float* ts;
    const uint8_t* sf_tiled = nullptr;   // scales in the tensor-core path's tiled layout
};
cudaError_t launch_gateup(const Shape& s, int T, const ExpertWeights& gate,
                          const ExpertWeights& up, float h_scale, const Workspace& ws,
                          cudaStream_t st);

// S6: down GEMV, weighted combine in slot order, optional residual.
cudaError_t launch_down(const Shape& s, int T, const ExpertWeights& down, float h_scale,
                        const Workspace& ws, const uint16_t* residual, float* y,
                        uint16_t* x_next, cudaStream_t st);

}  // namespace moe
