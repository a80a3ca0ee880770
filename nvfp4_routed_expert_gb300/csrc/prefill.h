// Tensor-core grouped GEMMs of the prefill path (prefill.cu).
#pragma once
#include <cstdint>
#include <cuda.h>   // CUtensorMap (the encoder is reached through the runtime's entry point)
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace moe {

struct GemmParams {
    // TMA tensor maps (128-byte swizzle, 128-byte inner box): B of every mode
    // (gate rows / down rows / Wr hi), the second B (up rows / Wr lo), and A
    // where its rows are contiguous (down: h rows; router: x rows)
    CUtensorMap tm_b, tm_b2, tm_a;
    CUtensorMap tm_out;           // down: the fp16 partials [P][H], 64 x 32 boxes (stores)
    int K;                        // contraction length (H for gate/up, I for down)
    int N_total;                  // rows of one expert's B matrix (I for gate/up, H for down)
    int k;                        // top-k
    float h_scale;                // static tensor scale of h
    const int4* mtiles;           // (expert, first row, rows, -) per 128-row M-tile
    const uint32_t* n_mtiles;     // device count of M-tiles
    const int32_t* perm;          // expert-grouped position -> pair id
    const uint8_t* a_codes;       // gate/up: x codes [T][H/2] (gathered by token)
    const uint8_t* a_scales;      // gate/up: x scales [T][H/16] (gathered by token)
    const uint8_t* a_sf_tiled;    // down: h scales, tiled per M-tile
    const float* a_tensor_scale;  // gate/up: s_x (device)
    const uint8_t* b_sf_tiled;    // gate (or down) weight scales, tiled per 128 rows
    const float* b_tensor_scale;
    const uint8_t* b2_sf_tiled;   // up weight scales, tiled (gate/up only)
    const float* b2_tensor_scale;
    uint8_t* out_codes;           // gate/up: hq [P][I/2]
    uint8_t* out_scales;          // gate/up: hs [P][I/16]
    uint8_t* out_sf_tiled;        // gate/up: hs again, tiled per M-tile (the down GEMM's A scales)
    const float* pair_w_perm;     // down: router weight of each expert-grouped position
    __half* partial;              // down: weighted fp16 outputs [P][H] (expert order)
    // router mode: logits[T][E] = x [T][H] (bf16) * (w_hi + w_lo)^T + bias
    int T, E;
    const uint16_t* x_bf16;
    const uint16_t* w_hi;         // bf16 [E][H], round-to-nearest of Wr
    const uint16_t* w_lo;         // bf16 [E][H], round-to-nearest of Wr - w_hi
    const float* bias;            // [E] or null
    float* logits;
    uint32_t* amax;               // router: max|x| as fp32 bits (atomicMax; the caller zeroes it), or null
    uint32_t* err;
};

enum class GemmMode { kGateUp, kDown, kRouter };

// Bytes of the packed router copy (bf16 hi and lo parts of Wr).
size_t router_split_bytes(const Shape& s);
// Fill the packed router copy from fp32 Wr.
cudaError_t launch_router_split(const float* Wr, int E, int H, uint16_t* hi, uint16_t* lo,
                                cudaStream_t st);
// S1 on the tensor cores: logits [T][E] (+ bias); with amax non-null also
// S3's max |x| (fp32 bits, atomicMax into a word the caller has zeroed).
cudaError_t launch_router_tc(const uint16_t* x, const uint16_t* w_hi, const uint16_t* w_lo,
                             const float* bias, int T, const Shape& s, float* logits,
                             uint32_t* amax, uint32_t* err, cudaStream_t st);
bool router_tc_supported(const Shape& s);

// Shapes the tensor-core path handles (H and I multiples of 256).
bool prefill_supported(const Shape& s);

// Block scales of a [rows][K] NVFP4 matrix (rows % 128 == 0, K % 256 == 0)
// in the tiled layout the grouped GEMM copies into tensor memory: for each
// 128-row group g and 256-element stage kb a 2 KB chunk at (g * K/256 + kb)
// * 2048 of four 512-byte k-steps [lane i][row quarter j][4 scale bytes of
// row 128 g + 32 j + i].  Same size as the scales.
size_t tiled_scale_bytes(size_t rows, int K);
cudaError_t launch_tile_scales(const uint8_t* scales, size_t rows, int K, uint8_t* tiled, cudaStream_t st);

// S5 (M-tile list + gate/up GEMM) for a call whose S1-S4 results are in ws.
cudaError_t launch_prefill_gateup(const Shape& s, const ExpertWeights& gate, const ExpertWeights& up,
                                  float h_scale, const Workspace& ws, uint32_t* err, cudaStream_t st);
// S6 (down GEMM + combine in slot order, residual).
cudaError_t launch_prefill_down(const Shape& s, int T, const ExpertWeights& down, float h_scale,
                                const Workspace& ws, const uint16_t* residual, float* y,
                                uint16_t* x_next, uint32_t* err, cudaStream_t st);

}  // namespace moe
