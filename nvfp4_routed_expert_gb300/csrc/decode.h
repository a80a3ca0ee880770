// Fused decode kernel (decode.cu): parameters and launch.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"

namespace moe {

constexpr int kDecodeMaxTokens = 8;
constexpr int kDecodeMaxPairs = 128;
constexpr int kDecodeMaxLayers = 64;
constexpr size_t kDecodeSmemBytes = 227 * 1024;

struct DecodeLayer {
    const float* wr;       // router [E][H]
    const float* bias;     // [E] or null
    const uint8_t* gc;     // gate codes / scales / tensor scales
    const uint8_t* gs;
    const float* gts;
    const uint8_t* uc;     // up
    const uint8_t* us;
    const float* uts;
    const uint8_t* dc;     // down
    const uint8_t* ds;
    const float* dts;
    float* y;              // [T][H] fp32 output of this layer, or null
};

struct DecodeParams {
    int L, T, H, E, k, I;
    float h_scale;
    uint32_t region_a_off, region_b_off;
    int slots_g, slots_d;
    uint32_t d_off;             // offset of the down ring inside region b
    int d_early;                // 1: the down ring has its own space and is filled during gate/up
    const uint16_t* x_in;       // layer-0 input [T][H]
    const uint16_t* residual0;  // layer-0 residual (null: layer 0 writes no x_next)
    uint16_t* x_out;            // last layer's bf16(residual + y), or null
    uint16_t* xbuf0;            // ping-pong activations between layers
    uint16_t* xbuf1;
    float* logits;              // [T][E]
    int32_t* idx;               // [T][k]
    float* w;
    int32_t* counts;            // [E]
    int32_t* offsets;           // [E+1]
    int32_t* perm;              // [T*k]
    int32_t* inv;
    uint8_t* xq;                // [T][H/2]
    uint8_t* xs;                // [T][H/16]
    float* sx;
    uint8_t* hq;                // [T*k][I/2]
    uint8_t* hs;                // [T*k][I/16]
    uint32_t* bar;              // grid-barrier counter (zeroed before each launch)
    uint32_t* err;              // device status word
    uint64_t* phase_ns;         // [2][16] globaltimer stamps of CTA 0 and the last CTA, or null
    DecodeLayer layer[kDecodeMaxLayers];
};

struct DecodeSmemPlan {
    bool ok;
    uint32_t region_a_off, region_b_off;
    int slots_g, slots_d;
    uint32_t d_off;
    int d_early;
    size_t bytes;
};

DecodeSmemPlan decode_smem_plan(const Shape& s, int T);
bool decode_supported(const Shape& s, int T);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st);

}  // namespace moe
