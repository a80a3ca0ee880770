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
    const uint8_t* resident;   // route-tail skip: experts never skipped [E], or null
    int keep;                  // route-tail skip: ranks always computed (k: every pick)
    float* y;              // [T][H] fp32 output of this layer, or null
};

// Shared-memory plan of one launch (depends on the shape, T and the grid).
struct DecodeSmemPlan {
    bool ok;
    uint32_t a_off;        // x as int8 + block scales + bf16 staging; later h as int8 + scales + per-pair outputs
    uint32_t wr_off;       // router rows of the CTA's experts, fp32 [wr_rows][H]
    uint32_t ring_off;     // logits, top-k candidates; then the weight slots
    uint32_t g_off;        // first gate/up slot (all offsets from the start of shared memory)
    uint32_t d_area_off;   // first down slot (after the gate/up slots)
    bool g_over_wr;        // gate/up slots also cover the x staging and the router rows,
                           // so the next layer's router rows are issued after gate/up
    int wr_rows;           // most router rows a CTA owns: ceil(E / grid)
    int d_rows;            // most output rows a CTA owns in the down step
    int slots_g;           // gate/up slots (one 16-feature item each)
    int slots_d;           // down slots in the down area
    int slots_d_total;     // down slots once the gate/up area is free as well
    size_t bytes;
};

struct DecodeParams {
    int L, T, H, E, k, I;
    float h_scale;
    DecodeSmemPlan plan;        // filled by launch_decode
    const uint16_t* x_in;       // layer-0 input [T][H]
    const uint16_t* residual0;  // layer-0 residual (null: layer 0 writes no x_next; needs L == 1)
    uint16_t* x_out;            // last layer's bf16(residual + y), or null
    uint64_t* tags;             // tagged exchange words, decode_tag_bytes(); zeroed per launch
    bool debug;                 // write the inspection outputs below (the caller asked for them)
    float* logits;              // [T][E]          (last layer's values, for inspection)
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
    uint32_t* err;              // device status word
    uint64_t* phase_ns;         // [2][16] globaltimer stamps of CTA 0 and the last CTA, or null
    DecodeLayer layer[kDecodeMaxLayers];
};

// Bytes of the tagged exchange area for T tokens (logits, h and x words of
// two consecutive layers).
size_t decode_tag_bytes(const Shape& s, int T);
DecodeSmemPlan decode_smem_plan(const Shape& s, int T, int grid);
bool decode_supported(const Shape& s, int T);
cudaError_t launch_decode(DecodeParams& p, cudaStream_t st);
// One CTA runs the bounded tagged-word poll over n never-written words and a
// bounded mbarrier wait; both must run out and set kDevErrTimeout in err[0], err[1].
cudaError_t launch_selftest_waits(const uint64_t* words, int n, uint32_t* err, cudaStream_t st);

}  // namespace moe
