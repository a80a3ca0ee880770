// The layer handle behind the C ABI's opaque moe_layer (host object).
#pragma once
#include <cuda_runtime.h>

#include "moe.h"

struct moe_layer {
    moe_layer_desc desc;
    const float* router_w;
    const float* router_bias;
    // bf16 hi and lo parts of the router weights (in the caller's packed
    // buffer) for the tensor-core S1; null when the layer never takes it
    const uint16_t* router_hi;
    const uint16_t* router_lo;
    // gate, up and down block scales in the grouped GEMM's tiled layout (in
    // the packed buffer too); null when the layer never takes that path
    const uint8_t* gate_sf_tiled;
    const uint8_t* up_sf_tiled;
    const uint8_t* down_sf_tiled;
    moe_nvfp4 gate, up, down;
    const uint8_t* resident;   // route-tail skip: experts never skipped [E], or null
    uint32_t* dev_status;
    int device;
    moe_step trace_step;
    cudaEvent_t trace_start, trace_end;
};
