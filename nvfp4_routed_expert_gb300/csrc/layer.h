// The layer handle behind the C ABI's opaque moe_layer (host object).
#pragma once
#include <cuda_runtime.h>

#include "moe.h"

struct moe_layer {
    moe_layer_desc desc;
    const float* router_w;
    const float* router_bias;
    moe_nvfp4 gate, up, down;
    uint32_t* dev_status;
    int device;
    moe_step trace_step;
    cudaEvent_t trace_start, trace_end;
};
