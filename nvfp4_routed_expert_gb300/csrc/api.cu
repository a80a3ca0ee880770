// C ABI of the NVFP4 MoE layer: argument checks, workspace carving and the
// launch sequence S1..S6 on the caller's stream.  No call here allocates
// device memory except moe_layer_create (one status word).
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>

#include "kernels.h"
#include "layer.h"
#include "moe.h"

namespace moe {

namespace {

constexpr size_t kAlign = 256;
std::atomic<uint64_t> g_launches{0};

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

}  // namespace

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

Workspace workspace_layout(const Shape& s, int Tm, void* base) {
    Workspace w{};
    const size_t Pm = (size_t)Tm * s.k;
    const size_t nchunks = (Pm + kPermChunk - 1) / kPermChunk;
    uint8_t* b = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* p = b ? b + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    w.scal = reinterpret_cast<uint32_t*>(take(sizeof(uint32_t) * kScalCount));
    w.logits = reinterpret_cast<float*>(take(sizeof(float) * (size_t)Tm * s.E));
    w.idx = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * Pm));
    w.w = reinterpret_cast<float*>(take(sizeof(float) * Pm));
    w.counts = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * s.E));
    w.offsets = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (s.E + 1)));
    w.active = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * s.E));
    w.chunk_cnt = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * nchunks * s.E));
    w.perm = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * Pm));
    w.inv = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * Pm));
    w.xq = take((size_t)Tm * s.H / 2);
    w.xs = take((size_t)Tm * s.H / 16);
    w.hq = take(Pm * s.I / 2);
    w.hs = take(Pm * s.I / 16);
    w.sx = w.scal ? reinterpret_cast<float*>(w.scal + kScalSx) : nullptr;
    w.bytes = off;
    return w;
}

}  // namespace moe

namespace {

using moe::Shape;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool desc_ok(const moe_layer_desc* d) {
    if (!d) return false;
    if (d->hidden < 64 || d->hidden > 8192 || d->hidden % 64) return false;
    if (d->inter < 64 || d->inter > 4096 || d->inter % 64) return false;
    if (d->num_experts < 1 || d->num_experts > 1024) return false;
    if (d->top_k < 1 || d->top_k > 32 || d->top_k > d->num_experts) return false;
    if (d->max_tokens < 1 || d->max_tokens > (1 << 20)) return false;
    if (d->flags != 0) return false;
    if (!(d->h_tensor_scale > 0.0f) || !std::isfinite(d->h_tensor_scale)) return false;
    return true;
}

Shape shape_of(const moe_layer_desc& d) { return Shape{d.hidden, d.num_experts, d.top_k, d.inter}; }

bool nvfp4_ok(const moe_nvfp4* w) {
    return w && w->codes && w->scales && w->tensor_scale && (reinterpret_cast<uintptr_t>(w->codes) & 15u) == 0;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARGUMENT: return "MOE_ERR_INVALID_ARGUMENT";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
        case MOE_ERR_OUT_OF_MEMORY: return "MOE_ERR_OUT_OF_MEMORY";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    }
    return "MOE_ERR_UNKNOWN";
}

size_t moe_workspace_bytes(const moe_layer_desc* desc) {
    if (!desc_ok(desc)) return 0;
    return moe::workspace_layout(shape_of(*desc), desc->max_tokens, nullptr).bytes;
}

size_t moe_packed_weight_bytes(const moe_layer_desc* desc) {
    (void)desc;
    return 0;
}

moe_status moe_layer_create(const moe_layer_desc* desc, const float* router_w,
                            const float* router_bias, const moe_nvfp4* gate, const moe_nvfp4* up,
                            const moe_nvfp4* down, void* packed, void* stream, moe_layer** out) {
    (void)packed;
    (void)stream;
    if (!out) return MOE_ERR_INVALID_ARGUMENT;
    *out = nullptr;
    if (!desc) return MOE_ERR_INVALID_ARGUMENT;
    if (!desc_ok(desc)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!router_w || !aligned16(router_w) || !nvfp4_ok(gate) || !nvfp4_ok(up) || !nvfp4_ok(down))
        return MOE_ERR_INVALID_ARGUMENT;
    moe_layer* L = new (std::nothrow) moe_layer{};
    if (!L) return MOE_ERR_OUT_OF_MEMORY;
    L->desc = *desc;
    L->router_w = router_w;
    L->router_bias = router_bias;
    L->gate = *gate;
    L->up = *up;
    L->down = *down;
    if (cudaGetDevice(&L->device) != cudaSuccess) {
        delete L;
        return MOE_ERR_CUDA;
    }
    cudaError_t e = cudaMalloc(&L->dev_status, 256);
    if (e != cudaSuccess) {
        delete L;
        return e == cudaErrorMemoryAllocation ? MOE_ERR_OUT_OF_MEMORY : MOE_ERR_CUDA;
    }
    e = cudaMemset(L->dev_status, 0, 256);
    if (e != cudaSuccess) {
        cudaFree(L->dev_status);
        delete L;
        return MOE_ERR_CUDA;
    }
    *out = L;
    return MOE_OK;
}

moe_status moe_quantize_act(moe_layer* L, const uint16_t* x, int32_t tokens, uint8_t* codes,
                            uint8_t* scales, float* tensor_scale, void* workspace, void* stream) {
    if (!L || !codes || !scales || !tensor_scale || !workspace) return MOE_ERR_INVALID_ARGUMENT;
    if (tokens < 0 || tokens > L->desc.max_tokens) return MOE_ERR_INVALID_ARGUMENT;
    if (tokens > 0 && (!x || !aligned16(x) || !aligned16(codes))) return MOE_ERR_INVALID_ARGUMENT;
    const moe::Workspace ws = moe::workspace_layout(shape_of(L->desc), L->desc.max_tokens, workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(moe::launch_quant_act(x, tokens, L->desc.hidden, codes, scales,
                                             tensor_scale, ws.scal + moe::kScalAmax, st));
}

moe_status moe_quantize_weights(const float* w, int32_t matrices, int32_t rows, int32_t cols,
                                uint8_t* codes, uint8_t* scales, float* tensor_scale, void* stream) {
    if (!w || !codes || !scales || !tensor_scale) return MOE_ERR_INVALID_ARGUMENT;
    if (matrices < 1 || rows < 1 || cols < 64 || cols % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(w) || !aligned16(codes)) return MOE_ERR_INVALID_ARGUMENT;
    if ((size_t)matrices * rows * cols / 16 > (size_t)0xFFFFFFFF * 256)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(moe::launch_quant_weights(w, matrices, rows, cols, codes, scales,
                                                 tensor_scale, st));
}

moe_status moe_forward(moe_layer* L, const uint16_t* x, const uint8_t* xq_codes,
                       const uint8_t* xq_scales, const float* xq_tensor_scale, int32_t tokens,
                       const uint16_t* residual, float* y, uint16_t* x_next, void* workspace,
                       const moe_debug* dbg, void* stream) {
    if (!L || !workspace) return MOE_ERR_INVALID_ARGUMENT;
    if (tokens < 0 || tokens > L->desc.max_tokens) return MOE_ERR_INVALID_ARGUMENT;
    if (tokens == 0) return MOE_OK;
    const bool have_xq = xq_codes || xq_scales || xq_tensor_scale;
    if (have_xq && !(xq_codes && xq_scales && xq_tensor_scale)) return MOE_ERR_INVALID_ARGUMENT;
    if (!x || !y || !aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARGUMENT;
    if (have_xq && !aligned16(xq_codes)) return MOE_ERR_INVALID_ARGUMENT;
    if (x_next && !residual) return MOE_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return MOE_ERR_INVALID_ARGUMENT;

    const Shape s = shape_of(L->desc);
    const int T = tokens;
    const size_t P = (size_t)T * s.k;
    moe::Workspace ws = moe::workspace_layout(s, L->desc.max_tokens, workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;

    auto trace = [&](moe_step step, bool end) {
        if (L->trace_step != step) return cudaSuccess;
        cudaEvent_t ev = end ? L->trace_end : L->trace_start;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t ce = cudaStreamIsCapturing(st, &cs);
        if (ce != cudaSuccess) return ce;
        // inside a capture only an "external" record becomes a graph node
        return cs == cudaStreamCaptureStatusActive
                   ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
                   : cudaEventRecord(ev, st);
    };
#define MOE_STEP(step, call)                                                   \
    do {                                                                       \
        if (trace(step, false) != cudaSuccess) return MOE_ERR_CUDA;            \
        if ((call) != cudaSuccess) return MOE_ERR_CUDA;                         \
        if (trace(step, true) != cudaSuccess) return MOE_ERR_CUDA;             \
    } while (0)

    // S3 (unless the caller passed the NVFP4 form of x)
    if (have_xq) {
        ws.xq = const_cast<uint8_t*>(xq_codes);
        ws.xs = const_cast<uint8_t*>(xq_scales);
        ws.sx = const_cast<float*>(xq_tensor_scale);
    } else {
        MOE_STEP(MOE_STEP_QUANT, moe::launch_quant_act(x, T, s.H, ws.xq, ws.xs, ws.sx,
                                                         ws.scal + moe::kScalAmax, st));
    }
    // S1 + S2
    MOE_STEP(MOE_STEP_ROUTER, moe::launch_router(x, L->router_w, L->router_bias, T, s, ws.logits,
                                                 ws.idx, ws.w, st));
    // S4
    MOE_STEP(MOE_STEP_PERMUTE, moe::launch_permute(ws.idx, T, s, ws, st));
    // S5
    const moe::ExpertWeights g{L->gate.codes, L->gate.scales, L->gate.tensor_scale};
    const moe::ExpertWeights u{L->up.codes, L->up.scales, L->up.tensor_scale};
    const moe::ExpertWeights d{L->down.codes, L->down.scales, L->down.tensor_scale};
    MOE_STEP(MOE_STEP_GATEUP, moe::launch_gateup(s, T, g, u, L->desc.h_tensor_scale, ws, st));
    // S6
    MOE_STEP(MOE_STEP_DOWN, moe::launch_down(s, T, d, L->desc.h_tensor_scale, ws, residual, y,
                                             x_next, st));
#undef MOE_STEP

    if (dbg) {
        struct Copy { void* dst; const void* src; size_t bytes; } copies[] = {
            {dbg->logits, ws.logits, sizeof(float) * (size_t)T * s.E},
            {dbg->idx, ws.idx, sizeof(int32_t) * P},
            {dbg->weights, ws.w, sizeof(float) * P},
            {dbg->counts, ws.counts, sizeof(int32_t) * s.E},
            {dbg->offsets, ws.offsets, sizeof(int32_t) * (s.E + 1)},
            {dbg->perm, ws.perm, sizeof(int32_t) * P},
            {dbg->inv, ws.inv, sizeof(int32_t) * P},
            {dbg->hq, ws.hq, P * s.I / 2},
            {dbg->hs, ws.hs, P * s.I / 16},
            {dbg->xq_codes, ws.xq, (size_t)T * s.H / 2},
            {dbg->xq_scales, ws.xs, (size_t)T * s.H / 16},
            {dbg->xq_tensor_scale, ws.sx, sizeof(float)},
        };
        for (const Copy& c : copies) {
            if (!c.dst) continue;
            e = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDeviceToDevice, st);
            if (e != cudaSuccess) return MOE_ERR_CUDA;
        }
    }
    return MOE_OK;
}

moe_status moe_layer_status(moe_layer* L, void* stream) {
    if (!L) return MOE_ERR_INVALID_ARGUMENT;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, L->dev_status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (word == 0) return MOE_OK;
    if (cudaMemset(L->dev_status, 0, sizeof(word)) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_ERR_DEVICE_TIMEOUT;
}

moe_status moe_layer_set_trace(moe_layer* L, moe_step step, void* start_event, void* end_event) {
    if (!L) return MOE_ERR_INVALID_ARGUMENT;
    if (step != MOE_STEP_NONE && step != MOE_STEP_ROUTER && step != MOE_STEP_QUANT &&
        step != MOE_STEP_PERMUTE && step != MOE_STEP_GATEUP && step != MOE_STEP_DOWN)
        return MOE_ERR_INVALID_ARGUMENT;
    if (step != MOE_STEP_NONE && (!start_event || !end_event)) return MOE_ERR_INVALID_ARGUMENT;
    L->trace_step = step;
    L->trace_start = static_cast<cudaEvent_t>(start_event);
    L->trace_end = static_cast<cudaEvent_t>(end_event);
    return MOE_OK;
}

uint64_t moe_kernel_launches(void) { return moe::g_launches.load(std::memory_order_relaxed); }

void moe_destroy(moe_layer* L) {
    if (!L) return;
    if (L->dev_status) cudaFree(L->dev_status);
    delete L;
}

}  // extern "C"
