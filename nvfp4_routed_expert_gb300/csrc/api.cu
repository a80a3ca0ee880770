// C ABI of the NVFP4 MoE layer: argument checks, workspace carving and the
// launch sequence S1..S6 on the caller's stream.  No call here allocates
// device memory except moe_layer_create (one status word).
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>

#include "common.cuh"
#include "decode.h"
#include "kernels.h"
#include "prefill.h"
#include "layer.h"
#include "moe.h"

namespace moe {

namespace {

constexpr size_t kAlign = 256;
std::atomic<uint64_t> g_launches{0};

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

}  // namespace

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

Workspace workspace_layout(const Shape& s, int Tm, void* base, bool with_prefill, bool with_decode) {
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
    const size_t ngroups = (size_t)perm_groups((int)nchunks);
    w.group_cnt = ngroups ? reinterpret_cast<int32_t*>(take(sizeof(int32_t) * ngroups * s.E)) : nullptr;
    w.perm = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * Pm));
    w.inv = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * Pm));
    w.xq = take((size_t)Tm * s.H / 2);
    w.xs = take((size_t)Tm * s.H / 16);
    w.hq = take(Pm * s.I / 2);
    w.hs = take(Pm * s.I / 16);
    const size_t Tx = Tm < 8 ? (size_t)Tm : 8;
    w.xbuf0 = reinterpret_cast<uint16_t*>(take(Tx * s.H * 2));
    w.xbuf1 = reinterpret_cast<uint16_t*>(take(Tx * s.H * 2));
    if (with_decode) w.tags = reinterpret_cast<uint64_t*>(take(decode_tag_bytes(s, (int)Tx)));
    if (with_prefill) {
        w.mtiles = reinterpret_cast<int4*>(take(sizeof(int4) * (Pm / 128 + s.E + 1)));
        w.hs_tiled = take((Pm / 128 + s.E + 1) * (size_t)(s.I / 16) * 128);
        w.partial = reinterpret_cast<__half*>(take(sizeof(__half) * Pm * s.H));
        w.wperm = reinterpret_cast<float*>(take(sizeof(float) * Pm));
    }
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
    if (d->flags & ~MOE_FLAG_MULTI_KERNEL) return false;
    if (!(d->h_tensor_scale > 0.0f) || !std::isfinite(d->h_tensor_scale)) return false;
    if (d->route_keep < 0 || d->route_keep > d->top_k) return false;
    return true;
}

Shape shape_of(const moe_layer_desc& d) { return Shape{d.hidden, d.num_experts, d.top_k, d.inter}; }

// Whether calls on this layer can take the tensor-core prefill path.
bool uses_prefill(const moe_layer_desc& d) {
    return d.max_tokens >= moe::kPrefillMinTokens && !(d.flags & MOE_FLAG_MULTI_KERNEL) &&
           moe::prefill_supported(shape_of(d));
}

// Whether S1 of the tensor-core path runs on the tensor cores (it needs the
// packed bf16 copy of the router weights).
bool uses_router_tc(const moe_layer_desc& d) {
    return uses_prefill(d) && moe::router_tc_supported(shape_of(d));
}

// Whether calls on this layer can take the fused decode kernel.
bool uses_decode(const moe_layer_desc& d) { return !(d.flags & MOE_FLAG_MULTI_KERNEL); }

// The packed buffer of a layer on the tensor-core path: the router's bf16 hi
// and lo parts, then the gate, up and down block scales in the tiled layout.
size_t packed_bytes(const Shape& s) {
    return moe::router_split_bytes(s) + 2 * moe::tiled_scale_bytes((size_t)s.E * s.I, s.H) +
           moe::tiled_scale_bytes((size_t)s.E * s.H, s.I);
}

moe::Workspace layout_of(const moe_layer_desc& d, void* base) {
    return moe::workspace_layout(shape_of(d), d.max_tokens, base, uses_prefill(d), uses_decode(d));
}

bool nvfp4_ok(const moe_nvfp4* w) {
    return w && w->codes && w->scales && w->tensor_scale && (reinterpret_cast<uintptr_t>(w->codes) & 15u) == 0;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Record the layer's trace start/end event on st; inside a stream capture only
// an "external" record becomes a graph node.
cudaError_t record_trace(const moe_layer* L, bool end, cudaStream_t st) {
    cudaEvent_t ev = end ? L->trace_end : L->trace_start;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t ce = cudaStreamIsCapturing(st, &cs);
    if (ce != cudaSuccess) return ce;
    return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
                                               : cudaEventRecord(ev, st);
}

// Ranks the route-tail skip always computes (top_k: every pick).
int route_keep(const moe_layer* L) {
    const int r = L->desc.route_keep;
    return r >= 1 && r < L->desc.top_k ? r : L->desc.top_k;
}

moe::DecodeLayer decode_layer(const moe_layer* L, float* y) {
    moe::DecodeLayer d{};
    d.wr = L->router_w;
    d.bias = L->router_bias;
    d.gc = L->gate.codes;
    d.gs = L->gate.scales;
    d.gts = L->gate.tensor_scale;
    d.uc = L->up.codes;
    d.us = L->up.scales;
    d.uts = L->up.tensor_scale;
    d.dc = L->down.codes;
    d.ds = L->down.scales;
    d.dts = L->down.tensor_scale;
    d.resident = L->resident;
    d.keep = route_keep(L);
    d.y = y;
    return d;
}

void fill_decode_params(moe::DecodeParams& p, const Shape& s, int T, const moe::Workspace& ws,
                        const moe_layer* L) {
    p.T = T;
    p.H = s.H;
    p.E = s.E;
    p.k = s.k;
    p.I = s.I;
    p.h_scale = L->desc.h_tensor_scale;
    p.tags = ws.tags;
    p.logits = ws.logits;
    p.idx = ws.idx;
    p.w = ws.w;
    p.counts = ws.counts;
    p.offsets = ws.offsets;
    p.perm = ws.perm;
    p.inv = ws.inv;
    p.xq = ws.xq;
    p.xs = ws.xs;
    p.sx = ws.sx;
    p.hq = ws.hq;
    p.hs = ws.hs;
    p.err = L->dev_status;
    p.phase_ns = nullptr;
    p.debug = false;
}

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
        case MOE_ERR_PARTIAL_OVERFLOW: return "MOE_ERR_PARTIAL_OVERFLOW";
    }
    return "MOE_ERR_UNKNOWN";
}

size_t moe_workspace_bytes(const moe_layer_desc* desc) {
    if (!desc_ok(desc)) return 0;
    return layout_of(*desc, nullptr).bytes;
}

size_t moe_packed_weight_bytes(const moe_layer_desc* desc) {
    if (!desc_ok(desc) || !uses_router_tc(*desc)) return 0;
    return packed_bytes(shape_of(*desc));
}

moe_status moe_layer_create(const moe_layer_desc* desc, const float* router_w,
                            const float* router_bias, const moe_nvfp4* gate, const moe_nvfp4* up,
                            const moe_nvfp4* down, void* packed, void* stream, moe_layer** out) {
    if (!out) return MOE_ERR_INVALID_ARGUMENT;
    *out = nullptr;
    if (!desc) return MOE_ERR_INVALID_ARGUMENT;
    if (!desc_ok(desc)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!router_w || !aligned16(router_w) || !nvfp4_ok(gate) || !nvfp4_ok(up) || !nvfp4_ok(down))
        return MOE_ERR_INVALID_ARGUMENT;
    const bool router_tc = uses_router_tc(*desc);
    if (router_tc && (!packed || !aligned16(packed))) return MOE_ERR_INVALID_ARGUMENT;
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
    if (e == cudaSuccess && router_tc) {
        const Shape s = shape_of(*desc);
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        uint16_t* hi = static_cast<uint16_t*>(packed);
        uint16_t* lo = hi + (size_t)s.E * s.H;
        e = moe::launch_router_split(router_w, s.E, s.H, hi, lo, st);
        L->router_hi = hi;
        L->router_lo = lo;
        uint8_t* t = static_cast<uint8_t*>(packed) + moe::router_split_bytes(s);
        const size_t gu = moe::tiled_scale_bytes((size_t)s.E * s.I, s.H);
        L->gate_sf_tiled = t;
        L->up_sf_tiled = t + gu;
        L->down_sf_tiled = t + 2 * gu;
        if (e == cudaSuccess) e = moe::launch_tile_scales(gate->scales, (size_t)s.E * s.I, s.H, t, st);
        if (e == cudaSuccess) e = moe::launch_tile_scales(up->scales, (size_t)s.E * s.I, s.H, t + gu, st);
        if (e == cudaSuccess)
            e = moe::launch_tile_scales(down->scales, (size_t)s.E * s.H, s.I, t + 2 * gu, st);
    }
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
    const moe::Workspace ws = layout_of(L->desc, workspace);
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
    // xq codes are read in 16-byte pieces, its scales in 4-byte pieces (the
    // tensor-core gather) and the tensor scale as one float
    if (have_xq && (!aligned16(xq_codes) || (reinterpret_cast<uintptr_t>(xq_scales) & 3u) ||
                    (reinterpret_cast<uintptr_t>(xq_tensor_scale) & 3u)))
        return MOE_ERR_INVALID_ARGUMENT;
    if (x_next && !residual) return MOE_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return MOE_ERR_INVALID_ARGUMENT;

    const Shape s = shape_of(L->desc);
    const int T = tokens;
    const size_t P = (size_t)T * s.k;
    moe::Workspace ws = layout_of(L->desc, workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    const bool fused = !have_xq && !(L->desc.flags & MOE_FLAG_MULTI_KERNEL) &&
                       moe::decode_supported(s, T);
    const bool tensor_core = !fused && uses_prefill(L->desc) && T >= moe::kPrefillMinTokens;

    auto trace = [&](moe_step step, bool end) {
        if (L->trace_step != step) return cudaSuccess;
        return record_trace(L, end, st);
    };
#define MOE_STEP(step, call)                                                   \
    do {                                                                       \
        if (trace(step, false) != cudaSuccess) return MOE_ERR_CUDA;            \
        if ((call) != cudaSuccess) return MOE_ERR_CUDA;                         \
        if (trace(step, true) != cudaSuccess) return MOE_ERR_CUDA;             \
    } while (0)

    if (fused) {
        // one kernel: every step is inside it, so any traced step brackets it
        moe::DecodeParams prm;
        fill_decode_params(prm, s, T, ws, L);
        prm.L = 1;
        prm.layer[0] = decode_layer(L, y);
        prm.x_in = x;
        prm.residual0 = residual;
        prm.x_out = x_next;
        prm.phase_ns = dbg ? dbg->phase_ns : nullptr;
        prm.debug = dbg != nullptr;   // the kernel writes its inspection outputs only when asked
        if (L->trace_step != MOE_STEP_NONE && trace(L->trace_step, false) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (moe::launch_decode(prm, st) != cudaSuccess) return MOE_ERR_CUDA;
        if (L->trace_step != MOE_STEP_NONE && trace(L->trace_step, true) != cudaSuccess)
            return MOE_ERR_CUDA;
    } else {
    if (have_xq) {   // the caller passed the NVFP4 form of x: no S3
        ws.xq = const_cast<uint8_t*>(xq_codes);
        ws.xs = const_cast<uint8_t*>(xq_scales);
        ws.sx = const_cast<float*>(xq_tensor_scale);
    }
    uint32_t* amax = ws.scal + moe::kScalAmax;
    if (tensor_core && L->router_hi) {
        // S1 on the tensor cores, which also takes S3's max |x| from the x
        // tiles it reads; S2; then S3's quantiser pass
        auto router_tc = [&]() {
            cudaError_t r = have_xq ? cudaSuccess : cudaMemsetAsync(amax, 0, sizeof(uint32_t), st);
            if (r == cudaSuccess)
                r = moe::launch_router_tc(x, L->router_hi, L->router_lo, L->router_bias, T, s, ws.logits,
                                          have_xq ? nullptr : amax, L->dev_status, st);
            return r != cudaSuccess ? r : moe::launch_topk(ws.logits, T, s, ws.idx, ws.w, st, route_keep(L),
                                                           L->resident);
        };
        MOE_STEP(MOE_STEP_ROUTER, router_tc());
        if (!have_xq)
            MOE_STEP(MOE_STEP_QUANT, moe::launch_quant_act_given_amax(x, T, s.H, ws.xq, ws.xs, ws.sx, amax, st));
    } else {
        // S3, then S1 + S2
        if (!have_xq) MOE_STEP(MOE_STEP_QUANT, moe::launch_quant_act(x, T, s.H, ws.xq, ws.xs, ws.sx, amax, st));
        MOE_STEP(MOE_STEP_ROUTER, moe::launch_router(x, L->router_w, L->router_bias, T, s, ws.logits,
                                                     ws.idx, ws.w, st, route_keep(L), L->resident));
    }
    // S4
    MOE_STEP(MOE_STEP_PERMUTE, moe::launch_permute(ws.idx, T, s, ws, st));
    const moe::ExpertWeights g{L->gate.codes, L->gate.scales, L->gate.tensor_scale, L->gate_sf_tiled};
    const moe::ExpertWeights u{L->up.codes, L->up.scales, L->up.tensor_scale, L->up_sf_tiled};
    const moe::ExpertWeights d{L->down.codes, L->down.scales, L->down.tensor_scale, L->down_sf_tiled};
    if (tensor_core) {
        // S5 and S6 (+ combine): block-scaled FP4 grouped GEMMs on the tensor cores
        MOE_STEP(MOE_STEP_GATEUP, moe::launch_prefill_gateup(s, g, u, L->desc.h_tensor_scale, ws,
                                                             L->dev_status, st));
        MOE_STEP(MOE_STEP_DOWN, moe::launch_prefill_down(s, T, d, L->desc.h_tensor_scale, ws, residual,
                                                         y, x_next, L->dev_status, st));
    } else {
        // S5
        MOE_STEP(MOE_STEP_GATEUP, moe::launch_gateup(s, T, g, u, L->desc.h_tensor_scale, ws, st));
        // S6
        MOE_STEP(MOE_STEP_DOWN, moe::launch_down(s, T, d, L->desc.h_tensor_scale, ws, residual, y,
                                                 x_next, st));
    }
#undef MOE_STEP
    }

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

moe_status moe_stack_forward(moe_layer* const* layers, int32_t n_layers, const uint16_t* x,
                             int32_t tokens, uint16_t* x_out, float* const* ys, void* workspace,
                             void* stream) {
    if (!layers || n_layers < 1 || !workspace || !x || !x_out) return MOE_ERR_INVALID_ARGUMENT;
    if (n_layers > moe::kDecodeMaxLayers) return MOE_ERR_UNSUPPORTED_SHAPE;
    const moe_layer* L0 = layers[0];
    if (!L0) return MOE_ERR_INVALID_ARGUMENT;
    for (int l = 1; l < n_layers; ++l) {
        const moe_layer* Ll = layers[l];
        if (!Ll) return MOE_ERR_INVALID_ARGUMENT;
        if (Ll->desc.hidden != L0->desc.hidden || Ll->desc.num_experts != L0->desc.num_experts ||
            Ll->desc.top_k != L0->desc.top_k || Ll->desc.inter != L0->desc.inter ||
            Ll->desc.h_tensor_scale != L0->desc.h_tensor_scale || Ll->device != L0->device)
            return MOE_ERR_INVALID_ARGUMENT;
    }
    if (tokens < 0 || tokens > L0->desc.max_tokens) return MOE_ERR_INVALID_ARGUMENT;
    if (tokens == 0) return MOE_OK;
    if (!aligned16(x) || !aligned16(x_out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MOE_ERR_INVALID_ARGUMENT;
    const Shape s = shape_of(L0->desc);
    if (!moe::decode_supported(s, tokens)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const moe::Workspace ws = layout_of(L0->desc, workspace);
    moe::DecodeParams prm;
    fill_decode_params(prm, s, tokens, ws, L0);
    prm.L = n_layers;
    for (int l = 0; l < n_layers; ++l) {
        float* y = ys ? ys[l] : nullptr;
        if (y && !aligned16(y)) return MOE_ERR_INVALID_ARGUMENT;
        prm.layer[l] = decode_layer(layers[l], y);
    }
    prm.x_in = x;
    prm.residual0 = x;
    prm.x_out = x_out;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // layers[0]'s trace (any step) brackets the single kernel of the stack
    const bool traced = L0->trace_step != MOE_STEP_NONE;
    if (traced && record_trace(L0, false, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (moe::launch_decode(prm, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (traced && record_trace(L0, true, st) != cudaSuccess) return MOE_ERR_CUDA;
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
    return (word & moe::kDevErrTimeout) ? MOE_ERR_DEVICE_TIMEOUT : MOE_ERR_PARTIAL_OVERFLOW;
}

moe_status moe_layer_set_resident(moe_layer* L, const uint8_t* resident) {
    if (!L) return MOE_ERR_INVALID_ARGUMENT;
    L->resident = resident;
    return MOE_OK;
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

moe_status moe_selftest_bounded_waits(void* scratch, uint32_t* status_out, void* stream) {
    if (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 15u)) return MOE_ERR_INVALID_ARGUMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t* err = static_cast<uint32_t*>(scratch);                   // 2 words
    const uint64_t* words = reinterpret_cast<const uint64_t*>(static_cast<uint8_t*>(scratch) + 256);
    const int n = (int)((MOE_SELFTEST_SCRATCH_BYTES - 256) / sizeof(uint64_t));
    if (cudaMemsetAsync(scratch, 0, MOE_SELFTEST_SCRATCH_BYTES, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (moe::launch_selftest_waits(words, n, err, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t h[2] = {0, 0};
    if (cudaMemcpy(h, err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (status_out) {
        status_out[0] = h[0];
        status_out[1] = h[1];
    }
    return (h[0] == moe::kDevErrTimeout && h[1] == moe::kDevErrTimeout) ? MOE_OK : MOE_ERR_CUDA;
}

uint64_t moe_kernel_launches(void) { return moe::g_launches.load(std::memory_order_relaxed); }

void moe_destroy(moe_layer* L) {
    if (!L) return;
    if (L->dev_status) cudaFree(L->dev_status);
    delete L;
}

}  // extern "C"
