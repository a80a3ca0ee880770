// moe_forward_noalloc: the layer forward for callers that cannot allocate
// device memory.  Its scratch is a fixed file-scope device array of the
// library instead of a caller-provided workspace; every other step is the
// same launch sequence as moe_forward.
#include <mutex>

#include <cuda.h>

#include "kernels.h"
#include "layer.h"
#include "moe.h"

namespace {

// Scratch of every moe_forward_noalloc call on a device.  Each device that
// loads the library holds one copy until the process exits.  In host code the
// name is only a stand-in: kernels get the device address looked up below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// The array's device address belongs to a CUDA context: a context created
// later on the same device (after cudaDeviceReset, for instance) loads the
// module again, possibly elsewhere.  So the address is cached per context,
// keyed on the context's unique id (cuCtxGetId: never reused within a
// process), and looked up again with that context current when the id is new.
// The two driver calls are reached through the runtime's entry-point query,
// so the library does not link the driver library itself.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CachedScratch {
    unsigned long long ctx_id;
    void* addr;
};
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mu;
CachedScratch g_scratch[kMaxContexts] = {};
int g_scratch_n = 0;

template <class Fn>
Fn driver_fn(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// Unique id of the context current on this thread for device `dev`.  A thread
// that has made no runtime call yet has none: cudaSetDevice makes the
// device's primary context current (it allocates nothing).
moe_status current_context_id(int dev, unsigned long long* id) {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id) return MOE_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
    if (ctx == nullptr) {
        if (cudaSetDevice(dev) != cudaSuccess) return MOE_ERR_CUDA;
        if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return MOE_ERR_CUDA;
    }
    return get_id(ctx, id) == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// Device address of g_noalloc_scratch in the current context, looked up once
// per context (with that context current) and cached.
moe_status scratch_in_current_context(int dev, void** out) {
    unsigned long long id = 0;
    const moe_status st = current_context_id(dev, &id);
    if (st != MOE_OK) return st;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    for (int i = 0; i < (g_scratch_n < kMaxContexts ? g_scratch_n : kMaxContexts); ++i) {
        if (g_scratch[i].ctx_id == id) {
            *out = g_scratch[i].addr;
            return MOE_OK;
        }
    }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    // a full table (more contexts than kMaxContexts in one process) recycles
    // its entries in the order they were made, oldest first
    const int slot = g_scratch_n < kMaxContexts ? g_scratch_n : g_scratch_n % kMaxContexts;
    ++g_scratch_n;
    g_scratch[slot] = CachedScratch{id, p};
    *out = p;
    return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_forward_noalloc(moe_layer* L, const uint16_t* x, int32_t tokens,
                                          const uint16_t* residual, float* y, uint16_t* x_next,
                                          void* stream) {
    if (!L) return MOE_ERR_INVALID_ARGUMENT;
    if (tokens < 0 || tokens > L->desc.max_tokens) return MOE_ERR_INVALID_ARGUMENT;
    if (tokens == 0) return MOE_OK;
    if (!x || !y || !aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARGUMENT;
    if (x_next && !residual) return MOE_ERR_INVALID_ARGUMENT;

    const moe::Shape s{L->desc.hidden, L->desc.num_experts, L->desc.top_k, L->desc.inter};
    // the scratch is laid out for exactly this call's token count
    if (moe::workspace_layout(s, tokens, nullptr, false).bytes > MOE_NOALLOC_SCRATCH_BYTES)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev != L->device) return MOE_ERR_INVALID_ARGUMENT;
    void* base = nullptr;
    const moe_status st0 = scratch_in_current_context(dev, &base);
    if (st0 != MOE_OK) return st0;

    const moe::Workspace ws = moe::workspace_layout(s, tokens, base, false);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const moe::ExpertWeights g{L->gate.codes, L->gate.scales, L->gate.tensor_scale};
    const moe::ExpertWeights u{L->up.codes, L->up.scales, L->up.tensor_scale};
    const moe::ExpertWeights d{L->down.codes, L->down.scales, L->down.tensor_scale};
    // the activation max-magnitude word is cleared inside launch_quant_act;
    // every other scratch region is fully written before it is read
    if (moe::launch_quant_act(x, tokens, s.H, ws.xq, ws.xs, ws.sx, ws.scal + moe::kScalAmax, st) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    const int keep = L->desc.route_keep >= 1 && L->desc.route_keep < s.k ? L->desc.route_keep : s.k;
    if (moe::launch_router(x, L->router_w, L->router_bias, tokens, s, ws.logits, ws.idx, ws.w, st, keep,
                           L->resident) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (moe::launch_permute(ws.idx, tokens, s, ws, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (moe::launch_gateup(s, tokens, g, u, L->desc.h_tensor_scale, ws, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (moe::launch_down(s, tokens, d, L->desc.h_tensor_scale, ws, residual, y, x_next, st) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
