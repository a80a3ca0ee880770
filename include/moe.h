/*
 * nvfp4_moe -- C ABI of the routed-expert NVFP4 (W4A4) MoE layer for one GB300.
 *
 * The layer is the one the capy-flash engine runs for every token of its
 * 125B mixture-of-experts model: 48 layers x 512 routed experts
 * ("capy-flash v0.7.1: a 125B MoE on 64 GB of RAM ...", "What shipped"),
 * with the expert weights and the activations both in NVIDIA's NVFP4 format
 * (the GPU expert path is W4A4 inside a captured CUDA graph: same page,
 * "Why it matters"; the engine was built for NVFP4: capy-flash status post,
 * feedman.me repost, "What it's for"), and every expert the router picks is
 * computed (same post, "Where it stands").  On one GB300 every expert sits in
 * HBM, so there is no expert cache and no host offload.
 *
 * Steps of moe_forward, in order:
 *   S1 router logits  l[t,e] = sum_h x[t,h] * Wr[e,h] (+ b[e]), fp32 accumulate
 *   S2 top-k          k largest logits, ties to the lower expert index; weights
 *                     w = softmax over the k picked logits (renormalised)
 *   S3 quantise x     NVFP4: E2M1 codes, one E4M3 scale per 16 elements of a
 *                     row, one fp32 tensor scale per call (amax / 2688)
 *   S4 permutation    pairs p = t*k + j grouped by expert (token order inside
 *                     an expert): counts, offsets, perm, inv
 *   S5 gate/up        h = silu(Wg x_hat) * (Wu x_hat), requantised to NVFP4
 *                     with the static tensor scale desc.h_tensor_scale
 *   S6 down/combine   y[t] = sum_j w[t,j] * (Wd h_hat)(t,j) in slot order;
 *                     optional residual: x_next = bf16(residual + y)
 *
 * Quantiser Q (S3 and the requantisation in S5), every operation one IEEE fp32
 * operation with round-to-nearest-even and no fused multiply-add:
 *   per 16-element block: a = max|x_i|; q = a / (6 * s); S = E4M3(q) (RNE,
 *   saturating at 448); if S == 0 all codes are 0, else c_i = E2M1(x_i / (S*s))
 *   (RNE on |x|, saturating at 6, sign bit = sign of x_i).
 *
 * Where each call comes from
 *   The pages describe the engine, not a library: they fix what the layer
 *   computes (the passages are cited on each call below) and print no API.
 *   The four calls that carry the layer -- moe_layer_create (hold the
 *   experts), moe_quantize_act (S3), moe_forward (S1..S6) and moe_destroy --
 *   are this library's surface for that computation; the other calls size
 *   buffers, read status or measure, and have no counterpart on the pages.
 *
 * Conventions
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - NVFP4 codes: two E2M1 codes per byte, the even element in the low nibble;
 *     16-element blocks run along the contraction axis of the matrix.
 *   - Calls that take a stream only enqueue work; they never synchronise,
 *     allocate device memory, print or abort (moe_layer_create and
 *     moe_layer_status are the exceptions, stated below).
 *   - Errors are reported by the return value; arguments are validated before
 *     anything is enqueued, so an error return means nothing was enqueued.
 *   - Device-side waits are bounded; one that runs out records
 *     MOE_ERR_DEVICE_TIMEOUT in the layer's status word (moe_layer_status).
 */
#ifndef NVFP4_MOE_H
#define NVFP4_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARGUMENT = 1,  /* NULL / misaligned pointer, bad count      */
    MOE_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the supported ranges below */
    MOE_ERR_OUT_OF_MEMORY = 3,     /* host or device allocation in create      */
    MOE_ERR_CUDA = 4,              /* a CUDA runtime call failed               */
    MOE_ERR_DEVICE_TIMEOUT = 5,    /* a bounded device-side wait ran out       */
    MOE_ERR_PARTIAL_OVERFLOW = 6   /* a weighted down partial of the tensor-core
                                      path left the fp16 range (|w o| >= 65520):
                                      that forward's y is not valid            */
} moe_status;

/* Layer shape.  Supported: hidden % 64 == 0 and 64 <= hidden <= 8192;
 * inter % 64 == 0 and 64 <= inter <= 4096; 1 <= num_experts <= 1024;
 * 1 <= top_k <= min(num_experts, 32); 1 <= max_tokens <= 1048576;
 * h_tensor_scale a positive finite float; 0 <= route_keep <= top_k.
 * Otherwise MOE_ERR_UNSUPPORTED_SHAPE.
 *
 * route_keep: the route-tail skip.  The capy-flash status post ("Where it
 * stands") attributes another engine's faster single-card decode mostly to a
 * route tail skip that drops low-ranked experts which miss its expert cache,
 * while capy-flash computes every pick.  With route_keep = r (1 <= r < top_k)
 * the picks of rank 0 .. r-1 are always computed and a pick of rank >= r only
 * if its expert is marked resident (moe_layer_set_resident; with no mask
 * nothing is resident, so the whole tail is dropped); the router weights are
 * renormalised over the kept picks.  A dropped pick reads as expert -1 with
 * weight 0 in the debug outputs and has no permutation position (inv = -1).
 * route_keep = 0 (or top_k) computes every pick. */
typedef struct moe_layer_desc {
    int32_t hidden;        /* H */
    int32_t num_experts;   /* E */
    int32_t top_k;         /* k */
    int32_t inter;         /* I, expert intermediate width */
    int32_t max_tokens;    /* largest T any call on this layer will pass */
    uint32_t flags;        /* MOE_FLAG_* bits; other bits must be 0 */
    float h_tensor_scale;  /* static fp32 tensor scale of the SwiGLU output h */
    int32_t route_keep;    /* route-tail skip: ranks always computed; 0 = every pick */
} moe_layer_desc;

/* desc.flags: run every call through the per-step CUDA-core kernels (no fused
 * decode kernel, no tensor-core GEMMs); same results within rounding, for
 * cross-checking and measurement. */
#define MOE_FLAG_MULTI_KERNEL 1u

/* One NVFP4 weight tensor holding all experts of one projection, N x K per
 * expert, row-major with K (the contraction axis) innermost:
 *   codes        uint8 [E][N][K/2]   (16-byte aligned)
 *   scales       uint8 [E][N][K/16]  unsigned E4M3 block scales
 *   tensor_scale fp32  [E]           one tensor scale per expert matrix
 * gate and up: N = I, K = H.  down: N = H, K = I. */
typedef struct moe_nvfp4 {
    const uint8_t* codes;
    const uint8_t* scales;
    const float* tensor_scale;
} moe_nvfp4;

/* Optional copies of the intermediate results of moe_forward (any member may
 * be NULL; T = tokens of the call, P = T * k):
 *   logits  fp32  [T][E]        idx    int32 [T][k]     weights fp32 [T][k]
 *   counts  int32 [E]           offsets int32 [E+1]
 *   perm    int32 [P]  pair id (t*k + j) at each expert-grouped position
 *   inv     int32 [P]  expert-grouped position of each pair id
 *   hq      uint8 [P][I/2]   hs uint8 [P][I/16]  requantised h, row r = pair perm[r]
 *   xq_codes uint8 [T][H/2]  xq_scales uint8 [T][H/16]  xq_tensor_scale fp32 [1]
 *           the NVFP4 form of x the experts used
 *   phase_ns uint64 [2][16]  fused decode kernel only: %globaltimer stamps
 *           (ns) of the first ([0][.]) and the last ([1][.]) CTA in layer 0,
 *           by index: 0 start, 1 x staged, 2 router logits published,
 *           3 x quantised, 4 all logits polled, 12 top-k threshold found,
 *           13 top-k ranks done, 14 permutation and active list done,
 *           15 weight copies issued (issuing warp), 5 issue and CTA barrier
 *           done, 6 first gate/up rows landed, 7 gate/up and h published,
 *           8 all h polled, 9 first down rows landed, 10 down done, 11 layer
 *           end (left untouched by the per-step kernels) */
typedef struct moe_debug {
    float* logits;
    int32_t* idx;
    float* weights;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* inv;
    uint8_t* hq;
    uint8_t* hs;
    uint8_t* xq_codes;
    uint8_t* xq_scales;
    float* xq_tensor_scale;
    uint64_t* phase_ns;
} moe_debug;

typedef struct moe_layer moe_layer;

/* Static string naming a status (never NULL).  Library mechanics: no
 * counterpart on the pages. */
const char* moe_status_string(moe_status status);

/* Bytes of scratch memory one moe_forward / moe_quantize_act call needs for
 * this shape (at desc->max_tokens tokens); 0 if desc is invalid.  The caller
 * allocates it (256-byte aligned); one workspace may serve any number of
 * calls that run one after another on one stream; calls that may overlap
 * need separate workspaces.  Library mechanics (the caller owns every device
 * allocation): no counterpart on the pages. */
size_t moe_workspace_bytes(const moe_layer_desc* desc);

/* Bytes of the layer-private buffer moe_layer_create fills for calls with
 * more than 8 tokens (the tensor-core path); library mechanics, no
 * counterpart on the pages:
 *   - the router weights split into two bf16 parts, hi = RN_bf16(Wr) and
 *     lo = RN_bf16(Wr - hi) ([E][H] each), from which S1 runs on the tensor
 *     cores (hi + lo equals Wr to about 2^-17 relative): 4 E H bytes;
 *   - the gate, up and down block scales rearranged into the tiles the
 *     block-scaled MMA reads (a permutation of each scale array, same size:
 *     E I H / 16 bytes each).
 * 0 when the layer never takes that path (max_tokens < 9,
 * MOE_FLAG_MULTI_KERNEL, or H, I not multiples of 256), and 0 if desc is
 * invalid. */
size_t moe_packed_weight_bytes(const moe_layer_desc* desc);

/* Create a layer handle: one routed-expert layer whose experts all stay
 * resident in device memory.  Defines: one layer of the 48-layer x 512-expert
 * model ("capy-flash v0.7.1: a 125B MoE on 64 GB of RAM ...", "What
 * shipped"), its experts in NVFP4 (capy-flash status post, feedman.me
 * repost, "What it's for").  The pages keep most experts in host RAM and a
 * VRAM cache ("Capy Flash 125B MoE on two consumer GPUs", "Where the experts
 * live"); here every expert is in HBM, so there is no cache to manage.
 *   router_w     fp32 [E][H]
 *   router_bias  fp32 [E] or NULL
 *   gate, up     NVFP4 [E][I][H];  down  NVFP4 [E][H][I]   (host structs
 *                holding device pointers; the structs are copied)
 *   packed       device buffer of moe_packed_weight_bytes(desc) bytes
 *                (16-byte aligned), or NULL when that is 0; filled from
 *                router_w and the weight scales by kernels on `stream`, so
 *                the first forward must be ordered after them (same stream,
 *                or a synchronize)
 * Weights and `packed` are BORROWED: they must stay valid and unchanged for
 * the life of the layer.  The handle is a host object; create allocates one
 * small device status word with cudaMalloc on the current device, which
 * moe_destroy frees.  On error *out is set to NULL. */
moe_status moe_layer_create(const moe_layer_desc* desc, const float* router_w,
                            const float* router_bias, const moe_nvfp4* gate,
                            const moe_nvfp4* up, const moe_nvfp4* down, void* packed,
                            void* stream, moe_layer** out);

/* S3 alone: quantise bf16 x [T][H] to NVFP4 with one dynamic tensor scale.
 * Defines: the activation side of the W4A4 expert path ("capy-flash v0.7.1",
 * "Why it matters"), in NVIDIA's NVFP4 format (status post, "What it's for");
 * the quantiser Q itself is this library's reading, stated at the top of
 * this file.
 *   codes uint8 [T][H/2], scales uint8 [T][H/16], tensor_scale fp32 [1]
 * 0 <= T <= max_tokens (T == 0 writes tensor_scale = 1).  x 16-byte aligned.
 * workspace: moe_workspace_bytes(desc) bytes. */
moe_status moe_quantize_act(moe_layer* layer, const uint16_t* x, int32_t tokens,
                            uint8_t* codes, uint8_t* scales, float* tensor_scale,
                            void* workspace, void* stream);

/* Quantise fp32 weight matrices to NVFP4, one tensor scale per matrix
 * (the weight side of the W4A4 path, "capy-flash v0.7.1", "Why it matters";
 * the experts ship in NVFP4, status post, "What it's for")
 * -- amax of that matrix / 2688: w fp32 [M][rows][cols] -> codes uint8
 * [M][rows][cols/2], scales uint8 [M][rows][cols/16], tensor_scale fp32 [M].
 * cols % 64 == 0; w 16-byte aligned.  Needs no layer and no workspace. */
moe_status moe_quantize_weights(const float* w, int32_t matrices, int32_t rows, int32_t cols,
                                uint8_t* codes, uint8_t* scales, float* tensor_scale,
                                void* stream);

/* The layer, S1..S6, for T tokens (0 <= T <= max_tokens; T == 0 is a no-op).
 * Defines: the routed-expert MoE layer of "capy-flash v0.7.1" ("What
 * shipped": 48 layers x 512 routed experts; "Why it matters": W4A4 experts
 * inside a captured CUDA graph, decode bound by memory bandwidth), computing
 * every expert the router picks (status post, "Where it stands").
 * Up to 8 tokens (with T*k <= 128, hidden <= 4096, inter <= 2048) and no
 * caller-supplied xq, the call runs as one fused, cooperatively launched
 * kernel over every SM (see moe_stack_forward).  With more tokens (and hidden,
 * inter multiples of 256) S5 and S6 run as block-scaled FP4 grouped GEMMs on
 * the tensor cores, S6 writing router-weighted fp16 per-pair outputs that a
 * combine step sums per token in slot order (its workspace holds those
 * outputs: 2 * max_tokens * k * H bytes).  MOE_FLAG_MULTI_KERNEL selects the
 * per-step CUDA-core kernels for every call.
 *   x          bf16 [T][H], router input (16-byte aligned)
 *   xq_codes, xq_scales, xq_tensor_scale
 *              the NVFP4 form of x from moe_quantize_act, or all three NULL to
 *              quantise x inside this call (same quantiser); codes 16-byte,
 *              scales and tensor scale 4-byte aligned
 *   residual   NULL or bf16 [T][H]
 *   y          fp32 [T][H] output
 *   x_next     NULL or bf16 [T][H]: bf16(residual + y), needs residual
 *   workspace  moe_workspace_bytes(desc) bytes of scratch
 *   dbg        NULL or host struct of optional device outputs (moe_debug)
 * Asynchronous on `stream`; no host synchronisation; capturable in a CUDA
 * graph (no allocation, no host-side dependence on device results). */
moe_status moe_forward(moe_layer* layer, const uint16_t* x, const uint8_t* xq_codes,
                       const uint8_t* xq_scales, const float* xq_tensor_scale, int32_t tokens,
                       const uint16_t* residual, float* y, uint16_t* x_next, void* workspace,
                       const moe_debug* dbg, void* stream);

/* Size of the device scratch array behind moe_forward_noalloc (per device). */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)

/* moe_forward without a workspace, for callers that cannot allocate device
 * memory (no counterpart on the pages): code that runs where its host owns every device allocation (a
 * framework's caching allocator, an inference-server plugin that is handed
 * only buffers and a stream), or a latency-critical loop that must not call
 * cudaMalloc, which can synchronise the device.  (The pages describe no such
 * call; it has no counterpart there.)
 *
 * Same computation and outputs as moe_forward with internal quantisation of x
 * (arguments as there).  Its scratch is one file-scope device array of
 * MOE_NOALLOC_SCRATCH_BYTES bytes inside this library, which every device
 * that loads the library holds until the process exits.  The call itself
 * allocates nothing.
 *   - Capacity: the call runs the per-step CUDA-core kernels and is refused
 *     with MOE_ERR_UNSUPPORTED_SHAPE when their scratch for `tokens` tokens
 *     exceeds MOE_NOALLOC_SCRATCH_BYTES (for hidden 2048, 512 experts,
 *     top-10, intermediate 512 that allows up to 658 tokens).
 *   - Shared scratch: all calls in the process share the array of their
 *     device and it keeps the last call's contents (each call clears what it
 *     needs cleared).  Calls on one stream run one after another and are
 *     safe; calls that can overlap on the GPU (other streams, other threads)
 *     race on the array and give wrong results.
 *   - The first call in a CUDA context looks up the array's device address
 *     (with that context current) and caches it under the context's unique
 *     id; a context created later (after cudaDeviceReset, say) gets a fresh
 *     lookup on its first call.  Make the first call before any stream
 *     capture.
 *   - The current device must be the one the layer was created on. */
moe_status moe_forward_noalloc(moe_layer* layer, const uint16_t* x, int32_t tokens,
                               const uint16_t* residual, float* y, uint16_t* x_next,
                               void* stream);

/* Batch-1..8 decode through a stack of layers in ONE kernel launch.
 * Defines: decode through the model's stacked MoE layers ("capy-flash
 * v0.7.1", "What shipped": 48 layers), each layer as in moe_forward, with
 * the residual add between layers:
 * x_{l+1} = bf16(x_l + y_l), l = 0 .. n_layers-1 (the residual add between
 * stacked MoE layers), all layers' S1..S6 inside one persistent kernel whose
 * phases are separated by bounded grid barriers.
 *   layers    host array of n_layers handles (1 <= n_layers <= 64), all with
 *             the same shape; the kernel runs on layers[0]'s device and
 *             reports timeouts in layers[0]'s status word
 *   x         bf16 [T][H] input of layer 0;  x_out  bf16 [T][H] output of the
 *             last layer (may alias nothing else)
 *   ys        NULL, or a host array of n_layers device pointers (each NULL
 *             or fp32 [T][H]) receiving every layer's y
 *   workspace moe_workspace_bytes(&layers[0]'s desc) bytes
 * Requires 1 <= T <= 8, T*k <= 128, hidden <= 4096, inter <= 2048, else
 * MOE_ERR_UNSUPPORTED_SHAPE (larger batches: call moe_forward per layer). */
moe_status moe_stack_forward(moe_layer* const* layers, int32_t n_layers, const uint16_t* x,
                             int32_t tokens, uint16_t* x_out, float* const* ys,
                             void* workspace, void* stream);

/* Route-tail skip: the experts that count as resident (never skipped) for
 * later forwards on this layer.  resident: NULL (no expert resident) or a
 * device array of num_experts bytes, nonzero = resident, BORROWED (it must stay
 * valid while forwards that use it run; its contents are read by those
 * forwards, so it may change between calls).  Only matters when
 * desc.route_keep is between 1 and top_k - 1.  Defines: the cache test of the
 * skip (status post, "Where it stands"); on one GB300 every expert is in HBM,
 * so "resident" is whatever the caller marks.  Host-only call. */
moe_status moe_layer_set_resident(moe_layer* layer, const uint8_t* resident);

/* Synchronise `stream`, then read and clear the layer's device status word.
 * Library mechanics (failure detection): no counterpart on the pages.
 * Returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT (takes precedence when both were
 * recorded), MOE_ERR_PARTIAL_OVERFLOW (the tensor-core path stores each
 * pair's weighted down output w * o as an fp16 partial before the combine; a
 * value at or beyond 65520 in magnitude would round to infinity, so the
 * epilogue records it instead of passing it on silently), or MOE_ERR_CUDA for
 * a failed synchronisation (e.g. a sticky error from an earlier launch). */
moe_status moe_layer_status(moe_layer* layer, void* stream);

/* Steps that moe_layer_set_trace can bracket with CUDA events. */
typedef enum moe_step {
    MOE_STEP_NONE = 0,
    MOE_STEP_ROUTER = 1,   /* S1 + S2 */
    MOE_STEP_QUANT = 3,    /* S3 (only when moe_forward quantises x itself) */
    MOE_STEP_PERMUTE = 4,  /* S4 */
    MOE_STEP_GATEUP = 5,   /* S5 */
    MOE_STEP_DOWN = 6      /* S6 (with the weighted combine) */
} moe_step;
/* A call that runs as the fused decode kernel (tokens <= 8) has one kernel for
 * all steps: any traced step brackets that kernel. */

/* Profiling hook (measurement; no counterpart on the pages): from now on
 * every moe_forward on this layer records
 * start_event (a cudaEvent_t, as void*) on its stream just before the kernels
 * of `step` and end_event just after them.  MOE_STEP_NONE (or NULL events)
 * turns it off.  The events are borrowed; a forward captured into a CUDA
 * graph captures the two records as event nodes.  Host-only call. */
moe_status moe_layer_set_trace(moe_layer* layer, moe_step step, void* start_event,
                               void* end_event);

/* Device scratch the wait self-test needs (caller-allocated, 16-byte aligned). */
#define MOE_SELFTEST_SCRATCH_BYTES 8192u

/* Self-test of the failure detection of the persistent kernels: on the current
 * device, one CTA runs the same bounded waits the fused decode kernel uses —
 * a poll of tagged words that nothing writes, then a wait on an mbarrier that
 * nothing arrives on — so both must run out (about a second each), set the
 * device timeout code in their status word, and return without leaving work
 * in flight; the CUDA context stays usable.  Clears `scratch`
 * (MOE_SELFTEST_SCRATCH_BYTES of device memory, 16-byte aligned) on `stream`,
 * synchronises the stream and copies the two status words to status_out[2]
 * (host memory; may be NULL).  Returns MOE_OK when both waits ran out and
 * reported, MOE_ERR_INVALID_ARGUMENT for a bad scratch pointer, MOE_ERR_CUDA
 * for a CUDA error or any other outcome.  A check of this library, not a step
 * of the layer (the pages have no counterpart). */
moe_status moe_selftest_bounded_waits(void* scratch, uint32_t* status_out, void* stream);

/* Number of CUDA kernels this library has launched (or added to a stream
 * capture) in this process so far; for launch accounting (measurement; no
 * counterpart on the pages). */
uint64_t moe_kernel_launches(void);

/* Free the handle and its status word.  NULL is a no-op.  Does not free the
 * borrowed weights or buffers.  The end of the layer's life in this library
 * (the counterpart of moe_layer_create; the pages have no API). */
void moe_destroy(moe_layer* layer);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_MOE_H */
