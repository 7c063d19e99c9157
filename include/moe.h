/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed-expert MoE FFN layer.
 *
 * One layer of a DeepSeek-V3-class mixture of experts with FP8 expert
 * weights:
 *
 *   logits   L[t][e] = x[t] . Wr[e] + b[e]                      (fp32)
 *   routing  ids[t] = top-k of L[t] (ties -> lower index),
 *            w[t][j] = softmax of the selected logits (renormalised)
 *   grouping tokens of one expert become contiguous rows
 *   experts  h = SiLU(x Wg^T) * (x Wu^T);  o = h Wd^T            (FP8, 128x128 block scales)
 *   combine  y[t] = o_shared(t) + sum_j w[t][j] * o_{ids[t][j]}(t)   (bf16)
 *
 * Sources (web pages; none published code):
 *  - "KTransformers deep dive" (chenxutan.com/d/5425.html), section 1.2:
 *    256 routed experts and 1 shared expert, a router sends every token to
 *    8 experts; section 2.2: tokens that hit the same expert are batched so
 *    that per-token GEMVs become one GEMM per expert; weights are repacked
 *    once at load time for the compute unit.
 *  - "CPU-GPU hybrid inference" article on the OSDI'26 paper (xingyun.xin):
 *    SmallEP section and Fig. 5 (gating and sorting before dispatch; expert
 *    outputs returned to their tokens and reduced with the gate weights);
 *    "Native FP8 GEMV" section and Fig. 9-10 (E4M3FN weights, one scale per
 *    128-element input block, block partial sums scaled once);
 *    "CPU fine-grained parallelism" section (gate and up side by side, then
 *    activation and elementwise product, then down).
 *  Readings where the pages are silent: softmax scoring with renormalised
 *  top-k, SiLU, shared-expert weight 1, per-token 1x128 E4M3 quantisation
 *  of the activations x and h (s = amax/448), no residual in y.
 *
 * Conventions
 *  - Every pointer in a struct or argument is a DEVICE pointer unless its
 *    comment says HOST.  Streams are cudaStream_t values passed as void*
 *    (NULL = the legacy default stream).
 *  - Asynchrony: calls validate their arguments on the host, enqueue work on
 *    the given stream and return; nothing waits for the GPU except
 *    moe_create(_ex), moe_destroy, moe_get_device_status, moe_profile_read
 *    and moe_forward_host.
 *  - Ownership: moe_create copies (and repacks) every weight into memory
 *    the layer owns; the caller may free its weight buffers once it
 *    returns.  Activations, outputs and the workspace are caller-owned;
 *    no call after moe_create allocates device memory.
 *  - Errors: every call returns a moe_status; argument errors are found
 *    before anything is enqueued; nothing aborts, traps or throws.  Faults
 *    found by the kernels (an expert id out of range, a pipeline wait that
 *    gave up) set bits in a device word read by moe_get_device_status.
 *    moe_last_error() gives a thread-local message for the last failure.
 *  - Limits: hidden and inter multiples of 128; 1 <= top_k <= 32;
 *    top_k <= n_experts <= 1024; shared_inter == inter; T*top_k < 2^31.
 *    x, y and all weight pointers 16-byte aligned; workspace 256-byte aligned.
 *  - Devices: a layer lives on the device that was current at moe_create.
 *    Every call that enqueues work must be made with that device current;
 *    otherwise it returns MOE_ERR_INVALID_ARG before enqueuing anything.
 *    moe_destroy selects the layer's device itself.
 *  - Thread safety: one handle may be used by one stream at a time; separate
 *    handles are independent.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1
#define MOE_DECODE_MAX_T 64      /* largest T accepted by moe_forward_decode */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,     /* null pointer, bad size, misaligned buffer  */
    MOE_ERR_UNSUPPORTED = 2,     /* shape outside the limits above             */
    MOE_ERR_WORKSPACE = 3,       /* workspace smaller than moe_workspace_bytes  */
    MOE_ERR_CUDA = 4,            /* a CUDA runtime call failed                 */
    MOE_ERR_DEVICE_CHECK = 5,    /* a kernel flagged bad data (device word)    */
    MOE_ERR_TIMEOUT = 6          /* a kernel wait gave up (device word)        */
} moe_status;

/* Bits of the device status word (moe_get_device_status).  The kernels
 * check every expert id and every permuted row they index with; a bad one
 * sets its bit and is clamped (ids) or skipped (rows), so no access leaves
 * the buffers.  The results of that call are then undefined. */
#define MOE_DEV_BAD_EXPERT_ID  0x1u   /* a routing id outside [0, n_experts)  */
#define MOE_DEV_BAD_ROW        0x2u   /* a permutation row outside its range  */
#define MOE_DEV_WAIT_TIMEOUT   0x4u   /* a pipeline wait hit its limit        */

typedef enum {
    MOE_MODE_ROUTE = 0,          /* moe_route / moe_route_from_logits          */
    MOE_MODE_PREFILL = 1,        /* moe_forward_prefill                        */
    MOE_MODE_DECODE = 2          /* moe_forward_decode                         */
} moe_mode;

typedef struct moe_layer moe_layer;  /* opaque; owned by the library */

typedef struct {
    int32_t hidden;              /* H: model width, multiple of 128            */
    int32_t inter;               /* I: routed-expert inner width, mult. of 128 */
    int32_t n_experts;           /* E: routed experts                          */
    int32_t top_k;               /* k: experts per token                       */
    int32_t n_shared;            /* 0 or 1 always-on shared expert             */
    int32_t shared_inter;        /* inner width of the shared expert (= inter) */
} moe_desc;

/* Weights, in checkpoint layout.  DEVICE pointers, caller-owned, read only
 * during moe_create.  E4M3FN codes are one byte per weight, row-major; the
 * fp32 multipliers give W = E4M3(q) * s per 128x128 block. */
typedef struct {
    const float* router_w;       /* [E][H] fp32                                 */
    const float* router_bias;    /* [E] fp32, or NULL for no bias               */
    const uint8_t* w_gate;       /* [E][I][H] E4M3FN                            */
    const uint8_t* w_up;         /* [E][I][H] E4M3FN                            */
    const uint8_t* w_down;       /* [E][H][I] E4M3FN                            */
    const float* s_gate;         /* [E][I/128][H/128]                           */
    const float* s_up;           /* [E][I/128][H/128]                           */
    const float* s_down;         /* [E][H/128][I/128]                           */
    const uint8_t* sh_gate;      /* shared expert, same layouts with E = 1;     */
    const uint8_t* sh_up;        /*   ignored when n_shared = 0                 */
    const uint8_t* sh_down;
    const float* sh_s_gate;
    const float* sh_s_up;
    const float* sh_s_down;
} moe_weights;

/* Optional outputs of the routing stage.  DEVICE pointers, caller-owned;
 * any may be NULL (then not written).  Row numbers index the expert-sorted
 * list of (token, slot) pairs: expert e owns rows [offsets[e], offsets[e+1]),
 * in ascending token order. */
typedef struct {
    float* logits;               /* [T][E] fp32 router logits (moe_route only)  */
    int32_t* topk_ids;           /* [T][k] selected experts, rank order         */
    float* topk_w;               /* [T][k] gate weights, rank order             */
    int32_t* expert_offsets;     /* [E+1] exclusive prefix sum of the counts    */
    int32_t* sorted_token;       /* [T*k] token of each row                     */
    int32_t* inv_row;            /* [T][k] row of (token, slot)                 */
    uint8_t* xq;                 /* [T][H] E4M3FN codes of x (forward only)     */
    float* sx;                   /* [T][H/128] multipliers of xq (forward only) */
    uint8_t* hq;                 /* [T][k+n_shared][I] E4M3FN codes of h per    */
                                 /*   (token, slot): routed slots in rank       */
                                 /*   order, then the shared expert (forward)   */
    float* sh;                   /* [T][k+n_shared][I/128] multipliers of hq    */
} moe_route_out;

/* Build a layer: validate desc, allocate the layer's device memory, repack
 * the weights into the tile layout the kernels stream, and synchronise
 * `stream`.  On success *out holds a handle for moe_destroy. */
moe_status moe_create(const moe_desc* desc, const moe_weights* w, void* stream, moe_layer** out);

/* moe_create with flags.  MOE_CREATE_HOST_TILES keeps the repacked expert
 * tile images (the bulk of the layer, 11.3 GB for a DeepSeek-V3 layer) in
 * pinned host memory instead of HBM: the Stream-Loading Prefill design of
 * the CPU-GPU hybrid inference article (its "Stream-Loading Prefill"
 * section: expert weights stay in CPU memory and stream into a GPU ring
 * buffer while the previous experts compute), here over NVLink-C2C from
 * Grace memory.  Such a layer runs only through moe_forward_tiles, on tiles
 * that moe_tiles_load brought into a device slot; routing entries work as
 * usual.  Scales, the router and the status word stay on the device. */
#define MOE_CREATE_HOST_TILES 1u
moe_status moe_create_ex(const moe_desc* desc, const moe_weights* w, uint32_t flags, void* stream, moe_layer** out);

/* Bytes of the layer's tile images ([gate/up][down]) = the size of a slot. */
moe_status moe_tiles_bytes(moe_layer* layer, size_t* bytes);

/* Enqueue the copy of a host-tile layer's tiles into `slot` (device,
 * 256-byte aligned, moe_tiles_bytes long) on `stream` (one copy-engine
 * transfer; order it against the forward that reads the slot with events). */
moe_status moe_tiles_load(moe_layer* layer, void* slot, void* stream);

/* The forward of a host-tile layer on the tiles in `slot`.  mode, x, T, y,
 * workspace and errors as for moe_forward_prefill / moe_forward_decode. */
moe_status moe_forward_tiles(moe_layer* layer, int32_t mode, const void* slot, const uint16_t* x, int32_t T,
                             uint16_t* y, void* ws, size_t ws_bytes, void* stream);

/* Release everything the layer owns (synchronises the device first). */
moe_status moe_destroy(moe_layer* layer);

/* Bytes of caller workspace a call of `mode` needs for T tokens (T >= 0). */
moe_status moe_workspace_bytes(const moe_layer* layer, int32_t T, int32_t mode, size_t* bytes);

/* Routing only: logits, top-k, gate weights and the expert grouping of the
 * bf16 activations x [T][H] (raw bf16 bits).  Results go to `out`. */
moe_status moe_route(moe_layer* layer, const uint16_t* x, int32_t T, const moe_route_out* out,
                     void* ws, size_t ws_bytes, void* stream);

/* Routing from given fp32 logits [T][E] (no router GEMM): top-k, gate
 * weights and grouping, with the same kernels the forward entries use. */
moe_status moe_route_from_logits(moe_layer* layer, const float* logits, int32_t T,
                                 const moe_route_out* out, void* ws, size_t ws_bytes, void* stream);

/* moe_route_from_logits without a workspace argument; this call allocates
 * no memory.  The source pages have no counterpart: it exists for callers
 * that cannot allocate device memory when they route -- serving runtimes
 * that give all of HBM to their own pools at start-up and forbid cudaMalloc
 * afterwards (which would also synchronise the device mid-step), and plain
 * C callers without an allocator to carve a workspace from.
 * Its scratch is a fixed array of MOE_NOALLOC_SCRATCH_BYTES (4 MiB) compiled
 * into the library; every GPU that loads the library holds it until the
 * process exits.  Outputs go to `out` bit for bit as moe_route_from_logits
 * writes them (for decode-sized batches the workspace entry fuses the
 * stages into one kernel and this entry runs them one by one; both call
 * the same device functions, so the results are identical).
 *  - Device: the layer's device must be current (MOE_ERR_INVALID_ARG
 *    otherwise).
 *  - Size limit: the routing scratch for (T, n_experts, top_k) must fit the
 *    array -- roughly 160 bytes per token at E = 256, k = 8 (T <= ~26,000) --
 *    otherwise MOE_ERR_UNSUPPORTED is returned and nothing runs.
 *  - Set-up: the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture on the device.
 *  - Sharing: every call uses the same array, which keeps the previous
 *    call's contents; every scratch word a call reads is first written by
 *    that call, so nothing needs clearing.  Calls that overlap on the GPU
 *    (other streams, other host threads) race on the array: serialise them. */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)
moe_status moe_route_from_logits_noalloc(moe_layer* layer, const float* logits, int32_t T,
                                         const moe_route_out* out, void* stream);

/* The whole layer for a prefill batch: x [T][H] bf16 -> y [T][H] bf16.
 * `dbg` (nullable) receives the routing, exactly as moe_route would write it.
 * T = 0 is a valid no-op. */
moe_status moe_forward_prefill(moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y,
                               const moe_route_out* dbg, void* ws, size_t ws_bytes, void* stream);

/* The same function for 1 <= T <= MOE_DECODE_MAX_T tokens, on the decode
 * kernels (one-CTA routing; expert GEMMs that stream only the touched
 * experts' weights, with 16-token tiles).  Enqueues a fixed sequence of kernels
 * whose grids do not depend on the routing and reads nothing back to the
 * host, so a CUDA graph may capture it. */
moe_status moe_forward_decode(moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y,
                              const moe_route_out* dbg, void* ws, size_t ws_bytes, void* stream);

/* End to end from HOST buffers: copies x_host [T][H] to the device, runs the
 * prefill (mode 1) or decode (mode 2) path, copies y back into y_host
 * [T][H] and synchronises `stream`.  Host buffers should be pinned for full
 * copy speed.  Workspace: moe_workspace_bytes(mode) + 4*T*H + 512 bytes. */
moe_status moe_forward_host(moe_layer* layer, int32_t mode, const uint16_t* x_host, int32_t T,
                            uint16_t* y_host, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- variants
 * The three entries below reuse the layer's kernels and change only how the
 * work is composed or combined. */

/* A stack of MoE layers as one call: layer l's output y is layer l+1's
 * input x ("LLM serving on heterogeneous hardware" lecture, section 4.3,
 * and KTransformers deep dive, section 2.4: a decode step runs every layer
 * back to back and is recorded as one CUDA graph).  mode: MOE_MODE_PREFILL or
 * MOE_MODE_DECODE for every layer.  `layers` is a host array of n_layers
 * handles, all with the same hidden size (they may be the same handle).
 * x, y: device [T][H] bf16.  The call enqueues work only (no host
 * synchronisation), so it can be captured into a CUDA graph.  Workspace:
 * moe_layers_workspace_bytes (the largest single-layer workspace plus two
 * T x H bf16 carry buffers).  Errors as for moe_forward_prefill. */
moe_status moe_layers_workspace_bytes(moe_layer* const* layers, int32_t n_layers, int32_t T, int32_t mode,
                                      size_t* bytes);
moe_status moe_forward_layers(moe_layer* const* layers, int32_t n_layers, int32_t mode, const uint16_t* x,
                              int32_t T, uint16_t* y, void* ws, size_t ws_bytes, void* stream);

/* The layer with the SmallEP combine emulated on one GPU (CPU-GPU hybrid
 * inference article, SmallEP section, Fig. 5: expert-parallel ranks each
 * combine their own experts, then the partial outputs are reduced).  The
 * routed experts are split into n_ranks contiguous groups, rank p holding
 * experts [ceil(pE/n_ranks), ceil((p+1)E/n_ranks)) and rank 0 also the
 * shared expert.  Each rank's partial is the fixed-order fp32 sum of its
 * slots; y = bf16 of the partials added in rank order.  n_ranks = 1 gives
 * bit for bit the output of moe_forward_prefill / moe_forward_decode; other
 * n_ranks are deterministic but round differently.  1 <= n_ranks <= E.
 * Workspace and errors as for the mode's entry. */
moe_status moe_forward_smallep(moe_layer* layer, int32_t mode, int32_t n_ranks, const uint16_t* x, int32_t T,
                               uint16_t* y, void* ws, size_t ws_bytes, void* stream);

/* Expert deferral ("LLM serving on heterogeneous hardware" lecture, section
 * 4.3: the results of some selected experts join the residual stream one
 * layer later, so the next layer can start; the lecture keeps at least two
 * experts per token undeferred, a policy left to the caller here).  defer: device uint8 [T][k], slot j of token t deferred
 * when non-zero, slots in the rank order of topk_ids.  Outputs, device
 * [T][H] bf16: y_now = O[shared] + the non-deferred w_j O_j, y_next = the
 * deferred w_j O_j, each summed in slot order in fp32 and rounded once.  All
 * experts are still computed in this call; the split is in the combine.
 * With no slot deferred, y_now equals moe_forward_* bit for bit and y_next
 * is zero.  Workspace and errors as for the mode's entry; y_next must be
 * 16-byte aligned. */
moe_status moe_forward_deferred(moe_layer* layer, int32_t mode, const uint16_t* x, int32_t T, const uint8_t* defer,
                                uint16_t* y_now, uint16_t* y_next, void* ws, size_t ws_bytes, void* stream);

/* Synchronise `stream`, then read and clear the device status word
 * (MOE_DEV_* bits).  Returns MOE_ERR_TIMEOUT if the timeout bit was set,
 * MOE_ERR_DEVICE_CHECK for any other bit, MOE_OK when clear. */
moe_status moe_get_device_status(moe_layer* layer, void* stream, uint32_t* flags);

/* Time limit, in microseconds of GPU wall clock, of every bounded wait in
 * the kernels (default 2,000,000).  A wait that expires sets
 * MOE_DEV_WAIT_TIMEOUT and its kernel returns early with undefined output.
 * Lowering it makes a wait that nothing satisfies return quickly (tests). */
moe_status moe_set_wait_limit(moe_layer* layer, uint32_t microseconds);

/* Test hook: run one bounded wait on an mbarrier that is never signalled,
 * so the timeout path can be exercised without a fault. */
moe_status moe_debug_timeout_probe(moe_layer* layer, void* stream);

/* Test hook (fault injection, host side): the next call on this layer that
 * routes (MOE_DEV_BAD_EXPERT_ID) or runs a forward entry (MOE_DEV_BAD_ROW)
 * overwrites one word of its own workspace -- the expert id of (token 0,
 * slot 0) with n_experts + 3, or the internal row of (token 0, slot 0) with
 * a row past the permuted buffers -- before the kernels that read it.
 * Those kernels must flag it in the device status word and clamp or skip
 * it, so nothing reads or writes outside the buffers; the call's outputs
 * are then undefined and moe_get_device_status returns
 * MOE_ERR_DEVICE_CHECK.  Each planted fault fires once.  Other bits:
 * MOE_ERR_INVALID_ARG. */
moe_status moe_debug_inject(moe_layer* layer, uint32_t faults);

/* Measurement hook.  With profiling enabled, every forward call records a
 * CUDA event on its stream at the boundaries of the timed stages:
 *   stage 0 routing (logits, top-k, grouping)   stage 1 x quantisation
 *   stage 2 gate/up GEMM + SiLU*up              stage 3 down GEMM
 *   stage 4 combine
 * `enable`: 0 disables; 1 times every stage; MOE_PROFILE_SELECT | mask
 * times only the stages whose bits (1 << s) are set in mask.  An event
 * between two kernels removes their programmatic-dependent-launch overlap
 * (a few microseconds each at decode sizes), so timing only the stage of
 * interest disturbs the layer least.  Other values: MOE_ERR_INVALID_ARG.
 * moe_profile_read synchronises the stream of the most recent call and
 * writes the elapsed milliseconds of its first n_stages stages, -1 for a
 * stage that is not timed.  Enabling creates the events (no device
 * memory); disabled by default. */
#define MOE_PROFILE_STAGES 5
#define MOE_PROFILE_SELECT 0x40000000
moe_status moe_profile_enable(moe_layer* layer, int32_t enable);
moe_status moe_profile_read(moe_layer* layer, float* stage_ms, int32_t n_stages);

const char* moe_status_string(moe_status s);
const char* moe_last_error(void);   /* thread-local; "" when none */
int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
