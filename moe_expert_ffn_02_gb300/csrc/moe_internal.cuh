// Internal definitions shared by the kernels and the C-ABI layer of the
// GB300 (sm_103a) MoE FFN library.  Nothing here is part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/moe.h"

namespace moe {

constexpr int QB = 128;               // quantisation / scale block edge
constexpr int TILE_BYTES = QB * QB;   // one 128x128 FP8 weight tile image
constexpr int MAX_TOPK = 32;
constexpr int MAX_EXPERTS = 1024;
constexpr int ROW_PAD = 256;          // spare rows after every permuted buffer
constexpr int ROW_ALIGN = 8;          // each group's rows start on a multiple of 8
constexpr int DEC_TILE_N = 16;        // token rows per group tile of the weight-streaming (decode) GEMMs;
                                      // routing-only entries build their group table with it too

// ---------------------------------------------------------------------------
// Permuted activation buffers (x codes, h codes) use the same 128-byte
// swizzle as the weight tiles, stored K-block-major:
//   buf[kb][row][128 B], 16-byte chunk c of (kb, row) at chunk c ^ (row & 7).
// Every group starts on a multiple of 8 rows, so the rows [r, r + n) of one
// K block are one contiguous, already-swizzled n x 128 B image: a single
// bulk copy moves an operand tile for either GEMM.  Their scales are
// K-block-major too: s[kb][row].
// ---------------------------------------------------------------------------
__host__ __device__ inline size_t act_offset(int kb, int row, int rows_pad) {
    return ((size_t)kb * rows_pad + row) * 128;
}

// ---------------------------------------------------------------------------
// Weight tile image.  A [R][C] FP8 matrix (C contiguous) is stored as tiles
// [R/128][C/128] of 16 KB; inside a tile, row r (0..127) occupies bytes
// [128 r, 128 r + 128) and its 16-byte chunk c is stored at chunk position
// c ^ (r & 7).  This is the K-major, 128-byte-swizzled operand layout of the
// Blackwell tensor-core descriptors (8-row x 128 B swizzle atoms stacked
// along the rows every 1024 B), so a tile can be moved into shared memory by
// one bulk copy and consumed as is.  Gate and up tiles of the same
// (row block, k block) sit next to each other (32 KB), gate first.
// ---------------------------------------------------------------------------
__host__ __device__ inline int swz_chunk(int r, int c) { return c ^ (r & 7); }

// Per-group work description built on the device from the routing.
// A "group" is one expert with at least one row (the shared expert is
// group expert = E with rows R..R+T-1).  Units of the expert GEMMs are
// (group, n tile of BN rows, m tile of 128 outputs), m fastest.
struct GroupTable {
    int32_t n_groups;
    int32_t n_pairs;        // sum over groups of ceil(rows / bn)
    int32_t bn;             // n-tile height used to build the table
    int32_t total_rows;     // internal rows in use (padded groups + shared)
    int32_t expert[MAX_EXPERTS + 1];
    int32_t row0[MAX_EXPERTS + 1];   // internal (8-aligned) first row
    int32_t rows[MAX_EXPERTS + 1];
    int32_t pair_start[MAX_EXPERTS + 2];
};

// Shared-memory copy of a GroupTable's per-group arrays, so the expert GEMMs
// decode their units without chains of dependent L2 loads.  gt_smem_bytes(cap)
// of dynamic shared memory hold up to cap - 1 groups; a table with more
// groups is read in place from global memory.  load_groups is called by
// every thread of the CTA before its first __syncthreads.
constexpr int GT_CAP = MAX_EXPERTS + 2;
__host__ __device__ constexpr int gt_smem_bytes(int cap) { return 4 * cap * 4; }
constexpr int GT_SMEM_BYTES = gt_smem_bytes(GT_CAP);

struct SGroups {
    int* expert;
    int* row0;
    int* rows;
    int* pair_start;
    int n_groups;
};

__device__ __forceinline__ SGroups load_groups(const GroupTable* gt, int* smem, int tid, int nthreads,
                                               int cap = GT_CAP) {
    SGroups g;
    g.n_groups = min(gt->n_groups, GT_CAP - 1);
    if (g.n_groups > cap - 1) {                   // too many groups for the copy: use the table in place
        g.expert = const_cast<int*>(gt->expert);
        g.row0 = const_cast<int*>(gt->row0);
        g.rows = const_cast<int*>(gt->rows);
        g.pair_start = const_cast<int*>(gt->pair_start);
        return g;
    }
    g.expert = smem;
    g.row0 = smem + cap;
    g.rows = smem + 2 * cap;
    g.pair_start = smem + 3 * cap;
    for (int i = tid; i < g.n_groups; i += nthreads) {
        g.expert[i] = gt->expert[i];
        g.row0[i] = gt->row0[i];
        g.rows[i] = gt->rows[i];
        g.pair_start[i] = gt->pair_start[i];
    }
    return g;
}

// Tile `pair` (a group's row tiles numbered consecutively over all groups)
// -> its group's expert, the tile's first internal row and its row count.
__device__ __forceinline__ void decode_pair(const SGroups& g, int pair, int tile_rows, int& expert, int& row_begin,
                                            int& valid) {
    int lo = 0, hi = g.n_groups - 1;              // last group with pair_start <= pair
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (g.pair_start[mid] <= pair) lo = mid; else hi = mid - 1;
    }
    const int nt = pair - g.pair_start[lo];
    expert = g.expert[lo];
    row_begin = g.row0[lo] + nt * tile_rows;
    valid = min(tile_rows, g.rows[lo] - nt * tile_rows);
}

// Workspace carve-up for one call (all offsets 256-byte aligned).
struct WsLayout {
    size_t logit_part;   // f32 [ksplit][T][E] router partial sums
    size_t logits;       // f32 [T][E]
    size_t ids;          // i32 [T][k]
    size_t w;            // f32 [T][k]
    size_t chunk_cnt;    // i32 [n_chunks][E]
    size_t chunk_base;   // i32 [n_chunks][E]
    size_t offsets;      // i32 [E+1]   canonical expert offsets
    size_t offsets_pad;  // i32 [E+1]   internal 8-aligned group starts (E: shared)
    size_t inv_row;      // i32 [T][k]  canonical row of (token, slot)
    size_t inv_int;      // i32 [T][k]  internal row of (token, slot)
    size_t table;        // GroupTable
    size_t xp;           // u8  [H/128][rows_pad][128]  permuted quantised x (swizzled)
    size_t sxT;          // f32 [H/128][rows_pad]
    size_t hq;           // u8  [I/128][rows_pad][128]  quantised h (swizzled)
    size_t shT;          // f32 [I/128][rows_pad]
    size_t o;            // f32 [rows_pad][H]           expert outputs (unweighted)
    size_t total;
    int ksplit, n_chunks, rows_pad;
    bool gemv;           // router logits by the split GEMV (decode batches)
};

constexpr int CHUNK_TOK = 64;         // tokens per permutation chunk (one warp)

}  // namespace moe

struct moe_layer {
    moe_desc d;
    int device;
    int num_sms;
    int n_groups_max;      // E + n_shared
    uint8_t* w_gu;         // [G][I/128][H/128][2][16 KB] gate/up tile images
    uint8_t* w_dn;         // [G][H/128][I/128][16 KB]    down tile images
    uint8_t* tiles_host;   // host-resident tiles ([gate/up][down], pinned) or NULL; then w_gu / w_dn
                           // point into a device slot only for the duration of moe_forward_tiles
    size_t gu_bytes, dn_bytes;
    float* s_gu;           // [G][I/128][H/128][2]
    float* s_dn;           // [G][H/128][I/128]
    float* r_gu;           // [G][I/128][H/128][4]: {gate, up, 0, 0} per k block (16-byte records)
    float* r_dn;           // [G][ceil(H/256)][I/128][4]: {s(2b), s(2b+1) or 0, 0, 0} per k block
    float* router_w;       // [E][H]
    uint16_t* router_w3;   // [3][E][H] bf16 terms of router_w (w = w1 + w2 + w3), prefill router GEMM
    float* router_b;       // [E] (zeros when no bias)
    uint32_t* dev_status;  // device status word
    uint32_t wait_limit;
    uint32_t profile;      // stages whose events forward calls record (bit s: stage s), 0 = off
    uint32_t inject;       // MOE_DEV_* bits of faults the next forward call plants (moe_debug_inject)
    cudaEvent_t ev[MOE_PROFILE_STAGES + 1];
    cudaStream_t ev_stream;
};

namespace moe {

// ---------------------------------------------------------------------------
// Device helpers (PTX wrappers).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps in hardware (up to hint_ns) instead of spinning, so waiting warps
// do not take issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: gives up after `limit_us` microseconds of wall time, or as
// soon as another thread of the CTA has given up (*abort != 0).  On expiry
// it sets the timeout bit of the device status word and *abort, and returns
// false; the caller then abandons its work.  Nothing traps.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit_us,
                                                  uint32_t* status, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (abort && *abort) return false;
        if (global_ns() - t0 > (uint64_t)limit_us * 1000ull) {
            atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
            if (abort) *abort = 1;
            return false;
        }
    }
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Prefetch [p, p + bytes) into L2 (bulk, asynchronous, no completion to wait
// for).  p 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch.  Kernels of the forward path are launched
// with launch_pdl; each calls pdl_wait() before it reads anything the
// preceding kernel wrote (the wait returns once that grid has completed and
// its memory is visible), so the launch, and whatever the kernel does before
// the wait, overlaps the preceding kernel.  Small kernels call pdl_trigger()
// on entry so their successor is launched at once; the persistent GEMMs
// trigger by exiting; the router kernels (the decode GEMV after its wait,
// the prefill GEMM by exiting) release their successors only once the layer
// input x is complete, so every later kernel of the layer may read x before
// its own wait (the quantiser does).  Both are no-ops for a kernel launched
// without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// Two fp32 -> two E4M3FN (round to nearest even, saturate to +-448);
// `lo` lands in the low byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
    return (uint32_t)f32x2_to_e4m3x2(a, b) | ((uint32_t)f32x2_to_e4m3x2(c, d) << 16);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// SiLU(g) * u, shared by the prefill and decode epilogues so both paths form
// the same h.  Fast divide: h only needs a few-ulp accuracy before its 1x128
// quantisation; for g < -87, exp(-g) = inf and the quotient is -0.  The
// quantisation that follows takes h / s as h * (1/s), within one ulp of the
// rounded quotient and far inside the E4M3 code spacing.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

}  // namespace moe

// Launchers (defined in the .cu files, called from api.cu).
namespace moe {

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per device:
// the attribute belongs to the device current when it is set, so a process
// that drives layers on several devices sets it on each of them.
template <auto Kernel>
cudaError_t ensure_smem_limit(int bytes) {
    static std::atomic<uint64_t> done{0};     // bit d: set on device d (< 64)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Launch with programmatic stream serialisation (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_repack(const moe_layer* L, const moe_weights* w, cudaStream_t s);
int router_gemv_splits(int H);
int router_tc_splits(int T, int H, int E, int num_sms);
size_t router_split_bytes(const moe_layer* L);
cudaError_t launch_split_router_weights(const moe_layer* L, cudaStream_t s);
cudaError_t launch_router_tc(const moe_layer* L, const uint16_t* x, int T, float* part, int ksplit, cudaStream_t s);
cudaError_t launch_router_logits(const moe_layer* L, const uint16_t* x, int T, float* part, int ksplit, bool gemv,
                                 cudaStream_t s);
cudaError_t launch_topk(const moe_layer* L, const float* part, int ksplit, bool add_bias, int T, float* logits_out,
                        int32_t* ids, float* w, cudaStream_t s);
cudaError_t launch_route_small(const moe_layer* L, const float* part, int ksplit, bool add_bias, int T,
                               float* logits_out, int32_t* ids, float* w, const WsLayout& lay, char* ws, int bn,
                               int32_t* offsets_out, int32_t* sorted_out, int32_t* inv_out, cudaStream_t s);
cudaError_t launch_permute(const moe_layer* L, const int32_t* ids, int T, const WsLayout& lay, char* ws, int bn,
                           int32_t* offsets_out, int32_t* sorted_out, int32_t* inv_out, cudaStream_t s);
cudaError_t launch_quant_scatter(const moe_layer* L, const uint16_t* x, int T, const WsLayout& lay, char* ws,
                                 uint8_t* xq_out, float* sx_out, cudaStream_t s);
cudaError_t launch_expert_dec_gate_up(const moe_layer* L, int T, const WsLayout& lay, char* ws, int bn,
                                      cudaStream_t s);
cudaError_t launch_expert_dec_down(const moe_layer* L, int T, const WsLayout& lay, char* ws, int bn, cudaStream_t s);
cudaError_t launch_h_gather(const moe_layer* L, int T, const WsLayout& lay, char* ws, uint8_t* hq_out, float* sh_out,
                            cudaStream_t s);
int tc_tile_n();
cudaError_t launch_expert_tc_gate_up(const moe_layer* L, int T, const WsLayout& lay, char* ws, cudaStream_t s);
cudaError_t launch_tc_scale_records(const moe_layer* L, cudaStream_t s);
cudaError_t launch_expert_tc_down(const moe_layer* L, int T, const WsLayout& lay, char* ws, cudaStream_t s);
cudaError_t launch_combine(const moe_layer* L, int T, const WsLayout& lay, char* ws, uint16_t* y, cudaStream_t s);
cudaError_t launch_combine_split(const moe_layer* L, int T, const WsLayout& lay, char* ws, int n_ranks,
                                 const uint8_t* defer, uint16_t* y, uint16_t* y_next, cudaStream_t s);
cudaError_t launch_timeout_probe(const moe_layer* L, cudaStream_t s);
cudaError_t launch_plant(int32_t* word, int32_t value, cudaStream_t s);
void set_last_error(const char* msg);   // message returned by moe_last_error()
}  // namespace moe
