// C ABI of the MoE layer (declared in include/moe.h): argument checks,
// workspace carve-up, layer ownership and the launch sequence of each entry.
#include "moe_internal.cuh"

#include <algorithm>
#include <cstddef>
#include <cstdarg>
#include <cstdio>
#include <string>

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MOE_CUDA(call, what)                        \
    do {                                            \
        cudaError_t e_ = (call);                    \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr uint32_t kDefaultWaitLimitUs = 2000000u;   // 2 s per bounded wait
constexpr int kBN = moe::DEC_TILE_N;                 // token tile of the decode expert GEMMs

moe::WsLayout make_layout(const moe_layer* L, int T, int mode) {
    moe::WsLayout l{};
    const size_t E = L->d.n_experts, k = L->d.top_k, H = L->d.hidden, I = L->d.inter;
    const size_t R = (size_t)T * k;
    // internal rows: every routed group padded to ROW_ALIGN, then the shared group
    const size_t rows = R + (L->d.n_shared ? (size_t)T : 0) + (size_t)moe::ROW_ALIGN * (E + 1);
    l.rows_pad = (int)up(rows + moe::ROW_PAD, 64);
    // router: T <= 64 -> the split GEMV; otherwise the tensor-core GEMM,
    // split along H.  Either way ksplit partial sums, added in order by the
    // top-k kernel.
    l.gemv = T <= 64;
    l.ksplit = l.gemv ? moe::router_gemv_splits((int)H) : moe::router_tc_splits(T, (int)H, (int)E, L->num_sms);
    l.n_chunks = (T + moe::CHUNK_TOK - 1) / moe::CHUNK_TOK;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = up(off + bytes, 256); return o; };
    l.logit_part = take((size_t)l.ksplit * T * E * 4);
    l.logits = l.logit_part;
    l.ids = take(R * 4);
    l.w = take(R * 4);
    l.chunk_cnt = take((size_t)l.n_chunks * E * 4);
    l.chunk_base = take((size_t)l.n_chunks * E * 4);
    l.offsets = take((E + 1) * 4);
    l.offsets_pad = take((E + 1) * 4);
    l.inv_row = take(R * 4);
    l.inv_int = take(R * 4);
    l.table = take(sizeof(moe::GroupTable));
    if (mode != MOE_MODE_ROUTE) {
        l.xp = take((size_t)l.rows_pad * H);
        l.sxT = take((H / moe::QB) * (size_t)l.rows_pad * 4);
        l.hq = take((size_t)l.rows_pad * I);
        l.shT = take((I / moe::QB) * (size_t)l.rows_pad * 4);
        l.o = take((size_t)l.rows_pad * H * 4);
    }
    l.total = off;
    return l;
}

// The host-side tests build a stand-in handle whose recorded device differs
// from the current one; they rely on `device` following the descriptor.
static_assert(offsetof(moe_layer, device) == sizeof(moe_desc), "moe_layer: device must follow the descriptor");

moe_status check_layer(const moe_layer* L) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    return MOE_OK;
}

// Every entry that enqueues work checks that the calling thread's current
// device is the one the layer lives on: a kernel launched on another device
// would dereference this layer's weights and workspace from the wrong GPU.
moe_status check_device(const moe_layer* L) {
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (cur != L->device)
        return fail(MOE_ERR_INVALID_ARG, "the current device (%d) is not the layer's device (%d)", cur, L->device);
    return MOE_OK;
}

moe_status check_layer_device(const moe_layer* L) {
    moe_status st = check_layer(L);
    return st != MOE_OK ? st : check_device(L);
}

moe_status check_call(moe_layer* L, int T, int mode, const void* x, const void* y, void* ws, size_t ws_bytes,
                      moe::WsLayout* lay) {
    moe_status st = check_layer_device(L);
    if (st == MOE_OK && mode != MOE_MODE_ROUTE && L->tiles_host && !L->w_gu)
        return fail(MOE_ERR_INVALID_ARG, "the layer keeps its tiles in host memory: run it with moe_forward_tiles");
    if (st != MOE_OK) return st;
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d is negative", T);
    if ((int64_t)T * L->d.top_k >= (int64_t)1 << 31) return fail(MOE_ERR_UNSUPPORTED, "T * top_k >= 2^31");
    if (mode == MOE_MODE_DECODE && (T < 1 || T > MOE_DECODE_MAX_T))
        return fail(MOE_ERR_UNSUPPORTED, "decode takes 1 <= T <= %d tokens (got %d)", MOE_DECODE_MAX_T, T);
    if (T > 0 && !x) return fail(MOE_ERR_INVALID_ARG, "input pointer is NULL");
    if (x && !aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "input pointer is not 16-byte aligned");
    if (mode != MOE_MODE_ROUTE && T > 0 && !y) return fail(MOE_ERR_INVALID_ARG, "output y is NULL");
    if (y && !aligned(y, 16)) return fail(MOE_ERR_INVALID_ARG, "output y is not 16-byte aligned");
    *lay = make_layout(L, T, mode);
    if (T > 0) {
        if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
        if (!aligned(ws, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
        if (ws_bytes < lay->total)
            return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, lay->total);
    }
    return MOE_OK;
}

// Routing stage shared by every entry.  `logits_in` != NULL: route from
// given logits (no router GEMM, no bias).
moe_status run_route(moe_layer* L, const uint16_t* x, const float* logits_in, int T, const moe::WsLayout& lay,
                     char* ws, const moe_route_out* dbg, cudaStream_t s, int bn = kBN) {
    const int k = L->d.top_k;
    int32_t* ids = reinterpret_cast<int32_t*>(ws + lay.ids);
    float* w = reinterpret_cast<float*>(ws + lay.w);
    // a decode-sized batch: top-k and grouping in one single-CTA kernel (not when a bad expert id is to be
    // planted between the two)
    const bool plant_id = (L->inject & MOE_DEV_BAD_EXPERT_ID) != 0;
    const bool small = lay.n_chunks == 1 && L->d.n_experts <= 512 && !plant_id;
    if (small) {
        const float* part = logits_in ? logits_in : reinterpret_cast<const float*>(ws + lay.logit_part);
        if (!logits_in)
            MOE_CUDA(moe::launch_router_logits(L, x, T, const_cast<float*>(part), lay.ksplit, lay.gemv, s),
                     "router logits");
        MOE_CUDA(moe::launch_route_small(L, part, logits_in ? 1 : lay.ksplit, !logits_in, T,
                                         (dbg && !logits_in) ? dbg->logits : nullptr, ids, w, lay, ws, bn,
                                         dbg ? dbg->expert_offsets : nullptr, dbg ? dbg->sorted_token : nullptr,
                                         dbg ? dbg->inv_row : nullptr, s),
                 "routing");
        if (dbg && dbg->topk_ids)
            MOE_CUDA(cudaMemcpyAsync(dbg->topk_ids, ids, sizeof(int32_t) * (size_t)T * k, cudaMemcpyDeviceToDevice, s),
                     "copy ids");
        if (dbg && dbg->topk_w)
            MOE_CUDA(cudaMemcpyAsync(dbg->topk_w, w, sizeof(float) * (size_t)T * k, cudaMemcpyDeviceToDevice, s),
                     "copy weights");
        return MOE_OK;
    }
    if (logits_in) {
        MOE_CUDA(moe::launch_topk(L, logits_in, 1, false, T, nullptr, ids, w, s), "top-k");
    } else {
        float* part = reinterpret_cast<float*>(ws + lay.logit_part);
        MOE_CUDA(moe::launch_router_logits(L, x, T, part, lay.ksplit, lay.gemv, s), "router logits");
        MOE_CUDA(moe::launch_topk(L, part, lay.ksplit, true, T, dbg ? dbg->logits : nullptr, ids,
                                  w, s),
                 "top-k");
    }
    if (plant_id) {                   // moe_debug_inject: an expert id outside [0, E) for (token 0, slot 0)
        MOE_CUDA(moe::launch_plant(ids, L->d.n_experts + 3, s), "fault injection");
        L->inject &= ~(uint32_t)MOE_DEV_BAD_EXPERT_ID;
    }
    if (dbg && dbg->topk_ids)
        MOE_CUDA(cudaMemcpyAsync(dbg->topk_ids, ids, sizeof(int32_t) * (size_t)T * k, cudaMemcpyDeviceToDevice, s),
                 "copy ids");
    if (dbg && dbg->topk_w)
        MOE_CUDA(cudaMemcpyAsync(dbg->topk_w, w, sizeof(float) * (size_t)T * k, cudaMemcpyDeviceToDevice, s),
                 "copy weights");
    MOE_CUDA(moe::launch_permute(L, ids, T, lay, ws, bn, dbg ? dbg->expert_offsets : nullptr,
                                 dbg ? dbg->sorted_token : nullptr, dbg ? dbg->inv_row : nullptr, s),
             "permutation");
    return MOE_OK;
}

// How the expert outputs are combined: the plain fixed-order sum, the SmallEP
// partial sums over n_ranks expert groups, or the deferral split.
struct CombineSpec {
    int n_ranks = 1;
    const uint8_t* defer = nullptr;
    uint16_t* y_next = nullptr;
};

moe_status run_forward(moe_layer* L, int mode, const uint16_t* x, int T, uint16_t* y, const moe_route_out* dbg,
                       void* ws_v, size_t ws_bytes, cudaStream_t s, const CombineSpec& cs = CombineSpec()) {
    moe::WsLayout lay;
    moe_status st = check_call(L, T, mode, x, y, ws_v, ws_bytes, &lay);
    if (st != MOE_OK) return st;
    if (T == 0) {
        if (dbg && dbg->expert_offsets)
            MOE_CUDA(cudaMemsetAsync(dbg->expert_offsets, 0, sizeof(int32_t) * (L->d.n_experts + 1), s), "memset");
        return MOE_OK;
    }
    char* ws = static_cast<char*>(ws_v);
    // event i opens stage i and closes stage i - 1; only the timed stages' events are recorded,
    // so an event-free stage boundary keeps its programmatic-dependent-launch overlap
    auto mark = [&](int i) -> cudaError_t {
        const uint32_t m = L->profile;
        if (!(((m >> i) & 1u) || (i > 0 && ((m >> (i - 1)) & 1u)))) return cudaSuccess;
        L->ev_stream = s;
        // inside a stream capture the events become record nodes of the graph (recorded at each launch)
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(s, &cap);
        if (e != cudaSuccess) return e;
        return cap == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(L->ev[i], s, cudaEventRecordExternal)
                                                    : cudaEventRecord(L->ev[i], s);
    };
    // prefill: tcgen05 grouped GEMMs (128-token tiles); decode: tcgen05 weight-streaming GEMMs with the
    // weights as the 128-row operand (16-token tiles)
    const bool tc_path = (mode == MOE_MODE_PREFILL);
    MOE_CUDA(mark(0), "profile event");
    st = run_route(L, x, nullptr, T, lay, ws, dbg, s, tc_path ? moe::tc_tile_n() : kBN);
    if (st != MOE_OK) return st;
    if (L->inject & MOE_DEV_BAD_ROW) {   // moe_debug_inject: an internal row outside the workspace for (0, 0)
        MOE_CUDA(moe::launch_plant(reinterpret_cast<int32_t*>(ws + lay.inv_int), lay.rows_pad + 5, s),
                 "fault injection");
        L->inject &= ~(uint32_t)MOE_DEV_BAD_ROW;
    }
    MOE_CUDA(mark(1), "profile event");
    MOE_CUDA(moe::launch_quant_scatter(L, x, T, lay, ws, dbg ? dbg->xq : nullptr, dbg ? dbg->sx : nullptr, s),
             "activation quantisation");
    MOE_CUDA(mark(2), "profile event");
    MOE_CUDA(tc_path ? moe::launch_expert_tc_gate_up(L, T, lay, ws, s) : moe::launch_expert_dec_gate_up(L, T, lay, ws, kBN, s),
             "gate/up GEMM");
    if (dbg && (dbg->hq || dbg->sh))
        MOE_CUDA(moe::launch_h_gather(L, T, lay, ws, dbg->hq, dbg->sh, s), "h debug copy");
    MOE_CUDA(mark(3), "profile event");
    MOE_CUDA(tc_path ? moe::launch_expert_tc_down(L, T, lay, ws, s) : moe::launch_expert_dec_down(L, T, lay, ws, kBN, s),
             "down GEMM");
    MOE_CUDA(mark(4), "profile event");
    if (cs.n_ranks == 1 && !cs.defer)
        MOE_CUDA(moe::launch_combine(L, T, lay, ws, y, s), "combine");
    else
        MOE_CUDA(moe::launch_combine_split(L, T, lay, ws, cs.n_ranks, cs.defer, y, cs.y_next, s), "combine");
    MOE_CUDA(mark(5), "profile event");
    return MOE_OK;
}

}  // namespace

namespace moe {
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }
}  // namespace moe

MOE_EXPORT int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

MOE_EXPORT const char* moe_last_error(void) { return g_last_error.c_str(); }

MOE_EXPORT const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    }
    return "MOE_ERR_UNKNOWN";
}

MOE_EXPORT moe_status moe_create(const moe_desc* d, const moe_weights* w, void* stream, moe_layer** out) {
    return moe_create_ex(d, w, 0, stream, out);
}

MOE_EXPORT moe_status moe_create_ex(const moe_desc* d, const moe_weights* w, uint32_t flags, void* stream,
                                    moe_layer** out) {
    g_last_error.clear();
    if (flags & ~(uint32_t)MOE_CREATE_HOST_TILES) return fail(MOE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    if (!d || !w || !out) return fail(MOE_ERR_INVALID_ARG, "desc, weights and out must be non-NULL");
    *out = nullptr;
    if (d->hidden <= 0 || d->inter <= 0 || d->hidden % moe::QB || d->inter % moe::QB)
        return fail(MOE_ERR_UNSUPPORTED, "hidden (%d) and inter (%d) must be positive multiples of 128", d->hidden,
                    d->inter);
    if (d->top_k < 1 || d->top_k > moe::MAX_TOPK || d->n_experts < d->top_k || d->n_experts > moe::MAX_EXPERTS)
        return fail(MOE_ERR_UNSUPPORTED, "need 1 <= top_k <= 32 and top_k <= n_experts <= 1024 (k=%d, E=%d)",
                    d->top_k, d->n_experts);
    if (d->n_shared != 0 && d->n_shared != 1) return fail(MOE_ERR_UNSUPPORTED, "n_shared must be 0 or 1");
    if (d->n_shared && d->shared_inter != 0 && d->shared_inter != d->inter)
        return fail(MOE_ERR_UNSUPPORTED, "shared_inter must equal inter");
    const void* req[] = {w->router_w, w->w_gate, w->w_up, w->w_down, w->s_gate, w->s_up, w->s_down};
    for (const void* p : req)
        if (!p || !aligned(p, 16)) return fail(MOE_ERR_INVALID_ARG, "a weight pointer is NULL or not 16-byte aligned");
    if (d->n_shared) {
        const void* sreq[] = {w->sh_gate, w->sh_up, w->sh_down, w->sh_s_gate, w->sh_s_up, w->sh_s_down};
        for (const void* p : sreq)
            if (!p || !aligned(p, 16))
                return fail(MOE_ERR_INVALID_ARG, "a shared-expert weight pointer is NULL or not 16-byte aligned");
    }
    if (w->router_bias && !aligned(w->router_bias, 4)) return fail(MOE_ERR_INVALID_ARG, "router_bias misaligned");

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    moe_layer* L = new moe_layer{};
    L->d = *d;
    if (!L->d.n_shared) L->d.shared_inter = 0;
    else L->d.shared_inter = d->inter;
    L->wait_limit = kDefaultWaitLimitUs;
    auto cleanup = [&](moe_status st) {
        cudaFree(L->w_gu); cudaFree(L->w_dn); cudaFree(L->s_gu); cudaFree(L->s_dn); cudaFree(L->r_gu); cudaFree(L->r_dn);
        cudaFree(L->router_w); cudaFree(L->router_w3); cudaFree(L->router_b); cudaFree(L->dev_status);
        delete L;
        return st;
    };
    cudaError_t e = cudaGetDevice(&L->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "device query"));
    const size_t H = d->hidden, I = d->inter, E = d->n_experts, G = E + L->d.n_shared;
    L->n_groups_max = (int)G;
    const size_t gu = G * I * H * 2, dn = G * H * I;
    L->gu_bytes = gu;
    L->dn_bytes = dn;
    const size_t sgu = G * (I / moe::QB) * (H / moe::QB) * 2 * 4, sdn = G * (H / moe::QB) * (I / moe::QB) * 4;
    if ((e = cudaMalloc(&L->w_gu, gu)) != cudaSuccess) return cleanup(cuda_fail(e, "allocating gate/up tiles"));
    if ((e = cudaMalloc(&L->w_dn, dn)) != cudaSuccess) return cleanup(cuda_fail(e, "allocating down tiles"));
    if ((e = cudaMalloc(&L->s_gu, sgu)) != cudaSuccess) return cleanup(cuda_fail(e, "allocating scales"));
    if ((e = cudaMalloc(&L->s_dn, sdn)) != cudaSuccess) return cleanup(cuda_fail(e, "allocating scales"));
    const size_t rgu = G * (I / moe::QB) * (H / moe::QB) * 16, rdn = G * ((H / moe::QB + 1) / 2) * (I / moe::QB) * 16;
    if ((e = cudaMalloc(&L->r_gu, rgu)) != cudaSuccess) return cleanup(cuda_fail(e, "allocating scale records"));
    if ((e = cudaMalloc(&L->r_dn, rdn)) != cudaSuccess) return cleanup(cuda_fail(e, "allocating scale records"));
    if ((e = cudaMalloc(&L->router_w, E * H * 4)) != cudaSuccess) return cleanup(cuda_fail(e, "allocating router"));
    if ((e = cudaMalloc(&L->router_w3, moe::router_split_bytes(L))) != cudaSuccess)
        return cleanup(cuda_fail(e, "allocating router terms"));
    if ((e = cudaMalloc(&L->router_b, E * 4)) != cudaSuccess) return cleanup(cuda_fail(e, "allocating bias"));
    if ((e = cudaMalloc(&L->dev_status, 4)) != cudaSuccess) return cleanup(cuda_fail(e, "allocating status"));
    if ((e = cudaMemsetAsync(L->dev_status, 0, 4, s)) != cudaSuccess) return cleanup(cuda_fail(e, "memset"));
    if ((e = cudaMemcpyAsync(L->router_w, w->router_w, E * H * 4, cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return cleanup(cuda_fail(e, "copying router weights"));
    e = w->router_bias ? cudaMemcpyAsync(L->router_b, w->router_bias, E * 4, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(L->router_b, 0, E * 4, s);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "copying router bias"));
    if ((e = moe::launch_split_router_weights(L, s)) != cudaSuccess) return cleanup(cuda_fail(e, "router split"));
    if ((e = moe::launch_repack(L, w, s)) != cudaSuccess) return cleanup(cuda_fail(e, "weight repack"));
    if ((e = moe::launch_tc_scale_records(L, s)) != cudaSuccess) return cleanup(cuda_fail(e, "scale records"));
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cleanup(cuda_fail(e, "moe_create synchronise"));
    if (flags & MOE_CREATE_HOST_TILES) {
        // keep the tile images in pinned host memory, [gate/up][down]; the device copies are released
        if ((e = cudaHostAlloc(&L->tiles_host, gu + dn, cudaHostAllocDefault)) != cudaSuccess)
            return cleanup(cuda_fail(e, "allocating host tiles"));
        if ((e = cudaMemcpy(L->tiles_host, L->w_gu, gu, cudaMemcpyDeviceToHost)) != cudaSuccess ||
            (e = cudaMemcpy(L->tiles_host + gu, L->w_dn, dn, cudaMemcpyDeviceToHost)) != cudaSuccess) {
            cudaFreeHost(L->tiles_host);
            L->tiles_host = nullptr;
            return cleanup(cuda_fail(e, "copying tiles to host"));
        }
        cudaFree(L->w_gu);
        cudaFree(L->w_dn);
        L->w_gu = L->w_dn = nullptr;
    }
    *out = L;
    return MOE_OK;
}

MOE_EXPORT moe_status moe_tiles_bytes(moe_layer* L, size_t* bytes) {
    moe_status st = check_layer(L);
    if (st != MOE_OK) return st;
    if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = L->gu_bytes + L->dn_bytes;
    return MOE_OK;
}

MOE_EXPORT moe_status moe_tiles_load(moe_layer* L, void* slot, void* stream) {
    moe_status st = check_layer_device(L);
    if (st != MOE_OK) return st;
    if (!L->tiles_host) return fail(MOE_ERR_INVALID_ARG, "the layer keeps its tiles on the device");
    if (!slot || !aligned(slot, 256)) return fail(MOE_ERR_INVALID_ARG, "slot NULL or not 256-byte aligned");
    MOE_CUDA(cudaMemcpyAsync(slot, L->tiles_host, L->gu_bytes + L->dn_bytes, cudaMemcpyHostToDevice,
                             static_cast<cudaStream_t>(stream)),
             "loading tiles");
    return MOE_OK;
}

MOE_EXPORT moe_status moe_forward_tiles(moe_layer* L, int32_t mode, const void* slot, const uint16_t* x, int32_t T,
                                        uint16_t* y, void* ws, size_t ws_bytes, void* stream) {
    moe_status st = check_layer_device(L);
    if (st != MOE_OK) return st;
    if (mode != MOE_MODE_PREFILL && mode != MOE_MODE_DECODE) return fail(MOE_ERR_INVALID_ARG, "mode must be 1 or 2");
    if (!L->tiles_host) return fail(MOE_ERR_INVALID_ARG, "the layer keeps its tiles on the device");
    if (!slot || !aligned(slot, 256)) return fail(MOE_ERR_INVALID_ARG, "slot NULL or not 256-byte aligned");
    // the kernels take the tile pointers by value at launch; the handle is used from one stream at a time
    L->w_gu = static_cast<uint8_t*>(const_cast<void*>(slot));
    L->w_dn = L->w_gu + L->gu_bytes;
    st = run_forward(L, mode, x, T, y, nullptr, ws, ws_bytes, static_cast<cudaStream_t>(stream));
    L->w_gu = L->w_dn = nullptr;
    return st;
}

MOE_EXPORT moe_status moe_destroy(moe_layer* L) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    // release on the layer's own device, whichever device the caller has current
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e == cudaSuccess && cur != L->device) e = cudaSetDevice(L->device);
    if (e != cudaSuccess) return cuda_fail(e, "moe_destroy: selecting the layer's device");
    e = cudaDeviceSynchronize();
    if (L->profile)
        for (cudaEvent_t ev : L->ev) cudaEventDestroy(ev);
    if (L->tiles_host) cudaFreeHost(L->tiles_host);
    cudaFree(L->w_gu); cudaFree(L->w_dn); cudaFree(L->s_gu); cudaFree(L->s_dn); cudaFree(L->r_gu); cudaFree(L->r_dn);
    cudaFree(L->router_w); cudaFree(L->router_w3); cudaFree(L->router_b); cudaFree(L->dev_status);
    const int dev = L->device;
    delete L;
    if (cur >= 0 && cur != dev) cudaSetDevice(cur);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_destroy synchronise");
}

MOE_EXPORT moe_status moe_workspace_bytes(const moe_layer* L, int32_t T, int32_t mode, size_t* bytes) {
    moe_status st = check_layer(L);
    if (st != MOE_OK) return st;
    if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T is negative");
    if (mode < MOE_MODE_ROUTE || mode > MOE_MODE_DECODE) return fail(MOE_ERR_INVALID_ARG, "unknown mode %d", mode);
    *bytes = make_layout(L, T, mode).total;
    return MOE_OK;
}

MOE_EXPORT moe_status moe_route(moe_layer* L, const uint16_t* x, int32_t T, const moe_route_out* out, void* ws,
                                size_t ws_bytes, void* stream) {
    moe::WsLayout lay;
    moe_status st = check_call(L, T, MOE_MODE_ROUTE, x, nullptr, ws, ws_bytes, &lay);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (out && out->expert_offsets)
            MOE_CUDA(cudaMemsetAsync(out->expert_offsets, 0, sizeof(int32_t) * (L->d.n_experts + 1), s), "memset");
        return MOE_OK;
    }
    return run_route(L, x, nullptr, T, lay, static_cast<char*>(ws), out, s);
}

MOE_EXPORT moe_status moe_route_from_logits(moe_layer* L, const float* logits, int32_t T, const moe_route_out* out,
                                            void* ws, size_t ws_bytes, void* stream) {
    moe::WsLayout lay;
    moe_status st = check_call(L, T, MOE_MODE_ROUTE, logits, nullptr, ws, ws_bytes, &lay);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (out && out->expert_offsets)
            MOE_CUDA(cudaMemsetAsync(out->expert_offsets, 0, sizeof(int32_t) * (L->d.n_experts + 1), s), "memset");
        return MOE_OK;
    }
    moe_route_out o = out ? *out : moe_route_out{};
    o.logits = nullptr;
    return run_route(L, nullptr, logits, T, lay, static_cast<char*>(ws), &o, s);
}

MOE_EXPORT moe_status moe_forward_prefill(moe_layer* L, const uint16_t* x, int32_t T, uint16_t* y,
                                          const moe_route_out* dbg, void* ws, size_t ws_bytes, void* stream) {
    return run_forward(L, MOE_MODE_PREFILL, x, T, y, dbg, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

MOE_EXPORT moe_status moe_forward_decode(moe_layer* L, const uint16_t* x, int32_t T, uint16_t* y,
                                         const moe_route_out* dbg, void* ws, size_t ws_bytes, void* stream) {
    return run_forward(L, MOE_MODE_DECODE, x, T, y, dbg, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

MOE_EXPORT moe_status moe_forward_smallep(moe_layer* L, int32_t mode, int32_t n_ranks, const uint16_t* x, int32_t T,
                                          uint16_t* y, void* ws, size_t ws_bytes, void* stream) {
    moe_status st = check_layer(L);
    if (st != MOE_OK) return st;
    if (mode != MOE_MODE_PREFILL && mode != MOE_MODE_DECODE) return fail(MOE_ERR_INVALID_ARG, "mode must be 1 or 2");
    if (n_ranks < 1 || n_ranks > L->d.n_experts)
        return fail(MOE_ERR_INVALID_ARG, "n_ranks (%d) must be in [1, n_experts]", n_ranks);
    CombineSpec cs;
    cs.n_ranks = n_ranks;
    return run_forward(L, mode, x, T, y, nullptr, ws, ws_bytes, static_cast<cudaStream_t>(stream), cs);
}

MOE_EXPORT moe_status moe_forward_deferred(moe_layer* L, int32_t mode, const uint16_t* x, int32_t T,
                                           const uint8_t* defer, uint16_t* y_now, uint16_t* y_next, void* ws,
                                           size_t ws_bytes, void* stream) {
    moe_status st = check_layer(L);
    if (st != MOE_OK) return st;
    if (mode != MOE_MODE_PREFILL && mode != MOE_MODE_DECODE) return fail(MOE_ERR_INVALID_ARG, "mode must be 1 or 2");
    if (T > 0 && (!defer || !y_next || !aligned(y_next, 16)))
        return fail(MOE_ERR_INVALID_ARG, "defer and a 16-byte aligned y_next are required");
    CombineSpec cs;
    cs.defer = defer;
    cs.y_next = y_next;
    return run_forward(L, mode, x, T, y_now, nullptr, ws, ws_bytes, static_cast<cudaStream_t>(stream), cs);
}

namespace {
// Workspace of a layer stack: the largest single-layer workspace, then two
// T x H bf16 activation buffers that carry y of layer l to layer l + 1.
moe_status layers_layout(moe_layer* const* layers, int n, int T, int mode, size_t* fwd, size_t* act) {
    if (!layers || n < 1) return fail(MOE_ERR_INVALID_ARG, "layers must be non-NULL and n_layers >= 1");
    if (mode != MOE_MODE_PREFILL && mode != MOE_MODE_DECODE) return fail(MOE_ERR_INVALID_ARG, "mode must be 1 or 2");
    if (T < 0 || (mode == MOE_MODE_DECODE && T > MOE_DECODE_MAX_T)) return fail(MOE_ERR_INVALID_ARG, "bad T (%d)", T);
    *fwd = 0;
    for (int l = 0; l < n; ++l) {
        if (!layers[l]) return fail(MOE_ERR_INVALID_ARG, "layer %d is NULL", l);
        if (layers[l]->d.hidden != layers[0]->d.hidden)
            return fail(MOE_ERR_INVALID_ARG, "layer %d has hidden %d, layer 0 has %d", l, layers[l]->d.hidden,
                        layers[0]->d.hidden);
        *fwd = std::max(*fwd, make_layout(layers[l], T, mode).total);
    }
    *act = up((size_t)T * layers[0]->d.hidden * 2, 256);
    return MOE_OK;
}
}  // namespace

MOE_EXPORT moe_status moe_layers_workspace_bytes(moe_layer* const* layers, int32_t n_layers, int32_t T, int32_t mode,
                                                 size_t* bytes) {
    size_t fwd = 0, act = 0;
    moe_status st = layers_layout(layers, n_layers, T, mode, &fwd, &act);
    if (st != MOE_OK) return st;
    if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = fwd + 2 * act;
    return MOE_OK;
}

MOE_EXPORT moe_status moe_forward_layers(moe_layer* const* layers, int32_t n_layers, int32_t mode, const uint16_t* x,
                                         int32_t T, uint16_t* y, void* ws, size_t ws_bytes, void* stream) {
    size_t fwd = 0, act = 0;
    moe_status st = layers_layout(layers, n_layers, T, mode, &fwd, &act);
    if (st != MOE_OK) return st;
    if (!ws || !aligned(ws, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
    if (ws_bytes < fwd + 2 * act) return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, fwd + 2 * act);
    char* base = static_cast<char*>(ws);
    uint16_t* buf[2] = {reinterpret_cast<uint16_t*>(base + fwd), reinterpret_cast<uint16_t*>(base + fwd + act)};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int l = 0; l < n_layers; ++l) {
        const uint16_t* in = l == 0 ? x : buf[(l - 1) & 1];
        uint16_t* out = l == n_layers - 1 ? y : buf[l & 1];
        st = run_forward(layers[l], mode, in, T, out, nullptr, base, fwd, s);
        if (st != MOE_OK) return st;
    }
    return MOE_OK;
}

MOE_EXPORT moe_status moe_forward_host(moe_layer* L, int32_t mode, const uint16_t* x_host, int32_t T,
                                       uint16_t* y_host, void* ws, size_t ws_bytes, void* stream) {
    moe_status st = check_layer_device(L);
    if (st != MOE_OK) return st;
    if (mode != MOE_MODE_PREFILL && mode != MOE_MODE_DECODE) return fail(MOE_ERR_INVALID_ARG, "mode must be 1 or 2");
    if (T < 0 || (T > 0 && (!x_host || !y_host))) return fail(MOE_ERR_INVALID_ARG, "bad host buffers or T");
    if (T == 0) return MOE_OK;
    const size_t fwd = make_layout(L, T, mode).total;
    const size_t xb = up((size_t)T * L->d.hidden * 2, 256);
    if (!ws || !aligned(ws, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
    if (ws_bytes < fwd + 2 * xb) return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, fwd + 2 * xb);
    char* base = static_cast<char*>(ws);
    uint16_t* xd = reinterpret_cast<uint16_t*>(base + fwd);
    uint16_t* yd = reinterpret_cast<uint16_t*>(base + fwd + xb);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)T * L->d.hidden * 2;
    MOE_CUDA(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s), "copy x to device");
    st = run_forward(L, mode, xd, T, yd, nullptr, base, fwd, s);
    if (st != MOE_OK) return st;
    MOE_CUDA(cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, s), "copy y to host");
    MOE_CUDA(cudaStreamSynchronize(s), "synchronise");
    return MOE_OK;
}

MOE_EXPORT moe_status moe_get_device_status(moe_layer* L, void* stream, uint32_t* flags) {
    moe_status st = check_layer_device(L);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    MOE_CUDA(cudaStreamSynchronize(s), "synchronise");
    MOE_CUDA(cudaMemcpy(&v, L->dev_status, 4, cudaMemcpyDeviceToHost), "read status");
    MOE_CUDA(cudaMemset(L->dev_status, 0, 4), "clear status");
    if (flags) *flags = v;
    if (v & MOE_DEV_WAIT_TIMEOUT) return fail(MOE_ERR_TIMEOUT, "a kernel wait gave up (status 0x%x)", v);
    if (v) return fail(MOE_ERR_DEVICE_CHECK, "a kernel flagged bad data (status 0x%x)", v);
    return MOE_OK;
}

MOE_EXPORT moe_status moe_set_wait_limit(moe_layer* L, uint32_t limit) {
    moe_status st = check_layer(L);
    if (st != MOE_OK) return st;
    if (limit == 0) return fail(MOE_ERR_INVALID_ARG, "limit must be positive");
    L->wait_limit = limit;
    return MOE_OK;
}

MOE_EXPORT moe_status moe_profile_enable(moe_layer* L, int32_t enable) {
    moe_status st = check_layer_device(L);
    if (st != MOE_OK) return st;
    const uint32_t all = (1u << MOE_PROFILE_STAGES) - 1u;
    uint32_t mask = 0;
    if (enable == 1) {
        mask = all;
    } else if (enable != 0) {
        if (!(enable & MOE_PROFILE_SELECT) || (enable & ~(MOE_PROFILE_SELECT | (int32_t)all)) != 0 ||
            (enable & (int32_t)all) == 0)
            return fail(MOE_ERR_INVALID_ARG, "profile selector %#x names no stage or an unknown one", (unsigned)enable);
        mask = (uint32_t)enable & all;
    }
    if (mask && !L->profile) {
        for (int i = 0; i <= MOE_PROFILE_STAGES; ++i) MOE_CUDA(cudaEventCreate(&L->ev[i]), "event create");
        L->ev_stream = nullptr;
    } else if (!mask && L->profile) {
        MOE_CUDA(cudaDeviceSynchronize(), "synchronise");
        for (int i = 0; i <= MOE_PROFILE_STAGES; ++i) cudaEventDestroy(L->ev[i]);
    }
    L->profile = mask;
    return MOE_OK;
}

MOE_EXPORT moe_status moe_profile_read(moe_layer* L, float* stage_ms, int32_t n) {
    moe_status st = check_layer(L);
    if (st != MOE_OK) return st;
    if (!L->profile) return fail(MOE_ERR_INVALID_ARG, "profiling is not enabled");
    if (!stage_ms || n < 1 || n > MOE_PROFILE_STAGES) return fail(MOE_ERR_INVALID_ARG, "bad stage buffer");
    int last = 0;                                       // the last recorded event closes the last timed stage
    for (int i = 0; i < MOE_PROFILE_STAGES; ++i)
        if ((L->profile >> i) & 1u) last = i + 1;
    MOE_CUDA(cudaEventSynchronize(L->ev[last]), "event synchronise");
    for (int i = 0; i < n; ++i) {
        if ((L->profile >> i) & 1u)
            MOE_CUDA(cudaEventElapsedTime(&stage_ms[i], L->ev[i], L->ev[i + 1]), "elapsed");
        else
            stage_ms[i] = -1.0f;
    }
    return MOE_OK;
}

MOE_EXPORT moe_status moe_debug_timeout_probe(moe_layer* L, void* stream) {
    moe_status st = check_layer_device(L);
    if (st != MOE_OK) return st;
    MOE_CUDA(moe::launch_timeout_probe(L, static_cast<cudaStream_t>(stream)), "timeout probe");
    return MOE_OK;
}

MOE_EXPORT moe_status moe_debug_inject(moe_layer* L, uint32_t faults) {
    moe_status st = check_layer(L);
    if (st != MOE_OK) return st;
    if (faults & ~(uint32_t)(MOE_DEV_BAD_EXPERT_ID | MOE_DEV_BAD_ROW))
        return fail(MOE_ERR_INVALID_ARG, "only MOE_DEV_BAD_EXPERT_ID and MOE_DEV_BAD_ROW can be planted (got %#x)",
                    faults);
    L->inject |= faults;
    return MOE_OK;
}
