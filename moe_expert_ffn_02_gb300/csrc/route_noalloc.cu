// moe_route_from_logits_noalloc: the routing stage (top-k, gate weights,
// expert grouping) from given logits, with its scratch memory in a
// fixed-size array compiled into this library instead of a caller-supplied
// workspace.
//
// Who needs it: callers that cannot allocate device memory when they route
// -- serving runtimes that hand all of HBM to their own pools (weights, KV
// cache) at start-up and forbid later cudaMalloc, and plain C programs that
// link this library without any allocator of their own.  For them a
// workspace argument is a burden, and a cudaMalloc in the middle of a step
// would also synchronise the whole device.
//
// The array costs every GPU that loads the library kStaticScratchBytes of
// device memory until the process exits.
#include "moe_internal.cuh"

#include <mutex>
#include <string>

namespace {

constexpr size_t kStaticScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;   // 4 MiB
constexpr int kMaxDevices = 64;

// The scratch itself.  Host code must not use this name as an address: on
// the host it is only a stand-in for the symbol; the device address comes
// from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

moe_status noalloc_fail(moe_status s, const std::string& msg) {
    moe::set_last_error(msg.c_str());
    return s;
}

inline size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Carve the routing scratch for (T, E, k) out of the array: the same pieces
// the workspace-based routing uses, without the router-GEMM partial sums and
// the expert-GEMM buffers (never touched when routing from logits).
moe::WsLayout route_layout(const moe_layer* L, int T) {
    moe::WsLayout l{};
    const size_t E = L->d.n_experts, k = L->d.top_k, R = (size_t)T * k;
    l.n_chunks = (T + moe::CHUNK_TOK - 1) / moe::CHUNK_TOK;
    l.ksplit = 1;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = up(off + bytes, 256); return o; };
    l.ids = take(R * 4);
    l.w = take(R * 4);
    l.chunk_cnt = take((size_t)l.n_chunks * E * 4);
    l.chunk_base = take((size_t)l.n_chunks * E * 4);
    l.offsets = take((E + 1) * 4);
    l.offsets_pad = take((E + 1) * 4);
    l.inv_row = take(R * 4);
    l.inv_int = take(R * 4);
    l.table = take(sizeof(moe::GroupTable));
    l.total = off;
    return l;
}

// Once per device: the device address of the array, looked up with that
// device current (the caller has checked that `device` is the current one).
// Runs on the first call of the entry point on each device.
moe_status scratch_on(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return noalloc_fail(MOE_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_addr[device]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess || !p)
            return noalloc_fail(MOE_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return MOE_OK;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) moe_status moe_route_from_logits_noalloc(
    moe_layer* L, const float* logits, int32_t T, const moe_route_out* out, void* stream) {
    moe::set_last_error("");
    if (!L) return noalloc_fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    int cur = -1;
    cudaError_t ge = cudaGetDevice(&cur);
    if (ge != cudaSuccess) return noalloc_fail(MOE_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ge));
    if (cur != L->device)
        return noalloc_fail(MOE_ERR_INVALID_ARG, "the current device (" + std::to_string(cur) +
                                                     ") is not the layer's device (" + std::to_string(L->device) + ")");
    if (T < 0) return noalloc_fail(MOE_ERR_INVALID_ARG, "T is negative");
    if (T > 0 && !logits) return noalloc_fail(MOE_ERR_INVALID_ARG, "logits is NULL");
    if (logits && (reinterpret_cast<uintptr_t>(logits) % 16))
        return noalloc_fail(MOE_ERR_INVALID_ARG, "logits is not 16-byte aligned");
    const moe::WsLayout lay = route_layout(L, T);
    if (lay.total > kStaticScratchBytes)
        return noalloc_fail(MOE_ERR_UNSUPPORTED,
                            "routing scratch for T=" + std::to_string(T) + " needs " + std::to_string(lay.total) +
                                " bytes; the built-in scratch holds " + std::to_string(kStaticScratchBytes));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (out && out->expert_offsets) {
            cudaError_t e = cudaMemsetAsync(out->expert_offsets, 0, sizeof(int32_t) * (L->d.n_experts + 1), s);
            if (e != cudaSuccess) return noalloc_fail(MOE_ERR_CUDA, cudaGetErrorString(e));
        }
        return MOE_OK;
    }
    void* base = nullptr;
    moe_status st = scratch_on(L->device, &base);
    if (st != MOE_OK) return st;
    char* ws = static_cast<char*>(base);
    const int k = L->d.top_k;
    int32_t* ids = reinterpret_cast<int32_t*>(ws + lay.ids);
    float* w = reinterpret_cast<float*>(ws + lay.w);
    cudaError_t e = moe::launch_topk(L, logits, 1, false, T, nullptr, ids, w, s);
    if (e == cudaSuccess && out && out->topk_ids)
        e = cudaMemcpyAsync(out->topk_ids, ids, sizeof(int32_t) * (size_t)T * k, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && out && out->topk_w)
        e = cudaMemcpyAsync(out->topk_w, w, sizeof(float) * (size_t)T * k, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
        e = moe::launch_permute(L, ids, T, lay, ws, moe::DEC_TILE_N, out ? out->expert_offsets : nullptr,
                                out ? out->sorted_token : nullptr, out ? out->inv_row : nullptr, s);
    if (e != cudaSuccess) return noalloc_fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    return MOE_OK;
}
