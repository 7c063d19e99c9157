// Combine of the expert outputs and the small kernels around the expert
// GEMMs: the weighted combine (and its split / deferred variant), the debug
// copy of h in token order, the repack of the checkpoint's FP8 weights into
// tile images at load time, the bounded-wait probe and the host-side fault
// injection.
#include "moe_internal.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Combine ("weighted reduction" after the experts, SmallEP section of the
// CPU-GPU hybrid inference article): per token, in this fixed order,
//   y = O[shared row] + w_0 O[row_0] + ... + w_{k-1} O[row_{k-1}]
// in fp32, rounded once to bf16.  CTA (token, blockIdx.y) owns 1024
// channels, 4 per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ O, const int32_t* __restrict__ inv_int,
                                                      const float* __restrict__ w, const int32_t* __restrict__ offsets_pad,
                                                      int T, int H, int k, int E, int n_shared, int ld,
                                                      uint16_t* __restrict__ y, uint32_t* status) {
    __shared__ int rows[MAX_TOPK];
    __shared__ float wt[MAX_TOPK];
    const int t = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x < k) {
        // a row outside the expert outputs is flagged and its slot left out (never read)
        const int row = inv_int[(size_t)t * k + threadIdx.x];
        const bool ok = row >= 0 && row < ld;
        if (!ok && blockIdx.y == 0) atomicOr(status, MOE_DEV_BAD_ROW);
        rows[threadIdx.x] = ok ? row : -1;
        wt[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
    }
    __syncthreads();
    const size_t shrow = (size_t)offsets_pad[E] + t;
    for (int c = (blockIdx.y * blockDim.x + threadIdx.x) * 4; c < H; c += gridDim.y * blockDim.x * 4) {
        float4 acc = n_shared ? *reinterpret_cast<const float4*>(O + shrow * H + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            if (rows[j] < 0) continue;
            const float4 o = *reinterpret_cast<const float4*>(O + (size_t)rows[j] * H + c);
            const float wj = wt[j];
            acc.x = __fmaf_rn(wj, o.x, acc.x);
            acc.y = __fmaf_rn(wj, o.y, acc.y);
            acc.z = __fmaf_rn(wj, o.z, acc.z);
            acc.w = __fmaf_rn(wj, o.w, acc.w);
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(y + (size_t)t * H + c) = pk;
    }
}

cudaError_t launch_combine(const moe_layer* L, int T, const WsLayout& lay, char* ws, uint16_t* y, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    // CTA (token, blockIdx.y) owns channels [1024 blockIdx.y, +1024): one float4 per thread
    const dim3 grid(T, (L->d.hidden + 1023) / 1024);
    return launch_pdl(combine_kernel, grid, dim3(256), 0, s, reinterpret_cast<const float*>(ws + lay.o),
                                     reinterpret_cast<const int32_t*>(ws + lay.inv_int),
                                     reinterpret_cast<const float*>(ws + lay.w),
                                     reinterpret_cast<const int32_t*>(ws + lay.offsets_pad), T, L->d.hidden, L->d.top_k,
                                     L->d.n_experts, L->d.n_shared, lay.rows_pad, y, L->dev_status);
}

// ---------------------------------------------------------------------------
// Split combines (same inputs as combine_kernel, same fp32 fused multiply-adds
// in slot order inside each part).
//
// SmallEP partial sums (SmallEP section of the CPU-GPU hybrid inference
// article, Fig. 5: each expert-parallel rank combines its own experts, then
// the partial outputs are reduced): the routed experts are split into
// n_ranks contiguous groups, rank p holding experts [ceil(p E / P),
// ceil((p+1) E / P)) and rank 0 also the shared expert.  Part p = (p == 0 ?
// O[shared] : 0) + sum over the slots j whose expert rank p holds, in slot
// order, of w_j O[row_j]; y = bf16(((part_0 + part_1) + part_2) + ...).  With
// one rank this is exactly combine_kernel.
//
// Deferral (when defer != NULL; n_ranks is then 1): the slots with
// defer[t][j] != 0 go to y_next = bf16(sum of their w_j O[row_j]), the others
// and the shared expert to y = bf16(O[shared] + sum of theirs).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_split_kernel(const float* __restrict__ O,
                                                            const int32_t* __restrict__ inv_int,
                                                            const int32_t* __restrict__ ids,
                                                            const float* __restrict__ w,
                                                            const int32_t* __restrict__ offsets_pad,
                                                            const uint8_t* __restrict__ defer, int T, int H, int k,
                                                            int E, int n_shared, int n_ranks, int ld,
                                                            uint16_t* __restrict__ y, uint16_t* __restrict__ y_next,
                                                            uint32_t* status) {
    __shared__ int rows[MAX_TOPK], part_of[MAX_TOPK];
    __shared__ float wt[MAX_TOPK];
    const int t = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x < k) {
        const int j = threadIdx.x;
        const int row = inv_int[(size_t)t * k + j];
        const bool ok = row >= 0 && row < ld;
        if (!ok && blockIdx.y == 0) atomicOr(status, MOE_DEV_BAD_ROW);
        rows[j] = ok ? row : -1;
        wt[j] = w[(size_t)t * k + j];
        if (defer) {
            part_of[j] = defer[(size_t)t * k + j] ? 1 : 0;
        } else {
            const int e = min(max(ids[(size_t)t * k + j], 0), E - 1);
            int p = 0;                              // largest p with ceil(p E / P) <= e
            while (p + 1 < n_ranks && (int)(((long long)(p + 1) * E + n_ranks - 1) / n_ranks) <= e) ++p;
            part_of[j] = p;
        }
    }
    __syncthreads();
    const int nparts = defer ? 2 : n_ranks;
    const size_t shrow = (size_t)offsets_pad[E] + t;
    for (int c = (blockIdx.y * blockDim.x + threadIdx.x) * 4; c < H; c += gridDim.y * blockDim.x * 4) {
        float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < nparts; ++p) {
            float4 acc = (p == 0 && n_shared) ? *reinterpret_cast<const float4*>(O + shrow * H + c)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < k; ++j) {
                if (part_of[j] != p || rows[j] < 0) continue;
                const float4 o = *reinterpret_cast<const float4*>(O + (size_t)rows[j] * H + c);
                const float wj = wt[j];
                acc.x = __fmaf_rn(wj, o.x, acc.x);
                acc.y = __fmaf_rn(wj, o.y, acc.y);
                acc.z = __fmaf_rn(wj, o.z, acc.z);
                acc.w = __fmaf_rn(wj, o.w, acc.w);
            }
            if (defer) {
                uint16_t* dst = (p == 0 ? y : y_next) + (size_t)t * H + c;
                const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
                *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                                                            *reinterpret_cast<const uint32_t*>(&hi));
            } else if (p == 0) {
                tot = acc;
            } else {
                tot.x = __fadd_rn(tot.x, acc.x);
                tot.y = __fadd_rn(tot.y, acc.y);
                tot.z = __fadd_rn(tot.z, acc.z);
                tot.w = __fadd_rn(tot.w, acc.w);
            }
        }
        if (!defer) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(tot.x, tot.y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(tot.z, tot.w);
            *reinterpret_cast<uint2*>(y + (size_t)t * H + c) = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                                                                           *reinterpret_cast<const uint32_t*>(&hi));
        }
    }
}

cudaError_t launch_combine_split(const moe_layer* L, int T, const WsLayout& lay, char* ws, int n_ranks,
                                 const uint8_t* defer, uint16_t* y, uint16_t* y_next, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const dim3 grid(T, (L->d.hidden + 1023) / 1024);
    return launch_pdl(combine_split_kernel, grid, dim3(256), 0, s, 
        reinterpret_cast<const float*>(ws + lay.o), reinterpret_cast<const int32_t*>(ws + lay.inv_int),
        reinterpret_cast<const int32_t*>(ws + lay.ids), reinterpret_cast<const float*>(ws + lay.w),
        reinterpret_cast<const int32_t*>(ws + lay.offsets_pad), defer, T, L->d.hidden, L->d.top_k, L->d.n_experts,
        L->d.n_shared, n_ranks, lay.rows_pad, y, y_next, L->dev_status);
}

// ---------------------------------------------------------------------------
// Debug copy of the h codes and scales per (token, slot), slots 0..k-1 the
// routed experts in rank order and slot k the shared expert, unswizzled:
// hq_out [T][S][I], sh_out [T][S][I/128].  One CTA per token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) h_gather_kernel(const uint8_t* __restrict__ hq, const float* __restrict__ shT,
                                                       int ld, const int32_t* __restrict__ inv_int,
                                                       const int32_t* __restrict__ offsets_pad, int E, int k, int S,
                                                       int I, uint8_t* __restrict__ hq_out, float* __restrict__ sh_out,
                                                       uint32_t* status) {
    const int t = blockIdx.x;
    const int IB = I / QB;
    for (int slot = 0; slot < S; ++slot) {
        const int row = slot < k ? inv_int[(size_t)t * k + slot] : offsets_pad[E] + t;
        if (row < 0 || row >= ld) {                     // flagged and skipped, never read
            if (threadIdx.x == 0) atomicOr(status, MOE_DEV_BAD_ROW);
            continue;
        }
        const size_t rec = (size_t)t * S + slot;
        if (hq_out)
            for (int c = threadIdx.x; c < IB * 8; c += blockDim.x) {
                const int ib = c >> 3, ch = c & 7;
                const uint4 v = *reinterpret_cast<const uint4*>(hq + act_offset(ib, row, ld) + ((ch ^ (row & 7)) * 16));
                *reinterpret_cast<uint4*>(hq_out + rec * I + ib * QB + ch * 16) = v;
            }
        if (sh_out)
            for (int ib = threadIdx.x; ib < IB; ib += blockDim.x) sh_out[rec * IB + ib] = shT[(size_t)ib * ld + row];
    }
}

cudaError_t launch_h_gather(const moe_layer* L, int T, const WsLayout& lay, char* ws, uint8_t* hq_out, float* sh_out,
                            cudaStream_t s) {
    if (T == 0 || (!hq_out && !sh_out)) return cudaSuccess;
    const int S = L->d.top_k + L->d.n_shared;
    h_gather_kernel<<<T, 128, 0, s>>>(reinterpret_cast<const uint8_t*>(ws + lay.hq),
                                      reinterpret_cast<const float*>(ws + lay.shT), lay.rows_pad,
                                      reinterpret_cast<const int32_t*>(ws + lay.inv_int),
                                      reinterpret_cast<const int32_t*>(ws + lay.offsets_pad), L->d.n_experts,
                                      L->d.top_k, S, L->d.inter, hq_out, sh_out, L->dev_status);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Weight repacking at load time (KTransformers deep dive, section 2.2:
// expert weights are laid out once for the compute unit).  Checkpoint
// [G][R][C] row-major codes -> tile images (see moe_internal.cuh); gate and
// up interleaved per (row block, k block).  One thread per 16-byte chunk.
// ---------------------------------------------------------------------------
__global__ void repack_kernel(const uint8_t* __restrict__ src0, const uint8_t* __restrict__ src1, int n_mat_per_tile,
                              int G, int R, int C, uint8_t* __restrict__ dst) {
    const size_t n_chunks = (size_t)G * R * C / 16 * n_mat_per_tile;
    const int RB = R / QB, CB = C / QB;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n_chunks; i += (size_t)gridDim.x * blockDim.x) {
        size_t rem = i;
        const int cpos = rem % 8; rem /= 8;
        const int r = rem % QB; rem /= QB;
        const int mat = rem % n_mat_per_tile; rem /= n_mat_per_tile;
        const int cb = rem % CB; rem /= CB;
        const int rb = rem % RB; rem /= RB;
        const int gidx = (int)rem;
        const int c = cpos ^ (r & 7);
        const uint8_t* src = mat ? src1 : src0;
        const uint4 v = *reinterpret_cast<const uint4*>(src + ((size_t)gidx * R + rb * QB + r) * C + cb * QB + c * 16);
        *reinterpret_cast<uint4*>(dst + i * 16) = v;
    }
}

__global__ void repack_scales_kernel(const float* __restrict__ s0, const float* __restrict__ s1, int n_mat, size_t n,
                                     float* __restrict__ dst) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        dst[i * n_mat] = s0[i];
        if (n_mat == 2) dst[i * 2 + 1] = s1[i];
    }
}

cudaError_t launch_repack(const moe_layer* L, const moe_weights* w, cudaStream_t s) {
    const int H = L->d.hidden, I = L->d.inter, E = L->d.n_experts;
    const size_t gu_per = (size_t)I * H * 2, dn_per = (size_t)H * I;
    const size_t sgu_per = (size_t)(I / QB) * (H / QB) * 2, sdn_per = (size_t)(H / QB) * (I / QB);
    const int threads = 256, blocks = 4 * L->num_sms;
    repack_kernel<<<blocks, threads, 0, s>>>(w->w_gate, w->w_up, 2, E, I, H, L->w_gu);
    repack_kernel<<<blocks, threads, 0, s>>>(w->w_down, w->w_down, 1, E, H, I, L->w_dn);
    repack_scales_kernel<<<blocks, threads, 0, s>>>(w->s_gate, w->s_up, 2, (size_t)E * (I / QB) * (H / QB), L->s_gu);
    repack_scales_kernel<<<blocks, threads, 0, s>>>(w->s_down, w->s_down, 1, (size_t)E * (H / QB) * (I / QB), L->s_dn);
    if (L->d.n_shared) {
        repack_kernel<<<blocks, threads, 0, s>>>(w->sh_gate, w->sh_up, 2, 1, I, H, L->w_gu + (size_t)E * gu_per);
        repack_kernel<<<blocks, threads, 0, s>>>(w->sh_down, w->sh_down, 1, 1, H, I, L->w_dn + (size_t)E * dn_per);
        repack_scales_kernel<<<blocks, threads, 0, s>>>(w->sh_s_gate, w->sh_s_up, 2, (size_t)(I / QB) * (H / QB),
                                                        L->s_gu + (size_t)E * sgu_per);
        repack_scales_kernel<<<blocks, threads, 0, s>>>(w->sh_s_down, w->sh_s_down, 1, (size_t)(H / QB) * (I / QB),
                                                        L->s_dn + (size_t)E * sdn_per);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// A bounded wait on an mbarrier nobody signals: exercises the timeout path
// (status bit set, kernel returns) without hanging or faulting.
// ---------------------------------------------------------------------------
__global__ void timeout_probe_kernel(uint32_t* status, uint32_t limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait_bounded(&bar, 0, limit, status, nullptr);
    }
}

cudaError_t launch_timeout_probe(const moe_layer* L, cudaStream_t s) {
    timeout_probe_kernel<<<1, 32, 0, s>>>(L->dev_status, L->wait_limit);
    return cudaGetLastError();
}

// Fault injection (moe_debug_inject): overwrite one routing word in the
// workspace with a value the checked kernels must flag and skip.
__global__ void plant_kernel(int32_t* word, int32_t value) { *word = value; }

cudaError_t launch_plant(int32_t* word, int32_t value, cudaStream_t s) {
    plant_kernel<<<1, 1, 0, s>>>(word, value);
    return cudaGetLastError();
}

}  // namespace moe
