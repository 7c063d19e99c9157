// Routing stage of the MoE layer on sm_103a: router logits, top-k with gate
// weights, expert grouping (histogram -> scan -> stable scatter) and the
// 1x128 E4M3 quantisation of x written straight into the grouped rows.
//
// Sources: "KTransformers deep dive" (chenxutan.com), section 1.2 (router
// picks 8 of 256 experts plus a shared one) and section 2.2 (tokens of one
// expert are batched so GEMV becomes GEMM); CPU-GPU hybrid inference article
// (xingyun.xin), SmallEP section / Fig. 5 (gating and sorting come before
// dispatch).  Scoring = softmax over the selected logits (renormalised
// top-k), ties to the lower expert index.
#include "moe_internal.cuh"

#include <math_constants.h>

namespace moe {

// ---------------------------------------------------------------------------
// Router logits for a decode batch (T <= 64): a GEMV over the fp32 router
// weights, which dominate the bytes.  The channels are split into ksplit
// slices (grid.y) and the experts into groups of 8 (grid.x); each CTA's
// weight and x slices come into shared memory by bulk copies (no per-thread
// load is in flight, so one round trip brings all of them), and the
// slice's partial sum goes to part[slice][t][e]; the top-k kernel adds the
// slices in order, so the result is deterministic.
// ---------------------------------------------------------------------------
constexpr int GEMV_WARPS = 8, GEMV_TC = 16;
constexpr size_t PF_CHUNK = 64 << 10;   // bytes per L2 prefetch instruction
constexpr int PF_MIN_TOKENS = 16;       // decode batches from this size on prefetch the shared expert

// The shared expert's gate/up tiles do not depend on the routing: their
// prefetch into L2, 64 KB pieces spread over the CTAs, overlaps routing and
// quantisation, and the gate/up GEMM takes the shared expert's units first.
__device__ __forceinline__ void prefetch_shared_expert(const uint8_t* pf, size_t pf_bytes) {
    if (pf && threadIdx.x == 0) {
        const size_t n_cta = (size_t)gridDim.x * gridDim.y;
        for (size_t off = ((size_t)blockIdx.y * gridDim.x + blockIdx.x) * PF_CHUNK; off < pf_bytes;
             off += n_cta * PF_CHUNK)
            l2_prefetch(pf + off, (uint32_t)min((size_t)PF_CHUNK, pf_bytes - off));
    }
}

// One CTA's share of the split GEMV: experts e_base .. e_base + 7 (warp w
// takes e_base + w), channels [z * slice, (z + 1) * slice) with z =
// blockIdx.y.  Thread 0 moves every operand into shared memory with bulk
// copies: the experts' weight rows in chunks of up to GEMV_WCH channels (two
// buffers), the tokens' x slices per pass of up to tc tokens.  The first
// weight chunk is issued before the programmatic-launch wait (the router
// weights do not depend on the preceding kernel), and a single-chunk slice is
// copied once for all passes.  Lane l accumulates channels 4l, 4l + 128, ...
// of the slice in ascending order, one product chain of four channels at a
// time; the lanes are combined by a fixed shuffle tree and the partial sum
// goes to part[z][t][e].  A thread whose wait timed out skips its waits and
// arithmetic from then on but still reaches every CTA barrier; nothing more is
// written or issued, and the copies in flight land before the CTA exits.
constexpr int GEMV_WCH = 1024;          // weight channels per chunk and expert (4 KB)

__global__ void __launch_bounds__(GEMV_WARPS * 32) router_gemv_kernel(const uint16_t* __restrict__ x,
                                                                      const float* __restrict__ W, int T, int H,
                                                                      int E, int slice, int tc,
                                                                      float* __restrict__ part,
                                                                      const uint8_t* __restrict__ pf,
                                                                      size_t pf_bytes, uint32_t* status,
                                                                      uint32_t wait_limit) {
    extern __shared__ __align__(128) uint8_t gsm[];
    const int wch = min(slice, GEMV_WCH);                        // channels per chunk
    const int nch = (slice + GEMV_WCH - 1) / GEMV_WCH;           // chunks per slice
    float* wbuf = reinterpret_cast<float*>(gsm);                 // [nch > 1 ? 2 : 1][GEMV_WARPS][wch]
    uint16_t* xs = reinterpret_cast<uint16_t*>(gsm + (size_t)(nch > 1 ? 2 : 1) * GEMV_WARPS * wch * 4);  // [tc][slice]
    __shared__ uint64_t wbar[2], xbar;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int z = blockIdx.y, h0 = z * slice;
    const int e_base = blockIdx.x * GEMV_WARPS;
    const int ne = min(GEMV_WARPS, E - e_base);
    const int e = e_base + warp;
    if (threadIdx.x == 0) {
        mbar_init(&wbar[0], 1);
        mbar_init(&wbar[1], 1);
        mbar_init(&xbar, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    volatile int* abort = &abort_flag;
    // chunk c of the slice into buffer (c & 1): ne weight rows of cw channels
    auto issue_w = [&](int c) {
        const int cw = min(wch, slice - c * GEMV_WCH);
        float* dst = wbuf + (size_t)(c & 1) * GEMV_WARPS * wch;
        mbar_arrive_expect_tx(&wbar[c & 1], (uint32_t)(ne * cw * 4));
        for (int w = 0; w < ne; ++w)
            bulk_g2s(dst + (size_t)w * wch, W + (size_t)(e_base + w) * H + h0 + (size_t)c * GEMV_WCH, cw * 4,
                     &wbar[c & 1]);
    };
    uint32_t wphase[2] = {0u, 0u}, xphase = 0u;
    uint32_t pend = 0;                 // bit b: wbar[b] armed and not yet waited; bit 2: xbar
    if (threadIdx.x == 0) {
        issue_w(0);
        pend |= 1u;
    }
    prefetch_shared_expert(pf, pf_bytes);
    pdl_wait();
    // the dependents launch only now, when the layer input x is complete: the quantiser reads x
    // before its own wait
    pdl_trigger();
    bool dead = false;
    for (int t0 = 0; t0 < T; t0 += tc) {
        const int nt = min(tc, T - t0);
        if (threadIdx.x == 0 && !dead) {
            mbar_arrive_expect_tx(&xbar, (uint32_t)(nt * slice * 2));
            for (int tt = 0; tt < nt; ++tt)
                bulk_g2s(xs + (size_t)tt * slice, x + (size_t)(t0 + tt) * H + h0, slice * 2, &xbar);
            pend |= 4u;
        }
        if (!dead) {
            if (mbar_wait_bounded(&xbar, xphase, wait_limit, status, abort)) {
                xphase ^= 1u;
                if (threadIdx.x == 0) pend &= ~4u;
            } else {
                dead = true;
            }
        }
        dead = __any_sync(0xFFFFFFFFu, dead);                      // warp-uniform (the shuffles below)
        float acc[GEMV_TC];
#pragma unroll
        for (int u = 0; u < GEMV_TC; ++u) acc[u] = 0.f;
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            if (nch > 1 && threadIdx.x == 0 && c + 1 < nch && !dead) {   // the next chunk into the other buffer
                issue_w(c + 1);
                pend |= 1u << ((c + 1) & 1);
            }
            // a single-chunk slice stays resident: its barrier is waited on in the first pass only
            if ((nch > 1 || t0 == 0) && !dead) {
                if (mbar_wait_bounded(&wbar[b], wphase[b], wait_limit, status, abort)) {
                    wphase[b] ^= 1u;
                    if (threadIdx.x == 0) pend &= ~(1u << b);
                } else {
                    dead = true;
                }
            }
            dead = __any_sync(0xFFFFFFFFu, dead);
            if (warp < ne && !dead) {
                const float* wr = wbuf + ((size_t)b * GEMV_WARPS + warp) * wch;
                const int cw = min(wch, slice - c * GEMV_WCH);
                const int cbase = c * GEMV_WCH;
                for (int cc = lane * 4; cc < cw; cc += 128) {
                    const float4 wv = *reinterpret_cast<const float4*>(wr + cc);
#pragma unroll
                    for (int u = 0; u < GEMV_TC; ++u) {
                        if (u < nt) {
                            const uint2 raw = *reinterpret_cast<const uint2*>(xs + (size_t)u * slice + cbase + cc);
                            float p = __fmul_rn(__uint_as_float(raw.x << 16), wv.x);
                            p = __fmaf_rn(__uint_as_float(raw.x & 0xFFFF0000u), wv.y, p);
                            p = __fmaf_rn(__uint_as_float(raw.y << 16), wv.z, p);
                            p = __fmaf_rn(__uint_as_float(raw.y & 0xFFFF0000u), wv.w, p);
                            acc[u] = __fadd_rn(acc[u], p);
                        }
                    }
                }
            }
            if (nch > 1) __syncthreads();                          // buffer b free for chunk c + 2
        }
        if (warp < ne && !dead) {
#pragma unroll
            for (int u = 0; u < GEMV_TC; ++u) {
                if (u < nt) {
                    float v = acc[u];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
                    if (lane == 0) part[((size_t)z * T + t0 + u) * E + e] = v;
                }
            }
        }
        __syncthreads();                                           // xs (and a resident chunk) reused next pass
        if (nch > 1 && t0 + tc < T && threadIdx.x == 0 && !dead) {   // the next pass starts from chunk 0 again
            issue_w(0);
            pend |= 1u;
        }
    }
    // copies still in flight after a timeout land before the CTA exits
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b)
            if ((pend >> b) & 1u) mbar_wait_bounded(&wbar[b], wphase[b], wait_limit, status, nullptr);
        if (pend & 4u) mbar_wait_bounded(&xbar, xphase, wait_limit, status, nullptr);
    }
}

// The shared expert's gate/up tile images (group E) to prefetch during the
// routing of a T-token decode batch, or none.  From 16 tokens on, the gate/up
// GEMM streams ~100 experts in many waves and is HBM-bound, and the shared
// expert's units, which it takes first, then read from L2.  Below that every
// unit runs in the first wave, bound by its SM's own stream rate, so the
// prefetch would only compete with the routing for HBM (measured: T = 1
// 132 -> 137 us, T = 16 770 -> 766 us with the prefetch at every T).
void shared_expert_prefetch(const moe_layer* L, int T, const uint8_t** pf, size_t* bytes) {
    *pf = nullptr;
    *bytes = 0;
    if (!L->d.n_shared || T < PF_MIN_TOKENS || !L->w_gu) return;
    const size_t gu_per = (size_t)L->d.inter * L->d.hidden * 2;
    *pf = L->w_gu + (size_t)L->d.n_experts * gu_per;
    *bytes = gu_per;
}

// Slices for the GEMV: the largest divisor of H/128 that is at most 8.
int router_gemv_splits(int H) {
    const int hb = H / QB;
    int d = 1;
    for (int c = 1; c <= 8; ++c)
        if (hb % c == 0) d = c;
    return d;
}

cudaError_t launch_router_logits(const moe_layer* L, const uint16_t* x, int T, float* part, int ksplit, bool gemv,
                                 cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int H = L->d.hidden, E = L->d.n_experts;
    if (gemv) {                                        // decode batch: split GEMV, ksplit partial sums
        const int slice = H / ksplit;
        const int tc = max(1, min(GEMV_TC, (128 * 1024) / (slice * 2)));
        const int nbuf = slice > GEMV_WCH ? 2 : 1;
        const size_t smem = (size_t)nbuf * GEMV_WARPS * min(slice, GEMV_WCH) * 4 + (size_t)tc * slice * 2;
        {
            cudaError_t e = ensure_smem_limit<router_gemv_kernel>(2 * GEMV_WARPS * GEMV_WCH * 4 + 128 * 1024);
            if (e != cudaSuccess) return e;
        }
        dim3 grid((E + GEMV_WARPS - 1) / GEMV_WARPS, ksplit);
        const uint8_t* pf = nullptr;
        size_t pf_bytes = 0;
        shared_expert_prefetch(L, T, &pf, &pf_bytes);
        return launch_pdl(router_gemv_kernel, grid, dim3(GEMV_WARPS * 32), smem, s, x, L->router_w, T, H, E, slice, tc,
                          part, pf, pf_bytes, L->dev_status, L->wait_limit);
    }
    return launch_router_tc(L, x, T, part, ksplit, s);      // prefill batch: tensor-core GEMM (router_tc.cu)
}

// ---------------------------------------------------------------------------
// exp in fp32 for the gate weights: Cody & Waite reduction x = n ln2 + r
// (ln2 split into a 15-significant-bit head, so n * head is exact for
// |n| < 512, and a tail), degree-7 Taylor polynomial of e^r on
// |r| <= ln2/2 by Horner's rule with fused multiply-adds, exact scaling by
// 2^n.  Arguments below -86 give 0 (keeps 2^n a normal number).  Every
// operation is an explicitly rounded fp32 intrinsic, so the result is fully
// determined by the argument.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float gate_exp(float x) {
    const float log2e = (float)1.4426950408889634;
    const float ln2_hi = 0x1.62e4p-1f;
    const float ln2_lo = (float)(0.69314718055994530942 - 0.693145751953125);
    const float c2 = (float)(1.0 / 2.0), c3 = (float)(1.0 / 6.0);
    const float c4 = (float)(1.0 / 24.0), c5 = (float)(1.0 / 120.0);
    const float c6 = (float)(1.0 / 720.0), c7 = (float)(1.0 / 5040.0);
    if (!(x >= -86.0f)) return 0.0f;
    if (x > 88.0f) return CUDART_INF_F;
    const float n = rintf(__fmul_rn(x, log2e));
    float r = __fmaf_rn(-n, ln2_hi, x);
    r = __fmaf_rn(-n, ln2_lo, r);
    float p = c7;
    p = __fmaf_rn(p, r, c6);
    p = __fmaf_rn(p, r, c5);
    p = __fmaf_rn(p, r, c4);
    p = __fmaf_rn(p, r, c3);
    p = __fmaf_rn(p, r, c2);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const float two_n = __int_as_float(((int)n + 127) << 23);
    return __fmul_rn(p, two_n);
}

// ---------------------------------------------------------------------------
// Top-k + gate weights, one warp per token.  Lane l holds experts
// l, l+32, ...; each of the k rounds takes the largest remaining logit,
// lower index on ties (-0 == +0; a NaN ranks below every number).  A round
// is two warp reductions: the maximum of an order-preserving integer key of
// the logits, then the minimum index among the lanes that hold it.
// Weights: m = L[id0]; e_j = exp(L[id_j] - m); S = e_0 + e_1 + ... summed
// left to right; w_j = e_j / S -- each step an IEEE-rounded fp32 op (lane j
// computes e_j and w_j; every lane forms S in the same order).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v != v) return 1u;                                    // NaN: below every number
    const uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v); // -0 -> +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);        // >= 0x007FFFFF for numbers
}

// `bias` may point to shared memory (a generic pointer: not read through the read-only path).
template <int PER>
__device__ void topk_token(const float* __restrict__ part, int ksplit, const float* bias, int T, int E,
                           int k, float* __restrict__ logits_out, int32_t* __restrict__ ids,
                           float* __restrict__ wout, int t, int lane, float* sel_v, int* sel_i) {
    // logits: the ksplit partial sums added in split order, then the bias.  The
    // partials are fetched ZB splits at a time for all PER experts of the lane
    // before any addition, so the loads are in flight together.
    constexpr int ZB = PER <= 8 ? 8 : (PER <= 16 ? 4 : 2);
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) v[i] = 0.f;
    for (int z0 = 0; z0 < ksplit; z0 += ZB) {
        float pv[PER][ZB];
#pragma unroll
        for (int i = 0; i < PER; ++i)
#pragma unroll
            for (int zz = 0; zz < ZB; ++zz) {
                const int e = lane + 32 * i, z = z0 + zz;
                pv[i][zz] = (e < E && z < ksplit) ? part[((size_t)z * T + t) * E + e] : 0.f;
            }
#pragma unroll
        for (int i = 0; i < PER; ++i)
#pragma unroll
            for (int zz = 0; zz < ZB; ++zz)
                if (z0 + zz < ksplit) v[i] = (z0 + zz == 0) ? pv[i][zz] : __fadd_rn(v[i], pv[i][zz]);
    }
    uint32_t key[PER];                    // 0: not an expert, or already taken
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0u;
        if (e < E) {
            if (bias) v[i] = __fadd_rn(v[i], bias[e]);
            if (logits_out) logits_out[(size_t)t * E + e] = v[i];
            key[i] = order_key(v[i]);
        }
    }
    // each lane orders its PER candidates once (key descending, index ascending: insertion into
    // a register list), then a round compares the lanes' heads and the winner pops its head
    uint32_t hk[PER];
    int hi[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) { hk[i] = 0u; hi[i] = 0x7FFFFFFF; }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        uint32_t ck = key[i];
        int ci = lane + 32 * i;                            // indices of a lane ascend with i
#pragma unroll
        for (int p = 0; p <= i; ++p) {                     // equal keys: the lower index first
            if (ck > hk[p] || (ck == hk[p] && ci < hi[p])) {
                const uint32_t tk = hk[p]; const int ti = hi[p];
                hk[p] = ck; hi[p] = ci;
                ck = tk; ci = ti;
            }
        }
    }
    for (int j = 0; j < k; ++j) {
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, hk[0]);
        const int win = (int)__reduce_min_sync(0xFFFFFFFFu, hk[0] == m ? (uint32_t)hi[0] : 0xFFFFFFFFu);
        if (win == hi[0]) {
#pragma unroll
            for (int i = 0; i < PER; ++i)
                if (i == (win >> 5)) sel_v[j] = v[i];
            sel_i[j] = win;
#pragma unroll
            for (int p = 0; p + 1 < PER; ++p) { hk[p] = hk[p + 1]; hi[p] = hi[p + 1]; }
            hk[PER - 1] = 0u;
            hi[PER - 1] = 0x7FFFFFFF;
        }
    }
    __syncwarp();
    const float m = sel_v[0];
    const float ej = lane < k ? gate_exp(__fsub_rn(sel_v[lane], m)) : 0.f;
    float S = 0.f;
    for (int j = 0; j < k; ++j) {
        const float ev = __shfl_sync(0xFFFFFFFFu, ej, j);
        S = (j == 0) ? ev : __fadd_rn(S, ev);
    }
    if (lane < k) {
        if (ids) ids[(size_t)t * k + lane] = sel_i[lane];
        if (wout) wout[(size_t)t * k + lane] = __fdiv_rn(ej, S);
    }
    __syncwarp();
}

template <int PER>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ part, int ksplit,
                                                   const float* __restrict__ bias, int T, int E, int k,
                                                   float* __restrict__ logits_out, int32_t* __restrict__ ids,
                                                   float* __restrict__ wout) {
    __shared__ float sel_v[8][MAX_TOPK];
    __shared__ int sel_i[8][MAX_TOPK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    pdl_trigger();
    pdl_wait();
    if (t >= T) return;
    topk_token<PER>(part, ksplit, bias, T, E, k, logits_out, ids, wout, t, lane, sel_v[warp], sel_i[warp]);
}

cudaError_t launch_topk(const moe_layer* L, const float* part, int ksplit, bool add_bias, int T, float* logits_out,
                        int32_t* ids, float* w, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int E = L->d.n_experts, k = L->d.top_k;
    const float* bias = add_bias ? L->router_b : nullptr;
    const int per = (E + 31) / 32;
    dim3 grid((T + 7) / 8);
#define MOE_TOPK_CASE(P)                                                                              \
    if (per <= P) {                                                                                   \
        return launch_pdl(topk_kernel<P>, grid, dim3(256), 0, s, part, ksplit, bias, T, E, k, logits_out, ids, w); \
    }
    MOE_TOPK_CASE(1) MOE_TOPK_CASE(2) MOE_TOPK_CASE(4) MOE_TOPK_CASE(8) MOE_TOPK_CASE(12)
    MOE_TOPK_CASE(16) MOE_TOPK_CASE(24) MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Expert grouping.  The (token, slot) pairs are cut into chunks of
// CHUNK_TOK tokens, one warp each.
//   count:   per chunk, per expert, how many pairs chose it;
//   scan:    one CTA turns the counts into the expert offsets (exclusive
//            prefix sum over experts) and, for every chunk, the first row
//            its pairs of expert e will take; it also builds the group
//            table the expert GEMMs iterate over;
//   scatter: each warp walks its chunk in token-major order, 32 pairs at a
//            time, ranks equal experts with a warp match, and writes
//            sorted_token / inv_row.  Rows inside an expert therefore
//            ascend with the token index, independent of scheduling.
// Ids outside [0, E) set MOE_DEV_BAD_EXPERT_ID and are clamped so that
// every later access stays in bounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int clamp_expert(int e, int E, uint32_t* status) {
    if (e < 0 || e >= E) {
        atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
        e = e < 0 ? 0 : E - 1;
    }
    return e;
}

// One warp counts chunk c (CHUNK_TOK tokens) into cnt (E ints of shared memory).
__device__ void count_chunk(const int32_t* __restrict__ ids, int T, int E, int k, int c, int32_t* cnt,
                            int32_t* __restrict__ chunk_cnt, uint32_t* status, int lane) {
    for (int e = lane; e < E; e += 32) cnt[e] = 0;
    __syncwarp();
    const int t0 = c * CHUNK_TOK;
    const int t1 = min(T, t0 + CHUNK_TOK);
    const int n = (t1 - t0) * k;
    for (int i = lane; i < n; i += 32) {
        const int e = clamp_expert(ids[(size_t)t0 * k + i], E, status);
        atomicAdd(&cnt[e], 1);
    }
    __syncwarp();
    for (int e = lane; e < E; e += 32) chunk_cnt[(size_t)c * E + e] = cnt[e];
}

__global__ void __launch_bounds__(128) perm_count_kernel(const int32_t* __restrict__ ids, int T, int E, int k,
                                                         int n_chunks, int32_t* __restrict__ chunk_cnt,
                                                         uint32_t* status) {
    extern __shared__ int32_t cnt_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x * 4 + warp;
    pdl_trigger();
    pdl_wait();
    if (c >= n_chunks) return;
    count_chunk(ids, T, E, k, c, cnt_smem + warp * E, chunk_cnt, status, lane);
}

// Exclusive scan across the block (blockDim.x a multiple of 32, at most
// 1024); returns this thread's prefix and writes the block total to *total.
__device__ int block_excl_scan_1024(int v, int* total) {
    __shared__ int warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int ws = lane < nwarps ? warp_sums[lane] : 0;
        int wi = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
            if (lane >= off) wi += o;
        }
        warp_sums[lane] = wi - ws;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int r = warp_sums[warp] + incl - v;
    __syncthreads();
    return r;
}

// Offsets, padded offsets and the group table from the per-expert pair
// counts; thread e of the block handles expert e (blockDim.x >= E) and
// passes tot = expert e's count (0 for e >= E).  Returns expert e's first
// row (*off_e) and first internal row (*poff_e).
__device__ void scan_counts(int tot, int T, int E, int n_shared, int bn, int32_t* __restrict__ offsets,
                            int32_t* __restrict__ offsets_pad, int32_t* __restrict__ offsets_out, GroupTable* gt,
                            int* off_e, int* poff_e) {
    __shared__ int total_s;
    const int e = threadIdx.x;
    const int off = block_excl_scan_1024(e < E ? tot : 0, &total_s);
    const int R = total_s;
    // internal row space: every group starts on a multiple of ROW_ALIGN rows
    const int padded = (e < E) ? (tot + ROW_ALIGN - 1) / ROW_ALIGN * ROW_ALIGN : 0;
    const int poff = block_excl_scan_1024(padded, &total_s);
    const int shared_row0 = total_s;
    if (e < E) {
        offsets[e] = off;
        offsets_pad[e] = poff;
        if (offsets_out) offsets_out[e] = off;
    }
    if (e == 0) {
        offsets[E] = R;
        offsets_pad[E] = shared_row0;
        if (offsets_out) offsets_out[E] = R;
    }
    *off_e = off;
    *poff_e = poff;
    // group table: the active routed experts in index order and the shared expert.  From
    // PF_MIN_TOKENS tokens on the shared expert comes first: its weights do not depend on the
    // routing, so the expert GEMMs start on them while the L2 prefetch of them issued during
    // routing is still resident; below that it comes last (measured: first costs a T = 1
    // decode layer ~3 us).  The order only schedules the units; every output row is computed
    // by one unit either way.
    const bool active = (e < E) && tot > 0;
    const int sh = (n_shared && T >= PF_MIN_TOKENS) ? 1 : 0;         // shared group in front
    const int sh_back = (n_shared && T > 0 && !sh) ? 1 : 0;          // shared group at the end
    const int sh_tiles = sh ? (T + bn - 1) / bn : 0;
    const int gidx = sh + block_excl_scan_1024(active ? 1 : 0, &total_s);
    const int n_routed = total_s;
    const int tiles = active ? (tot + bn - 1) / bn : 0;
    const int pstart = sh_tiles + block_excl_scan_1024(tiles, &total_s);
    const int routed_pairs = total_s;
    if (active) {
        gt->expert[gidx] = e;
        gt->row0[gidx] = poff;
        gt->rows[gidx] = tot;
        gt->pair_start[gidx] = pstart;
    }
    if (e == 0) {
        int ng = sh + n_routed, np = sh_tiles + routed_pairs;
        if (sh || sh_back) {
            const int g = sh ? 0 : ng;
            gt->expert[g] = E;
            gt->row0[g] = shared_row0;
            gt->rows[g] = T;
            gt->pair_start[g] = sh ? 0 : np;
            if (sh_back) {
                np += (T + bn - 1) / bn;
                ng += 1;
            }
        }
        gt->pair_start[ng] = np;
        gt->n_groups = ng;
        gt->n_pairs = np;
        gt->bn = bn;
        gt->total_rows = shared_row0 + (n_shared ? T : 0);
    }
}

// The same from the chunk counts of the multi-CTA grouping; also turns the
// counts into every chunk's first row per expert (chunk_base).
__device__ void scan_groups(const int32_t* __restrict__ chunk_cnt, int n_chunks, int T, int E, int k, int n_shared,
                            int bn, int32_t* __restrict__ chunk_base, int32_t* __restrict__ offsets,
                            int32_t* __restrict__ offsets_pad, int32_t* __restrict__ offsets_out, GroupTable* gt) {
    const int e = threadIdx.x;
    int tot = 0;
    if (e < E) {
        for (int c = 0; c < n_chunks; ++c) {
            const int v = chunk_cnt[(size_t)c * E + e];
            chunk_base[(size_t)c * E + e] = tot;
            tot += v;
        }
    }
    int off, poff;
    scan_counts(tot, T, E, n_shared, bn, offsets, offsets_pad, offsets_out, gt, &off, &poff);
    if (e < E)
        for (int c = 0; c < n_chunks; ++c) chunk_base[(size_t)c * E + e] += off;
}

__global__ void __launch_bounds__(1024) perm_scan_kernel(const int32_t* __restrict__ chunk_cnt, int n_chunks, int T,
                                                         int E, int k, int n_shared, int bn,
                                                         int32_t* __restrict__ chunk_base,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ offsets_pad,
                                                         int32_t* __restrict__ offsets_out, GroupTable* gt) {
    pdl_trigger();
    pdl_wait();
    scan_groups(chunk_cnt, n_chunks, T, E, k, n_shared, bn, chunk_base, offsets, offsets_pad, offsets_out, gt);
}

// One warp scatters chunk c: stable ranks within each expert from match_any
// over 32 assignments at a time and a running count per expert (E ints of
// shared memory in `run`).
__device__ void scatter_chunk(const int32_t* __restrict__ ids, int T, int E, int k, int c,
                              const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
                              const int32_t* __restrict__ offsets_pad, int32_t* __restrict__ sorted_token,
                              int32_t* __restrict__ inv_row, int32_t* __restrict__ inv_int, uint32_t* status,
                              int32_t* run, int lane) {
    for (int e = lane; e < E; e += 32) run[e] = 0;
    __syncwarp();
    const int t0 = c * CHUNK_TOK;
    const int t1 = min(T, t0 + CHUNK_TOK);
    const int n = (t1 - t0) * k;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int b = 0; b < n; b += 32) {
        const int i = b + lane;
        const bool valid = i < n;
        int e = valid ? clamp_expert(ids[(size_t)t0 * k + i], E, status) : -1 - lane;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
        const int rank = __popc(peers & lt_mask);
        if (valid) {
            const int row = chunk_base[(size_t)c * E + e] + run[e] + rank;
            const int t = t0 + i / k;
            if (sorted_token) sorted_token[row] = t;
            inv_row[(size_t)t0 * k + i] = row;
            inv_int[(size_t)t0 * k + i] = row - offsets[e] + offsets_pad[e];
        }
        __syncwarp();
        if (valid && (peers & lt_mask) == 0) run[e] += __popc(peers);
        __syncwarp();
    }
}

__global__ void __launch_bounds__(128) perm_scatter_kernel(const int32_t* __restrict__ ids, int T, int E, int k,
                                                           int n_chunks, const int32_t* __restrict__ chunk_base,
                                                           const int32_t* __restrict__ offsets,
                                                           const int32_t* __restrict__ offsets_pad,
                                                           int32_t* __restrict__ sorted_token,
                                                           int32_t* __restrict__ inv_row,
                                                           int32_t* __restrict__ inv_int, uint32_t* status) {
    extern __shared__ int32_t run_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x * 4 + warp;
    pdl_trigger();
    pdl_wait();
    if (c >= n_chunks) return;
    scatter_chunk(ids, T, E, k, c, chunk_base, offsets, offsets_pad, sorted_token, inv_row, inv_int, status,
                  run_smem + warp * E, lane);
}

// ---------------------------------------------------------------------------
// Routing of a decode batch (T <= CHUNK_TOK, E <= 512) in one CTA: top-k and
// gate weights (the device function of the multi-CTA top-k kernel), then the
// grouping with the ids, counts and offsets held in shared memory.  Rows
// inside an expert ascend with the pair index (token-major), as in the
// multi-CTA grouping, so the results are identical to it.
// ---------------------------------------------------------------------------
constexpr int SMALL_THREADS = 512;
constexpr int SMALL_PAIRS = CHUNK_TOK * MAX_TOPK;

template <int PER>
__global__ void __launch_bounds__(SMALL_THREADS) route_small_kernel(
    const float* __restrict__ part, int ksplit, const float* __restrict__ bias, int T, int E, int k, int n_shared,
    int bn, float* __restrict__ logits_out, int32_t* __restrict__ ids, float* __restrict__ wout,
    int32_t* __restrict__ offsets, int32_t* __restrict__ offsets_pad, int32_t* __restrict__ offsets_out,
    GroupTable* gt, int32_t* __restrict__ sorted_token, int32_t* __restrict__ inv_row, int32_t* __restrict__ inv_int,
    uint32_t* status) {
    __shared__ float sel_v[SMALL_THREADS / 32][MAX_TOPK];
    __shared__ int sel_i[SMALL_THREADS / 32][MAX_TOPK];
    __shared__ int32_t s_ids[SMALL_PAIRS];
    __shared__ int32_t cnt[512], s_off[512], s_pad[512];
    __shared__ float s_bias[512];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    // the router bias is a layer constant: fetched before the wait, off the critical path
    for (int e = threadIdx.x; e < E; e += SMALL_THREADS) {
        cnt[e] = 0;
        if (bias) s_bias[e] = bias[e];
    }
    __syncthreads();
    pdl_wait();
    for (int t = warp; t < T; t += SMALL_THREADS / 32) {
        topk_token<PER>(part, ksplit, bias ? s_bias : nullptr, T, E, k, logits_out, ids, wout, t, lane, sel_v[warp],
                        sel_i[warp]);
        if (lane < k) s_ids[t * k + lane] = sel_i[warp][lane];
    }
    __syncthreads();
    const int n = T * k;
    for (int i = threadIdx.x; i < n; i += SMALL_THREADS) {
        const int e = clamp_expert(s_ids[i], E, status);
        s_ids[i] = e;
        atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    {
        const int e = threadIdx.x;
        int off, poff;
        scan_counts(e < E ? cnt[e] : 0, T, E, n_shared, bn, offsets, offsets_pad, offsets_out, gt, &off, &poff);
        if (e < E) {
            s_off[e] = off;
            s_pad[e] = poff;
            cnt[e] = 0;                        // reused as the running count per expert
        }
    }
    __syncthreads();
    if (warp == 0) {
        // stable ranks: 32 pairs at a time in pair order, equal experts ranked by a warp match
        const uint32_t lt_mask = (1u << lane) - 1u;
        for (int b0 = 0; b0 < n; b0 += 32) {
            const int i = b0 + lane;
            const bool valid = i < n;
            const int e = valid ? s_ids[i] : -1 - lane;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
            const int rank = __popc(peers & lt_mask);
            if (valid) {
                const int r = cnt[e] + rank;
                const int row = s_off[e] + r;
                if (sorted_token) sorted_token[row] = i / k;
                inv_row[i] = row;
                inv_int[i] = s_pad[e] + r;
            }
            __syncwarp();
            if (valid && (peers & lt_mask) == 0) cnt[e] += __popc(peers);
            __syncwarp();
        }
    }
}

cudaError_t launch_route_small(const moe_layer* L, const float* part, int ksplit, bool add_bias, int T,
                               float* logits_out, int32_t* ids, float* w, const WsLayout& lay, char* ws, int bn,
                               int32_t* offsets_out, int32_t* sorted_out, int32_t* inv_out, cudaStream_t s) {
    const int E = L->d.n_experts, k = L->d.top_k;
    int32_t* inv_row = reinterpret_cast<int32_t*>(ws + lay.inv_row);
    const int per = (E + 31) / 32;
#define MOE_SMALL_CASE(P)                                                                                         \
    if (per <= P) {                                                                                               \
        err = launch_pdl(route_small_kernel<P>, dim3(1), dim3(SMALL_THREADS), 0, s,                               \
            part, ksplit, add_bias ? L->router_b : nullptr, T, E, k, L->d.n_shared, bn, logits_out, ids, w,       \
            reinterpret_cast<int32_t*>(ws + lay.offsets), reinterpret_cast<int32_t*>(ws + lay.offsets_pad),       \
            offsets_out, reinterpret_cast<GroupTable*>(ws + lay.table), sorted_out, inv_row,                      \
            reinterpret_cast<int32_t*>(ws + lay.inv_int), L->dev_status);                                         \
    } else
    cudaError_t err = cudaSuccess;
    MOE_SMALL_CASE(1) MOE_SMALL_CASE(2) MOE_SMALL_CASE(4) MOE_SMALL_CASE(8) MOE_SMALL_CASE(12) MOE_SMALL_CASE(16)
    return cudaErrorInvalidValue;
#undef MOE_SMALL_CASE
    if (err == cudaSuccess && inv_out)
        err = cudaMemcpyAsync(inv_out, inv_row, sizeof(int32_t) * (size_t)T * k, cudaMemcpyDeviceToDevice, s);
    return err;
}

cudaError_t launch_permute(const moe_layer* L, const int32_t* ids, int T, const WsLayout& lay, char* ws, int bn,
                           int32_t* offsets_out, int32_t* sorted_out, int32_t* inv_out, cudaStream_t s) {
    const int E = L->d.n_experts, k = L->d.top_k;
    int32_t* chunk_cnt = reinterpret_cast<int32_t*>(ws + lay.chunk_cnt);
    int32_t* chunk_base = reinterpret_cast<int32_t*>(ws + lay.chunk_base);
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + lay.offsets);
    int32_t* offsets_pad = reinterpret_cast<int32_t*>(ws + lay.offsets_pad);
    int32_t* sorted_token = sorted_out;   // only the caller needs it
    int32_t* inv_row = reinterpret_cast<int32_t*>(ws + lay.inv_row);
    int32_t* inv_int = reinterpret_cast<int32_t*>(ws + lay.inv_int);
    GroupTable* gt = reinterpret_cast<GroupTable*>(ws + lay.table);
    const int nc = lay.n_chunks;
    const size_t smem = 4 * E * sizeof(int32_t);
    if (nc > 0) {
        cudaError_t err = launch_pdl(perm_count_kernel, dim3((nc + 3) / 4), dim3(128), smem, s, ids, T, E, k, nc,
                                     chunk_cnt, L->dev_status);
        if (err != cudaSuccess) return err;
    }
    cudaError_t err = launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, s, chunk_cnt, nc, T, E, k, L->d.n_shared,
                                 bn, chunk_base, offsets, offsets_pad, offsets_out, gt);
    if (err != cudaSuccess) return err;
    if (nc > 0) {
        err = launch_pdl(perm_scatter_kernel, dim3((nc + 3) / 4), dim3(128), smem, s, ids, T, E, k, nc, chunk_base,
                         offsets, offsets_pad, sorted_token, inv_row, inv_int, L->dev_status);
        if (err != cudaSuccess) return err;
        if (inv_out)
            err = cudaMemcpyAsync(inv_out, inv_row, sizeof(int32_t) * (size_t)T * k, cudaMemcpyDeviceToDevice, s);
    }
    return err;
}

// ---------------------------------------------------------------------------
// 1x128 quantisation of x, written to every row the token owns.
// Per token t and 128-channel group g: amax = max |x|; s = amax / 448
// (s = 1 if amax = 0); q = E4M3FN(fp32(x / s)) rounded to nearest even with
// saturation.  Destination rows (internal, 8-aligned groups): inv_int[t][j]
// for the routed groups and shared_row0 + t for the shared group; the codes
// go to the swizzled K-block-major layout (see act_offset) and the scales
// to sxT[g][row], so one tile of rows is one contiguous run of both.  CTA
// (token, blockIdx.y) quantises groups 32 blockIdx.y .. +31, warp w the
// groups w, w + 8, w + 16, w + 24 of them (loads issued together), 4
// channels per lane.
// ---------------------------------------------------------------------------
constexpr int QUANT_GPW = 4;    // 128-channel groups per warp (loads in flight per lane)

__global__ void __launch_bounds__(256) quant_scatter_kernel(const uint16_t* __restrict__ x, int T, int H, int k,
                                                            int n_shared, const int32_t* __restrict__ inv_int,
                                                            const int32_t* __restrict__ offsets_pad, int E,
                                                            uint8_t* __restrict__ xp, float* __restrict__ sxT,
                                                            int ld, uint8_t* __restrict__ xq_out,
                                                            float* __restrict__ sx_out, uint32_t* status) {
    __shared__ int dest[MAX_TOPK + 1];
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    // x is read and quantised before the wait: this kernel is launched only after the router
    // kernel has passed its own wait, so the layer input is complete; only the destination rows
    // come from the routing
    const int G = H / QB;
    uint32_t qv[QUANT_GPW];
    float scv[QUANT_GPW];
    {
        uint2 raws[QUANT_GPW];
#pragma unroll
        for (int i = 0; i < QUANT_GPW; ++i) {
            const int g = blockIdx.y * 8 * QUANT_GPW + warp + 8 * i;
            raws[i] = g < G ? *reinterpret_cast<const uint2*>(x + (size_t)t * H + g * QB + lane * 4) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < QUANT_GPW; ++i) {
            const uint2 raw = raws[i];
            const float v0 = __uint_as_float(raw.x << 16), v1 = __uint_as_float(raw.x & 0xFFFF0000u);
            const float v2 = __uint_as_float(raw.y << 16), v3 = __uint_as_float(raw.y & 0xFFFF0000u);
            float am = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, off));
            const float sc = (am > 0.f) ? __fdiv_rn(am, 448.0f) : 1.0f;
            scv[i] = sc;
            qv[i] = pack4_e4m3(__fdiv_rn(v0, sc), __fdiv_rn(v1, sc), __fdiv_rn(v2, sc), __fdiv_rn(v3, sc));
        }
    }
    pdl_wait();
    const int nd = k + (n_shared ? 1 : 0);
    if (threadIdx.x < k) {
        // a row outside the permuted buffers is flagged and skipped, never written
        const int row = inv_int[(size_t)t * k + threadIdx.x];
        const bool ok = row >= 0 && row < ld;
        if (!ok && blockIdx.y == 0) atomicOr(status, MOE_DEV_BAD_ROW);
        dest[threadIdx.x] = ok ? row : -1;
    }
    if (threadIdx.x == 0 && n_shared) dest[k] = offsets_pad[E] + t;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < QUANT_GPW; ++i) {
        const int g = blockIdx.y * 8 * QUANT_GPW + warp + 8 * i;
        if (g >= G) break;
        const uint32_t q = qv[i];
        const float sc = scv[i];
        for (int d = 0; d < nd; ++d) {
            const int row = dest[d];
            if (row < 0) continue;
            const int chunk = (lane >> 2) ^ (row & 7);
            *reinterpret_cast<uint32_t*>(xp + act_offset(g, row, ld) + chunk * 16 + (lane & 3) * 4) = q;
            if (lane == 0) sxT[(size_t)g * ld + row] = sc;
        }
        if (xq_out) *reinterpret_cast<uint32_t*>(xq_out + (size_t)t * H + g * QB + lane * 4) = q;
        if (sx_out && lane == 0) sx_out[(size_t)t * G + g] = sc;
    }
}

cudaError_t launch_quant_scatter(const moe_layer* L, const uint16_t* x, int T, const WsLayout& lay, char* ws,
                                 uint8_t* xq_out, float* sx_out, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    // one warp per 128-channel group, QUANT_GPW groups per warp: grid.y covers the groups 8 * QUANT_GPW at a time
    const dim3 grid(T, (L->d.hidden / QB + 8 * QUANT_GPW - 1) / (8 * QUANT_GPW));
    return launch_pdl(quant_scatter_kernel, grid, dim3(256), 0, s, x, T, L->d.hidden, L->d.top_k, L->d.n_shared,
                                           reinterpret_cast<const int32_t*>(ws + lay.inv_int),
                                           reinterpret_cast<const int32_t*>(ws + lay.offsets_pad), L->d.n_experts,
                                           reinterpret_cast<uint8_t*>(ws + lay.xp),
                                           reinterpret_cast<float*>(ws + lay.sxT), lay.rows_pad, xq_out, sx_out,
                                           L->dev_status);
}

}  // namespace moe
