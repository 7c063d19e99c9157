// Router logits for prefill batches on the 5th-generation tensor cores
// (tcgen05, sm_103a): L = x W_r^T in fp32, the gating GEMM that precedes
// dispatch (KTransformers deep dive, section 1.2; CPU-GPU hybrid inference
// article, SmallEP section: gating and sorting come first).
//
// Exactness.  x is bf16, so it is an exact bf16 MMA operand.  Each fp32
// router weight is split once, at load time, into three bf16 terms
// w = w1 + w2 + w3 (w1 = bf16(w), w2 = bf16(w - w1), w3 = bf16(w - w1 - w2);
// each remainder is exact in fp32, and 3 x 8 significant bits cover the 24 of
// fp32).  Every product x * w_j is exact in fp32, but the tensor core's
// fp32 accumulation truncates: a long-lived accumulator, whose sign rarely
// changes, collects that bias linearly (measured: ~1e-5 on N(0,1) logits).
// So every 64-channel k step goes into a fresh TMEM accumulator (12 MMAs,
// partial sums ~0.1), and the epilogue warps add the k-step partials into
// fp32 registers in k order with IEEE adds; the truncation errors of
// independent steps then average out.  The K range is split over grid.z and
// the top-k kernel adds the splits in order.
//
// Tile: 128 tokens (TMEM lanes) x 64 experts, 64 channels per stage.  Both
// operands arrive by TMA (cp.async.bulk.tensor) with 128-byte swizzle, rows
// past T or E are zero-filled by the copy.  Warp 4 issues the copies, warp 5
// the MMAs (kind::f16, bf16 x bf16 -> f32, M128 N64 K16) into four rotating
// accumulators, and warps 0-3 (one TMEM lane quarter each) drain them.  Two
// CTAs fit on an SM (80 KB of shared memory and 256 TMEM columns each).
#include <cuda.h>
#include <mutex>

#include "moe_internal.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace rt {

constexpr int BM = 128;                  // tokens per tile
constexpr int BN = 64;                   // experts per tile
constexpr int BK = 64;                   // channels per k step (128 bytes of bf16)
constexpr int NTERM = 3;                 // bf16 terms of each fp32 router weight
constexpr int NACC = 4;                  // rotating accumulators
constexpr int STAGES = 2;
constexpr int A_BYTES = BM * BK * 2;     // 16 KB
constexpr int B_BYTES = BN * BK * 2;     // 8 KB per term
constexpr int STAGE = A_BYTES + NTERM * B_BYTES;
constexpr int SMEM = STAGES * STAGE + 1024;
constexpr uint32_t TMEM_COLS = NACC * BN;   // 256

// Instruction descriptor, kind::f16: D f32, A = B = bf16, both K-major, M = 128, N = 64.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

// part[z][t][e] = sum over the channels of split z of x[t][h] * W_r[e][h]
constexpr int NTHREADS = 192;

__global__ void __launch_bounds__(NTHREADS) router_tc_kernel(const __grid_constant__ CUtensorMap tx,
                                                        const __grid_constant__ CUtensorMap tw, int T, int E,
                                                        int ksteps, float* __restrict__ part, uint32_t* status,
                                                        uint32_t wait_limit) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[STAGES], empty[STAGES], tfull[NACC], tempty[NACC], mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * BN, t0 = blockIdx.y * BM, z = blockIdx.z;
    pdl_wait();                                   // x may come from the preceding kernel
    const int kx0 = z * ksteps * BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int a = 0; a < NACC; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], 4); }
        mbar_init(&mma_done, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 0) tc::tmem_alloc(&tmem_slot, TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int* abort = &abort_flag;

    if (warp == 4 && lane == 0) {
        // ------------------------------------------------------------ producer
        int issued = 0;
        for (int s = 0; s < ksteps; ++s) {
            const int st = s % STAGES;
            const uint32_t ph = (uint32_t)(s / STAGES) & 1u;
            if (!mbar_wait_bounded(&empty[st], ph ^ 1u, wait_limit, status, abort)) break;
            uint8_t* buf = smem + st * STAGE;
            mbar_arrive_expect_tx(&full[st], STAGE);
            const int kx = kx0 + s * BK;
            tma_load_2d(buf, &tx, kx, t0, &full[st]);
#pragma unroll
            for (int j = 0; j < NTERM; ++j) tma_load_3d(buf + A_BYTES + j * B_BYTES, &tw, kx, e0, j, &full[st]);
            ++issued;
        }
        // every issued copy must land before the CTA exits
        for (int s = max(0, issued - STAGES); s < issued; ++s)
            mbar_wait_bounded(&full[s % STAGES], (uint32_t)(s / STAGES) & 1u, wait_limit, status, nullptr);
    } else if (warp == 5 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        int issued = 0;
        for (int s = 0; s < ksteps; ++s) {
            const int st = s % STAGES, a = s % NACC;
            if (!mbar_wait_bounded(&tempty[a], ((uint32_t)(s / NACC) & 1u) ^ 1u, wait_limit, status, abort) ||
                !mbar_wait_bounded(&full[st], (uint32_t)(s / STAGES) & 1u, wait_limit, status, abort))
                break;
            tc::tc_fence_after();
            const uint32_t base = smem_addr(smem + st * STAGE);
            const uint64_t adesc = tc::sw128_desc(base);
            const uint32_t dt = tmem + (uint32_t)(a * BN);
#pragma unroll
            for (int j = 0; j < NTERM; ++j) {
                const uint64_t bdesc = tc::sw128_desc(base + A_BYTES + j * B_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    tc::mma_f16(dt, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (j == 0 && kk == 0) ? 0u : 1u);
            }
            tc::mma_commit(&empty[st]);
            tc::mma_commit(&tfull[a]);
            ++issued;
        }
        // every issued MMA must complete before the tensor memory is released
        if (issued) {
            tc::mma_commit(&mma_done);
            mbar_wait_bounded(&mma_done, 0u, wait_limit, status, nullptr);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue warps 0-3
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        float v[BN];
#pragma unroll
        for (int c = 0; c < BN; ++c) v[c] = 0.f;
        bool ok = true;
        for (int s = 0; s < ksteps; ++s) {
            const int a = s % NACC;
            if (ok && !mbar_wait_bounded(&tfull[a], (uint32_t)(s / NACC) & 1u, wait_limit, status, abort)) ok = false;
            ok = __all_sync(0xFFFFFFFFu, ok);          // tcgen05.ld below is warp-collective
            if (ok) {
                tc::tc_fence_after();
                uint32_t p0[32], p1[32];
                tc::tmem_ld32u(tl + (uint32_t)(a * BN), p0);
                tc::tmem_ld32u(tl + (uint32_t)(a * BN + 32), p1);
                tc::tmem_wait_ld();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[a]);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    v[c] = __fadd_rn(v[c], __uint_as_float(p0[c]));
                    v[32 + c] = __fadd_rn(v[32 + c], __uint_as_float(p1[c]));
                }
            }
        }
        const bool ready = ok;
        const int t = t0 + warp * 32 + lane;
        if (ready && t < T) {
            float* dst = part + ((size_t)z * T + t) * E + e0;
            if (e0 + BN <= E && (E & 3) == 0) {
#pragma unroll
                for (int c = 0; c < BN; c += 4) *reinterpret_cast<float4*>(dst + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (e0 + c < E) dst[c] = v[c];
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// w -> three bf16 terms, [3][E][H].
__global__ void split_router_weights_kernel(const float* __restrict__ w, size_t n, uint16_t* __restrict__ out) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float v = w[i];
        const __nv_bfloat16 b1 = __float2bfloat16_rn(v);
        const float r1 = __fsub_rn(v, __bfloat162float(b1));
        const __nv_bfloat16 b2 = __float2bfloat16_rn(r1);
        const float r2 = __fsub_rn(r1, __bfloat162float(b2));
        const __nv_bfloat16 b3 = __float2bfloat16_rn(r2);
        out[i] = __bfloat16_as_ushort(b1);
        out[n + i] = __bfloat16_as_ushort(b2);
        out[2 * n + i] = __bfloat16_as_ushort(b3);
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no
// link-time dependency on the driver library).
EncodeTiled encoder() {
    static std::once_flag once;
    static EncodeTiled fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

}  // namespace rt

size_t router_split_bytes(const moe_layer* L) { return (size_t)rt::NTERM * L->d.n_experts * L->d.hidden * 2; }

cudaError_t launch_split_router_weights(const moe_layer* L, cudaStream_t s) {
    const size_t n = (size_t)L->d.n_experts * L->d.hidden;
    rt::split_router_weights_kernel<<<4 * L->num_sms, 256, 0, s>>>(L->router_w, n, L->router_w3);
    return cudaGetLastError();
}

// K splits for a prefill batch: the smallest divisor d of H/64 that gives at
// least 4 CTAs per SM, keeping >= 4 k steps per CTA.
int router_tc_splits(int T, int H, int E, int num_sms) {
    const int kt = H / rt::BK;
    const int tiles = ((T + rt::BM - 1) / rt::BM) * ((E + rt::BN - 1) / rt::BN);
    int best = 1;
    for (int d = 1; d <= kt; ++d) {
        if (kt % d) continue;
        if (kt / d < rt::NACC) break;
        best = d;
        if (tiles * d >= 4 * num_sms) break;
    }
    return best;
}

cudaError_t launch_router_tc(const moe_layer* L, const uint16_t* x, int T, float* part, int ksplit, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int H = L->d.hidden, E = L->d.n_experts;
    rt::EncodeTiled enc = rt::encoder();
    if (!enc) return cudaErrorNotSupported;
    {
        cudaError_t e = ensure_smem_limit<rt::router_tc_kernel>(rt::SMEM);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tx, tw;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
        const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
        const cuuint32_t box[2] = {rt::BK, rt::BM};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)E, (cuuint64_t)rt::NTERM};
        const cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)E * H * 2};
        const cuuint32_t box[3] = {rt::BK, rt::BN, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, L->router_w3, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int ksteps = H / rt::BK / ksplit;
    dim3 grid((E + rt::BN - 1) / rt::BN, (T + rt::BM - 1) / rt::BM, ksplit);
    return launch_pdl(rt::router_tc_kernel, grid, dim3(rt::NTHREADS), rt::SMEM, s, tx, tw, T, E, ksteps, part,
                      L->dev_status, L->wait_limit);
}

}  // namespace moe
