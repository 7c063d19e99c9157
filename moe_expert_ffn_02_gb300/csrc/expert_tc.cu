// Grouped FP8 expert GEMMs for prefill on the 5th-generation tensor cores
// (tcgen05, sm_103a).
//
// Swap-AB tiles: A = 128 rows of an expert's weight matrix (output
// features), B = 128 token rows of the expert's group, K = 128 per stage.
// Both operands are 16 KB 128-byte-swizzled K-major images in global memory
// (weight tiles repacked at load time; activation tiles written so by the
// quantiser / gate-up epilogue), so the producer warp moves each with one
// bulk copy.  One thread of the MMA warp issues tcgen05.mma kind::f8f6f4
// (E4M3 x E4M3, fp32 accumulate in tensor memory) -- 4 instructions of
// K = 32 per stage, two accumulators (gate, up) in the gate/up kernel --
// and commits to mbarriers.  Accumulators are double-buffered in TMEM so
// the tensor core works on block kb+1 while the epilogue warps promote
// block kb.
//
// Scale promotion (FP8 GEMV section of the CPU-GPU hybrid inference
// article, Fig. 9-10: block partial sums are scaled once per 128-element
// block): every K block's partial D_kb is read out of TMEM (tcgen05.ld) and
// added as acc += D_kb * s_w[kb] * s_x[token][kb] in fp32 registers.
//
// Unit = (group, m tile, n tile), n fastest, so the n tiles of one weight
// row block run on neighbouring CTAs and share its bytes through L2.
#include "moe_internal.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;                 // weight rows per tile (TMEM lanes)
constexpr int BN = 128;                 // tokens per tile (TMEM columns per accumulator)
constexpr int EPI_WARPS = 8;            // 4 lane quarters x 2 column halves
constexpr int COLS = BN / 2;            // columns per epilogue thread
constexpr int NTHREADS = (2 + EPI_WARPS) * 32;
constexpr uint32_t TMEM_COLS = 512;

template <bool GU>
struct Cfg {
    static constexpr int W_BYTES = GU ? 2 * TILE_BYTES : TILE_BYTES;
    static constexpr int X_BYTES = BN * 128;
    static constexpr int STAGE = W_BYTES + X_BYTES;
    static constexpr int STAGES = GU ? 4 : 6;
    static constexpr int NACC = GU ? 2 : 1;
    static constexpr int BUF_COLS = NACC * BN;          // TMEM columns per buffer
    static constexpr int SCALE_BYTES = EPI_WARPS * 2 * NACC * COLS * 4;
    static constexpr int STAGING = GU ? BN * 144 + 2 * 4 * COLS * 4 : 0;
    static constexpr int SMEM = STAGES * STAGE + SCALE_BYTES + STAGING + 256;
};

struct Args {
    const uint8_t* w;         // tile images of all groups
    const float* wscale;      // [group][m tile][k tile] (x2 gate/up)
    const uint8_t* act;       // [K/128][rows_pad][128] swizzled E4M3
    const float* actsT;       // [K/128][rows_pad]
    int ld;                   // rows_pad
    int K, M;
    const GroupTable* gt;
    uint8_t* hq;              // gate/up output codes (same layout as act)
    float* shT;               // gate/up output scales
    float* out;               // down: [rows_pad][M] fp32
    uint32_t* status;
    uint32_t wait_limit;
};

struct Unit {
    int expert, mb, row_begin, valid;
};

// u -> (group, m tile, n tile) with n fastest inside a group.
__device__ __forceinline__ Unit decode_unit(const GroupTable* gt, int u, int MT) {
    int lo = 0, hi = gt->n_groups - 1;            // last group with MT * pair_start <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (gt->pair_start[mid] * MT <= u) lo = mid; else hi = mid - 1;
    }
    const int nt_g = gt->pair_start[lo + 1] - gt->pair_start[lo];
    const int local = u - gt->pair_start[lo] * MT;
    const int mb = local / nt_g, nt = local - mb * nt_g;
    Unit r;
    r.expert = gt->expert[lo];
    r.mb = mb;
    r.row_begin = gt->row0[lo] + nt * BN;
    r.valid = min(BN, gt->rows[lo] - nt * BN);
    return r;
}

// ------------------------------------------------------------------ tcgen05 PTX
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms
// 1024 B apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                 // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
    d |= (uint64_t)1 << 46;                 // version
    d |= (uint64_t)2 << 61;                 // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f8f6f4: D f32, A = B = E4M3, both K-major.
constexpr uint32_t IDESC = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(IDESC), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// 32 lanes x 32 columns of fp32 (one register per column per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

// ------------------------------------------------------------------ kernel
template <bool GU>
__global__ void __launch_bounds__(NTHREADS, 1) expert_tc_kernel(Args a) {
    using C = Cfg<GU>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    float* scl = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE);           // [EPI_WARPS][2][NACC][COLS]
    uint8_t* staging = smem + C::STAGES * C::STAGE + C::SCALE_BYTES;               // gate/up: codes + amax
    __shared__ uint64_t full[C::STAGES], empty[C::STAGES], tfull[2], tempty[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int MT = a.M / QB, KT = a.K / QB;
    const GroupTable* gt = a.gt;
    const int n_units = gt->n_pairs * MT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(&tfull[b], 1); mbar_init(&tempty[b], EPI_WARPS); }
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 1) tmem_alloc(&tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int* abort = &abort_flag;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit un = decode_unit(gt, u, MT);
                const uint8_t* wbase = a.w + ((size_t)(un.expert * MT + un.mb) * KT) * C::W_BYTES;
                for (int kb = 0; kb < KT; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, a.wait_limit, a.status, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = stages + stage * C::STAGE;
                    mbar_arrive_expect_tx(&full[stage], C::STAGE);
                    bulk_g2s(st, wbase + (size_t)kb * C::W_BYTES, C::W_BYTES, &full[stage]);
                    bulk_g2s(st + C::W_BYTES, a.act + act_offset(kb, un.row_begin, a.ld), C::X_BYTES, &full[stage]);
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            for (int s = 0; s < C::STAGES; ++s)
                if ((armed >> s) & 1u) mbar_wait_bounded(&full[s], (armed_par >> s) & 1u, a.wait_limit, a.status, nullptr);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, buf = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                for (int kb = 0; kb < KT; ++kb) {
                    if (!mbar_wait_bounded(&tempty[buf], tphase ^ 1u, a.wait_limit, a.status, abort) ||
                        !mbar_wait_bounded(&full[stage], phase, a.wait_limit, a.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sW = smem_addr(stages + stage * C::STAGE);
                    const uint32_t sX = sW + C::W_BYTES;
                    const uint32_t d0 = tmem + (uint32_t)(buf * C::BUF_COLS);
#pragma unroll
                    for (int k = 0; k < QB / 32; ++k) {
                        const uint64_t bdesc = sw128_desc(sX + k * 32);
                        mma_f8(d0, sw128_desc(sW + k * 32), bdesc, k > 0);
                        if (GU) mma_f8(d0 + BN, sw128_desc(sW + TILE_BYTES + k * 32), bdesc, k > 0);
                    }
                    mma_commit(&empty[stage]);
                    mma_commit(&tfull[buf]);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                    if (++buf == 2) { buf = 0; tphase ^= 1u; }
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int ew = warp - 2;                  // 0..7
        const int quarter = warp & 3;             // TMEM lanes this warp may read
        const int half = ew >> 2;                 // column half
        const int row = quarter * 32 + lane;      // output feature within the tile
        float* my_scl = scl + ew * (2 * C::NACC * COLS);
        int buf = 0;
        uint32_t tphase = 0;
        bool dead = false;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
            const Unit un = decode_unit(gt, u, MT);
            const float* wsc = a.wscale + ((size_t)(un.expert * MT + un.mb) * KT) * C::NACC;
            float acc[C::NACC][COLS];
#pragma unroll
            for (int j = 0; j < C::NACC; ++j)
#pragma unroll
                for (int c = 0; c < COLS; ++c) acc[j][c] = 0.f;
            // prefetch the activation scales of block 0 for this lane's two columns
            const int col0 = half * COLS + lane, col1 = col0 + 32;
            float sx0 = (col0 < un.valid) ? __ldg(a.actsT + un.row_begin + col0) : 0.f;
            float sx1 = (col1 < un.valid) ? __ldg(a.actsT + un.row_begin + col1) : 0.f;
            for (int kb = 0; kb < KT; ++kb) {
                // combined scale per column: s_w[kb] * s_x[col][kb]
                float* cs = my_scl + (kb & 1) * (C::NACC * COLS);
#pragma unroll
                for (int j = 0; j < C::NACC; ++j) {
                    const float sw = __ldg(wsc + (size_t)kb * C::NACC + j);
                    cs[j * COLS + lane] = sw * sx0;
                    cs[j * COLS + lane + 32] = sw * sx1;
                }
                if (kb + 1 < KT) {
                    sx0 = (col0 < un.valid) ? __ldg(a.actsT + (size_t)(kb + 1) * a.ld + un.row_begin + col0) : 0.f;
                    sx1 = (col1 < un.valid) ? __ldg(a.actsT + (size_t)(kb + 1) * a.ld + un.row_begin + col1) : 0.f;
                }
                __syncwarp();
                if (!dead && !mbar_wait_bounded(&tfull[buf], tphase, a.wait_limit, a.status, abort)) dead = true;
                if (!dead) {
                    tc_fence_after();
                    const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * C::BUF_COLS) +
                                           (uint32_t)(half * COLS);
#pragma unroll
                    for (int j = 0; j < C::NACC; ++j) {
#pragma unroll
                        for (int ch = 0; ch < COLS / 32; ++ch) {
                            float p[32];
                            tmem_ld32(tbase + (uint32_t)(j * BN + ch * 32), p);
                            tmem_wait_ld();
#pragma unroll
                            for (int c4 = 0; c4 < 8; ++c4) {
                                const float4 s4 = *reinterpret_cast<const float4*>(cs + j * COLS + ch * 32 + c4 * 4);
                                acc[j][ch * 32 + c4 * 4 + 0] = __fmaf_rn(p[c4 * 4 + 0], s4.x, acc[j][ch * 32 + c4 * 4 + 0]);
                                acc[j][ch * 32 + c4 * 4 + 1] = __fmaf_rn(p[c4 * 4 + 1], s4.y, acc[j][ch * 32 + c4 * 4 + 1]);
                                acc[j][ch * 32 + c4 * 4 + 2] = __fmaf_rn(p[c4 * 4 + 2], s4.z, acc[j][ch * 32 + c4 * 4 + 2]);
                                acc[j][ch * 32 + c4 * 4 + 3] = __fmaf_rn(p[c4 * 4 + 3], s4.w, acc[j][ch * 32 + c4 * 4 + 3]);
                            }
                        }
                    }
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
                if (++buf == 2) { buf = 0; tphase ^= 1u; }
            }

            if (GU) {
                // -------------------------------------- SiLU(g)*u and 1x128 E4M3 quantisation of h
                uint8_t* qst = staging;                                         // [BN][144]
                float* amax_s = reinterpret_cast<float*>(staging + BN * 144);   // [2 halves][4 quarters][COLS]
                float* h = acc[0];
#pragma unroll
                for (int c = 0; c < COLS; ++c) h[c] = silu_mul(acc[0][c], acc[GU ? 1 : 0][c]);
#pragma unroll
                for (int c = 0; c < COLS; ++c) {
                    float m = fabsf(h[c]);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
                    if (lane == 0) amax_s[(half * 4 + quarter) * COLS + c] = m;
                }
                named_bar_sync(1, EPI_WARPS * 32);
#pragma unroll
                for (int c = 0; c < COLS; ++c) {
                    const float* am = amax_s + half * 4 * COLS + c;
                    const float mx = fmaxf(fmaxf(am[0], am[COLS]), fmaxf(am[2 * COLS], am[3 * COLS]));
                    const float sc = (mx > 0.f) ? __fdiv_rn(mx, 448.0f) : 1.0f;
                    const uint16_t q2 = f32x2_to_e4m3x2(__fdiv_rn(h[c], sc), 0.f);
                    qst[(half * COLS + c) * 144 + row] = (uint8_t)(q2 & 0xFF);
                    if (quarter == 0 && lane == 0 && half * COLS + c < un.valid)
                        a.shT[(size_t)un.mb * a.ld + un.row_begin + half * COLS + c] = sc;
                }
                named_bar_sync(1, EPI_WARPS * 32);
                const int tid = threadIdx.x - 64;
                for (int rr = tid >> 3; rr < un.valid; rr += (EPI_WARPS * 32) >> 3) {
                    const uint4 v = lds128(qst + rr * 144 + (tid & 7) * 16);
                    const int pos = (tid & 7) ^ (rr & 7);
                    *reinterpret_cast<uint4*>(a.hq + act_offset(un.mb, un.row_begin + rr, a.ld) + pos * 16) = v;
                }
                named_bar_sync(1, EPI_WARPS * 32);
            } else {
                // -------------------------------------- fp32 expert output rows
                const int cbeg = half * COLS;
#pragma unroll
                for (int c = 0; c < COLS; ++c)
                    if (cbeg + c < un.valid)
                        a.out[(size_t)(un.row_begin + cbeg + c) * a.M + un.mb * QB + row] = acc[0][c];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

template <bool GU>
static cudaError_t launch(const moe_layer* L, const WsLayout& lay, char* ws, cudaStream_t s) {
    using C = Cfg<GU>;
    static bool attr[2] = {false, false};
    if (!attr[GU]) {
        cudaError_t e = cudaFuncSetAttribute(expert_tc_kernel<GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM + 1024);
        if (e != cudaSuccess) return e;
        attr[GU] = true;
    }
    Args a;
    const int H = L->d.hidden, I = L->d.inter;
    a.gt = reinterpret_cast<const GroupTable*>(ws + lay.table);
    a.ld = lay.rows_pad;
    a.status = L->dev_status;
    a.wait_limit = L->wait_limit;
    a.hq = reinterpret_cast<uint8_t*>(ws + lay.hq);
    a.shT = reinterpret_cast<float*>(ws + lay.shT);
    a.out = reinterpret_cast<float*>(ws + lay.o);
    if (GU) {
        a.w = L->w_gu; a.wscale = L->s_gu;
        a.act = reinterpret_cast<const uint8_t*>(ws + lay.xp);
        a.actsT = reinterpret_cast<const float*>(ws + lay.sxT);
        a.K = H; a.M = I;
    } else {
        a.w = L->w_dn; a.wscale = L->s_dn;
        a.act = reinterpret_cast<const uint8_t*>(ws + lay.hq);
        a.actsT = reinterpret_cast<const float*>(ws + lay.shT);
        a.K = I; a.M = H;
    }
    expert_tc_kernel<GU><<<L->num_sms, NTHREADS, C::SMEM + 1024, s>>>(a);
    return cudaGetLastError();
}

}  // namespace tc

int tc_tile_n() { return tc::BN; }

cudaError_t launch_expert_tc_gate_up(const moe_layer* L, int T, const WsLayout& lay, char* ws, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return tc::launch<true>(L, lay, ws, s);
}

cudaError_t launch_expert_tc_down(const moe_layer* L, int T, const WsLayout& lay, char* ws, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return tc::launch<false>(L, lay, ws, s);
}

}  // namespace moe
