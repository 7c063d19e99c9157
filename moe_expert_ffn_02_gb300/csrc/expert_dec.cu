// Grouped FP8 expert GEMMs for decode batches on the 5th-generation tensor
// cores (sm_103a): tcgen05 MMAs with the weights as the 128-row operand and
// the unit's few token rows as the narrow one.
//
// Decode batches give every expert a handful of tokens, so a unit is
// (group, token tile of <= 16 rows, weight block) as in the prefill kernel,
// but the roles of the operands are swapped: D[weight row][token] =
// W[128 rows x 128 K] * X[16 tokens x 128 K]^T.  A group with more tokens
// (the shared expert of a larger batch) has several tiles, whose units read
// the same weight blocks at about the same time, mostly from L2.  The layer streams its touched experts' weights once
// from HBM; the tensor core work per 32 KB stage is eight small MMAs issued
// by one thread, so the stream, not the arithmetic, sets the pace.
//
// Per 128-wide K block (the block of the 128x128 weight scales and of the
// 1x128 activation scales) the MMAs start a fresh accumulator in a TMEM
// buffer; the epilogue warps (one weight row per thread) read the block's
// N columns back, multiply by s_w[block] * s_x[token][block] and add to
// fp32 registers -- the post-scaling order of the FP8 GEMV section of the
// CPU-GPU hybrid inference article (xingyun.xin, Fig. 9-10).  Gate/up: the
// gate and up tiles of the same 128 inner features go to two column ranges
// of one buffer, and the unit's epilogue forms h = SiLU(g) * u and
// quantises each token's 128 values to E4M3 with s = amax / 448 (the
// activation and elementwise product between gate/up and down in the
// article's "CPU fine-grained parallelism" section).  Down: two consecutive
// 128-row output tiles take the places of gate and up, and the epilogue
// writes the unweighted fp32 expert output rows.
//
// Warp roles (256 threads, one persistent CTA per SM): warp 0 streams the
// stages (the block's two weight tiles, the tile's token rows, their scales
// and the weight-scale record, by bulk copies), warp 1 issues the MMAs,
// warps 4-7 drain TMEM (warp 4 + q reads lanes 32q..32q+31).  Barriers:
// full[s] (copies landed); tfull[b] (the block's MMAs done); empty[s],
// handed back by the epilogue warps as soon as tfull shows the MMAs done,
// so a stage is busy only for its copies and its MMAs; tempty[b], handed
// back once they have read the block's columns and scales.
#include "moe_internal.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace dec {

using tc::mma_commit;
using tc::mma_f8;
using tc::sw128_desc;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::tmem_alloc;
using tc::tmem_dealloc;
using tc::tmem_ld16u;
using tc::tmem_wait_ld;

constexpr int TN = DEC_TILE_N;           // token rows per unit = N of every MMA (16)
static_assert(TN == 16, "the epilogue holds one 16-column chunk per operand");
constexpr int CTRL_WARPS = 4;            // producer, MMA issuer, two idle
constexpr int EPI_WARPS = 4;             // one TMEM lane quarter each
constexpr int NTHREADS = (CTRL_WARPS + EPI_WARPS) * 32;
constexpr int STAGES = 6;
constexpr int NBUF = 8;                  // TMEM accumulator buffers of 2 x TN columns
constexpr uint32_t TMEM_COLS = 256;
static_assert(NBUF * 2 * TN <= (int)TMEM_COLS, "TMEM buffers");
constexpr int W_BYTES = 2 * TILE_BYTES;  // gate + up tile, or two consecutive down tiles
constexpr int X_BYTES = TN * 128;        // the tile's token rows (128-byte swizzled rows)
constexpr int STAGE = W_BYTES + X_BYTES; // a multiple of 1024: every stage stays 1024-byte aligned
static_assert(STAGE % 1024 == 0, "stage alignment");
// The block's scales (s_x of the tile's tokens, the weight-scale record) travel in their own ring
// of STAGES + 1 slots: the epilogue hands a stage back as soon as the block's MMAs are done and
// reads the scales later.  When the producer refills stage s for block n (block n - STAGES handed
// it back), the epilogue has finished every block up to n - STAGES - 1, the last user of slot
// n mod (STAGES + 1).
constexpr int S_BYTES = TN * 4;
constexpr int R_BYTES = 16;
constexpr int SC_SLOT = S_BYTES + R_BYTES;
constexpr int SC_SLOTS = STAGES + 1;
constexpr int GT_CAP_DEC = 386;          // groups held in the shared-memory table copy (+1)
constexpr int Q_STRIDE = 144;            // h-code staging row (token), bytes
constexpr int EPI_BYTES = SC_SLOTS * SC_SLOT + TN * Q_STRIDE + EPI_WARPS * TN * 4 + 2 * TN * 4;
constexpr int SMEM = STAGES * STAGE + EPI_BYTES + gt_smem_bytes(GT_CAP_DEC);
// dynamic (with 1024 bytes of alignment slack) + static (barriers) <= 227 KB
static_assert(SMEM + 1024 + 1024 <= 232448, "shared memory budget");

struct Args {
    const uint8_t* w;         // tile images of all groups
    const float* wrec;        // [group][weight block][k tile][4] weight-scale records
    const uint8_t* act;       // [K/128][rows_pad][128] swizzled E4M3
    const float* actsT;       // [K/128][rows_pad]
    int ld;                   // rows_pad
    int K, M;                 // reduction length; output features (I or H)
    const GroupTable* gt;
    uint8_t* hq;              // gate/up output codes (same layout as act)
    float* shT;               // gate/up output scales
    float* out;               // down: [rows_pad][M] fp32 expert outputs
    uint32_t* status;
    uint32_t wait_limit;
};

struct Unit {
    int expert, wb, row_begin, valid;
};

// u -> (group, token tile, weight block) with the weight block fastest.
__device__ __forceinline__ Unit decode_unit(const SGroups& g, int u, int NB) {
    const int pair = u / NB;
    Unit r;
    r.wb = u - pair * NB;
    decode_pair(g, pair, TN, r.expert, r.row_begin, r.valid);
    return r;
}

// Instruction descriptor, kind::f8f6f4: D f32, A = B = E4M3, both K-major,
// M = 128 (weight rows), N = TN (token rows).
constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(TN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

template <bool GU>
__global__ void __launch_bounds__(NTHREADS, 1) expert_dec_kernel(Args a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint8_t* scr = smem + STAGES * STAGE;                                  // [SC_SLOTS][SC_SLOT] block scales
    uint8_t* qst = scr + SC_SLOTS * SC_SLOT;                               // [TN][Q_STRIDE] h codes
    float* amax_s = reinterpret_cast<float*>(qst + TN * Q_STRIDE);          // [EPI_WARPS][TN]
    float* qs_s = amax_s + EPI_WARPS * TN;                                  // [2][TN]: s and 1/s per token
    int* gt_s = reinterpret_cast<int*>(scr + EPI_BYTES);
    __shared__ uint64_t full[STAGES], empty[STAGES], tfull[NBUF], tempty[NBUF], mdone;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = a.K / QB, MT = a.M / QB;
    const int NB = GU ? MT : (MT + 1) / 2;     // weight blocks per token tile
    const GroupTable* gt = a.gt;
    pdl_wait();                                // the group table and activations come from earlier kernels
    const int n_units = gt->n_pairs * NB;
    const SGroups sg = load_groups(gt, gt_s, threadIdx.x, NTHREADS, GT_CAP_DEC);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], EPI_WARPS); }
        for (int b = 0; b < NBUF; ++b) { mbar_init(&tfull[b], 1); mbar_init(&tempty[b], EPI_WARPS); }
        mbar_init(&mdone, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    // token rows past a tile's valid count are never copied: zero them once, so every column the
    // MMAs read holds finite codes (those columns' results are never used)
    for (int i = threadIdx.x; i < STAGES * (X_BYTES / 16); i += NTHREADS) {
        const int s = i / (X_BYTES / 16), c = i - s * (X_BYTES / 16);
        *reinterpret_cast<uint4*>(stages + (size_t)s * STAGE + W_BYTES + c * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 1) tmem_alloc(&tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int* abort = &abort_flag;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0, sslot = 0;
            uint32_t phase = 0, armed = 0, armed_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit un = decode_unit(sg, u, NB);
                const int t0 = GU ? un.wb : 2 * un.wb;
                const bool two = GU || t0 + 1 < MT;
                const uint8_t* wbase = a.w + ((size_t)(un.expert * MT + t0) * KT) * (GU ? W_BYTES : TILE_BYTES);
                for (int kb = 0; kb < KT; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, a.wait_limit, a.status, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = stages + (size_t)stage * STAGE;
                    uint8_t* tail = scr + sslot * SC_SLOT;
                    mbar_arrive_expect_tx(&full[stage],
                                          (two ? 2 : 1) * TILE_BYTES + un.valid * QB + S_BYTES + R_BYTES);
                    if (GU) {
                        bulk_g2s(st, wbase + (size_t)kb * W_BYTES, W_BYTES, &full[stage]);
                    } else {
                        bulk_g2s(st, wbase + (size_t)kb * TILE_BYTES, TILE_BYTES, &full[stage]);
                        if (two)
                            bulk_g2s(st + TILE_BYTES, wbase + ((size_t)KT + kb) * TILE_BYTES, TILE_BYTES, &full[stage]);
                    }
                    bulk_g2s(st + W_BYTES, a.act + act_offset(kb, un.row_begin, a.ld), un.valid * QB, &full[stage]);
                    bulk_g2s(tail, a.actsT + (size_t)kb * a.ld + un.row_begin, S_BYTES, &full[stage]);
                    bulk_g2s(tail + S_BYTES, a.wrec + (((size_t)un.expert * NB + un.wb) * KT + kb) * 4, R_BYTES,
                             &full[stage]);
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (++sslot == SC_SLOTS) sslot = 0;
                }
            }
            // every armed stage's copies land before the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) mbar_wait_bounded(&full[s], (armed_par >> s) & 1u, a.wait_limit, a.status, nullptr);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, buf = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true, issued = false;
            const uint64_t d0 = sw128_desc(smem_addr(stages));
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit un = decode_unit(sg, u, NB);
                const int t0 = GU ? un.wb : 2 * un.wb;
                const bool two = GU || t0 + 1 < MT;
                for (int kb = 0; kb < KT; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, a.wait_limit, a.status, abort) ||
                        !mbar_wait_bounded(&tempty[buf], tphase ^ 1u, a.wait_limit, a.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t w0 = d0 + (uint64_t)(((size_t)stage * STAGE) >> 4);              // tile 0
                    const uint64_t w1 = w0 + (uint64_t)(TILE_BYTES >> 4);                           // tile 1
                    const uint64_t xd = d0 + (uint64_t)(((size_t)stage * STAGE + W_BYTES) >> 4);    // tokens
                    const uint32_t dt = tmem + (uint32_t)(buf * 2 * TN);
#pragma unroll
                    for (int k = 0; k < 4; ++k) mma_f8(dt, w0 + 2 * k, xd + 2 * k, IDESC, k > 0 ? 1u : 0u);
                    if (two) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) mma_f8(dt + TN, w1 + 2 * k, xd + 2 * k, IDESC, k > 0 ? 1u : 0u);
                    }
                    mma_commit(&tfull[buf]);
                    issued = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (++buf == NBUF) { buf = 0; tphase ^= 1u; }
                }
            }
            // every issued MMA completes before the tensor memory is released
            if (issued) {
                mma_commit(&mdone);
                mbar_wait_bounded(&mdone, 0u, a.wait_limit, a.status, nullptr);
            }
        }
        __syncwarp();
    } else if (warp >= CTRL_WARPS) {
        // ------------------------------------------------------------ epilogue warps
        const int q4 = warp & 3;                       // TMEM lanes 32 q4 .. 32 q4 + 31
        const int r = q4 * 32 + lane;                  // weight row inside the 128-row tile
        const int et = threadIdx.x - CTRL_WARPS * 32;  // 0 .. 127
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        int buf = 0, slot = 0, sslot = 0;
        uint32_t tphase = 0;
        bool dead = false;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
            const Unit un = decode_unit(sg, u, NB);
            const int t0 = GU ? un.wb : 2 * un.wb;
            const bool two = GU || t0 + 1 < MT;
            float acc0[TN], acc1[TN];                  // tile 0 (gate / down t0), tile 1 (up / down t0 + 1)
#pragma unroll
            for (int i = 0; i < TN; ++i) { acc0[i] = 0.f; acc1[i] = 0.f; }
            for (int kb = 0; kb < KT; ++kb) {
                if (!dead && !mbar_wait_bounded(&tfull[buf], tphase, a.wait_limit, a.status, abort)) dead = true;
                dead = __any_sync(0xFFFFFFFFu, dead);      // warp-uniform: tcgen05.ld is warp-collective
                // the block's MMAs are done: its stage can be refilled
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
                if (!dead) {
                    tc_fence_after();
                    uint32_t v0[16], v1[16];
                    tmem_ld16u(trow + (uint32_t)(buf * 2 * TN), v0);
                    if (two) tmem_ld16u(trow + (uint32_t)(buf * 2 * TN + TN), v1);
                    const float* sx = reinterpret_cast<const float*>(scr + sslot * SC_SLOT);
                    const float2 sw = *reinterpret_cast<const float2*>(scr + sslot * SC_SLOT + S_BYTES);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < TN; ++j) {
                        const float s = sx[j];
                        acc0[j] = __fmaf_rn(__uint_as_float(v0[j]), __fmul_rn(sw.x, s), acc0[j]);
                        if (two) acc1[j] = __fmaf_rn(__uint_as_float(v1[j]), __fmul_rn(sw.y, s), acc1[j]);
                    }
                    tc_fence_before();
                }
                // the block is read: its buffer goes back
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
                if (++buf == NBUF) { buf = 0; tphase ^= 1u; }
                if (++slot == STAGES) slot = 0;
                if (++sslot == SC_SLOTS) sslot = 0;
            }

            if (GU) {
                // ---------------------------------------------- h = SiLU(g) * u, 1x128 E4M3 quantisation
                // thread r holds inner feature r of the 128-feature block for each token
                float h[TN];
#pragma unroll
                for (int i = 0; i < TN; ++i) {
                    h[i] = silu_mul(acc0[i], acc1[i]);
                    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(h[i])));
                    if (lane == 0) amax_s[q4 * TN + i] = __uint_as_float(m);   // |h| >= 0: bits order as values
                }
                named_bar_sync(1, EPI_WARPS * 32);
                if (et < TN) {                                  // token et's scale, once
                    float am = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < EPI_WARPS; ++w2) am = fmaxf(am, amax_s[w2 * TN + et]);
                    const float sc = (am > 0.f) ? __fdiv_rn(am, 448.0f) : 1.0f;
                    qs_s[et] = sc;
                    qs_s[TN + et] = __frcp_rn(sc);              // h / s as h * (1/s), as in prefill
                    if (et < un.valid) a.shT[(size_t)un.wb * a.ld + un.row_begin + et] = sc;
                }
                named_bar_sync(1, EPI_WARPS * 32);
#pragma unroll
                for (int i = 0; i < TN; i += 2) {
                    const uint16_t pq = f32x2_to_e4m3x2(h[i] * qs_s[TN + i], h[i + 1] * qs_s[TN + i + 1]);
                    qst[i * Q_STRIDE + r] = (uint8_t)(pq & 0xFF);
                    qst[(i + 1) * Q_STRIDE + r] = (uint8_t)(pq >> 8);
                }
                named_bar_sync(1, EPI_WARPS * 32);
                // 16 bytes per thread, 16 token rows per pass, into the swizzled K-block-major layout
                {
                    const int rr = et >> 3;
                    if (rr < un.valid) {
                        const uint4 v = lds128(qst + rr * Q_STRIDE + (et & 7) * 16);
                        const int pos = (et & 7) ^ (rr & 7);              // row_begin is a multiple of 8
                        *reinterpret_cast<uint4*>(a.hq + act_offset(un.wb, un.row_begin + rr, a.ld) + pos * 16) = v;
                    }
                }
                named_bar_sync(1, EPI_WARPS * 32);
            } else {
                // ---------------------------------------------- fp32 expert output rows: feature r of tiles
                // t0 and t0 + 1 for every valid token (a warp stores 128 contiguous bytes per row)
                float* dst = a.out + (size_t)un.row_begin * a.M + (size_t)t0 * QB + r;
#pragma unroll
                for (int i = 0; i < TN; ++i) {
                    if (i < un.valid) {
                        dst[(size_t)i * a.M] = acc0[i];
                        if (two) dst[(size_t)i * a.M + QB] = acc1[i];
                    }
                }
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
    {
        cudaError_t e = ensure_smem_limit<expert_dec_kernel<GU>>(SMEM + 1024);
        if (e != cudaSuccess) return e;
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
        a.w = L->w_gu; a.wrec = L->r_gu;
        a.act = reinterpret_cast<const uint8_t*>(ws + lay.xp);
        a.actsT = reinterpret_cast<const float*>(ws + lay.sxT);
        a.K = H; a.M = I;
    } else {
        a.w = L->w_dn; a.wrec = L->r_dn;
        a.act = reinterpret_cast<const uint8_t*>(ws + lay.hq);
        a.actsT = reinterpret_cast<const float*>(ws + lay.shT);
        a.K = I; a.M = H;
    }
    return launch_pdl(expert_dec_kernel<GU>, dim3(L->num_sms), dim3(NTHREADS), SMEM + 1024, s, a);
}

}  // namespace dec

cudaError_t launch_expert_dec_gate_up(const moe_layer* L, int T, const WsLayout& lay, char* ws, int bn,
                                      cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (bn != dec::TN) return cudaErrorInvalidValue;     // the group table must be built for TN-row tiles
    return dec::launch<true>(L, lay, ws, s);
}

cudaError_t launch_expert_dec_down(const moe_layer* L, int T, const WsLayout& lay, char* ws, int bn,
                                   cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (bn != dec::TN) return cudaErrorInvalidValue;
    return dec::launch<false>(L, lay, ws, s);
}

}  // namespace moe
