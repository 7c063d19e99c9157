// Grouped FP8 expert GEMMs on sm_103a (weight-streaming path).
//
// One persistent CTA per SM walks the units (group, n tile of <= 64 rows,
// weight block): a gate/up block is the gate and up tiles of 128 inner
// features, a down block two consecutive 128-row tiles of the output.  A
// producer warp streams, for every 128-wide K block, the block's two
// 128x128 weight tile images with bulk copies and
// the unit's activation rows (128 B each) with per-row bulk copies into a
// ring of shared-memory stages guarded by mbarriers; eight consumer warps
// run FP8 E4M3 tensor-core MMAs (m16n8k32, fp32 accumulate) on each stage.
//
// Scale promotion follows the post-scaling order of the FP8 GEMV section
// of the CPU-GPU hybrid inference article (xingyun.xin, Fig. 9-10): the
// products inside one 128-block are accumulated first (by the tensor core),
// then the block is scaled once, here by s_w[block] * s_a[row][block], and
// added to the fp32 accumulator.  Both scales travel in the stage with the
// operands (two more bulk copies), so the consumers never wait on a global
// load inside the K loop.
//
// Gate/up kernel: both projections of the same 128 rows of the expert's
// inner dimension share the activation fragments; the epilogue forms
// h = SiLU(g) * u (the activation and elementwise product that sit between
// gate/up and down in the article's "CPU fine-grained parallelism"
// section), quantises each token's 128 values of h to E4M3 with
// s = amax/448, and writes the codes and the scale.  Down kernel: the two
// output tiles take the places of gate and up (same fragments, second
// accumulator) and it writes the unweighted fp32 expert output rows of both.
//
// K permutation inside a 128-block: lane (g, q) of a warp owns the 32
// consecutive channels [32q, 32q+32) of the block; MMA m (0..3) takes
// channels 32q+8m .. 32q+8m+7 of them as its k-slots {4q..4q+3,
// 16+4q..16+4q+3}.  The same map is applied to the weight rows and to the
// activation rows, so the dot products are unchanged while every operand
// fragment comes from two 16-byte shared-memory loads.
#include "moe_internal.cuh"

namespace moe {

constexpr int BN = DEC_TILE_N;          // rows (tokens) per n tile
constexpr int CW = 8;                   // consumer warps (16 output rows each)
constexpr int NTHREADS = (CW + 1) * 32; // + producer warp
constexpr int XSTRIDE = 128;            // activation row in shared memory (swizzled)
constexpr int GT_CAP_DEC = 386;         // groups held in the shared-memory table copy (+1)

// Stage tail: the tile rows' activation scales of this k block (BN floats)
// and the 16-byte weight-scale record, brought by the producer with the
// operands; padded so the next stage's weight tiles stay 1024-byte aligned.
constexpr int S_BYTES = BN * 4;
constexpr int R_BYTES = 16;
constexpr int TAIL = 1024;

template <bool GU>
struct Cfg {
    static constexpr int W_BYTES = 2 * TILE_BYTES;      // gate + up tile, or two consecutive down tiles
    static constexpr int X_BYTES = BN * XSTRIDE;
    static constexpr int STAGE = W_BYTES + X_BYTES + TAIL;
    static constexpr int STAGES = GU ? 5 : 4;           // as deep as shared memory allows (HBM latency)
    static constexpr int EPI = GU ? (BN * 144 + CW * BN * 4) : (BN * 132 * 4);
    // + the group table copy for up to 385 groups (larger tables are read in place)
    static constexpr int SMEM = STAGES * STAGE + EPI + gt_smem_bytes(GT_CAP_DEC) + 2 * STAGES * 8 + 128;
};

struct ExpertArgs {
    const uint8_t* w;         // tile images of all groups
    const float* wrec;        // weight-scale records, [group][m tile (down: pair of m tiles)][k tile][4]
    const uint8_t* act;       // activations [K/128][rows_pad][128] (E4M3, swizzled)
    const float* actsT;       // activation scales [K/128][ld]
    int ld;                   // rows_pad of the permuted buffers
    int K, M;                 // reduction length, output features
    const GroupTable* gt;
    uint8_t* hq;              // gate/up: [M/128][rows_pad][128] E4M3 h (swizzled)
    float* shT;               // gate/up: [M/128][ld]
    float* out;               // down: [rows][M] fp32
    uint32_t* status;
    uint32_t wait_limit;
};

struct Unit {
    int expert, mb, row_begin, valid;
};

__device__ __forceinline__ Unit decode_unit(const SGroups& g, int u, int MT) {
    const int pair = u / MT;
    Unit r;
    r.mb = u - pair * MT;
    decode_pair(g, pair, BN, r.expert, r.row_begin, r.valid);
    return r;
}


template <bool GU>
__global__ void __launch_bounds__(NTHREADS, 1) expert_gemm_kernel(ExpertArgs a) {
    using C = Cfg<GU>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint8_t* epi = smem + C::STAGES * C::STAGE;
    int* gt_s = reinterpret_cast<int*>(epi + C::EPI);
    uint64_t* full = reinterpret_cast<uint64_t*>(epi + C::EPI + gt_smem_bytes(GT_CAP_DEC));
    uint64_t* empty = full + C::STAGES;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int MT = a.M / QB, KT = a.K / QB;
    // weight blocks per n tile: gate/up one 128-row tile pair (gate, up) each; down two consecutive
    // 128-row output tiles each (the last block of an odd tile count has one)
    const int NB = GU ? MT : (MT + 1) / 2;
    const GroupTable* gt = a.gt;
    pdl_wait();                                   // the group table and activations come from earlier kernels
    const int n_units = gt->n_pairs * NB;
    const SGroups sg = load_groups(gt, gt_s, threadIdx.x, NTHREADS, GT_CAP_DEC);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    volatile int* abort = &abort_flag;

    if (warp == CW) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t armed = 0, armed_par = 0;       // per stage: armed at least once / parity of last arm
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Unit un = decode_unit(sg, u, NB);
            const int t0 = GU ? un.mb : 2 * un.mb;
            const bool two = GU || t0 + 1 < MT;
            const uint8_t* wbase = a.w + ((size_t)(un.expert * MT + t0) * KT) * (GU ? C::W_BYTES : TILE_BYTES);
            for (int kb = 0; kb < KT; ++kb) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, a.wait_limit, a.status, abort)) { ok = false; break; }
                uint8_t* st = stages + stage * C::STAGE;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[stage],
                                          (two ? 2 : 1) * TILE_BYTES + un.valid * QB + S_BYTES + R_BYTES);
                    if (GU) {
                        bulk_g2s(st, wbase + (size_t)kb * C::W_BYTES, C::W_BYTES, &full[stage]);
                    } else {
                        bulk_g2s(st, wbase + (size_t)kb * TILE_BYTES, TILE_BYTES, &full[stage]);
                        if (two)
                            bulk_g2s(st + TILE_BYTES, wbase + ((size_t)KT + kb) * TILE_BYTES, TILE_BYTES, &full[stage]);
                    }
                    bulk_g2s(st + C::W_BYTES, a.act + act_offset(kb, un.row_begin, a.ld), un.valid * QB,
                             &full[stage]);
                    uint8_t* tail = st + C::W_BYTES + C::X_BYTES;
                    bulk_g2s(tail, a.actsT + (size_t)kb * a.ld + un.row_begin, S_BYTES, &full[stage]);
                    const size_t rec = ((size_t)un.expert * NB + un.mb) * KT + kb;
                    bulk_g2s(tail + S_BYTES, a.wrec + rec * 4, R_BYTES, &full[stage]);
                }
                __syncwarp();
                armed |= 1u << stage;
                armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        // drain: every armed stage's copies must have landed before exit
        for (int s = 0; s < C::STAGES; ++s)
            if ((armed >> s) & 1u) mbar_wait_bounded(&full[s], (armed_par >> s) & 1u, a.wait_limit, a.status, nullptr);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, q = lane & 3;
    const int r0 = warp * 16 + g;             // tile rows r0 and r0 + 8 (same swizzle phase g)
    const int c0 = ((2 * q) ^ g) * 16, c1 = ((2 * q + 1) ^ g) * 16;
    int stage = 0;
    uint32_t phase = 0;
    bool dead = false;    // a wait gave up: skip the math, keep the barriers

    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit un = decode_unit(sg, u, NB);
        const int nt_active = (un.valid + 7) >> 3;
        const int t0 = GU ? un.mb : 2 * un.mb;         // down: output tiles t0 (accg) and t0 + 1 (accu)
        const bool dual = GU || t0 + 1 < MT;
        float accg[BN / 8][4], accu[BN / 8][4];
#pragma unroll
        for (int nt = 0; nt < BN / 8; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) { accg[nt][i] = 0.f; accu[nt][i] = 0.f; }

        for (int kb = 0; kb < KT; ++kb) {
            if (!dead && !mbar_wait_bounded(&full[stage], phase, a.wait_limit, a.status, abort)) dead = true;
            if (dead) {
                if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                continue;
            }
            const uint8_t* st = stages + stage * C::STAGE;
            // scales from the stage tail: s_x of this lane's columns, the weight-scale record
            // (gate/up: {gate, up}; down: {tile 2b, tile 2b+1})
            const float* tail = reinterpret_cast<const float*>(st + C::W_BYTES + C::X_BYTES);
            const float2 rec = *reinterpret_cast<const float2*>(tail + BN);
            const float swg = rec.x;
            const float swu = rec.y;
            float sa[BN / 8][2];
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt) {
                const float2 v = *reinterpret_cast<const float2*>(tail + nt * 8 + 2 * q);
                sa[nt][0] = v.x;
                sa[nt][1] = v.y;
            }
            const uint8_t* X = st + C::W_BYTES;
            const uint4 ag0 = lds128(st + r0 * 128 + c0), ag1 = lds128(st + r0 * 128 + c1);
            const uint4 ag8 = lds128(st + (r0 + 8) * 128 + c0), ag9 = lds128(st + (r0 + 8) * 128 + c1);
            const uint32_t Ag[8] = {ag0.x, ag0.y, ag0.z, ag0.w, ag1.x, ag1.y, ag1.z, ag1.w};
            const uint32_t Ah[8] = {ag8.x, ag8.y, ag8.z, ag8.w, ag9.x, ag9.y, ag9.z, ag9.w};
            uint32_t Bg[8] = {0, 0, 0, 0, 0, 0, 0, 0}, Bh[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (dual) {
                const uint8_t* U = st + TILE_BYTES;
                const uint4 au0 = lds128(U + r0 * 128 + c0), au1 = lds128(U + r0 * 128 + c1);
                const uint4 au8 = lds128(U + (r0 + 8) * 128 + c0), au9 = lds128(U + (r0 + 8) * 128 + c1);
                Bg[0] = au0.x; Bg[1] = au0.y; Bg[2] = au0.z; Bg[3] = au0.w;
                Bg[4] = au1.x; Bg[5] = au1.y; Bg[6] = au1.z; Bg[7] = au1.w;
                Bh[0] = au8.x; Bh[1] = au8.y; Bh[2] = au8.z; Bh[3] = au8.w;
                Bh[4] = au9.x; Bh[5] = au9.y; Bh[6] = au9.z; Bh[7] = au9.w;
            }
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt) {
                if (nt < nt_active) {
                    const uint8_t* xr = X + (nt * 8 + g) * XSTRIDE;      // row & 7 == g: same swizzle as A
                    const uint4 xb0 = lds128(xr + c0), xb1 = lds128(xr + c1);
                    const uint32_t Bx[8] = {xb0.x, xb0.y, xb0.z, xb0.w, xb1.x, xb1.y, xb1.z, xb1.w};
                    float pg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        mma_e4m3_16832(pg, Ag[2 * m], Ah[2 * m], Ag[2 * m + 1], Ah[2 * m + 1], Bx[2 * m],
                                       Bx[2 * m + 1], pg);
                    const float s0 = swg * sa[nt][0], s1 = swg * sa[nt][1];
                    accg[nt][0] = __fmaf_rn(pg[0], s0, accg[nt][0]);
                    accg[nt][1] = __fmaf_rn(pg[1], s1, accg[nt][1]);
                    accg[nt][2] = __fmaf_rn(pg[2], s0, accg[nt][2]);
                    accg[nt][3] = __fmaf_rn(pg[3], s1, accg[nt][3]);
                    if (dual) {
                        float pu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int m = 0; m < 4; ++m)
                            mma_e4m3_16832(pu, Bg[2 * m], Bh[2 * m], Bg[2 * m + 1], Bh[2 * m + 1], Bx[2 * m],
                                           Bx[2 * m + 1], pu);
                        const float t0 = swu * sa[nt][0], t1 = swu * sa[nt][1];
                        accu[nt][0] = __fmaf_rn(pu[0], t0, accu[nt][0]);
                        accu[nt][1] = __fmaf_rn(pu[1], t1, accu[nt][1]);
                        accu[nt][2] = __fmaf_rn(pu[2], t0, accu[nt][2]);
                        accu[nt][3] = __fmaf_rn(pu[3], t1, accu[nt][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }

        if (GU) {
            // ---------------------------------------------- SiLU(g)*u, 1x128 quantisation
            uint8_t* qst = epi;                                   // [BN][144] codes (unswizzled)
            float* amax_s = reinterpret_cast<float*>(epi + BN * 144);   // [CW][BN]
            float h[BN / 8][4];
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt) {
                float m0 = 0.f, m1 = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) h[nt][i] = silu_mul(accg[nt][i], accu[nt][i]);
                m0 = fmaxf(fabsf(h[nt][0]), fabsf(h[nt][2]));
                m1 = fmaxf(fabsf(h[nt][1]), fabsf(h[nt][3]));
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    m0 = fmaxf(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, off));
                    m1 = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, off));
                }
                if (g == 0) {
                    amax_s[warp * BN + nt * 8 + 2 * q] = m0;
                    amax_s[warp * BN + nt * 8 + 2 * q + 1] = m1;
                }
            }
            named_bar_sync(1, CW * 32);
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt) {
                if (nt < nt_active) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int col = nt * 8 + 2 * q + j;
                        float am = 0.f;
#pragma unroll
                        for (int w2 = 0; w2 < CW; ++w2) am = fmaxf(am, amax_s[w2 * BN + col]);
                        const float sc = (am > 0.f) ? __fdiv_rn(am, 448.0f) : 1.0f;
                        const float rs = __frcp_rn(sc);                  // h / s as h * (1/s), as in prefill
                        const uint16_t pq = f32x2_to_e4m3x2(h[nt][j] * rs, h[nt][2 + j] * rs);
                        qst[col * 144 + r0] = (uint8_t)(pq & 0xFF);
                        qst[col * 144 + r0 + 8] = (uint8_t)(pq >> 8);
                        if (warp == 0 && g == 0 && col < un.valid)
                            a.shT[(size_t)un.mb * a.ld + un.row_begin + col] = sc;
                    }
                }
            }
            named_bar_sync(1, CW * 32);
            // 16 bytes per thread, 8 rows per pass, into the swizzled K-block-major layout
            const int tid = threadIdx.x;
            for (int rr = tid >> 3; rr < un.valid; rr += (CW * 32) >> 3) {
                const uint4 v = lds128(qst + rr * 144 + (tid & 7) * 16);
                const int pos = (tid & 7) ^ (rr & 7);                 // row_begin is a multiple of 8
                *reinterpret_cast<uint4*>(a.hq + act_offset(un.mb, un.row_begin + rr, a.ld) + pos * 16) = v;
            }
            named_bar_sync(1, CW * 32);
        } else {
            // ---------------------------------------------- fp32 expert output rows: tile t0 from accg,
            // tile t0 + 1 from accu, each staged through shared memory and stored row by row
            float* ost = reinterpret_cast<float*>(epi);           // [BN][132]
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                if (part == 1 && !dual) break;
                const float(&acc)[BN / 8][4] = part ? accu : accg;
#pragma unroll
                for (int nt = 0; nt < BN / 8; ++nt) {
                    if (nt < nt_active) {
                        const int col = nt * 8 + 2 * q;
                        ost[col * 132 + r0] = acc[nt][0];
                        ost[(col + 1) * 132 + r0] = acc[nt][1];
                        ost[col * 132 + r0 + 8] = acc[nt][2];
                        ost[(col + 1) * 132 + r0 + 8] = acc[nt][3];
                    }
                }
                named_bar_sync(1, CW * 32);
                const int tid = threadIdx.x;
                for (int rr = tid >> 5; rr < un.valid; rr += (CW * 32) >> 5) {
                    const float4 v = *reinterpret_cast<const float4*>(ost + rr * 132 + (tid & 31) * 4);
                    *reinterpret_cast<float4*>(a.out + (size_t)(un.row_begin + rr) * a.M + (t0 + part) * QB +
                                               (tid & 31) * 4) = v;
                }
                named_bar_sync(1, CW * 32);
            }
        }
    }
}

template <bool GU>
static cudaError_t launch_expert(const moe_layer* L, const WsLayout& lay, char* ws, cudaStream_t s) {
    using C = Cfg<GU>;
    {
        cudaError_t e = ensure_smem_limit<expert_gemm_kernel<GU>>(C::SMEM + 1024);
        if (e != cudaSuccess) return e;
    }
    ExpertArgs a;
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
    const int grid = L->num_sms;
    return launch_pdl(expert_gemm_kernel<GU>, dim3(grid), dim3(NTHREADS), C::SMEM + 1024, s, a);
}

cudaError_t launch_expert_gate_up(const moe_layer* L, int T, const WsLayout& lay, char* ws, int bn, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (bn != BN) return cudaErrorInvalidValue;       // the group table must be built for BN-row tiles
    return launch_expert<true>(L, lay, ws, s);
}

cudaError_t launch_expert_down(const moe_layer* L, int T, const WsLayout& lay, char* ws, int bn, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (bn != BN) return cudaErrorInvalidValue;
    return launch_expert<false>(L, lay, ws, s);
}

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
