// Grouped FP8 expert GEMMs for prefill on the 5th-generation tensor cores
// (tcgen05, sm_103a).
//
// Tile: A = 128 token rows of one expert's group, B = 256 weight rows, K =
// 128 per stage.  Gate/up: B = the expert's gate tile and up tile of the
// same 128 inner features, which sit next to each other in the repacked
// weights, so one M128 x N256 x K32 MMA covers both projections.  Down: B =
// two consecutive 128-row tiles of the down weights (256 outputs), written as
// fp32 expert-output rows.  Both
// operands are 128-byte-swizzled K-major images that one bulk copy each
// brings into shared memory.  One thread issues tcgen05.mma kind::f8f6f4
// (E4M3 x E4M3, fp32 accumulate in tensor memory), 4 per stage, with
// descriptors advanced by a constant; accumulators are double-buffered in
// TMEM (2 x 256 columns).
//
// Scale promotion (FP8 GEMV section of the CPU-GPU hybrid inference
// article, Fig. 9-10: a 128-element block's partial sum is scaled once):
// each TMEM lane is one token, so its activation scale s_x[token][kb] is a
// per-thread scalar and the weight scales s_w[kb] are uniform; the epilogue
// warps read each block's partial with tcgen05.ld, 16 columns at a time,
// and promote it into registers with packed fp32 FMAs (fma.rn.f32x2: two
// lanes of the same IEEE fma per instruction, half the issue slots of scalar
// FFMA).  Both scales are copied with the stage's operands into the stage's
// scale slot; the epilogue warps read them once the block's MMAs have
// completed and then hand the stage back themselves, so one commit per block
// (on the TMEM buffer) serves both the epilogue and the producer.  Gate/up
// then forms h = SiLU(g)*u and its
// 1x128 E4M3 codes (the activation and elementwise product between gate/up
// and down, "CPU fine-grained parallelism" section of the same article);
// down writes fp32 output rows.
//
// Unit = (group, token tile of 128, weight block), weight block fastest, so
// the CTAs working on one token tile at a time share its bytes through L2.
#include "moe_internal.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;                 // token rows per tile (TMEM lanes)
constexpr int BN = 256;                 // weight rows per tile (TMEM columns per buffer)
constexpr int EPI_WARPS = 8;            // 4 lane quarters x 2 column halves
constexpr int HALF = BN / 2;            // columns per epilogue thread (per buffer)
constexpr int CTRL_WARPS = 4;           // warpgroup 0: producer, MMA issuer, 2 idle
constexpr int NTHREADS = (CTRL_WARPS + EPI_WARPS) * 32;
// Register split (setmaxnreg acts per warpgroup): launched at 168 per thread
// (384 x 168 = 64,512); the control warpgroup drops to 32 and the two
// epilogue warpgroups rise to 232: 4*32*32 + 8*32*232 = 63,488.
constexpr int CTRL_REGS = 32, EPI_REGS = 232;
static_assert(CTRL_WARPS * 32 * CTRL_REGS + EPI_WARPS * 32 * EPI_REGS <= NTHREADS * 168, "register split");
constexpr uint32_t TMEM_COLS = 512;
constexpr int STAGES = 4;
constexpr int W_BYTES = 2 * TILE_BYTES;   // 256 weight rows
constexpr int X_BYTES = BM * 128;         // 128 token rows
constexpr int STAGE = W_BYTES + X_BYTES;
// Scale slot of each stage: the k block's 128 token activation scales
// (512 B) and the weight-scale record (16 B), copied with the stage's
// operands (counted on its full barrier).  The stage, slot included, is
// handed back by the epilogue warps (EPI_WARPS arrivals on its empty
// barrier) once they have read the scales, which is after the block's MMAs
// completed.
constexpr int S_BYTES = BM * 4;
constexpr int R_BYTES = 16;
constexpr int SSLOT = S_BYTES + R_BYTES;
// + amax exchange + the group table copy (units are decoded from shared
// memory; up to 385 groups, larger tables are read in place) + the down
// epilogue's per-warp staging tiles (32 rows x 16 floats, rows 20 floats
// apart so the row-wise writes are free of bank conflicts)
constexpr int GT_SMEM_CAP = 386;
constexpr int STG_STRIDE = 20;
constexpr int STG_BYTES = EPI_WARPS * 32 * STG_STRIDE * 4;
constexpr int SMEM = STAGES * STAGE + STAGES * SSLOT + 2 * 4 * 32 * 4 + gt_smem_bytes(GT_SMEM_CAP) + STG_BYTES + 256;
// dynamic (with 1024 bytes of alignment slack) + static (barriers, padded to 1024) <= 227 KB
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

// Instruction descriptor, kind::f8f6f4: D f32, A = B = E4M3, both K-major,
// M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_for(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// u -> (group, token tile, weight block) with the weight block fastest.
// NB = weight blocks per group (I/128 for gate/up, ceil(H/256) for down).
__device__ __forceinline__ Unit decode_unit(const SGroups& g, int u, int NB) {
    const int pair = u / NB;
    Unit r;
    r.wb = u - pair * NB;
    decode_pair(g, pair, BM, r.expert, r.row_begin, r.valid);
    return r;
}



// ------------------------------------------------------------------ kernel
template <bool GU>
__global__ void __launch_bounds__(NTHREADS, 1) expert_tc_kernel(Args a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint8_t* sring = smem + STAGES * STAGE;                                 // [STAGES][SSLOT]
    uint8_t* after = sring + STAGES * SSLOT;
    float* amax_x = reinterpret_cast<float*>(after);                       // [2 halves][4 quarters][32 lanes]
    int* gt_s = reinterpret_cast<int*>(after + 2 * 4 * 32 * 4);
    float* stg_all = reinterpret_cast<float*>(after + 2 * 4 * 32 * 4 + gt_smem_bytes(GT_SMEM_CAP));
    __shared__ uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = a.K / QB;
    const int MT128 = a.M / QB;                              // 128-row weight tiles per expert
    const int NB = GU ? MT128 : (MT128 + 1) / 2;             // weight blocks per unit row
    const GroupTable* gt = a.gt;
    pdl_wait();                                   // the group table and activations come from earlier kernels
    const int n_units = gt->n_pairs * NB;
    const SGroups sg = load_groups(gt, gt_s, threadIdx.x, NTHREADS, GT_SMEM_CAP);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], EPI_WARPS); }
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

    if (warp < CTRL_WARPS) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(CTRL_REGS));
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------------- producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit un = decode_unit(sg, u, NB);
                // gate/up: the gate+up pair of inner tile wb (32 KB, contiguous per k block);
                // down: tiles 2wb and 2wb+1 of the output rows (16 KB each, KT tiles apart)
                const int t0 = GU ? un.wb : 2 * un.wb;
                const bool two = GU || (t0 + 1 < MT128);
                const uint32_t wbytes = two ? (uint32_t)W_BYTES : (uint32_t)TILE_BYTES;
                const uint8_t* wbase = a.w + ((size_t)(un.expert * MT128 + t0) * KT) * (GU ? W_BYTES : TILE_BYTES);
                for (int kb = 0; kb < KT; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, a.wait_limit, a.status, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = stages + stage * STAGE;
                    uint8_t* ss = sring + stage * SSLOT;
                    mbar_arrive_expect_tx(&full[stage], wbytes + X_BYTES + S_BYTES + R_BYTES);
                    if (GU) {
                        bulk_g2s(st, wbase + (size_t)kb * W_BYTES, W_BYTES, &full[stage]);
                    } else {
                        bulk_g2s(st, wbase + (size_t)kb * TILE_BYTES, TILE_BYTES, &full[stage]);
                        if (two)
                            bulk_g2s(st + TILE_BYTES, wbase + ((size_t)KT + kb) * TILE_BYTES, TILE_BYTES, &full[stage]);
                    }
                    bulk_g2s(st + W_BYTES, a.act + act_offset(kb, un.row_begin, a.ld), X_BYTES, &full[stage]);
                    bulk_g2s(ss, a.actsT + (size_t)kb * a.ld + un.row_begin, S_BYTES, &full[stage]);
                    bulk_g2s(ss + S_BYTES, a.wrec + (((size_t)un.expert * NB + un.wb) * KT + kb) * 4, R_BYTES,
                             &full[stage]);
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) mbar_wait_bounded(&full[s], (armed_par >> s) & 1u, a.wait_limit, a.status, nullptr);
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------------- MMA issuer
            int stage = 0, buf = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true;
            const uint64_t d0 = sw128_desc(smem_addr(stages));        // stage 0, weight operand
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const int wb = u % NB;
                const bool two = GU || (2 * wb + 1 < MT128);
                const uint32_t idesc = idesc_for(two ? BN : BN / 2);
                for (int kb = 0; kb < KT; ++kb) {
                    // the stage's copies usually land long before the buffer is handed back:
                    // waiting for them first keeps that wait off the hand-off path
                    if (!mbar_wait_bounded(&full[stage], phase, a.wait_limit, a.status, abort) ||
                        !mbar_wait_bounded(&tempty[buf], tphase ^ 1u, a.wait_limit, a.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = d0 + (uint64_t)((stage * STAGE) >> 4);                   // weights
                    const uint64_t adesc = d0 + (uint64_t)((stage * STAGE + W_BYTES) >> 4);       // tokens
                    const uint32_t dt = tmem + (uint32_t)(buf * BN);
                    mma_f8(dt, adesc, bdesc, idesc, 0u);
                    mma_f8(dt, adesc + 2, bdesc + 2, idesc, 1u);
                    mma_f8(dt, adesc + 4, bdesc + 4, idesc, 1u);
                    mma_f8(dt, adesc + 6, bdesc + 6, idesc, 1u);
                    mma_commit(&tfull[buf]);          // the epilogue hands the stage back after this
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (++buf == 2) { buf = 0; tphase ^= 1u; }
                }
            }
        }
        __syncwarp();
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(EPI_REGS));
        // ------------------------------------------------------------ epilogue warps
        const int ew = warp - CTRL_WARPS;           // 0..7
        const int quarter = warp & 3;               // TMEM lanes this warp may read
        const int half = ew >> 2;                   // column half of the 256-column buffer
        const int r = quarter * 32 + lane;          // token row inside the tile
        int buf = 0, slot = 0;                        // slot: the stage of the block (scales, empty barrier)
        uint32_t tphase = 0;
        bool dead = false;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
            const Unit un = decode_unit(sg, u, NB);
            const bool rv = r < un.valid;
            const int t0 = GU ? un.wb : 2 * un.wb;
            const bool two = GU || (t0 + 1 < MT128);
            float acc[HALF];                          // 128 fp32 accumulators (my row, my columns)
#pragma unroll
            for (int c = 0; c < HALF; ++c) acc[c] = 0.f;
            for (int kb = 0; kb < KT; ++kb) {
                if (!dead && !mbar_wait_bounded(&tfull[buf], tphase, a.wait_limit, a.status, abort)) dead = true;
                dead = __any_sync(0xFFFFFFFFu, dead);      // warp-uniform: tcgen05.ld is warp-collective
                if (!dead) {
                    tc_fence_after();
                    // this block's scales from its stage's slot: s_x of my token, the record's weight
                    // scales; combined per 32-column chunk (gate/up: c0 gate, c1 up; down: my half's tile)
                    const uint8_t* tail = sring + slot * SSLOT;
                    const float sx = reinterpret_cast<const float*>(tail)[r];
                    const float2 sw = *reinterpret_cast<const float2*>(tail + S_BYTES);
                    const float c0 = (GU || half == 0) ? sw.x * sx : sw.y * sx;
                    const float c1 = sw.y * sx;
                    const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN);
                    // Eight 16-column pieces, software-pipelined: the next piece's tcgen05.ld is in
                    // flight while this piece's FMAs issue.  32-column chunk i = piece / 2 covers, for
                    // gate/up, gate (i even) or up (i odd) columns [64h + 32(i/2), +32) of its
                    // 128-column tile into accumulators 64(i%2) + 32(i/2); for down, columns
                    // [128h + 32i, +32) into accumulators 32i.
                    auto col_of = [&](int i) -> uint32_t {
                        return GU ? (uint32_t)((i & 1) * 128 + 64 * half + 32 * (i >> 1)) : (uint32_t)(128 * half + 32 * i);
                    };
                    uint32_t pa[16], pb[16];
                    tmem_ld16u(tb + col_of(0), pa);
                    // the scales are in registers and the block's MMAs are complete: the stage,
                    // scale slot included, can be refilled
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t(&cur)[16] = (j & 1) ? pb : pa;
                        uint32_t(&nxt)[16] = (j & 1) ? pa : pb;
                        if (j < 7) tmem_ld16u(tb + col_of((j + 1) >> 1) + 16 * ((j + 1) & 1), nxt);
                        const int i = j >> 1;
                        const float c = (GU && (i & 1)) ? c1 : c0;
                        const int base = 2 * (GU ? ((i & 1) * 32 + (i >> 1) * 16) : 16 * i) + 16 * (j & 1);
#pragma unroll
                        for (int q = 0; q < 16; q += 2) fma2(acc[base + q], acc[base + q + 1], cur[q], cur[q + 1], c);
                        if (j < 7) tmem_wait_ld();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[buf]);
                } else {
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[slot]);
                        mbar_arrive(&tempty[buf]);
                    }
                }
                if (++buf == 2) { buf = 0; tphase ^= 1u; }
                if (++slot == STAGES) slot = 0;
            }

            if (GU) {
                // ------------------------------------------ SiLU(g)*u, 1x128 E4M3 quantisation of h
                // this thread: features [64h, 64h+64) of the 128-feature tile; gate in acc[0..63],
                // up in acc[64..127]
                float h[64];
                float amax = 0.f;
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    h[e] = silu_mul(acc[e], acc[64 + e]);
                    amax = fmaxf(amax, fabsf(h[e]));
                }
                amax_x[(half * 4 + quarter) * 32 + lane] = amax;
                named_bar_sync(1, EPI_WARPS * 32);
                const float mx = fmaxf(amax, amax_x[((1 - half) * 4 + quarter) * 32 + lane]);
                const float sc = (mx > 0.f) ? __fdiv_rn(mx, 448.0f) : 1.0f;
                // h / s as h * (1/s): within one ulp of the rounded quotient, far inside
                // the E4M3 code spacing, so a code can differ only for h at a rounding
                // midpoint of the code grid
                const float rs = __frcp_rn(sc);
                if (rv) {
                    uint8_t* dst = a.hq + act_offset(un.wb, un.row_begin + r, a.ld);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {                 // 16-byte chunks 4h .. 4h+3
                        uint32_t w4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int e = c4 * 16 + k * 4;
                            w4[k] = pack4_e4m3(h[e] * rs, h[e + 1] * rs, h[e + 2] * rs, h[e + 3] * rs);
                        }
                        const int chunk = (half * 4 + c4) ^ (r & 7);     // row_begin is a multiple of 8
                        *reinterpret_cast<uint4*>(dst + chunk * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    if (half == 0) a.shT[(size_t)un.wb * a.ld + un.row_begin + r] = sc;
                }
                named_bar_sync(1, EPI_WARPS * 32);
            } else {
                // ------------------------------------------ fp32 expert output rows: 128 features
                // Through the warp's staging tile, 16 columns at a time: each lane writes its
                // row's 16 values, then lane l stores row 8p + l/4, columns 4(l%4)..+3, so one
                // store instruction covers 8 rows x 64 contiguous bytes (full sectors) instead
                // of 32 rows x 16 bytes.
                float* stg = stg_all + (size_t)ew * 32 * STG_STRIDE;
                const bool wr = half == 0 || two;
                float* dst0 = a.out + (size_t)un.row_begin * a.M + (size_t)un.wb * BN + half * HALF + 4 * (lane & 3);
#pragma unroll
                for (int c0 = 0; c0 < HALF; c0 += 16) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        *reinterpret_cast<float4*>(stg + lane * STG_STRIDE + 4 * i) =
                            make_float4(acc[c0 + 4 * i], acc[c0 + 4 * i + 1], acc[c0 + 4 * i + 2], acc[c0 + 4 * i + 3]);
                    __syncwarp();
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const int rr = 8 * p + (lane >> 2);
                        const float4 v = *reinterpret_cast<const float4*>(stg + rr * STG_STRIDE + 4 * (lane & 3));
                        const int row = quarter * 32 + rr;
                        if (wr && row < un.valid) *reinterpret_cast<float4*>(dst0 + (size_t)row * a.M + c0) = v;
                    }
                    __syncwarp();
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
        cudaError_t e = ensure_smem_limit<expert_tc_kernel<GU>>(SMEM + 1024);
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
    return launch_pdl(expert_tc_kernel<GU>, dim3(L->num_sms), dim3(NTHREADS), SMEM + 1024, s, a);
}

// Weight-scale records, built once at load time from the repacked scales:
// one 16-byte record per (group, weight block, k block), so each stage
// fetches its weight scales with one bulk copy.
__global__ void scale_records_kernel(const float* __restrict__ s_gu, const float* __restrict__ s_dn, int G, int IT,
                                     int HT, float4* __restrict__ r_gu, float4* __restrict__ r_dn) {
    const int NBD = (HT + 1) / 2;
    const size_t n_gu = (size_t)G * IT * HT, n_dn = (size_t)G * NBD * IT;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n_gu + n_dn; i += (size_t)gridDim.x * blockDim.x) {
        if (i < n_gu) {
            r_gu[i] = make_float4(s_gu[2 * i], s_gu[2 * i + 1], 0.f, 0.f);
        } else {
            const size_t j = i - n_gu;                 // (g, b, kb), kb fastest
            const int kb = (int)(j % IT);
            const int b = (int)((j / IT) % NBD);
            const size_t g = j / ((size_t)IT * NBD);
            const float lo = s_dn[(g * HT + 2 * b) * IT + kb];
            const float hi = (2 * b + 1 < HT) ? s_dn[(g * HT + 2 * b + 1) * IT + kb] : 0.f;
            r_dn[j] = make_float4(lo, hi, 0.f, 0.f);
        }
    }
}

}  // namespace tc

int tc_tile_n() { return tc::BM; }

cudaError_t launch_tc_scale_records(const moe_layer* L, cudaStream_t s) {
    const int G = L->n_groups_max, IT = L->d.inter / QB, HT = L->d.hidden / QB;
    tc::scale_records_kernel<<<4 * L->num_sms, 256, 0, s>>>(L->s_gu, L->s_dn, G, IT, HT,
                                                           reinterpret_cast<float4*>(L->r_gu),
                                                           reinterpret_cast<float4*>(L->r_dn));
    return cudaGetLastError();
}

cudaError_t launch_expert_tc_gate_up(const moe_layer* L, int T, const WsLayout& lay, char* ws, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return tc::launch<true>(L, lay, ws, s);
}

cudaError_t launch_expert_tc_down(const moe_layer* L, int T, const WsLayout& lay, char* ws, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return tc::launch<false>(L, lay, ws, s);
}

}  // namespace moe
