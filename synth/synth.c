/*
 * Seeded synthetic inputs for the routed-expert MoE FFN layer.
 *
 * This module only PRODUCES inputs: activations, router weights and FP8
 * expert weights in the checkpoint format the layer consumes (E4M3FN codes
 * plus one fp32 multiplier per 128x128 block).  It holds none of the
 * layer's arithmetic.  Both the CUDA path and the CPU oracle read the bytes
 * written here, so they see exactly the same inputs.
 *
 * Randomness is counter based: every value is a pure function of
 * (seed, stream, element index), so any block of any tensor can be
 * regenerated on its own, in any order, on any number of threads, on x86 or
 * Arm, with bit-identical results (integer arithmetic plus exact fp64 sums;
 * no libm call).
 *
 * Normal variates use the Irwin-Hall construction: the sum of twelve
 * independent U(0,1) draws minus 6 has mean 0 and variance 1 and is the
 * classic libm-free approximation of N(0,1) (tails bounded at +-6 sigma).
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>

#define SYNTH_API __attribute__((visibility("default")))

static inline uint64_t mix64(uint64_t z) {
    /* SplitMix64 output function (Steele, Lea, Flood 2014). */
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27; z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed * 0x9E3779B97F4A7C15ull + stream * 0xD1B54A32D192ED03ull + 1ull);
}

static inline uint64_t draw(uint64_t key, uint64_t idx, uint64_t j) {
    return mix64(key + (idx * 4ull + j + 1ull) * 0x9E3779B97F4A7C15ull);
}

/* One N(0,1) variate (Irwin-Hall, 12 uniforms of 16 bits) for element idx.
 * Every partial sum is a multiple of 2^-17 below 12, so the fp64 sum is exact. */
static inline double normal_at(uint64_t key, uint64_t idx) {
    double acc = 0.0;
    for (uint64_t j = 0; j < 3; ++j) {
        uint64_t r = draw(key, idx, j);
        for (int b = 0; b < 4; ++b) {
            uint32_t u = (uint32_t)((r >> (16 * b)) & 0xFFFFu);
            acc += ((double)u + 0.5) * (1.0 / 65536.0);
        }
    }
    return acc - 6.0;
}

static inline uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* float -> bf16 bits, round to nearest even (inputs here are always finite). */
static inline uint16_t to_bf16_rne(float f) {
    uint32_t u = f32_bits(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ---- E4M3FN encoder used only to write the weight checkpoint ----------
 * Table of the 127 non-negative finite code values, searched by bisection,
 * ties to the even code, saturating at 448.  */
static double g_e4m3_pos[127];
static int g_e4m3_ready = 0;

static void e4m3_table_init(void) {
    if (g_e4m3_ready) return;
    for (int c = 0; c < 127; ++c) {
        int e = c >> 3, m = c & 7;
        g_e4m3_pos[c] = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    }
    g_e4m3_ready = 1;
}

static uint8_t e4m3_from_float(float v) {
    uint8_t sign = (f32_bits(v) >> 31) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 126;
    int lo = 0, hi = 126;             /* invariant: table[lo] <= a < table[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (g_e4m3_pos[mid] <= a) lo = mid; else hi = mid;
    }
    double mid = 0.5 * (g_e4m3_pos[lo] + g_e4m3_pos[hi]);
    int c;
    if (a < mid) c = lo; else if (a > mid) c = hi; else c = (lo & 1) ? hi : lo;
    return sign | (uint8_t)c;
}

/* ---- public entry points ------------------------------------------------ */

/* out[i] = bf16(std * N(0,1)) for i in [0, n). */
SYNTH_API void synth_bf16_normal(uint64_t seed, uint64_t stream, int64_t n, double std_, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = to_bf16_rne((float)(std_ * normal_at(key, (uint64_t)i)));
}

/* out[i] = fp32(std * N(0,1)). */
SYNTH_API void synth_f32_normal(uint64_t seed, uint64_t stream, int64_t n, double std_, float* out) {
    uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(std_ * normal_at(key, (uint64_t)i));
}

/* A random permutation of 0..n-1 (Fisher-Yates driven by the counter stream). */
SYNTH_API void synth_permutation(uint64_t seed, uint64_t stream, int32_t n, int32_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int32_t i = 0; i < n; ++i) out[i] = i;
    for (int32_t i = n - 1; i > 0; --i) {
        uint64_t j = draw(key, (uint64_t)i, 0) % (uint64_t)(i + 1);
        int32_t t = out[i]; out[i] = out[j]; out[j] = t;
    }
}

/* FP8 checkpoint for n_mat matrices of [rows][cols] (rows, cols multiples of
 * 128).  The dense weight is W = fp32(std * N(0,1)); for each 128x128 block
 * the stored multiplier is s = amax/448 (s = 1 for an all-zero block) and the
 * stored code is E4M3FN(W/s).  Output layouts:
 *   q [n_mat][rows][cols]            (row-major, one byte per weight)
 *   s [n_mat][rows/128][cols/128]    (fp32)
 * Element (m, r, c) draws counter index (m*rows + r)*cols + c. */
SYNTH_API int synth_fp8_blocks(uint64_t seed, uint64_t stream, int32_t n_mat, int32_t rows, int32_t cols,
                               double std_, uint8_t* q, float* s) {
    if (rows % 128 || cols % 128 || n_mat <= 0) return -1;
    e4m3_table_init();
    uint64_t key = stream_key(seed, stream);
    const int64_t rb = rows / 128, cb = cols / 128;
    const int64_t nblk = (int64_t)n_mat * rb * cb;
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t b = 0; b < nblk; ++b) {
        int64_t m = b / (rb * cb), rem = b % (rb * cb);
        int64_t br = rem / cb, bc = rem % cb;
        float buf[128 * 128];
        float amax = 0.0f;
        for (int r = 0; r < 128; ++r) {
            int64_t row = br * 128 + r;
            uint64_t base = (uint64_t)((m * rows + row) * cols + bc * 128);
            for (int c = 0; c < 128; ++c) {
                float w = (float)(std_ * normal_at(key, base + (uint64_t)c));
                buf[r * 128 + c] = w;
                float a = fabsf(w);
                if (a > amax) amax = a;
            }
        }
        float sc = (amax > 0.0f) ? amax / 448.0f : 1.0f;
        s[b] = sc;
        for (int r = 0; r < 128; ++r) {
            int64_t row = br * 128 + r;
            uint8_t* dst = q + (m * rows + row) * (int64_t)cols + bc * 128;
            for (int c = 0; c < 128; ++c) dst[c] = e4m3_from_float(buf[r * 128 + c] / sc);
        }
    }
    return 0;
}

SYNTH_API int synth_version(void) { return 1; }
