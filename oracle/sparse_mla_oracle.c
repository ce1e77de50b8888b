/*
 * Sparse MLA forward: the plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file. Only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it. It shares no code, header, table or helper with the
 * CUDA library; the only thing both sides share is the seeded input generator.
 *
 * What it computes (sources, by page title and section):
 *
 *  - "Enable AITER sparse MLA on gfx942, including FP8 KV" (vLLM PR 60583),
 *    Overview / Details: sparse MLA over a rope-free latent cache, bf16 or fp8
 *    KV; with fp8 KV the q side is quantized per tile inside the kernel and the
 *    dots run in fp8 ("FP8 KV on gfx942"); the error envelope of that mode is
 *    given under "Numerics".
 *  - "Fuse decode QK-RoPE + Q-concat + KV-concat + KV-cache write for sparse
 *    MLA" (vLLM PR 47757), Test plan: the cache row is the latent part
 *    followed by the rope part; fp8 storage follows the scaled_fp8_quant
 *    convention, stored = x / scale, dequantized = code * scale.
 *  - The forward itself: for each query row t and head h, gather the rows
 *    named by indices[t] (-1 = masked) from the head-shared cache, logits
 *    s_i = scale * q[t,h] . kv[idx_i][:D_qk], softmax over the valid i,
 *    out[t,h] = sum_i p_i kv[idx_i][:D_v], lse[t,h] = log sum_i exp(s_i).
 *
 * Everything is fp64 except the two places where the method itself fixes a
 * float32 step: the scale division amax/448 and the quantization x/scale,
 * which decide integer codes and are therefore done in IEEE binary32 on both
 * sides. The e4m3 codec is written from the OCP 8-bit floating point format
 * definition (E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, largest finite 448).
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes): lse is the natural log of sum exp(scale * q.k); a row with no valid
 * index gives out = 0 and lse = -inf; an index < -1 or >= num_slots breaks the
 * contract and is treated as masked; duplicate indices each count; the q
 * "tile" of the fp8 mode is one (t, h) row of D_qk values with
 * s_q = amax/448 (1.0 when amax == 0); the per-tensor kv scale is
 * amax/448 over the whole source (1.0 when amax == 0); NaN is ignored by amax.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (no fast-math; IEEE semantics needed).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16: the top 16 bits of an IEEE binary32. Widening is exact.            */
/* ------------------------------------------------------------------------ */
static float bf16_to_float(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------ */
/* OCP E4M3 ("fn": finite + NaN) codec, from the format definition.         */
/* ------------------------------------------------------------------------ */

/* Value of an E4M3 code. exponent field 0 -> subnormal m/8 * 2^(1-7);
 * exponent field 15 with mantissa 7 -> NaN; otherwise (1 + m/8) * 2^(e-7). */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* The 127 non-negative finite magnitudes, by code 0x00..0x7E (ascending). */
static double g_e4m3_mag[127];
static int g_e4m3_ready = 0;

static void e4m3_init(void)
{
    if (g_e4m3_ready)
        return;
    for (int c = 0; c < 127; ++c)
        g_e4m3_mag[c] = oracle_e4m3_decode((uint8_t)c);
    g_e4m3_ready = 1;
}

/* Round-to-nearest-even onto the E4M3 grid, saturating to +-448 ("satfinite"):
 * the code whose value is nearest to x; on a tie, the code with an even
 * mantissa (even code). NaN -> 0x7F. */
uint8_t oracle_e4m3_encode(float x)
{
    e4m3_init();
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= g_e4m3_mag[126])
        return sign | 0x7E;
    /* largest code lo with mag[lo] <= a (binary search on the ascending grid) */
    int lo = 0, hi = 126;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (g_e4m3_mag[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    if (g_e4m3_mag[hi] <= a)
        lo = hi;
    int pick = lo;
    if (lo < 126) {
        double dlo = a - g_e4m3_mag[lo];
        double dhi = g_e4m3_mag[lo + 1] - a;
        if (dhi < dlo)
            pick = lo + 1;
        else if (dhi == dlo)
            pick = (lo % 2 == 0) ? lo : lo + 1;
    }
    return sign | (uint8_t)pick;
}

/* amax(|x|) over bf16 values, NaN ignored. Exact (max of exact values). */
float oracle_amax_bf16(const uint16_t *x, int64_t n)
{
    float amax = 0.0f;
#pragma omp parallel for reduction(max : amax) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float v = fabsf(bf16_to_float(x[i]));
        if (v > amax) /* false for NaN */
            amax = v;
    }
    return amax;
}

/* Per-tensor fp8 scale from an amax: amax / 448 in binary32; 1.0 if amax == 0. */
float oracle_fp8_scale_from_amax(float amax)
{
    volatile float a = amax; /* keep the division in binary32 */
    if (a == 0.0f)
        return 1.0f;
    return a / 448.0f;
}

float oracle_fp8_scale(const uint16_t *x, int64_t n)
{
    return oracle_fp8_scale_from_amax(oracle_amax_bf16(x, n));
}

/* Quantize src[N, D] (bf16) into cache[slot_mapping[n], :] as E4M3 codes of
 * x / kv_scale (binary32 division). slot -1 skips the row; a slot outside
 * [0, num_slots) also skips (contract violation). Returns rows written. */
int64_t oracle_fp8_cache_write(const uint16_t *src, const int64_t *slot_mapping,
                               int64_t N, int D, float kv_scale,
                               uint8_t *cache, int64_t num_slots)
{
    int64_t written = 0;
    e4m3_init();
#pragma omp parallel for reduction(+ : written) schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0 || slot >= num_slots)
            continue;
        for (int d = 0; d < D; ++d) {
            volatile float x = bf16_to_float(src[n * (int64_t)D + d]);
            float y = x / kv_scale;
            cache[slot * (int64_t)D + d] = oracle_e4m3_encode(y);
        }
        written += 1;
    }
    return written;
}

/* ------------------------------------------------------------------------ */
/* The sparse MLA forward.                                                  */
/* ------------------------------------------------------------------------ */

/* kv element (slot j, column d) as a double: bf16 widened exactly, or the
 * E4M3 value times kv_scale (exact in binary64: 4 x 24 significant bits). */
static double kv_value(const void *kv, int kv_is_fp8, double kv_scale,
                       int64_t j, int D_qk, int d)
{
    if (kv_is_fp8) {
        uint8_t c = ((const uint8_t *)kv)[j * (int64_t)D_qk + d];
        return oracle_e4m3_decode(c) * kv_scale;
    }
    return (double)bf16_to_float(((const uint16_t *)kv)[j * (int64_t)D_qk + d]);
}

/*
 * q        bf16 [T, H, D_qk]
 * kv       [num_slots, D_qk]: bf16 if kv_is_fp8 == 0, E4M3 codes otherwise
 * indices  int32 [T, topk]; -1 masked; any order; duplicates allowed
 * q_mode   0: q enters the dots as given (bf16, exact)
 *          1: q is first quantized per (t, h) row exactly as the fp8-dot mode
 *             prescribes: s_q = amax|q[t,h,:]| / 448 (1.0 if 0),
 *             q8 = E4M3(q / s_q), used value = q8 * s_q.
 * out      double [T, H, D_v]; lse double [T, H] (natural log, includes scale)
 * nthreads 0 = OpenMP default. Returns the number of out-of-range indices seen.
 */
int64_t oracle_sparse_mla(const uint16_t *q, const void *kv, int kv_is_fp8,
                          float kv_scale, const int32_t *indices,
                          int T, int H, int D_qk, int D_v, int64_t num_slots,
                          int topk, float scale, int q_mode,
                          double *out, double *lse, int nthreads)
{
    int64_t bad = 0;
    e4m3_init();
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#endif
#pragma omp parallel reduction(+ : bad)
    {
        double *qv = (double *)malloc(sizeof(double) * (size_t)D_qk);
        double *s = (double *)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
        int64_t *sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)(topk > 0 ? topk : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t th = 0; th < (int64_t)T * H; ++th) {
            int64_t t = th / H;
            const uint16_t *qrow = q + th * (int64_t)D_qk;
            double *orow = out + th * (int64_t)D_v;

            /* the q row as it enters the dots */
            if (q_mode == 1) {
                float amax = 0.0f;
                for (int d = 0; d < D_qk; ++d) {
                    float v = fabsf(bf16_to_float(qrow[d]));
                    if (v > amax)
                        amax = v;
                }
                float s_q = oracle_fp8_scale_from_amax(amax);
                for (int d = 0; d < D_qk; ++d) {
                    volatile float x = bf16_to_float(qrow[d]);
                    float y = x / s_q;
                    qv[d] = oracle_e4m3_decode(oracle_e4m3_encode(y)) * (double)s_q;
                }
            } else {
                for (int d = 0; d < D_qk; ++d)
                    qv[d] = (double)bf16_to_float(qrow[d]);
            }

            /* the selected rows, in index order (masked and invalid dropped) */
            int n = 0;
            for (int i = 0; i < topk; ++i) {
                int64_t j = indices[t * (int64_t)topk + i];
                if (j == -1)
                    continue;
                if (j < -1 || j >= num_slots) {
                    if (th % H == 0)
                        bad += 1;
                    continue;
                }
                sel[n++] = j;
            }
            if (n == 0) {
                for (int d = 0; d < D_v; ++d)
                    orow[d] = 0.0;
                lse[th] = -INFINITY;
                continue;
            }

            /* logits */
            double m = -INFINITY;
            for (int i = 0; i < n; ++i) {
                double acc = 0.0;
                for (int d = 0; d < D_qk; ++d)
                    acc += qv[d] * kv_value(kv, kv_is_fp8, kv_scale, sel[i], D_qk, d);
                s[i] = (double)scale * acc;
                if (s[i] > m)
                    m = s[i];
            }
            /* softmax normaliser and lse */
            double l = 0.0;
            for (int i = 0; i < n; ++i)
                l += exp(s[i] - m);
            lse[th] = m + log(l);
            /* weighted sum of the value rows (first D_v columns) */
            for (int d = 0; d < D_v; ++d)
                orow[d] = 0.0;
            for (int i = 0; i < n; ++i) {
                double p = exp(s[i] - m) / l;
                for (int d = 0; d < D_v; ++d)
                    orow[d] += p * kv_value(kv, kv_is_fp8, kv_scale, sel[i], D_qk, d);
            }
        }
        free(qv);
        free(s);
        free(sel);
    }
    return bad;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
