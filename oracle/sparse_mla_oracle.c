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
 *  - Same page, Summary and Test plan: the fused producer step. RoPE on the
 *    pre-RoPE q_pe and k_pe at each token's position (neox or GPT-J pairing),
 *    q_out = concat(ql_nope, RoPE(q_pe)) in bf16, or its scaled_fp8_quant
 *    with a per-tensor q_scale, and the cache row concat(kv_c, RoPE(k_pe)).
 *    The unfused chain stores the rotated values as bf16 before any
 *    quantization, so the rotation is rounded to bf16 first.
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
 * Readings for the producer step (the page gives no formula): the rotation
 * of a pair (a, b) by angle theta is (a cos - b sin, b cos + a sin); neox
 * pairs element i with i + R/2, GPT-J pairs 2i with 2i + 1; the cos/sin cache
 * row of a position holds cos(theta_0..theta_{R/2-1}) then the sines, as
 * binary32; the rotation is done in fp64 and rounded once to bf16 (mode 0),
 * or, where its bf16 value decides an fp8 code, mirrored in binary32 with
 * each product and the difference or sum rounded (mode 1), the precision the
 * device computes it in. A position outside [0, max_position) leaves the
 * token's outputs unwritten; slot -1 skips the cache row.
 *
 * Attention sinks ("Enable AITER sparse MLA on gfx942, including FP8 KV",
 * Limitations: sinks are passed through; the page gives no formula). Reading:
 * a per-head sink logit, in the units of scale * q.k, joins the softmax
 * denominator and has no value row: out = sum_i e^{s_i} v_i / (e^{sink} +
 * sum_j e^{s_j}), lse = log(e^{sink} + sum_j e^{s_j}); a row with no valid
 * index gives out = 0 and lse = sink.
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
/* The fused producer step (RoPE + q concat + cache write).                 */
/* ------------------------------------------------------------------------ */

/* bf16 bits of the binary32 value x, rounded to nearest even. */
static uint16_t float_to_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* bf16 bits of the binary64 value x, rounded to nearest even directly (no
 * intermediate binary32 rounding): keep 8 significant bits. */
static uint16_t double_to_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0u;
    if (x == 0.0)
        return signbit(x) ? 0x8000u : 0x0000u;
    double a = fabs(x);
    int e;
    frexp(a, &e);                       /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                      /* spacing of 8-bit significands at this binade */
    if (q < -133)
        q = -133;                       /* bf16 subnormal spacing 2^-133 */
    double r = ldexp(nearbyint(ldexp(a, -q)), q); /* default rounding: to nearest even */
    if (r > 3.3895313892515355e38)     /* above the largest finite bf16: infinity */
        r = INFINITY;
    float f = (float)r;                 /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)((u >> 16) | (signbit(x) ? 0x8000u : 0u));
}

/* Rotary embedding of x[0..R) with cos[0..R/2), sin[0..R/2), in fp64. */
void oracle_rope_f64(const double *x, int R, const double *cs, const double *sn, int is_neox, double *out)
{
    const int half = R / 2;
    for (int i = 0; i < half; ++i) {
        const int ia = is_neox ? i : 2 * i;
        const int ib = is_neox ? i + half : 2 * i + 1;
        const double a = x[ia], b = x[ib];
        out[ia] = a * cs[i] - b * sn[i];
        out[ib] = b * cs[i] + a * sn[i];
    }
}

/* One rotated pair as bf16 bits: mode 0 = fp64 rotation rounded once; mode 1 =
 * binary32 products and difference/sum, each rounded, then rounded to bf16. */
static void rope_pair_bf16(float a, float b, float c, float sn, int mode, uint16_t *oa, uint16_t *ob)
{
    if (mode == 0) {
        *oa = double_to_bf16_rne((double)a * c - (double)b * sn);
        *ob = double_to_bf16_rne((double)b * c + (double)a * sn);
    } else {
        volatile float p0 = a * c, p1 = b * sn, p2 = b * c, p3 = a * sn;
        volatile float ra = p0 - p1, rb = p2 + p3;
        *oa = float_to_bf16_rne(ra);
        *ob = float_to_bf16_rne(rb);
    }
}

/* One output row of Dn + Dr values: nope[0..Dn) copied, rope[0..Dr) rotated at
 * row `cs_row` of the cos/sin cache; stored as bf16 bits (fp8 == 0) or as the
 * E4M3 codes of bf16 / scale in binary32 (fp8 == 1). */
static void producer_row(const uint16_t *nope, int Dn, const uint16_t *rope, int Dr, const float *cs_row,
                         int is_neox, int mode, int fp8, float scale, void *dst)
{
    uint16_t tmp[4096];
    for (int d = 0; d < Dn; ++d)
        tmp[d] = nope[d];
    const int half = Dr / 2;
    for (int i = 0; i < half; ++i) {
        const int ia = is_neox ? i : 2 * i;
        const int ib = is_neox ? i + half : 2 * i + 1;
        rope_pair_bf16(bf16_to_float(rope[ia]), bf16_to_float(rope[ib]), cs_row[i], cs_row[half + i], mode,
                       &tmp[Dn + ia], &tmp[Dn + ib]);
    }
    const int D = Dn + Dr;
    if (!fp8) {
        memcpy(dst, tmp, (size_t)D * sizeof(uint16_t));
    } else {
        uint8_t *o = (uint8_t *)dst;
        for (int d = 0; d < D; ++d) {
            volatile float x = bf16_to_float(tmp[d]);
            float y = x / scale;
            o[d] = oracle_e4m3_encode(y);
        }
    }
}

/* The whole step over contiguous inputs: ql_nope [T,H,Dn], q_pe [T,H,Dr],
 * kv_c [T,Dn], k_pe [T,Dr] (bf16 bits), positions [T], cos_sin
 * [max_pos, Dr] binary32. q_out [T,H,Dn+Dr] (bf16 bits or E4M3 codes);
 * cache [num_slots, Dn+Dr] (bf16 bits or E4M3 codes) row slot_mapping[t]
 * (negative: skipped). Returns the number of tokens whose position or slot
 * was out of range (their outputs are left unwritten). */
int64_t oracle_fused_qk_rope_cache(const uint16_t *ql_nope, const uint16_t *q_pe, const uint16_t *kv_c,
                                   const uint16_t *k_pe, const int64_t *positions, const float *cos_sin,
                                   int64_t max_pos, int is_neox, const int64_t *slot_mapping, void *cache,
                                   int cache_fp8, int64_t num_slots, float kv_scale, void *q_out, int q_out_fp8,
                                   float q_scale, int T, int H, int Dn, int Dr, int mode)
{
    int64_t bad = 0;
    const int D = Dn + Dr;
    if (D > 4096 || Dr % 2 != 0)
        return -1;
    e4m3_init();
#pragma omp parallel for reduction(+ : bad) schedule(static)
    for (int t = 0; t < T; ++t) {
        const int64_t pos = positions[t];
        if (pos < 0 || pos >= max_pos) {
            bad += 1;
            continue;
        }
        const float *cs_row = cos_sin + pos * (int64_t)Dr;
        for (int h = 0; h < H; ++h) {
            const int64_t r = (int64_t)t * H + h;
            void *dst = q_out_fp8 ? (void *)((uint8_t *)q_out + r * D) : (void *)((uint16_t *)q_out + r * D);
            producer_row(ql_nope + r * Dn, Dn, q_pe + r * Dr, Dr, cs_row, is_neox, mode, q_out_fp8, q_scale, dst);
        }
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            bad += 1;
            continue;
        }
        void *dst = cache_fp8 ? (void *)((uint8_t *)cache + slot * D) : (void *)((uint16_t *)cache + slot * D);
        producer_row(kv_c + (int64_t)t * Dn, Dn, k_pe + (int64_t)t * Dr, Dr, cs_row, is_neox, mode, cache_fp8,
                     kv_scale, dst);
    }
    return bad;
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
static int64_t sparse_mla_core(const uint16_t *q, const double *qf, const void *kv, int kv_is_fp8,
                               float kv_scale, const int32_t *indices,
                               int T, int H, int D_qk, int D_v, int64_t num_slots,
                               int topk, float scale, int q_mode, const float *sinks,
                               double *out, double *lse, int nthreads);

int64_t oracle_sparse_mla(const uint16_t *q, const void *kv, int kv_is_fp8,
                          float kv_scale, const int32_t *indices,
                          int T, int H, int D_qk, int D_v, int64_t num_slots,
                          int topk, float scale, int q_mode,
                          double *out, double *lse, int nthreads)
{
    return sparse_mla_core(q, NULL, kv, kv_is_fp8, kv_scale, indices, T, H, D_qk, D_v, num_slots, topk, scale,
                           q_mode, NULL, out, lse, nthreads);
}

/* The forward with per-head sink logits sinks[H] (see the reading above);
 * sinks == NULL is the plain forward. q as in oracle_sparse_mla (q != NULL)
 * or as fp64 values (qf != NULL). */
int64_t oracle_sparse_mla_sinks(const uint16_t *q, const double *qf, const void *kv, int kv_is_fp8,
                                float kv_scale, const int32_t *indices,
                                int T, int H, int D_qk, int D_v, int64_t num_slots,
                                int topk, float scale, int q_mode, const float *sinks,
                                double *out, double *lse, int nthreads)
{
    return sparse_mla_core(q, qf, kv, kv_is_fp8, kv_scale, indices, T, H, D_qk, D_v, num_slots, topk, scale,
                           q_mode, sinks, out, lse, nthreads);
}

/*
 * The same forward with q given as the values that enter the dots, fp64
 * [T, H, D_qk]: a pre-quantized q is its E4M3 codes times its per-tensor
 * scale ("Enable AITER sparse MLA on gfx942, including FP8 KV", Details,
 * "FP8 KV on gfx942": gfx950 keeps the pre-quantized q).
 */
int64_t oracle_sparse_mla_qf64(const double *qf, const void *kv, int kv_is_fp8,
                               float kv_scale, const int32_t *indices,
                               int T, int H, int D_qk, int D_v, int64_t num_slots,
                               int topk, float scale, double *out, double *lse, int nthreads)
{
    return sparse_mla_core(NULL, qf, kv, kv_is_fp8, kv_scale, indices, T, H, D_qk, D_v, num_slots, topk, scale,
                           0, NULL, out, lse, nthreads);
}

static int64_t sparse_mla_core(const uint16_t *q, const double *qf, const void *kv, int kv_is_fp8,
                               float kv_scale, const int32_t *indices,
                               int T, int H, int D_qk, int D_v, int64_t num_slots,
                               int topk, float scale, int q_mode, const float *sinks,
                               double *out, double *lse, int nthreads)
{
    int64_t bad = 0;
    e4m3_init();
    /* the thread count applies to this call alone (no process-wide setting) */
#ifdef _OPENMP
    const int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    const int nt = 1;
    (void)nthreads;
#endif
#pragma omp parallel reduction(+ : bad) num_threads(nt)
    {
        double *qv = (double *)malloc(sizeof(double) * (size_t)D_qk);
        double *s = (double *)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
        int64_t *sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)(topk > 0 ? topk : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t th = 0; th < (int64_t)T * H; ++th) {
            int64_t t = th / H;
            const uint16_t *qrow = q ? q + th * (int64_t)D_qk : NULL;
            double *orow = out + th * (int64_t)D_v;

            /* the q row as it enters the dots */
            if (qf != NULL) {
                for (int d = 0; d < D_qk; ++d)
                    qv[d] = qf[th * (int64_t)D_qk + d];
            } else if (q_mode == 1) {
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
            /* the head's sink logit (-inf: none) */
            const double sink = sinks ? (double)sinks[th % H] : -INFINITY;
            if (n == 0) {
                for (int d = 0; d < D_v; ++d)
                    orow[d] = 0.0;
                lse[th] = sink;
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
            /* softmax normaliser (the sink joins it) and lse */
            if (sink > m)
                m = sink;
            double l = (sink == -INFINITY) ? 0.0 : exp(sink - m);
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
