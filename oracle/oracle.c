/*
 * Paged KV-cache attention oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of what the paged decode / prefill
 * path computes.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library.  It shares no code, header or
 * constant with the CUDA library; the product path never calls it.
 *
 * Sources (page title, section):
 *  [KVC-ES] "La caché de claves y valores: cuánto cuesta cada token"
 *           (gustavoai.dev), section "Las claves y los valores de una
 *           posición no cambian": row t of the output is the unmasked softmax
 *           of q_t against all t cached keys (its own included) applied to
 *           the t cached values; the new k_t, v_t are appended to the end of
 *           each head's cache before the attention step (step 2, then 3).
 *  [ATT-DE] "Aufmerksamkeit" feed (chatgpz.de), linear-attention article,
 *           class TraditionalAttention: scores = Q K^T / sqrt(d_k), softmax
 *           over the last axis, times V.
 *  [PA-DE]  same feed, PagedAttention article, SECTION 2 "Pages + Block
 *           Table": a block table maps logical page index -> physical page
 *           id, PAGE_SIZE tokens per page.
 *  [XF-DE]  same feed, xformers article, parts 4 (variable-length packed
 *           batch, BlockDiagonalMask / BlockDiagonalCausalMask) and 5
 *           (grouped-query attention, BMGHK: G KV heads, each shared by a
 *           contiguous group of query heads).
 *  [FA-DE]  same feed, FlashAttention article, "Was ist der mathematische
 *           Aspekt von Softmax?": per block keep the row maximum and the sum
 *           of exponentials; when merging, rescale both by
 *           e^(block max - global max).
 *
 * Every floating-point step is fp64.  fp16 inputs are passed as their IEEE
 * binary16 bit patterns and widened exactly.
 *
 * Parity pins (tests/test_oracle_*.py): brute-force full causal attention,
 * torch's float64 scaled_dot_product_attention, closed forms (one-token
 * context, identical keys, two-token logistic form), block-permutation and
 * prefix-sharing invariance, GQA == replicated-head MHA, and exhaustive
 * binary16 widening against numpy.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- IEEE 754 binary16 -> double, exact (sign, 5-bit exponent bias 15,
 *      10-bit fraction; subnormals scaled by 2^-24). ---- */
double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x400), expo - 25);
    }
    return sign ? -v : v;
}

void oracle_half_array_to_double(const uint16_t* src, double* dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_half_to_double(src[i]);
}

/* ---- fp8 e4m3 (the quantized-cache extension; the pages fix no KV format) ----
 * 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; exponent field 0 holds the
 * subnormals m * 2^-9 (m = 0..7); no infinities; exponent 15 with fraction 7 is NaN,
 * so the largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t c) {
    int sign = (c >> 7) & 1, expo = (c >> 3) & 0xf, frac = c & 7;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -9);
    } else if (expo == 15 && frac == 7) {
        v = NAN;
    } else {
        v = ldexp((double)(8 + frac), expo - 10);
    }
    return sign ? -v : v;
}

/* Round to the nearest e4m3 value, ties to the even fraction, magnitudes past 448 saturating to 448. */
uint8_t oracle_e4m3_from_float(float x) {
    if (isnan(x)) return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7e;
    if (a < ldexp(1.0, -6)) {                 /* subnormal range: steps of 2^-9 */
        double m = nearbyint(ldexp(a, 9));    /* default rounding: to nearest, ties to even */
        return sign | (uint8_t)m;             /* m == 8 is 2^-6, the first normal: code 0x08 */
    }
    int e2;
    frexp(a, &e2);                            /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;                           /* unbiased exponent, -6 .. 8 */
    double m = nearbyint(ldexp(a, 3 - E));    /* 8 .. 16 */
    if (m == 16.0) {
        m = 8.0;
        E += 1;
    }
    int code = ((E + 7) << 3) | ((int)m - 8);
    if (code > 0x7e) code = 0x7e;
    return sign | (uint8_t)code;
}

/* Quantize rows of D binary16 values: scale = absmax / 448 in binary32 (1 for an all-zero row),
 * code_i = e4m3(x_i / scale) with the quotient in binary32.  codes [rows][D], scales [rows]. */
void oracle_quantize_fp8(const uint16_t* x, int64_t rows, int D, uint8_t* codes, float* scales) {
    for (int64_t r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < D; ++c) {
            float v = (float)fabs(oracle_half_to_double(x[r * D + c]));
            if (v > amax) amax = v;
        }
        float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        scales[r] = s;
        for (int c = 0; c < D; ++c) codes[r * D + c] = oracle_e4m3_from_float((float)oracle_half_to_double(x[r * D + c]) / s);
    }
}

/* ---- a tiny static thread pool: run fn(i, ctx) for i in [0, n) ---- */
typedef void (*task_fn)(int64_t, void*);
typedef struct {
    task_fn fn;
    void* ctx;
    int64_t begin, end;
} span_t;

static void* run_span(void* p) {
    span_t* s = (span_t*)p;
    for (int64_t i = s->begin; i < s->end; ++i) s->fn(i, s->ctx);
    return NULL;
}

static void parallel_for(int64_t n, int nthreads, task_fn fn, void* ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) {
        for (int64_t i = 0; i < n; ++i) fn(i, ctx);
        return;
    }
    pthread_t th[256];
    span_t sp[256];
    for (int t = 0; t < nthreads; ++t) {
        sp[t].fn = fn;
        sp[t].ctx = ctx;
        sp[t].begin = n * t / nthreads;
        sp[t].end = n * (t + 1) / nthreads;
        pthread_create(&th[t], NULL, run_span, &sp[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* ---- softmax(q K^T * scale) V over n contiguous fp64 rows ([ATT-DE]) ----
 * q[D]; K, V: [n][D] with row stride ld; out[D].  x_j = scale * <q, k_j>,
 * m = max_j x_j, p_j = exp(x_j - m), o = sum_j p_j v_j / sum_j p_j. */
static void attend_row(const double* q, const double* K, const double* V, int64_t n, int D,
                       int64_t ld, double scale, double* x /* scratch [n] */, double* out) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double s = 0.0;
        for (int c = 0; c < D; ++c) s += q[c] * K[j * ld + c];
        x[j] = scale * s;
        if (x[j] > m) m = x[j];
    }
    double l = 0.0;
    for (int c = 0; c < D; ++c) out[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(x[j] - m);
        l += p;
        for (int c = 0; c < D; ++c) out[c] += p * V[j * ld + c];
    }
    for (int c = 0; c < D; ++c) out[c] /= l;
}

/* ======================================================================
 * Decode over a paged cache ([KVC-ES], [PA-DE], [XF-DE] part 5).
 *
 * q:            [B][Hq][D] binary16
 * k_cache/v_cache: one layer, [NB][Hkv][bs][D] binary16
 * block_table:  [B][max_blocks] physical block ids
 * context_lens: [B], the number of cached tokens INCLUDING the token
 *               appended in this step (it attends to itself)
 * out:          [B][Hq][D] fp64
 * Query head h reads KV head h / (Hq / Hkv).
 * Returns 0, or -1 when an index is out of range.
 * ====================================================================== */
typedef struct {
    const uint16_t *q, *k, *v;
    const uint8_t *kq, *vq;       /* fp8 cache instead of k, v when not NULL */
    const float *ks, *vs;         /* its per-row scales [NB][Hkv][bs] */
    const int32_t *table, *ctx;
    int max_blocks, B, Hq, Hkv, D, bs, NB;
    double scale;
    double* out;
    volatile int bad;
} decode_job;

static void decode_task(int64_t idx, void* p) {
    decode_job* J = (decode_job*)p;
    int b = (int)(idx / J->Hq), h = (int)(idx % J->Hq);
    int G = J->Hq / J->Hkv, hk = h / G, D = J->D;
    int64_t n = J->ctx[b];
    double* o = J->out + ((int64_t)b * J->Hq + h) * D;
    if (n < 1 || n > (int64_t)J->max_blocks * J->bs) {
        J->bad = 1;
        for (int c = 0; c < D; ++c) o[c] = 0.0;
        return;
    }
    /* gather this sequence's keys and values for KV head hk into contiguous rows */
    double* K = (double*)malloc(sizeof(double) * n * D);
    double* V = (double*)malloc(sizeof(double) * n * D);
    double* x = (double*)malloc(sizeof(double) * n);
    double qd[512];
    for (int64_t j = 0; j < n; ++j) {
        int32_t phys = J->table[(int64_t)b * J->max_blocks + j / J->bs];
        if (phys < 0 || phys >= J->NB) {
            J->bad = 1;
            phys = 0;
        }
        int64_t row = (((int64_t)phys * J->Hkv + hk) * J->bs + j % J->bs) * D;
        for (int c = 0; c < D; ++c) {
            if (J->kq) { /* dequantized: code value times the row's scale, exact in fp64 */
                K[j * D + c] = oracle_e4m3_to_double(J->kq[row + c]) * (double)J->ks[row / D];
                V[j * D + c] = oracle_e4m3_to_double(J->vq[row + c]) * (double)J->vs[row / D];
            } else {
                K[j * D + c] = oracle_half_to_double(J->k[row + c]);
                V[j * D + c] = oracle_half_to_double(J->v[row + c]);
            }
        }
    }
    for (int c = 0; c < D; ++c) qd[c] = oracle_half_to_double(J->q[((int64_t)b * J->Hq + h) * D + c]);
    attend_row(qd, K, V, n, D, D, J->scale, x, o);
    free(K);
    free(V);
    free(x);
}

int oracle_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                  const int32_t* block_table, int max_blocks, const int32_t* context_lens, int B,
                  int Hq, int Hkv, int D, int bs, int NB, double scale, double* out, int nthreads) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || D > 512 || bs <= 0) return -1;
    decode_job J = {q, k_cache, v_cache, NULL, NULL, NULL, NULL, block_table, context_lens, max_blocks, B, Hq,
                    Hkv, D, bs, NB, scale, out, 0};
    parallel_for((int64_t)B * Hq, nthreads, decode_task, &J);
    return J.bad ? -1 : 0;
}

/* Decode over an fp8 e4m3 cache with per-row scales (k_codes/v_codes [NB][Hkv][bs][D], scales [NB][Hkv][bs]):
 * every cached value is code value * scale; the rest is oracle_decode. */
int oracle_decode_fp8(const uint16_t* q, const uint8_t* k_codes, const uint8_t* v_codes, const float* k_scales,
                      const float* v_scales, const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                      int B, int Hq, int Hkv, int D, int bs, int NB, double scale, double* out, int nthreads) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || D > 512 || bs <= 0) return -1;
    decode_job J = {q, NULL, NULL, k_codes, v_codes, k_scales, v_scales, block_table, context_lens, max_blocks, B,
                    Hq, Hkv, D, bs, NB, scale, out, 0};
    parallel_for((int64_t)B * Hq, nthreads, decode_task, &J);
    return J.bad ? -1 : 0;
}

/* ======================================================================
 * Full causal self-attention on one contiguous sequence, written as the
 * n x n score matrix with -inf above the diagonal ([ATT-DE] plus the causal
 * mask of [KVC-ES]).  Q, K, V, O: [n][D] fp64.  This is the brute force that
 * the cached decode row must reproduce.
 * ====================================================================== */
int oracle_causal_attention(const double* Q, const double* K, const double* V, int n, int D,
                            double scale, double* O) {
    double* S = (double*)malloc(sizeof(double) * (size_t)n * n);
    if (!S) return -1;
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) {
            if (j > i) {
                S[(size_t)i * n + j] = -INFINITY;
                continue;
            }
            double s = 0.0;
            for (int c = 0; c < D; ++c) s += Q[i * D + c] * K[j * D + c];
            S[(size_t)i * n + j] = s * scale;
        }
    for (int i = 0; i < n; ++i) {
        double m = -INFINITY, l = 0.0;
        for (int j = 0; j < n; ++j) m = fmax(m, S[(size_t)i * n + j]);
        for (int j = 0; j < n; ++j) {
            S[(size_t)i * n + j] = exp(S[(size_t)i * n + j] - m);
            l += S[(size_t)i * n + j];
        }
        for (int c = 0; c < D; ++c) {
            double a = 0.0;
            for (int j = 0; j < n; ++j) a += S[(size_t)i * n + j] * V[j * D + c];
            O[i * D + c] = a / l;
        }
    }
    free(S);
    return 0;
}

/* ======================================================================
 * Varlen packed prefill ([XF-DE] parts 4 and 5).
 * q: [T][Hq][D], k, v: [T][Hkv][D] binary16, packed without padding;
 * cu_seqlens[nseq+1] segment starts.  Row i of segment s attends to rows j
 * of the same segment with j <= i (causal) or all of them (causal == 0).
 * out: [T][Hq][D] fp64.
 * ====================================================================== */
typedef struct {
    const uint16_t *q, *k, *v;
    const int32_t* cu;
    int nseq, Hq, Hkv, D, causal;
    double scale;
    double* out;
    int64_t T;
    volatile int bad;
} prefill_job;

static void prefill_task(int64_t idx, void* p) {
    prefill_job* J = (prefill_job*)p;
    int64_t t = idx / J->Hq;
    int h = (int)(idx % J->Hq), D = J->D, hk = h / (J->Hq / J->Hkv);
    int s = 0;
    while (s < J->nseq && !(J->cu[s] <= t && t < J->cu[s + 1])) ++s;
    double* o = J->out + (t * J->Hq + h) * D;
    if (s == J->nseq) {
        J->bad = 1;
        for (int c = 0; c < D; ++c) o[c] = 0.0;
        return;
    }
    int64_t beg = J->cu[s], end = J->causal ? t + 1 : J->cu[s + 1];
    int64_t n = end - beg;
    double* K = (double*)malloc(sizeof(double) * n * D);
    double* V = (double*)malloc(sizeof(double) * n * D);
    double* x = (double*)malloc(sizeof(double) * n);
    double qd[512];
    for (int64_t j = 0; j < n; ++j)
        for (int c = 0; c < D; ++c) {
            K[j * D + c] = oracle_half_to_double(J->k[((beg + j) * J->Hkv + hk) * D + c]);
            V[j * D + c] = oracle_half_to_double(J->v[((beg + j) * J->Hkv + hk) * D + c]);
        }
    for (int c = 0; c < D; ++c) qd[c] = oracle_half_to_double(J->q[(t * J->Hq + h) * D + c]);
    attend_row(qd, K, V, n, D, D, J->scale, x, o);
    free(K);
    free(V);
    free(x);
}

int oracle_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* cu_seqlens,
                   int nseq, int Hq, int Hkv, int D, double scale, int causal, double* out,
                   int nthreads) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || D > 512 || nseq < 0) return -1;
    for (int s = 0; s < nseq; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
    int64_t T = cu_seqlens[nseq] - cu_seqlens[0];
    prefill_job J = {q, k, v, cu_seqlens, nseq, Hq, Hkv, D, causal, scale, out, T, 0};
    parallel_for(T * Hq, nthreads, prefill_task, &J);
    return J.bad ? -1 : 0;
}

/* ======================================================================
 * Append ([KVC-ES] step 2, [PA-DE]): write row t of k_new/v_new
 * ([n][Hkv][D] binary16) into the slot slot_mapping[t] of one layer's cache
 * [NB][Hkv][bs][D]; the slot is physical_block * bs + offset.  A negative
 * slot is skipped.  Bit copy.  Returns -1 if a slot is out of range (that
 * row is then skipped).
 * ====================================================================== */
int oracle_append(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_new, const uint16_t* v_new,
                  const int64_t* slot_mapping, int n, int Hkv, int D, int bs, int NB) {
    int bad = 0;
    for (int t = 0; t < n; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)NB * bs) {
            bad = 1;
            continue;
        }
        int64_t blk = slot / bs, off = slot % bs;
        for (int h = 0; h < Hkv; ++h) {
            int64_t dst = ((blk * Hkv + h) * bs + off) * D;
            int64_t src = ((int64_t)t * Hkv + h) * D;
            memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * D);
            memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * D);
        }
    }
    return bad ? -1 : 0;
}

/* ======================================================================
 * Split-context partial softmax and its merge ([FA-DE]).
 * oracle_partial: over rows [j0, j1) of contiguous K, V ([n][D] fp64) it
 * returns the row maximum m, the sum of exponentials l = sum e^(x_j - m) and
 * the unnormalised accumulator acc = sum e^(x_j - m) v_j.  An empty range
 * gives m = -inf, l = 0, acc = 0.
 * oracle_merge: M = max_s m_s, o = sum_s e^(m_s - M) acc_s /
 * sum_s e^(m_s - M) l_s; parts with l_s == 0 contribute nothing.
 * ====================================================================== */
void oracle_partial(const double* q, const double* K, const double* V, int j0, int j1, int D,
                    double scale, double* m_out, double* l_out, double* acc) {
    double m = -INFINITY, l = 0.0;
    for (int c = 0; c < D; ++c) acc[c] = 0.0;
    for (int j = j0; j < j1; ++j) {
        double s = 0.0;
        for (int c = 0; c < D; ++c) s += q[c] * K[(int64_t)j * D + c];
        m = fmax(m, s * scale);
    }
    for (int j = j0; j < j1; ++j) {
        double s = 0.0;
        for (int c = 0; c < D; ++c) s += q[c] * K[(int64_t)j * D + c];
        double p = exp(s * scale - m);
        l += p;
        for (int c = 0; c < D; ++c) acc[c] += p * V[(int64_t)j * D + c];
    }
    *m_out = m;
    *l_out = l;
}

void oracle_merge(const double* m, const double* l, const double* acc, int nparts, int D, double* out) {
    double M = -INFINITY, L = 0.0;
    for (int s = 0; s < nparts; ++s)
        if (l[s] > 0.0) M = fmax(M, m[s]);
    for (int c = 0; c < D; ++c) out[c] = 0.0;
    for (int s = 0; s < nparts; ++s) {
        if (!(l[s] > 0.0)) continue;
        double w = exp(m[s] - M);
        L += w * l[s];
        for (int c = 0; c < D; ++c) out[c] += w * acc[(int64_t)s * D + c];
    }
    for (int c = 0; c < D; ++c) out[c] /= L;
}
