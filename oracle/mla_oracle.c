/*
 * Plain CPU oracle for MLA decode over a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct statement
 * of what the GPU path computes. Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it. The GPU library never links,
 * includes or calls anything here, and nothing here includes GPU code.
 *
 * Sources (web pages, cited by title and section):
 *  [P1] "sabi-mla-vllm" (PyPI README): intro paragraph (512-d latent plus one
 *       shared 64-d rotary key, 576 cached values per token); "What the plugin
 *       does" (paged 576-wide bf16 latent cache, no K/V stored); "B300 fix
 *       (0.2.0)" (the paged offset block_id x page_size x 576 must not be
 *       formed in 32-bit integers).
 *  [P2] "qwen-mla-vllm" README: "Speculative decoding (MTP)" (a verify step
 *       of 1+k query tokens reads the latent cache once per request).
 *  [P3] vLLM pull request #55543 (fp8_ds_mla for rope-free MLA on SM90):
 *       commit messages 3.1+3.2 and 5.1-5.4 and the PR description
 *       "Approach" / "Memory tradeoff" (656-byte row; NoPE bytes are a
 *       per-128-block fp8 quantisation; decode returns an LSE; rows with no
 *       valid token neutralise to (0, -inf)).
 *
 * Arithmetic: every floating-point step of the definition is evaluated in
 * fp64. bf16 and e4m3 inputs are exactly representable in fp64, so the
 * oracle is the definition up to fp64 rounding.  The two places where the
 * method itself fixes a lower precision are the fp8 cache write (scale and
 * quotient are fp32 IEEE divisions, see oracle_cache_write) and the stored
 * fp32 scale.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MLA_D 512      /* latent width (kv_lora_rank) [P1 intro] */
#define MLA_P 64       /* shared rotary key width [P1 intro] */
#define MLA_W 576      /* values per cached token = 512 + 64 [P1 intro] */
#define ROW_BF16 1152  /* bytes per bf16 row = 576 * 2 [P1 intro] */
#define ROW_FP8 656    /* bytes per fp8_ds_mla row [P3 "Memory tradeoff"] */

/* ---------------------------------------------------------------- codecs */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn") variant: 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 is subnormal (m * 2^-9); code
 * S.1111.111 is NaN; there is no infinity; the largest finite is 448. */
double oracle_e4m3_to_f64(uint8_t c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to nearest, ties to even, saturating to +-448 (what "satfinite"
 * means: a finite input never becomes NaN). NaN stays NaN. */
uint8_t oracle_f32_to_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: value = m * 2^-9, m in 0..8 (8 is the smallest
         * normal 2^-6, whose code 0x08 is also m = 8 read as e=1,m=0). */
        double m = nearbyint(a * 512.0);  /* exact scaling, RNE */
        return sign | (uint8_t)m;
    }
    int e2;
    double fr = frexp(a, &e2);        /* a = fr * 2^e2, fr in [0.5, 1) */
    int e = e2 - 1;                    /* a = (2 fr) * 2^e, 2fr in [1, 2) */
    double mant = (2.0 * fr - 1.0) * 8.0;  /* exact */
    double mr = nearbyint(mant);       /* RNE on the 3-bit mantissa */
    if (mr == 8.0) { mr = 0.0; e += 1; }
    int code = ((e + 7) << 3) | (int)mr;
    if (code > 0x7E) code = 0x7E;      /* cannot happen for a < 448 */
    return sign | (uint8_t)code;
}

/* Array form of oracle_f32_to_e4m3 (for exhaustive codec checks). */
void oracle_f32_to_e4m3_n(const float *x, uint8_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_e4m3(x[i]);
}

/* ----------------------------------------------------------- cache write */

/* Scatter one row per token into the paged pool.
 * [P1 "What the plugin does"], [P3 commit 3.1+3.2 "concat_and_cache_mla"]:
 *   kind 0: row = concat(latent[0:512], k_pe[0:64]) as 576 bf16 (1152 B).
 *   kind 1: fp8_ds_mla 656 B row [P3 commit 5.1-5.4, PR "Approach"]:
 *     bytes [0,512)   e4m3 codes of latent / scale_j, j = d / 128
 *     bytes [512,528) four fp32 scales, scale_j = absmax_j / 448 (1 if 0)
 *     bytes [528,656) the 64 bf16 k_pe values unchanged.
 * slot_mapping[t] < 0 means "no row for this token".
 * Returns 0, or -1 if a slot is out of range (nothing written for it). */
int oracle_cache_write(const uint16_t *latent, int64_t latent_stride,
                       const uint16_t *k_pe, int64_t k_pe_stride,
                       const int64_t *slot_mapping, int64_t num_tokens,
                       uint8_t *cache, int64_t num_slots, int kind) {
    int bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) { bad = 1; continue; }
        const uint16_t *x = latent + t * latent_stride;
        const uint16_t *r = k_pe + t * k_pe_stride;
        if (kind == 0) {
            uint8_t *row = cache + slot * (int64_t)ROW_BF16;
            memcpy(row, x, MLA_D * 2);
            memcpy(row + MLA_D * 2, r, MLA_P * 2);
        } else {
            uint8_t *row = cache + slot * (int64_t)ROW_FP8;
            for (int j = 0; j < 4; ++j) {
                float amax = 0.0f;
                for (int i = 0; i < 128; ++i) {
                    float v = (float)oracle_bf16_to_f64(x[128 * j + i]);
                    float av = fabsf(v);
                    if (av > amax) amax = av;
                }
                volatile float scale = (amax == 0.0f) ? 1.0f : amax / 448.0f;
                for (int i = 0; i < 128; ++i) {
                    float v = (float)oracle_bf16_to_f64(x[128 * j + i]);
                    volatile float q = v / scale;
                    row[128 * j + i] = oracle_f32_to_e4m3(q);
                }
                float sc = scale;
                memcpy(row + 512 + 4 * j, &sc, 4);
            }
            memcpy(row + 528, r, MLA_P * 2);
        }
    }
    return bad ? -1 : 0;
}

/* Read cached token `slot` back as 576 fp64 values (latent then k_pe). */
static void read_row(const uint8_t *cache, int kind, int64_t slot, double *v) {
    if (kind == 0) {
        const uint8_t *row = cache + slot * (int64_t)ROW_BF16;
        for (int d = 0; d < MLA_W; ++d) {
            uint16_t b;
            memcpy(&b, row + 2 * d, 2);
            v[d] = oracle_bf16_to_f64(b);
        }
    } else {
        const uint8_t *row = cache + slot * (int64_t)ROW_FP8;
        for (int d = 0; d < MLA_D; ++d) {
            float sc;
            memcpy(&sc, row + 512 + 4 * (d / 128), 4);
            v[d] = oracle_e4m3_to_f64(row[d]) * (double)sc;
        }
        for (int e = 0; e < MLA_P; ++e) {
            uint16_t b;
            memcpy(&b, row + 528 + 2 * e, 2);
            v[MLA_D + e] = oracle_bf16_to_f64(b);
        }
    }
}

/* ---------------------------------------------------- context gather */

/* bf16 bits of an fp32 value, round to nearest with ties to even (the 16
 * dropped bits decide; a NaN stays a quiet NaN). */
uint16_t oracle_f32_to_bf16(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* The prefill-context gather of an fp8_ds_mla pool [P3: the commit "derive
 * mla_dims from the runtime layers" and the PR description, where the
 * fp8_ds_mla context-gather path (cp_gather_and_upconvert_fp8_kv_cache)
 * fills a workspace whose rows must be 576 wide]. For request b < B and
 * context token j < cu[b+1] - cu[b]:
 *   slot = block_table[b][j / ps] * ps + j % ps                  (64-bit)
 *   dst[cu[b] + j][d]       = bf16(fp32(e4m3(code_d)) * scale_{d / 128})   d < 512
 *   dst[cu[b] + j][512 + e] = k_pe_e, the stored bf16 bits                 e < 64
 * The dequantised value is one fp32 multiply (the e4m3 value is exact in
 * fp32) rounded once more to bf16, round to nearest even: the two roundings
 * of the plainest reading (dequantise in fp32, store the 576-wide bf16 row).
 * Rows with cu[b] + j >= num_rows are skipped; other dst rows are untouched.
 * A page id outside the pool writes that row as zeros and the call returns
 * -1 (0 otherwise). */
int oracle_gather_upconvert(const uint8_t *cache, int64_t num_slots, int page_size,
                            const int32_t *block_table, int64_t bt_stride,
                            const int32_t *cu_seq_lens, int B, int64_t num_rows,
                            uint16_t *dst, int64_t dst_stride) {
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t r0 = cu_seq_lens[b], len = (int64_t)cu_seq_lens[b + 1] - r0;
        for (int64_t j = 0; j < len; ++j) {
            const int64_t r = r0 + j;
            if (r < 0 || r >= num_rows) continue;
            uint16_t *out = dst + r * dst_stride;
            const int64_t page = block_table[(int64_t)b * bt_stride + j / page_size];
            const int64_t slot = page * page_size + j % page_size;
            if (page < 0 || slot >= num_slots) {
                memset(out, 0, MLA_W * sizeof(uint16_t));
                bad = 1;
                continue;
            }
            const uint8_t *row = cache + slot * (int64_t)ROW_FP8;
            for (int d = 0; d < MLA_D; ++d) {
                float sc;
                memcpy(&sc, row + 512 + 4 * (d / 128), 4);
                const float v = (float)oracle_e4m3_to_f64(row[d]) * sc;  /* exact widening, one fp32 multiply */
                out[d] = oracle_f32_to_bf16(v);
            }
            for (int e = 0; e < MLA_P; ++e) memcpy(out + MLA_D + e, row + 528 + 2 * e, 2);
        }
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- decode */

/* Absorbed MLA decode, definition form.
 * For request b, query token qt (0..Qt-1), head h:
 *   visible tokens j = 0 .. T_b - Qt + qt   (a verify step of Qt tokens whose
 *     rows are already in the cache; token qt sees itself and its past)
 *   slot_j = block_table[b][j / ps] * ps + j % ps        (64-bit) [P1 "B300 fix"]
 *   s_j    = scale * (q_lat . c_j + q_pe . k_pe_j)
 *   out    = sum_j softmax(s)_j * c_j        (512 values; softmax over tokens)
 *   lse    = ln sum_j exp(s_j)
 * With no visible token: out = 0, lse = -inf [P3 commit 5.1-5.4].
 * Two passes over the tokens (max, then sums) in fp64.
 * `reqs` (n_reqs entries) restricts the work to those requests; NULL = all.
 * Rows of other requests in `out` / `lse` are left untouched.
 * Returns 0, or -1 if a slot or block id is out of range. */
/* One output row of the definition above: query token qt of a verify step
 * of Qt tokens over a request of T tokens whose block-table row is btr. */
static int decode_row(const uint16_t *ql, const uint16_t *qp, const uint8_t *cache, int kind,
                      int64_t num_slots, int page_size, const int32_t *btr, int64_t T,
                      int Qt, int qt, double scale, double *o, double *lse_out) {
    int64_t nvis = T - Qt + qt + 1;
    if (nvis < 0) nvis = 0;
    for (int d = 0; d < MLA_D; ++d) o[d] = 0.0;
    if (nvis == 0) { *lse_out = -INFINITY; return 0; }
    double q[MLA_W], c[MLA_W];
    for (int d = 0; d < MLA_D; ++d) q[d] = oracle_bf16_to_f64(ql[d]);
    for (int e = 0; e < MLA_P; ++e) q[MLA_D + e] = oracle_bf16_to_f64(qp[e]);
    double *s = (double *)malloc(sizeof(double) * (size_t)nvis);
    int64_t *slots = (int64_t *)malloc(sizeof(int64_t) * (size_t)nvis);
    for (int64_t j = 0; j < nvis; ++j) {
        int64_t blk = btr[j / page_size];
        int64_t slot = blk * (int64_t)page_size + j % page_size;
        if (blk < 0 || slot >= num_slots) { free(s); free(slots); *lse_out = NAN; return -1; }
        slots[j] = slot;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        read_row(cache, kind, slots[j], c);
        double dot = 0.0;
        for (int d = 0; d < MLA_W; ++d) dot += q[d] * c[d];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        double p = exp(s[j] - m);
        l += p;
        read_row(cache, kind, slots[j], c);
        for (int d = 0; d < MLA_D; ++d) o[d] += p * c[d];
    }
    for (int d = 0; d < MLA_D; ++d) o[d] /= l;
    *lse_out = m + log(l);
    free(s);
    free(slots);
    return 0;
}

int oracle_decode(const uint16_t *q_lat, const uint16_t *q_pe,
                  const uint8_t *cache, int kind, int64_t num_slots,
                  int page_size, const int32_t *block_table,
                  int64_t bt_stride, const int32_t *seq_lens, int B, int Qt,
                  int Hq, double scale, const int32_t *reqs, int n_reqs,
                  double *out, double *lse) {
    int nb = reqs ? n_reqs : B;
    int64_t ntask = (int64_t)nb * Qt * Hq;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t task = 0; task < ntask; ++task) {
        int bi = (int)(task / ((int64_t)Qt * Hq));
        int qt = (int)((task / Hq) % Qt);
        int h = (int)(task % Hq);
        int b = reqs ? reqs[bi] : bi;
        int64_t row = ((int64_t)b * Qt + qt) * Hq + h;
        if (decode_row(q_lat + row * MLA_D, q_pe + row * MLA_P, cache, kind, num_slots, page_size,
                       block_table + (int64_t)b * bt_stride, seq_lens[b], Qt, qt, scale,
                       out + row * MLA_D, lse + row))
            bad = 1;
    }
    return bad ? -1 : 0;
}

/* The same definition with a verify step of its own length per request (a
 * chunked verify batch; [P2 "Speculative decoding (MTP)"]: a verify step of
 * 1 + k query tokens reads the latent once per request, k per request):
 * request b's query tokens are cu_q[b] .. cu_q[b+1] - 1 (Qt_b of them, the
 * last Qt_b of its T_b tokens), its rows (cu_q[b] + qt) * Hq + h, and query
 * qt sees tokens 0 .. T_b - Qt_b + qt. All cu_q[B] * Hq rows are computed. */
int oracle_decode_varlen(const uint16_t *q_lat, const uint16_t *q_pe,
                         const uint8_t *cache, int kind, int64_t num_slots,
                         int page_size, const int32_t *block_table,
                         int64_t bt_stride, const int32_t *seq_lens,
                         const int32_t *cu_q, int B, int Hq, double scale,
                         double *out, double *lse) {
    int64_t ntask = (int64_t)cu_q[B] * Hq;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t row = 0; row < ntask; ++row) {
        int64_t tq = row / Hq;
        int b = 0;
        while (b + 1 < B && cu_q[b + 1] <= tq) ++b;
        int Qt = cu_q[b + 1] - cu_q[b];
        int qt = (int)(tq - cu_q[b]);
        if (decode_row(q_lat + row * MLA_D, q_pe + row * MLA_P, cache, kind, num_slots, page_size,
                       block_table + (int64_t)b * bt_stride, seq_lens[b], Qt, qt, scale,
                       out + row * MLA_D, lse + row))
            bad = 1;
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------- other latent widths */

/* The same absorbed decode for a bf16 cache whose rows hold a latent of D
 * values followed by a rotary key of P values (2 (D + P) bytes a row)
 * [P2 "How it works": the full-attention layers cache a per-layer latent of
 * rank 256, 768 or 1792 plus a small rotary and normalisation tail]. The
 * pages give neither the tail's rotary width nor what its normalisation
 * stores, so the reading is: the normalisation is applied before a row is
 * cached, and the decode sees [latent D | rope P] exactly as the 512-wide
 * definition above sees [latent 512 | rope 64]:
 *   s_j = scale * (q_lat . c_j[0:D] + q_pe . c_j[D:D+P])
 *   out = sum_j softmax(s)_j * c_j[0:D]   (D values),  lse = ln sum_j exp(s_j)
 * with the same visibility rule, (0, -inf) rows, 64-bit slot arithmetic and
 * fp64 two-pass softmax. q_lat rows are D values, q_pe rows P, out rows D.
 * Returns 0, or -1 if a block id or slot is out of range. */
static int decode_row_latent(const uint16_t *ql, const uint16_t *qp, const uint16_t *cache, int D, int P,
                             int64_t num_slots, int page_size, const int32_t *btr, int64_t T, int Qt,
                             int qt, double scale, double *o, double *lse_out) {
    const int Wd = D + P;
    int64_t nvis = T - Qt + qt + 1;
    if (nvis < 0) nvis = 0;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (nvis == 0) { *lse_out = -INFINITY; return 0; }
    double *q = (double *)malloc(sizeof(double) * (size_t)Wd);
    double *s = (double *)malloc(sizeof(double) * (size_t)nvis);
    int64_t *slots = (int64_t *)malloc(sizeof(int64_t) * (size_t)nvis);
    for (int d = 0; d < D; ++d) q[d] = oracle_bf16_to_f64(ql[d]);
    for (int e = 0; e < P; ++e) q[D + e] = oracle_bf16_to_f64(qp[e]);
    int bad = 0;
    for (int64_t j = 0; j < nvis; ++j) {
        int64_t blk = btr[j / page_size];
        int64_t slot = blk * (int64_t)page_size + j % page_size;
        if (blk < 0 || slot >= num_slots) { bad = 1; break; }
        slots[j] = slot;
    }
    if (bad) { free(q); free(s); free(slots); *lse_out = NAN; return -1; }
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        const uint16_t *c = cache + slots[j] * (int64_t)Wd;
        double dot = 0.0;
        for (int d = 0; d < Wd; ++d) dot += q[d] * oracle_bf16_to_f64(c[d]);
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        const uint16_t *c = cache + slots[j] * (int64_t)Wd;
        double pj = exp(s[j] - m);
        l += pj;
        for (int d = 0; d < D; ++d) o[d] += pj * oracle_bf16_to_f64(c[d]);
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    *lse_out = m + log(l);
    free(q);
    free(s);
    free(slots);
    return 0;
}

int oracle_decode_latent(const uint16_t *q_lat, const uint16_t *q_pe, const uint16_t *cache, int D, int P,
                         int64_t num_slots, int page_size, const int32_t *block_table, int64_t bt_stride,
                         const int32_t *seq_lens, int B, int Qt, int Hq, double scale, double *out,
                         double *lse) {
    if (D <= 0 || P < 0 || page_size <= 0) return -1;
    int64_t ntask = (int64_t)B * Qt * Hq;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t row = 0; row < ntask; ++row) {
        int b = (int)(row / ((int64_t)Qt * Hq));
        int qt = (int)((row / Hq) % Qt);
        if (decode_row_latent(q_lat + row * D, q_pe + row * P, cache, D, P, num_slots, page_size,
                              block_table + (int64_t)b * bt_stride, seq_lens[b], Qt, qt, scale,
                              out + row * D, lse + row))
            bad = 1;
    }
    return bad ? -1 : 0;
}

/* ----------------------------------------------------------------- merge */

/* Combine S partial results of the same rows computed over disjoint token
 * sets (flash-decoding split-KV / decode-context-parallel combine)
 * [P3 commit 5.1-5.4 "(0, -inf) per the DCP merge contract"]:
 *   L   = ln sum_i exp(lse_i)
 *   out = sum_i exp(lse_i - L) * o_i
 * Partials with lse = -inf carry no weight; if all are -inf the row is
 * (0, -inf). part_o: [S, N, 512] fp32, part_lse: [S, N] fp32. */
void oracle_merge(const float *part_o, const float *part_lse, int S, int64_t N,
                  double *out, double *lse) {
    for (int64_t n = 0; n < N; ++n) {
        double m = -INFINITY;
        for (int i = 0; i < S; ++i) {
            double v = part_lse[(int64_t)i * N + n];
            if (v > m) m = v;
        }
        double *o = out + n * MLA_D;
        for (int d = 0; d < MLA_D; ++d) o[d] = 0.0;
        if (m == -INFINITY) { lse[n] = -INFINITY; continue; }
        double wsum = 0.0;
        for (int i = 0; i < S; ++i) {
            double v = part_lse[(int64_t)i * N + n];
            if (v == -INFINITY) continue;
            wsum += exp(v - m);
        }
        double L = m + log(wsum);
        for (int i = 0; i < S; ++i) {
            double v = part_lse[(int64_t)i * N + n];
            if (v == -INFINITY) continue;
            double w = exp(v - L);
            const float *po = part_o + ((int64_t)i * N + n) * MLA_D;
            for (int d = 0; d < MLA_D; ++d) o[d] += w * (double)po[d];
        }
        lse[n] = L;
    }
}

/* Sets the threads the decode loops use from now on (no effect without
 * OpenMP); n < 1 is ignored. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Threads the decode loop uses (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Geometry constants, exposed so tests can check them against the pages. */
int oracle_row_values(void) { return MLA_W; }
int oracle_row_bytes(int kind) { return kind == 0 ? ROW_BF16 : ROW_FP8; }
