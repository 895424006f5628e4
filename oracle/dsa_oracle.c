/*
 * dsa_oracle.c -- plain, slow CPU oracle for the DSA sparse-attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent definition that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product library never links,
 * includes or calls it, and it shares no header, table or helper with the
 * CUDA path.
 *
 * Source: the web page "vLLM's Kimi K3.1 Pro day-0 support: sparse attention,
 * DCP, zero-mismatch RL" (agentlenshq.com/ja/blogs/5e91cd0c...), cited below
 * as [K31] with its section titles:
 *   [K31 "What changed"]          the table: top-2048 indexer, 32 heads x 128
 *                                 dims, FP8 keys; the text: one FP8 key per
 *                                 token of 132 bytes including its scale, every
 *                                 earlier token scored, the top 2048 kept, MLA
 *                                 run exactly on those tokens only.
 *   [K31 "Sparse attention cuts long-context decode bandwidth"]
 *                                 576-byte FP8 latent per token; full latents
 *                                 read only for the 2048 selected tokens.
 *   [K31 "Packed KV cache"]       widths: latent 576 B (FP8) / 352 B (NVFP4),
 *                                 index key 132 B (FP8) / 68 B (MXFP4); kernels
 *                                 see small fixed-size pages through a block
 *                                 table translated before each step.
 *   [K31 "Fused low-latency decode for DSA layers"]
 *                                 indexer query quantised with the head weights
 *                                 folded in; the new token's key and latent are
 *                                 written into the cache.
 *   [K31 "Native MXFP4 indexer"]  (AMD MI355X section) 68 B key with scales,
 *                                 fp32 accumulation, weighted reduction across
 *                                 heads.
 * The pages do not print the indexer formula.  The reading used here is
 *     S[t,s] = sum_h w[t,h] * ReLU( qhat[t,h,:] . khat[s,:] )
 * with a stable tie-break toward the lower token index, softmax scale
 * 1/sqrt(192), absorbed MLA with 96 heads x 576 dims, values = dims 0..511.
 *
 * Number formats are decoded from the published specifications, not from any
 * library: OCP 8-bit floating point (OFP8) E4M3, and the OCP Microscaling (MX)
 * E2M1 element and E8M0 scale formats.
 *
 * All arithmetic is IEEE double unless a step states fp32 (the cache writer
 * mirrors the fp32 steps the format fixes).  Compile without fast-math and
 * with -ffp-contract=off.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- cache page formats (one layer) ------------------------------------ */
#define PAGE_TOKENS 64
#define IDX_HEADS 32
#define IDX_DIM 128
#define LAT_DIM 576
#define V_DIM 512
#define MLA_HEADS 96
/* FP8 index page: 64 x 128 E4M3 key bytes, then 64 little-endian fp32 scales. */
#define FP8_KEY_BYTES_PER_TOKEN (IDX_DIM + 4)                      /* 132 */
#define FP8_PAGE_BYTES (PAGE_TOKENS * IDX_DIM + PAGE_TOKENS * 4)   /* 8448 */
/* MXFP4 index page: 64 x 64 packed E2M1 bytes (element 2i in the low nibble),
 * then 64 x 4 E8M0 block scales (one per 32 elements). */
#define MXFP4_KEY_BYTES_PER_TOKEN (IDX_DIM / 2 + IDX_DIM / 32)     /* 68 */
#define MXFP4_PAGE_BYTES (PAGE_TOKENS * IDX_DIM / 2 + PAGE_TOKENS * 4) /* 4352 */
/* Latent page: 64 x 576 E4M3 bytes, one scale per layer (passed separately). */
/* NVFP4 latent page ([K31 "Packed KV cache"]: 352 B per token; the split is
 * not printed -- reading: 64 rows of [256 B packed E2M1 of dims 0..511
 * (element 2i in the low nibble) | 32 E4M3 scales, one per block of 16
 * elements | 64 E4M3 bytes of dims 512..575]), one fp32 scale per layer. */
#define NVFP4_LAT_BYTES 352
#define NVFP4_LAT_PAGE_BYTES (PAGE_TOKENS * NVFP4_LAT_BYTES)
#define LAT_BYTES_PER_TOKEN LAT_DIM                                /* 576 */
#define LAT_PAGE_BYTES (PAGE_TOKENS * LAT_DIM)                     /* 36864 */

#define ORC_OK 0
#define ORC_BAD_ARG (-1)
#define ORC_BAD_PAGE (-2)
#define ORC_BAD_INDEX (-3)
#define ORC_NAN (-4)
#define ORC_NOMEM (-5)

int oracle_constants(int32_t* out, int32_t n) {
    const int32_t c[] = {PAGE_TOKENS, IDX_HEADS, IDX_DIM, LAT_DIM, V_DIM, MLA_HEADS,
                         FP8_KEY_BYTES_PER_TOKEN, FP8_PAGE_BYTES,
                         MXFP4_KEY_BYTES_PER_TOKEN, MXFP4_PAGE_BYTES,
                         LAT_BYTES_PER_TOKEN, LAT_PAGE_BYTES};
    int32_t m = (int32_t)(sizeof(c) / sizeof(c[0]));
    for (int32_t i = 0; i < n && i < m; ++i) out[i] = c[i];
    return m;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- number formats ------------------------------------------------------ */

/* OCP OFP8 E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits.  No
 * infinities; S.1111.111 is NaN; exponent field 0 is subnormal
 * (value = m/8 * 2^-6).  Largest finite value 448. */
double oracle_e4m3_decode(uint8_t code) {
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* OCP MX E2M1 element: sign, 2 exponent bits (bias 1), 1 mantissa bit; no
 * infinities or NaN; exponent field 0 is subnormal (value = m * 0.5). */
double oracle_e2m1_decode(uint8_t nibble) {
    int s = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 3;
    int m = nibble & 1;
    double v;
    if (e == 0) v = 0.5 * (double)m;
    else v = ldexp(1.0 + 0.5 * (double)m, e - 1);
    return s ? -v : v;
}

/* OCP MX E8M0 scale: 2^(code-127); 0xFF is NaN. */
double oracle_e8m0_decode(uint8_t code) {
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* bfloat16: the upper half of an IEEE binary32. */
double oracle_bf16_decode(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a binary32 value to E4M3, round-to-nearest-even, saturating finite
 * values beyond the largest normal to +-448 (OFP8 "satfinite" conversion).
 * The input is widened to double, where every step below is exact. */
uint8_t oracle_e4m3_encode(float xf) {
    double x = (double)xf;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: quantum 2^-9; q == 8 is the smallest normal */
        double q = rint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)q);
    }
    int e;
    (void)frexp(a, &e);             /* a = f * 2^e, f in [0.5, 1) */
    int E = e - 1;                   /* a in [2^E, 2^(E+1)) */
    double q = rint(ldexp(a, 3 - E)); /* significand with 3 fraction bits, in [8,16] */
    if (q == 16.0) { q = 8.0; E += 1; }
    if (E > 8 || (E == 8 && q > 14.0)) return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | ((int)q - 8)));
}

/* Decode a whole array (used by the tests to pin the decoder). */
void oracle_e4m3_decode_array(const uint8_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(in[i]);
}
void oracle_e4m3_encode_array(const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(in[i]);
}

/* ---- batch addressing ---------------------------------------------------- */

typedef struct {
    int32_t num_requests;
    const int32_t* q_offsets;  /* [B+1] */
    const int32_t* seq_lens;   /* [B]   */
    const int32_t* block_table;/* [B, max_pages] */
    int32_t max_pages;
    int32_t num_pages;
} obatch;

/* Query token t belongs to request b with q_offsets[b] <= t < q_offsets[b+1].
 * Its position is seq_len[b] - n_b + j (j = t - q_offsets[b]) and it sees the
 * positions 0 .. seq_len[b] - n_b + j: the causal rule of multi-token decode
 * (n_b = 1 for plain decode, n_b new tokens for prefill-append). */
static int locate(const obatch* bt, int32_t t, int32_t* b_out, int64_t* vis_out) {
    for (int32_t b = 0; b < bt->num_requests; ++b) {
        if (t >= bt->q_offsets[b] && t < bt->q_offsets[b + 1]) {
            int32_t nb = bt->q_offsets[b + 1] - bt->q_offsets[b];
            int32_t j = t - bt->q_offsets[b];
            *b_out = b;
            *vis_out = (int64_t)bt->seq_lens[b] - nb + j + 1;
            return ORC_OK;
        }
    }
    return ORC_BAD_ARG;
}

/* Physical page of logical token s of request b (the block-table lookup that
 * the page describes as translating cache slots to kernel page addresses). */
static int page_of(const obatch* bt, int32_t b, int64_t s, int64_t* page, int32_t* slot) {
    int64_t lp = s / PAGE_TOKENS;
    if (lp >= bt->max_pages) return ORC_BAD_PAGE;
    int32_t p = bt->block_table[(int64_t)b * bt->max_pages + lp];
    if (p < 0 || p >= bt->num_pages) return ORC_BAD_PAGE;
    *page = p;
    *slot = (int32_t)(s % PAGE_TOKENS);
    return ORC_OK;
}

static float load_f32(const uint8_t* p) {
    float f;
    memcpy(&f, p, 4);
    return f;
}

/* Dequantised index key khat[s, 0..127] of logical token s (request b). */
static int load_key(const obatch* bt, int32_t b, int64_t s, const uint8_t* pages,
                    int32_t key_format, double* k) {
    int64_t page;
    int32_t slot;
    int rc = page_of(bt, b, s, &page, &slot);
    if (rc) return rc;
    if (key_format == 0) {
        const uint8_t* base = pages + page * (int64_t)FP8_PAGE_BYTES;
        double scale = (double)load_f32(base + PAGE_TOKENS * IDX_DIM + slot * 4);
        for (int d = 0; d < IDX_DIM; ++d)
            k[d] = oracle_e4m3_decode(base[slot * IDX_DIM + d]) * scale;
    } else if (key_format == 1) {
        const uint8_t* base = pages + page * (int64_t)MXFP4_PAGE_BYTES;
        const uint8_t* vals = base + slot * (IDX_DIM / 2);
        const uint8_t* scl = base + PAGE_TOKENS * (IDX_DIM / 2) + slot * 4;
        for (int d = 0; d < IDX_DIM; ++d) {
            uint8_t byte = vals[d / 2];
            uint8_t nib = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            k[d] = oracle_e2m1_decode(nib) * oracle_e8m0_decode(scl[d / 32]);
        }
    } else {
        return ORC_BAD_ARG;
    }
    return ORC_OK;
}

/* ---- indexer scores ------------------------------------------------------ */

/* For every listed query row t = rows[r] and every visible position s:
 *   S[r, s] = sum_h w[t,h] * ReLU( sum_d qhat[t,h,d] * khat[s,d] )
 *   A[r, s] = sum_h |w[t,h]| * sum_d |qhat[t,h,d] * khat[s,d]|
 * with qhat = E4M3(q8) * qscale[t,h] and khat the dequantised key.  A is the
 * magnitude against which a fp32 implementation's rounding is judged.
 * Positions s in [visible, ld) get S = -inf and A = 0. */
static int index_scores_row(const obatch* bt, int32_t t, const uint8_t* q8,
                            const float* qscale, const float* w, const uint8_t* pages,
                            int32_t key_format, int64_t ld, double* S, double* A) {
    int32_t b;
    int64_t vis;
    int rc = locate(bt, t, &b, &vis);
    if (rc) return rc;
    if (vis > ld) return ORC_BAD_ARG;
    double* qh = (double*)malloc(sizeof(double) * IDX_HEADS * IDX_DIM);
    if (!qh) return ORC_NOMEM;
    for (int h = 0; h < IDX_HEADS; ++h) {
        double sc = (double)qscale[(int64_t)t * IDX_HEADS + h];
        for (int d = 0; d < IDX_DIM; ++d)
            qh[h * IDX_DIM + d] =
                oracle_e4m3_decode(q8[((int64_t)t * IDX_HEADS + h) * IDX_DIM + d]) * sc;
    }
    double k[IDX_DIM];
    for (int64_t s = 0; s < vis; ++s) {
        rc = load_key(bt, b, s, pages, key_format, k);
        if (rc) { free(qh); return rc; }
        double acc = 0.0, mag = 0.0;
        for (int h = 0; h < IDX_HEADS; ++h) {
            double dot = 0.0, adot = 0.0;
            for (int d = 0; d < IDX_DIM; ++d) {
                double p = qh[h * IDX_DIM + d] * k[d];
                dot += p;
                adot += fabs(p);
            }
            double wh = (double)w[(int64_t)t * IDX_HEADS + h];
            double relu = dot > 0.0 ? dot : 0.0;
            acc += wh * relu;
            mag += fabs(wh) * adot;
        }
        S[s] = acc;
        if (A) A[s] = mag;
    }
    for (int64_t s = vis; s < ld; ++s) {
        S[s] = -INFINITY;
        if (A) A[s] = 0.0;
    }
    free(qh);
    return ORC_OK;
}

int oracle_index_scores(int32_t num_requests, const int32_t* q_offsets,
                        const int32_t* seq_lens, const int32_t* block_table,
                        int32_t max_pages, int32_t num_pages, const uint8_t* q8,
                        const float* qscale, const float* w, const uint8_t* index_pages,
                        int32_t key_format, const int32_t* rows, int32_t nrows, int64_t ld,
                        double* S, double* A) {
    obatch bt = {num_requests, q_offsets, seq_lens, block_table, max_pages, num_pages};
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < nrows; ++r) {
        int rc = index_scores_row(&bt, rows[r], q8, qscale, w, index_pages, key_format, ld,
                                  S + (int64_t)r * ld, A ? A + (int64_t)r * ld : NULL);
        if (rc) {
#pragma omp critical
            err = rc;
        }
    }
    return err;
}

/* ---- exact top-k ---------------------------------------------------------- */

typedef struct {
    double v;
    int32_t i;
} scored;

/* Larger score first; equal scores: lower token index first.  (-0 and +0
 * compare equal, so they tie and fall back to the index.) */
static int cmp_scored(const void* pa, const void* pb) {
    const scored* a = (const scored*)pa;
    const scored* b = (const scored*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

static int cmp_i32(const void* pa, const void* pb) {
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

/* The k visible positions with the largest scores (ties to the lower index),
 * returned in ascending position order and padded with -1.  When at most k
 * positions are visible, all of them are returned. */
int oracle_topk_row(const double* scores, int64_t n_visible, int32_t k, int32_t* out) {
    if (n_visible < 0 || k <= 0) return ORC_BAD_ARG;
    scored* tmp = (scored*)malloc(sizeof(scored) * (size_t)(n_visible > 0 ? n_visible : 1));
    if (!tmp) return ORC_NOMEM;
    for (int64_t s = 0; s < n_visible; ++s) {
        if (isnan(scores[s])) { free(tmp); return ORC_NAN; }
        tmp[s].v = scores[s];
        tmp[s].i = (int32_t)s;
    }
    qsort(tmp, (size_t)n_visible, sizeof(scored), cmp_scored);
    int64_t m = n_visible < k ? n_visible : k;
    for (int64_t j = 0; j < m; ++j) out[j] = tmp[j].i;
    qsort(out, (size_t)m, sizeof(int32_t), cmp_i32);
    for (int64_t j = m; j < k; ++j) out[j] = -1;
    free(tmp);
    return ORC_OK;
}

/* Row-wise top-k: row r has n_visible[r] valid scores at scores[r*ld ...]. */
int oracle_topk(const double* scores, int64_t ld, const int64_t* n_visible, int32_t nrows,
                int32_t k, int32_t* out) {
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < nrows; ++r) {
        int rc = oracle_topk_row(scores + (int64_t)r * ld, n_visible[r], k,
                                 out + (int64_t)r * k);
        if (rc) {
#pragma omp critical
            err = rc;
        }
    }
    return err;
}

/* Visible count of each listed query row (host-side helper for the tests). */
int oracle_visible(int32_t num_requests, const int32_t* q_offsets, const int32_t* seq_lens,
                   const int32_t* rows, int32_t nrows, int64_t* vis) {
    obatch bt = {num_requests, q_offsets, seq_lens, NULL, 0, 0};
    for (int32_t r = 0; r < nrows; ++r) {
        int32_t b;
        int rc = locate(&bt, rows[r], &b, &vis[r]);
        if (rc) return rc;
    }
    return ORC_OK;
}

/* ---- latent rows ------------------------------------------------------------ */

/* Dequantised latent of one token, lhat[0..575], from its stored bytes.
 * format 0 (FP8):   lhat[d] = E4M3(row[d]) * kv_scale
 * format 1 (NVFP4): lhat[d] = E2M1(nibble d of row[0..255]) * E4M3(row[256 + d/16])
 *                             * kv_scale                       for d < 512
 *                   lhat[d] = E4M3(row[288 + d - 512]) * kv_scale  for d >= 512 */
int oracle_latent_row(int32_t format, const uint8_t* row, double kv_scale, double* out) {
    if (format == 0) {
        for (int d = 0; d < LAT_DIM; ++d) out[d] = oracle_e4m3_decode(row[d]) * kv_scale;
        return ORC_OK;
    }
    if (format != 1) return ORC_BAD_ARG;
    for (int d = 0; d < V_DIM; ++d) {
        const uint8_t byte = row[d / 2];
        const uint8_t nib = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
        out[d] = oracle_e2m1_decode(nib) * oracle_e4m3_decode(row[V_DIM / 2 + d / 16]) * kv_scale;
    }
    for (int d = V_DIM; d < LAT_DIM; ++d)
        out[d] = oracle_e4m3_decode(row[V_DIM / 2 + V_DIM / 16 + (d - V_DIM)]) * kv_scale;
    return ORC_OK;
}

/* ---- sparse MLA, absorbed form -------------------------------------------- */

/* For query row t and the selected positions I (entries >= 0 of indices[r,:]):
 *   lhat_s = E4M3(latent[s, :]) * kv_scale                       (576 dims)
 *   z[h,s] = sm_scale * sum_d qhat[t,h,d] * lhat_s[d]            (96 heads)
 *   p[h,s] = exp(z[h,s] - max_s z[h,s]) / sum_s exp(z[h,s] - max_s z[h,s])
 *   o[h,d] = sum_s p[h,s] * lhat_s[d]      for d < 512 (values = first 512 dims)
 *   lse[h] = max_s z[h,s] + log(sum_s exp(z[h,s] - max_s z[h,s]))
 * An empty selection gives o = 0 and lse = -inf. */
static int sparse_mla_row(const obatch* bt, int32_t t, const uint16_t* q_lat,
                          const uint8_t* latent_pages, int32_t lat_format, double kv_scale,
                          double sm_scale, const int32_t* idx, int32_t k, double* o,
                          double* lse) {
    int32_t b;
    int64_t vis;
    int rc = locate(bt, t, &b, &vis);
    if (rc) return rc;
    int64_t seq = bt->seq_lens[b];
    int32_t n = 0;
    for (int32_t j = 0; j < k; ++j) {
        if (idx[j] < 0) continue;
        if (idx[j] >= seq) return ORC_BAD_INDEX;
        ++n;
    }
    memset(o, 0, sizeof(double) * MLA_HEADS * V_DIM);
    if (n == 0) {
        for (int h = 0; h < MLA_HEADS; ++h) lse[h] = -INFINITY;
        return ORC_OK;
    }
    double* L = (double*)malloc(sizeof(double) * (size_t)n * LAT_DIM);
    double* q = (double*)malloc(sizeof(double) * MLA_HEADS * LAT_DIM);
    double* z = (double*)malloc(sizeof(double) * (size_t)n);
    if (!L || !q || !z) { free(L); free(q); free(z); return ORC_NOMEM; }
    int32_t c = 0;
    for (int32_t j = 0; j < k; ++j) {
        if (idx[j] < 0) continue;
        int64_t page;
        int32_t slot;
        rc = page_of(bt, b, idx[j], &page, &slot);
        if (rc) { free(L); free(q); free(z); return rc; }
        const int64_t row_bytes = lat_format == 1 ? NVFP4_LAT_BYTES : LAT_DIM;
        const uint8_t* src = latent_pages + (page * PAGE_TOKENS + slot) * row_bytes;
        rc = oracle_latent_row(lat_format, src, kv_scale, L + (int64_t)c * LAT_DIM);
        if (rc) { free(L); free(q); free(z); return rc; }
        ++c;
    }
    for (int i = 0; i < MLA_HEADS * LAT_DIM; ++i)
        q[i] = oracle_bf16_decode(q_lat[(int64_t)t * MLA_HEADS * LAT_DIM + i]);
    for (int h = 0; h < MLA_HEADS; ++h) {
        double zmax = -INFINITY;
        for (int32_t s = 0; s < n; ++s) {
            double dot = 0.0;
            for (int d = 0; d < LAT_DIM; ++d) dot += q[h * LAT_DIM + d] * L[(int64_t)s * LAT_DIM + d];
            z[s] = sm_scale * dot;
            if (z[s] > zmax) zmax = z[s];
        }
        double sum = 0.0;
        for (int32_t s = 0; s < n; ++s) {
            z[s] = exp(z[s] - zmax);
            sum += z[s];
        }
        for (int32_t s = 0; s < n; ++s) {
            double p = z[s] / sum;
            for (int d = 0; d < V_DIM; ++d) o[h * V_DIM + d] += p * L[(int64_t)s * LAT_DIM + d];
        }
        lse[h] = zmax + log(sum);
    }
    free(L);
    free(q);
    free(z);
    return ORC_OK;
}

int oracle_sparse_mla_fmt(int32_t num_requests, const int32_t* q_offsets,
                          const int32_t* seq_lens, const int32_t* block_table, int32_t max_pages,
                          int32_t num_pages, const uint16_t* q_lat, const uint8_t* latent_pages,
                          int32_t lat_format, double kv_scale, double sm_scale,
                          const int32_t* indices, int32_t k, const int32_t* rows, int32_t nrows,
                          double* out, double* lse) {
    obatch bt = {num_requests, q_offsets, seq_lens, block_table, max_pages, num_pages};
    if (lat_format != 0 && lat_format != 1) return ORC_BAD_ARG;
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < nrows; ++r) {
        int rc = sparse_mla_row(&bt, rows[r], q_lat, latent_pages, lat_format, kv_scale, sm_scale,
                                indices + (int64_t)r * k, k,
                                out + (int64_t)r * MLA_HEADS * V_DIM, lse + (int64_t)r * MLA_HEADS);
        if (rc) {
#pragma omp critical
            err = rc;
        }
    }
    return err;
}

int oracle_sparse_mla(int32_t num_requests, const int32_t* q_offsets, const int32_t* seq_lens,
                      const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                      const uint16_t* q_lat, const uint8_t* latent_pages, double kv_scale,
                      double sm_scale, const int32_t* indices, int32_t k, const int32_t* rows,
                      int32_t nrows, double* out, double* lse) {
    return oracle_sparse_mla_fmt(num_requests, q_offsets, seq_lens, block_table, max_pages,
                                 num_pages, q_lat, latent_pages, 0, kv_scale, sm_scale, indices,
                                 k, rows, nrows, out, lse);
}

/* ---- the whole decode step for a set of query rows ----------------------- */

/* scores -> top-k -> sparse MLA, row by row (what one layer's step computes for
 * those query tokens).  Outputs: indices [nrows, k], out [nrows, 96, 512],
 * lse [nrows, 96]. */
int oracle_decode_fmt(int32_t num_requests, const int32_t* q_offsets, const int32_t* seq_lens,
                      const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                      const uint8_t* q8, const float* qscale, const float* w,
                      const uint8_t* index_pages, int32_t key_format, const uint16_t* q_lat,
                      const uint8_t* latent_pages, int32_t lat_format, double kv_scale,
                      double sm_scale, int32_t k, const int32_t* rows, int32_t nrows,
                      int32_t* indices, double* out, double* lse) {
    obatch bt = {num_requests, q_offsets, seq_lens, block_table, max_pages, num_pages};
    if (lat_format != 0 && lat_format != 1) return ORC_BAD_ARG;
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < nrows; ++r) {
        int32_t b;
        int64_t vis;
        int rc = locate(&bt, rows[r], &b, &vis);
        double* S = NULL;
        if (!rc) {
            S = (double*)malloc(sizeof(double) * (size_t)(vis > 0 ? vis : 1));
            if (!S) rc = ORC_NOMEM;
        }
        if (!rc)
            rc = index_scores_row(&bt, rows[r], q8, qscale, w, index_pages, key_format, vis, S, NULL);
        if (!rc) rc = oracle_topk_row(S, vis, k, indices + (int64_t)r * k);
        if (!rc)
            rc = sparse_mla_row(&bt, rows[r], q_lat, latent_pages, lat_format, kv_scale,
                                sm_scale, indices + (int64_t)r * k, k,
                                out + (int64_t)r * MLA_HEADS * V_DIM, lse + (int64_t)r * MLA_HEADS);
        free(S);
        if (rc) {
#pragma omp critical
            err = rc;
        }
    }
    return err;
}

int oracle_decode(int32_t num_requests, const int32_t* q_offsets, const int32_t* seq_lens,
                  const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                  const uint8_t* q8, const float* qscale, const float* w,
                  const uint8_t* index_pages, int32_t key_format, const uint16_t* q_lat,
                  const uint8_t* latent_pages, double kv_scale, double sm_scale, int32_t k,
                  const int32_t* rows, int32_t nrows, int32_t* indices, double* out,
                  double* lse) {
    return oracle_decode_fmt(num_requests, q_offsets, seq_lens, block_table, max_pages,
                             num_pages, q8, qscale, w, index_pages, key_format, q_lat,
                             latent_pages, 0, kv_scale, sm_scale, k, rows, nrows, indices, out,
                             lse);
}

/* ---- cache append ---------------------------------------------------------- */

/* Write the n = q_offsets[B] new tokens (the last n_b positions of each
 * request, in q_offsets order) into the paged caches.
 *   index key (FP8 format): scale = amax/448 in fp32 (1 when amax == 0),
 *       code[d] = E4M3_rne_satfinite( x[d] / scale ) with an fp32 division;
 *       the 128 codes and the fp32 scale are stored in the token's slot.
 *   latent: code[d] = E4M3_rne_satfinite( x[d] / kv_scale ), fp32 division.
 * Either pointer pair may be NULL to skip that cache. */
int oracle_append_cache(int32_t num_requests, const int32_t* q_offsets, const int32_t* seq_lens,
                        const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                        const float* new_keys, const float* new_latent, float kv_scale,
                        uint8_t* index_pages, uint8_t* latent_pages, int32_t key_format) {
    obatch bt = {num_requests, q_offsets, seq_lens, block_table, max_pages, num_pages};
    if (key_format != 0) return ORC_BAD_ARG;
    int32_t n = q_offsets[num_requests];
    for (int32_t t = 0; t < n; ++t) {
        int32_t b;
        int64_t vis;
        int rc = locate(&bt, t, &b, &vis);
        if (rc) return rc;
        int64_t pos = vis - 1; /* the token's own position */
        int64_t page;
        int32_t slot;
        rc = page_of(&bt, b, pos, &page, &slot);
        if (rc) return rc;
        if (new_keys && index_pages) {
            const float* x = new_keys + (int64_t)t * IDX_DIM;
            float amax = 0.0f;
            for (int d = 0; d < IDX_DIM; ++d) {
                float a = fabsf(x[d]);
                if (a > amax) amax = a;
            }
            float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
            uint8_t* base = index_pages + page * (int64_t)FP8_PAGE_BYTES;
            for (int d = 0; d < IDX_DIM; ++d) {
                float y = x[d] / scale;
                base[slot * IDX_DIM + d] = oracle_e4m3_encode(y);
            }
            memcpy(base + PAGE_TOKENS * IDX_DIM + slot * 4, &scale, 4);
        }
        if (new_latent && latent_pages) {
            const float* x = new_latent + (int64_t)t * LAT_DIM;
            uint8_t* dst = latent_pages + page * (int64_t)LAT_PAGE_BYTES + slot * LAT_DIM;
            for (int d = 0; d < LAT_DIM; ++d) {
                float y = x[d] / kv_scale;
                dst[d] = oracle_e4m3_encode(y);
            }
        }
    }
    return ORC_OK;
}

/* ---- decode context parallelism: exact top-k merge and LSE combine -------- */

/* [K31 "Decode context parallelism with the sparse indexer"]: with DCP over W
 * ranks, rank r stores every W-th token (positions s = r mod W) and can only
 * rank its own tokens, so the global top-2048 has to be merged across ranks
 * before attention; partial attention outputs are combined by log-sum-exp.
 * [K31 "Exact top-k merge with about 10x less traffic"]: each rank sends only
 * its best ceil(1.5 * 2048 / W) candidates, chosen from BF16 scores (each
 * packed with its score into 32 bits); every rank selects the same global
 * top-2048 from the gathered candidates; the merge stays exact because a
 * rank that holds more of the top-2048 than it sent is detected and resends
 * its full local top-k for that row.
 *
 * The result the merge reaches is defined here directly: the k visible
 * positions with the largest BF16-rounded scores, ties to the lower position.
 * The resend decision is the one the protocol takes: rank r resends when every
 * candidate it sent is among the top k of all sent candidates and it holds
 * more visible tokens than it sent. */

/* bfloat16 code of a binary32 value: round to nearest, ties to even (the 16
 * dropped bits decide); infinities keep their code.  NaN is not an input. */
uint16_t oracle_bf16_encode(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof(u));
    if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void oracle_bf16_encode_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_encode(in[i]);
}

/* One row: scores[0 .. n_visible) (binary32), `world` ranks, `cand` candidates
 * sent per rank, k selected.  Writes the merged selection to out[0..k) in
 * ascending position order (padded with -1) and 1 / 0 to resend[0..world). */
int oracle_dcp_topk_row(const float* scores, int64_t n_visible, int32_t world, int32_t cand,
                        int32_t k, int32_t* out, int32_t* resend) {
    if (n_visible < 0 || world < 1 || cand < 1 || k < 1) return ORC_BAD_ARG;
    const size_t n = (size_t)n_visible;
    scored* ord = (scored*)malloc(sizeof(scored) * (n > 0 ? n : 1));
    int64_t* n_r = (int64_t*)calloc((size_t)world, sizeof(int64_t));
    int64_t* seen = (int64_t*)calloc((size_t)world, sizeof(int64_t));
    int64_t* taken = (int64_t*)calloc((size_t)world, sizeof(int64_t));
    char* sent = (char*)malloc(n > 0 ? n : 1);
    if (!ord || !n_r || !seen || !taken || !sent) {
        free(ord); free(n_r); free(seen); free(taken); free(sent);
        return ORC_NOMEM;
    }
    for (size_t s = 0; s < n; ++s) {
        if (isnan(scores[s])) {
            free(ord); free(n_r); free(seen); free(taken); free(sent);
            return ORC_NAN;
        }
        ord[s].v = oracle_bf16_decode(oracle_bf16_encode(scores[s]));
        ord[s].i = (int32_t)s;
        n_r[s % (size_t)world] += 1;
    }
    /* the global order: BF16 score descending, position ascending */
    qsort(ord, n, sizeof(scored), cmp_scored);
    const int64_t m = n_visible < k ? n_visible : k;
    for (int64_t j = 0; j < m; ++j) out[j] = ord[j].i;
    qsort(out, (size_t)m, sizeof(int32_t), cmp_i32);
    for (int64_t j = m; j < k; ++j) out[j] = -1;
    /* each rank's order is the global order restricted to its positions, so
     * its candidates are its first `cand` positions in the global order */
    int64_t n_sent = 0;
    for (size_t j = 0; j < n; ++j) {
        const int r = ord[j].i % world;
        sent[j] = (seen[r] < cand);
        seen[r] += 1;
        n_sent += sent[j];
    }
    /* the top k of everything sent, and how many of each rank's candidates
     * it holds */
    const int64_t g = n_sent < k ? n_sent : k;
    int64_t got = 0;
    for (size_t j = 0; j < n && got < g; ++j) {
        if (!sent[j]) continue;
        taken[ord[j].i % world] += 1;
        ++got;
    }
    for (int32_t r = 0; r < world; ++r) {
        const int64_t sr = n_r[r] < cand ? n_r[r] : cand;
        resend[r] = (sr > 0 && taken[r] == sr && n_r[r] > sr) ? 1 : 0;
    }
    free(ord); free(n_r); free(seen); free(taken); free(sent);
    return ORC_OK;
}

int oracle_dcp_topk(const float* scores, int64_t ld, const int64_t* n_visible, int32_t nrows,
                    int32_t world, int32_t cand, int32_t k, int32_t* out, int32_t* resend) {
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < nrows; ++r) {
        int rc = oracle_dcp_topk_row(scores + (int64_t)r * ld, n_visible[r], world, cand, k,
                                     out + (int64_t)r * k, resend + (int64_t)r * world);
        if (rc) {
#pragma omp critical
            err = rc;
        }
    }
    return err;
}

/* Log-sum-exp combine of `world` partial attention results over disjoint
 * token sets, row by row (a row is one (query token, head) pair):
 *   L = log sum_r exp(lse_r),  out = sum_r exp(lse_r - L) * part_r
 * part [world][nrows][dim], part_lse [world][nrows] (natural log; -inf for a
 * rank with no tokens).  A row with no tokens anywhere gives out = 0 and
 * lse = -inf. */
int oracle_lse_combine(int32_t world, int64_t nrows, int32_t dim, const double* part,
                       const double* part_lse, double* out, double* lse) {
    if (world < 1 || nrows < 0 || dim < 1) return ORC_BAD_ARG;
    for (int64_t i = 0; i < nrows; ++i) {
        double mx = -INFINITY;
        for (int32_t r = 0; r < world; ++r)
            if (part_lse[(int64_t)r * nrows + i] > mx) mx = part_lse[(int64_t)r * nrows + i];
        double* o = out + i * dim;
        for (int32_t d = 0; d < dim; ++d) o[d] = 0.0;
        if (mx == -INFINITY) {
            lse[i] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int32_t r = 0; r < world; ++r) sum += exp(part_lse[(int64_t)r * nrows + i] - mx);
        const double L = mx + log(sum);
        for (int32_t r = 0; r < world; ++r) {
            const double wgt = exp(part_lse[(int64_t)r * nrows + i] - L);
            const double* pr = part + ((int64_t)r * nrows + i) * dim;
            for (int32_t d = 0; d < dim; ++d) o[d] += wgt * pr[d];
        }
        lse[i] = L;
    }
    return ORC_OK;
}

/* ---- fused indexer front ---------------------------------------------------- */

/* [K31 "Fused low-latency decode for DSA layers"], second step: one kernel
 * does the query norm, the indexer query projection, FP8 quantisation with the
 * head weights folded in, and the new token's index key.  The pages give
 * neither dimensions nor formulas; the reading is
 *   inv_rms[t] = 1 / sqrt( (1/dq) sum_k q_c[t,k]^2 + 1e-6 )        (query norm;
 *                its gain is part of the synthetic projection W_q)
 *   q[t,j]     = inv_rms[t] * sum_k W_q[j,k] q_c[t,k]    j < 32*128: head j/128
 *   w[t,h]     = sum_k W_w[h,k] x[t,k]                   h < 32 head weights
 *   key[t,d]   = sum_k W_k[d,k] x[t,k]                   d < 128 the new index key
 * with q_c the token's query latent [dq], x its hidden state [dh], all bf16
 * inputs decoded exactly and the arithmetic in fp64.  Quantising q per head
 * and the key (and writing the key into the cache) follow the cache writer's
 * rule: oracle_quantize_rows below and oracle_append_cache. */
int oracle_indexer_front(int32_t T, int32_t dq, int32_t dh, const uint16_t* q_c, const uint16_t* x,
                         const uint16_t* w_q, const uint16_t* w_w, const uint16_t* w_k,
                         double* q, double* w, double* key, double* inv_rms) {
    if (T < 0 || dq < 1 || dh < 1) return ORC_BAD_ARG;
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t t = 0; t < T; ++t) {
        double* qc = (double*)malloc(sizeof(double) * (size_t)dq);
        double* xx = (double*)malloc(sizeof(double) * (size_t)dh);
        if (!qc || !xx) {
            free(qc); free(xx);
#pragma omp critical
            err = ORC_NOMEM;
            continue;
        }
        double ss = 0.0;
        for (int32_t k = 0; k < dq; ++k) {
            qc[k] = oracle_bf16_decode(q_c[(int64_t)t * dq + k]);
            ss += qc[k] * qc[k];
        }
        for (int32_t k = 0; k < dh; ++k) xx[k] = oracle_bf16_decode(x[(int64_t)t * dh + k]);
        const double r = 1.0 / sqrt(ss / dq + 1e-6);
        inv_rms[t] = r;
        for (int32_t j = 0; j < IDX_HEADS * IDX_DIM; ++j) {
            double acc = 0.0;
            for (int32_t k = 0; k < dq; ++k) acc += oracle_bf16_decode(w_q[(int64_t)j * dq + k]) * qc[k];
            q[(int64_t)t * IDX_HEADS * IDX_DIM + j] = r * acc;
        }
        for (int32_t h = 0; h < IDX_HEADS; ++h) {
            double acc = 0.0;
            for (int32_t k = 0; k < dh; ++k) acc += oracle_bf16_decode(w_w[(int64_t)h * dh + k]) * xx[k];
            w[(int64_t)t * IDX_HEADS + h] = acc;
        }
        for (int32_t d = 0; d < IDX_DIM; ++d) {
            double acc = 0.0;
            for (int32_t k = 0; k < dh; ++k) acc += oracle_bf16_decode(w_k[(int64_t)d * dh + k]) * xx[k];
            key[(int64_t)t * IDX_DIM + d] = acc;
        }
        free(qc);
        free(xx);
    }
    return err;
}

/* Per-row FP8 quantisation, the cache writer's rule: scale = amax/448 in fp32
 * (1 when amax == 0), code = E4M3_rne_satfinite(x / scale) with an fp32
 * division.  x [nrows][dim] binary32 -> codes [nrows][dim], scales [nrows]. */
int oracle_quantize_rows(const float* x, int64_t nrows, int32_t dim, uint8_t* codes,
                         float* scales) {
    if (nrows < 0 || dim < 1) return ORC_BAD_ARG;
    for (int64_t r = 0; r < nrows; ++r) {
        const float* v = x + r * dim;
        float amax = 0.0f;
        for (int32_t d = 0; d < dim; ++d) {
            const float a = fabsf(v[d]);
            if (a > amax) amax = a;
        }
        const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        for (int32_t d = 0; d < dim; ++d) codes[r * dim + d] = oracle_e4m3_encode(v[d] / scale);
        scales[r] = scale;
    }
    return ORC_OK;
}
