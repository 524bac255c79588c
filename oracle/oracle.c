/*
 * CPU oracle for the restricted-vocabulary draft head and the greedy verify
 * head.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the library path never does.  It
 * shares no code with the CUDA library (separate sources, headers and
 * build), and is deliberately plain and slow.
 *
 * What it computes (plain definitions, no blocking, fusion or reordering):
 *
 *  Draft head ("少读一张大表，草稿路径才真正快起来", cnblogs Qwen3.8 Flash
 *  dual-Spark log): the draft path scores only a smaller candidate table,
 *  takes the maximum score and returns the *global* token id of the winning
 *  candidate, plus the score.
 *      s[b,c]      = sum_{h=0}^{H-1} float(x[b,h]) * float(W[c,h])
 *                    (fp32, sequential in h)
 *      c*          = first c (lowest index) reaching max_c s[b,c]
 *      ids[b]      = cand_ids[c*],  maxlogit[b] = s[b,c*]
 *  Candidate ids are ascending, so the first maximum is also the lowest
 *  global id: ties go to the lowest global id.
 *
 *  Block-scaled 4-bit head (NVFP4: E2M1 values, one E4M3 scale per 16
 *  elements along H, one fp32 tensor scale g): every weight is decoded to
 *  fp32 as  w = float(e2m1(q)) * float(e4m3(s_blk)) * g  (the first product
 *  is exact, one rounding comes from * g), then scored as above.
 *
 *  Greedy verify (same page: the target keeps the full output head and
 *  verifies the draft; "长上下文推理优化" §5: MTP proposal -> target
 *  verification -> accept several tokens): row r = b*(k+1)+j of X is the
 *  target hidden state after the context plus draft tokens d[b,0..j-1].
 *      next_ids[r]   = argmax_v sum_h X[r,h] W[v,h]   (same rules, gid = v)
 *      accept_len[b] = number of leading j < k with next_ids[b(k+1)+j] == d[b,j]
 *
 * NaN scores are treated as -inf and -0 equals +0 (inputs here are finite).
 *
 * Compiled with -ffp-contract=off so that x86_64 and aarch64 agree bit for
 * bit.  Plain C99 + pthreads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 -> fp32: the bf16 bits are the upper half of the fp32 bits. */
float vh_oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* E2M1 (OCP MX FP4): sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent field 0 is subnormal: value = m * 2^(1-1) * 0.5.  Codes 0 and 8
 * are +0 and -0.  There is no Inf or NaN. */
float vh_oracle_e2m1_value(uint8_t code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return (float)(s ? -v : v);
}

/* E4M3 (OCP FP8 "e4m3fn"): sign bit 7, exponent bits 6..3 (bias 7),
 * mantissa bits 2..0.  Exponent field 0 is subnormal: m/8 * 2^-6.  Only
 * S.1111.111 is NaN (returned as NaN); there is no infinity. */
float vh_oracle_e4m3_value(uint8_t code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return (float)(s ? -v : v);
}

/* One 4-bit weight: element h of a row with codes q (two per byte, element
 * 2i in the low nibble) and block scales s (one per 16 elements). */
static inline float nvfp4_weight(const uint8_t* q, const uint8_t* s, float g, int64_t h) {
    uint8_t byte = q[h >> 1];
    uint8_t code = (h & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
    float ws = vh_oracle_e2m1_value(code) * vh_oracle_e4m3_value(s[h >> 4]);
    return ws * g;
}

/* fp32 dot product of bf16 vectors, summed sequentially over h. */
float vh_oracle_dot_bf16(const uint16_t* x, const uint16_t* w, int64_t H) {
    float acc = 0.0f;
    for (int64_t h = 0; h < H; ++h) acc += vh_oracle_bf16_to_f32(x[h]) * vh_oracle_bf16_to_f32(w[h]);
    return acc;
}

/* fp32 dot product of a bf16 vector with one decoded 4-bit row. */
float vh_oracle_dot_nvfp4(const uint16_t* x, const uint8_t* q, const uint8_t* s, float g, int64_t H) {
    float acc = 0.0f;
    for (int64_t h = 0; h < H; ++h) acc += vh_oracle_bf16_to_f32(x[h]) * nvfp4_weight(q, s, g, h);
    return acc;
}

/* ---------------------------------------------------------------------- */
/* Scores of one hidden row against rows [0, n) of a head, split over
 * threads by contiguous row ranges (each score is computed on its own, so
 * the split does not change any value).                                   */

typedef struct {
    const uint16_t* x;
    const uint16_t* W;  /* bf16 head, or NULL for the 4-bit head */
    const int32_t* rows; /* score W row rows[c] for entry c (NULL: row c) */
    const uint8_t* q;
    const uint8_t* s;
    float g;
    int64_t H;
    float* out;
    int64_t lo, hi;
} score_job;

static void* score_main(void* p) {
    score_job* j = (score_job*)p;
    for (int64_t c = j->lo; c < j->hi; ++c) {
        if (j->W)
            j->out[c] = vh_oracle_dot_bf16(j->x, j->W + (j->rows ? (int64_t)j->rows[c] : c) * j->H, j->H);
        else
            j->out[c] = vh_oracle_dot_nvfp4(j->x, j->q + c * (j->H / 2), j->s + c * (j->H / 16), j->g, j->H);
    }
    return NULL;
}

static void all_scores_rows(const uint16_t* x, const uint16_t* W, const int32_t* rows, const uint8_t* q,
                            const uint8_t* s, float g, int64_t n, int64_t H, float* out, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < 64) nthreads = 1;
    score_job jobs[256];
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        score_job j = {x, W, rows, q, s, g, H, out, n * t / nthreads, n * (t + 1) / nthreads};
        jobs[t] = j;
    }
    for (int t = 0; t + 1 < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, score_main, &jobs[t]) != 0) break;
        ++started;
    }
    for (int t = started; t < nthreads; ++t) score_main(&jobs[t]);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

static void all_scores(const uint16_t* x, const uint16_t* W, const uint8_t* q, const uint8_t* s, float g, int64_t n,
                       int64_t H, float* out, int nthreads) {
    all_scores_rows(x, W, NULL, q, s, g, n, H, out, nthreads);
}

/* Sequential scan: first index of the maximum (strict >), NaN as -inf,
 * -0 == +0.  Also reports the largest score among the other rows. */
static int64_t first_argmax(const float* sc, int64_t n, float* best_out, float* second_out) {
    int64_t best = -1;
    float bv = -INFINITY, sv = -INFINITY;
    for (int64_t c = 0; c < n; ++c) {
        float v = isnan(sc[c]) ? -INFINITY : sc[c];
        if (best < 0 || v > bv) {
            if (best >= 0 && bv > sv) sv = bv;
            best = c;
            bv = v;
        } else if (v > sv) {
            sv = v;
        }
    }
    if (best_out) *best_out = bv + 0.0f; /* canonical +0 */
    if (second_out) *second_out = sv;
    return best;
}

/* Draft head over bf16 candidate rows.
 *   x [B][H] bf16, W [Vc][H] bf16, cand_ids [Vc]  ->  ids [B], maxlogit [B],
 *   second [B] (nullable: best score among the other candidates).
 * Returns 0, or -1 on bad sizes / -2 on allocation failure. */
int vh_oracle_draft_argmax(const uint16_t* x, const uint16_t* W, const int32_t* cand_ids, int64_t B, int64_t H,
                           int64_t Vc, int32_t* ids, float* maxlogit, float* second, int nthreads) {
    if (B < 1 || H < 1 || Vc < 1) return -1;
    float* sc = (float*)malloc((size_t)Vc * sizeof(float));
    if (!sc) return -2;
    for (int64_t b = 0; b < B; ++b) {
        all_scores(x + b * H, W, NULL, NULL, 0.0f, Vc, H, sc, nthreads);
        float bv, sv;
        int64_t c = first_argmax(sc, Vc, &bv, &sv);
        ids[b] = cand_ids[c];
        maxlogit[b] = bv;
        if (second) second[b] = sv;
    }
    free(sc);
    return 0;
}

/* Draft head over 4-bit candidate rows: q [Vc][H/2], s [Vc][H/16], g. */
int vh_oracle_draft_argmax_nvfp4(const uint16_t* x, const uint8_t* q, const uint8_t* s, float g,
                                 const int32_t* cand_ids, int64_t B, int64_t H, int64_t Vc, int32_t* ids,
                                 float* maxlogit, float* second, int nthreads) {
    if (B < 1 || H < 16 || H % 16 != 0 || Vc < 1) return -1;
    float* sc = (float*)malloc((size_t)Vc * sizeof(float));
    if (!sc) return -2;
    for (int64_t b = 0; b < B; ++b) {
        all_scores(x + b * H, NULL, q, s, g, Vc, H, sc, nthreads);
        float bv, sv;
        int64_t c = first_argmax(sc, Vc, &bv, &sv);
        ids[b] = cand_ids[c];
        maxlogit[b] = bv;
        if (second) second[b] = sv;
    }
    free(sc);
    return 0;
}

/* Draft head over rows gathered from the full head (dynamic candidate rows):
 * entry i scores W row row_ids[i] (entries outside [0, V) are ignored); the
 * largest score wins and equal scores go to the lowest row id, whatever the
 * order of the list.  second[b] = best score among entries with another id.
 * Returns -3 if no entry is in range. */
int vh_oracle_draft_argmax_gather(const uint16_t* x, const uint16_t* W, const int32_t* row_ids, int64_t B, int64_t H,
                                  int64_t n, int64_t V, int32_t* ids, float* maxlogit, float* second, int nthreads) {
    if (B < 1 || H < 1 || n < 1 || V < 1) return -1;
    float* sc = (float*)malloc((size_t)n * sizeof(float));
    int32_t* rows = (int32_t*)malloc((size_t)n * sizeof(int32_t));
    if (!sc || !rows) { free(sc); free(rows); return -2; }
    for (int64_t i = 0; i < n; ++i) rows[i] = (row_ids[i] >= 0 && row_ids[i] < V) ? row_ids[i] : 0;
    for (int64_t b = 0; b < B; ++b) {
        all_scores_rows(x + b * H, W, rows, NULL, NULL, 0.0f, n, H, sc, nthreads);
        int64_t best = -1;
        float bv = -INFINITY;
        for (int64_t i = 0; i < n; ++i) {
            if (row_ids[i] < 0 || row_ids[i] >= V) continue;
            float v = isnan(sc[i]) ? -INFINITY : sc[i];
            if (best < 0 || v > bv || (v == bv && row_ids[i] < row_ids[best])) {
                best = i;
                bv = v;
            }
        }
        if (best < 0) { free(sc); free(rows); return -3; }
        float sv = -INFINITY;
        for (int64_t i = 0; i < n; ++i) {
            if (row_ids[i] < 0 || row_ids[i] >= V || row_ids[i] == row_ids[best]) continue;
            float v = isnan(sc[i]) ? -INFINITY : sc[i];
            if (v > sv) sv = v;
        }
        ids[b] = row_ids[best];
        maxlogit[b] = bv + 0.0f;
        if (second) second[b] = sv;
    }
    free(sc);
    free(rows);
    return 0;
}

/* Accepted-prefix length: leading positions where the target's greedy id
 * equals the draft id. */
int32_t vh_oracle_accept_len(const int32_t* next_ids_b, const int32_t* draft_b, int64_t k) {
    int32_t a = 0;
    while (a < k && next_ids_b[a] == draft_b[a]) ++a;
    return a;
}

/* Greedy verify over the full head (gid = row index of W).
 *   X [R][H], R = B*(k+1);  W [V][H];  draft [B][k]
 *   -> next_ids [R], accept_len [B], maxlogit [R] and second [R] (nullable).
 * Rows listed in `rows` (nrows of them, nullable = all R rows) are the only
 * ones scored; the others' outputs are left untouched, and accept_len is
 * written only when every row is scored. */
int vh_oracle_verify_greedy(const uint16_t* X, const uint16_t* W, const int32_t* draft, int64_t B, int64_t k,
                            int64_t H, int64_t V, const int32_t* rows, int64_t nrows, int32_t* next_ids,
                            int32_t* accept_len, float* maxlogit, float* second, int nthreads) {
    if (B < 1 || k < 0 || H < 1 || V < 1) return -1;
    const int64_t R = B * (k + 1);
    float* sc = (float*)malloc((size_t)V * sizeof(float));
    if (!sc) return -2;
    const int64_t n = rows ? nrows : R;
    for (int64_t i = 0; i < n; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= R) { free(sc); return -1; }
        all_scores(X + r * H, W, NULL, NULL, 0.0f, V, H, sc, nthreads);
        float bv, sv;
        int64_t v = first_argmax(sc, V, &bv, &sv);
        next_ids[r] = (int32_t)v;
        if (maxlogit) maxlogit[r] = bv;
        if (second) second[r] = sv;
    }
    free(sc);
    if (!rows && accept_len && draft)
        for (int64_t b = 0; b < B; ++b) accept_len[b] = vh_oracle_accept_len(next_ids + b * (k + 1), draft + b * k, k);
    return 0;
}

/* Greedy verify over a block-scaled 4-bit full head (codes q [V][H/2],
 * scales s [V][H/16], tensor scale g): the same rules as the bf16 verify,
 * every weight decoded as e2m1(q) * e4m3(s) * g. */
int vh_oracle_verify_greedy_nvfp4(const uint16_t* X, const uint8_t* q, const uint8_t* s, float g,
                                  const int32_t* draft, int64_t B, int64_t k, int64_t H, int64_t V,
                                  const int32_t* rows, int64_t nrows, int32_t* next_ids, int32_t* accept_len,
                                  float* maxlogit, float* second, int nthreads) {
    if (B < 1 || k < 0 || H < 16 || H % 16 != 0 || V < 1) return -1;
    const int64_t R = B * (k + 1);
    float* sc = (float*)malloc((size_t)V * sizeof(float));
    if (!sc) return -2;
    const int64_t n = rows ? nrows : R;
    for (int64_t i = 0; i < n; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= R) { free(sc); return -1; }
        all_scores(X + r * H, NULL, q, s, g, V, H, sc, nthreads);
        float bv, sv;
        int64_t v = first_argmax(sc, V, &bv, &sv);
        next_ids[r] = (int32_t)v;
        if (maxlogit) maxlogit[r] = bv;
        if (second) second[r] = sv;
    }
    free(sc);
    if (!rows && accept_len && draft)
        for (int64_t b = 0; b < B; ++b) accept_len[b] = vh_oracle_accept_len(next_ids + b * (k + 1), draft + b * k, k);
    return 0;
}

/* All scores of one hidden row against a bf16 head (for near-tie checks). */
void vh_oracle_scores_bf16(const uint16_t* x, const uint16_t* W, int64_t n, int64_t H, float* out, int nthreads) {
    all_scores(x, W, NULL, NULL, 0.0f, n, H, out, nthreads);
}

void vh_oracle_scores_nvfp4(const uint16_t* x, const uint8_t* q, const uint8_t* s, float g, int64_t n, int64_t H,
                            float* out, int nthreads) {
    all_scores(x, NULL, q, s, g, n, H, out, nthreads);
}

/* Decode a whole 4-bit head to fp32 [n][H] with the per-weight rule above. */
void vh_oracle_decode_nvfp4(const uint8_t* q, const uint8_t* s, float g, int64_t n, int64_t H, float* out) {
    for (int64_t c = 0; c < n; ++c)
        for (int64_t h = 0; h < H; ++h) out[c * H + h] = nvfp4_weight(q + c * (H / 2), s + c * (H / 16), g, h);
}
