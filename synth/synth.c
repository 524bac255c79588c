/*
 * Seeded synthetic inputs for the restricted-vocabulary draft head and the
 * greedy verify head.  Shared by the tests, the benchmark and the oracle
 * checks; it holds none of the head arithmetic (no dot products, no argmax,
 * no weight decoding for scoring, no acceptance scan).
 *
 * Every value is a pure function of (seed, stream, index): a splitmix64
 * counter generator (S. Vigna, "splitmix64.c", public domain reference
 * generator) mixed per stream, so multi-threaded generation is deterministic
 * and a single row can be regenerated without the rest of the tensor.
 *
 * Plain C99 + pthreads; no architecture-specific code.  Built with
 * -ffp-contract=off so x86_64 and aarch64 produce the same bits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* Key of one (seed, stream) pair. */
static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GOLDEN) ^ (stream * 0xD1B54A32D192ED03ull + 1));
}

/* The index-th output of the splitmix64 sequence started at key. */
static inline uint64_t draw(uint64_t key, uint64_t index) {
    return mix64(key + (index + 1) * GOLDEN);
}

/* Uniform double in [0, 1) with 53 random bits. */
static inline double unif01(uint64_t u) { return (double)(u >> 11) * 0x1.0p-53; }

/* Standard normal number `index` of a stream: Box-Muller on the pair
 * (2p, 2p+1), p = index/2; even indices take the cosine branch, odd the
 * sine branch. */
static inline double std_normal(uint64_t key, uint64_t index) {
    uint64_t p = index >> 1;
    double u1 = ((double)(draw(key, 2 * p) >> 11) + 1.0) * 0x1.0p-53; /* (0,1] */
    double u2 = unif01(draw(key, 2 * p + 1));
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586 * u2;
    return (index & 1) ? r * sin(a) : r * cos(a);
}

/* float -> bf16 bits, round to nearest even (finite inputs only). */
static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

/* ---------------------------------------------------------------------- */
/* Threading helper: split [0, n) into nthreads contiguous chunks.         */

typedef struct {
    void (*fn)(void* ctx, int64_t lo, int64_t hi);
    void* ctx;
    int64_t lo, hi;
} job_t;

static void* job_main(void* p) {
    job_t* j = (job_t*)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static void parallel_for(int64_t n, int nthreads, void (*fn)(void*, int64_t, int64_t), void* ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < (int64_t)nthreads * 4096 || nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t th[256];
    job_t jobs[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].lo = n * t / nthreads;
        jobs[t].hi = n * (t + 1) / nthreads;
        if (t == nthreads - 1) break;
        if (pthread_create(&th[t], NULL, job_main, &jobs[t]) != 0) break;
        ++started;
    }
    /* Whatever was not handed to a thread runs here. */
    for (int t = started; t < nthreads; ++t) fn(ctx, jobs[t].lo, jobs[t].hi);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------------- */
/* Normal tensors.                                                         */

typedef struct {
    uint64_t key;
    uint64_t offset;
    double sigma;
    uint16_t* out_bf16;
    float* out_f32;
} normal_ctx;

static void normal_bf16_body(void* c, int64_t lo, int64_t hi) {
    normal_ctx* x = (normal_ctx*)c;
    for (int64_t i = lo; i < hi; ++i)
        x->out_bf16[i] = f32_to_bf16_rne((float)(x->sigma * std_normal(x->key, x->offset + (uint64_t)i)));
}

static void normal_f32_body(void* c, int64_t lo, int64_t hi) {
    normal_ctx* x = (normal_ctx*)c;
    for (int64_t i = lo; i < hi; ++i)
        x->out_f32[i] = (float)(x->sigma * std_normal(x->key, x->offset + (uint64_t)i));
}

/* out[i] = bf16(sigma * N_i), N_i = normal number (offset + i) of (seed, stream). */
void vh_synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double sigma,
                          uint16_t* out, int nthreads) {
    normal_ctx c = {stream_key(seed, stream), offset, sigma, out, NULL};
    parallel_for(n, nthreads, normal_bf16_body, &c);
}

void vh_synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double sigma,
                         float* out, int nthreads) {
    normal_ctx c = {stream_key(seed, stream), offset, sigma, NULL, out};
    parallel_for(n, nthreads, normal_f32_body, &c);
}

typedef struct {
    uint64_t key;
    const int32_t* rows;
    int64_t H;
    double sigma;
    uint16_t* out;
} rows_ctx;

static void rows_body(void* c, int64_t lo, int64_t hi) {
    rows_ctx* x = (rows_ctx*)c;
    for (int64_t r = lo; r < hi; ++r) {
        uint64_t base = (uint64_t)x->rows[r] * (uint64_t)x->H;
        uint16_t* o = x->out + r * x->H;
        for (int64_t h = 0; h < x->H; ++h)
            o[h] = f32_to_bf16_rne((float)(x->sigma * std_normal(x->key, base + (uint64_t)h)));
    }
}

/* Rows `rows[0..nrows)` of the [*, H] bf16 normal tensor of (seed, stream):
 * out[r][h] equals element rows[r]*H + h of vh_synth_normal_bf16. */
void vh_synth_normal_bf16_rows(uint64_t seed, uint64_t stream, const int32_t* rows, int64_t nrows,
                               int64_t H, double sigma, uint16_t* out, int nthreads) {
    rows_ctx c = {stream_key(seed, stream), rows, H, sigma, out};
    parallel_for(nrows, nthreads, rows_body, &c);
}

/* ---------------------------------------------------------------------- */
/* Sorted distinct subset of [0, n_total) of size k (R. Floyd's sampling). */

int vh_synth_sorted_subset(uint64_t seed, uint64_t stream, int64_t n_total, int64_t k, int32_t* out) {
    if (k < 0 || k > n_total || n_total > 0x7FFFFFFF) return -1;
    uint64_t key = stream_key(seed, stream);
    int64_t words = (n_total + 63) / 64;
    uint64_t* bits = (uint64_t*)calloc((size_t)(words > 0 ? words : 1), 8);
    if (!bits) return -2;
    uint64_t ctr = 0;
    for (int64_t j = n_total - k; j < n_total; ++j) {
        uint64_t t = draw(key, ctr++) % (uint64_t)(j + 1);
        if (bits[t >> 6] & (1ull << (t & 63))) t = (uint64_t)j;
        bits[t >> 6] |= 1ull << (t & 63);
    }
    int64_t m = 0;
    for (int64_t i = 0; i < n_total; ++i)
        if (bits[i >> 6] & (1ull << (i & 63))) out[m++] = (int32_t)i;
    free(bits);
    return m == k ? 0 : -3;
}

/* ---------------------------------------------------------------------- */
/* Draft ids: the target's greedy ids corrupted independently per position.
 * With probability p position i is replaced by an id drawn uniformly from
 * [0, V) minus the true id (draw r in [0, V-1), id = r + (r >= t)). */

void vh_synth_corrupt_ids(uint64_t seed, uint64_t stream, const int32_t* truth, int64_t n, int32_t V,
                          double p, int32_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) {
        int32_t t = truth[i];
        if (unif01(draw(key, 2 * (uint64_t)i)) < p && V > 1) {
            int32_t r = (int32_t)(draw(key, 2 * (uint64_t)i + 1) % (uint64_t)(V - 1));
            out[i] = r + (r >= t ? 1 : 0);
        } else {
            out[i] = t;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Block-scaled 4-bit encoder (data generation only).
 *
 * Format (NVFP4 as used for Blackwell 4-bit weights): each element is an
 * E2M1 code (sign, 2 exponent bits with bias 1, 1 mantissa bit; magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6), two codes per byte with element 2i in the
 * low nibble; one E4M3 scale (OCP FP8: bias 7, subnormals, max 448) per 16
 * consecutive elements along H; one fp32 tensor scale g.
 *
 *   g     = amax(|w|) / (6 * 448)
 *   s_blk = RNE_e4m3(amax_blk / (6 g))
 *   q     = RNE_e2m1(w / (s_blk g)), saturating at +-6; s_blk = 0 gives q = 0.
 *
 * Encoding is a nearest-value search over the format's value grid with ties
 * to the even code; the grids are enumerated here from the bit layouts.
 */

static double e4m3_grid[127]; /* value of non-negative code c, c = 0..126 */
static const double e2m1_grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
static pthread_once_t grid_once = PTHREAD_ONCE_INIT;

static void build_grid(void) {
    for (int c = 0; c < 127; ++c) {
        int e = (c >> 3) & 15, m = c & 7;
        e4m3_grid[c] = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    }
}

/* Nearest grid index for a non-negative value, ties to the even index;
 * values above the top of the grid saturate. */
static int nearest_even(const double* grid, int n, double v) {
    if (!(v > 0.0)) return 0;
    if (v >= grid[n - 1]) return n - 1;
    int lo = 0, hi = n - 1; /* grid[lo] <= v < grid[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (grid[mid] <= v) lo = mid; else hi = mid;
    }
    double dl = v - grid[lo], dh = grid[hi] - v;
    if (dl < dh) return lo;
    if (dh < dl) return hi;
    return (lo & 1) ? hi : lo;
}

typedef struct {
    const float* w;
    int64_t H;
    double g;
    uint8_t* q;
    uint8_t* s;
} quant_ctx;

static void quant_body(void* c, int64_t lo, int64_t hi) {
    quant_ctx* x = (quant_ctx*)c;
    const int64_t H = x->H, nb = H / 16;
    for (int64_t r = lo; r < hi; ++r) {
        const float* w = x->w + r * H;
        uint8_t* q = x->q + r * (H / 2);
        uint8_t* s = x->s + r * nb;
        memset(q, 0, (size_t)(H / 2));
        for (int64_t b = 0; b < nb; ++b) {
            double amax = 0.0;
            for (int i = 0; i < 16; ++i) {
                double a = fabs((double)w[b * 16 + i]);
                if (a > amax) amax = a;
            }
            int sc = (x->g > 0.0) ? nearest_even(e4m3_grid, 127, amax / (6.0 * x->g)) : 0;
            s[b] = (uint8_t)sc;
            double step = e4m3_grid[sc] * x->g;
            for (int i = 0; i < 16; ++i) {
                int64_t h = b * 16 + i;
                double v = (double)w[h];
                int code = 0;
                if (step > 0.0) {
                    int mag = nearest_even(e2m1_grid, 8, fabs(v) / step);
                    code = (mag != 0 && v < 0.0) ? (mag | 8) : mag;
                }
                q[h >> 1] |= (uint8_t)((h & 1) ? (code << 4) : code);
            }
        }
    }
}

/* w: fp32 [rows][H] (H % 16 == 0).  Writes q [rows][H/2], s [rows][H/16] and
 * returns g through *g_out.  Returns 0 on success. */
int vh_synth_nvfp4_quantize(const float* w, int64_t rows, int64_t H, uint8_t* q, uint8_t* s,
                            float* g_out, int nthreads) {
    if (H <= 0 || H % 16 != 0 || rows < 0) return -1;
    pthread_once(&grid_once, build_grid);
    double amax = 0.0;
    for (int64_t i = 0; i < rows * H; ++i) {
        double a = fabs((double)w[i]);
        if (a > amax) amax = a;
    }
    float g = (float)(amax / (6.0 * 448.0));
    *g_out = g;
    quant_ctx c = {w, H, (double)g, q, s};
    parallel_for(rows, nthreads, quant_body, &c);
    return 0;
}

/* Encode with a caller-given tensor scale (g > 0). */
int vh_synth_nvfp4_quantize_with_g(const float* w, int64_t rows, int64_t H, float g, uint8_t* q,
                                   uint8_t* s, int nthreads) {
    if (H <= 0 || H % 16 != 0 || rows < 0 || !(g > 0.0f)) return -1;
    pthread_once(&grid_once, build_grid);
    quant_ctx c = {w, H, (double)g, q, s};
    parallel_for(rows, nthreads, quant_body, &c);
    return 0;
}

/* 64-bit FNV-1a over a byte buffer: fingerprints generated tensors so that
 * stored expected values can check the generator reproduces the same bits. */
uint64_t vh_synth_fingerprint(const void* data, int64_t nbytes) {
    const uint8_t* p = (const uint8_t*)data;
    uint64_t h = 0xCBF29CE484222325ull;
    for (int64_t i = 0; i < nbytes; ++i) {
        h ^= p[i];
        h *= 0x100000001B3ull;
    }
    return h;
}
