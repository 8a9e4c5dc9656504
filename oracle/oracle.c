/*
 * oracle.c -- plain, slow, fp64 CPU reference for the speculative-verify weight stream.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this file;
 * only the tests, the package smoke check and the bench's CPU-baseline leg use it.  It shares no
 * code, header, table or constant generator with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *  - "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max", section "What one token
 *    costs the bus" (the NVFP4/FP8 byte table) and section "Formats, and what runs where": NVFP4 is an
 *    E2M1 code, one FP8 E4M3 block scale per 16 weights and an FP32 tensor scale used as a
 *    MULTIPLIER; block-scale codes top out at exactly 448 (so E4M3 is the finite-only "FN" variant);
 *    arithmetic is weight-only with BF16 activations/residuals and FP32 (here: fp64) accumulation.
 *  - same page, section "The megakernel is per layer, not per step": the greedy acceptance scan
 *    (accept the longest prefix of drafts that equal the target's tokens, then commit the target's
 *    own token after it; a round commits 1..8 tokens).
 *  - "144 tok/s needs 502 GB/s" (Splash engine), section "The engine hard-codes the model": the
 *    geometry (64 layers, hidden 5120, vocab 248320, intermediate 17408, fullAttentionPeriod = 4).
 *  - "Beating Splash on an M5 Max", section "The bugs a second reviewer found": the argmax tie
 *    rule must be the same everywhere (here: lowest index among equal maxima).
 *  - "144 tok/s needs 502 GB/s", section "The engine hard-codes the model": the other engines'
 *    affine 4-bit format (32 bytes of codes + a bf16 scale + a bf16 bias per group of 64 inputs) --
 *    see orc_linear_q4().
 *
 * Readings where the pages are silent (the plainest choice the passages support):
 *  - E2M1 bit layout: bit 3 = sign, bits 2..1 = exponent (bias 1), bit 0 = mantissa (OCP MX).
 *  - Packing of two E2M1 codes per byte: element 2j is the LOW nibble of byte j.
 *  - Block scales run along K: scale[n][k/16].
 *  - Argmax: NaN is treated as -inf; -0 == +0; the lowest index among equal maxima wins.
 *  - Q4: unsigned codes, w = scale * q + bias, groups of 64 along K, low nibble first.
 *  - The verify-pass surrogate (mixer cores replaced by slices) -- see orc_verify_pass().
 *  - Sampled acceptance: candidates ordered by logit, ties to the lower index; top_p keeps the
 *    shortest prefix whose mass reaches top_p; a draw takes the first i whose cumulative weight
 *    exceeds u times the total; a zero residual draws from the target -- see orc_sample_accept().
 *  - Verify attention: scores q.k / sqrt(D); row j of a lane sees cache positions 0 .. ctx + j after
 *    the lane's 8 new keys are appended; q head h reads kv head h / (Hq / Hkv) -- see
 *    orc_attention_verify().
 *  - Gated DeltaNet: the published gated delta rule; the re-scan count is the lane's n_commit --
 *    see orc_gdn_scan().
 *  - Lookup drafts: the longest match of the history's suffix (at most max_match), the latest
 *    position among equals, its continuation then its last token repeated -- see orc_lookup_drafts().
 *
 * Pins: every building block (formats, linear, Q4, bf16 rounding, SiLU*up, RMSNorm, argmax,
 * acceptance, byte tables, the sampled-acceptance distribution, attention, the delta-rule scan,
 * the decode-loop pieces) is pinned by the tests against page values, closed forms, library
 * routines or brute force.  orc_verify_pass is pinned through its parts and an independent
 * composition on a tiny model; the long (64-layer) chain as a whole is parity unpinned -- end-to-end
 * comparisons against it check only decisions that are unique and report the drift.
 *
 * Everything is computed in fp64 from the plain definitions, with no blocking or reordering:
 * w[n][k] = e2m1(code) * e4m3(scale) * ts, y[m][n] = sum_k x[m][k] * w[n][k].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ formats */

/* E2M1 magnitudes for codes 0..7; codes 8..15 are their negatives (code 8 is -0). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1(int code) {
    code &= 15;
    double v = E2M1_MAG[code & 7];
    return (code & 8) ? -v : v;
}

/* E4M3 "FN": 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6);
 * S.1111.111 is NaN; there are no infinities, so the largest finite value is 1.75 * 2^8 = 448. */
double orc_e4m3(int byte) {
    byte &= 255;
    int s = byte >> 7, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

void orc_tables(double* e2m1_16, double* e4m3_256) {
    for (int c = 0; c < 16; ++c) e2m1_16[c] = orc_e2m1(c);
    for (int b = 0; b < 256; ++b) e4m3_256[b] = orc_e4m3(b);
}

/* bf16 bits -> value (exact). */
double orc_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

void orc_bf16_values(const uint16_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_value(in[i]);
}

/* fp64 -> bf16 with round-to-nearest-even, rounding once, directly from fp64. */
uint16_t orc_bf16_round1(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    frexp(a, &e);           /* a in [2^(e-1), 2^e) */
    int q = e - 8;          /* 8 significant bits -> quantum 2^(e-8) */
    if (q < -133) q = -133; /* bf16 subnormal quantum */
    double r = nearbyint(ldexp(a, -q)); /* default rounding mode: to nearest, ties to even */
    double rv = ldexp(r, q);
    if (rv >= 0x1p128) return sign | 0x7F80;
    float f = (float)rv; /* exact: rv has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

void orc_bf16_round(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round1(in[i]);
}

/* ------------------------------------------------------------------ threading */

typedef struct {
    void (*fn)(void* ctx, int64_t i);
    void* ctx;
    int64_t n;
    int tid, nthreads;
} orc_job;

static void* orc_job_run(void* p) {
    orc_job* j = (orc_job*)p;
    for (int64_t i = j->tid; i < j->n; i += j->nthreads) j->fn(j->ctx, i);
    return NULL;
}

/* Runs fn(ctx, i) for i in [0, n) on up to nthreads threads (rows are independent). */
static void orc_parallel(int nthreads, int64_t n, void (*fn)(void*, int64_t), void* ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    pthread_t th[256];
    orc_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].n = n; jobs[t].tid = t; jobs[t].nthreads = nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, orc_job_run, &jobs[t]) != 0) break;
        started = t;
    }
    orc_job_run(&jobs[0]);
    for (int t = started + 1; t < nthreads; ++t) orc_job_run(&jobs[t]); /* threads that failed to start */
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ linear layers */

/* Weight formats handled by orc_linear. */
enum { ORC_NVFP4 = 0, ORC_FP8 = 1 };

typedef struct {
    int fmt;
    const double* x; /* [M][K] activation values (bf16 values widened to fp64) */
    int M, K, N;
    const uint8_t* codes;  /* NVFP4: [N][K/2], element 2j = low nibble of byte j.  FP8: [N][K] */
    const uint8_t* scales; /* NVFP4: [N][K/16] E4M3 block scales; unused for FP8 */
    double ts;             /* NVFP4 tensor scale / FP8 per-tensor scale (a multiplier) */
    const int32_t* rows;   /* rows to compute (NULL = all N) */
    double* y;             /* [M][n_rows] */
    double* a;             /* [M][n_rows] sum |x*w| (may be NULL) */
    int64_t n_rows;
} orc_lin_ctx;

/* Dequantizes weight row n to fp64 by the definition, then forms the M dot products. */
static void orc_lin_row(void* p, int64_t i) {
    orc_lin_ctx* c = (orc_lin_ctx*)p;
    int64_t n = c->rows ? c->rows[i] : i;
    int K = c->K;
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
    if (!w) return;
    if (c->fmt == ORC_NVFP4) {
        const uint8_t* cr = c->codes + n * (int64_t)(K / 2);
        const uint8_t* sr = c->scales + n * (int64_t)(K / 16);
        for (int k = 0; k < K; ++k) {
            int byte = cr[k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            w[k] = orc_e2m1(code) * orc_e4m3(sr[k / 16]) * c->ts;
        }
    } else {
        const uint8_t* wr = c->codes + n * (int64_t)K;
        for (int k = 0; k < K; ++k) w[k] = orc_e4m3(wr[k]) * c->ts;
    }
    for (int m = 0; m < c->M; ++m) {
        const double* xr = c->x + (int64_t)m * K;
        double s = 0.0, sa = 0.0;
        for (int k = 0; k < K; ++k) {
            double p2 = xr[k] * w[k];
            s += p2;
            sa += fabs(p2);
        }
        c->y[(int64_t)m * c->n_rows + i] = s;
        if (c->a) c->a[(int64_t)m * c->n_rows + i] = sa;
    }
    free(w);
}

/* y[m][i] = sum_k x[m][k] * w[rows[i]][k] in fp64; a[m][i] = sum_k |x[m][k] * w[rows[i]][k]|.
 * x holds bf16 bit patterns [M][K].  Returns 0, or -1 on bad arguments. */
int orc_linear(int fmt, const uint16_t* x_bf16, int M, int K, int N, const uint8_t* codes,
               const uint8_t* scales, double ts, const int32_t* rows, int64_t n_rows, double* y,
               double* a, int nthreads) {
    if (M < 0 || K <= 0 || N <= 0 || !x_bf16 || !codes || !y) return -1;
    if (fmt == ORC_NVFP4 && (K % 16 != 0 || !scales)) return -1;
    if (fmt != ORC_NVFP4 && fmt != ORC_FP8) return -1;
    if (!rows) n_rows = N;
    for (int64_t i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= N) return -1;
    double* x = (double*)malloc(sizeof(double) * (size_t)M * (size_t)K + 8);
    if (!x) return -1;
    for (int64_t i = 0; i < (int64_t)M * K; ++i) x[i] = orc_bf16_value(x_bf16[i]);
    orc_lin_ctx c = {fmt, x, M, K, N, codes, scales, ts, rows, y, a, n_rows};
    orc_parallel(nthreads, n_rows, orc_lin_row, &c);
    free(x);
    return 0;
}

/* ------------------------------------------------------------------ affine INT4 ("Q4") linear
 *
 * "144 tok/s needs 502 GB/s, and Apple sells two M5 Max chips", section "The engine hard-codes the
 * model": the other engines' 4-bit format packs nine bytes per sixteen weights -- for every group of
 * 64 inputs, 32 bytes of 4-bit codes plus a bf16 scale and a bf16 bias.  Readings (the page gives no
 * formula): the code q is unsigned (0..15) and the weight is the affine map w = scale * q + bias;
 * groups run along K (scale[n][k/64]); element 2j is the low nibble of byte j (as for NVFP4).
 * "Beating Splash on an M5 Max", section "What actually moved the needle": the producers emit the
 * per-group input sums the Q4 tiles need -- that is an implementation route to the same y, not a
 * different result, so the oracle keeps the plain definition below. */

typedef struct {
    const double* x; /* [M][K] */
    int M, K, N;
    const uint8_t* codes;   /* [N][K/2] */
    const uint16_t* scales; /* [N][K/64] bf16 */
    const uint16_t* biases; /* [N][K/64] bf16 */
    const int32_t* rows;
    double* y;
    double* a; /* sum_k |x| (|scale * q| + |bias|): the magnitude of both terms of every weight */
    int64_t n_rows;
} orc_q4_ctx;

static void orc_q4_row(void* p, int64_t i) {
    orc_q4_ctx* c = (orc_q4_ctx*)p;
    int64_t n = c->rows ? c->rows[i] : i;
    int K = c->K;
    double* w = (double*)malloc(sizeof(double) * (size_t)K * 2);
    if (!w) return;
    double* wa = w + K;
    const uint8_t* cr = c->codes + n * (int64_t)(K / 2);
    const uint16_t* sr = c->scales + n * (int64_t)(K / 64);
    const uint16_t* br = c->biases + n * (int64_t)(K / 64);
    for (int k = 0; k < K; ++k) {
        int byte = cr[k / 2];
        int q = (k & 1) ? (byte >> 4) : (byte & 15);
        double sc = orc_bf16_value(sr[k / 64]), bi = orc_bf16_value(br[k / 64]);
        w[k] = sc * (double)q + bi;
        wa[k] = fabs(sc * (double)q) + fabs(bi);
    }
    for (int m = 0; m < c->M; ++m) {
        const double* xr = c->x + (int64_t)m * K;
        double s = 0.0, sa = 0.0;
        for (int k = 0; k < K; ++k) {
            s += xr[k] * w[k];
            sa += fabs(xr[k]) * wa[k];
        }
        c->y[(int64_t)m * c->n_rows + i] = s;
        if (c->a) c->a[(int64_t)m * c->n_rows + i] = sa;
    }
    free(w);
}

/* y[m][i] = sum_k x[m][k] * (scale * q + bias)[rows[i]][k] in fp64 (x: bf16 bit patterns [M][K]).
 * Returns 0, or -1 on bad arguments (K must be a multiple of 64). */
int orc_linear_q4(const uint16_t* x_bf16, int M, int K, int N, const uint8_t* codes, const uint16_t* scales,
                  const uint16_t* biases, const int32_t* rows, int64_t n_rows, double* y, double* a,
                  int nthreads) {
    if (M < 0 || K <= 0 || K % 64 != 0 || N <= 0 || !x_bf16 || !codes || !scales || !biases || !y) return -1;
    if (!rows) n_rows = N;
    for (int64_t i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= N) return -1;
    double* x = (double*)malloc(sizeof(double) * (size_t)M * (size_t)K + 8);
    if (!x) return -1;
    for (int64_t i = 0; i < (int64_t)M * K; ++i) x[i] = orc_bf16_value(x_bf16[i]);
    orc_q4_ctx c = {x, M, K, N, codes, scales, biases, rows, y, a, n_rows};
    orc_parallel(nthreads, n_rows, orc_q4_row, &c);
    free(x);
    return 0;
}

/* Packed bytes of an N x K Q4 matrix: per group of 64 weights, 32 bytes of codes + 2 + 2. */
int64_t orc_q4_bytes(int64_t N, int64_t K) { return N * (K / 64) * (32 + 2 + 2); }

/* ------------------------------------------------------------------ glue */

/* silu(g) = g / (1 + exp(-g)); out = silu(g) * u, fp64. */
void orc_silu_mul(const double* g, const double* u, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* RMSNorm with unit weight: r = bf16( h / sqrt(mean(h^2) + eps) ), per row, fp64 inside. */
void orc_rmsnorm(const uint16_t* h, int M, int D, double eps, uint16_t* r) {
    for (int m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int k = 0; k < D; ++k) {
            double v = orc_bf16_value(h[(int64_t)m * D + k]);
            ss += v * v;
        }
        double denom = sqrt(ss / (double)D + eps);
        for (int k = 0; k < D; ++k)
            r[(int64_t)m * D + k] = orc_bf16_round1(orc_bf16_value(h[(int64_t)m * D + k]) / denom);
    }
}

/* Lowest index of the maximum; NaN counts as -inf, and -0 == +0 (IEEE compare). */
int64_t orc_argmax(const double* v, int64_t n) {
    int64_t best = 0;
    double bv = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        double x = isnan(v[i]) ? -INFINITY : v[i];
        if (i == 0 || x > bv) {
            bv = x;
            best = i;
        }
    }
    return best;
}

/* Greedy acceptance per lane of R verify rows (the committed anchor token + R - 1 drafts).
 * t[R l + j] is the target's token at verify row j; pending[R l + j + 1] is draft j.
 * acc = number of leading drafts equal to the target's tokens (0..R-1);
 * n_commit = acc + 1 and committed[l][0..acc] = t[R l .. R l + acc] (accepted drafts, then the
 * target's own token); committed[l][acc+1..R-1] = -1.  The pages' verify has R = 8; lookup drafts
 * ("mlx-dspark", section "Lookup drafts") verify 16-32 rows. */
void orc_accept_rows(const int32_t* t, const int32_t* pending, int lanes, int R, int32_t* n_commit,
                     int32_t* committed) {
    for (int l = 0; l < lanes; ++l) {
        int base = R * l, acc = 0;
        while (acc < R - 1 && t[base + acc] == pending[base + acc + 1]) acc++;
        n_commit[l] = acc + 1;
        for (int j = 0; j < R; ++j) committed[R * l + j] = (j <= acc) ? t[base + j] : -1;
    }
}
void orc_accept(const int32_t* t, const int32_t* pending, int lanes, int32_t* n_commit,
                int32_t* committed) {
    orc_accept_rows(t, pending, lanes, 8, n_commit, committed);
}

/* ------------------------------------------------------------------ verify-pass surrogate */

/* Geometry of the pass.  Layer l is an attention layer when l % period == period - 1, otherwise a
 * Gated DeltaNet layer (fullAttentionPeriod = 4 on the Splash page). */
typedef struct {
    int n_layers, hidden, inter, vocab, period;
    int gdn_in, gdn_z;            /* GDN in-projection width (16384) and out-projection K (6144) */
    int attn_q, attn_kv, attn_z;  /* attention q (12288), kv (2048) widths, o-projection K (6144) */
    double eps;
} orc_geom;

/* Per layer, pointers in this order (canonical layouts, see orc_linear):
 *   [0] mixer in-projection  FP8 [gdn_in or attn_q][hidden]
 *   [1] attention kv         FP8 [attn_kv][hidden] (NULL on GDN layers; streamed, unused here)
 *   [2] mixer out-projection FP8 [hidden][gdn_z or attn_z]
 *   [3] gate codes [inter][hidden/2]  [4] gate scales [inter][hidden/16]
 *   [5] up codes                      [6] up scales
 *   [7] down codes [hidden][inter/2]  [8] down scales [hidden][inter/16]
 * and per layer the scales in this order: s_in, s_kv, s_out, ts_gate, ts_up, ts_down. */
#define ORC_PTRS_PER_LAYER 9
#define ORC_SCALES_PER_LAYER 6

static int orc_lin_bf16(int fmt, const uint16_t* x, int M, int K, int N, const uint8_t* codes,
                        const uint8_t* scales, double ts, double* y, int nthreads) {
    return orc_linear(fmt, x, M, K, N, codes, scales, ts, NULL, N, y, NULL, nthreads);
}

/*
 * The surrogate pass (mixer cores are outside the weight stream; the plainest shape-consistent
 * stand-in keeps every weight GEMM and replaces each core by a slice):
 *   h = x0
 *   for l in layers:
 *     r = RMSNorm(h)
 *     GDN:  u = FP8(in, r);  z = bf16(u[:, :gdn_z]);   h = bf16(h + FP8(out, z))
 *     attn: q = FP8(q, r);   (kv = FP8(kv, r) is streamed but unused);
 *           z = bf16(q[:, :attn_z]);                   h = bf16(h + FP8(o, z))
 *     r = RMSNorm(h);  a = bf16(silu(NVFP4(gate, r)) * NVFP4(up, r));  h = bf16(h + NVFP4(down, a))
 *   r = RMSNorm(h); logits = NVFP4(head, r); t = argmax per row; accept per lane.
 * Optional outputs: trace [2*n_layers][M][hidden] bf16 (h after each mixer block and each MLP
 * block), logits [M][vocab] fp64, final_r [M][hidden] bf16 (the head's input).
 */
int orc_verify_pass(const orc_geom* G, const uint8_t* const* layer_ptrs, const double* layer_scales,
                    const uint8_t* head_codes, const uint8_t* head_scales, double head_ts,
                    const uint16_t* x0, int M, const int32_t* pending, int32_t* argmax,
                    int32_t* n_commit, int32_t* committed, uint16_t* trace, double* logits_out,
                    uint16_t* final_r, int nthreads) {
    if (!G || M <= 0 || M % 8 != 0 || G->hidden % 16 || G->inter % 16) return -1;
    int H = G->hidden, I = G->inter, V = G->vocab;
    int wmax = G->gdn_in > G->attn_q ? G->gdn_in : G->attn_q;
    if (I > wmax) wmax = I;
    if (H > wmax) wmax = H;
    if (V > wmax) wmax = V;
    uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * H);
    uint16_t* r = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * H);
    uint16_t* z = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * wmax);
    double* y = (double*)malloc(sizeof(double) * (size_t)M * wmax);
    double* y2 = (double*)malloc(sizeof(double) * (size_t)M * wmax);
    int rc = -1;
    if (!h || !r || !z || !y || !y2) goto done;
    memcpy(h, x0, sizeof(uint16_t) * (size_t)M * H);
    for (int l = 0; l < G->n_layers; ++l) {
        const uint8_t* const* P = layer_ptrs + (int64_t)l * ORC_PTRS_PER_LAYER;
        const double* S = layer_scales + (int64_t)l * ORC_SCALES_PER_LAYER;
        int attn = (l % G->period) == G->period - 1;
        int n_in = attn ? G->attn_q : G->gdn_in;
        int kz = attn ? G->attn_z : G->gdn_z;
        /* mixer block */
        orc_rmsnorm(h, M, H, G->eps, r);
        if (orc_lin_bf16(ORC_FP8, r, M, H, n_in, P[0], NULL, S[0], y, nthreads)) goto done;
        for (int m = 0; m < M; ++m)
            for (int k = 0; k < kz; ++k) z[(int64_t)m * kz + k] = orc_bf16_round1(y[(int64_t)m * n_in + k]);
        if (orc_lin_bf16(ORC_FP8, z, M, kz, H, P[2], NULL, S[2], y, nthreads)) goto done;
        for (int64_t i = 0; i < (int64_t)M * H; ++i) h[i] = orc_bf16_round1(orc_bf16_value(h[i]) + y[i]);
        if (trace) memcpy(trace + (int64_t)(2 * l) * M * H, h, sizeof(uint16_t) * (size_t)M * H);
        /* MLP block */
        orc_rmsnorm(h, M, H, G->eps, r);
        if (orc_lin_bf16(ORC_NVFP4, r, M, H, I, P[3], P[4], S[3], y, nthreads)) goto done;
        if (orc_lin_bf16(ORC_NVFP4, r, M, H, I, P[5], P[6], S[4], y2, nthreads)) goto done;
        orc_silu_mul(y, y2, (int64_t)M * I, y);
        orc_bf16_round(y, z, (int64_t)M * I);
        if (orc_lin_bf16(ORC_NVFP4, z, M, I, H, P[7], P[8], S[5], y, nthreads)) goto done;
        for (int64_t i = 0; i < (int64_t)M * H; ++i) h[i] = orc_bf16_round1(orc_bf16_value(h[i]) + y[i]);
        if (trace) memcpy(trace + (int64_t)(2 * l + 1) * M * H, h, sizeof(uint16_t) * (size_t)M * H);
    }
    orc_rmsnorm(h, M, H, G->eps, r);
    if (final_r) memcpy(final_r, r, sizeof(uint16_t) * (size_t)M * H);
    {
        double* lg = logits_out ? logits_out : (double*)malloc(sizeof(double) * (size_t)M * V);
        if (!lg) goto done;
        if (orc_lin_bf16(ORC_NVFP4, r, M, H, V, head_codes, head_scales, head_ts, lg, nthreads)) {
            if (!logits_out) free(lg);
            goto done;
        }
        int32_t* t = (int32_t*)malloc(sizeof(int32_t) * (size_t)M);
        for (int m = 0; m < M; ++m) t[m] = (int32_t)orc_argmax(lg + (int64_t)m * V, V);
        for (int m = 0; m < M; ++m) argmax[m] = t[m];
        orc_accept(t, pending, M / 8, n_commit, committed);
        free(t);
        if (!logits_out) free(lg);
    }
    rc = 0;
done:
    free(h); free(r); free(z); free(y); free(y2);
    return rc;
}

/* ------------------------------------------------------------------ byte counts */

/* Bytes one NVFP4 matrix streams: N*K/2 code bytes + N*K/16 scale bytes (9 bytes per 16 weights). */
int64_t orc_nvfp4_code_bytes(int64_t N, int64_t K) { return N * K / 2; }
int64_t orc_nvfp4_scale_bytes(int64_t N, int64_t K) { return N * K / 16; }
int64_t orc_fp8_bytes(int64_t N, int64_t K) { return N * K; }

/* ------------------------------------------------------------------ verify attention over a KV cache
 *
 * "lithos-metal ...", section "The megakernel is per layer, not per step" (the full-attention figure
 * and the text after it): the attention core reads and appends a BF16 KV cache, runs a causal
 * softmax of q k^T weighting V, multiplies by the sigmoid of the gate, and the KV range is split
 * into partitions whose online-softmax partials are merged.  The partitions are an implementation
 * route to the same result, so the oracle computes the plain definition.  Readings: scores are
 * q . k / sqrt(D); the verify rows of lane l append their keys / values at positions
 * ctx[l] .. ctx[l] + 7 and row j sees positions 0 .. ctx[l] + j; q heads h share kv head
 * h / (Hq / Hkv); q and k arrive normalised and rotated (the page's Q/K RMSNorm and RoPE are
 * elementwise steps before this one).
 *
 * q, gate: bf16 [M][Hq][D]; k_new, v_new: bf16 [M][Hkv][D]; k_cache, v_cache: bf16
 * [L][Hkv][cap][D] holding positions 0 .. ctx[l] - 1; out, a: fp64 [M][Hq][D] with
 * a = sum_t p_t |v_t| * |sigmoid(gate)| (tolerance scale).  gate may be NULL (no gating). */
static double orc_bf(const uint16_t* p, int64_t i) { return orc_bf16_value(p[i]); }

int orc_attention_verify(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new, const uint16_t* k_cache,
                         const uint16_t* v_cache, const int32_t* ctx, int cap, const uint16_t* gate, int M, int Hq,
                         int Hkv, int D, double* out, double* a) {
    if (M < 8 || M % 8 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1 || !q || !k_new || !v_new || !k_cache ||
        !v_cache || !ctx || !out)
        return -1;
    const int G = Hq / Hkv, L = M / 8;
    for (int l = 0; l < L; ++l)
        if (ctx[l] < 0 || ctx[l] + 8 > cap) return -1;
    const double scale = 1.0 / sqrt((double)D);
    double* sc = (double*)malloc(sizeof(double) * ((size_t)cap + 8));
    if (!sc) return -1;
    for (int r = 0; r < M; ++r) {
        const int l = r / 8, j = r % 8, n = ctx[l] + j + 1;
        for (int h = 0; h < Hq; ++h) {
            const int g = h / G;
            const uint16_t* qr = q + ((int64_t)r * Hq + h) * D;
            /* key / value of position t for this lane and kv head */
            #define ORC_K(t, d) ((t) < ctx[l] ? orc_bf(k_cache, (((int64_t)l * Hkv + g) * cap + (t)) * D + (d)) \
                                              : orc_bf(k_new, ((int64_t)(8 * l + (t) - ctx[l]) * Hkv + g) * D + (d)))
            #define ORC_V(t, d) ((t) < ctx[l] ? orc_bf(v_cache, (((int64_t)l * Hkv + g) * cap + (t)) * D + (d)) \
                                              : orc_bf(v_new, ((int64_t)(8 * l + (t) - ctx[l]) * Hkv + g) * D + (d)))
            double mx = -INFINITY;
            for (int t = 0; t < n; ++t) {
                double s = 0.0;
                for (int d = 0; d < D; ++d) s += orc_bf(qr, d) * ORC_K(t, d);
                sc[t] = s * scale;
                if (sc[t] > mx) mx = sc[t];
            }
            double den = 0.0;
            for (int t = 0; t < n; ++t) {
                sc[t] = exp(sc[t] - mx);
                den += sc[t];
            }
            for (int d = 0; d < D; ++d) {
                double o = 0.0, oa = 0.0;
                for (int t = 0; t < n; ++t) {
                    const double v = ORC_V(t, d);
                    o += sc[t] * v;
                    oa += sc[t] * fabs(v);
                }
                double gt = 1.0;
                if (gate) gt = 1.0 / (1.0 + exp(-orc_bf(gate, ((int64_t)r * Hq + h) * D + d)));
                out[((int64_t)r * Hq + h) * D + d] = o / den * gt;
                if (a) a[((int64_t)r * Hq + h) * D + d] = oa / den * gt;
            }
            #undef ORC_K
            #undef ORC_V
        }
    }
    free(sc);
    return 0;
}

/* ------------------------------------------------------------------ Gated DeltaNet verify scan
 *
 * "Beating Splash on an M5 Max", section "What actually moved the needle": the fused GatedDeltaNet
 * step writes out of place from parity buffer A to parity buffer B; rejecting part of a round
 * re-scans only the committed rows from the still-intact A, and the state after every possible
 * number of kept tokens must match a reference scan exactly.  "lithos-metal ...", sections "What one
 * token costs the bus" (fp32 state (v_heads, dk, dv), 48 x 128 x 128 per layer) and "The megakernel
 * is per layer, not per step" (the commit pass recomputes the recurrence over the committed tokens,
 * whose count the accept scan wrote).  The pages name the layer (Gated DeltaNet) but do not print its
 * recurrence; the oracle takes the published gated delta rule (Yang, Kautz and Hatamizadeh, "Gated
 * Delta Networks: Improving Mamba2 with Delta Rule", 2024), per head with S a dv x dk matrix:
 *   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,   o_t = S_t q_t
 * (= S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T).  Readings: one q / k per v head;
 * q, k, v arrive after the layer's short convolution, activation and normalisation, and alpha, beta
 * after their gates (all producer steps); lane l scans its first rows[l] verify rows (8 for the
 * verify pass, the committed count for the re-scan).
 *
 * state_in, state_out: [L][H][dv][dk] (fp64 here); q, k: bf16 [M][H][dk]; v: bf16 [M][H][dv];
 * alpha, beta: [M][H]; out: [M][H][dv] (rows past rows[l] are left untouched). */
int orc_gdn_scan(const double* state_in, double* state_out, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                 const double* alpha, const double* beta, const int32_t* rows, int M, int H, int dk, int dv,
                 double* out) {
    if (M < 8 || M % 8 || H < 1 || dk < 1 || dv < 1 || !state_in || !state_out || !q || !k || !v || !alpha || !beta ||
        !rows)
        return -1;
    const int L = M / 8;
    double* u = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!u) return -1;
    for (int l = 0; l < L; ++l) {
        if (rows[l] < 0 || rows[l] > 8) { free(u); return -1; }
        for (int h = 0; h < H; ++h) {
            const int64_t so = ((int64_t)l * H + h) * dv * dk;
            double* S = state_out + so;
            memcpy(S, state_in + so, sizeof(double) * (size_t)dv * dk);
            for (int j = 0; j < rows[l]; ++j) {
                const int r = 8 * l + j;
                const uint16_t* kr = k + ((int64_t)r * H + h) * dk;
                const uint16_t* qr = q + ((int64_t)r * H + h) * dk;
                const uint16_t* vr = v + ((int64_t)r * H + h) * dv;
                const double a = alpha[(int64_t)r * H + h], b = beta[(int64_t)r * H + h];
                for (int i = 0; i < dv; ++i) {
                    double sk = 0.0;
                    for (int c = 0; c < dk; ++c) sk += S[(int64_t)i * dk + c] * orc_bf16_value(kr[c]);
                    u[i] = b * (orc_bf16_value(vr[i]) - a * sk);
                }
                for (int i = 0; i < dv; ++i)
                    for (int c = 0; c < dk; ++c)
                        S[(int64_t)i * dk + c] = a * S[(int64_t)i * dk + c] + u[i] * orc_bf16_value(kr[c]);
                if (out)
                    for (int i = 0; i < dv; ++i) {
                        double o = 0.0;
                        for (int c = 0; c < dk; ++c) o += S[(int64_t)i * dk + c] * orc_bf16_value(qr[c]);
                        out[((int64_t)r * H + h) * dv + i] = o;
                    }
            }
        }
    }
    free(u);
    return 0;
}

/* ------------------------------------------------------------------ decode loop pieces
 *
 * "lithos-metal ...", section "What one token costs the bus": the embedding is a gather of the
 * 4-bit table (the pass streams everything else).  "Speculative decoding" (mlx-dspark), sections
 * "Lookup (no drafter)" and "Lookup drafts": when the text being written already appeared earlier in
 * the context, the continuation of that earlier match is a free draft.  "The megakernel is per
 * layer, not per step": a round commits 1..8 tokens.  Readings: the embedding row is NVFP4 in the
 * canonical layout, x = bf16(e2m1 * e4m3 * ts) rounded once; the lookup takes the earlier position p
 * (continuation hist[p..]) whose preceding tokens match the history's last tokens for the most
 * positions (up to max_match), the most recent among equals, a match of at least one token; the 7
 * drafts are hist[p], hist[p+1], ... while p + j < T, then the last one repeated; with no match the
 * drafts are the anchor repeated; the anchor is the last committed token hist[T-1]. */

void orc_embed_nvfp4(const uint8_t* codes, const uint8_t* scales, double ts, const int32_t* tokens, int M, int K,
                     uint16_t* out) {
    for (int m = 0; m < M; ++m) {
        const int64_t t = tokens[m];
        for (int k = 0; k < K; ++k) {
            int byte = codes[t * (K / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            out[(int64_t)m * K + k] = orc_bf16_round1(orc_e2m1(code) * orc_e4m3(scales[t * (K / 16) + k / 16]) * ts);
        }
    }
}

/* Lane l: history hist[l * cap .. + T), T = hist_len[l] >= 1; writes pending[R l .. R l + R - 1]:
 * the anchor, then R - 1 drafts. */
void orc_lookup_drafts_rows(const int32_t* hist, const int32_t* hist_len, int L, int cap, int max_match, int R,
                            int32_t* pending) {
    for (int l = 0; l < L; ++l) {
        const int32_t* h = hist + (int64_t)l * cap;
        const int T = hist_len[l];
        int best_p = -1, best_len = 0;
        for (int p = 1; p < T; ++p) {  /* continuation starts at p; match hist[p-1-i] == hist[T-1-i] */
            int len = 0;
            while (len < max_match && p - 1 - len >= 0 && h[p - 1 - len] == h[T - 1 - len]) len++;
            if (len >= 1 && len >= best_len) { best_len = len; best_p = p; }  /* ties: the later p */
        }
        const int32_t anchor = h[T - 1];
        pending[R * l] = anchor;
        int32_t last = anchor;
        for (int j = 0; j < R - 1; ++j) {
            if (best_p >= 0 && best_p + j < T) last = h[best_p + j];
            pending[R * l + 1 + j] = last;
        }
    }
}
void orc_lookup_drafts(const int32_t* hist, const int32_t* hist_len, int L, int cap, int max_match,
                       int32_t* pending) {
    orc_lookup_drafts_rows(hist, hist_len, L, cap, max_match, 8, pending);
}

/* Appends committed[l][0 .. n_commit[l]) (rows of R entries) to lane l's history; returns -1 if one
 * would not fit. */
int orc_commit_append_rows(int32_t* hist, int32_t* hist_len, int L, int cap, int R, const int32_t* n_commit,
                           const int32_t* committed) {
    int rc = 0;
    for (int l = 0; l < L; ++l) {
        const int n = n_commit[l];
        if (hist_len[l] + n > cap) { rc = -1; continue; }
        for (int j = 0; j < n; ++j) hist[(int64_t)l * cap + hist_len[l] + j] = committed[R * l + j];
        hist_len[l] += n;
    }
    return rc;
}
int orc_commit_append(int32_t* hist, int32_t* hist_len, int L, int cap, const int32_t* n_commit,
                      const int32_t* committed) {
    return orc_commit_append_rows(hist, hist_len, L, cap, 8, n_commit, committed);
}

/* Probability the draft gave token t (0 when t is not among its 16 candidates). */
static double orc_q_of(const int32_t* dt, const double* dp, int32_t t) {
    for (int i = 0; i < 16; ++i) if (dt[i] == t) return dp[i];
    return 0.0;
}

/* ------------------------------------------------------------------ sampled acceptance
 *
 * "144 tok/s needs 502 GB/s", section "Exact, up to top-32": the acceptance test is standard
 * speculative sampling -- accept a draft token when u * q < p, else draw from max(p - q, 0) -- so the
 * output follows the target's distribution; the target's probabilities are temperature over its first
 * top_k (<= 32) entries, truncated by top_p, renormalised; a token outside those candidates has
 * probability zero.  "lithos-metal ...", section "How DSpark is wired in": with a greedy drafter the
 * draft is a point mass (q = 1 on the drafted token).  "Beating Splash on an M5 Max", section "What
 * actually moved the needle": one GPU kernel over the verify logits applies top-k and top-p, samples
 * and runs the acceptance rule.
 * Readings (the pages give the rule, not these details): candidates are ordered by logit, larger
 * first, ties to the lower token index; top_p keeps the shortest prefix whose mass reaches top_p; a
 * draw with uniform u from weights w over that order takes the first i with u * sum(w) < w_0 + .. + w_i;
 * if the residual max(p - q, 0) is zero everywhere (p == q) the draw is from p; the draft's
 * distribution for draft j of lane l is given as 16 (token, probability) pairs at row 8l + j, and a
 * token not among them has q = 0; the uniforms are inputs, two per row: u[r][0] for the test of the
 * draft checked at row r, u[r][1] for the draw at row r. */

/* The target distribution of one row: its top_k candidates in order, probabilities after
 * temperature, top_p and renormalisation.  Returns the number kept (1..top_k); *margin = the smallest
 * distance of a running mass to top_p (how close the truncation was to flipping). */
int orc_target_dist(const double* logits, int V, double temperature, int top_k, double top_p, int32_t* tok,
                    double* prob, double* margin) {
    if (V < 1 || top_k < 1 || top_k > 32 || top_k > V || !(temperature > 0.0) || !(top_p > 0.0)) return 0;
    int32_t best[32];
    double bv[32];
    int n = 0;
    /* top_k by insertion: larger logit first, the lower index first among equals; NaN as -inf */
    for (int i = 0; i < V; ++i) {
        double v = isnan(logits[i]) ? -INFINITY : logits[i];
        int pos = n;
        while (pos > 0 && v > bv[pos - 1]) pos--;
        if (pos >= top_k) continue;
        if (n < top_k) n++;
        for (int j = n - 1; j > pos; --j) { bv[j] = bv[j - 1]; best[j] = best[j - 1]; }
        bv[pos] = v;
        best[pos] = i;
    }
    double e[32], sum = 0.0;
    for (int i = 0; i < n; ++i) {
        e[i] = exp((bv[i] - bv[0]) / temperature);
        sum += e[i];
    }
    double cum = 0.0, mg = INFINITY;
    int keep = n;
    for (int i = 0; i < n; ++i) {
        cum += e[i] / sum;
        double d = fabs(cum - top_p);
        if (d < mg) mg = d;
        if (cum >= top_p) { keep = i + 1; break; }
    }
    double ksum = 0.0;
    for (int i = 0; i < keep; ++i) ksum += e[i];
    for (int i = 0; i < keep; ++i) { tok[i] = best[i]; prob[i] = e[i] / ksum; }
    if (margin) *margin = top_p >= 1.0 ? INFINITY : mg;
    return keep;
}

/* First i with u * W < w_0 + .. + w_i (W = the sum); *margin = distance of u * W to the nearest
 * boundary, relative to W. */
static int orc_draw(const double* w, int n, double u, double* margin) {
    double W = 0.0;
    for (int i = 0; i < n; ++i) W += w[i];
    double t = u * W, cum = 0.0;
    int pick = n - 1;
    double mg = INFINITY;
    for (int i = 0; i < n; ++i) {
        cum += w[i];
        double d = fabs(cum - t) / W;
        if (d < mg) mg = d;
        if (t < cum) { pick = i; break; }
    }
    if (margin) *margin = mg;
    return pick;
}

/* Per lane: speculative sampling of the 7 drafts against the target rows, then the bonus draw.
 * logits [M][V] (the GPU's fp32 values, widened); draft_tokens / draft_probs [M][16] or NULL
 * (point mass on each draft); uniforms [M][2].  margin[l] = the smallest margin of the lane's
 * decisions (acceptance tests |u q - p|, draws, top_p truncations).  Returns 0, or -1 on bad args. */
int orc_sample_accept(const double* logits, int M, int V, double temperature, int top_k, double top_p,
                      const int32_t* pending, const int32_t* draft_tokens, const double* draft_probs,
                      const double* uniforms, int32_t* n_commit, int32_t* committed, double* margin) {
    if (M < 8 || M % 8 || V < 1 || top_k < 1 || top_k > 32 || top_k > V || !(temperature > 0.0) ||
        !(top_p > 0.0) || !logits || !pending || !uniforms || !n_commit || !committed)
        return -1;
    for (int l = 0; l < M / 8; ++l) {
        double mg = INFINITY;
        int acc = 0, last = -1;
        for (int j = 0; j <= 7; ++j) {
            const int r = 8 * l + j;
            int32_t tok[32];
            double p[32], tm;
            const int n = orc_target_dist(logits + (int64_t)r * V, V, temperature, top_k, top_p, tok, p, &tm);
            if (tm < mg) mg = tm;
            double w[32], dm;
            if (j == 7) { /* all drafts accepted: the bonus token from p */
                last = tok[orc_draw(p, n, uniforms[2 * r + 1], &dm)];
                if (dm < mg) mg = dm;
                break;
            }
            const int32_t d = pending[8 * l + j + 1];
            double pd = 0.0, qd;
            for (int i = 0; i < n; ++i) if (tok[i] == d) pd = p[i];
            /* q of a token under the draft's distribution at this row */
            #define ORC_Q(t) (draft_probs ? orc_q_of(draft_tokens + (int64_t)r * 16, draft_probs + (int64_t)r * 16, (t)) \
                                          : ((t) == d ? 1.0 : 0.0))
            qd = ORC_Q(d);
            const double a = uniforms[2 * r] * qd;
            if (fabs(a - pd) < mg) mg = fabs(a - pd);
            if (a < pd) { acc++; continue; }
            double W = 0.0;
            for (int i = 0; i < n; ++i) { w[i] = fmax(p[i] - ORC_Q(tok[i]), 0.0); W += w[i]; }
            #undef ORC_Q
            const int pick = W > 0.0 ? orc_draw(w, n, uniforms[2 * r + 1], &dm) : orc_draw(p, n, uniforms[2 * r + 1], &dm);
            if (dm < mg) mg = dm;
            last = tok[pick];
            break;
        }
        n_commit[l] = acc + 1;
        for (int j = 0; j < 8; ++j)
            committed[8 * l + j] = j < acc ? pending[8 * l + j + 1] : (j == acc ? last : -1);
        if (margin) margin[l] = mg;
    }
    return 0;
}

/* Per-pass byte groups of the pass geometry, in the page's table order:
 * out[0] MLP codes, out[1] MLP block scales, out[2] GDN FP8, out[3] attention FP8, out[4] head
 * (codes + scales), out[5] total. */
void orc_pass_bytes(const orc_geom* G, int64_t* out) {
    int64_t H = G->hidden, I = G->inter;
    int64_t n_attn = 0, n_gdn = 0;
    for (int l = 0; l < G->n_layers; ++l) {
        if ((l % G->period) == G->period - 1) n_attn++;
        else n_gdn++;
    }
    int64_t L = G->n_layers;
    out[0] = L * (2 * orc_nvfp4_code_bytes(I, H) + orc_nvfp4_code_bytes(H, I));
    out[1] = L * (2 * orc_nvfp4_scale_bytes(I, H) + orc_nvfp4_scale_bytes(H, I));
    out[2] = n_gdn * (orc_fp8_bytes(G->gdn_in, H) + orc_fp8_bytes(H, G->gdn_z));
    out[3] = n_attn * (orc_fp8_bytes(G->attn_q, H) + orc_fp8_bytes(G->attn_kv, H) +
                       orc_fp8_bytes(H, G->attn_z));
    out[4] = orc_nvfp4_code_bytes(G->vocab, H) + orc_nvfp4_scale_bytes(G->vocab, H);
    out[5] = out[0] + out[1] + out[2] + out[3] + out[4];
}
