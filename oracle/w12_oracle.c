/*
 * W12 tree-verify ORACLE -- test infrastructure only.
 *
 * A plain, slow, single-source CPU implementation of what the verify pass
 * computes.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only through the seeded input generators.
 *
 * Sources (SpecPilot explainer, jaehun.me; SpecPilot summary, agihunt.info):
 *   - W12 format: explainer "4.1 W12: a 12-bit lossless weight format" and the
 *     summary's W12 paragraph: per output channel a window of 16 binades,
 *     in-window weights kept as sign + 4-bit exponent offset + 7 mantissa
 *     bits, everything else on a per-channel escape list restored exactly;
 *     12 KB records of 128x64 weights, first 8 KB the 8-bit view, last 4 KB
 *     the low mantissa bits.
 *   - Verify GEMM and LM-head argmax: explainer "1.1" (one row per token,
 *     target argmax per row) and "2.1".
 *   - Best-first tree under a shared budget: explainer "4.2" (path score is
 *     the sum of log p(child | parent)) and "4.4" (one budget shared by all
 *     requests, filled by highest path log-probability, prefix-closed).
 *   - Greedy acceptance: explainer "1.1" (accept the longest prefix equal to
 *     the target's argmax, then append that argmax as a bonus).
 *
 * Readings of points the pages leave open (each also listed in the design
 * notes):
 *   R1  window coordinate is the BF16 biased exponent field e in [1,254];
 *       the window is [b, b+15] with b in [1,239].
 *   R2  b maximises the number of the channel's normal weights inside the
 *       window; ties go to the largest b; no normal weights -> b = 1.
 *   R3  a weight escapes iff e < b or e > b+15 (this covers zeros,
 *       denormals, Inf and NaN); the escape keeps all 16 BF16 bits.
 *   R4  view byte = [sign:1][offset:4][mantissa high 3]; the low plane keeps
 *       the low 4 mantissa bits.
 *   R5  an escaped slot stores a zero 12-bit code.
 *   R6  record = 128 channels x 64 K; tiles ordered n-tile major.
 *       Inside the 8 KB view plane: four 16-K groups, each 128 channels x
 *       16 bytes; inside a 16-byte chunk weight kk (0..15) sits at byte
 *       pos(kk) = 4*((kk%8)/2) + 2*(kk/8) + kk%2.  Inside the 4 KB low plane:
 *       two 32-K groups, each 128 channels x 16 bytes; weight kk of the
 *       first 16 K of the group is the low nibble of byte pos(kk), weight kk
 *       of the second 16 K the high nibble.
 *   R7  escape index: esc_tile_off[tiles+1] (prefix counts per record) and
 *       entries u32 = n_local<<22 | k_local<<16 | bf16 sorted by
 *       (n_local, k_local) inside each record.
 *   R9  argmax ties go to the lowest index; NaN never wins.
 *   R11 the lattice gives log-probabilities; edge score = logp[pos][cand]
 *       (or logp[pos][parent rank][cand] for a parent-conditioned lattice,
 *       the root using parent rank 0).  Path score is accumulated in FP32,
 *       root to leaf.
 *   R12 the budget counts every request's root row (score 0, depth 0).
 *   R13 order key: score desc, depth asc, request asc, path asc (path = the
 *       candidate ranks from the root, 4 bits each, most significant first).
 *       Rows are emitted grouped by request, best-first inside a request.
 *   R14 a child at depth d uses position d (1-based); depth <= P_r.
 *   R15 chain mode = only rank-0 candidates (n_cand = 1).
 *   R16 if two accepted siblings had the same token the lowest row wins.
 *   R19 quick pass: in-window weights from the view byte with the four low
 *       mantissa bits set to 0b1000; escaped weights exact.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)

#define TILE_N 128
#define TILE_K 64
#define REC_BYTES 12288
#define VIEW_BYTES 8192

/* ------------------------------------------------------------------------ */
/* BF16 helpers                                                              */
/* ------------------------------------------------------------------------ */

static int bf16_exp(uint16_t h) { return (h >> 7) & 0xFF; }

static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* position of weight kk (0..15) inside a 16-byte chunk (R6) */
static int chunk_pos(int kk) { return 4 * ((kk % 8) / 2) + 2 * (kk / 8) + (kk % 2); }

/* ------------------------------------------------------------------------ */
/* W12: window choice, pack, unpack                                          */
/* ------------------------------------------------------------------------ */

/* R2: the window base for one channel. */
static int choose_base(const uint16_t *row, int64_t k)
{
    int64_t hist[256];
    memset(hist, 0, sizeof hist);
    int64_t normals = 0;
    for (int64_t i = 0; i < k; ++i) {
        int e = bf16_exp(row[i]);
        if (e >= 1 && e <= 254) {
            hist[e]++;
            normals++;
        }
    }
    if (normals == 0) return 1;
    int best_b = 1;
    int64_t best = -1;
    for (int b = 1; b <= 239; ++b) {
        int64_t cnt = 0;
        for (int e = b; e <= b + 15; ++e) cnt += hist[e];
        if (cnt >= best) { /* ">=": ties move to the larger b */
            best = cnt;
            best_b = b;
        }
    }
    return best_b;
}

static int is_escape(uint16_t h, int b)
{
    int e = bf16_exp(h);
    return e < b || e > b + 15;
}

/* Window bases for every channel and the total escape count. */
int orc_w12_layout(const uint16_t *w, int64_t n, int64_t k, uint8_t *base, int64_t *n_escapes)
{
    if (!w || !base || !n_escapes || n <= 0 || k <= 0 || n % TILE_N || k % TILE_K) return ORC_EINVAL;
    int64_t cnt = 0;
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t *row = w + i * k;
        int b = choose_base(row, k);
        base[i] = (uint8_t)b;
        for (int64_t j = 0; j < k; ++j) cnt += is_escape(row[j], b);
    }
    *n_escapes = cnt;
    return ORC_OK;
}

/* Byte offsets inside a record for (channel c, K index kl). */
static int64_t view_off(int c, int kl) { return (int64_t)((kl / 16) * TILE_N + c) * 16 + chunk_pos(kl % 16); }
static int64_t nib_off(int c, int kl) { return VIEW_BYTES + (int64_t)((kl / 32) * TILE_N + c) * 16 + chunk_pos(kl % 16); }
static int nib_shift(int kl) { return ((kl % 32) / 16) * 4; }

int orc_w12_pack(const uint16_t *w, int64_t n, int64_t k, const uint8_t *base, uint8_t *rec,
                 int32_t *esc_tile_off, uint32_t *esc)
{
    if (!w || !base || !rec || !esc_tile_off || n <= 0 || k <= 0 || n % TILE_N || k % TILE_K) return ORC_EINVAL;
    int64_t nt_count = n / TILE_N, kt_count = k / TILE_K;
    int64_t e_idx = 0;
    memset(rec, 0, (size_t)(nt_count * kt_count * REC_BYTES));
    for (int64_t nt = 0; nt < nt_count; ++nt) {
        for (int64_t kt = 0; kt < kt_count; ++kt) {
            int64_t t = nt * kt_count + kt;
            uint8_t *r = rec + t * REC_BYTES;
            esc_tile_off[t] = (int32_t)e_idx;
            for (int c = 0; c < TILE_N; ++c) {
                int64_t ch = nt * TILE_N + c;
                int b = base[ch];
                for (int kl = 0; kl < TILE_K; ++kl) {
                    uint16_t h = w[ch * k + kt * TILE_K + kl];
                    if (is_escape(h, b)) {
                        /* R5: the slot keeps a zero code; R7: the entry keeps all bits */
                        if (esc) esc[e_idx] = ((uint32_t)c << 22) | ((uint32_t)kl << 16) | h;
                        e_idx++;
                        continue;
                    }
                    int s = h >> 15;
                    int o = bf16_exp(h) - b;
                    int m = h & 0x7F;
                    r[view_off(c, kl)] = (uint8_t)((s << 7) | (o << 3) | (m >> 4));
                    r[nib_off(c, kl)] |= (uint8_t)((m & 0xF) << nib_shift(kl));
                }
            }
        }
    }
    esc_tile_off[nt_count * kt_count] = (int32_t)e_idx;
    return ORC_OK;
}

/* Decode rows [row0, row0+nrows) of a packed tensor to BF16 bits. */
int orc_w12_unpack_rows(const uint8_t *rec, const uint8_t *base, const int32_t *esc_tile_off,
                        const uint32_t *esc, int64_t n, int64_t k, int64_t row0, int64_t nrows,
                        uint16_t *out)
{
    if (!rec || !base || !esc_tile_off || !out || n % TILE_N || k % TILE_K || row0 < 0 || nrows < 0 ||
        row0 + nrows > n)
        return ORC_EINVAL;
    int64_t kt_count = k / TILE_K;
    for (int64_t ch = row0; ch < row0 + nrows; ++ch) {
        int64_t nt = ch / TILE_N;
        int c = (int)(ch % TILE_N);
        int b = base[ch];
        for (int64_t kt = 0; kt < kt_count; ++kt) {
            int64_t t = nt * kt_count + kt;
            const uint8_t *r = rec + t * REC_BYTES;
            for (int kl = 0; kl < TILE_K; ++kl) {
                int v = r[view_off(c, kl)];
                int ml = (r[nib_off(c, kl)] >> nib_shift(kl)) & 0xF;
                int s = v >> 7, o = (v >> 3) & 0xF, mh = v & 7;
                uint16_t h = (uint16_t)((s << 15) | ((b + o) << 7) | (mh << 4) | ml);
                out[(ch - row0) * k + kt * TILE_K + kl] = h;
            }
            /* restore the escaped slots of this channel in this record */
            for (int32_t e = esc_tile_off[t]; e < esc_tile_off[t + 1]; ++e) {
                uint32_t en = esc[e];
                int nl = (int)(en >> 22) & 0x7F, kl = (int)(en >> 16) & 0x3F;
                if (nl != c) continue;
                out[(ch - row0) * k + kt * TILE_K + kl] = (uint16_t)(en & 0xFFFF);
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* FP64 GEMM and the argmax over an LM head                                  */
/* ------------------------------------------------------------------------ */

static int pick_threads(int nthreads)
{
    if (nthreads > 0) return nthreads;
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

typedef struct {
    const uint16_t *x, *w;
    int64_t R, n, k, n0, n1;
    double *y;
} gemm_job;

static void *gemm_worker(void *p)
{
    gemm_job *j = (gemm_job *)p;
    for (int64_t c = j->n0; c < j->n1; ++c) {
        const uint16_t *wr = j->w + c * j->k;
        for (int64_t r = 0; r < j->R; ++r) {
            const uint16_t *xr = j->x + r * j->k;
            double acc = 0.0;
            for (int64_t i = 0; i < j->k; ++i) acc += bf16_to_double(xr[i]) * bf16_to_double(wr[i]);
            j->y[r * j->n + c] = acc;
        }
    }
    return NULL;
}

/* R19: the quick pass (explainer 4.1 "the 8-bit view is what the Q pass reads";
 * 4.3: the Q pass reads the view nested in the record with the discarded
 * mantissa bits set to the midpoint).  In-window weights keep sign, exponent
 * and the three high mantissa bits from the view byte and take 0b1000 as the
 * low four; escaped weights keep their exact value (the escape list is part
 * of the record's weight and is read as is). */
int orc_w12_unpack_rows_q(const uint8_t *rec, const uint8_t *base, const int32_t *esc_tile_off,
                          const uint32_t *esc, int64_t n, int64_t k, int64_t row0, int64_t nrows,
                          uint16_t *out)
{
    if (!rec || !base || !esc_tile_off || !out || n % TILE_N || k % TILE_K || row0 < 0 || nrows < 0 ||
        row0 + nrows > n)
        return ORC_EINVAL;
    int64_t kt_count = k / TILE_K;
    for (int64_t ch = row0; ch < row0 + nrows; ++ch) {
        int64_t nt = ch / TILE_N;
        int c = (int)(ch % TILE_N);
        int b = base[ch];
        for (int64_t kt = 0; kt < kt_count; ++kt) {
            int64_t t = nt * kt_count + kt;
            const uint8_t *r = rec + t * REC_BYTES;
            for (int kl = 0; kl < TILE_K; ++kl) {
                int v = r[view_off(c, kl)];
                int s = v >> 7, o = (v >> 3) & 0xF, mh = v & 7;
                out[(ch - row0) * k + kt * TILE_K + kl] = (uint16_t)((s << 15) | ((b + o) << 7) | (mh << 4) | 0x8);
            }
            for (int32_t e = esc_tile_off[t]; e < esc_tile_off[t + 1]; ++e) {
                uint32_t en = esc[e];
                int nl = (int)(en >> 22) & 0x7F, kl = (int)(en >> 16) & 0x3F;
                if (nl != c) continue;
                out[(ch - row0) * k + kt * TILE_K + kl] = (uint16_t)(en & 0xFFFF);
            }
        }
    }
    return ORC_OK;
}

/* y[r][c] = sum_i x[r][i] * w[c][i], FP64 accumulation in index order. */
int orc_gemm_f64(const uint16_t *x, int64_t R, const uint16_t *w, int64_t n, int64_t k, double *y,
                 int nthreads)
{
    if (!x || !w || !y || R <= 0 || n <= 0 || k <= 0) return ORC_EINVAL;
    int T = pick_threads(nthreads);
    if (T > n) T = (int)n;
    pthread_t th[256];
    gemm_job jobs[256];
    if (T > 256) T = 256;
    for (int t = 0; t < T; ++t) {
        jobs[t] = (gemm_job){x, w, R, n, k, n * t / T, n * (t + 1) / T, y};
        pthread_create(&th[t], NULL, gemm_worker, &jobs[t]);
    }
    for (int t = 0; t < T; ++t) pthread_join(th[t], NULL);
    return ORC_OK;
}

typedef struct {
    const uint16_t *h, *w;
    const double *bias;
    int64_t R, V, k, v0, v1;
    double *top1, *top2;
    int32_t *arg;
} head_job;

/* R9: a value beats the current best iff it is larger; NaN never wins. */
static void head_update(double val, int64_t v, double *t1, double *t2, int32_t *a)
{
    if (isnan(val)) return;
    if (*a < 0 || val > *t1) {
        if (*a >= 0) *t2 = *t1;
        *t1 = val;
        *a = (int32_t)v;
    } else if (val > *t2 || isnan(*t2)) {
        *t2 = val;
    }
}

static void *head_worker(void *p)
{
    head_job *j = (head_job *)p;
    for (int64_t r = 0; r < j->R; ++r) {
        j->top1[r] = NAN;
        j->top2[r] = -INFINITY;
        j->arg[r] = -1;
    }
    for (int64_t v = j->v0; v < j->v1; ++v) {
        const uint16_t *wr = j->w + v * j->k;
        for (int64_t r = 0; r < j->R; ++r) {
            const uint16_t *hr = j->h + r * j->k;
            double acc = 0.0;
            for (int64_t i = 0; i < j->k; ++i) acc += bf16_to_double(hr[i]) * bf16_to_double(wr[i]);
            if (j->bias) acc += j->bias[v];
            head_update(acc, v, &j->top1[r], &j->top2[r], &j->arg[r]);
        }
    }
    return NULL;
}

/*
 * logits = h . W_head^T in FP64 (optionally + bias[v], a hook the tests use
 * to plant a defect), then per row: argmax (R9), top-1 value and the margin
 * top1 - top2.  Vocabulary chunks are scanned in increasing index order so
 * the lowest index wins ties.
 */
int orc_head_argmax(const uint16_t *h, int64_t R, const uint16_t *w, int64_t V, int64_t k,
                    const double *bias, int32_t *argmax, double *top1, double *margin, int nthreads)
{
    if (!h || !w || !argmax || R <= 0 || V <= 0 || k <= 0) return ORC_EINVAL;
    int T = pick_threads(nthreads);
    if (T > 256) T = 256;
    if (T > V) T = (int)V;
    head_job *jobs = calloc((size_t)T, sizeof *jobs);
    pthread_t *th = calloc((size_t)T, sizeof *th);
    double *t1 = malloc(sizeof(double) * (size_t)(R * T));
    double *t2 = malloc(sizeof(double) * (size_t)(R * T));
    int32_t *ar = malloc(sizeof(int32_t) * (size_t)(R * T));
    if (!jobs || !th || !t1 || !t2 || !ar) {
        free(jobs), free(th), free(t1), free(t2), free(ar);
        return ORC_ENOMEM;
    }
    for (int t = 0; t < T; ++t) {
        jobs[t] = (head_job){h, w, bias, R, V, k, V * t / T, V * (t + 1) / T, t1 + R * t, t2 + R * t, ar + R * t};
        pthread_create(&th[t], NULL, head_worker, &jobs[t]);
    }
    for (int t = 0; t < T; ++t) pthread_join(th[t], NULL);
    for (int64_t r = 0; r < R; ++r) {
        double b1 = NAN, b2 = -INFINITY;
        int32_t a = -1;
        for (int t = 0; t < T; ++t) { /* chunks in index order */
            if (ar[R * t + r] < 0) continue;
            double c1 = t1[R * t + r], c2 = t2[R * t + r];
            if (a < 0 || c1 > b1) {
                if (a >= 0 && b1 > b2) b2 = b1;
                b1 = c1;
                a = ar[R * t + r];
            } else if (c1 > b2) {
                b2 = c1;
            }
            if (c2 > b2) b2 = c2;
        }
        argmax[r] = a < 0 ? 0 : a;
        if (top1) top1[r] = b1;
        if (margin) margin[r] = (a < 0) ? 0.0 : b1 - b2;
    }
    free(jobs), free(th), free(t1), free(t2), free(ar);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Best-first tree under a shared budget                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    float score;
    int32_t depth, req, parent_row, token, rank;
    uint64_t path;
} node;

/* R13: nonzero iff a comes before b */
static int node_before(const node *a, const node *b)
{
    if (a->score != b->score) return a->score > b->score;
    if (a->depth != b->depth) return a->depth < b->depth;
    if (a->req != b->req) return a->req < b->req;
    return a->path < b->path;
}

/*
 * Priority-queue expansion: start from every request's root; repeatedly take
 * the best node of the frontier into the tree and put its children on the
 * frontier, until the budget is spent or the frontier is empty.  Log
 * probabilities must be finite and <= 0 (checked for every entry used).
 * Output rows: grouped by request, in the order they were taken.
 */
int orc_tree_build(int32_t n_req, int32_t p_max, int32_t n_cand, int32_t conditional,
                   const int32_t *p_r, const int32_t *root_tok, const int32_t *cand_tok,
                   const float *cand_logp, int32_t budget, int32_t *parent, int32_t *token,
                   uint8_t *depth, int32_t *req, float *score, uint8_t *rank, int32_t *req_row_off,
                   int32_t *R_out)
{
    if (n_req < 1 || p_max < 0 || p_max > 16 || n_cand < 1 || n_cand > 16 || budget < n_req || !p_r ||
        !root_tok || !R_out || (p_max > 0 && (!cand_tok || !cand_logp)))
        return ORC_EINVAL;
    for (int32_t r = 0; r < n_req; ++r) {
        if (p_r[r] < 0 || p_r[r] > p_max) return ORC_EINVAL;
        for (int32_t d = 0; d < p_r[r]; ++d) {
            int rows = conditional ? n_cand : 1;
            for (int pc = 0; pc < rows; ++pc)
                for (int j = 0; j < n_cand; ++j) {
                    int64_t idx = conditional ? ((((int64_t)r * p_max + d) * 16 + pc) * 16 + j)
                                              : (((int64_t)r * p_max + d) * 16 + j);
                    float lp = cand_logp[idx];
                    if (!(lp <= 0.0f) || isinf(lp)) return ORC_EINVAL;
                }
        }
    }
    int64_t cap = (int64_t)budget * 16 + n_req + 16;
    node *front = malloc(sizeof(node) * (size_t)cap);
    node *taken = malloc(sizeof(node) * (size_t)budget);
    if (!front || !taken) {
        free(front), free(taken);
        return ORC_ENOMEM;
    }
    int64_t nf = 0;
    for (int32_t r = 0; r < n_req; ++r)
        front[nf++] = (node){0.0f, 0, r, -1, root_tok[r], 0, 0};
    int32_t nt = 0;
    while (nt < budget && nf > 0) {
        int64_t best = 0;
        for (int64_t i = 1; i < nf; ++i)
            if (node_before(&front[i], &front[best])) best = i;
        node x = front[best];
        front[best] = front[--nf];
        taken[nt] = x;
        int32_t my_idx = nt++;
        if (x.depth < p_r[x.req]) {
            int32_t d = x.depth + 1; /* child depth; uses position d (R14) */
            for (int j = 0; j < n_cand; ++j) {
                int64_t pos = (int64_t)x.req * p_max + (d - 1);
                float e = conditional ? cand_logp[(pos * 16 + x.rank) * 16 + j] : cand_logp[pos * 16 + j];
                node c;
                c.score = x.score + e; /* FP32 add, root to leaf (R11) */
                c.depth = d;
                c.req = x.req;
                c.parent_row = my_idx; /* index into taken[] for now */
                c.token = cand_tok[pos * 16 + j];
                c.rank = j;
                c.path = x.path | ((uint64_t)j << (64 - 4 * d));
                front[nf++] = c;
            }
        }
    }
    /* emit grouped by request, keeping the taken order inside a request */
    int32_t *row_of = malloc(sizeof(int32_t) * (size_t)(nt > 0 ? nt : 1));
    int32_t R = 0;
    for (int32_t r = 0; r < n_req; ++r) {
        if (req_row_off) req_row_off[r] = R;
        for (int32_t i = 0; i < nt; ++i) {
            if (taken[i].req != r) continue;
            row_of[i] = R;
            if (parent) parent[R] = taken[i].parent_row < 0 ? -1 : row_of[taken[i].parent_row];
            if (token) token[R] = taken[i].token;
            if (depth) depth[R] = (uint8_t)taken[i].depth;
            if (req) req[R] = r;
            if (score) score[R] = taken[i].score;
            if (rank) rank[R] = (uint8_t)taken[i].rank;
            R++;
        }
    }
    if (req_row_off) req_row_off[n_req] = R;
    *R_out = R;
    free(front), free(taken), free(row_of);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Greedy acceptance                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Per request: the root is accepted; a node is accepted iff its parent is
 * and its token equals the target's argmax at the parent.  Output: the draft
 * tokens of the deepest accepted node's path, then the bonus token (the
 * argmax at that node).  acc_len = tau = depth + 1.  acc_tok rows are padded
 * with -1 up to p_max + 1 entries.
 */
int orc_tree_accept(int32_t R, const int32_t *parent, const int32_t *token, const uint8_t *depth,
                    const int32_t *req_row_off, int32_t n_req, int32_t p_max, const int32_t *argmax,
                    int32_t *acc_tok, int32_t *acc_len, int32_t *acc_node)
{
    if (R < 1 || !parent || !token || !depth || !req_row_off || !argmax || !acc_tok || !acc_len || n_req < 1)
        return ORC_EINVAL;
    for (int32_t r = 0; r < n_req; ++r) {
        int32_t lo = req_row_off[r], hi = req_row_off[r + 1];
        int32_t *out = acc_tok + (int64_t)r * (p_max + 1);
        for (int i = 0; i <= p_max; ++i) out[i] = -1;
        if (lo >= hi) {
            acc_len[r] = 0;
            if (acc_node) acc_node[r] = -1;
            continue;
        }
        int32_t cur = lo, n = 0;
        for (;;) {
            int32_t next = -1;
            for (int32_t j = lo; j < hi; ++j)
                if (parent[j] == cur && token[j] == argmax[cur]) {
                    next = j; /* lowest row wins (R16) */
                    break;
                }
            if (next < 0) break;
            out[n++] = token[next];
            cur = next;
        }
        out[n] = argmax[cur];
        acc_len[r] = depth[cur] + 1;
        if (acc_node) acc_node[r] = cur;
    }
    return ORC_OK;
}
