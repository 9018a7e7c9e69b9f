/*
 * w12.h -- C ABI of the W12 tree-verify library (GB300, sm_103a).
 *
 * The verify pass of tree-based speculative decoding over weights stored in
 * the W12 12-bit lossless format:
 *
 *   lattice --w12_tree_build--> draft tree of R rows
 *   rows    --w12_gemm (per linear)-------------------> Y = X . W^T
 *   rows    --w12_lmhead_argmax--> target argmax per row
 *   tree + argmax --w12_tree_accept--> accepted tokens + lengths
 *
 * Around it: the quick pass on the 8-bit view planes (w12_gemm_q,
 * w12_lmhead_argmax_q, w12_verify_step_q), the certified LM head
 * (w12_head_cert_norms, w12_lmhead_argmax_certified), the TLV splice of two
 * trees (w12_tlv_chain, w12_tlv_splice) and a recurrent (Gated DeltaNet)
 * layer over a tree (w12_gdn_tree_verify, w12_gdn_commit).
 *
 * Sources (SpecPilot explainer at jaehun.me, "SpecPilot: Autonomous Algorithm
 * Discovery and Systems Optimization for Speculative Decoding"; the summary
 * page at agihunt.info; the poot-llm speculative-decoding docs):
 *   - W12: explainer section 4.1 "W12: a 12-bit lossless weight format".
 *   - verify rows / greedy acceptance: explainer 1.1; poot-llm "What a round
 *     guarantees".
 *   - best-first tree / shared budget: explainer 4.2 and 4.4.
 *   - quick pass, certified head, TLV: explainer 4.1 and 4.3.
 *   - recurrent layers over a tree (path walk, WY form): explainer 4.2.
 *   - typed refusal before anything runs: poot-llm "What is refused".
 *
 * Conventions for every entry point:
 *   - Every argument is validated before any launch; a bad argument returns
 *     a typed status and launches nothing.
 *   - Device pointers are caller-owned (e.g. torch tensors).  The library
 *     allocates no device memory and keeps no global state except cached
 *     device properties, its driver entry point and the fixed scratch array
 *     of w12_gemm_static_scratch.
 *   - Device work is asynchronous on the caller's stream unless stated.
 *     Launch failures map to W12_E_CUDA.
 *   - Conditions found on the device (a timed-out wait, bad lattice values)
 *     are written to a status word in the workspace and read back with
 *     w12_status_fetch(); no kernel traps.
 *   - Limits: N % 128 == 0, K % 64 == 0, 1 <= R <= 256 rows, budget <= 512,
 *     p_max <= 16, 16 candidates per position; anything else is
 *     W12_E_UNSUPPORTED.
 *   - There is no CPU fallback: every device step runs in this library's
 *     CUDA kernels.
 */
#ifndef W12_H
#define W12_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *w12_stream_t;

typedef enum {
    W12_OK = 0,
    W12_E_INVAL = -1,        /* malformed argument (null pointer, bad size, ...) */
    W12_E_UNSUPPORTED = -2,  /* well-formed but outside the limits above */
    W12_E_MISMATCH = -3,     /* a bit-exact check failed (pack / load check) */
    W12_E_CUDA = -4,         /* a CUDA call failed */
    W12_E_TIMEOUT = -5,      /* a bounded device wait ran out */
    W12_E_WORKSPACE = -6     /* workspace null, too small or misaligned */
} w12_status;

/* Human-readable name of a status code (static storage). */
const char *w12_status_str(int status);

/* ABI version of this header: major*100 + minor. */
int w12_abi_version(void);

/* ------------------------------------------------------------------------
 * W12 packing (host memory, caller-owned)
 *
 * Format (explainer 4.1): for every output channel n a window base b_n (the
 * BF16 biased exponent field of the window's lowest binade, 1..239) chosen
 * to hold the most normal weights of the channel (ties: largest b_n).  A
 * weight whose exponent field e lies in [b_n, b_n + 15] is stored in 12 bits:
 * an 8-bit view byte [sign:1][e - b_n:4][mantissa bits 6..4] and a low nibble
 * (mantissa bits 3..0).  Any other weight (zero, denormal, Inf, NaN, out of
 * window) is stored as a zero code plus an exact 16-bit escape entry.
 *
 * Records: one 12288-byte record per 128x64 tile, tiles ordered n-tile major
 * (t = n_tile * (K/64) + k_tile).  Bytes 0..8191 (the 8-bit view):
 * four 16-K groups g, each 128 channels c x 16 bytes at (g*128 + c)*16, the
 * weight kk of the group at byte pos(kk) = 4*((kk%8)/2) + 2*(kk/8) + kk%2.
 * Bytes 8192..12287 (low nibbles): two 32-K groups h, each 128 channels x 16
 * bytes at 8192 + (h*128 + c)*16; weight kk of the group's first 16 K is the
 * low nibble of byte pos(kk), weight kk of the second 16 K the high nibble.
 *
 * Escapes: esc_tile_off[t] .. esc_tile_off[t+1] index the entries of record
 * t in esc[], each u32 = n_local << 22 | k_local << 16 | bf16 bits, sorted
 * by (n_local, k_local).
 * ---------------------------------------------------------------------- */

typedef struct {
    int64_t n, k;            /* output channels, input features */
    int64_t n_tiles, k_tiles;
    int64_t n_escapes;
    size_t rec_bytes;        /* n_tiles * k_tiles * 12288 */
    size_t base_bytes;       /* n */
    size_t esc_off_bytes;    /* (n_tiles * k_tiles + 1) * 4 */
    size_t esc_bytes;        /* n_escapes * 4 */
} w12_layout;

/*
 * Sizes of the packed buffers of a row-major BF16 tensor w_bf16[n][k].
 * Reads the whole tensor (window choice and escape count).
 * Errors: W12_E_INVAL (null pointer, n or k <= 0), W12_E_UNSUPPORTED
 * (n % 128 or k % 64 nonzero).
 */
w12_status w12_pack_query(const uint16_t *w_bf16, int64_t n, int64_t k, w12_layout *out);

/*
 * Pack w_bf16[n][k] into caller buffers of the sizes w12_pack_query gave
 * (esc may be NULL when n_escapes == 0).  The packer then decodes its own
 * output on the host and compares it bit for bit with the source (the load
 * check of explainer 4.1); any difference returns W12_E_MISMATCH.
 * Runs on host threads; thread-safe for distinct outputs.
 */
w12_status w12_pack(const uint16_t *w_bf16, int64_t n, int64_t k, const w12_layout *layout,
                    void *rec, uint8_t *base, int32_t *esc_tile_off, uint32_t *esc);

/* ------------------------------------------------------------------------
 * Device views.  All pointers below are device pointers owned by the caller.
 * ---------------------------------------------------------------------- */

typedef struct {
    const void *rec;             /* records, 16-byte aligned */
    const uint8_t *base;         /* [n] window bases */
    const int32_t *esc_tile_off; /* [tiles + 1] */
    const uint32_t *esc;         /* [n_escapes] (may be NULL if none) */
    int64_t n, k;
    int64_t n_escapes;
} w12_weight;

/*
 * Workspace: one caller-owned device buffer, 256-byte aligned, at least
 * w12_workspace_bytes(...) bytes for the largest call made with it, and set
 * to zero once with w12_workspace_init before first use.  Calls that share
 * a workspace must be ordered on one stream.
 *   R       rows (<= 256), max_n: largest N of any weight, vocab: LM-head N,
 *   n_req   requests of the tree (<= 512).
 */
size_t w12_workspace_bytes(int32_t R, int64_t max_n, int64_t vocab, int32_t n_req);
w12_status w12_workspace_init(void *ws, size_t ws_bytes, w12_stream_t stream);

/*
 * Read and clear the device status word (synchronises the stream).
 * Returns W12_OK or the first device-detected condition since the last
 * fetch (W12_E_TIMEOUT, W12_E_INVAL for bad lattice values, ...).
 */
w12_status w12_status_fetch(void *ws, w12_stream_t stream);

/*
 * Decode a packed tensor to row-major BF16 dst[n][k] (device), escapes
 * restored: the exact restore of explainer 4.1 "W12: a 12-bit lossless
 * weight format" (each in-window weight rebuilt from its sign, exponent
 * offset against the channel's window and seven mantissa bits; each escaped
 * weight from its 16-bit escape entry).  dst is caller-owned, 16-byte
 * aligned.  Asynchronous on the stream.  Errors: W12_E_INVAL (null or
 * misaligned pointer, malformed weight), W12_E_UNSUPPORTED (n % 128 or
 * k % 64 not zero), W12_E_CUDA.
 */
w12_status w12_unpack(const w12_weight *w, uint16_t *dst_bf16, w12_stream_t stream);

/*
 * Load-time bit-exact check (explainer 4.1: "checks the restored tensors
 * bit-for-bit against the checkpoint"): decodes w on the device and compares
 * every weight with src_bf16[n][k] (device).  Synchronises the stream and
 * writes the number of differing weights to *mismatches (host).
 * Returns W12_OK if none differ, W12_E_MISMATCH otherwise.
 */
w12_status w12_load_check(const w12_weight *w, const uint16_t *src_bf16, int64_t *mismatches,
                          void *ws, size_t ws_bytes, w12_stream_t stream);

/*
 * Verify GEMM (explainer 4.1 "W12 GEMM", 2.1): y[R][n] = x[R][k] . W^T with W
 * decoded exactly from W12 inside the kernel, FP32 accumulation, BF16
 * (round to nearest even) output.  x, y row-major BF16, 16-byte aligned
 * rows (k % 64 == 0 already gives that).  Deterministic: the K-split points
 * and the reduction order depend only on the shapes and the device.
 */
w12_status w12_gemm(const w12_weight *w, const uint16_t *x, int32_t R, uint16_t *y, void *ws,
                    size_t ws_bytes, w12_stream_t stream);

/*
 * w12_gemm without a workspace, for callers that cannot allocate device
 * memory where they call it: plugin hosts that give kernels no device
 * allocations of their own, and processes that must keep a fixed device
 * footprint (an allocation there could fail or stall mid-run).  The paper
 * has no counterpart to this entry point; it computes exactly what w12_gemm
 * computes, with the same kernel.
 *   - Scratch (split-tile partial sums, tile arrival counters, a status word)
 *     is a file-scope device array of about 4.1 MiB that every GPU loading
 *     the library holds until the process exits.  The call allocates and
 *     frees nothing.
 *   - Limits: 1 <= R <= 16 rows and n <= 16384 * 128 output channels; larger
 *     sizes return W12_E_UNSUPPORTED before anything runs.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call on a device shares the array and leaves its contents
 *     behind; each call zeroes the counters and status word it uses.  Calls
 *     whose kernels overlap on the GPU (different streams, no ordering)
 *     race on the array: order them on one stream.
 *   - Device-detected conditions (a timed-out wait) are recorded only in the
 *     array's status word, which this entry point does not report.
 * Arguments, layout and errors otherwise as w12_gemm.
 */
w12_status w12_gemm_static_scratch(const w12_weight *w, const uint16_t *x, int32_t R, uint16_t *y,
                                   w12_stream_t stream);

/*
 * LM head + argmax: logits = h[R][k] . W_head^T in FP32 (never stored), then
 * per row the index of the largest logit (lowest index on ties; NaN never
 * wins) into argmax[R]; maxlogit[R] (nullable) gets the winning logit.
 */
w12_status w12_lmhead_argmax(const w12_weight *head, const uint16_t *h, int32_t R, int32_t *argmax,
                             float *maxlogit, void *ws, size_t ws_bytes, w12_stream_t stream);

/*
 * Quick pass (SpecPilot explainer, 4.1 "the 8-bit view is what the Q pass
 * reads" and 4.3 TLV: the Q pass reads the view already nested in the W12
 * record, its first 2/3, with the discarded mantissa bits set to the
 * midpoint).  Same contract as w12_gemm and w12_lmhead_argmax, computed with
 * the quick weights: every in-window weight keeps its sign, exponent and
 * three high mantissa bits and takes 0b1000 as its four low mantissa bits;
 * escaped weights keep their exact value.  Only the 8 KB view plane of each
 * record is read (about 2/3 of the W12 bytes).  Takes the same GEMM path as
 * the exact pass for the same weight and row count.
 */
w12_status w12_gemm_q(const w12_weight *w, const uint16_t *x, int32_t R, uint16_t *y, void *ws, size_t ws_bytes,
                      w12_stream_t stream);
w12_status w12_lmhead_argmax_q(const w12_weight *head, const uint16_t *h, int32_t R, int32_t *argmax,
                               float *maxlogit, void *ws, size_t ws_bytes, w12_stream_t stream);

/*
 * Certified LM head (explainer 4.1 and 4.3: a cheap pass, a per-row
 * Cauchy-Schwarz error bound that discards every token proven unable to be
 * the argmax, exact rescoring of the survivors; the argmax never changes).
 * The cheap pass is the quick pass above (the 8-bit view in each record,
 * where the pages keep a separate INT8 copy), so nothing extra is stored.
 *
 * w12_head_cert_norms: load time.  norms (device, float[2][head->n]) gets
 * per token v, rounded up: norms[v] = ||w_v - w^_v|| and
 * norms[n + v] = ||w^_v||, with w^ the quick weights.  Asynchronous.
 *
 * w12_lmhead_argmax_certified: per row r, with s^ the quick logits (BF16)
 * and eps_v = ||h_r|| (norms[v] + tau norms[n + v]) + 2^-8 |s^_v|
 * (tau = k * 2^-22 covers the FP32 accumulation of the cheap pass):
 * L = max_v (s^_v - eps_v); survivors are the tokens with s^_v + eps_v >= L;
 * their exact logits (W12 decoded exactly, FP64 accumulation) decide
 * argmax[r] (lowest index on ties); maxlogit[r] (nullable) gets that logit
 * in FP32; n_survivors[r] (device, nullable) the survivor count.
 * ws: the w12_lmhead_argmax workspace for R rows and n = vocab; cws: device,
 * 256-byte aligned, w12_cert_workspace_bytes(R, vocab) bytes (room for every
 * token of every row to survive).  The rescoring costs one exact row decode
 * and a K-long FP64 dot product per survivor: cheap when a row's top logit
 * stands out, slow (but still exact) when the view's bound keeps much of the
 * vocabulary, as for unstructured rows.
 */
w12_status w12_head_cert_norms(const w12_weight *head, float *norms, w12_stream_t stream);
size_t w12_cert_workspace_bytes(int32_t R, int64_t vocab);
w12_status w12_lmhead_argmax_certified(const w12_weight *head, const float *norms, const uint16_t *h, int32_t R,
                                       int32_t *argmax, float *maxlogit, int32_t *n_survivors, void *ws,
                                       size_t ws_bytes, void *cws, size_t cws_bytes, w12_stream_t stream);

/* ------------------------------------------------------------------------
 * Draft tree
 * ---------------------------------------------------------------------- */

typedef struct {
    int32_t n_req;              /* requests */
    int32_t p_max;              /* drafted positions per request (<= 16) */
    int32_t n_cand;             /* candidates used per position (1 = chain, <= 16) */
    int32_t conditional;        /* 0: logp[n_req][p_max][16]; 1: logp[n_req][p_max][16][16] */
    const int32_t *p_r;         /* HOST [n_req]: positions drafted by request r (0..p_max) */
    const int32_t *root_tok;    /* device [n_req]: last committed token */
    const int32_t *cand_tok;    /* device [n_req][p_max][16] */
    const float *cand_logp;     /* device, layout per `conditional`; finite and <= 0 */
} w12_lattice;

typedef struct {
    int32_t R;                  /* rows, set by w12_tree_build */
    int32_t *parent;            /* device [budget]: parent row, -1 for a root */
    int32_t *token;             /* device [budget] */
    uint8_t *depth;             /* device [budget] */
    int32_t *req;               /* device [budget] */
    float *score;               /* device [budget]: FP32 path log-probability */
    uint8_t *rank;              /* device [budget]: candidate rank at its depth */
    int32_t *req_row_off;       /* device [n_req + 1] */
} w12_tree;

/*
 * Best-first tree under one shared node budget (explainer 4.2, 4.4): the
 * rows are the `budget` nodes (roots included, score 0) ranked first by
 * (path score desc, depth asc, request asc, candidate-rank path asc), where
 * a child at depth d takes position d's candidates and its score is the
 * FP32 sum of edge log-probabilities from the root.  The set is
 * prefix-closed.  Rows are emitted grouped by request, best-first inside a
 * request (so every parent precedes its children).  out->R is set on the
 * host (min(budget, nodes available)) before anything runs.
 * Device check: a used log-probability that is positive or not finite sets
 * W12_E_INVAL in the status word.
 */
w12_status w12_tree_build(const w12_lattice *lat, int32_t budget, w12_tree *out, void *ws, size_t ws_bytes,
                          w12_stream_t stream);

/*
 * Greedy acceptance (explainer 1.1): per request the root is accepted and a
 * node is accepted iff its parent is and its token equals the argmax at the
 * parent.  acc_tok[n_req][p_max + 1] gets the deepest accepted node's draft
 * tokens followed by the bonus token (argmax at that node), padded with -1;
 * acc_len[n_req] = tau = depth + 1; acc_node[n_req] (nullable) the row.
 * p_max: the tree's deepest row depth or more (<= 33, which covers a
 * spliced TLV tree); the row stride of acc_tok is p_max + 1.
 */
w12_status w12_tree_accept(const w12_tree *tree, int32_t n_req, int32_t p_max, const int32_t *argmax,
                           int32_t *acc_tok, int32_t *acc_len, int32_t *acc_node, w12_stream_t stream);

/* ------------------------------------------------------------------------
 * Recurrent (Gated DeltaNet) layer over a draft tree (explainer 4.2)
 *
 * A GDN head keeps a d x d state S per request, updated by each token with
 * gate a, write strength b, key k, value v:  S <- a S (I - b k k^T) + b v k^T,
 * and outputs o = S q.  Every tree row is a token; the root applies its
 * update to the request's committed state, a child to its parent's state.
 * No per-node state is stored: the outputs are recomputed along root paths.
 * ---------------------------------------------------------------------- */

typedef struct {
    int32_t n_heads;             /* H (>= 1) */
    int32_t head_dim;            /* d = d_k = d_v; must be 128 */
    const float *S0;             /* device [n_req][H][d][d] FP32, S0[r][h][v][k]; 16-byte aligned */
    const uint16_t *q, *k;       /* device BF16 [R][H][d], 16-byte aligned */
    const uint16_t *v;           /* device BF16 [R][H][d], 4-byte aligned */
    const float *alpha, *beta;   /* device [R][H] */
} w12_gdn_layer;

#define W12_GDN_WY 0     /* WY form: one triangular solve per request and head, state products on tensor cores */
#define W12_GDN_PATH 1   /* path walk: every row replays its root path on a copy of the committed state */

/*
 * Per-row outputs o (device FP32 [R][H][d]) of one layer over a tree
 * (tree->R rows; parent and req_row_off used; rows of a request list every
 * parent before its children, at most 64 rows per request).  W12_GDN_WY
 * multiplies the FP32 state as three BF16 pieces that add up to it exactly,
 * with FP32 accumulation; both methods match the FP64 path walk to FP32
 * rounding.  Device checks: a request with more than 64 rows sets
 * W12_E_UNSUPPORTED, a parent outside its request or after its child
 * W12_E_INVAL in the status word (ws as for w12_tree_build); with
 * W12_GDN_WY, row offsets outside [0, tree->R] also set W12_E_INVAL, and a
 * bad row range anywhere leaves the whole output unwritten.  W12_GDN_WY on
 * a tree of several requests uses tensor memory and 226 KB of shared memory
 * per CTA (one CTA per SM), and its bounded waits report W12_E_TIMEOUT.
 */
w12_status w12_gdn_tree_verify(const w12_gdn_layer *layer, const w12_tree *tree, int32_t n_req, int32_t method,
                               float *o, void *ws, size_t ws_bytes, w12_stream_t stream);

/*
 * The committed states after acceptance: state[r] (device FP32, same layout
 * as S0; may be S0 itself) = S0[r] replayed along the root path of row
 * acc_node[r] (device [n_req], from w12_tree_accept).  Device check: a row
 * outside the request sets W12_E_INVAL (the state is then left as S0[r]).
 */
w12_status w12_gdn_commit(const w12_gdn_layer *layer, const w12_tree *tree, int32_t n_req, const int32_t *acc_node,
                          float *state, void *ws, size_t ws_bytes, w12_stream_t stream);

/*
 * The WY form with its vectors kept for the commit (explainer 4.2, TreeWY):
 * the outputs o as w12_gdn_tree_verify(W12_GDN_WY) gives them, and
 * u (device FP32 [R][H][d], caller-owned) with u_j = b_j (v_j - a_j S k_j),
 * S the state row j's update applies to.  The state after row j is then
 * g_j S0 + sum over i on j's root path of (g_j / g_i) u_i k_i^T, g the
 * product of the gates along the path.  Same checks and status words as
 * w12_gdn_tree_verify; o and u must not be NULL.
 */
w12_status w12_gdn_wy_verify(const w12_gdn_layer *layer, const w12_tree *tree, int32_t n_req, float *o, float *u,
                             void *ws, size_t ws_bytes, w12_stream_t stream);

/*
 * The committed states from those vectors, in one pass over S0 (no replay):
 * state[r] = g S0[r] + sum over i on acc_node[r]'s root path of (g / g_i) u_i k_i^T,
 * with u from w12_gdn_wy_verify on the same layer and tree (16-byte
 * aligned).  state as for w12_gdn_commit (16-byte aligned; may be S0 itself).  Device checks: a row
 * outside the request sets W12_E_INVAL (the state is then left as S0[r]).
 */
w12_status w12_gdn_wy_commit(const w12_gdn_layer *layer, const w12_tree *tree, int32_t n_req, const int32_t *acc_node,
                             const float *u, float *state, void *ws, size_t ws_bytes, w12_stream_t stream);

/* ------------------------------------------------------------------------
 * The verify step
 * ---------------------------------------------------------------------- */

typedef struct {
    int32_t n_linear;
    const w12_weight *lin;         /* HOST array [n_linear] */
    const uint16_t *const *x;      /* HOST array [n_linear] of device x_l[R][lin[l].k] */
    uint16_t *const *y;            /* HOST array [n_linear] of device y_l[R][lin[l].n] */
    const w12_weight *head;
    const uint16_t *h;             /* device h[R][head->k] */
    int32_t *argmax;               /* device [R] */
} w12_step;

/*
 * One verify pass over a built tree (explainer 1.1 and 2.1: the target
 * model verifies every draft row of the tree in one forward pass, keeps the
 * drafts equal to the target's argmax at their parent and appends the bonus
 * token; poot-llm "What a round guarantees": the accepted tokens are exactly
 * the greedy autoregressive ones).  Every linear in order (each may start
 * streaming its weights while the previous one finishes), then the LM head
 * with per-row argmax, then greedy acceptance; same outputs as the
 * individual calls (w12_gemm, w12_lmhead_argmax, w12_tree_accept).
 * step: host arrays of device pointers (x_l[R][k_l], y_l[R][n_l], h[R][k],
 * argmax[R]); rows = tree->R; acc_tok[n_req][p_max + 1], acc_len[n_req],
 * acc_node[n_req] (nullable) as for w12_tree_accept.  ws sized by
 * w12_workspace_bytes(R, max n_l, head n, n_req).  Asynchronous.  Errors:
 * W12_E_INVAL / W12_E_UNSUPPORTED / W12_E_WORKSPACE before any launch,
 * W12_E_CUDA on a failed launch; device conditions in the status word.
 */
w12_status w12_verify_step(const w12_step *step, const w12_tree *tree, int32_t n_req, int32_t p_max,
                           int32_t *acc_tok, int32_t *acc_len, int32_t *acc_node, void *ws, size_t ws_bytes,
                           w12_stream_t stream);

/*
 * The Q pass of TLV (explainer 4.3): the same pass on the quick weights
 * (w12_gemm_q semantics for every linear and the head).  Its acceptance
 * output is the commit chain C: per request the Q-accepted draft tokens and
 * the Q bonus token (acc_tok), their count (acc_len) and the deepest
 * Q-accepted row (acc_node).  Same arguments and workspace as
 * w12_verify_step.
 */
w12_status w12_verify_step_q(const w12_step *step, const w12_tree *tree, int32_t n_req, int32_t p_max,
                             int32_t *acc_tok, int32_t *acc_len, int32_t *acc_node, void *ws, size_t ws_bytes,
                             w12_stream_t stream);

/* ------------------------------------------------------------------------
 * TLV: two-level verification (explainer 4.3)
 *
 *   tree T1 --w12_verify_step_q--> chain C (device)
 *   C lengths + T1 row offsets (read to the host) --w12_tlv_chain--> m, subtree budget
 *   lattice drafted from each chain end --w12_tree_build(budget)--> subtree T2
 *   T1 + C + T2 --w12_tlv_splice--> combined tree --w12_verify_step--> accepted tokens
 *
 * Only the exact pass over the combined tree accepts tokens; C is a
 * proposal, so the output is lossless whatever the Q pass chose.
 * ---------------------------------------------------------------------- */

/*
 * Host only, no device work.  c_len[n_req]: the chain lengths (acc_len of
 * the Q pass); t1_row_off[n_req + 1]: T1's req_row_off; budget: the node
 * budget N the exact pass keeps.  Request q commits
 * m[q] = min(c_len[q], N_q - 1) chain tokens, N_q being its rows in T1 (the
 * cap only drops the bonus, when the whole share was accepted, so every
 * request keeps a row for its subtree root); *sub_budget = N - sum(m): the
 * budget of the fresh subtrees, counting their roots, which are the chain
 * ends (for one request: N - |C|).  W12_E_INVAL if c_len[q] is not in
 * [1, N_q] or the offsets are not those of a tree of at most N rows.
 */
w12_status w12_tlv_chain(const int32_t *c_len, const int32_t *t1_row_off, int32_t n_req, int32_t budget, int32_t *m,
                         int32_t *sub_budget);

/*
 * The combined tree (device, asynchronous).  t1: the first tree (R set);
 * c_tok[n_req][p1_max + 1], c_len[n_req], c_node[n_req]: the Q pass's
 * acceptance outputs for t1 (device); m: HOST [n_req] from w12_tlv_chain;
 * t2: the subtree built with the lattice whose roots are the chain ends
 * (R set, req required).  Per request the rows are t1's root, the first m[q]
 * tokens of the chain as a path (draft rows keep t1's rank and score; the
 * bonus row takes rank 255 and its parent's score), then t2's non-root rows
 * of q under the chain end (depth + m[q], FP32 score + the chain end's).
 * out->R = sum(m) + t2->R is set on the host; out's arrays hold that many
 * rows, req_row_off n_req + 1.  Device check: a chain that is not t1's path
 * from the root to c_node, a t2 root that is not the chain end, or
 * inconsistent row offsets set W12_E_INVAL in the status word (ws as for
 * w12_tree_build); no write goes past out->R rows.
 */
w12_status w12_tlv_splice(const w12_tree *t1, const int32_t *c_tok, const int32_t *c_len, const int32_t *c_node,
                          int32_t n_req, int32_t p1_max, const int32_t *m, const w12_tree *t2, w12_tree *out,
                          void *ws, size_t ws_bytes, w12_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W12_H */
