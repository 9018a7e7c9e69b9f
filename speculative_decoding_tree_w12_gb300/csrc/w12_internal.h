// Internal declarations shared by the host ABI layer and the CUDA kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "w12.h"

namespace w12i {

constexpr int kTileN = 128;          // output channels per W12 record
constexpr int kTileK = 64;           // input features per W12 record
constexpr int kRecBytes = 12288;     // one record: 8 KB view plane + 4 KB low nibbles
constexpr int kViewBytes = 8192;
constexpr int kMaxRows = 256;
constexpr int kMaxBudget = 512;
constexpr int kMaxPositions = 16;
constexpr int kMaxDepth = 2 * kMaxPositions + 1;   // deepest row of a spliced tree
constexpr int kCands = 16;
constexpr int kGemmSlots = 2;        // consecutive GEMMs alternate workspace slots
constexpr int kGridWords = 4096;     // GEMM-chain words: an abort word + one per GEMM of a step

// Device status word values (first condition wins).
constexpr int32_t kDevOk = 0;

// Byte layout of the caller's workspace.  Every region is 256-byte aligned.
struct WsLayout {
    size_t status;        // int32[64]: [0] status, [1] detail, [8] mismatch count (int64)
    size_t grid;          // uint32[kGridWords]: [0] abort word of a GEMM chain, [1 + j] CTAs done with GEMM j
    size_t counters;      // int32[kGemmSlots][max_tiles_n]: split-tile arrival counters
    size_t partial;       // float[kGemmSlots][max_ctas][2][rows8][128]
    size_t stage1_val;    // float[rows][vocab_tiles]
    size_t stage1_idx;    // int32[rows][vocab_tiles]
    size_t tree;          // tree-build scratch
    size_t total;
    int64_t max_tiles_n, max_ctas, rows8, vocab_tiles;
    int32_t rows;
};

WsLayout ws_layout(int32_t R, int64_t max_n, int64_t vocab, int32_t n_req, int num_sms);
size_t tree_ws_bytes(int32_t n_req);

// ---------------------------------------------------------------------------
// kernel launchers (defined in the .cu files); all return cudaError_t as int
// ---------------------------------------------------------------------------

struct DevWeight {
    const uint8_t *rec;
    const uint8_t *base;
    const int32_t *esc_off;
    const uint32_t *esc;
    int32_t n_tiles, k_tiles;
    int64_t n, k;
};

int launch_unpack(const DevWeight &w, uint16_t *dst, const uint16_t *cmp, int64_t *mismatch, int32_t *status,
                  void *stream);

enum GemmMode : int32_t { kModeLinear = 0, kModeHead = 1 };

struct GemmArgs {
    DevWeight w;
    const uint16_t *x;       // [R][k] row-major BF16
    int32_t R;
    int32_t mode;
    uint16_t *y;             // linear: [R][n]
    float *stage1_val;       // head: [R][n_tiles]
    int32_t *stage1_idx;
    float *partial;          // this call's slot
    int32_t *counters;       // this call's slot
    int32_t *status;
    int num_sms;
    bool pdl;                // launched as a programmatic dependent of the previous kernel
    bool qview;              // quick pass: view planes only, low mantissa bits = 0b1000 (warp-MMA path)
    int32_t debug_flags;
    uint64_t timeout_ns;
};

// The verify pass's GEMM chain in one persistent launch per up to
// chain_max_jobs() GEMMs (k_chain.cu): GEMM j + 1 reads its activations only
// after every CTA has counted itself in grid_bar[j].
struct ChainJob {
    DevWeight w;
    const uint16_t *x;       // [R][k] row-major BF16
    int32_t mode;
    uint16_t *y;             // linear: [R][n]
    float *s1_val;           // head: [R][n_tiles]
    int32_t *s1_idx;
};

struct ChainArgs {
    const ChainJob *jobs;
    int32_t n_jobs;
    int32_t R;
    float *partial;          // one partial slot (ws.partial(0))
    int32_t *counters;       // one counter slot, zero on entry
    int32_t *status;
    uint32_t *grid_bar;      // [n_jobs], zero on entry (may be null for one GEMM)
    int32_t *grid_abort;     // zero on entry
    uint64_t *trace;         // optional timing stamps (w12_debug_chain_trace)
    int num_sms;
    bool pdl;
    bool qview;
    int32_t debug_flags;
    uint64_t timeout_ns;
};

int launch_chain(const ChainArgs &a, void *stream);
int chain_max_jobs();

int launch_gemm(const GemmArgs &a, void *stream);      // warp-MMA path, R <= 64 per launch
int launch_gemm_tc(const GemmArgs &a, void *stream);   // tensor-memory path, R <= 256
// same kernel, scratch in a file-scope device array (no workspace argument)
int launch_gemm_static_scratch(const GemmArgs &a, void *stream);
int static_scratch_limits(int32_t *max_rows, int32_t *max_tiles);
int launch_argmax_stage2(const float *s1_val, const int32_t *s1_idx, int32_t R, int32_t n_tiles, int32_t *argmax,
                         float *maxlogit, bool pdl, void *stream);

struct TreeArgs {
    int32_t n_req, p_max, n_cand, conditional, budget, R;
    const int32_t *p_r_host;     // [n_req], host memory (copied into the launch parameters)
    const int32_t *root_tok;
    const int32_t *cand_tok;
    const float *cand_logp;
    int32_t *parent, *token, *req, *req_row_off;
    uint8_t *depth, *rank;
    float *score;
    void *scratch;
    int32_t *status;
};

int launch_tree_build(const TreeArgs &a, void *stream);

// certified LM head (k_cert.cu)
constexpr int kCertParts = 64;   // CTAs rescoring one row's survivors
int launch_cert_norms(const DevWeight &w, float *err, float *qnorm, void *stream);
int launch_cert_select(const uint16_t *shat, const uint16_t *h, const float *err, const float *qnorm, int32_t R,
                       int64_t V, int64_t K, int32_t *surv, int32_t *cnt, float *part_lo, void *stream);
int launch_cert_rescore(const DevWeight &w, const uint16_t *h, int32_t R, const int32_t *surv, const int32_t *cnt,
                        double *part_v, int32_t *part_i, int32_t *argmax, float *maxlogit, int32_t *cnt_out,
                        void *stream);
// recurrent-layer tree verification (k_gdn.cu)
constexpr int kGdnWy = 0, kGdnPath = 1, kGdnCommit = 2, kGdnCommitWy = 3;
constexpr int kGdnDim = 128;        // head dimension
constexpr int kGdnMaxRows = 64;     // tree rows of one request
struct GdnArgs {
    int32_t H, n_req, R;
    int num_sms;             // SMs of the device (sizes the WY kernel's grid)
    uint64_t timeout_ns;     // bounded waits of the WY kernel
    const float *S0;
    const uint16_t *q, *k, *v;
    const float *alpha, *beta;
    const int32_t *parent, *req_row_off, *acc_node;
    float *out;
    float *u;                // WY vectors [R][H][d]: written by kGdnWy when not null, read by kGdnCommitWy
    int32_t *status;
    int32_t debug_flags;     // w12_debug_set flags (bit 0: the tensor-memory WY kernel's test hook)
};
int launch_gdn(const GdnArgs &a, int mode, void *stream);

// TLV splice (k_tlv.cu)
struct SpliceArgs {
    int32_t n_req, p1_max, t1_R, t2_R, R;
    const int32_t *m_host;       // [n_req], host memory (copied into the launch parameters)
    const int32_t *t1_parent, *t1_token, *t1_off;
    const uint8_t *t1_rank;
    const float *t1_score;
    const int32_t *c_tok, *c_len, *c_node;
    const int32_t *t2_parent, *t2_token, *t2_req, *t2_off;
    const uint8_t *t2_depth, *t2_rank;
    const float *t2_score;
    int32_t *parent, *token, *req, *off;
    uint8_t *depth, *rank;
    float *score;
    int32_t *status;
};
int launch_tlv_splice(const SpliceArgs &a, void *stream);

int launch_tree_accept(const int32_t *parent, const int32_t *token, const uint8_t *depth,
                       const int32_t *req_row_off, int32_t R, int32_t n_req, int32_t p_max, const int32_t *argmax,
                       int32_t *acc_tok, int32_t *acc_len, int32_t *acc_node, bool pdl, void *stream);

}  // namespace w12i
