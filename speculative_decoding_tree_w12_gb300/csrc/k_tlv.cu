// TLV splice (sm_103a): the combined tree that one exact pass verifies.
//
// SpecPilot explainer, 4.3: the Q pass (quick weights) over the first tree
// picks the commit chain C (its greedy-accepted path plus the bonus token);
// the drafter then builds a fresh subtree from the end of C, cut to the
// budget that C leaves, and the exact pass verifies C with the subtree hung
// under its last token.  Per request q the combined rows are: the first
// tree's root, the first m_q tokens of C as a path (the chain's draft rows
// keep the first tree's rank and score, the bonus row takes rank 255 and its
// parent's score), then the subtree's non-root rows (its root is the chain
// end) with depth + m_q and score + the chain end's score.
//
// One CTA: both trees are staged in shared memory (<= 512 rows each), one
// thread per request lays out its chain, one thread per subtree row moves
// it.  Every index read from the inputs is range-checked first; a
// malformed input sets W12_E_INVAL in the status word and nothing is
// written past the host-sized output.
#include <cuda_runtime.h>

#include "w12_device.cuh"

using namespace w12d;

namespace {

constexpr int kRows = w12i::kMaxBudget;
constexpr int kThreads = kRows;

struct SpliceParams {
    int32_t n_req, p1_max, t1_R, t2_R, R;
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
    int16_t m[kRows];
};

struct SpliceShared {
    int32_t t1_parent[kRows], t1_token[kRows];
    float t1_score[kRows];
    uint8_t t1_rank[kRows];
    int32_t base[kRows + 1];
    int32_t end_tok[kRows];
    float end_score[kRows];
    int32_t warp_sum[kThreads / 32];
    int32_t bad;
};

__device__ __forceinline__ void flag(SpliceShared &s) { s.bad = 1; }

__global__ void __launch_bounds__(kThreads, 1) k_tlv_splice(const SpliceParams p)
{
    __shared__ SpliceShared s;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int n_req = p.n_req;
    if (tid == 0) s.bad = 0;
    for (int j = tid; j < p.t1_R; j += kThreads) {
        s.t1_parent[j] = p.t1_parent[j];
        s.t1_token[j] = p.t1_token[j];
        s.t1_score[j] = p.t1_score[j];
        s.t1_rank[j] = p.t1_rank[j];
    }
    __syncthreads();

    // rows of request q in the combined tree: m_q chain rows + its subtree
    int32_t cnt = 0;
    if (tid < n_req) {
        const int32_t lo = p.t2_off[tid], hi = p.t2_off[tid + 1];
        const int32_t a = p.t1_off[tid], b = p.t1_off[tid + 1];
        if (lo < 0 || hi <= lo || hi > p.t2_R || a < 0 || b <= a || b > p.t1_R) flag(s);
        cnt = p.m[tid] + (hi - lo);
    }
    // block-wide exclusive scan of cnt
    int32_t x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s.warp_sum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int32_t w = lane < kThreads / 32 ? s.warp_sum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kThreads / 32) s.warp_sum[lane] = w;   // inclusive warp totals
    }
    __syncthreads();
    const int32_t incl = x + (wid ? s.warp_sum[wid - 1] : 0);
    if (tid < n_req) s.base[tid] = incl - cnt;
    if (tid == n_req - 1 && incl != p.R) flag(s);
    __syncthreads();
    if (s.bad) {
        if (tid == 0) atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
        return;
    }

    // chains: one thread per request walks the first tree up from the
    // Q-accepted node (shared memory), writing the rows it commits
    if (tid < n_req) {
        const int q = tid;
        const int32_t base = s.base[q], mq = p.m[q], len = p.c_len[q];
        const int32_t a = p.t1_off[q], b = p.t1_off[q + 1];
        const int32_t *ct = p.c_tok + (int64_t)q * (p.p1_max + 1);
        int32_t j = p.c_node[q];
        bool ok = len >= 1 && len <= p.p1_max + 1 && mq <= len && j >= a && j < b;
        const int d = len - 1;
        float s_end = 0.f, s_last = 0.f;
        int32_t t_end = 0;
        // path row i = d, d-1, ..., 0 (i = 0 is the root)
        for (int i = d; ok && i >= 0; --i) {
            const int32_t par = s.t1_parent[j];
            const bool bad_step = i == 0 ? (par != -1 || j != a) : (par < a || par >= j || s.t1_token[j] != ct[i - 1]);
            if (bad_step) {
                ok = false;
                break;
            }
            if (i == d) s_last = s.t1_score[j];
            if (i <= mq) {
                const int32_t o = base + i;
                p.parent[o] = i ? base + i - 1 : -1;
                p.token[o] = s.t1_token[j];
                p.depth[o] = (uint8_t)i;
                p.req[o] = q;
                p.score[o] = s.t1_score[j];
                p.rank[o] = s.t1_rank[j];
                if (i == mq) {
                    s_end = s.t1_score[j];
                    t_end = s.t1_token[j];
                }
            }
            if (i) j = par;
        }
        if (ok && mq == len) {   // the bonus token closes the chain
            const int32_t o = base + mq;
            p.parent[o] = o - 1;
            p.token[o] = ct[d];
            p.depth[o] = (uint8_t)mq;
            p.req[o] = q;
            p.score[o] = s_last;
            p.rank[o] = 255;
            s_end = s_last;
            t_end = ct[d];
        }
        if (!ok) flag(s);
        s.end_tok[q] = t_end;
        s.end_score[q] = s_end;
        p.off[q] = base;
        if (q == n_req - 1) p.off[n_req] = p.R;
    }
    __syncthreads();
    if (s.bad) {
        if (tid == 0) atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
        return;
    }

    // subtree rows: the root must be the chain end; the rest move under it
    for (int j = tid; j < p.t2_R; j += kThreads) {
        const int32_t q = p.t2_req[j];
        if (q < 0 || q >= n_req) {
            flag(s);
            continue;
        }
        const int32_t lo = p.t2_off[q], hi = p.t2_off[q + 1];
        if (j < lo || j >= hi) {
            flag(s);
            continue;
        }
        if (j == lo) {
            if (p.t2_token[j] != s.end_tok[q] || p.t2_parent[j] != -1) flag(s);
            continue;
        }
        const int32_t par = p.t2_parent[j];
        if (par < lo || par >= j) {
            flag(s);
            continue;
        }
        const int32_t end = s.base[q] + p.m[q];
        const int32_t o = end + (j - lo);
        p.parent[o] = end + (par - lo);
        p.token[o] = p.t2_token[j];
        p.depth[o] = (uint8_t)(p.m[q] + p.t2_depth[j]);
        p.req[o] = q;
        p.score[o] = __fadd_rn(s.end_score[q], p.t2_score[j]);
        p.rank[o] = p.t2_rank[j];
    }
    __syncthreads();
    if (tid == 0 && s.bad) atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
}

}  // namespace

namespace w12i {

int launch_tlv_splice(const SpliceArgs &a, void *stream)
{
    if (a.n_req < 1 || a.n_req > kRows || a.t1_R > kRows || a.t2_R > kRows || a.R > kRows)
        return (int)cudaErrorInvalidValue;
    SpliceParams p{};
    p.n_req = a.n_req;
    p.p1_max = a.p1_max;
    p.t1_R = a.t1_R;
    p.t2_R = a.t2_R;
    p.R = a.R;
    p.t1_parent = a.t1_parent;
    p.t1_token = a.t1_token;
    p.t1_off = a.t1_off;
    p.t1_rank = a.t1_rank;
    p.t1_score = a.t1_score;
    p.c_tok = a.c_tok;
    p.c_len = a.c_len;
    p.c_node = a.c_node;
    p.t2_parent = a.t2_parent;
    p.t2_token = a.t2_token;
    p.t2_req = a.t2_req;
    p.t2_off = a.t2_off;
    p.t2_depth = a.t2_depth;
    p.t2_rank = a.t2_rank;
    p.t2_score = a.t2_score;
    p.parent = a.parent;
    p.token = a.token;
    p.req = a.req;
    p.off = a.off;
    p.depth = a.depth;
    p.rank = a.rank;
    p.score = a.score;
    p.status = a.status;
    for (int q = 0; q < a.n_req; ++q) p.m[q] = (int16_t)a.m_host[q];
    k_tlv_splice<<<1, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace w12i
