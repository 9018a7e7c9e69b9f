// Best-first draft tree under a shared node budget, and greedy acceptance
// (sm_103a).
//
// SpecPilot explainer, 4.2: keep the N nodes with the highest path score
// sum log p(child | parent); 4.4: one budget for all requests, filled from
// the highest path log-probability, prefix-closed per request.  Explainer
// 1.1: greedy verification keeps the drafts equal to the target's argmax and
// appends that argmax as a bonus.
//
// Tree build, one CTA.  With every edge log-probability <= 0 a child never
// outranks its parent, so the budget's best nodes at depth d are among the
// best (budget - n_req) children of the nodes kept at depth d-1.  The kernel
// keeps exactly those per depth (radix select on the score, ties by
// (request, path) which is the storage order), then takes the best `R` of
// all kept nodes (ties by depth, then storage order) and sorts them into
// request-grouped, best-first rows.
#include <cuda_runtime.h>

#include <algorithm>

#include "w12_device.cuh"

using namespace w12d;

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kInvalid = 0xFFFFFFFFu;

struct TreeParams {
    int32_t n_req, p_max, n_cand, conditional, budget, R;
    int32_t cand_shift;      // log2(n_cand) when n_cand is a power of two, else -1
    int32_t stage_lattice;   // the lattice (log-probs + tokens) is copied to shared memory
    // shared-memory carve-up (byte offsets), sized on the host
    int32_t off_keys, off_score, off_token, off_parent, off_req, off_meta, off_sort, off_lp, off_lt;
    const int32_t *root_tok;
    const int32_t *cand_tok;
    const float *cand_logp;
    int32_t *parent, *token, *req, *req_row_off;
    uint8_t *depth, *rank;
    float *score;
    int32_t *status;
    uint8_t p_r[w12i::kMaxBudget];
};

struct Hdr {
    uint8_t p_r[w12i::kMaxBudget];
    uint32_t hist[256];
    int32_t red[kWarps];
    int32_t bcast[2];
    int32_t lvl_begin[w12i::kMaxPositions + 2];
    int32_t lvl_end[w12i::kMaxPositions + 2];
};

// ascending key == descending score (a total order on non-NaN floats)
__device__ __forceinline__ uint32_t score_key(float s)
{
    const uint32_t u = __float_as_uint(s);
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ~ord;
}

__device__ __forceinline__ int warp_incl_scan(int x)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// block-wide sum (2 barriers)
__device__ int block_sum(int v, Hdr &h)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) h.red[threadIdx.x >> 5] = v;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += h.red[w];
    __syncthreads();
    return t;
}

// block-wide exclusive scan of one int per thread (2 barriers)
__device__ int block_excl_scan(int v, Hdr &h)
{
    const int incl = warp_incl_scan(v);
    if ((threadIdx.x & 31) == 31) h.red[threadIdx.x >> 5] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < (int)(threadIdx.x >> 5); ++w) before += h.red[w];
    __syncthreads();
    return before + incl - v;
}

// The K smallest of keys[0..n) (1 <= K <= n): threshold tau, and how many of
// the keys equal to tau are taken (the lowest-index ones).  Expects h.hist
// zeroed and leaves it zeroed.  2 barriers per 8-bit pass.
__device__ void radix_select(const uint32_t *keys, int n, int K, uint32_t &tau, int &take_eq, Hdr &h)
{
    uint32_t prefix = 0, mask = 0;
    int krem = K;
    const int rounds = (n + kThreads - 1) / kThreads;   // uniform trip count: whole warps vote
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int it = 0; it < rounds; ++it) {
            const int i = it * kThreads + threadIdx.x;
            const uint32_t k = i < n ? keys[i] : 0u;
            const bool counted = i < n && (k & mask) == prefix;
            const uint32_t bin = counted ? ((k >> shift) & 255u) : 256u;
            // one atomic per distinct bin per warp: scores of one depth share
            // their top bits, so per-key atomics would serialise on one bin
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (counted && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h.hist[bin], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            int c[8], sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                c[q] = (int)h.hist[lane * 8 + q];
                h.hist[lane * 8 + q] = 0;
                sum += c[q];
            }
            const int incl = warp_incl_scan(sum);
            const int before = incl - sum;
            if (before < krem && incl >= krem) {
                int b = before;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (b + c[q] >= krem) {
                        h.bcast[0] = lane * 8 + q;
                        h.bcast[1] = b;
                        break;
                    }
                    b += c[q];
                }
            }
        }
        __syncthreads();
        prefix |= (uint32_t)h.bcast[0] << shift;
        mask |= 255u << shift;
        krem -= h.bcast[1];
    }
    tau = prefix;
    take_eq = krem;
}

// Walk keys[0..n) in index order and call emit(i, out) for every selected
// key: key < tau, or key == tau among the first take_eq such keys.  `out`
// numbers the selected keys in index order.  Each thread owns a contiguous
// chunk; one packed (less, equal) scan gives every position (2 barriers).
template <class Emit>
__device__ int select_ordered(const uint32_t *keys, int n, uint32_t tau, int take_eq, Hdr &h, Emit emit)
{
    const int chunk = (n + kThreads - 1) / kThreads;
    const int lo = min(n, (int)threadIdx.x * chunk), hi = min(n, lo + chunk);
    int lt = 0, eq = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t k = keys[i];
        lt += k < tau;
        eq += k == tau;
    }
    const int packed_before = block_excl_scan((lt << 16) | eq, h);
    int lt_before = packed_before >> 16, eq_before = packed_before & 0xFFFF;
    for (int i = lo; i < hi; ++i) {
        const uint32_t k = keys[i];
        if (k < tau) {
            emit(i, lt_before + min(eq_before, take_eq));
            ++lt_before;
        } else if (k == tau) {
            if (eq_before < take_eq) emit(i, lt_before + eq_before);
            ++eq_before;
        }
    }
    int total_lt = 0, total_eq = 0;
    if (threadIdx.x == kThreads - 1) h.bcast[0] = lt_before, h.bcast[1] = eq_before;
    __syncthreads();
    total_lt = h.bcast[0];
    total_eq = h.bcast[1];
    __syncthreads();
    return total_lt + min(total_eq, take_eq);
}

__global__ void __launch_bounds__(kThreads, 1) k_tree_build(const TreeParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    Hdr &h = *reinterpret_cast<Hdr *>(smem);
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + p.off_keys);
    float *u_score = reinterpret_cast<float *>(smem + p.off_score);
    int32_t *u_token = reinterpret_cast<int32_t *>(smem + p.off_token);
    int16_t *u_parent = reinterpret_cast<int16_t *>(smem + p.off_parent);
    int16_t *u_req = reinterpret_cast<int16_t *>(smem + p.off_req);
    uint16_t *u_meta = reinterpret_cast<uint16_t *>(smem + p.off_meta);   // depth << 8 | rank
    unsigned long long *sortbuf = reinterpret_cast<unsigned long long *>(smem + p.off_sort);
    float *lp_s = reinterpret_cast<float *>(smem + p.off_lp);
    int32_t *lt_s = reinterpret_cast<int32_t *>(smem + p.off_lt);
    const int tid = threadIdx.x;
    const int K = p.budget - p.n_req;   // non-root rows available

    pdl_wait();
    for (int i = tid; i < 256; i += kThreads) h.hist[i] = 0;
    for (int r = tid; r < p.n_req; r += kThreads) h.p_r[r] = p.p_r[r];
    if (p.stage_lattice) {
        const int n = p.n_req * p.p_max * 16;
        for (int i = tid; i < n; i += kThreads) {
            lp_s[i] = p.cand_logp[i];
            lt_s[i] = p.cand_tok[i];
        }
    }
    // depth 0: the roots, in request order
    for (int r = tid; r < p.n_req; r += kThreads) {
        u_score[r] = 0.f;
        u_parent[r] = -1;
        u_req[r] = (int16_t)r;
        u_token[r] = p.root_tok[r];
        u_meta[r] = 0;
    }
    if (tid == 0) h.lvl_begin[0] = 0, h.lvl_end[0] = p.n_req;
    __syncthreads();

    auto edge = [&](int r, int d, int prank, int j) -> float {
        const int64_t pos = (int64_t)r * p.p_max + (d - 1);
        if (p.conditional) return p.cand_logp[(pos * 16 + prank) * 16 + j];
        return p.stage_lattice ? lp_s[pos * 16 + j] : p.cand_logp[pos * 16 + j];
    };
    auto cand_token = [&](int r, int d, int j) -> int32_t {
        const int64_t pos = (int64_t)r * p.p_max + (d - 1);
        return p.stage_lattice ? lt_s[pos * 16 + j] : p.cand_tok[pos * 16 + j];
    };
    auto split = [&](int ci, int &par_local, int &j) {
        if (p.cand_shift >= 0) {
            par_local = ci >> p.cand_shift;
            j = ci & ((1 << p.cand_shift) - 1);
        } else {
            par_local = ci / p.n_cand;
            j = ci - par_local * p.n_cand;
        }
    };

    int nU = p.n_req;
    bool bad_input = false;
    for (int d = 1; d <= p.p_max && K > 0; ++d) {
        const int pb = h.lvl_begin[d - 1], pe = h.lvl_end[d - 1];
        const int ncand = (pe - pb) * p.n_cand;
        if (ncand == 0) break;
        int valid = 0;
        for (int ci = tid; ci < ncand; ci += kThreads) {
            int pl, j;
            split(ci, pl, j);
            const int par = pb + pl;
            const int r = u_req[par];
            uint32_t key = kInvalid;
            if (d <= h.p_r[r]) {
                const float e = edge(r, d, u_meta[par] & 0xFF, j);
                if (!(e <= 0.f) || isinf(e)) bad_input = true;
                key = score_key(__fadd_rn(u_score[par], e));
                ++valid;
            }
            keys[ci] = key;
        }
        const int nvalid = block_sum(valid, h);
        if (nvalid == 0) break;
        uint32_t tau = kInvalid;   // with take_eq = 0: every valid key is taken
        int take = 0;
        if (nvalid > K) radix_select(keys, ncand, K, tau, take, h);
        const int base = nU;
        const int nsel = select_ordered(keys, ncand, tau, take, h, [&](int ci, int out) {
            int pl, j;
            split(ci, pl, j);
            const int par = pb + pl;
            const int r = u_req[par];
            const int u = base + out;
            u_score[u] = __fadd_rn(u_score[par], edge(r, d, u_meta[par] & 0xFF, j));
            u_parent[u] = (int16_t)par;
            u_req[u] = (int16_t)r;
            u_token[u] = cand_token(r, d, j);
            u_meta[u] = (uint16_t)((d << 8) | j);
        });
        nU += nsel;
        if (tid == 0) h.lvl_begin[d] = base, h.lvl_end[d] = nU;
        __syncthreads();
    }
    if (bad_input) atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);

    // the best R of every kept node: score desc, then storage position
    // (depth, request, path)
    for (int i = tid; i < nU; i += kThreads) keys[i] = score_key(u_score[i]);
    __syncthreads();
    const int R = min(p.R, nU);
    uint32_t tau = kInvalid;
    int take = 0;
    if (R < nU) radix_select(keys, nU, R, tau, take, h);
    select_ordered(keys, nU, tau, take, h, [&](int u, int out) {
        sortbuf[out] = ((unsigned long long)u_req[u] << 46) | ((unsigned long long)keys[u] << 14) |
                       (unsigned long long)u;
    });
    // output row of each selected node = its rank under (request, score desc,
    // storage position); then storage position -> row (reusing the keys)
    int32_t *row_of = reinterpret_cast<int32_t *>(keys);
    for (int i = tid; i < R; i += kThreads) {
        const unsigned long long mine = sortbuf[i];
        int rank_i = 0;
        for (int j = 0; j < R; ++j) rank_i += sortbuf[j] < mine;
        row_of[mine & 0x3FFFull] = rank_i;
    }
    __syncthreads();
    for (int i = tid; i < R; i += kThreads) {
        const int u = (int)(sortbuf[i] & 0x3FFFull);
        const int row = row_of[u];
        const int pu = u_parent[u];
        p.parent[row] = pu < 0 ? -1 : row_of[pu];
        p.token[row] = u_token[u];
        p.req[row] = u_req[u];
        p.score[row] = u_score[u];
        p.depth[row] = (uint8_t)(u_meta[u] >> 8);
        p.rank[row] = (uint8_t)(u_meta[u] & 0xFF);
    }
    // request row offsets: rows before request r = selected nodes of requests < r
    for (int r = tid; r <= p.n_req; r += kThreads) {
        int c = 0;
        for (int j = 0; j < R; ++j) c += (int)(sortbuf[j] >> 46) < r;
        p.req_row_off[r] = c;
    }
    pdl_launch_dependents();
}

// one warp per request: walk down from the root along children whose token
// equals the argmax at their parent (children follow their parent in row order)
__global__ void __launch_bounds__(128) k_tree_accept(const int32_t *parent, const int32_t *token, const uint8_t *depth,
                                                     const int32_t *req_row_off, int32_t n_req, int32_t p_max,
                                                     const int32_t *argmax, int32_t *acc_tok, int32_t *acc_len,
                                                     int32_t *acc_node)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (r >= n_req) return;
    const int lo = req_row_off[r], hi = req_row_off[r + 1];
    int32_t *out = acc_tok + (int64_t)r * (p_max + 1);
    for (int i = lane; i <= p_max; i += 32) out[i] = -1;
    __syncwarp();
    if (lo >= hi) {
        if (lane == 0) {
            acc_len[r] = 0;
            if (acc_node) acc_node[r] = -1;
        }
        return;
    }
    int cur = lo, n = 0;
    for (int guard = 0; guard < p_max; ++guard) {   // a path holds at most p_max drafts
        const int32_t want = argmax[cur];
        int next = -1;
        for (int j0 = cur + 1; j0 < hi && next < 0; j0 += 32) {
            const int j = j0 + lane;
            const bool hit = j < hi && parent[j] == cur && token[j] == want;
            const unsigned m = __ballot_sync(0xffffffffu, hit);
            if (m) next = j0 + __ffs(m) - 1;
        }
        if (next < 0) break;
        if (lane == 0) out[n] = token[next];
        ++n;
        cur = next;
    }
    if (lane == 0) {
        out[n] = argmax[cur];
        acc_len[r] = depth[cur] + 1;
        if (acc_node) acc_node[r] = cur;
    }
}

}  // namespace

namespace w12i {

size_t tree_ws_bytes(int32_t n_req)
{
    (void)n_req;
    return 256;
}

int launch_tree_build(const TreeArgs &a, void *stream)
{
    TreeParams p{};
    p.n_req = a.n_req;
    p.p_max = a.p_max;
    p.n_cand = a.n_cand;
    p.conditional = a.conditional;
    p.budget = a.budget;
    p.R = a.R;
    p.cand_shift = -1;
    for (int sft = 0; sft <= 4; ++sft)
        if (a.n_cand == (1 << sft)) p.cand_shift = sft;
    p.root_tok = a.root_tok;
    p.cand_tok = a.cand_tok;
    p.cand_logp = a.cand_logp;
    p.parent = a.parent;
    p.token = a.token;
    p.req = a.req;
    p.req_row_off = a.req_row_off;
    p.depth = a.depth;
    p.rank = a.rank;
    p.score = a.score;
    p.status = a.status;
    for (int r = 0; r < a.n_req; ++r) p.p_r[r] = (uint8_t)a.p_r_host[r];
    // capacities: kept nodes of all depths, candidates of one depth, rows
    const int K = a.budget - a.n_req;
    const int umax = a.n_req + a.p_max * std::max(K, 0);
    const int cmax = std::max(a.n_req, K) * a.n_cand;
    const int kcap = std::max(umax, cmax);
    auto up = [](int x) { return (x + 15) & ~15; };
    int o = up((int)sizeof(Hdr));
    p.off_keys = o, o = up(o + 4 * kcap);
    p.off_score = o, o = up(o + 4 * umax);
    p.off_token = o, o = up(o + 4 * umax);
    p.off_parent = o, o = up(o + 2 * umax);
    p.off_req = o, o = up(o + 2 * umax);
    p.off_meta = o, o = up(o + 2 * umax);
    p.off_sort = o, o = up(o + 8 * std::max(a.R, 1));
    const int lat = a.n_req * a.p_max * 16;
    const int limit = 227 * 1024;
    p.stage_lattice = (!a.conditional && o + 8 * lat <= limit) ? 1 : 0;
    p.off_lp = o;
    p.off_lt = o + 4 * lat;
    if (p.stage_lattice) o += 8 * lat;
    if (o > limit) return (int)cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(k_tree_build, cudaFuncAttributeMaxDynamicSharedMemorySize, o);
    if (e != cudaSuccess) return (int)e;
    k_tree_build<<<1, kThreads, o, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

int launch_tree_accept(const int32_t *parent, const int32_t *token, const uint8_t *depth, const int32_t *req_row_off,
                       int32_t R, int32_t n_req, int32_t p_max, const int32_t *argmax, int32_t *acc_tok,
                       int32_t *acc_len, int32_t *acc_node, bool pdl, void *stream)
{
    (void)R;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((n_req + 3) / 4);
    cfg.blockDim = dim3(128);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return (int)cudaLaunchKernelEx(&cfg, k_tree_accept, parent, token, depth, req_row_off, n_req, p_max, argmax,
                                   acc_tok, acc_len, acc_node);
}

}  // namespace w12i
