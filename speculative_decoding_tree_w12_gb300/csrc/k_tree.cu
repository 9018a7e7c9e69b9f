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

#include "w12_device.cuh"

using namespace w12d;

namespace {

constexpr int kThreads = 1024;
constexpr int kMaxU = w12i::kMaxBudget + w12i::kMaxPositions * w12i::kMaxBudget;   // kept nodes, all depths
constexpr uint32_t kInvalid = 0xFFFFFFFFu;

struct TreeParams {
    int32_t n_req, p_max, n_cand, conditional, budget, R;
    const int32_t *root_tok;
    const int32_t *cand_tok;
    const float *cand_logp;
    int32_t *parent, *token, *req, *req_row_off;
    uint8_t *depth, *rank;
    float *score;
    // scratch (global): kept nodes of every depth
    float *u_score;
    int32_t *u_parent, *u_req, *u_token, *u_meta;   // meta = depth << 8 | rank
    int32_t *status;
    uint8_t p_r[w12i::kMaxBudget];
};

// ascending key == descending score (a total order on non-NaN floats)
__device__ __forceinline__ uint32_t score_key(float s)
{
    const uint32_t u = __float_as_uint(s);
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ~ord;
}

struct Shared {
    uint32_t hist[256];
    int32_t scan[32];
    int32_t bcast[4];
    int32_t lvl_begin[w12i::kMaxPositions + 2];
    int32_t lvl_end[w12i::kMaxPositions + 2];
    unsigned long long sortbuf[w12i::kMaxBudget];
    uint32_t keys[kMaxU];
};

// exclusive block scan of one int per thread; returns the block total
__device__ int block_scan(int v, int &total, Shared &sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = sh.scan[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh.scan[lane] = w;
    }
    __syncthreads();
    total = sh.scan[31];
    const int before = (warp > 0 ? sh.scan[warp - 1] : 0) + x - v;
    __syncthreads();
    return before;
}

// K smallest of keys[0..n) (1 <= K <= n): threshold tau and how many keys
// equal to tau are taken (the lowest-index ones)
__device__ void radix_select(const uint32_t *keys, int n, int K, uint32_t &tau, int &take_eq, Shared &sh)
{
    uint32_t prefix = 0, mask = 0;
    int krem = K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kThreads) sh.hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += kThreads) {
            const uint32_t k = keys[i];
            if ((k & mask) == prefix) atomicAdd(&sh.hist[(k >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            int c[8], s = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) c[q] = (int)sh.hist[lane * 8 + q], s += c[q];
            int incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int before = incl - s;
            if (before < krem && incl >= krem) {
                int b = before;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (b + c[q] >= krem) {
                        sh.bcast[0] = lane * 8 + q;
                        sh.bcast[1] = b;
                        break;
                    }
                    b += c[q];
                }
            }
        }
        __syncthreads();
        const uint32_t bin = (uint32_t)sh.bcast[0];
        krem -= sh.bcast[1];
        prefix |= bin << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    tau = prefix;
    take_eq = krem;
}

// flags for "selected": key < tau, or key == tau among the first take_eq of
// those; returns each thread's chunk selection via out positions (exclusive)
// Elements are owned in contiguous chunks per thread to keep index order.
template <class Emit>
__device__ int select_and_compact(const uint32_t *keys, int n, uint32_t tau, int take_eq, bool take_all_valid,
                                  Shared &sh, Emit emit)
{
    const int chunk = (n + kThreads - 1) / kThreads;
    const int lo = min(n, (int)threadIdx.x * chunk), hi = min(n, lo + chunk);
    int eq = 0;
    if (!take_all_valid)
        for (int i = lo; i < hi; ++i) eq += keys[i] == tau;
    int eq_total;
    int eq_before = block_scan(eq, eq_total, sh);
    int sel = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t k = keys[i];
        bool s;
        if (take_all_valid) s = k != kInvalid;
        else if (k < tau) s = true;
        else if (k == tau) s = (eq_before++ < take_eq);
        else s = false;
        sel += s;
    }
    int sel_total;
    int pos = block_scan(sel, sel_total, sh);
    if (!take_all_valid) eq_before -= eq;   // rewind to this chunk's start
    for (int i = lo; i < hi; ++i) {
        const uint32_t k = keys[i];
        bool s;
        if (take_all_valid) s = k != kInvalid;
        else if (k < tau) s = true;
        else if (k == tau) s = (eq_before++ < take_eq);
        else s = false;
        if (s) emit(i, pos++);
    }
    __syncthreads();
    return sel_total;
}

__global__ void __launch_bounds__(kThreads, 1) k_tree_build(const TreeParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Shared &sh = *reinterpret_cast<Shared *>(smem_raw);
    const int tid = threadIdx.x;
    const int K = p.budget - p.n_req;   // non-root rows available

    // depth 0: the roots, in request order
    for (int r = tid; r < p.n_req; r += kThreads) {
        p.u_score[r] = 0.f;
        p.u_parent[r] = -1;
        p.u_req[r] = r;
        p.u_token[r] = p.root_tok[r];
        p.u_meta[r] = 0;
    }
    if (tid == 0) sh.lvl_begin[0] = 0, sh.lvl_end[0] = p.n_req;
    __syncthreads();
    int nU = p.n_req;
    bool bad_input = false;

    for (int d = 1; d <= p.p_max && K > 0; ++d) {
        const int pb = sh.lvl_begin[d - 1], pe = sh.lvl_end[d - 1];
        const int ncand = (pe - pb) * p.n_cand;
        if (ncand == 0) break;
        int valid = 0;
        for (int ci = tid; ci < ncand; ci += kThreads) {
            const int par = pb + ci / p.n_cand, j = ci % p.n_cand;
            const int r = p.u_req[par];
            uint32_t key = kInvalid;
            if (d <= p.p_r[r]) {
                const int64_t pos = (int64_t)r * p.p_max + (d - 1);
                const int prank = p.u_meta[par] & 0xFF;
                const float e = p.conditional ? p.cand_logp[(pos * 16 + prank) * 16 + j] : p.cand_logp[pos * 16 + j];
                if (!(e <= 0.f) || isinf(e)) bad_input = true;
                key = score_key(__fadd_rn(p.u_score[par], e));
                ++valid;
            }
            sh.keys[ci] = key;
        }
        int nvalid;
        block_scan(valid, nvalid, sh);
        if (nvalid == 0) break;
        uint32_t tau = 0;
        int take = 0;
        const bool all = nvalid <= K;
        if (!all) radix_select(sh.keys, ncand, K, tau, take, sh);
        const int base = nU;
        const int nsel = select_and_compact(sh.keys, ncand, tau, take, all, sh, [&](int ci, int out) {
            const int par = pb + ci / p.n_cand, j = ci % p.n_cand;
            const int r = p.u_req[par];
            const int64_t pos = (int64_t)r * p.p_max + (d - 1);
            const int prank = p.u_meta[par] & 0xFF;
            const float e = p.conditional ? p.cand_logp[(pos * 16 + prank) * 16 + j] : p.cand_logp[pos * 16 + j];
            const int u = base + out;
            p.u_score[u] = __fadd_rn(p.u_score[par], e);
            p.u_parent[u] = par;
            p.u_req[u] = r;
            p.u_token[u] = p.cand_tok[pos * 16 + j];
            p.u_meta[u] = (d << 8) | j;
        });
        nU += nsel;
        if (tid == 0) sh.lvl_begin[d] = base, sh.lvl_end[d] = nU;
        __threadfence_block();
        __syncthreads();
    }
    if (bad_input) atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);

    // best R of every kept node: score desc, then storage position (depth, request, path)
    for (int i = tid; i < nU; i += kThreads) sh.keys[i] = score_key(p.u_score[i]);
    __syncthreads();
    const int R = min(p.R, nU);
    uint32_t tau = 0;
    int take = 0;
    const bool all = (R == nU);
    if (!all) radix_select(sh.keys, nU, R, tau, take, sh);
    int npow = 1;
    while (npow < R) npow <<= 1;
    for (int i = tid; i < npow; i += kThreads) sh.sortbuf[i] = ~0ull;
    __syncthreads();
    select_and_compact(sh.keys, nU, tau, take, all, sh, [&](int u, int out) {
        sh.sortbuf[out] = ((unsigned long long)p.u_req[u] << 46) | ((unsigned long long)sh.keys[u] << 14) |
                          (unsigned long long)u;
    });
    // bitonic sort: request, then score desc, then storage position
    for (int k = 2; k <= npow; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < npow; i += kThreads) {
                const int ix = i ^ j;
                if (ix > i) {
                    const unsigned long long a = sh.sortbuf[i], b = sh.sortbuf[ix];
                    const bool up = (i & k) == 0;
                    if ((a > b) == up) sh.sortbuf[i] = b, sh.sortbuf[ix] = a;
                }
            }
            __syncthreads();
        }
    }
    // storage position -> output row (reuse the key buffer)
    int32_t *row_of = reinterpret_cast<int32_t *>(sh.keys);
    for (int i = tid; i < R; i += kThreads) row_of[sh.sortbuf[i] & 0x3FFFull] = i;
    __syncthreads();
    for (int i = tid; i < R; i += kThreads) {
        const int u = (int)(sh.sortbuf[i] & 0x3FFFull);
        const int pu = p.u_parent[u];
        p.parent[i] = pu < 0 ? -1 : row_of[pu];
        p.token[i] = p.u_token[u];
        p.req[i] = p.u_req[u];
        p.score[i] = p.u_score[u];
        p.depth[i] = (uint8_t)(p.u_meta[u] >> 8);
        p.rank[i] = (uint8_t)(p.u_meta[u] & 0xFF);
    }
    // request row offsets: first row whose request is >= r
    for (int r = tid; r <= p.n_req; r += kThreads) {
        int lo = 0, hi = R;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((int)(sh.sortbuf[mid] >> 46) < r) lo = mid + 1;
            else hi = mid;
        }
        p.req_row_off[r] = lo;
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
    return (size_t)kMaxU * (4 * 5) + 256;
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
    uint8_t *s = static_cast<uint8_t *>(a.scratch);
    p.u_score = reinterpret_cast<float *>(s);
    p.u_parent = reinterpret_cast<int32_t *>(s + 4 * kMaxU);
    p.u_req = reinterpret_cast<int32_t *>(s + 8 * kMaxU);
    p.u_token = reinterpret_cast<int32_t *>(s + 12 * kMaxU);
    p.u_meta = reinterpret_cast<int32_t *>(s + 16 * kMaxU);
    p.status = a.status;
    for (int r = 0; r < a.n_req; ++r) p.p_r[r] = (uint8_t)a.p_r_host[r];
    const int smem = (int)sizeof(Shared);
    cudaError_t e = cudaFuncSetAttribute(k_tree_build, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    k_tree_build<<<1, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
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
