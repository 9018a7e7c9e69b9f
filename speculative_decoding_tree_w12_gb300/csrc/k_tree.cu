// Best-first draft tree under a shared node budget, and greedy acceptance
// (sm_103a).
//
// SpecPilot explainer, 4.2: keep the N nodes with the highest path score
// sum log p(child | parent); 4.4: one budget for all requests, filled from
// the highest path log-probability, prefix-closed per request.  Explainer
// 1.1: greedy verification keeps the drafts equal to the target's argmax and
// appends that argmax as a bonus.
//
// Tree build, one CTA.  Order of nodes: score descending, then depth, then
// request, then path (candidate indices from the root).  Every edge
// log-probability is <= 0, so a child comes after its parent, and a node's
// children, ranked by their own FP32 score and then candidate index, come in
// that order too.  Best-first selection therefore only ever needs, for each
// selected node, its best child not yet taken: the next node of the tree is
// the best of those "frontier" children.  One warp runs the R selections
// (each lane keeps the best frontier child of the nodes it owns, a warp
// argmax picks the winner, the winner's parent advances to its next child
// and the new node's children are ranked by 16 lanes); the other warps check
// and stage the lattice before, and write the request-grouped rows after.
#include <cuda_runtime.h>

#include <algorithm>

#include "w12_device.cuh"

using namespace w12d;

namespace {

constexpr int kThreads = 256;
constexpr int kCap = w12i::kMaxBudget;   // selected nodes

struct TreeParams {
    int32_t n_req, p_max, n_cand, conditional, budget, R;
    int32_t stage_lattice;   // non-conditional log-probs and tokens copied to shared memory
    const int32_t *root_tok;
    const int32_t *cand_tok;
    const float *cand_logp;
    int32_t *parent, *token, *req, *req_row_off;
    uint8_t *depth, *rank;
    float *score;
    int32_t *status;
    uint8_t p_r[w12i::kMaxBudget];
};

// Selected nodes, in selection order, plus the frontier child of each.
struct Nodes {
    unsigned long long key1[kCap];     // frontier child: ordered score << 32 | ~(depth << 16 | request); 0 = none
    unsigned long long key2[kCap];     // frontier child: ~path
    unsigned long long path[kCap];     // candidate index of depth d at bits 64 - 4d
    unsigned long long perm[kCap];     // children ranked best first, 4 bits each
    float score[kCap];
    uint32_t dr[kCap];                 // depth << 16 | request
    int32_t tok[kCap];
    int32_t row[kCap];
    int16_t par[kCap];
    uint8_t rank[kCap];
    uint8_t next[kCap];                // rank position of the frontier child
    uint8_t nch[kCap];                 // children available (0 at the depth limit)
    uint8_t p_r[w12i::kMaxBudget];
    int32_t n_sel;
    int32_t bad;
    __device__ __forceinline__ void store(int x, float s, uint32_t d, unsigned long long pa, int j, int pr, int32_t t,
                                          unsigned long long pm, int nc, unsigned long long k1, unsigned long long k2)
    {
        score[x] = s, dr[x] = d, path[x] = pa, rank[x] = (uint8_t)j, par[x] = (int16_t)pr, tok[x] = t;
        perm[x] = pm, next[x] = 0, nch[x] = (uint8_t)nc, key1[x] = k1, key2[x] = k2;
    }
};

// Order-preserving map of a finite float to an unsigned integer (larger
// float, larger integer; -0 and +0 map alike, as they compare equal).
__device__ __forceinline__ uint32_t ord_score(float s)
{
    const uint32_t u = __float_as_uint(__fadd_rn(s, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord_score(uint32_t o)
{
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
// the tree order as one comparison: larger (key1, key2) comes first
__device__ __forceinline__ unsigned long long make_key1(float s, uint32_t dr)
{
    return ((unsigned long long)ord_score(s) << 32) | (unsigned long long)(~dr);
}

// ---------------------------------------------------------------------------
// shared pieces of both build kernels
// ---------------------------------------------------------------------------

// Every log-probability a node could use must be finite and <= 0; sets *bad.
// Then copies the non-conditional lattice to shared memory when asked.
__device__ void check_and_stage(const TreeParams &p, const uint8_t *p_r, int32_t *bad, float *lp_s, int32_t *lt_s)
{
    const int tid = threadIdx.x, nth = blockDim.x;
    const int NC = p.n_cand, PM = p.p_max;
    bool b = false;
    const int rows = p.conditional ? NC : 1;
    const int per_req = PM * 16 * (p.conditional ? 16 : 1);
    for (int64_t i = tid; i < (int64_t)p.n_req * per_req; i += nth) {
        const int r = (int)(i / per_req), rem = (int)(i - (int64_t)r * per_req);
        const int d = p.conditional ? rem / 256 : rem / 16;
        const int pc = p.conditional ? (rem / 16) & 15 : 0, j = rem & 15;
        if (d < p_r[r] && pc < rows && j < NC) {
            const float v = p.cand_logp[i];
            if (!(v <= 0.f) || isinf(v)) b = true;
        }
    }
    if (b) *bad = 1;
    if (p.stage_lattice) {
        const int lat = p.n_req * PM * 16;
        for (int i = tid; i < lat; i += nth) {
            lp_s[i] = p.cand_logp[i];
            lt_s[i] = p.cand_tok[i];
        }
    }
}

// edge log-probability into child candidate j at depth d (1-based position)
// of request r whose parent has candidate rank prank; the child's token
struct Lattice {
    const TreeParams *p;
    const float *lp_s;
    const int32_t *lt_s;
    __device__ __forceinline__ float edge(int r, int d, int prank, int j) const
    {
        const int64_t pos = (int64_t)r * p->p_max + (d - 1);
        if (p->conditional) return p->cand_logp[(pos * 16 + prank) * 16 + j];
        return p->stage_lattice ? lp_s[pos * 16 + j] : p->cand_logp[pos * 16 + j];
    }
    __device__ __forceinline__ int32_t token(int r, int d, int j) const
    {
        const int64_t pos = (int64_t)r * p->p_max + (d - 1);
        return p->stage_lattice ? lt_s[pos * 16 + j] : p->cand_tok[pos * 16 + j];
    }
};

// Node x (score sx, depth/request dr, path, candidate rank jx) was just
// selected: the warp ranks its children by FP32 score then candidate index
// (lane k scores child k) and returns the key of its best child (k1 = 0 when
// it has none) and the ranking (4 bits per child, best first).
__device__ __forceinline__ void rank_children(const Lattice &L, int NC, int p_r, float sx, uint32_t dr,
                                              unsigned long long path, int jx, unsigned long long &perm,
                                              unsigned long long &k1, unsigned long long &k2, bool &has)
{
    const int lane = threadIdx.x & 31;
    const int d = (int)(dr >> 16), r = (int)(dr & 0xFFFF);
    has = d < p_r;
    float cs = -INFINITY;
    if (has && lane < NC) cs = __fadd_rn(sx, L.edge(r, d + 1, jx, lane));
    // rank = children before this one; branch-free so the warp stays converged
    int pos = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float o = __shfl_sync(0xffffffffu, cs, k);
        pos += (int)((k < NC) & ((o > cs) | ((o == cs) & (k < lane))));
    }
    const unsigned long long mine = (has && lane < NC) ? ((unsigned long long)lane << (4 * pos)) : 0ull;
    const uint32_t lo = __reduce_or_sync(0xffffffffu, (uint32_t)mine);
    const uint32_t hi = __reduce_or_sync(0xffffffffu, (uint32_t)(mine >> 32));
    perm = ((unsigned long long)hi << 32) | lo;
    const int j0 = (int)(perm & 15ull);
    const float best = __shfl_sync(0xffffffffu, cs, j0);
    k1 = has ? make_key1(best, dr + (1u << 16)) : 0ull;
    k2 = has ? ~(path | ((unsigned long long)j0 << (64 - 4 * (d + 1)))) : 0ull;
}

// warp argmax of the lanes' (b1, b2), most significant word first; M1 = 0
// when no lane holds a key
struct WarpMax {
    uint32_t M1, M2, M3, M4;
    int lane;
};
__device__ __forceinline__ WarpMax warp_max(unsigned long long b1, unsigned long long b2)
{
    const uint32_t h1 = (uint32_t)(b1 >> 32), l1 = (uint32_t)b1, h2 = (uint32_t)(b2 >> 32), l2 = (uint32_t)b2;
    WarpMax w;
    w.M1 = __reduce_max_sync(0xffffffffu, h1);
    bool m = h1 == w.M1;
    const uint32_t top = __ballot_sync(0xffffffffu, m);
    if ((top & (top - 1)) == 0) {
        // one lane holds the best score: its other words come by shuffle
        w.lane = __ffs(top) - 1;
        w.M2 = __shfl_sync(0xffffffffu, l1, w.lane);
        w.M3 = __shfl_sync(0xffffffffu, h2, w.lane);
        w.M4 = __shfl_sync(0xffffffffu, l2, w.lane);
        return w;
    }
    w.M2 = __reduce_max_sync(0xffffffffu, m ? l1 : 0u);
    m = m && l1 == w.M2;
    w.M3 = __reduce_max_sync(0xffffffffu, m ? h2 : 0u);
    m = m && h2 == w.M3;
    w.M4 = __reduce_max_sync(0xffffffffu, m ? l2 : 0u);
    m = m && l2 == w.M4;
    w.lane = __ffs(__ballot_sync(0xffffffffu, m)) - 1;
    return w;
}

// One warp's best-first selection over a node store: the store holds the
// nodes selected so far (index order = selection order) and, per node, its
// frontier child (best child not yet taken).  NodeStore provides the arrays
// and `cap`; `req_of_root` maps root index -> request for the initial roots.
// Selects nodes t .. limit-1 (fewer when the frontier empties); lane-local
// bests (b1, b2, bx) persist between calls.  Returns the new count.
template <class S>
__device__ int best_first(S &n, const Lattice &L, int NC, const uint8_t *p_r, int t, int limit,
                          unsigned long long &b1, unsigned long long &b2, int &bx)
{
    const int lane = threadIdx.x & 31;
    for (; t < limit; ++t) {
        const WarpMax w = warp_max(b1, b2);
        if (w.M1 == 0) break;   // every node of the lattice is taken
        const int wx = __shfl_sync(0xffffffffu, bx, w.lane);
        // node t = the frontier child of wx
        const float st = unord_score(w.M1);
        const uint32_t drt = ~w.M2;
        const unsigned long long patht = ~(((unsigned long long)w.M3 << 32) | w.M4);
        const int dt = (int)(drt >> 16);
        const int j = (int)((patht >> (64 - 4 * dt)) & 15ull);
        const int rt = (int)(drt & 0xFFFF);
        const int32_t tok = L.token(rt, dt, j);
        // the parent moves on to its next child: every lane computes its new
        // key from broadcast loads, issued before the new node's stores so
        // that both chains overlap
        const int nx = n.next[wx] + 1;
        const unsigned long long pperm = n.perm[wx], ppath = n.path[wx];
        const uint32_t pdr = n.dr[wx];
        const float psc = n.score[wx];
        const int prk = n.rank[wx], pnch = n.nch[wx];
        const int pdc = (int)(pdr >> 16) + 1;
        const int j2 = (int)((pperm >> (4 * (nx & 15))) & 15ull);
        const bool more = nx < pnch;
        const float pe = more ? L.edge((int)(pdr & 0xFFFF), pdc, prk, j2) : 0.f;
        unsigned long long perm, k1, k2;
        bool has;
        rank_children(L, NC, p_r[rt], st, drt, patht, j, perm, k1, k2, has);
        if (lane == 0) n.store(t, st, drt, patht, j, wx, tok, perm, has ? NC : 0, k1, k2);
        // the parent's owner lane rescans
        {
            const unsigned long long p1 = more ? make_key1(__fadd_rn(psc, pe), pdr + (1u << 16)) : 0ull;
            const unsigned long long p2 = more ? ~(ppath | ((unsigned long long)j2 << (64 - 4 * pdc))) : 0ull;
            __syncwarp();
            if (lane == 0) {
                n.next[wx] = (uint8_t)nx;
                n.key1[wx] = p1;
                n.key2[wx] = p2;
            }
            __syncwarp();
            if (lane == w.lane) {
                b1 = 0, b2 = 0, bx = -1;
                for (int x = lane; x < t; x += 32) {
                    const unsigned long long q1 = n.key1[x], q2 = n.key2[x];
                    const bool better = (q1 > b1) | ((q1 == b1) & (q2 > b2));
                    b1 = better ? q1 : b1;
                    b2 = better ? q2 : b2;
                    bx = better ? x : bx;
                }
                if (b1 == 0) bx = -1;
            }
        }
        {
            const bool better = (lane == (t & 31)) & (k1 != 0) & ((k1 > b1) | ((k1 == b1) & (k2 > b2)));
            b1 = better ? k1 : b1;
            b2 = better ? k2 : b2;
            bx = better ? t : bx;
        }
        __syncwarp();
    }
    return t;
}

// a root (node index x, request r) enters the store; the owner lane of x
// takes its best child as its lane-local best
template <class S>
__device__ void add_root(S &n, const Lattice &L, int NC, const uint8_t *p_r, int x, int r, int32_t tok,
                         unsigned long long &b1, unsigned long long &b2, int &bx)
{
    const int lane = threadIdx.x & 31;
    unsigned long long perm, k1, k2;
    bool has;
    rank_children(L, NC, p_r[r], 0.f, (uint32_t)r, 0ull, 0, perm, k1, k2, has);
    if (lane == 0) n.store(x, 0.f, (uint32_t)r, 0ull, 0, -1, tok, perm, has ? NC : 0, k1, k2);
    if (lane == (x & 31) && k1 != 0 && (k1 > b1 || (k1 == b1 && k2 > b2))) b1 = k1, b2 = k2, bx = x;
    __syncwarp();
}

// The whole budget with one warp, over every request (the store holds them
// all); then rows grouped by request in selection order.  Used for a single
// request, for many requests and when the per-request stores overflow.
__device__ void build_single(Nodes &n, const TreeParams &p, const Lattice &L)
{
    const int tid = threadIdx.x, nth = blockDim.x;
    if (tid < 32) {
        unsigned long long b1 = 0, b2 = 0;
        int bx = -1;
        for (int r = 0; r < p.n_req; ++r) add_root(n, L, p.n_cand, n.p_r, r, r, p.root_tok[r], b1, b2, bx);
        const int t = best_first(n, L, p.n_cand, n.p_r, p.n_req, min(p.R, kCap), b1, b2, bx);
        if (tid == 0) n.n_sel = t;
    }
    __syncthreads();
    // rows: grouped by request, selection order inside
    const int R = n.n_sel;
    for (int i = tid; i < R; i += nth) {
        const int r = (int)(n.dr[i] & 0xFFFF);
        int row = 0;
        for (int k = 0; k < R; ++k) {
            const int rk = (int)(n.dr[k] & 0xFFFF);
            row += rk < r || (rk == r && k < i);
        }
        n.row[i] = row;
    }
    __syncthreads();
    for (int i = tid; i < R; i += nth) {
        const int row = n.row[i];
        p.parent[row] = n.par[i] < 0 ? -1 : n.row[n.par[i]];
        p.token[row] = n.tok[i];
        p.req[row] = (int32_t)(n.dr[i] & 0xFFFF);
        p.score[row] = n.score[i];
        p.depth[row] = (uint8_t)(n.dr[i] >> 16);
        p.rank[row] = n.rank[i];
    }
    for (int r = tid; r <= p.n_req; r += nth) {
        int c = 0;
        for (int k = 0; k < R; ++k) c += (int)(n.dr[k] & 0xFFFF) < r;
        p.req_row_off[r] = c;
    }
}

// ---------------------------------------------------------------------------
// one warp for the whole budget
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads, 1) k_tree_build(const TreeParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    Nodes &n = *reinterpret_cast<Nodes *>(smem);
    float *lp_s = reinterpret_cast<float *>(smem + sizeof(Nodes));
    const int32_t lat = p.n_req * p.p_max * 16;
    int32_t *lt_s = reinterpret_cast<int32_t *>(smem + sizeof(Nodes) + 4 * (p.stage_lattice ? lat : 0));
    const int tid = threadIdx.x;

    // the next kernel (the first verify GEMM) may start now: it streams weights
    // into its shared memory and waits for this grid before it reads rows
    pdl_launch_dependents();
    pdl_wait();
    if (tid == 0) n.bad = 0;
    for (int r = tid; r < p.n_req; r += kThreads) n.p_r[r] = p.p_r[r];
    __syncthreads();
    check_and_stage(p, n.p_r, &n.bad, lp_s, lt_s);
    __syncthreads();
    if (n.bad) {
        if (tid == 0) atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
        return;
    }
    const Lattice L{&p, lp_s, lt_s};
    build_single(n, p, L);
}

// ---------------------------------------------------------------------------
// one warp per request (2 .. 32 requests), or per child of the root (one request)
// ---------------------------------------------------------------------------
//
// The selected set is the first R - n_req non-root nodes of the tree order
// over all requests, and every request's share of it is a prefix of its own
// best-first sequence.  Each warp generates its request's sequence on its
// own, up to a limit; then the CTA checks every unfinished request: once at
// least R - n_req generated nodes come before the request's next node, none
// of its later nodes can be selected.  Requests that are not settled raise
// their limit and go on.  The selection is the first R - n_req generated
// nodes in tree order; each request's count follows from a binary search of
// ranks, where a node's rank is the number of generated nodes before it.
// A request that needs more nodes than its store holds sends the CTA to the
// one-warp build.  With one request the same argument holds for the subtrees
// of the root's children: each is generated by its own warp, and a selected
// node's row is one more than the number of selected nodes before it.

constexpr int kPW = 64;   // nodes per request store (root included)

struct ReqNodes {
    unsigned long long key1[kPW];   // frontier child: ordered score << 32 | ~(depth << 16 | request); 0 = none
    unsigned long long key2[kPW];   // frontier child: ~path
    unsigned long long path[kPW];
    unsigned long long perm[kPW];
    float score[kPW];
    uint32_t dr[kPW];
    int32_t tok[kPW];
    int8_t par[kPW];
    uint8_t rank[kPW];
    uint8_t next[kPW];
    uint8_t nch[kPW];
    __device__ __forceinline__ void store(int x, float s, uint32_t d, unsigned long long pa, int j, int pr, int32_t t,
                                          unsigned long long pm, int nc, unsigned long long k1, unsigned long long k2)
    {
        score[x] = s, dr[x] = d, path[x] = pa, rank[x] = (uint8_t)j, par[x] = (int8_t)pr, tok[x] = t;
        perm[x] = pm, next[x] = 0, nch[x] = (uint8_t)nc, key1[x] = k1, key2[x] = k2;
    }
    // a generated node's own place in the tree order
    __device__ __forceinline__ unsigned long long own1(int x) const { return make_key1(score[x], dr[x]); }
    __device__ __forceinline__ unsigned long long own2(int x) const { return ~path[x]; }
};

struct ParShared {
    ReqNodes rn[32];
    unsigned long long head1[32], head2[32];   // key of the request's next node (0 = none)
    int32_t n_gen[32];                         // nodes generated, root included
    int32_t k_sel[32];                         // non-root nodes selected
    int32_t row_off[33];
    int32_t pending, overflow;
};

constexpr size_t kParSmem = sizeof(ParShared) > sizeof(Nodes) ? sizeof(ParShared) : sizeof(Nodes);

// number of generated nodes (positions first.. of every sequence) that come
// before (h1, h2); lane q searches sequence q, which is in tree order
__device__ __forceinline__ int count_before(const ParShared &s, int n_seq, unsigned long long h1,
                                            unsigned long long h2, int first)
{
    const int lane = threadIdx.x & 31;
    int c = 0;
    if (lane < n_seq) {
        const ReqNodes &q = s.rn[lane];
        int lo = first, hi = s.n_gen[lane];   // first position in [first, n_gen) not before h
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const unsigned long long a1 = q.own1(mid), a2 = q.own2(mid);
            const bool before = (a1 > h1) | ((a1 == h1) & (a2 > h2));
            lo = before ? mid + 1 : lo;
            hi = before ? hi : mid;
        }
        c = lo - first;
    }
    return (int)__reduce_add_sync(0xffffffffu, (uint32_t)c);
}

__global__ void __launch_bounds__(1024, 1) k_tree_build_par(const TreeParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    ParShared &s = *reinterpret_cast<ParShared *>(smem);
    Nodes &n1 = *reinterpret_cast<Nodes *>(smem);   // the one-warp fallback reuses the space
    uint8_t *p_r = smem + kParSmem;
    int32_t *bad = reinterpret_cast<int32_t *>(smem + kParSmem + 512);
    float *lp_s = reinterpret_cast<float *>(smem + kParSmem + 528);
    const int32_t lat = p.n_req * p.p_max * 16;
    int32_t *lt_s = reinterpret_cast<int32_t *>(smem + kParSmem + 528 + 4 * (p.stage_lattice ? lat : 0));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NR = p.n_req, NC = p.n_cand;

    pdl_launch_dependents();
    pdl_wait();
    if (tid == 0) *bad = 0, s.pending = 0, s.overflow = 0;
    for (int r = tid; r < NR; r += blockDim.x) p_r[r] = p.p_r[r];
    __syncthreads();
    check_and_stage(p, p_r, bad, lp_s, lt_s);
    __syncthreads();
    if (*bad) {
        if (tid == 0) atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
        return;
    }
    const Lattice L{&p, lp_s, lt_s};
    const int R = min(p.R, kCap);
    // sequences: one per request, or (one request) one per child of the root,
    // whose subtree is a sequence of its own; position 0 of a request sequence
    // is its root, of a subtree sequence the child, which counts as selected
    const bool sub = NR == 1;
    const int NS = sub ? NC : NR, first = sub ? 0 : 1;
    const int B = max(R - NR, 0);   // non-root nodes to select

    // generation passes
    unsigned long long b1 = 0, b2 = 0;
    int bx = -1, t = 1;
    // first limit: the average share plus a little; unsettled sequences grow
    // their limit by half each pass
    int limit = min(kPW, 1 + (B + NS - 1) / NS + 2);
    ReqNodes &q = s.rn[warp];
    if (sub) {
        // child `warp` of the root: its score is the edge itself (0 + e)
        const float sc = __fadd_rn(0.f, L.edge(0, 1, 0, warp));
        const uint32_t dr = 1u << 16;
        const unsigned long long path = (unsigned long long)warp << 60;
        unsigned long long perm, k1, k2;
        bool has;
        rank_children(L, NC, p_r[0], sc, dr, path, warp, perm, k1, k2, has);
        if (lane == 0) q.store(0, sc, dr, path, warp, -1, L.token(0, 1, warp), perm, has ? NC : 0, k1, k2);
        if (lane == 0 && k1 != 0) b1 = k1, b2 = k2, bx = 0;
        __syncwarp();
    } else {
        add_root(q, L, NC, p_r, 0, warp, p.root_tok[warp], b1, b2, bx);
    }
    bool settled = false;
    for (;;) {
        if (!settled) {
            t = best_first(q, L, NC, p_r, t, limit, b1, b2, bx);
            const WarpMax w = warp_max(b1, b2);
            if (lane == 0) {
                s.n_gen[warp] = t;
                s.head1[warp] = w.M1 ? (((unsigned long long)w.M1 << 32) | w.M2) : 0ull;
                s.head2[warp] = ((unsigned long long)w.M3 << 32) | w.M4;
            }
        }
        __syncthreads();
        if (!settled) {
            const unsigned long long h1 = s.head1[warp], h2 = s.head2[warp];
            settled = h1 == 0 || count_before(s, NS, h1, h2, first) >= B;
            if (!settled && lane == 0) {
                atomicAdd(&s.pending, 1);
                if (limit == kPW) s.overflow = 1;
            }
            if (!settled) limit = min(kPW, limit + max(2, limit / 2));
        }
        __syncthreads();
        const int pending = s.pending, overflow = s.overflow;
        __syncthreads();
        if (overflow) break;
        if (pending == 0) break;
        if (tid == 0) s.pending = 0;
    }
    if (s.overflow) {
        __syncthreads();
        for (int r = tid; r < NR; r += blockDim.x) n1.p_r[r] = p_r[r];
        __syncthreads();
        build_single(n1, p, L);
        return;
    }

    // selection: sequence q keeps its nodes at positions first .. first + k_q - 1,
    // the largest k_q whose last node has fewer than B generated nodes before it
    {
        const int ng = s.n_gen[warp];
        int lo = 0, hi = ng - first;   // k in [lo, hi]
        while (lo < hi) {
            const int k = (lo + hi + 1) >> 1;
            const int x = first + k - 1;
            const int before = count_before(s, NS, q.own1(x), q.own2(x), first);
            if (before < B) lo = k; else hi = k - 1;
        }
        if (lane == 0) s.k_sel[warp] = lo;
    }
    __syncthreads();
    if (sub) {
        // one request: row 0 is the root, a selected node's row is one more than
        // the number of selected nodes before it in the tree order
        const int cnt = s.k_sel[warp];
        for (int i = 0; i < cnt; ++i) {
            const int rk = count_before(s, NS, q.own1(i), q.own2(i), 0);
            if (lane == 0) q.key1[i] = (unsigned long long)(1 + rk);   // the node's row (frontier keys are done with)
        }
        __syncwarp();
        for (int i = lane; i < cnt; i += 32) {
            const int row = (int)q.key1[i];
            p.parent[row] = q.par[i] < 0 ? 0 : (int)q.key1[q.par[i]];
            p.token[row] = q.tok[i];
            p.req[row] = 0;
            p.score[row] = q.score[i];
            p.depth[row] = (uint8_t)(q.dr[i] >> 16);
            p.rank[row] = q.rank[i];
        }
        if (tid == 0) {
            int total = 1;
            for (int w = 0; w < NS; ++w) total += s.k_sel[w];
            p.parent[0] = -1;
            p.token[0] = p.root_tok[0];
            p.req[0] = 0;
            p.score[0] = 0.f;
            p.depth[0] = 0;
            p.rank[0] = 0;
            p.req_row_off[0] = 0;
            p.req_row_off[1] = total;
        }
        return;
    }
    if (tid == 0) {
        int o = 0;
        for (int r = 0; r < NR; ++r) s.row_off[r] = o, o += 1 + s.k_sel[r];
        s.row_off[NR] = o;
    }
    __syncthreads();
    // rows: request order, tree order inside (root first)
    {
        const int base = s.row_off[warp], cnt = 1 + s.k_sel[warp];
        for (int i = lane; i < cnt; i += 32) {
            const int row = base + i;
            p.parent[row] = q.par[i] < 0 ? -1 : base + q.par[i];
            p.token[row] = q.tok[i];
            p.req[row] = warp;
            p.score[row] = q.score[i];
            p.depth[row] = (uint8_t)(q.dr[i] >> 16);
            p.rank[row] = q.rank[i];
        }
    }
    for (int r = tid; r <= NR; r += blockDim.x) p.req_row_off[r] = s.row_off[r];
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
        acc_len[r] = n + 1;   // the tokens written: n drafts and the bonus
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
    if (a.n_req > kCap || a.budget > kCap || a.R > kCap) return (int)cudaErrorInvalidValue;
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
    p.status = a.status;
    for (int r = 0; r < a.n_req; ++r) p.p_r[r] = (uint8_t)a.p_r_host[r];
    const int lat = a.n_req * a.p_max * 16;
    const int limit = 227 * 1024;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool sub = a.n_req == 1 && a.n_cand >= 2 && a.p_max >= 1 && a.p_r_host[0] >= 1;
    if ((a.n_req >= 2 && a.n_req <= 32) || sub) {
        // one warp per request, or (one request) per child of the root
        int o = (int)kParSmem + 528;
        p.stage_lattice = (!a.conditional && o + 8 * lat <= limit) ? 1 : 0;
        if (p.stage_lattice) o += 8 * lat;
        cudaError_t e = cudaFuncSetAttribute(k_tree_build_par, cudaFuncAttributeMaxDynamicSharedMemorySize, o);
        if (e != cudaSuccess) return (int)e;
        k_tree_build_par<<<1, 32 * (sub ? a.n_cand : a.n_req), o, st>>>(p);
        return (int)cudaGetLastError();
    }
    int o = (int)sizeof(Nodes);
    p.stage_lattice = (!a.conditional && o + 8 * lat <= limit) ? 1 : 0;
    if (p.stage_lattice) o += 8 * lat;
    cudaError_t e = cudaFuncSetAttribute(k_tree_build, cudaFuncAttributeMaxDynamicSharedMemorySize, o);
    if (e != cudaSuccess) return (int)e;
    k_tree_build<<<1, kThreads, o, st>>>(p);
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
