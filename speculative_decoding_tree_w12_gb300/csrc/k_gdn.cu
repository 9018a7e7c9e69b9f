// Recurrent (Gated DeltaNet) layer over a draft tree (sm_103a).
//
// SpecPilot explainer, 4.2: a GDN head keeps a fixed-size state S (d_v x
// d_k) updated by one rank-one step per token,
//     S <- a S (I - b k k^T) + b v k^T,      o = S q,
// and over a tree the state is recomputed along each root path from the
// committed state instead of being snapshotted per node.  Two methods give
// the per-node outputs:
//
//  * k_gdn_path: the path walk.  Every node replays its root path on a copy
//    of the committed state (FP32).  One CTA owns 32 state rows (rows of S
//    update independently), each warp 4 of them in registers.
//  * the WY form (TreeWY, explainer 4.2).  With g_j the product of gates
//    along node j's root path, u_j = b_j (v_j - a_j S_parent k_j) and
//    S_j = g_j S0 + sum over i on j's path of (g_j/g_i) u_i k_i^T,
//        (I + A) U = B,  A[j,i] = b_j (g_j/g_i) k_i.k_j  (i a strict ancestor)
//                        B[j]   = b_j (v_j - g_j S0 k_j)
//        o_j = g_j S0 q_j + sum over i on j's path of (g_j/g_i) (k_i.q_j) u_i.
//    The state products S0 k and S0 q take S0 as three BF16 pieces that add
//    up to the FP32 value exactly (bit masks and exact subtractions, no
//    rounding), each piece times the BF16 keys/queries (exact products) with
//    FP32 accumulation; k.k and q.k are BF16 products too.  Two kernels:
//      - k_gdn_wy_slice, for a tree of one request: CTAs of (window, head,
//        32 state rows), the products on warp-level MMAs, the solve by depth
//        level across the CTA's warps;
//      - k_gdn_wy, for several requests: CTAs of (window, head) holding all
//        128 state rows in tensor memory, the products on tcgen05 MMAs, each
//        state row's column solved by its own threads.
//    On this part a warp-level m16n8k16 MMA costs tens of cycles of the
//    tensor pipe, so the sliced kernel pays per request; the tensor-memory
//    kernel pays a fixed cost per CTA (tensor memory, the state staged by
//    TMA) and little per request.
//
// The committed-state update after acceptance either replays the accepted
// path (k_gdn_path<true>, like the path kernel) or, given the WY vectors u the
// WY form wrote, adds the path's rank-one terms to the committed state in one
// pass (k_gdn_wy_commit).
//
// Grid of the path walk and the commit: (request, head, d_v / 32); of the WY
// kernels: windows of first rows (several requests per CTA), see below.  Rows
// of one request are its tree rows [req_row_off[r], req_row_off[r+1]), at
// most 64; a larger request sets W12_E_UNSUPPORTED in the status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "w12_device.cuh"

using namespace w12d;

namespace {

constexpr int kD = 128;       // head dimension (d_k = d_v)
constexpr int kVS = 32;       // state rows per CTA
constexpr int kNR = 64;       // rows per request
constexpr int kKS = kD + 16;  // BF16 row stride of K / Q in the slice kernel (rows 8 banks apart)
constexpr int kPS = kVS + 1;  // FP32 row stride of N x 32 matrices
constexpr int kMS = kNR + 1;  // FP32 row stride of N x N matrices
constexpr int kSliceWin = 64; // slice kernel: first rows of the requests one CTA owns
constexpr int kThreads = 256;

struct GdnParams {
    int32_t H, n_req, R, win;
    uint64_t timeout_ns;
    const float *S0;
    const uint16_t *q, *k, *v;
    const float *alpha, *beta;
    const int32_t *parent, *req_row_off, *acc_node;
    float *out;          // o [R][H][d] or, for the commit, the state [n_req][H][d][d]
    float *u;            // the WY vectors u [R][H][d]: written by the WY form when not null, read by its commit
    int32_t *status;
    int32_t debug_flags; // bit 0: CTA (0, 0) of the tensor-memory WY kernel never copies its first state (test hook)
};

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// x = hi + mid + lo exactly, each a BF16 value: hi is x cut to its top 8
// significant bits (its upper 16 bits), mid the same cut of the remainder,
// lo what is left (at most 8 significant bits).  Both subtractions are exact,
// and so is the sum for |x| >= 2^-110 (below that only bits under 2^-126 can
// drop).  Returned as the BF16 pairs of (x0, x1).
__device__ __forceinline__ void split3(float x0, float x1, uint32_t &h, uint32_t &m, uint32_t &l)
{
    const uint32_t a0 = __float_as_uint(x0), a1 = __float_as_uint(x1);
    const float r0 = x0 - __uint_as_float(a0 & 0xffff0000u), r1 = x1 - __uint_as_float(a1 & 0xffff0000u);
    const uint32_t b0 = __float_as_uint(r0), b1 = __float_as_uint(r1);
    const float q0 = r0 - __uint_as_float(b0 & 0xffff0000u), q1 = r1 - __uint_as_float(b1 & 0xffff0000u);
    h = __byte_perm(a0, a1, 0x7632);
    m = __byte_perm(b0, b1, 0x7632);
    l = __byte_perm(__float_as_uint(q0), __float_as_uint(q1), 0x7632);
}

__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bring [ptr, ptr + bytes) into L2 without waiting (16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void *ptr, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

// rows of request r, or -1 (and the status word set) when there are too many
__device__ __forceinline__ int request_rows(const GdnParams &p, int r, int &row0)
{
    row0 = p.req_row_off[r];
    const int n = p.req_row_off[r + 1] - row0;
    if (n < 0 || n > kNR) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, (int32_t)W12_E_UNSUPPORTED);
        return -1;
    }
    return n;
}

// Per-row tree data of one request and head, in shared memory.  Parents,
// gates and strengths load in parallel; then every row walks up its own
// parent chain (shared memory, <= 64 steps) for its ancestor set, depth and
// cumulative gate.  A parent outside the request or not before its child
// sets W12_E_INVAL and makes the row a root.
struct TreeInfo {
    float g[kNR], ginv[kNR], alpha[kNR], beta[kNR];
    unsigned long long anc[kNR];
    int32_t par[kNR], depth[kNR];
};

__device__ __forceinline__ void tree_info(const GdnParams &p, TreeInfo &t, int row0, int n, int h)
{
    const int H = p.H;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        const int pr = p.parent[row0 + j];
        int pl = pr < 0 ? -1 : pr - row0;
        if (pr >= 0 && (pl < 0 || pl >= j)) {
            atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
            pl = -1;
        }
        t.par[j] = pl;
        t.alpha[j] = p.alpha[(size_t)(row0 + j) * H + h];
        t.beta[j] = p.beta[(size_t)(row0 + j) * H + h];
    }
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        unsigned long long m = 0ull;
        float g = t.alpha[j];
        int d = 0;
        for (int i = t.par[j]; i >= 0; i = t.par[i]) {   // strictly decreasing: ends within n steps
            m |= 1ull << i;
            g *= t.alpha[i];
            ++d;
        }
        t.anc[j] = m;
        t.g[j] = g;
        t.ginv[j] = 1.0f / g;
        t.depth[j] = d;
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// WY form for a single request: state-row slices
// ---------------------------------------------------------------------------
//
// Grid (window, head, d_v / 32).  A CTA owns the requests whose first row lies
// in its window of kSliceWin rows and takes them in packs: runs of whole requests
// that span at most 64 rows.  One pass over a pack serves all of its requests
// at once: the ancestor sets, the k.k and q.k products, the solve by depth
// level and the outputs are per row, and rows of different requests never
// meet (a parent lies in its child's request).  Only the state products
// S0 k and S0 q differ by request: each warp takes the pack's requests in
// turn, its B fragments read straight from the request's state slice in
// global memory, the next request's fragments loaded while the current
// one's products run.
//
// Inside every 16-wide k step the products pair MMA k-slot 2t + e with
// feature 4t + e and slot 2t + 8 + e with feature 4t + 2 + e (t = lane % 4,
// e = 0, 1), for both operands: a sum over k does not depend on the order, and
// each lane then reads four consecutive features with one load.

struct SliceShared {
    __nv_bfloat16 K[kNR * kKS], Q[kNR * kKS];
    float V[kNR * kPS], P[kNR * kPS], Rq[kNR * kPS], U[kNR * kPS];
    float KK[kNR * kMS], QK[kNR * kMS];
    TreeInfo t;
    unsigned long long starts;   // bit i: a request of the pack starts at pack row i
    int32_t rq[kNR];             // the request that starts at pack row i
    int32_t lvl_cnt[kNR];        // rows per depth level, then each row's place in its level
    int8_t lidx[kNR];
    int8_t order[kNR];
    int8_t lvl_off[kNR + 2];
    int32_t maxd, pack_end;
};

// B fragments of one 8-row tile of a request's state slice: lane (g, t) holds
// S[row g][16 s + 4 t .. 16 s + 4 t + 3] for the eight k steps s
__device__ __forceinline__ const float *state_rows(const GdnParams &p, int r, int h, int vrow)
{
    return p.S0 + (((size_t)r * p.H + h) * kD + vrow) * kD;
}

__device__ __forceinline__ void mma_a(const __nv_bfloat16 *X, int row, int col, uint32_t a[4])
{
    const uint2 lo = *reinterpret_cast<const uint2 *>(&X[row * kKS + col]);
    const uint2 hi = *reinterpret_cast<const uint2 *>(&X[(row + 8) * kKS + col]);
    a[0] = lo.x;
    a[2] = lo.y;
    a[1] = hi.x;
    a[3] = hi.y;
}

__global__ void __launch_bounds__(kThreads, 2) k_gdn_wy_slice(const GdnParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SliceShared &s = *reinterpret_cast<SliceShared *>(smem_raw);
    const int h = blockIdx.y, vs = blockIdx.z * kVS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int H = p.H;
    const int w0 = blockIdx.x * kSliceWin, w1 = w0 + kSliceWin;

    // the requests whose first row lies in [w0, w1): [r_lo, r_hi).  Every CTA
    // checks every request's row range first, so all of them agree on the
    // requests' places (or all stop).
    int r_lo = 0, r_hi = 0, bad = 0;
    for (int base = 0; base < p.n_req; base += kThreads) {
        const int r = base + tid;
        int lo = 0, hi = 0;
        if (r < p.n_req) {
            const int o0 = p.req_row_off[r], o1 = p.req_row_off[r + 1];
            const int code = (o1 - o0 < 0 || o1 - o0 > kNR) ? (int)W12_E_UNSUPPORTED
                             : (o0 < 0 || o1 > p.R)         ? (int)W12_E_INVAL
                                                            : 0;
            if (code) {
                atomicCAS(p.status, 0, code);
                bad = 1;
            }
            lo = o0 < w0;
            hi = o0 < w1;
        }
        r_lo += __syncthreads_count(lo);
        r_hi += __syncthreads_count(hi);
    }
    if (__syncthreads_or(bad) || r_lo >= r_hi) return;

    int a = p.req_row_off[r_lo];
    const int row_end = p.req_row_off[r_hi];
    while (a < row_end) {
        // this pack: the requests that start at or after row a and end by a + 64
        if (tid == 0) {
            s.pack_end = a;
            s.starts = 0ull;
            s.maxd = 0;
        }
        if (tid < kNR) s.lvl_cnt[tid] = 0;
        __syncthreads();
        // (each request's state slice starts on its way to L2 at once: the
        // warps read the slices one request after another)
        for (int r = r_lo + tid; r < r_hi; r += kThreads) {
            const int o0 = p.req_row_off[r], o1 = p.req_row_off[r + 1];
            if (o0 >= a && o1 <= a + kNR && o1 > o0) {
                atomicMax(&s.pack_end, o1);
                atomicOr(&s.starts, 1ull << (o0 - a));
                s.rq[o0 - a] = r;
                prefetch_l2(state_rows(p, r, h, vs), kVS * kD * sizeof(float));
            }
        }
        __syncthreads();
        const int n = s.pack_end - a, n16 = (n + 15) & ~15;
        const unsigned long long starts = s.starts;

        // every global read of the pack issued before its first shared-memory
        // store: K and Q rows (16-byte pieces, zero padding to 16-row tiles),
        // the value slice, the rows' parents, gates and strengths, and this
        // warp's fragments of the first request's state
        const int mat = warp >> 2, nt = (warp & 3) * 8;
        const float *srow = state_rows(p, s.rq[0], h, vs + nt + g8) + 4 * t4;
        float4 sf[kD / 16];
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) sf[ks] = *reinterpret_cast<const float4 *>(srow + 16 * ks);
        uint4 kv[kNR * 16 / kThreads], qv[kNR * 16 / kThreads];
        uint32_t vv[kNR * 16 / kThreads];
#pragma unroll
        for (int i = 0; i < kNR * 16 / kThreads; ++i) {
            const int e = tid + i * kThreads, j = e >> 4;
            kv[i] = qv[i] = make_uint4(0, 0, 0, 0);
            vv[i] = 0;
            if (j < n) {
                const size_t base = ((size_t)(a + j) * H + h) * kD;
                kv[i] = *reinterpret_cast<const uint4 *>(p.k + base + (e & 15) * 8);
                qv[i] = *reinterpret_cast<const uint4 *>(p.q + base + (e & 15) * 8);
                vv[i] = *reinterpret_cast<const uint32_t *>(p.v + base + vs + (e & 15) * 2);
            }
        }
        int pr = -1;
        float al = 0.f, be = 0.f;
        if (tid < n) {
            pr = p.parent[a + tid];
            al = p.alpha[(size_t)(a + tid) * H + h];
            be = p.beta[(size_t)(a + tid) * H + h];
        }
#pragma unroll
        for (int i = 0; i < kNR * 16 / kThreads; ++i) {
            const int e = tid + i * kThreads, j = e >> 4;
            if (j < n16) {
                *reinterpret_cast<uint4 *>(&s.K[j * kKS + (e & 15) * 8]) = kv[i];
                *reinterpret_cast<uint4 *>(&s.Q[j * kKS + (e & 15) * 8]) = qv[i];
            }
            if (j < n) {
                s.V[j * kPS + (e & 15) * 2] = __uint_as_float(vv[i] << 16);
                s.V[j * kPS + (e & 15) * 2 + 1] = __uint_as_float(vv[i] & 0xffff0000u);
            }
        }
        // parents: inside the row's own request and before the row, else
        // W12_E_INVAL and the row becomes a root
        if (tid < n) {
            const int rs = 63 - __clzll((long long)(starts & (~0ull >> (63 - tid))));   // the request's first row
            int pl = pr < 0 ? -1 : pr - a;
            if (pr >= 0 && (pl < rs || pl >= tid)) {
                atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
                pl = -1;
            }
            s.t.par[tid] = pl;
            s.t.alpha[tid] = al;
            s.t.beta[tid] = be;
        }
        __syncthreads();
        // ancestor sets, cumulative gates, depths
        if (tid < n) {
            unsigned long long m = 0ull;
            float g = s.t.alpha[tid];
            int d = 0;
            for (int i = s.t.par[tid]; i >= 0; i = s.t.par[i]) {   // strictly decreasing: ends within n steps
                m |= 1ull << i;
                g *= s.t.alpha[i];
                ++d;
            }
            s.t.anc[tid] = m;
            s.t.g[tid] = g;
            s.t.ginv[tid] = 1.0f / g;
            s.t.depth[tid] = d;
            atomicMax(&s.maxd, d);
            s.lidx[tid] = (int8_t)atomicAdd(&s.lvl_cnt[d], 1);
        }
        __syncthreads();
        // rows ordered by depth level (rows of different requests share
        // levels; the order inside a level does not matter): warp 0 scans the
        // level counts and places the rows while the other warps go on
        if (warp == 0) {
            const int maxd = s.maxd;
            const int c0 = lane <= maxd ? s.lvl_cnt[lane] : 0, c1 = lane + 32 <= maxd ? s.lvl_cnt[lane + 32] : 0;
            int i0 = c0, i1 = c1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u0 = __shfl_up_sync(0xffffffffu, i0, o), u1 = __shfl_up_sync(0xffffffffu, i1, o);
                if (lane >= o) {
                    i0 += u0;
                    i1 += u1;
                }
            }
            i1 += __shfl_sync(0xffffffffu, i0, 31);
            s.lvl_off[lane] = (int8_t)(i0 - c0);
            s.lvl_off[lane + 32] = (int8_t)(i1 - c1);
            if (lane == 0) s.lvl_off[kNR] = (int8_t)n;
            __syncwarp();
            for (int j = lane; j < n; j += 32) s.order[s.lvl_off[s.t.depth[j]] + s.lidx[j]] = (int8_t)j;
        }

        // KK = K K^T and QK = Q K^T: warp -> (matrix, two 8-column tiles).  A
        // tile pair is skipped when no row of it can be an ancestor (or the
        // row itself) of a row of the other in the same request; those
        // entries are never read.
        const __nv_bfloat16 *X = mat ? s.Q : s.K;
        const int mt_n = n16 / 16;
        {
            float *Y = mat ? s.QK : s.KK;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int n0 = ((warp & 3) * 2 + half) * 8;
                if (n0 >= n16) continue;
                bool need[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int m0 = m * 16, m1 = m0 + 16;
                    // rows i in [n0, n0 + 8) and j in [m0, m1), i <= j, one request:
                    // overlapping ranges, or the request of row m0 starts before n0 + 8
                    const int rs_m0 = 63 - __clzll((long long)(starts & (~0ull >> (63 - m0))));
                    need[m] = m < mt_n && n0 < m1 && (n0 + 8 > m0 || rs_m0 < n0 + 8);
                }
                float acc[4][4];
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[m][e] = 0.f;
#pragma unroll 2
                for (int ks = 0; ks < kD; ks += 16) {
                    const uint2 b = *reinterpret_cast<const uint2 *>(&s.K[(n0 + g8) * kKS + ks + t4 * 4]);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        if (need[m]) {
                            uint32_t af[4];
                            mma_a(X, m * 16 + g8, ks + t4 * 4, af);
                            mma_bf16(acc[m], af, b.x, b.y);
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    if (need[m]) {
                        const int r0 = m * 16 + g8, c0 = n0 + t4 * 2;
                        Y[r0 * kMS + c0] = acc[m][0];
                        Y[r0 * kMS + c0 + 1] = acc[m][1];
                        Y[(r0 + 8) * kMS + c0] = acc[m][2];
                        Y[(r0 + 8) * kMS + c0 + 1] = acc[m][3];
                    }
                }
            }
        }

        // state products, request by request: P = K S^T folded at once into
        // B = b (v - g P), and Rq = Q S^T.  Warp -> (matrix, 8-column tile);
        // two accumulators per 16-row tile (even and odd k steps).
        {
            unsigned long long m = starts;
            while (m) {
                const int st = __ffsll((long long)m) - 1;
                m &= m - 1;
                const int en = m ? __ffsll((long long)m) - 1 : n;
                const float *nrow = m ? state_rows(p, s.rq[en], h, vs + nt + g8) + 4 * t4 : nullptr;
                const int t0 = st >> 4, t1 = (en - 1) >> 4;
                float acc[4][2][4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[u][q][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    uint32_t bh0, bm0, bl0, bh1, bm1, bl1;
                    split3(sf[ks].x, sf[ks].y, bh0, bm0, bl0);
                    split3(sf[ks].z, sf[ks].w, bh1, bm1, bl1);
                    if (nrow) sf[ks] = *reinterpret_cast<const float4 *>(nrow + 16 * ks);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (t0 + u <= t1) {
                            uint32_t af[4];
                            mma_a(X, (t0 + u) * 16 + g8, 16 * ks + t4 * 4, af);
                            mma_bf16(acc[u][ks & 1], af, bl0, bl1);
                            mma_bf16(acc[u][ks & 1], af, bm0, bm1);
                            mma_bf16(acc[u][ks & 1], af, bh0, bh1);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (t0 + u <= t1) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = (t0 + u) * 16 + g8 + (e >> 1) * 8, c = nt + t4 * 2 + (e & 1);
                            if (j >= st && j < en) {
                                const float y = acc[u][0][e] + acc[u][1][e];
                                if (mat)
                                    s.Rq[j * kPS + c] = y;
                                else
                                    s.P[j * kPS + c] = s.t.beta[j] * (s.V[j * kPS + c] - s.t.g[j] * y);
                            }
                        }
                    }
                }
            }
        }
        __syncthreads();

        // forward substitution by depth level: U[j] = B[j] - b_j g_j sum_anc (k_i.k_j / g_i) U[i]
        const int c = tid & 31, slot = tid >> 5;
        const int n_lvl = s.maxd + 1;
        for (int L = 0; L < n_lvl; ++L) {
            const int lo = s.lvl_off[L], hi = s.lvl_off[L + 1];
            for (int t = lo + slot; t < hi; t += kThreads / 32) {
                const int j = s.order[t];
                float sum = 0.f;
                unsigned long long am = s.t.anc[j];
                while (am) {
                    const int i = __ffsll((long long)am) - 1;
                    am &= am - 1;
                    sum = fmaf(s.KK[j * kMS + i] * s.t.ginv[i], s.U[i * kPS + c], sum);
                }
                s.U[j * kPS + c] = s.P[j * kPS + c] - s.t.beta[j] * s.t.g[j] * sum;
            }
            __syncthreads();
        }
        // outputs: o_j = g_j (S0 q_j + sum over the path (k_i.q_j / g_i) u_i)
        for (int j = slot; j < n; j += kThreads / 32) {
            float sum = s.Rq[j * kPS + c];
            unsigned long long am = s.t.anc[j] | (1ull << j);
            while (am) {
                const int i = __ffsll((long long)am) - 1;
                am &= am - 1;
                sum = fmaf(s.QK[j * kMS + i] * s.t.ginv[i], s.U[i * kPS + c], sum);
            }
            p.out[((size_t)(a + j) * H + h) * kD + vs + c] = s.t.g[j] * sum;
            if (p.u) p.u[((size_t)(a + j) * H + h) * kD + vs + c] = s.U[j * kPS + c];
        }
        a += n;
        __syncthreads();   // the next pack reuses every buffer
    }
}

// ---------------------------------------------------------------------------
// WY form for several requests: tensor memory
// ---------------------------------------------------------------------------
//
// Grid (window, head), one CTA per SM.  A CTA owns the requests whose first
// row lies in its window of p.win rows and takes them in packs: runs of at
// most kPackReqs whole requests spanning at most 64 rows.  At a pack's start
// the tree data of its rows is built (ancestor sets, cumulative gates), the
// key and query rows go to shared memory as BF16 blocks, one per request (its
// keys, its queries, zero rows up to a multiple of 16).
//
// Two warp roles then run the pack's requests as a pipeline:
//  * splitters (warps 8..11, one state row each: TMEM lane = state row c,
//    columns = features): the request's state arrives in shared memory by
//    TMA (sixteen 32 x 32 FP32 boxes, 128-byte swizzle, so that every thread
//    reads its own row without bank conflicts); once read, the next
//    request's copy starts.  Once the tensor cores have released the A
//    columns, the splitters write the state as three exact BF16 pieces into
//    tensor memory (A of the state products), the threads of the first 2n
//    lanes also the request's key and query rows (A of k.k and q.k); one
//    thread issues the MMAs (M = 128, N = the request's block rows):
//        D [c][  j ] = S0 k_j  and  D [c][n + j] = S0 q_j   (3 pieces x 8 k steps)
//        D2[j][  i ] = k_j.k_i and  D2[n + j][i] = q_j.k_i  (8 k steps);
//  * solvers (warps 0..7): copy D and D2 out of tensor memory (which frees
//    them for the next request), then take the request's rows by depth, a
//    group of rows of one depth at a time (none is an ancestor of another),
//    each thread for its own state row's column:
//        u_j = b_j (v_j - g_j S0 k_j) - sum over the ancestors (b_j g_j k_i.k_j / g_i) u_i,
//        o_j = g_j S0 q_j + sum over the path (g_j k_i.q_j / g_i) u_i,
//    one pass over the ancestors for both sums.  When every request of the
//    pack has at most 45 rows, two groups of four warps take alternate
//    requests (one thread per column, each group with its own half of the
//    k.k / q.k buffers); otherwise all eight warps take each request, two
//    threads per column sharing each depth group.
//
// Hand-offs: request r's MMAs complete bar_mma[r % 2] (a waiter has always
// seen request r - 2 complete, so its parity is never two phases ahead);
// bar_dfree counts the solver warps that have copied D and D2 out; bar_stage
// the state copies.  Every wait is bounded; each role decides to stop with a
// barrier reduction, so that a stop never leaves a named barrier short.

constexpr int kWyThreads = 384;
constexpr int kSolvers = 256;       // warps 0..7: two per quarter of the state rows
constexpr int kSplitters = 128;     // warps 8..11: one state row per thread
constexpr int kPackReqs = 8;        // requests per pack: bounds the blocks' zero padding
constexpr int kXRows = 248;         // block rows: at most 2 * 64 + 14 * kPackReqs
constexpr uint32_t kStageBytes = kD * kD * sizeof(float);   // one request's state (one head)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColPiece = 0;   // S0 as three BF16 pieces, 64 columns each
constexpr uint32_t kColX = 192;     // the request's key and query rows
constexpr uint32_t kColD = 256;     // state products, up to 128 columns
constexpr uint32_t kColD2 = 384;    // k.k and q.k, up to 64 columns
constexpr int kBarSplit = 1, kBarSolve = 2;   // named barriers of the two roles
constexpr int kBarGroup = 3;                  // and of the two solver groups (3, 4)
constexpr int kHalfTri = 1040;                // a group's k.k / q.k entries: requests of up to 45 rows
constexpr int kTri = kNR * (kNR + 1) / 2;     // entries (j, i), i <= j, of an N x N lower triangle

__device__ __forceinline__ int tri(int j, int i) { return j * (j + 1) / 2 + i; }

struct WyShared {
    uint8_t stage[kStageBytes];   // the state being split: box (row quarter, feature quarter) = 32 rows x 128 B
    uint8_t X[2][kXRows * 128];   // key/query blocks, BF16, K-major, 128-byte swizzle: [feature half][row][64]
    float PU[kNR * kD];           // S0 k, replaced row by row by u: [pack row][state row]
    float Rq[kNR * kD];           // S0 q
    float KK[kTri], QK[kTri];     // b_j g_j k_i.k_j / g_i and g_j q_j.k_i / g_i of the current request (lower triangles)
    uint16_t V[kNR * kD];         // value rows (BF16): [pack row][state row]
    TreeInfo t;
    unsigned long long starts;    // bit i: a request of the pack starts at pack row i
    int32_t rq[kNR];              // the request starting at pack row i
    int32_t blk[kNR];             // its block's first row
    int8_t order[kNR];            // each request's rows by depth (a request's entries start at its first row)
    int8_t run[kNR];              // entries from this one on with its depth, in its request (at most 8)
    int32_t pack_end;
    int32_t two_groups;           // the pack's requests are solved by two groups of solvers
    uint32_t tmem;
    int32_t abort;
    unsigned long long bar_mma[2];   // request r's MMAs are done: bar_mma[r % 2], phase r / 2
    unsigned long long bar_dfree; // the solvers have copied D and D2 out
    unsigned long long bar_stage; // the request's state is in shared memory
};

static_assert(sizeof(WyShared) + 1024 <= 227 * 1024, "WY shared memory above the per-CTA limit");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ bool elect_lane()
{
    uint32_t e;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
    return e != 0;
}

// 32 lanes x 16 columns of 32 bits: register j of lane i <- TMEM (lane base + i, col + j)
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// named barrier `id` over `threads` threads that also ANDs `v` across them
__device__ __forceinline__ bool bar_all(int id, int threads, bool v)
{
    uint32_t out;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(out)
                 : "r"((uint32_t)v), "r"(id), "r"(threads)
                 : "memory");
    return out != 0;
}

// byte offset of 16-byte piece `chunk` (features 8 chunk .. 8 chunk + 7 of
// the half) of block row `row` in one feature half of X
__device__ __forceinline__ uint32_t x_off(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

__global__ void __launch_bounds__(kWyThreads, 1) k_gdn_wy(const __grid_constant__ CUtensorMap smap, const GdnParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    WyShared &s = *reinterpret_cast<WyShared *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    const int h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H;
    const int w0 = blockIdx.x * p.win, w1 = w0 + p.win;

    // the requests whose first row lies in [w0, w1): [r_lo, r_hi).  Every CTA
    // checks every request's row range first, so all of them agree on the
    // requests' places (or all stop).
    int r_lo = 0, r_hi = 0, bad = 0;
    for (int base = 0; base < p.n_req; base += kWyThreads) {
        const int r = base + tid;
        int lo = 0, hi = 0;
        if (r < p.n_req) {
            const int o0 = p.req_row_off[r], o1 = p.req_row_off[r + 1];
            const int code = (o1 - o0 < 0 || o1 - o0 > kNR) ? (int)W12_E_UNSUPPORTED
                             : (o0 < 0 || o1 > p.R)         ? (int)W12_E_INVAL
                                                            : 0;
            if (code) {
                atomicCAS(p.status, 0, code);
                bad = 1;
            }
            lo = o0 < w0;
            hi = o0 < w1;
        }
        r_lo += __syncthreads_count(lo);
        r_hi += __syncthreads_count(hi);
    }
    if (__syncthreads_or(bad) || r_lo >= r_hi) return;

    // (two barriers for the MMAs: a waiter for request r has always seen
    // request r - 2 complete, so the parity it waits for is never two phases
    // ahead, whichever solver group takes r)
    const uint32_t bar_mma0 = smem_u32(&s.bar_mma[0]), bar_dfree = smem_u32(&s.bar_dfree);
    auto bar_mma = [&](uint32_t r) { return bar_mma0 + 8u * (r & 1u); };
    auto mma_par = [](uint32_t r) { return (r >> 1) & 1u; };
    const uint32_t bar_stage = smem_u32(&s.bar_stage), stage = smem_u32(s.stage);
    if (tid == 0) {
        mbar_init(bar_mma(0), 1);
        mbar_init(bar_mma(1), 1);
        mbar_init(bar_dfree, 4);   // one arrival per warp of the solver group (or of warps 0..3)
        mbar_init(bar_stage, 1);
        prefetch_tmap(&smap);
        s.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&s.tmem), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;   // this warp's TMEM lane quarter
    const uint32_t x0 = smem_u32(s.X[0]), x1 = smem_u32(s.X[1]);
    const bool splitter = warp >= 8;
    const int c = (warp & 3) * 32 + lane;           // state row: TMEM lane
    const int hs = (warp >> 2) & 1;                 // a solver's half of the work on its row
    // request r's state (head h) into the stage: sixteen 32 x 32 boxes
    auto stage_state = [&](int r) {
        mbar_expect_tx(bar_stage, kStageBytes);
        const int row0 = (r * H + h) * kD;
#pragma unroll
        for (int b = 0; b < 16; ++b)
            tma_load_2d(stage + b * 4096, &smap, (b & 3) * 32, row0 + (b >> 2) * 32, bar_stage);
    };
    uint32_t rc = 0;                                // requests taken so far (barrier phases)
    uint32_t n_staged = 0;                          // thread kSolvers: state copies issued
    bool go = true;
    bool issue_ok = true;                           // warp 8: the last MMA issue went ahead

    int a = p.req_row_off[r_lo];
    const int row_end = p.req_row_off[r_hi];
    while (a < row_end && go) {
        // reads that need only the pack's first row, issued before the pack is
        // known (all in bounds; rows past the pack are never used): the rows'
        // parents, gates and strengths, and the value rows
        int pr = -1;
        float al = 0.f, be = 0.f;
        const int rows_avail = min(kNR, p.R - a);
        if (tid < rows_avail) {
            pr = p.parent[a + tid];
            al = p.alpha[(size_t)(a + tid) * H + h];
            be = p.beta[(size_t)(a + tid) * H + h];
        }
        for (int e = tid; e < rows_avail * 16; e += kWyThreads) {
            const int j = e >> 4, ch = e & 15;
            cp_async16(smem_u32(&s.V[j * kD + ch * 8]), p.v + ((size_t)(a + j) * H + h) * kD + ch * 8);
        }
        // this pack: up to kPackReqs requests that start at or after row a and end by a + 64
        if (tid == 0) {
            s.pack_end = a;
            s.starts = 0ull;
        }
        __syncthreads();
        for (int r = r_lo + tid; r < r_hi; r += kWyThreads) {
            const int o0 = p.req_row_off[r], o1 = p.req_row_off[r + 1];
            if (o0 >= a && o1 <= a + kNR && o1 > o0) {
                atomicOr(&s.starts, 1ull << (o0 - a));
                s.rq[o0 - a] = r;
                s.blk[o0 - a] = o1 - o0;   // rows, for the block offsets below
            }
        }
        __syncthreads();
        if (tid == 0) {
            unsigned long long m = s.starts;
            int blk = 0, end = 0, q = 0, big = 0;
            for (; q < kPackReqs && m; ++q) {
                const int st = __ffsll((long long)m) - 1;
                m &= m - 1;
                const int rows = s.blk[st];
                s.blk[st] = blk;
                blk += (2 * rows + 15) & ~15;
                end = st + rows;
                big |= rows * (rows + 1) / 2 > kHalfTri;
            }
            if (m) s.starts &= (1ull << (__ffsll((long long)m) - 1)) - 1;   // the rest goes to the next pack
            s.pack_end = a + end;
            s.two_groups = q > 1 && !big;
        }
        __syncthreads();
        const int n = s.pack_end - a;
        const unsigned long long starts = s.starts;
        if (tid == kSolvers) {   // the first request's state
            const bool withheld = (p.debug_flags & 1) && blockIdx.x == 0 && blockIdx.y == 0 && rc == 0;
            if (!withheld) {   // (the test hook leaves the first copy out: the splitters' wait runs out)
                stage_state(s.rq[0]);
                ++n_staged;
            }
        }

        // the rest of the pack's reads: the key / query blocks (asynchronous
        // copies into shared memory; each later request's state is copied by
        // TMA once the previous one has been split)
        {
            unsigned long long m = starts;
            while (m) {
                const int st = __ffsll((long long)m) - 1;
                m &= m - 1;
                const int en = m ? __ffsll((long long)m) - 1 : n, nr = en - st;
                const int blk = s.blk[st], brows = (2 * nr + 15) & ~15;
                for (int e = tid; e < brows * 16; e += kWyThreads) {
                    const int q = e >> 4, ch = e & 15, row = blk + q;
                    if (q < 2 * nr) {
                        const uint16_t *src = (q < nr ? p.k + ((size_t)(a + st + q) * H + h) * kD
                                                      : p.q + ((size_t)(a + st + q - nr) * H + h) * kD) + ch * 8;
                        cp_async16((ch < 8 ? x0 : x1) + x_off(row, ch & 7), src);
                    } else {
                        *reinterpret_cast<uint4 *>(&s.X[ch >> 3][x_off(row, ch & 7)]) = make_uint4(0, 0, 0, 0);
                    }
                }
            }
        }
        if (tid < n) {
            // parents: inside the row's own request and before the row, else
            // W12_E_INVAL and the row becomes a root
            const int rs = 63 - __clzll((long long)(starts & (~0ull >> (63 - tid))));   // the request's first row
            int pl = pr < 0 ? -1 : pr - a;
            if (pr >= 0 && (pl < rs || pl >= tid)) {
                atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
                pl = -1;
            }
            s.t.par[tid] = pl;
            s.t.alpha[tid] = al;
            s.t.beta[tid] = be;
        }
        __syncthreads();
        // ancestor sets and cumulative gates
        if (tid < n) {
            unsigned long long m = 0ull;
            float g = s.t.alpha[tid];
            for (int i = s.t.par[tid]; i >= 0; i = s.t.par[i]) {   // strictly decreasing: ends within n steps
                m |= 1ull << i;
                g *= s.t.alpha[i];
            }
            s.t.anc[tid] = m;
            s.t.g[tid] = g;
            s.t.ginv[tid] = 1.0f / g;
            s.t.depth[tid] = __popcll(m);
        }
        __syncthreads();
        // each request's rows ordered by depth, then by row
        if (tid < n) {
            const unsigned long long below = starts & (~0ull >> (63 - tid));
            const unsigned long long above = starts & ~below;
            const int rs = 63 - __clzll((long long)below), re = above ? __ffsll((long long)above) - 1 : n;
            const int dj = s.t.depth[tid];
            int pos = rs;
            for (int i = rs; i < re; ++i) {
                const int di = s.t.depth[i];
                pos += (di < dj) || (di == dj && i < tid);
            }
            s.order[pos] = (int8_t)tid;
            // the run of entries with this depth from position pos on
            int later = 0;
            for (int i = rs; i < re; ++i) later += s.t.depth[i] == dj && i > tid;
            s.run[pos] = (int8_t)min(later + 1, 8);
        }
        cp_async_wait_all();
        __syncthreads();

        unsigned long long m = starts;
        if (splitter) {
            // ------------------------------------------------------------ splitters
            while (m && go) {
                const int st = __ffsll((long long)m) - 1;
                m &= m - 1;
                const int en = m ? __ffsll((long long)m) - 1 : n, nr = en - st;
                const int blk = s.blk[st];
                // the state is staged and the previous request's MMAs have read
                // the A columns: warp 8 polls, the other splitters wait in the
                // barrier (every splitter decides alike: a stop anywhere stops
                // them all here)
                bool ok = issue_ok;
                if (warp == 8) {
                    if (rc > 0) ok = ok && mbar_wait(bar_mma(rc - 1), mma_par(rc - 1), p.timeout_ns, p.status, &s.abort);
                    ok = ok && mbar_wait(bar_stage, rc & 1u, p.timeout_ns, p.status, &s.abort);
                    ok = __all_sync(0xffffffffu, ok);
                }
                if (!bar_all(kBarSplit, kSplitters, ok)) {
                    go = false;
                    break;
                }
                tc_fence_after();
                uint32_t w[32];
#pragma unroll 1
                for (int kh = 0; kh < 2; ++kh) {
                    // features [64 kh, 64 kh + 64) of state row c: feature quarters 2 kh, 2 kh + 1
                    float4 sv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t box = (uint32_t)((warp & 3) * 4 + 2 * kh + (i >> 3)) * 4096u;
                        sv[i] = *reinterpret_cast<const float4 *>(s.stage + box + lane * 128 + (((i & 7) ^ (lane & 7)) << 4));
                    }
#pragma unroll
                    for (int piece = 0; piece < 3; ++piece) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint32_t b0 = __float_as_uint(sv[i].x), b1 = __float_as_uint(sv[i].y);
                            const uint32_t b2 = __float_as_uint(sv[i].z), b3 = __float_as_uint(sv[i].w);
                            w[2 * i] = __byte_perm(b0, b1, 0x7632);
                            w[2 * i + 1] = __byte_perm(b2, b3, 0x7632);
                            if (piece < 2) {   // the remainder after this piece (exact), two at a time
                                const float2 m1 = make_float2(-1.f, -1.f);
                                const float2 lo = __ffma2_rn(make_float2(__uint_as_float(b0 & 0xffff0000u),
                                                                         __uint_as_float(b1 & 0xffff0000u)),
                                                             m1, make_float2(sv[i].x, sv[i].y));
                                const float2 hi = __ffma2_rn(make_float2(__uint_as_float(b2 & 0xffff0000u),
                                                                         __uint_as_float(b3 & 0xffff0000u)),
                                                             m1, make_float2(sv[i].z, sv[i].w));
                                sv[i] = make_float4(lo.x, lo.y, hi.x, hi.y);
                            }
                        }
                        // (the source registers are read at issue: one completion wait below)
                        tmem_st_x32(tmem + lane_base + kColPiece + 64 * piece + 32 * kh, w);
                    }
                    // the request's key and query rows (lanes below 2 nr; the
                    // other lanes of those warps copy a valid row, never read)
                    if ((warp & 3) * 32 < 2 * nr) {
                        const int row = blk + min(c, 2 * nr - 1);
                        const uint8_t *xs = s.X[kh];
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(xs + x_off(row, ch));
                            w[4 * ch] = v.x;
                            w[4 * ch + 1] = v.y;
                            w[4 * ch + 2] = v.z;
                            w[4 * ch + 3] = v.w;
                        }
                        tmem_st_x32(tmem + lane_base + kColX + 32 * kh, w);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                named_bar(kBarSplit, kSplitters);   // the stage is read, the A columns written
                if (tid == kSolvers && m) {   // the next request's state (this thread issues every copy)
                    stage_state(s.rq[en]);
                    ++n_staged;
                }
                if (warp == 8) {
                    // the solvers have copied the previous request's D and D2 out
                    bool ok = rc == 0 || mbar_wait(bar_dfree, (rc - 1) & 1u, p.timeout_ns, p.status, &s.abort);
                    ok = __all_sync(0xffffffffu, ok);
                    tc_fence_after();
                    if (ok && elect_lane()) {
                        const uint32_t N = (2 * nr + 15) & ~15, N2 = (nr + 15) & ~15;
                        const uint32_t id = idesc_bf16_f32(128, N), id2 = idesc_bf16_f32(128, N2);
                        const uint64_t b0 = smem_desc_sw128(x0 + blk * 128), b1 = smem_desc_sw128(x1 + blk * 128);
#pragma unroll
                        for (int piece = 0; piece < 3; ++piece)
#pragma unroll
                            for (int ks = 0; ks < 8; ++ks)
                                tc_mma_ts(tmem + kColD, tmem + kColPiece + 64 * piece + 8 * ks,
                                          (ks < 4 ? b0 : b1) + (uint64_t)((ks & 3) * 2), id, (piece | ks) ? 1u : 0u);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc_mma_ts(tmem + kColD2, tmem + kColX + 8 * ks,
                                      (ks < 4 ? b0 : b1) + (uint64_t)((ks & 3) * 2), id2, ks ? 1u : 0u);
                        tc_commit(bar_mma(rc));
                    }
                    __syncwarp();
                    if (!ok) {
                        issue_ok = false;   // the other splitters see it at their next vote,
                        s.abort = 1;        // the solvers' waits end at once
                    }
                }
                ++rc;
            }
        } else {
            // -------------------------------------------------------------- solvers
            // Two groups of four warps take alternate requests when every
            // request of the pack fits half of the k.k / q.k buffers; else all
            // eight warps take each request, two threads per column.
            const bool two = s.two_groups != 0;
            const int grp = warp >> 2;                          // 0: warps 0..3, 1: warps 4..7
            const int bar_id = two ? kBarGroup + grp : kBarSolve, bar_n = two ? 128 : kSolvers;
            const int nsplit = two ? 1 : 2, part = two ? 0 : hs;   // column chunks / group rows shared by nsplit warps
            const int poller = two ? 4 * grp : 0;
            float *KKb = s.KK + (two ? grp * kHalfTri : 0), *QKb = s.QK + (two ? grp * kHalfTri : 0);
            uint32_t rq_i = rc;                                   // this request's number
            for (int q = 0; m && go; ++q, ++rq_i) {
                const int st = __ffsll((long long)m) - 1;
                m &= m - 1;
                const int en = m ? __ffsll((long long)m) - 1 : n, nr = en - st;
                if (two && (q & 1) != grp) continue;
                // the MMAs are done: one warp polls, the others wait in the barrier
                bool ok = true;
                if (warp == poller)
                    ok = __all_sync(0xffffffffu, mbar_wait(bar_mma(rq_i), mma_par(rq_i), p.timeout_ns, p.status, &s.abort));
                if (!bar_all(bar_id, bar_n, ok)) {
                    go = false;
                    break;
                }
                tc_fence_after();
                // D -> S0 k and S0 q rows; D2 -> the scaled k.k and q.k rows
                const bool d2 = (warp & 3) * 32 < 2 * nr;   // this warp's lanes hold rows of D2
                for (int c0 = 16 * part; c0 < 2 * nr; c0 += 16 * nsplit) {
                    uint32_t v[16], v2[16];
                    tmem_ld_x16(tmem + lane_base + kColD + c0, v);
                    if (d2 && c0 < nr) tmem_ld_x16(tmem + lane_base + kColD2 + c0, v2);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int col = c0 + i;
                        if (col < nr)
                            s.PU[(st + col) * kD + c] = __uint_as_float(v[i]);
                        else if (col < 2 * nr)
                            s.Rq[(st + col - nr) * kD + c] = __uint_as_float(v[i]);
                    }
                    if (d2 && c0 < nr && c < 2 * nr) {
                        const int jj = c < nr ? c : c - nr, j = st + jj;
                        const float f = c < nr ? s.t.beta[j] * s.t.g[j] : s.t.g[j];
                        float *dst = c < nr ? KKb : QKb;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (c0 + i <= jj) dst[tri(jj, c0 + i)] = __uint_as_float(v2[i]) * s.t.ginv[st + c0 + i] * f;
                    }
                }
                tc_fence_before();
                named_bar(bar_id, bar_n);
                if ((two || warp < 4) && lane == 0) mbar_arrive(bar_dfree);   // D, D2 free for the next MMAs
                // rows by depth, a run of rows of one depth at a time (none is an
                // ancestor of another, and all have `depth` ancestors), up to four
                // per thread: one pass over the ancestors for u_j and o_j
                for (int t = st; t < en;) {
                    const int d = s.t.depth[s.order[t]], gsz = min((int)s.run[t], 4 * nsplit);
                    const int mine = (gsz - part + nsplit - 1) / nsplit;   // entries part, part + nsplit, ...
                    if (mine > 0) {
                        int jr[4], tb[4];
                        float u[4], o[4];
                        unsigned long long am[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int j = s.order[t + part + nsplit * min(k, mine - 1)];   // the last one again past the end
                            jr[k] = j;
                            tb[k] = tri(j - st, 0) - st;                                    // entry (j, i) at index tb + i
                            const float vj = __uint_as_float((uint32_t)s.V[j * kD + c] << 16);
                            u[k] = s.t.beta[j] * (vj - s.t.g[j] * s.PU[j * kD + c]);
                            o[k] = s.t.g[j] * s.Rq[j * kD + c];
                            am[k] = s.t.anc[j];
                        }
                        for (int step = 0; step < d; ++step) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int i = __ffsll((long long)am[k]) - 1;
                                am[k] &= am[k] - 1;
                                const float ui = s.PU[i * kD + c];
                                u[k] = fmaf(-KKb[tb[k] + i], ui, u[k]);
                                o[k] = fmaf(QKb[tb[k] + i], ui, o[k]);
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (k < mine) {
                                s.PU[jr[k] * kD + c] = u[k];
                                p.out[((size_t)(a + jr[k]) * H + h) * kD + c] = fmaf(QKb[tb[k] + jr[k]], u[k], o[k]);
                                if (p.u) p.u[((size_t)(a + jr[k]) * H + h) * kD + c] = u[k];
                            }
                        }
                    }
                    t += gsz;
                    // the next depth reads these rows' u: with two threads per
                    // column a barrier; with one, the thread's own order (and
                    // the vote before the group's next request orders the
                    // solve before that request's k.k / q.k writes)
                    if (!two) named_bar(bar_id, bar_n);
                }
            }
            rc += __popcll(starts);   // (both roles count the pack's requests)
        }
        if (__syncthreads_or(!go)) go = false;   // the pack is done (or stopped) on both sides
        a += n;
    }

    // release tensor memory once no MMA is in flight and leave no copy into
    // shared memory running: after a stop, one more bounded wait for the last
    // commit and the last state copy
    if (!go && rc > 0) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar_mma(rc - 1), mma_par(rc - 1)) && globaltimer() - t0 < p.timeout_ns) {
        }
    }
    if (!go && tid == kSolvers && n_staged > 0) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar_stage, (n_staged - 1) & 1u) && globaltimer() - t0 < p.timeout_ns) {
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// path walk (and the commit replay)
// ---------------------------------------------------------------------------

struct PathShared {
    float S[kVS * kD];
    float K[kNR * kD];
    float V[kNR * kVS];
    TreeInfo t;
};

// One walk: a warp's 4 state rows (lane holds columns lane + 32 e) start from
// the committed state and take the update of every row in `path` (a row set
// closed under parents; ascending row order is root first).
__device__ __forceinline__ void walk(const PathShared &s, unsigned long long path, int vrow0, int lane, float w[4][4])
{
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) w[r][e] = s.S[(vrow0 + r) * kD + lane + 32 * e];
    while (path) {
        const int i = __ffsll((long long)path) - 1;
        path &= path - 1;
        float kk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) kk[e] = s.K[i * kD + lane + 32 * e];
        const float a = s.t.alpha[i], b = s.t.beta[i];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float d = w[r][0] * kk[0];
#pragma unroll
            for (int e = 1; e < 4; ++e) d = fmaf(w[r][e], kk[e], d);
#pragma unroll
            for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            // a (S - b (S k) k^T) + b v k^T, row by row
            const float coef = b * (s.V[i * kVS + vrow0 + r] - a * d);
#pragma unroll
            for (int e = 0; e < 4; ++e) w[r][e] = fmaf(coef, kk[e], a * w[r][e]);
        }
    }
}

template <bool kCommit>
__global__ void __launch_bounds__(kThreads, 1) k_gdn_path(const GdnParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    PathShared &s = *reinterpret_cast<PathShared *>(smem_raw);
    const int r = blockIdx.x, h = blockIdx.y, vs = blockIdx.z * kVS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H;
    const float *S0 = p.S0 + (((size_t)r * H + h) * kD + vs) * kD;
    for (int e = tid; e < kVS * kD / 4; e += kThreads)
        *reinterpret_cast<float4 *>(&s.S[e * 4]) = *reinterpret_cast<const float4 *>(S0 + (size_t)e * 4);
    int row0;
    const int n = request_rows(p, r, row0);
    if (n <= 0) return;
    const int vrow = warp * 4;   // this warp's first row inside the slice
    float w[4][4];
    if constexpr (kCommit) {
        // the accepted row's path first, then only its rows' keys and values
        tree_info(p, s.t, row0, n, h);
        const int node = p.acc_node[r] - row0;
        unsigned long long path = 0ull;
        if (node >= 0 && node < n) {
            path = s.t.anc[node] | (1ull << node);
        } else if (tid == 0) {
            atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
        }
        for (int e = tid; e < n * kD; e += kThreads) {
            const int j = e / kD, c = e % kD;
            if ((path >> j) & 1ull) s.K[j * kD + c] = bf(p.k[((size_t)(row0 + j) * H + h) * kD + c]);
        }
        for (int e = tid; e < n * kVS; e += kThreads) {
            const int j = e / kVS, c = e % kVS;
            if ((path >> j) & 1ull) s.V[j * kVS + c] = bf(p.v[((size_t)(row0 + j) * H + h) * kD + vs + c]);
        }
        __syncthreads();
        // every read of S0 happened before tree_info's barriers: writing in place is safe
        walk(s, path, vrow, lane, w);
        float *dst = p.out + (((size_t)r * H + h) * kD + vs) * kD;
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[(size_t)(vrow + rr) * kD + lane + 32 * e] = w[rr][e];
    } else {
        for (int e = tid; e < n * kD; e += kThreads) {
            const int j = e / kD, c = e % kD;
            s.K[j * kD + c] = bf(p.k[((size_t)(row0 + j) * H + h) * kD + c]);
        }
        for (int e = tid; e < n * kVS; e += kThreads) {
            const int j = e / kVS, c = e % kVS;
            s.V[j * kVS + c] = bf(p.v[((size_t)(row0 + j) * H + h) * kD + vs + c]);
        }
        tree_info(p, s.t, row0, n, h);
        for (int node = 0; node < n; ++node) {
            walk(s, s.t.anc[node] | (1ull << node), vrow, lane, w);
            float qq[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) qq[e] = bf(p.q[((size_t)(row0 + node) * H + h) * kD + lane + 32 * e]);
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                float d = w[rr][0] * qq[0];
#pragma unroll
                for (int e = 1; e < 4; ++e) d = fmaf(w[rr][e], qq[e], d);
#pragma unroll
                for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                if (lane == 0) p.out[((size_t)(row0 + node) * H + h) * kD + vs + vrow + rr] = d;
            }
        }
    }
}


// ---------------------------------------------------------------------------
// commit from the WY vectors
// ---------------------------------------------------------------------------
//
// The state after the accepted row j in WY form (explainer 4.2):
//     S_j = g_j S0 + sum over i on j's root path of (g_j / g_i) u_i k_i^T,
// with the u_i the WY form wrote.  One pass over the committed state: each
// thread reads four float4 of the slice, adds the path's rank-one terms and
// writes them back (in place if the state is S0).  Grid (request, head,
// d_v / 32).

struct WyCommitShared {
    uint16_t K[kNR * kD];  // keys of the request's rows (BF16)
    float Uc[kNR * kVS];   // their WY vectors, this CTA's 32 state rows
    float coef[kNR];       // g_acc / g_i per path entry
    int32_t path[kNR];     // the accepted row's root path, accepted row first
    int32_t par[kNR];
    float alpha[kNR];
    int32_t plen;
    float gacc;
};

__global__ void __launch_bounds__(kThreads) k_gdn_wy_commit(const GdnParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    WyCommitShared &s = *reinterpret_cast<WyCommitShared *>(smem_raw);
    const int r = blockIdx.x, h = blockIdx.y, vs = blockIdx.z * kVS;
    const int tid = threadIdx.x;
    const int H = p.H;
    // every read issued before the path is known: the committed slice (rows
    // vs .. vs + 31), the keys and this slice of the WY vectors of all the
    // request's rows (asynchronous copies), the rows' parents and gates
    const float *S0 = p.S0 + (((size_t)r * H + h) * kD + vs) * kD;
    float4 sv[kVS * kD / 4 / kThreads];
#pragma unroll
    for (int i = 0; i < kVS * kD / 4 / kThreads; ++i)
        sv[i] = *reinterpret_cast<const float4 *>(S0 + (size_t)(tid + i * kThreads) * 4);
    int row0;
    const int n = request_rows(p, r, row0);
    if (n <= 0) return;
    if (row0 < 0 || row0 + n > p.R) {   // rows past the tree: nothing read, nothing written
        if (tid == 0) atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
        return;
    }
    for (int e = tid; e < n * 16; e += kThreads) {
        const int j = e >> 4, ch = e & 15;
        cp_async16(smem_u32(&s.K[j * kD + ch * 8]), p.k + ((size_t)(row0 + j) * H + h) * kD + ch * 8);
    }
    for (int e = tid; e < n * (kVS / 4); e += kThreads) {
        const int j = e / (kVS / 4), ch = e % (kVS / 4);
        cp_async16(smem_u32(&s.Uc[j * kVS + ch * 4]), p.u + ((size_t)(row0 + j) * H + h) * kD + vs + ch * 4);
    }
    if (tid < n) {
        const int pr = p.parent[row0 + tid];
        int pl = pr < 0 ? -1 : pr - row0;
        if (pr >= 0 && (pl < 0 || pl >= tid)) {
            atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);
            pl = -1;
        }
        s.par[tid] = pl;
        s.alpha[tid] = p.alpha[(size_t)(row0 + tid) * H + h];
    }
    __syncthreads();
    if (tid == 0) {
        // the accepted row's root path (strictly decreasing rows: at most n
        // steps), then the cumulative gates from the root down
        const int node = p.acc_node[r] - row0;
        int len = 0;
        if (node >= 0 && node < n) {
            for (int i = node; i >= 0; i = s.par[i]) s.path[len++] = i;
        } else {
            atomicCAS(p.status, 0, (int32_t)W12_E_INVAL);   // the state stays S0[r]
        }
        float g = 1.f;
        for (int q = len - 1; q >= 0; --q) {
            g *= s.alpha[s.path[q]];
            s.coef[q] = g;
        }
        s.gacc = g;
        for (int q = 0; q < len; ++q) s.coef[q] = g / s.coef[q];
        s.plen = len;
    }
    cp_async_wait_all();
    __syncthreads();
    const int len = s.plen;
    const float gacc = s.gacc;
    float *dst = p.out + (((size_t)r * H + h) * kD + vs) * kD;
#pragma unroll
    for (int i = 0; i < kVS * kD / 4 / kThreads; ++i) {
        const int e = tid + i * kThreads, row = e >> 5, c4 = (e & 31) * 4;
        float4 x = make_float4(gacc * sv[i].x, gacc * sv[i].y, gacc * sv[i].z, gacc * sv[i].w);
        for (int q = 0; q < len; ++q) {
            const int j = s.path[q];
            const float w = s.coef[q] * s.Uc[j * kVS + row];
            const uint2 kb = *reinterpret_cast<const uint2 *>(&s.K[j * kD + c4]);
            x.x = fmaf(w, __uint_as_float(kb.x << 16), x.x);
            x.y = fmaf(w, __uint_as_float(kb.x & 0xffff0000u), x.y);
            x.z = fmaf(w, __uint_as_float(kb.y << 16), x.z);
            x.w = fmaf(w, __uint_as_float(kb.y & 0xffff0000u), x.w);
        }
        *reinterpret_cast<float4 *>(dst + (size_t)row * kD + c4) = x;
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_gdn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

}  // namespace

namespace w12i {

int launch_gdn(const GdnArgs &a, int mode, void *stream)
{
    if (a.H < 1 || a.n_req < 1 || a.R < 1) return (int)cudaErrorInvalidValue;
    GdnParams p{};
    p.H = a.H;
    p.n_req = a.n_req;
    p.R = a.R;
    p.timeout_ns = a.timeout_ns;
    p.S0 = a.S0;
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.parent = a.parent;
    p.req_row_off = a.req_row_off;
    p.acc_node = a.acc_node;
    p.out = a.out;
    p.u = a.u;
    p.debug_flags = a.debug_flags;
    p.status = a.status;
    // plain launches: with an early start the next layer's CTAs would share
    // SMs with this one's and leave others idle (one CTA per SM is the
    // balanced placement of a 128-CTA layer)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.n_req, a.H, kD / kVS);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    if (mode == kGdnWy && a.n_req == 1) {
        // one request: (window, head, 32-row slice) CTAs, two per SM
        cfg.gridDim = dim3((a.R + kSliceWin - 1) / kSliceWin, a.H, kD / kVS);
        cfg.dynamicSmemBytes = sizeof(SliceShared);
        cudaError_t e = cudaFuncSetAttribute(k_gdn_wy_slice, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return (int)e;
        return (int)cudaLaunchKernelEx(&cfg, k_gdn_wy_slice, p);
    }
    if (mode == kGdnWy) {
        // several requests: windows sized so that the (window, head) CTAs fit one wave
        const int wins = std::max(1, a.num_sms / a.H);
        p.win = (a.R + wins - 1) / wins;
        cfg.gridDim = dim3((a.R + p.win - 1) / p.win, a.H);
        cfg.blockDim = dim3(kWyThreads);
        cfg.dynamicSmemBytes = sizeof(WyShared) + 1024;
        // the states as rows of 128 FP32 features, copied in 32 x 32 boxes
        EncodeTiledFn enc = encode_fn_gdn();
        if (!enc) return (int)cudaErrorNotSupported;
        CUtensorMap smap;
        const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)a.n_req * a.H * kD};
        const cuuint64_t strides[1] = {(cuuint64_t)kD * sizeof(float)};
        const cuuint32_t box[2] = {32, 32}, estr[2] = {1, 1};
        if (enc(&smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(a.S0), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return (int)cudaErrorInvalidValue;
        cudaError_t e = cudaFuncSetAttribute(k_gdn_wy, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return (int)e;
        return (int)cudaLaunchKernelEx(&cfg, k_gdn_wy, smap, p);
    }
    if (mode == kGdnCommitWy) {
        cfg.dynamicSmemBytes = sizeof(WyCommitShared);
        cudaError_t e = cudaFuncSetAttribute(k_gdn_wy_commit, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return (int)e;
        return (int)cudaLaunchKernelEx(&cfg, k_gdn_wy_commit, p);
    }
    cfg.dynamicSmemBytes = sizeof(PathShared);
    const auto kern = mode == kGdnCommit ? k_gdn_path<true> : k_gdn_path<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.dynamicSmemBytes);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace w12i
