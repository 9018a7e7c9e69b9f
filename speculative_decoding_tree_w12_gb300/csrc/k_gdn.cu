// Recurrent (Gated DeltaNet) layer over a draft tree (sm_103a).
//
// SpecPilot explainer, 4.2: a GDN head keeps a fixed-size state S (d_v x
// d_k) updated by one rank-one step per token,
//     S <- a S (I - b k k^T) + b v k^T,      o = S q,
// and over a tree the state is recomputed along each root path from the
// committed state instead of being snapshotted per node.  Two kernels give
// the per-node outputs:
//
//  * k_gdn_path: the path walk.  Every node replays its root path on a copy
//    of the committed state (FP32).  One CTA owns 32 state rows (rows of S
//    update independently), each warp 4 of them in registers.
//  * k_gdn_wy: the WY form (TreeWY, explainer 4.2).  With g_j the product
//    of gates along node j's root path, u_j = b_j (v_j - a_j S_parent k_j)
//    and S_j = g_j S0 + sum over i on j's path of (g_j/g_i) u_i k_i^T,
//        (I + A) U = B,  A[j,i] = b_j (g_j/g_i) k_i.k_j  (i a strict ancestor)
//                        B[j]   = b_j (v_j - g_j S0 k_j)
//        o_j = g_j S0 q_j + sum over i on j's path of (g_j/g_i) (k_i.q_j) u_i.
//    The state products S0 k and S0 q run on tensor cores: S0 is split into
//    three BF16 pieces that add up to the FP32 value exactly, each piece is
//    multiplied by the BF16 keys/queries (exact products) with FP32
//    accumulation.  k.k and k.q are BF16 products too.  The triangular solve
//    (by depth level) and the output sums run on the FP32 pipes.
//
// The committed-state update after acceptance (k_gdn_commit) replays the
// accepted path, like the path kernel, and writes the state.
//
// Grid of every kernel: (request, head, d_v / 32).  Rows of one request are
// its tree rows [req_row_off[r], req_row_off[r+1]), at most 64; a larger
// request sets W12_E_UNSUPPORTED in the status word.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "w12_device.cuh"

using namespace w12d;

namespace {

constexpr int kD = 128;       // head dimension (d_k = d_v)
constexpr int kVS = 32;       // state rows per CTA
constexpr int kNR = 64;       // rows per request
constexpr int kThreads = 256;
constexpr int kKS = kD + 8;   // BF16 row stride of K / Q in shared memory
constexpr int kSS = kD + 4;   // FP32 row stride of the state slice
constexpr int kPS = kVS + 1;  // FP32 row stride of N x 32 matrices
constexpr int kMS = kNR + 1;  // FP32 row stride of N x N matrices

struct GdnParams {
    int32_t H, n_req;
    const float *S0;
    const uint16_t *q, *k, *v;
    const float *alpha, *beta;
    const int32_t *parent, *req_row_off, *acc_node;
    float *out;          // o [R][H][d] or, for the commit, the state [n_req][H][d][d]
    int32_t *status;
};

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 lo, __nv_bfloat16 hi)
{
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// x = hi + mid + lo exactly (24 significand bits in three 8-bit pieces)
__device__ __forceinline__ void split3(float x, __nv_bfloat16 &h, __nv_bfloat16 &m, __nv_bfloat16 &l)
{
    h = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(h);
    m = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(m);
    l = __float2bfloat16_rn(r2);
}

__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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
// WY form
// ---------------------------------------------------------------------------

struct WyShared {
    __nv_bfloat16 K[kNR * kKS], Q[kNR * kKS];
    float S[kVS * kSS];
    float P[kNR * kPS], Rq[kNR * kPS], U[kNR * kPS];
    float KK[kNR * kMS], QK[kNR * kMS];
    TreeInfo t;
    int8_t order[kNR];
    int8_t lvl_off[kNR + 2];
    int32_t maxd;
};

__global__ void __launch_bounds__(kThreads, 1) k_gdn_wy(const GdnParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    WyShared &s = *reinterpret_cast<WyShared *>(smem_raw);
    const int r = blockIdx.x, h = blockIdx.y, vs = blockIdx.z * kVS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H;
    int row0;
    const int n = request_rows(p, r, row0);
    if (n <= 0) return;
    const int n16 = (n + 15) & ~15;
    if (tid == 0) s.maxd = 0;

    // every global read issued before the first shared-memory store: the
    // state slice, K and Q rows (16-byte pieces, zero padding to 16-row
    // tiles) and the value slice (kept in registers until the state slice's
    // space is free)
    const float *S0 = p.S0 + (((size_t)r * H + h) * kD + vs) * kD;
    float4 sv[kVS * kD / 4 / kThreads];
#pragma unroll
    for (int i = 0; i < kVS * kD / 4 / kThreads; ++i)
        sv[i] = *reinterpret_cast<const float4 *>(S0 + (size_t)(tid + i * kThreads) * 4);
    uint4 kv[kNR * 16 / kThreads], qv[kNR * 16 / kThreads];
    uint32_t vv[kNR * 16 / kThreads];
#pragma unroll
    for (int i = 0; i < kNR * 16 / kThreads; ++i) {
        const int e = tid + i * kThreads, j = e >> 4;
        kv[i] = qv[i] = make_uint4(0, 0, 0, 0);
        vv[i] = 0;
        if (j < n) {
            const size_t base = ((size_t)(row0 + j) * H + h) * kD;
            kv[i] = *reinterpret_cast<const uint4 *>(p.k + base + (e & 15) * 8);
            qv[i] = *reinterpret_cast<const uint4 *>(p.q + base + (e & 15) * 8);
            vv[i] = *reinterpret_cast<const uint32_t *>(p.v + base + vs + (e & 15) * 2);
        }
    }
#pragma unroll
    for (int i = 0; i < kVS * kD / 4 / kThreads; ++i) {
        const int e = tid + i * kThreads, v = e / (kD / 4), c4 = (e % (kD / 4)) * 4;
        *reinterpret_cast<float4 *>(&s.S[v * kSS + c4]) = sv[i];
    }
#pragma unroll
    for (int i = 0; i < kNR * 16 / kThreads; ++i) {
        const int e = tid + i * kThreads, j = e >> 4;
        if (j < n16) {
            *reinterpret_cast<uint4 *>(&s.K[j * kKS + (e & 15) * 8]) = kv[i];
            *reinterpret_cast<uint4 *>(&s.Q[j * kKS + (e & 15) * 8]) = qv[i];
        }
    }
    // ancestor sets and cumulative gates, then rows ordered by depth level
    tree_info(p, s.t, row0, n, h);
    for (int j = tid; j < n; j += kThreads) {
        const int dj = s.t.depth[j];
        atomicMax(&s.maxd, dj);
        int pos = 0;
        for (int i = 0; i < n; ++i) {
            const int di = s.t.depth[i];
            pos += (di < dj) || (di == dj && i < j);
        }
        s.order[pos] = (int8_t)j;
    }
    __syncthreads();
    for (int L = tid; L <= s.maxd + 1; L += kThreads) {
        int c = 0;
        for (int i = 0; i < n; ++i) c += s.t.depth[i] < L;
        s.lvl_off[L] = (int8_t)c;
    }
    __syncthreads();

    const int g8 = lane >> 2, t4 = lane & 3;
    const int mt_n = n16 / 16;
    // P = K S^T and Rq = Q S^T (N x 32): warp -> (matrix, 8-column tile), all row tiles
    {
        const __nv_bfloat16 *X = (warp >> 2) ? s.Q : s.K;
        float *Y = (warp >> 2) ? s.Rq : s.P;
        const int nt = (warp & 3) * 8;
        float acc[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[m][e] = 0.f;
#pragma unroll 2
        for (int ks = 0; ks < kD; ks += 16) {
            // B fragment: B[k][n] = S[n][k], split into three BF16 pieces
            const float *srow = &s.S[(nt + g8) * kSS + ks + t4 * 2];
            __nv_bfloat16 h0, m0, l0, h1, m1, l1, h2, m2, l2, h3, m3, l3;
            split3(srow[0], h0, m0, l0);
            split3(srow[1], h1, m1, l1);
            split3(srow[8], h2, m2, l2);
            split3(srow[9], h3, m3, l3);
            const uint32_t bh0 = pack2(h0, h1), bh1 = pack2(h2, h3);
            const uint32_t bm0 = pack2(m0, m1), bm1 = pack2(m2, m3);
            const uint32_t bl0 = pack2(l0, l1), bl1 = pack2(l2, l3);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (m < mt_n) {
                    const __nv_bfloat16 *xr = &X[(m * 16 + g8) * kKS + ks + t4 * 2];
                    uint32_t a[4];
                    a[0] = *reinterpret_cast<const uint32_t *>(xr);
                    a[1] = *reinterpret_cast<const uint32_t *>(xr + 8 * kKS);
                    a[2] = *reinterpret_cast<const uint32_t *>(xr + 8);
                    a[3] = *reinterpret_cast<const uint32_t *>(xr + 8 * kKS + 8);
                    mma_bf16(acc[m], a, bl0, bl1);
                    mma_bf16(acc[m], a, bm0, bm1);
                    mma_bf16(acc[m], a, bh0, bh1);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            if (m < mt_n) {
                const int r0 = m * 16 + g8, c0 = nt + t4 * 2;
                Y[r0 * kPS + c0] = acc[m][0];
                Y[r0 * kPS + c0 + 1] = acc[m][1];
                Y[(r0 + 8) * kPS + c0] = acc[m][2];
                Y[(r0 + 8) * kPS + c0 + 1] = acc[m][3];
            }
        }
    }
    // KK = K K^T and QK = Q K^T (N x N): warp -> (matrix, two 8-column tiles)
    {
        const __nv_bfloat16 *X = (warp >> 2) ? s.Q : s.K;
        float *Y = (warp >> 2) ? s.QK : s.KK;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int nt = ((warp & 3) * 2 + half) * 8;
            if (nt >= n16) continue;
            float acc[4][4];
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[m][e] = 0.f;
#pragma unroll 2
            for (int ks = 0; ks < kD; ks += 16) {
                const __nv_bfloat16 *kr = &s.K[(nt + g8) * kKS + ks + t4 * 2];
                const uint32_t b0 = *reinterpret_cast<const uint32_t *>(kr);
                const uint32_t b1 = *reinterpret_cast<const uint32_t *>(kr + 8);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    if (m < mt_n) {
                        const __nv_bfloat16 *xr = &X[(m * 16 + g8) * kKS + ks + t4 * 2];
                        uint32_t a[4];
                        a[0] = *reinterpret_cast<const uint32_t *>(xr);
                        a[1] = *reinterpret_cast<const uint32_t *>(xr + 8 * kKS);
                        a[2] = *reinterpret_cast<const uint32_t *>(xr + 8);
                        a[3] = *reinterpret_cast<const uint32_t *>(xr + 8 * kKS + 8);
                        mma_bf16(acc[m], a, b0, b1);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (m < mt_n) {
                    const int r0 = m * 16 + g8, c0 = nt + t4 * 2;
                    Y[r0 * kMS + c0] = acc[m][0];
                    Y[r0 * kMS + c0 + 1] = acc[m][1];
                    Y[(r0 + 8) * kMS + c0] = acc[m][2];
                    Y[(r0 + 8) * kMS + c0 + 1] = acc[m][3];
                }
            }
        }
    }
    __syncthreads();

    // the value slice moves into the state slice's space, no longer read
    float *Vf = s.S;
#pragma unroll
    for (int i = 0; i < kNR * 16 / kThreads; ++i) {
        const int e = tid + i * kThreads, j = e >> 4;
        if (j < n) {
            Vf[j * kPS + (e & 15) * 2] = __uint_as_float(vv[i] << 16);
            Vf[j * kPS + (e & 15) * 2 + 1] = __uint_as_float(vv[i] & 0xffff0000u);
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
            unsigned long long m = s.t.anc[j];
            while (m) {
                const int i = __ffsll((long long)m) - 1;
                m &= m - 1;
                sum = fmaf(s.KK[j * kMS + i] * s.t.ginv[i], s.U[i * kPS + c], sum);
            }
            const float bj = s.t.beta[j], gj = s.t.g[j];
            const float B = bj * (Vf[j * kPS + c] - gj * s.P[j * kPS + c]);
            s.U[j * kPS + c] = B - bj * gj * sum;
        }
        __syncthreads();
    }
    // outputs: o_j = g_j (S0 q_j + sum over the path (k_i.q_j / g_i) u_i)
    for (int j = slot; j < n; j += kThreads / 32) {
        float sum = s.Rq[j * kPS + c];
        unsigned long long m = s.t.anc[j] | (1ull << j);
        while (m) {
            const int i = __ffsll((long long)m) - 1;
            m &= m - 1;
            sum = fmaf(s.QK[j * kMS + i] * s.t.ginv[i], s.U[i * kPS + c], sum);
        }
        p.out[((size_t)(row0 + j) * H + h) * kD + vs + c] = s.t.g[j] * sum;
    }
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
    extern __shared__ __align__(16) uint8_t smem_raw[];
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

}  // namespace

namespace w12i {

int launch_gdn(const GdnArgs &a, int mode, void *stream)
{
    if (a.H < 1 || a.n_req < 1) return (int)cudaErrorInvalidValue;
    GdnParams p{};
    p.H = a.H;
    p.n_req = a.n_req;
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
    p.status = a.status;
    // plain launches: with an early start the next layer's CTAs would share
    // SMs with this one's and leave others idle (one CTA per SM is the
    // balanced placement of a 128-CTA layer)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.n_req, a.H, kD / kVS);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    if (mode == kGdnWy) {
        cfg.dynamicSmemBytes = sizeof(WyShared);
        cudaError_t e = cudaFuncSetAttribute(k_gdn_wy, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return (int)e;
        return (int)cudaLaunchKernelEx(&cfg, k_gdn_wy, p);
    }
    cfg.dynamicSmemBytes = sizeof(PathShared);
    const auto kern = mode == kGdnCommit ? k_gdn_path<true> : k_gdn_path<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.dynamicSmemBytes);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace w12i
