// Certified LM head (sm_103a).
//
// SpecPilot explainer, sections 4.1 and 4.3: a cheap pass over the head, a
// per-row Cauchy-Schwarz error bound that discards every token proven unable
// to be the argmax, and exact rescoring of the survivors, so the argmax never
// changes.  The pages' cheap pass reads an INT8 copy of the head; here it is
// the quick pass over the 8-bit view already in every W12 record (w^: view
// byte, low mantissa nibble 0b1000, escapes exact), so nothing extra is
// stored.  For row r and token v the bound is ||h_r|| * ||w_v - w^_v||, with
// slack for the FP32 accumulation and the BF16 output of the cheap pass.
//
//   k_cert_norms    load time: ||w_v - w^_v|| and ||w^_v|| per token (FP64
//                   sums over the decoded record rows, rounded up to FP32)
//   k_cert_lo/surv  64 CTAs per row: ||h_r||, the best lower bound
//                   L = max(s^ - eps) and the survivors s^ + eps >= L (FP32
//                   with directed rounding; an unordered list with room for
//                   the whole vocabulary)
//   k_cert_rescore  64 CTAs per row, one survivor at a time per CTA: exact
//                   FP64 logits from the W12 records (exact decode, escapes
//                   patched), each CTA's best; k_cert_final: one warp per
//                   row, the row's argmax (lowest index on ties)
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>

#include "w12_device.cuh"

using namespace w12d;

namespace {

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// the 16 weights of channel c in the 16-K group kg of a record, exact (nib =
// the record's low-nibble word) or quick (nib = 0x88888888); escaped slots
// of the group take their exact value
__device__ __forceinline__ void decode16(const uint8_t *r, int c, int kg, ChanConst cc, bool quick,
                                         const int32_t *esc_off, const uint32_t *esc, int64_t t, float (&w)[16])
{
    const uint4 v4 = __ldg(reinterpret_cast<const uint4 *>(r + (kg * 128 + c) * 16));
    const uint32_t vw[4] = {v4.x, v4.y, v4.z, v4.w};
    uint32_t nw[4] = {0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u};
    if (!quick) {
        const uint4 n4 = __ldg(reinterpret_cast<const uint4 *>(r + w12i::kViewBytes + ((kg >> 1) * 128 + c) * 16));
        nw[0] = n4.x >> ((kg & 1) * 4), nw[1] = n4.y >> ((kg & 1) * 4);
        nw[2] = n4.z >> ((kg & 1) * 4), nw[3] = n4.w >> ((kg & 1) * 4);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t pp, pq;
        decode_word(vw[i], nw[i], cc, 16u, pp, pq);
        w[2 * i] = bf16f(pp & 0xFFFFu), w[2 * i + 1] = bf16f(pp >> 16);
        w[2 * i + 8] = bf16f(pq & 0xFFFFu), w[2 * i + 9] = bf16f(pq >> 16);
    }
    const int32_t e0 = __ldg(esc_off + t), e1 = __ldg(esc_off + t + 1);
    for (int32_t e = e0; e < e1; ++e) {
        const uint32_t en = __ldg(esc + e);
        const int nl = (en >> 22) & 0x7F, kl = (en >> 16) & 0x3F;
        if (nl != c || (kl >> 4) != kg) continue;
        const float x = bf16f(en & 0xFFFFu);
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j == (kl & 15)) w[j] = x;
    }
}

__global__ void __launch_bounds__(128) k_cert_norms(const uint8_t *__restrict__ rec, const uint8_t *__restrict__ base,
                                                    const int32_t *__restrict__ esc_off,
                                                    const uint32_t *__restrict__ esc, int32_t k_tiles, float *err,
                                                    float *qnorm)
{
    const int nt = blockIdx.x, c = threadIdx.x;
    const ChanConst cc = chan_const(__ldg(base + nt * w12i::kTileN + c));
    double d2 = 0.0, q2 = 0.0;
    for (int kt = 0; kt < k_tiles; ++kt) {
        const int64_t t = (int64_t)nt * k_tiles + kt;
        const uint8_t *r = rec + t * w12i::kRecBytes;
        for (int kg = 0; kg < 4; ++kg) {
            float we[16], wq[16];
            decode16(r, c, kg, cc, false, esc_off, esc, t, we);
            decode16(r, c, kg, cc, true, esc_off, esc, t, wq);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const double d = (double)we[j] - (double)wq[j];
                d2 += d * d;
                q2 += (double)wq[j] * (double)wq[j];
            }
        }
    }
    // round up: the bound must not shrink
    err[nt * w12i::kTileN + c] = __double2float_ru(sqrt(d2) * (1.0 + 1e-12));
    qnorm[nt * w12i::kTileN + c] = __double2float_ru(sqrt(q2) * (1.0 + 1e-12));
}

template <typename T, typename Op>
__device__ T block_reduce(T v, Op op, T *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, off));
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    T r = scratch[0];
    for (int i = 1; i < nw; ++i) r = op(r, scratch[i]);
    return r;
}

// grid R: hn[r] = ||h_r|| rounded up to FP32 (FP64 sum)
__global__ void __launch_bounds__(256) k_cert_hnorm(const uint16_t *__restrict__ h, int64_t K, float *hn)
{
    __shared__ double scratch[32];
    const uint16_t *hr = h + blockIdx.x * K;
    double s = 0.0;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
        const double x = bf16f(__ldg(hr + k));
        s += x * x;
    }
    s = block_reduce(s, [](double a, double b) { return a + b; }, scratch);
    if (threadIdx.x == 0) hn[blockIdx.x] = __double2float_ru(sqrt(s) * (1.0 + 1e-12));
}

// eps of token v, rounded up: the Cauchy-Schwarz bound, the FP32
// accumulation of the cheap pass (tau ||h|| ||w^||) and its BF16 output
// (2^-8 |s^|)
__device__ __forceinline__ float eps_up(float hn, float e, float q, float tau, float sh)
{
    return __fadd_ru(__fmul_ru(hn, __fadd_ru(e, __fmul_ru(tau, q))), __fmul_ru(0x1p-8f, fabsf(sh)));
}

// grid (R, parts): part_lo[r][b] = max over CTA b's tokens of s^ - eps (rounded down)
__global__ void __launch_bounds__(256) k_cert_lo(const uint16_t *__restrict__ shat, const float *__restrict__ hnorm,
                                                 const float *__restrict__ err, const float *__restrict__ qnorm,
                                                 int64_t V, float tau, float *part_lo, int32_t *cnt)
{
    __shared__ float fscratch[32];
    const int r = blockIdx.x, b = blockIdx.y, parts = gridDim.y;
    const float hn = hnorm[r];
    const uint16_t *sr = shat + r * V;
    float lo = -FLT_MAX;
    for (int64_t v = (int64_t)b * blockDim.x + threadIdx.x; v < V; v += (int64_t)parts * blockDim.x) {
        const float sh = bf16f(__ldg(sr + v));
        lo = fmaxf(lo, __fsub_rd(sh, eps_up(hn, __ldg(err + v), __ldg(qnorm + v), tau, sh)));
    }
    lo = block_reduce(lo, [](float x, float y) { return fmaxf(x, y); }, fscratch);
    if (threadIdx.x == 0) {
        part_lo[(int64_t)r * parts + b] = lo;
        if (b == 0) cnt[r] = 0;
    }
}

// grid (R, parts): the survivors s^ + eps >= L (L = the row's best lower bound)
__global__ void __launch_bounds__(256) k_cert_surv(const uint16_t *__restrict__ shat, const float *__restrict__ hnorm,
                                                   const float *__restrict__ err, const float *__restrict__ qnorm,
                                                   int64_t V, float tau, const float *part_lo, int32_t *surv,
                                                   int32_t *cnt)
{
    const int r = blockIdx.x, b = blockIdx.y, parts = gridDim.y;
    const float hn = hnorm[r];
    float L = -FLT_MAX;
    for (int i = 0; i < parts; ++i) L = fmaxf(L, part_lo[(int64_t)r * parts + i]);
    const uint16_t *sr = shat + r * V;
    for (int64_t v = (int64_t)b * blockDim.x + threadIdx.x; v < V; v += (int64_t)parts * blockDim.x) {
        const float sh = bf16f(__ldg(sr + v));
        if (__fadd_ru(sh, eps_up(hn, __ldg(err + v), __ldg(qnorm + v), tau, sh)) >= L) {
            const int i = atomicAdd(cnt + r, 1);
            surv[(int64_t)r * V + i] = (int32_t)v;   // at most V survivors: the list never overflows
        }
    }
}

// grid (R, parts): CTA (r, b) rescores survivors b*8 + warp, b*8 + warp + 8*parts, ...
// of row r and writes its best (logit, token) to part_v/part_i[r][b]
// better (logit, token): larger logit, then the lower token id
__device__ __forceinline__ bool better(double v, int32_t i, double bv, int32_t bi)
{
    return v > bv || (v == bv && i < bi);
}

// grid (R, parts): CTA (r, b) rescores survivors b, b + parts, ... of row r,
// each with all 256 threads (one 16-K group of the channel per thread and
// step), and writes its best (logit, token) to part_v/part_i[r][b]
__global__ void __launch_bounds__(256) k_cert_rescore(const uint8_t *__restrict__ rec, const uint8_t *__restrict__ base,
                                                      const int32_t *__restrict__ esc_off,
                                                      const uint32_t *__restrict__ esc, int32_t k_tiles, int64_t K,
                                                      const uint16_t *__restrict__ h, const int32_t *__restrict__ surv,
                                                      const int32_t *__restrict__ cnt, int64_t cap, double *part_v,
                                                      int32_t *part_i)
{
    __shared__ double red[8];
    const int r = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int parts = gridDim.y, b = blockIdx.y;
    const int64_t n = min((int64_t)cnt[r], cap);
    const uint16_t *hr = h + r * K;
    double bv = -DBL_MAX;
    int32_t bi = INT_MAX;
    for (int64_t i = b; i < n; i += parts) {   // uniform over the CTA
        const int32_t v = surv[(int64_t)r * cap + i];
        const int nt = v >> 7, c = v & 127;
        const ChanConst cc = chan_const(__ldg(base + v));
        double acc = 0.0;
        for (int j = threadIdx.x; j < 4 * k_tiles; j += 256) {
            const int kt = j >> 2, kg = j & 3;
            const int64_t t = (int64_t)nt * k_tiles + kt;
            float w[16];
            decode16(rec + t * w12i::kRecBytes, c, kg, cc, false, esc_off, esc, t, w);
            const uint16_t *hk = hr + kt * 64 + kg * 16;
#pragma unroll
            for (int q = 0; q < 16; ++q) acc += (double)w[q] * (double)bf16f(__ldg(hk + q));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            double tot = red[0];
            for (int w = 1; w < 8; ++w) tot += red[w];
            if (better(tot, v, bv, bi)) bv = tot, bi = v;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        part_v[(int64_t)r * parts + b] = bv;
        part_i[(int64_t)r * parts + b] = bi;
    }
}

// one warp per row: the best of the row's parts (lowest token id on ties)
__global__ void __launch_bounds__(128) k_cert_final(const double *part_v, const int32_t *part_i, int32_t R,
                                                    int32_t parts, int32_t *argmax, float *maxlogit,
                                                    const int32_t *cnt, int32_t *cnt_out)
{
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (r >= R) return;
    double bv = -DBL_MAX;
    int32_t bi = INT_MAX;
    for (int b = lane; b < parts; b += 32) {
        const double v = part_v[(int64_t)r * parts + b];
        const int32_t i = part_i[(int64_t)r * parts + b];
        if (better(v, i, bv, bi)) bv = v, bi = i;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const double ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ov, oi, bv, bi)) bv = ov, bi = oi;
    }
    if (lane == 0) {
        if (cnt_out) cnt_out[r] = cnt[r];
        argmax[r] = (bi == INT_MAX) ? 0 : bi;
        if (maxlogit) maxlogit[r] = (float)bv;
    }
}

}  // namespace

namespace w12i {

int launch_cert_norms(const DevWeight &w, float *err, float *qnorm, void *stream)
{
    k_cert_norms<<<w.n_tiles, 128, 0, static_cast<cudaStream_t>(stream)>>>(w.rec, w.base, w.esc_off, w.esc,
                                                                           w.k_tiles, err, qnorm);
    return (int)cudaGetLastError();
}

int launch_cert_select(const uint16_t *shat, const uint16_t *h, const float *err, const float *qnorm, int32_t R,
                       int64_t V, int64_t K, int32_t *surv, int32_t *cnt, float *part_lo, void *stream)
{
    // FP32 accumulation of K products: |error| <= K * 2^-23 * ||h|| ||w^|| with
    // room to spare (2^-22 per product)
    const float tau = (float)K * 0x1p-22f;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *hn = part_lo + (size_t)R * kCertParts;   // R more floats after the partial bounds
    k_cert_hnorm<<<R, 256, 0, st>>>(h, K, hn);
    if (cudaError_t e = cudaGetLastError()) return (int)e;
    k_cert_lo<<<dim3(R, kCertParts), 256, 0, st>>>(shat, hn, err, qnorm, V, tau, part_lo, cnt);
    if (cudaError_t e = cudaGetLastError()) return (int)e;
    k_cert_surv<<<dim3(R, kCertParts), 256, 0, st>>>(shat, hn, err, qnorm, V, tau, part_lo, surv, cnt);
    return (int)cudaGetLastError();
}

int launch_cert_rescore(const DevWeight &w, const uint16_t *h, int32_t R, const int32_t *surv, const int32_t *cnt,
                        double *part_v, int32_t *part_i, int32_t *argmax, float *maxlogit, int32_t *cnt_out,
                        void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    k_cert_rescore<<<dim3(R, kCertParts), 256, 0, st>>>(w.rec, w.base, w.esc_off, w.esc, w.k_tiles, w.k, h, surv, cnt,
                                                        w.n, part_v, part_i);
    if (cudaError_t e = cudaGetLastError()) return (int)e;
    k_cert_final<<<(R + 3) / 4, 128, 0, st>>>(part_v, part_i, R, kCertParts, argmax, maxlogit, cnt, cnt_out);
    return (int)cudaGetLastError();
}

}  // namespace w12i
