// W12 decode to BF16 and the load-time bit-exact check (sm_103a).
//
// SpecPilot explainer, section 4.1: the server restores the W12 tensors and
// checks them bit for bit against the checkpoint at load time.  One CTA
// decodes one 128x64 record into shared memory with the same register decode
// the GEMM uses, patches the record's escapes, then either writes the tile
// out or compares it with the source tensor.
#include <cuda_runtime.h>

#include "w12_device.cuh"

using namespace w12d;

namespace {

constexpr int kThreads = 256;
constexpr int kRowHalves = w12i::kTileK + 8;   // padded tile row (uint16 elements)

__global__ void __launch_bounds__(kThreads) k_unpack(const uint8_t *__restrict__ rec, const uint8_t *__restrict__ base,
                                                     const int32_t *__restrict__ esc_off,
                                                     const uint32_t *__restrict__ esc, int32_t k_tiles, int64_t k,
                                                     int64_t tiles, uint16_t *dst, const uint16_t *cmp,
                                                     unsigned long long *mismatch)
{
    __shared__ __align__(16) uint16_t tile[w12i::kTileN * kRowHalves];
    const uint32_t mul16 = 16u + (uint32_t)(k < 0);   // k >= 0: stays 16, opaque to strength reduction
    unsigned long long bad = 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t nt = t / k_tiles, kt = t % k_tiles;
        const uint8_t *r = rec + t * w12i::kRecBytes;
        {
            // thread -> (channel c, 32-K half h): 2 view chunks + 1 nibble chunk
            const int c = threadIdx.x & 127, h = threadIdx.x >> 7;
            const ChanConst cc = chan_const(__ldg(base + nt * w12i::kTileN + c));
            const uint4 nib = __ldg(reinterpret_cast<const uint4 *>(r + w12i::kViewBytes + (h * 128 + c) * 16));
            const uint32_t nw[4] = {nib.x, nib.y, nib.z, nib.w};
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int kg = 2 * h + q;
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(r + (kg * 128 + c) * 16));
                const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t pp, pq;
                    decode_word(vw[i], nw[i] >> (4 * q), cc, mul16, pp, pq);
                    *reinterpret_cast<uint32_t *>(&tile[c * kRowHalves + kg * 16 + 2 * i]) = pp;
                    *reinterpret_cast<uint32_t *>(&tile[c * kRowHalves + kg * 16 + 2 * i + 8]) = pq;
                }
            }
        }
        __syncthreads();
        const int32_t e0 = __ldg(esc_off + t), e1 = __ldg(esc_off + t + 1);
        for (int32_t e = e0 + threadIdx.x; e < e1; e += kThreads) {
            const uint32_t en = __ldg(esc + e);
            tile[((en >> 22) & 0x7F) * kRowHalves + ((en >> 16) & 0x3F)] = static_cast<uint16_t>(en & 0xFFFF);
        }
        __syncthreads();
        // 128 rows x 128 bytes: 8 threads per row, 16 bytes each
        for (int i = threadIdx.x; i < w12i::kTileN * 8; i += kThreads) {
            const int c = i >> 3, part = i & 7;
            const uint4 val = *reinterpret_cast<const uint4 *>(&tile[c * kRowHalves + part * 8]);
            const int64_t off = (nt * w12i::kTileN + c) * k + kt * w12i::kTileK + part * 8;
            if (dst) *reinterpret_cast<uint4 *>(dst + off) = val;
            if (cmp) {
                const uint4 ref = __ldg(reinterpret_cast<const uint4 *>(cmp + off));
                const uint32_t a[4] = {val.x, val.y, val.z, val.w}, b[4] = {ref.x, ref.y, ref.z, ref.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    bad += (unsigned long long)(((a[j] ^ b[j]) & 0xFFFFu) != 0) + ((((a[j] ^ b[j]) >> 16)) != 0);
            }
        }
        __syncthreads();
    }
    if (cmp) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, off);
        if ((threadIdx.x & 31) == 0 && bad) atomicAdd(mismatch, bad);
    }
}

}  // namespace

namespace w12i {

int launch_unpack(const DevWeight &w, uint16_t *dst, const uint16_t *cmp, int64_t *mismatch, int32_t *status,
                  void *stream)
{
    (void)status;
    const int64_t tiles = (int64_t)w.n_tiles * w.k_tiles;
    const int grid = (int)(tiles < 65535 * 8 ? tiles : 65535 * 8);
    k_unpack<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        w.rec, w.base, w.esc_off, w.esc, w.k_tiles, w.k, tiles, dst, cmp,
        reinterpret_cast<unsigned long long *>(mismatch));
    return (int)cudaGetLastError();
}

}  // namespace w12i
