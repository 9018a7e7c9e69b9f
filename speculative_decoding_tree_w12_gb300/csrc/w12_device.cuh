// Device primitives for the W12 kernels (sm_103a): inline-PTX wrappers, bounded
// mbarrier waits and the in-register W12 decode.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "w12_internal.h"

namespace w12d {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// bit manipulation
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// d = a ? b : c, bitwise
__device__ __forceinline__ uint32_t bitmux(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xCA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t mad_u32(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------------------------
// W12 decode
//
// A view word holds the view bytes of weights kk = 2i, 2i+1, 2i+8, 2i+9 of a
// 16-K group (bytes 0..3); the nibble word holds their low mantissa nibbles in
// the low nibble of the same byte positions.  Output: two BF16x2 registers,
// pair P = (2i, 2i+1) and pair Q = (2i+8, 2i+9), low half = lower k.
//
// Per pair: W = [0, v1, 0, v0] (bytes), S = [sign(v1)*0xFF, n1, sign(v0)*0xFF, n0],
//   Z = S ? C1 : C2 (bitwise), out = W * 16 + Z
// with C2 = P0 | P0<<16, P0 = b<<7, and C1 = P1 | P1<<16, P1 = (b<<7) + 0x7800
// with its low nibble set.  For a positive weight: W*16 = o<<7 | mh<<4 and Z =
// b<<7 | ml; for a negative one W*16 carries the sign at bit 11 and Z adds
// 0x7800 more, moving it to bit 15.  No half overflows into the other.
// ---------------------------------------------------------------------------

struct ChanConst {
    uint32_t c1, c2;
};

__device__ __forceinline__ ChanConst chan_const(uint32_t b)
{
    const uint32_t p0 = b << 7;
    const uint32_t p1 = (p0 + 0x7800u) | 0xFu;
    return ChanConst{p1 | (p1 << 16), p0 | (p0 << 16)};
}

__device__ __forceinline__ void decode_word(uint32_t v, uint32_t nib, ChanConst cc, uint32_t mul16, uint32_t &pairP,
                                            uint32_t &pairQ)
{
    const uint32_t wP = prmt(v, 0u, 0x4140u);
    const uint32_t wQ = prmt(v, 0u, 0x4342u);
    const uint32_t sP = prmt(v, nib, 0x9584u);
    const uint32_t sQ = prmt(v, nib, 0xB7A6u);
    pairP = mad_u32(wP, mul16, bitmux(sP, cc.c1, cc.c2));
    pairQ = mad_u32(wQ, mul16, bitmux(sQ, cc.c1, cc.c2));
}

// position of weight kk (0..15) of a 16-K group inside its 16-byte chunk
__device__ __forceinline__ int chunk_pos(int kk) { return ((kk & 7) >> 1) * 4 + (kk >> 3) * 2 + (kk & 1); }

// Reference decode of one weight from its view byte and low nibble.
__device__ __forceinline__ uint16_t decode_one(uint32_t view, uint32_t nib, uint32_t b)
{
    return static_cast<uint16_t>(((view & 0x80u) << 8) | (((view & 0x7Fu) << 4) + (b << 7)) | (nib & 0xFu));
}

// ---------------------------------------------------------------------------
// mbarrier, bulk copies, TMA, programmatic dependent launch
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of parity `parity` to complete.  Gives up after
// `timeout_ns` (checked every 256 polls), records W12_E_TIMEOUT in *status
// and returns false.  Also returns false early once *abort is set.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns, int32_t *status,
                                          volatile int32_t *abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > timeout_ns) {
                atomicCAS(status, 0, static_cast<int32_t>(W12_E_TIMEOUT));
                *abort = 1;
                return false;
            }
        }
    }
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 2-D tiled TMA load (box from the tensor map) at element coordinates (x, y).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int32_t x, int32_t y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ void named_bar(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------------------
// warp-level MMA (legacy path for the memory-bound row counts)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// ldmatrix at [addr + OFF] with OFF a compile-time byte offset
template <int OFF>
__device__ __forceinline__ void ldsm_x4_off(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4+%5];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr), "n"(OFF));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// two floats -> BF16x2 (round to nearest even), `lo` in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// argmax combine: (v, i) beats (bv, bi) iff v > bv, or v == bv and i < bi;
// NaN never beats anything, anything non-NaN beats NaN.
__device__ __forceinline__ bool beats(float v, int32_t i, float bv, int32_t bi)
{
    if (v != v) return false;
    if (bv != bv) return true;
    return v > bv || (v == bv && i < bi);
}

}  // namespace w12d
