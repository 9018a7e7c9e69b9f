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

// Escape patch: put the exact BF16 value `val` in the upper (upper = true) or
// lower half of a[idx], where idx is known only at run time.  A switch keeps
// a[] in registers at the cost of one jump; a compare-and-select over every
// entry costs a few instructions per entry.
template <int N>
__device__ __forceinline__ void patch_half(uint32_t (&a)[N], int idx, uint32_t val, bool upper)
{
    static_assert(N <= 32, "at most 32 registers");
    switch (idx) {
#define W12_PATCH_CASE(k)                                                                        \
    case k:                                                                                      \
        if constexpr (k < N)                                                                     \
            a[k] = upper ? ((a[k] & 0x0000FFFFu) | (val << 16)) : ((a[k] & 0xFFFF0000u) | val); \
        break;
    W12_PATCH_CASE(0)
    W12_PATCH_CASE(1)
    W12_PATCH_CASE(2)
    W12_PATCH_CASE(3)
    W12_PATCH_CASE(4)
    W12_PATCH_CASE(5)
    W12_PATCH_CASE(6)
    W12_PATCH_CASE(7)
    W12_PATCH_CASE(8)
    W12_PATCH_CASE(9)
    W12_PATCH_CASE(10)
    W12_PATCH_CASE(11)
    W12_PATCH_CASE(12)
    W12_PATCH_CASE(13)
    W12_PATCH_CASE(14)
    W12_PATCH_CASE(15)
    W12_PATCH_CASE(16)
    W12_PATCH_CASE(17)
    W12_PATCH_CASE(18)
    W12_PATCH_CASE(19)
    W12_PATCH_CASE(20)
    W12_PATCH_CASE(21)
    W12_PATCH_CASE(22)
    W12_PATCH_CASE(23)
    W12_PATCH_CASE(24)
    W12_PATCH_CASE(25)
    W12_PATCH_CASE(26)
    W12_PATCH_CASE(27)
    W12_PATCH_CASE(28)
    W12_PATCH_CASE(29)
    W12_PATCH_CASE(30)
    W12_PATCH_CASE(31)
#undef W12_PATCH_CASE
    default: break;
    }
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
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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

// As mbar_try_wait, with a suspend-time hint: a thread whose phase is not yet
// complete sleeps until it completes or about `hint_ns` pass, instead of
// returning after the (short) system default and polling again.  A sleeping
// warp issues nothing, so it leaves the issue slots of its scheduler to the
// warps that have work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase (never suspends the thread, unlike try_wait):
// for a thread that polls several barriers in turn.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
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
// `timeout_ns`, records W12_E_TIMEOUT in *status and returns false.  Also
// returns false once *abort is set.  After one plain poll the thread sleeps
// in try_wait (woken by the phase, or after kWaitSleepNs to look at the clock
// and the abort flag), so a waiting warp does not take issue slots from the
// warps of its scheduler that have work.
constexpr uint32_t kWaitSleepNs = 20000;

// A wait that guards the reuse of a named barrier (an arrival must not come
// twice before the barrier's sync) gets this many wait limits: the other side
// may first sit out one bounded wait of its own, and must get there first.
constexpr uint64_t kReuseWaits = 4;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns, int32_t *status,
                                          volatile int32_t *abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
#pragma unroll 1
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > timeout_ns) {
            atomicCAS(status, 0, static_cast<int32_t>(W12_E_TIMEOUT));
            *abort = 1;
            return false;
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

// ---------------------------------------------------------------------------
// 5th-generation tensor cores (tcgen05) and tensor memory (TMEM)
// ---------------------------------------------------------------------------

// whole warp: allocate `cols` TMEM columns, base address written to smem
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t cols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem desc]; kind::f16 (BF16 in, FP32 accumulate)
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-wide forms: every lane executes the instruction stream, one elected
// lane issues (the warp stays converged around the tensor-core issue).
__device__ __forceinline__ void tc_mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit_elect(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// arrive (once) on an mbarrier when all prior tcgen05 ops of this thread complete
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (rows of 128 bytes), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1u << 16;                          // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset: next 8-row group
    d |= (uint64_t)1u << 46;                          // version
    d |= (uint64_t)2u << 61;                          // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: FP32 D, BF16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4)                   // D format: F32
           | (1u << 7)                 // A format: BF16
           | (1u << 10)                // B format: BF16
           | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 32 lanes x 32 columns of 32 bits: register j of lane i -> TMEM (lane base + i, col + j)
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// argmax combine: (v, i) beats (bv, bi) iff v > bv, or v == bv and i < bi;
// NaN never beats anything, anything non-NaN beats NaN.
__device__ __forceinline__ bool beats(float v, int32_t i, float bv, int32_t bi)
{
    if (v != v) return false;
    if (bv != bv) return true;
    return v > bv || (v == bv && i < bi);
}

}  // namespace w12d
