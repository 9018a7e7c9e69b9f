// The verify pass's chain of W12 GEMMs in one persistent launch, on the
// 5th-generation tensor cores (tcgen05), sm_103a.
//
// SpecPilot explainer, section 2.1: the verify step is a chain of
// weight-streaming GEMMs whose time is the weight traffic; section 4.1 "W12
// GEMM": 12 KB records (128 x 64 weights) restored in registers and fed to
// the tensor cores, with a fixed-order stream-K split.  Here every GEMM of a
// step -- the linears in layer order, then the LM head with its per-tile
// argmax -- runs inside one grid of one CTA per SM, so the weight stream
// never drains between GEMMs.
//
// The unit of work is a record pair: two consecutive records of one GEMM
// (one at the end of a CTA's share of an odd length).  Per pair:
//
//   producer warp    one thread: a 24 KB bulk copy of the pair (L2
//                    evict-first) into a ring slot; pairs of GEMM j+1 stream
//                    as soon as ring slots free up
//   activation warp  one thread: the pair's two activation blocks (2-D TMA,
//                    128-byte swizzle) into an activation ring slot, once the
//                    MMAs of the slot's previous pair are done.  GEMM j+1's
//                    activations are read once every CTA has finished GEMM j.
//                    A copy instruction occupies its issuing thread for
//                    hundreds of cycles under load, so the two streams get a
//                    thread each
//   decode groups    one to four groups of four warps (one per tensor-memory
//                    lane quarter); group g takes every G-th pair.  Thread =
//                    output channel: per record six 16-byte shared loads,
//                    in-register decode of its 64 weights, escape patch and a
//                    tcgen05.st of 32 columns into the group's 64-column A
//                    buffer; then one non-blocking arrive on the buffer's
//                    named barrier
//   MMA warp         takes the pairs in order: one named-barrier sync, one
//                    tensor-memory fence, the activation wait, then one
//                    elected lane issues four MMAs per record (M = 128
//                    channels, N = rows rounded up to 32, K = 16) into the
//                    tile's FP32 accumulator in tensor memory, and one commit
//                    each that frees the A buffer and the activation slot
//                    (plus one per finished tile)
//   epilogue warps   tcgen05.ld of a finished tile: BF16 rows, or the tile's
//                    (max, index) per row for the LM head; a tile split
//                    between CTAs is published as a partial and finished by
//                    the last contributor in CTA order.  After its last tile
//                    of GEMM j a CTA counts itself in GEMM j's arrival word
//   meta warp        per GEMM, one GEMM ahead, the CTA's escape offsets and
//                    entries, a per-record mask of the 32-channel quarters
//                    holding escapes, and the window bases of its n-tiles,
//                    into one of two shared buffers.
//
// Handing over pairs instead of single records halves the MMA warp's
// barrier syncs, fences and commits per record: measured per role, that
// warp's serial chain of shared-memory and tensor-memory operations (each
// queued behind the decode warps' loads and stores) set the pace, not the
// MMAs or the decode arithmetic.
//
// The dependency between GEMMs is the model's: in a decoder the activations
// of GEMM j+1 are computed from GEMM j's outputs, so they are read only
// after all of GEMM j is written.  The weights depend on nothing; the copy,
// decode and escape work of GEMM j+1 overlap the end of GEMM j.
//
// Every wait is bounded.  A wait that runs out records W12_E_TIMEOUT and
// raises the CTA's abort flag and the grid's abort word; the named-barrier
// hand-off between decode warps and the MMA warp never hangs (decode warps
// arrive once for every pair they own, the MMA warp syncs and commits once
// for every pair, aborted or not).  Issued copies and MMAs are waited for
// and tensor memory is released before a CTA exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "w12_device.cuh"

using namespace w12d;

namespace {

constexpr int kProducerWarp = 0;   // also allocates tensor memory
constexpr int kGroupWarp0 = 1;     // decode group g = warps 1 + 4g .. 4 + 4g
constexpr int kMaxGroups = 4;
constexpr int kMmaWarp = 1 + 4 * kMaxGroups;    // warp 17
constexpr int kEpiWarp0 = kMmaWarp + 1;          // warps 18..21
constexpr int kMetaWarp = kEpiWarp0 + 4;         // warp 22
constexpr int kXWarp = kMetaWarp + 1;            // warp 23
constexpr int kThreads = (kXWarp + 1) * 32;      // 24 warps
constexpr int kRecPair = 2 * w12i::kRecBytes;
constexpr int kACols = 64;         // tensor-memory columns of one A buffer (a record pair)
constexpr uint32_t kTmemCols = 512;
constexpr int kBarA0 = 1;          // named barrier of A buffer (g, a): kBarA0 + g * a_bufs + a (<= 15)
constexpr int kMaxJobs = 144;      // GEMMs per launch (the parameter block stays under 32 KB)

struct Job {
    const uint8_t *rec;
    const uint8_t *base;
    const int32_t *esc_off;
    const uint32_t *esc;
    uint16_t *y;          // linear: [R][ldy]
    float *s1_val;        // head: [R][n_tiles]
    int32_t *s1_idx;
    int64_t ldy;
    int32_t n_tiles, k_tiles, mode, ctas;
};

struct ChainParams {
    CUtensorMap xmap[kMaxJobs];   // activations of each GEMM: box 64 K x nr rows, 128-byte swizzle
    Job job[kMaxJobs];
    float *partial;               // [ctas][2][nr][128]
    int32_t *counters;            // split-tile arrival counters, [max n_tiles]
    int32_t *status;
    uint32_t *grid_bar;           // [n_jobs] arrivals of CTAs that finished each GEMM (null: one GEMM)
    int32_t *grid_abort;          // raised by a CTA that gave up waiting
    uint64_t *trace;              // optional: [n_jobs + 1][trace_stride] global-timer stamps (GEMM ends, CTA start)
    uint64_t timeout_ns;
    int32_t trace_stride;
    int32_t n_jobs, R, nr;
    int32_t groups;               // decode groups (1..4)
    int32_t a_bufs;               // A buffers (record pairs) per group
    int32_t d_bufs;               // tile accumulators (1 or 2)
    int32_t stages;               // record-pair slots
    int32_t x_slots;              // activation pair slots
    int32_t max_recs, esc_cap, base_tiles;
    int32_t debug_flags;
};

// Shared-memory plan.  q = A buffers over all groups; sx = activation pair slots.
struct Plan {
    int rec, x, bars, misc, meta, red, total;
    int meta_bytes, m_escoff, m_esc, m_emask, m_base;
};

__host__ __device__ inline Plan plan(int stages, int q, int sx, int nr, int max_recs, int esc_cap, int base_tiles)
{
    Plan p;
    int o = 0;
    p.rec = o;
    o += stages * kRecPair;                   // 24 KB per slot keeps the 1024-byte alignment
    p.x = o;
    o += sx * 2 * nr * 128;
    p.bars = o;
    // rec full/empty, A done, x full/done, acc full/empty, epilogue, meta full/empty
    o += 8 * (2 * stages + q + 2 * sx + 2 * 2 + 1 + 2 * 2);
    p.misc = o;
    o += 64;
    int m = 0;
    p.m_escoff = m;
    m += ((max_recs + 1) * 4 + 15) / 16 * 16;
    p.m_esc = m;
    m += esc_cap * 4;
    p.m_emask = m;
    m += (max_recs + 15) / 16 * 16;
    p.m_base = m;
    m += base_tiles * w12i::kTileN;
    p.meta_bytes = m;
    p.meta = o;
    o += 2 * m;
    p.red = o;
    o += 4 * nr * 8;      // head epilogue: per warp, per row (max, index)
    p.total = o + 1024;   // slack for the 1024-byte alignment
    return p;
}

// A CTA's share of one GEMM: records [rb, rb + nrec) in (n-tile, k-tile) order.
struct Span {
    int64_t rb;
    int nrec;
    int kt0;           // k-tile of record rb
    int64_t nt_first;  // n-tile of record rb
};

__device__ __forceinline__ Span span_of(const Job &jb, int cta)
{
    Span s;
    const int64_t T = (int64_t)jb.n_tiles * jb.k_tiles;
    if (cta < jb.ctas) {
        s.rb = (int64_t)cta * T / jb.ctas;
        s.nrec = (int)((int64_t)(cta + 1) * T / jb.ctas - s.rb);
    } else {
        s.rb = 0;
        s.nrec = 0;
    }
    s.nt_first = s.rb / jb.k_tiles;
    s.kt0 = (int)(s.rb - s.nt_first * jb.k_tiles);
    return s;
}

__device__ __forceinline__ int cta_of_record(int64_t r, int G, int64_t T) { return (int)(((r + 1) * G - 1) / T); }
__device__ __forceinline__ int64_t first_record(int c, int G, int64_t T) { return (int64_t)c * T / G; }

__device__ __forceinline__ bool elect_one()
{
    uint32_t e;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
    return e != 0;
}

__device__ __forceinline__ void named_arrive(int id, int threads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Per-GEMM meta info kept beside the two shared meta buffers.
struct MetaInfo {
    int32_t e_lo;          // first escape entry of the CTA's records
    int32_t esc_cached;    // entries copied into the shared buffer
    int32_t base_cached;   // window bases of the CTA's n-tiles copied
    int32_t pad;
};

// QV: the quick pass (only the 8 KB view plane of each record is copied; the
// low mantissa bits of in-window weights are the midpoint 0b1000)
template <bool QV>
__global__ void __launch_bounds__(kThreads, 1) k_w12_chain(const __grid_constant__ ChainParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages, NR = p.nr, GR = p.groups, NAG = p.a_bufs, DB = p.d_bufs, SX = p.x_slots;
    const int Q = GR * NAG;
    const int J = p.n_jobs;
    const Plan pl = plan(S, Q, SX, NR, p.max_recs, p.esc_cap, p.base_tiles);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;

    const uint32_t rec_s = smem_u32(smem + pl.rec), x_s = smem_u32(smem + pl.x);
    const uint32_t xb = (uint32_t)NR * 128;
    const uint32_t bar0 = smem_u32(smem + pl.bars);
    const uint32_t bar_rfull = bar0, bar_rempty = bar0 + 8 * S;
    const uint32_t bar_done = bar_rempty + 8 * S;
    const uint32_t bar_xfull = bar_done + 8 * Q, bar_xdone = bar_xfull + 8 * SX;
    const uint32_t bar_accfull = bar_xdone + 8 * SX, bar_accempty = bar_accfull + 16;
    const uint32_t bar_epi = bar_accempty + 16;
    const uint32_t bar_mfull = bar_epi + 8, bar_mempty = bar_mfull + 16;
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + pl.misc);
    int32_t *last_flag = reinterpret_cast<int32_t *>(smem + pl.misc + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + pl.misc + 8);
    MetaInfo *minfo = reinterpret_cast<MetaInfo *>(smem + pl.misc + 16);   // [2]
    auto meta_escoff = [&](int b) { return reinterpret_cast<int32_t *>(smem + pl.meta + b * pl.meta_bytes + pl.m_escoff); };
    auto meta_esc = [&](int b) { return reinterpret_cast<uint32_t *>(smem + pl.meta + b * pl.meta_bytes + pl.m_esc); };
    auto meta_emask = [&](int b) { return smem + pl.meta + b * pl.meta_bytes + pl.m_emask; };
    auto meta_base = [&](int b) { return smem + pl.meta + b * pl.meta_bytes + pl.m_base; };

    const bool drop_first = (p.debug_flags & 1) && cta == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_rfull + 8 * s, 1);    // producer's expect_tx arrival + the copy's bytes
            mbar_init(bar_rempty + 8 * s, 4);   // the group's four warps have read the pair
        }
        for (int s = 0; s < Q; ++s) mbar_init(bar_done + 8 * s, 1);   // one commit per pair
        for (int s = 0; s < SX; ++s) {
            mbar_init(bar_xfull + 8 * s, 1);    // producer's expect_tx arrival + the blocks' bytes
            mbar_init(bar_xdone + 8 * s, 1);    // one commit per pair: its MMAs are done
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(bar_accfull + 8 * d, 1);    // commit after a tile's last MMA
            mbar_init(bar_accempty + 8 * d, 4);   // the four epilogue warps have read the accumulator
        }
        mbar_init(bar_epi, 4);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_mfull + 8 * b, 1);         // the meta warp filled the buffer
            mbar_init(bar_mempty + 8 * b, 4 * GR);   // every decode warp left the buffer's GEMM
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarp) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    const uint32_t d_col0 = (uint32_t)(Q * kACols);
    auto a_col = [&](int g, int a) { return (uint32_t)((g * NAG + a) * kACols); };
    auto d_col = [&](int d) { return d_col0 + (uint32_t)(d * NR); };

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- record producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // record stream: GEMM jr, its pair mr; global pair count qr -> slot sl, fill round ru
            int jr = 0, mr = 0;
            Span sr = span_of(p.job[0], cta);
            int64_t qr = 0;
            int sl = 0;
            uint32_t ru = 0;
            auto rec_skip = [&]() {
                while (jr < J && 2 * mr >= sr.nrec) {
                    ++jr;
                    mr = 0;
                    if (jr < J) sr = span_of(p.job[jr], cta);
                }
            };
            auto issue_r = [&]() {
                const Job &jb = p.job[jr];
                const int n = min(2, sr.nrec - 2 * mr);
                const uint8_t *src = jb.rec + (sr.rb + 2 * mr) * (int64_t)w12i::kRecBytes;
                const uint32_t fb = bar_rfull + 8 * sl;
                if constexpr (QV) {
                    // the view plane of each record: its first 8 KB, at the record's place in the slot
                    mbar_expect_tx(fb, (uint32_t)(n * w12i::kViewBytes));
                    if (!(drop_first && qr == 0))
                        for (int r = 0; r < n; ++r)
                            bulk_g2s(rec_s + sl * kRecPair + r * w12i::kRecBytes, src + r * w12i::kRecBytes,
                                     (uint32_t)w12i::kViewBytes, fb, pol);
                } else {
                    mbar_expect_tx(fb, (uint32_t)(n * w12i::kRecBytes));
                    if (!(drop_first && qr == 0))
                        bulk_g2s(rec_s + sl * kRecPair, src, (uint32_t)(n * w12i::kRecBytes), fb, pol);
                }
                ++mr;
                ++qr;
                if (++sl == S) sl = 0, ++ru;
            };
            if (p.trace) p.trace[(int64_t)J * p.trace_stride + cta] = globaltimer();
            // weights do not depend on earlier kernels: the record stream runs
            // without the programmatic-dependency wait
            rec_skip();
            bool stalled = false;
            uint64_t t_idle = 0;
            while (jr < J && !stalled) {
                bool moved = false;
                // slot sl's previous pair (qr - S) has been read by its decode group
                if (qr < S || mbar_try_wait(bar_rempty + 8 * sl, (ru - 1u) & 1u)) {
                    issue_r();
                    rec_skip();
                    moved = true;
                }
                if (moved) {
                    t_idle = 0;
                } else if (*abort_flag || (p.grid_abort && *(volatile int32_t *)p.grid_abort)) {
                    *abort_flag = 1;
                    stalled = true;
                } else if (t_idle == 0) {
                    t_idle = globaltimer();
                } else if (globaltimer() - t_idle > p.timeout_ns) {
                    atomicCAS(p.status, 0, static_cast<int32_t>(W12_E_TIMEOUT));
                    *abort_flag = 1;
                    stalled = true;
                }
            }
            if (*abort_flag) {
                if (p.grid_abort) *(volatile int32_t *)p.grid_abort = 1;
                // leave no copy in flight: the last use of every slot that was filled
                int32_t no_abort = 0;
                for (int64_t q = (qr > S ? qr - S : 0); q < qr; ++q) {
                    if (drop_first && q == 0) continue;
                    mbar_wait(bar_rfull + 8 * (int)(q % S), (uint32_t)((q / S) & 1), p.timeout_ns, p.status,
                              &no_abort);
                }
            }
        }
    } else if (warp < kMmaWarp) {
        // --------------------------------------------------------------- decode
        const int g = (warp - kGroupWarp0) >> 2;
        const int quarter = warp & 3;                // tensor-memory lanes this warp may touch
        const int c = quarter * 32 + lane;           // output channel of this thread
        if (g < GR) {
            // cursor over the CTA's pair sequence (all GEMMs concatenated):
            // GEMM j starts at global pair pstart
            int j = 0;
            Span sp = span_of(p.job[0], cta);
            int pstart = 0;
            int npj = (sp.nrec + 1) >> 1;
            int entered = -1;             // last GEMM whose meta buffer this warp waited for
            int cur_pair = 0;             // ring slot s (fill round parity sph) of global pair cur_pair
            int s = 0;
            uint32_t sph = 0;
            int ab = 0, iq = g;           // A buffer, A-buffer done slot (parity iph) of pair q
            uint32_t iph = 0;
            int job_cur = -1;             // GEMM of the tile cursor
            int nt = 0, nt_cur = -1;      // n-tile, relative to the CTA's first n-tile of the GEMM
            int kt = 0, KT = 1;
            ChanConst cc{0, 0};
            auto enter = [&](int jj) {
                mbar_wait(bar_mfull + 8 * (jj & 1), (uint32_t)((jj >> 1) & 1), p.timeout_ns, p.status, abort_flag);
                entered = jj;
            };
            auto leave = [&](int jj) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_mempty + 8 * (jj & 1));
            };
            int n_done = 0;
            for (int q = g;; q += GR) {
                while (j < J && q >= pstart + npj) {
                    // this warp is done with GEMM j's meta buffer (waiting for it
                    // first keeps the buffer's phases in order)
                    if (entered < j) enter(j);
                    leave(j);
                    pstart += npj;
                    ++j;
                    if (j < J) {
                        sp = span_of(p.job[j], cta);
                        npj = (sp.nrec + 1) >> 1;
                    }
                }
                if (j >= J) break;
                if (entered < j) enter(j);
                const int r0 = 2 * (q - pstart);               // first record of the pair in GEMM j
                const int n = min(2, sp.nrec - r0);
                const int mb = j & 1;
                if (j != job_cur) {
                    job_cur = j;
                    KT = p.job[j].k_tiles;
                    // record r0 of the share: kt0 + r0 k-tiles past the first n-tile
                    const int t = sp.kt0 + r0;
                    nt = t / KT;
                    kt = t - nt * KT;
                    nt_cur = -1;
                } else {
                    kt += 2 * GR;
                    while (kt >= KT) kt -= KT, ++nt;
                }
                while (cur_pair < q) {
                    ++cur_pair;
                    if (++s == S) s = 0, sph ^= 1u;
                }
                if (n_done > 0) {
                    if (++ab == NAG) ab = 0;
                    iq += GR;
                    if (iq >= Q) iq -= Q, iph ^= 1u;
                }
                ++n_done;
                // A buffer ab last held pair q - Q: its MMAs must be done before
                // the buffer is written.  The wait sits after the first record's
                // loads and decode, so that those overlap the MMAs of pair q - Q.
                // The MMA warp commits every pair, so the wait ends even after an
                // abort; it is never skipped (the buffer's named barrier is
                // reused only after its sync: a second arrival before that sync
                // would leave the MMA warp waiting at the barrier for good).  The
                // MMA warp may itself sit in one bounded wait before it commits,
                // so this wait is allowed several of those limits.
                bool buf_free = q < Q;
                auto wait_buffer = [&]() {
                    if (buf_free) return true;
                    buf_free = true;
                    int32_t no_abort = 0;
                    return mbar_wait(bar_done + 8 * iq, iph ^ 1u, kReuseWaits * p.timeout_ns, p.status, &no_abort);
                };
                bool ok = !*abort_flag;
                if (ok) ok = mbar_wait(bar_rfull + 8 * s, sph, p.timeout_ns, p.status, abort_flag);
                ok = __all_sync(0xffffffffu, ok && !*abort_flag);
                if (ok) {
                    const MetaInfo mi = minfo[mb];
                    const uint8_t *emask = meta_emask(mb);
                    int ntr = nt;
                    int ktr = kt;
#pragma unroll 1
                    for (int u = 0; u < n; ++u) {
                        if (u == 1 && ++ktr == KT) ktr = 0, ++ntr;
                        const int r = r0 + u;
                        if (ntr != nt_cur) {
                            nt_cur = ntr;
                            const uint32_t b = mi.base_cached
                                                   ? meta_base(mb)[ntr * w12i::kTileN + c]
                                                   : __ldg(p.job[j].base + (sp.nt_first + ntr) * w12i::kTileN + c);
                            cc = chan_const(b);
                        }
                        const uint8_t *rb = smem + pl.rec + s * kRecPair + u * w12i::kRecBytes;
                        uint4 v[4], nb[2];
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) v[k4] = *reinterpret_cast<const uint4 *>(rb + (k4 * 128 + c) * 16);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            nb[h] = QV ? make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u)
                                       : *reinterpret_cast<const uint4 *>(rb + w12i::kViewBytes + (h * 128 + c) * 16);
                        if (u == n - 1) {
                            // the whole pair has been read: hand the slot back
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar_rempty + 8 * s);
                        }
                        uint32_t a[32];
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const uint32_t vw[4] = {v[k4].x, v[k4].y, v[k4].z, v[k4].w};
                            const uint4 n4 = nb[k4 >> 1];
                            const uint32_t nw[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
                            for (int w = 0; w < 4; ++w)
                                decode_word(vw[w], nw[w] >> ((k4 & 1) * 4), cc, 16u, a[8 * k4 + w], a[8 * k4 + 4 + w]);
                        }
                        if ((emask[r] >> quarter) & 1u) {
                            // escaped slots of this channel: the exact value replaces the filler
                            const int32_t *eo = meta_escoff(mb);
                            const uint32_t *es = meta_esc(mb);
                            const int32_t e0 = eo[r] - mi.e_lo, e1 = eo[r + 1] - mi.e_lo;
                            for (int e = e0; e < e1; ++e) {
                                const uint32_t en = mi.esc_cached ? es[e] : __ldg(p.job[j].esc + mi.e_lo + e);
                                const int nl = (en >> 22) & 0x7F;
                                if ((nl >> 5) != quarter) continue;   // warp-uniform skip
                                const int kl = (en >> 16) & 0x3F;
                                if (nl == c) patch_half(a, kl >> 1, en & 0xFFFFu, kl & 1);
                            }
                        }
                        if (u == 0) wait_buffer();
                        tmem_st_x32(tmem + ((uint32_t)(quarter * 32) << 16) + a_col(g, ab) + (uint32_t)(u * 32), a);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                }
                wait_buffer();
                __syncwarp();
                named_arrive(kBarA0 + g * NAG + ab, 160);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA
        const uint32_t idesc = idesc_bf16_f32(128, NR);
        int tcount = 0, dcur = 0;
        // group g, A buffer ab and A-buffer done slot aq of the next pair;
        // activation pair slot xsl (fill parity xph) of the next pair
        int g = 0, ab = 0, aq = 0, xsl = 0;
        uint32_t xph = 0;
        int64_t q_glob = 0;
        for (int j = 0; j < J; ++j) {
            const Span sp = span_of(p.job[j], cta);
            const int KT = p.job[j].k_tiles;
            int kt = sp.kt0;
            for (int r0 = 0; r0 < sp.nrec; r0 += 2) {
                const int n = min(2, sp.nrec - r0);
                named_bar(kBarA0 + g * NAG + ab, 160);
                // the whole warp runs this part (it stays converged); one elected
                // lane issues the tensor-core instructions
                tc_fence_after();
                bool go = !*abort_flag;
                if (go) go = mbar_wait(bar_xfull + 8 * xsl, xph, p.timeout_ns, p.status, abort_flag);
                go = __all_sync(0xffffffffu, go);
                const uint32_t a_t = tmem + a_col(g, ab);
                const uint32_t xa = x_s + (uint32_t)(xsl * 2) * xb;
#pragma unroll 1
                for (int u = 0; u < n; ++u) {
                    const int r = r0 + u;
                    const bool first = (r == 0) || kt == 0;
                    const bool last = (r == sp.nrec - 1) || kt == KT - 1;
                    if (first) {
                        dcur = tcount % DB;
                        if (go && tcount >= DB)
                            go = mbar_wait(bar_accempty + 8 * dcur, ((tcount / DB) - 1) & 1, p.timeout_ns, p.status,
                                           abort_flag);
                        go = __all_sync(0xffffffffu, go);
                        tc_fence_after();
                    }
                    if (elect_one()) {
                        if (go) {
                            const uint32_t d_t = tmem + d_col(dcur), au = a_t + (uint32_t)(u * 32);
                            const uint64_t bd = smem_desc_sw128(xa + (uint32_t)u * xb);
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                tc_mma_ts(d_t, au + ks * 8, bd + (uint64_t)(ks * 2), idesc,
                                          (first && ks == 0) ? 0u : 1u);
                            if (last) tc_commit(bar_accfull + 8 * dcur);
                        }
                        if (u == n - 1) {
                            tc_commit(bar_done + 8 * aq);      // always: frees the A buffer
                            tc_commit(bar_xdone + 8 * xsl);    // always: frees the activation slot
                        }
                    }
                    __syncwarp();
                    if (last) ++tcount;
                    if (++kt == KT) kt = 0;
                }
                if (++g == GR) {
                    g = 0;
                    if (++ab == NAG) ab = 0;
                }
                if (++aq == Q) aq = 0;
                if (++xsl == SX) xsl = 0, xph ^= 1u;
                ++q_glob;
            }
        }
        // tensor memory is released only after every issued MMA finished
        if (q_glob > 0) {
            int32_t no_abort = 0;
            mbar_wait(bar_done + 8 * (int)((q_glob - 1) % Q), (uint32_t)(((q_glob - 1) / Q) & 1), p.timeout_ns,
                      p.status, &no_abort);
        }
    } else if (warp < kMetaWarp) {
        // ------------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int c = quarter * 32 + lane;
        const int ew = warp - kEpiWarp0;
        const int etid = ew * 32 + lane;   // 0..127
        const int rows = p.R;
        float *red_v = reinterpret_cast<float *>(smem + pl.red);
        int32_t *red_i = reinterpret_cast<int32_t *>(smem + pl.red + 4 * NR * 4);
        uint32_t eph = 0;
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_epi);
            const bool ok = mbar_wait(bar_epi, eph, p.timeout_ns, p.status, abort_flag);
            eph ^= 1u;
            return __all_sync(0xffffffffu, ok);
        };
        int tcount = 0;
        bool alive = true;
        for (int j = 0; j < J && alive; ++j) {
            const Job &jb = p.job[j];
            const Span sp = span_of(jb, cta);
            const int G = jb.ctas, KT = jb.k_tiles;
            const int64_t T = (int64_t)jb.n_tiles * KT;
            const int64_t rec_end = sp.rb + sp.nrec;
            const int64_t nt_last = sp.nrec ? (rec_end - 1) / KT : sp.nt_first - 1;
            // write (or reduce, for the LM head) 32 rows r0..r0+31 of this channel
            auto emit_rows = [&](int64_t nt, int r0, const float (&v)[32]) {
                if (jb.mode == w12i::kModeLinear) {
                    uint16_t *yc = jb.y + nt * w12i::kTileN + c;
#pragma unroll
                    for (int u = 0; u < 32; ++u)
                        if (r0 + u < rows) yc[(int64_t)(r0 + u) * jb.ldy] = (uint16_t)(pack_bf16x2(v[u], 0.f) & 0xFFFFu);
                } else {
                    // (max, lowest index) over the warp's 32 channels for 32 rows at
                    // once: at each of five steps a lane keeps half of its rows,
                    // trades the other half with its partner and combines; lane l
                    // ends with row r0 + l
                    float bv[32];
                    int32_t bi[32];
#pragma unroll
                    for (int u = 0; u < 32; ++u) bv[u] = v[u], bi[u] = c;
#pragma unroll
                    for (int h = 16; h > 0; h >>= 1) {
                        const bool upper = (lane & h) != 0;
#pragma unroll
                        for (int k = 0; k < h; ++k) {
                            const float keep_v = upper ? bv[h + k] : bv[k], send_v = upper ? bv[k] : bv[h + k];
                            const int32_t keep_i = upper ? bi[h + k] : bi[k], send_i = upper ? bi[k] : bi[h + k];
                            const float ov = __shfl_xor_sync(0xffffffffu, send_v, h);
                            const int32_t oi = __shfl_xor_sync(0xffffffffu, send_i, h);
                            const bool take = beats(ov, oi, keep_v, keep_i);
                            bv[k] = take ? ov : keep_v;
                            bi[k] = take ? oi : keep_i;
                        }
                    }
                    if (r0 + lane < rows) red_v[ew * NR + r0 + lane] = bv[0], red_i[ew * NR + r0 + lane] = bi[0];
                }
            };
            // LM head: combine the four warps' per-row winners into the tile's (max, index)
            auto head_finish = [&](int64_t nt) -> bool {
                if (jb.mode != w12i::kModeHead) return true;
                if (!epi_sync()) return false;
                for (int r = etid; r < rows; r += 128) {
                    float bv = red_v[r];
                    int32_t bi = red_i[r];
                    for (int w = 1; w < 4; ++w)
                        if (beats(red_v[w * NR + r], red_i[w * NR + r], bv, bi))
                            bv = red_v[w * NR + r], bi = red_i[w * NR + r];
                    jb.s1_val[(int64_t)r * jb.n_tiles + nt] = bv;
                    jb.s1_idx[(int64_t)r * jb.n_tiles + nt] = (int32_t)(nt * w12i::kTileN + bi);
                }
                return epi_sync();
            };
            for (int64_t nt = sp.nt_first; nt <= nt_last; ++nt) {
                const int64_t t0 = nt * KT, t1 = t0 + KT;
                const int dsel = tcount % DB;
                const bool ok =
                    mbar_wait(bar_accfull + 8 * dsel, (tcount / DB) & 1, p.timeout_ns, p.status, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                const bool owned = sp.rb <= t0 && rec_end >= t1;
                const int slot = (nt == sp.nt_first) ? 0 : 1;
                float *mine = p.partial + ((int64_t)(cta * 2 + slot) * NR) * w12i::kTileN;
                const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
                for (int r0 = 0; r0 < NR; r0 += 32) {
                    uint32_t raw[32];
                    tmem_ld_x32(lane_base + d_col(dsel) + r0, raw);
                    tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int u = 0; u < 32; ++u) v[u] = __uint_as_float(raw[u]);
                    if (owned) {
                        emit_rows(nt, r0, v);
                    } else {
#pragma unroll
                        for (int u = 0; u < 32; ++u)
                            if (r0 + u < rows) __stcg(mine + (r0 + u) * w12i::kTileN + c, v[u]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_accempty + 8 * dsel);
                ++tcount;
                if (owned) {
                    if (!head_finish(nt)) {
                        alive = false;
                        break;
                    }
                    continue;
                }
                // split tile: publish, count arrivals, the last contributor finishes it
                __threadfence();
                if (!epi_sync()) {
                    alive = false;
                    break;
                }
                const int c_first = cta_of_record(t0, G, T), c_last = cta_of_record(t1 - 1, G, T);
                if (etid == 0) *last_flag = (atomicAdd(p.counters + nt, 1) == c_last - c_first);
                if (!epi_sync()) {
                    alive = false;
                    break;
                }
                if (*last_flag == 0) continue;
                __threadfence();
                for (int r0 = 0; r0 < NR; r0 += 32) {
                    float v[32];
#pragma unroll
                    for (int u = 0; u < 32; ++u) v[u] = 0.f;
                    for (int cc2 = c_first; cc2 <= c_last; ++cc2) {
                        const int sl = (nt == first_record(cc2, G, T) / KT) ? 0 : 1;
                        const float *src = p.partial + ((int64_t)(cc2 * 2 + sl) * NR) * w12i::kTileN;
#pragma unroll
                        for (int u = 0; u < 32; ++u)
                            if (r0 + u < rows) v[u] += __ldcg(src + (r0 + u) * w12i::kTileN + c);
                    }
                    emit_rows(nt, r0, v);
                }
                if (etid == 0) p.counters[nt] = 0;   // ready for the next GEMM using this tile
                if (!head_finish(nt)) {
                    alive = false;
                    break;
                }
            }
            if (!alive) break;
            // every output of this CTA for GEMM j is written: count the CTA in
            // GEMM j's arrival word (the next GEMM's activations wait for all)
            if (p.grid_bar) {
                if (!epi_sync()) {
                    alive = false;
                    break;
                }
                if (etid == 0) {
                    __threadfence();
                    atomicAdd(p.grid_bar + j, 1u);
                }
            }
            if (p.trace && etid == 0) p.trace[(int64_t)j * p.trace_stride + cta] = globaltimer();
        }
        if (!alive && p.grid_abort && etid == 0) *(volatile int32_t *)p.grid_abort = 1;
    } else if (warp == kMetaWarp) {
        // ------------------------------------------------------------------ meta
        for (int j = 0; j < J; ++j) {
            const int b = j & 1;
            if (j >= 2) {
                // every decode warp has left GEMM j - 2, the buffer's previous user
                if (!mbar_wait(bar_mempty + 8 * b, (uint32_t)(((j >> 1) - 1) & 1), p.timeout_ns, p.status,
                               abort_flag))
                    break;
            }
            const Job &jb = p.job[j];
            const Span sp = span_of(jb, cta);
            int32_t *eo = meta_escoff(b);
            uint32_t *es = meta_esc(b);
            uint8_t *em = meta_emask(b);
            uint8_t *bs = meta_base(b);
            if (sp.nrec > 0) {
                for (int i = lane; i <= sp.nrec; i += 32) eo[i] = __ldg(jb.esc_off + sp.rb + i);
                __syncwarp();
                const int32_t e_lo = eo[0], n_e = eo[sp.nrec] - e_lo;
                const bool esc_cached = n_e <= p.esc_cap;
                if (esc_cached)
                    for (int i = lane; i < n_e; i += 32) es[i] = __ldg(jb.esc + e_lo + i);
                __syncwarp();
                // per record, a bit for every 32-channel quarter that holds an escape
                for (int i = lane; i < sp.nrec; i += 32) {
                    uint32_t msk = 0;
                    for (int e = eo[i]; e < eo[i + 1]; ++e) {
                        const uint32_t en = esc_cached ? es[e - e_lo] : __ldg(jb.esc + e);
                        msk |= 1u << ((en >> 27) & 3u);
                    }
                    em[i] = (uint8_t)msk;
                }
                const int64_t nt_last = (sp.rb + sp.nrec - 1) / jb.k_tiles;
                const int span_tiles = (int)(nt_last - sp.nt_first + 1);
                const bool base_cached = span_tiles <= p.base_tiles;
                if (base_cached)
                    for (int i = lane; i < span_tiles * w12i::kTileN; i += 32)
                        bs[i] = __ldg(jb.base + sp.nt_first * w12i::kTileN + i);
                if (lane == 0) {
                    minfo[b].e_lo = e_lo;
                    minfo[b].esc_cached = esc_cached ? 1 : 0;
                    minfo[b].base_cached = base_cached ? 1 : 0;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_mfull + 8 * b);
        }
    } else if (lane == 0) {
        // ----------------------------------------------------------- activations
        // pair q of the CTA's sequence into slot q % SX once the MMAs of pair
        // q - SX are done (the MMA warp commits every pair, aborted or not)
        const uint32_t G_all = gridDim.x;
        int64_t qx = 0;
        int xsl = 0;
        uint32_t xu = 0;
        bool ok = true;
        prefetch_tmap(&p.xmap[0]);
        // the first GEMM's activations may come from the previous kernel
        pdl_wait();
        for (int j = 0; j < J && ok; ++j) {
            const Job &jb = p.job[j];
            const Span sp = span_of(jb, cta);
            if (sp.nrec == 0) continue;
            if (j + 1 < J) prefetch_tmap(&p.xmap[j + 1]);
            if (j > 0) {
                // GEMM j reads activations computed from GEMM j - 1: wait until
                // every CTA has finished that GEMM
                uint64_t t0 = 0;
                for (uint32_t it = 0;; ++it) {
                    if (ld_acquire_u32(p.grid_bar + (j - 1)) >= G_all) break;
                    if ((it & 31u) == 31u) {
                        if (*abort_flag || (p.grid_abort && *(volatile int32_t *)p.grid_abort)) {
                            ok = false;
                            break;
                        }
                        const uint64_t now = globaltimer();
                        if (t0 == 0) {
                            t0 = now;
                        } else if (now - t0 > p.timeout_ns) {
                            atomicCAS(p.status, 0, static_cast<int32_t>(W12_E_TIMEOUT));
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok) break;
                fence_proxy_async();
            }
            const int KT = jb.k_tiles;
            int kx = sp.kt0;
            for (int m = 0; 2 * m < sp.nrec; ++m) {
                if (qx >= SX && !mbar_wait(bar_xdone + 8 * xsl, (xu - 1u) & 1u, p.timeout_ns, p.status, abort_flag)) {
                    ok = false;
                    break;
                }
                const int n = min(2, sp.nrec - 2 * m);
                const uint32_t fb = bar_xfull + 8 * xsl;
                mbar_expect_tx(fb, (uint32_t)n * xb);
                if (!(drop_first && qx == 0))
                    for (int r = 0; r < n; ++r) {
                        const int kt = (kx + r < KT) ? kx + r : kx + r - KT;
                        tma_load_2d(x_s + (uint32_t)(xsl * 2 + r) * xb, &p.xmap[j], kt * w12i::kTileK, 0, fb);
                    }
                kx += 2;
                while (kx >= KT) kx -= KT;
                ++qx;
                if (++xsl == SX) xsl = 0, ++xu;
            }
        }
        if (!ok) {
            // this CTA stops too: its MMA warp must not wait a full limit for
            // activations that will not come
            *abort_flag = 1;
            if (p.grid_abort) *(volatile int32_t *)p.grid_abort = 1;
        }
        // leave no copy in flight: the last use of every slot that was filled
        int32_t no_abort = 0;
        for (int64_t q = (qx > SX ? qx - SX : 0); q < qx; ++q) {
            if (drop_first && q == 0) continue;
            mbar_wait(bar_xfull + 8 * (int)(q % SX), (uint32_t)((q / SX) & 1), p.timeout_ns, p.status, &no_abort);
        }
    }

    // all roles done (or stopped): release tensor memory
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kProducerWarp) tmem_dealloc(tmem, kTmemCols);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
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

// Buffer plan for MMA width nr: groups x pair A buffers x 64 columns plus
// accumulators x nr columns within 512 tensor-memory columns; the activation
// ring and the record-pair ring within the shared-memory budget.
// The record ring holds a multiple of the group count: then pair q's slot is
// only ever used by pair q's group, and the slot's previous fill is that
// group's own earlier pair, which it has already consumed.  A waiter is thus
// never two fills ahead of a slot, where a parity wait would report the fill
// from two rounds back as complete.
// Preference: two accumulators (the epilogue of one tile overlaps the next
// tile's MMAs), then more decode groups, then as many record-pair slots
// (bytes in flight), then activation slots, as possible.
bool chain_buffer_plan(int nr, int max_recs, int esc_cap, int base_tiles, int budget, int *groups, int *a_bufs,
                       int *d_bufs, int *stages, int *x_slots)
{
    // (groups, A buffers per group, accumulators); named barriers 1 .. groups * A buffers stay <= 15
    static const int cand[][3] = {{4, 1, 2}, {3, 2, 2}, {3, 1, 2}, {2, 2, 2}, {2, 1, 2},
                                  {4, 1, 1}, {3, 1, 1}, {2, 2, 1}, {2, 1, 1}, {1, 2, 1}, {1, 1, 1}};
    int best = -1, best_st = 0, best_sx = 0;
    for (int k = 0; k < (int)(sizeof(cand) / sizeof(cand[0])); ++k) {
        const int g = cand[k][0], na = cand[k][1], db = cand[k][2];
        if (g * na * kACols + db * nr > (int)kTmemCols) continue;
        // the deepest record ring whose activation ring still gets min(S, 4)
        // slots (else the deepest that fits at all)
        int st = 0, sx = 0, fb_st = 0, fb_sx = 0;
        for (int s = 8 / g * g; s >= g && s >= 2 && st == 0; s -= g)
            for (int x = s + 2; x >= 2; --x)
                if (plan(s, g * na, x, nr, max_recs, esc_cap, base_tiles).total <= budget) {
                    if (x >= std::min(s, 4)) st = s, sx = x;
                    else if (fb_st == 0) fb_st = s, fb_sx = x;
                    break;
                }
        if (st == 0) st = fb_st, sx = fb_sx;
        if (st == 0) continue;
        if (best < 0 || (db > cand[best][2]) || (db == cand[best][2] && g > cand[best][0]) ||
            (db == cand[best][2] && g == cand[best][0] && (st > best_st || (st == best_st && sx > best_sx))))
            best = k, best_st = st, best_sx = sx;
    }
    if (best < 0) return false;
    *groups = cand[best][0], *a_bufs = cand[best][1], *d_bufs = cand[best][2], *stages = best_st, *x_slots = best_sx;
    return true;
}

}  // namespace

namespace w12i {

int chain_max_jobs() { return kMaxJobs; }

// One launch over jobs [0, n) (n <= kMaxJobs).
static int launch_chain_part(const ChainArgs &a, const ChainJob *jobs, int n, uint32_t *grid_bar, bool pdl,
                             void *stream)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return (int)cudaErrorNotSupported;
    if (a.R < 1 || a.R > kMaxRows || n < 1 || n > kMaxJobs) return (int)cudaErrorInvalidValue;
    if (n > 1 && !grid_bar) return (int)cudaErrorInvalidValue;
    const int nr = std::max(32, (a.R + 31) / 32 * 32);
    // A tile split between CTAs costs each contributor an nr x 128 FP32
    // partial and the last one a read of all of them; with many rows and few
    // records (a small linear at 256 rows) that reduction outweighs the
    // records, so every CTA gets at least nr / 8 records.
    const int64_t min_recs = std::max(1, nr / 8);
    ChainParams p{};
    int grid = 1, max_recs = 1, base_tiles = 2;
    for (int j = 0; j < n; ++j) {
        const ChainJob &cj = jobs[j];
        const int64_t T = (int64_t)cj.w.n_tiles * cj.w.k_tiles;
        const int G = (int)std::max<int64_t>(1, std::min<int64_t>(a.num_sms, T / min_recs));
        grid = std::max(grid, G);
        const int mr = (int)((T + G - 1) / G);
        max_recs = std::max(max_recs, mr);
        base_tiles = std::max(base_tiles, mr / cj.w.k_tiles + 2);
        CUtensorMap &m = p.xmap[j];
        const cuuint64_t dims[2] = {(cuuint64_t)cj.w.k, (cuuint64_t)a.R};
        const cuuint64_t strides[1] = {(cuuint64_t)cj.w.k * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)nr};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(cj.x), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return (int)cudaErrorInvalidValue;
        Job &jb = p.job[j];
        jb.rec = cj.w.rec;
        jb.base = cj.w.base;
        jb.esc_off = cj.w.esc_off;
        jb.esc = cj.w.esc;
        jb.y = cj.y;
        jb.s1_val = cj.s1_val;
        jb.s1_idx = cj.s1_idx;
        jb.ldy = cj.w.n;
        jb.n_tiles = cj.w.n_tiles;
        jb.k_tiles = cj.w.k_tiles;
        jb.mode = cj.mode;
        jb.ctas = G;
    }
    p.partial = a.partial;
    p.counters = a.counters;
    p.status = a.status;
    p.grid_bar = n > 1 ? grid_bar : nullptr;
    p.grid_abort = n > 1 ? a.grid_abort : nullptr;
    p.trace = a.trace;
    p.trace_stride = a.num_sms;
    p.timeout_ns = a.timeout_ns;
    p.n_jobs = n;
    p.R = a.R;
    p.nr = nr;
    p.max_recs = max_recs;
    p.esc_cap = 1024;
    p.base_tiles = std::min(64, base_tiles);
    p.debug_flags = a.debug_flags;
    const int budget = 227 * 1024;
    if (!chain_buffer_plan(nr, p.max_recs, p.esc_cap, p.base_tiles, budget, &p.groups, &p.a_bufs, &p.d_bufs,
                           &p.stages, &p.x_slots))
        return (int)cudaErrorInvalidConfiguration;
    const int smem = plan(p.stages, p.groups * p.a_bufs, p.x_slots, nr, p.max_recs, p.esc_cap, p.base_tiles).total;
    if (smem > budget) return (int)cudaErrorInvalidConfiguration;
    const auto kern = a.qview ? k_w12_chain<true> : k_w12_chain<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return (int)cudaLaunchKernelEx(&cfg, kern, p);
}

int launch_chain(const ChainArgs &a, void *stream)
{
    if (a.n_jobs < 1) return (int)cudaErrorInvalidValue;
    // GEMM counts beyond one launch's parameter block go to consecutive
    // launches of balanced size; each launch has its own arrival words
    const int parts = (a.n_jobs + kMaxJobs - 1) / kMaxJobs;
    int j0 = 0;
    for (int k = 0; k < parts; ++k) {
        const int n = (a.n_jobs - j0) / (parts - k);
        ChainArgs ak = a;
        // each launch stamps its own block of the trace: (n + 1) x grid words
        if (a.trace) ak.trace = a.trace + (int64_t)(j0 + k) * a.num_sms;
        const int e = launch_chain_part(ak, a.jobs + j0, n, a.grid_bar ? a.grid_bar + j0 : nullptr,
                                        a.pdl || k > 0, stream);
        if (e) return e;
        j0 += n;
    }
    return 0;
}

}  // namespace w12i
