// W12 verify GEMM on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// Same contract as the stream-K kernel in k_gemm.cu (SpecPilot explainer,
// section 4.1 "W12 GEMM": records restored in registers and fed to the tensor
// cores, a fixed-order stream-K split), laid out for Blackwell's tensor
// memory:
//
//   record producer  one 24 KB bulk copy per pair of consecutive records (L2
//                    evict-first) into a ring, and right behind it the pair's
//                    two activation blocks (2-D TMA, 128-byte swizzle) into an
//                    activation ring; a record slot is handed back as soon as
//                    the decode warps have read the pair into registers, an
//                    activation slot once the pair's MMAs are done
//   decode groups    one to four groups of four warps (one per tensor-memory
//                    lane quarter); a group takes every G-th record of the
//                    CTA.  Thread = output channel: six 16-byte shared loads,
//                    in-register decode of its 64 weights, escape patch, one
//                    tcgen05.st of 32 columns into one of the group's A
//                    buffers, then a non-blocking arrive on that buffer's
//                    named barrier
//   MMA warp         takes the records in order: a named-barrier sync on the
//                    record's A buffer, then one elected lane issues the
//                    record's four MMAs (M = 128 channels, N = rows rounded up
//                    to 32, K = 16) into the tile's FP32 accumulator, a commit
//                    that frees the A buffer and, after a pair, one that frees
//                    the activation slot
//   epilogue warps   tcgen05.ld of a finished tile's accumulator; BF16 rows,
//                    or the tile's (max, index) per row for the LM head; a
//                    tile split between CTAs is published as a partial and
//                    finished by the last contributor in CTA order.
//
// Every mbarrier wait is bounded.  The named-barrier hand-off cannot hang:
// decode warps arrive once for every record they own and the MMA warp syncs
// once for every record, in order, whether or not a timeout has
// stopped the work; the MMA warp commits every record, so an A buffer's next
// arrival always follows the previous sync.  Issued MMAs and copies are
// waited for, and tensor memory is released, before the CTA exits.
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
constexpr int kThreads = (kEpiWarp0 + 4) * 32;   // 22 warps
constexpr int kRecPair = 2 * w12i::kRecBytes;
constexpr int kACols = 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kBarCaches = 1;      // named barrier: decode threads after filling the shared caches
constexpr int kBarA0 = 2;          // named barrier of A buffer (g, a): kBarA0 + g * a_bufs + a (<= 13)

struct TcParams {
    const uint8_t *rec;
    const uint8_t *base;
    const int32_t *esc_off;
    const uint32_t *esc;
    int32_t n_tiles, k_tiles, R, mode;
    int32_t nr;          // MMA N: rows rounded up to 32
    int32_t groups;      // decode groups (1 or 2)
    int32_t a_bufs;      // A buffers per group
    int32_t d_bufs;      // tile accumulators (1 or 2)
    int32_t x_slots;     // activation ring: slots of one record pair's activation blocks
    uint16_t *y;
    int64_t ldy;
    float *s1_val;
    int32_t *s1_idx;
    float *partial;      // [ctas][2][nr][128]
    int32_t *counters;
    int32_t *status;
    uint32_t mul16;
    int32_t debug_flags;
    uint64_t timeout_ns;
    int32_t stages;      // record-pair slots; the activation ring and the done
                         // barriers have groups * a_bufs slots
    int32_t max_recs, esc_cap, base_tiles;
};

struct Plan {
    int rec, x, bars, misc, escoff, esc, emask, base, red, total;
};

// q = A buffers over all groups; sx = activation pair slots
__host__ __device__ inline Plan plan(int stages, int q, int sx, int nr, int max_recs, int esc_cap, int base_tiles)
{
    Plan p;
    int o = 0;
    p.rec = o;
    o += stages * kRecPair;                   // 24 KB per slot keeps the 1024-byte alignment
    p.x = o;
    o += sx * 2 * nr * 128;
    p.bars = o;
    o += 8 * (2 * stages + q + 2 * sx + 2 * 2 + 1);   // rec full/empty, A done, x full/done, acc full/empty, epilogue
    p.misc = o;
    o += 32;
    p.escoff = o;
    o += ((max_recs + 1) * 4 + 15) / 16 * 16;
    p.esc = o;
    o += esc_cap * 4;
    p.emask = o;
    o += (max_recs + 15) / 16 * 16;
    p.base = o;
    o += (base_tiles * w12i::kTileN + 15) / 16 * 16;
    p.red = o;
    o += 4 * nr * 8;      // head epilogue: per warp, per row (max, index)
    p.total = o + 1024;   // slack for the 1024-byte alignment
    return p;
}

__device__ __forceinline__ int cta_of_record(int64_t r, int G, int64_t T) { return (int)(((r + 1) * G - 1) / T); }
__device__ __forceinline__ int64_t first_record(int c, int G, int64_t T) { return (int64_t)c * T / G; }

// one lane of a converged warp
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

// kChunk: records the MMA warp takes per tensor-memory fence (see the MMA warp);
// QV: the quick pass (only the 8 KB view plane of each record is copied; the low
// mantissa bits of in-window weights are taken as the midpoint 0b1000)
template <int kChunk, bool QV>
__global__ void __launch_bounds__(kThreads, 1) k_w12_gemm_tc(const __grid_constant__ CUtensorMap xmap, const TcParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages, NR = p.nr, GR = p.groups, NAG = p.a_bufs, DB = p.d_bufs, SX = p.x_slots;
    const int Q = GR * NAG;
    const Plan pl = plan(S, Q, SX, NR, p.max_recs, p.esc_cap, p.base_tiles);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int KT = p.k_tiles;
    const int64_t T = (int64_t)p.n_tiles * KT;
    const int64_t rec_begin = first_record(cta, G, T), rec_end = first_record(cta + 1, G, T);
    const int nrec = (int)(rec_end - rec_begin);
    const int npairs = (nrec + 1) / 2;
    const int64_t nt_first = rec_begin / KT, nt_last = (rec_end - 1) / KT;

    const uint32_t rec_s = smem_u32(smem + pl.rec), x_s = smem_u32(smem + pl.x);
    const uint32_t xb = (uint32_t)NR * 128;
    const uint32_t bar0 = smem_u32(smem + pl.bars);
    const uint32_t bar_rfull = bar0, bar_rempty = bar0 + 8 * S;
    const uint32_t bar_done = bar_rempty + 8 * S;
    const uint32_t bar_xfull = bar_done + 8 * Q, bar_xdone = bar_xfull + 8 * SX;
    const uint32_t bar_accfull = bar_xdone + 8 * SX, bar_accempty = bar_accfull + 16;
    const uint32_t bar_epi = bar_accempty + 16;
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + pl.misc);
    int32_t *last_flag = reinterpret_cast<int32_t *>(smem + pl.misc + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + pl.misc + 8);
    int32_t *esc_off_s = reinterpret_cast<int32_t *>(smem + pl.escoff);
    uint32_t *esc_s = reinterpret_cast<uint32_t *>(smem + pl.esc);
    uint8_t *emask_s = smem + pl.emask;
    uint8_t *base_s = smem + pl.base;

    const bool drop_first = (p.debug_flags & 1) && cta == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_rfull + 8 * s, 1);    // producer's expect_tx arrival + the copy's bytes
            mbar_init(bar_rempty + 8 * s, 8);   // the decode warps have read both records of the pair
        }
        for (int s = 0; s < Q; ++s) mbar_init(bar_done + 8 * s, 1);   // one commit per record: its MMAs are done
        for (int s = 0; s < SX; ++s) {
            mbar_init(bar_xfull + 8 * s, 1);    // producer's expect_tx arrival + the pair's activation blocks
            mbar_init(bar_xdone + 8 * s, 1);    // one commit per pair: the MMAs reading the slot are done
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(bar_accfull + 8 * d, 1);    // commit after a tile's last MMA
            mbar_init(bar_accempty + 8 * d, 4);   // the four epilogue warps have read the accumulator
        }
        mbar_init(bar_epi, 4);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarp) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    const uint32_t d_col0 = (uint32_t)(GR * NAG * kACols);
    auto a_col = [&](int g, int a) { return (uint32_t)((g * NAG + a) * kACols); };
    auto d_col = [&](int d) { return d_col0 + (uint32_t)(d * NR); };

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- record producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            auto issue = [&](int m, int sl) {
                const int n = min(2, nrec - 2 * m);
                if constexpr (QV) {
                    // the view plane of each record: its first 8 KB, at the record's place in the slot
                    mbar_expect_tx(bar_rfull + 8 * sl, (uint32_t)(n * w12i::kViewBytes));
                    if (!(drop_first && m == 0))
                        for (int r = 0; r < n; ++r)
                            bulk_g2s(rec_s + sl * kRecPair + r * w12i::kRecBytes,
                                     p.rec + (rec_begin + 2 * m + r) * (int64_t)w12i::kRecBytes,
                                     (uint32_t)w12i::kViewBytes, bar_rfull + 8 * sl, pol);
                } else {
                    mbar_expect_tx(bar_rfull + 8 * sl, (uint32_t)(n * w12i::kRecBytes));
                    if (!(drop_first && m == 0))
                        bulk_g2s(rec_s + sl * kRecPair, p.rec + (rec_begin + 2 * m) * (int64_t)w12i::kRecBytes,
                                 (uint32_t)(n * w12i::kRecBytes), bar_rfull + 8 * sl, pol);
                }
            };
            // activation blocks of pair m (k-tile kt0 for its first record) into
            // pair slot xsl, right behind the pair's records in the copy queue
            auto issue_x = [&](int m, int xsl, int kt0) {
                const int n = min(2, nrec - 2 * m);
                mbar_expect_tx(bar_xfull + 8 * xsl, (uint32_t)n * xb);
                if (drop_first && m == 0) return;
                for (int r = 0; r < n; ++r) {
                    const int kt = (kt0 + r < KT) ? kt0 + r : kt0 + r - KT;
                    tma_load_2d(x_s + (uint32_t)(xsl * 2 + r) * xb, &xmap, kt * w12i::kTileK, 0, bar_xfull + 8 * xsl);
                }
            };
            prefetch_tmap(&xmap);
            // weights do not depend on earlier kernels: they start before the
            // programmatic-dependency wait, the activations after it
            const int pre = min(S, npairs);
            for (int m = 0; m < pre; ++m) issue(m, m);
            pdl_wait();
            int kt0 = (int)(rec_begin - nt_first * KT);   // k-tile of record 2m
            auto adv = [&]() {
                kt0 += 2;
                while (kt0 >= KT) kt0 -= KT;
            };
            // Records and activations advance on their own: record pair mr waits
            // for its slot (the decode warps read pair mr - S), activation pair mx
            // for its slot (the MMAs of pair mx - SX), and neither holds up the
            // other.  Slots and reuse parities are advanced without divisions.
            int mr = pre, mx = 0;
            int sl = pre % S, xsl = 0;
            uint32_t rph = (uint32_t)((pre / S) - 1) & 1u, xph = 1u;
            bool stalled = false;
            uint64_t t_idle = 0;
            while ((mr < npairs || mx < npairs) && !stalled) {
                bool moved = false;
                if (mr < npairs && mbar_try_wait(bar_rempty + 8 * sl, rph)) {
                    issue(mr, sl);
                    ++mr;
                    if (++sl == S) sl = 0, rph ^= 1u;
                    moved = true;
                }
                if (mx < npairs && (mx < SX || mbar_try_wait(bar_xdone + 8 * xsl, xph))) {
                    issue_x(mx, xsl, kt0);
                    adv();
                    ++mx;
                    if (++xsl == SX) xsl = 0, xph ^= 1u;
                    moved = true;
                }
                if (moved) {
                    t_idle = 0;
                    continue;
                }
                // both rings full: back off so that this warp's polls do not
                // take issue slots from the decode warps of its scheduler
                __nanosleep(64);
                if (*abort_flag) {
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
                // leave no copy in flight
                int32_t no_abort = 0;
                for (int m = max(0, mr - S); m < mr; ++m) {
                    if (drop_first && m == 0) continue;
                    mbar_wait(bar_rfull + 8 * (m % S), (m / S) & 1, p.timeout_ns, p.status, &no_abort);
                }
                for (int m = max(0, mx - SX); m < mx; ++m) {
                    if (drop_first && m == 0) continue;
                    mbar_wait(bar_xfull + 8 * (m % SX), (m / SX) & 1, p.timeout_ns, p.status, &no_abort);
                }
            }
        }
    } else if (warp < kMmaWarp) {
        // --------------------------------------------------------------- decode
        const int g = (warp - kGroupWarp0) >> 2;
        const int wq = (warp - kGroupWarp0) & 3;     // warp within the group
        const int quarter = warp & 3;                // tensor-memory lanes this warp may touch
        const int c = quarter * 32 + lane;           // output channel of this thread
        if (g < GR) {
            const int dtid = g * 128 + wq * 32 + lane;
            const int ndec = GR * 128;
            // shared caches: escape offsets/entries of the CTA's records, window bases
            const int nt_span = (int)(nt_last - nt_first + 1);
            const bool base_cached = nt_span <= p.base_tiles;
            for (int i = dtid; i <= nrec; i += ndec) esc_off_s[i] = __ldg(p.esc_off + rec_begin + i);
            if (base_cached)
                for (int i = dtid; i < nt_span * w12i::kTileN; i += ndec)
                    base_s[i] = __ldg(p.base + nt_first * w12i::kTileN + i);
            named_bar(kBarCaches, ndec);
            const int32_t e_lo = esc_off_s[0];
            const bool esc_cached = (esc_off_s[nrec] - e_lo) <= p.esc_cap;
            if (esc_cached)
                for (int i = dtid; i < esc_off_s[nrec] - e_lo; i += ndec) esc_s[i] = __ldg(p.esc + e_lo + i);
            // per record, a bit for every 32-channel quarter that holds an
            // escape: the other quarters' warps skip the escape list
            for (int i = dtid; i < nrec; i += ndec) {
                uint32_t msk = 0;
                for (int e = esc_off_s[i]; e < esc_off_s[i + 1]; ++e) msk |= 1u << ((__ldg(p.esc + e) >> 27) & 3u);
                emask_s[i] = (uint8_t)msk;
            }
            named_bar(kBarCaches, ndec);

            int64_t nt_cur = -1;
            ChanConst cc{0, 0};
            // every record of the group is visited: work is skipped after a
            // timeout, but the hand-off to the MMA warp always takes place
            // per-record indices advanced without divisions: pair m = i / 2 in
            // slot s (fill parity sph), tile nt / k-tile kt of record i, A
            // buffer ab, activation slot iq (fill parity iph)
            // record g sits in pair g / 2 (slot g / 2: there are at least two slots)
            int m = g >> 1, s = g >> 1;
            uint32_t sph = 0;
            int64_t nt = (rec_begin + g) / KT;
            int kt = (int)((rec_begin + g) - nt * KT);
            int ab = 0, iq = g;
            uint32_t iph = 0;
            for (int j = 0;; ++j) {
                const int i = g + j * GR;
                if (i >= nrec) break;
                if (j > 0) {
                    while (m < (i >> 1)) {   // record pair m holds records 2m, 2m + 1
                        ++m;
                        if (++s == S) s = 0, sph ^= 1u;
                    }
                    kt += GR;
                    while (kt >= KT) kt -= KT, ++nt;
                    if (++ab == NAG) ab = 0;
                    iq += GR;
                    if (iq >= Q) iq -= Q, iph ^= 1u;
                }
                const bool has_esc = (emask_s[i] >> quarter) & 1u;
                bool ok = !*abort_flag;
                if (ok) ok = mbar_wait(bar_rfull + 8 * s, sph, p.timeout_ns, p.status, abort_flag);
                if (i >= Q) {
                    // A buffer ab last held record i - Q: its MMAs must be done.
                    // The MMA warp commits every record, so this wait ends even
                    // after an abort; it is never skipped (the buffer's named
                    // barrier is reused only after its sync: a second arrival
                    // before that sync would leave the MMA warp waiting at the
                    // barrier for good).  The MMA warp may itself sit in one
                    // bounded wait before it commits, so this wait is allowed
                    // several of those limits and never gives up first.
                    int32_t no_abort = 0;
                    if (!mbar_wait(bar_done + 8 * iq, iph ^ 1u, kReuseWaits * p.timeout_ns, p.status, &no_abort))
                        ok = false;
                }
                ok = __all_sync(0xffffffffu, ok && !*abort_flag);
                if (ok) {
                    if (nt != nt_cur) {
                        nt_cur = nt;
                        const uint32_t b = base_cached ? base_s[(nt - nt_first) * w12i::kTileN + c]
                                                       : __ldg(p.base + nt * w12i::kTileN + c);
                        cc = chan_const(b);
                    }
                    const uint8_t *rb = smem + pl.rec + s * kRecPair + (i & 1) * w12i::kRecBytes;
                    uint4 v[4], nb[2];
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[q] = *reinterpret_cast<const uint4 *>(rb + (q * 128 + c) * 16);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        nb[h] = QV ? make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u)
                                   : *reinterpret_cast<const uint4 *>(rb + w12i::kViewBytes + (h * 128 + c) * 16);
                    // the record is in registers: hand the slot back to the producer
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_rempty + 8 * s);
                    uint32_t a[32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t vw[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
                        const uint4 n4 = nb[q >> 1];
                        const uint32_t nw[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
                        for (int w = 0; w < 4; ++w)
                            decode_word(vw[w], nw[w] >> ((q & 1) * 4), cc, p.mul16, a[8 * q + w], a[8 * q + 4 + w]);
                    }
                    // escaped slots of this channel: the exact value replaces the filler
                    const int32_t e0 = has_esc ? esc_off_s[i] - e_lo : 0, e1 = has_esc ? esc_off_s[i + 1] - e_lo : 0;
                    for (int e = e0; e < e1; ++e) {
                        const uint32_t en = esc_cached ? esc_s[e] : __ldg(p.esc + e_lo + e);
                        const int nl = (en >> 22) & 0x7F;
                        if ((nl >> 5) != quarter) continue;   // warp-uniform skip
                        const int kl = (en >> 16) & 0x3F;
                        if (nl == c) patch_half(a, kl >> 1, en & 0xFFFFu, kl & 1);
                    }
                    tmem_st_x32(tmem + ((uint32_t)(quarter * 32) << 16) + a_col(g, ab), a);
                    tmem_st_wait();
                    tc_fence_before();
                }
                __syncwarp();
                named_arrive(kBarA0 + g * NAG + ab, 160);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA
        const uint32_t idesc = idesc_bf16_f32(128, NR);
        int tcount = 0, dcur = 0;
        int kt = (int)(rec_begin - nt_first * KT);
        if constexpr (kChunk == 1) {
            // group g, A buffer ab, A-buffer done slot aq and activation pair slot
            // xsl (fill parity xph) of record i, advanced without divisions
            int g = 0, ab = 0, aq = 0, xsl = 0;
            uint32_t xph = 0;
            for (int i = 0; i < nrec; ++i) {
                if (i > 0) {
                    if (++g == GR) {
                        g = 0;
                        if (++ab == NAG) ab = 0;
                    }
                    if (++aq == Q) aq = 0;
                }
                named_bar(kBarA0 + g * NAG + ab, 160);
                // the whole warp runs this part (it stays converged); one elected
                // lane issues the tensor-core instructions
                tc_fence_after();
                const bool first = (i == 0) || kt == 0;
                const bool last = (i == nrec - 1) || kt == KT - 1;
                const bool pair_end = (i & 1) || i == nrec - 1;
                bool go = !*abort_flag;
                if (go && (i & 1) == 0) go = mbar_wait(bar_xfull + 8 * xsl, xph, p.timeout_ns, p.status, abort_flag);
                go = __all_sync(0xffffffffu, go);
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
                        const uint32_t d_t = tmem + d_col(dcur), a_t = tmem + a_col(g, ab);
                        const uint64_t bd = smem_desc_sw128(x_s + (uint32_t)(xsl * 2 + (i & 1)) * xb);
    #pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc_mma_ts(d_t, a_t + ks * 8, bd + (uint64_t)(ks * 2), idesc, (first && ks == 0) ? 0u : 1u);
                    }
                    tc_commit(bar_done + 8 * aq);                 // always: frees the A buffer
                    if (pair_end) tc_commit(bar_xdone + 8 * xsl);   // always: frees the activation slot
                    if (last && go) tc_commit(bar_accfull + 8 * dcur);
                }
                __syncwarp();
                if (last) ++tcount;
                if (pair_end && ++xsl == SX) xsl = 0, xph ^= 1u;
                if (++kt == KT) kt = 0;
            }
        } else {
            // group g, A buffer ab, A-buffer done slot aq and activation pair slot
            // xsl (fill parity xph) of the next record, advanced without divisions.
            // The records are taken in chunks of up to kChunk within one tile: one
            // tensor-memory fence per chunk, after the chunk's named-barrier syncs.
            // Up to 64 rows the host picks 4 (LM head at 32 rows 269 -> 252 us);
            // wider MMAs want each record issued as soon as it is decoded, so
            // there it picks 1 (a separate instantiation: sharing one with the
            // chunked loop made the wide launches 1.5x slower).
            int g = 0, ab = 0, aq = 0, xsl = 0;
            uint32_t xph = 0;
            for (int i = 0; i < nrec;) {
                int n = min(kChunk, nrec - i);
                n = min(n, KT - kt);   // a chunk never crosses a tile boundary
                n = min(n, Q);         // record r's buffer waits for record r - Q's commit
                int cg[kChunk], cab[kChunk], caq[kChunk], cxs[kChunk];
                uint32_t cxp[kChunk];
                bool cpe[kChunk];
    #pragma unroll
                for (int j = 0; j < kChunk; ++j) {
                    if (j < n) {
                        const int r = i + j;
                        if (r > 0) {
                            if (++g == GR) {
                                g = 0;
                                if (++ab == NAG) ab = 0;
                            }
                            if (++aq == Q) aq = 0;
                            if ((r & 1) == 0 && ++xsl == SX) xsl = 0, xph ^= 1u;   // a new pair starts
                        }
                        cg[j] = g, cab[j] = ab, caq[j] = aq, cxs[j] = xsl, cxp[j] = xph;
                        cpe[j] = (r & 1) || r == nrec - 1;
                        named_bar(kBarA0 + g * NAG + ab, 160);
                    }
                }
                // the whole warp runs this part (it stays converged); one elected
                // lane issues the tensor-core instructions
                tc_fence_after();
                const bool first = (i == 0) || kt == 0;
                const bool last = (i + n == nrec) || kt + n == KT;
                bool go = !*abort_flag;
    #pragma unroll
                for (int j = 0; j < kChunk; ++j)
                    if (j < n && go && ((i + j) & 1) == 0)
                        go = mbar_wait(bar_xfull + 8 * cxs[j], cxp[j], p.timeout_ns, p.status, abort_flag);
                go = __all_sync(0xffffffffu, go);
                if (first) {
                    dcur = tcount % DB;
                    if (go && tcount >= DB)
                        go = mbar_wait(bar_accempty + 8 * dcur, ((tcount / DB) - 1) & 1, p.timeout_ns, p.status,
                                       abort_flag);
                    go = __all_sync(0xffffffffu, go);
                    tc_fence_after();
                }
                if (elect_one()) {
    #pragma unroll
                    for (int j = 0; j < kChunk; ++j) {
                        if (j < n) {
                            if (go) {
                                const uint32_t d_t = tmem + d_col(dcur), a_t = tmem + a_col(cg[j], cab[j]);
                                const uint64_t bd = smem_desc_sw128(x_s + (uint32_t)(cxs[j] * 2 + ((i + j) & 1)) * xb);
    #pragma unroll
                                for (int ks = 0; ks < 4; ++ks)
                                    tc_mma_ts(d_t, a_t + ks * 8, bd + (uint64_t)(ks * 2), idesc,
                                              (first && j == 0 && ks == 0) ? 0u : 1u);
                            }
                            tc_commit(bar_done + 8 * caq[j]);                    // always: frees the A buffer
                            if (cpe[j]) tc_commit(bar_xdone + 8 * cxs[j]);       // always: frees the activation slot
                        }
                    }
                    if (last && go) tc_commit(bar_accfull + 8 * dcur);
                }
                __syncwarp();
                if (last) ++tcount;
                kt += n;
                if (kt == KT) kt = 0;
                i += n;
            }
        }
        // tensor memory is released only after every issued MMA finished
        if (nrec > 0) {
            int32_t no_abort = 0;
            mbar_wait(bar_done + 8 * ((nrec - 1) % Q), ((nrec - 1) / Q) & 1, p.timeout_ns, p.status, &no_abort);
        }
    } else {
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
        // write (or reduce, for the LM head) 32 rows r0..r0+31 of this channel
        auto emit_rows = [&](int64_t nt, int r0, const float (&v)[32]) {
            if (p.mode == w12i::kModeLinear) {
                uint16_t *yc = p.y + nt * w12i::kTileN + c;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (r0 + j < rows) yc[(int64_t)(r0 + j) * p.ldy] = (uint16_t)(pack_bf16x2(v[j], 0.f) & 0xFFFFu);
            } else {
                // (max, lowest index) over the warp's 32 channels for 32 rows at
                // once: at each of five steps a lane keeps half of its rows,
                // trades the other half with its partner and combines; lane l
                // ends with row r0 + l (31 trades instead of 32 x 5)
                float bv[32];
                int32_t bi[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) bv[j] = v[j], bi[j] = c;
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
            if (p.mode != w12i::kModeHead) return true;
            if (!epi_sync()) return false;
            for (int r = etid; r < rows; r += 128) {
                float bv = red_v[r];
                int32_t bi = red_i[r];
                for (int w = 1; w < 4; ++w)
                    if (beats(red_v[w * NR + r], red_i[w * NR + r], bv, bi))
                        bv = red_v[w * NR + r], bi = red_i[w * NR + r];
                p.s1_val[(int64_t)r * p.n_tiles + nt] = bv;
                p.s1_idx[(int64_t)r * p.n_tiles + nt] = (int32_t)(nt * w12i::kTileN + bi);
            }
            return epi_sync();
        };
        for (int64_t nt = nt_first; nt <= nt_last; ++nt) {
            const int64_t t0 = nt * KT, t1 = t0 + KT;
            const int dsel = tcount % DB;
            const bool ok = mbar_wait(bar_accfull + 8 * dsel, (tcount / DB) & 1, p.timeout_ns, p.status, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const bool owned = rec_begin <= t0 && rec_end >= t1;
            const int slot = (nt == nt_first) ? 0 : 1;
            float *mine = p.partial + ((int64_t)(cta * 2 + slot) * NR) * w12i::kTileN;
            const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
            for (int r0 = 0; r0 < NR; r0 += 32) {
                uint32_t raw[32];
                tmem_ld_x32(lane_base + d_col(dsel) + r0, raw);
                tmem_ld_wait();
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
                if (owned) {
                    emit_rows(nt, r0, v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (r0 + j < rows) __stcg(mine + (r0 + j) * w12i::kTileN + c, v[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_accempty + 8 * dsel);
            ++tcount;
            if (owned) {
                if (!head_finish(nt)) break;
                continue;
            }
            // split tile: publish, count arrivals, the last contributor finishes it
            __threadfence();
            if (!epi_sync()) break;
            const int c_first = cta_of_record(t0, G, T), c_last = cta_of_record(t1 - 1, G, T);
            if (etid == 0) *last_flag = (atomicAdd(p.counters + nt, 1) == c_last - c_first);
            if (!epi_sync()) break;
            if (*last_flag == 0) continue;
            __threadfence();
            for (int r0 = 0; r0 < NR; r0 += 32) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
                for (int cc2 = c_first; cc2 <= c_last; ++cc2) {
                    const int sl = (nt == first_record(cc2, G, T) / KT) ? 0 : 1;
                    const float *src = p.partial + ((int64_t)(cc2 * 2 + sl) * NR) * w12i::kTileN;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (r0 + j < rows) v[j] += __ldcg(src + (r0 + j) * w12i::kTileN + c);
                }
                emit_rows(nt, r0, v);
            }
            if (etid == 0) p.counters[nt] = 0;   // ready for the next launch using this slot
            if (!head_finish(nt)) break;
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

EncodeTiledFn encode_fn_tc()
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

// Buffer plan for MMA width nr: groups x A buffers x 32 columns plus
// accumulators x nr columns within 512 tensor-memory columns; the activation
// ring (groups x A buffers slots of nr x 128 bytes) and at least two
// record-pair slots within the shared-memory budget.  Preference: two
// accumulators (the epilogue of one tile overlaps the next tile's MMAs), then
// more decode groups, then as many record-pair slots (bytes in flight) as
// possible.
bool tc_buffer_plan(int nr, int max_recs, int esc_cap, int base_tiles, int budget, int *groups, int *a_bufs,
                    int *d_bufs, int *stages, int *x_slots)
{
    // (groups, A buffers per group, accumulators); named barriers 2 .. 2 + groups * A buffers - 1 stay below 16
    static const int cand[][3] = {{4, 3, 2}, {4, 2, 2}, {4, 2, 1}, {3, 4, 2}, {3, 3, 2}, {3, 2, 2}, {3, 2, 1},
                                  {2, 4, 2}, {2, 3, 2}, {2, 2, 2}, {2, 4, 1}, {2, 2, 1}, {1, 4, 2}, {1, 4, 1}, {1, 2, 1}};
    int best = -1, best_st = 0, best_sx = 0;
    for (int k = 0; k < (int)(sizeof(cand) / sizeof(cand[0])); ++k) {
        const int g = cand[k][0], na = cand[k][1], db = cand[k][2];
        if (g * na * kACols + db * nr > (int)kTmemCols) continue;
        // the most record-pair slots, then an activation ring up to two pairs deeper
        int st = 0, sx = 0;
        // Group g takes records g, g + G, ...; pair slot P % S last held pair
        // P - S.  With 4 groups a group reads every other pair, with 3 groups
        // two pairs in three, so an even S (4 groups) or a multiple of 3 (3
        // groups) makes pair P - S one the group itself has already consumed:
        // a group waiting on a slot is then never two fills ahead of it, where
        // a parity wait would report the fill from two rounds back as done.
        const int s_step = g == 4 ? 2 : g == 3 ? 3 : 1;
        for (int s = 8 / s_step * s_step; s >= 2 && st == 0; s -= s_step)
            for (int x = s + 2; x >= s; --x)
                if (plan(s, g * na, x, nr, max_recs, esc_cap, base_tiles).total <= budget) {
                    st = s, sx = x;
                    break;
                }
        if (st == 0) continue;
        if (best < 0 || (db > cand[best][2]) || (db == cand[best][2] && g > cand[best][0]) ||
            (db == cand[best][2] && g == cand[best][0] && (st > best_st || (st == best_st && sx > best_sx))))
            best = k, best_st = st, best_sx = sx;
    }
    if (best < 0) return false;
    *groups = cand[best][0], *a_bufs = cand[best][1], *d_bufs = cand[best][2], *stages = best_st, *x_slots = best_sx;
    return true;
}

int launch_gemm_tc(const GemmArgs &a, void *stream)
{
    EncodeTiledFn enc = encode_fn_tc();
    if (!enc) return (int)cudaErrorNotSupported;
    if (a.R < 1 || a.R > kMaxRows) return (int)cudaErrorInvalidValue;
    const int nr = std::max(32, (a.R + 31) / 32 * 32);
    CUtensorMap xmap;
    const cuuint64_t dims[2] = {(cuuint64_t)a.w.k, (cuuint64_t)a.R};
    const cuuint64_t strides[1] = {(cuuint64_t)a.w.k * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)nr};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a.x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return (int)cudaErrorInvalidValue;
    const int64_t T = (int64_t)a.w.n_tiles * a.w.k_tiles;
    // A tile split between CTAs costs each contributor an nr x 128 FP32
    // partial and the last one a read of all of them; with many rows and few
    // records (a small linear at 256 rows) that reduction outweighs the
    // records, so every CTA gets at least nr / 8 records.
    const int64_t min_recs = std::max(1, nr / 8);
    const int G = (int)std::max<int64_t>(1, std::min<int64_t>(a.num_sms, T / min_recs));
    TcParams p{};
    p.rec = a.w.rec;
    p.base = a.w.base;
    p.esc_off = a.w.esc_off;
    p.esc = a.w.esc;
    p.n_tiles = a.w.n_tiles;
    p.k_tiles = a.w.k_tiles;
    p.R = a.R;
    p.mode = a.mode;
    p.nr = nr;

    p.y = a.y;
    p.ldy = a.w.n;
    p.s1_val = a.stage1_val;
    p.s1_idx = a.stage1_idx;
    p.partial = a.partial;
    p.counters = a.counters;
    p.status = a.status;
    p.mul16 = 16u;
    p.debug_flags = a.debug_flags;
    p.timeout_ns = a.timeout_ns;
    p.max_recs = (int)((T + G - 1) / G);
    p.esc_cap = 2048;
    p.base_tiles = std::min<int>(64, (int)(p.max_recs / a.w.k_tiles + 2));
    const int budget = 227 * 1024;
    if (!tc_buffer_plan(nr, p.max_recs, p.esc_cap, p.base_tiles, budget, &p.groups, &p.a_bufs, &p.d_bufs, &p.stages,
                        &p.x_slots))
        return (int)cudaErrorInvalidConfiguration;
    const int smem = plan(p.stages, p.groups * p.a_bufs, p.x_slots, nr, p.max_recs, p.esc_cap, p.base_tiles).total;
    if (smem > budget) return (int)cudaErrorInvalidConfiguration;
    // chunks of four records per fence up to 64 rows with two accumulators
    const bool chunked = nr <= 64 && p.d_bufs == 2;
    const auto kern = a.qview ? (chunked ? k_w12_gemm_tc<4, true> : k_w12_gemm_tc<1, true>)
                              : (chunked ? k_w12_gemm_tc<4, false> : k_w12_gemm_tc<1, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return (int)cudaLaunchKernelEx(&cfg, kern, xmap, p);
}

}  // namespace w12i
