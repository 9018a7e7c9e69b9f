// W12 verify GEMM on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// Same contract as the stream-K kernel in k_gemm.cu (SpecPilot explainer,
// section 4.1 "W12 GEMM": records restored in registers and fed to the tensor
// cores, a fixed-order stream-K split), laid out for Blackwell's tensor
// memory instead of warp-level MMA fragments:
//
//   producer warp   bulk copy of each 12 KB record + 2-D TMA of the matching
//                   activation block (128-byte swizzle) into a shared ring
//   decode warps    two groups of four, alternating records; thread = output
//                   channel: six 16-byte shared loads, in-register decode of
//                   its 64 weights, escape patch, one tcgen05.st of 32
//                   columns into a tensor-memory A buffer (4 buffers)
//   MMA thread      per record four tcgen05.mma (M=128 channels, N = rows
//                   rounded up to 32, K=16) with A from tensor memory and the
//                   activations from shared memory, FP32 accumulator in
//                   tensor memory (two accumulators while N <= 192)
//   epilogue warps  tcgen05.ld of a finished tile; BF16 rows, or the tile's
//                   (max, index) per row for the LM head; a tile split between
//                   CTAs is published as a partial and finished by the last
//                   contributor in CTA order (deterministic, no waiting)
//
// Every wait is bounded: on a timeout the kernel records W12_E_TIMEOUT, all
// roles stop, the MMA thread waits for its issued work, and tensor memory is
// released before the CTA exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "w12_device.cuh"

using namespace w12d;

namespace {

constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kDecodeWarp0 = 2;   // warps 2..9: group 0 = 2..5, group 1 = 6..9
constexpr int kEpiWarp0 = 10;     // warps 10..13
constexpr int kThreads = 14 * 32;
constexpr int kMaxABufs = 8;      // tensor-memory A buffers of 32 columns (8 while N <= 128, else 4)
constexpr int kACols = 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kRecsPerStage = 1;  // records per shared-memory stage
constexpr int kBatch = 4;         // records per MMA batch: one wait round, 16 MMAs, two commits

struct TcParams {
    const uint8_t *rec;
    const uint8_t *base;
    const int32_t *esc_off;
    const uint32_t *esc;
    int32_t n_tiles, k_tiles, R, mode;
    int32_t nr;          // MMA N: rows rounded up to 32
    int32_t d_bufs;      // accumulators in tensor memory (1 or 2)
    int32_t a_bufs;      // A buffers in tensor memory (4 or 8); accumulators start after them
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
    int32_t stages, max_recs, esc_cap, base_tiles;
};

struct Plan {
    int rec, x, bars, misc, escoff, esc, base, red, total;
};

__host__ __device__ inline Plan plan(int stages, int nr, int max_recs, int esc_cap, int base_tiles)
{
    Plan p;
    int o = 0;
    p.rec = o;
    o += stages * kRecsPerStage * w12i::kRecBytes;
    p.x = o;
    o += stages * kRecsPerStage * nr * 128;
    p.bars = o;
    o += 8 * (2 * stages + 2 * kMaxABufs + 4 + 2);   // full + slot-empty, A ready + A free, acc, syncs
    p.misc = o;
    o += 32;
    p.escoff = o;
    o += ((max_recs + 1) * 4 + 15) / 16 * 16;
    p.esc = o;
    o += esc_cap * 4;
    p.base = o;
    o += (base_tiles * w12i::kTileN + 15) / 16 * 16;
    p.red = o;
    o += 4 * nr * 8;      // head epilogue: per warp, per row (max, index)
    p.total = o + 1024;   // slack for the 1024-byte alignment
    return p;
}

__device__ __forceinline__ int cta_of_record(int64_t r, int G, int64_t T) { return (int)(((r + 1) * G - 1) / T); }
__device__ __forceinline__ int64_t first_record(int c, int G, int64_t T) { return (int64_t)c * T / G; }

__global__ void __launch_bounds__(kThreads, 1) k_w12_gemm_tc(const __grid_constant__ CUtensorMap xmap, const TcParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages, NR = p.nr;
    const Plan pl = plan(S, NR, p.max_recs, p.esc_cap, p.base_tiles);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int KT = p.k_tiles;
    const int64_t T = (int64_t)p.n_tiles * KT;
    const int64_t rec_begin = first_record(cta, G, T), rec_end = first_record(cta + 1, G, T);
    const int nrec = (int)(rec_end - rec_begin);
    const int64_t nt_first = rec_begin / KT, nt_last = (rec_end - 1) / KT;

    const uint32_t rec_s = smem_u32(smem + pl.rec), x_s = smem_u32(smem + pl.x);
    const uint32_t bar0 = smem_u32(smem + pl.bars);
    const uint32_t bar_full = bar0, bar_empty = bar0 + 8 * S;
    const uint32_t bar_afull = bar_empty + 8 * S, bar_afree = bar_afull + 8 * kMaxABufs;
    const uint32_t bar_accfull = bar_afree + 8 * kMaxABufs, bar_accempty = bar_accfull + 16;
    const int NA = p.a_bufs;
    const int kDCol0 = NA * kACols;
    const uint32_t bar_epi = bar_accempty + 16, bar_dec = bar_epi + 8;
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + pl.misc);
    int32_t *last_flag = reinterpret_cast<int32_t *>(smem + pl.misc + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + pl.misc + 8);
    int32_t *esc_off_s = reinterpret_cast<int32_t *>(smem + pl.escoff);
    uint32_t *esc_s = reinterpret_cast<uint32_t *>(smem + pl.esc);
    uint8_t *base_s = smem + pl.base;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 4 * kBatch + 1);   // per slot of kBatch stages: 4 decode warps per record + 1 commit
        }
        for (int b = 0; b < kMaxABufs; ++b) {
            mbar_init(bar_afull + 8 * b, 4);    // per A buffer: the 4 decode warps that filled it
            mbar_init(bar_afree + 8 * b, 1);    // per batch of A buffers: one MMA commit
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(bar_accfull + 8 * d, 1);
            mbar_init(bar_accempty + 8 * d, 4);
        }
        mbar_init(bar_epi, 4);     // one arrival per epilogue warp
        mbar_init(bar_dec, 8);     // one arrival per decode warp
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp == kProducerWarp) {
        // -------------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tmap(&xmap);
            const uint64_t pol = policy_evict_first();
            const uint32_t xb = (uint32_t)NR * 128;
            const bool drop_first = (p.debug_flags & 1) && cta == 0;
            const int nst = (nrec + kRecsPerStage - 1) / kRecsPerStage;
            auto recs_in = [&](int j) { return min(kRecsPerStage, nrec - j * kRecsPerStage); };
            auto issue_w = [&](int j, int sl) {
                const int n = recs_in(j);
                mbar_expect_tx(bar_full + 8 * sl, (uint32_t)n * (w12i::kRecBytes + xb));
                if (!(drop_first && j == 0))
                    bulk_g2s(rec_s + sl * kRecsPerStage * w12i::kRecBytes,
                             p.rec + (rec_begin + j * kRecsPerStage) * (int64_t)w12i::kRecBytes,
                             (uint32_t)n * w12i::kRecBytes, bar_full + 8 * sl, pol);
            };
            auto issue_x = [&](int j, int sl) {
                if (drop_first && j == 0) return;
                for (int r = 0; r < recs_in(j); ++r) {
                    const int kt = (int)((rec_begin + j * kRecsPerStage + r) % KT);
                    tma_load_2d(x_s + (sl * kRecsPerStage + r) * xb, &xmap, kt * w12i::kTileK, 0, bar_full + 8 * sl);
                }
            };
            const int pre = min(S, nst);
            for (int j = 0; j < pre; ++j) issue_w(j, j);
            pdl_wait();
            for (int j = 0; j < pre; ++j) issue_x(j, j);
            int issued = pre;
            for (int j = pre; j < nst; ++j) {
                const int sl = j % S;
                // the first stage of a slot waits until the whole slot is released
                if (sl % kBatch == 0 &&
                    !mbar_wait(bar_empty + 8 * (sl / kBatch), ((j / S) - 1) & 1, p.timeout_ns, p.status, abort_flag))
                    break;
                issue_w(j, sl);
                issue_x(j, sl);
                issued = j + 1;
            }
            if (*abort_flag) {
                int32_t no_abort = 0;
                for (int j = max(0, issued - S); j < issued; ++j) {
                    if (drop_first && j == 0) continue;
                    mbar_wait(bar_full + 8 * (j % S), (j / S) & 1, p.timeout_ns, p.status, &no_abort);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------- MMA issue
        const uint32_t idesc = idesc_bf16_f32(128, NR);
        int kt = (int)(rec_begin - nt_first * KT);
        int dbuf = 0;
        uint32_t duse[2] = {0, 0};
        int last_i = -1;
        for (int i0 = 0; i0 < nrec; i0 += kBatch) {
            // lanes wait in parallel: lane l < kBatch on record i0+l's A buffer,
            // lane kBatch+l on its shared-memory stage
            bool ok = true;
            if (lane < 2 * kBatch) {
                const int i = i0 + (lane % kBatch);
                if (i < nrec) {
                    if (lane < kBatch)
                        ok = mbar_wait(bar_afull + 8 * (i % NA), (i / NA) & 1, p.timeout_ns, p.status, abort_flag);
                    else
                        ok = mbar_wait(bar_full + 8 * (i % S), (i / S) & 1, p.timeout_ns, p.status, abort_flag);
                }
            }
            if (__any_sync(0xffffffffu, !ok)) break;
            if (lane == 0) {
                tc_fence_after();
                const int n = min(kBatch, nrec - i0);
                bool stop = false;
                for (int r = 0; r < n && !stop; ++r) {
                    const int i = i0 + r;
                    const bool first = (i == 0) || kt == 0;
                    const bool last = (i == nrec - 1) || kt == KT - 1;
                    if (first && duse[dbuf] > 0) {
                        if (!mbar_wait(bar_accempty + 8 * dbuf, (duse[dbuf] - 1) & 1, p.timeout_ns, p.status,
                                       abort_flag)) {
                            stop = true;
                            break;
                        }
                        tc_fence_after();
                    }
                    const uint32_t d_t = tmem + kDCol0 + dbuf * NR;
                    const uint32_t a_t = tmem + (i % NA) * kACols;
                    const uint64_t bd = smem_desc_sw128(x_s + (i % S) * NR * 128);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc_mma_ts(d_t, a_t + ks * 8, bd + (uint64_t)(ks * 2), idesc, (first && ks == 0) ? 0u : 1u);
                    if (last) {
                        tc_commit(bar_accfull + 8 * dbuf);
                        ++duse[dbuf];
                        if (p.d_bufs == 2) dbuf ^= 1;
                    }
                    last_i = i;
                    if (++kt == KT) kt = 0;
                }
                // one commit frees the batch's A buffers, one its shared-memory slot
                tc_commit(bar_afree + 8 * ((i0 / kBatch) % (NA / kBatch)));
                tc_commit(bar_empty + 8 * ((i0 % S) / kBatch));
                if (stop) *abort_flag = 1;
            }
            __syncwarp();
            if (*abort_flag) break;
        }
        // tensor memory is released only after every issued MMA has finished
        if (lane == 0 && last_i >= 0) {
            int32_t no_abort = 0;
            mbar_wait(bar_afree + 8 * ((last_i / kBatch) % (NA / kBatch)), (last_i / NA) & 1, p.timeout_ns, p.status,
                      &no_abort);
        }
    } else if (warp < kEpiWarp0) {
        // --------------------------------------------------------------- decode
        const int dw = warp - kDecodeWarp0;
        const int grp = dw >> 2;
        const int quarter = warp & 3;          // tensor-memory lanes this warp may touch
        const int c = quarter * 32 + lane;     // output channel of this thread
        const int dtid = dw * 32 + lane;       // 0..255
        // shared caches: escape offsets/entries of the CTA's records, window bases
        const int nt_span = (int)(nt_last - nt_first + 1);
        const bool base_cached = nt_span <= p.base_tiles;
        for (int i = dtid; i <= nrec; i += 256) esc_off_s[i] = __ldg(p.esc_off + rec_begin + i);
        if (base_cached)
            for (int i = dtid; i < nt_span * w12i::kTileN; i += 256)
                base_s[i] = __ldg(p.base + nt_first * w12i::kTileN + i);
        uint32_t dph = 0;
        auto dec_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_dec);
            const bool ok = mbar_wait(bar_dec, dph, p.timeout_ns, p.status, abort_flag);
            dph ^= 1u;
            return ok;
        };
        bool ok = dec_sync();
        const int32_t e_lo = esc_off_s[0];
        const bool esc_cached = (esc_off_s[nrec] - e_lo) <= p.esc_cap;
        if (ok && esc_cached)
            for (int i = dtid; i < esc_off_s[nrec] - e_lo; i += 256) esc_s[i] = __ldg(p.esc + e_lo + i);
        ok = ok && dec_sync();

        int64_t nt = -1;
        ChanConst cc{0, 0};
        int kt = (int)(rec_begin - nt_first * KT) + grp;
        int64_t ntc = nt_first;
        while (kt >= KT) kt -= KT, ++ntc;
        for (int i = grp; ok && i < nrec; i += 2) {
            if (ntc != nt) {
                nt = ntc;
                const uint32_t b = base_cached ? base_s[(nt - nt_first) * w12i::kTileN + c]
                                               : __ldg(p.base + nt * w12i::kTileN + c);
                cc = chan_const(b);
            }
            const int j = i / kRecsPerStage, ab = i % NA;
            const int s = j % S;
            if (!mbar_wait(bar_full + 8 * s, (j / S) & 1, p.timeout_ns, p.status, abort_flag)) break;
            if (i >= NA && !mbar_wait(bar_afree + 8 * ((i / kBatch) % (NA / kBatch)), ((i / NA) - 1) & 1, p.timeout_ns,
                                      p.status, abort_flag))
                break;
            const uint8_t *rb = smem + pl.rec + (s * kRecsPerStage + i % kRecsPerStage) * w12i::kRecBytes;
            uint4 v[4], nb[2];
#pragma unroll
            for (int g = 0; g < 4; ++g) v[g] = *reinterpret_cast<const uint4 *>(rb + (g * 128 + c) * 16);
#pragma unroll
            for (int h = 0; h < 2; ++h)
                nb[h] = *reinterpret_cast<const uint4 *>(rb + w12i::kViewBytes + (h * 128 + c) * 16);
            uint32_t a[32];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint32_t vw[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
                const uint4 n4 = nb[g >> 1];
                const uint32_t nw[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    decode_word(vw[q], nw[q] >> ((g & 1) * 4), cc, p.mul16, a[8 * g + q], a[8 * g + 4 + q]);
            }
            // escaped slots of this channel: the exact value replaces the filler
            const int32_t e0 = esc_off_s[i] - e_lo, e1 = esc_off_s[i + 1] - e_lo;
            for (int e = e0; e < e1; ++e) {
                const uint32_t en = esc_cached ? esc_s[e] : __ldg(p.esc + e_lo + e);
                const int nl = (en >> 22) & 0x7F;
                if ((nl >> 5) != quarter) continue;              // warp-uniform skip
                const int kl = (en >> 16) & 0x3F, col = kl >> 1;
                const uint32_t val = en & 0xFFFFu;
                const bool mine = nl == c, upper = kl & 1;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (mine && j == col)
                        a[j] = upper ? ((a[j] & 0x0000FFFFu) | (val << 16)) : ((a[j] & 0xFFFF0000u) | val);
            }
            tmem_st_x32(tmem + ((uint32_t)(quarter * 32) << 16) + ab * kACols, a);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_afull + 8 * ab);
                mbar_arrive(bar_empty + 8 * (s / kBatch));
            }
            kt += 2;
            while (kt >= KT) kt -= KT, ++ntc;
        }
    } else {
        // ------------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int c = quarter * 32 + lane;
        const int etid = (warp - kEpiWarp0) * 32 + lane;   // 0..127
        const int ew = warp - kEpiWarp0;
        const int rows = p.R;
        float *red_v = reinterpret_cast<float *>(smem + pl.red);
        int32_t *red_i = reinterpret_cast<int32_t *>(smem + pl.red + 4 * NR * 4);
        uint32_t eph = 0;
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_epi);
            const bool ok = mbar_wait(bar_epi, eph, p.timeout_ns, p.status, abort_flag);
            eph ^= 1u;
            return ok;
        };
        int dbuf = 0;
        uint32_t duse[2] = {0, 0};
        // write (or reduce, for the LM head) 32 rows r0..r0+31 of this channel
        auto emit_rows = [&](int64_t nt, int r0, const float (&v)[32]) {
            if (p.mode == w12i::kModeLinear) {
                uint16_t *yc = p.y + nt * w12i::kTileN + c;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (r0 + j < rows) yc[(int64_t)(r0 + j) * p.ldy] = (uint16_t)(pack_bf16x2(v[j], 0.f) & 0xFFFFu);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (r0 + j >= rows) break;
                    float bv = v[j];
                    int32_t bi = c;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                        const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, off);
                        if (beats(ov, oi, bv, bi)) bv = ov, bi = oi;
                    }
                    if (lane == 0) red_v[ew * NR + r0 + j] = bv, red_i[ew * NR + r0 + j] = bi;
                }
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
            if (!mbar_wait(bar_accfull + 8 * dbuf, duse[dbuf] & 1, p.timeout_ns, p.status, abort_flag)) break;
            tc_fence_after();
            const int64_t t0 = nt * KT, t1 = t0 + KT;
            const bool owned = rec_begin <= t0 && rec_end >= t1;
            const int slot = (nt == nt_first) ? 0 : 1;
            float *mine = p.partial + ((int64_t)(cta * 2 + slot) * NR) * w12i::kTileN;
            const uint32_t d_t = tmem + ((uint32_t)(quarter * 32) << 16) + kDCol0 + dbuf * NR;
            for (int r0 = 0; r0 < NR; r0 += 32) {
                uint32_t raw[32];
                tmem_ld_x32(d_t + r0, raw);
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
            if (lane == 0) mbar_arrive(bar_accempty + 8 * dbuf);
            ++duse[dbuf];
            if (p.d_bufs == 2) dbuf ^= 1;
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
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
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
    const int G = (int)std::min<int64_t>(a.num_sms, T);
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
    // 8 A buffers (four records of slack per decode group) while the two
    // accumulators still fit next to them; otherwise 4
    p.a_bufs = (8 * kACols + 2 * nr <= (int)kTmemCols) ? 8 : 4;
    p.d_bufs = (p.a_bufs * kACols + 2 * nr <= (int)kTmemCols) ? 2 : 1;
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
    int stages = 16;   // a multiple of kBatch, as many as fit
    while (stages > kBatch && plan(stages, nr, p.max_recs, p.esc_cap, p.base_tiles).total > budget) stages -= kBatch;
    p.stages = stages;
    const int smem = plan(stages, nr, p.max_recs, p.esc_cap, p.base_tiles).total;
    if (smem > budget) return (int)cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(k_w12_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
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
    return (int)cudaLaunchKernelEx(&cfg, k_w12_gemm_tc, xmap, p);
}

}  // namespace w12i
