// Stream-K W12 verify GEMM and fused LM-head tile argmax (sm_103a).
//
// SpecPilot explainer, section 4.1 "W12 GEMM": 12 KB records (128x64 weights)
// are restored in registers and fed to the tensor cores; a stream-K split of
// the reduction loop in a fixed order keeps the GEMM deterministic.  That
// kernel was written for H100 (wgmma register operands); this one is built
// for GB300:
//   * one persistent CTA per SM; each CTA owns a contiguous run of records in
//     (n-tile, k-tile) order, i.e. a contiguous slice of the packed buffer;
//   * a producer warp streams records with 1-D bulk copies (cp.async.bulk,
//     L2 evict-first) and the matching activation block with a 2-D TMA load
//     (128-byte swizzle, out-of-range rows zero-filled) into an mbarrier ring;
//   * consumer warps decode the records in registers straight into mma.sync
//     A fragments (output channels are M, tree rows are N), patch escapes,
//     and accumulate in FP32;
//   * at a tile's end the consumer warps drop their accumulators in shared
//     memory and go on with the next tile; an epilogue warp writes the tile,
//     or publishes its partial sum when the tile is split between CTAs, and
//     the last CTA to arrive at a split tile sums the partials in CTA order
//     (no waiting, deterministic).  The CTA's last tile, whose end is the
//     launch's critical path, is finished the same way by all consumer
//     threads;
//   * the LM-head epilogue reduces each 128-token tile to (max, index) per row.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <mutex>
#include <type_traits>

#include "w12_device.cuh"

using namespace w12d;

namespace {

struct KParams {
    const uint8_t *rec;
    const uint8_t *base;
    const int32_t *esc_off;
    const uint32_t *esc;
    int32_t n_tiles, k_tiles, R, mode;
    uint16_t *y;
    int64_t ldy;
    float *s1_val;
    int32_t *s1_idx;
    float *partial;
    int32_t *counters;
    int32_t *status;
    uint32_t mul16;
    int32_t debug_flags;
    uint64_t timeout_ns;
    int32_t stages;
    int32_t max_recs;       // records of the largest CTA share
    int32_t esc_cap;        // escape entries that fit the shared cache
    int32_t base_tiles;     // n-tiles whose window bases fit the shared cache
};

// QV: the quick pass (only the 8 KB view plane of each record is read; the
// low mantissa bits of in-window weights are taken as the midpoint 0b1000)
template <int NB8, int WK, int RPS, bool QV = false, int MB = 2>
struct Cfg {
    static constexpr int kRecStride = QV ? w12i::kViewBytes : w12i::kRecBytes;   // bytes kept per record
    static constexpr int kRows = NB8 * 8;                     // rows per activation block
    static constexpr int kXBytes = kRows * 128;               // activation block: rows x 64 BF16
    static constexpr int kWarpsN = 8 / MB;                    // consumer warps across the 128 channels (16 * MB each)
    static constexpr int kConsumerWarps = kWarpsN * WK;
    static constexpr int kConsumers = kConsumerWarps * 32;
    static constexpr int kProducerWarp = kConsumerWarps;
    static constexpr int kEpilogueWarp = kConsumerWarps + 1;
    static constexpr int kThreads = kConsumers + 64;          // + producer and epilogue warps
    static constexpr int kKgPerWarp = 4 / WK;                 // 16-K groups per consumer warp
    static constexpr int kRedStride = 132;                    // padded row stride of the reduction tile
    static constexpr int kRedBytes = WK * kRows * kRedStride * 4;
};

struct SmemPlan {
    int rec_off, x_off, red_off, bar_off, flag_off, escoff_off, esc_off, emask_off, base_off, total;
};

template <int NB8, int WK, int RPS, bool QV, int MB>
__host__ __device__ inline SmemPlan smem_plan(int stages, int max_recs, int esc_cap, int base_tiles)
{
    using C = Cfg<NB8, WK, RPS, QV, MB>;
    SmemPlan s;
    int o = 0;
    s.rec_off = o;
    o += stages * RPS * C::kRecStride;
    s.x_off = o;
    o += stages * RPS * C::kXBytes;
    s.red_off = o;
    o += C::kRedBytes;
    s.bar_off = o;
    o += 2 * stages * 8 + 24;
    s.flag_off = o;
    o += 16;
    s.escoff_off = o;
    o += ((max_recs + 1) * 4 + 15) / 16 * 16;
    s.esc_off = o;
    o += esc_cap * 4;
    s.emask_off = o;
    o += (max_recs * 2 + 15) / 16 * 16;
    s.base_off = o;
    o += base_tiles * w12i::kTileN;
    s.total = o + 1024;   // slack to align the window to 1024 bytes at run time
    return s;
}

__device__ __forceinline__ int cta_of_record(int64_t r, int G, int64_t T) { return (int)(((r + 1) * G - 1) / T); }
__device__ __forceinline__ int64_t first_record(int c, int G, int64_t T) { return (int64_t)c * T / G; }

template <int NB8, int WK, int RPS, bool QV, int MB>
__global__ void __launch_bounds__(Cfg<NB8, WK, RPS, QV, MB>::kThreads, 1)
    k_w12_gemm(const __grid_constant__ CUtensorMap xmap, const KParams p)
{
    using C = Cfg<NB8, WK, RPS, QV, MB>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte swizzle of the activation blocks needs 1024-byte alignment
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const SmemPlan sp = smem_plan<NB8, WK, RPS, QV, MB>(p.stages, p.max_recs, p.esc_cap, p.base_tiles);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int KT = p.k_tiles;
    const int64_t T = (int64_t)p.n_tiles * KT;
    const int64_t rec_begin = first_record(cta, G, T), rec_end = first_record(cta + 1, G, T);
    const int nrec = (int)(rec_end - rec_begin);
    const int S = p.stages;

    const uint32_t rec_s = smem_u32(smem + sp.rec_off);
    const uint32_t x_s = smem_u32(smem + sp.x_off);
    float *red = reinterpret_cast<float *>(smem + sp.red_off);
    const uint32_t bar_full = smem_u32(smem + sp.bar_off);
    const uint32_t bar_empty = bar_full + 8 * S;
    const uint32_t bar_cons = bar_empty + 8 * S;
    const uint32_t bar_red_full = bar_cons + 8;    // the consumers' accumulators are in red
    const uint32_t bar_red_empty = bar_cons + 16;  // the epilogue has read them
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + sp.flag_off);
    int32_t *last_flag = reinterpret_cast<int32_t *>(smem + sp.flag_off + 4);
    int32_t *esc_off_s = reinterpret_cast<int32_t *>(smem + sp.escoff_off);
    uint32_t *esc_s = reinterpret_cast<uint32_t *>(smem + sp.esc_off);
    uint16_t *emask_s = reinterpret_cast<uint16_t *>(smem + sp.emask_off);
    uint8_t *base_s = smem + sp.base_off;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, C::kConsumerWarps);
        }
        mbar_init(bar_cons, C::kConsumerWarps);   // one arrival per consumer warp
        mbar_init(bar_red_full, C::kConsumerWarps);
        mbar_init(bar_red_empty, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == C::kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&xmap);
            const uint64_t pol = policy_evict_first();
            const bool drop_first = (p.debug_flags & 1) && cta == 0;
            const int nst = (nrec + RPS - 1) / RPS;
            auto recs_in = [&](int j) { return min(RPS, nrec - j * RPS); };
            auto issue_w = [&](int j, int sl) {
                const int n = recs_in(j);
                mbar_expect_tx(bar_full + 8 * sl, (uint32_t)n * (C::kRecStride + C::kXBytes));
                if (!(drop_first && j == 0)) {
                    if constexpr (QV) {
                        // the view plane of each record: its first 8 KB
                        for (int r = 0; r < n; ++r)
                            bulk_g2s(rec_s + (sl * RPS + r) * C::kRecStride,
                                     p.rec + (rec_begin + j * RPS + r) * (int64_t)w12i::kRecBytes,
                                     (uint32_t)w12i::kViewBytes, bar_full + 8 * sl, pol);
                    } else {
                        bulk_g2s(rec_s + sl * RPS * w12i::kRecBytes,
                                 p.rec + (rec_begin + j * RPS) * (int64_t)w12i::kRecBytes, (uint32_t)n * w12i::kRecBytes,
                                 bar_full + 8 * sl, pol);
                    }
                }
            };
            auto issue_x = [&](int j, int sl) {
                if (drop_first && j == 0) return;
                for (int r = 0; r < recs_in(j); ++r)
                    tma_load_2d(x_s + (sl * RPS + r) * C::kXBytes, &xmap,
                                (int)((rec_begin + j * RPS + r) % KT) * w12i::kTileK, 0, bar_full + 8 * sl);
            };
            const int pre = min(S, nst);
            // weights do not depend on earlier kernels: start them before the
            // programmatic-dependency wait
            for (int j = 0; j < pre; ++j) issue_w(j, j);
            pdl_wait();
            for (int j = 0; j < pre; ++j) issue_x(j, j);
            int issued = pre;
            int sl = pre % S;
            uint32_t use = pre / S;                 // how many times stage sl has been filled
            for (int j = pre; j < nst; ++j) {
                if (!mbar_wait(bar_empty + 8 * sl, (use - 1) & 1, p.timeout_ns, p.status, abort_flag)) break;
                issue_w(j, sl);
                issue_x(j, sl);
                issued = j + 1;
                if (++sl == S) sl = 0, ++use;
            }
            if (*abort_flag) {
                // leave no copy in flight: wait (bounded, ignoring the abort
                // flag) for the last use of every stage that was issued
                int32_t dummy_abort = 0;
                for (int j = max(0, issued - S); j < issued; ++j) {
                    if (drop_first && j == 0) continue;
                    mbar_wait(bar_full + 8 * (j % S), (j / S) & 1, p.timeout_ns, p.status, &dummy_abort);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------- finishing a tile
    // Tile nt from the K-slice sums in red, by the nthr threads tid = 0 ..
    // nthr - 1 (whole warps): written when this CTA holds all of its records;
    // else this CTA's partial sum is published (slot 0 for the CTA's first
    // tile, 1 for its last) and the last of the tile's contributors to arrive
    // sums every partial in CTA order and writes the result.  red_read() runs
    // as soon as red has been read; sync() is a barrier over the threads
    // (false: aborted); *flag is a shared word for the last-arrival decision.
    const int64_t nt_first = rec_begin / KT;
    auto finish_tile = [&](int64_t nt, int tid, int nthr, auto &&sync, auto &&red_read, int32_t *flag) -> bool {
        const int rows = min(p.R, C::kRows);
        const int wi = tid >> 5, nw = nthr >> 5;
        auto from_red = [&](int row, int c4) {
            float4 v = *reinterpret_cast<const float4 *>(red + row * C::kRedStride + c4);
#pragma unroll
            for (int sl = 1; sl < WK; ++sl) {
                const float4 w = *reinterpret_cast<const float4 *>(red + (sl * C::kRows + row) * C::kRedStride + c4);
                v.x += w.x, v.y += w.y, v.z += w.z, v.w += w.w;
            }
            return v;
        };
        // BF16 (round to nearest even) rows of 128 channels, or per row the
        // (max, lowest index) over the tile's 128 tokens (a warp reduces four
        // of its rows side by side); get(row, c4) gives 4 channels from c4
        auto emit = [&](auto &&get) {
            if (p.mode == w12i::kModeLinear) {
#pragma unroll 4
                for (int e = tid; e < rows * 32; e += nthr) {
                    const int row = e >> 5, c4 = (e & 31) * 4;
                    const float4 v = get(row, c4);
                    uint2 packed;
                    packed.x = pack_bf16x2(v.x, v.y);
                    packed.y = pack_bf16x2(v.z, v.w);
                    *reinterpret_cast<uint2 *>(p.y + row * p.ldy + nt * w12i::kTileN + c4) = packed;
                }
                return;
            }
            constexpr int kU = 4;
            const int lane = tid & 31;
            for (int r0 = wi; r0 < rows; r0 += kU * nw) {
                float bv[kU];
                int32_t bi[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    bv[u] = __int_as_float(0x7fc00000);
                    bi[u] = 0x7fffffff;
                    const int row = r0 + u * nw;
                    if (row < rows) {
                        const float4 v = get(row, lane * 4);
                        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (beats(vv[q], lane * 4 + q, bv[u], bi[u])) bv[u] = vv[q], bi[u] = lane * 4 + q;
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bv[u], off);
                        const int32_t oi = __shfl_xor_sync(0xffffffffu, bi[u], off);
                        if (beats(ov, oi, bv[u], bi[u])) bv[u] = ov, bi[u] = oi;
                    }
                if (lane == 0) {
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int row = r0 + u * nw;
                        if (row < rows) {
                            p.s1_val[(int64_t)row * p.n_tiles + nt] = bv[u];
                            p.s1_idx[(int64_t)row * p.n_tiles + nt] = (bi[u] == 0x7fffffff)
                                                                          ? (int32_t)(nt * w12i::kTileN)
                                                                          : (int32_t)(nt * w12i::kTileN + bi[u]);
                        }
                    }
                }
            }
        };

        const int64_t t0 = nt * KT, t1 = t0 + KT;
        if (rec_begin <= t0 && rec_end >= t1) {
            emit(from_red);
            red_read();
            return sync();
        }
        float *mine = p.partial + ((int64_t)(cta * 2 + (nt == nt_first ? 0 : 1)) * C::kRows) * w12i::kTileN;
        for (int e = tid; e < rows * 32; e += nthr) {
            const int row = e >> 5, c4 = (e & 31) * 4;
            __stcg(reinterpret_cast<float4 *>(mine + row * w12i::kTileN + c4), from_red(row, c4));
        }
        red_read();
        __threadfence();
        if (!sync()) return false;
        const int c_first = cta_of_record(t0, G, T), c_last = cta_of_record(t1 - 1, G, T);
        if (tid == 0) *flag = (atomicAdd(p.counters + nt, 1) == c_last - c_first);
        if (!sync()) return false;
        if (*reinterpret_cast<volatile int32_t *>(flag) == 0) return true;
        __threadfence();
        // Every contributor after the first starts inside this tile (its slot
        // 0); the first one's slot depends on where it starts.
        const int sl_first = (first_record(c_first, G, T) >= t0) ? 0 : 1;
        const float *part0 = p.partial + (int64_t)(c_first * 2 + sl_first) * C::kRows * w12i::kTileN;
        const float *part1 = p.partial + (int64_t)((c_first + 1) * 2) * C::kRows * w12i::kTileN;
        constexpr int64_t kSlot2 = 2 * (int64_t)C::kRows * w12i::kTileN;   // floats between CTAs' slot 0
        const int n_later = c_last - c_first;
        emit([&](int row, int c4) {
            const int off = row * w12i::kTileN + c4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 w0 = __ldcg(reinterpret_cast<const float4 *>(part0 + off));
            v.x += w0.x, v.y += w0.y, v.z += w0.z, v.w += w0.w;
            for (int c = 0; c < n_later; ++c) {
                const float4 w = __ldcg(reinterpret_cast<const float4 *>(part1 + c * kSlot2 + off));
                v.x += w.x, v.y += w.y, v.z += w.z, v.w += w.w;
            }
            return v;
        });
        if (tid == 0) p.counters[nt] = 0;   // ready for the next launch using this slot
        return sync();
    };

    if (warp == C::kEpilogueWarp) {
        // ------------------------------------------------------------ epilogue
        // The tiles the consumers hand over (all of this CTA's but the last),
        // in order.  red goes back to the consumers as soon as it has been read.
        const int64_t nt_last = (rec_end - 1) / KT;
        int32_t *eflag = last_flag + 1;
        auto wsync = [&]() -> bool {
            __syncwarp();
            return true;
        };
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_red_empty);
        };
        uint32_t ph = 0;
        for (int64_t nt = nt_first; nt < nt_last; ++nt) {
            const bool ok = mbar_wait(bar_red_full, ph, p.timeout_ns, p.status, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) return;
            ph ^= 1u;
            if (!finish_tile(nt, lane, 32, wsync, release, eflag)) return;
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp;                 // consumer warp 0 .. kConsumerWarps-1
    constexpr int kWarpsN = C::kWarpsN;
    const int mw = cw % kWarpsN, wk = cw / kWarpsN;
    const int g = lane >> 2, t = lane & 3;
    const int ctid = threadIdx.x;        // 0 .. kConsumers-1

    uint32_t cons_phase0 = 0;
    auto cons_sync0 = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cons);
        const bool ok = mbar_wait(bar_cons, cons_phase0, p.timeout_ns, p.status, abort_flag);
        cons_phase0 ^= 1u;
        return ok;
    };
    // shared caches: escape offsets/entries of this CTA's records, window bases
    const int nt_span = (int)((rec_end - 1) / KT - nt_first + 1);
    const bool base_cached = nt_span <= p.base_tiles;
    for (int i = ctid; i <= nrec; i += C::kConsumers) esc_off_s[i] = __ldg(p.esc_off + rec_begin + i);
    if (base_cached)
        for (int i = ctid; i < nt_span * w12i::kTileN; i += C::kConsumers)
            base_s[i] = __ldg(p.base + nt_first * w12i::kTileN + i);
    if (!cons_sync0()) return;
    const int32_t e_lo = esc_off_s[0];
    const bool esc_cached = (esc_off_s[nrec] - e_lo) <= p.esc_cap;
    if (esc_cached)
        for (int i = ctid; i < esc_off_s[nrec] - e_lo; i += C::kConsumers) esc_s[i] = __ldg(p.esc + e_lo + i);
    // per record, a bit for every consumer warp whose part of the record
    // holds an escape: the record loop skips the escape list without reading it
    static_assert(C::kConsumerWarps <= 16, "one 16-bit mask per record");
    for (int i = ctid; i < nrec; i += C::kConsumers) {
        uint32_t m = 0;
        for (int e = esc_off_s[i]; e < esc_off_s[i + 1]; ++e) {
            const uint32_t en = __ldg(p.esc + e);
            const int nl = (en >> 22) & 0x7F, kg = ((en >> 16) & 0x3F) >> 4;
            m |= 1u << (nl / (16 * MB) + kWarpsN * (kg / C::kKgPerWarp));
        }
        emask_s[i] = (uint16_t)m;
    }
    if (!cons_sync0()) return;

    float acc[MB][NB8][4];
    ChanConst cc[MB][2];
    int64_t cur_nt = -1;
    uint32_t cons_phase = cons_phase0;
    // barrier over the consumer threads with a bounded wait; false = aborted
    auto cons_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cons);
        const bool ok = mbar_wait(bar_cons, cons_phase, p.timeout_ns, p.status, abort_flag);
        cons_phase ^= 1u;
        return ok;
    };

    auto load_consts = [&](int64_t nt) {
#pragma unroll
        for (int mb = 0; mb < MB; ++mb)
#pragma unroll
            for (int hi = 0; hi < 2; ++hi) {
                const int ch = mw * 16 * MB + mb * 16 + hi * 8 + g;
                const uint32_t b = base_cached ? base_s[(nt - nt_first) * w12i::kTileN + ch]
                                               : __ldg(p.base + nt * w12i::kTileN + ch);
                cc[mb][hi] = chan_const(b);
            }
#pragma unroll
        for (int mb = 0; mb < MB; ++mb)
#pragma unroll
            for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[mb][nb][q] = 0.f;
    };

    // End of tile nt.  In the record loop the warps drop their accumulators
    // into red (once the epilogue warp has read the previous ones), hand the
    // tile to the epilogue warp and go on; the CTA's last tile, whose end is
    // the critical path, is finished by all consumer threads.
    uint32_t n_handed = 0;   // tiles handed to the epilogue warp
    auto drop_acc = [&]() -> bool {
        if (*abort_flag) return false;
        if (n_handed > 0 && !mbar_try_wait(bar_red_empty, (n_handed - 1) & 1u) &&
            !mbar_wait(bar_red_empty, (n_handed - 1) & 1u, p.timeout_ns, p.status, abort_flag))
            return false;
        // red[wk][row][ch]
#pragma unroll
        for (int mb = 0; mb < MB; ++mb)
#pragma unroll
            for (int nb = 0; nb < NB8; ++nb) {
                const int ch = mw * 16 * MB + mb * 16 + g;
                const int row = nb * 8 + 2 * t;
                float *rb = red + (wk * C::kRows) * C::kRedStride;
                rb[row * C::kRedStride + ch] = acc[mb][nb][0];
                rb[(row + 1) * C::kRedStride + ch] = acc[mb][nb][1];
                rb[row * C::kRedStride + ch + 8] = acc[mb][nb][2];
                rb[(row + 1) * C::kRedStride + ch + 8] = acc[mb][nb][3];
            }
        return true;
    };
    auto flush = [&](int64_t) -> bool {
        if (!drop_acc()) return false;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_red_full);
        ++n_handed;
        return true;
    };
    auto flush_last = [&](int64_t nt) -> bool {
        if (!drop_acc() || !cons_sync()) return false;
        return finish_tile(nt, ctid, C::kConsumers, cons_sync, [] {}, last_flag);
    };

    int64_t nt = nt_first;
    int kt = (int)(rec_begin - nt_first * KT);
    int s = 0;
    uint32_t full_phase = 0;
    // Per-thread parts of every shared-memory address, hoisted out of the
    // record loop; what varies inside it is a compile-time offset.
    //   view word (kg, mb, hi): thread base + kg*2048 + mb*256 + hi*128
    //   nibble word:            thread base + 8192 + (kg/2)*2048 + mb*256 + hi*128
    const uint8_t *rec_thread = smem + sp.rec_off + (mw * 16 * MB + g) * 16 + 4 * t;
    uint32_t x_thread[C::kKgPerWarp];
#pragma unroll
    for (int kgl = 0; kgl < C::kKgPerWarp; ++kgl) {
        const int kg = wk * C::kKgPerWarp + kgl;
        if constexpr (NB8 == 1) {
            const int chunk = 2 * kg + ((lane >> 3) & 1);
            x_thread[kgl] = (lane & 7) * 128 + ((chunk ^ (lane & 7)) << 4);
        } else {
            const int q = lane >> 3, chunk = 2 * kg + (q & 1);
            x_thread[kgl] = ((q >> 1) * 8 + (lane & 7)) * 128 + ((chunk ^ (lane & 7)) << 4);
        }
    }
    using Frag = uint32_t[MB][C::kKgPerWarp][4];
    // decode this warp's 16 * MB channels x (16 * kKgPerWarp) K of one record
    auto decode_rec = [&](const uint32_t *rw, Frag &fa) {
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
            uint32_t nib_lo = 0, nib_hi = 0;
#pragma unroll
            for (int kgl = 0; kgl < C::kKgPerWarp; ++kgl) {
                const int kg = wk * C::kKgPerWarp + kgl;
                if constexpr (QV) {
                    nib_lo = nib_hi = 0x88888888u;   // every low mantissa nibble = 0b1000
                } else if (kgl == 0 || (kg & 1) == 0) {
                    nib_lo = rw[(w12i::kViewBytes + (kg >> 1) * 2048 + mb * 256) / 4];
                    nib_hi = rw[(w12i::kViewBytes + (kg >> 1) * 2048 + mb * 256 + 128) / 4];
                }
                const uint32_t sh = (kg & 1) * 4;
                const uint32_t v_lo = rw[(kg * 2048 + mb * 256) / 4];
                const uint32_t v_hi = rw[(kg * 2048 + mb * 256 + 128) / 4];
                decode_word(v_lo, nib_lo >> sh, cc[mb][0], p.mul16, fa[mb][kgl][0], fa[mb][kgl][2]);
                decode_word(v_hi, nib_hi >> sh, cc[mb][1], p.mul16, fa[mb][kgl][1], fa[mb][kgl][3]);
            }
        }
    };
    // escaped slots of record i: the warp reads up to 32 entries at once,
    // keeps the ones inside its 16 * MB channels x (16 * kKgPerWarp) K, and the
    // owning lane replaces the filler by the exact value
    auto patch_rec = [&](int i, Frag &fa, bool has) {
        if (!has) return;
        const int32_t e0 = esc_off_s[i] - e_lo, e1 = esc_off_s[i + 1] - e_lo;
        for (int eb = e0; eb < e1; eb += 32) {
            const int e = eb + lane;
            uint32_t en = 0;
            bool own = false;
            if (e < e1) {
                en = esc_cached ? esc_s[e] : __ldg(p.esc + e_lo + e);
                const int nl = (en >> 22) & 0x7F, kg = ((en >> 16) & 0x3F) >> 4;
                own = nl / (16 * MB) == mw && (kg / C::kKgPerWarp) == wk;
            }
            uint32_t mine = __ballot_sync(0xffffffffu, own);
            while (mine) {
                const int src = __ffs(mine) - 1;
                mine &= mine - 1;
                const uint32_t ent = __shfl_sync(0xffffffffu, en, src);
                const int nl = (ent >> 22) & 0x7F, kl = (ent >> 16) & 0x3F;
                const int kk = kl & 15;
                if (lane != ((nl & 7) * 4 + ((kk & 7) >> 1))) continue;
                const int mb_e = (nl >> 4) % MB, kgl_e = (kl >> 4) % C::kKgPerWarp;
                const int j_e = (kk >> 3) * 2 + ((nl >> 3) & 1);
                // fa[mb][kgl][j] as one array of MB * kKgPerWarp * 4 registers
                patch_half(reinterpret_cast<uint32_t(&)[MB * C::kKgPerWarp * 4]>(fa),
                           (mb_e * C::kKgPerWarp + kgl_e) * 4 + j_e, ent & 0xFFFFu, kk & 1);
            }
        }
    };
    // activations (B operand) from the swizzled TMA block, then MMA
    auto mma_rec = [&](uint32_t xb, const Frag &fa) {
#pragma unroll
        for (int kgl = 0; kgl < C::kKgPerWarp; ++kgl) {
            const uint32_t xa = xb + x_thread[kgl];
            if constexpr (NB8 == 1) {
                uint32_t b0, b1;
                ldsm_x2(xa, b0, b1);
#pragma unroll
                for (int mb = 0; mb < MB; ++mb) mma_bf16_16816(acc[mb][0], fa[mb][kgl], b0, b1);
            } else {
                uint32_t b[NB8][2];
                ldsm_x4_off<0>(xa, b[0][0], b[0][1], b[1][0], b[1][1]);
                if constexpr (NB8 >= 4) ldsm_x4_off<2048>(xa, b[2][0], b[2][1], b[3][0], b[3][1]);
                if constexpr (NB8 >= 8) {
                    ldsm_x4_off<4096>(xa, b[4][0], b[4][1], b[5][0], b[5][1]);
                    ldsm_x4_off<6144>(xa, b[6][0], b[6][1], b[7][0], b[7][1]);
                }
#pragma unroll
                for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb) mma_bf16_16816(acc[mb][nb], fa[mb][kgl], b[nb][0], b[nb][1]);
            }
        }
    };
    auto rec_words = [&](int q) {
        return reinterpret_cast<const uint32_t *>(rec_thread + (s * RPS + q) * C::kRecStride);
    };
    auto rec_x = [&](int q) { return x_s + (s * RPS + q) * C::kXBytes; };

    for (int i = 0; i < nrec;) {
        // escape bits of the stage's records (bit 16 * r + cw: record i + r)
        using EscBits = std::conditional_t<(RPS > 2), uint64_t, uint32_t>;
        EscBits em = 0;
#pragma unroll
        for (int r = 0; r < RPS; ++r)
            if (i + r < nrec) em |= (EscBits)emask_s[i + r] << (16 * r);
        if (!mbar_try_wait(bar_full + 8 * s, full_phase) &&
            !mbar_wait(bar_full + 8 * s, full_phase, p.timeout_ns, p.status, abort_flag))
            return;
        int q = 0;
        while (q < RPS && i < nrec) {
            if (nt != cur_nt) {
                if (cur_nt >= 0 && !flush(cur_nt)) return;
                cur_nt = nt;
                load_consts(nt);
            }
            // two records of the stage in this tile: interleave them (with two
            // records a stage, only as its first and second)
            if (RPS >= 2 && (RPS == 2 ? q == 0 : q + 1 < RPS) && i + 1 < nrec && kt + 1 < KT) {
                const int q0 = RPS == 2 ? 0 : q;
                Frag f0, f1;
                decode_rec(rec_words(q0), f0);
                decode_rec(rec_words(q0 + 1), f1);
                patch_rec(i, f0, (uint32_t)(em >> (16 * q0 + cw)) & 1u);
                patch_rec(i + 1, f1, (uint32_t)(em >> (16 * (q0 + 1) + cw)) & 1u);
                mma_rec(rec_x(q0), f0);
                mma_rec(rec_x(q0 + 1), f1);
                q += 2, i += 2, kt += 2;
                if (kt == KT) kt = 0, ++nt;
            } else {
                Frag f0;
                decode_rec(rec_words(q), f0);
                patch_rec(i, f0, (uint32_t)(em >> (16 * q + cw)) & 1u);
                mma_rec(rec_x(q), f0);
                ++q, ++i;
                if (++kt == KT) kt = 0, ++nt;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        if (++s == S) s = 0, full_phase ^= 1u;
    }
    if (cur_nt >= 0) flush_last(cur_nt);
}

// second stage of the LM-head argmax: one CTA per row, fixed-order reduction
__global__ void __launch_bounds__(256) k_argmax_stage2(const float *s1_val, const int32_t *s1_idx, int32_t n_tiles,
                                                       int32_t *argmax, float *maxlogit)
{
    pdl_wait();
    const int row = blockIdx.x;
    float bv = __int_as_float(0x7fc00000);
    int32_t bi = 0x7fffffff;
    for (int i = threadIdx.x; i < n_tiles; i += blockDim.x) {
        const float v = s1_val[(int64_t)row * n_tiles + i];
        const int32_t ix = s1_idx[(int64_t)row * n_tiles + i];
        if (beats(v, ix, bv, bi)) bv = v, bi = ix;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (beats(ov, oi, bv, bi)) bv = ov, bi = oi;
    }
    __shared__ float sv[8];
    __shared__ int32_t si[8];
    if ((threadIdx.x & 31) == 0) sv[threadIdx.x >> 5] = bv, si[threadIdx.x >> 5] = bi;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            if (beats(sv[w], si[w], bv, bi)) bv = sv[w], bi = si[w];
        argmax[row] = (bi == 0x7fffffff) ? 0 : bi;
        if (maxlogit) maxlogit[row] = bv;
    }
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

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

template <int NB8, int WK, int RPS, bool QV = false, int MB = 2>
int launch_t(const w12i::GemmArgs &a, const CUtensorMap &xmap, cudaStream_t st)
{
    using C = Cfg<NB8, WK, RPS, QV, MB>;
    const int64_t T = (int64_t)a.w.n_tiles * a.w.k_tiles;
    const int G = (int)std::min<int64_t>(a.num_sms, T);
    const int max_recs = (int)((T + G - 1) / G);
    KParams p{};
    p.rec = a.w.rec;
    p.base = a.w.base;
    p.esc_off = a.w.esc_off;
    p.esc = a.w.esc;
    p.n_tiles = a.w.n_tiles;
    p.k_tiles = a.w.k_tiles;
    p.R = a.R;
    p.mode = a.mode;
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
    p.max_recs = max_recs;
    p.esc_cap = 2048;
    p.base_tiles = std::min<int>(64, (int)(max_recs / a.w.k_tiles + 2));
    const int budget = 227 * 1024;
    int stages = 8;
    while (stages > 2 && smem_plan<NB8, WK, RPS, QV, MB>(stages, max_recs, p.esc_cap, p.base_tiles).total > budget)
        --stages;
    p.stages = stages;
    const int smem = smem_plan<NB8, WK, RPS, QV, MB>(stages, max_recs, p.esc_cap, p.base_tiles).total;
    if (smem > budget) return (int)cudaErrorInvalidConfiguration;
    cudaError_t e =
        cudaFuncSetAttribute(k_w12_gemm<NB8, WK, RPS, QV, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, k_w12_gemm<NB8, WK, RPS, QV, MB>);
    if (e != cudaSuccess) return (int)e;
    if (fa.maxThreadsPerBlock < C::kThreads) return (int)cudaErrorLaunchOutOfResources;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return (int)cudaLaunchKernelEx(&cfg, k_w12_gemm<NB8, WK, RPS, QV, MB>, xmap, p);
}

}  // namespace

namespace w12i {

int launch_gemm(const GemmArgs &a, void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    EncodeTiledFn enc = encode_fn();
    if (!enc) return (int)cudaErrorNotSupported;
    int nb8 = (a.R + 7) / 8;
    nb8 = nb8 <= 1 ? 1 : nb8 <= 2 ? 2 : nb8 <= 4 ? 4 : 8;
    CUtensorMap xmap;
    const cuuint64_t dims[2] = {(cuuint64_t)a.w.k, (cuuint64_t)a.R};
    const cuuint64_t strides[1] = {(cuuint64_t)a.w.k * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)(nb8 * 8)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a.x), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
    // Two 16-K groups of consumer warps, 16 warps of 16 channels: more warps
    // hide the decode chain's latency, and the four on a scheduler overlap one
    // another's decode and MMAs (the register cap of 576 threads still fits
    // every row count).  Records per stage: four up to 16 rows (one wait and
    // one release per 48 KB: at these row counts the per-stage work is a large
    // part of a record's), two at 17-32 rows (with 32-row activation blocks
    // four would leave fewer records in flight), one at 64 rows.
    if (a.qview) {
        switch (nb8) {
        case 1: return launch_t<1, 2, 2, true, 1>(a, xmap, st);
        case 2: return launch_t<2, 2, 2, true, 1>(a, xmap, st);
        case 4: return launch_t<4, 2, 2, true, 1>(a, xmap, st);
        default: return launch_t<8, 2, 1, true, 1>(a, xmap, st);
        }
    }
    switch (nb8) {
    case 1: return launch_t<1, 2, 4, false, 1>(a, xmap, st);
    case 2: return launch_t<2, 2, 4, false, 1>(a, xmap, st);
    case 4: return launch_t<4, 2, 2, false, 1>(a, xmap, st);
    default: return launch_t<8, 2, 1, false, 1>(a, xmap, st);
    }
}

// ---------------------------------------------------------------------------
// Scratch of the allocation-free GEMM entry point (w12_gemm_static_scratch).
//
// Some callers cannot allocate device memory at the point where they run the
// GEMM (code inside a CUDA stream capture, hosts that hand out no device
// allocations to plugins, processes that must keep a fixed footprint).  For
// them the split-tile partial sums, the tile arrival counters and a status
// word live in this file-scope array instead of a caller workspace.  Every
// GPU that loads the library keeps it (about 4.1 MiB) until the process exits.
// Limits: R <= kStaticMaxRows rows, at most kStaticMaxTiles output tiles of
// 128 channels, at most kStaticMaxCtas CTAs.
// ---------------------------------------------------------------------------
constexpr int kStaticMaxRows = 16;
constexpr int kStaticMaxCtas = 256;
constexpr int kStaticMaxTiles = 16384;
constexpr size_t kStaticStatusBytes = 256;
constexpr size_t kStaticCounterBytes = (size_t)kStaticMaxTiles * 4;
constexpr size_t kStaticPartialBytes = (size_t)kStaticMaxCtas * 2 * kStaticMaxRows * kTileN * 4;
constexpr size_t kStaticScratchBytes = kStaticStatusBytes + kStaticCounterBytes + kStaticPartialBytes;

}  // namespace w12i

static __device__ __align__(256) unsigned char g_static_scratch[w12i::kStaticScratchBytes];

namespace w12i {

// Device address of g_static_scratch on the current device, looked up once per
// device (with that device current) and cached.  A host-side name of a
// __device__ array is not a device address, so it is never passed directly.
static int static_scratch_on_current_device(unsigned char **out)
{
    static std::mutex mu;
    static unsigned char *cache[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= 128) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return (int)e;
        cache[dev] = static_cast<unsigned char *>(p);
    }
    *out = cache[dev];
    return 0;
}

int static_scratch_limits(int32_t *max_rows, int32_t *max_tiles)
{
    *max_rows = kStaticMaxRows;
    *max_tiles = kStaticMaxTiles;
    return 0;
}

int launch_gemm_static_scratch(const GemmArgs &in, void *stream)
{
    if (in.R < 1 || in.R > kStaticMaxRows || in.w.n_tiles > kStaticMaxTiles) return (int)cudaErrorInvalidValue;
    unsigned char *base = nullptr;
    if (int e = static_scratch_on_current_device(&base)) return e;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    GemmArgs a = in;
    // a device with more SMs than the array has partial slots for runs a
    // smaller grid (the split points follow the grid, so the result is that
    // of w12_gemm on a device of kStaticMaxCtas SMs)
    a.num_sms = std::min(in.num_sms, kStaticMaxCtas);
    a.status = reinterpret_cast<int32_t *>(base);
    a.counters = reinterpret_cast<int32_t *>(base + kStaticStatusBytes);
    a.partial = reinterpret_cast<float *>(base + kStaticStatusBytes + kStaticCounterBytes);
    // the status word and the arrival counters of this call start at zero
    cudaError_t e = cudaMemsetAsync(base, 0, kStaticStatusBytes + (size_t)a.w.n_tiles * 4, st);
    if (e != cudaSuccess) return (int)e;
    return launch_gemm(a, stream);
}

int launch_argmax_stage2(const float *s1_val, const int32_t *s1_idx, int32_t R, int32_t n_tiles, int32_t *argmax,
                         float *maxlogit, bool pdl, void *stream)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(R);
    cfg.blockDim = dim3(256);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return (int)cudaLaunchKernelEx(&cfg, k_argmax_stage2, s1_val, s1_idx, n_tiles, argmax, maxlogit);
}

}  // namespace w12i
