// Host-side W12 packer with its bit-exact self check.
//
// Format: SpecPilot explainer, section 4.1 "W12: a 12-bit lossless weight
// format" -- a 16-binade window per output channel, in-window weights as
// sign + 4-bit exponent offset + 7 mantissa bits, the rest on an escape list
// restored exactly; 12 KB records of 128x64 weights with the 8-bit view in
// the first 8 KB and the low mantissa bits in the last 4 KB.  The byte
// placement inside a record is documented in include/w12.h.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <thread>
#include <vector>

#include "w12.h"
#include "w12_internal.h"

namespace {

constexpr int kTileN = w12i::kTileN;
constexpr int kTileK = w12i::kTileK;
constexpr int kRecBytes = w12i::kRecBytes;
constexpr int kViewBytes = w12i::kViewBytes;

// weight kk (0..15) of a 16-K group sits at this byte of its 16-byte chunk
constexpr int kChunkPos[16] = {0, 1, 4, 5, 8, 9, 12, 13, 2, 3, 6, 7, 10, 11, 14, 15};

inline int exp_field(uint16_t v) { return (v >> 7) & 0xFF; }

// Window base of one channel: the lowest binade b of the 16-binade window
// [b, b+15] that holds the most normal weights; ties go to the larger b; a
// channel without normal weights gets b = 1.
int window_base(const uint16_t *row, int64_t k)
{
    int count[256] = {0};
    bool any = false;
    for (int64_t i = 0; i < k; ++i) {
        const int e = exp_field(row[i]);
        if (e != 0 && e != 255) {
            ++count[e];
            any = true;
        }
    }
    if (!any) return 1;
    // sliding sum over the 16 fields [b, b+15], b = 1 .. 239
    int64_t run = 0;
    for (int e = 1; e <= 16; ++e) run += count[e];
    int64_t best = run;
    int best_b = 1;
    for (int b = 2; b <= 239; ++b) {
        run += count[b + 15] - count[b - 1];
        if (run >= best) {
            best = run;
            best_b = b;
        }
    }
    return best_b;
}

inline bool in_window(uint16_t v, int b)
{
    const int e = exp_field(v);
    return e >= b && e <= b + 15;
}

template <class F>
void parallel_for(int64_t n, F &&fn)
{
    unsigned hw = std::thread::hardware_concurrency();
    int64_t nthreads = std::max<int64_t>(1, std::min<int64_t>(hw ? hw : 1, n));
    if (nthreads == 1) {
        fn(0, n);
        return;
    }
    std::vector<std::thread> pool;
    for (int64_t t = 0; t < nthreads; ++t)
        pool.emplace_back([&, t] { fn(n * t / nthreads, n * (t + 1) / nthreads); });
    for (auto &th : pool) th.join();
}

bool shape_ok(int64_t n, int64_t k) { return n > 0 && k > 0; }
bool shape_supported(int64_t n, int64_t k) { return n % kTileN == 0 && k % kTileK == 0; }

}  // namespace

extern "C" w12_status w12_pack_query(const uint16_t *w_bf16, int64_t n, int64_t k, w12_layout *out)
{
    if (!w_bf16 || !out || !shape_ok(n, k)) return W12_E_INVAL;
    if (!shape_supported(n, k)) return W12_E_UNSUPPORTED;
    std::atomic<int64_t> esc{0};
    parallel_for(n, [&](int64_t lo, int64_t hi) {
        int64_t local = 0;
        for (int64_t r = lo; r < hi; ++r) {
            const uint16_t *row = w_bf16 + r * k;
            const int b = window_base(row, k);
            for (int64_t i = 0; i < k; ++i) local += !in_window(row[i], b);
        }
        esc += local;
    });
    out->n = n;
    out->k = k;
    out->n_tiles = n / kTileN;
    out->k_tiles = k / kTileK;
    out->n_escapes = esc.load();
    out->rec_bytes = static_cast<size_t>(out->n_tiles * out->k_tiles) * kRecBytes;
    out->base_bytes = static_cast<size_t>(n);
    out->esc_off_bytes = static_cast<size_t>(out->n_tiles * out->k_tiles + 1) * 4;
    out->esc_bytes = static_cast<size_t>(out->n_escapes) * 4;
    return W12_OK;
}

extern "C" w12_status w12_pack(const uint16_t *w_bf16, int64_t n, int64_t k, const w12_layout *layout, void *rec,
                               uint8_t *base, int32_t *esc_tile_off, uint32_t *esc)
{
    if (!w_bf16 || !layout || !rec || !base || !esc_tile_off || !shape_ok(n, k)) return W12_E_INVAL;
    if (!shape_supported(n, k)) return W12_E_UNSUPPORTED;
    if (layout->n != n || layout->k != k) return W12_E_INVAL;
    if (layout->n_escapes > 0 && !esc) return W12_E_INVAL;
    const int64_t nt = n / kTileN, kt = k / kTileK, tiles = nt * kt;
    uint8_t *recb = static_cast<uint8_t *>(rec);

    // 1. window bases
    parallel_for(n, [&](int64_t lo, int64_t hi) {
        for (int64_t r = lo; r < hi; ++r) base[r] = static_cast<uint8_t>(window_base(w_bf16 + r * k, k));
    });

    // 2. escape counts per tile -> prefix offsets
    std::vector<int64_t> tile_cnt(static_cast<size_t>(tiles), 0);
    parallel_for(nt, [&](int64_t lo, int64_t hi) {
        for (int64_t a = lo; a < hi; ++a)
            for (int64_t c = 0; c < kTileN; ++c) {
                const int64_t ch = a * kTileN + c;
                const uint16_t *row = w_bf16 + ch * k;
                for (int64_t j = 0; j < k; ++j)
                    if (!in_window(row[j], base[ch])) ++tile_cnt[static_cast<size_t>(a * kt + j / kTileK)];
            }
    });
    int64_t acc = 0;
    for (int64_t t = 0; t < tiles; ++t) {
        esc_tile_off[t] = static_cast<int32_t>(acc);
        acc += tile_cnt[static_cast<size_t>(t)];
    }
    esc_tile_off[tiles] = static_cast<int32_t>(acc);
    if (acc != layout->n_escapes || acc > INT32_MAX) return W12_E_INVAL;

    // 3. records and escape entries, one tile at a time
    parallel_for(tiles, [&](int64_t lo, int64_t hi) {
        for (int64_t t = lo; t < hi; ++t) {
            const int64_t a = t / kt, bk = t % kt;
            uint8_t *r = recb + t * kRecBytes;
            std::memset(r, 0, kRecBytes);
            uint32_t *e = esc ? esc + esc_tile_off[t] : nullptr;
            for (int c = 0; c < kTileN; ++c) {
                const int64_t ch = a * kTileN + c;
                const int b = base[ch];
                const uint16_t *src = w_bf16 + ch * k + bk * kTileK;
                for (int kl = 0; kl < kTileK; ++kl) {
                    const uint16_t v = src[kl];
                    if (!in_window(v, b)) {
                        *e++ = (static_cast<uint32_t>(c) << 22) | (static_cast<uint32_t>(kl) << 16) | v;
                        continue;
                    }
                    const int group = kl >> 4, kk = kl & 15;
                    const uint32_t view = (v & 0x8000u) >> 8 | static_cast<uint32_t>(exp_field(v) - b) << 3 |
                                          ((v >> 4) & 7u);
                    r[(group * kTileN + c) * 16 + kChunkPos[kk]] = static_cast<uint8_t>(view);
                    const int half = kl >> 5, upper = (kl >> 4) & 1;
                    r[kViewBytes + (half * kTileN + c) * 16 + kChunkPos[kk]] |=
                        static_cast<uint8_t>((v & 0xFu) << (upper * 4));
                }
            }
        }
    });

    // 4. self check: decode everything back and compare bit for bit
    std::atomic<int64_t> bad{0};
    parallel_for(tiles, [&](int64_t lo, int64_t hi) {
        int64_t local = 0;
        uint16_t tile[kTileN * kTileK];
        for (int64_t t = lo; t < hi; ++t) {
            const int64_t a = t / kt, bk = t % kt;
            const uint8_t *r = recb + t * kRecBytes;
            for (int c = 0; c < kTileN; ++c) {
                const uint32_t b7 = static_cast<uint32_t>(base[a * kTileN + c]) << 7;
                for (int kl = 0; kl < kTileK; ++kl) {
                    const int group = kl >> 4, kk = kl & 15;
                    const uint32_t view = r[(group * kTileN + c) * 16 + kChunkPos[kk]];
                    const uint32_t nib = (r[kViewBytes + ((kl >> 5) * kTileN + c) * 16 + kChunkPos[kk]] >>
                                          (((kl >> 4) & 1) * 4)) & 0xFu;
                    tile[c * kTileK + kl] =
                        static_cast<uint16_t>(((view & 0x80u) << 8) | (((view & 0x7Fu) << 4) + b7) | nib);
                }
            }
            if (esc)
                for (int32_t i = esc_tile_off[t]; i < esc_tile_off[t + 1]; ++i) {
                    const uint32_t en = esc[i];
                    tile[((en >> 22) & 0x7F) * kTileK + ((en >> 16) & 0x3F)] = static_cast<uint16_t>(en & 0xFFFF);
                }
            for (int c = 0; c < kTileN; ++c) {
                const uint16_t *src = w_bf16 + (a * kTileN + c) * k + bk * kTileK;
                for (int kl = 0; kl < kTileK; ++kl) local += tile[c * kTileK + kl] != src[kl];
            }
        }
        bad += local;
    });
    return bad.load() == 0 ? W12_OK : W12_E_MISMATCH;
}
