// C ABI of the W12 tree-verify library: argument validation (before any
// launch), workspace layout and the sequencing of the CUDA kernels.
//
// Typed refusal before anything runs follows the poot-llm speculative
// decoding docs ("What is refused": a typed error before anything compiles or
// uploads).  Everything that touches data on the device is a kernel of this
// library; nothing here computes on the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <vector>

#include "w12.h"
#include "w12_debug.h"
#include "w12_internal.h"

using namespace w12i;

namespace {

int32_t g_debug_flags = 0;
uint64_t g_timeout_ns = 2000000000ull;   // 2 s per bounded wait

constexpr int kMaxCtas = 256;            // persistent grids never exceed this

// benchmark timing hook (see w12_debug.h)
bool g_profile = false;
constexpr int kProfMax = 1024;
cudaEvent_t g_prof_ev[kProfMax + 1];
int g_prof_created = 0, g_prof_used = 0;

int prof_mark(cudaStream_t st)
{
    if (!g_profile || g_prof_used > kProfMax) return 0;
    if (g_prof_used >= g_prof_created) {
        if (cudaEventCreate(&g_prof_ev[g_prof_created]) != cudaSuccess) return 1;
        ++g_prof_created;
    }
    return (int)cudaEventRecord(g_prof_ev[g_prof_used++], st);
}
constexpr int kPartialRows = 64;         // rows per warp-MMA launch (larger R is sliced)

// rows of one CTA's partial tile: the warp-MMA path pads to <= 64, the
// tensor-memory path to a multiple of 32
int partial_rows(int32_t R) { return std::max(kPartialRows, (R + 31) / 32 * 32); }

// Path choice: the tensor-memory kernel streams the weights once for any
// R <= 256; the warp-MMA kernel covers R <= 64 per pass.  Measured on GB300
// (27B-like shapes, microseconds per launch, warp-MMA against tcgen05):
//   16 rows: warp-MMA faster for every weight (LM head 246 / 265);
//   32 rows: tcgen05 faster for gate/up (78 / 73) and the LM head (292 / 266),
//            warp-MMA for QKV, O and down (under 100 records per SM);
//   64 rows: tcgen05 faster from down (72 records per SM: 58 / 56) up,
//            warp-MMA for QKV and O.
// Debug flag bit 1 forces the tensor-memory path, bit 2 the warp-MMA path.
int num_sms();

bool use_tc(int32_t R, int64_t records)
{
    if (g_debug_flags & 2) return true;
    if (g_debug_flags & 4) return false;
    if (R > kPartialRows) return true;
    if (R <= 16) return false;
    const int64_t per_sm = records / num_sms();
    return R <= 32 ? per_sm >= 100 : per_sm >= 50;
}

// GEMM-chain timing hook (w12_debug_chain_trace)
uint64_t *g_trace = nullptr;
size_t g_trace_words = 0;

int chain_parts(int n_jobs) { return (n_jobs + chain_max_jobs() - 1) / chain_max_jobs(); }

// The verify step runs its GEMMs as one persistent chain (k_chain.cu) when
// debug flag bit 4 asks for it, unless bit 2 (warp-MMA kernel) or bit 3 (one
// launch per GEMM) is set or the step has more GEMMs than the workspace has
// chain words for.  Measured on GB300, one launch per GEMM with the per-row-count
// kernel choice is faster on the 27B-like shapes, so it is the default.
bool use_chain(int n_jobs)
{
    if (g_debug_flags & (4 | 8)) return false;
    if (!(g_debug_flags & 16)) return false;
    return n_jobs + 1 <= kGridWords;
}

// SM count of the current device, looked up once per device.  Each device
// has its own cache entry (an atomic, so host threads driving different
// devices never read one another's count); devices beyond the table are
// looked up on every call.
int num_sms()
{
    constexpr int kDevCache = 64;
    static std::atomic<int> cached[kDevCache];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kMaxCtas;
    if (dev >= 0 && dev < kDevCache) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return kMaxCtas;
    n = std::min(n, kMaxCtas);
    if (dev >= 0 && dev < kDevCache) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

w12_status weight_ok(const w12_weight *w)
{
    if (!w || !w->rec || !w->base || !w->esc_tile_off) return W12_E_INVAL;
    if (w->n <= 0 || w->k <= 0 || w->n_escapes < 0) return W12_E_INVAL;
    if (w->n_escapes > 0 && !w->esc) return W12_E_INVAL;
    if (w->n % kTileN || w->k % kTileK) return W12_E_UNSUPPORTED;
    if (w->n / kTileN > INT32_MAX || w->k / kTileK > INT32_MAX) return W12_E_UNSUPPORTED;
    if (!aligned(w->rec, 16)) return W12_E_INVAL;
    return W12_OK;
}

DevWeight dev_weight(const w12_weight *w)
{
    DevWeight d;
    d.rec = static_cast<const uint8_t *>(w->rec);
    d.base = w->base;
    d.esc_off = w->esc_tile_off;
    d.esc = w->esc;
    d.n_tiles = static_cast<int32_t>(w->n / kTileN);
    d.k_tiles = static_cast<int32_t>(w->k / kTileK);
    d.n = w->n;
    d.k = w->k;
    return d;
}

int g_last_cuda_error = 0;

w12_status cuda_status(int e)
{
    if (e == 0) return W12_OK;
    g_last_cuda_error = e;
    return W12_E_CUDA;
}

struct Ws {
    uint8_t *base;
    WsLayout L;
    int32_t *status() const { return reinterpret_cast<int32_t *>(base + L.status); }
    int64_t *mismatch() const { return reinterpret_cast<int64_t *>(base + L.status + 64); }
    int32_t *counters(int slot) const
    {
        return reinterpret_cast<int32_t *>(base + L.counters) + static_cast<size_t>(slot) * L.max_tiles_n;
    }
    float *partial(int slot) const
    {
        return reinterpret_cast<float *>(base + L.partial) +
               static_cast<size_t>(slot) * kMaxCtas * 2 * partial_rows(L.rows) * kTileN;
    }
    // arrival counters start at zero for every call (the kernels also reset
    // each counter they finish with, so launches inside one call need no memset)
    int clear_counters(cudaStream_t st) const
    {
        return (int)cudaMemsetAsync(base + L.counters, 0, static_cast<size_t>(kGemmSlots) * L.max_tiles_n * 4, st);
    }
    // the same, plus the GEMM-chain words of n_jobs GEMMs (the region sits just
    // before the counters, so one memset clears both)
    int clear_chain(int n_jobs, cudaStream_t st) const
    {
        const size_t lead = static_cast<size_t>(1 + n_jobs) * 4;
        return (int)cudaMemsetAsync(base + L.counters - lead, 0,
                                    lead + static_cast<size_t>(kGemmSlots) * L.max_tiles_n * 4, st);
    }
    // a chain of n_jobs GEMMs uses the last 1 + n_jobs words of the region:
    // its abort word, then one arrival word per GEMM
    int32_t *grid_abort(int n_jobs) const
    {
        return reinterpret_cast<int32_t *>(base + L.counters - static_cast<size_t>(1 + n_jobs) * 4);
    }
    uint32_t *grid_bar(int n_jobs) const { return reinterpret_cast<uint32_t *>(grid_abort(n_jobs) + 1); }
    float *s1_val() const { return reinterpret_cast<float *>(base + L.stage1_val); }
    int32_t *s1_idx() const { return reinterpret_cast<int32_t *>(base + L.stage1_idx); }
    void *tree() const { return base + L.tree; }
};

// The layout depends only on the sizes, so a workspace sized for a call is
// laid out identically by every call whose sizes it covers.
WsLayout layout_for(int32_t R, int64_t max_n, int64_t vocab, int32_t n_req)
{
    WsLayout L{};
    L.rows8 = (std::max<int32_t>(R, 1) + 7) / 8 * 8;
    L.rows = std::max<int32_t>(R, 1);
    L.max_tiles_n = std::max<int64_t>(std::max<int64_t>(max_n, vocab), kTileN) / kTileN;
    L.vocab_tiles = std::max<int64_t>(vocab, kTileN) / kTileN;
    L.max_ctas = kMaxCtas;
    size_t o = 0;
    L.status = o;
    o += 256;
    // the chain words end exactly where the counters start
    L.grid = o;
    o += static_cast<size_t>(kGridWords) * 4;
    L.counters = o;
    o = align256(o + static_cast<size_t>(kGemmSlots) * L.max_tiles_n * 4);
    L.partial = o;
    o = align256(o + static_cast<size_t>(kGemmSlots) * kMaxCtas * 2 * partial_rows(L.rows) * kTileN * 4);
    L.stage1_val = o;
    o = align256(o + static_cast<size_t>(L.rows8) * L.vocab_tiles * 4);
    L.stage1_idx = o;
    o = align256(o + static_cast<size_t>(L.rows8) * L.vocab_tiles * 4);
    L.tree = o;
    o = align256(o + tree_ws_bytes(n_req));
    L.total = o;
    return L;
}

w12_status ws_check(void *ws, size_t ws_bytes, const WsLayout &L)
{
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return W12_E_WORKSPACE;
    return W12_OK;
}

int gemm_slices(const DevWeight &dw, const uint16_t *x, int32_t R, int mode, uint16_t *y, const Ws &ws, int &slot,
                bool pdl, cudaStream_t st, bool qview = false)
{
    const bool tc = use_tc(R, (int64_t)dw.n_tiles * dw.k_tiles);
    const int32_t step = tc ? R : kPartialRows;
    for (int32_t r0 = 0; r0 < R; r0 += step) {
        GemmArgs a{};
        a.w = dw;
        a.x = x + static_cast<int64_t>(r0) * dw.k;
        a.R = std::min<int32_t>(step, R - r0);
        a.mode = mode;
        a.y = y ? y + static_cast<int64_t>(r0) * dw.n : nullptr;
        a.stage1_val = ws.s1_val() + static_cast<int64_t>(r0) * dw.n_tiles;
        a.stage1_idx = ws.s1_idx() + static_cast<int64_t>(r0) * dw.n_tiles;
        a.partial = ws.partial(slot);
        a.counters = ws.counters(slot);
        a.status = ws.status();
        a.num_sms = num_sms();
        a.pdl = pdl;
        a.debug_flags = g_debug_flags;
        a.timeout_ns = g_timeout_ns;
        a.qview = qview;
        const int e = tc ? launch_gemm_tc(a, st) : launch_gemm(a, st);
        if (e) return e;
        if (int pe = prof_mark(st)) return pe;
        slot = (slot + 1) % kGemmSlots;
        pdl = true;
    }
    return 0;
}

w12_status tree_ok(const w12_tree *t, bool need_rows)
{
    if (!t || !t->parent || !t->token || !t->depth || !t->req_row_off) return W12_E_INVAL;
    if (need_rows && (t->R < 1 || t->R > kMaxBudget)) return t->R < 1 ? W12_E_INVAL : W12_E_UNSUPPORTED;
    return W12_OK;
}

}  // namespace

namespace w12i {
WsLayout ws_layout(int32_t R, int64_t max_n, int64_t vocab, int32_t n_req, int)
{
    return layout_for(R, max_n, vocab, n_req);
}
}  // namespace w12i

extern "C" {

const char *w12_status_str(int status)
{
    switch (status) {
    case W12_OK: return "W12_OK";
    case W12_E_INVAL: return "W12_E_INVAL";
    case W12_E_UNSUPPORTED: return "W12_E_UNSUPPORTED";
    case W12_E_MISMATCH: return "W12_E_MISMATCH";
    case W12_E_CUDA: return "W12_E_CUDA";
    case W12_E_TIMEOUT: return "W12_E_TIMEOUT";
    case W12_E_WORKSPACE: return "W12_E_WORKSPACE";
    default: return "W12_E_UNKNOWN";
    }
}

int w12_abi_version(void) { return 100; }

void w12_debug_set(int32_t flags, uint64_t timeout_ns)
{
    g_debug_flags = flags;
    g_timeout_ns = timeout_ns ? timeout_ns : 2000000000ull;
}

int32_t w12_debug_num_sms(void) { return num_sms(); }

void w12_debug_chain_trace(void *dev_words, size_t n_words)
{
    g_trace = static_cast<uint64_t *>(dev_words);
    g_trace_words = dev_words ? n_words : 0;
}

int32_t w12_debug_chain_parts(int32_t n_gemms) { return n_gemms > 0 ? chain_parts(n_gemms) : 0; }

int32_t w12_debug_last_cuda_error(char *buf, int32_t len)
{
    if (buf && len > 0) {
        const char *name = g_last_cuda_error ? cudaGetErrorName(static_cast<cudaError_t>(g_last_cuda_error)) : "";
        std::strncpy(buf, name, static_cast<size_t>(len - 1));
        buf[len - 1] = 0;
    }
    return g_last_cuda_error;
}

void w12_debug_profile(int32_t enable)
{
    g_profile = enable != 0;
    g_prof_used = 0;
}

int32_t w12_debug_profile_read(float *ms, int32_t max)
{
    if (!ms || max < 0) return W12_E_INVAL;
    if (g_prof_used < 2) return 0;
    if (cudaEventSynchronize(g_prof_ev[g_prof_used - 1]) != cudaSuccess) return W12_E_CUDA;
    const int n = std::min(g_prof_used - 1, max);
    for (int i = 0; i < n; ++i)
        if (cudaEventElapsedTime(&ms[i], g_prof_ev[i], g_prof_ev[i + 1]) != cudaSuccess) return W12_E_CUDA;
    return g_prof_used - 1;
}

size_t w12_workspace_bytes(int32_t R, int64_t max_n, int64_t vocab, int32_t n_req)
{
    if (R < 1 || R > kMaxRows || max_n < 0 || vocab < 0 || n_req < 0 || n_req > kMaxBudget) return 0;
    return layout_for(R, max_n, vocab, n_req).total;
}

w12_status w12_workspace_init(void *ws, size_t ws_bytes, w12_stream_t stream)
{
    if (!ws || !aligned(ws, 256) || ws_bytes < 256) return W12_E_WORKSPACE;
    return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

w12_status w12_status_fetch(void *ws, w12_stream_t stream)
{
    if (!ws || !aligned(ws, 256)) return W12_E_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return W12_E_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof v, st) != cudaSuccess) return W12_E_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return W12_E_CUDA;
    return static_cast<w12_status>(v);
}

w12_status w12_unpack(const w12_weight *w, uint16_t *dst_bf16, w12_stream_t stream)
{
    w12_status s = weight_ok(w);
    if (s != W12_OK) return s;
    if (!dst_bf16 || !aligned(dst_bf16, 16)) return W12_E_INVAL;
    return cuda_status(launch_unpack(dev_weight(w), dst_bf16, nullptr, nullptr, nullptr, stream));
}

w12_status w12_load_check(const w12_weight *w, const uint16_t *src_bf16, int64_t *mismatches, void *ws,
                          size_t ws_bytes, w12_stream_t stream)
{
    w12_status s = weight_ok(w);
    if (s != W12_OK) return s;
    if (!src_bf16 || !mismatches || !aligned(src_bf16, 16)) return W12_E_INVAL;
    if (!ws || !aligned(ws, 256) || ws_bytes < 256) return W12_E_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int64_t *dev_count = reinterpret_cast<int64_t *>(static_cast<uint8_t *>(ws) + 64);
    if (cudaMemsetAsync(dev_count, 0, sizeof(int64_t), st) != cudaSuccess) return W12_E_CUDA;
    if (launch_unpack(dev_weight(w), nullptr, src_bf16, dev_count, nullptr, stream)) return W12_E_CUDA;
    int64_t host = 0;
    if (cudaMemcpyAsync(&host, dev_count, sizeof host, cudaMemcpyDeviceToHost, st) != cudaSuccess) return W12_E_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return W12_E_CUDA;
    *mismatches = host;
    return host == 0 ? W12_OK : W12_E_MISMATCH;
}

namespace {

w12_status gemm_entry(const w12_weight *w, const uint16_t *x, int32_t R, uint16_t *y, void *ws, size_t ws_bytes,
                      w12_stream_t stream, bool qview)
{
    w12_status s = weight_ok(w);
    if (s != W12_OK) return s;
    if (!x || !y || !aligned(x, 16) || !aligned(y, 16)) return W12_E_INVAL;
    if (R < 1) return W12_E_INVAL;
    if (R > kMaxRows) return W12_E_UNSUPPORTED;
    const WsLayout L = layout_for(R, w->n, 0, 0);
    if ((s = ws_check(ws, ws_bytes, L)) != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (int ce = W.clear_counters(st)) return cuda_status(ce);
    int slot = 0;
    return cuda_status(gemm_slices(dev_weight(w), x, R, kModeLinear, y, W, slot, false, st, qview));
}

}  // namespace

w12_status w12_gemm(const w12_weight *w, const uint16_t *x, int32_t R, uint16_t *y, void *ws, size_t ws_bytes,
                    w12_stream_t stream)
{
    return gemm_entry(w, x, R, y, ws, ws_bytes, stream, false);
}

w12_status w12_gemm_q(const w12_weight *w, const uint16_t *x, int32_t R, uint16_t *y, void *ws, size_t ws_bytes,
                      w12_stream_t stream)
{
    return gemm_entry(w, x, R, y, ws, ws_bytes, stream, true);
}

w12_status w12_gemm_static_scratch(const w12_weight *w, const uint16_t *x, int32_t R, uint16_t *y,
                                   w12_stream_t stream)
{
    w12_status s = weight_ok(w);
    if (s != W12_OK) return s;
    if (!x || !y || !aligned(x, 16) || !aligned(y, 16)) return W12_E_INVAL;
    if (R < 1) return W12_E_INVAL;
    int32_t max_rows = 0, max_tiles = 0;
    static_scratch_limits(&max_rows, &max_tiles);
    if (R > max_rows || w->n / kTileN > max_tiles) return W12_E_UNSUPPORTED;
    GemmArgs a{};
    a.w = dev_weight(w);
    a.x = x;
    a.R = R;
    a.mode = kModeLinear;
    a.y = y;
    a.num_sms = num_sms();
    a.pdl = false;
    a.debug_flags = 0;
    a.timeout_ns = g_timeout_ns;
    return cuda_status(launch_gemm_static_scratch(a, stream));
}

namespace {

w12_status head_entry(const w12_weight *head, const uint16_t *h, int32_t R, int32_t *argmax, float *maxlogit,
                      void *ws, size_t ws_bytes, w12_stream_t stream, bool qview)
{
    w12_status s = weight_ok(head);
    if (s != W12_OK) return s;
    if (!h || !argmax || !aligned(h, 16)) return W12_E_INVAL;
    if (R < 1) return W12_E_INVAL;
    if (R > kMaxRows) return W12_E_UNSUPPORTED;
    const WsLayout L = layout_for(R, 0, head->n, 0);
    if ((s = ws_check(ws, ws_bytes, L)) != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (int ce = W.clear_counters(st)) return cuda_status(ce);
    int slot = 0;
    const DevWeight dw = dev_weight(head);
    if (int e = gemm_slices(dw, h, R, kModeHead, nullptr, W, slot, false, st, qview)) return cuda_status(e);
    return cuda_status(launch_argmax_stage2(W.s1_val(), W.s1_idx(), R, dw.n_tiles, argmax, maxlogit, true, st));
}

}  // namespace

w12_status w12_lmhead_argmax(const w12_weight *head, const uint16_t *h, int32_t R, int32_t *argmax, float *maxlogit,
                             void *ws, size_t ws_bytes, w12_stream_t stream)
{
    return head_entry(head, h, R, argmax, maxlogit, ws, ws_bytes, stream, false);
}

w12_status w12_lmhead_argmax_q(const w12_weight *head, const uint16_t *h, int32_t R, int32_t *argmax,
                               float *maxlogit, void *ws, size_t ws_bytes, w12_stream_t stream)
{
    return head_entry(head, h, R, argmax, maxlogit, ws, ws_bytes, stream, true);
}

// ---------------------------------------------------------------------------
// certified LM head
// ---------------------------------------------------------------------------

w12_status w12_head_cert_norms(const w12_weight *head, float *norms, w12_stream_t stream)
{
    w12_status s = weight_ok(head);
    if (s != W12_OK) return s;
    if (!norms || !aligned(norms, 4)) return W12_E_INVAL;
    const DevWeight dw = dev_weight(head);
    return cuda_status(launch_cert_norms(dw, norms, norms + head->n, stream));
}

size_t w12_cert_workspace_bytes(int32_t R, int64_t vocab)
{
    if (R < 1 || vocab < 1) return 0;
    const size_t shat = ((size_t)R * (size_t)vocab * 2 + 255) / 256 * 256;
    const size_t surv = ((size_t)R * (size_t)vocab * 4 + 255) / 256 * 256;
    const size_t cnt = ((size_t)R * 4 + 255) / 256 * 256;
    const size_t part = ((size_t)R * kCertParts * 16 + (size_t)R * 4 + 255) / 256 * 256;
    return shat + surv + cnt + part;
}

w12_status w12_lmhead_argmax_certified(const w12_weight *head, const float *norms, const uint16_t *h, int32_t R,
                                       int32_t *argmax, float *maxlogit, int32_t *n_survivors, void *ws,
                                       size_t ws_bytes, void *cws, size_t cws_bytes, w12_stream_t stream)
{
    w12_status s = weight_ok(head);
    if (s != W12_OK) return s;
    if (!norms || !h || !argmax || !aligned(h, 16) || !cws || !aligned(cws, 256)) return W12_E_INVAL;
    if (R < 1) return W12_E_INVAL;
    if (R > kMaxRows) return W12_E_UNSUPPORTED;
    if (cws_bytes < w12_cert_workspace_bytes(R, head->n)) return W12_E_WORKSPACE;
    const WsLayout L = layout_for(R, head->n, 0, 0);
    if ((s = ws_check(ws, ws_bytes, L)) != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (int ce = W.clear_counters(st)) return cuda_status(ce);
    uint8_t *c = static_cast<uint8_t *>(cws);
    uint16_t *shat = reinterpret_cast<uint16_t *>(c);
    int32_t *surv = reinterpret_cast<int32_t *>(c + ((size_t)R * head->n * 2 + 255) / 256 * 256);
    int32_t *cnt = surv + ((size_t)R * head->n * 4 + 255) / 256 * 256 / 4;
    double *part_v = reinterpret_cast<double *>(reinterpret_cast<uint8_t *>(cnt) + ((size_t)R * 4 + 255) / 256 * 256);
    int32_t *part_i = reinterpret_cast<int32_t *>(part_v + (size_t)R * kCertParts);
    float *part_lo = reinterpret_cast<float *>(part_i + (size_t)R * kCertParts);
    const DevWeight dw = dev_weight(head);
    int slot = 0;
    // 1. cheap pass: the quick-pass logits of every token, BF16 [R][V]
    if (int e = gemm_slices(dw, h, R, kModeLinear, shat, W, slot, false, st, true)) return cuda_status(e);
    // 2. per row: the bound and the survivors
    if (int e = launch_cert_select(shat, h, norms, norms + head->n, R, head->n, head->k, surv, cnt, part_lo, st))
        return cuda_status(e);
    // 3. exact FP64 rescoring of the survivors
    return cuda_status(launch_cert_rescore(dw, h, R, surv, cnt, part_v, part_i, argmax, maxlogit, n_survivors, st));
}

w12_status w12_tree_build(const w12_lattice *lat, int32_t budget, w12_tree *out, void *ws, size_t ws_bytes,
                          w12_stream_t stream)
{
    if (!lat || !out || !lat->p_r || !lat->root_tok) return W12_E_INVAL;
    if (lat->n_req < 1 || lat->p_max < 0 || lat->n_cand < 1 || budget < 1) return W12_E_INVAL;
    if (lat->p_max > 0 && (!lat->cand_tok || !lat->cand_logp)) return W12_E_INVAL;
    if (lat->n_req > kMaxBudget || lat->p_max > kMaxPositions || lat->n_cand > kCands || budget > kMaxBudget)
        return W12_E_UNSUPPORTED;
    if (budget < lat->n_req) return W12_E_INVAL;
    if (!out->parent || !out->token || !out->depth || !out->req || !out->score || !out->rank || !out->req_row_off)
        return W12_E_INVAL;
    // rows = min(budget, nodes the lattice can hold), known before any launch
    int64_t nodes = 0;
    for (int32_t r = 0; r < lat->n_req; ++r) {
        const int32_t pr = lat->p_r[r];
        if (pr < 0 || pr > lat->p_max) return W12_E_INVAL;
        int64_t level = 1, sum = 1;
        for (int32_t d = 1; d <= pr && sum < budget; ++d) {
            level = std::min<int64_t>(level * lat->n_cand, budget);
            sum += level;
        }
        nodes = std::min<int64_t>(nodes + sum, budget);
    }
    const WsLayout L = layout_for(1, 0, 0, lat->n_req);
    w12_status s = ws_check(ws, ws_bytes, L);
    if (s != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    out->R = static_cast<int32_t>(nodes);
    TreeArgs a{};
    a.n_req = lat->n_req;
    a.p_max = lat->p_max;
    a.n_cand = lat->n_cand;
    a.conditional = lat->conditional ? 1 : 0;
    a.budget = budget;
    a.R = out->R;
    a.p_r_host = lat->p_r;
    a.root_tok = lat->root_tok;
    a.cand_tok = lat->cand_tok;
    a.cand_logp = lat->cand_logp;
    a.parent = out->parent;
    a.token = out->token;
    a.req = out->req;
    a.req_row_off = out->req_row_off;
    a.depth = out->depth;
    a.rank = out->rank;
    a.score = out->score;
    a.scratch = W.tree();
    a.status = W.status();
    return cuda_status(launch_tree_build(a, stream));
}

w12_status w12_tree_accept(const w12_tree *tree, int32_t n_req, int32_t p_max, const int32_t *argmax, int32_t *acc_tok,
                           int32_t *acc_len, int32_t *acc_node, w12_stream_t stream)
{
    w12_status s = tree_ok(tree, true);
    if (s != W12_OK) return s;
    if (!argmax || !acc_tok || !acc_len) return W12_E_INVAL;
    if (n_req < 1 || p_max < 0) return W12_E_INVAL;
    if (n_req > kMaxBudget || p_max > kMaxDepth) return W12_E_UNSUPPORTED;
    return cuda_status(launch_tree_accept(tree->parent, tree->token, tree->depth, tree->req_row_off, tree->R, n_req,
                                          p_max, argmax, acc_tok, acc_len, acc_node, false, stream));
}

}  // extern "C"

namespace {

w12_status verify_step_entry(const w12_step *step, const w12_tree *tree, int32_t n_req, int32_t p_max,
                             int32_t *acc_tok, int32_t *acc_len, int32_t *acc_node, void *ws, size_t ws_bytes,
                             w12_stream_t stream, bool qview)
{
    if (!step || step->n_linear < 0 || (step->n_linear > 0 && (!step->lin || !step->x || !step->y)))
        return W12_E_INVAL;
    w12_status s = tree_ok(tree, true);
    if (s != W12_OK) return s;
    if (!acc_tok || !acc_len || !step->h || !step->argmax || !aligned(step->h, 16)) return W12_E_INVAL;
    if (n_req < 1 || p_max < 0) return W12_E_INVAL;
    if (n_req > kMaxBudget || p_max > kMaxDepth) return W12_E_UNSUPPORTED;
    const int32_t R = tree->R;
    if (R > kMaxRows) return W12_E_UNSUPPORTED;
    if ((s = weight_ok(step->head)) != W12_OK) return s;
    int64_t max_n = 0;
    for (int32_t l = 0; l < step->n_linear; ++l) {
        if ((s = weight_ok(&step->lin[l])) != W12_OK) return s;
        if (!step->x[l] || !step->y[l] || !aligned(step->x[l], 16) || !aligned(step->y[l], 16)) return W12_E_INVAL;
        max_n = std::max<int64_t>(max_n, step->lin[l].n);
    }
    const WsLayout L = layout_for(R, max_n, step->head->n, n_req);
    if ((s = ws_check(ws, ws_bytes, L)) != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const DevWeight hw = dev_weight(step->head);
    const int n_jobs = step->n_linear + 1;
    if (use_chain(n_jobs)) {
        // every GEMM of the step in one persistent launch (two or more for
        // steps beyond one launch's parameter block)
        if (int ce = W.clear_chain(n_jobs, st)) return cuda_status(ce);
        g_prof_used = 0;
        if (prof_mark(st)) return W12_E_CUDA;
        std::vector<ChainJob> jobs(static_cast<size_t>(n_jobs));
        for (int32_t l = 0; l < step->n_linear; ++l)
            jobs[l] = ChainJob{dev_weight(&step->lin[l]), step->x[l], kModeLinear, step->y[l], nullptr, nullptr};
        jobs[step->n_linear] = ChainJob{hw, step->h, kModeHead, nullptr, W.s1_val(), W.s1_idx()};
        ChainArgs ca{};
        ca.jobs = jobs.data();
        ca.n_jobs = n_jobs;
        ca.R = R;
        ca.partial = W.partial(0);
        ca.counters = W.counters(0);
        ca.status = W.status();
        ca.grid_bar = W.grid_bar(n_jobs);
        ca.grid_abort = W.grid_abort(n_jobs);
        ca.num_sms = num_sms();
        ca.pdl = true;
        ca.qview = qview;
        ca.debug_flags = g_debug_flags;
        ca.timeout_ns = g_timeout_ns;
        if (g_trace && g_trace_words >= (size_t)(n_jobs + chain_parts(n_jobs)) * (size_t)ca.num_sms)
            ca.trace = g_trace;
        if (int e = launch_chain(ca, st)) return cuda_status(e);
        if (int pe = prof_mark(st)) return cuda_status(pe);
    } else {
        if (int ce = W.clear_counters(st)) return cuda_status(ce);
        g_prof_used = 0;
        if (prof_mark(st)) return W12_E_CUDA;
        int slot = 0;
        for (int32_t l = 0; l < step->n_linear; ++l)
            if (int e = gemm_slices(dev_weight(&step->lin[l]), step->x[l], R, kModeLinear, step->y[l], W, slot, true,
                                    st, qview))
                return cuda_status(e);
        if (int e = gemm_slices(hw, step->h, R, kModeHead, nullptr, W, slot, true, st, qview)) return cuda_status(e);
    }
    if (int e = launch_argmax_stage2(W.s1_val(), W.s1_idx(), R, hw.n_tiles, step->argmax, nullptr, true, st))
        return cuda_status(e);
    if (prof_mark(st)) return W12_E_CUDA;
    if (int e = launch_tree_accept(tree->parent, tree->token, tree->depth, tree->req_row_off, R, n_req, p_max,
                                   step->argmax, acc_tok, acc_len, acc_node, true, stream))
        return cuda_status(e);
    return prof_mark(st) ? W12_E_CUDA : W12_OK;
}

}  // namespace

extern "C" {

w12_status w12_verify_step(const w12_step *step, const w12_tree *tree, int32_t n_req, int32_t p_max, int32_t *acc_tok,
                           int32_t *acc_len, int32_t *acc_node, void *ws, size_t ws_bytes, w12_stream_t stream)
{
    return verify_step_entry(step, tree, n_req, p_max, acc_tok, acc_len, acc_node, ws, ws_bytes, stream, false);
}

w12_status w12_verify_step_q(const w12_step *step, const w12_tree *tree, int32_t n_req, int32_t p_max,
                             int32_t *acc_tok, int32_t *acc_len, int32_t *acc_node, void *ws, size_t ws_bytes,
                             w12_stream_t stream)
{
    return verify_step_entry(step, tree, n_req, p_max, acc_tok, acc_len, acc_node, ws, ws_bytes, stream, true);
}

}  // extern "C"

namespace {

w12_status gdn_args(const w12_gdn_layer *L, const w12_tree *tree, int32_t n_req, GdnArgs &a)
{
    if (!L || !tree || !tree->parent || !tree->req_row_off || !L->S0 || !L->q || !L->k || !L->v || !L->alpha ||
        !L->beta)
        return W12_E_INVAL;
    if (L->n_heads < 1 || n_req < 1 || tree->R < 1) return W12_E_INVAL;
    if (L->head_dim != kGdnDim || L->n_heads > 65535 || n_req > kMaxBudget || tree->R > kMaxBudget)
        return W12_E_UNSUPPORTED;
    if (!aligned(L->S0, 16) || !aligned(L->q, 16) || !aligned(L->k, 16) || !aligned(L->v, 4)) return W12_E_INVAL;
    a = GdnArgs{};
    a.H = L->n_heads;
    a.n_req = n_req;
    a.R = tree->R;
    a.num_sms = num_sms();
    a.timeout_ns = g_timeout_ns;
    a.debug_flags = g_debug_flags;
    a.S0 = L->S0;
    a.q = L->q;
    a.k = L->k;
    a.v = L->v;
    a.alpha = L->alpha;
    a.beta = L->beta;
    a.parent = tree->parent;
    a.req_row_off = tree->req_row_off;
    return W12_OK;
}

}  // namespace

extern "C" {

w12_status w12_gdn_tree_verify(const w12_gdn_layer *layer, const w12_tree *tree, int32_t n_req, int32_t method,
                               float *o, void *ws, size_t ws_bytes, w12_stream_t stream)
{
    GdnArgs a;
    w12_status s = gdn_args(layer, tree, n_req, a);
    if (s != W12_OK) return s;
    if (!o || (method != W12_GDN_WY && method != W12_GDN_PATH)) return W12_E_INVAL;
    const WsLayout L = layout_for(1, 0, 0, n_req);
    if ((s = ws_check(ws, ws_bytes, L)) != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    a.out = o;
    a.status = W.status();
    return cuda_status(launch_gdn(a, method == W12_GDN_WY ? kGdnWy : kGdnPath, stream));
}

w12_status w12_gdn_wy_verify(const w12_gdn_layer *layer, const w12_tree *tree, int32_t n_req, float *o, float *u,
                             void *ws, size_t ws_bytes, w12_stream_t stream)
{
    GdnArgs a;
    w12_status s = gdn_args(layer, tree, n_req, a);
    if (s != W12_OK) return s;
    if (!o || !u) return W12_E_INVAL;
    const WsLayout L = layout_for(1, 0, 0, n_req);
    if ((s = ws_check(ws, ws_bytes, L)) != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    a.out = o;
    a.u = u;
    a.status = W.status();
    return cuda_status(launch_gdn(a, kGdnWy, stream));
}

w12_status w12_gdn_wy_commit(const w12_gdn_layer *layer, const w12_tree *tree, int32_t n_req, const int32_t *acc_node,
                             const float *u, float *state, void *ws, size_t ws_bytes, w12_stream_t stream)
{
    GdnArgs a;
    w12_status s = gdn_args(layer, tree, n_req, a);
    if (s != W12_OK) return s;
    if (!acc_node || !u || !state || !aligned(state, 16) || !aligned(u, 16)) return W12_E_INVAL;
    const WsLayout L = layout_for(1, 0, 0, n_req);
    if ((s = ws_check(ws, ws_bytes, L)) != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    a.acc_node = acc_node;
    a.u = const_cast<float *>(u);
    a.out = state;
    a.status = W.status();
    return cuda_status(launch_gdn(a, kGdnCommitWy, stream));
}

w12_status w12_gdn_commit(const w12_gdn_layer *layer, const w12_tree *tree, int32_t n_req, const int32_t *acc_node,
                          float *state, void *ws, size_t ws_bytes, w12_stream_t stream)
{
    GdnArgs a;
    w12_status s = gdn_args(layer, tree, n_req, a);
    if (s != W12_OK) return s;
    if (!acc_node || !state || !aligned(state, 16)) return W12_E_INVAL;
    const WsLayout L = layout_for(1, 0, 0, n_req);
    if ((s = ws_check(ws, ws_bytes, L)) != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    a.acc_node = acc_node;
    a.out = state;
    a.status = W.status();
    return cuda_status(launch_gdn(a, kGdnCommit, stream));
}

w12_status w12_tlv_chain(const int32_t *c_len, const int32_t *t1_row_off, int32_t n_req, int32_t budget, int32_t *m,
                         int32_t *sub_budget)
{
    if (!c_len || !t1_row_off || !m || !sub_budget || n_req < 1 || budget < 1) return W12_E_INVAL;
    if (n_req > kMaxBudget || budget > kMaxBudget) return W12_E_UNSUPPORTED;
    if (t1_row_off[0] != 0 || t1_row_off[n_req] > budget) return W12_E_INVAL;
    int64_t used = 0;
    for (int32_t q = 0; q < n_req; ++q) {
        const int32_t rows = t1_row_off[q + 1] - t1_row_off[q];
        if (rows < 1 || c_len[q] < 1 || c_len[q] > rows) return W12_E_INVAL;
        m[q] = std::min(c_len[q], rows - 1);
        used += m[q];
    }
    *sub_budget = static_cast<int32_t>(budget - used);
    return W12_OK;
}

w12_status w12_tlv_splice(const w12_tree *t1, const int32_t *c_tok, const int32_t *c_len, const int32_t *c_node,
                          int32_t n_req, int32_t p1_max, const int32_t *m, const w12_tree *t2, w12_tree *out,
                          void *ws, size_t ws_bytes, w12_stream_t stream)
{
    w12_status s = tree_ok(t1, true);
    if (s != W12_OK) return s;
    if ((s = tree_ok(t2, true)) != W12_OK) return s;
    if (!t1->score || !t1->rank || !t2->req || !t2->score || !t2->rank) return W12_E_INVAL;
    if (!out || !out->parent || !out->token || !out->depth || !out->req || !out->score || !out->rank ||
        !out->req_row_off)
        return W12_E_INVAL;
    if (!c_tok || !c_len || !c_node || !m || n_req < 1 || p1_max < 0) return W12_E_INVAL;
    if (n_req > kMaxBudget || p1_max > kMaxPositions) return W12_E_UNSUPPORTED;
    int64_t R = t2->R;
    for (int32_t q = 0; q < n_req; ++q) {
        if (m[q] < 0 || m[q] > p1_max + 1) return W12_E_INVAL;
        R += m[q];
    }
    if (R > kMaxBudget) return W12_E_UNSUPPORTED;
    const WsLayout L = layout_for(1, 0, 0, n_req);
    if ((s = ws_check(ws, ws_bytes, L)) != W12_OK) return s;
    Ws W{static_cast<uint8_t *>(ws), L};
    out->R = static_cast<int32_t>(R);
    SpliceArgs a{};
    a.n_req = n_req;
    a.p1_max = p1_max;
    a.t1_R = t1->R;
    a.t2_R = t2->R;
    a.R = out->R;
    a.m_host = m;
    a.t1_parent = t1->parent;
    a.t1_token = t1->token;
    a.t1_off = t1->req_row_off;
    a.t1_rank = t1->rank;
    a.t1_score = t1->score;
    a.c_tok = c_tok;
    a.c_len = c_len;
    a.c_node = c_node;
    a.t2_parent = t2->parent;
    a.t2_token = t2->token;
    a.t2_req = t2->req;
    a.t2_off = t2->req_row_off;
    a.t2_depth = t2->depth;
    a.t2_rank = t2->rank;
    a.t2_score = t2->score;
    a.parent = out->parent;
    a.token = out->token;
    a.req = out->req;
    a.off = out->req_row_off;
    a.depth = out->depth;
    a.rank = out->rank;
    a.score = out->score;
    a.status = W.status();
    return cuda_status(launch_tlv_splice(a, stream));
}

}  // extern "C"
