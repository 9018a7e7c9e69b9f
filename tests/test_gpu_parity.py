"""GPU parity of every step of the W12 verify pass against the CPU oracle,
called through the C ABI (marked gpu)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_w12_gb300 import synth
from tests import helpers as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w12():
    from speculative_decoding_tree_w12_gb300 import build
    build.build()
    import speculative_decoding_tree_w12_gb300 as m
    m.lib()
    return m


@pytest.fixture(params=["warp_mma", "tcgen05"])
def path(request, w12):
    """Run the test on one GEMM kernel: the warp-MMA kernel (flag 4) or the
    tensor-memory kernel (flag 2)."""
    w12.debug_set(4 if request.param == "warp_mma" else 2, 0)
    yield request.param
    w12.debug_set(0, 0)


def _dev_bf16(bits: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _bits(t) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _packed(w12, w):
    return w12.DeviceWeight(w12.w12_pack(w))


# ---------------------------------------------------------------------------
# decode and load check
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", ["tiny", "exhaustive", "specials", "wide"])
def test_unpack_and_load_check_bit_exact(w12, case):
    if case == "tiny":
        w = synth.weights(1024, 512, 0, synth.STREAM_LINEAR, 0.01, 0.01)
    elif case == "exhaustive":
        g = np.random.default_rng(3)
        w = g.permutation(np.arange(65536, dtype=np.uint32).astype(np.uint16)).reshape(1024, 64)
    elif case == "specials":
        w = synth.weights(384, 640, 2, 9)
        g = np.random.default_rng(4)
        idx = g.choice(w.size, 5000, replace=False)
        w.reshape(-1)[idx] = g.integers(0, 65536, size=5000).astype(np.uint16)
    else:
        w = synth.weights(5120, 1024, 5, 1)
    dw = _packed(w12, w)
    out = w12.w12_unpack(dw)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), w)
    ws = w12.Workspace(1, 128)
    assert w12.w12_load_check(dw, _dev_bf16(w), ws) == 0
    # a single flipped bit in the source is caught
    w2 = w.copy()
    w2[7, 13] ^= 0x0010
    assert w12.w12_load_check(dw, _dev_bf16(w2), ws) == 1


def test_load_check_catches_corrupted_record(w12):
    w = synth.weights(256, 256, 6, 1)
    hp = w12.w12_pack(w)
    hp.rec[100] ^= 0x08          # flips an exponent-offset bit of one weight
    dw = w12.DeviceWeight(hp)
    ws = w12.Workspace(1, 256)
    assert w12.w12_load_check(dw, _dev_bf16(w), ws) == 1


# ---------------------------------------------------------------------------
# GEMM
# ---------------------------------------------------------------------------

GEMM_CASES = [
    # (n, k, R, outlier, zeros)
    (1024, 512, 8, 0.01, 0.01),      # the small workload's linear
    (1024, 512, 1, 0.01, 0.01),
    (512, 1536, 3, 0.0, 0.0),
    (768, 2048, 16, 0.001, 0.001),
    (1024, 1024, 24, 0.0, 0.0),
    (640, 4096, 32, 0.0, 0.0),
    (384, 3072, 40, 0.0, 0.0),
    (256, 5120, 64, 0.0, 0.0),
    (512, 1024, 100, 0.0, 0.0),      # two row slices
    (256, 640, 192, 0.0, 0.001),
    (128, 512, 256, 0.0, 0.0),
    (128, 64, 5, 0.0, 0.0),          # a single record
    (9 * 128, 64 * 37, 12, 0.0, 0.0),
    (65536, 128, 8, 0.01, 0.0),      # tiles of two records: a tile end every other record
]


@pytest.mark.parametrize("n,k,R,outl,zero", GEMM_CASES)
def test_gemm_matches_oracle(w12, path, n, k, R, outl, zero):
    w = synth.weights(n, k, n + k + R, 11, outl, zero)
    x = synth.activations(R, k, n + k + R, 12)
    dw = _packed(w12, w)
    ws = w12.Workspace(R, n)
    y = w12.w12_gemm(dw, _dev_bf16(x), ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    got = synth.bf16_bits_to_f32(_bits(y)).astype(np.float64)
    ref = oracle.gemm_f64(x, oracle.w12_unpack(oracle.w12_pack(w)))
    assert H.gemm_rel_err(got, ref) <= H.GEMM_REL_TOL
    assert H.gemm_norm_err(got, ref) <= H.GEMM_REL_TOL
    # deterministic: a second run gives the same bits
    y2 = w12.w12_gemm(dw, _dev_bf16(x), ws)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_gemm_exact_integer_case(w12, path):
    """Products and sums exact in FP32 -> the BF16 output is the BF16 rounding
    of the exact integer result."""
    g = np.random.default_rng(7)
    n, k, R = 384, 1024, 20
    wi = g.choice([-1, 1], size=(n, k)) * g.integers(1, 8, size=(n, k)) * (2 ** g.integers(0, 5, size=(n, k)))
    xi = g.integers(-3, 4, size=(R, k))
    w = synth.f32_to_bf16_bits(wi.astype(np.float32))
    x = synth.f32_to_bf16_bits(xi.astype(np.float32))
    dw = _packed(w12, w)
    ws = w12.Workspace(R, n)
    y = w12.w12_gemm(dw, _dev_bf16(x), ws)
    exact = (xi.astype(np.int64) @ wi.astype(np.int64).T).astype(np.float32)
    assert np.array_equal(_bits(y), synth.f32_to_bf16_bits(exact))


# ---------------------------------------------------------------------------
# LM head argmax
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("V,K,R", [(4096, 512, 8), (8192, 1024, 33), (1280, 2560, 70), (2048, 384, 256),
                                   (65536, 128, 8)])
def test_lmhead_argmax_matches_oracle(w12, path, V, K, R):
    wh = synth.weights(V, K, V + R, 2000, 0.005, 0.005)
    h = synth.activations(R, K, V + R, 5)
    dw = _packed(w12, wh)
    ws = w12.Workspace(R, 0, V)
    maxl = torch.empty(R, dtype=torch.float32, device="cuda")
    am = w12.w12_lmhead_argmax(dw, _dev_bf16(h), ws, maxlogit=maxl)
    torch.cuda.synchronize()
    assert ws.status() == 0
    ref_am, ref_t1, ref_mg = oracle.head_argmax(h, wh)
    gated = ref_mg > H.MARGIN_GATE
    assert gated.sum() >= 0.8 * R
    got = am.cpu().numpy()
    assert np.array_equal(got[gated], ref_am[gated])
    assert np.allclose(maxl.cpu().numpy()[gated], ref_t1[gated], rtol=1e-3, atol=1e-3)


def test_lmhead_argmax_detects_planted_defect(w12):
    """The checker must fail against an oracle with the pages' planted logit
    bias (+2 on every 7th id): the mutation is caught on the GPU results."""
    V, K, R = 2048, 256, 48
    wh = synth.weights(V, K, 31, 2000)
    h = synth.activations(R, K, 31, 5)
    dw = _packed(w12, wh)
    ws = w12.Workspace(R, 0, V)
    got = w12.w12_lmhead_argmax(dw, _dev_bf16(h), ws).cpu().numpy()
    bias = np.zeros(V)
    bias[::7] = 2.0
    bad_am, _, bad_mg = oracle.head_argmax(h, wh, bias=bias)
    gated = bad_mg > H.MARGIN_GATE
    assert (got[gated] != bad_am[gated]).mean() > 0.5


# ---------------------------------------------------------------------------
# quick pass (view planes only)
# ---------------------------------------------------------------------------

QUICK_GEMM_CASES = [
    (1024, 512, 8, 0.01, 0.01),
    (640, 4096, 32, 0.0, 0.0),
    (256, 5120, 64, 0.0, 0.001),
    (512, 1024, 100, 0.0, 0.0),      # two row slices
    (128, 64, 5, 0.0, 0.0),
]


@pytest.mark.parametrize("n,k,R,outl,zero", QUICK_GEMM_CASES)
def test_gemm_quick_matches_oracle(w12, path, n, k, R, outl, zero):
    w = synth.weights(n, k, n + k + R, 21, outl, zero)
    x = synth.activations(R, k, n + k + R, 22)
    pk = oracle.w12_pack(w)
    ref = oracle.gemm_f64(x, oracle.w12_unpack_q(pk))
    dw = _packed(w12, w)
    ws = w12.Workspace(R, n)
    y = w12.w12_gemm(dw, _dev_bf16(x), ws, quick=True)
    y2 = w12.w12_gemm(dw, _dev_bf16(x), ws, quick=True)
    torch.cuda.synchronize()
    assert ws.status() == 0
    got = synth.bf16_bits_to_f32(_bits(y)).astype(np.float64)
    assert H.gemm_rel_err(got, ref) <= H.GEMM_REL_TOL
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))   # deterministic


@pytest.mark.parametrize("V,K,R", [(4096, 512, 8), (8192, 1024, 33), (2048, 384, 70), (4096, 640, 200)])
def test_lmhead_argmax_quick_matches_oracle(w12, path, V, K, R):
    wh = synth.weights(V, K, V + K, 23)
    pk = oracle.w12_pack(wh)
    wq = oracle.w12_unpack_q(pk)
    h = synth.activations(R, K, V + K, 24)
    am, _, mg = oracle.head_argmax(h, wq)
    dw = _packed(w12, wh)
    ws = w12.Workspace(R, 0, V)
    got = w12.w12_lmhead_argmax(dw, _dev_bf16(h), ws, quick=True)
    torch.cuda.synchronize()
    assert ws.status() == 0
    gated = mg > H.MARGIN_GATE
    assert gated.mean() > 0.9
    assert np.array_equal(got.cpu().numpy()[gated], am[gated])


# ---------------------------------------------------------------------------
# certified LM head: the argmax of exact FP64 logits, on every row
# ---------------------------------------------------------------------------

def _planted_rows(wh, R, seed, alpha=8.0):
    g = np.random.default_rng(seed)
    t = g.integers(0, wh.shape[0], size=R)
    hf = alpha * synth.bf16_bits_to_f32(wh[t]) + g.standard_normal((R, wh.shape[1]), dtype=np.float32)
    return synth.f32_to_bf16_bits(hf.astype(np.float32))


@pytest.mark.parametrize("V,K,R,planted", [(4096, 512, 8, True), (8192, 1024, 33, True), (2048, 384, 70, False),
                                           (4096, 640, 200, True), (1024, 256, 5, False)])
def test_lmhead_certified_matches_dense_fp64(w12, path, V, K, R, planted):
    wh = synth.weights(V, K, V + K, 31, 0.001, 0.001)
    pk = oracle.w12_pack(wh)
    h = _planted_rows(wh, R, V + R) if planted else synth.activations(R, K, V + K, 32)
    dense, _, _ = oracle.head_argmax(h, oracle.w12_unpack(pk))
    _, surv_ref, err_ref, qn_ref = oracle.certified_head(h, pk)
    dw = _packed(w12, wh)
    norms = w12.w12_head_cert_norms(dw)
    ws = w12.Workspace(R, V, V)
    cws = w12.CertWorkspace(R, V)
    surv = torch.empty(R, dtype=torch.int32, device="cuda")
    got = w12.w12_lmhead_argmax_certified(dw, norms, _dev_bf16(h), ws, cws, survivors=surv)
    got2 = w12.w12_lmhead_argmax_certified(dw, norms, _dev_bf16(h), ws, cws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert np.array_equal(got.cpu().numpy(), dense)               # every row, no margin gate
    assert torch.equal(got, got2)
    n = surv.cpu().numpy()
    assert (n >= 1).all() and (n <= 1024).all()
    nm = norms.cpu().numpy().astype(np.float64)
    assert (nm[0] >= err_ref * (1 - 1e-6)).all() and np.allclose(nm[0], err_ref, rtol=1e-5, atol=1e-12)
    assert (nm[1] >= qn_ref * (1 - 1e-6)).all() and np.allclose(nm[1], qn_ref, rtol=1e-5)


def test_lmhead_certified_separates_tokens_the_view_cannot(w12):
    """Token 1 is token 0 with other low mantissa nibbles (same view bytes):
    the quick argmax takes token 0, the certified and dense argmax token 1."""
    base = synth.weights(256, 256, 5, 45)
    g = np.random.default_rng(46)
    wh = base.copy()
    wh[1] = (wh[0] & np.uint16(0xFFF0)) | g.integers(0, 16, size=256).astype(np.uint16)
    h = np.ascontiguousarray(np.vstack([wh[1]] * 4))
    pk = oracle.w12_pack(wh)
    dense, _, _ = oracle.head_argmax(h, oracle.w12_unpack(pk))
    dw = _packed(w12, wh)
    norms = w12.w12_head_cert_norms(dw)
    ws = w12.Workspace(4, 256, 256)
    cws = w12.CertWorkspace(4, 256)
    surv = torch.empty(4, dtype=torch.int32, device="cuda")
    got = w12.w12_lmhead_argmax_certified(dw, norms, _dev_bf16(h), ws, cws, survivors=surv)
    quick = w12.w12_lmhead_argmax(dw, _dev_bf16(h), ws, quick=True)
    torch.cuda.synchronize()
    assert (dense == 1).all()
    assert (got.cpu().numpy() == 1).all() and (surv.cpu().numpy() >= 2).all()
    assert (quick.cpu().numpy() == 0).all()


# ---------------------------------------------------------------------------
# tree build and acceptance
# ---------------------------------------------------------------------------

TREE_CASES = [
    ("tiny", {}),
    ("single_27b", dict(vocab=4096, hidden=512)),
    ("batched_27b", dict(vocab=4096, hidden=512)),
    ("b4_tree", dict(vocab=4096, hidden=512)),
    ("b4_chain", dict(vocab=4096, hidden=512)),
    ("batched_27b", dict(vocab=4096, hidden=512, conditional=True, seed=3)),
    ("batched_27b", dict(vocab=4096, hidden=512, budget=512, seed=4)),
    ("batched_27b", dict(vocab=4096, hidden=512, budget=24, seed=5)),       # roots only
    ("single_27b", dict(vocab=4096, hidden=512, positions=(2,), budget=500, n_cand=3, seed=6)),  # exhausted
    ("single_27b", dict(vocab=4096, hidden=512, conditional=True, seed=7)),
    ("single_27b", dict(vocab=4096, hidden=512, budget=200, seed=8)),       # a subtree outgrows its store
    ("single_27b", dict(vocab=4096, hidden=512, budget=120, n_cand=5, seed=9)),
    ("single_27b", dict(vocab=4096, hidden=512, positions=(1,), budget=20, seed=10)),  # depth 1 only
]


def _tree_equal(t_gpu, t_ref):
    assert t_gpu["parent"].tolist() == t_ref.parent.tolist()
    assert t_gpu["token"].tolist() == t_ref.token.tolist()
    assert t_gpu["depth"].tolist() == t_ref.depth.tolist()
    assert t_gpu["req"].tolist() == t_ref.req.tolist()
    assert t_gpu["rank"].tolist() == t_ref.rank.tolist()
    assert t_gpu["score"].tobytes() == t_ref.score.tobytes()
    assert t_gpu["req_row_off"].tolist() == t_ref.req_row_off.tolist()


@pytest.mark.parametrize("name,kw", TREE_CASES)
def test_tree_build_bit_exact(w12, name, kw):
    w = synth.scaled(synth.WORKLOADS[name], **kw)
    lat = synth.lattice(w)
    ref = oracle.tree_build(lat, w.budget)
    dl = w12.DeviceLattice(lat)
    ws = w12.Workspace(1, 0, 0, w.n_req)
    t = w12.w12_tree_build(dl, w.budget, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert t.R == ref.R
    _tree_equal(t.host(), ref)


def _tree_case(w12, lat, budget):
    ref = oracle.tree_build(lat, budget)
    dl = w12.DeviceLattice(lat)
    ws = w12.Workspace(1, 0, 0, lat.n_req)
    t = w12.w12_tree_build(dl, budget, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert t.R == ref.R
    _tree_equal(t.host(), ref)


@pytest.mark.parametrize("n_req,budget", [(2, 40), (3, 7), (31, 200), (33, 100)])
def test_tree_build_request_counts(w12, n_req, budget):
    """One warp per request covers 2..32 requests; 33 goes to the one-warp build."""
    w = synth.scaled(synth.WORKLOADS["batched_27b"], vocab=4096, hidden=512, n_req=n_req, budget=budget, seed=11)
    _tree_case(w12, synth.lattice(w), budget)


def test_tree_build_one_request_dominates(w12):
    """A request whose edges are almost free takes nearly the whole budget:
    more nodes than a per-request store holds, so the build falls back to the
    one-warp selection."""
    w = synth.scaled(synth.WORKLOADS["batched_27b"], vocab=4096, hidden=512, n_req=4, budget=200, seed=12)
    lat = synth.lattice(w)
    lat.cand_logp[0] = np.float32(-1e-4)
    lat.p_r[0] = 16
    _tree_case(w12, lat, 200)


def test_tree_build_equal_scores(w12):
    """Every edge has the same log-probability: the order falls to depth,
    request and path, across the per-request warps."""
    w = synth.scaled(synth.WORKLOADS["batched_27b"], vocab=4096, hidden=512, n_req=8, budget=120, seed=13)
    lat = synth.lattice(w)
    lat.cand_logp[:] = np.float32(-0.5)
    _tree_case(w12, lat, 120)


def test_tree_build_one_request_equal_scores(w12):
    """One request split over the root's children, every edge equal: the
    order falls to depth and path across the subtree warps."""
    w = synth.scaled(synth.WORKLOADS["single_27b"], vocab=4096, hidden=512, budget=40, seed=14)
    lat = synth.lattice(w)
    lat.cand_logp[:] = np.float32(-0.5)
    _tree_case(w12, lat, 40)


def test_tree_build_flags_positive_logp(w12):
    w = synth.scaled(synth.WORKLOADS["single_27b"], vocab=4096, hidden=512)
    lat = synth.lattice(w)
    lat.cand_logp[0, 0, 0] = 0.25
    ws = w12.Workspace(1, 0, 0, 1)
    w12.w12_tree_build(w12.DeviceLattice(lat), w.budget, ws)
    assert ws.status() == w12.W12_E_INVAL


def _oracle_step(w: synth.Workload, lat, wh, n2, seed=0):
    tree = oracle.tree_build(lat, w.budget)
    h = synth.hidden_rows(tree.req, tree.parent, tree.token, lat.truth, wh, seed, head_norm2=n2)
    am, t1, mg = oracle.head_argmax(h, wh)
    tok, ln, node = oracle.tree_accept(tree, am, w.n_req, w.p_max)
    return tree, h, am, mg, tok, ln, node


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("single_27b", dict(vocab=8192, hidden=512, linears=((1024, 512), (512, 1024)))),
    ("batched_27b", dict(vocab=8192, hidden=512, linears=((1024, 512),))),
    ("b4_tree", dict(vocab=4096, hidden=256, linears=((768, 256), (256, 768)))),
    ("b4_chain", dict(vocab=4096, hidden=256, linears=((256, 256),))),
])
def test_verify_step_matches_oracle(w12, path, name, kw):
    """Whole pass through the C ABI: tree -> linears -> head argmax -> accept,
    against the oracle (accepted tokens bit-exact on margin-passing requests)."""
    w = synth.scaled(synth.WORKLOADS[name], **kw)
    lat = synth.lattice(w)
    wh = synth.weights(w.vocab, w.hidden, w.seed, synth.STREAM_HEAD, w.outlier_frac, w.zero_frac)
    n2 = synth.head_norms(wh)
    tree, h, am, mg, tok, ln, node = _oracle_step(w, lat, wh, n2, w.seed)
    R = tree.R
    lin_w = [synth.weights(n, k, w.seed, synth.STREAM_LINEAR + i, w.outlier_frac, w.zero_frac)
             for i, (n, k) in enumerate(w.linears)]
    xs = [synth.activations(R, k, w.seed, synth.STREAM_X + i) for i, (n, k) in enumerate(w.linears)]
    dls = [_packed(w12, lw) for lw in lin_w]
    dh = _packed(w12, wh)
    ws = w12.Workspace(R, max(n for n, _ in w.linears), w.vocab, w.n_req)
    dl = w12.DeviceLattice(lat)
    t = w12.w12_tree_build(dl, w.budget, ws)
    _tree_equal(t.host(), tree)
    xd = [_dev_bf16(x) for x in xs]
    yd = [torch.empty((R, n), dtype=torch.bfloat16, device="cuda") for n, _ in w.linears]
    hd = _dev_bf16(h)
    amd = torch.empty(R, dtype=torch.int32, device="cuda")
    step = w12.VerifyStep(dls, xd, yd, dh, hd, amd)
    acc_tok = torch.empty((w.n_req, w.p_max + 1), dtype=torch.int32, device="cuda")
    acc_len = torch.empty(w.n_req, dtype=torch.int32, device="cuda")
    acc_node = torch.empty(w.n_req, dtype=torch.int32, device="cuda")
    w12.w12_verify_step(step, t, w.n_req, w.p_max, ws, acc_tok, acc_len, acc_node)
    torch.cuda.synchronize()
    assert ws.status() == 0
    # linears
    for i, (lw, x) in enumerate(zip(lin_w, xs)):
        ref = oracle.gemm_f64(x, lw)
        got = synth.bf16_bits_to_f32(_bits(yd[i])).astype(np.float64)
        assert H.gemm_rel_err(got, ref) <= H.GEMM_REL_TOL
    # argmax on margin-passing rows
    gated = mg > H.MARGIN_GATE
    assert np.array_equal(amd.cpu().numpy()[gated], am[gated])
    compared, mism, near = H.accepted_parity(acc_tok.cpu().numpy(), acc_len.cpu().numpy(), tok, ln, node,
                                             tree.parent, mg, w.n_req)
    assert not mism, (mism, near)
    assert len(compared) >= 0.9 * w.n_req
    assert np.all(acc_len.cpu().numpy() >= 1)


@pytest.mark.parametrize("kernel_flag", [4, 2])
def test_bounded_wait_times_out_cleanly(w12, kernel_flag):
    """A GEMM whose first record is never copied (test hook) records
    W12_E_TIMEOUT and returns; the context stays usable."""
    w = synth.weights(1024, 512, 1, 1)
    x = synth.activations(8, 512, 1, 2)
    dw = _packed(w12, w)
    ws = w12.Workspace(8, 1024)
    w12.debug_set(1 | kernel_flag, 50_000_000)      # 50 ms limit
    try:
        w12.w12_gemm(dw, _dev_bf16(x), ws)
        torch.cuda.synchronize()
        assert ws.status() == w12.W12_E_TIMEOUT
    finally:
        w12.debug_set(0, 0)
    ws2 = w12.Workspace(8, 1024)
    y = w12.w12_gemm(dw, _dev_bf16(x), ws2)
    torch.cuda.synchronize()
    assert ws2.status() == 0
    ref = oracle.gemm_f64(x, w)
    assert H.gemm_rel_err(synth.bf16_bits_to_f32(_bits(y)).astype(np.float64), ref) <= H.GEMM_REL_TOL
