"""Pins of the CPU oracle against facts fixed by the pages and by
mathematics, not against the oracle itself (CPU only).

Each test names what it pins and the passage it follows (SpecPilot
explainer sections unless stated otherwise)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_w12_gb300 import synth
from tests import helpers as H


# ---------------------------------------------------------------------------
# W12 (explainer 4.1; summary's W12 paragraph)
# ---------------------------------------------------------------------------

def _roundtrip(w):
    p = oracle.w12_pack(w)
    assert np.array_equal(oracle.w12_unpack(p), w)
    return p


def test_w12_exhaustive_bf16_ordered():
    """Every BF16 bit pattern restores bit-exactly (lossless, 4.1)."""
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(1024, 64)
    p = _roundtrip(allp)
    # each row of 64 consecutive patterns holds one exponent field; only the
    # rows whose field is 0 (zeros, denormals) or 255 (Inf, NaN) escape:
    # 4 rows each (two signs, two halves of the mantissa) -> 8 * 64 slots
    assert p.n_escapes == 8 * 64


def test_w12_exhaustive_bf16_shuffled():
    """All 65536 patterns scattered over channels, so windows mix binades."""
    g = np.random.default_rng(1)
    allp = g.permutation(np.arange(65536, dtype=np.uint32).astype(np.uint16)).reshape(1024, 64)
    _roundtrip(allp)
    allp2 = g.permutation(allp.reshape(-1)).reshape(256, 256)
    _roundtrip(allp2)


def test_w12_special_values():
    """Signed zeros, denormals, Inf and NaN payloads are restored verbatim."""
    w = synth.weights(128, 128, 5, 0)
    specials = np.array([0x0000, 0x8000, 0x0001, 0x807F, 0x7F80, 0xFF80, 0x7FC1, 0xFFFF, 0x0080, 0x7F7F],
                        np.uint16)
    g = np.random.default_rng(2)
    idx = g.choice(w.size, size=400, replace=False)
    w.reshape(-1)[idx] = specials[np.arange(400) % specials.size]
    _roundtrip(w)


def test_w12_golden_record_bytes():
    """Hand-derived record bytes, window bases and escape entries."""
    fx = H.load_golden("w12_record_bytes.json")
    w = np.full((fx["n"], fx["k"]), fx["fill"], np.uint16)
    for e in fx["weights"]:
        w[e["n"], e["k"]] = int(e["bf16"], 16)
    p = oracle.w12_pack(w)
    assert np.all(p.base == fx["base_all"])
    expect = np.zeros(12288, np.uint8)
    for off, val in fx["nonzero_record_bytes"].items():
        expect[int(off)] = val
    assert np.array_equal(p.rec, expect)
    assert [hex(int(v)) for v in p.esc] == [hex(int(v, 16)) for v in fx["escapes"]]
    assert p.esc_tile_off.tolist() == fx["esc_tile_off"]


def _channel_with_exponents(counts, k=64, sign_mix=False):
    """One channel (padded to 128 identical rows) whose weights have the given
    exponent-field multiset; remaining slots are +0."""
    row = np.zeros(k, np.uint16)
    i = 0
    for e, c in counts.items():
        for _ in range(c):
            s = (i % 2) if sign_mix else 0
            row[i] = (s << 15) | (e << 7) | (i % 128)
            i += 1
    return np.tile(row, (128, 1))


@pytest.mark.parametrize("counts,expect_b", [
    ({100: 10, 120: 5, 130: 20}, 120),   # 120 and 130 fit one window; largest base wins ties
    ({121: 64}, 121),                    # one binade: any base in [106,121] covers it -> 121
    ({250: 30, 240: 2}, 239),            # the window cannot start above 239
    ({1: 40}, 1),                        # smallest normal exponent
    ({}, 1),                             # no normal weights at all -> base 1, all escape
    ({110: 8, 126: 8, 127: 1}, 126),     # 110 never shares a window with 126; [112..126, +15] hold 9
    ({110: 8, 125: 9, 127: 1}, 110),     # [110,125] holds 17, beating [112..125, +15] with 10
])
def test_w12_window_choice_hand_cases(counts, expect_b):
    """Window = 16 binades covering most of the channel's weights (4.1)."""
    w = _channel_with_exponents(counts, sign_mix=True)
    p = _roundtrip(w)
    assert int(p.base[0]) == expect_b
    inside = sum(c for e, c in counts.items() if expect_b <= e <= expect_b + 15)
    assert p.n_escapes == 128 * (64 - inside)


def test_w12_single_binade_offsets_constant():
    """A channel whose weights share one binade stores one offset value."""
    w = _channel_with_exponents({121: 64})
    p = oracle.w12_pack(w)
    view = p.rec[:8192].reshape(4, 128, 16)
    offs = (view >> 3) & 0xF
    assert np.all(offs == 0) and np.all((view >> 7) == 0)


def test_w12_zero_channel_all_escapes():
    w = np.zeros((128, 64), np.uint16)
    w[:, ::2] = 0x8000
    p = _roundtrip(w)
    assert p.n_escapes == 128 * 64 and np.all(p.rec == 0)


def test_w12_gaussian_escape_rate_and_bits():
    """Soft check against the page's 7.33e-5 escapes and 12.013-12.020
    bits/weight (4.1): Gaussian synthetic weights land in the same regime."""
    w = synth.weights(2048, 2048, 0, 77)
    p = _roundtrip(w)
    rate = p.n_escapes / w.size
    bits = 8.0 * p.bytes / w.size
    assert 1e-5 < rate < 3e-4, rate
    assert 12.0 < bits < 12.03, bits


# ---------------------------------------------------------------------------
# Quick pass (explainer 4.1, 4.3; reading R19)
# ---------------------------------------------------------------------------

def _quick_closed_form(w: np.ndarray, base: np.ndarray) -> np.ndarray:
    """From the source bits alone: escaped weights (exponent field outside
    [b, b+15]) stay exact; every other weight keeps its upper 12 bits and
    takes 0b1000 as its low mantissa nibble."""
    e = (w.astype(np.int64) >> 7) & 0xFF
    b = base.astype(np.int64)[:, None]
    escaped = (e < b) | (e > b + 15)
    return np.where(escaped, w, (w & 0xFFF0) | 0x0008).astype(np.uint16)


def test_quick_decode_closed_form_gaussian_with_escapes():
    w = synth.weights(512, 256, 4, 31, 0.01, 0.01)
    p = oracle.w12_pack(w)
    assert p.n_escapes > 0
    assert np.array_equal(oracle.w12_unpack_q(p), _quick_closed_form(w, p.base))


def test_quick_decode_closed_form_every_bf16_pattern():
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(1024, 64)
    p = oracle.w12_pack(w)
    assert np.array_equal(oracle.w12_unpack_q(p), _quick_closed_form(w, p.base))


def test_quick_decode_is_exact_when_low_nibble_is_the_midpoint():
    w = synth.weights(256, 128, 5, 32)
    w = ((w & 0xFFF0) | 0x0008).astype(np.uint16)
    p = oracle.w12_pack(w)
    assert np.array_equal(oracle.w12_unpack_q(p), oracle.w12_unpack(p))


def test_quick_decode_error_bound():
    """An in-window quick weight differs from the exact one by at most half
    of its low-nibble range: |q - w| <= 8 units of the last mantissa place."""
    w = synth.weights(256, 128, 6, 33)
    p = oracle.w12_pack(w)
    q = oracle.w12_unpack_q(p)
    diff = np.abs((q.astype(np.int64) & 0xF) - (w.astype(np.int64) & 0xF))
    assert diff.max() <= 8
    assert np.array_equal(q & 0xFFF0, w & 0xFFF0)


# ---------------------------------------------------------------------------
# GEMM (explainer 1.1, 2.1) and LM-head argmax
# ---------------------------------------------------------------------------

def test_gemm_matches_numpy_float64():
    w = synth.weights(256, 512, 3, 1, 0.01, 0.01)
    x = synth.activations(9, 512, 3, 2)
    y = oracle.gemm_f64(x, oracle.w12_unpack(oracle.w12_pack(w)))
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ synth.bf16_bits_to_f32(w).astype(np.float64).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_gemm_exact_integer_case():
    """Weights +-2^j * m and small-integer activations: the exact sum is an
    integer computed here with Python ints."""
    g = np.random.default_rng(4)
    n, k, R = 128, 192, 5
    mant = g.integers(1, 8, size=(n, k))
    expo = g.integers(0, 6, size=(n, k))
    sign = g.choice([-1, 1], size=(n, k))
    wi = sign * mant * (2 ** expo)
    xi = g.integers(-4, 5, size=(R, k))
    w = synth.f32_to_bf16_bits(wi.astype(np.float32))
    x = synth.f32_to_bf16_bits(xi.astype(np.float32))
    y = oracle.gemm_f64(x, w)
    exact = np.array([[sum(int(a) * int(b) for a, b in zip(xi[r], wi[c])) for c in range(n)] for r in range(R)])
    assert np.array_equal(y, exact.astype(np.float64))


def test_head_argmax_planted_rows():
    """Rows planted on a token pick that token with a wide margin."""
    V, K = 2048, 512
    wh = synth.weights(V, K, 6, 2000)
    n2 = synth.head_norms(wh)
    truth = np.asarray([[5, 77, 1999, 3]], np.int32)
    rows = np.stack([synth.hidden_row(0, list(truth[0, :d]), truth, wh, n2, 0) for d in range(3)])
    am, t1, mg = oracle.head_argmax(rows, wh)
    assert am.tolist() == [int(truth[0, d]) for d in range(3)]
    assert np.all(mg > 1.0)


def test_head_argmax_ties_nan_and_numpy():
    """Lowest index on ties, NaN never wins; argmax and margins agree with
    NumPy on FP64 logits (a library routine)."""
    V, K = 512, 64
    wh = np.zeros((V, K), np.uint16)
    one = 0x3F80
    wh[[7, 9, 300], 0] = one        # three tokens share the top logit
    wh[11, 0] = 0x3F00              # 0.5
    h = np.zeros((2, K), np.uint16)
    h[0, 0] = one
    h[1, 1] = 0x7FC0                # NaN input to column 1 -> logits of tokens with w[:,1] != 0 are NaN
    wh[400, 1] = one
    am, t1, mg = oracle.head_argmax(h, wh)
    assert am[0] == 7 and mg[0] == 0.0 and t1[0] == 1.0
    # row 1: every logit is 0 except token 400, whose logit is NaN * 1 = NaN
    assert am[1] == 0
    g = np.random.default_rng(8)
    wh2 = synth.weights(V, K, 9, 1)
    h2 = synth.activations(6, K, 9, 2)
    am2, t12, mg2 = oracle.head_argmax(h2, wh2, nthreads=3)
    lg = synth.bf16_bits_to_f32(h2).astype(np.float64) @ synth.bf16_bits_to_f32(wh2).astype(np.float64).T
    assert am2.tolist() == np.argmax(lg, axis=1).tolist()
    srt = np.sort(lg, axis=1)
    assert np.allclose(mg2, srt[:, -1] - srt[:, -2], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# best-first tree (explainer 4.2, 4.4)
# ---------------------------------------------------------------------------

def _tiny_lattice(n_req, p_max, n_cand, conditional, seed, positions=None):
    w = synth.Workload("t", ((128, 64),), vocab=97, hidden=64, n_req=n_req,
                       positions=positions or (p_max,), budget=1, n_cand=n_cand,
                       conditional=conditional, seed=seed)
    return synth.lattice(w)


def _check_tree_vs_brute(lat, budget):
    t = oracle.tree_build(lat, budget)
    ref = H.brute_tree(lat, budget)
    assert t.R == len(ref)
    for i, row in enumerate(ref):
        assert t.parent[i] == row["parent"], i
        assert t.token[i] == row["token"], i
        assert t.depth[i] == row["depth"], i
        assert t.req[i] == row["req"], i
        assert t.score[i].tobytes() == np.float32(row["score"]).tobytes(), i
        assert t.rank[i] == row["rank"], i
    return t


@pytest.mark.parametrize("n_req,p_max,n_cand,cond,budget,seed", [
    (1, 4, 4, False, 20, 0),
    (3, 4, 4, False, 40, 1),
    (2, 3, 5, True, 30, 2),
    (4, 2, 16, False, 64, 3),
    (2, 4, 4, True, 200, 4),     # budget larger than some requests' trees
    (5, 3, 3, False, 5, 5),      # roots only
])
def test_tree_matches_brute_force_top_budget(n_req, p_max, n_cand, cond, budget, seed):
    """Best-first = the top-budget nodes under the order key, found here by
    enumerating every node of the lattice (4.2: keep the N nodes with the
    highest path score)."""
    lat = _tiny_lattice(n_req, p_max, n_cand, cond, seed)
    _check_tree_vs_brute(lat, budget)


def test_tree_varied_depth_limits_brute_force():
    lat = _tiny_lattice(4, 4, 3, False, 11, positions=(1, 2, 4))
    _check_tree_vs_brute(lat, 50)


def test_tree_invariants_shared_budget():
    """Prefix-closed, every root present, scores never rise along a path,
    each request's share is a valid tree (4.4)."""
    w = synth.scaled(synth.WORKLOADS["batched_27b"], vocab=4096, hidden=512)
    lat = synth.lattice(w)
    t = oracle.tree_build(lat, w.budget)
    assert t.R == w.budget
    for r in range(w.n_req):
        lo, hi = t.req_row_off[r], t.req_row_off[r + 1]
        assert hi > lo and t.parent[lo] == -1 and t.depth[lo] == 0 and t.token[lo] == lat.root_tok[r]
        for j in range(lo + 1, hi):
            p = t.parent[j]
            assert lo <= p < j and t.depth[j] == t.depth[p] + 1 and t.req[j] == r
            assert t.score[j] <= t.score[p]
            assert t.depth[j] <= lat.p_r[r]
            assert t.token[j] == lat.cand_tok[r, t.depth[j] - 1, t.rank[j]]


def test_tree_chain_mode_is_rank0_chain():
    """n_cand = 1 reduces to stock's chain: depth d holds position d's top
    candidate (1.1, 2.1)."""
    lat = _tiny_lattice(1, 8, 1, False, 3)
    t = oracle.tree_build(lat, 9)
    assert t.R == 9
    assert t.parent.tolist() == [-1] + list(range(8))
    assert t.token[1:].tolist() == lat.cand_tok[0, :, 0].tolist()


def test_tree_rejects_positive_logp():
    lat = _tiny_lattice(1, 3, 4, False, 3)
    lat.cand_logp[0, 1, 2] = 0.5
    with pytest.raises(ValueError):
        oracle.tree_build(lat, 10)


# ---------------------------------------------------------------------------
# greedy acceptance (explainer 1.1; poot-llm docs: greedy rows keep drafts
# equal to the argmax, then the target's own token)
# ---------------------------------------------------------------------------

def test_accept_matches_brute_force_paths():
    g = np.random.default_rng(12)
    lat = _tiny_lattice(3, 4, 4, False, 12)
    t = oracle.tree_build(lat, 60)
    for trial in range(30):
        # argmax rows biased towards the tree's own tokens so long paths occur
        am = g.integers(0, 97, size=t.R).astype(np.int32)
        for j in range(t.R):
            kids = [c for c in range(t.R) if t.parent[c] == j]
            if kids and g.random() < 0.7:
                am[j] = t.token[kids[g.integers(len(kids))]]
        tok, ln, node = oracle.tree_accept(t, am, lat.n_req, lat.p_max)
        best = H.brute_accept(t.parent, t.token, t.depth, t.req, lat.n_req, am)
        for r in range(lat.n_req):
            d = best[r]
            assert node[r] == d and ln[r] == t.depth[d] + 1
            assert 1 <= ln[r] <= lat.p_r[r] + 1
            path = []
            cur = d
            while t.parent[cur] >= 0:
                path.append(int(t.token[cur]))
                cur = t.parent[cur]
            assert tok[r, :ln[r]].tolist() == path[::-1] + [int(am[d])]


def test_accept_chain_reduces_to_prefix_rule():
    """On a chain, tau = 1 + longest prefix of drafts equal to the argmax of
    the previous position (1.1)."""
    g = np.random.default_rng(13)
    lat = _tiny_lattice(1, 8, 1, False, 13)
    t = oracle.tree_build(lat, 9)
    drafts = t.token[1:].tolist()
    for _ in range(20):
        am = g.integers(0, 97, size=9).astype(np.int32)
        m = g.integers(0, 9)
        am[:m] = drafts[:m]
        tok, ln, node = oracle.tree_accept(t, am, 1, 8)
        n = 0
        while n < 8 and am[n] == drafts[n]:
            n += 1
        assert ln[0] == n + 1 and tok[0, :n + 1].tolist() == drafts[:n] + [int(am[n])]


def _target_argmax_for_tree(t, truth, wh, n2, seed=0):
    rows = synth.hidden_rows(t.req, t.parent, t.token, truth, wh, seed, head_norm2=n2)
    am, _, mg = oracle.head_argmax(rows, wh)
    return am, mg


def test_worked_example_chain_vs_tree():
    """Section 2.4's scenario: the chain commits 'mat is a' (tau 3); the tree
    keeps mat -> is -> a -> place and accepts four drafts plus the bonus."""
    fx = H.load_golden("worked_example_2_4.json")
    V, K = 256, 64
    wh = synth.weights(V, K, 21, 2000)
    n2 = synth.head_norms(wh)
    inv = {v: k for k, v in fx["tokens"].items()}
    for mode, n_cand, budget, exp in (("chain", 1, fx["positions"] + 1, fx["chain_expected"]),
                                      ("tree", 16, fx["tree_budget"], fx["tree_expected"])):
        lat, tok = H.lattice_from_fixture(fx, n_cand=n_cand)
        t = oracle.tree_build(lat, budget)
        am, mg = _target_argmax_for_tree(t, lat.truth, wh, n2)
        acc, ln, node = oracle.tree_accept(t, am, 1, lat.p_max)
        assert ln[0] == exp["tau"], mode
        assert [inv.get(int(v), v) for v in acc[0, :ln[0]]] == exp["tokens"], mode


@pytest.mark.parametrize("n_req,budget,seed", [(1, 32, 0), (6, 60, 1), (3, 40, 2)])
def test_accept_equals_greedy_autoregressive(n_req, budget, seed):
    """The pages' invariant (explainer 1.2; poot-llm docs 'What a round
    guarantees' and its digest check): with a target whose row depends only on
    the root path, the accepted tokens are exactly the first tau tokens of
    greedy decoding without speculation, and tau - 1 is the longest prefix of
    that sequence present as a root path of the tree."""
    V, K = 1024, 128
    w = synth.Workload("ar", ((128, 64),), vocab=V, hidden=K, n_req=n_req,
                       positions=(6, 4), budget=budget, seed=seed)
    lat = synth.lattice(w)
    wh = synth.weights(V, K, seed, 2000)
    n2 = synth.head_norms(wh)
    t = oracle.tree_build(lat, budget)
    am, mg = _target_argmax_for_tree(t, lat.truth, wh, n2, seed)
    acc, ln, node = oracle.tree_accept(t, am, n_req, lat.p_max)
    paths = synth.tree_paths(t.parent, t.token)
    for r in range(n_req):
        # greedy autoregressive decoding with the same row function
        seq = []
        for step in range(int(lat.p_r[r]) + 1):
            row = synth.hidden_row(r, seq, lat.truth, wh, n2, seed)
            a, _, m = oracle.head_argmax(row[None, :], wh)
            assert m[0] > H.MARGIN_GATE
            seq.append(int(a[0]))
        mine = {tuple(paths[j]) for j in range(t.R) if t.req[j] == r}
        n = 0
        while n < lat.p_r[r] and tuple(seq[:n + 1]) in mine:
            n += 1
        assert ln[r] == n + 1
        assert acc[r, :ln[r]].tolist() == seq[:n + 1]


def test_planted_defect_is_caught():
    """The pages' defective system (summary: a logit bias of 2 on every 7th
    vocabulary id) must break argmax parity against the unmutated oracle on
    rows whose target preference is not decisive."""
    V, K = 2048, 256
    wh = synth.weights(V, K, 31, 2000)
    h = synth.activations(64, K, 31, 5)
    am, _, mg = oracle.head_argmax(h, wh)
    bias = np.zeros(V)
    bias[::7] = 2.0
    am_bad, _, _ = oracle.head_argmax(h, wh, bias=bias)
    gated = mg > H.MARGIN_GATE
    assert gated.sum() > 32
    assert (am_bad[gated] != am[gated]).mean() > 0.5
    assert (am_bad % 7 == 0).mean() > 0.9


# ---------------------------------------------------------------------------
# Certified LM head (explainer "4.1"/"4.3": cheap pass, per-row Cauchy-Schwarz
# bound, exact rescoring of the survivors; the argmax never changes)
# ---------------------------------------------------------------------------

def test_certified_head_equals_dense_argmax():
    w = synth.weights(640, 256, 3, 41, 0.002, 0.002)      # Gaussian, with escapes
    h = synth.activations(24, 256, 3, 42)
    p = oracle.w12_pack(w)
    am, surv, err, qn = oracle.certified_head(h, p)
    dense, _, _ = oracle.head_argmax(h, oracle.w12_unpack(p))
    assert np.array_equal(am, dense)
    assert (surv >= 1).all() and (surv < 640).all()
    assert (err >= 0).all() and (qn > 0).all()


def test_certified_head_bound_holds():
    """|h.w_v - h.w^_v| <= ||h|| ||w_v - w^_v|| for every row and token
    (Cauchy-Schwarz), checked on logits computed separately."""
    w = synth.weights(384, 192, 4, 43, 0.003, 0.003)
    h = synth.activations(16, 192, 4, 44)
    p = oracle.w12_pack(w)
    _, _, err, _ = oracle.certified_head(h, p)
    s = oracle.gemm_f64(h, oracle.w12_unpack(p))
    sq = oracle.gemm_f64(h, oracle.w12_unpack_q(p))
    hn = np.sqrt((synth.bf16_bits_to_f32(h).astype(np.float64) ** 2).sum(axis=1))
    assert (np.abs(s - sq) <= hn[:, None] * err[None, :] * (1 + 1e-9) + 1e-12).all()


def test_certified_head_separates_tokens_the_view_cannot():
    """Token 1 is token 0 with other low mantissa nibbles: the two share their
    view bytes, so the cheap pass scores them alike.  With h = w_1 the exact
    argmax is token 1; the cheap argmax (lowest index on its tie) is token 0;
    the certified head keeps both and returns token 1."""
    base = synth.weights(128, 128, 5, 45)
    g = np.random.default_rng(46)
    w = base.copy()
    w[1] = (w[0] & np.uint16(0xFFF0)) | g.integers(0, 16, size=128).astype(np.uint16)
    h = np.ascontiguousarray(np.vstack([w[1], w[1]]))
    p = oracle.w12_pack(w)
    dense, _, _ = oracle.head_argmax(h, oracle.w12_unpack(p))
    quick, _, _ = oracle.head_argmax(h, oracle.w12_unpack_q(p))
    am, surv, _, _ = oracle.certified_head(h, p)
    assert (dense == 1).all() and (quick == 0).all()
    assert np.array_equal(am, dense) and (surv >= 2).all()
