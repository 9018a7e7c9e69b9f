"""Pins of the oracle's TLV commit chain and splice (SpecPilot explainer,
4.3: Q pass over the first tree, commit chain, fresh subtree from the chain
end truncated to the budget left, one exact pass over the combined tree).

Each pin checks the oracle against something other than its own code: trees
written out by hand from the rules, greedy autoregressive decoding under a
toy target (the exact pass over the combined tree must reproduce it whatever
the Q pass got wrong), and the structural invariants of a best-first tree."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_w12_gb300 import synth
from tests import helpers as H


def _tree(parent, token, score, rank, row_off, req=None):
    parent = np.asarray(parent, np.int32)
    depth = np.zeros(len(parent), np.uint8)
    for j, p in enumerate(parent):
        depth[j] = 0 if p < 0 else depth[p] + 1
    if req is None:
        req = np.zeros(len(parent), np.int32)
    return oracle.Tree(len(parent), parent, np.asarray(token, np.int32), depth, np.asarray(req, np.int32),
                       np.asarray(score, np.float32), np.asarray(rank, np.uint8), np.asarray(row_off, np.int32))


def _cycle(w, p2, err, seed):
    """One TLV cycle in the oracle, the target being the toy greedy target."""
    truth = H.tlv_truth(w, p2, seed)
    lat1 = synth.lattice(w, seed, truth=truth[:, :w.p_max + 1])
    t1 = oracle.tree_build(lat1, w.budget)
    exact1 = H.target_argmax(t1, truth, w.vocab, seed)
    qarg = H.q_argmax(exact1, err, w.vocab, seed)
    c_tok, c_len, c_node = oracle.tree_accept(t1, qarg, w.n_req, w.p_max)
    m, sub = oracle.tlv_chain(c_len, t1.req_row_off, w.budget)
    w2 = synth.scaled(w, positions=(p2,))
    lat2 = H.second_lattice(w2, lat1, c_tok, m, truth, seed)
    t2 = oracle.tree_build(lat2, sub)
    tc = oracle.tlv_splice(t1, c_tok, c_len, c_node, m, t2, w.n_req)
    p_comb = w.p_max + 1 + p2
    exact = H.target_argmax(tc, truth, w.vocab, seed)
    a_tok, a_len, a_node = oracle.tree_accept(tc, exact, w.n_req, p_comb)
    s_tok, s_len, _ = oracle.tree_accept(t1, exact1, w.n_req, w.p_max)
    return dict(truth=truth, t1=t1, c_tok=c_tok, c_len=c_len, c_node=c_node, m=m, sub=sub, t2=t2, tc=tc,
                a_tok=a_tok, a_len=a_len, s_len=s_len, p_comb=p_comb)


def test_hand_example_with_bonus():
    # first tree: root 5 -> {7 (row 1), 9 (row 2)}, 7 -> 3 (row 3); the Q pass
    # prefers 7 at the root, 3 after 7 and 11 after 3
    t1 = _tree([-1, 0, 0, 1], [5, 7, 9, 3], [0, -0.5, -1.0, -1.25], [0, 0, 1, 0], [0, 4])
    qarg = np.array([7, 3, 8, 11], np.int32)
    c_tok, c_len, c_node = oracle.tree_accept(t1, qarg, 1, 2)
    assert list(c_tok[0]) == [7, 3, 11] and c_len[0] == 3 and c_node[0] == 3
    m, sub = oracle.tlv_chain(c_len, t1.req_row_off, 6)
    assert list(m) == [3] and sub == 3          # N - |C| with N = 6, |C| = 3
    # fresh subtree from the chain end 11: 11 -> {4, 6}
    t2 = _tree([-1, 0, 0], [11, 4, 6], [0, -0.25, -2.0], [0, 0, 1], [0, 3])
    tc = oracle.tlv_splice(t1, c_tok, c_len, c_node, m, t2, 1)
    assert tc.R == 6
    assert list(tc.parent) == [-1, 0, 1, 2, 3, 3]
    assert list(tc.token) == [5, 7, 3, 11, 4, 6]
    assert list(tc.depth) == [0, 1, 2, 3, 4, 4]
    assert list(tc.rank) == [0, 0, 0, oracle.BONUS_RANK, 0, 1]
    assert list(tc.score) == [0.0, -0.5, -1.25, -1.25, -1.5, -3.25]
    assert list(tc.req_row_off) == [0, 6]


def test_hand_example_cap_drops_the_bonus():
    # the whole first tree is the accepted chain root 5 -> 7 -> 3, so the
    # chain keeps 7, 3 (N_q - 1 = 2) and the subtree hangs under 3
    t1 = _tree([-1, 0, 1], [5, 7, 3], [0, -0.5, -1.0], [0, 0, 0], [0, 3])
    qarg = np.array([7, 3, 11], np.int32)
    c_tok, c_len, c_node = oracle.tree_accept(t1, qarg, 1, 2)
    assert c_len[0] == 3
    m, sub = oracle.tlv_chain(c_len, t1.req_row_off, 3)
    assert list(m) == [2] and sub == 1
    t2 = _tree([-1], [3], [0], [0], [0, 1])
    tc = oracle.tlv_splice(t1, c_tok, c_len, c_node, m, t2, 1)
    assert list(tc.parent) == [-1, 0, 1] and list(tc.token) == [5, 7, 3] and list(tc.rank) == [0, 0, 0]


def test_hand_example_two_requests_shared_budget():
    # request 0: root 5 -> 7 (accepted, bonus 2); request 1: root 8 -> {1, 4},
    # Q argmax at its root is 6 (no child): chain = the bonus 6 alone
    t1 = _tree([-1, 0, -1, 2, 2], [5, 7, 8, 1, 4], [0, -0.1, 0, -0.3, -0.9], [0, 0, 0, 0, 1], [0, 2, 5],
               req=[0, 0, 1, 1, 1])
    qarg = np.array([7, 2, 6, 0, 0], np.int32)
    c_tok, c_len, c_node = oracle.tree_accept(t1, qarg, 2, 1)
    assert list(c_len) == [2, 1]
    m, sub = oracle.tlv_chain(c_len, t1.req_row_off, 5)
    assert list(m) == [1, 1] and sub == 3       # request 0 keeps N_0 - 1 = 1: the bonus goes
    t2 = _tree([-1, -1, 1], [7, 6, 9], [0, 0, -0.5], [0, 0, 3], [0, 1, 3], req=[0, 1, 1])
    tc = oracle.tlv_splice(t1, c_tok, c_len, c_node, m, t2, 2)
    assert list(tc.req_row_off) == [0, 2, 5]
    assert list(tc.parent) == [-1, 0, -1, 2, 3]
    assert list(tc.token) == [5, 7, 8, 6, 9]
    assert list(tc.depth) == [0, 1, 0, 1, 2]
    assert list(tc.rank) == [0, 0, 0, oracle.BONUS_RANK, 3]


def test_splice_refuses_inconsistent_inputs():
    t1 = _tree([-1, 0], [5, 7], [0, -0.5], [0, 0], [0, 2])
    qarg = np.array([7, 3], np.int32)
    c_tok, c_len, c_node = oracle.tree_accept(t1, qarg, 1, 1)
    m, _ = oracle.tlv_chain(c_len, t1.req_row_off, 4)
    bad_root = _tree([-1, 0], [99, 4], [0, -0.5], [0, 0], [0, 2])
    with pytest.raises(ValueError):
        oracle.tlv_splice(t1, c_tok, c_len, c_node, m, bad_root, 1)
    with pytest.raises(ValueError):
        oracle.tlv_splice(t1, c_tok, c_len, c_node, np.array([3], np.int32), bad_root, 1)


CASES = [
    ("single", dict(n_req=1, positions=(8,), budget=24, vocab=64, n_cand=16), 6),
    ("single_deep", dict(n_req=1, positions=(16,), budget=32, vocab=64, n_cand=16), 16),
    ("batched", dict(n_req=5, positions=(2, 4, 6), budget=40, vocab=64, n_cand=16), 5),
    ("chain", dict(n_req=3, positions=(6,), budget=12, vocab=64, n_cand=1), 4),
    ("roots_only_left", dict(n_req=4, positions=(3,), budget=8, vocab=64, n_cand=16), 3),
]


@pytest.mark.parametrize("name,kw,p2", CASES)
@pytest.mark.parametrize("err", [0.0, 0.35, 1.0])
def test_exact_pass_over_spliced_tree_is_greedy_ar(name, kw, p2, err):
    """Losslessness: whatever the Q pass chose, the exact pass over the
    combined tree accepts a prefix of greedy autoregressive decoding."""
    for seed in range(6):
        w = synth.scaled(synth.WORKLOADS["tiny"], hit_rate=0.9, seed=seed, **kw)
        c = _cycle(w, p2, err, seed)
        for q in range(w.n_req):
            n = int(c["a_len"][q])
            assert n >= 1
            ar = H.greedy_ar(q, c["truth"], w.vocab, seed, n)
            assert list(c["a_tok"][q][:n]) == ar, (name, seed, q)


@pytest.mark.parametrize("name,kw,p2", CASES)
def test_perfect_q_pass_commits_the_whole_chain(name, kw, p2):
    """With a Q pass that agrees with the exact one everywhere, the exact
    pass accepts every committed chain token plus at least one more, so it
    never accepts fewer tokens than a single pass over the first tree."""
    for seed in range(6):
        w = synth.scaled(synth.WORKLOADS["tiny"], hit_rate=0.9, seed=seed, **kw)
        c = _cycle(w, p2, 0.0, seed)
        assert np.all(c["a_len"] >= c["m"] + 1)
        assert np.all(c["a_len"] >= c["s_len"])


@pytest.mark.parametrize("name,kw,p2", CASES)
@pytest.mark.parametrize("err", [0.0, 0.5])
def test_spliced_tree_invariants(name, kw, p2, err):
    for seed in range(4):
        w = synth.scaled(synth.WORKLOADS["tiny"], hit_rate=0.9, seed=seed, **kw)
        c = _cycle(w, p2, err, seed)
        tc, t1, t2, m = c["tc"], c["t1"], c["t2"], c["m"]
        assert tc.R == int(m.sum()) + t2.R <= w.budget
        assert c["sub"] >= w.n_req
        off = tc.req_row_off
        for q in range(w.n_req):
            lo, hi = int(off[q]), int(off[q + 1])
            assert hi - lo == int(m[q]) + int(t2.req_row_off[q + 1] - t2.req_row_off[q])
            assert tc.parent[lo] == -1 and tc.token[lo] == t1.token[t1.req_row_off[q]]
            assert np.all(tc.req[lo:hi] == q)
            # the chain is the committed prefix of C, one row per depth
            assert list(tc.token[lo + 1:lo + 1 + int(m[q])]) == list(c["c_tok"][q][:int(m[q])])
            for j in range(lo + 1, hi):
                p = int(tc.parent[j])
                assert lo <= p < j
                assert tc.depth[j] == tc.depth[p] + 1
                assert tc.score[j] <= tc.score[p]
            # siblings carry distinct tokens
            kids = {}
            for j in range(lo + 1, hi):
                kids.setdefault(int(tc.parent[j]), []).append(int(tc.token[j]))
            assert all(len(v) == len(set(v)) for v in kids.values())
