"""Pins of the oracle's recurrent-layer tree verification (SpecPilot
explainer, 4.2: a Gated DeltaNet head keeps a fixed-size state updated by
one rank-one step per token; over a tree the state is recomputed along each
root path from the committed state).

Each pin checks the oracle against something other than its own loop:
special cases with closed forms (no write: pure decay; a unit key written
with full strength reads back its value), independence of a node's output
from rows off its root path, and an independent restatement of the whole
tree as one triangular solve plus matrix products (the WY form the CUDA
kernel follows), which must agree to FP64 rounding."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_w12_gb300 import synth
from tests import helpers as H


def _tree(lat_kw, seed):
    w = synth.scaled(synth.WORKLOADS["tiny"], hit_rate=0.9, seed=seed, **lat_kw)
    return oracle.tree_build(synth.lattice(w, seed), w.budget), w


TREES = [
    dict(n_req=1, positions=(16,), budget=32, vocab=64, n_cand=16),
    dict(n_req=1, positions=(8,), budget=9, vocab=64, n_cand=1),
    dict(n_req=3, positions=(2, 4, 6), budget=30, vocab=64, n_cand=16),
]


def _path(tree, j):
    p = []
    while j >= 0:
        p.append(j)
        j = int(tree.parent[j])
    return p[::-1]


@pytest.mark.parametrize("kw", TREES)
def test_no_write_is_pure_decay(kw):
    t, w = _tree(kw, 1)
    x = synth.gdn_inputs(t.R, w.n_req, 3, 16, seed=2)
    beta = np.zeros_like(x.beta)
    o = oracle.gdn_tree_path(x.S0, x.q, x.k, x.v, x.alpha, beta, t)
    qf = synth.bf16_bits_to_f32(x.q).astype(np.float64)
    for j in range(t.R):
        g = np.prod([x.alpha[i].astype(np.float64) for i in _path(t, j)], axis=0)       # [H]
        ref = g[:, None] * np.einsum("hvk,hk->hv", x.S0[t.req[j]].astype(np.float64), qf[j])
        assert np.allclose(o[j], ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("kw", TREES)
def test_unit_key_written_at_full_strength_reads_back_its_value(kw):
    t, w = _tree(kw, 3)
    Hh, d = 2, 16
    x = synth.gdn_inputs(t.R, w.n_req, Hh, d, seed=4)
    g = np.random.default_rng(5)
    basis = g.integers(0, d, size=(t.R, Hh))
    k = np.zeros((t.R, Hh, d), np.float32)
    for j in range(t.R):
        for h in range(Hh):
            k[j, h, basis[j, h]] = 1.0
    kb = synth.f32_to_bf16_bits(k)
    o = oracle.gdn_tree_path(x.S0, kb, kb, x.v, np.ones_like(x.alpha), np.ones_like(x.beta), t)
    vf = synth.bf16_bits_to_f32(x.v).astype(np.float64)
    assert np.array_equal(o, vf)


@pytest.mark.parametrize("kw", TREES)
def test_rows_off_the_root_path_do_not_matter(kw):
    t, w = _tree(kw, 6)
    x = synth.gdn_inputs(t.R, w.n_req, 2, 16, seed=7)
    o = oracle.gdn_tree_path(x.S0, x.q, x.k, x.v, x.alpha, x.beta, t)
    g = np.random.default_rng(8)
    for j in g.choice(t.R, size=min(6, t.R), replace=False):
        on = set(_path(t, int(j)))
        x2 = synth.gdn_inputs(t.R, w.n_req, 2, 16, seed=99)     # fresh values everywhere off the path
        for f in ("q", "k", "v", "alpha", "beta"):
            a = getattr(x2, f)
            a[list(on)] = getattr(x, f)[list(on)]
        x2.S0[:] = x.S0
        o2 = oracle.gdn_tree_path(x2.S0, x2.q, x2.k, x2.v, x2.alpha, x2.beta, t)
        assert np.array_equal(o2[j], o[j])


def _wy_reference(S0, q, k, v, alpha, beta, tree, u_out=None):
    """The tree in WY form, written independently of the oracle's loop: per
    request and head, with g the cumulative gate along each root path and
    anc/path the strict/inclusive ancestor relations,
      (I + A) U = B,  A[j,i] = b_j (g_j / g_i) k_i.k_j  (i a strict ancestor of j),
                      B[j]   = b_j (v_j - g_j S0 k_j),
      o_j = g_j S0 q_j + sum over i on j's path of (g_j / g_i) (k_i.q_j) u_i."""
    qf, kf, vf = (synth.bf16_bits_to_f32(a).astype(np.float64) for a in (q, k, v))
    R, Hh, _ = qf.shape
    out = np.zeros((R, Hh, vf.shape[2]))
    off = tree.req_row_off
    for r in range(len(off) - 1):
        rows = np.arange(off[r], off[r + 1])
        n = len(rows)
        loc = {int(j): a for a, j in enumerate(rows)}
        anc = np.zeros((n, n), bool)
        for a, j in enumerate(rows):
            p = int(tree.parent[j])
            if p >= 0:
                anc[a] = anc[loc[p]]
                anc[a, loc[p]] = True
        incl = anc | np.eye(n, dtype=bool)
        for h in range(Hh):
            al, be = alpha[rows, h].astype(np.float64), beta[rows, h].astype(np.float64)
            gcum = np.array([np.prod(al[incl[a]]) for a in range(n)])
            K, Q, V = kf[rows, h], qf[rows, h], vf[rows, h]
            S = S0[r, h].astype(np.float64)
            ratio = gcum[:, None] / gcum[None, :]
            A = np.where(anc, be[:, None] * ratio * (K @ K.T), 0.0)
            B = be[:, None] * (V - gcum[:, None] * (K @ S.T))
            U = np.linalg.solve(np.eye(n) + A, B)
            C = np.where(incl, ratio * (Q @ K.T), 0.0)
            out[rows, h] = gcum[:, None] * (Q @ S.T) + C @ U
            if u_out is not None:
                u_out[rows, h] = U
    return out


@pytest.mark.parametrize("kw", TREES)
def test_path_walk_equals_wy_form(kw):
    t, w = _tree(kw, 9)
    x = synth.gdn_inputs(t.R, w.n_req, 3, 32, seed=10)
    o = oracle.gdn_tree_path(x.S0, x.q, x.k, x.v, x.alpha, x.beta, t)
    ref = _wy_reference(x.S0, x.q, x.k, x.v, x.alpha, x.beta, t)
    assert np.max(np.abs(o - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("kw", TREES)
def test_commit_state_reproduces_the_accepted_rows_output(kw):
    t, w = _tree(kw, 11)
    x = synth.gdn_inputs(t.R, w.n_req, 2, 16, seed=12)
    o = oracle.gdn_tree_path(x.S0, x.q, x.k, x.v, x.alpha, x.beta, t)
    g = np.random.default_rng(13)
    acc = np.asarray([g.integers(t.req_row_off[r], t.req_row_off[r + 1]) for r in range(w.n_req)], np.int32)
    S = oracle.gdn_commit(x.S0, x.k, x.v, x.alpha, x.beta, t, acc)
    qf = synth.bf16_bits_to_f32(x.q).astype(np.float64)
    for r, j in enumerate(acc):
        assert np.allclose(np.einsum("hvk,hk->hv", S[r], qf[j]), o[j], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("kw", TREES)
def test_wy_vectors_equal_the_triangular_solve(kw):
    """oracle.gdn_wy_u (u_j from the state each row's update applies to)
    against U of the independent WY restatement, (I + A) U = B by a dense
    solve."""
    t, w = _tree(kw, 15)
    x = synth.gdn_inputs(t.R, w.n_req, 3, 32, seed=16)
    U = np.zeros((t.R, 3, 32))
    _wy_reference(x.S0, x.q, x.k, x.v, x.alpha, x.beta, t, u_out=U)
    u = oracle.gdn_wy_u(x.S0, x.k, x.v, x.alpha, x.beta, t)
    assert np.max(np.abs(u - U)) <= 1e-12 * max(1.0, np.max(np.abs(U)))


@pytest.mark.parametrize("kw", TREES)
def test_commit_from_wy_vectors_equals_the_replay(kw):
    """The accepted state in WY form, g S0 + sum over the path of (g / g_i)
    u_i k_i^T, against the committed state replayed step by step."""
    t, w = _tree(kw, 17)
    x = synth.gdn_inputs(t.R, w.n_req, 2, 16, seed=18)
    g = np.random.default_rng(19)
    acc = np.asarray([g.integers(t.req_row_off[r], t.req_row_off[r + 1]) for r in range(w.n_req)], np.int32)
    ref = oracle.gdn_commit(x.S0, x.k, x.v, x.alpha, x.beta, t, acc)
    u = oracle.gdn_wy_u(x.S0, x.k, x.v, x.alpha, x.beta, t)
    kf = synth.bf16_bits_to_f32(x.k).astype(np.float64)
    a64 = x.alpha.astype(np.float64)
    for r, j in enumerate(acc):
        path = []
        i = int(j)
        while i >= 0:
            path.append(i)
            i = int(t.parent[i])
        gcum = {}
        run = np.ones(2)
        for i in reversed(path):
            run = run * a64[i]
            gcum[i] = run.copy()
        gacc = gcum[int(j)]
        S = gacc[:, None, None] * x.S0[r].astype(np.float64)
        for i in path:
            S += (gacc / gcum[i])[:, None, None] * u[i][:, :, None] * kf[i][:, None, :]
        assert np.allclose(S, ref[r], rtol=1e-11, atol=1e-13)
