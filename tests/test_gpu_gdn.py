"""GPU parity of the recurrent-layer tree verification (SpecPilot explainer,
4.2) through the C ABI: both kernels (WY form, path walk) and the commit
replay against the FP64 oracle (marked gpu).

Tolerance: the pages hold the WY kernel to one BF16 ulp of the path
kernel's output.  Both kernels here compute in FP32 (the WY state products
on BF16 pieces that add up to the FP32 state exactly, with FP32
accumulation), so the test asks each of them for that bound against the
FP64 oracle: per row and head, max |o - o_ref| <= 2^-8 max |o_ref|."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_w12_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2.0 ** -8


@pytest.fixture(scope="module")
def w12():
    from speculative_decoding_tree_w12_gb300 import build
    build.build()
    import speculative_decoding_tree_w12_gb300 as m
    m.lib()
    return m


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _layer(w12, x):
    return w12.GdnLayer(torch.from_numpy(x.S0).cuda(), _bf16(x.q), _bf16(x.k), _bf16(x.v),
                        torch.from_numpy(x.alpha).cuda(), torch.from_numpy(x.beta).cuda())


def _rel_err(got, ref):
    """max over (row, head) of max_c |got - ref| / max_c |ref|"""
    num = np.abs(got - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return float((num / den).max())


CASES = [
    ("single_32", dict(n_req=1, positions=(16,), budget=32, n_cand=16), 4),
    ("chain_17", dict(n_req=1, positions=(16,), budget=17, n_cand=1), 2),
    ("requests_3", dict(n_req=3, positions=(2, 4, 6), budget=30, n_cand=16), 3),
    ("full_64", dict(n_req=1, positions=(16,), budget=64, n_cand=16), 2),
    ("many_small", dict(n_req=24, positions=(8, 12, 16), budget=192, n_cand=16), 2),
    ("roots_only", dict(n_req=5, positions=(4,), budget=5, n_cand=16), 3),
    # the shapes the bench times: 32 heads over the single_27b and batched_27b trees
    ("bench_single", dict(n_req=1, positions=(16,), budget=32, n_cand=16), 32),
    ("bench_batched", dict(n_req=24, positions=(16, 12, 8), budget=192, n_cand=16), 32),
]


def _case(kw, H, seed):
    w = synth.scaled(synth.WORKLOADS["tiny"], vocab=4096, hit_rate=0.9, seed=seed, **kw)
    lat = synth.lattice(w, seed)
    t = oracle.tree_build(lat, w.budget)
    x = synth.gdn_inputs(t.R, w.n_req, H, 128, seed=seed)
    return w, lat, t, x


@pytest.mark.parametrize("name,kw,H", CASES)
def test_gdn_tree_outputs_match_fp64_path_walk(w12, name, kw, H):
    w, lat, t, x = _case(kw, H, 5)
    ref = oracle.gdn_tree_path(x.S0, x.q, x.k, x.v, x.alpha, x.beta, t)
    ws = w12.Workspace(1, 0, 0, w.n_req)
    tree = w12.w12_tree_build(w12.DeviceLattice(lat), w.budget, ws)
    layer = _layer(w12, x)
    o_wy = w12.w12_gdn_tree_verify(layer, tree, w.n_req, ws, w12.W12_GDN_WY)
    o_path = w12.w12_gdn_tree_verify(layer, tree, w.n_req, ws, w12.W12_GDN_PATH)
    torch.cuda.synchronize()
    assert ws.status() == 0
    e_wy = _rel_err(o_wy.cpu().numpy().astype(np.float64), ref)
    e_path = _rel_err(o_path.cpu().numpy().astype(np.float64), ref)
    assert e_wy <= TOL and e_path <= TOL, (e_wy, e_path)
    # both kernels compute in FP32: far inside the bound on these inputs
    assert e_wy <= 1e-4 and e_path <= 1e-4, (e_wy, e_path)


@pytest.mark.parametrize("name,kw,H", CASES[:3] + CASES[4:5])
def test_gdn_commit_matches_fp64_replay(w12, name, kw, H):
    w, lat, t, x = _case(kw, H, 7)
    g = np.random.default_rng(8)
    acc = np.asarray([g.integers(t.req_row_off[r], t.req_row_off[r + 1]) for r in range(w.n_req)], np.int32)
    ref = oracle.gdn_commit(x.S0, x.k, x.v, x.alpha, x.beta, t, acc)
    ws = w12.Workspace(1, 0, 0, w.n_req)
    tree = w12.w12_tree_build(w12.DeviceLattice(lat), w.budget, ws)
    layer = _layer(w12, x)
    st = w12.w12_gdn_commit(layer, tree, w.n_req, torch.from_numpy(acc).cuda(), ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    got = st.cpu().numpy().astype(np.float64)
    assert _rel_err(got.reshape(-1, 128), ref.reshape(-1, 128)) <= 1e-4
    # in place: the committed state overwrites S0
    st2 = w12.w12_gdn_commit(layer, tree, w.n_req, torch.from_numpy(acc).cuda(), ws, state=layer.S0)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert np.array_equal(st2.cpu().numpy(), st.cpu().numpy())


def test_gdn_flags_a_request_over_64_rows(w12):
    w, lat, t, x = _case(dict(n_req=1, positions=(16,), budget=80, n_cand=16), 1, 9)
    ws = w12.Workspace(1, 0, 0, w.n_req)
    tree = w12.w12_tree_build(w12.DeviceLattice(lat), w.budget, ws)
    layer = _layer(w12, x)
    w12.w12_gdn_tree_verify(layer, tree, w.n_req, ws, w12.W12_GDN_WY)
    torch.cuda.synchronize()
    assert ws.status() == w12.W12_E_UNSUPPORTED
    w12.w12_gdn_tree_verify(layer, tree, w.n_req, ws, w12.W12_GDN_PATH)
    torch.cuda.synchronize()
    assert ws.status() == w12.W12_E_UNSUPPORTED
