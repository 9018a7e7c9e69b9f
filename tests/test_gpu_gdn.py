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


def _hand_tree(w12, sizes, seed, extra_root=0.1):
    """A tree with the given rows per request (zero allowed): each request's
    first row is a root, every later row hangs under a random earlier row of
    its request or, with probability extra_root, is one more root."""
    g = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    parent = np.full(R, -1, np.int32)
    req = np.empty(R, np.int32)
    for r, n in enumerate(sizes):
        o = int(off[r])
        req[o:o + n] = r
        for j in range(1, n):
            parent[o + j] = -1 if g.random() < extra_root else o + int(g.integers(0, j))
    z = np.zeros(R, np.int32)
    t = oracle.Tree(R, parent, z, z.astype(np.uint8), req, z.astype(np.float32), z.astype(np.uint8), off)
    dt = w12.DeviceTree(max(R, 1), len(sizes))
    dt.parent[:R] = torch.from_numpy(parent).cuda()
    dt.req_row_off.copy_(torch.from_numpy(off))
    dt.c.R = R
    return t, dt


PACKS = [
    # windows holding one 64-row request, several packs, a request that crosses
    # a window edge, an empty request, and runs of 16-row requests
    ("mixed", [64, 1, 1, 63, 5, 40, 24, 0, 7, 33, 31, 2, 16, 16, 16, 16, 3], 3),
    # 60 requests of 1 to 4 rows: up to 64 requests start in one window
    ("tiny", [1, 4, 2, 3] * 15, 2),
    # every size from 1 to 12
    ("ramp", list(range(1, 13)), 2),
    # the two-solver-group threshold: with 64 heads the windows are wide, so
    # a 45-row request shares a pack with small ones (two groups) and a
    # 46-row one does too (one group)
    ("threshold", [45, 46, 3, 1, 45], 64),
    ("threshold_big", [3, 46, 1], 64),
    # 64 heads: the tensor-memory kernel's windows shrink to fit one wave
    ("heads_64", [8] * 6, 64),
    # 500 one-row requests: more requests than threads in the row-range check
    ("many_requests", [1] * 500, 1),
]


@pytest.mark.parametrize("name,sizes,H", PACKS)
def test_gdn_wy_packs_requests_of_mixed_sizes(w12, name, sizes, H):
    """The WY kernel takes the requests whose first row lies in one 64-row
    window together, in runs of at most 64 rows; outputs must not depend on
    where a request falls."""
    t, dt = _hand_tree(w12, sizes, 11)
    x = synth.gdn_inputs(t.R, len(sizes), H, 128, seed=13)
    ref = oracle.gdn_tree_path(x.S0, x.q, x.k, x.v, x.alpha, x.beta, t)
    ws = w12.Workspace(1, 0, 0, len(sizes))
    layer = _layer(w12, x)
    o_wy = w12.w12_gdn_tree_verify(layer, dt, len(sizes), ws, w12.W12_GDN_WY)
    o_path = w12.w12_gdn_tree_verify(layer, dt, len(sizes), ws, w12.W12_GDN_PATH)
    torch.cuda.synchronize()
    assert ws.status() == 0
    e_wy = _rel_err(o_wy.cpu().numpy().astype(np.float64), ref)
    e_path = _rel_err(o_path.cpu().numpy().astype(np.float64), ref)
    assert e_wy <= 1e-4 and e_path <= 1e-4, (e_wy, e_path)


def test_gdn_wy_flags_row_offsets_past_the_tree(w12):
    """Row offsets that run past the tree's rows: the WY kernel checks every
    request's range before any other read, sets W12_E_INVAL and writes nothing."""
    t, dt = _hand_tree(w12, [10, 6], 3)
    x = synth.gdn_inputs(t.R, 2, 1, 128, seed=3)
    ws = w12.Workspace(1, 0, 0, 2)
    layer = _layer(w12, x)
    dt.req_row_off.copy_(torch.tensor([0, 10, 20], dtype=torch.int32))
    o = torch.full((t.R, 1, 128), 7.0, device="cuda")
    w12.w12_gdn_tree_verify(layer, dt, 2, ws, w12.W12_GDN_WY, out=o)
    torch.cuda.synchronize()
    assert ws.status() == w12.W12_E_INVAL
    assert bool((o == 7.0).all())


WY_COMMIT_CASES = CASES[:6] + [("bench_batched", dict(n_req=24, positions=(16, 12, 8), budget=192, n_cand=16), 32)]


@pytest.mark.parametrize("name,kw,H", WY_COMMIT_CASES)
def test_gdn_wy_vectors_and_commit_match_fp64(w12, name, kw, H):
    """w12_gdn_wy_verify's outputs equal w12_gdn_tree_verify's (same
    kernels), its WY vectors match oracle.gdn_wy_u, and w12_gdn_wy_commit's
    states match the replayed FP64 commit (also written in place over S0)."""
    w, lat, t, x = _case(kw, H, 21)
    ws = w12.Workspace(1, 0, 0, w.n_req)
    tree = w12.w12_tree_build(w12.DeviceLattice(lat), w.budget, ws)
    layer = _layer(w12, x)
    o, u = w12.w12_gdn_wy_verify(layer, tree, w.n_req, ws)
    o_ref = w12.w12_gdn_tree_verify(layer, tree, w.n_req, ws, w12.W12_GDN_WY)
    g = np.random.default_rng(22)
    acc = np.asarray([g.integers(t.req_row_off[r], t.req_row_off[r + 1]) for r in range(w.n_req)], np.int32)
    st = w12.w12_gdn_wy_commit(layer, tree, w.n_req, torch.from_numpy(acc).cuda(), u, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert torch.equal(o, o_ref)
    u_ref = oracle.gdn_wy_u(x.S0, x.k, x.v, x.alpha, x.beta, t)
    assert _rel_err(u.cpu().numpy().astype(np.float64), u_ref) <= 1e-4
    ref = oracle.gdn_commit(x.S0, x.k, x.v, x.alpha, x.beta, t, acc)
    assert _rel_err(st.cpu().numpy().astype(np.float64).reshape(-1, 128), ref.reshape(-1, 128)) <= 1e-4
    st2 = w12.w12_gdn_wy_commit(layer, tree, w.n_req, torch.from_numpy(acc).cuda(), u, ws, state=layer.S0)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert torch.equal(st2, st)


def test_gdn_wy_commit_flags_a_row_outside_its_request(w12):
    w, lat, t, x = _case(dict(n_req=3, positions=(2, 4, 6), budget=30, n_cand=16), 2, 23)
    ws = w12.Workspace(1, 0, 0, w.n_req)
    tree = w12.w12_tree_build(w12.DeviceLattice(lat), w.budget, ws)
    layer = _layer(w12, x)
    _, u = w12.w12_gdn_wy_verify(layer, tree, w.n_req, ws)
    acc = np.asarray([t.req_row_off[0], t.req_row_off[0], t.req_row_off[2]], np.int32)   # request 1: a row of request 0
    st = w12.w12_gdn_wy_commit(layer, tree, w.n_req, torch.from_numpy(acc).cuda(), u, ws)
    torch.cuda.synchronize()
    assert ws.status() == w12.W12_E_INVAL
    assert torch.equal(st[1], layer.S0[1])



@pytest.mark.parametrize("name,sizes,H", PACKS + [("one_of_64_then_tiny", [64] + [1] * 20, 2)])
def test_gdn_wy_vectors_and_commit_on_hand_packs(w12, name, sizes, H):
    """w12_gdn_wy_verify and w12_gdn_wy_commit on the hand-made packs: the
    outputs, the WY vectors and the committed states of non-empty requests
    (an empty request has no row to accept and keeps no state) against the
    FP64 oracle."""
    t, dt = _hand_tree(w12, sizes, 31)
    n_req = len(sizes)
    x = synth.gdn_inputs(t.R, n_req, H, 128, seed=32)
    ws = w12.Workspace(1, 0, 0, n_req)
    layer = _layer(w12, x)
    o, u = w12.w12_gdn_wy_verify(layer, dt, n_req, ws)
    g = np.random.default_rng(33)
    off = t.req_row_off
    acc = np.asarray([g.integers(off[r], off[r + 1]) if sizes[r] else off[r] for r in range(n_req)], np.int32)
    st = w12.w12_gdn_wy_commit(layer, dt, n_req, torch.from_numpy(acc).cuda(), u, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    o_ref = oracle.gdn_tree_path(x.S0, x.q, x.k, x.v, x.alpha, x.beta, t)
    u_ref = oracle.gdn_wy_u(x.S0, x.k, x.v, x.alpha, x.beta, t)
    assert _rel_err(o.cpu().numpy().astype(np.float64), o_ref) <= 1e-4
    assert _rel_err(u.cpu().numpy().astype(np.float64), u_ref) <= 1e-4
    full = [r for r in range(n_req) if sizes[r]]
    s_ref = oracle.gdn_commit(x.S0[full], x.k, x.v, x.alpha, x.beta, t, acc[full])
    got = st.cpu().numpy().astype(np.float64)[full]
    assert _rel_err(got.reshape(-1, 128), s_ref.reshape(-1, 128)) <= 1e-4


def test_gdn_wy_tensor_memory_wait_times_out_cleanly(w12):
    """CTA (0, 0) of the tensor-memory WY kernel never copies its first
    request's state (test hook): its splitters give up after 50 ms, both warp
    roles stop, tensor memory is released, the status word reads
    W12_E_TIMEOUT, and the context stays usable: the same call without the
    hook matches the oracle."""
    w, lat, t, x = _case(dict(n_req=3, positions=(2, 4, 6), budget=30, n_cand=16), 2, 41)
    ws = w12.Workspace(1, 0, 0, w.n_req)
    tree = w12.w12_tree_build(w12.DeviceLattice(lat), w.budget, ws)
    layer = _layer(w12, x)
    torch.cuda.synchronize()
    assert ws.status() == 0
    w12.debug_set(1, 50_000_000)
    try:
        w12.w12_gdn_tree_verify(layer, tree, w.n_req, ws, w12.W12_GDN_WY)
        torch.cuda.synchronize()
        assert ws.status() == w12.W12_E_TIMEOUT
    finally:
        w12.debug_set(0, 0)
    o = w12.w12_gdn_tree_verify(layer, tree, w.n_req, ws, w12.W12_GDN_WY)
    torch.cuda.synchronize()
    assert ws.status() == 0
    ref = oracle.gdn_tree_path(x.S0, x.q, x.k, x.v, x.alpha, x.beta, t)
    assert _rel_err(o.cpu().numpy().astype(np.float64), ref) <= 1e-4
