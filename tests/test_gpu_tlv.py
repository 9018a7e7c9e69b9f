"""GPU parity of the TLV cycle (SpecPilot explainer, 4.3) through the C ABI:
the Q pass's chain, the host chain rule, the fresh subtree and the splice,
bit-exact against the oracle; then a whole cycle with real W12 GEMMs whose
exact pass must accept what greedy decoding would (marked gpu)."""
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


def _tree_equal(got: dict, ref: oracle.Tree):
    R = ref.R
    assert len(got["parent"]) == R
    for k in ("parent", "token", "depth", "req", "rank"):
        assert np.array_equal(got[k], getattr(ref, k)), k
    assert np.array_equal(got["score"].view(np.uint32), ref.score.view(np.uint32))
    assert np.array_equal(got["req_row_off"][:len(ref.req_row_off)], ref.req_row_off)


CASES = [
    ("single", dict(n_req=1, positions=(16,), budget=32, vocab=4096, n_cand=16), 16),
    ("single_short", dict(n_req=1, positions=(6,), budget=24, vocab=4096, n_cand=16), 8),
    ("batched", dict(n_req=6, positions=(2, 4, 8), budget=64, vocab=4096, n_cand=16), 8),
    ("chain", dict(n_req=3, positions=(8,), budget=18, vocab=4096, n_cand=1), 6),
    ("many_requests", dict(n_req=96, positions=(2, 3, 4), budget=400, vocab=4096, n_cand=16), 4),
    ("roots_tight", dict(n_req=40, positions=(3,), budget=80, vocab=4096, n_cand=16), 3),
    ("full_budget", dict(n_req=16, positions=(16,), budget=512, vocab=4096, n_cand=16, conditional=True), 16),
]


@pytest.mark.parametrize("name,kw,p2", CASES)
@pytest.mark.parametrize("err", [0.0, 0.35, 1.0])
def test_tlv_splice_bit_exact(w12, name, kw, p2, err):
    seed = 3
    w = synth.scaled(synth.WORKLOADS["tiny"], hit_rate=0.9, seed=seed, **kw)
    truth = H.tlv_truth(w, p2, seed)
    lat1 = synth.lattice(w, seed, truth=truth[:, :w.p_max + 1])
    # oracle cycle
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

    # the same cycle through the library
    ws = w12.Workspace(1, 0, 0, w.n_req)
    d1 = w12.w12_tree_build(w12.DeviceLattice(lat1), w.budget, ws)
    _tree_equal(d1.host(), t1)
    q_dev = torch.from_numpy(qarg).cuda()
    g_tok, g_len, g_node = w12.w12_tree_accept(d1, w.n_req, w.p_max, q_dev)
    torch.cuda.synchronize()
    assert np.array_equal(g_tok.cpu().numpy(), c_tok)
    assert np.array_equal(g_len.cpu().numpy(), c_len)
    assert np.array_equal(g_node.cpu().numpy(), c_node)
    gm, gsub = w12.w12_tlv_chain(g_len.cpu().numpy(), d1.req_row_off.cpu().numpy(), w.budget)
    assert np.array_equal(gm, m) and gsub == sub
    d2 = w12.w12_tree_build(w12.DeviceLattice(lat2), gsub, ws)
    _tree_equal(d2.host(), t2)
    dc = w12.w12_tlv_splice(d1, g_tok, g_len, g_node, gm, d2, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    _tree_equal(dc.host(), tc)
    assert dc.R <= w.budget
    ex_dev = torch.from_numpy(exact).cuda()
    e_tok, e_len, e_node = w12.w12_tree_accept(dc, w.n_req, p_comb, ex_dev)
    torch.cuda.synchronize()
    assert np.array_equal(e_tok.cpu().numpy(), a_tok)
    assert np.array_equal(e_len.cpu().numpy(), a_len)
    assert np.array_equal(e_node.cpu().numpy(), a_node)


def test_tlv_splice_flags_a_chain_that_is_not_the_tree_path(w12):
    seed = 4
    w = synth.scaled(synth.WORKLOADS["tiny"], n_req=2, positions=(6,), budget=20, vocab=4096, hit_rate=0.9,
                     seed=seed)
    truth = H.tlv_truth(w, 4, seed)
    lat1 = synth.lattice(w, seed, truth=truth[:, :w.p_max + 1])
    ws = w12.Workspace(1, 0, 0, w.n_req)
    d1 = w12.w12_tree_build(w12.DeviceLattice(lat1), w.budget, ws)
    t1 = oracle.tree_build(lat1, w.budget)
    exact1 = H.target_argmax(t1, truth, w.vocab, seed)
    g_tok, g_len, g_node = w12.w12_tree_accept(d1, w.n_req, w.p_max, torch.from_numpy(exact1).cuda())
    m, sub = w12.w12_tlv_chain(g_len.cpu().numpy(), d1.req_row_off.cpu().numpy(), w.budget)
    c_tok, c_len, _ = oracle.tree_accept(t1, exact1, w.n_req, w.p_max)
    w2 = synth.scaled(w, positions=(4,))
    d2 = w12.w12_tree_build(w12.DeviceLattice(H.second_lattice(w2, lat1, c_tok, m, truth, seed)), sub, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    # a chain length that disagrees with the node's depth
    bad_len = g_len.clone()
    bad_len[0] += 1
    w12.w12_tlv_splice(d1, g_tok, bad_len, g_node, np.minimum(m, (bad_len.cpu().numpy() - 1)), d2, ws)
    torch.cuda.synchronize()
    assert ws.status() == w12.W12_E_INVAL
    # a chain token that is not the tree's
    if int(c_len[0]) >= 2:
        bad_tok = g_tok.clone()
        bad_tok[0, 0] += 1
        w12.w12_tlv_splice(d1, bad_tok, g_len, g_node, m, d2, ws)
        torch.cuda.synchronize()
        assert ws.status() == w12.W12_E_INVAL
    # the good call still works afterwards
    dc = w12.w12_tlv_splice(d1, g_tok, g_len, g_node, m, d2, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0 and dc.R == int(m.sum()) + d2.R


@pytest.mark.parametrize("n_req,positions,budget,p2", [(1, (16,), 32, 16), (4, (4, 8), 48, 8)])
def test_tlv_cycle_with_w12_gemms(w12, path, n_req, positions, budget, p2):
    """A whole cycle: Q pass (quick weights) over the first tree, chain,
    subtree, splice, exact pass over the combined tree; every stage against
    the oracle on margin-passing rows, and the accepted tokens against
    greedy decoding of the same target."""
    seed = 9
    w = synth.scaled(synth.WORKLOADS["single_27b"], vocab=8192, hidden=512, linears=((1024, 512),), n_req=n_req,
                     positions=positions, budget=budget, hit_rate=0.9, seed=seed)
    truth = H.tlv_truth(w, p2, seed)
    lat1 = synth.lattice(w, seed, truth=truth[:, :w.p_max + 1])
    wh = synth.weights(w.vocab, w.hidden, seed, synth.STREAM_HEAD, 0.001, 0.001)
    n2 = synth.head_norms(wh)
    pk = oracle.w12_pack(wh)
    wq = oracle.w12_unpack_q(pk)
    lw = synth.weights(1024, 512, seed, synth.STREAM_LINEAR)
    dh = w12.DeviceWeight(w12.w12_pack(wh))
    dl = w12.DeviceWeight(w12.w12_pack(lw))

    # oracle: Q pass over T1 on the quick head
    t1 = oracle.tree_build(lat1, w.budget)
    h1 = synth.hidden_rows(t1.req, t1.parent, t1.token, truth, wh, seed, head_norm2=n2)
    qam, _, qmg = oracle.head_argmax(h1, wq)
    c_tok, c_len, c_node = oracle.tree_accept(t1, qam, w.n_req, w.p_max)

    # library: Q pass
    ws = w12.Workspace(w.budget, 1024, w.vocab, w.n_req)
    d1 = w12.w12_tree_build(w12.DeviceLattice(lat1), w.budget, ws)
    R1 = d1.R
    x1 = _dev_bf16(synth.activations(R1, 512, seed, synth.STREAM_X))
    y1 = torch.empty((R1, 1024), dtype=torch.bfloat16, device="cuda")
    am1 = torch.empty(R1, dtype=torch.int32, device="cuda")
    step1 = w12.VerifyStep([dl], [x1], [y1], dh, _dev_bf16(h1), am1)
    g_tok = torch.empty((w.n_req, w.p_max + 1), dtype=torch.int32, device="cuda")
    g_len = torch.empty(w.n_req, dtype=torch.int32, device="cuda")
    g_node = torch.empty(w.n_req, dtype=torch.int32, device="cuda")
    w12.w12_verify_step_q(step1, d1, w.n_req, w.p_max, ws, g_tok, g_len, g_node)
    torch.cuda.synchronize()
    assert ws.status() == 0
    compared, mism, near = H.accepted_parity(g_tok.cpu().numpy(), g_len.cpu().numpy(), c_tok, c_len, c_node,
                                             t1.parent, qmg, w.n_req)
    assert not mism and not near, (mism, near)     # these inputs keep every consulted row clear of ties
    assert np.array_equal(g_node.cpu().numpy(), c_node)

    # chain, subtree, splice
    m, sub = oracle.tlv_chain(c_len, t1.req_row_off, w.budget)
    gm, gsub = w12.w12_tlv_chain(g_len.cpu().numpy(), d1.req_row_off.cpu().numpy(), w.budget)
    assert np.array_equal(gm, m) and gsub == sub
    w2 = synth.scaled(w, positions=(p2,))
    lat2 = H.second_lattice(w2, lat1, c_tok, m, truth, seed)
    t2 = oracle.tree_build(lat2, sub)
    tc = oracle.tlv_splice(t1, c_tok, c_len, c_node, m, t2, w.n_req)
    d2 = w12.w12_tree_build(w12.DeviceLattice(lat2), gsub, ws)
    dc = w12.w12_tlv_splice(d1, g_tok, g_len, g_node, gm, d2, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    _tree_equal(dc.host(), tc)

    # exact pass over the combined tree
    p_comb = w.p_max + 1 + p2
    hc = synth.hidden_rows(tc.req, tc.parent, tc.token, truth, wh, seed, head_norm2=n2)
    am, _, mg = oracle.head_argmax(hc, wh)
    a_tok, a_len, a_node = oracle.tree_accept(tc, am, w.n_req, p_comb)
    Rc = dc.R
    xc = _dev_bf16(synth.activations(Rc, 512, seed, synth.STREAM_X + 1))
    yc = torch.empty((Rc, 1024), dtype=torch.bfloat16, device="cuda")
    amc = torch.empty(Rc, dtype=torch.int32, device="cuda")
    stepc = w12.VerifyStep([dl], [xc], [yc], dh, _dev_bf16(hc), amc)
    e_tok = torch.empty((w.n_req, p_comb + 1), dtype=torch.int32, device="cuda")
    e_len = torch.empty(w.n_req, dtype=torch.int32, device="cuda")
    e_node = torch.empty(w.n_req, dtype=torch.int32, device="cuda")
    w12.w12_verify_step(stepc, dc, w.n_req, p_comb, ws, e_tok, e_len, e_node)
    torch.cuda.synchronize()
    assert ws.status() == 0
    compared, mism, near = H.accepted_parity(e_tok.cpu().numpy(), e_len.cpu().numpy(), a_tok, a_len, a_node,
                                             tc.parent, mg, w.n_req)
    assert not mism, (mism, near)
    assert len(compared) >= 0.75 * w.n_req
    # greedy decoding of the same target (the FP64 argmax of each prefix's
    # hidden row), one token at a time
    for q in compared:
        n = int(a_len[q])
        ar = []
        for _ in range(n):
            hrow = synth.hidden_row(q, ar, truth, wh, n2, seed)
            ar.append(int(oracle.head_argmax(hrow[None, :], wh)[0][0]))
        assert list(e_tok.cpu().numpy()[q][:n]) == ar
    # where the Q pass agreed with the exact one along the chain, the exact
    # pass accepts the whole committed chain and one token more
    am1, _, _ = oracle.head_argmax(h1, wh)
    for q in compared:
        rows, j = [], int(c_node[q])
        while j >= 0:
            rows.append(j)
            j = int(t1.parent[j])
        if all(qam[j] == am1[j] for j in rows):
            assert int(e_len[q]) >= int(m[q]) + 1
