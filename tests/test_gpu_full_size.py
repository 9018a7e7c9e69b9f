"""Parity at the full workload sizes, in the launch configuration the
benchmark times (the tree build and the whole verify step captured in one
CUDA graph, default GEMM path choice).

The oracle cannot run every output of every linear at these sizes in
seconds, so the linears are checked on sampled output channels (random ones
plus the first channels of the tiles where stream-K splits CTA shares); for
the 64-layer stack, in the first, a middle and the last layer.  The tree,
the full LM-head argmax and the accepted tokens are checked whole.
"""
import os
import sys

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_w12_gb300 import synth
from tests import helpers as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _sample_channels(n, k, n_sms, rng, n_random=96):
    k_tiles = k // 64
    T = (n // 128) * k_tiles
    ch = set(rng.choice(n, size=min(n, n_random), replace=False).tolist())
    for c in range(0, n_sms, 7):
        tile = (c * T // n_sms) // k_tiles          # n-tile holding CTA c's first record
        ch.update({tile * 128, tile * 128 + 77, min(n - 1, tile * 128 + 127)})
    ch.update({0, n - 1})
    return np.array(sorted(ch), dtype=np.int64)


@pytest.mark.parametrize("name", ["single_27b", "batched_27b", "b4_tree", "full_depth_27b"])
def test_full_size_verify_step(name):
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_tree_w12_gb300 import build
    build.build()
    import speculative_decoding_tree_w12_gb300 as w12

    w12.debug_set(0, 0)
    dev = torch.device("cuda", 0)
    wk = bench.Workload(name, 0, dev)
    # the benchmark's launch configuration: one eager step on a side stream,
    # then the step captured in a graph and replayed
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        wk.step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for y in wk.ys:
        y.zero_()
    wk.argmax.fill_(-1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wk.step()
    g.replay()
    torch.cuda.synchronize()
    assert wk.ws.status() == 0

    w = wk.wl
    ref_tree = oracle.tree_build(wk.lat, w.budget)
    t = wk.tree.host()
    assert t["parent"].tolist() == ref_tree.parent.tolist()
    assert t["token"].tolist() == ref_tree.token.tolist()
    assert t["score"].tobytes() == ref_tree.score.tobytes()
    assert t["req_row_off"].tolist() == ref_tree.req_row_off.tolist()

    rng = np.random.default_rng(1234)
    n_sms = w12.num_sms()
    n_lin = len(w.linears)
    # stacked layers: the first, one past the middle and the last layer (three
    # of the four distinct weight sets; every layer streams its own copy)
    layers = sorted({0, w.layers // 2 + 1, w.layers - 1}) if w.layers > 1 else [0]
    for layer in layers:
        for i, x in enumerate(wk.x_bits):
            if layer == 0:
                bits = wk.lin_bits[i]
            else:
                n, k = w.linears[i]
                bits = synth.weights(n, k, w.seed, synth.STREAM_LINEAR + 100 * (layer % 4) + i,
                                     w.outlier_frac, w.zero_frac)
            n, k = bits.shape
            cols = _sample_channels(n, k, n_sms, rng)
            ref = oracle.gemm_f64(x, np.ascontiguousarray(bits[cols]))
            got = np.ascontiguousarray(_bits(wk.ys[layer * n_lin + i])[:, cols])
            got = synth.bf16_bits_to_f32(got).astype(np.float64)
            assert H.gemm_rel_err(got, ref) <= H.GEMM_REL_TOL, (name, layer, i)

    am, _, mg = oracle.head_argmax(wk.h_bits, wk.head_bits)
    gated = mg > H.MARGIN_GATE
    assert gated.mean() > 0.9
    got_am = wk.argmax.cpu().numpy()
    assert np.array_equal(got_am[gated], am[gated])

    tok, ln, node = oracle.tree_accept(ref_tree, am, w.n_req, w.p_max)
    compared, mism, near = H.accepted_parity(wk.acc_tok.cpu().numpy(), wk.acc_len.cpu().numpy(), tok, ln,
                                             node, ref_tree.parent, mg, w.n_req)
    assert not mism, (mism, near)
    assert len(compared) >= 0.9 * w.n_req
