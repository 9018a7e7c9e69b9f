"""The verify step's persistent GEMM chain (one launch for every linear and the
LM head), through the C ABI.

The chain runs the same tensor-memory GEMM as the one-launch-per-GEMM path,
with the same stream-K split and the same accumulation order, so its outputs
must be bit-identical to that path's: every linear's BF16 output, the head
argmax and the acceptance outputs.  The linears are also checked against the
FP64 oracle.  Cases cover 1 to 192 rows, GEMMs small enough that most CTAs
have no records, escapes, the quick pass, a step longer than one launch's
parameter block (two launches) and a wait that runs out."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_w12_gb300 import synth
from tests import helpers as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FORCE_TC = 2        # debug flag: every GEMM on the tensor-memory kernel
NO_CHAIN = 8        # debug flag: one launch per GEMM
CHAIN = 16          # debug flag: the verify step as one GEMM-chain launch


@pytest.fixture(scope="module")
def w12():
    from speculative_decoding_tree_w12_gb300 import build
    build.build()
    import speculative_decoding_tree_w12_gb300 as m
    m.lib()
    yield m
    m.debug_set(0, 0)


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class _Step:
    """A one-request tree of `budget` rows and a step over `linears` + head."""

    def __init__(self, w12, budget, linears, vocab, hidden, outl=0.0, zero=0.0, seed=3):
        w = synth.scaled(synth.WORKLOADS["single_27b"], linears=tuple(linears), vocab=vocab, hidden=hidden,
                         budget=budget, outlier_frac=outl, zero_frac=zero, seed=seed)
        self.w = w
        lat = synth.lattice(w)
        self.ws = w12.Workspace(budget, max(n for n, _ in linears), vocab, w.n_req)
        self.tree = w12.w12_tree_build(w12.DeviceLattice(lat), w.budget, self.ws)
        torch.cuda.synchronize()
        R = self.R = self.tree.R
        self.lin_bits = [synth.weights(n, k, seed, synth.STREAM_LINEAR + i, outl, zero)
                         for i, (n, k) in enumerate(linears)]
        self.lin = [w12.DeviceWeight(w12.w12_pack(b)) for b in self.lin_bits]
        self.head = w12.DeviceWeight(w12.w12_pack(synth.weights(vocab, hidden, seed, synth.STREAM_HEAD, outl, zero)))
        self.x_bits = [synth.activations(R, k, seed, synth.STREAM_X + i) for i, (_, k) in enumerate(linears)]
        self.xs = [_dev(x) for x in self.x_bits]
        self.h = _dev(synth.activations(R, hidden, seed, synth.STREAM_X + 999))

    def run(self, w12, flags, quick=False):
        R, w = self.R, self.w
        ys = [torch.full((R, d.n), float("nan"), dtype=torch.bfloat16, device="cuda") for d in self.lin]
        am = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        step = w12.VerifyStep(self.lin, self.xs, ys, self.head, self.h, am)
        tok = torch.full((w.n_req, w.p_max + 1), -7, dtype=torch.int32, device="cuda")
        ln = torch.full((w.n_req,), -7, dtype=torch.int32, device="cuda")
        node = torch.full((w.n_req,), -7, dtype=torch.int32, device="cuda")
        w12.debug_set(flags, 0)
        try:
            fn = w12.w12_verify_step_q if quick else w12.w12_verify_step
            fn(step, self.tree, w.n_req, w.p_max, self.ws, tok, ln, node)
            torch.cuda.synchronize()
        finally:
            w12.debug_set(0, 0)
        assert self.ws.status() == 0
        return [_bits(y) for y in ys], am.cpu().numpy(), tok.cpu().numpy(), ln.cpu().numpy(), node.cpu().numpy()


LIN_SMALL = ((1536, 1024), (1024, 1536), (4096, 1024), (1024, 4096))


@pytest.mark.parametrize("budget", [1, 7, 32, 64, 100, 192])
def test_chain_bit_identical_to_one_launch_per_gemm(w12, budget):
    st = _Step(w12, budget, LIN_SMALL, vocab=8192, hidden=1024, outl=0.002, zero=0.002)
    got = st.run(w12, CHAIN)
    ref = st.run(w12, FORCE_TC | NO_CHAIN)
    for i, (a, b) in enumerate(zip(got[0], ref[0])):
        assert np.array_equal(a, b), ("linear", i)
    for a, b, what in zip(got[1:], ref[1:], ("argmax", "acc_tok", "acc_len", "acc_node")):
        assert np.array_equal(a, b), what
    # and the linears against the FP64 oracle
    for i, (lw, x) in enumerate(zip(st.lin_bits, st.x_bits)):
        y = synth.bf16_bits_to_f32(got[0][i]).astype(np.float64)
        assert H.gemm_rel_err(y, oracle.gemm_f64(x, lw)) <= H.GEMM_REL_TOL, i


def test_chain_tiny_gemms_and_heavy_escapes(w12):
    """GEMMs of 2 to 8 records (one to two CTAs busy, the rest pass through)
    with 1% outliers and 1% zeros, i.e. escape lists beyond the shared cache
    of some CTAs."""
    lin = ((128, 64), (256, 512), (384, 128), (128, 448))
    st = _Step(w12, 16, lin, vocab=1024, hidden=512, outl=0.01, zero=0.01)
    got = st.run(w12, CHAIN)
    ref = st.run(w12, FORCE_TC | NO_CHAIN)
    for a, b in zip(got[0], ref[0]):
        assert np.array_equal(a, b)
    for a, b in zip(got[1:], ref[1:]):
        assert np.array_equal(a, b)
    for i, (lw, x) in enumerate(zip(st.lin_bits, st.x_bits)):
        y = synth.bf16_bits_to_f32(got[0][i]).astype(np.float64)
        assert H.gemm_rel_err(y, oracle.gemm_f64(x, lw)) <= H.GEMM_REL_TOL, i


@pytest.mark.parametrize("budget", [8, 96])
def test_chain_quick_pass_bit_identical(w12, budget):
    st = _Step(w12, budget, LIN_SMALL[:2], vocab=8192, hidden=1024, outl=0.001, zero=0.001)
    got = st.run(w12, CHAIN, quick=True)
    ref = st.run(w12, FORCE_TC | NO_CHAIN, quick=True)
    for a, b in zip(got[0], ref[0]):
        assert np.array_equal(a, b)
    for a, b in zip(got[1:], ref[1:]):
        assert np.array_equal(a, b)


def test_chain_longer_than_one_launch(w12):
    """150 linears + head: more GEMMs than one launch's parameter block holds,
    so the chain runs as two launches with their own arrival words."""
    lin = [(512, 256), (256, 512), (768, 256)] * 50
    st = _Step(w12, 24, lin, vocab=2048, hidden=256, outl=0.001, zero=0.001)
    got = st.run(w12, CHAIN)
    ref = st.run(w12, FORCE_TC | NO_CHAIN)
    for i, (a, b) in enumerate(zip(got[0], ref[0])):
        assert np.array_equal(a, b), i
    for a, b in zip(got[1:], ref[1:]):
        assert np.array_equal(a, b)


def test_chain_bounded_wait_times_out_cleanly(w12):
    """CTA 0's first record pair is announced but never copied (test hook): its
    decode warps give up after 50 ms, the CTA raises the grid's abort word, every
    other CTA stops at its next GEMM boundary, the status word reads
    W12_E_TIMEOUT and the context stays usable."""
    st = _Step(w12, 32, LIN_SMALL, vocab=8192, hidden=1024)
    R, w = st.R, st.w
    ys = [torch.empty((R, d.n), dtype=torch.bfloat16, device="cuda") for d in st.lin]
    am = torch.empty(R, dtype=torch.int32, device="cuda")
    step = w12.VerifyStep(st.lin, st.xs, ys, st.head, st.h, am)
    tok = torch.empty((w.n_req, w.p_max + 1), dtype=torch.int32, device="cuda")
    ln = torch.empty(w.n_req, dtype=torch.int32, device="cuda")
    node = torch.empty(w.n_req, dtype=torch.int32, device="cuda")
    w12.debug_set(1 | CHAIN, 50_000_000)
    try:
        w12.w12_verify_step(step, st.tree, w.n_req, w.p_max, st.ws, tok, ln, node)
        torch.cuda.synchronize()
        assert st.ws.status() == w12.W12_E_TIMEOUT
    finally:
        w12.debug_set(0, 0)
    got = st.run(w12, CHAIN)
    ref = st.run(w12, FORCE_TC | NO_CHAIN)
    for a, b in zip(got[0], ref[0]):
        assert np.array_equal(a, b)
