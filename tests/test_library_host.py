"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every symbol the headers declare, its packer writes exactly the bytes of the
oracle's packer (two independent implementations of one written format), and
malformed calls are refused with a typed status before anything launches."""
from __future__ import annotations

import ctypes as C
import glob
import os
import re

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_w12_gb300 import synth
import speculative_decoding_tree_w12_gb300 as w12
from speculative_decoding_tree_w12_gb300 import build as w12build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    w12build.build()
    return w12.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(w12_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert {"w12_pack", "w12_gemm", "w12_verify_step", "w12_tree_build", "w12_tree_accept",
            "w12_lmhead_argmax", "w12_load_check", "w12_unpack"} <= names
    for n in sorted(names):
        assert hasattr(L, n), n


def _lib_pack(w):
    return w12.w12_pack(w)


@pytest.mark.parametrize("case", ["tiny", "specials", "exhaustive", "zeros", "wide"])
def test_host_packer_bytes_equal_oracle(L, case):
    if case == "tiny":
        w = synth.weights(1024, 512, 0, synth.STREAM_LINEAR, 0.01, 0.01)
    elif case == "specials":
        w = synth.weights(256, 384, 4, 1)
        g = np.random.default_rng(0)
        idx = g.choice(w.size, 3000, replace=False)
        w.reshape(-1)[idx] = g.integers(0, 65536, size=3000).astype(np.uint16)
    elif case == "exhaustive":
        g = np.random.default_rng(1)
        w = g.permutation(np.arange(65536, dtype=np.uint32).astype(np.uint16)).reshape(512, 128)
    elif case == "zeros":
        w = np.zeros((128, 64), np.uint16)
    else:
        w = synth.weights(384, 2048, 9, 2, 0.002, 0.0)
    a = _lib_pack(w)
    b = oracle.w12_pack(w)
    assert np.array_equal(a.base, b.base)
    assert np.array_equal(a.esc_tile_off, b.esc_tile_off)
    assert np.array_equal(a.esc, b.esc)
    assert np.array_equal(a.rec, b.rec)
    # and the oracle decodes the library's bytes back to the source
    assert np.array_equal(oracle.w12_unpack(oracle.Packed(a.n, a.k, a.rec, a.base, a.esc_tile_off, a.esc)), w)


def test_pack_refuses_bad_shapes(L):
    w = np.zeros((100, 64), np.uint16)
    lay = w12.Layout()
    assert L.w12_pack_query(w.ctypes.data_as(C.c_void_p), 100, 64, C.byref(lay)) == w12.W12_E_UNSUPPORTED
    assert L.w12_pack_query(None, 128, 64, C.byref(lay)) == w12.W12_E_INVAL
    assert L.w12_pack_query(w.ctypes.data_as(C.c_void_p), 0, 64, C.byref(lay)) == w12.W12_E_INVAL


def _stream_k_bounds(T, G):
    return [c * T // G for c in range(G + 1)]


@pytest.mark.parametrize("T,G", [(64, 64), (3200, 152), (94960, 152), (4480, 152), (21760, 152), (7, 3),
                                 (152 * 80 + 5, 152), (1000003, 148)])
def test_stream_k_owner_formula(T, G):
    """The kernel finds the CTA owning record r as ((r+1)*G - 1) // T; check
    it against the CTA ranges [c*T//G, (c+1)*T//G)."""
    b = _stream_k_bounds(T, G)
    rs = np.unique(np.concatenate([np.arange(min(T, 5000)), np.asarray(b[1:-1]) - 1, np.asarray(b[1:-1]),
                                   [T - 1]]))
    for r in rs:
        c = ((int(r) + 1) * G - 1) // T
        assert b[c] <= r < b[c + 1], (r, c)


def test_refusals_before_launch(L):
    """Malformed calls return a typed status and launch nothing (these run
    without a GPU because validation precedes every CUDA call)."""
    fake = C.c_void_p(0x1000)   # never dereferenced: validation fails first
    wt = w12.Weight(0x1000, 0x1000, 0x1000, None, 128, 64, 0)
    ws = C.c_void_p(0x100000)
    # null weight / null x
    assert L.w12_gemm(None, fake, 4, fake, ws, 1 << 30, None) == w12.W12_E_INVAL
    assert L.w12_gemm(C.byref(wt), None, 4, fake, ws, 1 << 30, None) == w12.W12_E_INVAL
    # rows out of range
    assert L.w12_gemm(C.byref(wt), fake, 0, fake, ws, 1 << 30, None) == w12.W12_E_INVAL
    assert L.w12_gemm(C.byref(wt), fake, 257, fake, ws, 1 << 30, None) == w12.W12_E_UNSUPPORTED
    # unsupported shape
    bad = w12.Weight(0x1000, 0x1000, 0x1000, None, 100, 64, 0)
    assert L.w12_gemm(C.byref(bad), fake, 4, fake, ws, 1 << 30, None) == w12.W12_E_UNSUPPORTED
    # escapes announced but no list
    noesc = w12.Weight(0x1000, 0x1000, 0x1000, None, 128, 64, 5)
    assert L.w12_gemm(C.byref(noesc), fake, 4, fake, ws, 1 << 30, None) == w12.W12_E_INVAL
    # workspace too small / misaligned
    assert L.w12_gemm(C.byref(wt), fake, 4, fake, ws, 16, None) == w12.W12_E_WORKSPACE
    assert L.w12_gemm(C.byref(wt), fake, 4, fake, C.c_void_p(0x100010), 1 << 30, None) == w12.W12_E_WORKSPACE
    # tree: budget below the number of requests, too many positions
    pr = np.asarray([4, 4], np.int32)
    lat = w12.LatticeC(2, 4, 16, 0, pr.ctypes.data, 0x1000, 0x1000, 0x1000)
    tr = w12.TreeC(0, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    assert L.w12_tree_build(C.byref(lat), 1, C.byref(tr), ws, 1 << 30, None) == w12.W12_E_INVAL
    lat17 = w12.LatticeC(2, 17, 16, 0, pr.ctypes.data, 0x1000, 0x1000, 0x1000)
    assert L.w12_tree_build(C.byref(lat17), 8, C.byref(tr), ws, 1 << 30, None) == w12.W12_E_UNSUPPORTED
    prbad = np.asarray([5, 1], np.int32)
    latb = w12.LatticeC(2, 4, 16, 0, prbad.ctypes.data, 0x1000, 0x1000, 0x1000)
    assert L.w12_tree_build(C.byref(latb), 8, C.byref(tr), ws, 1 << 30, None) == w12.W12_E_INVAL
    assert L.w12_tree_build(C.byref(lat), 600, C.byref(tr), ws, 1 << 30, None) == w12.W12_E_UNSUPPORTED
    # accept with a tree of zero rows
    assert L.w12_tree_accept(C.byref(tr), 2, 4, fake, fake, fake, None, None) == w12.W12_E_INVAL
    assert L.w12_workspace_bytes(0, 128, 0, 1) == 0
    assert L.w12_workspace_bytes(257, 128, 0, 1) == 0
    assert w12.status_str(w12.W12_E_TIMEOUT) == "W12_E_TIMEOUT"


def test_tlv_chain_equals_oracle(L):
    """The library's host-side TLV chain rule against the oracle's, on random
    first-tree shares and chain lengths (no device work)."""
    g = np.random.default_rng(5)
    for _ in range(300):
        n_req = int(g.integers(1, 20))
        rows = g.integers(1, 12, size=n_req)
        off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
        budget = int(off[-1] + g.integers(0, 5))
        c_len = np.asarray([g.integers(1, r + 1) for r in rows], np.int32)
        m, sub = w12.w12_tlv_chain(c_len, off, budget)
        m_ref, sub_ref = oracle.tlv_chain(c_len, off, budget)
        assert np.array_equal(m, m_ref) and sub == sub_ref
        assert sub >= n_req


def test_tlv_refusals_before_launch(L):
    m = np.zeros(1, np.int32)
    sub = C.c_int32(0)
    c_len = np.asarray([3], np.int32)
    off = np.asarray([0, 2], np.int32)   # a chain longer than the request's rows
    assert L.w12_tlv_chain(c_len.ctypes.data, off.ctypes.data, 1, 4, m.ctypes.data, C.byref(sub)) == w12.W12_E_INVAL
    off_big = np.asarray([0, 9], np.int32)   # more rows than the budget
    assert L.w12_tlv_chain(c_len.ctypes.data, off_big.ctypes.data, 1, 4, m.ctypes.data,
                           C.byref(sub)) == w12.W12_E_INVAL
    fake = C.c_void_p(0x1000)
    ws = C.c_void_p(0x100000)
    t = w12.TreeC(4, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    out = w12.TreeC(0, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    mm = np.asarray([2], np.int32)
    assert L.w12_tlv_splice(C.byref(t), None, fake, fake, 1, 4, mm.ctypes.data, C.byref(t), C.byref(out), ws,
                            1 << 30, None) == w12.W12_E_INVAL
    m_bad = np.asarray([6], np.int32)   # more than p1_max + 1 chain tokens
    assert L.w12_tlv_splice(C.byref(t), fake, fake, fake, 1, 4, m_bad.ctypes.data, C.byref(t), C.byref(out), ws,
                            1 << 30, None) == w12.W12_E_INVAL
    t_big = w12.TreeC(510, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    m5 = np.asarray([5], np.int32)      # 510 + 5 rows: over the 512-row cap
    assert L.w12_tlv_splice(C.byref(t), fake, fake, fake, 1, 4, m5.ctypes.data, C.byref(t_big), C.byref(out), ws,
                            1 << 30, None) == w12.W12_E_UNSUPPORTED
    assert L.w12_tree_accept(C.byref(t), 1, 34, fake, fake, fake, None, None) == w12.W12_E_UNSUPPORTED


def test_gdn_refusals_before_launch(L):
    ws = C.c_void_p(0x100000)
    tr = w12.TreeC(32, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    good = w12.GdnLayerC(4, 128, 0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000)
    out = C.c_void_p(0x70000)
    # head dimension other than 128
    bad_d = w12.GdnLayerC(4, 64, 0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000)
    assert L.w12_gdn_tree_verify(C.byref(bad_d), C.byref(tr), 1, 0, out, ws, 1 << 30, None) == w12.W12_E_UNSUPPORTED
    # null state, misaligned keys, unknown method
    no_s = w12.GdnLayerC(4, 128, None, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000)
    assert L.w12_gdn_tree_verify(C.byref(no_s), C.byref(tr), 1, 0, out, ws, 1 << 30, None) == w12.W12_E_INVAL
    mis = w12.GdnLayerC(4, 128, 0x10000, 0x20000, 0x30008, 0x40000, 0x50000, 0x60000)
    assert L.w12_gdn_tree_verify(C.byref(mis), C.byref(tr), 1, 0, out, ws, 1 << 30, None) == w12.W12_E_INVAL
    assert L.w12_gdn_tree_verify(C.byref(good), C.byref(tr), 1, 7, out, ws, 1 << 30, None) == w12.W12_E_INVAL
    # workspace too small, commit without accepted rows
    assert L.w12_gdn_tree_verify(C.byref(good), C.byref(tr), 1, 0, out, ws, 16, None) == w12.W12_E_WORKSPACE
    assert L.w12_gdn_commit(C.byref(good), C.byref(tr), 1, None, out, ws, 1 << 30, None) == w12.W12_E_INVAL
    # the WY form's own entry points: outputs, vectors, alignment, workspace
    u = C.c_void_p(0x80000)
    node = C.c_void_p(0x90000)
    assert L.w12_gdn_wy_verify(C.byref(bad_d), C.byref(tr), 1, out, u, ws, 1 << 30, None) == w12.W12_E_UNSUPPORTED
    assert L.w12_gdn_wy_verify(C.byref(good), C.byref(tr), 1, None, u, ws, 1 << 30, None) == w12.W12_E_INVAL
    assert L.w12_gdn_wy_verify(C.byref(good), C.byref(tr), 1, out, None, ws, 1 << 30, None) == w12.W12_E_INVAL
    assert L.w12_gdn_wy_verify(C.byref(good), C.byref(tr), 1, out, u, ws, 16, None) == w12.W12_E_WORKSPACE
    assert L.w12_gdn_wy_commit(C.byref(good), C.byref(tr), 1, None, u, out, ws, 1 << 30, None) == w12.W12_E_INVAL
    assert L.w12_gdn_wy_commit(C.byref(good), C.byref(tr), 1, node, None, out, ws, 1 << 30, None) == w12.W12_E_INVAL
    assert L.w12_gdn_wy_commit(C.byref(good), C.byref(tr), 1, node, u, C.c_void_p(0x70004), ws, 1 << 30,
                               None) == w12.W12_E_INVAL
    assert L.w12_gdn_wy_commit(C.byref(good), C.byref(tr), 1, node, C.c_void_p(0x80008), out, ws, 1 << 30,
                               None) == w12.W12_E_INVAL
    assert L.w12_gdn_wy_commit(C.byref(good), C.byref(tr), 1, node, u, out, ws, 16, None) == w12.W12_E_WORKSPACE


def test_binding_signatures_match_the_header(L):
    """Every declared entry point that the binding marshals has as many
    arguments there as in its C declaration."""
    import ctypes
    src = ""
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src += re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
    decl = {}
    for m in re.finditer(r"\b(w12_\w+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
        args = m.group(2).strip()
        decl[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    checked = 0
    for name, n in decl.items():
        f = getattr(L, name)
        if getattr(f, "argtypes", None) is None:
            continue
        assert len(f.argtypes) == n, (name, len(f.argtypes), n)
        checked += 1
    assert checked >= 25


def test_tlv_chain_edge_cases(L):
    # 512 requests holding one row each: nothing can be committed, every row is a subtree root
    n = 512
    off = np.arange(n + 1, dtype=np.int32)
    m, sub = w12.w12_tlv_chain(np.ones(n, np.int32), off, 512)
    assert not m.any() and sub == 512
    # one request whose whole share (a 32-row chain) was accepted: the bonus is dropped
    m, sub = w12.w12_tlv_chain(np.asarray([32], np.int32), np.asarray([0, 32], np.int32), 32)
    assert list(m) == [31] and sub == 1
    # the first tree held fewer rows than the budget (lattice exhausted): the rest goes to the subtrees
    m, sub = w12.w12_tlv_chain(np.asarray([2, 1], np.int32), np.asarray([0, 3, 5], np.int32), 40)
    assert list(m) == [2, 1] and sub == 37
