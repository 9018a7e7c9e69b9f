"""CPU oracle for the W12 tree-verify pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``w12_oracle.c`` (plain C,
FP64 accumulation, ``-ffp-contract=off``) through ctypes and shares no code
with the CUDA library.  Each wrapper names the passage it follows; the C file
lists the readings taken where the pages are silent.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(exhaustive round trip, hand-computed window cases, NumPy cross-check,
exact integer GEMM, brute-force tree and acceptance enumeration, the greedy
autoregressive invariant and the planted-defect mutation); the TLV chain and
splice by ``tests/test_oracle_tlv.py`` (hand-built trees, greedy
autoregressive decoding through the combined tree under any Q-pass argmax,
tree invariants); the recurrent-layer tree functions by
``tests/test_oracle_gdn.py`` (closed forms for pure decay and for a unit key
written at full strength, independence from rows off the root path, an
independent WY-form restatement (outputs and the WY vectors u), the commit
state, and the commit rebuilt from the WY vectors).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w12_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

TILE_N, TILE_K, REC_BYTES = 128, 64, 12288


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (host code; same flags on x86 and Arm)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        p = C.c_void_p
        i64, i32 = C.c_int64, C.c_int32
        L.orc_w12_layout.argtypes = [p, i64, i64, p, p]
        L.orc_w12_pack.argtypes = [p, i64, i64, p, p, p, p]
        L.orc_w12_unpack_rows.argtypes = [p, p, p, p, i64, i64, i64, i64, p]
        L.orc_w12_unpack_rows_q.argtypes = [p, p, p, p, i64, i64, i64, i64, p]
        L.orc_gemm_f64.argtypes = [p, i64, p, i64, i64, p, C.c_int]
        L.orc_head_argmax.argtypes = [p, i64, p, i64, i64, p, p, p, p, C.c_int]
        L.orc_tree_build.argtypes = [i32, i32, i32, i32, p, p, p, p, i32, p, p, p, p, p, p, p, p]
        L.orc_tree_accept.argtypes = [i32, p, p, p, p, i32, i32, p, p, p, p]
        for f in (L.orc_w12_layout, L.orc_w12_pack, L.orc_w12_unpack_rows, L.orc_w12_unpack_rows_q, L.orc_gemm_f64,
                  L.orc_head_argmax, L.orc_tree_build, L.orc_tree_accept):
            f.restype = C.c_int
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


# ---------------------------------------------------------------------------
# W12 (SpecPilot explainer "4.1 W12: a 12-bit lossless weight format")
# ---------------------------------------------------------------------------

class Packed:
    """Host-side W12 tensor: records, per-channel window base, escape index."""

    def __init__(self, n, k, rec, base, esc_tile_off, esc):
        self.n, self.k = n, k
        self.rec, self.base, self.esc_tile_off, self.esc = rec, base, esc_tile_off, esc

    @property
    def n_escapes(self) -> int:
        return int(self.esc.shape[0])

    @property
    def bytes(self) -> int:
        return self.rec.nbytes + self.base.nbytes + self.esc_tile_off.nbytes + self.esc.nbytes


def w12_pack(w: np.ndarray) -> Packed:
    """Pack BF16 bits ``w[n][k]`` into W12 (window choice, records, escapes)."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    n, k = w.shape
    L = lib()
    base = np.empty(n, dtype=np.uint8)
    ne = np.zeros(1, dtype=np.int64)
    _check(L.orc_w12_layout(_ptr(w), n, k, _ptr(base), _ptr(ne)), "w12_layout")
    tiles = (n // TILE_N) * (k // TILE_K)
    rec = np.empty(tiles * REC_BYTES, dtype=np.uint8)
    off = np.empty(tiles + 1, dtype=np.int32)
    esc = np.empty(int(ne[0]), dtype=np.uint32)
    _check(L.orc_w12_pack(_ptr(w), n, k, _ptr(base), _ptr(rec), _ptr(off), _ptr(esc) if esc.size else None),
           "w12_pack")
    return Packed(n, k, rec, base, off, esc)


def w12_unpack(p: Packed, row0: int = 0, nrows: Optional[int] = None) -> np.ndarray:
    """Decode rows ``[row0, row0 + nrows)`` back to BF16 bits."""
    nrows = p.n - row0 if nrows is None else nrows
    out = np.empty((nrows, p.k), dtype=np.uint16)
    esc = p.esc if p.esc.size else np.zeros(1, dtype=np.uint32)
    _check(lib().orc_w12_unpack_rows(_ptr(p.rec), _ptr(p.base), _ptr(p.esc_tile_off), _ptr(esc),
                                     p.n, p.k, row0, nrows, _ptr(out)), "w12_unpack")
    return out


def w12_unpack_q(p: Packed, row0: int = 0, nrows: Optional[int] = None) -> np.ndarray:
    """Quick-pass weights of rows ``[row0, row0 + nrows)`` as BF16 bits (R19:
    view byte with the low mantissa nibble 0b1000; escapes exact)."""
    nrows = p.n - row0 if nrows is None else nrows
    out = np.empty((nrows, p.k), dtype=np.uint16)
    esc = p.esc if p.esc.size else np.zeros(1, dtype=np.uint32)
    _check(lib().orc_w12_unpack_rows_q(_ptr(p.rec), _ptr(p.base), _ptr(p.esc_tile_off), _ptr(esc),
                                       p.n, p.k, row0, nrows, _ptr(out)), "w12_unpack_q")
    return out


# ---------------------------------------------------------------------------
# Verify GEMM and LM-head argmax (explainer "1.1", "2.1")
# ---------------------------------------------------------------------------

def gemm_f64(x: np.ndarray, w: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """``y = x . w^T`` with BF16 inputs and FP64 accumulation."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    R, k = x.shape
    n = w.shape[0]
    assert w.shape[1] == k
    y = np.empty((R, n), dtype=np.float64)
    _check(lib().orc_gemm_f64(_ptr(x), R, _ptr(w), n, k, _ptr(y), nthreads), "gemm_f64")
    return y


def head_argmax(h: np.ndarray, w_head: np.ndarray, bias: Optional[np.ndarray] = None,
                nthreads: int = 0) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Per row of ``h``: argmax over ``h . w_head^T`` (+ bias), the top-1 logit
    and the top1 - top2 margin, all from FP64 logits."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    w_head = np.ascontiguousarray(w_head, dtype=np.uint16)
    R, k = h.shape
    V = w_head.shape[0]
    am = np.empty(R, dtype=np.int32)
    t1 = np.empty(R, dtype=np.float64)
    mg = np.empty(R, dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    _check(lib().orc_head_argmax(_ptr(h), R, _ptr(w_head), V, k, _ptr(b), _ptr(am), _ptr(t1), _ptr(mg),
                                 nthreads), "head_argmax")
    return am, t1, mg


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def certified_head(h: np.ndarray, p: Packed):
    """Certified LM head (explainer "4.1"/"4.3": a cheap pass over the head,
    a per-row Cauchy-Schwarz error bound that discards tokens proven unable
    to be the argmax, exact rescoring of the survivors; the argmax equals the
    dense one).  Reading: the cheap pass reads each record's 8-bit view (the
    quick-pass weights w^), not a separate INT8 copy, so the bound for row r
    and token v is ||h_r|| * ||w_v - w^_v||.  All in FP64.

    Returns (argmax per row, survivors per row, the per-token norms
    ||w_v - w^_v|| and ||w^_v||)."""
    hf = _bf16_to_f64(h)
    w = _bf16_to_f64(w12_unpack(p))
    wq = _bf16_to_f64(w12_unpack_q(p))
    err = np.sqrt(((w - wq) ** 2).sum(axis=1))
    qn = np.sqrt((wq ** 2).sum(axis=1))
    sq = hf @ wq.T
    eps = np.sqrt((hf ** 2).sum(axis=1))[:, None] * err[None, :]
    low = (sq - eps).max(axis=1)
    surv = (sq + eps) >= low[:, None]
    am = np.empty(hf.shape[0], dtype=np.int32)
    for r in range(hf.shape[0]):
        idx = np.nonzero(surv[r])[0]
        s = w[idx] @ hf[r]
        am[r] = idx[int(np.argmax(s))]          # first maximum: lowest index on ties
    return am, surv.sum(axis=1).astype(np.int64), err, qn


# ---------------------------------------------------------------------------
# Best-first tree (explainer "4.2", "4.4") and acceptance ("1.1")
# ---------------------------------------------------------------------------

class Tree:
    def __init__(self, R, parent, token, depth, req, score, rank, req_row_off):
        self.R = R
        self.parent, self.token, self.depth, self.req = parent, token, depth, req
        self.score, self.rank, self.req_row_off = score, rank, req_row_off


def tree_build(lat, budget: int) -> Tree:
    """Best-first tree over a lattice (``synth.Lattice``) with a shared budget."""
    n_req, p_max = lat.n_req, lat.p_max
    out = dict(parent=np.empty(budget, np.int32), token=np.empty(budget, np.int32),
               depth=np.empty(budget, np.uint8), req=np.empty(budget, np.int32),
               score=np.empty(budget, np.float32), rank=np.empty(budget, np.uint8))
    off = np.empty(n_req + 1, np.int32)
    R = np.zeros(1, np.int32)
    ct = np.ascontiguousarray(lat.cand_tok, np.int32)
    cl = np.ascontiguousarray(lat.cand_logp, np.float32)
    rc = lib().orc_tree_build(n_req, p_max, lat.n_cand, int(bool(lat.conditional)),
                              _ptr(np.ascontiguousarray(lat.p_r, np.int32)),
                              _ptr(np.ascontiguousarray(lat.root_tok, np.int32)), _ptr(ct), _ptr(cl), budget,
                              _ptr(out["parent"]), _ptr(out["token"]), _ptr(out["depth"]), _ptr(out["req"]),
                              _ptr(out["score"]), _ptr(out["rank"]), _ptr(off), _ptr(R))
    _check(rc, "tree_build")
    r = int(R[0])
    return Tree(r, *(out[k][:r] for k in ("parent", "token", "depth", "req", "score", "rank")), off)


def tree_accept(tree: Tree, argmax: np.ndarray, n_req: int, p_max: int):
    """Greedy acceptance on every request's share of the tree."""
    acc_tok = np.empty((n_req, p_max + 1), np.int32)
    acc_len = np.empty(n_req, np.int32)
    acc_node = np.empty(n_req, np.int32)
    am = np.ascontiguousarray(argmax, np.int32)
    _check(lib().orc_tree_accept(tree.R, _ptr(tree.parent), _ptr(tree.token), _ptr(tree.depth),
                                 _ptr(tree.req_row_off), n_req, p_max, _ptr(am), _ptr(acc_tok),
                                 _ptr(acc_len), _ptr(acc_node)), "tree_accept")
    return acc_tok, acc_len, acc_node


# ---------------------------------------------------------------------------
# TLV: commit chain and splice (explainer "4.3")
# ---------------------------------------------------------------------------

BONUS_RANK = 255     # rank of the chain's bonus token: not a drafted candidate


def tlv_chain(c_len: np.ndarray, t1_row_off: np.ndarray, budget: int):
    """Commit chain lengths and the fresh subtree's budget (explainer "4.3").

    The Q pass's greedy acceptance over the first tree gives, per request q,
    the chain C_q: its accepted draft tokens and the bonus token, c_len[q] of
    them.  Reading: the exact pass keeps the first tree's budget N; request
    q commits m_q = min(c_len[q], N_q - 1) chain tokens, N_q being its row
    count in the first tree (the cap only ever drops the bonus, when the
    request's whole share was accepted), so every request keeps one row for
    its subtree root.  The fresh subtrees, drafted from the chain ends, share
    N - sum(m_q) rows counting their roots, which are the chain ends: for one
    request that is the pages' N - |C|."""
    n_req = len(c_len)
    m = np.zeros(n_req, np.int32)
    for q in range(n_req):
        rows_q = int(t1_row_off[q + 1]) - int(t1_row_off[q])
        m[q] = max(0, min(int(c_len[q]), rows_q - 1))
    return m, int(budget) - int(m.sum())


def tlv_splice(t1: Tree, c_tok: np.ndarray, c_len: np.ndarray, c_node: np.ndarray, m: np.ndarray,
               t2: Tree, n_req: int) -> Tree:
    """The combined tree of one TLV cycle (explainer "4.3"): per request the
    first tree's root, then the first m_q tokens of the commit chain as a
    path, then the fresh subtree (drafted from the chain end, its root being
    that end) attached under the chain's last row.

    Rows stay grouped by request, parents before children.  Chain rows copy
    the first tree's rank and score along the Q-accepted path; the bonus row
    takes rank BONUS_RANK and its parent's score; a subtree row's depth is
    m_q plus its own and its score is the chain end's plus its own (FP32)."""
    par, tok, dep, req, sc, rk = [], [], [], [], [], []
    off = [0]
    for q in range(n_req):
        base = len(par)
        path = []
        j = int(c_node[q])
        while j >= 0:
            path.append(j)
            j = int(t1.parent[j])
        path.reverse()
        if len(path) != int(c_len[q]) or not 0 <= int(m[q]) <= int(c_len[q]):
            raise ValueError("commit chain of request %d does not match the first tree" % q)
        root = path[0]
        par.append(-1); tok.append(int(t1.token[root])); dep.append(0); req.append(q)
        sc.append(np.float32(t1.score[root])); rk.append(int(t1.rank[root]))
        for i in range(1, int(m[q]) + 1):
            t = int(c_tok[q][i - 1])
            if i < len(path):
                if t != int(t1.token[path[i]]):
                    raise ValueError("chain token %d of request %d is not the tree's" % (i, q))
                s, r = np.float32(t1.score[path[i]]), int(t1.rank[path[i]])
            else:
                s, r = sc[-1], BONUS_RANK
            par.append(base + i - 1); tok.append(t); dep.append(i); req.append(q); sc.append(s); rk.append(r)
        end = base + int(m[q])
        lo, hi = int(t2.req_row_off[q]), int(t2.req_row_off[q + 1])
        if hi <= lo or int(t2.token[lo]) != tok[end]:
            raise ValueError("subtree of request %d is not rooted at the chain end" % q)
        for j in range(lo + 1, hi):
            par.append(end + int(t2.parent[j]) - lo); tok.append(int(t2.token[j]))
            dep.append(int(m[q]) + int(t2.depth[j])); req.append(q)
            sc.append(np.float32(sc[end] + np.float32(t2.score[j]))); rk.append(int(t2.rank[j]))
        off.append(len(par))
    R = len(par)
    return Tree(R, np.asarray(par, np.int32), np.asarray(tok, np.int32), np.asarray(dep, np.uint8),
                np.asarray(req, np.int32), np.asarray(sc, np.float32), np.asarray(rk, np.uint8),
                np.asarray(off, np.int32))


# ---------------------------------------------------------------------------
# Gated DeltaNet layer over a draft tree (explainer "4.2": a recurrent head
# keeps a fixed-size state updated once per token; the tree recomputes the
# state along each root path from the committed state)
# ---------------------------------------------------------------------------

def gdn_tree_path(S0: np.ndarray, q: np.ndarray, k: np.ndarray, v: np.ndarray, alpha: np.ndarray,
                  beta: np.ndarray, tree: Tree):
    """Per-node outputs of one GDN layer over a tree, in FP64, by walking every
    node's root path from its request's committed state.

    Reading (the pages name the layer and its rank-one updates; the update is
    the published gated delta rule): per head, with state S (d_v x d_k), a
    token with gate a, strength b, key k, value v, query q does
        S <- a * S (I - b k k^T) + b v k^T,      output o = S q.
    Every row of the tree is a token: the root applies its update to the
    committed state S0[request], a child to its parent's state.

    S0: float [n_req][H][d_v][d_k]; q, k: BF16 bits [R][H][d_k]; v: BF16 bits
    [R][H][d_v]; alpha, beta: float [R][H].  Returns o float64 [R][H][d_v]."""
    qf, kf, vf = _bf16_to_f64(q), _bf16_to_f64(k), _bf16_to_f64(v)
    a64, b64 = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    R, H, dk = qf.shape
    dv = vf.shape[2]
    out = np.empty((R, H, dv), np.float64)
    for j in range(R):
        path = []
        i = j
        while i >= 0:
            path.append(i)
            i = int(tree.parent[i])
        path.reverse()
        S = np.array(S0[int(tree.req[j])], np.float64)            # [H][d_v][d_k]
        for i in path:
            Sk = np.einsum("hvk,hk->hv", S, kf[i])
            S = a64[i][:, None, None] * (S - b64[i][:, None, None] * Sk[:, :, None] * kf[i][:, None, :]) \
                + b64[i][:, None, None] * vf[i][:, :, None] * kf[i][:, None, :]
        out[j] = np.einsum("hvk,hk->hv", S, qf[j])
    return out


def gdn_wy_u(S0: np.ndarray, k: np.ndarray, v: np.ndarray, alpha: np.ndarray, beta: np.ndarray, tree: Tree):
    """The WY vectors of every tree row (FP64), by their definition (SpecPilot
    explainer 4.2, TreeWY): u_j = b_j (v_j - a_j S_p k_j), where S_p is the
    state the row's update applies to (its parent's state after the parent's
    update, or the request's committed state for a root), found by walking
    the root path as gdn_tree_path does.  With them the state after row j is
    g_j S0 + sum over i on j's root path of (g_j / g_i) u_i k_i^T (g the
    product of the gates along the path).  Returns float64 [R][H][d_v]."""
    kf, vf = _bf16_to_f64(k), _bf16_to_f64(v)
    a64, b64 = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    R, H, _ = kf.shape
    out = np.empty((R, H, vf.shape[2]), np.float64)
    for j in range(R):
        path = []
        i = int(tree.parent[j])
        while i >= 0:
            path.append(i)
            i = int(tree.parent[i])
        S = np.array(S0[int(tree.req[j])], np.float64)
        for i in reversed(path):
            Sk = np.einsum("hvk,hk->hv", S, kf[i])
            S = a64[i][:, None, None] * (S - b64[i][:, None, None] * Sk[:, :, None] * kf[i][:, None, :]) \
                + b64[i][:, None, None] * vf[i][:, :, None] * kf[i][:, None, :]
        Sk = np.einsum("hvk,hk->hv", S, kf[j])
        out[j] = b64[j][:, None] * (vf[j] - a64[j][:, None] * Sk)
    return out


def gdn_commit(S0: np.ndarray, k: np.ndarray, v: np.ndarray, alpha: np.ndarray, beta: np.ndarray, tree: Tree,
               acc_node: np.ndarray):
    """The committed state after acceptance (FP64): each request's state
    replayed along the root path of its deepest accepted row."""
    kf, vf = _bf16_to_f64(k), _bf16_to_f64(v)
    a64, b64 = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    out = np.array(S0, np.float64)
    for r, node in enumerate(acc_node):
        path = []
        i = int(node)
        while i >= 0:
            path.append(i)
            i = int(tree.parent[i])
        S = out[r]
        for i in reversed(path):
            Sk = np.einsum("hvk,hk->hv", S, kf[i])
            S = a64[i][:, None, None] * (S - b64[i][:, None, None] * Sk[:, :, None] * kf[i][:, None, :]) \
                + b64[i][:, None, None] * vf[i][:, :, None] * kf[i][:, None, :]
        out[r] = S
    return out
