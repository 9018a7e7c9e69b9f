"""Shared test helpers: brute-force enumerations, lattice fixtures and the
margin-gated parity comparison.  Test infrastructure only."""
from __future__ import annotations

import itertools
import json
import os
from typing import Dict, List, Tuple

import numpy as np

from speculative_decoding_tree_w12_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# accepted tokens are compared only on requests whose consulted rows all have
# a top-2 logit margin above this (FP64 oracle logits)
MARGIN_GATE = 1e-2
# GEMM tolerance: max |y - y_ref| / max(|y_ref|, 1e-3 * max_row |y_ref|)
GEMM_REL_TOL = 2e-2


def load_golden(name: str) -> Dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# brute force over tiny lattices
# ---------------------------------------------------------------------------

def enumerate_nodes(lat: synth.Lattice) -> List[Tuple]:
    """Every node of every request's full candidate tree, as
    (score, depth, req, path_ranks, tokens, parent_ranks).  Scores are summed
    in float32 root to leaf."""
    out = []
    for r in range(lat.n_req):
        out.append((np.float32(0.0), 0, r, (), (int(lat.root_tok[r]),)))
        frontier = [((), np.float32(0.0))]
        for d in range(1, int(lat.p_r[r]) + 1):
            nxt = []
            for ranks, s in frontier:
                prev = ranks[-1] if ranks else 0
                for j in range(lat.n_cand):
                    if lat.conditional:
                        e = np.float32(lat.cand_logp[r, d - 1, prev, j])
                    else:
                        e = np.float32(lat.cand_logp[r, d - 1, j])
                    s2 = np.float32(s + e)
                    nr = ranks + (j,)
                    toks = tuple(int(lat.cand_tok[r, dd, rr]) for dd, rr in enumerate(nr))
                    out.append((s2, d, r, nr, toks))
                    nxt.append((nr, s2))
            frontier = nxt
    return out


def path_key(ranks) -> int:
    v = 0
    for d, j in enumerate(ranks, start=1):
        v |= j << (64 - 4 * d)
    return v


def brute_tree(lat: synth.Lattice, budget: int):
    """Top-``budget`` nodes under (score desc, depth asc, req asc, path asc),
    emitted grouped by request in that order.  Returns rows as dicts."""
    nodes = enumerate_nodes(lat)
    nodes.sort(key=lambda t: (-float(t[0]), t[1], t[2], path_key(t[3])))
    top = nodes[:budget]
    rows = []
    for r in range(lat.n_req):
        rows.extend([t for t in top if t[2] == r])
    index = {(t[2], t[3]): i for i, t in enumerate(rows)}
    res = []
    for t in rows:
        s, d, r, ranks, toks = t
        par = -1 if d == 0 else index[(r, ranks[:-1])]
        tok = toks[0] if d == 0 else toks[-1]
        res.append(dict(score=np.float32(s), depth=d, req=r, parent=par, token=tok,
                        rank=(ranks[-1] if ranks else 0)))
    return res


def brute_accept(parent, token, depth, req, n_req, argmax):
    """Deepest node whose whole root path matches the argmax chain, by
    enumerating every node's root path."""
    best = {}
    for j in range(len(parent)):
        ok, cur = True, j
        while parent[cur] >= 0:
            p = parent[cur]
            if token[cur] != argmax[p]:
                ok = False
                break
            cur = p
        if not ok:
            continue
        r = int(req[j])
        if r not in best or depth[j] > depth[best[r]] or (depth[j] == depth[best[r]] and j < best[r]):
            best[r] = j
    return best


def lattice_from_fixture(fx: Dict, vocab_pad: int = 64, n_cand: int = 16) -> Tuple[synth.Lattice, Dict]:
    tok = fx["tokens"]
    P = fx["positions"]
    cand_tok = np.zeros((1, P, 16), np.int32)
    cand_logp = np.full((1, P, 16), np.float32(fx["filler_logp"]), np.float32)
    for c in fx["candidates"]:
        p = c["pos"] - 1
        ids = [tok[w] for w in c["ranked"]]
        fill = [v for v in range(vocab_pad, vocab_pad + 64) if v not in ids][: 16 - len(ids)]
        cand_tok[0, p] = np.asarray(ids + fill, np.int32)
        for i, lp in enumerate(c["logp"]):
            cand_logp[0, p, i] = np.float32(lp)
        # filler log-probs strictly below the listed ones, distinct, sorted
        for i in range(len(ids), 16):
            cand_logp[0, p, i] = np.float32(fx["filler_logp"] - 0.01 * i)
    truth = np.asarray([[tok[w] for w in fx["target_greedy"]]], np.int32)
    lat = synth.Lattice(n_req=1, p_max=P, n_cand=n_cand, conditional=False,
                        p_r=np.asarray([P], np.int32), root_tok=np.asarray([fx["root_tok"]], np.int32),
                        cand_tok=cand_tok, cand_logp=cand_logp, truth=truth)
    return lat, tok


# ---------------------------------------------------------------------------
# parity
# ---------------------------------------------------------------------------

def gemm_rel_err(y: np.ndarray, y_ref: np.ndarray) -> float:
    """max |y - y_ref| / max(|y_ref|, 1e-3 * max over the row of |y_ref|)."""
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    row_max = np.abs(y_ref).max(axis=-1, keepdims=True)
    den = np.maximum(np.abs(y_ref), 1e-3 * row_max)
    den = np.where(den > 0, den, 1.0)
    return float((np.abs(y - y_ref) / den).max())


def gemm_norm_err(y: np.ndarray, y_ref: np.ndarray) -> float:
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    return float(np.linalg.norm(y - y_ref) / max(np.linalg.norm(y_ref), 1e-300))


def accepted_parity(acc_tok, acc_len, ref_tok, ref_len, ref_node, parent, margin, n_req):
    """Compare accepted tokens/lengths per request, gated by the oracle's
    margins on every row whose argmax the reference acceptance consulted:
    the accepted path from the root down to the deepest accepted node (its
    argmax picks the next child or the bonus token).  Returns
    (compared, mismatched, near_tie) request lists."""
    compared, mismatched, near = [], [], []
    for r in range(n_req):
        node = int(ref_node[r])
        path = []
        cur = node
        while cur >= 0:
            path.append(cur)
            cur = int(parent[cur])
        if any(margin[j] <= MARGIN_GATE for j in path):
            near.append(r)
            continue
        compared.append(r)
        n = int(ref_len[r])
        if int(acc_len[r]) != n or not np.array_equal(np.asarray(acc_tok[r][:n]), np.asarray(ref_tok[r][:n])):
            mismatched.append(r)
    return compared, mismatched, near


# ---------------------------------------------------------------------------
# TLV cycle inputs (explainer 4.3): a long true continuation per request, the
# first lattice over its start, a toy target that prefers the true next token
# on the true path, a Q-pass argmax that may disagree with it, and the second
# lattice drafted from each chain end
# ---------------------------------------------------------------------------

def tlv_truth(w: synth.Workload, p2: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed * 7 + 3)
    return g.integers(0, w.vocab, size=(w.n_req, w.p_max + p2 + 2)).astype(np.int32)


def target_argmax(tree, truth_long: np.ndarray, vocab: int, seed: int) -> np.ndarray:
    """The toy target's greedy token at every row: a function of the row's
    (request, root path) only."""
    paths = synth.tree_paths(tree.parent, tree.token)
    return np.asarray([synth.planted_token(int(tree.req[j]), paths[j], truth_long, vocab, seed)
                       for j in range(len(paths))], np.int32)


def q_argmax(exact: np.ndarray, err: float, vocab: int, seed: int) -> np.ndarray:
    """A Q-pass argmax that differs from the exact one at a fraction ``err``
    of the rows."""
    g = np.random.default_rng(seed * 11 + 5)
    q = exact.copy()
    bad = g.random(len(q)) < err
    q[bad] = g.integers(0, vocab, size=int(bad.sum()))
    return q


def greedy_ar(req: int, truth_long: np.ndarray, vocab: int, seed: int, n: int) -> List[int]:
    """n tokens of greedy autoregressive decoding under the toy target."""
    out: List[int] = []
    for _ in range(n):
        out.append(synth.planted_token(req, out, truth_long, vocab, seed))
    return out


def second_lattice(w2: synth.Workload, lat1: synth.Lattice, c_tok: np.ndarray, m: np.ndarray,
                   truth_long: np.ndarray, seed: int) -> synth.Lattice:
    """The lattice drafted from each request's chain end: its root is the
    last committed chain token (the first tree's root when m = 0); where the
    chain follows the true continuation the drafter is offered the rest of
    it, elsewhere a drawn one."""
    p2 = w2.p_max
    g = np.random.default_rng(seed * 13 + 7)
    truth2 = g.integers(0, w2.vocab, size=(w2.n_req, p2 + 1)).astype(np.int32)
    root2 = np.asarray(lat1.root_tok, np.int32).copy()
    for q in range(w2.n_req):
        mq = int(m[q])
        if mq:
            root2[q] = int(c_tok[q][mq - 1])
        if np.array_equal(np.asarray(c_tok[q][:mq]), truth_long[q, :mq]):
            truth2[q] = truth_long[q, mq:mq + p2 + 1]
    return synth.lattice(w2, seed + 101, truth=truth2, root_tok=root2)
