"""Seeded synthetic inputs for the W12 tree-verify pass.

This module is shared by the tests, the benchmark and the CPU oracle's drivers.
It draws random numbers and arranges them into the shapes the pass consumes;
it holds none of the method's arithmetic (no W12 coding, no GEMM, no argmax,
no tree selection, no acceptance).

What it stands in for (SpecPilot explainer, "5.1 Measurement conditions"):
the pages measure on real models and real benchmark prompts, which are not
available here.  Every input below is synthetic, with the shapes of the
pages' workloads:

* weights  - BF16 ``W[N][K]`` (PyTorch Linear layout), N(0, 0.02) times a
  per-row scale U[0.5, 2], rounded to BF16 with round-to-nearest-even;
  optional outliers (x64) and exact zeros force escapes ("4.1 W12");
* lattice  - per request and drafted position, 16 candidate tokens with
  log-probabilities (a DFlash2-like top-16 output, "1.1"), or a
  parent-conditioned table (DSpark-like, "1.1" and "4.2");
* hidden rows - a toy target whose row for a tree node depends only on the
  node's root path: ``h = a_t * W_head[t] + N(0, 1)`` with ``t`` the planted
  next token, so the target's greedy token is known by construction.

Seeds: every stream is ``numpy.random.default_rng(SeedSequence([seed, stream]))``.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# --------------------------------------------------------------------------
# random streams and BF16 bit handling
# --------------------------------------------------------------------------

STREAM_LINEAR = 1000   # + linear index (+ 100 * layer for stacked layers)
STREAM_HEAD = 2000
STREAM_X = 3000        # + linear index
STREAM_LATTICE = 4000
STREAM_TRUTH = 5000


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(stream)]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to BF16 (round to nearest, ties to even); NaN stays NaN."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    lsb = (u >> 16) & 1
    r = ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# weights and activations
# --------------------------------------------------------------------------

def weights(n: int, k: int, seed: int, stream: int, outlier_frac: float = 0.0,
            zero_frac: float = 0.0, chunk_rows: int = 4096) -> np.ndarray:
    """BF16 bits ``[n][k]``: N(0, 0.02) * U[0.5, 2] per row, plus optional
    x64 outliers and exact zeros (each a fraction of all entries).

    Rows are drawn in chunks of ``chunk_rows``, chunk i from the child stream
    SeedSequence([seed, stream, i]); chunks are filled on a thread pool."""
    import concurrent.futures as cf
    import os

    out = np.empty((n, k), dtype=np.uint16)

    def fill(i):
        r0, r1 = i * chunk_rows, min(n, (i + 1) * chunk_rows)
        g = np.random.default_rng(np.random.SeedSequence([int(seed), int(stream), i]))
        w = g.standard_normal((r1 - r0, k), dtype=np.float32)
        w *= np.float32(0.02)
        w *= g.uniform(0.5, 2.0, size=(r1 - r0, 1)).astype(np.float32)
        if outlier_frac > 0.0:
            m = g.random((r1 - r0, k)) < outlier_frac
            w[m] *= np.float32(64.0)
        if zero_frac > 0.0:
            m = g.random((r1 - r0, k)) < zero_frac
            w[m] = 0.0
        out[r0:r1] = f32_to_bf16_bits(w)

    chunks = (n + chunk_rows - 1) // chunk_rows
    if chunks == 1:
        fill(0)
    else:
        with cf.ThreadPoolExecutor(max_workers=min(chunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(chunks)))
    return out


def activations(rows: int, k: int, seed: int, stream: int) -> np.ndarray:
    """BF16 bits ``[rows][k]`` drawn from N(0, 1)."""
    g = rng(seed, stream)
    return f32_to_bf16_bits(g.standard_normal((rows, k), dtype=np.float32))


# --------------------------------------------------------------------------
# workload shapes (named by what they are)
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    linears: Tuple[Tuple[int, int], ...]   # (N, K) per linear, in launch order
    vocab: int
    hidden: int
    n_req: int
    positions: Tuple[int, ...]             # drafted positions a request may pick
    budget: int                            # node budget (roots included)
    n_cand: int = 16                       # 1 = chain (rank-0 candidates only)
    conditional: bool = False
    layers: int = 1                        # stacked copies of the linears
    outlier_frac: float = 0.0
    zero_frac: float = 0.0
    hit_rate: float = 0.8
    seed: int = 0

    @property
    def p_max(self) -> int:
        return max(self.positions)


LAYER_27B = ((7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408))
LAYER_4B = ((3584, 2560), (2560, 2560), (19456, 2560), (2560, 9728))

WORKLOADS: Dict[str, Workload] = {
    # one small linear + small head, an 8-row chain over 8 drafted positions
    "tiny": Workload("tiny", ((1024, 512),), vocab=4096, hidden=512, n_req=1,
                     positions=(8,), budget=8, n_cand=1, outlier_frac=0.01,
                     zero_frac=0.01),
    # one 27B-like decoder layer + 151936x5120 head, single request, 32-node tree
    "single_27b": Workload("single_27b", LAYER_27B, vocab=151936, hidden=5120,
                           n_req=1, positions=(16,), budget=32),
    # same shapes, 24 requests sharing a 192-node budget, 16/12/8 positions
    "batched_27b": Workload("batched_27b", LAYER_27B, vocab=151936, hidden=5120,
                            n_req=24, positions=(16, 12, 8), budget=192),
    # 4B-like layer + head, 32 requests, 256-node budget (trees)
    "b4_tree": Workload("b4_tree", LAYER_4B, vocab=151936, hidden=2560,
                        n_req=32, positions=(8, 12, 16), budget=256),
    # the same with chains (rank-0 candidates only)
    "b4_chain": Workload("b4_chain", LAYER_4B, vocab=151936, hidden=2560,
                         n_req=32, positions=(8, 12, 16), budget=256, n_cand=1),
    # 64 stacked 27B-like layers + head; one request's 32-node tree by
    # default, rows swept by the caller
    "full_depth_27b": Workload("full_depth_27b", LAYER_27B, vocab=151936,
                               hidden=5120, n_req=1, positions=(16,),
                               budget=32, layers=64),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller test cases)."""
    return dataclasses.replace(w, **kw)


# --------------------------------------------------------------------------
# drafter lattice
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Lattice:
    n_req: int
    p_max: int
    n_cand: int
    conditional: bool
    p_r: np.ndarray          # int32 [n_req]
    root_tok: np.ndarray     # int32 [n_req]
    cand_tok: np.ndarray     # int32 [n_req][p_max][16]
    cand_logp: np.ndarray    # float32 [n_req][p_max][16] or [n_req][p_max][16][16]
    truth: np.ndarray        # int32 [n_req][p_max + 1]: target's greedy continuation


def _log_softmax_sorted(g: np.random.Generator, shape) -> np.ndarray:
    """Drafter scores: 16 sorted N(0, 1.5) logits plus one 'rest' bucket,
    log-softmax over the 17, keep the 16 (all <= 0, descending)."""
    logits = g.normal(0.0, 1.5, size=tuple(shape) + (17,)).astype(np.float64)
    cand = -np.sort(-logits[..., :16], axis=-1)
    allv = np.concatenate([cand, logits[..., 16:]], axis=-1)
    mx = allv.max(axis=-1, keepdims=True)
    lse = mx + np.log(np.exp(allv - mx).sum(axis=-1, keepdims=True))
    return (cand - lse).astype(np.float32)


def lattice(w: Workload, seed: Optional[int] = None, truth: Optional[np.ndarray] = None,
            root_tok: Optional[np.ndarray] = None) -> Lattice:
    """Drafter lattice of workload ``w``.  ``truth`` ([n_req][p_max + 1]) and
    ``root_tok`` ([n_req]) replace the drawn continuation and roots when given
    (a second draft from the end of a committed chain); the random streams are
    consumed the same way either way."""
    seed = w.seed if seed is None else seed
    g = rng(seed, STREAM_LATTICE)
    gt = rng(seed, STREAM_TRUTH)
    n_req, p_max, V = w.n_req, w.p_max, w.vocab
    p_r = g.choice(np.asarray(w.positions), size=n_req).astype(np.int32)
    drawn_truth = gt.integers(0, V, size=(n_req, p_max + 1)).astype(np.int32)
    drawn_root = gt.integers(0, V, size=n_req).astype(np.int32)
    truth = drawn_truth if truth is None else np.ascontiguousarray(truth, np.int32).reshape(n_req, p_max + 1)
    root_tok = drawn_root if root_tok is None else np.ascontiguousarray(root_tok, np.int32).reshape(n_req)
    cand_tok = np.zeros((n_req, p_max, 16), dtype=np.int32)
    if w.conditional:
        logp = _log_softmax_sorted(g, (n_req, p_max, 16))
    else:
        logp = _log_softmax_sorted(g, (n_req, p_max))
    for r in range(n_req):
        for p in range(p_max):
            toks = g.choice(V, size=16, replace=False).astype(np.int32)
            # place the true token with probability hit_rate, at a rank drawn
            # from the drafter's own probabilities at this position
            if g.random() < w.hit_rate:
                lp = logp[r, p] if not w.conditional else logp[r, p, 0]
                pr = np.exp(lp.astype(np.float64))
                pr /= pr.sum()
                rank = int(g.choice(16, p=pr))
                t = truth[r, p]
                hit = np.nonzero(toks == t)[0]
                if hit.size:
                    toks[hit[0]] = toks[rank]
                toks[rank] = t
            else:
                # make sure the true token is absent
                while (toks == truth[r, p]).any():
                    bad = np.nonzero(toks == truth[r, p])[0][0]
                    toks[bad] = int(g.integers(0, V))
                    if len(set(toks.tolist())) != 16:
                        toks = g.choice(V, size=16, replace=False).astype(np.int32)
            cand_tok[r, p] = toks
    return Lattice(n_req=n_req, p_max=p_max, n_cand=w.n_cand,
                   conditional=w.conditional, p_r=p_r, root_tok=root_tok,
                   cand_tok=cand_tok, cand_logp=np.ascontiguousarray(logp),
                   truth=truth)


# --------------------------------------------------------------------------
# toy target: hidden rows as a function of (request, root path)
# --------------------------------------------------------------------------

PLANT_LOGIT = 30.0
NOISE_STD = 1.0


def _path_hash(req: int, path: Sequence[int], salt: int) -> int:
    h = hashlib.blake2b(digest_size=8)
    h.update(np.asarray([salt, req, len(path)], dtype=np.int64).tobytes())
    h.update(np.asarray(path, dtype=np.int64).tobytes())
    return int.from_bytes(h.digest(), "little")


def planted_token(req: int, path: Sequence[int], truth: np.ndarray, vocab: int,
                  seed: int) -> int:
    """The token a node's hidden row is built to prefer.

    On-path nodes (path equal to the request's true continuation so far)
    prefer the next true token; any other node prefers a token derived from
    a hash of its path.  Depends only on (request, path)."""
    d = len(path)
    if d < truth.shape[1] and all(int(path[i]) == int(truth[req, i]) for i in range(d)):
        return int(truth[req, d])
    return _path_hash(req, path, seed * 7919 + 1) % vocab


def hidden_row(req: int, path: Sequence[int], truth: np.ndarray,
               w_head_bits: np.ndarray, head_norm2: np.ndarray, seed: int,
               plant_logit: float = PLANT_LOGIT,
               noise_std: float = NOISE_STD) -> np.ndarray:
    """BF16 bits of the hidden row of the node reached by ``path`` in request
    ``req``: ``a_t * W_head[t] + N(0, noise_std)`` with ``t`` the planted
    token and ``a_t = plant_logit / ||W_head[t]||^2``."""
    vocab, kh = w_head_bits.shape
    t = planted_token(req, path, truth, vocab, seed)
    g = np.random.default_rng(_path_hash(req, path, seed * 7919 + 2))
    noise = g.standard_normal(kh, dtype=np.float32) * np.float32(noise_std)
    n2 = float(head_norm2[t])
    a = np.float32(plant_logit / n2) if n2 > 0 else np.float32(0.0)
    wt = bf16_bits_to_f32(w_head_bits[t])
    return f32_to_bf16_bits(a * wt + noise)


def head_norms(w_head_bits: np.ndarray, chunk: int = 8192) -> np.ndarray:
    out = np.empty(w_head_bits.shape[0], dtype=np.float64)
    for i in range(0, w_head_bits.shape[0], chunk):
        f = bf16_bits_to_f32(w_head_bits[i:i + chunk]).astype(np.float64)
        out[i:i + chunk] = (f * f).sum(axis=1)
    return out


def tree_paths(parent: np.ndarray, token: np.ndarray) -> List[List[int]]:
    """Root path (draft tokens, root excluded) of every row of a tree whose
    rows list each parent before its children."""
    paths: List[List[int]] = []
    for j in range(len(parent)):
        p = int(parent[j])
        paths.append([] if p < 0 else paths[p] + [int(token[j])])
    return paths


def hidden_rows(req: np.ndarray, parent: np.ndarray, token: np.ndarray,
                truth: np.ndarray, w_head_bits: np.ndarray, seed: int,
                plant_logit: float = PLANT_LOGIT,
                noise_std: float = NOISE_STD,
                head_norm2: Optional[np.ndarray] = None) -> np.ndarray:
    """Hidden rows ``[R][K_h]`` (BF16 bits) for every row of a tree."""
    if head_norm2 is None:
        head_norm2 = head_norms(w_head_bits)
    paths = tree_paths(parent, token)
    rows = np.empty((len(parent), w_head_bits.shape[1]), dtype=np.uint16)
    for j, path in enumerate(paths):
        rows[j] = hidden_row(int(req[j]), path, truth, w_head_bits, head_norm2,
                             seed, plant_logit, noise_std)
    return rows


# --------------------------------------------------------------------------
# recurrent (Gated DeltaNet) layer inputs over a draft tree
# --------------------------------------------------------------------------

STREAM_GDN = 6000


@dataclasses.dataclass
class GdnInputs:
    S0: np.ndarray       # float32 [n_req][H][d_v][d_k]: committed states
    q: np.ndarray        # BF16 bits [R][H][d_k]
    k: np.ndarray        # BF16 bits [R][H][d_k], rows of unit L2 norm before rounding
    v: np.ndarray        # BF16 bits [R][H][d_v]
    alpha: np.ndarray    # float32 [R][H], gates in [0.85, 1)
    beta: np.ndarray     # float32 [R][H], write strengths in [0.05, 0.95]


def gdn_inputs(R: int, n_req: int, H: int, d: int = 128, seed: int = 0, state_std: float = 0.05) -> GdnInputs:
    """Seeded synthetic inputs of one recurrent layer for R tree rows: keys
    and queries of unit norm (as the layer normalises them), N(0, 1) values,
    gates near 1 and write strengths spread over (0, 1), committed states
    N(0, state_std)."""
    g = rng(seed, STREAM_GDN)
    S0 = (g.standard_normal((n_req, H, d, d)) * state_std).astype(np.float32)
    k = g.standard_normal((R, H, d))
    k /= np.linalg.norm(k, axis=2, keepdims=True)
    q = g.standard_normal((R, H, d))
    q /= np.linalg.norm(q, axis=2, keepdims=True)
    v = g.standard_normal((R, H, d)).astype(np.float32)
    alpha = g.uniform(0.85, 1.0, size=(R, H)).astype(np.float32)
    beta = g.uniform(0.05, 0.95, size=(R, H)).astype(np.float32)
    return GdnInputs(S0=S0, q=f32_to_bf16_bits(q.astype(np.float32)), k=f32_to_bf16_bits(k.astype(np.float32)),
                     v=f32_to_bf16_bits(v), alpha=alpha, beta=beta)
