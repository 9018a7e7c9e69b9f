"""W12 tree-verify pass on GB300 (sm_103a): Python binding of ``libw12.so``.

A thin ctypes layer over the C ABI in ``include/w12.h``: it marshals torch
tensors (device memory) and numpy arrays (host memory) into the C structs and
calls the library.  Every step of the pass runs in the library's CUDA
kernels; if ``libw12.so`` is missing or cannot load, importing the functions
below raises -- there is no fallback.

Entry points (same names as the C ABI): ``w12_pack``, ``w12_unpack``,
``w12_load_check``, ``w12_gemm``, ``w12_lmhead_argmax``, ``w12_tree_build``,
``w12_tree_accept``, ``w12_verify_step``, the TLV calls (``w12_verify_step_q``,
``w12_tlv_chain``, ``w12_tlv_splice``), plus the workspace helpers.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw12.so")

W12_OK, W12_E_INVAL, W12_E_UNSUPPORTED, W12_E_MISMATCH, W12_E_CUDA, W12_E_TIMEOUT, W12_E_WORKSPACE = \
    0, -1, -2, -3, -4, -5, -6

TILE_N, TILE_K, REC_BYTES = 128, 64, 12288


class W12Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status == W12_E_CUDA:
            buf = C.create_string_buffer(96)
            code = lib().w12_debug_last_cuda_error(buf, 96)
            detail = f" [{buf.value.decode()} = {code}]"
        super().__init__(f"{what}: {status_str(status)} ({status}){detail}")


# ---------------------------------------------------------------------------
# C structs (mirror include/w12.h)
# ---------------------------------------------------------------------------

class Layout(C.Structure):
    _fields_ = [("n", C.c_int64), ("k", C.c_int64), ("n_tiles", C.c_int64), ("k_tiles", C.c_int64),
                ("n_escapes", C.c_int64), ("rec_bytes", C.c_size_t), ("base_bytes", C.c_size_t),
                ("esc_off_bytes", C.c_size_t), ("esc_bytes", C.c_size_t)]


class Weight(C.Structure):
    _fields_ = [("rec", C.c_void_p), ("base", C.c_void_p), ("esc_tile_off", C.c_void_p), ("esc", C.c_void_p),
                ("n", C.c_int64), ("k", C.c_int64), ("n_escapes", C.c_int64)]


class LatticeC(C.Structure):
    _fields_ = [("n_req", C.c_int32), ("p_max", C.c_int32), ("n_cand", C.c_int32), ("conditional", C.c_int32),
                ("p_r", C.c_void_p), ("root_tok", C.c_void_p), ("cand_tok", C.c_void_p), ("cand_logp", C.c_void_p)]


class TreeC(C.Structure):
    _fields_ = [("R", C.c_int32), ("parent", C.c_void_p), ("token", C.c_void_p), ("depth", C.c_void_p),
                ("req", C.c_void_p), ("score", C.c_void_p), ("rank", C.c_void_p), ("req_row_off", C.c_void_p)]


class StepC(C.Structure):
    _fields_ = [("n_linear", C.c_int32), ("lin", C.c_void_p), ("x", C.c_void_p), ("y", C.c_void_p),
                ("head", C.c_void_p), ("h", C.c_void_p), ("argmax", C.c_void_p)]


_lib = None


def lib():
    """Load libw12.so (raises if it is missing: no fallback path exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "speculative_decoding_tree_w12_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        p, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
        sigs = {
            "w12_status_str": ([C.c_int], C.c_char_p),
            "w12_abi_version": ([], C.c_int),
            "w12_pack_query": ([p, i64, i64, p], C.c_int),
            "w12_pack": ([p, i64, i64, p, p, p, p, p], C.c_int),
            "w12_workspace_bytes": ([i32, i64, i64, i32], sz),
            "w12_workspace_init": ([p, sz, p], C.c_int),
            "w12_status_fetch": ([p, p], C.c_int),
            "w12_unpack": ([p, p, p], C.c_int),
            "w12_load_check": ([p, p, p, p, sz, p], C.c_int),
            "w12_gemm": ([p, p, i32, p, p, sz, p], C.c_int),
            "w12_gemm_static_scratch": ([p, p, i32, p, p], C.c_int),
            "w12_lmhead_argmax": ([p, p, i32, p, p, p, sz, p], C.c_int),
            "w12_gemm_q": ([p, p, i32, p, p, sz, p], C.c_int),
            "w12_lmhead_argmax_q": ([p, p, i32, p, p, p, sz, p], C.c_int),
            "w12_head_cert_norms": ([p, p, p], C.c_int),
            "w12_cert_workspace_bytes": ([i32, i64], sz),
            "w12_lmhead_argmax_certified": ([p, p, p, i32, p, p, p, p, sz, p, sz, p], C.c_int),
            "w12_tree_build": ([p, i32, p, p, sz, p], C.c_int),
            "w12_tree_accept": ([p, i32, i32, p, p, p, p, p], C.c_int),
            "w12_verify_step": ([p, p, i32, i32, p, p, p, p, sz, p], C.c_int),
            "w12_verify_step_q": ([p, p, i32, i32, p, p, p, p, sz, p], C.c_int),
            "w12_tlv_chain": ([p, p, i32, i32, p, p], C.c_int),
            "w12_gdn_tree_verify": ([p, p, i32, i32, p, p, sz, p], C.c_int),
            "w12_gdn_commit": ([p, p, i32, p, p, p, sz, p], C.c_int),
            "w12_gdn_wy_verify": ([p, p, i32, p, p, p, sz, p], C.c_int),
            "w12_gdn_wy_commit": ([p, p, i32, p, p, p, p, sz, p], C.c_int),
            "w12_tlv_splice": ([p, p, p, p, i32, i32, p, p, p, p, sz, p], C.c_int),
            "w12_debug_set": ([i32, C.c_uint64], None),
            "w12_debug_num_sms": ([], i32),
            "w12_debug_profile": ([i32], None),
            "w12_debug_last_cuda_error": ([p, i32], i32),
            "w12_debug_profile_read": ([p, i32], i32),
            "w12_debug_chain_trace": ([p, sz], None),
            "w12_debug_chain_parts": ([i32], i32),
        }
        for name, (args, res) in sigs.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_str(s: int) -> str:
    return lib().w12_status_str(int(s)).decode()


def _check(s: int, what: str):
    if s != W12_OK:
        raise W12Error(s, what)


def _stream(stream=None):
    import torch
    st = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(st.cuda_stream)


def _dp(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _np(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------------------
# host packing
# ---------------------------------------------------------------------------

class HostPacked:
    """W12 buffers in host memory (numpy), as produced by ``w12_pack``."""

    def __init__(self, n, k, rec, base, esc_tile_off, esc):
        self.n, self.k = n, k
        self.rec, self.base, self.esc_tile_off, self.esc = rec, base, esc_tile_off, esc

    @property
    def n_escapes(self) -> int:
        return int(self.esc.shape[0])

    @property
    def nbytes(self) -> int:
        return self.rec.nbytes + self.base.nbytes + self.esc_tile_off.nbytes + self.esc.nbytes


def w12_pack(w_bf16_bits: np.ndarray) -> HostPacked:
    """Pack a host BF16 tensor (uint16 bits, [n][k]) into W12.  The library
    checks its own output bit for bit before returning."""
    w = np.ascontiguousarray(w_bf16_bits, dtype=np.uint16)
    n, k = w.shape
    L = Layout()
    _check(lib().w12_pack_query(_np(w), n, k, C.byref(L)), "w12_pack_query")
    rec = np.empty(L.rec_bytes, np.uint8)
    base = np.empty(L.base_bytes, np.uint8)
    off = np.empty(L.esc_off_bytes // 4, np.int32)
    esc = np.empty(L.esc_bytes // 4, np.uint32)
    _check(lib().w12_pack(_np(w), n, k, C.byref(L), _np(rec), _np(base), _np(off),
                          _np(esc) if esc.size else None), "w12_pack")
    return HostPacked(n, k, rec, base, off, esc)


# ---------------------------------------------------------------------------
# device tensors
# ---------------------------------------------------------------------------

class DeviceWeight:
    """A packed W12 tensor resident on the GPU (torch tensors) plus its C view."""

    def __init__(self, hp: HostPacked, device="cuda", rec=None):
        import torch
        self.n, self.k, self.n_escapes = hp.n, hp.k, hp.n_escapes
        self.rec = rec if rec is not None else torch.from_numpy(hp.rec).to(device)
        self.base = torch.from_numpy(hp.base).to(device)
        self.esc_tile_off = torch.from_numpy(hp.esc_tile_off).to(device)
        self.esc = torch.from_numpy(hp.esc.view(np.int32)).to(device) if hp.n_escapes else None
        self.c = Weight(self.rec.data_ptr(), self.base.data_ptr(), self.esc_tile_off.data_ptr(),
                        _dp(self.esc), self.n, self.k, self.n_escapes)

    @property
    def nbytes(self) -> int:
        b = self.rec.numel() + self.base.numel() + 4 * self.esc_tile_off.numel()
        return b + (4 * self.esc.numel() if self.esc is not None else 0)


class Workspace:
    """Zero-initialised device workspace sized for the given call shapes."""

    def __init__(self, R: int, max_n: int = 0, vocab: int = 0, n_req: int = 1, device="cuda"):
        import torch
        nbytes = int(lib().w12_workspace_bytes(int(R), int(max_n), int(vocab), int(n_req)))
        if nbytes == 0:
            raise W12Error(W12_E_UNSUPPORTED, "w12_workspace_bytes")
        self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.nbytes = nbytes
        _check(lib().w12_workspace_init(self.ptr, nbytes, _stream()), "w12_workspace_init")

    @property
    def ptr(self):
        return C.c_void_p(self.buf.data_ptr())

    def status(self, stream=None) -> int:
        return int(lib().w12_status_fetch(self.ptr, _stream(stream)))


def w12_unpack(w: DeviceWeight, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((w.n, w.k), dtype=torch.bfloat16, device=w.rec.device)
    _check(lib().w12_unpack(C.byref(w.c), C.c_void_p(out.data_ptr()), _stream(stream)), "w12_unpack")
    return out


def w12_load_check(w: DeviceWeight, src_bf16, ws: Workspace, stream=None) -> int:
    """Bit-exact device check against the source tensor; returns the number of
    differing weights (0 = identical).  Synchronises the stream."""
    mism = C.c_int64(0)
    s = lib().w12_load_check(C.byref(w.c), C.c_void_p(src_bf16.data_ptr()), C.byref(mism), ws.ptr, ws.nbytes,
                             _stream(stream))
    if s not in (W12_OK, W12_E_MISMATCH):
        raise W12Error(s, "w12_load_check")
    return int(mism.value)


def w12_gemm(w: DeviceWeight, x, ws: Workspace, y=None, stream=None, quick: bool = False):
    """``y = x . W^T`` (x: bf16 [R][k] on the device) -> bf16 [R][n].
    ``quick``: the quick pass (``w12_gemm_q``, view planes only)."""
    import torch
    R = x.shape[0]
    if y is None:
        y = torch.empty((R, w.n), dtype=torch.bfloat16, device=x.device)
    fn, name = (lib().w12_gemm_q, "w12_gemm_q") if quick else (lib().w12_gemm, "w12_gemm")
    _check(fn(C.byref(w.c), C.c_void_p(x.data_ptr()), R, C.c_void_p(y.data_ptr()), ws.ptr, ws.nbytes,
              _stream(stream)), name)
    return y


def w12_lmhead_argmax(head: DeviceWeight, h, ws: Workspace, argmax=None, maxlogit=None, stream=None,
                      quick: bool = False):
    """Argmax over ``h . W_head^T`` per row -> int32 [R].  ``quick``: the quick
    pass (``w12_lmhead_argmax_q``, view planes only)."""
    import torch
    R = h.shape[0]
    if argmax is None:
        argmax = torch.empty(R, dtype=torch.int32, device=h.device)
    fn, name = (lib().w12_lmhead_argmax_q, "w12_lmhead_argmax_q") if quick else \
        (lib().w12_lmhead_argmax, "w12_lmhead_argmax")
    _check(fn(C.byref(head.c), C.c_void_p(h.data_ptr()), R, C.c_void_p(argmax.data_ptr()),
              C.c_void_p(_dp(maxlogit)) if maxlogit is not None else None, ws.ptr, ws.nbytes,
              _stream(stream)), name)
    return argmax


def w12_head_cert_norms(head: DeviceWeight, out=None, stream=None):
    """Per token: ||w_v - w^_v|| and ||w^_v|| (w^: quick weights) -> float32
    [2][n] on the device (load time, for the certified head)."""
    import torch
    if out is None:
        out = torch.empty((2, head.n), dtype=torch.float32, device="cuda")
    _check(lib().w12_head_cert_norms(C.byref(head.c), C.c_void_p(out.data_ptr()), _stream(stream)),
           "w12_head_cert_norms")
    return out


class CertWorkspace:
    """Device buffer for the certified head's quick logits and survivor lists."""

    def __init__(self, R: int, vocab: int, device="cuda"):
        import torch
        self.nbytes = int(lib().w12_cert_workspace_bytes(int(R), int(vocab)))
        if self.nbytes == 0:
            raise W12Error(W12_E_INVAL, "w12_cert_workspace_bytes")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)

    @property
    def ptr(self):
        return C.c_void_p(self.buf.data_ptr())


def w12_lmhead_argmax_certified(head: DeviceWeight, norms, h, ws: Workspace, cws: CertWorkspace, argmax=None,
                                maxlogit=None, survivors=None, stream=None):
    """Certified argmax over ``h . W_head^T`` per row -> int32 [R]: quick-pass
    logits, per-row Cauchy-Schwarz bound, exact FP64 rescoring of the
    survivors.  ``survivors`` (int32 [R], optional) gets the survivor counts."""
    import torch
    R = h.shape[0]
    if argmax is None:
        argmax = torch.empty(R, dtype=torch.int32, device=h.device)
    _check(lib().w12_lmhead_argmax_certified(C.byref(head.c), C.c_void_p(norms.data_ptr()), C.c_void_p(h.data_ptr()),
                                             R, C.c_void_p(argmax.data_ptr()),
                                             C.c_void_p(_dp(maxlogit)) if maxlogit is not None else None,
                                             C.c_void_p(_dp(survivors)) if survivors is not None else None,
                                             ws.ptr, ws.nbytes, cws.ptr, cws.nbytes, _stream(stream)),
           "w12_lmhead_argmax_certified")
    return argmax


class DeviceLattice:
    def __init__(self, lat, device="cuda"):
        import torch
        self.n_req, self.p_max, self.n_cand = int(lat.n_req), int(lat.p_max), int(lat.n_cand)
        self.conditional = int(bool(lat.conditional))
        self.p_r = np.ascontiguousarray(lat.p_r, np.int32)        # host memory by contract
        self.root_tok = torch.from_numpy(np.ascontiguousarray(lat.root_tok, np.int32)).to(device)
        self.cand_tok = torch.from_numpy(np.ascontiguousarray(lat.cand_tok, np.int32)).to(device)
        self.cand_logp = torch.from_numpy(np.ascontiguousarray(lat.cand_logp, np.float32)).to(device)
        self.c = LatticeC(self.n_req, self.p_max, self.n_cand, self.conditional, _np(self.p_r).value,
                          self.root_tok.data_ptr(), self.cand_tok.data_ptr(), self.cand_logp.data_ptr())


class DeviceTree:
    def __init__(self, budget: int, n_req: int, device="cuda"):
        import torch
        z = lambda dt, n: torch.zeros(n, dtype=dt, device=device)
        self.parent, self.token, self.req = z(torch.int32, budget), z(torch.int32, budget), z(torch.int32, budget)
        self.depth, self.rank = z(torch.uint8, budget), z(torch.uint8, budget)
        self.score = z(torch.float32, budget)
        self.req_row_off = z(torch.int32, n_req + 1)
        self.c = TreeC(0, *(t.data_ptr() for t in (self.parent, self.token, self.depth, self.req, self.score,
                                                    self.rank, self.req_row_off)))

    @property
    def R(self) -> int:
        return int(self.c.R)

    def host(self):
        R = self.R
        return dict(parent=self.parent[:R].cpu().numpy(), token=self.token[:R].cpu().numpy(),
                    depth=self.depth[:R].cpu().numpy(), req=self.req[:R].cpu().numpy(),
                    score=self.score[:R].cpu().numpy(), rank=self.rank[:R].cpu().numpy(),
                    req_row_off=self.req_row_off.cpu().numpy())


def w12_tree_build(lat: DeviceLattice, budget: int, ws: Workspace, tree: Optional[DeviceTree] = None,
                   stream=None) -> DeviceTree:
    if tree is None:
        tree = DeviceTree(budget, lat.n_req, device=lat.root_tok.device)
    _check(lib().w12_tree_build(C.byref(lat.c), int(budget), C.byref(tree.c), ws.ptr, ws.nbytes, _stream(stream)),
           "w12_tree_build")
    return tree


def w12_tree_accept(tree: DeviceTree, n_req: int, p_max: int, argmax, acc_tok=None, acc_len=None, acc_node=None,
                    stream=None):
    import torch
    dev = argmax.device
    acc_tok = acc_tok if acc_tok is not None else torch.empty((n_req, p_max + 1), dtype=torch.int32, device=dev)
    acc_len = acc_len if acc_len is not None else torch.empty(n_req, dtype=torch.int32, device=dev)
    acc_node = acc_node if acc_node is not None else torch.empty(n_req, dtype=torch.int32, device=dev)
    _check(lib().w12_tree_accept(C.byref(tree.c), n_req, p_max, C.c_void_p(argmax.data_ptr()),
                                 C.c_void_p(acc_tok.data_ptr()), C.c_void_p(acc_len.data_ptr()),
                                 C.c_void_p(acc_node.data_ptr()), _stream(stream)), "w12_tree_accept")
    return acc_tok, acc_len, acc_node


class VerifyStep:
    """Marshalled arguments of ``w12_verify_step`` (kept alive between calls so
    the call can be captured in a CUDA graph and replayed)."""

    def __init__(self, linears: Sequence[DeviceWeight], xs, ys, head: DeviceWeight, h, argmax):
        self.linears, self.xs, self.ys, self.head, self.h, self.argmax = list(linears), list(xs), list(ys), head, h, argmax
        n = len(self.linears)
        self._lin = (Weight * max(n, 1))(*[w.c for w in self.linears])
        self._x = (C.c_void_p * max(n, 1))(*[x.data_ptr() for x in self.xs])
        self._y = (C.c_void_p * max(n, 1))(*[y.data_ptr() for y in self.ys])
        self.c = StepC(n, C.cast(self._lin, C.c_void_p), C.cast(self._x, C.c_void_p), C.cast(self._y, C.c_void_p),
                       C.cast(C.pointer(head.c), C.c_void_p), h.data_ptr(), argmax.data_ptr())


def w12_verify_step(step: VerifyStep, tree: DeviceTree, n_req: int, p_max: int, ws: Workspace, acc_tok, acc_len,
                    acc_node=None, stream=None):
    _check(lib().w12_verify_step(C.byref(step.c), C.byref(tree.c), n_req, p_max, C.c_void_p(acc_tok.data_ptr()),
                                 C.c_void_p(acc_len.data_ptr()), C.c_void_p(_dp(acc_node)) if acc_node is not None
                                 else None, ws.ptr, ws.nbytes, _stream(stream)), "w12_verify_step")


def w12_verify_step_q(step: VerifyStep, tree: DeviceTree, n_req: int, p_max: int, ws: Workspace, acc_tok,
                      acc_len, acc_node=None, stream=None):
    """The TLV Q pass: ``w12_verify_step`` on the quick weights; its
    acceptance outputs are the commit chain."""
    _check(lib().w12_verify_step_q(C.byref(step.c), C.byref(tree.c), n_req, p_max, C.c_void_p(acc_tok.data_ptr()),
                                   C.c_void_p(acc_len.data_ptr()), C.c_void_p(_dp(acc_node)) if acc_node is not None
                                   else None, ws.ptr, ws.nbytes, _stream(stream)), "w12_verify_step_q")


def w12_tlv_chain(c_len_host, t1_row_off_host, budget: int):
    """Host call: chain tokens committed per request and the subtree budget."""
    c_len = np.ascontiguousarray(c_len_host, np.int32)
    off = np.ascontiguousarray(t1_row_off_host, np.int32)
    n_req = len(c_len)
    if len(off) != n_req + 1:
        raise ValueError("t1_row_off needs n_req + 1 entries")
    m = np.empty(n_req, np.int32)
    sub = C.c_int32(0)
    _check(lib().w12_tlv_chain(_np(c_len), _np(off), n_req, int(budget), _np(m), C.byref(sub)), "w12_tlv_chain")
    return m, int(sub.value)


def w12_tlv_splice(t1: DeviceTree, c_tok, c_len, c_node, m_host, t2: DeviceTree, ws: Workspace,
                   out: Optional[DeviceTree] = None, stream=None) -> DeviceTree:
    """The combined tree of one TLV cycle (device)."""
    m = np.ascontiguousarray(m_host, np.int32)
    n_req = len(m)
    p1_max = int(c_tok.shape[1]) - 1
    if out is None:
        out = DeviceTree(max(1, int(m.sum()) + t2.R), n_req, device=c_tok.device)
    _check(lib().w12_tlv_splice(C.byref(t1.c), C.c_void_p(c_tok.data_ptr()), C.c_void_p(c_len.data_ptr()),
                                C.c_void_p(c_node.data_ptr()), n_req, p1_max, _np(m), C.byref(t2.c),
                                C.byref(out.c), ws.ptr, ws.nbytes, _stream(stream)), "w12_tlv_splice")
    return out


class GdnLayerC(C.Structure):
    _fields_ = [("n_heads", C.c_int32), ("head_dim", C.c_int32), ("S0", C.c_void_p), ("q", C.c_void_p),
                ("k", C.c_void_p), ("v", C.c_void_p), ("alpha", C.c_void_p), ("beta", C.c_void_p)]


W12_GDN_WY, W12_GDN_PATH = 0, 1


class GdnLayer:
    """Device inputs of one recurrent layer over a tree: committed states
    S0 (float32 [n_req][H][d][d]), q/k/v (bfloat16 [R][H][d]), alpha/beta
    (float32 [R][H]); kept alive with the marshalled struct."""

    def __init__(self, S0, q, k, v, alpha, beta):
        self.S0, self.q, self.k, self.v, self.alpha, self.beta = S0, q, k, v, alpha, beta
        self.H, self.d = int(q.shape[1]), int(q.shape[2])
        self.c = GdnLayerC(self.H, self.d, S0.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                           alpha.data_ptr(), beta.data_ptr())


def w12_gdn_tree_verify(layer: GdnLayer, tree: DeviceTree, n_req: int, ws: Workspace, method: int = W12_GDN_WY,
                        out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((tree.R, layer.H, layer.d), dtype=torch.float32, device=layer.q.device)
    _check(lib().w12_gdn_tree_verify(C.byref(layer.c), C.byref(tree.c), int(n_req), int(method),
                                     C.c_void_p(out.data_ptr()), ws.ptr, ws.nbytes, _stream(stream)),
           "w12_gdn_tree_verify")
    return out


def w12_gdn_commit(layer: GdnLayer, tree: DeviceTree, n_req: int, acc_node, ws: Workspace, state=None, stream=None):
    import torch
    if state is None:
        state = torch.empty_like(layer.S0)
    _check(lib().w12_gdn_commit(C.byref(layer.c), C.byref(tree.c), int(n_req), C.c_void_p(acc_node.data_ptr()),
                                C.c_void_p(state.data_ptr()), ws.ptr, ws.nbytes, _stream(stream)), "w12_gdn_commit")
    return state


def w12_gdn_wy_verify(layer: GdnLayer, tree: DeviceTree, n_req: int, ws: Workspace, out=None, u=None, stream=None):
    """WY-form outputs and the WY vectors u (both float32 [R][H][d])."""
    import torch
    if out is None:
        out = torch.empty((tree.R, layer.H, layer.d), dtype=torch.float32, device=layer.q.device)
    if u is None:
        u = torch.empty((tree.R, layer.H, layer.d), dtype=torch.float32, device=layer.q.device)
    _check(lib().w12_gdn_wy_verify(C.byref(layer.c), C.byref(tree.c), int(n_req), C.c_void_p(out.data_ptr()),
                                   C.c_void_p(u.data_ptr()), ws.ptr, ws.nbytes, _stream(stream)), "w12_gdn_wy_verify")
    return out, u


def w12_gdn_wy_commit(layer: GdnLayer, tree: DeviceTree, n_req: int, acc_node, u, ws: Workspace, state=None,
                      stream=None):
    """The committed states from the WY vectors u of w12_gdn_wy_verify."""
    import torch
    if state is None:
        state = torch.empty_like(layer.S0)
    _check(lib().w12_gdn_wy_commit(C.byref(layer.c), C.byref(tree.c), int(n_req), C.c_void_p(acc_node.data_ptr()),
                                   C.c_void_p(u.data_ptr()), C.c_void_p(state.data_ptr()), ws.ptr, ws.nbytes,
                                   _stream(stream)), "w12_gdn_wy_commit")
    return state


def debug_set(flags: int = 0, timeout_ns: int = 0):
    lib().w12_debug_set(int(flags), int(timeout_ns))


def profile(enable: bool):
    lib().w12_debug_profile(1 if enable else 0)


def profile_read(max_launches: int = 1024) -> List[float]:
    buf = (C.c_float * max_launches)()
    n = int(lib().w12_debug_profile_read(buf, max_launches))
    if n < 0:
        raise W12Error(n, "w12_debug_profile_read")
    return [float(buf[i]) for i in range(min(n, max_launches))]


def num_sms() -> int:
    return int(lib().w12_debug_num_sms())


class ChainTrace:
    """Per-GEMM end times inside the verify step's GEMM chain (debug hook):
    while enabled, each chain launch stamps the global timer per CTA at its
    start and when the CTA has written its last output of each GEMM."""

    def __init__(self, n_gemms: int, device="cuda"):
        import torch
        self.n = int(n_gemms)
        self.parts = int(lib().w12_debug_chain_parts(self.n))
        self.S = num_sms()
        self.buf = torch.zeros(((self.n + self.parts) * self.S,), dtype=torch.int64, device=device)

    def __enter__(self):
        lib().w12_debug_chain_trace(C.c_void_p(self.buf.data_ptr()), self.buf.numel())
        return self

    def __exit__(self, *exc):
        lib().w12_debug_chain_trace(None, 0)

    def gemm_us(self) -> List[float]:
        """Per GEMM: the time from the previous GEMM's end (for each launch's
        first GEMM, from the launch's first CTA start) to the last CTA's stamp."""
        t = self.buf.view(self.n + self.parts, self.S).cpu().numpy().astype(np.float64)
        out, j0 = [], 0
        for k in range(self.parts):
            m = (self.n - j0) // (self.parts - k)
            rows = t[j0 + k: j0 + k + m]
            start = t[j0 + k + m]
            starts = start[start > 0]
            prev = starts.min() if starts.size else rows[0].max()
            for r in rows:
                end = r.max()
                out.append((end - prev) / 1e3)
                prev = end
            j0 += m
        return out
