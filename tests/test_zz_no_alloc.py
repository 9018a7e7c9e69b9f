"""The allocation-free GEMM entry point (w12_gemm_static_scratch), called
through the C ABI, against the workspace entry point (w12_gemm) and the
FP64 oracle.

This entry point exists for callers that cannot allocate device memory
where they run the GEMM (plugin hosts that give kernels no allocations of
their own, processes that must keep a fixed device footprint): its scratch
lives in a device array inside the library.  It runs the same kernel with
the same split points as w12_gemm, so two calls in a row must both give
w12_gemm's output bit for bit (which also shows that each call clears the
shared counters it uses), and both must match the oracle within the GEMM
tolerance."""
from __future__ import annotations

import ctypes as C

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


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("n,k,R", [(1024, 512, 8), (2048, 1536, 16), (640, 5120, 3)])
def test_static_scratch_gemm_matches_workspace_gemm(w12, n, k, R):
    w = synth.weights(n, k, 17 + R, 3, 0.005, 0.005)
    x = synth.activations(R, k, 17 + R, 4)
    dw = w12.DeviceWeight(w12.w12_pack(w))
    xd = _dev(x)
    ws = w12.Workspace(R, n)
    ref = w12.w12_gemm(dw, xd, ws)
    torch.cuda.synchronize()
    ref_bits = ref.view(torch.int16).cpu().numpy()
    exact = oracle.gemm_f64(x, w)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        y = torch.full((R, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        s = w12.lib().w12_gemm_static_scratch(C.byref(dw.c), C.c_void_p(xd.data_ptr()), R,
                                              C.c_void_p(y.data_ptr()), stream)
        assert s == w12.W12_OK, (call, w12.status_str(s))
        torch.cuda.synchronize()
        assert np.array_equal(y.view(torch.int16).cpu().numpy(), ref_bits), call
        got = y.float().cpu().numpy().astype(np.float64)
        assert H.gemm_rel_err(got, exact) <= H.GEMM_REL_TOL, call


def test_static_scratch_gemm_refuses_sizes_beyond_its_limit(w12):
    w = synth.weights(256, 128, 1, 1)
    dw = w12.DeviceWeight(w12.w12_pack(w))
    x = _dev(synth.activations(17, 128, 1, 2))
    y = torch.empty((17, 256), dtype=torch.bfloat16, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert w12.lib().w12_gemm_static_scratch(C.byref(dw.c), C.c_void_p(x.data_ptr()), 17,
                                             C.c_void_p(y.data_ptr()), stream) == w12.W12_E_UNSUPPORTED
