"""q4_argmax_noalloc: the argmax for callers that cannot allocate device
memory (for example a plug-in whose host application owns all GPU memory, or
a decode loop that must not call cudaMalloc while it runs).  It keeps its
pass-1 pairs in a fixed array inside the library instead of a caller
workspace.  Called through the C ABI, it must give the same results as
q4_argmax, call after call, and reject shapes its fixed array cannot hold.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import q4_workloads as wl
from parity import check, dev_weight, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def q4():
    import bit_weight_quantized_q4_gb300 as m
    m.build()
    m.lib()
    return m


def _noalloc_c(q4, W, x, gamma, eps, nb):
    """Call the C entry point directly (ctypes, no Python wrapper)."""
    idx = torch.full((nb,), -1, dtype=torch.int32, device="cuda")
    val = torch.empty(nb, dtype=torch.float32, device="cuda")
    logits = torch.empty((nb, W.n), dtype=torch.float32, device="cuda")
    st = q4.lib().q4_argmax_noalloc(
        W.cref(), ctypes.c_void_p(x.data_ptr()),
        None if gamma is None else ctypes.c_void_p(gamma.data_ptr()), ctypes.c_float(eps),
        ctypes.c_int32(nb), ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(val.data_ptr()),
        ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, q4.STATUS.get(st, st)
    return idx, val, logits


def test_noalloc_matches_workspace_argmax_twice(q4):
    rng = np.random.default_rng(77)
    cases = [(wl.draw_q4_0(rng, 65536, 2048), 1, True), (wl.draw_affine(rng, 3000, 512), 5, False)]
    for H, nb, norm in cases:                       # two calls in a row, different shapes
        W = dev_weight(H)
        x = torch.from_numpy(wl.draw_x(rng, nb, H.k)).cuda()
        gamma = torch.from_numpy(wl.draw_gamma(rng, H.k)).cuda() if norm else None
        i1, v1, l1 = _noalloc_c(q4, W, x, gamma, 1e-6, nb)
        i0, v0, l0 = q4.q4_argmax(W, x, gamma, 1e-6, want_val=True, want_logits=True)
        torch.cuda.synchronize()
        check(to_np(l1), to_np(l0), np.abs(to_np(l0)), what="noalloc logits")
        assert torch.equal(i1, i0)
        assert np.allclose(v1.cpu().numpy(), v0.cpu().numpy(), rtol=1e-3, atol=1e-6)


def test_noalloc_rejects_beyond_its_fixed_array(q4):
    # 2^22 rows of 32 at nb = 16 need more (max, index) pairs than the array
    # holds.  The buffers are real device memory (contents unused), so that a
    # call accepted by mistake would compute on them, never touch a bogus
    # address.
    n, k, nb = 1 << 22, 32, 16
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups = q4.plan(0, n // 16, 1, nb, False, sms)["groups"]
    assert groups * nb * 8 > 128 * 1024
    wbuf = torch.empty(q4.packed_bytes(0, n, k), dtype=torch.uint8, device="cuda")
    x = torch.zeros((nb, k), dtype=torch.float32, device="cuda")
    idx = torch.empty(nb, dtype=torch.int32, device="cuda")
    c = q4._CWeight(0, n, k, wbuf.data_ptr(), wbuf.numel())
    st = q4.lib().q4_argmax_noalloc(ctypes.byref(c), ctypes.c_void_p(x.data_ptr()), None, ctypes.c_float(0.0),
                                    ctypes.c_int32(nb), ctypes.c_void_p(idx.data_ptr()), None, None, None)
    torch.cuda.synchronize()
    assert st == 5        # Q4_ERR_WORKSPACE, nothing launched
