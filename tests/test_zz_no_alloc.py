"""q4_argmax_noalloc: the argmax for callers that cannot allocate device
memory (for example a plug-in whose host application owns all GPU memory, or
a decode loop that must not call cudaMalloc while it runs).  It keeps its
pass-1 pairs in a fixed array inside the library instead of a caller
workspace.  Called through the C ABI, it must give the same bits as
q4_argmax (both run the same kernels) and match the f64 oracle, call after
call, at a size that fills most of the fixed array, and reject shapes the
array cannot hold.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import oracle
import q4_workloads as wl
from parity import check, check_argmax, dev_weight, host_weight, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SCRATCH_BYTES = 128 * 1024     # the library's fixed array


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


def _same_as_workspace_call_and_oracle(q4, H, x, gamma, eps, what):
    nb = x.shape[0]
    W = dev_weight(H)
    i1, v1, l1 = _noalloc_c(q4, W, x, gamma, eps, nb)
    i0, v0, l0 = q4.q4_argmax(W, x, gamma, eps, want_val=True, want_logits=True)
    torch.cuda.synchronize()
    # the same kernels on the same inputs: the same bits
    assert torch.equal(i1, i0) and torch.equal(v1, v0) and torch.equal(l1, l0), what
    # and the oracle's logits and argmax
    g = None if gamma is None else gamma.cpu().numpy()
    _, lref, S = oracle.q4_argmax(host_weight(H), x.cpu().numpy(), g, eps)
    check(to_np(l1), lref, S, what=what + " logits")
    check_argmax(i1.cpu().numpy(), lref, what=what + " argmax")
    rows = np.arange(nb)
    assert np.all(to_np(v1) == to_np(l1)[rows, i1.cpu().numpy()]), what + " value of the argmax"


def test_noalloc_matches_workspace_argmax_and_oracle_twice(q4):
    rng = np.random.default_rng(77)
    cases = [(wl.draw_q4_0(rng, 65536, 2048), 1, True), (wl.draw_affine(rng, 3000, 512), 5, False)]
    for H, nb, norm in cases:                       # two calls in a row, different shapes
        x = torch.from_numpy(wl.draw_x(rng, nb, H.k)).cuda()
        gamma = torch.from_numpy(wl.draw_gamma(rng, H.k)).cuda() if norm else None
        _same_as_workspace_call_and_oracle(q4, H, x, gamma, 1e-6, "noalloc %dx%d nb=%d" % (H.n, H.k, nb))


def test_noalloc_near_its_capacity(q4):
    # 2183168 x 32 at nb = 15 plans 1064 groups: 15960 (max, index) pairs,
    # 127680 of the array's 131072 bytes
    n, k, nb = 2183168, 32, 15
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups = q4.plan(0, n // 16, 1, nb, False, sms)["groups"]
    used = ((groups * nb * 4 + 15) // 16) * 16 + groups * nb * 4
    assert used <= SCRATCH_BYTES
    rng = np.random.default_rng(78)
    H = wl.draw_q4_0(rng, n, k)
    x = torch.from_numpy(wl.draw_x(rng, nb, k)).cuda()
    for _ in range(2):
        _same_as_workspace_call_and_oracle(q4, H, x, None, 0.0, "noalloc %d pairs" % (groups * nb))


def test_noalloc_rejects_beyond_its_fixed_array(q4):
    # 2^22 rows of 32 at nb = 16 need more (max, index) pairs than the array
    # holds.  The buffers are real device memory (contents unused), so that a
    # call accepted by mistake would compute on them, never touch a bogus
    # address.
    n, k, nb = 1 << 22, 32, 16
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups = q4.plan(0, n // 16, 1, nb, False, sms)["groups"]
    assert groups * nb * 8 > SCRATCH_BYTES
    wbuf = torch.empty(q4.packed_bytes(0, n, k), dtype=torch.uint8, device="cuda")
    x = torch.zeros((nb, k), dtype=torch.float32, device="cuda")
    idx = torch.empty(nb, dtype=torch.int32, device="cuda")
    c = q4._CWeight(0, n, k, wbuf.data_ptr(), wbuf.numel())
    st = q4.lib().q4_argmax_noalloc(ctypes.byref(c), ctypes.c_void_p(x.data_ptr()), None, ctypes.c_float(0.0),
                                    ctypes.c_int32(nb), ctypes.c_void_p(idx.data_ptr()), None, None, None)
    torch.cuda.synchronize()
    assert st == 5        # Q4_ERR_WORKSPACE, nothing launched
