"""The kernels' bounded waits give up cleanly.

Every wait in the library's kernels is bounded.  Here each kind is made to
run out on purpose through the library's testing hook
(q4_debug_wait_limits): a grid barrier of the persistent decode step that
expects one arrival more than there are CTAs, and a weight-copy stage of a
per-call GEMV (and of the prefill GEMM and the decode attention) that
expects 16 bytes more than its copies bring.  None faults or hangs: the kernel records the failure, waits (bounded) for its
copies in flight and returns.  The check call then reports Q4_ERR_CUDA, and
the next normal call gives the same bits as before."""
import numpy as np
import pytest

import q4_workloads as wl
from parity import dev_weight

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def q4():
    import bit_weight_quantized_q4_gb300 as m
    m.build()
    m.lib()
    yield m
    m.q4_debug_wait_limits()     # defaults, whatever happened


def test_grid_barrier_gives_up_and_the_next_step_is_unchanged(q4):
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    cfg = wl.cfg4(seed=21, layers=2, hidden=256, kv=64, inter=384, vocab=500, nb=1)
    step = DecodeStep(cfg)
    step.run_fused()
    q4.q4_decode_check(step.step_ws)
    idx0, val0, hid0 = step.idx.clone(), step.val.clone(), step.hid.clone()
    q4.q4_debug_wait_limits(barrier_polls=256, barrier_extra=1)
    try:
        step.run_fused()
        with pytest.raises(q4.Q4Error) as e:
            q4.q4_decode_check(step.step_ws)
        assert e.value.status == 6
    finally:
        q4.q4_debug_wait_limits()
    step.run_fused()
    q4.q4_decode_check(step.step_ws)
    assert torch.equal(step.idx, idx0) and torch.equal(step.val, val0) and torch.equal(step.hid, hid0)


def test_copy_wait_gives_up_and_the_next_call_is_unchanged(q4):
    rng = np.random.default_rng(22)
    H = wl.draw_q4_0(rng, 300, 1024)
    W = dev_weight(H)
    x = torch.from_numpy(wl.draw_x(rng, 1, 1024)).cuda()
    y0 = q4.q4_gemv(W, x)
    q4.q4_device_check()
    q4.q4_debug_wait_limits(copy_wait_cycles=200000, copy_extra_bytes=16)
    try:
        q4.q4_gemv(W, x)
        with pytest.raises(q4.Q4Error) as e:
            q4.q4_device_check()          # reads and clears the flag
        assert e.value.status == 6
    finally:
        q4.q4_debug_wait_limits()
    y1 = q4.q4_gemv(W, x)
    q4.q4_device_check()
    assert torch.equal(y1, y0)


def test_attention_copy_wait_gives_up_and_the_next_call_is_unchanged(q4):
    rng = np.random.default_rng(23)
    H, Hkv, D, ms, pos = 32, 8, 64, 2048, 2047
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    q, kn, vn = T(rng.standard_normal((H, D))), T(rng.standard_normal((Hkv, D))), T(rng.standard_normal((Hkv, D)))
    kc, vc = T(rng.standard_normal((Hkv, ms, D))), T(rng.standard_normal((Hkv, ms, D)))
    ws = torch.zeros(int(q4.lib().q4_attn_workspace_bytes(H, D, ms)), dtype=torch.uint8, device="cuda")
    o0 = q4.q4_attn_decode(q, kn, vn, kc, vc, pos, workspace=ws)
    q4.q4_device_check()
    q4.q4_debug_wait_limits(copy_wait_cycles=200000, copy_extra_bytes=16)
    try:
        q4.q4_attn_decode(q, kn, vn, kc, vc, pos, workspace=ws)
        with pytest.raises(q4.Q4Error) as e:
            q4.q4_device_check()
        assert e.value.status == 6
    finally:
        q4.q4_debug_wait_limits()
    # the split counters are zero again and the result is the same
    assert torch.equal(q4.q4_attn_decode(q, kn, vn, kc, vc, pos, workspace=ws), o0)
    q4.q4_device_check()


# the 16-row and the 64-row activation tiles of the mma.sync form, and the
# tensor-memory form (Q4_0 and Q8_0 from 17 rows) at its three column-tile
# widths (128, 256, 512)
@pytest.mark.parametrize("fmt,nb", [("q4_0", 9), ("affine", 40), ("q4_0", 40), ("q4_0", 200), ("q4_0", 300),
                                    ("q8_0", 80)])
def test_gemm_copy_wait_gives_up_and_the_next_call_is_unchanged(q4, fmt, nb):
    rng = np.random.default_rng(24 + nb)
    H = wl._draw_fmt(fmt)(rng, 300, 1024)
    W = dev_weight(H)
    x = torch.from_numpy(wl.draw_x(rng, nb, 1024)).cuda()
    y0 = q4.q4_gemm(W, x)
    q4.q4_device_check()
    q4.q4_debug_wait_limits(copy_wait_cycles=200000, copy_extra_bytes=16)
    try:
        q4.q4_gemm(W, x)
        with pytest.raises(q4.Q4Error) as e:
            q4.q4_device_check()
        assert e.value.status == 6
    finally:
        q4.q4_debug_wait_limits()
    y1 = q4.q4_gemm(W, x)
    q4.q4_device_check()
    assert torch.equal(y1, y0)
