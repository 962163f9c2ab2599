"""HalfSet activations (Module gpu, Struct HalfSet: f16 even/odd streams plus
per-32 group sums, the input format of the multi-row Q4 matvecs), through the
C ABI: q4_pack_half must round like numpy's float16 and sum groups like
q4_group_sums; q4_gemv_half must match the f64 oracle on the decoded f16 rows
at every batch class, and give the same bits as q4_gemv on the same f16
values widened to fp32."""
import numpy as np
import pytest

import oracle
import q4_workloads as wl
from parity import case_seed, check, dev_weight, fmt_k, host_weight, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def q4():
    import bit_weight_quantized_q4_gb300 as m
    m.build()
    m.lib()
    return m


def _draw(fmt, rng, n, k):
    return wl._draw_fmt(fmt)(rng, n, k)


@pytest.mark.parametrize("nb,k", [(1, 32), (3, 544), (16, 4096)])
def test_pack_rounds_and_sums(q4, nb, k):
    rng = np.random.default_rng(case_seed("pack", nb, k))
    x = wl.draw_x(rng, nb, k) * 3.0
    xd = torch.from_numpy(x).cuda()
    xe, xo, gs = q4.q4_pack_half(xd)
    x16 = x.astype(np.float16)
    assert np.array_equal(xe.cpu().numpy().view(np.uint16), x16[:, 0::2].view(np.uint16))
    assert np.array_equal(xo.cpu().numpy().view(np.uint16), x16[:, 1::2].view(np.uint16))
    ref = q4.q4_group_sums(torch.from_numpy(x16.astype(np.float32)).cuda())
    assert torch.equal(gs, ref)


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("nb", [1, 3, 5, 9, 16])
@pytest.mark.parametrize("n,k", [(33, 160), (700, 1024), (64, 8192)])
def test_gemv_half_parity(q4, fmt, nb, n, k):
    k = fmt_k(fmt, k)
    rng = np.random.default_rng(case_seed("half", fmt, nb, n, k))
    H = _draw(fmt, rng, n, k)
    x16 = wl.draw_x(rng, nb, k).astype(np.float16)
    xe = torch.from_numpy(np.ascontiguousarray(x16[:, 0::2])).cuda()
    xo = torch.from_numpy(np.ascontiguousarray(x16[:, 1::2])).cuda()
    W = dev_weight(H)
    y = q4.q4_gemv_half(W, xe, xo)
    ref, S = oracle.q4_gemv_half(host_weight(H), x16[:, 0::2].view(np.uint16), x16[:, 1::2].view(np.uint16))
    check(to_np(y), ref, S, what="gemv_half %s nb=%d %dx%d" % (fmt, nb, n, k))
    # the same bits as the fp32 path on the same values, with or without
    # the caller's group sums
    y32 = q4.q4_gemv(W, torch.from_numpy(x16.astype(np.float32)).cuda())
    assert torch.equal(y, y32)
    _, _, gs = q4.q4_pack_half(torch.from_numpy(x16.astype(np.float32)).cuda())
    assert torch.equal(q4.q4_gemv_half(W, xe, xo, gsum=gs), y32)


def test_gemv_half_workload_shape(q4):
    # the affine 14336 x 4096 matvec at the speculative-verify width
    c = wl.cfg3()
    x = c.x[:16]
    W = dev_weight(c.W)
    xe, xo, gs = q4.q4_pack_half(torch.from_numpy(x).cuda())
    y = q4.q4_gemv_half(W, xe, xo, gsum=gs)
    ref, S = oracle.q4_gemv_half(host_weight(c.W), xe.cpu().numpy().view(np.uint16),
                                 xo.cpu().numpy().view(np.uint16))
    check(to_np(y), ref, S, what="gemv_half 14336x4096 nb=16")


def test_gemv_half_rejects_bad_streams(q4):
    rng = np.random.default_rng(5)
    H = wl.draw_q4_0(rng, 16, 64)
    W = dev_weight(H)
    good = torch.zeros((2, 32), dtype=torch.float16, device="cuda")
    with pytest.raises(TypeError):
        q4.q4_gemv_half(W, good.float(), good)
    with pytest.raises(ValueError):
        q4.q4_gemv_half(W, good[:, :16].contiguous(), good)
