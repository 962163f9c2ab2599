"""GPU parity of every epilogue when the planner splits K over a thread-block
cluster of 2, 4 and 8 CTAs (each rank folds a slice of the group's tiles from
the partials the other ranks push into its shared memory): plain store,
RMSNorm (the slices' sums of squares exchanged), residual, SwiGLU over
gate/up pairs and the per-group argmax, for single-row, hi/lo-pair and
single-f16 batch classes.  Shapes are picked from the planner so that each
split is exercised; the check is the oracle's tolerance."""
import numpy as np
import pytest

import oracle
import q4_workloads as wl
from parity import (FMT_ID, case_seed, check, check_argmax, check_residual, check_swiglu, dev_weight, host_weight,
                    to_np)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CANDIDATES = [(n, k) for k in (2048, 4096, 8192, 16384) for n in (32, 48, 96, 160, 256, 512, 1024, 2048)]


@pytest.fixture(scope="module")
def q4():
    import bit_weight_quantized_q4_gb300 as m
    m.build()
    m.lib()
    return m


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _shape(q4, fmt, nb, S, pairs=False):
    """The smallest candidate (n, k) whose plan splits K over S ranks."""
    f = FMT_ID[fmt]
    for n, k in sorted(CANDIDATES, key=lambda s: s[0] * s[1]):
        tiles = 2 * ((n + 15) // 16) if pairs else (n + 15) // 16
        if q4.plan(f, tiles, (k + 127) // 128, nb, pairs, _sms())["S"] == S:
            return n, k
    pytest.skip("no candidate shape splits K over %d ranks for nb=%d" % (S, nb))


def _draw(fmt, rng, n, k):
    return wl._draw_fmt(fmt)(rng, n, k)


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("nb", [1, 4, 16])
@pytest.mark.parametrize("S", [2, 4, 8])
def test_split_store_and_norm(q4, fmt, nb, S):
    n, k = _shape(q4, fmt, nb, S)
    rng = np.random.default_rng(case_seed("split", fmt, nb, S))
    H = _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    gamma = wl.draw_gamma(rng, k)
    W = dev_weight(H)
    xd, gd = torch.from_numpy(x).cuda(), torch.from_numpy(gamma).cuda()
    y = q4.q4_gemv(W, xd)
    assert torch.equal(y, q4.q4_gemv(W, xd))  # the ranks' shares are added in a fixed order
    y_ref, Sr = oracle.q4_gemv(host_weight(H), x)
    check(to_np(y), y_ref, Sr, what="split gemv %s nb=%d S=%d %dx%d" % (fmt, nb, S, n, k))
    y = q4.q4_nrm_gemv(W, xd, gd, 1e-6)
    assert torch.equal(y, q4.q4_nrm_gemv(W, xd, gd, 1e-6))
    y_ref, Sr = oracle.q4_nrm_gemv(host_weight(H), x, gamma, 1e-6)
    check(to_np(y), y_ref, Sr, what="split nrm %s nb=%d S=%d %dx%d" % (fmt, nb, S, n, k))


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("nb", [1, 16])
@pytest.mark.parametrize("S", [2, 8])
def test_split_residual(q4, fmt, nb, S):
    n, k = _shape(q4, fmt, nb, S)
    rng = np.random.default_rng(case_seed("split-res", fmt, nb, S))
    H = _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    r = wl.draw_x(rng, nb, n)
    y = q4.q4_res_gemv(dev_weight(H), torch.from_numpy(x).cuda(), torch.from_numpy(r).cuda())
    y_ref, Sr = oracle.q4_res_gemv(host_weight(H), x, r)
    check_residual(to_np(y), y_ref, Sr, what="split res %s nb=%d S=%d" % (fmt, nb, S))


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("nb", [1, 8])
@pytest.mark.parametrize("S", [2, 4, 8])
def test_split_swiglu(q4, fmt, nb, S):
    n, k = _shape(q4, fmt, nb, S, pairs=True)
    rng = np.random.default_rng(case_seed("split-gus", fmt, nb, S))
    Hg, Hu = _draw(fmt, rng, n, k), _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    gamma = wl.draw_gamma(rng, k)
    h = q4.q4_gus_nrm(dev_weight(Hg), dev_weight(Hu), torch.from_numpy(x).cuda(),
                      torch.from_numpy(gamma).cuda(), 1e-6)
    _, g, Sg, u, Su = oracle.q4_gus_nrm(host_weight(Hg), host_weight(Hu), x, gamma, 1e-6)
    check_swiglu(to_np(h), g, Sg, u, Su, what="split gus %s nb=%d S=%d %dx%d" % (fmt, nb, S, n, k))


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("nb", [1, 3])
@pytest.mark.parametrize("S", [2, 8])
def test_split_argmax(q4, fmt, nb, S):
    n, k = _shape(q4, fmt, nb, S)
    rng = np.random.default_rng(case_seed("split-am", fmt, nb, S))
    H = _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    gamma = wl.draw_gamma(rng, k)
    idx, val, logits = q4.q4_argmax(dev_weight(H), torch.from_numpy(x).cuda(), torch.from_numpy(gamma).cuda(),
                                    1e-6, want_val=True, want_logits=True)
    idx_ref, lref, Sr = oracle.q4_argmax(host_weight(H), x, gamma, 1e-6)
    check(to_np(logits), lref, Sr, what="split argmax logits %s nb=%d S=%d" % (fmt, nb, S))
    check_argmax(idx.cpu().numpy(), lref, what="split argmax")
    lg = logits.cpu().numpy()
    assert np.array_equal(idx.cpu().numpy(), np.argmax(lg, axis=1))
    assert np.array_equal(val.cpu().numpy(), lg.max(axis=1))
