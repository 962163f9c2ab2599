"""GPU parity of every libq4gemv call against the f64 CPU oracle, on seeded
inputs at sizes spanning several tiles, chunks and ragged tails, plus the
method's degenerate cases and invariants.  Calls go through the C ABI (via
the ctypes binding)."""
import numpy as np
import pytest

import oracle
import q4_workloads as wl
from parity import (case_seed, check, check_argmax, check_residual, check_swiglu, dev_weight, fmt_k, host_weight,
                    to_np)

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


SHAPES = [(1, 32), (7, 96), (33, 160), (100, 544), (512, 2048), (1000, 4096), (48, 8192)]


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("nb", [1, 2, 3, 4, 5, 8, 9, 16])
@pytest.mark.parametrize("n,k", SHAPES)
def test_gemv(q4, fmt, nb, n, k):
    k = fmt_k(fmt, k)
    rng = np.random.default_rng(case_seed(fmt, nb, n, k))
    H = _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    y = q4.q4_gemv(dev_weight(H), torch.from_numpy(x).cuda())
    y_ref, S = oracle.q4_gemv(host_weight(H), x)
    check(to_np(y), y_ref, S, what="gemv %s nb=%d %dx%d" % (fmt, nb, n, k))


@pytest.mark.parametrize("nb", [1, 4, 16])
def test_affine_with_given_group_sums(q4, nb):
    rng = np.random.default_rng(31)
    n, k = 300, 1024
    H = wl.draw_affine(rng, n, k)
    x = torch.from_numpy(wl.draw_x(rng, nb, k)).cuda()
    W = dev_weight(H)
    gs = q4.q4_group_sums(x)
    ref_gs = x.cpu().numpy().reshape(nb, k // 32, 32).astype(np.float64).sum(-1)
    assert np.allclose(to_np(gs), ref_gs, rtol=1e-5, atol=1e-5)
    y1 = q4.q4_gemv(W, x, gsum=gs)
    y2 = q4.q4_gemv(W, x)
    assert torch.equal(y1, y2)      # in-kernel sums are added in the same order
    y_ref, S = oracle.q4_gemv(host_weight(H), x.cpu().numpy())
    check(to_np(y1), y_ref, S, what="affine given gsum")


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("nb", [1, 3, 16])
@pytest.mark.parametrize("n,k", [(64, 64), (2048, 2048), (37, 4096), (130, 8192)])
def test_nrm_gemv(q4, fmt, nb, n, k):
    k = fmt_k(fmt, k)
    rng = np.random.default_rng(case_seed("nrm", fmt, nb, n, k))
    H = _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    gamma = wl.draw_gamma(rng, k)
    y = q4.q4_nrm_gemv(dev_weight(H), torch.from_numpy(x).cuda(), torch.from_numpy(gamma).cuda(), 1e-6)
    y_ref, S = oracle.q4_nrm_gemv(host_weight(H), x, gamma, 1e-6)
    check(to_np(y), y_ref, S, what="nrm %s nb=%d %dx%d" % (fmt, nb, n, k))


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("na,nbr,k,nb", [(512, 512, 2048, 1), (40, 17, 96, 2), (2048, 512, 2048, 4)])
def test_dual(q4, fmt, norm, na, nbr, k, nb):
    k = fmt_k(fmt, k)
    rng = np.random.default_rng(case_seed("dual", fmt, norm, na, nbr, k, nb))
    Ha, Hb = _draw(fmt, rng, na, k), _draw(fmt, rng, nbr, k)
    x = wl.draw_x(rng, nb, k)
    gamma = wl.draw_gamma(rng, k) if norm else None
    ya, yb = q4.q4_dual_gemv(dev_weight(Ha), dev_weight(Hb), torch.from_numpy(x).cuda(),
                             None if gamma is None else torch.from_numpy(gamma).cuda(), 1e-6)
    ra, Sa, rb, Sb = oracle.q4_dual_gemv(host_weight(Ha), host_weight(Hb), x, gamma, 1e-6)
    check(to_np(ya), ra, Sa, what="dual a")
    check(to_np(yb), rb, Sb, what="dual b")


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("n,k,nb", [(8192, 2048, 1), (40, 96, 3), (1000, 1024, 8), (256, 512, 16)])
def test_gus_nrm(q4, fmt, n, k, nb):
    k = fmt_k(fmt, k)
    rng = np.random.default_rng(case_seed("gus", fmt, n, k, nb))
    Hg, Hu = _draw(fmt, rng, n, k), _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    gamma = wl.draw_gamma(rng, k)
    h = q4.q4_gus_nrm(dev_weight(Hg), dev_weight(Hu), torch.from_numpy(x).cuda(),
                      torch.from_numpy(gamma).cuda(), 1e-6)
    _, g, Sg, u, Su = oracle.q4_gus_nrm(host_weight(Hg), host_weight(Hu), x, gamma, 1e-6)
    check_swiglu(to_np(h), g, Sg, u, Su, what="gus %s %dx%d nb=%d" % (fmt, n, k, nb))


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("n,k,nb", [(2048, 8192, 1), (2048, 2048, 1), (33, 160, 5), (700, 1024, 16)])
@pytest.mark.parametrize("inplace", [False, True])
def test_res_gemv(q4, fmt, n, k, nb, inplace):
    k = fmt_k(fmt, k)
    rng = np.random.default_rng(case_seed("res", fmt, n, k, nb))
    H = _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    r = wl.draw_x(rng, nb, n)
    rd = torch.from_numpy(r).cuda()
    out = rd if inplace else None
    y = q4.q4_res_gemv(dev_weight(H), torch.from_numpy(x).cuda(), rd, out=out)
    if inplace:
        assert y.data_ptr() == rd.data_ptr()
    y_ref, S = oracle.q4_res_gemv(host_weight(H), x, r)
    check_residual(to_np(y), y_ref, S, what="res %s" % fmt)


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
@pytest.mark.parametrize("n,k,nb,norm", [(65536, 2048, 1, True), (1000, 256, 3, False), (77, 96, 16, True)])
def test_argmax(q4, fmt, n, k, nb, norm):
    k = fmt_k(fmt, k)
    rng = np.random.default_rng(case_seed("am", fmt, n, k, nb))
    H = _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    gamma = wl.draw_gamma(rng, k) if norm else None
    idx, val, logits = q4.q4_argmax(dev_weight(H), torch.from_numpy(x).cuda(),
                                    None if gamma is None else torch.from_numpy(gamma).cuda(), 1e-6,
                                    want_val=True, want_logits=True)
    idx_ref, lref, S = oracle.q4_argmax(host_weight(H), x, gamma, 1e-6)
    check(to_np(logits), lref, S, what="argmax logits")
    check_argmax(idx.cpu().numpy(), lref, what="argmax")
    # the index is exact against the device's own logits, ties to the lowest
    lg = logits.cpu().numpy()
    assert np.array_equal(idx.cpu().numpy(), np.argmax(lg, axis=1))
    assert np.array_equal(val.cpu().numpy(), lg.max(axis=1))


def test_argmax_planted_and_ties(q4):
    n, k = 5000, 64
    q = np.full((n, k), 8, np.uint8)
    q[3123, :] = 15                         # unique max for x = 1
    d = np.full((n, k // 32), 0x3C00, np.uint16)
    W = dev_weight(wl.Q4_0Host(n, k, wl.pack_q4_0(q, d)))
    x = torch.ones((2, k), device="cuda")
    x[1] = -1.0                             # row 1: every logit ties at 0 except row 3123 (-448)
    idx, val, _ = q4.q4_argmax(W, x, want_val=True)
    assert idx.cpu().tolist() == [3123, 0]
    assert val.cpu().tolist() == [7.0 * 64, 0.0]


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
def test_zero_weights_exact(q4, fmt):
    rng = np.random.default_rng(41)
    n, k = 200, 1024
    if fmt == "q4_0":
        d = rng.uniform(0.005, 0.02, (n, k // 32)).astype(np.float16).view(np.uint16)
        H = wl.Q4_0Host(n, k, wl.pack_q4_0(np.full((n, k), 8, np.uint8), d))
    elif fmt == "q8_0":
        d = rng.uniform(0.0003, 0.0012, (n, k // 32)).astype(np.float16).view(np.uint16)
        H = wl.Q8_0Host(n, k, wl.pack_q8_0(np.zeros((n, k), np.int16), d))
    elif fmt == "q1":
        # random signs, every scale zero
        z = np.zeros((n, k // 128), np.uint16)
        H = wl.Q1Host(n, k, wl.pack_q1(rng.integers(0, 2, (n, k), dtype=np.uint8), z))
    elif fmt == "q4_k":
        # nonzero nibbles, d and dmin; every sub-block scale and min zero
        d = rng.uniform(1e-4, 4e-4, (n, k // 256)).astype(np.float16).view(np.uint16)
        z = np.zeros((n, k // 32), int)
        H = wl.Q4_KHost(n, k, wl.pack_q4_k(rng.integers(1, 16, (n, k), dtype=np.uint8), z, z, d, d))
    else:
        z = np.zeros((n, k // 32), np.uint16)
        H = wl.AffineHost(n, k, rng.integers(0, 256, (n, k // 2), dtype=np.uint8), z, z)
    x = torch.from_numpy(wl.draw_x(rng, 4, k)).cuda()
    y = q4.q4_gemv(dev_weight(H), x)
    assert torch.count_nonzero(y).item() == 0
    r = torch.from_numpy(wl.draw_x(rng, 4, n)).cuda()
    yr = q4.q4_res_gemv(dev_weight(H), x, r)
    assert torch.equal(yr, r)


def test_power_of_two_scaling_bitwise(q4):
    rng = np.random.default_rng(42)
    n, k = 333, 2048
    H = wl.draw_q4_0(rng, n, k)
    b2 = H.blocks.copy()
    dd = (b2[:, :, 0].astype(np.uint16) | (b2[:, :, 1].astype(np.uint16) << 8)) + 0x0400
    b2[:, :, 0] = (dd & 0xFF).astype(np.uint8)
    b2[:, :, 1] = (dd >> 8).astype(np.uint8)
    x = torch.from_numpy(wl.draw_x(rng, 2, k)).cuda()
    y1 = q4.q4_gemv(dev_weight(H), x)
    y2 = q4.q4_gemv(dev_weight(wl.Q4_0Host(n, k, b2)), x)
    assert torch.equal(y2, 2.0 * y1)
    y4 = q4.q4_gemv(dev_weight(H), 4.0 * x)
    assert torch.equal(y4, 4.0 * y1)
    # Q8_0: d -> 2d doubles every output exactly too
    H8 = wl.draw_q8_0(rng, n, k)
    b8 = H8.blocks8.copy()
    dd = (b8[:, :, 0].astype(np.uint16) | (b8[:, :, 1].astype(np.uint16) << 8)) + 0x0400
    b8[:, :, 0] = (dd & 0xFF).astype(np.uint8)
    b8[:, :, 1] = (dd >> 8).astype(np.uint8)
    z1 = q4.q4_gemv(dev_weight(H8), x)
    assert torch.equal(q4.q4_gemv(dev_weight(wl.Q8_0Host(n, k, b8)), x), 2.0 * z1)
    # Q4_K: d -> 2d and dmin -> 2 dmin together
    HK = wl.draw_q4_k(rng, n, k)
    bk = HK.blocks_k.copy()
    for o in (0, 2):
        dd = (bk[:, :, o].astype(np.uint16) | (bk[:, :, o + 1].astype(np.uint16) << 8)) + 0x0400
        bk[:, :, o] = (dd & 0xFF).astype(np.uint8)
        bk[:, :, o + 1] = (dd >> 8).astype(np.uint8)
    k1 = q4.q4_gemv(dev_weight(HK), x)
    assert torch.equal(q4.q4_gemv(dev_weight(wl.Q4_KHost(n, k, bk)), x), 2.0 * k1)
    # Q1: d -> 2d
    H1 = wl.draw_q1(rng, n, k)
    b1 = H1.blocks1.copy()
    dd = (b1[:, :, 0].astype(np.uint16) | (b1[:, :, 1].astype(np.uint16) << 8)) + 0x0400
    b1[:, :, 0] = (dd & 0xFF).astype(np.uint8)
    b1[:, :, 1] = (dd >> 8).astype(np.uint8)
    o1 = q4.q4_gemv(dev_weight(H1), x)
    assert torch.equal(q4.q4_gemv(dev_weight(wl.Q1Host(n, k, b1)), x), 2.0 * o1)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q4_k", "q1"])
def test_one_hot_columns(q4, fmt):
    rng = np.random.default_rng(43)
    n, k = 96, 256
    H = _draw(fmt, rng, n, k)
    cols = [0, 5, 16, 31, 32, 130, 255]
    x = np.zeros((len(cols), k), np.float32)
    for r, c in enumerate(cols):
        x[r, c] = 1.0
    y = to_np(q4.q4_gemv(dev_weight(H), torch.from_numpy(x).cuda()))
    dense = oracle.dequant(host_weight(H))
    for r, c in enumerate(cols):
        assert np.array_equal(y[r], dense[:, c].astype(np.float32).astype(np.float64))


def test_rows_independent_and_deterministic(q4):
    rng = np.random.default_rng(44)
    n, k, nb = 1024, 2048, 4
    H = wl.draw_q4_0(rng, n, k)
    W = dev_weight(H)
    x = torch.from_numpy(wl.draw_x(rng, nb, k)).cuda()
    y = q4.q4_gemv(W, x)
    assert torch.equal(y, q4.q4_gemv(W, x))          # run to run
    same_plan = q4.plan(0, 64, 16, nb, False, torch.cuda.get_device_properties(0).multi_processor_count) == \
        q4.plan(0, 64, 16, 1, False, torch.cuda.get_device_properties(0).multi_processor_count)
    for r in range(nb):
        yr = q4.q4_gemv(W, x[r:r + 1].contiguous())
        if same_plan:
            assert torch.equal(yr[0], y[r])
        else:
            assert torch.allclose(yr[0], y[r], rtol=1e-5, atol=1e-5)


def test_nrm_constant_vector(q4):
    rng = np.random.default_rng(45)
    n, k, c, eps = 64, 512, 0.75, 1e-6
    H = wl.draw_q4_0(rng, n, k)
    gamma = wl.draw_gamma(rng, k)
    W = dev_weight(H)
    y = q4.q4_nrm_gemv(W, torch.full((1, k), c, device="cuda"), torch.from_numpy(gamma).cuda(), eps)
    ref, S = oracle.q4_gemv(host_weight(H), gamma.astype(np.float64) * (c / np.sqrt(c * c + eps)))
    check(to_np(y), ref, S, what="nrm constant")


@pytest.mark.parametrize("nb", [3, 5, 9])
@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q8_0", "q4_k", "q1"])
def test_large_dynamic_range(q4, fmt, nb):
    # activations far outside f16 range in both directions, and 32-column
    # blocks of very different magnitude inside one row, stay within
    # tolerance: each block carries its own power-of-two scale (hi + lo f16
    # parts for nb <= 4, one f16 for larger batches)
    rng = np.random.default_rng(case_seed("range", fmt, nb))
    n, k = 128, 1024
    H = _draw(fmt, rng, n, k)
    x = wl.draw_x(rng, nb, k)
    x[0] *= 1e6
    x[1] *= 1e-9
    x[2, ::7] *= 3e4
    for r in range(3, nb):
        x[r] *= np.repeat(10.0 ** rng.integers(-15, 16, size=k // 32), 32).astype(np.float32)
    y = q4.q4_gemv(dev_weight(H), torch.from_numpy(x).cuda())
    y_ref, S = oracle.q4_gemv(host_weight(H), x)
    check(to_np(y), y_ref, S, what="dynamic range %s nb=%d" % (fmt, nb))
    gamma = wl.draw_gamma(rng, k)
    y = q4.q4_nrm_gemv(dev_weight(H), torch.from_numpy(x).cuda(), torch.from_numpy(gamma).cuda(), 1e-6)
    y_ref, S = oracle.q4_nrm_gemv(host_weight(H), x, gamma, 1e-6)
    check(to_np(y), y_ref, S, what="dynamic range nrm %s nb=%d" % (fmt, nb))


def test_device_check_clear_after_calls(q4):
    # every kernel above finished its bounded weight-copy waits
    rng = np.random.default_rng(47)
    H = wl.draw_q4_0(rng, 4096, 2048)
    x = torch.from_numpy(wl.draw_x(rng, 2, 2048)).cuda()
    for _ in range(3):
        q4.q4_gemv(dev_weight(H), x)
    q4.q4_device_check()
