"""GPU parity of q4_gemm (the prefill GEMM: y = x W^T for wide activation
batches; crate inferencelayer, gemm_q4_src) against the f64 oracle, through
the C ABI: every weight format, batch widths in the 16-row activation tile
(1, 9, 16) and around and far above one 64-row (Q4_0: 128-row tensor-memory)
tile, ragged n and k, the accumulate form, scales over many binades, exact
zeros and run-to-run determinism."""
import numpy as np
import pytest

import oracle
import q4_workloads as wl
from parity import case_seed, check, check_residual, dev_weight, fmt_k, host_weight, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FMTS = ["q4_0", "affine", "q8_0", "q4_k", "q1"]


@pytest.fixture(scope="module")
def q4():
    import bit_weight_quantized_q4_gb300 as m
    m.build()
    m.lib()
    return m


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("nb", [1, 9, 16, 17, 64, 100, 257])
@pytest.mark.parametrize("n,k", [(33, 160), (64, 1024), (200, 544), (1000, 2048)])
def test_gemm_parity(q4, fmt, nb, n, k):
    k = fmt_k(fmt, k)
    rng = np.random.default_rng(case_seed("gemm", fmt, nb, n, k))
    H = wl._draw_fmt(fmt)(rng, n, k)
    x = wl.draw_x(rng, nb, k)
    y = q4.q4_gemm(dev_weight(H), torch.from_numpy(x).cuda())
    ref, S = oracle.q4_gemv(host_weight(H), x)
    check(to_np(y), ref, S, what="gemm %s nb=%d %dx%d" % (fmt, nb, n, k))


@pytest.mark.parametrize("fmt", ["q4_0", "affine", "q1"])
def test_gemm_accumulate(q4, fmt):
    rng = np.random.default_rng(case_seed("gemm-acc", fmt))
    n, k, nb = 300, fmt_k(fmt, 1024), 80
    H = wl._draw_fmt(fmt)(rng, n, k)
    x = wl.draw_x(rng, nb, k)
    r = wl.draw_x(rng, nb, n)
    y = torch.from_numpy(r.copy()).cuda()
    q4.q4_gemm(dev_weight(H), torch.from_numpy(x).cuda(), accumulate=True, out=y)
    ref, S = oracle.q4_res_gemv(host_weight(H), x, r)
    check_residual(to_np(y), ref, S, what="gemm accumulate " + fmt)


def test_gemm_workload_shape_and_determinism(q4):
    # the 14336 x 4096 projection over a 256-row prefill chunk: sampled rows
    # against the oracle, and the same bits twice
    rng = np.random.default_rng(77)
    H = wl.draw_q4_0(rng, 14336, 4096)
    W = dev_weight(H)
    x = wl.draw_x(rng, 256, 4096)
    xd = torch.from_numpy(x).cuda()
    y = q4.q4_gemm(W, xd)
    assert torch.equal(y, q4.q4_gemm(W, xd))
    rows = np.sort(rng.choice(14336, 40, replace=False))
    sub = wl.Q4_0Host(40, 4096, H.blocks[rows])
    ref, S = oracle.q4_gemv(host_weight(sub), x)
    check(to_np(y)[:, rows], ref, S, what="gemm 14336x4096 nb=256 (sampled rows)")


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
@pytest.mark.parametrize("nb", [17, 130, 257])
def test_gemm_scale_range(q4, fmt, nb):
    # Q4_0 and Q8_0 from 17 rows run on the tensor-memory form, whose operands
    # carry a power of two per weight row and per activation row: weight rows
    # whose block scales span 2^-14 .. 2^15 (2^-14 .. 2^11 for Q8_0, whose
    # weights reach 128 d; a few rows all zero), activation rows from 1e-12 to
    # 1e12, against the oracle at the plain tolerance
    rng = np.random.default_rng(80 + nb)
    n, k = 200, 1024
    top = 14 if fmt == "q4_0" else 10
    e = rng.integers(-13, top, (n, 1)) + rng.integers(-6, 1, (n, k // 32))
    d = (rng.uniform(1.0, 2.0, (n, k // 32)) * 2.0 ** e).astype(np.float16)
    d[rng.choice(n, 4, replace=False)] = 0
    if fmt == "q4_0":
        H = wl.Q4_0Host(n, k, wl.pack_q4_0(rng.integers(0, 16, (n, k), dtype=np.uint8), d.view(np.uint16)))
    else:
        H = wl.Q8_0Host(n, k, wl.pack_q8_0(rng.integers(-128, 128, (n, k), dtype=np.int16), d.view(np.uint16)))
    x = wl.draw_x(rng, nb, k) * (10.0 ** rng.integers(-12, 13, (nb, 1))).astype(np.float32)
    y = q4.q4_gemm(dev_weight(H), torch.from_numpy(x).cuda())
    ref, S = oracle.q4_gemv(host_weight(H), x)
    check(to_np(y), ref, S, what="gemm scale range %s nb=%d" % (fmt, nb))


def test_gemm_zero_weights_exact(q4):
    rng = np.random.default_rng(78)
    n, k, nb = 100, 512, 70
    d = rng.uniform(0.005, 0.02, (n, k // 32)).astype(np.float16).view(np.uint16)
    H = wl.Q4_0Host(n, k, wl.pack_q4_0(np.full((n, k), 8, np.uint8), d))
    y = q4.q4_gemm(dev_weight(H), torch.from_numpy(wl.draw_x(rng, nb, k)).cuda())
    assert torch.count_nonzero(y).item() == 0


def test_gemm_rejects(q4):
    rng = np.random.default_rng(79)
    W = dev_weight(wl.draw_q4_0(rng, 16, 64))
    L = q4.lib()
    x = torch.zeros((32, 64), device="cuda")
    y = torch.zeros((32, 16), device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert L.q4_gemm(W.cref(), x.data_ptr(), 32, y.data_ptr(), 0, ws.data_ptr(), ws.numel(), None) == 5
    assert L.q4_gemm(W.cref(), x.data_ptr(), 0, y.data_ptr(), 0, ws.data_ptr(), ws.numel(), None) == 2
    q4.q4_device_check()
