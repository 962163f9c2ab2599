"""Shared helpers of the GPU parity tests: oracle weights from generator
output, device weights through the library, and the tolerance checks
(per output |y - y_ref| <= 1e-3 * sum|w||x| + 1e-6, propagated through the
fused epilogues)."""
import zlib

import numpy as np

import oracle

TOL_REL = 1e-3
TOL_ABS = 1e-6


def case_seed(*key):
    """A seed fixed by the test case's parameters (Python's str hash varies
    from process to process; this does not)."""
    return zlib.crc32(repr(key).encode()) & 0xFFFF


FMT_ID = {"q4_0": 0, "affine": 1, "q8_0": 2, "q4_k": 3, "q1": 4}
_SUPERBLOCK = {"q4_k": 256, "q1": 128}


def fmt_k(fmt, k):
    """A test shape's k for a format: Q4_K and Q1 rows are whole 256- and
    128-column superblocks, so their k is rounded up to one."""
    sb = _SUPERBLOCK.get(fmt, 32)
    return -(-k // sb) * sb


def host_weight(H):
    if hasattr(H, "blocks8"):
        return oracle.HostWeight.q8_0(H.blocks8, H.n, H.k)
    if hasattr(H, "blocks_k"):
        return oracle.HostWeight.q4_k(H.blocks_k, H.n, H.k)
    if hasattr(H, "blocks1"):
        return oracle.HostWeight.q1(H.blocks1, H.n, H.k)
    if hasattr(H, "blocks"):
        return oracle.HostWeight.q4_0(H.blocks, H.n, H.k)
    return oracle.HostWeight.affine(H.nib, H.s, H.m, H.n, H.k)


def dev_weight(H, device="cuda"):
    import bit_weight_quantized_q4_gb300 as q4
    if hasattr(H, "blocks8"):
        return q4.Q4Weight.from_q8_0(H.blocks8, H.n, H.k, device)
    if hasattr(H, "blocks_k"):
        return q4.Q4Weight.from_q4_k(H.blocks_k, H.n, H.k, device)
    if hasattr(H, "blocks1"):
        return q4.Q4Weight.from_q1(H.blocks1, H.n, H.k, device)
    if hasattr(H, "blocks"):
        return q4.Q4Weight.from_q4_0(H.blocks, H.n, H.k, device)
    return q4.Q4Weight.from_affine(H.nib, H.s, H.m, H.n, H.k, device)


def to_np(t):
    return t.detach().cpu().numpy().astype(np.float64)


def check(y, y_ref, S, extra=0.0, what=""):
    """Assert the plain tolerance; return the worst error / bound ratio."""
    y = np.asarray(y, dtype=np.float64)
    bound = TOL_REL * S + TOL_ABS + extra
    err = np.abs(y - y_ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d outputs out of tolerance; first %s: got %r want %r bound %r"
                             % (what, int(bad.sum()), tuple(i), y[tuple(i)], y_ref[tuple(i)], bound[tuple(i)]))
    return float(np.max(err / bound))


def check_residual(y, y_ref, S, what=""):
    return check(y, y_ref, S, extra=2.0 ** -23 * np.abs(y_ref), what=what)


def check_swiglu(h, g_ref, Sg, u_ref, Su, what=""):
    silu = g_ref / (1.0 + np.exp(-g_ref))
    h_ref = silu * u_ref
    bound = TOL_REL * (1.1 * np.abs(u_ref) * Sg + np.abs(silu) * Su) + TOL_ABS
    err = np.abs(np.asarray(h, np.float64) - h_ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d outputs out of tolerance; first %s: got %r want %r"
                             % (what, int(bad.sum()), tuple(i), h[tuple(i)], h_ref[tuple(i)]))
    return float(np.max(err / bound))


def check_argmax(idx, logits_ref, margin=1e-3, what=""):
    """The index is exact where the f64 top-1 beats the top-2 by more than
    `margin`; elsewhere its f64 logit must be within `margin` of the max."""
    idx = np.asarray(idx).ravel()
    for r in range(logits_ref.shape[0]):
        row = logits_ref[r]
        best = int(np.argmax(row))
        top2 = np.partition(row, -2)[-2] if row.size > 1 else -np.inf
        if row[best] - top2 > margin:
            assert idx[r] == best, "%s row %d: got %d want %d" % (what, r, idx[r], best)
        else:
            assert row[idx[r]] >= row[best] - margin, "%s row %d: index %d not within margin" % (what, r, idx[r])
