"""GPU parity of q4_attn_decode (decode attention of one token: RoPE, KV
append, GQA, sliding window; honeycrisp/mod.rs, gpu_attention and the fused
RoPE + KV-append + SDPA dispatch) against the f64 oracle, through the C ABI.

Cache rows past the token hold NaN, so any read of them shows in the output;
every other row must come back untouched, the appended v bitwise.  Shapes
span one and many sequence chunks, every supported head grouping and both
head sizes."""
import numpy as np
import pytest

import oracle
from parity import case_seed, check, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def q4():
    import bit_weight_quantized_q4_gb300 as m
    m.build()
    m.lib()
    return m


def _case(rng, H, Hkv, D, max_seq, position):
    q = rng.standard_normal((H, D)).astype(np.float32)
    kn = rng.standard_normal((Hkv, D)).astype(np.float32)
    vn = rng.standard_normal((Hkv, D)).astype(np.float32)
    kc = rng.standard_normal((Hkv, max_seq, D)).astype(np.float32)
    vc = rng.standard_normal((Hkv, max_seq, D)).astype(np.float32)
    kc[:, position:] = np.nan
    vc[:, position:] = np.nan
    return q, kn, vn, kc, vc


def _run(q4, H, Hkv, D, max_seq, position, window, rope, seed):
    rng = np.random.default_rng(seed)
    q, kn, vn, kc, vc = _case(rng, H, Hkv, D, max_seq, position)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kcd, vcd = T(kc), T(vc)
    scale = 1.0 / np.sqrt(D)
    tables = None
    cos64 = sin64 = None
    if rope:
        c, s = q4.rope_table(max_seq, D, 10000.0)
        tables = (T(c), T(s))
        cos64, sin64 = oracle.rope_table(max_seq, D, 10000.0)
    out = q4.q4_attn_decode(T(q), T(kn), T(vn), kcd, vcd, position, window, scale, rope=tables)
    ref, bound, kc2, vc2 = oracle.attn_decode(q, kn, vn, kc, vc, position, window, scale, cos64, sin64)
    what = "attn H=%d Hkv=%d D=%d pos=%d win=%d rope=%s" % (H, Hkv, D, position, window, rope)
    check(to_np(out), ref, bound, what=what)
    assert torch.isfinite(out).all(), what
    # the cache: row `position` appended (v bitwise), everything else untouched
    kg, vg = kcd.cpu().numpy(), vcd.cpu().numpy()
    assert np.array_equal(vg[:, position], vn), what
    kref = kc2[:, position]
    assert np.all(np.abs(kg[:, position] - kref) <= 1e-6 * (1 + np.abs(kref))), what
    others = np.ones(max_seq, bool)
    others[position] = False
    assert np.array_equal(kg[:, others], kc[:, others], equal_nan=True), what
    assert np.array_equal(vg[:, others], vc[:, others], equal_nan=True), what
    return out


# (H, Hkv, D): every supported grouping for both head sizes
GEOMS = [(32, 8, 64), (8, 8, 64), (6, 3, 64), (16, 1, 64), (16, 4, 128), (8, 1, 128), (4, 4, 128), (4, 2, 128)]


@pytest.mark.parametrize("H,Hkv,D", GEOMS)
@pytest.mark.parametrize("position,window", [(0, 0), (7, 0), (300, 0), (2999, 0), (2999, 100), (2999, 1)])
def test_attn_parity(q4, H, Hkv, D, position, window):
    _run(q4, H, Hkv, D, 3000, position, window, False, case_seed("attn", H, Hkv, D, position, window))


@pytest.mark.parametrize("H,Hkv,D", [(32, 8, 64), (16, 4, 128), (16, 1, 64)])
@pytest.mark.parametrize("position,window", [(0, 0), (513, 0), (8191, 0), (8191, 4000)])
def test_attn_parity_rope(q4, H, Hkv, D, position, window):
    _run(q4, H, Hkv, D, 8192, position, window, True, case_seed("attn-rope", H, Hkv, D, position, window))


def test_attn_first_token_is_v(q4):
    # one attended position: every head's output is its group's new v, bitwise
    out = _run(q4, 8, 2, 64, 16, 0, 0, True, 7)
    rng = np.random.default_rng(7)
    _, _, vn, _, _ = _case(rng, 8, 2, 64, 16, 0)
    assert np.array_equal(out.cpu().numpy(), np.repeat(vn, 4, axis=0))


def test_attn_deterministic_and_window_larger_than_context(q4):
    rng = np.random.default_rng(8)
    H, Hkv, D, ms, pos = 32, 8, 64, 4096, 4095
    q, kn, vn, kc, vc = _case(rng, H, Hkv, D, ms, pos)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    args = (T(q), T(kn), T(vn), T(kc), T(vc), pos)
    a = q4.q4_attn_decode(*args, window=0)
    b = q4.q4_attn_decode(*args, window=0)
    c = q4.q4_attn_decode(*args, window=100000)
    assert torch.equal(a, b) and torch.equal(a, c)


def test_attn_rejects(q4):
    T = lambda *s: torch.zeros(s, dtype=torch.float32, device="cuda")
    with pytest.raises(q4.Q4Error) as e:   # 3 query heads per kv head
        q4.q4_attn_decode(T(9, 64), T(3, 64), T(3, 64), T(3, 32, 64), T(3, 32, 64), 4)
    assert e.value.status == 4
    with pytest.raises(q4.Q4Error) as e:   # head size 96
        q4.q4_attn_decode(T(4, 96), T(4, 96), T(4, 96), T(4, 32, 96), T(4, 32, 96), 4)
    assert e.value.status == 4
    with pytest.raises(q4.Q4Error) as e:   # position past the cache
        q4.q4_attn_decode(T(4, 64), T(4, 64), T(4, 64), T(4, 32, 64), T(4, 32, 64), 32)
    assert e.value.status == 2
    # a workspace too small for the chunks this call needs
    L = q4.lib()
    kc = T(8, 4096, 64)
    out = T(32, 64)
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    st = L.q4_attn_decode(T(32, 64).data_ptr(), T(8, 64).data_ptr(), T(8, 64).data_ptr(), kc.data_ptr(),
                          T(8, 4096, 64).data_ptr(), 4096, 4095, 32, 8, 64, 0, 0.125, None, None, out.data_ptr(),
                          ws.data_ptr(), ws.numel(), None)
    assert st == 5
    assert q4.lib().q4_device_check(None) == 0
