"""Host-side tests of libq4gemv that need no GPU: the library loads and
exports every function its header declares, the repack is lossless, the
launch planner keeps its invariants, and invalid arguments are rejected
before anything is launched."""
import ctypes

import numpy as np
import pytest

import bit_weight_quantized_q4_gb300 as q4
import q4_workloads as wl


@pytest.fixture(scope="module", autouse=True)
def built():
    q4.build()


def test_exports_every_declared_symbol():
    L = q4.lib()
    names = q4.header_functions()
    assert len(names) >= 16
    for n in names:
        assert hasattr(L, n), n


def test_status_strings():
    L = q4.lib()
    for s in range(7):
        assert L.q4_status_str(s).decode().startswith(q4.STATUS[s])


@pytest.mark.parametrize("n,k", [(1, 32), (16, 128), (17, 96), (33, 160), (100, 544), (64, 1024)])
def test_repack_roundtrip_random(n, k):
    rng = np.random.default_rng(n * 1000 + k)
    H = wl.draw_q4_0(rng, n, k)
    P = q4.repack_q4_0(H.blocks, n, k)
    assert P.size == q4.packed_bytes(0, n, k)
    assert np.array_equal(q4.unpack_q4_0(P, n, k), H.blocks)
    A = wl.draw_affine(rng, n, k)
    P = q4.repack_affine(A.nib, A.s, A.m, n, k)
    nib, s, m = q4.unpack_affine(P, n, k)
    assert np.array_equal(nib, A.nib) and np.array_equal(s, A.s) and np.array_equal(m, A.m)
    Q = wl.draw_q8_0(rng, n, k)
    P = q4.repack_q8_0(Q.blocks8, n, k)
    assert P.size == q4.packed_bytes(2, n, k)
    assert np.array_equal(q4.unpack_q8_0(P, n, k), Q.blocks8)


def test_q8_0_layout_bytes():
    # the device record of a 16 x 128 Q8_0 tile holds exactly the 2048 biased
    # weight bytes (q + 128) and the 64 fp16 scales: nothing else, no padding
    rng = np.random.default_rng(11)
    Q = wl.draw_q8_0(rng, 16, 128)
    P = q4.repack_q8_0(Q.blocks8, 16, 128)
    assert P.size == 2176 == q4.weight_bytes(2, 16, 128)
    assert np.array_equal(np.sort(P[:2048]), np.sort((Q.blocks8[:, :, 2:] ^ 0x80).ravel()))
    assert np.array_equal(np.sort(P[2048:].view(np.uint16)), np.sort(Q.blocks8[:, :, :2].copy().view(np.uint16).ravel()))


@pytest.mark.parametrize("n,k", [(1, 256), (16, 256), (17, 512), (33, 768), (100, 1024)])
def test_repack_roundtrip_q4_k(n, k):
    rng = np.random.default_rng(n * 7 + k)
    H = wl.draw_q4_k(rng, n, k)
    P = q4.repack_q4_k(H.blocks_k, n, k)
    assert P.size == q4.packed_bytes(3, n, k)
    assert np.array_equal(q4.unpack_q4_k(P, n, k), H.blocks_k)


@pytest.mark.parametrize("n,k", [(1, 128), (16, 128), (17, 384), (33, 1024), (100, 256)])
def test_repack_roundtrip_q1(n, k):
    rng = np.random.default_rng(n * 11 + k)
    H = wl.draw_q1(rng, n, k)
    P = q4.repack_q1(H.blocks1, n, k)
    assert P.size == q4.packed_bytes(4, n, k) == -(-n // 16) * (k // 128) * 288
    assert np.array_equal(q4.unpack_q1(P, n, k), H.blocks1)


def test_q1_layout_bytes():
    # a 16 x 128 tile is one 288-byte record: the 2048 sign bits, each
    # inverted (a set stored bit is -d), then the 16 rows' fp16 d
    rng = np.random.default_rng(13)
    H = wl.draw_q1(rng, 16, 128)
    P = q4.repack_q1(H.blocks1, 16, 128)
    assert P.size == 288 and q4.weight_bytes(4, 16, 128) == 16 * 18
    signs = np.unpackbits(H.blocks1[:, 0, 2:], axis=1, bitorder="little")
    stored = np.unpackbits(P[:256], bitorder="little")
    assert int(stored.sum()) == int((1 - signs).sum())   # the same bits, inverted
    d = P[256:288].view(np.uint16).reshape(8, 2)
    dh = H.blocks1[:, 0, 0:2].copy().view(np.uint16)[:, 0]
    assert np.array_equal(d[:, 0], dh[:8]) and np.array_equal(d[:, 1], dh[8:])


def test_q4_k_layout_bytes():
    # one 16 x 256 superblock row-set is two 1216-byte records; each holds the
    # 1024 nibble bytes of its half, one byte word per (row pair, block) with
    # the 6-bit scale and min, and the rows' fp16 d and dmin
    rng = np.random.default_rng(12)
    H = wl.draw_q4_k(rng, 16, 256)
    P = q4.repack_q4_k(H.blocks_k, 16, 256)
    assert P.size == 2 * 1216 and q4.weight_bytes(3, 16, 256) == 16 * 144
    b = H.blocks_k[:, 0, :]
    for c in range(2):
        r = P[c * 1216:(c + 1) * 1216]
        d = r[1152:1184].view(np.uint16).reshape(8, 2)
        dm = r[1184:1216].view(np.uint16).reshape(8, 2)
        assert np.array_equal(d[:, 0], b[0:8, 0:2].copy().view(np.uint16)[:, 0])
        assert np.array_equal(d[:, 1], b[8:16, 0:2].copy().view(np.uint16)[:, 0])
        assert np.array_equal(dm[:, 0], b[0:8, 2:4].copy().view(np.uint16)[:, 0])
        w = r[1024:1152].reshape(8, 4, 4)            # [g][block][sc_g, mn_g, sc_g8, mn_g8]
        assert w.max() < 64
        for g in range(8):
            for j in range(4):
                sc, mn = oracle_free_q4k_field(b[g, 4:16], 4 * c + j)
                assert (w[g, j, 0], w[g, j, 1]) == (sc, mn)


def oracle_free_q4k_field(scale_bytes, j):
    # the generator's bit-position table read backwards
    vals = []
    for f in range(2):
        v = 0
        for bit in range(6):
            byte, pos = wl.Q4K_SCALE_BITS[f, j, bit]
            v |= ((int(scale_bytes[byte]) >> int(pos)) & 1) << bit
        vals.append(v)
    return tuple(vals)


def test_repack_roundtrip_edge_values():
    # scales: +-0, smallest subnormal, largest finite, inf; every nibble value
    n, k = 5, 64
    q = np.tile(np.arange(16, dtype=np.uint8), (n, k // 16))
    d = np.array([[0x0000, 0x8000], [0x0001, 0x7BFF], [0xFBFF, 0x7C00], [0x3C00, 0xBC00], [0x0400, 0x03FF]],
                 dtype=np.uint16)
    blocks = wl.pack_q4_0(q, d)
    P = q4.repack_q4_0(blocks, n, k)
    assert np.array_equal(q4.unpack_q4_0(P, n, k), blocks)


def test_packed_sizes_and_padding():
    # full tiles and chunks: the packed size is the algorithmic size plus
    # nothing for Q4_0 payload+scales (1152 B per 16x128 = 18 B per 32 weights)
    assert q4.packed_bytes(0, 14336, 4096) == q4.weight_bytes(0, 14336, 4096) == 33030144
    assert q4.packed_bytes(1, 14336, 4096) == q4.weight_bytes(1, 14336, 4096) == 36700160
    assert q4.weight_bytes(0, 1, 32) == 18 and q4.weight_bytes(1, 1, 32) == 20
    assert q4.packed_bytes(0, 1, 32) == 1152       # one padded tile chunk
    assert q4.packed_bytes(0, 0, 32) == 0 and q4.packed_bytes(0, 4, 33) == 0
    assert q4.packed_bytes(2, 14336, 4096) == q4.weight_bytes(2, 14336, 4096) == 14336 * 128 * 34
    assert q4.weight_bytes(2, 1, 32) == 34 and q4.packed_bytes(2, 1, 32) == 2176
    assert q4.packed_bytes(3, 4, 32) == 0 and q4.packed_bytes(3, 4, 128) == 0   # Q4_K: whole superblocks
    assert q4.packed_bytes(3, 14336, 4096) == 896 * 32 * 1216
    assert q4.weight_bytes(3, 14336, 4096) == 14336 * 16 * 144
    assert q4.packed_bytes(4, 4, 64) == 0 and q4.packed_bytes(4, 4, 256) == 2 * 288   # Q1: whole 128-superblocks
    assert q4.weight_bytes(4, 14336, 4096) == 14336 * 32 * 18
    assert q4.packed_bytes(5, 4, 256) == 0


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("tiles,chunks,pairs", [(896, 32, False), (1024, 16, True), (128, 16, False),
                                                (64, 16, False), (4096, 16, False), (1, 1, False),
                                                (2, 1, True), (7, 3, False), (128, 64, False)])
@pytest.mark.parametrize("nb", [1, 3, 8, 16])
def test_plan_invariants(fmt, tiles, chunks, pairs, nb):
    sms = 152
    p = q4.plan(fmt, tiles, chunks, nb, pairs, sms)
    # work is handed out in tile pairs, or single tiles when pairs would
    # leave CTAs idle (never for gate/up jobs)
    upt = 2 if pairs or (tiles + 1) // 2 >= max(1, sms // p["S"]) else 1
    units = -(-tiles // upt)
    assert 1 <= p["S"] <= 8 and (p["S"] & (p["S"] - 1)) == 0
    assert p["S"] * p["Cs"] >= chunks and p["Cs"] >= 1
    assert (p["S"] - 1) * p["Cs"] < chunks         # no empty K-slice
    assert 1 <= p["groups"] <= units
    # balanced contiguous ranges of units: the busiest group holds TG tiles
    assert p["TG"] == min(upt * -(-units // p["groups"]), tiles)
    assert p["groups"] * p["TG"] >= tiles
    assert p["ctas"] == p["groups"] * p["S"]
    # one wave of CTAs (one per SM) unless the partial sums of a one-wave
    # plan would not fit shared memory (large nb x many tiles)
    if nb <= 4:
        assert p["ctas"] <= sms
    assert p["ctas"] <= 8 * sms
    assert p["smem"] <= 227 * 1024
    if pairs:
        assert p["TG"] % 2 == 0
    # the activation slice fits the staging budget: f16 hi + lo parts (4 bytes
    # a value) for nb <= 4, the f16 value alone (2 bytes) for larger batches
    bytes_per_value = 4 if nb <= 4 else 2
    assert bytes_per_value * nb * p["Cs"] * 128 <= 64 * 1024 or p["S"] == 8


def test_plan_rejects_bad_arguments():
    with pytest.raises(q4.Q4Error):
        q4.plan(0, 0, 1, 1, False, 152)
    with pytest.raises(q4.Q4Error):
        q4.plan(0, 3, 1, 1, True, 152)    # pairs need an even tile count
    with pytest.raises(q4.Q4Error):
        q4.plan(0, 8, 1, 17, False, 152)
    with pytest.raises(q4.Q4Error):
        q4.plan(5, 8, 1, 1, False, 152)


def _cw(fmt=0, n=16, k=64, dev=0x1000, nbytes=None):
    if nbytes is None:
        nbytes = q4.packed_bytes(fmt, n, k)
    return q4._CWeight(fmt, n, k, dev, nbytes)


A = 0x10000    # a 16-byte aligned fake device address: never dereferenced, since
               # every case below fails validation before any CUDA call


@pytest.mark.parametrize("case,expect", [
    ("null_weight", 1), ("null_x", 1), ("null_y", 1), ("bad_fmt", 4), ("bad_k", 2), ("bad_n", 2),
    ("small_bytes", 2), ("misaligned_w", 3), ("misaligned_x", 3), ("nb0", 4), ("nb17", 4),
])
def test_gemv_validation(case, expect):
    L = q4.lib()
    W = _cw()
    x, y, nb = A, A + 4096, 1
    if case == "null_weight":
        W.dev = None
    elif case == "null_x":
        x = None
    elif case == "null_y":
        y = None
    elif case == "bad_fmt":
        W.fmt = 7
    elif case == "bad_k":
        W.k = 48
    elif case == "bad_n":
        W.n = 0
    elif case == "small_bytes":
        W.bytes = 100
    elif case == "misaligned_w":
        W.dev = A + 8
    elif case == "misaligned_x":
        x = A + 4
    elif case == "nb0":
        nb = 0
    elif case == "nb17":
        nb = 17
    assert L.q4_gemv(ctypes.byref(W), x, None, nb, y, None) == expect


def test_fused_validation():
    L = q4.lib()
    Wa, Wb = _cw(0, 16, 64), _cw(1, 16, 64)
    # mixed formats
    assert L.q4_dual_gemv(ctypes.byref(Wa), ctypes.byref(Wb), A, None, 0.0, 1, A, A, None) == 4
    assert L.q4_gus_nrm(ctypes.byref(Wa), ctypes.byref(Wb), A, A, 1e-6, 1, A, None) == 4
    # mismatched k / n
    Wc = _cw(0, 16, 96)
    assert L.q4_dual_gemv(ctypes.byref(Wa), ctypes.byref(Wc), A, None, 0.0, 1, A, A, None) == 2
    Wd = _cw(0, 32, 64)
    assert L.q4_gus_nrm(ctypes.byref(Wa), ctypes.byref(Wd), A, A, 1e-6, 1, A, None) == 2
    # gamma is required by nrm and gus
    assert L.q4_nrm_gemv(ctypes.byref(Wa), A, None, 1e-6, 1, A, None) == 1
    assert L.q4_gus_nrm(ctypes.byref(Wa), ctypes.byref(Wa), A, None, 1e-6, 1, A, None) == 1
    # residual pointer required
    assert L.q4_res_gemv(ctypes.byref(Wa), A, None, 1, A, None) == 1
    # argmax: workspace missing / too small / misaligned, idx missing
    ws = q4.q4_argmax_workspace_bytes(16, 1)
    assert ws > 0
    assert L.q4_argmax(ctypes.byref(Wa), A, None, 0.0, 1, A, None, None, None, ws, None) == 5
    assert L.q4_argmax(ctypes.byref(Wa), A, None, 0.0, 1, A, None, None, A, ws - 1, None) == 5
    assert L.q4_argmax(ctypes.byref(Wa), A, None, 0.0, 1, A, None, None, A + 4, ws, None) == 3
    assert L.q4_argmax(ctypes.byref(Wa), A, None, 0.0, 1, None, None, None, A, ws, None) == 1
    # group sums
    assert L.q4_group_sums(A, 1, 48, A, None) == 2
    assert L.q4_group_sums(None, 1, 64, A, None) == 1


def test_q4_k_rejects_partial_superblocks():
    L = q4.lib()
    buf = np.zeros(1 << 16, np.uint8)
    assert L.q4_repack_q4_k(buf.ctypes.data, 16, 128, buf.ctypes.data, buf.size) == 2
    assert L.q4_repack_q4_k(None, 16, 256, buf.ctypes.data, buf.size) == 1
    # a Q4_K weight view whose k is not whole superblocks fails before launch
    W = _cw(3, 16, 128, nbytes=1 << 20)
    assert L.q4_gemv(ctypes.byref(W), A, None, 1, A + 4096, None) == 2
    with pytest.raises(ValueError):
        q4.repack_q4_k(np.zeros((16, 1, 144), np.uint8), 16, 128)


def test_q1_rejects_partial_superblocks():
    L = q4.lib()
    buf = np.zeros(1 << 16, np.uint8)
    assert L.q4_repack_q1(buf.ctypes.data, 16, 96, buf.ctypes.data, buf.size) == 2
    W = _cw(4, 16, 96, nbytes=1 << 20)
    assert L.q4_gemv(ctypes.byref(W), A, None, 1, A + 4096, None) == 2


def test_rope_table_host():
    import oracle
    c, s = q4.rope_table(300, 64, 10000.0)
    co, so = oracle.rope_table(300, 64, 10000.0)
    assert np.abs(c - co).max() <= 6e-8 and np.abs(s - so).max() <= 6e-8
    L = q4.lib()
    buf = np.zeros(64, np.float32)
    assert L.q4_rope_table(4, 7, 10000.0, buf.ctypes.data, buf.ctypes.data) == 2
    assert L.q4_rope_table(4, 8, 0.0, buf.ctypes.data, buf.ctypes.data) == 2
    assert L.q4_rope_table(4, 8, 10000.0, None, buf.ctypes.data) == 1


def test_attn_workspace_bytes():
    L = q4.lib()
    assert L.q4_attn_workspace_bytes(32, 64, 4096) == 128 + 256 * 32 * 66 * 4
    assert L.q4_attn_workspace_bytes(32, 96, 4096) == 0 and L.q4_attn_workspace_bytes(0, 64, 16) == 0


@pytest.mark.parametrize("case,expect", [("ok_shape_g3", 4), ("d96", 4), ("pos_past", 2), ("neg_window", 2),
                                         ("null_q", 1), ("one_table", 1), ("misaligned_q", 3)])
def test_attn_validation(case, expect):
    # every case fails before any CUDA call (fake 16-byte aligned addresses)
    L = q4.lib()
    H, Hkv, D, ms, pos, win = 32, 8, 64, 128, 5, 0
    q, cs, sn = A, A, A
    if case == "ok_shape_g3":
        H, Hkv = 9, 3
    elif case == "d96":
        D = 96
    elif case == "pos_past":
        pos = ms
    elif case == "neg_window":
        win = -1
    elif case == "null_q":
        q = None
    elif case == "one_table":
        sn = None
    elif case == "misaligned_q":
        q = A + 4
    st = L.q4_attn_decode(q, A, A, A, A, ms, pos, H, Hkv, D, win, 0.125, cs, sn, A, A, 1 << 20, None)
    assert st == expect


def test_step_attn_workspace_bytes():
    L = q4.lib()
    assert L.q4_decode_attn_workspace_bytes(32, 8, 64) == 80 + 8 * 1024 + (1024 // 8) * 32 * 66 * 4
    assert L.q4_decode_attn_workspace_bytes(8, 2, 64) == 80 + 8 * 1024 + 512 * 8 * 66 * 4
    assert L.q4_decode_attn_workspace_bytes(4, 2, 64) == 0      # two query heads per kv head
    assert L.q4_decode_attn_workspace_bytes(16, 4, 128) == 0    # head size 128
    assert L.q4_decode_attn_workspace_bytes(68, 17, 64) == 0    # more than 16 kv heads


@pytest.mark.parametrize("case,expect", [("null_att", 1), ("g2", 4), ("d128", 4), ("width", 2), ("pos_past", 2),
                                         ("neg_window", 2), ("null_caches", 1), ("misaligned_cache", 3),
                                         ("one_table", 1), ("misaligned_out", 3), ("ws_small", 5),
                                         ("too_many_layers", 4)])
def test_step_attn_validation(case, expect):
    # every case fails before any CUDA call (fake 16-byte aligned addresses)
    L = q4.lib()
    hidden, kv, inter, nl = 512, 128, 256, 2
    heads, kv_heads, D, ms, pos, win = 8, 2, 64, 128, 100, 0
    caches = [A, A]
    cos, sin, out = A, A, A

    def layer():
        return q4._CDecodeLayer(_cw(0, hidden, hidden), _cw(0, kv, hidden), _cw(0, kv, hidden),
                                _cw(0, hidden, hidden), _cw(0, inter, hidden), _cw(0, inter, hidden),
                                _cw(0, hidden, inter), A, A, None)
    if case == "g2":
        heads, kv_heads = 4, 2
    elif case == "d128":
        D = 128
    elif case == "width":
        heads, kv_heads = 16, 4
    elif case == "pos_past":
        pos = ms
    elif case == "neg_window":
        win = -1
    elif case == "misaligned_cache":
        caches = [A, A + 4]
    elif case == "one_table":
        sin = None
    elif case == "misaligned_out":
        out = A + 8
    elif case == "too_many_layers":
        nl = 26
    layers = (q4._CDecodeLayer * nl)(*[layer() for _ in range(nl)])
    kc = (ctypes.c_void_p * nl)(*(caches + [A] * (nl - len(caches))))
    att = q4._CStepAttention(ctypes.cast(kc, ctypes.c_void_p), ctypes.cast(kc, ctypes.c_void_p), cos, sin, out, ms,
                             pos, win, heads, kv_heads, D, 0.0)
    if case == "null_caches":
        att.k_caches = None
    ws = L.q4_decode_attn_workspace_bytes(8, 2, 64) - (1 if case == "ws_small" else 0)
    Wl = _cw(0, 500, hidden)
    st = L.q4_decode_step_attn(ctypes.cast(layers, ctypes.c_void_p), nl, None if case == "null_att" else
                               ctypes.byref(att), ctypes.byref(Wl), A, 1e-6, A, A, A, A, A, A, A, A, A, ws, None)
    assert st == expect


def test_gemm_validation():
    # every case fails before any CUDA call (fake 16-byte aligned addresses)
    L = q4.lib()
    W = _cw()
    ws = q4.lib().q4_gemm_workspace_bytes(40, 64)
    # from 17 rows, the larger of the two forms' images: one 64-row tile of
    # one chunk (18432 bytes), or the tensor-memory form's 128 rows x 128 f16
    # columns plus 128 row factors (33280 bytes)
    assert ws == max(1 * 1 * (4 * 8 * 32 * 16 + 2 * 4 * 64 * 4), 128 * 128 * 2 + 128 * 4)
    assert L.q4_gemm_workspace_bytes(16, 64) == 4 * 2 * 32 * 16 + 2 * 4 * 16 * 4  # one 16-row tile
    assert L.q4_gemm_workspace_bytes(80, 64) == max(2 * 18432, 128 * 128 * 2 + 128 * 4)
    # 256-row column tiles above 128 rows, 512-row above 256
    assert L.q4_gemm_workspace_bytes(200, 128) == max(4 * 18432, 256 * 128 * 2 + 256 * 4)
    assert L.q4_gemm_workspace_bytes(300, 128) == max(5 * 18432, 512 * 128 * 2 + 512 * 4)
    assert L.q4_gemm_workspace_bytes(0, 64) == 0 and L.q4_gemm_workspace_bytes(8, 48) == 0
    assert L.q4_gemm(ctypes.byref(W), None, 40, A, 0, A, ws, None) == 1
    assert L.q4_gemm(ctypes.byref(W), A + 4, 40, A, 0, A, ws, None) == 3
    assert L.q4_gemm(ctypes.byref(W), A, 0, A, 0, A, ws, None) == 2
    assert L.q4_gemm(ctypes.byref(W), A, 40, A, 0, A, ws - 16, None) == 5
    assert L.q4_gemm(ctypes.byref(W), A, 40, A, 0, None, ws, None) == 5
    assert L.q4_gemm(ctypes.byref(W), A, 40, A, 0, A + 8, ws, None) == 3


def test_repack_validation():
    L = q4.lib()
    buf = np.zeros(4096, np.uint8)
    assert L.q4_repack_q4_0(None, 1, 32, buf.ctypes.data, buf.size) == 1
    assert L.q4_repack_q4_0(buf.ctypes.data, 1, 33, buf.ctypes.data, buf.size) == 2
    assert L.q4_repack_q4_0(buf.ctypes.data, 1, 32, buf.ctypes.data, 10) == 2


def test_debug_wait_limits_validation():
    L = q4.lib()
    assert L.q4_debug_wait_limits(0, 2, 0, 0) == 2          # at most one extra arrival
    assert L.q4_debug_wait_limits(0, -1, 0, 0) == 2
    assert L.q4_debug_wait_limits(0, 0, 0, 8) == 2          # bytes in multiples of 16
    assert L.q4_debug_wait_limits(0, 0, 0, 8192) == 2
    assert L.q4_debug_wait_limits(0, 0, 0, 0) == 0          # the defaults


def test_record_lane_words_hold_the_tensor_memory_gemm_column_pairs():
    # The tcgen05 GEMM's dequant reads, for row r and block j of a chunk, the
    # 32-bit word of lane-position t (offset (r // 8) * 512 + (4 (r % 8) + t)
    # * 16 + 4 j) and takes nibble m as element 8 m + 2 t and nibble m + 4 as
    # element 8 m + 2 t + 1 of the block, m = 0..3.  Pin that against the
    # library's own repack: every element gets a distinct nibble pattern.
    # The scale word of (row pair g, g + 8; block j) sits at 1024 + 16 g + 4 j:
    # row g's fp16 d in its low half, row g + 8's in its high half.
    n, k = 16, 128
    rng = np.random.default_rng(21)
    q = rng.integers(0, 16, (n, k), dtype=np.uint8)
    d = (0x3C00 + np.arange(n * (k // 32), dtype=np.uint16)).reshape(n, k // 32)
    P = q4.repack_q4_0(wl.pack_q4_0(q, d), n, k)
    for g in range(8):
        for j in range(4):
            sw = int(P[1024 + 16 * g + 4 * j:1024 + 16 * g + 4 * j + 4].view(np.uint32)[0])
            assert sw & 0xFFFF == d[g, j] and sw >> 16 == d[g + 8, j]
    for r in range(n):
        for j in range(4):
            for t in range(4):
                off = (r // 8) * 512 + (4 * (r % 8) + t) * 16 + 4 * j
                word = int(P[off:off + 4].view(np.uint32)[0])
                for m in range(4):
                    assert (word >> (4 * m)) & 15 == q[r, 32 * j + 8 * m + 2 * t]
                    assert (word >> (4 * m + 16)) & 15 == q[r, 32 * j + 8 * m + 2 * t + 1]
