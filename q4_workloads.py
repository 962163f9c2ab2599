"""Seeded synthetic inputs for the Q4 dequant-in-GEMV workloads.

Shared by the tests, the smoke check and the benchmark.  This module holds
none of the method's arithmetic: only random draws (numpy PCG64,
``default_rng(seed)``) and their *storage encodings* (fp16 / bf16 rounding of
the drawn scales, nibble packing into the host byte layouts).  Both the
oracle and the CUDA library consume exactly the bytes produced here.

Host storage formats (the readings of the pages, stated once):

* Q4_0: ``uint8[n, k/32, 18]``; bytes 0-1 = fp16 scale ``d`` little endian;
  bytes 2..17 = 16 nibble bytes, byte ``i`` holding element ``i`` in its low
  nibble and element ``i + 16`` in its high nibble (GGUF order).
* Q8_0: ``uint8[n, k/32, 34]``; bytes 0-1 = fp16 scale ``d``; bytes 2..33 =
  the 32 weights as signed bytes (two's complement).
* Q4_K: ``uint8[n, k/256, 144]``; bytes 0-1 = fp16 ``d``, 2-3 = fp16 ``dmin``,
  4..15 = the eight sub-blocks' 6-bit scales and mins (GGUF pack, see
  ``Q4K_SCALE_BITS``), 16..143 = four runs of 32 nibble bytes, run ``r``
  holding sub-block ``2r`` in its low nibbles and ``2r + 1`` in its high ones.
* Q1: ``uint8[n, k/128, 18]``; bytes 0-1 = fp16 scale ``d``; bytes 2..17 =
  the sign bits, byte ``i`` holding elements ``8i..8i+7`` from its lowest
  bit (1 for ``+d``, 0 for ``-d``).
* affine-Q4: nibbles ``uint8[n, k/2]`` with byte ``i`` holding element ``2i``
  (low nibble) and ``2i + 1`` (high nibble); ``s`` and ``m`` as bf16 bit
  patterns ``uint16[n, k/32]``.

Draw order for every weight matrix: nibbles ``q`` (``integers(0, 16,
(n, k))``), then scales, then (affine) mins.  Activations are drawn after the
weights of the same configuration, in the order documented per builder.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

D_RANGE = (0.005, 0.02)       # fp16 scale d ~ U[0.005, 0.02]
S_RANGE = (0.005, 0.02)       # bf16 scale s ~ U[0.005, 0.02]
M_RANGE = (-0.1, 0.0)         # bf16 min m ~ U[-0.1, 0]
EPS = 1e-6


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def pack_q4_0(q: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """Pack nibbles ``q[n, k]`` (0..15) and fp16 scale bits ``d_bits[n, k/32]``
    into Q4_0 host blocks ``uint8[n, k/32, 18]``."""
    n, k = q.shape
    nb = k // 32
    qb = q.reshape(n, nb, 32).astype(np.uint8)
    out = np.empty((n, nb, 18), dtype=np.uint8)
    d = np.ascontiguousarray(d_bits, dtype=np.uint16).reshape(n, nb)
    out[:, :, 0] = (d & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d >> 8).astype(np.uint8)
    out[:, :, 2:] = qb[:, :, :16] | (qb[:, :, 16:] << 4)
    return out


def pack_q8_0(q: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """Pack signed bytes ``q[n, k]`` (-128..127) and fp16 scale bits
    ``d_bits[n, k/32]`` into Q8_0 host blocks ``uint8[n, k/32, 34]``."""
    n, k = q.shape
    nb = k // 32
    out = np.empty((n, nb, 34), dtype=np.uint8)
    d = np.ascontiguousarray(d_bits, dtype=np.uint16).reshape(n, nb)
    out[:, :, 0] = (d & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d >> 8).astype(np.uint8)
    out[:, :, 2:] = q.astype(np.int8).reshape(n, nb, 32).view(np.uint8)
    return out


def _q4k_scale_bits():
    """Where each bit of the Q4_K 6-bit fields lives in the 12 scale bytes:
    ``table[f, j, b] = (byte, bit)`` for field f (0 scale, 1 min) of sub-block
    j, bit b.  Sub-blocks 0-3: six bits in bytes j (scale) and j + 4 (min).
    Sub-blocks 4-7: the low four bits in byte j + 4 (scale in the low nibble,
    min in the high one), the top two in bits 6-7 of byte j - 4 (scale) and of
    byte j (min)."""
    t = np.zeros((2, 8, 6, 2), dtype=np.int64)
    for j in range(8):
        for b in range(6):
            if j < 4:
                t[0, j, b] = (j, b)
                t[1, j, b] = (j + 4, b)
            elif b < 4:
                t[0, j, b] = (j + 4, b)
                t[1, j, b] = (j + 4, b + 4)
            else:
                t[0, j, b] = (j - 4, b + 2)
                t[1, j, b] = (j, b + 2)
    return t


Q4K_SCALE_BITS = _q4k_scale_bits()


def pack_q4_k(q: np.ndarray, sc: np.ndarray, mn: np.ndarray, d_bits: np.ndarray,
              dmin_bits: np.ndarray) -> np.ndarray:
    """Pack nibbles ``q[n, k]`` (0..15), 6-bit sub-block scales and mins
    ``sc, mn[n, k/32]`` (0..63) and fp16 bits ``d_bits, dmin_bits[n, k/256]``
    into Q4_K host superblocks ``uint8[n, k/256, 144]``."""
    n, k = q.shape
    assert k % 256 == 0
    ns = k // 256
    out = np.zeros((n, ns, 144), dtype=np.uint8)
    d = np.ascontiguousarray(d_bits, dtype=np.uint16).reshape(n, ns)
    dm = np.ascontiguousarray(dmin_bits, dtype=np.uint16).reshape(n, ns)
    out[:, :, 0], out[:, :, 1] = (d & 0xFF).astype(np.uint8), (d >> 8).astype(np.uint8)
    out[:, :, 2], out[:, :, 3] = (dm & 0xFF).astype(np.uint8), (dm >> 8).astype(np.uint8)
    fields = (np.asarray(sc).reshape(n, ns, 8).astype(np.int64), np.asarray(mn).reshape(n, ns, 8).astype(np.int64))
    for f in range(2):
        for j in range(8):
            for b in range(6):
                byte, bit = Q4K_SCALE_BITS[f, j, b]
                out[:, :, 4 + byte] |= (((fields[f][:, :, j] >> b) & 1) << bit).astype(np.uint8)
    qq = q.reshape(n, ns, 4, 2, 32).astype(np.uint8)   # superblock, run, low / high, element
    out[:, :, 16:] = (qq[:, :, :, 0, :] | (qq[:, :, :, 1, :] << 4)).reshape(n, ns, 128)
    return out


def pack_q1(bits: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """Pack sign bits ``bits[n, k]`` (1 for +d, 0 for -d) and fp16 scale bits
    ``d_bits[n, k/128]`` into Q1 host superblocks ``uint8[n, k/128, 18]``."""
    n, k = bits.shape
    assert k % 128 == 0
    ns = k // 128
    out = np.empty((n, ns, 18), dtype=np.uint8)
    d = np.ascontiguousarray(d_bits, dtype=np.uint16).reshape(n, ns)
    out[:, :, 0] = (d & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d >> 8).astype(np.uint8)
    out[:, :, 2:] = np.packbits(bits.astype(np.uint8).reshape(n, ns, 128), axis=2, bitorder="little")
    return out


def pack_affine_nibbles(q: np.ndarray) -> np.ndarray:
    """Pack nibbles ``q[n, k]`` into ``uint8[n, k/2]`` (even element low)."""
    q = q.astype(np.uint8)
    return np.ascontiguousarray(q[:, 0::2] | (q[:, 1::2] << 4))


@dataclass
class Q4_0Host:
    n: int
    k: int
    blocks: np.ndarray          # uint8[n, k/32, 18]


@dataclass
class Q8_0Host:
    n: int
    k: int
    blocks8: np.ndarray         # uint8[n, k/32, 34]


@dataclass
class Q4_KHost:
    n: int
    k: int
    blocks_k: np.ndarray        # uint8[n, k/256, 144]


@dataclass
class Q1Host:
    n: int
    k: int
    blocks1: np.ndarray         # uint8[n, k/128, 18]


@dataclass
class AffineHost:
    n: int
    k: int
    nib: np.ndarray             # uint8[n, k/2]
    s: np.ndarray               # uint16[n, k/32] bf16 bits
    m: np.ndarray               # uint16[n, k/32] bf16 bits


def draw_q4_0(rng: np.random.Generator, n: int, k: int, d_range=D_RANGE) -> Q4_0Host:
    """q ~ U{0..15}, d ~ U[d_range] rounded to fp16."""
    assert k % 32 == 0
    q = rng.integers(0, 16, size=(n, k), dtype=np.uint8)
    d = rng.uniform(d_range[0], d_range[1], size=(n, k // 32)).astype(np.float16)
    return Q4_0Host(n, k, pack_q4_0(q, d.view(np.uint16)))


def draw_q8_0(rng: np.random.Generator, n: int, k: int, d_range=(0.0003, 0.0012)) -> Q8_0Host:
    """q ~ U{-128..127}, d ~ U[d_range] rounded to fp16 (the scale range gives
    weights of the magnitude of the Q4_0 draws)."""
    assert k % 32 == 0
    q = rng.integers(-128, 128, size=(n, k), dtype=np.int16)
    d = rng.uniform(d_range[0], d_range[1], size=(n, k // 32)).astype(np.float16)
    return Q8_0Host(n, k, pack_q8_0(q, d.view(np.uint16)))


def q4_0_to_q8_0(H: Q4_0Host) -> Q8_0Host:
    """The lossless upcast of Q4_0 blocks to Q8_0 (same d, q8 = nibble - 8):
    a storage re-encoding, used by the tests as an identity between formats."""
    b = H.blocks
    nib = np.concatenate([b[:, :, 2:] & 0x0F, b[:, :, 2:] >> 4], axis=2).astype(np.int16) - 8
    out = np.empty((H.n, H.k // 32, 34), dtype=np.uint8)
    out[:, :, :2] = b[:, :, :2]
    out[:, :, 2:] = nib.astype(np.int8).view(np.uint8)
    return Q8_0Host(H.n, H.k, out)


def draw_q4_k(rng: np.random.Generator, n: int, k: int, d_range=(0.0001, 0.0004),
              dmin_range=(0.0002, 0.0008)) -> Q4_KHost:
    """q ~ U{0..15}, sub-block scales and mins ~ U{0..63}, d and dmin ~
    U[range] rounded to fp16 (weights of about the Q4_0 draws' magnitude)."""
    assert k % 256 == 0
    q = rng.integers(0, 16, size=(n, k), dtype=np.uint8)
    sc = rng.integers(0, 64, size=(n, k // 32))
    mn = rng.integers(0, 64, size=(n, k // 32))
    d = rng.uniform(d_range[0], d_range[1], size=(n, k // 256)).astype(np.float16)
    dm = rng.uniform(dmin_range[0], dmin_range[1], size=(n, k // 256)).astype(np.float16)
    return Q4_KHost(n, k, pack_q4_k(q, sc, mn, d.view(np.uint16), dm.view(np.uint16)))


def draw_q1(rng: np.random.Generator, n: int, k: int, d_range=(0.02, 0.06)) -> Q1Host:
    """Signs ~ U{0, 1}, d ~ U[d_range] rounded to fp16 (weights of the Q4_0
    draws' magnitude)."""
    assert k % 128 == 0
    bits = rng.integers(0, 2, size=(n, k), dtype=np.uint8)
    d = rng.uniform(d_range[0], d_range[1], size=(n, k // 128)).astype(np.float16)
    return Q1Host(n, k, pack_q1(bits, d.view(np.uint16)))


def draw_affine(rng: np.random.Generator, n: int, k: int,
                s_range=S_RANGE, m_range=M_RANGE) -> AffineHost:
    """q ~ U{0..15}, s ~ U[s_range], m ~ U[m_range], both rounded to bf16."""
    assert k % 32 == 0
    q = rng.integers(0, 16, size=(n, k), dtype=np.uint8)
    s = rng.uniform(s_range[0], s_range[1], size=(n, k // 32)).astype(np.float32)
    m = rng.uniform(m_range[0], m_range[1], size=(n, k // 32)).astype(np.float32)
    return AffineHost(n, k, pack_affine_nibbles(q), f32_to_bf16_bits(s), f32_to_bf16_bits(m))


def draw_x(rng: np.random.Generator, nb: int, k: int) -> np.ndarray:
    """Activations ~ N(0, 1), fp32 ``[nb, k]``."""
    return rng.standard_normal((nb, k)).astype(np.float32)


def draw_gamma(rng: np.random.Generator, k: int) -> np.ndarray:
    """RMSNorm weight gamma = 1 + 0.1 * N(0, 1), fp32 ``[k]``."""
    return (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32)


# ------------------------------------------------------------ configurations

@dataclass
class Cfg0:
    """Q4_0 GEMV, nb = 1, N = K = 1024; seed 0.  Draws: W, x."""
    W: Q4_0Host
    x: np.ndarray


def cfg0(seed: int = 0, n: int = 1024, k: int = 1024) -> Cfg0:
    rng = np.random.default_rng(seed)
    W = draw_q4_0(rng, n, k)
    return Cfg0(W, draw_x(rng, 1, k))


@dataclass
class Cfg1:
    """Fused RMSNorm + Q4_0 q-projection (2048 x 2048) and the dual K/V pair
    (2 x 512 x 2048) over one normed x; nb = 1; seed 1.
    Draws: x, gamma, Wq, Wk, Wv."""
    x: np.ndarray
    gamma: np.ndarray
    Wq: Q4_0Host
    Wk: Q4_0Host
    Wv: Q4_0Host
    eps: float = EPS


def cfg1(seed: int = 1, hidden: int = 2048, kv: int = 512, nb: int = 1) -> Cfg1:
    rng = np.random.default_rng(seed)
    x = draw_x(rng, nb, hidden)
    gamma = draw_gamma(rng, hidden)
    Wq = draw_q4_0(rng, hidden, hidden)
    Wk = draw_q4_0(rng, kv, hidden)
    Wv = draw_q4_0(rng, kv, hidden)
    return Cfg1(x, gamma, Wq, Wk, Wv)


@dataclass
class Cfg2:
    """MLP block, nb = 1, hidden 2048, intermediate 8192, all Q4_0; seed 2.
    Draws: x, gamma, Wg, Wu, Wd, residual r."""
    x: np.ndarray
    gamma: np.ndarray
    Wg: Q4_0Host
    Wu: Q4_0Host
    Wd: Q4_0Host
    r: np.ndarray
    eps: float = EPS


def cfg2(seed: int = 2, hidden: int = 2048, inter: int = 8192, nb: int = 1) -> Cfg2:
    rng = np.random.default_rng(seed)
    x = draw_x(rng, nb, hidden)
    gamma = draw_gamma(rng, hidden)
    Wg = draw_q4_0(rng, inter, hidden)
    Wu = draw_q4_0(rng, inter, hidden)
    Wd = draw_q4_0(rng, hidden, inter)
    r = draw_x(rng, nb, hidden)
    return Cfg2(x, gamma, Wg, Wu, Wd, r)


@dataclass
class Cfg3:
    """Affine-Q4 multi-row matvec, K = 4096, N = 14336, nb in {1,2,4,8,16};
    seed 3.  Draws: W, then x for nb = 16 (smaller nb take the first rows)."""
    W: AffineHost
    x: np.ndarray


def cfg3(seed: int = 3, n: int = 14336, k: int = 4096, nb_max: int = 16) -> Cfg3:
    rng = np.random.default_rng(seed)
    W = draw_affine(rng, n, k)
    return Cfg3(W, draw_x(rng, nb_max, k))


@dataclass
class Layer:
    gamma_in: np.ndarray
    Wq: Q4_0Host
    Wk: Q4_0Host
    Wv: Q4_0Host
    Wo: Q4_0Host
    attn: np.ndarray            # N(0,1) stand-in for the attention output
    gamma_post: np.ndarray
    Wg: Q4_0Host
    Wu: Q4_0Host
    Wd: Q4_0Host


@dataclass
class Cfg4:
    """Synthetic decode step: ``layers`` decoder blocks, nb = 1, hidden 2048,
    then a final RMSNorm, a Q4_0 logits projection and argmax.

    Seeds: the step input x and the final gamma / logits weight come from
    ``default_rng(seed)``; layer ``l`` draws from ``default_rng(seed*1000+l)``
    in the order gamma_in, Wq, Wk, Wv, Wo, attn, gamma_post, Wg, Wu, Wd."""
    x: np.ndarray
    layers: list = field(default_factory=list)
    gamma_final: np.ndarray | None = None
    Wlogits: Q4_0Host | AffineHost | None = None
    eps: float = EPS


def _draw_fmt(fmt: str):
    if fmt == "q4_0":
        return draw_q4_0
    if fmt == "affine":
        return draw_affine
    if fmt == "q8_0":
        return draw_q8_0
    if fmt == "q4_k":
        return draw_q4_k
    if fmt == "q1":
        return draw_q1
    raise ValueError("fmt must be 'q4_0', 'affine', 'q8_0', 'q4_k' or 'q1'")


def cfg4_layer(seed: int, layer: int, hidden: int = 2048, kv: int = 512,
               inter: int = 8192, nb: int = 1, fmt: str = "q4_0") -> Layer:
    draw = _draw_fmt(fmt)
    rng = np.random.default_rng(seed * 1000 + layer)
    gamma_in = draw_gamma(rng, hidden)
    Wq = draw(rng, hidden, hidden)
    Wk = draw(rng, kv, hidden)
    Wv = draw(rng, kv, hidden)
    Wo = draw(rng, hidden, hidden)
    attn = draw_x(rng, nb, hidden)
    gamma_post = draw_gamma(rng, hidden)
    Wg = draw(rng, inter, hidden)
    Wu = draw(rng, inter, hidden)
    Wd = draw(rng, hidden, inter)
    return Layer(gamma_in, Wq, Wk, Wv, Wo, attn, gamma_post, Wg, Wu, Wd)


def cfg4(seed: int = 4, layers: int = 16, hidden: int = 2048, kv: int = 512,
         inter: int = 8192, vocab: int = 65536, nb: int = 1, fmt: str = "q4_0") -> Cfg4:
    """``fmt`` picks the weight format of every matrix (the workload itself is
    Q4_0; the affine variant serves the parity tests)."""
    draw = _draw_fmt(fmt)
    rng = np.random.default_rng(seed)
    x = draw_x(rng, nb, hidden)
    gamma_final = draw_gamma(rng, hidden)
    Wlogits = draw(rng, vocab, hidden)
    c = Cfg4(x, [], gamma_final, Wlogits)
    for l in range(layers):
        c.layers.append(cfg4_layer(seed, l, hidden, kv, inter, nb, fmt))
    return c


@dataclass
class AttnSpec:
    """Decode attention inside the step (the real step the stand-in replaces):
    ``heads`` x ``head_dim`` must be the hidden size and ``kv_heads`` x
    ``head_dim`` the k/v width; the token sits at ``position`` of caches of
    ``max_seq`` rows."""
    heads: int = 32
    kv_heads: int = 8
    head_dim: int = 64
    max_seq: int = 4096
    position: int = 4095
    window: int = 0
    rope_theta: float = 10000.0


def draw_kv_caches(seed: int, layers: int, spec: AttnSpec):
    """Per layer the K and V caches ``[kv_heads, max_seq, head_dim]`` fp32:
    rows before ``position`` (the earlier tokens) ~ N(0, 1), the rest zero."""
    out = []
    for l in range(layers):
        rng = np.random.default_rng(seed * 1000 + 500 + l)
        shape = (spec.kv_heads, spec.max_seq, spec.head_dim)
        kc = np.zeros(shape, np.float32)
        vc = np.zeros(shape, np.float32)
        kc[:, :spec.position] = rng.standard_normal((spec.kv_heads, spec.position, spec.head_dim))
        vc[:, :spec.position] = rng.standard_normal((spec.kv_heads, spec.position, spec.head_dim))
        out.append((kc, vc))
    return out


def q4_0_weight_bytes(n: int, k: int) -> int:
    """Algorithmic Q4_0 bytes: 18 per 32 weights."""
    return n * (k // 32) * 18


def affine_weight_bytes(n: int, k: int) -> int:
    """Algorithmic affine-Q4 bytes: 16 nibble bytes + 2 + 2 per 32 weights."""
    return n * (k // 32) * 20


def decode_step_weight_bytes(layers: int = 16, hidden: int = 2048, kv: int = 512,
                             inter: int = 8192, vocab: int = 65536) -> int:
    per_layer = (q4_0_weight_bytes(hidden, hidden) * 2 + q4_0_weight_bytes(kv, hidden) * 2
                 + q4_0_weight_bytes(inter, hidden) * 2 + q4_0_weight_bytes(hidden, inter))
    return layers * per_layer + q4_0_weight_bytes(vocab, hidden)
