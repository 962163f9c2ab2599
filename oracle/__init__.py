"""CPU oracle for the Q4 dequant-in-GEMV family (f64, plain C behind ctypes).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it.

Every function here takes the weights in their *host* storage format (the
bytes before any device repack) and computes in IEEE double precision:

* ``q4_0``:  blocks ``uint8[n, k/32, 18]`` -- fp16 scale ``d`` (little
  endian) then 16 nibble bytes; element ``i`` of a block is the low nibble of
  byte ``i`` and element ``i+16`` its high nibble; ``w = d*(q-8)``
  (crate inferencelayer, Functions: q4_0_to_q8_0n, gemv_q1_k_lcpp_src).
* ``q8_0``: blocks ``uint8[n, k/32, 34]`` -- fp16 scale ``d`` then 32
  signed bytes; ``w = d*q`` (crate inferencelayer, Functions: q4_0_to_q8_0n,
  gemv_q8_0n_k_lcpp_src).
* ``q4_k``: superblocks ``uint8[n, k/256, 144]`` -- fp16 ``d``, fp16
  ``dmin``, 12 bytes of 6-bit sub-scales and sub-mins (GGUF pack), 128 nibble
  bytes (runs of 32 holding sub-blocks 2r / 2r+1 in the low / high nibbles);
  ``w = d*sc*q - dmin*mn`` (crate inferencelayer, Functions:
  gemv_q5k_k_lcpp_src; honeycrisp/mod.rs, quant_matmul's Q4_K branch).
* ``q1``: superblocks ``uint8[n, k/128, 18]`` -- fp16 ``d`` then 16 bytes of
  sign bits, byte ``i`` holding elements ``8i..8i+7`` from its lowest bit;
  ``w = +d`` for a set bit, ``-d`` for a clear one (crate inferencelayer,
  Functions: gemv_q1_k_lcpp_src, gemm_q1_src).
* ``affine``: nibbles ``uint8[n, k/2]`` (element ``2i`` low nibble of byte
  ``i``, ``2i+1`` high nibble), ``s`` and ``m`` as bf16 bits
  ``uint16[n, k/32]``; ``w = s*q + m`` (Module gpu, Structs Q and HalfSet).

The composed calls below mirror the library's C entry points one for one;
each is the plain definition written out (decode, sequential dot, then the
fused neighbour), with the passage it follows named in its docstring.

Parity note: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, exhaustive decodes, exact rationals, invariants, brute force);
the decode-step composition (``decode_layer``, ``decode_step``) by
``tests/test_oracle_decode_pin.py`` (an independent numpy composition, and
wiring mutants it must catch).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_LIB = os.path.join(_HERE, "libq4oracle.so")

FMT_Q4_0 = 0
FMT_AFFINE = 1
FMT_Q8_0 = 2
FMT_Q4_K = 3
FMT_Q1 = 4


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no fused multiply-add)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
             "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None
_threads = 1


def set_threads(n: int) -> int:
    """Run the GEMV's output rows on ``n`` host threads (rows are
    independent; every output is computed by the same code either way, so
    the results do not depend on ``n``).  Returns the previous setting."""
    global _threads
    old, _threads = _threads, max(1, int(n))
    return old


def lib() -> ctypes.CDLL:
    """The compiled oracle.  ``Q4_ORACLE_LIB`` may name another build of the
    same source (the mutant tests use it to plant mistakes on the CPU)."""
    global _lib
    if _lib is None:
        path = os.environ.get("Q4_ORACLE_LIB")
        if not path:
            path = build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.q4o_half.restype = ctypes.c_double
        L.q4o_half.argtypes = [ctypes.c_uint16]
        L.q4o_bf16.restype = ctypes.c_double
        L.q4o_bf16.argtypes = [ctypes.c_uint16]
        L.q4o_q4_0_row.argtypes = [P, I64, I64, P]
        L.q4o_q8_0_row.argtypes = [P, I64, I64, P]
        L.q4o_q4_k_row.argtypes = [P, I64, I64, P]
        L.q4o_q1_row.argtypes = [P, I64, I64, P]
        L.q4o_q4_k_scale_min.argtypes = [P, ctypes.c_int, P, P]
        L.q4o_affine_row.argtypes = [P, P, P, I64, I64, P]
        L.q4o_gemv.argtypes = [ctypes.c_int, P, P, P, I64, I64, P, I64, P, P, P]
        L.q4o_gemv_rows.argtypes = [ctypes.c_int, P, P, P, I64, I64, P, I64, P, P, P, I64, I64]
        L.q4o_rmsnorm.argtypes = [P, P, I64, I64, ctypes.c_double, P]
        L.q4o_halfset_rows.argtypes = [P, P, I64, I64, P]
        L.q4o_silu.restype = ctypes.c_double
        L.q4o_silu.argtypes = [ctypes.c_double]
        L.q4o_swiglu.argtypes = [P, P, I64, P]
        L.q4o_add.argtypes = [P, P, I64, P]
        L.q4o_argmax.restype = I64
        L.q4o_rope_table.argtypes = [I64, I64, ctypes.c_double, P, P]
        L.q4o_rope_apply.argtypes = [P, I64, P, P]
        L.q4o_attn_decode.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I64, ctypes.c_double,
                                      P, P, P, P, P]
        L.q4o_argmax.argtypes = [P, I64]
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


@dataclass
class HostWeight:
    """A quantised weight matrix in its host storage format (see module doc)."""
    fmt: int
    n: int
    k: int
    a: np.ndarray                   # q4_0 / q8_0 / q4_k: blocks; affine: nibbles
    s: np.ndarray | None = None     # affine: bf16 scale bits
    m: np.ndarray | None = None     # affine: bf16 min bits

    def __post_init__(self):
        assert self.k % 32 == 0 and self.n >= 1
        self.a = np.ascontiguousarray(self.a, dtype=np.uint8)
        if self.fmt == FMT_Q4_0:
            assert self.a.size == self.n * (self.k // 32) * 18
        elif self.fmt == FMT_Q8_0:
            assert self.a.size == self.n * (self.k // 32) * 34
        elif self.fmt == FMT_Q4_K:
            assert self.k % 256 == 0 and self.a.size == self.n * (self.k // 256) * 144
        elif self.fmt == FMT_Q1:
            assert self.k % 128 == 0 and self.a.size == self.n * (self.k // 128) * 18
        else:
            assert self.a.size == self.n * self.k // 2
            self.s = np.ascontiguousarray(self.s, dtype=np.uint16)
            self.m = np.ascontiguousarray(self.m, dtype=np.uint16)
            assert self.s.size == self.m.size == self.n * self.k // 32

    @staticmethod
    def q4_0(blocks: np.ndarray, n: int, k: int) -> "HostWeight":
        return HostWeight(FMT_Q4_0, n, k, blocks)

    @staticmethod
    def q8_0(blocks: np.ndarray, n: int, k: int) -> "HostWeight":
        return HostWeight(FMT_Q8_0, n, k, blocks)

    @staticmethod
    def q4_k(blocks: np.ndarray, n: int, k: int) -> "HostWeight":
        return HostWeight(FMT_Q4_K, n, k, blocks)

    @staticmethod
    def q1(blocks: np.ndarray, n: int, k: int) -> "HostWeight":
        return HostWeight(FMT_Q1, n, k, blocks)

    @staticmethod
    def affine(nib: np.ndarray, s: np.ndarray, m: np.ndarray, n: int, k: int) -> "HostWeight":
        return HostWeight(FMT_AFFINE, n, k, nib, s, m)


# ---------------------------------------------------------------- primitives

def half_to_f64(bits: int) -> float:
    """IEEE binary16 bits -> value."""
    return lib().q4o_half(int(bits) & 0xFFFF)


def bf16_to_f64(bits: int) -> float:
    """bfloat16 bits -> value."""
    return lib().q4o_bf16(int(bits) & 0xFFFF)


def dequant_row(W: HostWeight, row: int) -> np.ndarray:
    """Row ``row`` of W as f64 weights (the format's value formula)."""
    out = np.empty(W.k, dtype=np.float64)
    if W.fmt == FMT_Q4_0:
        lib().q4o_q4_0_row(_p(W.a), W.k, row, _p(out))
    elif W.fmt == FMT_Q8_0:
        lib().q4o_q8_0_row(_p(W.a), W.k, row, _p(out))
    elif W.fmt == FMT_Q4_K:
        lib().q4o_q4_k_row(_p(W.a), W.k, row, _p(out))
    elif W.fmt == FMT_Q1:
        lib().q4o_q1_row(_p(W.a), W.k, row, _p(out))
    else:
        lib().q4o_affine_row(_p(W.a), _p(W.s), _p(W.m), W.k, row, _p(out))
    return out


def q4_k_scale_min(scale_bytes, j: int) -> tuple[int, int]:
    """Sub-block ``j``'s 6-bit (scale, min) from a Q4_K superblock's 12 scale
    bytes."""
    sb = np.ascontiguousarray(np.asarray(scale_bytes, dtype=np.uint8))
    assert sb.size == 12 and 0 <= j < 8
    sc, mn = ctypes.c_int(), ctypes.c_int()
    lib().q4o_q4_k_scale_min(_p(sb), j, ctypes.byref(sc), ctypes.byref(mn))
    return sc.value, mn.value


def dequant(W: HostWeight) -> np.ndarray:
    """All of W as f64 ``[n, k]`` (small matrices only)."""
    return np.stack([dequant_row(W, i) for i in range(W.n)])


def gemv(W: HostWeight, x) -> tuple[np.ndarray, np.ndarray]:
    """``y[r, i] = sum_k w[i, k] x[r, k]`` and the tolerance scale
    ``S[r, i] = sum_k |w[i, k]| |x[r, k]|``, both f64 ``[nb, n]``.

    x is ``[nb, k]`` (any float dtype; fp32 inputs convert exactly)."""
    x = _f64(x)
    if x.ndim == 1:
        x = x[None, :]
    nb, k = x.shape
    assert k == W.k
    y = np.empty((nb, W.n), dtype=np.float64)
    S = np.empty((nb, W.n), dtype=np.float64)
    b = W.s if W.s is not None else W.a
    c = W.m if W.m is not None else W.a
    T = min(_threads, W.n)
    if T <= 1:
        wrow = np.empty(W.k, dtype=np.float64)
        lib().q4o_gemv(W.fmt, _p(W.a), _p(b), _p(c), W.n, W.k, _p(x), nb, _p(y), _p(S), _p(wrow))
        return y, S
    # disjoint row ranges on a thread pool (ctypes releases the GIL during
    # the call), each thread with its own scratch row
    from concurrent.futures import ThreadPoolExecutor
    L = lib()
    cuts = [W.n * t // T for t in range(T + 1)]

    def part(t):
        wrow = np.empty(W.k, dtype=np.float64)
        L.q4o_gemv_rows(W.fmt, _p(W.a), _p(b), _p(c), W.n, W.k, _p(x), nb, _p(y), _p(S), _p(wrow),
                        cuts[t], cuts[t + 1])

    with ThreadPoolExecutor(max_workers=T) as ex:
        list(ex.map(part, range(T)))
    return y, S


def rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """``xhat = x / sqrt(mean(x^2) + eps) * gamma`` per row (honeycrisp/mod.rs,
    Op::RmsNorm: eps and width d = len(gamma) are its parameters)."""
    x = _f64(x)
    if x.ndim == 1:
        x = x[None, :]
    g = _f64(gamma)
    nb, k = x.shape
    assert g.shape == (k,)
    out = np.empty_like(x)
    lib().q4o_rmsnorm(_p(x), _p(g), nb, k, float(eps), _p(out))
    return out


def silu(t: float) -> float:
    return lib().q4o_silu(float(t))


def swiglu(g, u) -> np.ndarray:
    """``h = silu(g) * u`` elementwise (honeycrisp/mod.rs, fused_ffn_residual step 4)."""
    g = _f64(g)
    u = _f64(u)
    assert g.shape == u.shape
    h = np.empty_like(g)
    lib().q4o_swiglu(_p(g), _p(u), g.size, _p(h))
    return h


def add(a, b) -> np.ndarray:
    a = _f64(a)
    b = _f64(b)
    assert a.shape == b.shape
    out = np.empty_like(a)
    lib().q4o_add(_p(a), _p(b), a.size, _p(out))
    return out


def argmax(v) -> int:
    """Index of the maximum of a 1-D vector, lowest index on ties."""
    v = _f64(v).ravel()
    return int(lib().q4o_argmax(_p(v), v.size))


# ------------------------------------------------------------ composed calls
# One per library entry point; the fused steps are applied in the order the
# pages' fused kernels apply them.

def q4_gemv(W: HostWeight, x):
    """Plain dequant-in-GEMV: returns (y, S)."""
    return gemv(W, x)


def halfset_rows(x_even, x_odd) -> np.ndarray:
    """HalfSet activations as f64 rows ``[nb, k]``: element ``2i`` of a row
    from the even stream, ``2i+1`` from the odd one (f16 bit patterns,
    ``uint16[nb, k/2]`` each; Module gpu, Struct HalfSet)."""
    xe = np.ascontiguousarray(x_even, dtype=np.uint16)
    xo = np.ascontiguousarray(x_odd, dtype=np.uint16)
    if xe.ndim == 1:
        xe, xo = xe[None, :], xo[None, :]
    assert xe.shape == xo.shape
    nb, h = xe.shape
    x = np.empty((nb, 2 * h), dtype=np.float64)
    lib().q4o_halfset_rows(_p(xe), _p(xo), nb, 2 * h, _p(x))
    return x


def q4_gemv_half(W: HostWeight, x_even, x_odd):
    """GEMV over a HalfSet batch (the multi-row matvec's input format):
    returns (y, S) as ``q4_gemv`` on the decoded rows."""
    return gemv(W, halfset_rows(x_even, x_odd))


def q4_nrm_gemv(W: HostWeight, x, gamma, eps):
    """RMSNorm prologue then GEMV (honeycrisp/mod.rs, forward_decode_fused_layers
    step "1+2 Q matmul with inline input_norm").  Returns (y, S) with S taken
    over the normed activations."""
    return gemv(W, rmsnorm(x, gamma, eps))


def q4_dual_gemv(Wa: HostWeight, Wb: HostWeight, x, gamma=None, eps=0.0):
    """Two weight streams over one (optionally normed) activation batch
    (forward_decode_fused_layers step 3, K+V with inline input_norm).
    Returns (ya, Sa, yb, Sb)."""
    xh = rmsnorm(x, gamma, eps) if gamma is not None else _f64(x)
    ya, Sa = gemv(Wa, xh)
    yb, Sb = gemv(Wb, xh)
    return ya, Sa, yb, Sb


def q4_gus_nrm(Wg: HostWeight, Wu: HostWeight, x, gamma, eps):
    """RMSNorm, gate and up GEMVs, then ``h = silu(g) * u`` (honeycrisp/mod.rs,
    post_norm + gate + up + silu fused).  Returns (h, g, Sg, u, Su)."""
    xh = rmsnorm(x, gamma, eps)
    g, Sg = gemv(Wg, xh)
    u, Su = gemv(Wu, xh)
    return swiglu(g, u), g, Sg, u, Su


def q4_res_gemv(W: HostWeight, x, r):
    """``y = W x + r`` (honeycrisp/mod.rs, fused matmul + residual).
    Returns (y, S)."""
    y, S = gemv(W, x)
    r = _f64(r)
    if r.ndim == 1:
        r = r[None, :]
    return add(y, r), S


def q4_argmax(W: HostWeight, x, gamma=None, eps=0.0):
    """Logits projection (optionally behind an RMSNorm) and greedy argmax per
    activation row (Module gpu, module sampling).  Returns (idx, logits, S)."""
    xh = rmsnorm(x, gamma, eps) if gamma is not None else _f64(x)
    logits, S = gemv(W, xh)
    idx = np.array([argmax(logits[r]) for r in range(logits.shape[0])], dtype=np.int64)
    return idx, logits, S


# ---------------------------------------------------------------- decode step
# The synthetic decode step of honeycrisp/mod.rs, forward_decode_fused_layers
# (per layer: Q with inline input_norm, K+V dual with inline input_norm,
# o projection + residual, post_norm + gate + up + silu, down + residual),
# followed by the final norm, logits projection and greedy argmax of Module
# gpu, module sampling.  The attention output is the layer's given stand-in.

def _hw(H) -> HostWeight:
    """The oracle's view of a generator's host weight (any format)."""
    if hasattr(H, "blocks8"):
        return HostWeight.q8_0(H.blocks8, H.n, H.k)
    if hasattr(H, "blocks_k"):
        return HostWeight.q4_k(H.blocks_k, H.n, H.k)
    if hasattr(H, "blocks1"):
        return HostWeight.q1(H.blocks1, H.n, H.k)
    if hasattr(H, "blocks"):
        return HostWeight.q4_0(H.blocks, H.n, H.k)
    return HostWeight.affine(H.nib, H.s, H.m, H.n, H.k)


def layer_attention(q, k, v, kc, vc, spec, cosv=None, sinv=None):
    """Decode attention of one token inside a layer: q ``[1, heads*head_dim]``,
    k and v ``[1, kv_heads*head_dim]`` as heads, against the layer's caches
    ``[kv_heads, max_seq, head_dim]``; scale 1/sqrt(head_dim).  Returns
    ``(out [1, heads*head_dim], bound, kc', vc')``."""
    H, Hkv, D = spec.heads, spec.kv_heads, spec.head_dim
    out, bound, kc2, vc2 = attn_decode(_f64(q).reshape(H, D), _f64(k).reshape(Hkv, D), _f64(v).reshape(Hkv, D),
                                       kc, vc, spec.position, spec.window, 1.0 / np.sqrt(D), cosv, sinv)
    return out.reshape(1, H * D), bound.reshape(1, H * D), kc2, vc2


def decode_layer(L, src, eps: float, attention=None) -> dict:
    """One layer on f64 activations ``src [nb, hidden]``; returns every
    intermediate (and its tolerance scale) as f64 arrays.  With
    ``attention = (spec, kc, vc, cosv, sinv)`` (nb = 1) the o projection takes
    the token's attention output (honeycrisp/mod.rs, gpu_attention between the
    K+V and the o projection) instead of the layer's stand-in; the result then
    also holds ``attn`` and the appended caches ``kc``, ``vc``."""
    src = _f64(src)
    q, Sq = q4_nrm_gemv(_hw(L.Wq), src, L.gamma_in, eps)
    k, Sk, v, Sv = q4_dual_gemv(_hw(L.Wk), _hw(L.Wv), src, L.gamma_in, eps)
    extra = {}
    o_in = L.attn
    if attention is not None:
        spec, kc, vc, cosv, sinv = attention
        o_in, Sa, kc2, vc2 = layer_attention(q, k, v, kc, vc, spec, cosv, sinv)
        extra = dict(attn=o_in, Sa=Sa, kc=kc2, vc=vc2)
    hid_o, So = q4_res_gemv(_hw(L.Wo), o_in, src)
    h, g, Sg, u, Su = q4_gus_nrm(_hw(L.Wg), _hw(L.Wu), hid_o, L.gamma_post, eps)
    hid, Sd = q4_res_gemv(_hw(L.Wd), h, hid_o)
    return dict(q=q, Sq=Sq, k=k, Sk=Sk, v=v, Sv=Sv, hid_o=hid_o, So=So, h=h, g=g, Sg=Sg, u=u, Su=Su,
                hid=hid, Sd=Sd, **extra)


def decode_step(cfg, layers=None, attention=None):
    """The whole step in f64 from ``cfg.x``; returns (idx, logits, hidden).
    ``attention = (spec, caches)`` runs each layer's real attention against
    its ``(kc, vc)`` caches (see decode_layer)."""
    hid = _f64(cfg.x)
    Ls = cfg.layers if layers is None else cfg.layers[:layers]
    tables = None
    if attention is not None:
        spec, caches = attention
        tables = rope_table(spec.max_seq, spec.head_dim, spec.rope_theta)
    for l, L in enumerate(Ls):
        att = None if attention is None else (spec, caches[l][0], caches[l][1], tables[0], tables[1])
        hid = decode_layer(L, hid, cfg.eps, att)["hid"]
    idx, logits, _ = q4_argmax(_hw(cfg.Wlogits), hid, cfg.gamma_final, cfg.eps)
    return idx, logits, hid


# ---------------------------------------------------------------- attention
# Decode attention of honeycrisp/mod.rs (attn_state, gpu_attention, and the
# fused RoPE + KV-append + SDPA dispatch of forward_decode_fused_layers).

def rope_table(max_seq: int, d: int, rope_theta: float):
    """cos and sin tables ``[max_seq, d/2]`` (f64) of theta = pos /
    rope_theta^(2j/d)."""
    c = np.empty((max_seq, d // 2), np.float64)
    s = np.empty((max_seq, d // 2), np.float64)
    lib().q4o_rope_table(max_seq, d, float(rope_theta), _p(c), _p(s))
    return c, s


def rope_apply(x, c_row, s_row) -> np.ndarray:
    """One head vector rotated by a table row (element j pairs with j + d/2)."""
    x = _f64(x).copy()
    c_row, s_row = _f64(c_row), _f64(s_row)
    lib().q4o_rope_apply(_p(x), x.size, _p(c_row), _p(s_row))
    return x


def attn_decode(q, k_new, v_new, k_cache, v_cache, position: int, window: int, scale: float,
                cosv=None, sinv=None):
    """Decode attention of one token.  q ``[H, d]``, k_new / v_new
    ``[Hkv, d]``, caches ``[Hkv, max_seq, d]`` (not modified: the appended
    copies are returned), tables ``[max_seq, d/2]`` or None.  Returns
    ``(out [H, d], bound [H, d], k_cache', v_cache')``, all f64."""
    q, k_new, v_new = _f64(q), _f64(k_new), _f64(v_new)
    kc, vc = _f64(k_cache).copy(), _f64(v_cache).copy()
    H, d = q.shape
    Hkv, max_seq, _ = kc.shape
    assert H % Hkv == 0 and 0 <= position < max_seq
    out = np.empty((H, d), np.float64)
    bound = np.empty((H, d), np.float64)
    scratch = np.empty(max_seq + 2 * d, np.float64)
    cp = sp = None
    if cosv is not None:
        cosv, sinv = _f64(cosv), _f64(sinv)
        assert cosv.shape == (max_seq, d // 2) and sinv.shape == (max_seq, d // 2)
        cp, sp = _p(cosv), _p(sinv)
    lib().q4o_attn_decode(_p(q), _p(k_new), _p(v_new), _p(kc), _p(vc), max_seq, position, H, Hkv, d,
                          int(window), float(scale), cp, sp, _p(out), _p(bound), _p(scratch))
    return out, bound, kc, vc
