"""Python binding of libq4gemv (weight-only 4-bit dequant-in-GEMV for sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libq4gemv.so``; this module checks tensor dtypes and devices,
passes raw pointers and the current CUDA stream, and raises on a non-OK
status.  PyTorch provides device memory and streams, nothing else.  There is
no CPU fallback: if the library is missing the calls raise.

Entry points (same names as the C ABI in ``include/q4gemv.h``):
``q4_gemv``, ``q4_nrm_gemv``, ``q4_dual_gemv``, ``q4_gus_nrm``,
``q4_res_gemv``, ``q4_argmax``, ``q4_group_sums``, ``q4_pack_half``,
``q4_gemv_half``, ``q4_gemm``, ``q4_decode_step``, ``q4_attn_decode``; plus ``Q4Weight``
for repacking host weights into the device layout and ``rope_table``.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
LIB_PATH = os.path.join(_HERE, "libq4gemv.so")
HEADER_PATH = os.path.join(_ROOT, "include", "q4gemv.h")

Q4_FMT_Q4_0 = 0
Q4_FMT_AFFINE = 1
Q4_FMT_Q8_0 = 2
Q4_FMT_Q4_K = 3
Q4_FMT_Q1 = 4
MAX_NB = 16

STATUS = {0: "Q4_OK", 1: "Q4_ERR_NULL", 2: "Q4_ERR_SHAPE", 3: "Q4_ERR_ALIGN",
          4: "Q4_ERR_UNSUPPORTED", 5: "Q4_ERR_WORKSPACE", 6: "Q4_ERR_CUDA"}


class Q4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s" % (what, STATUS.get(status, status)))


class _CWeight(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("n", ctypes.c_int32), ("k", ctypes.c_int32),
                ("dev", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


class _CDecodeLayer(ctypes.Structure):
    _fields_ = [("Wq", _CWeight), ("Wk", _CWeight), ("Wv", _CWeight), ("Wo", _CWeight), ("Wg", _CWeight),
                ("Wu", _CWeight), ("Wd", _CWeight), ("gamma_in", ctypes.c_void_p),
                ("gamma_post", ctypes.c_void_p), ("attn", ctypes.c_void_p)]


class _CStepAttention(ctypes.Structure):
    _fields_ = [("k_caches", ctypes.c_void_p), ("v_caches", ctypes.c_void_p), ("rope_cos", ctypes.c_void_p),
                ("rope_sin", ctypes.c_void_p), ("out", ctypes.c_void_p), ("max_seq", ctypes.c_int32),
                ("position", ctypes.c_int32), ("window", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("scale", ctypes.c_float)]


_lib = None


def build(force: bool = False) -> str:
    """Compile libq4gemv.so in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libq4gemv.so is not built (run __graft_entry__.build() or "
                               "bit_weight_quantized_q4_gb300.build())")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
        W = ctypes.POINTER(_CWeight)
        sig = {
            "q4_packed_bytes": (SZ, [I32, I32, I32]),
            "q4_weight_bytes": (SZ, [I32, I32, I32]),
            "q4_repack_q4_0": (I32, [P, I32, I32, P, SZ]),
            "q4_repack_affine": (I32, [P, P, P, I32, I32, P, SZ]),
            "q4_repack_q8_0": (I32, [P, I32, I32, P, SZ]),
            "q4_unpack_q8_0": (I32, [P, SZ, I32, I32, P]),
            "q4_repack_q4_k": (I32, [P, I32, I32, P, SZ]),
            "q4_unpack_q4_k": (I32, [P, SZ, I32, I32, P]),
            "q4_repack_q1": (I32, [P, I32, I32, P, SZ]),
            "q4_unpack_q1": (I32, [P, SZ, I32, I32, P]),
            "q4_unpack_q4_0": (I32, [P, SZ, I32, I32, P]),
            "q4_unpack_affine": (I32, [P, SZ, I32, I32, P, P, P]),
            "q4_group_sums": (I32, [P, I32, I32, P, P]),
            "q4_gemv": (I32, [W, P, P, I32, P, P]),
            "q4_pack_half": (I32, [P, I32, I32, P, P, P, P]),
            "q4_gemv_half": (I32, [W, P, P, P, I32, P, P]),
            "q4_nrm_gemv": (I32, [W, P, P, F, I32, P, P]),
            "q4_dual_gemv": (I32, [W, W, P, P, F, I32, P, P, P]),
            "q4_gus_nrm": (I32, [W, W, P, P, F, I32, P, P]),
            "q4_res_gemv": (I32, [W, P, P, I32, P, P]),
            "q4_argmax_workspace_bytes": (SZ, [I32, I32]),
            "q4_argmax": (I32, [W, P, P, F, I32, P, P, P, P, SZ, P]),
            "q4_argmax_noalloc": (I32, [W, P, P, F, I32, P, P, P, P]),
            "q4_decode_workspace_bytes": (SZ, [I32]),
            "q4_decode_step": (I32, [P, I32, W, P, F, I32, P, P, P, P, P, P, P, P, P, SZ, P]),
            "q4_decode_attn_workspace_bytes": (SZ, [I32, I32, I32]),
            "q4_decode_step_attn": (I32, [P, I32, P, W, P, F, P, P, P, P, P, P, P, P, P, SZ, P]),
            "q4_decode_check": (I32, [P, P]),
            "q4_device_check": (I32, [P]),
            "q4_debug_wait_limits": (I32, [ctypes.c_int64, I32, ctypes.c_int64, I32]),
            "q4_plan": (I32, [I32, I32, I32, I32, I32, I32, ctypes.POINTER(ctypes.c_int32)]),
            "q4_attn_workspace_bytes": (SZ, [I32, I32, I32]),
            "q4_gemm_workspace_bytes": (SZ, [I32, I32]),
            "q4_gemm": (I32, [W, P, I32, P, I32, P, SZ, P]),
            "q4_attn_decode": (I32, [P, P, P, P, P, I32, I32, I32, I32, I32, I32, F, P, P, P, P, SZ, P]),
            "q4_rope_table": (I32, [I32, I32, ctypes.c_double, P, P]),
            "q4_status_str": (ctypes.c_char_p, [I32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions ``include/q4gemv.h`` declares."""
    src = open(HEADER_PATH).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(q4_[a-z0-9_]+)\s*\(", src)))


def _check(status: int, what: str):
    if status != 0:
        raise Q4Error(status, what)


# ------------------------------------------------------------------ host side

def packed_bytes(fmt: int, n: int, k: int) -> int:
    return int(lib().q4_packed_bytes(fmt, n, k))


def weight_bytes(fmt: int, n: int, k: int) -> int:
    return int(lib().q4_weight_bytes(fmt, n, k))


def repack_q4_0(blocks: np.ndarray, n: int, k: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    if blocks.size != n * (k // 32) * 18:
        raise ValueError("Q4_0 blocks must be uint8[n, k/32, 18]")
    nbytes = packed_bytes(Q4_FMT_Q4_0, n, k)
    if nbytes == 0:
        raise ValueError("bad shape n=%d k=%d" % (n, k))
    out = np.empty(nbytes, dtype=np.uint8)
    _check(lib().q4_repack_q4_0(blocks.ctypes.data, n, k, out.ctypes.data, nbytes), "q4_repack_q4_0")
    return out


def repack_q8_0(blocks: np.ndarray, n: int, k: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    if blocks.size != n * (k // 32) * 34:
        raise ValueError("Q8_0 blocks must be uint8[n, k/32, 34]")
    nbytes = packed_bytes(Q4_FMT_Q8_0, n, k)
    if nbytes == 0:
        raise ValueError("bad shape n=%d k=%d" % (n, k))
    out = np.empty(nbytes, dtype=np.uint8)
    _check(lib().q4_repack_q8_0(blocks.ctypes.data, n, k, out.ctypes.data, nbytes), "q4_repack_q8_0")
    return out


def unpack_q8_0(packed: np.ndarray, n: int, k: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros((n, k // 32, 34), dtype=np.uint8)
    _check(lib().q4_unpack_q8_0(packed.ctypes.data, packed.size, n, k, out.ctypes.data), "q4_unpack_q8_0")
    return out


def repack_q4_k(blocks: np.ndarray, n: int, k: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    if k % 256 != 0 or blocks.size != n * (k // 256) * 144:
        raise ValueError("Q4_K superblocks must be uint8[n, k/256, 144] with k a multiple of 256")
    nbytes = packed_bytes(Q4_FMT_Q4_K, n, k)
    if nbytes == 0:
        raise ValueError("bad shape n=%d k=%d" % (n, k))
    out = np.empty(nbytes, dtype=np.uint8)
    _check(lib().q4_repack_q4_k(blocks.ctypes.data, n, k, out.ctypes.data, nbytes), "q4_repack_q4_k")
    return out


def unpack_q4_k(packed: np.ndarray, n: int, k: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros((n, k // 256, 144), dtype=np.uint8)
    _check(lib().q4_unpack_q4_k(packed.ctypes.data, packed.size, n, k, out.ctypes.data), "q4_unpack_q4_k")
    return out


def repack_q1(blocks: np.ndarray, n: int, k: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    if k % 128 != 0 or blocks.size != n * (k // 128) * 18:
        raise ValueError("Q1 superblocks must be uint8[n, k/128, 18] with k a multiple of 128")
    nbytes = packed_bytes(Q4_FMT_Q1, n, k)
    if nbytes == 0:
        raise ValueError("bad shape n=%d k=%d" % (n, k))
    out = np.empty(nbytes, dtype=np.uint8)
    _check(lib().q4_repack_q1(blocks.ctypes.data, n, k, out.ctypes.data, nbytes), "q4_repack_q1")
    return out


def unpack_q1(packed: np.ndarray, n: int, k: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros((n, k // 128, 18), dtype=np.uint8)
    _check(lib().q4_unpack_q1(packed.ctypes.data, packed.size, n, k, out.ctypes.data), "q4_unpack_q1")
    return out


def repack_affine(nib: np.ndarray, s: np.ndarray, m: np.ndarray, n: int, k: int) -> np.ndarray:
    nib = np.ascontiguousarray(nib, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    m = np.ascontiguousarray(m, dtype=np.uint16)
    if nib.size != n * k // 2 or s.size != n * k // 32 or m.size != n * k // 32:
        raise ValueError("affine weights must be nib uint8[n, k/2], s/m uint16[n, k/32]")
    nbytes = packed_bytes(Q4_FMT_AFFINE, n, k)
    if nbytes == 0:
        raise ValueError("bad shape n=%d k=%d" % (n, k))
    out = np.empty(nbytes, dtype=np.uint8)
    _check(lib().q4_repack_affine(nib.ctypes.data, s.ctypes.data, m.ctypes.data, n, k,
                                  out.ctypes.data, nbytes), "q4_repack_affine")
    return out


def unpack_q4_0(packed: np.ndarray, n: int, k: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros((n, k // 32, 18), dtype=np.uint8)
    _check(lib().q4_unpack_q4_0(packed.ctypes.data, packed.size, n, k, out.ctypes.data), "q4_unpack_q4_0")
    return out


def unpack_affine(packed: np.ndarray, n: int, k: int):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    nib = np.zeros((n, k // 2), dtype=np.uint8)
    s = np.zeros((n, k // 32), dtype=np.uint16)
    m = np.zeros((n, k // 32), dtype=np.uint16)
    _check(lib().q4_unpack_affine(packed.ctypes.data, packed.size, n, k, nib.ctypes.data,
                                  s.ctypes.data, m.ctypes.data), "q4_unpack_affine")
    return nib, s, m


def plan(fmt: int, tiles: int, chunks: int, nb: int, pairs: bool, num_sms: int) -> dict:
    out = (ctypes.c_int32 * 6)()
    _check(lib().q4_plan(fmt, tiles, chunks, nb, int(pairs), num_sms, out), "q4_plan")
    return dict(zip(("TG", "S", "Cs", "groups", "ctas", "smem"), list(out)))


# ---------------------------------------------------------------- device side

def _torch():
    import torch
    return torch


class Q4Weight:
    """A repacked weight matrix resident in device memory (owns its tensor)."""

    def __init__(self, fmt: int, n: int, k: int, packed: np.ndarray, device="cuda"):
        torch = _torch()
        self.fmt, self.n, self.k = int(fmt), int(n), int(k)
        self.tensor = torch.from_numpy(packed).to(device)
        self.nbytes = int(packed.size)
        self._c = _CWeight(self.fmt, self.n, self.k, self.tensor.data_ptr(), self.nbytes)

    @classmethod
    def from_q4_0(cls, blocks: np.ndarray, n: int, k: int, device="cuda") -> "Q4Weight":
        return cls(Q4_FMT_Q4_0, n, k, repack_q4_0(blocks, n, k), device)

    @classmethod
    def from_q8_0(cls, blocks: np.ndarray, n: int, k: int, device="cuda") -> "Q4Weight":
        return cls(Q4_FMT_Q8_0, n, k, repack_q8_0(blocks, n, k), device)

    @classmethod
    def from_q4_k(cls, blocks: np.ndarray, n: int, k: int, device="cuda") -> "Q4Weight":
        return cls(Q4_FMT_Q4_K, n, k, repack_q4_k(blocks, n, k), device)

    @classmethod
    def from_q1(cls, blocks: np.ndarray, n: int, k: int, device="cuda") -> "Q4Weight":
        return cls(Q4_FMT_Q1, n, k, repack_q1(blocks, n, k), device)

    @classmethod
    def from_affine(cls, nib, s, m, n: int, k: int, device="cuda") -> "Q4Weight":
        return cls(Q4_FMT_AFFINE, n, k, repack_affine(nib, s, m, n, k), device)

    @property
    def weight_bytes(self) -> int:
        """Algorithmic bytes: 18 (Q4_0), 20 (affine) or 34 (Q8_0) per 32
        weights, 144 per 256 (Q4_K), 18 per 128 (Q1)."""
        return weight_bytes(self.fmt, self.n, self.k)

    def cref(self):
        return ctypes.byref(self._c)


def _stream():
    return _torch().cuda.current_stream().cuda_stream


def _dev_f32(t, name, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError("%s must be a CUDA float32 tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    return t


def _dev_buf(t, name, dtype, shape, device, min_numel=None):
    """A caller-supplied output or workspace: a contiguous CUDA tensor of
    `dtype` on `device`, of exactly `shape` (or, for a workspace, at least
    `min_numel` elements).  The C ABI carries no sizes for these buffers, so
    everything is checked here, before any launch."""
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype:
        raise TypeError("%s must be a CUDA %s tensor" % (name, dtype))
    if t.device != device:
        raise ValueError("%s is on %s, the activations on %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if min_numel is not None:
        if t.numel() < min_numel:
            raise ValueError("%s has %d elements, needs at least %d" % (name, t.numel(), min_numel))
    elif tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    return t


def _argmax_outs(W, x, nb, want_val, want_logits, idx, val, logits):
    torch = _torch()
    if idx is None:
        idx = torch.empty(nb, dtype=torch.int32, device=x.device)
    idx = _dev_buf(idx, "idx", torch.int32, (nb,), x.device)
    if want_val and val is None:
        val = torch.empty(nb, dtype=torch.float32, device=x.device)
    if val is not None:
        val = _dev_buf(val, "val", torch.float32, (nb,), x.device)
    if want_logits and logits is None:
        logits = torch.empty((nb, W.n), dtype=torch.float32, device=x.device)
    if logits is not None:
        logits = _dev_buf(logits, "logits", torch.float32, (nb, W.n), x.device)
    return idx, val, logits


def _rows(x, k):
    x = _dev_f32(x, "x")
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.dim() != 2 or x.shape[1] != k:
        raise ValueError("x must be [nb, %d]" % k)
    return x, x.shape[0]


def _out(out, shape, like):
    torch = _torch()
    if out is None:
        return torch.empty(shape, dtype=torch.float32, device=like.device)
    return _dev_f32(out, "out", shape)


def q4_group_sums(x, out=None):
    torch = _torch()
    x = _dev_f32(x, "x")
    if x.dim() == 1:
        x = x.view(1, -1)
    nb, k = x.shape
    out = _out(out, (nb, k // 32), x)
    _check(lib().q4_group_sums(x.data_ptr(), nb, k, out.data_ptr(), _stream()), "q4_group_sums")
    return out


def q4_gemv(W: Q4Weight, x, gsum=None, out=None):
    x, nb = _rows(x, W.k)
    out = _out(out, (nb, W.n), x)
    gp = None
    if gsum is not None:
        gp = _dev_f32(gsum, "gsum", (nb, W.k // 32)).data_ptr()
    _check(lib().q4_gemv(W.cref(), x.data_ptr(), gp, nb, out.data_ptr(), _stream()), "q4_gemv")
    return out


def q4_pack_half(x, with_gsum: bool = True):
    """The HalfSet of fp32 activations ``x [nb, k]``: ``(x_even, x_odd,
    gsum)`` -- float16 ``[nb, k/2]`` streams of the even- and odd-indexed
    elements and the fp32 per-32 group sums of the f16 values (or None)."""
    torch = _torch()
    x = _dev_f32(x, "x")
    if x.dim() == 1:
        x = x.view(1, -1)
    nb, k = x.shape
    xe = torch.empty((nb, k // 2), dtype=torch.float16, device=x.device)
    xo = torch.empty((nb, k // 2), dtype=torch.float16, device=x.device)
    gs = torch.empty((nb, k // 32), dtype=torch.float32, device=x.device) if with_gsum else None
    _check(lib().q4_pack_half(x.data_ptr(), nb, k, xe.data_ptr(), xo.data_ptr(),
                              None if gs is None else gs.data_ptr(), _stream()), "q4_pack_half")
    return xe, xo, gs


def q4_gemv_half(W: Q4Weight, x_even, x_odd, gsum=None, out=None):
    """``y = W x`` for a batch given as a HalfSet (see ``q4_pack_half``)."""
    torch = _torch()
    if x_even.dim() == 1:
        x_even, x_odd = x_even.view(1, -1), x_odd.view(1, -1)
    nb = x_even.shape[0]
    dev = x_even.device
    x_even = _dev_buf(x_even, "x_even", torch.float16, (nb, W.k // 2), dev)
    x_odd = _dev_buf(x_odd, "x_odd", torch.float16, (nb, W.k // 2), dev)
    gp = None
    if gsum is not None:
        gp = _dev_buf(gsum, "gsum", torch.float32, (nb, W.k // 32), dev).data_ptr()
    out = _out(out, (nb, W.n), x_even)
    _check(lib().q4_gemv_half(W.cref(), x_even.data_ptr(), x_odd.data_ptr(), gp, nb, out.data_ptr(), _stream()),
           "q4_gemv_half")
    return out


def q4_nrm_gemv(W: Q4Weight, x, gamma, eps: float, out=None):
    x, nb = _rows(x, W.k)
    gamma = _dev_f32(gamma, "gamma", (W.k,))
    out = _out(out, (nb, W.n), x)
    _check(lib().q4_nrm_gemv(W.cref(), x.data_ptr(), gamma.data_ptr(), float(eps), nb, out.data_ptr(),
                             _stream()), "q4_nrm_gemv")
    return out


def q4_dual_gemv(Wa: Q4Weight, Wb: Q4Weight, x, gamma=None, eps: float = 0.0, out_a=None, out_b=None):
    x, nb = _rows(x, Wa.k)
    gp = None if gamma is None else _dev_f32(gamma, "gamma", (Wa.k,)).data_ptr()
    out_a = _out(out_a, (nb, Wa.n), x)
    out_b = _out(out_b, (nb, Wb.n), x)
    _check(lib().q4_dual_gemv(Wa.cref(), Wb.cref(), x.data_ptr(), gp, float(eps), nb, out_a.data_ptr(),
                              out_b.data_ptr(), _stream()), "q4_dual_gemv")
    return out_a, out_b


def q4_gus_nrm(Wg: Q4Weight, Wu: Q4Weight, x, gamma, eps: float, out=None):
    x, nb = _rows(x, Wg.k)
    gamma = _dev_f32(gamma, "gamma", (Wg.k,))
    out = _out(out, (nb, Wg.n), x)
    _check(lib().q4_gus_nrm(Wg.cref(), Wu.cref(), x.data_ptr(), gamma.data_ptr(), float(eps), nb,
                            out.data_ptr(), _stream()), "q4_gus_nrm")
    return out


def q4_res_gemv(W: Q4Weight, x, r, out=None):
    """``out = W x + r``; pass ``out=r`` for the in-place residual stream."""
    x, nb = _rows(x, W.k)
    r = _dev_f32(r, "r", (nb, W.n)) if _torch().is_tensor(r) and r.dim() == 2 else _dev_f32(r, "r").view(nb, W.n)
    out = _out(out, (nb, W.n), x)
    _check(lib().q4_res_gemv(W.cref(), x.data_ptr(), r.data_ptr(), nb, out.data_ptr(), _stream()),
           "q4_res_gemv")
    return out


def q4_argmax_workspace_bytes(n: int, nb: int) -> int:
    return int(lib().q4_argmax_workspace_bytes(n, nb))


def q4_argmax(W: Q4Weight, x, gamma=None, eps: float = 0.0, want_val=False, want_logits=False,
              workspace=None, idx=None, val=None, logits=None):
    """Greedy argmax of the logits ``W xhat`` per activation row.  Returns
    ``(idx int32[nb], val or None, logits or None)``."""
    torch = _torch()
    x, nb = _rows(x, W.k)
    gp = None if gamma is None else _dev_f32(gamma, "gamma", (W.k,)).data_ptr()
    ws_bytes = q4_argmax_workspace_bytes(W.n, nb)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    workspace = _dev_buf(workspace, "workspace", torch.uint8, None, x.device, min_numel=ws_bytes)
    idx, val, logits = _argmax_outs(W, x, nb, want_val, want_logits, idx, val, logits)
    _check(lib().q4_argmax(W.cref(), x.data_ptr(), gp, float(eps), nb, idx.data_ptr(),
                           None if val is None else val.data_ptr(),
                           None if logits is None else logits.data_ptr(),
                           workspace.data_ptr(), workspace.numel(), _stream()), "q4_argmax")
    return idx, val, logits


def q4_argmax_noalloc(W: Q4Weight, x, gamma=None, eps: float = 0.0, want_val=False, want_logits=False,
                      idx=None, val=None, logits=None):
    """Like ``q4_argmax`` but without a workspace: the pass-1 pairs live in a
    fixed array inside the library (for callers that cannot allocate device
    memory; see ``q4_argmax_noalloc`` in the C header for the size limit and
    the sharing rules).  Returns ``(idx, val or None, logits or None)``."""
    x, nb = _rows(x, W.k)
    gp = None if gamma is None else _dev_f32(gamma, "gamma", (W.k,)).data_ptr()
    idx, val, logits = _argmax_outs(W, x, nb, want_val, want_logits, idx, val, logits)
    _check(lib().q4_argmax_noalloc(W.cref(), x.data_ptr(), gp, float(eps), nb, idx.data_ptr(),
                                   None if val is None else val.data_ptr(),
                                   None if logits is None else logits.data_ptr(), _stream()),
           "q4_argmax_noalloc")
    return idx, val, logits


def q4_decode_workspace_bytes(nb: int) -> int:
    return int(lib().q4_decode_workspace_bytes(nb))


class DecodeLayers:
    """Host array of q4_decode_layer descriptors (keeps the tensors alive)."""

    def __init__(self, layers):
        self.layers = list(layers)
        arr = (_CDecodeLayer * len(self.layers))()
        for i, L in enumerate(self.layers):
            arr[i] = _CDecodeLayer(L.Wq._c, L.Wk._c, L.Wv._c, L.Wo._c, L.Wg._c, L.Wu._c, L.Wd._c,
                                   _dev_f32(L.gamma_in, "gamma_in").data_ptr(),
                                   _dev_f32(L.gamma_post, "gamma_post").data_ptr(),
                                   _dev_f32(L.attn, "attn").data_ptr())
        self.arr = arr

    def __len__(self):
        return len(self.layers)


def q4_decode_attn_workspace_bytes(heads: int, kv_heads: int, head_dim: int) -> int:
    return int(lib().q4_decode_attn_workspace_bytes(heads, kv_heads, head_dim))


class StepAttention:
    """The decode attention of ``q4_decode_step_attn``: per-layer caches
    (``[kv_heads][max_seq][head_dim]`` float32 CUDA tensors), optional RoPE
    tables, the attention output buffer ``out`` (``[1, heads*head_dim]``)
    and the geometry.  Keeps the tensors and the host pointer arrays alive."""

    def __init__(self, caches, out, position: int, window: int = 0, rope=None, scale: float | None = None):
        torch = _torch()
        self.caches = [(_dev_f32(kc, "k_cache"), _dev_f32(vc, "v_cache")) for kc, vc in caches]
        if not self.caches:
            raise ValueError("no caches")
        kv_heads, max_seq, head_dim = self.caches[0][0].shape
        for kc, vc in self.caches:
            if tuple(kc.shape) != (kv_heads, max_seq, head_dim) or tuple(vc.shape) != (kv_heads, max_seq, head_dim):
                raise ValueError("every cache must be [kv_heads, max_seq, head_dim] like the first")
        self.out = _dev_f32(out, "out")
        heads = self.out.numel() // head_dim
        if heads * head_dim != self.out.numel():
            raise ValueError("out must hold heads * head_dim values")
        self.rope = None
        if rope is not None:
            c, sn = (_dev_f32(t, "rope table") for t in rope)
            if tuple(c.shape) != (max_seq, head_dim // 2) or tuple(sn.shape) != (max_seq, head_dim // 2):
                raise ValueError("rope tables must be [max_seq, head_dim/2]")
            self.rope = (c, sn)
        self._k = (ctypes.c_void_p * len(self.caches))(*[kc.data_ptr() for kc, _ in self.caches])
        self._v = (ctypes.c_void_p * len(self.caches))(*[vc.data_ptr() for _, vc in self.caches])
        self.c = _CStepAttention(ctypes.cast(self._k, ctypes.c_void_p), ctypes.cast(self._v, ctypes.c_void_p),
                                 None if self.rope is None else self.rope[0].data_ptr(),
                                 None if self.rope is None else self.rope[1].data_ptr(), self.out.data_ptr(),
                                 max_seq, int(position), int(window), heads, kv_heads, head_dim,
                                 0.0 if scale is None else float(scale))
        self.heads, self.kv_heads, self.head_dim = heads, kv_heads, head_dim

    def __len__(self):
        return len(self.caches)


def q4_decode_step_attn(layers: DecodeLayers, att: StepAttention, Wlogits: Q4Weight, gamma_final, eps: float, x_in,
                        hid, q, k, v, h, idx, val, workspace, n_layers: int | None = None):
    """The real decode step (each layer's decode attention between its q/k/v
    and o projections) as a single persistent kernel (``q4_decode_step_attn``
    in the C header); nb = 1.  All buffers are caller-owned CUDA tensors."""
    torch = _torch()
    n = len(layers) if n_layers is None else int(n_layers)
    if n > len(att):
        raise ValueError("fewer caches than layers")
    x_in = _dev_f32(x_in, "x_in")
    if x_in.shape[0] != 1:
        raise ValueError("the attention step takes one activation row")
    idx = _dev_buf(idx, "idx", torch.int32, (1,), x_in.device)
    if val is not None:
        val = _dev_buf(val, "val", torch.float32, (1,), x_in.device)
    workspace = _dev_buf(workspace, "workspace", torch.uint8, None, x_in.device,
                         min_numel=max(1, q4_decode_attn_workspace_bytes(att.heads, att.kv_heads, att.head_dim)))
    L0 = layers.layers[0]
    hidden = L0.Wo.n
    for t, name, width in ((x_in, "x_in", hidden), (hid, "hid", hidden), (q, "q", L0.Wq.n), (k, "k", L0.Wk.n),
                           (v, "v", L0.Wv.n), (h, "h", L0.Wg.n)):
        _dev_buf(t, name, torch.float32, (1, width), x_in.device)
    _check(lib().q4_decode_step_attn(ctypes.cast(layers.arr, ctypes.c_void_p), n, ctypes.byref(att.c),
                                     Wlogits.cref(), _dev_f32(gamma_final, "gamma_final").data_ptr(), float(eps),
                                     x_in.data_ptr(), _dev_f32(hid, "hid").data_ptr(), _dev_f32(q, "q").data_ptr(),
                                     _dev_f32(k, "k").data_ptr(), _dev_f32(v, "v").data_ptr(),
                                     _dev_f32(h, "h").data_ptr(), idx.data_ptr(),
                                     None if val is None else val.data_ptr(), workspace.data_ptr(),
                                     workspace.numel(), _stream()), "q4_decode_step_attn")


def q4_decode_step(layers: DecodeLayers, Wlogits: Q4Weight, gamma_final, eps: float, x_in, hid, q, k, v, h,
                   idx, val, workspace, n_layers: int | None = None):
    """One decode step as a single persistent kernel (see ``q4_decode_step``
    in the C header).  All buffers are caller-owned CUDA tensors."""
    torch = _torch()
    n = len(layers) if n_layers is None else int(n_layers)
    x_in = _dev_f32(x_in, "x_in")
    nb = x_in.shape[0]
    idx = _dev_buf(idx, "idx", torch.int32, (nb,), x_in.device)
    if val is not None:
        val = _dev_buf(val, "val", torch.float32, (nb,), x_in.device)
    workspace = _dev_buf(workspace, "workspace", torch.uint8, None, x_in.device,
                         min_numel=q4_decode_workspace_bytes(nb))
    L0 = layers.layers[0]
    hidden = L0.Wo.n
    for t, name, width in ((x_in, "x_in", hidden), (hid, "hid", hidden), (q, "q", L0.Wq.n), (k, "k", L0.Wk.n),
                           (v, "v", L0.Wv.n), (h, "h", L0.Wg.n)):
        _dev_buf(t, name, torch.float32, (nb, width), x_in.device)
    _check(lib().q4_decode_step(ctypes.cast(layers.arr, ctypes.c_void_p), n, Wlogits.cref(),
                                _dev_f32(gamma_final, "gamma_final").data_ptr(), float(eps), nb,
                                _dev_f32(x_in, "x_in").data_ptr(), _dev_f32(hid, "hid").data_ptr(),
                                _dev_f32(q, "q").data_ptr(), _dev_f32(k, "k").data_ptr(),
                                _dev_f32(v, "v").data_ptr(), _dev_f32(h, "h").data_ptr(), idx.data_ptr(),
                                None if val is None else val.data_ptr(), workspace.data_ptr(),
                                workspace.numel(), _stream()), "q4_decode_step")


def q4_decode_check(workspace):
    workspace = _dev_buf(workspace, "workspace", _torch().uint8, None, workspace.device, min_numel=16)
    _check(lib().q4_decode_check(workspace.data_ptr(), _stream()), "q4_decode_check")


def q4_debug_wait_limits(barrier_polls: int = 0, barrier_extra: int = 0, copy_wait_cycles: int = 0,
                         copy_extra_bytes: int = 0):
    """Testing hook: shorten the kernels' wait bounds and make their waits
    expect arrivals or bytes that never come (see ``q4_debug_wait_limits`` in
    the C header).  ``q4_debug_wait_limits()`` restores the defaults."""
    _check(lib().q4_debug_wait_limits(int(barrier_polls), int(barrier_extra), int(copy_wait_cycles),
                                      int(copy_extra_bytes)), "q4_debug_wait_limits")


def q4_device_check():
    """Synchronise the current stream; raise if a GEMV-family kernel gave up
    waiting for its weight copies since the last check (the flag is cleared)."""
    _check(lib().q4_device_check(_stream()), "q4_device_check")


# ---------------------------------------------------------------- attention

def rope_table(max_seq: int, d: int, rope_theta: float = 10000.0):
    """Host RoPE tables (cos, sin), float32 ``[max_seq, d/2]`` (q4_rope_table)."""
    c = np.empty((max_seq, d // 2), np.float32)
    sn = np.empty((max_seq, d // 2), np.float32)
    _check(lib().q4_rope_table(max_seq, d, float(rope_theta), c.ctypes.data, sn.ctypes.data), "q4_rope_table")
    return c, sn


def q4_attn_decode(q, k_new, v_new, k_cache, v_cache, position: int, window: int = 0, scale=None, rope=None,
                   out=None, workspace=None):
    """Decode attention of one token: q ``[H, D]``, k_new / v_new ``[Hkv, D]``,
    caches ``[Hkv, max_seq, D]`` (row ``position`` is written), ``rope`` an
    optional (cos, sin) pair of ``[max_seq, D/2]`` device tables.  Returns
    out ``[H, D]``; ``scale`` defaults to 1/sqrt(D)."""
    torch = _torch()
    q = _dev_f32(q, "q")
    if q.dim() != 2:
        raise ValueError("q must be [H, D]")
    H, D = q.shape
    dev = q.device
    k_cache = _dev_buf(k_cache, "k_cache", torch.float32, None, dev, min_numel=0)
    if k_cache.dim() != 3 or k_cache.shape[2] != D:
        raise ValueError("k_cache must be [Hkv, max_seq, D]")
    Hkv, max_seq = int(k_cache.shape[0]), int(k_cache.shape[1])
    _dev_buf(v_cache, "v_cache", torch.float32, (Hkv, max_seq, D), dev)
    _dev_buf(k_new, "k_new", torch.float32, (Hkv, D), dev)
    _dev_buf(v_new, "v_new", torch.float32, (Hkv, D), dev)
    cp = sp = None
    if rope is not None:
        cos_t, sin_t = rope
        cp = _dev_buf(cos_t, "rope cos", torch.float32, (max_seq, D // 2), dev).data_ptr()
        sp = _dev_buf(sin_t, "rope sin", torch.float32, (max_seq, D // 2), dev).data_ptr()
    if out is None:
        out = torch.empty((H, D), dtype=torch.float32, device=dev)
    else:
        _dev_buf(out, "out", torch.float32, (H, D), dev)
    wsb = int(lib().q4_attn_workspace_bytes(H, D, max_seq))
    if workspace is None:  # zero-filled: its split counters start at zero
        workspace = torch.zeros(max(16, wsb), dtype=torch.uint8, device=dev)
    else:
        _dev_buf(workspace, "workspace", torch.uint8, None, dev, min_numel=wsb)
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    _check(lib().q4_attn_decode(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                                v_cache.data_ptr(), max_seq, int(position), H, Hkv, D, int(window), float(scale),
                                cp, sp, out.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream()),
           "q4_attn_decode")
    return out


# ---------------------------------------------------------------- prefill GEMM

def q4_gemm(W: Q4Weight, x, accumulate: bool = False, out=None, workspace=None):
    """y = x W^T for any batch width (meant for nb > 16): x ``[nb, k]``
    float32 CUDA; with ``accumulate`` the product is added to ``out``."""
    torch = _torch()
    x = _dev_f32(x, "x")
    if x.dim() != 2 or x.shape[1] != W.k:
        raise ValueError("x must be [nb, %d]" % W.k)
    nb = int(x.shape[0])
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs out")
        out = torch.empty((nb, W.n), dtype=torch.float32, device=x.device)
    else:
        _dev_buf(out, "out", torch.float32, (nb, W.n), x.device)
    wsb = int(lib().q4_gemm_workspace_bytes(nb, W.k))
    if workspace is None:
        workspace = torch.empty(max(16, wsb), dtype=torch.uint8, device=x.device)
    else:
        _dev_buf(workspace, "workspace", torch.uint8, None, x.device, min_numel=wsb)
    _check(lib().q4_gemm(W.cref(), x.data_ptr(), nb, out.data_ptr(), int(bool(accumulate)), workspace.data_ptr(),
                         workspace.numel(), _stream()), "q4_gemm")
    return out
