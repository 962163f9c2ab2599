"""Pin of the oracle's decode-step composition (``oracle.decode_layer`` and
``oracle.decode_step``) against an independent composition, and mutants that
the pin must catch.

The independent side decodes the host weight bytes with numpy alone (its own
fp16 / bf16 and nibble decode, not the oracle's C), multiplies with numpy's
f64 matmul and applies RMSNorm, SwiGLU and the residual adds with numpy, in
the order of the pages' fused layer loop (honeycrisp/mod.rs,
forward_decode_fused_layers: Q with inline input_norm; K+V with inline
input_norm; o projection of the attention output plus the residual; post_norm
+ gate + up + silu; down plus the residual), then the final norm, the logits
projection and the greedy argmax (Module gpu, module sampling).  The shapes
are tiny and ragged; gamma_in, gamma_post and gamma_final differ, and the
attention stand-in is not zero, so a swapped operand anywhere changes the
result.

Each mutant plants one wiring mistake in a copy of the oracle's composition
(on the CPU, never in the library) and must fail the same comparison.
"""
import os
import sys
import types

import numpy as np
import pytest

import oracle
import q4_workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_PY = os.path.join(os.path.dirname(HERE), "oracle", "__init__.py")


# ---------------------------------------------------------------- numpy side

def _np_weights(H):
    """Dequantise a generator's host weight with numpy only."""
    if hasattr(H, "blocks"):
        b = H.blocks
        d = b[:, :, 0:2].copy().view("<f2")[:, :, 0].astype(np.float64)          # [n, k/32]
        lo = (b[:, :, 2:] & 0x0F).astype(np.float64)
        hi = (b[:, :, 2:] >> 4).astype(np.float64)
        q = np.concatenate([lo, hi], axis=2)                                     # element i, then i + 16
        return (d[:, :, None] * (q - 8.0)).reshape(H.n, H.k)
    nib = H.nib
    q = np.empty((H.n, H.k), dtype=np.float64)
    q[:, 0::2] = nib & 0x0F
    q[:, 1::2] = nib >> 4
    bf = lambda bits: (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    s = np.repeat(bf(H.s), 32, axis=1)
    m = np.repeat(bf(H.m), 32, axis=1)
    return s * q + m


def _np_norm(x, g, eps):
    return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps) * g


def _np_layer(L, src, eps):
    W = {nm: _np_weights(getattr(L, nm)) for nm in ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")}
    xn = _np_norm(src, L.gamma_in.astype(np.float64), eps)
    q, k, v = xn @ W["Wq"].T, xn @ W["Wk"].T, xn @ W["Wv"].T
    hid_o = L.attn.astype(np.float64) @ W["Wo"].T + src
    hn = _np_norm(hid_o, L.gamma_post.astype(np.float64), eps)
    g, u = hn @ W["Wg"].T, hn @ W["Wu"].T
    h = g / (1.0 + np.exp(-g)) * u
    hid = h @ W["Wd"].T + hid_o
    return dict(q=q, k=k, v=v, hid_o=hid_o, h=h, hid=hid)


def _np_attention(q, k, v, kc, vc, spec):
    """One token's attention with numpy alone: its own RoPE angles (pos /
    theta^(2j/D), element j paired with j + D/2), the append, a max-shifted
    softmax over the attended positions and the weighted sum of V."""
    H, Hkv, D, pos = spec.heads, spec.kv_heads, spec.head_dim, spec.position
    ang = pos / spec.rope_theta ** (2.0 * np.arange(D // 2) / D)
    c, s = np.cos(ang), np.sin(ang)

    def rot(x):
        a, b = x[..., :D // 2], x[..., D // 2:]
        return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)

    qh, kh, vh = rot(q.reshape(H, D)), rot(k.reshape(Hkv, D)), v.reshape(Hkv, D)
    kc, vc = kc.astype(np.float64).copy(), vc.astype(np.float64).copy()
    kc[:, pos], vc[:, pos] = kh, vh
    lo = max(0, pos + 1 - spec.window) if spec.window > 0 else 0
    out = np.empty((H, D))
    for h in range(H):
        j = h // (H // Hkv)
        sc = kc[j, lo:pos + 1] @ qh[h] / np.sqrt(D)
        p = np.exp(sc - sc.max())
        out[h] = (p / p.sum()) @ vc[j, lo:pos + 1]
    return out.reshape(1, H * D)


def _np_layer_attention(L, src, eps, spec, kc, vc):
    W = {nm: _np_weights(getattr(L, nm)) for nm in ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")}
    xn = _np_norm(src, L.gamma_in.astype(np.float64), eps)
    q, k, v = xn @ W["Wq"].T, xn @ W["Wk"].T, xn @ W["Wv"].T
    att = _np_attention(q, k, v, kc, vc, spec)
    hid_o = att @ W["Wo"].T + src
    hn = _np_norm(hid_o, L.gamma_post.astype(np.float64), eps)
    g, u = hn @ W["Wg"].T, hn @ W["Wu"].T
    h = g / (1.0 + np.exp(-g)) * u
    hid = h @ W["Wd"].T + hid_o
    return dict(q=q, k=k, v=v, attn=att, hid_o=hid_o, h=h, hid=hid)


def _np_step(cfg):
    hid = cfg.x.astype(np.float64)
    for L in cfg.layers:
        hid = _np_layer(L, hid, cfg.eps)["hid"]
    logits = _np_norm(hid, cfg.gamma_final.astype(np.float64), cfg.eps) @ _np_weights(cfg.Wlogits).T
    return np.argmax(logits, axis=1), logits, hid


# ------------------------------------------------------------------ the pin

def _close(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return a.shape == b.shape and np.allclose(a, b, rtol=1e-9, atol=1e-9 * max(1.0, float(np.abs(b).max())))


def pin_holds(orc, fmt, nb):
    """True when ``orc``'s decode_layer and decode_step agree with the numpy
    composition on a tiny two-layer step."""
    cfg = wl.cfg4(seed=11, layers=2, hidden=96, kv=32, inter=160, vocab=70, nb=nb, fmt=fmt)
    src = cfg.x.astype(np.float64)
    for L in cfg.layers:
        got = orc.decode_layer(L, src, cfg.eps)
        want = _np_layer(L, src, cfg.eps)
        for key in want:
            if not _close(got[key], want[key]):
                return False
        src = want["hid"]
    idx, logits, hid = orc.decode_step(cfg)
    widx, wlogits, whid = _np_step(cfg)
    return _close(hid, whid) and _close(logits, wlogits) and np.array_equal(np.asarray(idx), widx)


def attention_pin_holds(orc):
    """True when ``orc``'s composition with the real attention agrees with
    the numpy one on a tiny two-layer step (4 heads over 2 kv heads)."""
    spec = wl.AttnSpec(heads=4, kv_heads=2, head_dim=64, max_seq=40, position=30, window=0)
    cfg = wl.cfg4(seed=12, layers=2, hidden=256, kv=128, inter=160, vocab=70, nb=1)
    caches = wl.draw_kv_caches(12, 2, spec)
    tables = orc.rope_table(spec.max_seq, spec.head_dim, spec.rope_theta)
    src = cfg.x.astype(np.float64)
    for l, L in enumerate(cfg.layers):
        got = orc.decode_layer(L, src, cfg.eps, (spec, caches[l][0], caches[l][1], tables[0], tables[1]))
        want = _np_layer_attention(L, src, cfg.eps, spec, *caches[l])
        for key in want:
            if not _close(got[key], want[key]):
                return False
        src = want["hid"]
    idx, logits, hid = orc.decode_step(cfg, attention=(spec, caches))
    return _close(hid, src) and idx[0] == int(np.argmax(_np_norm(src, cfg.gamma_final.astype(np.float64), cfg.eps)
                                                         @ _np_weights(cfg.Wlogits).T))


@pytest.mark.parametrize("fmt,nb", [("q4_0", 1), ("q4_0", 3), ("affine", 2)])
def test_decode_composition_matches_numpy(fmt, nb):
    assert pin_holds(oracle, fmt, nb)


def test_decode_composition_with_attention_matches_numpy():
    assert attention_pin_holds(oracle)


def test_gammas_and_standin_are_distinct():
    # the pin only separates the wirings below if these differ
    cfg = wl.cfg4(seed=11, layers=2, hidden=96, kv=32, inter=160, vocab=70, nb=1)
    for L in cfg.layers:
        assert not np.array_equal(L.gamma_in, L.gamma_post)
        assert np.abs(L.attn).max() > 0
    assert not np.array_equal(cfg.gamma_final, cfg.layers[-1].gamma_post)


# ---------------------------------------------------------------- mutants

MUTANTS = {
    "gammas swapped": [("q4_nrm_gemv(_hw(L.Wq), src, L.gamma_in, eps)", "q4_nrm_gemv(_hw(L.Wq), src, L.gamma_post, eps)"),
                       ("_hw(L.Wv), src, L.gamma_in, eps)", "_hw(L.Wv), src, L.gamma_post, eps)"),
                       ("hid_o, L.gamma_post, eps)", "hid_o, L.gamma_in, eps)")],
    "o input and residual swapped": [("q4_res_gemv(_hw(L.Wo), o_in, src)", "q4_res_gemv(_hw(L.Wo), src, o_in)")],
    "down residual from the layer input": [("q4_res_gemv(_hw(L.Wd), h, hid_o)", "q4_res_gemv(_hw(L.Wd), h, src)")],
    "gate and up swapped": [("q4_gus_nrm(_hw(L.Wg), _hw(L.Wu),", "q4_gus_nrm(_hw(L.Wu), _hw(L.Wg),")],
    "k and v swapped": [("q4_dual_gemv(_hw(L.Wk), _hw(L.Wv),", "q4_dual_gemv(_hw(L.Wv), _hw(L.Wk),")],
    "gate/up fed the layer input": [("_hw(L.Wu), hid_o, L.gamma_post", "_hw(L.Wu), src, L.gamma_post")],
    "final norm dropped": [("hid, cfg.gamma_final, cfg.eps)", "hid)")],
    "final norm with the last layer's gamma": [("hid, cfg.gamma_final, cfg.eps)", "hid, Ls[-1].gamma_post, cfg.eps)")],
}


ATTN_MUTANTS = {
    "attention given v for k": [("layer_attention(q, k, v, kc, vc, spec, cosv, sinv)",
                                 "layer_attention(q, v, k, kc, vc, spec, cosv, sinv)")],
    "o fed the stand-in": [("hid_o, So = q4_res_gemv(_hw(L.Wo), o_in, src)",
                            "hid_o, So = q4_res_gemv(_hw(L.Wo), L.attn, src)")],
    "caches of the wrong layer": [("caches[l][0], caches[l][1], tables[0]", "caches[0][0], caches[0][1], tables[0]")],
}


def _mutant(edits):
    src = open(ORACLE_PY).read()
    for old, new in edits:
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    name = "oracle_mutant_%d" % abs(hash(tuple(edits)))
    mod = types.ModuleType(name)
    mod.__file__ = ORACLE_PY
    sys.modules[name] = mod            # dataclasses look their module up while the class is built
    try:
        exec(compile(src, ORACLE_PY, "exec"), mod.__dict__)
    finally:
        del sys.modules[name]
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    m = _mutant(MUTANTS[name])
    assert not (pin_holds(m, "q4_0", 1) and pin_holds(m, "q4_0", 3) and pin_holds(m, "affine", 2)), name


@pytest.mark.parametrize("name", sorted(ATTN_MUTANTS))
def test_attention_mutant_is_caught(name):
    m = _mutant(ATTN_MUTANTS[name])
    assert not attention_pin_holds(m), name
