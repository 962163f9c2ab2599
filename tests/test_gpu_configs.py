"""Parity at the full workload sizes: the Q4_0 GEMV (1024 x 1024), the fused
RMSNorm q projection and dual K/V (2048 x 2048, 2 x 512 x 2048), the MLP
block (gate/up 8192 x 2048 + SwiGLU, down 2048 x 8192 + residual), the affine
14336 x 4096 matvec at nb = 1, 2, 4, 8, 16, and the whole 16-layer decode step
in the launch configuration the benchmark times (teacher-forced: each call is
checked against the oracle run on that call's own GPU inputs)."""
import numpy as np
import pytest

import oracle
import q4_workloads as wl
from parity import check, check_argmax, check_residual, check_swiglu, dev_weight, host_weight, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def q4():
    import bit_weight_quantized_q4_gb300 as m
    m.build()
    m.lib()
    return m


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_q4_0_gemv_1024(q4):
    c = wl.cfg0()
    y = q4.q4_gemv(dev_weight(c.W), T(c.x))
    ref, S = oracle.q4_gemv(host_weight(c.W), c.x)
    check(to_np(y), ref, S, what="1024x1024")


def test_nrm_q_and_dual_kv_2048(q4):
    c = wl.cfg1()
    y = q4.q4_nrm_gemv(dev_weight(c.Wq), T(c.x), T(c.gamma), c.eps)
    ref, S = oracle.q4_nrm_gemv(host_weight(c.Wq), c.x, c.gamma, c.eps)
    check(to_np(y), ref, S, what="nrm q")
    yk, yv = q4.q4_dual_gemv(dev_weight(c.Wk), dev_weight(c.Wv), T(c.x), T(c.gamma), c.eps)
    ra, Sa, rb, Sb = oracle.q4_dual_gemv(host_weight(c.Wk), host_weight(c.Wv), c.x, c.gamma, c.eps)
    check(to_np(yk), ra, Sa, what="dual k")
    check(to_np(yv), rb, Sb, what="dual v")


def test_mlp_block_2048_8192(q4):
    c = wl.cfg2()
    h = q4.q4_gus_nrm(dev_weight(c.Wg), dev_weight(c.Wu), T(c.x), T(c.gamma), c.eps)
    _, g, Sg, u, Su = oracle.q4_gus_nrm(host_weight(c.Wg), host_weight(c.Wu), c.x, c.gamma, c.eps)
    check_swiglu(to_np(h), g, Sg, u, Su, what="gus")
    r = T(c.r)
    y = q4.q4_res_gemv(dev_weight(c.Wd), h, r)
    ref, S = oracle.q4_res_gemv(host_weight(c.Wd), h.cpu().numpy(), c.r)   # teacher-forced on the GPU h
    check_residual(to_np(y), ref, S, what="down+res")


@pytest.fixture(scope="module")
def cfg3():
    return wl.cfg3()


@pytest.mark.parametrize("nb", [1, 2, 4, 8, 16])
def test_affine_14336x4096(q4, cfg3, nb):
    x = cfg3.x[:nb]
    W = dev_weight(cfg3.W)
    y = q4.q4_gemv(W, T(x))
    ref, S = oracle.q4_gemv(host_weight(cfg3.W), x)
    check(to_np(y), ref, S, what="affine nb=%d" % nb)
    gs = q4.q4_group_sums(T(x))
    assert torch.equal(q4.q4_gemv(W, T(x), gsum=gs), y)


def test_decode_step_teacher_forced(q4):
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    cfg = wl.cfg4()
    step = DecodeStep(cfg)
    snaps = []

    def hook(name, l):
        if name == "q":
            snaps.append({"src": (step.x_in if l == 0 else step.hid).clone(), "q": step.q.clone()})
        elif name == "kv":
            snaps[-1].update(k=step.k.clone(), v=step.v.clone())
        elif name == "o":
            snaps[-1]["hid_o"] = step.hid.clone()
        elif name == "gus":
            snaps[-1]["h"] = step.h.clone()
        elif name == "down":
            snaps[-1]["hid"] = step.hid.clone()
        elif name == "argmax":
            snaps.append({"idx": step.idx.clone(), "val": step.val.clone(), "final": step.hid.clone()})

    step.run(hook=hook)
    torch.cuda.synchronize()
    for l, L in enumerate(cfg.layers):
        s = snaps[l]
        src = s["src"].cpu().numpy()
        q, Sq = oracle.q4_nrm_gemv(oracle._hw(L.Wq), src, L.gamma_in, cfg.eps)
        check(to_np(s["q"]), q, Sq, what="layer %d q" % l)
        ka, Ska, kb, Skb = oracle.q4_dual_gemv(oracle._hw(L.Wk), oracle._hw(L.Wv), src, L.gamma_in, cfg.eps)
        check(to_np(s["k"]), ka, Ska, what="layer %d k" % l)
        check(to_np(s["v"]), kb, Skb, what="layer %d v" % l)
        ho, So = oracle.q4_res_gemv(oracle._hw(L.Wo), L.attn, src)
        check_residual(to_np(s["hid_o"]), ho, So, what="layer %d o" % l)
        _, g, Sg, u, Su = oracle.q4_gus_nrm(oracle._hw(L.Wg), oracle._hw(L.Wu), s["hid_o"].cpu().numpy(),
                                            L.gamma_post, cfg.eps)
        check_swiglu(to_np(s["h"]), g, Sg, u, Su, what="layer %d gus" % l)
        hd, Sd = oracle.q4_res_gemv(oracle._hw(L.Wd), s["h"].cpu().numpy(), s["hid_o"].cpu().numpy())
        check_residual(to_np(s["hid"]), hd, Sd, what="layer %d down" % l)
    fin = snaps[-1]
    _, lref, Sl = oracle.q4_argmax(oracle._hw(cfg.Wlogits), fin["final"].cpu().numpy(), cfg.gamma_final, cfg.eps)
    check_argmax(fin["idx"].cpu().numpy(), lref, what="decode argmax")
    assert abs(float(fin["val"][0]) - lref[0].max()) <= 1e-3 * Sl[0].max() + 1e-6

    # the captured graph the benchmark replays gives the same bits as the
    # eager run checked above
    g = step.capture()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(step.idx, fin["idx"]) and torch.equal(step.val, fin["val"])
    assert torch.equal(step.hid, fin["final"])


def test_decode_step_with_attention_teacher_forced(q4):
    """The real step (decode attention between K+V and the o projection, over
    each layer's KV cache) at the workload's widths -- 2048 = 32 heads x 64,
    512 = 8 kv heads x 64 -- with 1000 cached positions, layer by layer
    against the oracle on the GPU's own inputs."""
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    spec = wl.AttnSpec(max_seq=1024, position=1000)
    cfg = wl.cfg4(seed=16, layers=2)
    caches = wl.draw_kv_caches(16, 2, spec)
    step = DecodeStep(cfg, attention=(spec, caches))
    snaps = []

    def hook(name, l):
        if name == "q":
            snaps.append({"src": (step.x_in if l == 0 else step.hid).clone(), "q": step.q.clone()})
        elif name == "kv":
            snaps[-1].update(k=step.k.clone(), v=step.v.clone())
        elif name == "attn":
            snaps[-1]["attn"] = step.att.clone()
        elif name == "o":
            snaps[-1]["hid_o"] = step.hid.clone()
        elif name == "gus":
            snaps[-1]["h"] = step.h.clone()
        elif name == "down":
            snaps[-1]["hid"] = step.hid.clone()
        elif name == "argmax":
            snaps.append({"idx": step.idx.clone(), "final": step.hid.clone()})

    step.run(hook=hook)
    torch.cuda.synchronize()
    assert step.n_kernels == 6 * 2 + 2
    cosv, sinv = oracle.rope_table(spec.max_seq, spec.head_dim, spec.rope_theta)
    for l, L in enumerate(cfg.layers):
        s = snaps[l]
        src = s["src"].cpu().numpy()
        q, Sq = oracle.q4_nrm_gemv(oracle._hw(L.Wq), src, L.gamma_in, cfg.eps)
        check(to_np(s["q"]), q, Sq, what="attn step layer %d q" % l)
        ka, Ska, kb, Skb = oracle.q4_dual_gemv(oracle._hw(L.Wk), oracle._hw(L.Wv), src, L.gamma_in, cfg.eps)
        check(to_np(s["k"]), ka, Ska, what="attn step layer %d k" % l)
        check(to_np(s["v"]), kb, Skb, what="attn step layer %d v" % l)
        ar, Sa, kc2, vc2 = oracle.layer_attention(to_np(s["q"]), to_np(s["k"]), to_np(s["v"]), caches[l][0],
                                                  caches[l][1], spec, cosv, sinv)
        check(to_np(s["attn"]), ar, Sa, what="attn step layer %d attention" % l)
        kd, vd = step.caches[l][0].cpu().numpy(), step.caches[l][1].cpu().numpy()
        assert np.array_equal(vd[:, spec.position], vc2[:, spec.position])
        assert np.allclose(kd[:, spec.position], kc2[:, spec.position], rtol=1e-5, atol=1e-5)
        assert np.array_equal(kd[:, :spec.position], caches[l][0][:, :spec.position])
        ho, So = oracle.q4_res_gemv(oracle._hw(L.Wo), s["attn"].cpu().numpy(), src)
        check_residual(to_np(s["hid_o"]), ho, So, what="attn step layer %d o" % l)
        _, g, Sg, u, Su = oracle.q4_gus_nrm(oracle._hw(L.Wg), oracle._hw(L.Wu), s["hid_o"].cpu().numpy(),
                                            L.gamma_post, cfg.eps)
        check_swiglu(to_np(s["h"]), g, Sg, u, Su, what="attn step layer %d gus" % l)
        hd, Sd = oracle.q4_res_gemv(oracle._hw(L.Wd), s["h"].cpu().numpy(), s["hid_o"].cpu().numpy())
        check_residual(to_np(s["hid"]), hd, Sd, what="attn step layer %d down" % l)
    fin = snaps[-1]
    _, lref, _ = oracle.q4_argmax(oracle._hw(cfg.Wlogits), fin["final"].cpu().numpy(), cfg.gamma_final, cfg.eps)
    check_argmax(fin["idx"].cpu().numpy(), lref, what="attn step argmax")
    # the captured graph gives the same bits (the appended rows are rewritten
    # with the same values)
    g = step.capture()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(step.idx, fin["idx"]) and torch.equal(step.hid, fin["final"])


@pytest.mark.parametrize("fmt,window", [("q4_0", 0), ("affine", 40), ("q8_0", 0), ("q4_k", 17), ("q1", 0)])
def test_decode_step_with_attention_every_format(q4, fmt, window):
    """The real step at small widths (4 heads / 2 kv heads of 64) in every
    weight format, with and without a sliding window: its final hidden state
    and argmax against the oracle's real step (not teacher-forced: two layers
    stay well inside the tolerance scale)."""
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    spec = wl.AttnSpec(heads=4, kv_heads=2, head_dim=64, max_seq=128, position=100, window=window)
    cfg = wl.cfg4(seed=17, layers=2, hidden=256, kv=128, inter=512, vocab=500, nb=1, fmt=fmt)
    caches = wl.draw_kv_caches(17, 2, spec)
    step = DecodeStep(cfg, attention=(spec, caches))
    step.run()
    torch.cuda.synchronize()
    idx_ref, lref, hid_ref = oracle.decode_step(cfg, attention=(spec, caches))
    check_argmax(step.idx.cpu().numpy(), lref, what="real step %s argmax" % fmt)
    assert np.allclose(to_np(step.hid), hid_ref, rtol=2e-3, atol=2e-3), "real step %s hidden state" % fmt


def test_fused_decode_step_with_attention_teacher_forced(q4):
    """The real step as one persistent kernel (q4_decode_step_attn: each
    layer's attention a job of the kernel) at the workload's widths -- 32 / 8
    heads of 64 -- over 1000 cached positions, layer by layer: running it on
    the first L layers leaves layer L-1's q, k, v, attention output and h, so
    each is checked against the oracle on the GPU's own inputs of that layer.
    Then the argmax, a graph replay (same bits) and the call-by-call real
    step."""
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    spec = wl.AttnSpec(max_seq=1024, position=1000)
    cfg = wl.cfg4(seed=18, layers=2)
    caches = wl.draw_kv_caches(18, 2, spec)
    step = DecodeStep(cfg, attention=(spec, caches))
    assert step.step_att is not None
    cosv, sinv = oracle.rope_table(spec.max_seq, spec.head_dim, spec.rope_theta)
    prev = cfg.x.astype(np.float64)
    for L in range(1, len(cfg.layers) + 1):
        step.run_fused(n_layers=L)
        q4.q4_decode_check(step.check_ws)
        lay = cfg.layers[L - 1]
        tag = "fused real step layer %d" % (L - 1)
        q, Sq = oracle.q4_nrm_gemv(oracle._hw(lay.Wq), prev, lay.gamma_in, cfg.eps)
        check(to_np(step.q), q, Sq, what=tag + " q")
        ka, Ska, kb, Skb = oracle.q4_dual_gemv(oracle._hw(lay.Wk), oracle._hw(lay.Wv), prev, lay.gamma_in, cfg.eps)
        check(to_np(step.k), ka, Ska, what=tag + " k")
        check(to_np(step.v), kb, Skb, what=tag + " v")
        ar, Sa, kc2, vc2 = oracle.layer_attention(to_np(step.q), to_np(step.k), to_np(step.v), caches[L - 1][0],
                                                  caches[L - 1][1], spec, cosv, sinv)
        check(to_np(step.att), ar, Sa, what=tag + " attention")
        kd, vd = step.caches[L - 1][0].cpu().numpy(), step.caches[L - 1][1].cpu().numpy()
        assert np.array_equal(vd[:, spec.position], vc2[:, spec.position])
        assert np.allclose(kd[:, spec.position], kc2[:, spec.position], rtol=1e-5, atol=1e-5)
        assert np.array_equal(kd[:, :spec.position], caches[L - 1][0][:, :spec.position])
        hid_o, So = oracle.q4_res_gemv(oracle._hw(lay.Wo), to_np(step.att), prev)
        _, g, Sg, u, Su = oracle.q4_gus_nrm(oracle._hw(lay.Wg), oracle._hw(lay.Wu), hid_o, lay.gamma_post, cfg.eps)
        check_swiglu(to_np(step.h), g, Sg, u, Su, what=tag + " gus")
        hid_ref, Sd = oracle.q4_res_gemv(oracle._hw(lay.Wd), to_np(step.h), hid_o)
        bound_extra = 1e-3 * So + 2.0 ** -22 * np.abs(hid_ref)
        check(to_np(step.hid), hid_ref, Sd, extra=bound_extra, what=tag + " hid")
        prev = to_np(step.hid)
    _, lref, Sl = oracle.q4_argmax(oracle._hw(cfg.Wlogits), prev, cfg.gamma_final, cfg.eps)
    check_argmax(step.idx.cpu().numpy(), lref, what="fused real step argmax")
    assert abs(float(step.val[0]) - lref[0].max()) <= 1e-3 * Sl[0].max() + 1e-6
    fused_idx, fused_hid = step.idx.clone(), step.hid.clone()
    g = step.capture(fused=True)
    g.replay()
    torch.cuda.synchronize()
    q4.q4_decode_check(step.check_ws)
    assert torch.equal(step.idx, fused_idx) and torch.equal(step.hid, fused_hid)
    step.run()
    torch.cuda.synchronize()
    assert float((step.hid - fused_hid).abs().max()) <= 1e-4 * float(fused_hid.abs().max())


@pytest.mark.parametrize("fmt,window", [("q4_0", 0), ("affine", 40), ("q8_0", 0), ("q4_k", 17), ("q1", 0),
                                        ("q4_0", 1)])
def test_fused_decode_step_with_attention_every_format(q4, fmt, window):
    """The persistent real step at small widths (8 query / 2 kv heads of 64)
    in every weight format, with and without a sliding window: the final
    hidden state and argmax against the oracle's real step, and against the
    call-by-call real step."""
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    spec = wl.AttnSpec(heads=8, kv_heads=2, head_dim=64, max_seq=128, position=100, window=window)
    cfg = wl.cfg4(seed=19, layers=2, hidden=512, kv=128, inter=512, vocab=500, nb=1, fmt=fmt)
    caches = wl.draw_kv_caches(19, 2, spec)
    step = DecodeStep(cfg, attention=(spec, caches))
    step.run_fused()
    q4.q4_decode_check(step.check_ws)
    idx_ref, lref, hid_ref = oracle.decode_step(cfg, attention=(spec, caches))
    check_argmax(step.idx.cpu().numpy(), lref, what="fused real step %s argmax" % fmt)
    assert np.allclose(to_np(step.hid), hid_ref, rtol=2e-3, atol=2e-3), "fused real step %s hidden state" % fmt
    fused_hid = step.hid.clone()
    step.run()
    torch.cuda.synchronize()
    assert float((step.hid - fused_hid).abs().max()) <= 1e-4 * float(fused_hid.abs().max())


def test_fused_decode_step_with_attention_rejects(q4):
    """Geometries the persistent form does not take fall back to run()."""
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    spec = wl.AttnSpec(heads=4, kv_heads=2, head_dim=64, max_seq=128, position=100)
    cfg = wl.cfg4(seed=20, layers=1, hidden=256, kv=128, inter=512, vocab=100, nb=1)
    step = DecodeStep(cfg, attention=(spec, wl.draw_kv_caches(20, 1, spec)))
    assert step.step_att is None
    with pytest.raises(ValueError):
        step.run_fused()


def test_fused_decode_step_teacher_forced(q4):
    """The persistent-kernel step, layer by layer: running it on the first L
    layers gives that prefix's hidden state (the same per-layer arithmetic
    for every L), so layer L-1 is checked against the oracle run on the
    GPU's own layer input.  Then the whole step against the call-by-call
    step and the oracle argmax."""
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    cfg = wl.cfg4()
    step = DecodeStep(cfg)
    prev = cfg.x.astype(np.float64)
    for L in range(1, len(cfg.layers) + 1):
        step.run_fused(n_layers=L)
        q4.q4_decode_check(step.step_ws)
        lay = cfg.layers[L - 1]
        ref = oracle.decode_layer(lay, prev, cfg.eps)
        check(to_np(step.q), ref["q"], ref["Sq"], what="fused layer %d q" % (L - 1))
        check(to_np(step.k), ref["k"], ref["Sk"], what="fused layer %d k" % (L - 1))
        check(to_np(step.v), ref["v"], ref["Sv"], what="fused layer %d v" % (L - 1))
        check_swiglu(to_np(step.h), ref["g"], ref["Sg"], ref["u"], ref["Su"], what="fused layer %d gus" % (L - 1))
        # hid = hid_o + Wd h: bound both residual adds with the oracle's scales
        bound_extra = 1e-3 * ref["So"] + 2.0 ** -22 * np.abs(ref["hid"])
        check(to_np(step.hid), ref["hid"], ref["Sd"], extra=bound_extra, what="fused layer %d hid" % (L - 1))
        prev = to_np(step.hid)
    _, lref, Sl = oracle.q4_argmax(oracle._hw(cfg.Wlogits), prev, cfg.gamma_final, cfg.eps)
    check_argmax(step.idx.cpu().numpy(), lref, what="fused argmax")
    assert abs(float(step.val[0]) - lref[0].max()) <= 1e-3 * Sl[0].max() + 1e-6
    fused_idx, fused_hid = step.idx.clone(), step.hid.clone()
    # the captured graph of the fused step gives the same bits
    g = step.capture(fused=True)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(step.idx, fused_idx) and torch.equal(step.hid, fused_hid)
    # and agrees with the call-by-call step
    step.run()
    torch.cuda.synchronize()
    # (different but fixed summation orders: compare on the vector's scale)
    assert float((step.hid - fused_hid).abs().max()) <= 1e-4 * float(fused_hid.abs().max())


def test_fused_decode_step_small_shapes(q4):
    """Ragged shapes and nb > 1 through the persistent kernel, against the
    oracle step."""
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    for (hidden, kv, inter, vocab, nb, layers) in [(256, 64, 384, 1000, 1, 3), (160, 48, 96, 333, 3, 2)]:
        cfg = wl.cfg4(seed=9, layers=layers, hidden=hidden, kv=kv, inter=inter, vocab=vocab, nb=nb)
        step = DecodeStep(cfg)
        step.run_fused()
        q4.q4_decode_check(step.step_ws)
        idx_ref, lref, hid_ref = oracle.decode_step(cfg)
        check_argmax(step.idx.cpu().numpy(), lref, what="small fused argmax")
        assert np.allclose(to_np(step.hid), hid_ref, rtol=2e-3, atol=2e-3)


def _teacher_forced_step(q4, cfg, what):
    """The persistent-kernel step on the first L layers for L = 1..layers:
    layer L-1's outputs against the oracle run on the GPU's own input of that
    layer, then the argmax against the oracle on the GPU's final state.

    Within a layer the down projection is checked on the GPU's own h (the
    kernel keeps the last layer's h): its reference is Wd h_gpu + hid_o, with
    hid_o the oracle's o projection plus residual of the GPU's layer input.
    Checking it on the oracle's h instead would charge the down projection
    with the gate/up error amplified by the SwiGLU, which the per-output
    bound does not cover when activations are carried as one f16 (nb > 4)."""
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    step = DecodeStep(cfg)
    prev = cfg.x.astype(np.float64)
    for L in range(1, len(cfg.layers) + 1):
        step.run_fused(n_layers=L)
        q4.q4_decode_check(step.step_ws)
        ref = oracle.decode_layer(cfg.layers[L - 1], prev, cfg.eps)
        tag = "%s layer %d" % (what, L - 1)
        check(to_np(step.q), ref["q"], ref["Sq"], what=tag + " q")
        check(to_np(step.k), ref["k"], ref["Sk"], what=tag + " k")
        check(to_np(step.v), ref["v"], ref["Sv"], what=tag + " v")
        check_swiglu(to_np(step.h), ref["g"], ref["Sg"], ref["u"], ref["Su"], what=tag + " gus")
        hid_ref, Sd = oracle.q4_res_gemv(oracle._hw(cfg.layers[L - 1].Wd), to_np(step.h), ref["hid_o"])
        bound_extra = 1e-3 * ref["So"] + 2.0 ** -22 * np.abs(hid_ref)
        check(to_np(step.hid), hid_ref, Sd, extra=bound_extra, what=tag + " hid")
        prev = to_np(step.hid)
    _, lref, Sl = oracle.q4_argmax(oracle._hw(cfg.Wlogits), prev, cfg.gamma_final, cfg.eps)
    check_argmax(step.idx.cpu().numpy(), lref, what=what + " argmax")
    rows = np.arange(cfg.x.shape[0])
    best = lref[rows, step.idx.cpu().numpy()]
    assert np.all(np.abs(to_np(step.val) - best) <= 1e-3 * Sl.max(axis=1) + 1e-6), what + " argmax value"
    return step


# (fmt, nb, layers, hidden, kv, inter, vocab): every batch class, every
# format, ragged shapes, and the 32-layer maximum
STEP_CASES = [
    ("affine", 1, 3, 256, 64, 384, 1000),
    ("affine", 3, 2, 160, 48, 96, 333),
    ("q4_0", 5, 2, 256, 64, 384, 1000),
    ("affine", 5, 2, 192, 32, 320, 777),
    ("q4_0", 8, 2, 192, 64, 320, 500),
    ("affine", 8, 2, 256, 64, 384, 1000),
    ("q4_0", 16, 2, 256, 64, 384, 1000),
    ("affine", 16, 2, 160, 48, 224, 333),
    ("q8_0", 1, 2, 256, 64, 384, 1000),
    ("q8_0", 4, 2, 160, 48, 224, 333),
    ("q8_0", 9, 2, 128, 32, 192, 300),
    ("q4_k", 1, 2, 256, 64, 512, 1000),
    ("q4_k", 3, 2, 256, 48, 256, 333),
    ("q4_k", 9, 2, 256, 32, 256, 300),
    ("q1", 1, 2, 256, 64, 384, 1000),
    ("q1", 4, 2, 128, 48, 256, 333),
    ("q1", 9, 2, 128, 32, 128, 300),
    ("q4_0", 1, 32, 128, 32, 192, 300),
    ("affine", 2, 32, 128, 32, 192, 300),
]


@pytest.mark.parametrize("fmt,nb,layers,hidden,kv,inter,vocab", STEP_CASES)
def test_fused_step_every_class_and_format(q4, fmt, nb, layers, hidden, kv, inter, vocab):
    cfg = wl.cfg4(seed=13, layers=layers, hidden=hidden, kv=kv, inter=inter, vocab=vocab, nb=nb, fmt=fmt)
    _teacher_forced_step(q4, cfg, "fused %s nb=%d L=%d" % (fmt, nb, layers))


def test_fused_step_full_size_nb5(q4):
    # the workload's shapes (hidden 2048, inter 8192, 65536 logits) with a
    # batch of 5 rows: the one-f16 activation class
    cfg = wl.cfg4(seed=14, layers=2, nb=5)
    _teacher_forced_step(q4, cfg, "fused full nb=5")


@pytest.mark.parametrize("nb", [8, 16])
def test_fused_step_rejects_what_one_cta_cannot_stage(q4, nb):
    # at inter 8192 a batch of 8 or more rows needs more shared memory per
    # CTA than there is: the call says so and launches nothing
    from bit_weight_quantized_q4_gb300.decode import DecodeStep
    cfg = wl.cfg4(seed=15, layers=1, hidden=2048, kv=512, inter=8192, vocab=256, nb=nb)
    step = DecodeStep(cfg)
    with pytest.raises(q4.Q4Error) as e:
        step.run_fused()
    assert e.value.status == 4
