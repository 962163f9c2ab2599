"""The synthetic Q4 decode step: per layer RMSNorm + q projection, dual K/V,
o projection + residual (its input an attention stand-in), RMSNorm + gate/up
+ SwiGLU, down + residual; then a final RMSNorm, the logits projection and
the greedy argmax.

Two ways to run it, same arithmetic per call:
* ``run_fused()``: one ``q4_decode_step`` call -- a single persistent kernel
  whose jobs are separated by grid-wide barriers while the weight stream runs
  ahead across them (the benchmark's step); with ``attention``, one
  ``q4_decode_step_attn`` call, the layers' attention as jobs of the kernel;
* ``run()``: the individual library calls (82 kernels for 16 layers) on one
  stream, e.g. captured as a CUDA graph.

The step order is the fused decode path of honeycrisp/mod.rs
(forward_decode_fused_layers: one command buffer per step) with the final
logits projection and greedy argmax of Module gpu (module sampling).  The
attention output is replaced by a fixed seeded vector per layer, so the q, k
and v projections are computed and stored but not consumed -- unless the
step is built with ``attention`` (a ``q4_workloads.AttnSpec`` and per-layer KV
caches): then ``run()`` adds each layer's decode attention (``q4_attn_decode``:
RoPE, append, softmax(q K^T) V over the layer's caches, q/k/v read as heads)
between the K+V and the o projection, which takes its output: the real step.

Kernels per step: 5 per layer + 2 for the argmax (82 for 16 layers), one more
per layer with attention.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import DecodeLayers, Q4Weight, StepAttention, lib, q4_argmax, q4_argmax_workspace_bytes, q4_attn_decode, \
    q4_decode_attn_workspace_bytes, q4_decode_step, q4_decode_step_attn, q4_decode_workspace_bytes, q4_dual_gemv, \
    q4_gus_nrm, q4_nrm_gemv, q4_res_gemv, rope_table


@dataclass
class DeviceLayer:
    gamma_in: torch.Tensor
    Wq: Q4Weight
    Wk: Q4Weight
    Wv: Q4Weight
    Wo: Q4Weight
    attn: torch.Tensor
    gamma_post: torch.Tensor
    Wg: Q4Weight
    Wu: Q4Weight
    Wd: Q4Weight


KERNELS_PER_LAYER = 5
KERNELS_FINAL = 2


class DecodeStep:
    """Device-resident weights and activation buffers of one decode step.

    ``cfg`` is a ``q4_workloads.Cfg4`` (host weights).  ``x_in`` holds the
    step input; after ``run()`` (or a graph replay) ``idx`` / ``val`` hold
    the argmax and ``hid`` the final hidden state."""

    def __init__(self, cfg, device="cuda", attention=None):
        T = lambda a: torch.from_numpy(a.copy()).to(device)
        W = lambda H: (Q4Weight.from_q8_0(H.blocks8, H.n, H.k, device) if hasattr(H, "blocks8")
                       else Q4Weight.from_q4_k(H.blocks_k, H.n, H.k, device) if hasattr(H, "blocks_k")
                       else Q4Weight.from_q1(H.blocks1, H.n, H.k, device) if hasattr(H, "blocks1")
                       else Q4Weight.from_q4_0(H.blocks, H.n, H.k, device) if hasattr(H, "blocks")
                       else Q4Weight.from_affine(H.nib, H.s, H.m, H.n, H.k, device))
        self.eps = float(cfg.eps)
        nb, hidden = cfg.x.shape
        # the step's inputs -- x and every layer's attention stand-in -- in one
        # device buffer, so that a caller brings them in with one copy
        self.inputs = torch.from_numpy(np.concatenate([cfg.x.reshape(-1)] + [L.attn.reshape(-1) for L in cfg.layers])
                                       .astype(np.float32)).to(device)
        rows = lambda i: self.inputs[i * nb * hidden:(i + 1) * nb * hidden].view(nb, hidden)
        self.layers = [DeviceLayer(T(L.gamma_in), W(L.Wq), W(L.Wk), W(L.Wv), W(L.Wo), rows(1 + l),
                                   T(L.gamma_post), W(L.Wg), W(L.Wu), W(L.Wd)) for l, L in enumerate(cfg.layers)]
        self.gamma_final = T(cfg.gamma_final)
        self.Wlogits = W(cfg.Wlogits)
        L0 = self.layers[0]
        f32 = dict(dtype=torch.float32, device=device)
        self.nb, self.hidden = nb, hidden
        self.x_in = rows(0)
        self.hid = torch.empty((nb, hidden), **f32)
        self.q = torch.empty((nb, L0.Wq.n), **f32)
        self.k = torch.empty((nb, L0.Wk.n), **f32)
        self.v = torch.empty((nb, L0.Wv.n), **f32)
        self.h = torch.empty((nb, L0.Wg.n), **f32)
        # the step's results -- the argmax indices, then (16-byte aligned) their
        # logits -- in one device buffer, read back with one copy
        self.results = torch.empty(32, dtype=torch.int32, device=device)
        self.idx = self.results[:nb]
        self.val = self.results[16:16 + nb].view(torch.float32)
        self.ws = torch.empty(q4_argmax_workspace_bytes(self.Wlogits.n, nb), dtype=torch.uint8, device=device)
        self.step_ws = torch.empty(q4_decode_workspace_bytes(nb), dtype=torch.uint8, device=device)
        self.descs = DecodeLayers(self.layers)
        # the real step: the attention spec, per-layer device caches, RoPE
        # tables, the attention output and its workspace
        self.attention = None
        if attention is not None:
            spec, caches = attention
            if nb != 1 or spec.heads * spec.head_dim != hidden or spec.kv_heads * spec.head_dim != L0.Wk.n:
                raise ValueError("attention needs nb = 1, heads*head_dim = hidden and kv_heads*head_dim = k width")
            self.attention = spec
            self.caches = [(T(kc), T(vc)) for kc, vc in caches]
            c, sn = rope_table(spec.max_seq, spec.head_dim, spec.rope_theta)
            self.rope = (T(c), T(sn))
            self.att = torch.empty((1, hidden), **f32)
            self.attn_ws = torch.zeros(int(lib().q4_attn_workspace_bytes(spec.heads, spec.head_dim, spec.max_seq)),
                                       dtype=torch.uint8, device=device)
            # the persistent form (run_fused): its attention descriptor and
            # workspace, where its geometry is one the kernel takes
            self.step_att = None
            nbytes = q4_decode_attn_workspace_bytes(spec.heads, spec.kv_heads, spec.head_dim)
            if nbytes:
                self.step_att = StepAttention(self.caches, self.att, spec.position, spec.window, rope=self.rope)
                self.step_att_ws = torch.empty(nbytes, dtype=torch.uint8, device=device)

    @property
    def n_kernels(self) -> int:
        return (KERNELS_PER_LAYER + (self.attention is not None)) * len(self.layers) + KERNELS_FINAL

    @property
    def kv_bytes(self) -> int:
        """Cache bytes the step's attention reads (0 without attention)."""
        a = self.attention
        if a is None:
            return 0
        lo = max(0, a.position + 1 - a.window) if a.window > 0 else 0
        return len(self.layers) * 2 * a.kv_heads * (a.position + 1 - lo) * a.head_dim * 4

    @property
    def weight_bytes(self) -> int:
        b = self.Wlogits.weight_bytes
        for L in self.layers:
            b += sum(w.weight_bytes for w in (L.Wq, L.Wk, L.Wv, L.Wo, L.Wg, L.Wu, L.Wd))
        return b

    def run(self, hook=None, around=None):
        """Enqueue one step.  ``hook(name, layer)`` runs after each call
        (tests use it to snapshot intermediates); ``around(name, layer, fn)``
        may wrap a call (the benchmark brackets one kernel with events)."""
        call = around or (lambda name, l, fn: fn())
        src = self.x_in
        eps = self.eps
        for l, L in enumerate(self.layers):
            call("q", l, lambda: q4_nrm_gemv(L.Wq, src, L.gamma_in, eps, out=self.q))
            hook and hook("q", l)
            call("kv", l, lambda: q4_dual_gemv(L.Wk, L.Wv, src, L.gamma_in, eps, out_a=self.k, out_b=self.v))
            hook and hook("kv", l)
            o_in = L.attn
            a = self.attention
            if a is not None:
                kc, vc = self.caches[l]
                call("attn", l, lambda: q4_attn_decode(
                    self.q.view(a.heads, a.head_dim), self.k.view(a.kv_heads, a.head_dim),
                    self.v.view(a.kv_heads, a.head_dim), kc, vc, a.position, a.window, None, rope=self.rope,
                    out=self.att.view(a.heads, a.head_dim), workspace=self.attn_ws))
                hook and hook("attn", l)
                o_in = self.att
            call("o", l, lambda: q4_res_gemv(L.Wo, o_in, src, out=self.hid))
            hook and hook("o", l)
            call("gus", l, lambda: q4_gus_nrm(L.Wg, L.Wu, self.hid, L.gamma_post, eps, out=self.h))
            hook and hook("gus", l)
            call("down", l, lambda: q4_res_gemv(L.Wd, self.h, self.hid, out=self.hid))
            hook and hook("down", l)
            src = self.hid
        call("argmax", len(self.layers),
             lambda: q4_argmax(self.Wlogits, self.hid, self.gamma_final, eps, workspace=self.ws,
                               idx=self.idx, val=self.val))
        hook and hook("argmax", len(self.layers))

    def run_fused(self, n_layers=None):
        """Enqueue the step as one persistent kernel (the first ``n_layers``
        layers then the logits argmax): with attention, its layers' attention
        as jobs of the kernel (``q4_decode_step_attn``)."""
        if self.attention is not None:
            if self.step_att is None:
                raise ValueError("the persistent step's attention takes head size 64 and four query heads per kv "
                                 "head; run() takes the others")
            q4_decode_step_attn(self.descs, self.step_att, self.Wlogits, self.gamma_final, self.eps, self.x_in,
                                self.hid, self.q, self.k, self.v, self.h, self.idx, self.val, self.step_att_ws,
                                n_layers=n_layers)
            return
        q4_decode_step(self.descs, self.Wlogits, self.gamma_final, self.eps, self.x_in, self.hid, self.q, self.k,
                       self.v, self.h, self.idx, self.val, self.step_ws, n_layers=n_layers)

    @property
    def check_ws(self):
        """The workspace q4_decode_check reads after run_fused()."""
        return self.step_att_ws if self.attention is not None else self.step_ws

    @property
    def n_kernels_fused(self) -> int:
        return 1

    def capture(self, around=None, fused=False) -> torch.cuda.CUDAGraph:
        """Capture one step as a CUDA graph (after one eager warm-up run)."""
        fn = (lambda: self.run_fused()) if fused else (lambda: self.run(around=around))
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run_fused() if fused else self.run()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g
