"""One full training step of a decoder stack, driven through librdt.so.

``DecoderTrainer`` owns the device-resident state in a few flat buffers:

* ``w``  fp32 master weights of every trainable tensor, laid out as
  [block 0 | block 1 | ... | block L-1 | final-norm gain | LM head], each
  block in the library's block layout (``rdt.block_param_offsets``);
* ``wb`` the bf16 shadow of ``w`` (GEMM operands), refreshed by AdamW;
* ``g``, ``m``, ``v`` the gradients and AdamW moments, same layout.

A step is: every block forward (saving its activations), the fused final
norm + LM head + cross-entropy (forward and backward), every block backward
in reverse, one squared sum over all gradients, the clip scale, and one AdamW
launch over all parameters.

Activation checkpointing (``checkpoint_segments`` = n > 0; the segmented
recompute of cuda_trainer.rs, ``recompute_segment`` and the saved-layer mask
of ``CudaTransformerTrainer::new``): the layers form n segments of
ceil(L / n); activations are held for one segment only. Every layer input
h[l] is kept, so the backward of a segment first re-runs that segment's block
forwards from their inputs (the last segment's are still current from the
forward pass), then runs its block backwards in reverse. The kernels are
deterministic, so the gradients are bit-identical to the step without
checkpointing.

Gradient accumulation (``accumulation_steps`` = n > 1; cuda_trainer.rs
R-038 / ``GpuGradientAccumulator``, loss scale 1/seq_len/accumulation_steps in
``train_step_inner``): a step takes n micro-batches of the shape's tokens;
each runs forward and backward with the CE loss scaled by 1/(T n), the
gradient producers adding into ``g`` after the first; the clip's squared sum
is taken from the accumulated values on the last micro-batch, then one AdamW.

Device embedding (``embedding=True``; cuda_trainer.rs ``gpu_forward`` lookup and
``embed_backward``, C-EMBED-GRAD-001, both moved from the host to the GPU): the
step takes token ids; x = E[ids] by a gather kernel; the activation gradient
leaving the first block is clipped by its own norm and scatter-added into the
table's gradient (deterministically, in token order); the table has its own
AdamW, outside the global clip.

CUDA graph (``train_step_graph``): the whole step (every micro-batch, the clip
and AdamW) is captured once into one graph that reads its inputs from the
trainer's staging buffers and is replayed each step; the optimizer's step
count lives on the device (``rdt_step_advance``), so the replayed graph needs
no host-side update. The loss partials stay on the device until the
caller reads them. Every launch is a librdt kernel; torch is used only to
allocate buffers and for the stream.
"""
from __future__ import annotations

import torch

from . import rdt
from .synth import OPTIM, DecoderShape


def _align(n: int, a: int = 64) -> int:
    return (n + a - 1) // a * a


class DecoderTrainer:
    def __init__(self, shape: DecoderShape, device="cuda", optim=None, checkpoint_segments=0,
                 accumulation_steps=1, embedding=False):
        self.shape = s = shape
        self.accumulation_steps = n_acc = max(1, int(accumulation_steps))
        self.device = torch.device(device)
        self.optim = dict(OPTIM if optim is None else optim)
        self.cfg = rdt.Config.from_shape(s)
        rdt.check_config(self.cfg)
        self.per_block = rdt.block_param_count(self.cfg)
        self.offsets = rdt.block_param_offsets(self.cfg)
        L, H, V, T = s.layers, s.hidden, s.vocab, s.tokens
        self.off_gf = L * self.per_block
        self.off_lm = self.off_gf + _align(H)
        self.n_params = self.off_lm + V * H
        dev = self.device
        f32 = dict(dtype=torch.float32, device=dev)
        self.w = torch.zeros(self.n_params, **f32)
        self.wb = torch.zeros(self.n_params, dtype=torch.bfloat16, device=dev)
        self.g = torch.zeros(self.n_params, **f32)
        self.m = torch.zeros(self.n_params, **f32)
        self.v = torch.zeros(self.n_params, **f32)
        self.saved_bytes = rdt.block_saved_bytes(self.cfg, s.batch, s.seq)
        self.checkpoint_segments = int(checkpoint_segments)
        if self.checkpoint_segments > 0:
            self.segment_size = -(-L // min(self.checkpoint_segments, L))
        else:
            self.segment_size = L
        self.saved = torch.empty(self.segment_size * self.saved_bytes, dtype=torch.uint8,
                                 device=dev)
        self.h = torch.empty((L + 1, T, H), **f32)
        # output of the recomputed block forwards (equal to h[l + 1]; never read)
        self.h_rc = torch.empty((T, H), **f32) if self.checkpoint_segments > 0 else None
        self.dh = torch.empty((T, H), **f32)
        self.block_ws = torch.empty(rdt.block_workspace_bytes(self.cfg, s.batch, s.seq),
                                    dtype=torch.uint8, device=dev)
        self.head_ws = torch.empty(rdt.head_workspace_bytes(self.cfg, T), dtype=torch.uint8,
                                   device=dev)
        self.sumsq = torch.zeros(1, dtype=torch.float64, device=dev)
        self.scale = torch.ones(1, **f32)
        self.nonfinite = torch.zeros(1, dtype=torch.int32, device=dev)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)  # AdamW's step count
        self.graph = None
        self.loss_partials = torch.zeros(n_acc * T, **f32)
        self.targets = torch.zeros(T, dtype=torch.int32, device=dev)
        self.embedding = bool(embedding)
        if self.embedding:
            self.emb = torch.zeros((V, H), **f32)
            self.emb_g = torch.zeros((V, H), **f32)
            self.emb_m = torch.zeros((V, H), **f32)
            self.emb_v = torch.zeros((V, H), **f32)
            self.ids = torch.zeros(n_acc * T, dtype=torch.int32, device=dev)
            self.emb_ws = torch.empty(rdt.embedding_workspace_bytes(T), dtype=torch.uint8,
                                      device=dev)
            self.emb_sumsq = torch.zeros(1, dtype=torch.float64, device=dev)
            self.emb_scale = torch.ones(1, **f32)
            self.emb_nonfinite = torch.zeros(1, dtype=torch.int32, device=dev)
            # rdt_sq_sum_noalloc looks up the device address of its static
            # scratch on its first call on a device; make that call now, on
            # the trainer's device, so that no later call (a captured step's)
            # does it
            with torch.cuda.device(dev):
                rdt.sq_sum_noalloc([self.emb_scale], self.emb_sumsq)
        self.step_count = 0

    # -------------------------------------------------------------- views
    def block_slice(self, buf, layer):
        return buf[layer * self.per_block:(layer + 1) * self.per_block]

    def tensor(self, buf, layer, name):
        """View of one trainable tensor inside a flat buffer (shape [out, in] or [n])."""
        s = self.shape
        if layer == "head":
            if name == "g_final":
                return buf[self.off_gf:self.off_gf + s.hidden]
            if name == "w_lm":
                return buf[self.off_lm:self.off_lm + s.vocab * s.hidden].view(s.vocab, s.hidden)
            raise KeyError(name)
        off, cnt = self.offsets[name]
        base = layer * self.per_block + off
        flat = buf[base:base + cnt]
        from .synth import block_shapes
        return flat.view(block_shapes(s)[name])

    def saved_slice(self, layer):
        """Activation slot of a layer: its own without checkpointing, else its
        position within its segment."""
        slot = layer % self.segment_size
        return self.saved[slot * self.saved_bytes:(slot + 1) * self.saved_bytes]

    # ------------------------------------------------------------- set-up
    def load(self, blocks, head, emb=None):
        """Copy parameter dicts (from ``synth``) into the flat masters and cast
        the bf16 shadow; emb: the embedding table [V, H] (device embedding)."""
        for li, p in enumerate(blocks):
            for name, t in p.items():
                self.tensor(self.w, li, name).copy_(t)
        for name, t in head.items():
            self.tensor(self.w, "head", name).copy_(t)
        if emb is not None:
            self.emb.copy_(emb)
        self.refresh_shadow()

    def init_random(self, seed=0, std=0.02):
        """Random-init on the device: matrices ~N(0, std), gains 1 (same
        distribution as ``synth``, drawn by a device generator)."""
        gen = torch.Generator(device=self.device)
        gen.manual_seed(seed)
        for li in range(self.shape.layers):
            for name in rdt.TENSOR_NAMES:
                t = self.tensor(self.w, li, name)
                if name.startswith("g_"):
                    t.fill_(1.0)
                else:
                    t.normal_(0.0, std, generator=gen)
        self.tensor(self.w, "head", "g_final").fill_(1.0)
        self.tensor(self.w, "head", "w_lm").normal_(0.0, std, generator=gen)
        if self.embedding:
            # rows ~N(0, 1): the looked-up hidden states have the workloads' statistics
            self.emb.normal_(0.0, 1.0, generator=gen)
        self.refresh_shadow()

    def refresh_shadow(self):
        rdt.cast_bf16(self.w, self.wb)

    def reset_optimizer(self):
        self.m.zero_()
        self.v.zero_()
        self.step_dev.zero_()
        if self.embedding:
            self.emb_m.zero_()
            self.emb_v.zero_()
        self.step_count = 0

    # --------------------------------------------------------------- step
    def forward_backward(self, x=None, targets=None, micro=0, ids=None):
        """Forward, fused CE and full backward of one (micro-)batch; gradients
        land in ``self.g`` (added to it for micro > 0). x [T, H] fp32 and
        targets [T] int32 on the device (or already copied into ``self.h[0]``
        / ``self.targets`` when None)."""
        s, cfg = self.shape, self.cfg
        n = self.accumulation_steps
        acc = micro > 0
        sq = self.sumsq if micro == n - 1 else None
        T = s.tokens
        if ids is not None:
            self.ids[micro * T:(micro + 1) * T].copy_(ids)
        if self.embedding:
            rdt.embedding_forward(self.emb, self.ids[micro * T:(micro + 1) * T], self.h[0])
        elif x is not None:
            self.h[0].copy_(x)
        if targets is not None:
            self.targets.copy_(targets)
        for li in range(s.layers):
            rdt.block_forward(cfg, s.batch, s.seq, self.block_slice(self.w, li),
                              self.block_slice(self.wb, li), self.h[li], self.h[li + 1],
                              self.saved_slice(li), self.block_ws)
        rdt.fused_cross_entropy(cfg, T, self.h[s.layers], self.tensor(self.w, "head", "g_final"),
                                self.tensor(self.wb, "head", "w_lm"), self.targets,
                                1.0 / (T * n), self.loss_partials[micro * T:(micro + 1) * T],
                                self.dh, self.tensor(self.g, "head", "g_final"),
                                self.tensor(self.g, "head", "w_lm"), self.head_ws,
                                grad_sq=sq, accumulate=acc)
        L, seg = s.layers, self.segment_size
        nseg = -(-L // seg)
        for k in reversed(range(nseg)):
            lo, hi = k * seg, min(L, (k + 1) * seg)
            if k != nseg - 1:
                # recompute this segment's activations from the kept layer inputs
                for li in range(lo, hi):
                    rdt.block_forward(cfg, s.batch, s.seq, self.block_slice(self.w, li),
                                      self.block_slice(self.wb, li), self.h[li], self.h_rc,
                                      self.saved_slice(li), self.block_ws)
            for li in reversed(range(lo, hi)):
                rdt.block_backward(cfg, s.batch, s.seq, self.block_slice(self.w, li),
                                   self.block_slice(self.wb, li), self.h[li],
                                   self.saved_slice(li), self.dh, self.dh,
                                   self.block_slice(self.g, li), self.block_ws,
                                   grad_sq=sq, accumulate=acc)
        if self.embedding:
            # C-EMBED-GRAD-001: the activation gradient clipped by its own norm,
            # then scatter-added into the table's gradient
            rdt.sq_sum_noalloc([self.dh], self.emb_sumsq)
            rdt.clip_scale(self.emb_sumsq, self.optim["max_norm"], self.emb_scale,
                           self.emb_nonfinite)
            rdt.embedding_backward(self.ids[micro * T:(micro + 1) * T], self.dh, self.emb_g,
                                   self.emb_ws, scale=self.emb_scale, accumulate=acc)
        return self.loss_partials

    def clip_and_update(self):
        """Global-norm clip from the squared sum of every gradient (summed by
        the backward calls into ``self.sumsq`` as they produce the gradients),
        then one AdamW over all parameters (skipped on a non-finite norm)."""
        o = self.optim
        rdt.clip_scale(self.sumsq, o["max_norm"], self.scale, self.nonfinite)
        self.step_count += 1
        rdt.step_advance(self.step_dev)
        rdt.adamw_step(self.w, self.g, self.m, self.v, None, o["lr"], o["beta1"], o["beta2"],
                       o["eps"], o["weight_decay"], scale=self.scale, skip=self.nonfinite,
                       w_bf16=self.wb, step_dev=self.step_dev)
        if self.embedding:
            rdt.adamw_step(self.emb, self.emb_g, self.emb_m, self.emb_v, None, o["lr"],
                           o["beta1"], o["beta2"], o["eps"], o["weight_decay"],
                           skip=self.emb_nonfinite, step_dev=self.step_dev)

    def train_step(self, x=None, targets=None, ids=None):
        """One full step; returns the device tensor of per-token loss partials.
        x: hidden states [n T, H] (or, with the device embedding, ids: int32
        token ids [n T]); targets [n T]: n micro-batches of T tokens, in order
        (n = 1 without accumulation)."""
        n, T = self.accumulation_steps, self.shape.tokens

        def part(a, i):
            return None if a is None else a[i * T:(i + 1) * T]

        for i in range(n):
            self.forward_backward(part(x, i), part(targets, i), micro=i, ids=part(ids, i))
        self.clip_and_update()
        return self.loss_partials

    # --------------------------------------------------------- CUDA graph
    def train_step_graph(self, x=None, targets=None, ids=None):
        """train_step as one CUDA graph replay. The inputs (as for train_step)
        are copied into staging buffers first; the graph is captured on the
        first call, which must follow at least one eager train_step (the
        library's one-time set-up runs there, outside any capture)."""
        n, T = self.accumulation_steps, self.shape.tokens
        if self.graph is None:
            self.tg_stage = torch.zeros(n * T, dtype=torch.int32, device=self.device)
            if not self.embedding:
                self.x_stage = torch.zeros((n * T, self.shape.hidden), dtype=torch.float32,
                                           device=self.device)
            torch.cuda.synchronize(self.device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._staged_step()
            self.graph = g
        if x is not None:
            self.x_stage.copy_(x, non_blocking=True)
        if ids is not None:
            self.ids.copy_(ids, non_blocking=True)
        if targets is not None:
            self.tg_stage.copy_(targets, non_blocking=True)
        self.graph.replay()
        return self.loss_partials

    def _staged_step(self):
        n, T = self.accumulation_steps, self.shape.tokens
        for i in range(n):
            x = None if self.embedding else self.x_stage[i * T:(i + 1) * T]
            self.forward_backward(x, self.tg_stage[i * T:(i + 1) * T], micro=i)
        self.clip_and_update()
        return self.loss_partials
