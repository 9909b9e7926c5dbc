"""Adapters-only training step of the NF4-frozen block with LoRA adapters,
driven through librdt.so (the CudaNf4TransformerBlock of the aprender-train
cuda_block.rs page, with lora_scale = alpha / rank as in cuda_trainer.rs).

``Nf4LoraTrainer`` owns the device-resident state:

* ``codes`` / ``scales`` the frozen projections as packed 4-bit NormalFloat
  codes and one fp32 scale per 64 weights (``rdt.nf4_offsets`` layout),
  ``gains`` the frozen norm gains;
* ``lora`` the fp32 adapter masters (``rdt.lora_param_offsets`` layout),
  ``shadow`` their bf16 operand copy, ``g``, ``m``, ``v`` the adapter
  gradients and AdamW moments.

A step is the block forward, the block backward (adapter gradients only), the
squared sum of the adapter gradients, the clip scale, AdamW over the adapters
and the shadow refresh. Every launch is a librdt kernel; torch only allocates
buffers and supplies the stream.
"""
from __future__ import annotations

import torch

from . import rdt
from .synth import LORA, NF4_PROJECTIONS, OPTIM, DecoderShape


class Nf4LoraTrainer:
    def __init__(self, shape: DecoderShape, rank=None, alpha=None, device="cuda", optim=None):
        self.shape = s = shape
        self.rank = int(rank or LORA["rank"])
        self.alpha = float(alpha if alpha is not None else LORA["alpha"])
        self.device = dev = torch.device(device)
        self.optim = dict(OPTIM if optim is None else optim)
        self.cfg = rdt.Config.from_shape(s)
        rdt.nf4_check(self.cfg, self.rank)
        n_codes, n_scales = rdt.nf4_sizes(self.cfg)
        self.nf4_offsets = rdt.nf4_offsets(self.cfg)
        self.lora_offsets = rdt.lora_param_offsets(self.cfg, self.rank)
        self.n_params = rdt.lora_param_count(self.cfg, self.rank)
        f32 = dict(dtype=torch.float32, device=dev)
        self.codes = torch.zeros(n_codes, dtype=torch.uint8, device=dev)
        self.scales = torch.zeros(n_scales, **f32)
        self.gains = torch.ones(2 * s.hidden + 2 * s.head_dim, **f32)
        self.lora = torch.zeros(self.n_params, **f32)
        self.shadow = torch.zeros(rdt.lora_shadow_count(self.cfg, self.rank),
                                  dtype=torch.bfloat16, device=dev)
        self.g = torch.zeros(self.n_params, **f32)
        self.m = torch.zeros(self.n_params, **f32)
        self.v = torch.zeros(self.n_params, **f32)
        self.saved = torch.empty(rdt.nf4_saved_bytes(self.cfg, self.rank, s.batch, s.seq),
                                 dtype=torch.uint8, device=dev)
        self.ws = torch.empty(rdt.nf4_workspace_bytes(self.cfg, self.rank, s.batch, s.seq),
                              dtype=torch.uint8, device=dev)
        self.y = torch.empty((s.tokens, s.hidden), **f32)
        self.dx = torch.empty((s.tokens, s.hidden), **f32)
        self.sumsq = torch.zeros(1, dtype=torch.float64, device=dev)
        self.scale = torch.ones(1, **f32)
        self.nonfinite = torch.zeros(1, dtype=torch.int32, device=dev)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)  # AdamW's step count
        self.step_count = 0
        self.graph = None
        # rdt_sq_sum_noalloc looks up the device address of its static
        # scratch on its first call on a device; make that call now, on the
        # trainer's device, so that no later call (a captured step's) does it
        with torch.cuda.device(dev):
            rdt.sq_sum_noalloc([self.scale], self.sumsq)

    # ------------------------------------------------------------- views
    def adapter(self, name):
        """View of one adapter tensor of ``lora`` (A: [rank, in], B: [out, rank])."""
        return self.tensor(self.lora, name)

    def tensor(self, buf, name):
        from .synth import block_shapes
        out, inn = block_shapes(self.shape)["w" + name[2:]]
        o, c = self.lora_offsets[name]
        return buf[o:o + c].view((self.rank, inn) if name.startswith("a_") else (out, self.rank))

    # ------------------------------------------------------------ set-up
    def load(self, base, gains, lora):
        """Copy the ``synth.draw_nf4_block`` dicts into the device buffers."""
        for name in NF4_PROJECTIONS:
            co, so = self.nf4_offsets[name]
            packed, absmax = base[name]
            self.codes[co:co + packed.numel()].copy_(packed.reshape(-1))
            self.scales[so:so + absmax.numel()].copy_(absmax.reshape(-1))
        s = self.shape
        parts = [gains[k].reshape(-1) for k in ("g_attn", "g_ffn", "g_q", "g_k")]
        self.gains.copy_(torch.cat(parts).to(self.device))
        for name, t in lora.items():
            self.adapter(name).copy_(t)
        self.refresh_shadow()
        assert self.gains.numel() == 2 * s.hidden + 2 * s.head_dim

    def init_random(self, seed=0, b_std=0.0):
        """The workload's distributions drawn on the device: codes uniform over
        all bytes (two uniform 4-bit codes each), scales 3|N(0, 0.02)|, gains 1,
        A ~ N(0, 0.02), B = 0 (or N(0, b_std))."""
        gen = torch.Generator(device=self.device)
        gen.manual_seed(seed)
        self.codes.copy_(torch.randint(0, 256, self.codes.shape, generator=gen,
                                       device=self.device, dtype=torch.int32).to(torch.uint8))
        self.scales.normal_(0.0, 0.02, generator=gen).abs_().mul_(3.0)
        self.gains.fill_(1.0)
        for name in rdt.LORA_NAMES:
            t = self.adapter(name)
            if name.startswith("a_"):
                t.normal_(0.0, 0.02, generator=gen)
            elif b_std > 0:
                t.normal_(0.0, b_std, generator=gen)
            else:
                t.zero_()
        self.refresh_shadow()

    def refresh_shadow(self):
        rdt.lora_shadow(self.cfg, self.rank, self.lora, self.shadow)

    # -------------------------------------------------------------- step
    def forward_backward(self, x, dy):
        """Block forward and backward: y, dx and the adapter gradients g."""
        s = self.shape
        rdt.nf4_block_forward(self.cfg, self.rank, self.alpha, s.batch, s.seq, self.codes,
                              self.scales, self.gains, self.shadow, x, self.y, self.saved,
                              self.ws)
        rdt.nf4_block_backward(self.cfg, self.rank, self.alpha, s.batch, s.seq, self.codes,
                               self.scales, self.gains, self.shadow, x, self.saved, dy, self.dx,
                               self.g, self.ws)

    def clip_and_update(self):
        """Squared sum of the adapter gradients, clip scale, AdamW over the
        adapters, shadow refresh."""
        o = self.optim
        self.step_count += 1
        rdt.sq_sum_noalloc([self.g], self.sumsq)
        rdt.clip_scale(self.sumsq, o["max_norm"], self.scale, self.nonfinite)
        rdt.step_advance(self.step_dev)
        rdt.adamw_step(self.lora, self.g, self.m, self.v, None, o["lr"], o["beta1"],
                       o["beta2"], o["eps"], o["weight_decay"], scale=self.scale,
                       skip=self.nonfinite, step_dev=self.step_dev)
        self.refresh_shadow()

    def train_step(self, x, dy):
        """One adapters-only step on input x and upstream gradient dy (fp32
        [tokens, hidden], on the device). Returns the block output y."""
        self.forward_backward(x, dy)
        self.clip_and_update()
        return self.y

    def train_step_graph(self, x=None, dy=None):
        """train_step as one CUDA graph replay: x and dy (when given) are
        copied into staging buffers, then the step captured on the first call
        (which must follow an eager train_step) replays."""
        if self.graph is None:
            self.x_stage = torch.zeros_like(self.y)
            self.dy_stage = torch.zeros_like(self.y)
            torch.cuda.synchronize(self.device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.forward_backward(self.x_stage, self.dy_stage)
                self.clip_and_update()
            self.graph = g
        if x is not None:
            self.x_stage.copy_(x, non_blocking=True)
        if dy is not None:
            self.dy_stage.copy_(dy, non_blocking=True)
        self.graph.replay()
        return self.y
