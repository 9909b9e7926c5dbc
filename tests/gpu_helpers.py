"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare with the FP64 oracle on the same seeded fp32 inputs."""
import numpy as np
import torch

from resident_decoder_trainer_gb300 import build, rdt, synth

# Tolerances. The CUDA path rounds GEMM operands to bf16 (relative error
# 2^-9 per element) and accumulates in fp32; the oracle is fp64 on the fp32
# masters. A chain of ~6 such roundings gives a relative L2 error of a few
# 1e-3 on every output, so:
LOSS_REL = 1e-3      # loss relative error
GRAD_REL_L2 = 1e-2   # per-tensor gradient relative L2 error
FWD_REL_L2 = 1e-2    # block output (y - x) relative L2 error
ADAMW_REL = 1e-5     # AdamW updated weights given identical gradients


def ensure_built():
    build.build()
    rdt.lib()


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / max(den, 1e-300))


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


SQ_START = 0.25  # grad_sq value before a block backward adds its squared sum


def gpu_block(shape, p, x, dy, with_sq=False, fill=None):
    """Block forward + backward on the GPU. p: dict of CPU fp32 tensors.
    with_sq: also return the fused squared sum the backward added to a
    scalar that held SQ_START. fill: a byte value the saved-activation and
    workspace buffers are filled with first, and the workspace again between
    the forward and the backward (default: left uninitialised)."""
    cfg = rdt.Config.from_shape(shape)
    n = rdt.block_param_count(cfg)
    offs = rdt.block_param_offsets(cfg)
    w = torch.zeros(n, dtype=torch.float32, device="cuda")
    for name, (o, c) in offs.items():
        w[o:o + c] = p[name].reshape(-1).to("cuda")
    wb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    rdt.cast_bf16(w, wb)
    saved = torch.empty(rdt.block_saved_bytes(cfg, shape.batch, shape.seq), dtype=torch.uint8,
                        device="cuda")
    ws = torch.empty(rdt.block_workspace_bytes(cfg, shape.batch, shape.seq), dtype=torch.uint8,
                     device="cuda")
    if fill is not None:
        saved.fill_(fill)
        ws.fill_(fill)
    xd = x.to("cuda").contiguous()
    y = torch.empty_like(xd)
    rdt.block_forward(cfg, shape.batch, shape.seq, w, wb, xd, y, saved, ws)
    if fill is not None:
        ws.fill_(fill)  # the backward keeps nothing of the forward's scratch
    dyd = dy.to("cuda").contiguous()
    dx = torch.empty_like(xd)
    grads = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    sq = torch.full((1,), SQ_START, dtype=torch.float64, device="cuda")
    rdt.block_backward(cfg, shape.batch, shape.seq, w, wb, xd, saved, dyd, dx, grads, ws,
                       grad_sq=sq if with_sq else None)
    torch.cuda.synchronize()
    g = {name: grads[o:o + c].view(synth.block_shapes(shape)[name]) for name, (o, c) in
         offs.items()}
    if with_sq:
        return y, dx, g, float(sq)
    return y, dx, g


def gpu_head(shape, h, g_final, w_lm, targets, fill=None):
    """Fused LM-head cross-entropy on the GPU; fill: a byte value the
    workspace is filled with first (default: left uninitialised)."""
    cfg = rdt.Config.from_shape(shape)
    T = h.shape[0]
    hd = h.to("cuda").contiguous()
    gf = g_final.to("cuda").contiguous()
    wl = w_lm.to("cuda").to(torch.bfloat16).contiguous()
    tg = targets.to("cuda").to(torch.int32).contiguous()
    ws = torch.empty(rdt.head_workspace_bytes(cfg, T), dtype=torch.uint8, device="cuda")
    if fill is not None:
        ws.fill_(fill)
    loss = torch.empty(T, dtype=torch.float32, device="cuda")
    dh = torch.empty_like(hd)
    dgf = torch.empty_like(gf)
    dwl = torch.empty(w_lm.shape, dtype=torch.float32, device="cuda")
    sq = torch.full((1,), float("nan"), dtype=torch.float64, device="cuda")
    rdt.fused_cross_entropy(cfg, T, hd, gf, wl, tg, 1.0 / T, loss, dh, dgf, dwl, ws, grad_sq=sq)
    torch.cuda.synchronize()
    gpu_head.last_sq = float(sq)
    return loss, dh, dgf, dwl


def ragged_shape(**kw):
    """Several tiles in every dimension plus ragged tails (S not a multiple of
    64/128, FFN width not a multiple of 128, vocab not a multiple of 256)."""
    base = dict(layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, intermediate=688,
                vocab=1008, seq=200, batch=2, eps=1e-6, theta=1e4)
    base.update(kw)
    return synth.DecoderShape(**base)


def nf4_buffers(shape, rank, base, gains, lora):
    """Device buffers of the NF4 + LoRA block in the library's layouts: codes
    (uint8), scales, gains, lora (fp32) and the bf16 adapter shadow."""
    cfg = rdt.Config.from_shape(shape)
    nc, ns = rdt.nf4_sizes(cfg)
    offs = rdt.nf4_offsets(cfg)
    codes = torch.zeros(nc, dtype=torch.uint8)
    scales = torch.zeros(ns, dtype=torch.float32)
    for name, (co, so) in offs.items():
        packed, absmax = base[name]
        codes[co:co + packed.numel()] = packed.reshape(-1)
        scales[so:so + absmax.numel()] = absmax.reshape(-1)
    g = torch.cat([gains[k].reshape(-1) for k in ("g_attn", "g_ffn", "g_q", "g_k")])
    lo = rdt.lora_param_offsets(cfg, rank)
    lw = torch.zeros(rdt.lora_param_count(cfg, rank), dtype=torch.float32)
    for name, (o, c) in lo.items():
        lw[o:o + c] = lora[name].reshape(-1)
    lw = lw.cuda()
    shadow = torch.empty(rdt.lora_shadow_count(cfg, rank), dtype=torch.bfloat16, device="cuda")
    rdt.lora_shadow(cfg, rank, lw, shadow)
    return cfg, codes.cuda(), scales.cuda(), g.cuda(), lw, shadow


def gpu_nf4_block(shape, rank, alpha, base, gains, lora, x, dy, fill=None):
    """NF4 + LoRA block forward + backward on the GPU: (y, dx, adapter grads
    {name: tensor}, fused squared sum added to SQ_START). fill: a byte value
    the saved-activation and workspace buffers are filled with first, and the
    workspace again between the forward and the backward."""
    cfg, codes, scales, g, lw, shadow = nf4_buffers(shape, rank, base, gains, lora)
    B, S = shape.batch, shape.seq
    saved = torch.empty(rdt.nf4_saved_bytes(cfg, rank, B, S), dtype=torch.uint8, device="cuda")
    ws = torch.empty(rdt.nf4_workspace_bytes(cfg, rank, B, S), dtype=torch.uint8, device="cuda")
    if fill is not None:
        saved.fill_(fill)
        ws.fill_(fill)
    xd = x.to("cuda").contiguous()
    y = torch.empty_like(xd)
    rdt.nf4_block_forward(cfg, rank, alpha, B, S, codes, scales, g, shadow, xd, y, saved, ws)
    if fill is not None:
        ws.fill_(fill)  # the backward keeps nothing of the forward's scratch
    dx = torch.empty_like(xd)
    grads = torch.full_like(lw, float("nan"))
    sq = torch.full((1,), SQ_START, dtype=torch.float64, device="cuda")
    rdt.nf4_block_backward(cfg, rank, alpha, B, S, codes, scales, g, shadow, xd, saved,
                           dy.to("cuda").contiguous(), dx, grads, ws, grad_sq=sq)
    torch.cuda.synchronize()
    out = {name: grads[o:o + c].view(lora[name].shape)
           for name, (o, c) in rdt.lora_param_offsets(cfg, rank).items()}
    return y, dx, out, float(sq)
