"""FP64 CPU oracle for the NF4-frozen block with LoRA adapters.

TEST INFRASTRUCTURE ONLY (same rules as ``oracle.model``): only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs may use it; it shares
no code, table or constant with the CUDA path.

What it computes, and from where (aprender-train docs.rs pages):

* cuda_block.rs (0.32.0) -- ``CudaNf4TransformerBlock``: the seven projection
  weights are frozen and stored as packed 4-bit NF4 codes plus one fp32 scale
  per block of 64 consecutive elements of the row-major [out, in] weight
  (``quantize_nf4(weights, total / NF4_BLOCK_SIZE, NF4_BLOCK_SIZE)``); the
  block is otherwise the fp32 block (QK-norm, RoPE, GQA attention, SwiGLU).
* cuda_trainer.rs (0.34.0) -- ``lora_scale = lora_alpha / lora_rank``.
* wgpu_trainer.rs (0.38.0) -- ``lora_forward``: y = x W^T + (alpha/rank)
  (x A^T) B^T with A [rank, in], B [out, rank].

Readings (the pages leave them open): the 16 NF4 levels are the published
NormalFloat-4 table (QLoRA, Dettmers et al. 2023), typed below and pinned in
the tests against its construction from normal quantiles; a packed byte holds
element 2j in its low nibble and 2j+1 in its high nibble; adapters sit on all
seven projections (the fifth workload), the norm gains are frozen, and only
the adapters are clipped and updated.

Exact in real arithmetic and used here: the LoRA projection equals one
projection with the merged weight W + s B A, so the block is the pinned fp64
block of ``oracle.model`` with merged weights, and the adapter gradients are
the projections of that block's weight gradient dW: dA = s B^T dW,
dB = s dW A^T.
"""
from __future__ import annotations

import numpy as np

from oracle import model as om

# NormalFloat-4 levels (QLoRA), ascending; index = 4-bit code.
NF4_LEVELS = np.array([
    -1.0, -0.6961928009986877, -0.5250730514526367, -0.39491748809814453,
    -0.28444138169288635, -0.18477343022823334, -0.09105003625154495, 0.0,
    0.07958029955625534, 0.16093020141124725, 0.24611230194568634, 0.33791524171829224,
    0.44070982933044434, 0.5626170039176941, 0.7229568362236023, 1.0,
], dtype=np.float64)

NF4_BLOCK = 64
PROJECTIONS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def nf4_unpack(packed, rows, cols):
    """Codes [rows, cols] from bytes [rows, cols/2]: element 2j is the low
    nibble of byte j, element 2j+1 the high nibble."""
    b = np.asarray(packed, dtype=np.uint8).reshape(rows, cols // 2)
    codes = np.empty((rows, cols), dtype=np.int64)
    codes[:, 0::2] = b & 0x0F
    codes[:, 1::2] = b >> 4
    return codes


def nf4_dequantize(packed, absmax, rows, cols):
    """W [rows, cols] fp64: level[code] times the scale of the element's block
    (blocks of 64 consecutive elements of the row-major weight)."""
    codes = nf4_unpack(packed, rows, cols)
    scale = np.repeat(np.asarray(absmax, dtype=np.float64), NF4_BLOCK)
    return NF4_LEVELS[codes] * scale.reshape(rows, cols)


def lora_scale(rank, alpha):
    return float(alpha) / float(rank)


def merged_params(base, gains, lora, s):
    """Block parameters for ``oracle.model.block_forward``: W + s B A per
    projection (base: dict of fp64 dequantized weights)."""
    p = {}
    for name in PROJECTIONS:
        a = om._f64(lora["a_" + name[1:]])
        b = om._f64(lora["b_" + name[1:]])
        p[name] = om._f64(base[name]) + s * (b @ a)
    for g in ("g_attn", "g_ffn", "g_q", "g_k"):
        p[g] = om._f64(gains[g])
    return p


def lora_forward_backward(base, gains, lora, x, dy, shape, rank, alpha):
    """Block forward and backward with frozen base weights and gains.
    Returns (y, dx, adapter grads {a_q, b_q, ..., a_d, b_d})."""
    s = lora_scale(rank, alpha)
    p = merged_params(base, gains, lora, s)
    y, cache = om.block_forward(p, x, shape)
    dx, grads = om.block_backward(cache, dy, shape)
    g = {}
    for name in PROJECTIONS:
        dw = grads[name]
        a = om._f64(lora["a_" + name[1:]])
        b = om._f64(lora["b_" + name[1:]])
        g["a_" + name[1:]] = s * (b.T @ dw)
        g["b_" + name[1:]] = s * (dw @ a.T)
    return y, dx, g


def lora_step(base, gains, lora, x, dy, shape, rank, alpha, optim, state=None, step=1):
    """One adapters-only step: forward, backward, global-norm clip over the
    adapter gradients, AdamW on the adapters (fp32 masters in ``lora``)."""
    y, dx, g = lora_forward_backward(base, gains, lora, x, dy, shape, rank, alpha)
    scale, norm, ok = om.clip_scale([om.squared_sum(v) for v in g.values()], optim["max_norm"])
    new = {}
    for k, gk in g.items():
        m, v = state[k] if state else (np.zeros(gk.shape), np.zeros(gk.shape))
        new[k], _, _ = om.adamw(lora[k], gk, m, v, step, optim["lr"], optim["beta1"],
                                optim["beta2"], optim["eps"], optim["weight_decay"], scale)
    return dict(y=y, dx=dx, grads=g, norm=norm, scale=scale, params=new)
