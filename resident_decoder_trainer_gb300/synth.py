"""Seeded synthetic inputs for the decoder training step.

This module only draws random numbers in a fixed, documented order; it holds
none of the training step's arithmetic. Both the FP64 oracle (tests) and the
CUDA path (tests, bench) take their inputs from here, so the two sides see
identical fp32 values.

Workloads (shapes of the Qwen3-style decoder stacks the training step is
defined on; the pages train Qwen3-4B and smaller decoders on token corpora,
which are stood in for by these synthetic draws):

* ``tiny``      2 layers, hidden 64, 4/2 heads, head_dim 16, FFN 176, vocab 256,
                seq 32, batch 1, eps 1e-6, RoPE theta 1e4.
* ``small``     8 layers, hidden 1024, 16/8 heads, head_dim 64, FFN 2816,
                vocab 32000, seq 1024, batch 4.
* ``q4b_block`` one Qwen3-4B-shaped block: hidden 2560, 32/8 heads, head_dim
                128, FFN 9728, theta 1e6, seq 2048, batch 1 (forward+backward
                of the block only, upstream gradient ~N(0, 1e-3)).
* ``q4b_full``  36 Qwen3-4B-shaped blocks + vocab-151936 LM head, seq 1024,
                batch 4.

Draw order (one ``torch.Generator`` seeded with ``seed``):
for each block: Wq, Wk, Wv, Wo, Wgate, Wup, Wdown ~ N(0, 0.02) in [out, in]
row-major; then (head) W_lm ~ N(0, 0.02) [vocab, hidden]; then the input hidden
states x ~ N(0, 1) [batch*seq, hidden]; then target ids ~ U{0..vocab-1}
[batch*seq]; then (block-only workloads) the upstream gradient dy ~ N(0, 1e-3).
Every norm gain (input, post-attention, q-norm, k-norm, final) is 1.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class DecoderShape:
    layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    seq: int
    batch: int
    eps: float = 1e-6
    theta: float = 1e4

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def replace(self, **kw) -> "DecoderShape":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": DecoderShape(layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16,
                         intermediate=176, vocab=256, seq=32, batch=1, eps=1e-6, theta=1e4),
    "small": DecoderShape(layers=8, hidden=1024, n_heads=16, n_kv_heads=8, head_dim=64,
                          intermediate=2816, vocab=32000, seq=1024, batch=4, eps=1e-6, theta=1e4),
    "q4b_block": DecoderShape(layers=1, hidden=2560, n_heads=32, n_kv_heads=8, head_dim=128,
                              intermediate=9728, vocab=151936, seq=2048, batch=1, eps=1e-6,
                              theta=1e6),
    # the NF4-frozen block with LoRA adapters runs at the single-block shape
    "q4b_nf4": DecoderShape(layers=1, hidden=2560, n_heads=32, n_kv_heads=8, head_dim=128,
                            intermediate=9728, vocab=151936, seq=2048, batch=1, eps=1e-6,
                            theta=1e6),
    "q4b_full": DecoderShape(layers=36, hidden=2560, n_heads=32, n_kv_heads=8, head_dim=128,
                             intermediate=9728, vocab=151936, seq=1024, batch=4, eps=1e-6,
                             theta=1e6),
}

# AdamW / clip hyper-parameters used by every workload.
OPTIM = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0)

BLOCK_MATRICES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")
BLOCK_GAINS = ("g_attn", "g_ffn", "g_q", "g_k")


def block_shapes(s: DecoderShape) -> dict[str, tuple[int, ...]]:
    """Shapes of one block's trainable tensors, [out, in] for matrices."""
    return {
        "wq": (s.q_dim, s.hidden), "wk": (s.kv_dim, s.hidden), "wv": (s.kv_dim, s.hidden),
        "wo": (s.hidden, s.q_dim), "wg": (s.intermediate, s.hidden),
        "wu": (s.intermediate, s.hidden), "wd": (s.hidden, s.intermediate),
        "g_attn": (s.hidden,), "g_ffn": (s.hidden,), "g_q": (s.head_dim,), "g_k": (s.head_dim,),
    }


def _normal(shape, std, gen, device):
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device) * std


def make_generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_blocks(s: DecoderShape, gen: torch.Generator, device="cpu", layers=None):
    """Per-block parameter dicts (fp32), in the documented draw order."""
    out = []
    for _ in range(s.layers if layers is None else layers):
        shp = block_shapes(s)
        p = {name: _normal(shp[name], 0.02, gen, device) for name in BLOCK_MATRICES}
        for name in BLOCK_GAINS:
            p[name] = torch.ones(shp[name], dtype=torch.float32, device=device)
        out.append(p)
    return out


def draw_head(s: DecoderShape, gen: torch.Generator, device="cpu"):
    return {"g_final": torch.ones(s.hidden, dtype=torch.float32, device=device),
            "w_lm": _normal((s.vocab, s.hidden), 0.02, gen, device)}


def draw_batch(s: DecoderShape, gen: torch.Generator, device="cpu"):
    """Input hidden states x [T, H] ~ N(0,1) and target ids [T] ~ U{0..V-1}."""
    x = _normal((s.tokens, s.hidden), 1.0, gen, device)
    targets = torch.randint(0, s.vocab, (s.tokens,), generator=gen, dtype=torch.int64,
                            device=device).to(torch.int32)
    return x, targets


def draw_upstream(s: DecoderShape, gen: torch.Generator, device="cpu", std=1e-3):
    return _normal((s.tokens, s.hidden), std, gen, device)


def make_model_inputs(s: DecoderShape, seed: int = 0, device="cpu"):
    """Full-model workload: (blocks, head, x, targets)."""
    gen = make_generator(seed, device)
    blocks = draw_blocks(s, gen, device)
    head = draw_head(s, gen, device)
    x, targets = draw_batch(s, gen, device)
    return blocks, head, x, targets


def make_block_inputs(s: DecoderShape, seed: int = 0, device="cpu"):
    """Single-block workload: (block params, x, dy)."""
    gen = make_generator(seed, device)
    (blk,) = draw_blocks(s, gen, device, layers=1)
    x = _normal((s.tokens, s.hidden), 1.0, gen, device)
    dy = draw_upstream(s, gen, device)
    return blk, x, dy


# ------------------------------------------------------------------ NF4 + LoRA
# The NF4-frozen block workload: packed 4-bit codes uniform over 0..15 (two
# per byte), one fp32 scale per 64 consecutive weight elements drawn as
# 3|N(0, 0.02)|, frozen gains of 1, LoRA rank 16 / alpha 32 on all seven
# projections with A ~ N(0, 0.02) [rank, in] and B = 0 [out, rank] (or
# N(0, b_std) when a test wants the adapter path live).
LORA = dict(rank=16, alpha=32.0)
NF4_PROJECTIONS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def draw_nf4_block(s: DecoderShape, gen: torch.Generator, rank=None, b_std=0.0, device="cpu"):
    """(base, gains, lora): base[name] = (packed uint8 [out, in/2], absmax fp32
    [out*in/64]); gains fp32 ones; lora['a_q'..'a_d'] fp32 [rank, in] and
    lora['b_q'..'b_d'] fp32 [out, rank]."""
    rank = rank or LORA["rank"]
    shp = block_shapes(s)
    base = {}
    for name in NF4_PROJECTIONS:
        out, inn = shp[name]
        packed = torch.randint(0, 256, (out, inn // 2), generator=gen, dtype=torch.int32,
                               device=device).to(torch.uint8)
        absmax = (_normal((out * inn // 64,), 0.02, gen, device).abs() * 3.0)
        base[name] = (packed, absmax)
    gains = {g: torch.ones(shp[g], dtype=torch.float32, device=device)
             for g in ("g_attn", "g_ffn", "g_q", "g_k")}
    lora = {}
    for name in NF4_PROJECTIONS:
        out, inn = shp[name]
        lora["a_" + name[1:]] = _normal((rank, inn), 0.02, gen, device)
    for name in NF4_PROJECTIONS:
        out, inn = shp[name]
        lora["b_" + name[1:]] = (_normal((out, rank), b_std, gen, device) if b_std > 0
                                 else torch.zeros((out, rank), dtype=torch.float32, device=device))
    return base, gains, lora


def make_nf4_inputs(s: DecoderShape, seed: int = 0, rank=None, b_std=0.0, device="cpu"):
    """NF4 block workload: (base, gains, lora, x, dy)."""
    gen = make_generator(seed, device)
    base, gains, lora = draw_nf4_block(s, gen, rank=rank, b_std=b_std, device=device)
    x = _normal((s.tokens, s.hidden), 1.0, gen, device)
    dy = draw_upstream(s, gen, device)
    return base, gains, lora, x, dy
