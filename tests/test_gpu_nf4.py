"""GPU parity of the NF4-frozen path with the FP64 oracle (``oracle/nf4.py``):
the NF4 GEMM (codes decoded into the tensor-core operand tiles, plus the bf16
tail that carries the LoRA term) against an fp64 matmul of the same decoded
weights, and the NF4 + LoRA block forward/backward and adapters-only step."""
import numpy as np
import pytest
import torch

from oracle import model as om
from oracle import nf4 as on
from resident_decoder_trainer_gb300 import rdt, synth

from gpu_helpers import (FWD_REL_L2, GRAD_REL_L2, ADAMW_REL, SQ_START, ensure_built,
                         gpu_nf4_block, nf4_buffers, rel_l2, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    assert rdt.device_error() == 0


def _nf4_weight(rows, cols, g):
    codes = torch.randint(0, 256, (rows, cols // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    scales = (torch.randn(rows * cols // 64, generator=g) * 0.02).abs() * 3.0
    return codes, scales


def _decoded(codes, scales, rows, cols):
    """W as the GPU's operand: level * scale in fp32, rounded to bf16 (RNE)."""
    w = on.nf4_dequantize(codes.numpy(), scales.numpy().astype(np.float32), rows, cols)
    lv = on.NF4_LEVELS.astype(np.float32)[on.nf4_unpack(codes.numpy(), rows, cols)]
    w32 = lv * np.repeat(scales.numpy().astype(np.float32), 64).reshape(rows, cols)
    assert np.max(np.abs(w32.astype(np.float64) - w)) <= 1e-6 * np.max(np.abs(w))
    return torch.from_numpy(w32).to(torch.bfloat16).double()


@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("k2", [0, 16, 48])
@pytest.mark.parametrize("M,rows,cols", [(300, 320, 512), (128, 192, 256), (700, 512, 1024)])
def test_nf4_gemm_matches_fp64_of_decoded_weights(b_mn, k2, M, rows, cols):
    if b_mn and k2 == 48 and rows == 192:
        pytest.skip("covered by the other shapes")
    g = torch.Generator().manual_seed(M + rows + 7 * cols + k2 + b_mn)
    codes, scales = _nf4_weight(rows, cols, g)
    w = _decoded(codes, scales, rows, cols)           # [rows, cols]
    N, K1 = (cols, rows) if b_mn else (rows, cols)
    a = torch.randn(M, K1, generator=g).to(torch.bfloat16)
    ref = a.double() @ (w if b_mn else w.T)
    a2 = b2 = None
    if k2:
        a2 = torch.randn(M, k2, generator=g).to(torch.bfloat16)
        b2 = torch.randn(k2, N, generator=g).to(torch.bfloat16) if b_mn else \
            torch.randn(N, k2, generator=g).to(torch.bfloat16)
        ref = ref + a2.double() @ (b2.double() if b_mn else b2.double().T)
    ldc = (N + 3) // 4 * 4
    c = torch.full((M, ldc), float("nan"), device="cuda")
    rdt.gemm_nf4(a.cuda(), codes.cuda(), scales.cuda(), rows, cols, b_mn, c,
                 None if a2 is None else a2.cuda(), None if b2 is None else b2.cuda())
    torch.cuda.synchronize()
    out = c[:, :N].double().cpu()
    assert torch.isfinite(out).all()
    assert rel_l2(out.numpy(), ref.numpy()) < 1e-5


@pytest.mark.parametrize("b_mn,rows,cols,k2", [(0, 2560, 9728, 16), (1, 19456, 2560, 32),
                                              (0, 2560, 4096, 0), (1, 6144, 2560, 48)])
def test_nf4_gemm_split_k_matches_fp64(b_mn, rows, cols, k2):
    """2048 rows against a 2560-wide output: 80 pair tiles, so the GEMM runs as
    K-slices (the LoRA tail in the last slice) summed in slice order."""
    M = 2048
    g = torch.Generator().manual_seed(rows + cols + k2 + b_mn)
    codes, scales = _nf4_weight(rows, cols, g)
    w = _decoded(codes, scales, rows, cols)
    N, K1 = (cols, rows) if b_mn else (rows, cols)
    a = torch.randn(M, K1, generator=g).to(torch.bfloat16)
    ref = a.double() @ (w if b_mn else w.T)
    a2 = b2 = None
    if k2:
        a2 = torch.randn(M, k2, generator=g).to(torch.bfloat16)
        b2 = torch.randn(k2, N, generator=g).to(torch.bfloat16) if b_mn else \
            torch.randn(N, k2, generator=g).to(torch.bfloat16)
        ref = ref + a2.double() @ (b2.double() if b_mn else b2.double().T)
    ws = torch.empty(4 * M * N, device="cuda")
    outs = []
    for split in (ws, ws, None):
        c = torch.full((M, N + 4), float("nan"), device="cuda")
        rdt.gemm_nf4(a.cuda(), codes.cuda(), scales.cuda(), rows, cols, b_mn, c,
                     None if a2 is None else a2.cuda(), None if b2 is None else b2.cuda(),
                     split_ws=split)
        torch.cuda.synchronize()
        outs.append(c)
    # fp32 accumulation over K up to 19456: typical error sqrt(K) 2^-24 = 8e-6
    tol = 2e-5
    out = outs[0][:, :N].double().cpu()
    assert torch.isfinite(out).all()
    assert rel_l2(out.numpy(), ref.numpy()) < tol
    assert torch.isnan(outs[0][:, N:]).all()
    assert torch.equal(outs[0][:, :N], outs[1][:, :N])  # fixed summation order
    assert rel_l2(outs[2][:, :N].double().cpu().numpy(), ref.numpy()) < tol


# ------------------------------------------------------- NF4 + LoRA block
def _nf4_shape(**kw):
    base = dict(layers=1, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, intermediate=512,
                vocab=256, seq=200, batch=2, eps=1e-6, theta=1e4)
    base.update(kw)
    return synth.DecoderShape(**base)


def _oracle_inputs(shape, base, gains, lora, x, dy):
    shp = synth.block_shapes(shape)
    deq = {k: on.nf4_dequantize(p.numpy(), a.numpy(), *shp[k]) for k, (p, a) in base.items()}
    g64 = {k: v.numpy().astype(np.float64) for k, v in gains.items()}
    l64 = {k: v.numpy().astype(np.float64) for k, v in lora.items()}
    return deq, g64, l64, om._f64(x), om._f64(dy)


def _random_gains(shape, gains, seed):
    g = torch.Generator().manual_seed(seed)
    return {k: 1.0 + 0.1 * torch.randn(v.shape, generator=g) for k, v in gains.items()}


def _nf4_block_case(shape, rank, alpha, b_std, seed=0, gains_random=True):
    base, gains, lora, x, dy = synth.make_nf4_inputs(shape, seed=seed, rank=rank, b_std=b_std)
    if gains_random:
        gains = _random_gains(shape, gains, seed + 1)
    y_ref, dx_ref, g_ref = on.lora_forward_backward(
        *_oracle_inputs(shape, base, gains, lora, x, dy), shape, rank, alpha)
    y, dx, g, sq = gpu_nf4_block(shape, rank, alpha, base, gains, lora, x, dy)
    x64 = to_np(x)
    assert rel_l2(to_np(y) - x64, y_ref - x64) < FWD_REL_L2
    assert rel_l2(to_np(dx), dx_ref) < GRAD_REL_L2
    for name, ref in g_ref.items():
        if not np.any(ref):
            continue
        err = rel_l2(to_np(g[name]), ref)
        assert err < GRAD_REL_L2, f"{name}: rel L2 {err:.3e}"
    # the squared sum fused into the adapter-gradient epilogues
    ref_sq = SQ_START + sum(float(np.sum(to_np(t) ** 2)) for t in g.values())
    assert abs(sq - ref_sq) / ref_sq < 1e-6, (sq, ref_sq)
    return y, dx, g


@pytest.mark.parametrize("rank,alpha", [(16, 32.0), (8, 16.0)])
def test_nf4_block_parity_ragged_gqa(rank, alpha):
    _nf4_block_case(_nf4_shape(), rank, alpha, b_std=0.05)


def test_nf4_block_parity_head_dim_128_odd_seq():
    _nf4_block_case(_nf4_shape(hidden=512, n_heads=4, n_kv_heads=1, head_dim=128,
                               intermediate=768, seq=131, batch=1), 16, 32.0, b_std=0.05, seed=4)


@pytest.mark.parametrize("shape", [
    _nf4_shape(),
    _nf4_shape(hidden=512, n_heads=4, n_kv_heads=1, head_dim=128, intermediate=768, seq=131,
               batch=1),
], ids=["d64-s200", "d128-s131"])
def test_nf4_block_ignores_stale_workspace_contents(shape):
    """Zeros or all-ones bytes (NaN) in the saved-activation and workspace
    buffers before the call give bit-identical outputs, input gradients,
    adapter gradients and squared sums."""
    base, gains, lora, x, dy = synth.make_nf4_inputs(shape, seed=2, rank=16, b_std=0.05)
    gains = _random_gains(shape, gains, 3)
    r0 = gpu_nf4_block(shape, 16, 32.0, base, gains, lora, x, dy, fill=0x00)
    r1 = gpu_nf4_block(shape, 16, 32.0, base, gains, lora, x, dy, fill=0xFF)
    assert torch.isfinite(r1[0]).all() and torch.isfinite(r1[1]).all()
    assert torch.equal(r0[0], r1[0]) and torch.equal(r0[1], r1[1])
    for name in r0[2]:
        assert torch.equal(r0[2][name], r1[2][name]), name
    assert r0[3] == r1[3]


def test_nf4_block_zero_b_gives_exactly_zero_da():
    """B = 0 (the adapters' initial state): U = s dY B vanishes exactly, so every
    dA is exactly zero and dB, y, dx are those of the plain NF4 block."""
    shape = _nf4_shape(seq=96, batch=1)
    _, _, g = _nf4_block_case(shape, 16, 32.0, b_std=0.0, seed=2)
    for name in ("a_q", "a_k", "a_v", "a_o", "a_g", "a_u", "a_d"):
        assert float(g[name].abs().max()) == 0.0, name


def test_lora_shadow_layout_is_bit_exact():
    """The bf16 operand copy: the A's in the adapter layout, then the stacked
    block-diagonal [Bq; Bk; Bv] and [Bg; Bu] and the plain Bo, Bd."""
    shape = _nf4_shape()
    rank = 16
    base, gains, lora, _, _ = synth.make_nf4_inputs(shape, seed=5, rank=rank, b_std=0.1)
    cfg, _, _, _, lw, shadow = nf4_buffers(shape, rank, base, gains, lora)
    torch.cuda.synchronize()
    sh = shadow.cpu()
    bf = {k: v.to(torch.bfloat16) for k, v in lora.items()}
    n_a = sum(bf["a_" + n[1:]].numel() for n in synth.NF4_PROJECTIONS)
    assert torch.equal(sh[:n_a], torch.cat([bf["a_" + n[1:]].reshape(-1)
                                            for n in synth.NF4_PROJECTIONS]))
    o = n_a
    for names in (("b_q", "b_k", "b_v"), ("b_o",), ("b_g", "b_u"), ("b_d",)):
        rows = sum(bf[k].shape[0] for k in names)
        want = torch.zeros(rows, len(names) * rank, dtype=torch.bfloat16)
        r0 = 0
        for j, k in enumerate(names):
            want[r0:r0 + bf[k].shape[0], j * rank:(j + 1) * rank] = bf[k]
            r0 += bf[k].shape[0]
        got = sh[o:o + want.numel()].view(want.shape)
        assert torch.equal(got, want), names
        o += want.numel()
    assert o == sh.numel()


def test_nf4_adapters_only_step():
    """One adapters-only step: fused squared sum -> clip scale -> AdamW on the
    fp32 adapters, then the shadow refresh. AdamW against the oracle's update
    given the same gradients; the clip against the oracle's norm of them."""
    shape = _nf4_shape(seq=128, batch=1)
    rank, alpha = 16, 32.0
    base, gains, lora, x, dy = synth.make_nf4_inputs(shape, seed=8, rank=rank, b_std=0.05)
    dy = dy * 1e4  # a gradient norm above max_norm, so the clip is active
    cfg, codes, scales, g, lw, shadow = nf4_buffers(shape, rank, base, gains, lora)
    B, S = shape.batch, shape.seq
    saved = torch.empty(rdt.nf4_saved_bytes(cfg, rank, B, S), dtype=torch.uint8, device="cuda")
    ws = torch.empty(rdt.nf4_workspace_bytes(cfg, rank, B, S), dtype=torch.uint8, device="cuda")
    xd = x.cuda()
    y = torch.empty_like(xd)
    dx = torch.empty_like(xd)
    grads = torch.empty_like(lw)
    sumsq = torch.zeros(1, dtype=torch.float64, device="cuda")
    scale = torch.ones(1, device="cuda")
    nonfinite = torch.zeros(1, dtype=torch.int32, device="cuda")
    m = torch.zeros_like(lw)
    v = torch.zeros_like(lw)
    w0 = lw.cpu().numpy().astype(np.float64)
    o = synth.OPTIM
    rdt.nf4_block_forward(cfg, rank, alpha, B, S, codes, scales, g, shadow, xd, y, saved, ws)
    rdt.nf4_block_backward(cfg, rank, alpha, B, S, codes, scales, g, shadow, xd, saved,
                           dy.cuda(), dx, grads, ws, grad_sq=sumsq)
    rdt.clip_scale(sumsq, o["max_norm"], scale, nonfinite)
    rdt.adamw_step(lw, grads, m, v, 1, o["lr"], o["beta1"], o["beta2"], o["eps"],
                   o["weight_decay"], scale=scale, skip=nonfinite)
    rdt.lora_shadow(cfg, rank, lw, shadow)
    torch.cuda.synchronize()
    g64 = to_np(grads)
    want_scale, norm, ok = om.clip_scale([om.squared_sum(g64)], o["max_norm"])
    assert ok and norm > o["max_norm"] and int(nonfinite) == 0
    assert abs(float(scale) - want_scale) / want_scale < 1e-6
    w_ref, _, _ = om.adamw(w0, g64, np.zeros_like(w0), np.zeros_like(w0), 1, o["lr"],
                           o["beta1"], o["beta2"], o["eps"], o["weight_decay"], want_scale)
    assert np.max(np.abs(to_np(lw) - w_ref)) <= ADAMW_REL * np.max(np.abs(w_ref))
    n_a = sum(lora["a_" + n[1:]].numel() for n in synth.NF4_PROJECTIONS)
    assert torch.equal(shadow[:n_a].cpu(), lw[:n_a].cpu().to(torch.bfloat16))


def test_q4b_nf4_block_at_full_size():
    """The NF4 + LoRA block at the single-block Qwen3-4B shape (hidden 2560,
    32/8 heads of 128, FFN 9728, 2048 tokens, rank 16, alpha 32), adapters
    live (B drawn nonzero) so every adapter gradient is checked."""
    shape = synth.WORKLOADS["q4b_nf4"]
    _nf4_block_case(shape, synth.LORA["rank"], synth.LORA["alpha"], b_std=0.02, seed=0,
                    gains_random=False)
