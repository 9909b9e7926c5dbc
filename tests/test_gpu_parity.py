"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle on
the same seeded inputs. Tolerances are set in tests/gpu_helpers.py."""
import math

import numpy as np
import pytest
import torch

from oracle import model as om
from resident_decoder_trainer_gb300 import rdt, synth
from resident_decoder_trainer_gb300.step import DecoderTrainer

from gpu_helpers import (ADAMW_REL, FWD_REL_L2, GRAD_REL_L2, LOSS_REL, SQ_START, ensure_built,
                         gpu_block, gpu_head, ragged_shape, rel_l2, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    assert rdt.device_error() == 0


# ------------------------------------------------------------------ GEMM
# every tile shape the host picks (128 x 192, 128 x 256, CTA-pair 256 x 256),
# with ragged M, N and K edges
GEMM_SHAPES = [(128, 256, 64), (300, 520, 200), (37, 40, 24), (1, 16, 16), (257, 513, 1000),
               (100, 38912, 64), (2048, 2048, 192), (5000, 5000, 40)]


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_matches_fp32_matmul_of_bf16_operands(a_mn, b_mn, M, N, K):
    g = torch.Generator(device="cpu").manual_seed(M * 7 + N * 13 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T

    def stored(X, mn):  # [rows, K] -> operand as stored; pad ld to a multiple of 8
        Y = X.T.contiguous() if mn else X.contiguous()
        ld = (Y.shape[1] + 7) // 8 * 8
        buf = torch.zeros(Y.shape[0], ld, dtype=torch.bfloat16)
        buf[:, :Y.shape[1]] = Y
        return buf.cuda()

    a, b = stored(A, a_mn), stored(B, b_mn)
    ldc = (N + 3) // 4 * 4
    c = torch.full((M, ldc), float("nan"), device="cuda")
    rdt.gemm(a, a_mn, b, b_mn, M, N, K, c)
    torch.cuda.synchronize()
    out = c[:, :N].double().cpu()
    assert torch.isfinite(out).all()
    assert rel_l2(out.numpy(), ref.numpy()) < 1e-5
    assert torch.isnan(c[:, N:]).all()  # nothing written past N


SPLITK_SHAPES = [(2048, 16, 2560, 0, 0), (2048, 48, 9728, 0, 1), (16, 2560, 2048, 1, 1),
                 (40, 1000, 3000, 1, 1), (300, 24, 4100, 0, 1), (9728, 16, 2048, 1, 1)]


@pytest.mark.parametrize("M,N,K,a_mn,b_mn", SPLITK_SHAPES)
def test_split_k_gemm_matches_fp64(M, N, K, a_mn, b_mn):
    """Skinny problems (few 128 x 256 output tiles, long K) given scratch run as
    K-slices summed in slice order: same values as the fp64 product, nothing
    written past N, and bit-identical on a second run."""
    g = torch.Generator(device="cpu").manual_seed(M + 3 * N + 7 * K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T

    def stored(X, mn):
        Y = X.T.contiguous() if mn else X.contiguous()
        ld = (Y.shape[1] + 7) // 8 * 8
        buf = torch.zeros(Y.shape[0], ld, dtype=torch.bfloat16)
        buf[:, :Y.shape[1]] = Y
        return buf.cuda()

    a, b = stored(A, a_mn), stored(B, b_mn)
    ldc = (N + 3) // 4 * 4 + 4
    ws = torch.empty(16 << 20, device="cuda")
    outs = []
    for _ in range(2):
        c = torch.full((M, ldc), float("nan"), device="cuda")
        rdt.gemm(a, a_mn, b, b_mn, M, N, K, c, split_ws=ws)
        torch.cuda.synchronize()
        outs.append(c)
    out = outs[0][:, :N].double().cpu()
    assert torch.isfinite(out).all()
    assert rel_l2(out.numpy(), ref.numpy()) < 1e-5
    assert torch.isnan(outs[0][:, N:]).all()
    assert torch.equal(outs[0][:, :N], outs[1][:, :N])


@pytest.mark.parametrize("b_mn", [0, 1])
def test_pair_split_k_gemm_matches_fp64(b_mn):
    """A 2048 x 2560 output (80 CTA-pair tiles on 76 pairs) over K = 8192
    runs as K-slices on the pair kernel; same values as the fp64 product,
    nothing written past N, bit-identical on a second run."""
    M, N, K = 2048, 2560, 8192
    g = torch.Generator(device="cpu").manual_seed(17 + b_mn)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    Bm = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = A.double() @ Bm.double().T
    b = (Bm.T.contiguous() if b_mn else Bm).cuda()
    ws = torch.empty(4 * M * N, device="cuda")
    outs = []
    for _ in range(2):
        c = torch.full((M, N + 4), float("nan"), device="cuda")
        rdt.gemm(A.cuda(), 0, b, b_mn, M, N, K, c, split_ws=ws)
        torch.cuda.synchronize()
        outs.append(c)
    assert rel_l2(outs[0][:, :N].double().cpu().numpy(), ref.numpy()) < 1e-5
    assert torch.isnan(outs[0][:, N:]).all()
    assert torch.equal(outs[0][:, :N], outs[1][:, :N])


# ------------------------------------------------------------------ block
def _block_case(shape, seed=0):
    blk, x, dy = synth.make_block_inputs(shape, seed)
    y_ref, cache = om.block_forward(blk, x, shape)
    dx_ref, g_ref = om.block_backward(cache, dy, shape)
    y, dx, g, sq = gpu_block(shape, blk, x, dy, with_sq=True)
    x64 = to_np(x)
    # the squared sum the backward fused into its weight-gradient epilogues
    # and gain reductions is the sum of squares of the gradients it returned
    ref_sq = SQ_START + sum(float(np.sum(to_np(t) ** 2)) for t in g.values())
    assert abs(sq - ref_sq) / ref_sq < 1e-6, (sq, ref_sq)
    assert rel_l2(to_np(y) - x64, y_ref - x64) < FWD_REL_L2
    assert rel_l2(to_np(dx), dx_ref) < GRAD_REL_L2
    for name in g_ref:
        err = rel_l2(to_np(g[name]), g_ref[name])
        assert err < GRAD_REL_L2, f"{name}: rel L2 {err:.3e}"


def test_block_parity_tiny():
    _block_case(synth.WORKLOADS["tiny"].replace(layers=1))


def test_block_parity_ragged_multi_tile():
    _block_case(ragged_shape(layers=1))


def test_block_parity_head_dim_128_mha_odd_seq():
    _block_case(ragged_shape(layers=1, hidden=512, n_heads=4, n_kv_heads=4, head_dim=128,
                             intermediate=1376, seq=131, batch=1), seed=3)


def test_block_parity_head_dim_128_gqa4_two_sequences():
    _block_case(ragged_shape(layers=1, hidden=512, n_heads=8, n_kv_heads=2, head_dim=128,
                             intermediate=1376, seq=300, batch=2), seed=7)


def test_block_parity_head_dim_128_long_sequence():
    # several 128-key tiles per sequence: online-softmax rescaling, multi-tile dK/dV
    _block_case(ragged_shape(layers=1, hidden=256, n_heads=2, n_kv_heads=1, head_dim=128,
                             intermediate=512, seq=700, batch=1), seed=9)


def test_block_parity_head_dim_64_gqa4_long_sequence():
    # head_dim 64 on the tensor-core kernels: several 128-key tiles, ragged tail
    _block_case(ragged_shape(layers=1, hidden=256, n_heads=8, n_kv_heads=2, head_dim=64,
                             intermediate=512, seq=650, batch=1), seed=13)


@pytest.mark.parametrize("shape", [
    ragged_shape(layers=1, hidden=512, n_heads=4, n_kv_heads=4, head_dim=128, intermediate=1376,
                 seq=131, batch=1),
    ragged_shape(layers=1, hidden=256, n_heads=8, n_kv_heads=2, head_dim=64, intermediate=512,
                 seq=650, batch=1),
], ids=["d128-s131", "d64-s650"])
def test_block_ignores_stale_workspace_contents(shape):
    """Whatever the saved-activation and workspace buffers held before the
    call (zeros, or all-ones bytes: NaN in fp32 and bf16), the block's output,
    input gradient and weight gradients are the same to the bit: no kernel
    reads a position it did not write first (padded segments included). The
    tensor-core head dims only: the head_dim 16/32 attention backward adds dQ
    with vector reductions, so its last bits may differ between two runs."""
    blk, x, dy = synth.make_block_inputs(shape, 11)
    runs = [gpu_block(shape, blk, x, dy, fill=f) for f in (0x00, 0xFF)]
    (y0, dx0, g0), (y1, dx1, g1) = runs
    assert torch.isfinite(y1).all() and torch.isfinite(dx1).all()
    assert torch.equal(y0, y1) and torch.equal(dx0, dx1)
    for name in g0:
        assert torch.equal(g0[name], g1[name]), name


def test_block_parity_head_dim_32_gqa4():
    _block_case(ragged_shape(layers=1, hidden=128, n_heads=8, n_kv_heads=2, head_dim=32,
                             intermediate=352, seq=97, batch=3), seed=5)


# ------------------------------------------------------------------- head
# 2048 tokens x 70,000 entries: two vocabulary chunks (the library keeps a
# chunk's bf16 dz at or below 128 M elements: 65,536 columns here), the second
# ragged, so the running log-sum-exp merge and the dh accumulation across
# chunks are exercised
TWO_CHUNKS = ragged_shape(hidden=256, vocab=70000, seq=1024, batch=2)


def _head_inputs(shape):
    g = torch.Generator().manual_seed(11)
    h = torch.randn(shape.tokens, shape.hidden, generator=g)
    gf = 1.0 + 0.1 * torch.randn(shape.hidden, generator=g)
    wl = 0.02 * torch.randn(shape.vocab, shape.hidden, generator=g)
    tg = torch.randint(0, shape.vocab, (shape.tokens,), generator=g)
    return h, gf, wl, tg


@pytest.mark.parametrize("shape", [synth.WORKLOADS["tiny"], ragged_shape(), TWO_CHUNKS],
                         ids=["tiny", "ragged", "two-chunks"])
def test_fused_cross_entropy_parity(shape):
    h, gf, wl, tg = _head_inputs(shape)
    ref = om.head_forward_backward(h, gf, wl, tg.numpy(), shape)
    loss, dh, dgf, dwl = gpu_head(shape, h, gf, wl, tg)
    lp = to_np(loss)
    assert np.max(np.abs(lp - ref["loss_partials"]) / ref["loss_partials"]) < LOSS_REL
    assert abs(lp.mean() - ref["loss"]) / ref["loss"] < LOSS_REL
    assert rel_l2(to_np(dh), ref["dh"]) < GRAD_REL_L2
    assert rel_l2(to_np(dgf), ref["g_final"]) < GRAD_REL_L2
    assert rel_l2(to_np(dwl), ref["w_lm"]) < GRAD_REL_L2
    ref_sq = float(np.sum(to_np(dgf) ** 2) + np.sum(to_np(dwl) ** 2))
    assert abs(gpu_head.last_sq - ref_sq) / ref_sq < 1e-6


@pytest.mark.parametrize("shape", [ragged_shape(), TWO_CHUNKS], ids=["ragged", "two-chunks"])
def test_head_ignores_stale_workspace_contents(shape):
    """The loss partials and gradients of the fused cross-entropy do not
    depend on what its workspace held before the call (zeros, or all-ones
    bytes: NaN in fp32 and bf16)."""
    h, gf, wl, tg = _head_inputs(shape)
    r0 = gpu_head(shape, h, gf, wl, tg, fill=0x00)
    sq0 = gpu_head.last_sq
    r1 = gpu_head(shape, h, gf, wl, tg, fill=0xFF)
    assert gpu_head.last_sq == sq0
    for a, b in zip(r0, r1):
        assert torch.isfinite(b).all()
        assert torch.equal(a, b)


def test_cross_entropy_of_zero_head_is_log_vocab():
    shape = ragged_shape()
    h = torch.randn(shape.tokens, shape.hidden)
    loss, dh, dgf, dwl = gpu_head(shape, h, torch.ones(shape.hidden),
                                  torch.zeros(shape.vocab, shape.hidden),
                                  torch.randint(0, shape.vocab, (shape.tokens,)))
    assert np.allclose(to_np(loss), math.log(shape.vocab), rtol=1e-6)
    assert float(dh.abs().max()) == 0.0


# ------------------------------------------------------- clip and AdamW
def test_sq_sum_and_clip_scale():
    g = torch.Generator().manual_seed(1)
    bufs = [torch.randn(n, generator=g) for n in (1, 7, 4096, 100003)]
    ref = sum(om.squared_sum(b) for b in bufs)
    dbufs = [b.cuda() for b in bufs]
    sumsq = torch.zeros(1, dtype=torch.float64, device="cuda")
    ws = torch.empty(rdt.sq_sum_workspace_bytes(), dtype=torch.uint8, device="cuda")
    rdt.sq_sum(dbufs, sumsq, ws)
    torch.cuda.synchronize()
    assert abs(float(sumsq) - ref) / ref < 1e-6
    scale = torch.zeros(1, device="cuda")
    flag = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    for max_norm in (0.5 * math.sqrt(ref), math.sqrt(ref) * 2.0):
        rdt.clip_scale(sumsq, max_norm, scale, flag)
        s_ref, _, _ = om.clip_scale([ref], max_norm)
        assert abs(float(scale) - s_ref) < 1e-6 and int(flag) == 0
    sumsq.fill_(float("inf"))
    rdt.clip_scale(sumsq, 1.0, scale, flag)
    assert int(flag) == 1 and float(scale) == 1.0


def test_adamw_matches_oracle_and_skip_flag_freezes_state():
    g = torch.Generator().manual_seed(2)
    n = 10001
    w, gr = torch.randn(n, generator=g), 1e-2 * torch.randn(n, generator=g)
    m, v = 1e-3 * torch.randn(n, generator=g), 1e-5 * torch.rand(n, generator=g)
    o = synth.OPTIM
    wr, mr, vr = om.adamw(w, gr, m, v, 3, o["lr"], o["beta1"], o["beta2"], o["eps"],
                          o["weight_decay"], scale=0.7)
    wd, gd, md, vd = w.cuda(), gr.cuda(), m.cuda(), v.cuda()
    scale = torch.full((1,), 0.7, device="cuda")
    wbf = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    rdt.adamw_step(wd, gd, md, vd, 3, o["lr"], o["beta1"], o["beta2"], o["eps"],
                   o["weight_decay"], scale=scale, w_bf16=wbf)
    torch.cuda.synchronize()
    assert rel_l2(to_np(wd), wr) < ADAMW_REL
    assert np.max(np.abs(to_np(wd) - wr)) < ADAMW_REL * np.max(np.abs(wr))
    assert rel_l2(to_np(md), mr) < ADAMW_REL and rel_l2(to_np(vd), vr) < ADAMW_REL
    assert torch.equal(wbf.cpu(), wd.cpu().to(torch.bfloat16))
    before = [t.clone() for t in (wd, md, vd)]
    skip = torch.ones(1, dtype=torch.int32, device="cuda")
    rdt.adamw_step(wd, gd, md, vd, 4, o["lr"], o["beta1"], o["beta2"], o["eps"],
                   o["weight_decay"], scale=scale, skip=skip)
    torch.cuda.synchronize()
    for a, b in zip(before, (wd, md, vd)):
        assert torch.equal(a, b)


# ------------------------------------------------------------- full step
def _full_step_case(shape, seed=0):
    blocks, head, x, tg = synth.make_model_inputs(shape, seed)
    ref = om.train_step(blocks, head, x, tg.numpy(), shape, step=1, optim=synth.OPTIM)
    tr = DecoderTrainer(shape)
    tr.load(blocks, head)
    loss = tr.forward_backward(x.cuda(), tg.cuda())
    torch.cuda.synchronize()
    lp = to_np(loss)
    assert abs(lp.mean() - ref["loss"]) / ref["loss"] < LOSS_REL
    assert np.max(np.abs(lp - ref["loss_partials"]) / ref["loss_partials"]) < LOSS_REL
    worst = 0.0
    for (li, name), gref in ref["grads"].items():
        err = rel_l2(to_np(tr.tensor(tr.g, li, name)), gref)
        worst = max(worst, err)
        assert err < GRAD_REL_L2, f"{li}.{name}: rel L2 {err:.3e}"
    # clip on the GPU's own gradients: the squared sum the backward fused into
    # its gradient producers, norm from it (not re-squared)
    g_all = to_np(tr.g)
    assert abs(float(tr.sumsq) - float(np.sum(g_all * g_all))) / float(np.sum(g_all * g_all)) < 1e-6
    assert abs(math.sqrt(float(tr.sumsq)) - ref["norm"]) / ref["norm"] < GRAD_REL_L2
    # AdamW given identical gradients: feed the oracle's gradients and their
    # squared sum (the standalone rdt_sq_sum)
    for (li, name), gref in ref["grads"].items():
        tr.tensor(tr.g, li, name).copy_(torch.from_numpy(gref).float())
    ws = torch.empty(rdt.sq_sum_workspace_bytes(), dtype=torch.uint8, device="cuda")
    rdt.sq_sum([tr.g], tr.sumsq, ws)
    tr.clip_and_update()
    torch.cuda.synchronize()
    for (li, name), wref in ref["params"].items():
        err = rel_l2(to_np(tr.tensor(tr.w, li, name)), wref)
        assert err < ADAMW_REL, f"AdamW {li}.{name}: rel L2 {err:.3e}"
    assert abs(float(tr.scale) - ref["scale"]) / ref["scale"] < 1e-5
    return worst


def test_full_step_parity_tiny():
    _full_step_case(synth.WORKLOADS["tiny"])


def test_full_step_parity_ragged_two_layers():
    _full_step_case(ragged_shape())


def test_training_reduces_loss_tiny():
    shape = synth.WORKLOADS["tiny"]
    blocks, head, x, tg = synth.make_model_inputs(shape, 0)
    tr = DecoderTrainer(shape, optim=dict(synth.OPTIM, lr=1e-2))
    tr.load(blocks, head)
    xd, td = x.cuda(), tg.cuda()
    losses = [float(tr.train_step(xd, td).mean()) for _ in range(15)]
    assert losses[0] == pytest.approx(math.log(256), rel=0.05)
    assert min(losses) < 0.9 * losses[0]
