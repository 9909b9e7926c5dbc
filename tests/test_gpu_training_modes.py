"""GPU tests of the step driver's training modes beyond the plain step:
activation checkpointing (segmented recompute, cuda_trainer.rs
``recompute_segment``) and gradient accumulation over micro-batches (R-038,
``GpuGradientAccumulator``). The kernels are deterministic, so a mode that
only changes when or how often the same block calls run must reproduce the
plain step bit for bit; accumulation is checked against the FP64 oracle's
accumulated step."""
import numpy as np
import pytest
import torch

from oracle import model as om
from resident_decoder_trainer_gb300 import rdt, synth
from resident_decoder_trainer_gb300.step import DecoderTrainer

from gpu_helpers import (ADAMW_REL, GRAD_REL_L2, LOSS_REL, ensure_built, ragged_shape, rel_l2,
                         to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    assert rdt.device_error() == 0


def _run(shape, steps=2, **kw):
    blocks, head, x, tg = synth.make_model_inputs(shape, 5)
    tr = DecoderTrainer(shape, **kw)
    tr.load(blocks, head)
    xd, td = x.cuda(), tg.cuda()
    losses = []
    for _ in range(steps):
        losses.append(tr.train_step(xd, td).clone())
    torch.cuda.synchronize()
    return tr, losses


@pytest.mark.parametrize("segments", [1, 2, 5])
def test_checkpointing_is_bit_identical(segments):
    """5 layers in 1, 2 (3 + 2) or 5 segments: the recomputed activations, and
    so the losses, gradients, weights and moments after two steps, equal the
    plain step's exactly."""
    shape = ragged_shape(layers=5)
    ref, ref_losses = _run(shape)
    tr, losses = _run(shape, checkpoint_segments=segments)
    assert tr.segment_size == -(-5 // segments)
    assert tr.saved.numel() == tr.segment_size * tr.saved_bytes
    for a, b in zip(losses, ref_losses):
        assert torch.equal(a, b)
    for name in ("g", "w", "m", "v", "wb"):
        assert torch.equal(getattr(tr, name), getattr(ref, name)), name
    assert float(tr.sumsq) == float(ref.sumsq)


# ------------------------------------------------------- gradient accumulation
def test_accumulated_step_matches_oracle():
    """Two micro-batches of two 200-token sequences each: gradients summed in
    place by the gradient producers (dW GEMM epilogues with the old value as
    the residual, gain reductions adding), the clip's squared sum taken from
    the accumulated values."""
    shape = ragged_shape()
    n, T = 2, shape.tokens
    blocks, head, _, _ = synth.make_model_inputs(shape, 2)
    g = torch.Generator().manual_seed(9)
    x = torch.randn(n * T, shape.hidden, generator=g)
    tg = torch.randint(0, shape.vocab, (n * T,), generator=g, dtype=torch.int64)
    ref = om.train_step_accumulated(blocks, head, [x[:T], x[T:]],
                                    [tg[:T].numpy(), tg[T:].numpy()], shape, step=1,
                                    optim=synth.OPTIM)
    tr = DecoderTrainer(shape, accumulation_steps=n)
    tr.load(blocks, head)
    for i in range(n):
        tr.forward_backward(x[i * T:(i + 1) * T].cuda(), tg[i * T:(i + 1) * T].int().cuda(),
                            micro=i)
    torch.cuda.synchronize()
    lp = to_np(tr.loss_partials)
    assert abs(lp.mean() - ref["loss"]) / ref["loss"] < LOSS_REL
    for (li, name), gref in ref["grads"].items():
        err = rel_l2(to_np(tr.tensor(tr.g, li, name)), gref)
        assert err < GRAD_REL_L2, f"{li}.{name}: rel L2 {err:.3e}"
    g_all = to_np(tr.g)
    want = float(np.sum(g_all * g_all))
    assert abs(float(tr.sumsq) - want) / want < 1e-6
    assert abs(np.sqrt(float(tr.sumsq)) - ref["norm"]) / ref["norm"] < GRAD_REL_L2


def test_accumulation_of_sequences_matches_the_whole_batch_on_gpu():
    """Micro-batches that are the sequences of one batch: the accumulated GPU
    gradients equal the one-pass GPU gradients of that batch up to fp32
    summation order."""
    whole_shape = ragged_shape(batch=2)
    micro_shape = ragged_shape(batch=1)
    blocks, head, x, tg = synth.make_model_inputs(whole_shape, 3)
    whole = DecoderTrainer(whole_shape)
    whole.load(blocks, head)
    whole.forward_backward(x.cuda(), tg.cuda())
    acc = DecoderTrainer(micro_shape, accumulation_steps=2)
    acc.load(blocks, head)
    T = micro_shape.tokens
    for i in range(2):
        acc.forward_backward(x[i * T:(i + 1) * T].cuda(), tg[i * T:(i + 1) * T].cuda(), micro=i)
    torch.cuda.synchronize()
    # per-token losses: same rows, possibly another tiling of the vocabulary
    assert torch.allclose(acc.loss_partials, whole.loss_partials, rtol=1e-6, atol=0)
    assert rel_l2(to_np(acc.g), to_np(whole.g)) < 1e-4
    assert abs(float(acc.sumsq) - float(whole.sumsq)) / float(whole.sumsq) < 1e-4


def test_accumulated_train_step_runs_and_updates():
    shape = ragged_shape()
    tr, losses = _run(shape, steps=1, accumulation_steps=1)
    tr2 = DecoderTrainer(shape, accumulation_steps=2)
    blocks, head, x, tg = synth.make_model_inputs(shape, 5)
    tr2.load(blocks, head)
    xs = torch.cat([x, x]).cuda()
    ts = torch.cat([tg, tg]).cuda()
    tr2.train_step(xs, ts)
    torch.cuda.synchronize()
    # the same micro-batch twice with loss scale 1/(2T): the gradient of the
    # single batch, so the update matches the plain step's closely
    assert rel_l2(to_np(tr2.w), to_np(tr.w)) < 1e-6
    assert torch.equal(tr2.loss_partials[:shape.tokens], losses[0])


# ------------------------------------------------------------ device embedding
from oracle import embedding as oe  # noqa: E402


def test_embedding_lookup_is_exact_and_flags_bad_ids():
    g = torch.Generator().manual_seed(1)
    V, H, T = 1000, 256, 777
    table = torch.randn(V, H, generator=g).cuda()
    ids = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    ids[5] = ids[9] = 17
    x = torch.full((T, H), float("nan"), device="cuda")
    rdt.embedding_forward(table, ids.cuda(), x)
    torch.cuda.synchronize()
    assert torch.equal(x, table[ids.long().cuda()])
    assert rdt.device_error() == 0
    ids[3] = V  # out of range: a zero row and RDT_EINDEX, no fault
    rdt.embedding_forward(table, ids.cuda(), x)
    assert rdt.device_error() == rdt.RDT_EINDEX
    assert float(x[3].abs().max()) == 0.0
    assert torch.equal(x[4:], table[ids[4:].long().cuda()])


@pytest.mark.parametrize("V,H,T,distinct", [(5000, 512, 3000, 40), (300, 64, 1, 1),
                                            (151936, 2560, 4096, 151936)])
def test_embedding_scatter_add_matches_oracle(V, H, T, distinct):
    """Duplicate-heavy, single-token and Qwen3-4B-sized cases: the scatter-add
    against the oracle on the rows the tokens touch (compact re-indexing keeps
    the oracle small), untouched rows exactly zero, accumulation adding, and
    the same bits on a second run."""
    g = torch.Generator().manual_seed(V + T)
    ids = torch.randint(0, distinct, (T,), generator=g, dtype=torch.int32)
    dx = torch.randn(T, H, generator=g)
    scale = torch.tensor([0.37], device="cuda")
    dtable = torch.full((V, H), float("nan"), device="cuda")
    ws = torch.empty(rdt.embedding_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    idd, dxd = ids.cuda(), dx.cuda()
    rdt.embedding_backward(idd, dxd, dtable, ws, scale=scale)
    first = dtable.clone()
    rdt.embedding_backward(idd, dxd, dtable, ws, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(first, dtable)  # deterministic
    used, compact = torch.unique(ids.long(), return_inverse=True)
    ref, _ = oe.embedding_grad(compact.numpy(), dx.numpy(), len(used))
    got = dtable[used.cuda()].double().cpu().numpy()
    assert np.max(np.abs(got - 0.37 * ref)) <= 1e-6 * max(1.0, np.max(np.abs(ref)))
    mask = torch.ones(V, dtype=torch.bool)
    mask[used] = False
    assert float(dtable[mask.cuda()].abs().max() if mask.any() else 0.0) == 0.0
    rdt.embedding_backward(idd, dxd, dtable, ws, scale=scale, accumulate=True)
    torch.cuda.synchronize()
    got2 = dtable[used.cuda()].double().cpu().numpy()
    assert np.max(np.abs(got2 - 2 * 0.37 * ref)) <= 2e-6 * max(1.0, np.max(np.abs(ref)))


def test_embedded_step_matches_oracle():
    """The step fed by token ids: lookup, model, the first block's activation
    gradient clipped by its own norm and scatter-added, the table's own AdamW
    next to the global clip + AdamW of the rest."""
    shape = ragged_shape()
    blocks, head, _, tg = synth.make_model_inputs(shape, 4)
    g = torch.Generator().manual_seed(8)
    table = torch.randn(shape.vocab, shape.hidden, generator=g)
    ids = torch.randint(0, 50, (shape.tokens,), generator=g, dtype=torch.int32)
    ref = oe.train_step_embedded(table.numpy(), blocks, head, ids.numpy(), tg.numpy(), shape,
                                 step=1, optim=synth.OPTIM)
    tr = DecoderTrainer(shape, embedding=True)
    tr.load(blocks, head, emb=table)
    tr.train_step(targets=tg.cuda(), ids=ids.cuda())
    torch.cuda.synchronize()
    lp = to_np(tr.loss_partials)
    assert abs(lp.mean() - ref["loss"]) / ref["loss"] < LOSS_REL
    assert abs(float(tr.emb_scale) - ref["emb_scale"]) / ref["emb_scale"] < GRAD_REL_L2
    err = rel_l2(to_np(tr.emb_g), ref["emb_grad"])
    assert err < GRAD_REL_L2, err
    # the table's AdamW given the same gradient (its own, no global scale)
    o = synth.OPTIM
    w0 = table.numpy().astype(np.float64)
    want, _, _ = om.adamw(w0, to_np(tr.emb_g), np.zeros_like(w0), np.zeros_like(w0), 1, o["lr"],
                          o["beta1"], o["beta2"], o["eps"], o["weight_decay"], 1.0)
    assert np.max(np.abs(to_np(tr.emb) - want)) <= ADAMW_REL * np.max(np.abs(want))
    assert rdt.device_error() == 0


# ------------------------------------------------------------------ CUDA graph
@pytest.mark.parametrize("mode", [{}, {"accumulation_steps": 2}, {"embedding": True},
                                  {"checkpoint_segments": 2}])
def test_graph_replay_is_bit_identical(mode):
    """One eager step, then the captured step replayed twice on new inputs:
    losses, gradients, weights and moments equal three eager steps exactly
    (the AdamW step count lives on the device)."""
    shape = ragged_shape(layers=3)
    n = mode.get("accumulation_steps", 1)
    T = shape.tokens
    blocks, head, _, _ = synth.make_model_inputs(shape, 7)
    g = torch.Generator().manual_seed(11)
    table = torch.randn(shape.vocab, shape.hidden, generator=g)
    steps = []
    for _ in range(3):
        tg = torch.randint(0, shape.vocab, (n * T,), generator=g, dtype=torch.int32).cuda()
        if mode.get("embedding"):
            steps.append(dict(targets=tg, ids=torch.randint(0, shape.vocab, (n * T,),
                                                            generator=g,
                                                            dtype=torch.int32).cuda()))
        else:
            steps.append(dict(targets=tg, x=torch.randn(n * T, shape.hidden,
                                                         generator=g).cuda()))
    runs = []
    for graph in (False, True):
        tr = DecoderTrainer(shape, **mode)
        tr.load(blocks, head, emb=table if mode.get("embedding") else None)
        losses = []
        for i, kw in enumerate(steps):
            fn = tr.train_step_graph if (graph and i > 0) else tr.train_step
            losses.append(fn(**kw).clone())
        torch.cuda.synchronize()
        runs.append((tr, losses))
    (a, la), (b, lb) = runs
    for x, y in zip(la, lb):
        assert torch.equal(x, y)
    for name in ("w", "wb", "g", "m", "v", "step_dev"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    if mode.get("embedding"):
        assert torch.equal(a.emb, b.emb)
    assert int(b.step_dev) == 3
