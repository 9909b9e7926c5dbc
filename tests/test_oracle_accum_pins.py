"""Pins for the oracle's gradient accumulation (``oracle.model.accumulated_gradients``
/ ``train_step_accumulated``): micro-batches that are the sequences of one
batch must give exactly (up to fp64 rounding) the gradients of that batch in
one pass, since the loss is the mean over all tokens and the sequences are
independent; one micro-batch is ``train_step`` itself; and a planted mistake
(the 1/n loss scale dropped) is caught."""
import numpy as np

from oracle import model as om
from resident_decoder_trainer_gb300 import synth

SHAPE = synth.WORKLOADS["tiny"].replace(layers=2)


def _inputs(batch, seed=4):
    s = SHAPE.replace(batch=batch)
    blocks, head, x, tg = synth.make_model_inputs(s, seed)
    return s, blocks, head, om._f64(x), tg.numpy()


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def test_micro_batches_of_sequences_equal_the_whole_batch():
    s3, blocks, head, x, tg = _inputs(batch=3)
    T = SHAPE.seq
    whole = om.train_step(blocks, head, x, tg, s3, step=1, optim=synth.OPTIM)
    s1 = SHAPE.replace(batch=1)
    xs = [x[i * T:(i + 1) * T] for i in range(3)]
    ts = [tg[i * T:(i + 1) * T] for i in range(3)]
    acc = om.train_step_accumulated(blocks, head, xs, ts, s1, step=1, optim=synth.OPTIM)
    assert abs(acc["loss"] - whole["loss"]) < 1e-12 * whole["loss"]
    assert np.max(np.abs(acc["loss_partials"] - whole["loss_partials"])) < 1e-12
    for key, g in whole["grads"].items():
        assert _rel(acc["grads"][key], g) < 1e-12, key
    assert abs(acc["norm"] - whole["norm"]) < 1e-12 * whole["norm"]
    for key, w in whole["params"].items():
        assert np.max(np.abs(acc["params"][key] - w)) < 1e-12, key


def test_one_micro_batch_is_the_plain_step():
    s1, blocks, head, x, tg = _inputs(batch=1)
    plain = om.train_step(blocks, head, x, tg, s1, step=1, optim=synth.OPTIM)
    acc = om.train_step_accumulated(blocks, head, [x], [tg], s1, step=1, optim=synth.OPTIM)
    for key, g in plain["grads"].items():
        assert np.array_equal(acc["grads"][key], g), key
    for key, w in plain["params"].items():
        assert np.array_equal(acc["params"][key], w), key


def test_planted_missing_loss_scale_is_caught():
    """Summing micro-batch gradients of the per-micro-batch mean loss (1/T
    instead of 1/(T n)) gives n times the whole-batch gradient."""
    s2, blocks, head, x, tg = _inputs(batch=2)
    T = SHAPE.seq
    whole = om.train_step(blocks, head, x, tg, s2, step=1, optim=synth.OPTIM)
    s1 = SHAPE.replace(batch=1)
    total = None
    for i in range(2):
        res, bgrads = om.model_forward_backward(blocks, head, x[i * T:(i + 1) * T],
                                                tg[i * T:(i + 1) * T], s1, loss_scale=1.0 / T)
        total = res["w_lm"] if total is None else total + res["w_lm"]
    assert _rel(total, whole["grads"][("head", "w_lm")]) > 0.5
