"""Oracle checks against fixtures stored under tests/golden/, each holding the
inputs and the pass criterion a page prints (the file's "source" names it).

wgpu_toy_convergence.json: the toy convergence test of the wgpu_trainer.rs
page (FALSIFY-WGPU-002) trains the LM head alone on fixed hidden states and
requires the best loss of 50 AdamW steps at learning rate 5e-2 to fall below
0.9 of the first. Reading: the head here is this path's (final RMSNorm with a
unit gain, the LM head, mean cross-entropy), the optimizer this path's AdamW
with its global clip; the other hyper-parameters are the workload's."""
import json
import os
import types

import numpy as np

from oracle import model as om
from resident_decoder_trainer_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def test_fixture_holds_the_pages_generator_values():
    fx = _load("wgpu_toy_convergence.json")
    H, V = fx["hidden_size"], fx["vocab_size"]
    T = len(fx["target_ids"])
    assert len(fx["hidden"]) == T * H and len(fx["lm_head"]) == V * H
    # the page's generators, evaluated independently of the stored lists
    assert fx["hidden"] == [((i * 7 + 3) % 100) / 100.0 - 0.5 for i in range(T * H)]
    assert fx["lm_head"] == [((i * 13 + 7) % 100) / 100.0 - 0.5 for i in range(V * H)]
    assert all(0 <= t < V for t in fx["target_ids"])


def test_lm_head_toy_training_converges_as_the_page_requires():
    fx = _load("wgpu_toy_convergence.json")
    H, V = fx["hidden_size"], fx["vocab_size"]
    T = len(fx["target_ids"])
    h = np.asarray(fx["hidden"], dtype=np.float64).reshape(T, H)
    w = np.asarray(fx["lm_head"], dtype=np.float64).reshape(V, H)
    tg = np.asarray(fx["target_ids"])
    o = dict(synth.OPTIM)
    shape = types.SimpleNamespace(eps=synth.WORKLOADS["tiny"].eps)
    m = np.zeros_like(w)
    v = np.zeros_like(w)
    losses = []
    for step in range(1, fx["steps"] + 1):
        res = om.head_forward_backward(h, np.ones(H), w, tg, shape)
        losses.append(res["loss"])
        scale, _, finite = om.clip_scale([om.squared_sum(res["w_lm"])], o["max_norm"])
        assert finite
        w, m, v = om.adamw(w, res["w_lm"], m, v, step, fx["lr"], o["beta1"], o["beta2"],
                           o["eps"], o["weight_decay"], scale)
    assert np.isfinite(losses[0])
    assert min(losses) < fx["best_over_first_below"] * losses[0], (losses[0], min(losses))
    # a sign error in the update (ascent) fails the same criterion
    w0 = np.asarray(fx["lm_head"], dtype=np.float64).reshape(V, H)
    wa, ma, va = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    asc = []
    for step in range(1, fx["steps"] + 1):
        res = om.head_forward_backward(h, np.ones(H), wa, tg, shape)
        asc.append(res["loss"])
        wa, ma, va = om.adamw(wa, -res["w_lm"], ma, va, step, fx["lr"], o["beta1"], o["beta2"],
                              o["eps"], o["weight_decay"])
    assert not min(asc) < fx["best_over_first_below"] * asc[0]
