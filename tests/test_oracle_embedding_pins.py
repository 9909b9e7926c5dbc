"""Pins for the embedding oracle (``oracle/embedding.py``): the scatter-add
gradient against finite differences of a linear functional of the lookup
(duplicate ids included, so an assignment instead of a sum is caught), the
clip scale in closed form, skipped out-of-range ids, and the embedded
model's gradient against finite differences of the model loss."""
import numpy as np

from oracle import embedding as oe
from oracle import model as om
from resident_decoder_trainer_gb300 import synth


def test_scatter_add_gradient_matches_finite_differences():
    rng = np.random.default_rng(0)
    V, H, T = 11, 6, 9
    table = rng.standard_normal((V, H))
    ids = np.array([3, 7, 3, 0, 10, 3, 7, 5, 1])  # id 3 three times, 7 twice
    w = rng.standard_normal((T, H))

    def f(e):
        return float(np.sum(w * oe.embedding_forward(e, ids)))

    de, scale = oe.embedding_grad(ids, w, V)
    assert scale == 1.0
    h = 1e-3
    for r in range(V):
        for c in range(H):
            ep, em = table.copy(), table.copy()
            ep[r, c] += h
            em[r, c] -= h
            fd = (f(ep) - f(em)) / (2 * h)
            assert abs(fd - de[r, c]) < 1e-9
    assert np.all(de[[2, 4, 6, 8, 9]] == 0.0)  # rows no token uses


def test_planted_assignment_instead_of_sum_is_caught():
    rng = np.random.default_rng(1)
    ids = np.array([2, 2, 1])
    w = rng.standard_normal((3, 4))
    wrong = np.zeros((4, 4))
    for t, tid in enumerate(ids):
        wrong[tid] = w[t]  # the mistake: duplicates overwrite
    de, _ = oe.embedding_grad(ids, w, 4)
    assert np.max(np.abs(de - wrong)) > 0.1


def test_clip_scale_closed_form_and_skipped_ids():
    """Distinct ids: ||dE|| = min(||dx||, max_norm); an id outside [0, V)
    contributes nothing (but still counts in dx's norm)."""
    rng = np.random.default_rng(2)
    dx = rng.standard_normal((5, 8)) * 10.0
    norm = float(np.sqrt(np.sum(dx * dx)))
    de, scale = oe.embedding_grad(np.array([0, 1, 2, 3, 4]), dx, 5, max_norm=1.0)
    assert abs(scale - 1.0 / norm) < 1e-15
    assert abs(np.sqrt(np.sum(de * de)) - 1.0) < 1e-12
    de2, s2 = oe.embedding_grad(np.array([0, 1, 2, 3, 99]), dx, 5, max_norm=1e9)
    assert s2 == 1.0
    assert np.array_equal(de2[:4], dx[:4]) and np.all(de2[4] == 0.0)


def test_embedded_model_gradient_matches_finite_differences():
    shape = synth.WORKLOADS["tiny"].replace(layers=1, seq=8)
    blocks, head, _, _ = synth.make_model_inputs(shape, 6)
    rng = np.random.default_rng(3)
    table = rng.standard_normal((shape.vocab, shape.hidden))
    ids = rng.integers(0, 12, shape.tokens)  # few distinct ids: duplicates
    tg = rng.integers(0, shape.vocab, shape.tokens)

    def loss(e):
        res, _ = om.model_forward_backward(blocks, head, oe.embedding_forward(e, ids), tg, shape)
        return res["loss"]

    res, _ = om.model_forward_backward(blocks, head, oe.embedding_forward(table, ids), tg, shape)
    de, _ = oe.embedding_grad(ids, res["dx"], shape.vocab)
    h = 1e-5
    for tid in sorted(set(ids.tolist()))[:3]:
        for c in (0, 5, shape.hidden - 1):
            ep, em = table.copy(), table.copy()
            ep[tid, c] += h
            em[tid, c] -= h
            fd = (loss(ep) - loss(em)) / (2 * h)
            assert abs(fd - de[tid, c]) < 1e-7 * max(1.0, abs(fd)), (tid, c)
