"""Pins for the FP64 oracle: each check ties the oracle to something other
than itself -- finite differences, closed forms, invariants, brute-force loops
over the definition, or a library routine for a special case. Chosen so that a
dropped term, a wrong sign or index, or a transposed operand anywhere in
``oracle.model`` fails at least one of them (``test_planted_mistakes_are_caught``
plants such mistakes and checks that they are)."""
import math

import numpy as np
import pytest

from oracle import model as om
from resident_decoder_trainer_gb300 import synth

TINY = synth.WORKLOADS["tiny"]


def _rand_block(shape, rng, std=0.06, gain_jitter=0.2):
    """Tiny block with gains away from 1 so that a dropped gain shows up."""
    shp = synth.block_shapes(shape)
    p = {}
    for k, s in shp.items():
        if k.startswith("g_"):
            p[k] = 1.0 + gain_jitter * rng.standard_normal(s)
        else:
            p[k] = std * rng.standard_normal(s)
    return p


def _small_shape(**kw):
    base = dict(layers=2, hidden=16, n_heads=4, n_kv_heads=2, head_dim=4, intermediate=24,
                vocab=11, seq=5, batch=2, eps=1e-6, theta=100.0)
    base.update(kw)
    return synth.DecoderShape(**base)


def _model(shape, seed=0):
    rng = np.random.default_rng(seed)
    blocks = [_rand_block(shape, rng) for _ in range(shape.layers)]
    head = {"g_final": 1.0 + 0.2 * rng.standard_normal(shape.hidden),
            "w_lm": 0.3 * rng.standard_normal((shape.vocab, shape.hidden))}
    x = rng.standard_normal((shape.tokens, shape.hidden))
    tg = rng.integers(0, shape.vocab, shape.tokens)
    return blocks, head, x, tg


def _loss(blocks, head, x, tg, shape):
    h = x
    for p in blocks:
        h, _ = om.block_forward(p, h, shape)
    return om.head_forward_backward(h, head["g_final"], head["w_lm"], tg, shape)["loss"]


# --------------------------------------------------------------------------
# Whole backward vs central finite differences (fp64)
# --------------------------------------------------------------------------
def _fd_check(shape, seed=0, per_tensor=12, rel_tol=1e-6):
    blocks, head, x, tg = _model(shape, seed)
    res, bgrads = om.model_forward_backward(blocks, head, x, tg, shape)
    rng = np.random.default_rng(seed + 100)
    worst = 0.0

    def check(arr, grad, name):
        nonlocal worst
        flat = arr.reshape(-1)
        gflat = grad.reshape(-1)
        idx = rng.choice(flat.size, size=min(per_tensor, flat.size), replace=False)
        fd = np.empty(idx.size)
        for j, i in enumerate(idx):
            h = 1e-6 * max(1.0, abs(flat[i]))
            old = flat[i]
            flat[i] = old + h
            lp = _loss(blocks, head, x, tg, shape)
            flat[i] = old - h
            lm = _loss(blocks, head, x, tg, shape)
            flat[i] = old
            fd[j] = (lp - lm) / (2 * h)
        an = gflat[idx]
        scale = max(np.max(np.abs(an)), 1e-12)
        err = np.max(np.abs(fd - an)) / scale
        worst = max(worst, err)
        assert err < rel_tol, f"{name}: fd vs analytic rel err {err:.3e}"

    for li, p in enumerate(blocks):
        for k in p:
            check(p[k], bgrads[li][k], f"block{li}.{k}")
    check(head["g_final"], res["g_final"], "g_final")
    check(head["w_lm"], res["w_lm"], "w_lm")
    check(x, res["dx"], "x")
    return worst


def test_finite_difference_whole_backward():
    _fd_check(_small_shape())


def test_finite_difference_mha_and_single_sequence():
    _fd_check(_small_shape(n_kv_heads=4, batch=1, seq=7, layers=1), seed=3)


def test_finite_difference_tiny_workload_shape():
    # the tiny workload's own shape, with its N(0, 0.02) weights and unit gains
    blocks, head, x, tg = synth.make_model_inputs(TINY, seed=0)
    blocks = [{k: om._f64(v) for k, v in b.items()} for b in blocks]
    head = {k: om._f64(v) for k, v in head.items()}
    x = om._f64(x)
    tg = np.asarray(tg)
    res, bgrads = om.model_forward_backward(blocks, head, x, tg, TINY)
    rng = np.random.default_rng(7)
    for arr, grad in [(blocks[0]["wq"], bgrads[0]["wq"]), (blocks[1]["wd"], bgrads[1]["wd"]),
                      (blocks[0]["g_k"], bgrads[0]["g_k"]), (head["w_lm"], res["w_lm"])]:
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        idx = np.argsort(-np.abs(gflat))[:4].tolist() + rng.choice(flat.size, 4).tolist()
        for i in idx:
            h = 1e-5
            old = flat[i]
            flat[i] = old + h
            lp = _loss(blocks, head, x, tg, TINY)
            flat[i] = old - h
            lm = _loss(blocks, head, x, tg, TINY)
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - gflat[i]) <= 1e-6 * np.max(np.abs(gflat)) + 1e-10


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------
def test_causal_softmax_rows_sum_to_one_and_zero_above_diagonal():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((9, 8)), rng.standard_normal((9, 8))
    P = om.attention_probs(q, k)
    assert np.allclose(P.sum(axis=-1), 1.0, atol=1e-14)
    assert np.all(P[np.triu_indices(9, 1)] == 0.0)
    assert np.all(P[np.tril_indices(9)] > 0.0)


def _attention_loops(q, k, v, batch, seq):
    """Brute force: explicit loops, the causal mask as loop bounds."""
    T, nh, d = q.shape
    nkv = k.shape[1]
    o = np.zeros_like(q)
    for b in range(batch):
        for h in range(nh):
            g = h * nkv // nh
            for i in range(seq):
                ti = b * seq + i
                s = [sum(q[ti, h, c] * k[b * seq + j, g, c] for c in range(d)) / math.sqrt(d)
                     for j in range(i + 1)]
                mx = max(s)
                w = [math.exp(sj - mx) for sj in s]
                den = sum(w)
                for c in range(d):
                    o[ti, h, c] = sum(w[j] * v[b * seq + j, g, c] for j in range(i + 1)) / den
    return o


def test_attention_matches_brute_force_loops():
    rng = np.random.default_rng(2)
    batch, seq, nh, nkv, d = 2, 5, 4, 2, 3
    q = rng.standard_normal((batch * seq, nh, d))
    k = rng.standard_normal((batch * seq, nkv, d))
    v = rng.standard_normal((batch * seq, nkv, d))
    assert np.allclose(om.attention(q, k, v, batch, seq), _attention_loops(q, k, v, batch, seq),
                       atol=1e-13)


def test_gqa_equals_expanded_mha_forward_and_backward():
    rng = np.random.default_rng(3)
    batch, seq, nh, nkv, d = 1, 6, 4, 2, 5
    q = rng.standard_normal((seq, nh, d))
    k = rng.standard_normal((seq, nkv, d))
    v = rng.standard_normal((seq, nkv, d))
    do = rng.standard_normal((seq, nh, d))
    ke, ve = np.repeat(k, nh // nkv, axis=1), np.repeat(v, nh // nkv, axis=1)
    assert np.allclose(om.attention(q, k, v, batch, seq), om.attention(q, ke, ve, batch, seq),
                       atol=1e-14)
    dq, dk, dv = om.attention_backward(do, q, k, v, batch, seq)
    dqe, dke, dve = om.attention_backward(do, q, ke, ve, batch, seq)
    assert np.allclose(dq, dqe, atol=1e-13)
    assert np.allclose(dk, dke.reshape(seq, nkv, nh // nkv, d).sum(axis=2), atol=1e-13)
    assert np.allclose(dv, dve.reshape(seq, nkv, nh // nkv, d).sum(axis=2), atol=1e-13)


def test_attention_single_position_returns_v():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((3, 4, 8))
    k = rng.standard_normal((3, 2, 8))
    v = rng.standard_normal((3, 2, 8))
    o = om.attention(q, k, v, batch=3, seq=1)
    assert np.allclose(o, np.repeat(v, 2, axis=1), atol=1e-15)


# --------------------------------------------------------------------------
# RMSNorm
# --------------------------------------------------------------------------
def test_rmsnorm_unit_rms_with_unit_gain():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 33)) * 3.0
    eps = 1e-6
    y, _ = om.rmsnorm(x, np.ones(33), eps)
    ms = np.mean(x * x, axis=-1)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0 / np.sqrt(1.0 + eps / ms), atol=1e-14)


def test_rmsnorm_gain_scales_columns():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((4, 9))
    gam = rng.standard_normal(9)
    y1, _ = om.rmsnorm(x, np.ones(9), 1e-6)
    y2, _ = om.rmsnorm(x, gam, 1e-6)
    assert np.allclose(y2, y1 * gam, atol=1e-14)


def test_rmsnorm_backward_orthogonal_to_input():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 16))
    dy = rng.standard_normal((5, 16))
    _, cache = om.rmsnorm(x, np.ones(16), 0.0)
    dx, _ = om.rmsnorm_backward(dy, cache, np.ones(16))
    assert np.allclose(np.sum(dx * x, axis=-1), 0.0, atol=1e-12)


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------
def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((1, 3, 8))
    c, s = om.rope_angles([0], 8, 1e4)
    assert np.array_equal(om.rope(x, c, s), x)


def test_rope_is_complex_multiplication():
    rng = np.random.default_rng(9)
    d, theta = 8, 1e4
    pos = np.array([0, 1, 5, 1000])
    x = rng.standard_normal((4, 2, d))
    c, s = om.rope_angles(pos, d, theta)
    y = om.rope(x, c, s)
    for t, p in enumerate(pos):
        for h in range(2):
            for i in range(d // 2):
                ang = p / theta ** (2 * i / d)
                z = complex(x[t, h, i], x[t, h, i + d // 2]) * complex(math.cos(ang),
                                                                       math.sin(ang))
                assert abs(y[t, h, i] - z.real) < 1e-12
                assert abs(y[t, h, i + d // 2] - z.imag) < 1e-12


def test_rope_backward_is_inverse_rotation():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((6, 3, 16))
    c, s = om.rope_angles(np.arange(6) * 37, 16, 1e6)
    y = om.rope(x, c, s)
    assert np.allclose(om.rope_backward(y, c, s), x, atol=1e-13)
    half = 8
    assert np.allclose(y[..., :half] ** 2 + y[..., half:] ** 2,
                       x[..., :half] ** 2 + x[..., half:] ** 2, atol=1e-12)


# --------------------------------------------------------------------------
# Cross-entropy head
# --------------------------------------------------------------------------
def test_cross_entropy_of_zero_logits_is_log_vocab():
    shape = _small_shape(vocab=37)
    rng = np.random.default_rng(11)
    h = rng.standard_normal((shape.tokens, shape.hidden))
    tg = rng.integers(0, 37, shape.tokens)
    r = om.head_forward_backward(h, np.ones(shape.hidden), np.zeros((37, shape.hidden)), tg,
                                 shape, keep_dz=True)
    assert np.allclose(r["loss_partials"], math.log(37), atol=1e-14)
    T = shape.tokens
    expect = np.full((T, 37), 1.0 / 37)
    expect[np.arange(T), tg] -= 1.0
    assert np.allclose(r["dz"], expect / T, atol=1e-15)
    assert np.allclose(r["dz"].sum(axis=-1), 0.0, atol=1e-15)
    assert np.all(r["dh"] == 0.0)


def test_cross_entropy_matches_scipy_logsumexp_and_loops():
    scipy_special = pytest.importorskip("scipy.special")
    shape = _small_shape(vocab=13)
    rng = np.random.default_rng(12)
    h = rng.standard_normal((shape.tokens, shape.hidden))
    g = 1.0 + 0.1 * rng.standard_normal(shape.hidden)
    w = rng.standard_normal((13, shape.hidden))
    tg = rng.integers(0, 13, shape.tokens)
    r = om.head_forward_backward(h, g, w, tg, shape)
    for t in range(shape.tokens):
        ms = sum(hv * hv for hv in h[t]) / shape.hidden
        hn = [h[t, c] / math.sqrt(ms + shape.eps) * g[c] for c in range(shape.hidden)]
        z = [sum(hn[c] * w[vv, c] for c in range(shape.hidden)) for vv in range(13)]
        nll = scipy_special.logsumexp(z) - z[tg[t]]
        assert abs(r["loss_partials"][t] - nll) < 1e-12
    assert abs(r["loss"] - np.mean(r["loss_partials"])) < 1e-15


# --------------------------------------------------------------------------
# Clip and AdamW
# --------------------------------------------------------------------------
def test_clip_rule_uses_sum_of_squared_sums_without_resquaring():
    # two buffers whose squared sums add to 4 * max_norm^2 -> norm = 2 max_norm
    g1 = np.array([1.2, -0.4, 0.0])
    g2 = np.array([np.sqrt(4.0 - om.squared_sum(g1))])
    sq = [om.squared_sum(g1), om.squared_sum(g2)]
    s, n, ok = om.clip_scale(sq, 1.0)
    assert ok and abs(n - 2.0) < 1e-15 and abs(s - 0.5) < 1e-15
    s, n, ok = om.clip_scale(sq, 2.0)
    assert s == 1.0
    s, n, ok = om.clip_scale(sq, 5.0)
    assert s == 1.0 and abs(n - 2.0) < 1e-15
    s, n, ok = om.clip_scale([1.0, float("inf")], 1.0)
    assert not ok
    s, n, ok = om.clip_scale([1.0, float("nan")], 1.0)
    assert not ok


def test_adamw_first_step_closed_form():
    rng = np.random.default_rng(13)
    w = rng.standard_normal(50)
    g = rng.standard_normal(50) * 1e-3
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.95, 1e-8, 0.1
    w1, m1, v1 = om.adamw(w, g, np.zeros(50), np.zeros(50), 1, lr, b1, b2, eps, wd)
    expect = w - lr * g / (np.abs(g) + eps) - lr * wd * w
    assert np.allclose(w1, expect, rtol=0, atol=1e-15)
    assert np.allclose(m1, (1 - b1) * g) and np.allclose(v1, (1 - b2) * g * g)
    # with a clip scale the first step is unchanged in direction (scale-invariant
    # up to eps) and the moments carry the scaled gradient
    w2, m2, _ = om.adamw(w, g, np.zeros(50), np.zeros(50), 1, lr, b1, b2, eps, wd, scale=0.5)
    assert np.allclose(m2, (1 - b1) * 0.5 * g)
    assert np.allclose(w2, w - lr * 0.5 * g / (np.abs(0.5 * g) + eps) - lr * wd * w, atol=1e-15)


def test_adamw_second_step_bias_correction():
    w, g1, g2 = np.array([0.5]), np.array([0.2]), np.array([-0.1])
    lr, b1, b2, eps, wd = 1e-2, 0.9, 0.95, 1e-8, 0.0
    w1, m1, v1 = om.adamw(w, g1, np.zeros(1), np.zeros(1), 1, lr, b1, b2, eps, wd)
    w2, m2, v2 = om.adamw(w1, g2, m1, v1, 2, lr, b1, b2, eps, wd)
    m = 0.9 * 0.1 * 0.2 + 0.1 * -0.1
    v = 0.95 * 0.05 * 0.04 + 0.05 * 0.01
    step = (m / (1 - 0.81)) / (math.sqrt(v / (1 - 0.9025)) + eps)
    assert abs(w2[0] - (w1[0] - lr * step)) < 1e-15


# --------------------------------------------------------------------------
# Block-level special cases with closed forms
# --------------------------------------------------------------------------
def test_block_is_identity_when_output_projections_are_zero():
    shape = _small_shape()
    rng = np.random.default_rng(14)
    p = _rand_block(shape, rng)
    p["wo"][:] = 0.0
    p["wd"][:] = 0.0
    x = rng.standard_normal((shape.tokens, shape.hidden))
    y, cache = om.block_forward(p, x, shape)
    assert np.array_equal(y, x)
    dy = rng.standard_normal(x.shape)
    dx, grads = om.block_backward(cache, dy, shape)
    assert np.allclose(dx, dy, atol=1e-15)
    assert np.allclose(grads["wd"], dy.T @ cache["sw"])


def test_block_attention_is_causal_mean_of_values_when_queries_vanish():
    shape = _small_shape()
    rng = np.random.default_rng(15)
    p = _rand_block(shape, rng)
    p["wq"][:] = 0.0  # q = 0 -> QK-norm(0) = 0 -> all scores 0 -> uniform causal weights
    p["wd"][:] = 0.0
    x = rng.standard_normal((shape.tokens, shape.hidden))
    y, _ = om.block_forward(p, x, shape)
    xn, _ = om.rmsnorm(x, p["g_attn"], shape.eps)
    v = (xn @ p["wv"].T).reshape(shape.tokens, shape.n_kv_heads, shape.head_dim)
    o = np.zeros((shape.tokens, shape.n_heads, shape.head_dim))
    rep = shape.n_heads // shape.n_kv_heads
    for b in range(shape.batch):
        for i in range(shape.seq):
            t = b * shape.seq + i
            for h in range(shape.n_heads):
                o[t, h] = v[b * shape.seq:t + 1, h // rep].mean(axis=0)
    assert np.allclose(y, x + o.reshape(shape.tokens, -1) @ p["wo"].T, atol=1e-13)


def test_ffn_matches_elementwise_loops():
    shape = _small_shape(hidden=6, intermediate=5, seq=2, batch=1)
    rng = np.random.default_rng(16)
    p = _rand_block(shape, rng)
    p["wo"][:] = 0.0  # r1 = x
    x = rng.standard_normal((shape.tokens, shape.hidden))
    y, _ = om.block_forward(p, x, shape)
    H, I = shape.hidden, shape.intermediate
    for t in range(shape.tokens):
        ms = sum(x[t, c] ** 2 for c in range(H)) / H
        xn = [x[t, c] / math.sqrt(ms + shape.eps) * p["g_ffn"][c] for c in range(H)]
        s = []
        for j in range(I):
            gg = sum(xn[c] * p["wg"][j, c] for c in range(H))
            uu = sum(xn[c] * p["wu"][j, c] for c in range(H))
            s.append(gg / (1.0 + math.exp(-gg)) * uu)
        for c in range(H):
            ref = x[t, c] + sum(s[j] * p["wd"][c, j] for j in range(I))
            assert abs(y[t, c] - ref) < 1e-13


def test_toy_training_loss_falls():
    # the pages' toy-convergence contract, as a sanity check of the whole step
    shape = TINY
    blocks, head, x, tg = synth.make_model_inputs(shape, seed=0)
    blocks = [{k: om._f64(v) for k, v in b.items()} for b in blocks]
    head = {k: om._f64(v) for k, v in head.items()}
    optim = dict(synth.OPTIM, lr=1e-2)
    state, losses = None, []
    for step in range(1, 16):
        r = om.train_step(blocks, head, x, np.asarray(tg), shape, state=state, step=step,
                          optim=optim)
        losses.append(r["loss"])
        state = r["state"]
        for (li, name), w in r["params"].items():
            (head if li == "head" else blocks[li])[name] = w
    assert losses[0] == pytest.approx(math.log(256), rel=0.05)
    assert min(losses) < 0.9 * losses[0]


# --------------------------------------------------------------------------
# Planted mistakes must be caught by the pins above
# --------------------------------------------------------------------------
def _planted(monkeypatch, name, fn):
    monkeypatch.setattr(om, name, fn)


def test_planted_mistakes_are_caught(monkeypatch):
    orig_rope_bwd = om.rope_backward
    orig_silu_grad = om.silu_grad
    orig_rms_bwd = om.rmsnorm_backward
    orig_attn_bwd = om.attention_backward
    mistakes = {
        "rope_backward sign": ("rope_backward",
                               lambda dy, c, s: orig_rope_bwd(dy, c, -s)),
        "silu' dropped term": ("silu_grad", lambda z: om.sigmoid(z)),
        "rmsnorm dgamma dropped": ("rmsnorm_backward",
                                   lambda dy, cache, g: (orig_rms_bwd(dy, cache, g)[0],
                                                         0 * orig_rms_bwd(dy, cache, g)[1])),
        "rmsnorm gain not applied in dx": ("rmsnorm_backward",
                                           lambda dy, cache, g: orig_rms_bwd(dy, cache,
                                                                             np.ones_like(g))),
        "attention dk transposed": ("attention_backward",
                                    lambda do, q, k, v, b, s: (
                                        orig_attn_bwd(do, q, k, v, b, s)[0],
                                        orig_attn_bwd(do, q, k, v, b, s)[1][:, ::-1],
                                        orig_attn_bwd(do, q, k, v, b, s)[2])),
    }
    for label, (name, fn) in mistakes.items():
        with monkeypatch.context() as mp:
            mp.setattr(om, name, fn)
            with pytest.raises(AssertionError):
                _fd_check(_small_shape(layers=1), per_tensor=6)
        del label
    # the unmodified oracle passes the same check
    _fd_check(_small_shape(layers=1), per_tensor=6)
    assert om.silu_grad is orig_silu_grad
