"""Pin of the oracle's block composition against per-token loops.

The pieces of ``oracle.model.block_forward`` are pinned one by one elsewhere
(RMSNorm, RoPE, attention, the FFN). What those pins cannot see is how the
block puts them together on the q/k path, as cuda_block.rs describes it in
``compute_attention_cuda`` and in the NF4 block forward's stated order
"projection -> QK-norm -> RoPE -> attention": the per-head RMSNorm over
head_dim comes first and uses gamma_q for queries and gamma_k for keys, the
rotation follows it, and a token's rotation angle is its position inside its
own sequence (p = t mod S), so every sequence of a batch starts at 0.

A mistake in that composition, made the same way in the forward and in the
backward, keeps the finite-difference pins green, because those check only
that the backward is the derivative of whatever the forward computes.
``test_composition_mistakes_pass_finite_differences_but_not_the_loops``
plants three such mistakes consistently and shows both facts.

The loops below use the ``math`` module only: nothing from the oracle, and no
array library, so that they restate the definition independently.
"""
import math

import numpy as np
import pytest

from oracle import model as om

from test_oracle_pins import _fd_check, _rand_block, _small_shape


def _loop_block_forward(p, x, sh):
    """One decoder block written out token by token."""
    B, S, H = sh.batch, sh.seq, sh.hidden
    nh, nkv, d, I = sh.n_heads, sh.n_kv_heads, sh.head_dim, sh.intermediate
    eps, theta = sh.eps, sh.theta
    T, rep, half = B * S, nh // nkv, d // 2
    P = {k: np.asarray(v, dtype=np.float64).tolist() for k, v in p.items()}
    X = np.asarray(x, dtype=np.float64).tolist()

    def norm(vec, gain):
        r = 1.0 / math.sqrt(sum(a * a for a in vec) / len(vec) + eps)
        return [a * r * g for a, g in zip(vec, gain)]

    def matvec(W, vec):
        return [sum(row[j] * vec[j] for j in range(len(vec))) for row in W]

    def rotate(vec, pos):
        out = list(vec)
        for i in range(half):
            ang = pos * theta ** (-2.0 * i / d)
            c, s = math.cos(ang), math.sin(ang)
            out[i] = vec[i] * c - vec[i + half] * s
            out[i + half] = vec[i + half] * c + vec[i] * s
        return out

    Q, K, Vv = [], [], []
    for t in range(T):
        pos = t % S  # position inside the token's own sequence
        xn = norm(X[t], P["g_attn"])
        q, k, v = matvec(P["wq"], xn), matvec(P["wk"], xn), matvec(P["wv"], xn)
        Q.append([rotate(norm(q[h * d:(h + 1) * d], P["g_q"]), pos) for h in range(nh)])
        K.append([rotate(norm(k[g * d:(g + 1) * d], P["g_k"]), pos) for g in range(nkv)])
        Vv.append([v[g * d:(g + 1) * d] for g in range(nkv)])
    Y = []
    for t in range(T):
        first = (t // S) * S  # keys of the same sequence, up to and including t
        o = []
        for h in range(nh):
            g = h // rep
            sc = [sum(a * b for a, b in zip(Q[t][h], K[j][g])) / math.sqrt(d)
                  for j in range(first, t + 1)]
            m = max(sc)
            e = [math.exp(a - m) for a in sc]
            z = sum(e)
            o.extend(sum(e[j - first] / z * Vv[j][g][c] for j in range(first, t + 1))
                     for c in range(d))
        a = matvec(P["wo"], o)
        r1 = [X[t][c] + a[c] for c in range(H)]
        xn2 = norm(r1, P["g_ffn"])
        gg, uu = matvec(P["wg"], xn2), matvec(P["wu"], xn2)
        s = [gg[j] / (1.0 + math.exp(-gg[j])) * uu[j] for j in range(I)]
        down = matvec(P["wd"], s)
        Y.append([r1[c] + down[c] for c in range(H)])
    return np.array(Y), np.array(Q), np.array(K)


def _model(sh, seed):
    rng = np.random.default_rng(seed)
    p = _rand_block(sh, rng, std=0.3, gain_jitter=0.4)
    x = rng.standard_normal((sh.tokens, sh.hidden))
    return p, x


def _loop_mismatch(sh, seed=21):
    """Largest difference between the oracle and the loops over the block
    output and the rotated queries and keys the oracle keeps for the backward.
    (A position offset shared by a whole sequence leaves the output unchanged,
    since the rotation makes scores depend on position differences only; the
    rotated q and k show it.)"""
    p, x = _model(sh, seed)
    y, cache = om.block_forward(p, x, sh)
    y_l, q_l, k_l = _loop_block_forward(p, x, sh)
    return float(max(np.max(np.abs(y - y_l)), np.max(np.abs(cache["qr"] - q_l)),
                     np.max(np.abs(cache["kr"] - k_l))))


def test_block_forward_matches_token_loops():
    sh = _small_shape()  # 2 sequences of 5, 4 query / 2 kv heads of 4
    p, x = _model(sh, 21)
    # the inputs exercise the q/k path: live projections, distinct q and k gains
    assert min(np.abs(p[k]).max() for k in ("wq", "wk", "wv")) > 0.1
    assert np.abs(p["g_q"] - p["g_k"]).max() > 0.1
    assert sh.batch >= 2 and sh.n_heads != sh.n_kv_heads
    assert _loop_mismatch(sh) < 1e-12


def test_block_forward_matches_token_loops_mha_three_sequences():
    sh = _small_shape(n_kv_heads=2, batch=3, seq=4, head_dim=8, hidden=16, n_heads=2,
                      theta=50.0)
    assert _loop_mismatch(sh, seed=22) < 1e-12


def _rope_before_norm(mp, sh):
    """RoPE applied to the raw projections and the QK RMSNorm after it: the
    per-head norm (3-D input) rotates first, the rotation step is skipped."""
    orig_norm, orig_norm_bwd = om.rmsnorm, om.rmsnorm_backward
    orig_rope, orig_rope_bwd = om.rope, om.rope_backward
    cos, sin = om.rope_angles(om.positions_of(sh.batch, sh.seq), sh.head_dim, sh.theta)

    def norm(x, gamma, eps):
        if np.ndim(x) == 3:
            return orig_norm(orig_rope(x, cos, sin), gamma, eps)
        return orig_norm(x, gamma, eps)

    def norm_bwd(dy, cache, gamma):
        dx, dg = orig_norm_bwd(dy, cache, gamma)
        if np.ndim(dy) == 3:
            dx = orig_rope_bwd(dx, cos, sin)
        return dx, dg

    mp.setattr(om, "rope", lambda x, c, s: x)
    mp.setattr(om, "rope_backward", lambda dy, c, s: dy)
    mp.setattr(om, "rmsnorm", norm)
    mp.setattr(om, "rmsnorm_backward", norm_bwd)


def _gains_swapped(mp, sh):
    """gamma_k applied to the queries and gamma_q to the keys (and their
    gradients reported under each other's name)."""
    orig_f, orig_b = om.block_forward, om.block_backward

    def fwd(p, x, shape):
        p2 = dict(p)
        p2["g_q"], p2["g_k"] = p["g_k"], p["g_q"]
        return orig_f(p2, x, shape)

    def bwd(cache, dy, shape):
        dx, g = orig_b(cache, dy, shape)
        g = dict(g)
        g["g_q"], g["g_k"] = g["g_k"], g["g_q"]
        return dx, g

    mp.setattr(om, "block_forward", fwd)
    mp.setattr(om, "block_backward", bwd)


def _positions_over_batch(mp, sh):
    """Positions counted over the whole batch instead of restarting at 0 in
    every sequence."""
    mp.setattr(om, "positions_of", lambda batch, seq: np.arange(batch * seq))


@pytest.mark.parametrize("plant", [_rope_before_norm, _gains_swapped, _positions_over_batch],
                         ids=["rope-before-qk-norm", "gamma-q-k-swapped",
                              "positions-over-batch"])
def test_composition_mistakes_pass_finite_differences_but_not_the_loops(monkeypatch, plant):
    sh = _small_shape(layers=1)
    with monkeypatch.context() as mp:
        plant(mp, sh)
        # forward and backward agree with each other: the derivative pins pass
        _fd_check(sh, per_tensor=6)
        # ... but the block no longer computes the definition
        assert _loop_mismatch(sh) > 1e-4
    # unplanted, both hold
    _fd_check(sh, per_tensor=6)
    assert _loop_mismatch(sh) < 1e-12
