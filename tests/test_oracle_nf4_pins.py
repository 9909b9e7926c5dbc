"""Pins for the NF4 + LoRA oracle (``oracle/nf4.py``): the NF4 levels against
their construction from normal quantiles, the unpacking order and block
scales against hand-built bytes, the LoRA projection against the two-step
loops of its definition, the adapter gradients against finite differences,
and the special cases (B = 0 gives the base block and dA = 0; AdamW's first
step in closed form). A planted mistake in each gradient formula is caught."""
import numpy as np
import pytest

from oracle import model as om
from oracle import nf4
from resident_decoder_trainer_gb300 import synth

# tiny NF4 block: every projection's input width a multiple of 64
SHAPE = synth.DecoderShape(layers=1, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16,
                           intermediate=128, vocab=256, seq=24, batch=1, eps=1e-6, theta=1e4)
RANK, ALPHA = 4, 8.0


def _inputs(b_std=0.05, seed=3):
    base_q, gains, lora, x, dy = synth.make_nf4_inputs(SHAPE, seed=seed, rank=RANK, b_std=b_std)
    shp = synth.block_shapes(SHAPE)
    base = {k: nf4.nf4_dequantize(p.numpy(), a.numpy(), *shp[k]) for k, (p, a) in base_q.items()}
    gains = {k: v.numpy().astype(np.float64) for k, v in gains.items()}
    lora = {k: v.numpy().astype(np.float64) for k, v in lora.items()}
    return base, gains, lora, om._f64(x), om._f64(dy)


# ------------------------------------------------------------------ NF4 levels
def test_nf4_levels_are_the_normal_quantile_construction():
    """QLoRA's NormalFloat-4: 8 positive levels at the normal quantiles of 8
    points evenly spaced from `offset` down to 1/2, 7 negative levels the same
    with 7 points, and 0; all divided by the largest. offset = 1 - (1/30 +
    1/32)/2 puts the extreme quantile half-way between the outermost
    probabilities of a 15- and a 16-level grid."""
    from scipy.stats import norm
    offset = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    pos = norm.ppf(np.linspace(offset, 0.5, 9)[:-1])
    neg = -norm.ppf(np.linspace(offset, 0.5, 8)[:-1])
    levels = np.sort(np.concatenate([pos, [0.0], neg]))
    levels /= levels.max()
    assert len(nf4.NF4_LEVELS) == 16
    assert np.max(np.abs(levels - nf4.NF4_LEVELS)) < 1e-6
    assert nf4.NF4_LEVELS[7] == 0.0 and nf4.NF4_LEVELS[0] == -1.0 and nf4.NF4_LEVELS[15] == 1.0
    assert np.all(np.diff(nf4.NF4_LEVELS) > 0)


def test_nf4_unpack_order_and_block_scales():
    # one row of 128 elements = two blocks of 64; byte j -> elements 2j (low), 2j+1 (high)
    packed = np.zeros((1, 64), dtype=np.uint8)
    packed[0, 0] = 0x5A          # element 0 = code 10, element 1 = code 5
    packed[0, 31] = 0xF0         # element 62 = code 0, element 63 = code 15
    packed[0, 32] = 0x77         # elements 64, 65 = code 7 (the zero level)
    packed[0, 1:31] = 0x77
    packed[0, 33:] = 0x77
    absmax = np.array([2.0, 0.5])
    w = nf4.nf4_dequantize(packed, absmax, 1, 128)
    assert w[0, 0] == nf4.NF4_LEVELS[10] * 2.0
    assert w[0, 1] == nf4.NF4_LEVELS[5] * 2.0
    assert w[0, 62] == -2.0 and w[0, 63] == 2.0
    assert np.all(w[0, 64:] == 0.0)
    # blocks run over the flattened row-major weight, across rows
    rng = np.random.default_rng(0)
    packed = rng.integers(0, 256, (6, 16), dtype=np.uint8)  # [6, 32] weight, 192 elements
    absmax = np.abs(rng.standard_normal(3)) + 0.1
    w = nf4.nf4_dequantize(packed, absmax, 6, 32)
    flat = w.reshape(-1)
    for b in range(3):
        assert np.max(np.abs(flat[64 * b:64 * (b + 1)])) <= absmax[b] + 1e-15


# ---------------------------------------------------------------- LoRA forward
def test_lora_projection_equals_its_two_step_loops():
    """x (W + s B A)^T == x W^T + s (x A^T) B^T, the latter as explicit loops
    (wgpu_trainer.rs `lora_forward`)."""
    rng = np.random.default_rng(1)
    t, inn, out, r = 5, 7, 6, 3
    x = rng.standard_normal((t, inn))
    w = rng.standard_normal((out, inn))
    a = rng.standard_normal((r, inn))
    b = rng.standard_normal((out, r))
    s = nf4.lora_scale(r, 6.0)
    merged = x @ (w + s * (b @ a)).T
    y = np.zeros((t, out))
    for i in range(t):
        h = [sum(x[i, p] * a[j, p] for p in range(inn)) for j in range(r)]
        for o in range(out):
            base = sum(x[i, p] * w[o, p] for p in range(inn))
            y[i, o] = base + s * sum(h[j] * b[o, j] for j in range(r))
    assert np.max(np.abs(merged - y)) < 1e-12


def test_zero_b_gives_the_base_block_and_zero_da():
    base, gains, lora, x, dy = _inputs(b_std=0.0)
    y, dx, g = nf4.lora_forward_backward(base, gains, lora, x, dy, SHAPE, RANK, ALPHA)
    p = dict(base)
    p.update(gains)
    y0, cache = om.block_forward(p, x, SHAPE)
    dx0, _ = om.block_backward(cache, dy, SHAPE)
    assert np.array_equal(y, y0) and np.array_equal(dx, dx0)
    for name in nf4.PROJECTIONS:
        assert np.all(g["a_" + name[1:]] == 0.0)
        assert np.any(g["b_" + name[1:]] != 0.0)


# --------------------------------------------------------------- LoRA backward
def _loss(base, gains, lora, x, r):
    p = nf4.merged_params(base, gains, lora, nf4.lora_scale(RANK, ALPHA))
    y, _ = om.block_forward(p, x, SHAPE)
    return float(np.sum(y * r))


def _fd_check(grad_fn, base, gains, lora, x, dy, n_samples=3, seed=0):
    _, _, g = grad_fn(base, gains, lora, x, dy, SHAPE, RANK, ALPHA)
    rng = np.random.default_rng(seed)
    worst = 0.0
    for key in sorted(g):
        for _ in range(n_samples):
            idx = tuple(rng.integers(0, n) for n in lora[key].shape)
            h = 1e-4 * max(1.0, abs(lora[key][idx]))  # central: O(h^2) truncation
            lp = {k: v.copy() for k, v in lora.items()}
            lm = {k: v.copy() for k, v in lora.items()}
            lp[key][idx] += h
            lm[key][idx] -= h
            fd = (_loss(base, gains, lp, x, dy) - _loss(base, gains, lm, x, dy)) / (2 * h)
            scale = max(abs(fd), 1e-3 * float(np.max(np.abs(g[key]))), 1e-12)
            worst = max(worst, abs(g[key][idx] - fd) / scale)
    return worst


def test_adapter_gradients_match_finite_differences():
    base, gains, lora, x, dy = _inputs(b_std=0.05)
    assert _fd_check(nf4.lora_forward_backward, base, gains, lora, x, dy) < 1e-6


@pytest.mark.parametrize("mistake", ["da_no_scale", "db_transposed_a"])
def test_planted_adapter_gradient_mistakes_are_caught(mistake):
    base, gains, lora, x, dy = _inputs(b_std=0.05)

    def wrong(base, gains, lora, x, dy, shape, rank, alpha):
        s = nf4.lora_scale(rank, alpha)
        p = nf4.merged_params(base, gains, lora, s)
        y, cache = om.block_forward(p, x, shape)
        dx, grads = om.block_backward(cache, dy, shape)
        g = {}
        for name in nf4.PROJECTIONS:
            dw, a, b = grads[name], lora["a_" + name[1:]], lora["b_" + name[1:]]
            g["a_" + name[1:]] = (b.T @ dw) if mistake == "da_no_scale" else s * (b.T @ dw)
            if mistake == "db_transposed_a":
                # B-gradient formed from A's transpose taken over the wrong axis
                g["b_" + name[1:]] = s * (dw @ np.flip(a, axis=1).T)
            else:
                g["b_" + name[1:]] = s * (dw @ a.T)
        return y, dx, g

    assert _fd_check(wrong, base, gains, lora, x, dy) > 1e-3


# ----------------------------------------------------------------------- step
def test_adapters_only_step_first_adamw_step_closed_form():
    base, gains, lora, x, dy = _inputs(b_std=0.05)
    o = synth.OPTIM
    res = nf4.lora_step(base, gains, lora, x, dy, SHAPE, RANK, ALPHA, o)
    assert res["scale"] == 1.0  # tiny gradients, far below max_norm
    for k, g in res["grads"].items():
        w = lora[k]
        want = w - o["lr"] * (g / (np.abs(g) + o["eps"]) + o["weight_decay"] * w)
        assert np.max(np.abs(res["params"][k] - want)) < 1e-12
