"""FP64 CPU oracle for one training step of a Qwen3-style decoder block stack.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module: only
the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg
of ``bench.py`` may call it. It shares no code with the CUDA path; its inputs
come from ``resident_decoder_trainer_gb300.synth`` (random draws only).

Everything here is a plain definition written out in float64 with numpy. A
matrix product (``@``) and ``exp``/``log``/``sqrt`` are the only library steps;
there is no tiling, fusion or reordering beyond the definitions.

Sources (aprender-train docs.rs pages, module ``entrenar``):

* cuda_block.rs (0.32.0) -- ``CudaTransformerBlock::forward`` (block forward),
  ``compute_attention_cuda`` (QK-norm, RoPE-neox, causal GQA attention),
  ``backward`` / ``backward_ffn`` / ``backward_post_attn_norm`` /
  ``backward_attention`` / ``reduce_gqa_gradients`` /
  ``backward_residual_and_input_norm`` (block backward), ``optimizer_step``
  (AdamW per tensor), and the NF4 block's forward for the fused residual+RMSNorm
  and the stated "projection -> QK-norm -> RoPE -> attention" order.
* cuda_trainer.rs (0.34.0) -- ``train_step_inner`` (fused cross-entropy with
  loss scale 1/T), ``gpu_forward`` (final RMSNorm, LM head), ``gpu_backward``
  (LM-head backward, final-norm backward), ``compute_workspace_clip_scale_gpu``
  / ``fused_clip_workspace_gradients`` (squared-sum clip, C-CLIP-001),
  ``run_nonblock_optimizer_step`` (AdamW, step counted from 1); R-038 gradient
  accumulation (loss scale 1/seq_len/accumulation_steps in
  ``train_step_inner``, micro-batch gradients summed before one step).
* wgpu_trainer.rs (0.38.0) -- ``train_step`` CPU cross-entropy loop (loss and
  softmax-minus-one-hot gradient) and ``ffn_backward`` (SiLU derivative).

Readings where the pages are silent or disagree (each is also listed in the
design notes): weights are [out, in] and y = x W^T; RMSNorm is
x / sqrt(mean(x^2) + eps) * gamma with the configured eps in forward and
backward alike; QK-norm gains are trainable and get the full backward the
fp32 block path omits; RoPE pairs (i, i + d/2) with angle p * theta^(-2i/d),
p the position inside its own sequence; one step covers the whole batch with
the loss averaged over all B*S tokens; one global clip over every trainable
tensor, scale = min(1, max_norm / ||g||) with no epsilon; a non-finite norm
skips the update.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against finite differences, closed forms, invariants and brute-force loops.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.asarray(a, dtype=F64)


# ----------------------------------------------------------------------------
# RMSNorm (cuda_block.rs: rms_norm_forward / rms_norm_backward call sites)
# ----------------------------------------------------------------------------
def rmsnorm(x, gamma, eps):
    """y = x * rsqrt(mean(x^2) + eps) * gamma over the last axis.

    Returns (y, cache) with cache = (xhat, rstd)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(ms + eps)
    xhat = x * rstd
    return xhat * gamma, (xhat, rstd)


def rmsnorm_backward(dy, cache, gamma):
    """Reverse of ``rmsnorm``: returns (dx, dgamma).

    With xhat = x * r and r = (mean(x^2)+eps)^-1/2:
    dx = r * (dxhat - xhat * mean(dxhat * xhat)), dxhat = dy * gamma,
    dgamma = sum over every leading index of dy * xhat."""
    xhat, rstd = cache
    dxhat = dy * gamma
    dx = rstd * (dxhat - xhat * np.mean(dxhat * xhat, axis=-1, keepdims=True))
    dgamma = (dy * xhat).reshape(-1, xhat.shape[-1]).sum(axis=0)
    return dx, dgamma


# ----------------------------------------------------------------------------
# RoPE-neox (compute_attention_cuda: batched_rope_neox_forward;
# backward_attention: "R^T(-theta)" inverse rotation)
# ----------------------------------------------------------------------------
def rope_angles(positions, head_dim, theta):
    """cos/sin tables [T, d/2]: angle(p, i) = p * theta^(-2i/d)."""
    half = head_dim // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=F64)) / head_dim)
    ang = np.asarray(positions, dtype=F64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def rope(x, cos, sin):
    """Rotate pairs (i, i + d/2) of x [T, heads, d] by the per-token angles."""
    half = x.shape[-1] // 2
    x0, x1 = x[..., :half], x[..., half:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([x0 * c - x1 * s, x1 * c + x0 * s], axis=-1)


def rope_backward(dy, cos, sin):
    """Transpose of the rotation: dx0 = dy0 cos + dy1 sin, dx1 = dy1 cos - dy0 sin."""
    half = dy.shape[-1] // 2
    d0, d1 = dy[..., :half], dy[..., half:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([d0 * c + d1 * s, d1 * c - d0 * s], axis=-1)


# ----------------------------------------------------------------------------
# Causal grouped-query attention (compute_attention_cuda, C-ATTN-001 and
# C-CAUSAL-001; backward_attention + reduce_gqa_gradients)
# ----------------------------------------------------------------------------
def attention_probs(q_h, k_g):
    """Causal softmax(q k^T / sqrt(d)) for one sequence and one head: [S, S]."""
    d = q_h.shape[-1]
    scores = (q_h @ k_g.T) / np.sqrt(d)
    S = scores.shape[0]
    mask = np.triu(np.ones((S, S), dtype=bool), k=1)  # key j > query i is masked
    scores = np.where(mask, -np.inf, scores)
    m = scores.max(axis=-1, keepdims=True)
    e = np.exp(scores - m)
    return e / e.sum(axis=-1, keepdims=True)


def attention(q, k, v, batch, seq):
    """q [T, nh, d], k/v [T, nkv, d] -> o [T, nh, d] (query head h reads kv
    head h // (nh/nkv)); every sequence of the batch attends only to itself."""
    T, nh, d = q.shape
    nkv = k.shape[1]
    rep = nh // nkv
    o = np.zeros_like(q)
    for b in range(batch):
        sl = slice(b * seq, (b + 1) * seq)
        for h in range(nh):
            g = h // rep
            P = attention_probs(q[sl, h], k[sl, g])
            o[sl, h] = P @ v[sl, g]
    return o


def attention_backward(do, q, k, v, batch, seq):
    """Reverse of ``attention``: dP = dO V^T, dS = P o (dP - rowsum(dP o P)),
    dQ = dS K / sqrt(d), dK_g = sum_{h in g} dS^T Q / sqrt(d),
    dV_g = sum_{h in g} P^T dO."""
    T, nh, d = q.shape
    nkv = k.shape[1]
    rep = nh // nkv
    c = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(batch):
        sl = slice(b * seq, (b + 1) * seq)
        for h in range(nh):
            g = h // rep
            P = attention_probs(q[sl, h], k[sl, g])
            dP = do[sl, h] @ v[sl, g].T
            dS = P * (dP - np.sum(dP * P, axis=-1, keepdims=True))
            dq[sl, h] = c * (dS @ k[sl, g])
            dk[sl, g] += c * (dS.T @ q[sl, h])
            dv[sl, g] += P.T @ do[sl, h]
    return dq, dk, dv


# ----------------------------------------------------------------------------
# SwiGLU (fused_swiglu_forward; ffn_backward's silu' = sig * (1 + x - x*sig))
# ----------------------------------------------------------------------------
def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def silu_grad(z):
    sg = sigmoid(z)
    return sg * (1.0 + z - z * sg)


# ----------------------------------------------------------------------------
# One decoder block (CudaTransformerBlock::forward / ::backward)
# ----------------------------------------------------------------------------
def positions_of(batch, seq):
    return np.tile(np.arange(seq), batch)


def block_forward(p, x, shape):
    """Pre-norm Qwen3 block. p: dict of fp32/fp64 arrays (wq, wk, wv, wo, wg,
    wu, wd [out, in]; g_attn, g_ffn [H]; g_q, g_k [d]); x [T, H].
    Returns (y, cache)."""
    s = shape
    p = {k_: _f64(v_) for k_, v_ in p.items()}
    x = _f64(x)
    T = x.shape[0]
    nh, nkv, d = s.n_heads, s.n_kv_heads, s.head_dim
    xn, c1 = rmsnorm(x, p["g_attn"], s.eps)
    q = (xn @ p["wq"].T).reshape(T, nh, d)
    k = (xn @ p["wk"].T).reshape(T, nkv, d)
    v = (xn @ p["wv"].T).reshape(T, nkv, d)
    # projection -> per-head QK RMSNorm -> RoPE -> attention
    qn, cq = rmsnorm(q, p["g_q"], s.eps)
    kn, ck = rmsnorm(k, p["g_k"], s.eps)
    cos, sin = rope_angles(positions_of(s.batch, s.seq), d, s.theta)
    qr = rope(qn, cos, sin)
    kr = rope(kn, cos, sin)
    o = attention(qr, kr, v, s.batch, s.seq).reshape(T, nh * d)
    a = o @ p["wo"].T
    r1 = x + a
    xn2, c2 = rmsnorm(r1, p["g_ffn"], s.eps)
    g = xn2 @ p["wg"].T
    u = xn2 @ p["wu"].T
    sw = silu(g) * u
    y = r1 + sw @ p["wd"].T
    cache = dict(p=p, x=x, xn=xn, c1=c1, qr=qr, kr=kr, v=v, cq=cq, ck=ck, cos=cos,
                 sin=sin, o=o, r1=r1, xn2=xn2, c2=c2, g=g, u=u, sw=sw)
    return y, cache


def block_backward(cache, dy, shape):
    """Exact reverse-mode of ``block_forward``. Returns (dx, grads dict)."""
    s = shape
    c = cache
    p = c["p"]
    dy = _f64(dy)
    T = dy.shape[0]
    nh, nkv, d = s.n_heads, s.n_kv_heads, s.head_dim
    # FFN: y = r1 + (silu(g) * u) Wd^T
    dsw = dy @ p["wd"]
    dwd = dy.T @ c["sw"]
    dg = dsw * c["u"] * silu_grad(c["g"])
    du = dsw * silu(c["g"])
    dxn2 = dg @ p["wg"] + du @ p["wu"]
    dwg = dg.T @ c["xn2"]
    dwu = du.T @ c["xn2"]
    # post-attention RMSNorm, then the identity skip added after it
    dr1, dg_ffn = rmsnorm_backward(dxn2, c["c2"], p["g_ffn"])
    dr1 = dr1 + dy
    # O projection
    do = dr1 @ p["wo"]
    dwo = dr1.T @ c["o"]
    # attention, then inverse RoPE, then the per-head QK-norm backward
    dqr, dkr, dv = attention_backward(do.reshape(T, nh, d), c["qr"], c["kr"], c["v"],
                                      s.batch, s.seq)
    dqn = rope_backward(dqr, c["cos"], c["sin"])
    dkn = rope_backward(dkr, c["cos"], c["sin"])
    dq, dg_q = rmsnorm_backward(dqn, c["cq"], p["g_q"])
    dk, dg_k = rmsnorm_backward(dkn, c["ck"], p["g_k"])
    dq = dq.reshape(T, nh * d)
    dk = dk.reshape(T, nkv * d)
    dv = dv.reshape(T, nkv * d)
    dxn = dq @ p["wq"] + dk @ p["wk"] + dv @ p["wv"]
    dwq = dq.T @ c["xn"]
    dwk = dk.T @ c["xn"]
    dwv = dv.T @ c["xn"]
    # input RMSNorm, then the identity skip
    dx, dg_attn = rmsnorm_backward(dxn, c["c1"], p["g_attn"])
    dx = dx + dr1
    grads = dict(wq=dwq, wk=dwk, wv=dwv, wo=dwo, wg=dwg, wu=dwu, wd=dwd,
                 g_attn=dg_attn, g_ffn=dg_ffn, g_q=dg_q, g_k=dg_k)
    return dx, grads


# ----------------------------------------------------------------------------
# Final RMSNorm + LM head + cross-entropy (gpu_forward, train_step_inner's
# fused_cross_entropy_cuda, gpu_backward; CPU loop in wgpu_trainer train_step)
# ----------------------------------------------------------------------------
def head_forward_backward(h, g_final, w_lm, targets, shape, loss_scale=None, keep_dz=False):
    """Returns dict(loss_partials [T] = per-token NLL (unscaled), loss = mean,
    dh [T, H], g_final grad [H], w_lm grad [V, H], lse [T]; dz [T, V] when
    ``keep_dz``)."""
    s = shape
    h = _f64(h)
    g_final = _f64(g_final)
    w_lm = _f64(w_lm)
    tg = np.asarray(targets, dtype=np.int64)
    T = h.shape[0]
    if loss_scale is None:
        loss_scale = 1.0 / T
    hn, cf = rmsnorm(h, g_final, s.eps)
    z = hn @ w_lm.T
    m = z.max(axis=-1, keepdims=True)
    lse = (m + np.log(np.sum(np.exp(z - m), axis=-1, keepdims=True)))[:, 0]
    rows = np.arange(T)
    partials = lse - z[rows, tg]
    dz = np.exp(z - lse[:, None])
    dz[rows, tg] -= 1.0
    dz *= loss_scale
    dhn = dz @ w_lm
    dw_lm = dz.T @ hn
    dh, dg_final = rmsnorm_backward(dhn, cf, g_final)
    out = dict(loss_partials=partials, loss=float(partials.mean()), dh=dh,
               g_final=dg_final, w_lm=dw_lm, lse=lse)
    if keep_dz:
        out["dz"] = dz
    return out


# ----------------------------------------------------------------------------
# Global-norm clip (C-CLIP-001) and AdamW (optimizer_step / adamw_step_cuda)
# ----------------------------------------------------------------------------
def squared_sum(g):
    g = _f64(g)
    return float(np.sum(g * g))


def clip_scale(per_buffer_sq_sums, max_norm):
    """||g||^2 is the plain sum of the per-buffer squared sums (never squared
    again); scale = max_norm / ||g|| when ||g|| > max_norm, else exactly 1.
    Returns (scale, norm, finite)."""
    total = float(np.sum(np.asarray(per_buffer_sq_sums, dtype=F64)))
    norm = float(np.sqrt(total))
    if not np.isfinite(norm):
        return 1.0, norm, False
    scale = max_norm / norm if norm > max_norm else 1.0
    return scale, norm, True


def adamw(w, g, m, v, step, lr, beta1, beta2, eps, weight_decay, scale=1.0):
    """One AdamW update at step t >= 1 with decoupled weight decay, on the
    clipped gradient g' = scale * g. Returns (w, m, v) new arrays."""
    assert step >= 1
    w, g, m, v = _f64(w), _f64(g), _f64(m), _f64(v)
    gs = scale * g
    m = beta1 * m + (1.0 - beta1) * gs
    v = beta2 * v + (1.0 - beta2) * gs * gs
    mhat = m / (1.0 - beta1 ** step)
    vhat = v / (1.0 - beta2 ** step)
    w = w - lr * (mhat / (np.sqrt(vhat) + eps) + weight_decay * w)
    return w, m, v


# ----------------------------------------------------------------------------
# The whole step
# ----------------------------------------------------------------------------
def model_forward_backward(blocks, head, x, targets, shape, loss_scale=None):
    """Forward through every block and the head, then the full backward.
    Returns (head result dict, list of per-block grads dicts)."""
    h = _f64(x)
    caches = []
    for p in blocks:
        h, cache = block_forward(p, h, shape)
        caches.append(cache)
    res = head_forward_backward(h, head["g_final"], head["w_lm"], targets, shape,
                                loss_scale=loss_scale)
    dh = res["dh"]
    block_grads = [None] * len(blocks)
    for i in reversed(range(len(blocks))):
        dh, block_grads[i] = block_backward(caches[i], dh, shape)
    res["dx"] = dh
    return res, block_grads


def train_step(blocks, head, x, targets, shape, state=None, step=1, optim=None):
    """One full training step: forward, fused CE, backward, one global clip
    over every trainable tensor, AdamW on every trainable tensor.

    ``state`` holds the AdamW moments as {(layer or 'head', name): (m, v)};
    missing entries start at zero. Returns a dict with the loss, the per-token
    loss partials, the gradients, the clip norm/scale and the updated
    parameters and moments."""
    res, bgrads = model_forward_backward(blocks, head, x, targets, shape)
    named = []
    for i, g in enumerate(bgrads):
        for k_, v_ in g.items():
            named.append(((i, k_), blocks[i][k_], v_))
    named.append((("head", "g_final"), head["g_final"], res["g_final"]))
    named.append((("head", "w_lm"), head["w_lm"], res["w_lm"]))
    out = _clip_adamw(named, state, step, optim)
    out.update(loss=res["loss"], loss_partials=res["loss_partials"], dx=res["dx"])
    return out


def accumulated_gradients(blocks, head, micro_xs, micro_targets, shape):
    """Gradient accumulation over n micro-batches (cuda_trainer.rs: R-038,
    ``train_step_inner`` scales the CE loss by 1/seq_len/accumulation_steps;
    the accumulator sums the micro-batch gradients before one optimizer step):
    each micro-batch runs the full forward and backward with the loss scaled
    by 1/(T n), T its token count, and the gradients are summed in micro-batch
    order. Returns (list of (key, parameter, gradient) like ``train_step``'s,
    concatenated per-token loss partials)."""
    n = len(micro_xs)
    total, partials = {}, []
    for x, tg in zip(micro_xs, micro_targets):
        T = np.asarray(x).shape[0]
        res, bgrads = model_forward_backward(blocks, head, x, tg, shape,
                                             loss_scale=1.0 / (T * n))
        partials.append(res["loss_partials"])
        items = [((i, k_), v_) for i, g in enumerate(bgrads) for k_, v_ in g.items()]
        items += [(("head", "g_final"), res["g_final"]), (("head", "w_lm"), res["w_lm"])]
        for key, g in items:
            total[key] = g if key not in total else total[key] + g
    named = [(key, blocks[key[0]][key[1]] if key[0] != "head" else head[key[1]], g)
             for key, g in total.items()]
    return named, np.concatenate(partials)


def train_step_accumulated(blocks, head, micro_xs, micro_targets, shape, state=None, step=1,
                           optim=None):
    """One step over n micro-batches: accumulated gradients, then the same
    global clip and AdamW as ``train_step``."""
    named, partials = accumulated_gradients(blocks, head, micro_xs, micro_targets, shape)
    out = _clip_adamw(named, state, step, optim)
    out.update(loss=float(partials.mean()), loss_partials=partials)
    return out


def _clip_adamw(named, state, step, optim):
    """The global clip over every (key, parameter, gradient) and AdamW on each."""
    o = dict(optim)
    sq = [squared_sum(g) for _, _, g in named]
    scale, norm, finite = clip_scale(sq, o["max_norm"])
    state = {} if state is None else state
    new_params, new_state = {}, {}
    for key, w, g in named:
        w = _f64(w)
        m, v = state.get(key, (np.zeros_like(w), np.zeros_like(w)))
        if finite:
            w2, m2, v2 = adamw(w, g, m, v, step, o["lr"], o["beta1"], o["beta2"], o["eps"],
                               o["weight_decay"], scale)
        else:
            w2, m2, v2 = w, _f64(m), _f64(v)
        new_params[key] = w2
        new_state[key] = (m2, v2)
    return dict(grads={key: g for key, _, g in named}, sq_sums=sq, norm=norm, scale=scale,
                finite=finite, params=new_params, state=new_state)
