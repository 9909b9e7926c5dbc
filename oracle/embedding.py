"""FP64 CPU oracle for the token embedding (lookup and scatter-add backward).

TEST INFRASTRUCTURE ONLY (same rules as ``oracle.model``): only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs may use it; it shares
no code, table or constant with the CUDA path.

What it computes (aprender-train docs.rs pages, cuda_trainer.rs 0.34.0):

* ``gpu_forward`` -- the block stack's input is the embedding row of every
  token: x[t] = E[ids[t]].
* ``embed_backward`` (contract C-EMBED-GRAD-001) -- the activation gradient
  that leaves the first block is clipped by its own norm to max_grad_norm
  (scale = max_norm / ||dx|| when ||dx|| > max_norm, else 1), then
  scatter-added into the embedding gradient: dE[ids[t]] += scale dx[t]; ids
  outside [0, vocab) are skipped.
* ``optimizer_step`` -- the embedding has its own AdamW (same hyper-parameters
  and step count as the rest), outside the global clip of the other weights.

Readings: the embedding's gradient is that of one step (or of the step's
micro-batches, each clipped on its own as the pages do per batch); its AdamW
is the same decoupled-decay AdamW as every other tensor's.
"""
from __future__ import annotations

import numpy as np

from oracle import model as om


def embedding_forward(table, ids):
    """x [T, H] = the rows of ``table`` [V, H] picked by ``ids`` [T]."""
    return om._f64(table)[np.asarray(ids, dtype=np.int64)]


def embedding_grad(ids, dx, vocab, max_norm=None):
    """dE [V, H]: token t adds scale * dx[t] to row ids[t] (skipped when the
    id is outside [0, vocab)); scale is dx's own clip scale (1 when max_norm
    is None). Returns (dE, scale)."""
    dx = om._f64(dx)
    scale = 1.0
    if max_norm is not None:
        scale, _, _ = om.clip_scale([om.squared_sum(dx)], max_norm)
    de = np.zeros((vocab, dx.shape[1]))
    for t, tid in enumerate(np.asarray(ids, dtype=np.int64)):
        if 0 <= tid < vocab:
            de[tid] += scale * dx[t]
    return de, scale


def train_step_embedded(table, blocks, head, ids, targets, shape, state=None, emb_state=None,
                        step=1, optim=None):
    """One step of the model fed by the embedding: ``oracle.model.train_step``
    on x = E[ids], then the embedding's clipped scatter-add gradient and its
    own AdamW. Returns train_step's dict plus emb_grad, emb_scale, emb (the
    updated table) and emb_state (its moments)."""
    o = dict(optim)
    x = embedding_forward(table, ids)
    out = om.train_step(blocks, head, x, targets, shape, state=state, step=step, optim=o)
    de, scale = embedding_grad(ids, out["dx"], np.asarray(table).shape[0], o["max_norm"])
    w = om._f64(table)
    m, v = emb_state if emb_state else (np.zeros_like(w), np.zeros_like(w))
    w2, m2, v2 = om.adamw(w, de, m, v, step, o["lr"], o["beta1"], o["beta2"], o["eps"],
                          o["weight_decay"], 1.0)
    out.update(emb_grad=de, emb_scale=scale, emb=w2, emb_state=(m2, v2))
    return out
