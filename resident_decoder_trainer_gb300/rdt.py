"""Thin ctypes binding of librdt.so (include/rdt.h): argument marshalling only.

Every function takes device pointers as torch tensors (or raw ints) and the
current torch CUDA stream, calls the C entry point of the same name and
raises ``RdtError`` with the library's message on a non-zero status. No
computation happens here; if librdt.so is missing the import fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librdt.so")

RDT_OK, RDT_EINVAL, RDT_ECUDA, RDT_ETIMEOUT, RDT_ENONFINITE, RDT_EINDEX = 0, 1, 2, 3, 4, 5
TENSOR_NAMES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "g_attn", "g_ffn", "g_q", "g_k")
NF4_NAMES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")
LORA_NAMES = ("a_q", "a_k", "a_v", "a_o", "a_g", "a_u", "a_d",
              "b_q", "b_k", "b_v", "b_o", "b_g", "b_u", "b_d")

EXPORTS = (
    "rdt_check_config", "rdt_block_param_count", "rdt_block_param_offsets",
    "rdt_block_saved_bytes", "rdt_block_workspace_bytes", "rdt_head_workspace_bytes",
    "rdt_sq_sum_workspace_bytes", "rdt_block_forward", "rdt_block_backward",
    "rdt_fused_cross_entropy", "rdt_sq_sum", "rdt_clip_scale", "rdt_adamw_step",
    "rdt_gemm", "rdt_cast_bf16", "rdt_last_error", "rdt_device_error",
    "rdt_gemm_timing_arm", "rdt_gemm_timing_disarm", "rdt_launch_count",
    "rdt_sq_sum_noalloc", "rdt_gemm_nf4", "rdt_nf4_check", "rdt_nf4_code_bytes",
    "rdt_nf4_scale_count", "rdt_nf4_offsets", "rdt_lora_param_count", "rdt_lora_param_offsets",
    "rdt_lora_shadow_count", "rdt_lora_shadow", "rdt_nf4_saved_bytes", "rdt_nf4_workspace_bytes",
    "rdt_nf4_block_forward", "rdt_nf4_block_backward", "rdt_embedding_workspace_bytes",
    "rdt_embedding_forward", "rdt_embedding_backward", "rdt_step_advance", "rdt_wait_probe",
)


class RdtError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"librdt status {status}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]

    @classmethod
    def from_shape(cls, s) -> "Config":
        return cls(s.hidden, s.n_heads, s.n_kv_heads, s.head_dim, s.intermediate, s.vocab,
                   s.eps, s.theta)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m resident_decoder_trainer_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, F32, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    CP = ctypes.POINTER(Config)
    sig = {
        "rdt_check_config": (I32, [CP]),
        "rdt_block_param_count": (I64, [CP]),
        "rdt_block_param_offsets": (I32, [CP, P, P]),
        "rdt_block_saved_bytes": (SZ, [CP, I32, I32]),
        "rdt_block_workspace_bytes": (SZ, [CP, I32, I32]),
        "rdt_head_workspace_bytes": (SZ, [CP, I32]),
        "rdt_sq_sum_workspace_bytes": (SZ, []),
        "rdt_block_forward": (I32, [CP, I32, I32, P, P, P, P, P, SZ, P, SZ, P]),
        "rdt_block_backward": (I32, [CP, I32, I32, P, P, P, P, SZ, P, P, P, I32, P, P, SZ, P]),
        "rdt_fused_cross_entropy": (I32, [CP, I32, P, P, P, P, F32, P, P, P, P, I32, P, P, SZ,
                                          P]),
        "rdt_sq_sum": (I32, [P, P, I32, P, P, SZ, P]),
        "rdt_clip_scale": (I32, [P, F32, P, P, P]),
        "rdt_adamw_step": (I32, [P, P, P, P, I64, P, P, I32, P, F32, F32, F32, F32, F32, P, P]),
        "rdt_step_advance": (I32, [P, P]),
        "rdt_gemm": (I32, [P, I32, I64, P, I32, I64, I32, I32, I32, P, I64, P, I64, P]),
        "rdt_gemm_nf4": (I32, [P, I64, P, P, I64, I64, I32, P, I64, P, I64, I32, I32, P, I64, P, I64,
                               P]),
        "rdt_cast_bf16": (I32, [P, P, I64, P]),
        "rdt_last_error": (ctypes.c_char_p, []),
        "rdt_device_error": (I32, [P]),
        "rdt_wait_probe": (I32, [I64, I32, P, P]),
        "rdt_gemm_timing_arm": (I32, [P, P, P, I32]),
        "rdt_gemm_timing_disarm": (I64, []),
        "rdt_launch_count": (I64, []),
        "rdt_sq_sum_noalloc": (I32, [P, P, I32, P, P]),
        "rdt_embedding_workspace_bytes": (SZ, [I32]),
        "rdt_embedding_forward": (I32, [P, I64, I32, P, I32, P, P]),
        "rdt_embedding_backward": (I32, [P, I32, P, I32, P, P, I64, I32, P, SZ, P]),
        "rdt_nf4_check": (I32, [CP, I32]),
        "rdt_nf4_code_bytes": (I64, [CP]),
        "rdt_nf4_scale_count": (I64, [CP]),
        "rdt_nf4_offsets": (I32, [CP, P, P]),
        "rdt_lora_param_count": (I64, [CP, I32]),
        "rdt_lora_param_offsets": (I32, [CP, I32, P, P]),
        "rdt_lora_shadow_count": (I64, [CP, I32]),
        "rdt_lora_shadow": (I32, [CP, I32, P, P, P]),
        "rdt_nf4_saved_bytes": (SZ, [CP, I32, I32, I32]),
        "rdt_nf4_workspace_bytes": (SZ, [CP, I32, I32, I32]),
        "rdt_nf4_block_forward": (I32, [CP, I32, F32, I32, I32, P, P, P, P, P, P, P, SZ, P, SZ,
                                        P]),
        "rdt_nf4_block_backward": (I32, [CP, I32, F32, I32, I32, P, P, P, P, P, P, SZ, P, P, P,
                                         P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int):
    if status != RDT_OK:
        raise RdtError(status, lib().rdt_last_error().decode())


# ------------------------------------------------------------------ layout
def check_config(cfg: Config):
    _check(lib().rdt_check_config(ctypes.byref(cfg)))


def block_param_count(cfg: Config) -> int:
    n = lib().rdt_block_param_count(ctypes.byref(cfg))
    if n < 0:
        check_config(cfg)
    return n


def block_param_offsets(cfg: Config) -> dict[str, tuple[int, int]]:
    off = (ctypes.c_int64 * len(TENSOR_NAMES))()
    cnt = (ctypes.c_int64 * len(TENSOR_NAMES))()
    _check(lib().rdt_block_param_offsets(ctypes.byref(cfg), off, cnt))
    return {n: (off[i], cnt[i]) for i, n in enumerate(TENSOR_NAMES)}


def block_saved_bytes(cfg: Config, batch: int, seq: int) -> int:
    return lib().rdt_block_saved_bytes(ctypes.byref(cfg), batch, seq)


def block_workspace_bytes(cfg: Config, batch: int, seq: int) -> int:
    return lib().rdt_block_workspace_bytes(ctypes.byref(cfg), batch, seq)


def head_workspace_bytes(cfg: Config, tokens: int) -> int:
    return lib().rdt_head_workspace_bytes(ctypes.byref(cfg), tokens)


def sq_sum_workspace_bytes() -> int:
    return lib().rdt_sq_sum_workspace_bytes()


# ------------------------------------------------------------------- calls
def block_forward(cfg, batch, seq, w, w_bf16, x, y, saved, ws, stream=None):
    _check(lib().rdt_block_forward(ctypes.byref(cfg), batch, seq, _ptr(w), _ptr(w_bf16), _ptr(x),
                                   _ptr(y), _ptr(saved), saved.numel() * saved.element_size(),
                                   _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def block_backward(cfg, batch, seq, w, w_bf16, x, saved, dy, dx, grads, ws, grad_sq=None,
                   accumulate=False, stream=None):
    """grad_sq: optional fp64 device scalar; += the squared sum of grads.
    accumulate: add to grads instead of overwriting them."""
    _check(lib().rdt_block_backward(ctypes.byref(cfg), batch, seq, _ptr(w), _ptr(w_bf16), _ptr(x),
                                    _ptr(saved), saved.numel() * saved.element_size(), _ptr(dy),
                                    _ptr(dx), _ptr(grads), int(bool(accumulate)),
                                    None if grad_sq is None else _ptr(grad_sq), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)))


def fused_cross_entropy(cfg, tokens, h, gamma_f, w_lm, targets, loss_scale, loss_partials, dh,
                        dgamma_f, dw_lm, ws, grad_sq=None, accumulate=False, stream=None):
    """grad_sq: optional fp64 device scalar; = the squared sum of dgamma_f and
    dw_lm. accumulate: add to dgamma_f and dw_lm instead of overwriting them."""
    _check(lib().rdt_fused_cross_entropy(ctypes.byref(cfg), tokens, _ptr(h), _ptr(gamma_f),
                                         _ptr(w_lm), _ptr(targets), float(loss_scale),
                                         _ptr(loss_partials), _ptr(dh), _ptr(dgamma_f),
                                         _ptr(dw_lm), int(bool(accumulate)), None if grad_sq is None else _ptr(grad_sq),
                                         _ptr(ws), ws.numel() * ws.element_size(),
                                         _stream(stream)))


def sq_sum(bufs, sumsq, ws, stream=None):
    n = len(bufs)
    ptrs = (ctypes.c_void_p * n)(*[_ptr(b) for b in bufs])
    lens = (ctypes.c_int64 * n)(*[b.numel() for b in bufs])
    _check(lib().rdt_sq_sum(ptrs, lens, n, _ptr(sumsq), _ptr(ws),
                            ws.numel() * ws.element_size(), _stream(stream)))


def sq_sum_noalloc(bufs, sumsq, stream=None):
    """rdt_sq_sum without a workspace: for callers that cannot allocate
    (the scratch is a fixed array inside the library; see include/rdt.h)."""
    n = len(bufs)
    ptrs = (ctypes.c_void_p * n)(*[_ptr(b) for b in bufs])
    lens = (ctypes.c_int64 * n)(*[b.numel() for b in bufs])
    _check(lib().rdt_sq_sum_noalloc(ptrs, lens, n, _ptr(sumsq), _stream(stream)))


def clip_scale(sumsq, max_norm, scale, nonfinite=None, stream=None):
    _check(lib().rdt_clip_scale(_ptr(sumsq), float(max_norm), _ptr(scale), _ptr(nonfinite),
                                _stream(stream)))


def adamw_step(w, g, m, v, step, lr, beta1, beta2, eps, weight_decay, scale=None, skip=None,
               w_bf16=None, n=None, step_dev=None, stream=None):
    """step: host int (>= 1), or None with step_dev: a device int32 holding it."""
    n = w.numel() if n is None else n
    _check(lib().rdt_adamw_step(_ptr(w), _ptr(g), _ptr(m), _ptr(v), n, _ptr(scale), _ptr(skip),
                                int(step or 0), _ptr(step_dev), float(lr), float(beta1),
                                float(beta2), float(eps), float(weight_decay), _ptr(w_bf16),
                                _stream(stream)))


def step_advance(step_dev, stream=None):
    """step_dev (device int32) += 1."""
    _check(lib().rdt_step_advance(_ptr(step_dev), _stream(stream)))


def gemm(a, a_mn, b, b_mn, M, N, K, c, split_ws=None, stream=None):
    """c[M, N] = a' b'^T (see include/rdt.h); a, b bf16 2-D, c fp32 2-D;
    split_ws: optional fp32 scratch for the split-K path."""
    _check(lib().rdt_gemm(_ptr(a), int(a_mn), a.stride(0), _ptr(b), int(b_mn), b.stride(0), M, N,
                          K, _ptr(c), c.stride(0), _ptr(split_ws),
                          0 if split_ws is None else split_ws.numel(), _stream(stream)))


def gemm_nf4(a, codes, scales, w_rows, w_cols, b_mn, c, a2=None, b2=None, split_ws=None,
             stream=None):
    """c[M, N] = a B^T (+ a2 b2'^T) with B decoded from NF4 (see include/rdt.h);
    a, a2, b2 bf16 2-D, codes uint8, scales fp32, c fp32 2-D; split_ws:
    optional fp32 scratch for the split-K path."""
    k2 = 0 if a2 is None else a2.shape[1]
    _check(lib().rdt_gemm_nf4(_ptr(a), a.stride(0), _ptr(codes), _ptr(scales), w_rows, w_cols,
                              int(b_mn), _ptr(a2), 0 if a2 is None else a2.stride(0), _ptr(b2),
                              0 if b2 is None else b2.stride(0), k2, a.shape[0], _ptr(c),
                              c.stride(0), _ptr(split_ws),
                              0 if split_ws is None else split_ws.numel(), _stream(stream)))


# ------------------------------------------------- NF4 + LoRA block
def nf4_check(cfg: Config, rank: int):
    _check(lib().rdt_nf4_check(ctypes.byref(cfg), int(rank)))


def nf4_sizes(cfg: Config) -> tuple[int, int]:
    """(code bytes, scale elements) of the seven frozen projections."""
    nc = lib().rdt_nf4_code_bytes(ctypes.byref(cfg))
    ns = lib().rdt_nf4_scale_count(ctypes.byref(cfg))
    if nc < 0 or ns < 0:
        nf4_check(cfg, 16)
    return nc, ns


def nf4_offsets(cfg: Config) -> dict[str, tuple[int, int]]:
    """{projection: (code byte offset, scale element offset)}."""
    co = (ctypes.c_int64 * 7)()
    so = (ctypes.c_int64 * 7)()
    _check(lib().rdt_nf4_offsets(ctypes.byref(cfg), co, so))
    return {n: (co[i], so[i]) for i, n in enumerate(NF4_NAMES)}


def lora_param_count(cfg: Config, rank: int) -> int:
    n = lib().rdt_lora_param_count(ctypes.byref(cfg), int(rank))
    if n < 0:
        nf4_check(cfg, rank)
    return n


def lora_param_offsets(cfg: Config, rank: int) -> dict[str, tuple[int, int]]:
    off = (ctypes.c_int64 * len(LORA_NAMES))()
    cnt = (ctypes.c_int64 * len(LORA_NAMES))()
    _check(lib().rdt_lora_param_offsets(ctypes.byref(cfg), int(rank), off, cnt))
    return {n: (off[i], cnt[i]) for i, n in enumerate(LORA_NAMES)}


def lora_shadow_count(cfg: Config, rank: int) -> int:
    n = lib().rdt_lora_shadow_count(ctypes.byref(cfg), int(rank))
    if n < 0:
        nf4_check(cfg, rank)
    return n


def lora_shadow(cfg, rank, lora, shadow, stream=None):
    _check(lib().rdt_lora_shadow(ctypes.byref(cfg), int(rank), _ptr(lora), _ptr(shadow),
                                 _stream(stream)))


def nf4_saved_bytes(cfg: Config, rank: int, batch: int, seq: int) -> int:
    return lib().rdt_nf4_saved_bytes(ctypes.byref(cfg), int(rank), batch, seq)


def nf4_workspace_bytes(cfg: Config, rank: int, batch: int, seq: int) -> int:
    return lib().rdt_nf4_workspace_bytes(ctypes.byref(cfg), int(rank), batch, seq)


def nf4_block_forward(cfg, rank, alpha, batch, seq, codes, scales, gains, shadow, x, y, saved, ws,
                      stream=None):
    _check(lib().rdt_nf4_block_forward(ctypes.byref(cfg), int(rank), float(alpha), batch, seq,
                                       _ptr(codes), _ptr(scales), _ptr(gains), _ptr(shadow),
                                       _ptr(x), _ptr(y), _ptr(saved),
                                       saved.numel() * saved.element_size(), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(stream)))


def nf4_block_backward(cfg, rank, alpha, batch, seq, codes, scales, gains, shadow, x, saved, dy,
                       dx, lora_grads, ws, grad_sq=None, stream=None):
    """grad_sq: optional fp64 device scalar; += the squared sum of lora_grads."""
    _check(lib().rdt_nf4_block_backward(ctypes.byref(cfg), int(rank), float(alpha), batch, seq,
                                        _ptr(codes), _ptr(scales), _ptr(gains), _ptr(shadow),
                                        _ptr(x), _ptr(saved),
                                        saved.numel() * saved.element_size(), _ptr(dy), _ptr(dx),
                                        _ptr(lora_grads),
                                        None if grad_sq is None else _ptr(grad_sq), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(stream)))


# ---------------------------------------------------------------- embedding
def embedding_workspace_bytes(tokens: int) -> int:
    return lib().rdt_embedding_workspace_bytes(int(tokens))


def embedding_forward(table, ids, x, stream=None):
    """x[t] = table[ids[t]]; table fp32 [V, H], ids int32 [T], x fp32 [T, H]."""
    _check(lib().rdt_embedding_forward(_ptr(table), table.shape[0], table.shape[1], _ptr(ids),
                                       ids.numel(), _ptr(x), _stream(stream)))


def embedding_backward(ids, dx, dtable, ws, scale=None, accumulate=False, stream=None):
    """dtable[id] (=, or += when accumulate) scale * sum of dx over the tokens with that id."""
    _check(lib().rdt_embedding_backward(_ptr(ids), ids.numel(), _ptr(dx), dx.shape[1], _ptr(scale),
                                        _ptr(dtable), dtable.shape[0], int(bool(accumulate)),
                                        _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)))


def cast_bf16(src, dst, n=None, stream=None):
    n = src.numel() if n is None else n
    _check(lib().rdt_cast_bf16(_ptr(src), _ptr(dst), n, _stream(stream)))


def wait_probe(limit_ns, arrive, waited=None, stream=None):
    """One warp waits on an mbarrier for at most limit_ns (see rdt_wait_probe);
    waited: optional int64 device tensor of one element for the duration."""
    _check(lib().rdt_wait_probe(int(limit_ns), 1 if arrive else 0,
                                None if waited is None else _ptr(waited), _stream(stream)))


def device_error() -> int:
    code = ctypes.c_int32(0)
    _check(lib().rdt_device_error(ctypes.byref(code)))
    return code.value


def launch_count() -> int:
    """Kernels launched through librdt so far in this process."""
    return lib().rdt_launch_count()


class GemmTimer:
    """Per-launch CUDA-event timing of every tensor-core GEMM launched while
    the context is active (rdt_gemm_timing_arm / _disarm)."""

    def __init__(self, capacity: int):
        self.capacity = capacity
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for ev in self.events:  # torch creates the CUDA event lazily, on first record
            ev.record()
        torch.cuda.synchronize()
        self._handles = (ctypes.c_void_p * (2 * capacity))(*[ev.cuda_event for ev in self.events])
        self._flops = (ctypes.c_double * capacity)()
        self._kinds = (ctypes.c_int32 * capacity)()
        self.seen = 0

    def __enter__(self):
        _check(lib().rdt_gemm_timing_arm(self._handles, self._flops, self._kinds,
                                         self.capacity))
        return self

    def __exit__(self, *exc):
        self.seen = lib().rdt_gemm_timing_disarm()

    KINDS = ("single", "pair", "nf4")

    def results(self, with_kind=False):
        """[(flops, milliseconds)] (or (flops, ms, kind) with kind one of
        KINDS) for every recorded launch (call after a sync)."""
        n = min(self.seen, self.capacity)
        out = []
        for i in range(n):
            ms = self.events[2 * i].elapsed_time(self.events[2 * i + 1])
            out.append((self._flops[i], ms, self.KINDS[self._kinds[i]]) if with_kind
                       else (self._flops[i], ms))
        return out
