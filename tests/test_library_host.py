"""Host-side checks of librdt.so that need no GPU: it loads, exports every
symbol include/rdt.h declares, and its layout / size / validation logic is
right. (No compute call is made here.)"""
import ctypes
import os
import re

import pytest

from resident_decoder_trainer_gb300 import build, rdt, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return rdt.lib()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "rdt.h")) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rdt_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/rdt.h but not exported"
    assert set(names) == set(rdt.EXPORTS)


def test_block_layout_matches_tensor_shapes(lib):
    for key in ("tiny", "small", "q4b_block"):
        s = synth.WORKLOADS[key]
        cfg = rdt.Config.from_shape(s)
        offs = rdt.block_param_offsets(cfg)
        shapes = synth.block_shapes(s)
        pos = 0
        for name in rdt.TENSOR_NAMES:
            off, cnt = offs[name]
            assert off == pos and off % 16 == 0
            n = 1
            for d in shapes[name]:
                n *= d
            assert cnt == n
            pos += cnt
        assert rdt.block_param_count(cfg) == pos
    q4b = rdt.Config.from_shape(synth.WORKLOADS["q4b_block"])
    assert rdt.block_param_count(q4b) == 100_930_816  # 100.93 M per Qwen3-4B block


def test_sizes_are_positive_and_aligned(lib):
    s = synth.WORKLOADS["q4b_full"]
    cfg = rdt.Config.from_shape(s)
    for n in (rdt.block_saved_bytes(cfg, s.batch, s.seq),
              rdt.block_workspace_bytes(cfg, s.batch, s.seq),
              rdt.head_workspace_bytes(cfg, s.tokens)):
        assert n > 0 and n % 256 == 0
    # the head never holds the logits of every token: its scratch is a few
    # [T, H] buffers and one vocabulary chunk (at most 256 MB), well below the
    # bf16 [T, V] logits
    head = rdt.head_workspace_bytes(cfg, s.tokens)
    assert head < 2 * s.tokens * s.vocab // 2
    assert head < 32 * s.tokens * s.hidden + (272 << 20)
    # ... and it grows with the vocabulary only by the clip's per-tile slots
    wide = rdt.Config.from_shape(s.replace(vocab=4 * s.vocab))
    assert rdt.head_workspace_bytes(wide, s.tokens) - head < (16 << 20)
    assert rdt.sq_sum_workspace_bytes() >= 8


@pytest.mark.parametrize("field,value", [("hidden", 40), ("hidden", 8192), ("head_dim", 48),
                                         ("n_kv_heads", 3), ("intermediate", 100),
                                         ("vocab", 1000)])
def test_bad_configs_are_rejected(lib, field, value):
    cfg = rdt.Config.from_shape(synth.WORKLOADS["tiny"])
    setattr(cfg, field, value)
    with pytest.raises(rdt.RdtError) as ei:
        rdt.check_config(cfg)
    assert ei.value.status == rdt.RDT_EINVAL
    assert lib.rdt_block_param_count(ctypes.byref(cfg)) == -1
    assert rdt.block_saved_bytes(cfg, 1, 32) == 0


def test_null_and_misaligned_arguments_fail_before_any_launch(lib):
    cfg = rdt.Config.from_shape(synth.WORKLOADS["tiny"])
    P = ctypes.c_void_p
    st = lib.rdt_block_forward(ctypes.byref(cfg), 1, 32, None, None, None, None, None, 0, None,
                               0, None)
    assert st == rdt.RDT_EINVAL and b"null" in lib.rdt_last_error()
    st = lib.rdt_adamw_step(P(16), P(16), P(16), P(16), 4, None, None, 0, None, 1e-3, 0.9, 0.95,
                            1e-8, 0.0, None, None)
    assert st == rdt.RDT_EINVAL and b"step" in lib.rdt_last_error()
    st = lib.rdt_adamw_step(P(18), P(16), P(16), P(16), 4, None, None, 1, None, 1e-3, 0.9, 0.95,
                            1e-8, 0.0, None, None)
    assert st == rdt.RDT_EINVAL and b"aligned" in lib.rdt_last_error()
    st = lib.rdt_clip_scale(P(16), ctypes.c_float(0.0), P(16), None, None)
    assert st == rdt.RDT_EINVAL
    st = lib.rdt_gemm(P(16), 0, 12, P(16), 0, 16, 8, 8, 8, P(16), 8, None, 0, None)
    assert st == rdt.RDT_EINVAL


def test_nf4_and_lora_layouts_match_tensor_shapes(lib):
    s = synth.WORKLOADS["q4b_nf4"]
    cfg = rdt.Config.from_shape(s)
    rank = synth.LORA["rank"]
    rdt.nf4_check(cfg, rank)
    shapes = synth.block_shapes(s)
    offs = rdt.nf4_offsets(cfg)
    pc = ps = 0
    for name in rdt.NF4_NAMES:
        out, inn = shapes[name]
        assert offs[name] == (pc, ps)
        pc += out * inn // 2
        ps += out * inn // 64
    assert rdt.nf4_sizes(cfg) == (pc, ps)
    # 4.5 bits per frozen weight: 4-bit codes plus one fp32 scale per 64
    n_w = 2 * pc
    assert n_w == rdt.block_param_count(cfg) - 2 * s.hidden - 2 * s.head_dim
    lo = rdt.lora_param_offsets(cfg, rank)
    pos = 0
    for name in rdt.LORA_NAMES:
        proj = "w" + name[2:]
        out, inn = shapes[proj]
        want = rank * inn if name.startswith("a_") else out * rank
        assert lo[name] == (pos, want)
        pos += want
    assert rdt.lora_param_count(cfg, rank) == pos
    n_a = sum(rank * shapes[p][1] for p in rdt.NF4_NAMES)
    stacked = (s.q_dim + 2 * s.kv_dim) * 3 * rank + s.hidden * rank + \
        2 * s.intermediate * 2 * rank + s.hidden * rank
    assert rdt.lora_shadow_count(cfg, rank) == n_a + stacked
    for n in (rdt.nf4_saved_bytes(cfg, rank, s.batch, s.seq),
              rdt.nf4_workspace_bytes(cfg, rank, s.batch, s.seq)):
        assert n > 0 and n % 256 == 0
    assert rdt.nf4_saved_bytes(cfg, rank, s.batch, s.seq) > \
        rdt.block_saved_bytes(cfg, s.batch, s.seq)


@pytest.mark.parametrize("field,value,rank", [("hidden", 320, 16), ("intermediate", 688, 16),
                                              ("hidden", 2576, 16), ("hidden", 256, 4),
                                              ("hidden", 256, 32)])
def test_nf4_constraints_are_enforced(lib, field, value, rank):
    cfg = rdt.Config.from_shape(synth.WORKLOADS["q4b_nf4"])
    setattr(cfg, field, value)
    with pytest.raises(rdt.RdtError) as ei:
        rdt.nf4_check(cfg, rank)
    assert ei.value.status == rdt.RDT_EINVAL
    assert lib.rdt_lora_param_count(ctypes.byref(cfg), rank) == -1
    assert rdt.nf4_saved_bytes(cfg, rank, 1, 32) == 0


def test_product_path_has_no_oracle_or_cpu_fallback():
    pkg = os.path.join(ROOT, "resident_decoder_trainer_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            with open(os.path.join(pkg, fn)) as fh:
                src = fh.read()
            assert not re.search(r"^\s*(import|from)\s+oracle", src, flags=re.M), fn
    with open(os.path.join(pkg, "rdt.py")) as fh:
        src = fh.read()
    assert "raise ImportError" in src  # a missing library fails loudly


def test_newer_entry_points_validate_before_any_launch(lib):
    """The embedding, NF4 GEMM and step-counter calls reject bad arguments on
    the host with RDT_EINVAL and a message (no device is touched)."""
    P = ctypes.c_void_p

    def einval(st, text):
        assert st == rdt.RDT_EINVAL, st
        assert text in lib.rdt_last_error(), lib.rdt_last_error()

    einval(lib.rdt_step_advance(None, None), b"null")
    # embedding: null ids, hidden not a multiple of 4, misaligned table, short workspace
    einval(lib.rdt_embedding_forward(P(16), 8, 8, None, 4, P(16), None), b"null")
    einval(lib.rdt_embedding_forward(P(16), 8, 6, P(16), 4, P(16), None), b"multiple of 4")
    einval(lib.rdt_embedding_forward(P(20), 8, 8, P(16), 4, P(16), None), b"aligned")
    einval(lib.rdt_embedding_backward(P(16), 4, P(16), 8, None, P(16), 8, 0, P(256), 0, None),
           b"workspace")
    # NF4 GEMM: a tail wider than one 64-deep step, W not a multiple of 256 columns,
    # misaligned codes
    einval(lib.rdt_gemm_nf4(P(16), 256, P(16), P(16), 64, 256, 0, P(16), 72, P(16), 72, 72, 8,
                            P(16), 64, None, 0, None), b"K2")
    einval(lib.rdt_gemm_nf4(P(16), 256, P(16), P(16), 64, 200, 0, None, 0, None, 0, 0, 8,
                            P(16), 64, None, 0, None), b"cols % 256")
    einval(lib.rdt_gemm_nf4(P(16), 256, P(24), P(16), 64, 256, 0, None, 0, None, 0, 0, 8,
                            P(16), 64, None, 0, None), b"16-byte")
    # NF4 block: rank outside {8, 16}
    cfg = rdt.Config.from_shape(synth.WORKLOADS["q4b_nf4"])
    einval(lib.rdt_lora_shadow(ctypes.byref(cfg), 12, P(16), P(16), None), b"rank")


def test_wait_probe_validates_its_limit_before_any_launch(lib):
    """The bounded-wait test hook rejects limits outside [1 us, 10 s] and a
    misaligned duration pointer on the host (no device is touched)."""
    P = ctypes.c_void_p
    for bad in (0, 999, 10_000_000_001):
        assert lib.rdt_wait_probe(bad, 1, None, None) == rdt.RDT_EINVAL
        assert b"limit_ns" in lib.rdt_last_error()
    assert lib.rdt_wait_probe(1_000_000, 0, P(12), None) == rdt.RDT_EINVAL
    assert b"aligned" in lib.rdt_last_error()
