"""The allocation-free squared sum (rdt_sq_sum_noalloc) against the
workspace version (rdt_sq_sum). It is meant for callers that cannot allocate
device memory; its scratch is a fixed array inside the library, shared by
every call, so two calls in a row must each give the right answer.
Collected last on purpose, so a failure here leaves every other test run."""
import ctypes

import pytest
import torch

from resident_decoder_trainer_gb300 import rdt

from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu

SQ_SUM_REL = 1e-6  # the relative tolerance of the squared-sum parity test


def _workspace_sq_sum(bufs):
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    ws = torch.empty(rdt.sq_sum_workspace_bytes(), dtype=torch.uint8, device="cuda")
    rdt.sq_sum(bufs, out, ws)
    return out


def _noalloc_sq_sum(bufs):
    out = torch.full((1,), float("nan"), dtype=torch.float64, device="cuda")
    n = len(bufs)
    ptrs = (ctypes.c_void_p * n)(*[b.data_ptr() for b in bufs])
    lens = (ctypes.c_int64 * n)(*[b.numel() for b in bufs])
    st = rdt.lib().rdt_sq_sum_noalloc(ptrs, lens, n, out.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    assert st == rdt.RDT_OK, rdt.lib().rdt_last_error()
    return out


def test_noalloc_sq_sum_matches_workspace_version_on_two_calls_in_a_row():
    ensure_built()
    g = torch.Generator(device="cuda").manual_seed(123)
    cases = [[torch.randn(n, device="cuda", generator=g) for n in (5, 4099, 1 << 20)],
             [3.0 * torch.randn(n, device="cuda", generator=g) for n in (1 << 23, 3, 17)]]
    for bufs in cases:
        want = float(_workspace_sq_sum(bufs))
        got = float(_noalloc_sq_sum(bufs))
        assert abs(got - want) <= SQ_SUM_REL * want, (got, want)
    torch.cuda.synchronize()


def test_noalloc_sq_sum_rejects_more_buffers_than_it_handles():
    ensure_built()
    bufs = [torch.ones(4, device="cuda") for _ in range(65)]
    with pytest.raises(rdt.RdtError) as ei:
        rdt.sq_sum_noalloc(bufs, torch.zeros(1, dtype=torch.float64, device="cuda"))
    assert ei.value.status == rdt.RDT_EINVAL and "64" in str(ei.value)
