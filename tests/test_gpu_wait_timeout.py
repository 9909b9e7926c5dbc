"""The bounded device waits: a wait that gives up records RDT_ETIMEOUT in the
device error word and the kernel returns (it releases its tensor memory and
does not trap), so the CUDA context stays usable and the host learns of the
failure from rdt_device_error. cuda_trainer.rs's train_step_inner reports a
poisoned CUDA context after a device-side failure; the bounds exist so that a
wait that never completes ends as an error status instead.

The failure is made with rdt_wait_probe: one warp waits on an mbarrier that
nothing arrives on, with a 1 ms limit, through the same bounded-wait helper
the GEMM and attention kernels use."""
import pytest
import torch

from resident_decoder_trainer_gb300 import rdt

from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu

RDT_ETIMEOUT = 3
LIMIT_NS = 1_000_000


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    rdt.device_error()  # start from a clear error word
    yield
    assert rdt.device_error() == 0


def test_wait_that_completes_records_nothing():
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    rdt.wait_probe(LIMIT_NS, arrive=True, waited=waited)
    assert rdt.device_error() == 0
    assert int(waited) < LIMIT_NS


def test_wait_that_runs_out_records_a_timeout_and_the_context_stays_usable():
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    rdt.wait_probe(LIMIT_NS, arrive=False, waited=waited)
    assert rdt.device_error() == RDT_ETIMEOUT
    # it waited for its limit, then gave up
    assert LIMIT_NS <= int(waited) < 1000 * LIMIT_NS
    # the read cleared the word
    assert rdt.device_error() == 0
    # the probe freed its tensor memory: a tensor-core GEMM whose CTAs cover
    # every SM (each allocates tensor memory) runs and is right
    g = torch.Generator(device="cuda").manual_seed(3)
    M, N, K = 4096, 4096, 256
    a = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    b = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    c = torch.empty(M, N, device="cuda")
    rdt.gemm(a, 0, b, 0, M, N, K, c)
    torch.cuda.synchronize()
    want = a.double() @ b.double().T
    err = float((c.double() - want).norm() / want.norm())
    assert err < 1e-5
    assert rdt.device_error() == 0
    # and the probe itself runs again, completing this time
    rdt.wait_probe(LIMIT_NS, arrive=True)
    assert rdt.device_error() == 0


def test_probe_rejects_limits_out_of_range():
    for bad in (0, 999, 10_000_000_001):
        with pytest.raises(rdt.RdtError):
            rdt.wait_probe(bad, arrive=True)
