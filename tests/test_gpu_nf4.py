"""GPU parity of the NF4-frozen path with the FP64 oracle (``oracle/nf4.py``):
the NF4 GEMM (codes decoded into the tensor-core operand tiles, plus the bf16
tail that carries the LoRA term) against an fp64 matmul of the same decoded
weights, and the NF4 + LoRA block forward/backward and adapters-only step."""
import numpy as np
import pytest
import torch

from oracle import nf4 as on
from resident_decoder_trainer_gb300 import rdt

from gpu_helpers import ensure_built, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    assert rdt.device_error() == 0


def _nf4_weight(rows, cols, g):
    codes = torch.randint(0, 256, (rows, cols // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    scales = (torch.randn(rows * cols // 64, generator=g) * 0.02).abs() * 3.0
    return codes, scales


def _decoded(codes, scales, rows, cols):
    """W as the GPU's operand: level * scale in fp32, rounded to bf16 (RNE)."""
    w = on.nf4_dequantize(codes.numpy(), scales.numpy().astype(np.float32), rows, cols)
    lv = on.NF4_LEVELS.astype(np.float32)[on.nf4_unpack(codes.numpy(), rows, cols)]
    w32 = lv * np.repeat(scales.numpy().astype(np.float32), 64).reshape(rows, cols)
    assert np.max(np.abs(w32.astype(np.float64) - w)) <= 1e-6 * np.max(np.abs(w))
    return torch.from_numpy(w32).to(torch.bfloat16).double()


@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("k2", [0, 16, 48])
@pytest.mark.parametrize("M,rows,cols", [(300, 320, 512), (128, 192, 256), (700, 512, 1024)])
def test_nf4_gemm_matches_fp64_of_decoded_weights(b_mn, k2, M, rows, cols):
    if b_mn and k2 == 48 and rows == 192:
        pytest.skip("covered by the other shapes")
    g = torch.Generator().manual_seed(M + rows + 7 * cols + k2 + b_mn)
    codes, scales = _nf4_weight(rows, cols, g)
    w = _decoded(codes, scales, rows, cols)           # [rows, cols]
    N, K1 = (cols, rows) if b_mn else (rows, cols)
    a = torch.randn(M, K1, generator=g).to(torch.bfloat16)
    ref = a.double() @ (w if b_mn else w.T)
    a2 = b2 = None
    if k2:
        a2 = torch.randn(M, k2, generator=g).to(torch.bfloat16)
        b2 = torch.randn(k2, N, generator=g).to(torch.bfloat16) if b_mn else \
            torch.randn(N, k2, generator=g).to(torch.bfloat16)
        ref = ref + a2.double() @ (b2.double() if b_mn else b2.double().T)
    ldc = (N + 3) // 4 * 4
    c = torch.full((M, ldc), float("nan"), device="cuda")
    rdt.gemm_nf4(a.cuda(), codes.cuda(), scales.cuda(), rows, cols, b_mn, c,
                 None if a2 is None else a2.cuda(), None if b2 is None else b2.cuda())
    torch.cuda.synchronize()
    out = c[:, :N].double().cpu()
    assert torch.isfinite(out).all()
    assert rel_l2(out.numpy(), ref.numpy()) < 1e-5
