"""The tcgen05 / TMA layout conventions in isolation: one 128 x N x 128 bf16
GEMM per operand-layout family used by the attention kernels, against an fp64
matrix product of the same bf16 values."""
import numpy as np
import pytest
import torch

import exact_io_aware_27_gb300 as fa

pytestmark = pytest.mark.gpu


def _ref(mode, A, B):
    a, b = A.double(), B.double()
    if mode in (0, 4):
        return a @ b.T
    if mode in (1, 2):
        return a @ b
    return a.T @ b  # mode 3


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_selftest_mma(mode):
    fa.build()
    g = torch.Generator().manual_seed(100 + mode)
    A = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    b_shape = {0: (128, 128), 1: (128, 128), 2: (128, 128), 3: (128, 64), 4: (64, 128)}[mode]
    B = torch.randn(*b_shape, generator=g).to(torch.bfloat16)
    D = fa.fa_selftest_mma(mode, A.cuda(), B.cuda())
    torch.cuda.synchronize()
    ref = _ref(mode, A, B).numpy()
    err = float(np.max(np.abs(D.double().cpu().numpy() - ref)))
    assert err <= 1e-3, f"mode {mode}: max abs err {err}"
