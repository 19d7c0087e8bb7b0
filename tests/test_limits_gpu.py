"""GPU parity at the plans' limits: the warp-MMA kernel at the widest index
list its shared memory takes (16-way split, 1600 keys a CTA), and the spread
kernel at its largest grid of work (1024 units of (row, 128 heads), pieces
in a dozen rounds over the cooperative grid). The CPU side checks that one
more key or one more unit is refused or planned elsewhere."""
from __future__ import annotations

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs
from test_parity_gpu import check, gpu_decode, oracle_decode

pytestmark = pytest.mark.gpu

MMA_MAX_W = 25600


def test_mma_kernel_at_its_widest_rows(cuda):
    from sparse_mla_decode_gb300 import binding
    p = binding.smd_plan(2, 16, MMA_MAX_W)
    assert p.kernel == binding.SMD_KERNEL_MMA and p.split == 16
    with pytest.raises(binding.SmdError):
        binding.smd_plan(2, 16, MMA_MAX_W + 1)
    case = inputs.random_case(901, B=2, H=16, W=MMA_MAX_W, N=60000, counts=[MMA_MAX_W, 12345])
    out_g, lse_g = gpu_decode(case, cuda)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, "warp MMA at W = 25600")


def test_spread_kernel_at_its_unit_cap(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    B, H, W = 1024, 128, 700
    force = {"kernel": binding.SMD_KERNEL_TC_SPREAD}
    nb = binding.smd_workspace_bytes_ex(B, H, W, force)
    assert nb > 0 and binding.smd_workspace_bytes_ex(B + 1, H, W, force) == 0
    rng = np.random.default_rng(902)
    counts = rng.integers(0, W + 1, size=B)
    counts[[5, 700]] = 0
    counts[[0, 1023]] = W
    case = inputs.random_case(902, B=B, H=H, W=W, N=20000, counts=counts.tolist())
    ws = torch.zeros(nb, dtype=torch.uint8, device=cuda)
    out_g, lse_g = gpu_decode(case, cuda, plan=force, workspace=ws)
    rows = [0, 5, 511, 512, 700, 1023]
    out_o, lse_o = oracle_decode(case, rows)
    check(out_g[rows], lse_g[rows], out_o, lse_o, "spread at 1024 units")
