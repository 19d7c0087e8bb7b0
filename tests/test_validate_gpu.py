"""smd_validate_indices on the GPU: the range check of an index list that a
caller runs before a decode. It must flag exactly the lists that hold an
entry outside [0, N) among a row's first clamp(count, 0, W) entries, and
must not read anything else. The lists with bad entries here go to the
check only, never to a decode."""
from __future__ import annotations

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs

pytestmark = pytest.mark.gpu


def check(indices, counts, N, dev, status0=0):
    import torch
    from sparse_mla_decode_gb300 import binding
    idx = torch.from_numpy(np.ascontiguousarray(indices, dtype=np.int32)).to(dev)
    cnt = torch.from_numpy(np.ascontiguousarray(counts, dtype=np.int32)).to(dev)
    status = torch.full((1,), status0, dtype=torch.int32, device=dev)
    binding.validate_indices(idx, cnt, N, status=status)
    torch.cuda.synchronize()
    return int(status.item())


def test_valid_lists_pass(cuda):
    from sparse_mla_decode_gb300 import binding
    for name in ("tiny", "latency", "dsa"):
        case = inputs.config(name)
        assert check(case.indices, case.counts, case.N, cuda) == binding.SMD_OK, name


@pytest.mark.parametrize("bad", [-1, -(2 ** 31), "N", 2 ** 31 - 1])
def test_an_entry_outside_the_pool_inside_a_count_is_flagged(cuda, bad):
    from sparse_mla_decode_gb300 import binding
    N, B, W = 1000, 7, 300
    rng = np.random.default_rng(1)
    idx = rng.integers(0, N, size=(B, W), dtype=np.int64).astype(np.int32)
    counts = np.array([300, 0, 5, 299, 1, 150, 300], dtype=np.int32)
    idx[3, 298] = N if bad == "N" else bad  # the last valid entry of row 3
    assert check(idx, counts, N, cuda) == binding.SMD_ERR_INDEX
    idx[3, 298] = N - 1  # the last row of the pool is in range
    assert check(idx, counts, N, cuda) == binding.SMD_OK


def test_entries_past_a_count_are_not_read(cuda):
    from sparse_mla_decode_gb300 import binding
    N, B, W = 500, 5, 64
    rng = np.random.default_rng(2)
    counts = np.array([64, 10, 0, -3, 63], dtype=np.int32)
    idx = rng.integers(0, N, size=(B, W), dtype=np.int64).astype(np.int32)
    for b, n in enumerate(counts):
        idx[b, max(n, 0):] = -7  # garbage wherever the decode reads nothing
    assert check(idx, counts, N, cuda) == binding.SMD_OK
    idx[4, 62] = N + 5
    assert check(idx, counts, N, cuda) == binding.SMD_ERR_INDEX


def test_counts_above_the_width_are_clamped(cuda):
    from sparse_mla_decode_gb300 import binding
    N = 100
    idx = np.arange(32, dtype=np.int32).reshape(2, 16)
    assert check(idx, [1000, 16], N, cuda) == binding.SMD_OK
    idx[0, 15] = 100
    assert check(idx, [1000, 0], N, cuda) == binding.SMD_ERR_INDEX
    assert check(idx, [15, 16], N, cuda) == binding.SMD_OK


def test_many_rows_one_bad_entry_in_the_last(cuda):
    """More rows than the grid has blocks (each block takes several)."""
    from sparse_mla_decode_gb300 import binding
    N, B, W = 2 ** 20, 5000, 40
    rng = np.random.default_rng(3)
    idx = rng.integers(0, N, size=(B, W), dtype=np.int64).astype(np.int32)
    counts = rng.integers(0, W + 1, size=B).astype(np.int32)
    counts[-1] = W
    assert check(idx, counts, N, cuda) == binding.SMD_OK
    idx[-1, 0] = -1
    assert check(idx, counts, N, cuda) == binding.SMD_ERR_INDEX


def test_zero_width_and_an_earlier_status_are_kept(cuda):
    from sparse_mla_decode_gb300 import binding
    assert check(np.zeros((3, 0), dtype=np.int32), [0, 4, 9], 10, cuda) == binding.SMD_OK
    bad = np.full((2, 4), 50, dtype=np.int32)
    # the first writer wins: an earlier device status is not overwritten
    assert check(bad, [4, 4], 10, cuda, status0=binding.SMD_ERR_TIMEOUT) == binding.SMD_ERR_TIMEOUT
    assert check(bad, [4, 4], 10, cuda) == binding.SMD_ERR_INDEX
