"""Pins of the top-k select oracle (oracle/topk.py) against facts that do not
come from it: the key order against the float order of every bf16 pattern,
the selected values against torch.topk, and hand-worked tie, NaN, row-end,
signed-zero and infinity cases (the topk_exchange page: push_local_topk's
select, threshold and tie rule)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import topk as ot


def bits_of(values) -> np.ndarray:
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def values_of(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def test_key_order_is_the_value_order_for_every_bf16_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    key, valid = ot.order_keys(bits)
    vals = values_of(bits)
    assert np.array_equal(valid, ~np.isnan(vals))
    assert np.all(key[~valid] == 0) and np.all(key[valid] > 0)
    k, v, b = key[valid], vals[valid], bits[valid]
    order = np.argsort(k, kind="stable")
    # keys are distinct per pattern and ascending keys give non-decreasing values
    assert np.unique(k).size == k.size
    assert np.all(np.diff(v[order].astype(np.float64)) >= 0)
    # the only equal neighbours are -0 then +0
    eq = np.nonzero(np.diff(v[order].astype(np.float64)) == 0)[0]
    assert eq.size == 1
    assert b[order][eq[0]] == 0x8000 and b[order][eq[0] + 1] == 0x0000


@pytest.mark.parametrize("seed,L,K", [(0, 5000, 64), (1, 70000, 2048), (2, 300, 299), (3, 1000, 1)])
def test_selected_values_are_torch_topk(seed, L, K):
    """Rows with many equal values (bf16 of a narrow normal): the multiset of
    selected values equals torch.topk's, the count is K, indices are unique."""
    g = np.random.default_rng(seed)
    vals = (g.standard_normal((3, L)) * 0.05).astype(np.float32)
    bits = bits_of(vals)
    idx, cnt = ot.topk_select(bits, K)
    tv = torch.from_numpy(values_of(bits)).to(torch.float64)
    ref = torch.topk(tv, K, dim=1).values.numpy()
    for r in range(3):
        assert cnt[r] == K and np.unique(idx[r]).size == K
        got = np.sort(values_of(bits[r])[idx[r]].astype(np.float64))[::-1]
        assert np.array_equal(got, ref[r])


def test_ties_go_last_in_index_order():
    bits = bits_of([3, 1, 3, 2, 3, 3])
    idx, cnt = ot.topk_select(bits[None], 3)
    assert cnt[0] == 3 and idx[0].tolist() == [0, 2, 4]     # v = 3: the first three 3s
    idx, cnt = ot.topk_select(bits[None], 5)
    assert idx[0].tolist() == [0, 2, 4, 5, 3]               # v = 2: every 3, then the 2


def test_nan_is_never_selected_and_short_rows_return_every_valid_index():
    bits = bits_of([1.0, float("nan"), 2.0, float("nan"), -1.0])
    idx, cnt = ot.topk_select(bits[None], 4)
    assert cnt[0] == 3 and idx[0].tolist() == [0, 2, 4, -1]
    idx, cnt = ot.topk_select(bits[None], 2)
    assert idx[0].tolist() == [2, 0]


def test_exactly_k_valid_takes_the_threshold_order():
    """K valid logits: the threshold is the smallest, so it goes last."""
    bits = bits_of([5.0, 1.0, 7.0])
    idx, cnt = ot.topk_select(bits[None], 3)
    assert cnt[0] == 3 and idx[0].tolist() == [0, 2, 1]


def test_row_end_and_signed_zero_and_infinities():
    bits = bits_of([0.0, -0.0, float("-inf"), float("inf"), 9.0, 8.0])
    idx, cnt = ot.topk_select(np.stack([bits, bits]), 2, row_ends=[4, -3])
    assert idx[0].tolist() == [3, 0]      # +inf, then +0 above -0
    assert cnt[1] == 0 and idx[1].tolist() == [-1, -1]
    idx, cnt = ot.topk_select(bits[None], 7, row_ends=[99])
    assert idx[0].tolist() == [0, 1, 2, 3, 4, 5, -1]  # every logit (end clamped to L)
