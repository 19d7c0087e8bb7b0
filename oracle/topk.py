"""Top-k select oracle -- plain, slow, obviously correct CPU code (numpy).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
CPU-baseline leg call this file. The decode library never imports it, and it
shares no code with the library.

What it computes (the topk_exchange page: the select of push_local_topk,
its radix histogram passes over bf16 logits, the threshold and the tie rule;
read for one GPU, without the exchange's packing):

  for row r with end = min(L, clamp(row_ends[r], 0, L)) logits x_0 .. x_{end-1}
  (bf16 bit patterns):
    valid    x_i is not a NaN: (bits & 0x7FFF) <= 0x7F80 (infinities count)
    key      o_i = the bf16 bits mapped to an unsigned 16-bit key whose order
             is the order of the values: bits | 0x8000 for a positive sign,
             ~bits for a negative one (so -0 sorts just below +0)
    if fewer than K logits are valid: all valid i, ascending
    else     v = the K-th largest key among the valid ones (the page finds it
             whenever the histogram's running count reaches K);
             first every i with o_i > v (ascending i), then the i with o_i == v
             in ascending order until K are taken
  count[r] = min(K, number of valid logits); entries past the count are -1.

The page finds v with two histogram passes (the high 9 bits of the key, then
the low 7 bits inside the threshold bucket); the K-th largest key is the same
number however it is found, so the oracle takes it from a sort.
"""
from __future__ import annotations

import numpy as np

NO_INDEX = -1


def order_keys(bits: np.ndarray) -> np.ndarray:
    """bf16 bits (uint16) -> order-preserving uint16 keys (0 for NaN)."""
    b = np.asarray(bits, np.uint16).astype(np.uint32)
    key = np.where(b & 0x8000, (~b) & 0xFFFF, b | 0x8000)
    valid = (b & 0x7FFF) <= 0x7F80
    return np.where(valid, key, 0).astype(np.uint32), valid


def select_row(bits: np.ndarray, K: int) -> np.ndarray:
    """The selected positions of one row (its first `end` logits), in output
    order."""
    key, valid = order_keys(bits)
    idx = np.nonzero(valid)[0]
    if idx.size < K:
        return idx.astype(np.int32)
    v = np.sort(key[idx])[::-1][K - 1]  # the K-th largest key
    gt = np.nonzero(valid & (key > v))[0]
    eq = np.nonzero(valid & (key == v))[0][: K - gt.size]
    return np.concatenate([gt, eq]).astype(np.int32)


def topk_select(logits_bits: np.ndarray, K: int, row_ends=None):
    """logits_bits uint16 [B, L] (bf16 bits), row_ends int32 [B] or None.
    Returns (indices int32 [B, K], counts int32 [B])."""
    x = np.asarray(logits_bits, np.uint16)
    assert x.ndim == 2
    B, L = x.shape
    out = np.full((B, K), NO_INDEX, np.int32)
    counts = np.zeros(B, np.int32)
    for r in range(B):
        end = L if row_ends is None else int(min(L, max(0, int(row_ends[r]))))
        sel = select_row(x[r, :end], K)
        out[r, : sel.size] = sel
        counts[r] = sel.size
    return out, counts
