"""Pins of the CPU oracle against facts that do not come from the oracle.

Each check is chosen so that a plausible mistake in the oracle fails it:
the E4M3 and BF16 codecs against torch's independent conversions and the
format's anchor values; exact logits against rational arithmetic; closed forms
(equal logits -> plain mean of V, one dominant key -> its V row, count 1,
count 0 -> zeros and -inf); the index-order invariance that the row-max anchor
gives; the E4M3-P error bound against the unquantized fp64 reference; and a
brute-force rational re-implementation on tiny inputs. For the bf16-query
variant: the split exponent's defining inequality, exactness of hi + lo over
every bf16 value where the residual fits, the reduction to the E4M3 decode,
and the removal of the query rounding against an unrounded reference.

The method these follow is the "attn_sparse" page (SparseDcpDecode): module
docstring paragraphs "Per CTA", "Precision" and "Rows of count 0", and the
merge method's epilogue.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_decode_gb300 import inputs

# ---------------------------------------------------------------- helpers ---

_E4M3_VALUES = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
    torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def dec(codes) -> np.ndarray:
    """E4M3 codes -> values through torch's float8 conversion (not the oracle)."""
    return _E4M3_VALUES[np.asarray(codes, np.int64)]


def bf16_of_fraction(x: Fraction) -> int:
    """BF16 bits nearest to the exact rational x (ties to even), found by
    comparing exact distances to the two bf16 neighbours of float(x)."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    f = np.float32(float(a))
    bits = int(np.array([f], np.float32).view(np.uint32)[0]) >> 16
    cands = [max(bits - 1, 0), bits, bits + 1]

    def val(b):
        return Fraction(float(np.array([b << 16], np.uint32).view(np.float32)[0]))

    best = min(cands, key=lambda b: (abs(val(b) - a), b & 1))
    return sign | best


def f32_of_bits(bits) -> np.ndarray:
    return oracle.bf16_bits_to_f32(np.asarray(bits, np.uint16))


def ulp_diff(a_bits, b_bits) -> np.ndarray:
    """Distance in bf16 ulps between bf16 bit patterns (same-sign ordering)."""
    a = np.asarray(a_bits, np.int64)
    b = np.asarray(b_bits, np.int64)
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)


def blank_case(B, H, W, N, counts, sm_scale=1.0, q_scale=1.0, k_scale=1.0):
    return inputs.Case("blank", np.zeros((B, H, 576), np.uint8), np.zeros((N, 576), np.uint8),
                       np.zeros((B, W), np.int32), np.asarray(counts, np.int32),
                       float(np.float32(sm_scale)), float(np.float32(q_scale)),
                       float(np.float32(k_scale)))


def run(case, mode=oracle.MODE_RECIPE):
    return oracle.sparse_mla_decode(case.q8, case.kv8, case.indices, case.counts,
                                    case.sm_scale, case.q_scale, case.k_scale, mode=mode)


# ------------------------------------------------------------ E4M3 codec ---

def test_e4m3_decode_matches_torch_and_anchor_values():
    ours = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(_E4M3_VALUES)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], _E4M3_VALUES[~nan])
    # The format's anchors: max finite 448, min normal 2^-6, min subnormal 2^-9.
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0
    assert math.copysign(1.0, ours[0x80]) == -1.0 and ours[0x80] == 0.0


def test_e4m3_encode_roundtrip_every_finite_code():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert oracle.e4m3_encode(v) == c, hex(c)


def test_e4m3_encode_matches_torch_rne_including_ties():
    rng = np.random.default_rng(7)
    mags = np.exp2(rng.uniform(-13, 8.9, 20000))
    xs = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    # Exact midpoints between neighbouring codes (ties go to the even code).
    finite = np.sort(np.unique(np.abs(_E4M3_VALUES[~np.isnan(_E4M3_VALUES)])))
    mids = ((finite[1:] + finite[:-1]) / 2).astype(np.float32)
    xs = np.concatenate([xs, mids, -mids])
    ref = torch.from_numpy(np.clip(xs, -448, 448)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(x)) for x in xs], np.uint8)
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates_and_flushes():
    assert oracle.e4m3_encode(1e9) == 0x7E
    assert oracle.e4m3_encode(-1e9) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00  # tie between 0 and 2^-9 -> even
    assert oracle.e4m3_encode(2.0 ** -10 * 1.0001) == 0x01


# ------------------------------------------------------------ BF16 codec ---

def test_bf16_rne_matches_torch_on_float32_values():
    rng = np.random.default_rng(11)
    xs = (rng.standard_normal(20000) * np.exp2(rng.uniform(-30, 30, 20000))).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    ours = np.array([oracle.bf16_rne(float(x)) for x in xs], np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rne_rounds_once_from_double():
    # 1 + 2^-8 is a bf16 tie; a hair above it must round up. Rounding to fp32
    # first would land on the tie and round down to 1.0.
    assert oracle.bf16_rne(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert oracle.bf16_rne(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_rne(-(1.0 + 3 * 2.0 ** -8)) == 0xBF82


# ------------------------------------------------------------ the decode ---

def test_logits_are_exact():
    case = inputs.random_case(3, B=1, H=2, W=5, N=50, counts=[5])
    for h in range(2):
        S, s, P, P8, m = oracle.row_head_terms(case.q8, case.kv8, case.indices, case.counts,
                                               0, h, case.sm_scale, case.q_scale, case.k_scale)
        qv = [Fraction(float(v)) for v in dec(case.q8[0, h])]
        for i, j in enumerate(case.indices[0, :5]):
            kv = [Fraction(float(v)) for v in dec(case.kv8[j])]
            exact = sum(a * b for a, b in zip(qv, kv))
            assert Fraction(S[i]) == exact
        # P is anchored at 448 of the row maximum: the max key gets 448.
        assert np.all(P <= np.float32(448.0) * np.float32(1 + 2 ** -20))
        assert P8[int(np.argmax(s))] == 0x7E
        assert m == s.max()


def test_count_zero_negative_and_clamp():
    base = inputs.random_case(5, B=4, H=16, W=24, N=300, counts=[0, -5, 24, 3])
    out, _, lse = run(base)
    assert np.all(out[0] == 0) and np.all(out[1] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[1]))
    big = inputs.Case("big", base.q8, base.kv8, base.indices,
                      np.array([0, -5, 10 ** 6, 3], np.int32),
                      base.sm_scale, base.q_scale, base.k_scale)
    out2, _, lse2 = run(big)
    assert np.array_equal(out2, out) and np.array_equal(lse2, lse)
    assert np.all(np.isfinite(lse[2:]))


def test_equal_logits_give_plain_mean_of_v():
    """q = 0 makes every logit 0: P = 448 for every key, so the output is
    BF16(k_s * mean of the gathered V rows) and LSE = ln n."""
    rng = np.random.default_rng(1)
    N, W = 64, 20
    case = blank_case(2, 16, W, N, [20, 7], sm_scale=0.07, q_scale=0.3, k_scale=0.0123)
    case.kv8[:] = rng.integers(0, 256, size=(N, 576)).astype(np.uint8)
    case.kv8[(case.kv8 & 0x7F) == 0x7F] = 0x3C  # no NaN codes in the pool
    for b in range(2):
        case.indices[b] = rng.choice(N, W, replace=False)
    out, _, lse = run(case)
    ks = Fraction(case.k_scale)
    for b, n in enumerate([20, 7]):
        V = dec(case.kv8[case.indices[b, :n], :512])
        for c in range(0, 512, 37):
            mean = sum(Fraction(float(v)) for v in V[:, c]) / n
            want = bf16_of_fraction(ks * mean)
            assert np.all(out[b, :, c] == want), (b, c)
        assert np.allclose(lse[b], math.log(n), rtol=0, atol=1e-12)


def test_equal_logits_from_rope_columns_only():
    """Keys that agree on columns 512..575 and q that is zero on columns
    0..511: every logit is the same non-zero value, so the output is still
    the plain mean of V over columns 0..511 (QK reads all 576 columns, PV
    only the first 512)."""
    rng = np.random.default_rng(2)
    N, W, n = 40, 16, 13
    case = blank_case(1, 16, W, N, [n], sm_scale=0.05, q_scale=0.02, k_scale=0.03)
    case.q8[0, :, 512:] = rng.integers(0x30, 0x40, size=(16, 64)).astype(np.uint8)
    shared = rng.integers(0x28, 0x48, size=64).astype(np.uint8)
    case.kv8[:, 512:] = shared
    case.kv8[:, :512] = rng.integers(0, 0x7E, size=(N, 512)).astype(np.uint8)
    case.indices[0] = rng.choice(N, W, replace=False)
    out, _, lse = run(case)
    V = dec(case.kv8[case.indices[0, :n], :512])
    for c in range(0, 512, 29):
        mean = sum(Fraction(float(v)) for v in V[:, c]) / n
        assert np.all(out[0, :, c] == bf16_of_fraction(Fraction(case.k_scale) * mean))
    # lse = ln n + ln2 * s, with s the common logit (non-zero here).
    S, s, _, _, _ = oracle.row_head_terms(case.q8, case.kv8, case.indices, case.counts, 0, 0,
                                          case.sm_scale, case.q_scale, case.k_scale)
    assert np.all(s == s[0]) and s[0] != 0.0
    assert abs(lse[0, 0] - (math.log(n) + math.log(2) * float(s[0]))) < 1e-5


@pytest.mark.parametrize("n,pos", [(1, 0), (9, 4), (64, 63)])
def test_dominant_key_returns_its_v_row(n, pos):
    """One key whose logit beats every other by > 40 (log2 units): every other
    P rounds to 0 in E4M3 and weighs < 2^-40 in the sum, so the output is
    BF16(k_s * V_dom) and LSE = ln2 * lambda * S_dom (to fp32 rounding)."""
    rng = np.random.default_rng(100 + n)
    N, W = 96, 64
    ks = 0.0371
    sm = 2.2e-3 / (ks * math.log2(math.e))  # lambda ~ 2.2e-3: s_dom ~ 63, others 0
    case = blank_case(1, 16, W, N, [n], sm_scale=sm, q_scale=1.0, k_scale=ks)
    case.q8[0, :, 512:] = 0x38  # 1.0
    case.kv8[:, :512] = rng.integers(0, 0x7E, size=(N, 512)).astype(np.uint8)
    keys = rng.choice(N, W, replace=False)
    case.indices[0] = keys
    dom = keys[pos]
    case.kv8[dom, 512:] = 0x7E  # 448: S_dom = 64 * 448
    out, _, lse = run(case)
    V = dec(case.kv8[dom, :512])
    want = np.array([bf16_of_fraction(Fraction(case.k_scale) * Fraction(float(v))) for v in V])
    assert np.all(out[0] == want[None, :])
    lam = case.sm_scale * case.q_scale * case.k_scale * math.log2(math.e)
    assert lam * 64 * 448 > 40
    assert np.allclose(lse[0], math.log(2) * lam * 64 * 448, rtol=1e-6)


def test_count_one_returns_that_v_row():
    case = inputs.random_case(9, B=3, H=32, W=8, N=200, counts=[1, 1, 1])
    out, _, lse = run(case)
    for b in range(3):
        V = dec(case.kv8[case.indices[b, 0], :512])
        want = np.array([bf16_of_fraction(Fraction(case.k_scale) * Fraction(float(v))) for v in V])
        assert ulp_diff(out[b], want[None, :]).max() <= 1
        assert (ulp_diff(out[b], want[None, :]) == 0).mean() > 0.99
        for h in range(32):
            _, s, _, _, _ = oracle.row_head_terms(case.q8, case.kv8, case.indices, case.counts,
                                                  b, h, case.sm_scale, case.q_scale, case.k_scale)
            assert abs(lse[b, h] - math.log(2) * float(s[0])) < 1e-5


def test_index_order_does_not_matter():
    """With the anchor at the row maximum, P8 of a key does not depend on
    where the key sits in the list: a permutation changes only sum order."""
    case = inputs.random_case(12, B=4, H=16, W=96, N=5000, counts=[96, 50, 1, 77],
                              heavy_frac=0.05)
    out, o64, lse = run(case)
    perm_idx = case.indices.copy()
    rng = np.random.default_rng(5)
    for b, n in enumerate(case.counts):
        perm_idx[b, :n] = perm_idx[b, rng.permutation(n)]
    shuffled = inputs.Case("perm", case.q8, case.kv8, perm_idx, case.counts,
                           case.sm_scale, case.q_scale, case.k_scale)
    out2, o642, lse2 = run(shuffled)
    assert ulp_diff(out, out2).max() <= 1
    assert np.max(np.abs(lse - lse2)) < 1e-12
    assert np.max(np.abs(o64 - o642)) <= 1e-12 * np.max(np.abs(o64))


def test_e4m3_p_error_bound_against_unquantized():
    """|out - out_u| <= k_s/T * sum_i |P8_i - P_i| |V_ic|
                     <= k_s * max_i |V_ic| * (2^-4 + n 2^-10 / T)
    since an E4M3 rounding moves P by at most max(2^-4 P, 2^-10)."""
    case = inputs.random_case(21, B=3, H=16, W=128, N=4000, counts=[128, 64, 5],
                              heavy_frac=0.02)
    _, o_q, _ = run(case, oracle.MODE_RECIPE)
    _, o_u, lse_u = run(case, oracle.MODE_UNQUANT)
    assert np.max(np.abs(o_q - o_u)) > 0  # the E4M3 rounding does act
    for b in range(case.B):
        n = int(case.counts[b])
        V = np.abs(dec(case.kv8[case.indices[b, :n], :512]))
        vmax = V.max(axis=0)
        for h in range(case.H):
            S, s, P, P8, m = oracle.row_head_terms(case.q8, case.kv8, case.indices, case.counts,
                                                   b, h, case.sm_scale, case.q_scale, case.k_scale)
            T = float(np.sum(P.astype(np.float64)))
            assert T >= 448.0 * (1 - 1e-6)
            bound = case.k_scale * vmax * (2.0 ** -4 + n * 2.0 ** -10 / T)
            assert np.all(np.abs(o_q[b, h] - o_u[b, h]) <= bound * (1 + 1e-12))


def _brute_force(case):
    """The decode written again from the definition, with exact rationals for
    every sum and torch / numpy for the codecs and the fp32 roundings."""
    B, H, W = case.B, case.H, case.W
    lam = np.float32(np.float64(np.float32(case.sm_scale)) * np.float64(np.float32(case.q_scale))
                     * np.float64(np.float32(case.k_scale)) * math.log2(math.e))
    l448 = np.float32(math.log2(448.0))
    out = np.zeros((B, H, 512), np.uint16)
    lse = np.zeros((B, H))
    for b in range(B):
        n = min(max(int(case.counts[b]), 0), W)
        keys = case.indices[b, :n]
        for h in range(H):
            if n == 0:
                lse[b, h] = -math.inf
                continue
            qv = [Fraction(float(v)) for v in dec(case.q8[b, h])]
            s = []
            for j in keys:
                kv = [Fraction(float(v)) for v in dec(case.kv8[j])]
                S = np.float32(float(sum(a * c for a, c in zip(qv, kv))))
                s.append(np.float32(lam * S))
            m = max(s)
            bias = np.float32(m - l448)
            P = [np.float32(2.0 ** float(np.float32(x - bias))) for x in s]
            P8 = dec(torch.tensor(np.array(P, np.float32)).clamp(-448, 448).to(
                torch.float8_e4m3fn).view(torch.uint8).numpy())
            T = sum(Fraction(float(p)) for p in P)
            for c in range(512):
                A = sum(Fraction(float(p8)) * Fraction(float(dec(case.kv8[j, c])))
                        for p8, j in zip(P8, keys))
                out[b, h, c] = bf16_of_fraction(Fraction(float(case.k_scale)) * A / T)
            lse[b, h] = math.log(2) * (float(m) - math.log2(448.0) + math.log2(float(T)))
    return out, lse


def test_brute_force_rational_reimplementation():
    case = inputs.random_case(31, B=2, H=16, W=6, N=64, counts=[6, 3], heavy_frac=0.1)
    sub = inputs.Case("bf", case.q8[:, :2].copy(), case.kv8, case.indices, case.counts,
                      case.sm_scale, case.q_scale, case.k_scale)
    want_out, want_lse = _brute_force(sub)
    out, _, lse = run(sub)
    assert np.array_equal(out, want_out)
    assert np.allclose(lse, want_lse, rtol=0, atol=1e-9)


def test_golden_fixture_regression():
    """A small stored case (inputs and outputs written by
    tests/golden/make_golden.py, which calls only the oracle)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "small_case.json")
    with open(path) as f:
        g = json.load(f)
    q8 = np.frombuffer(bytes.fromhex(g["q8"]), np.uint8).reshape(g["B"], g["H"], 576)
    kv8 = np.frombuffer(bytes.fromhex(g["kv8"]), np.uint8).reshape(g["N"], 576)
    idx = np.array(g["indices"], np.int32).reshape(g["B"], g["W"])
    counts = np.array(g["counts"], np.int32)
    out, _, lse = oracle.sparse_mla_decode(q8, kv8, idx, counts, g["sm_scale"],
                                           g["q_scale"], g["k_scale"])
    assert np.array_equal(out.reshape(-1), np.array(g["out_bf16"], np.uint16))
    want_lse = np.array([(-math.inf if v is None else v) for v in g["lse"]])
    assert np.allclose(lse.reshape(-1), want_lse, rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(lse.reshape(-1)), np.isneginf(want_lse))


# ------------------------------------------- the bf16 query, split hi + lo ---
# The mla_attn page: "q_split" (the bf16 Q rows to "E4M3 hi, lo of q 2^k") and
# "fp8_split4" (x ~ hi + lo). Reading: one power-of-two scale per (row, head).

def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 values that are exactly bf16 -> their bits."""
    x = np.ascontiguousarray(x, np.float32)
    bits = x.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)
    return (bits >> 16).astype(np.uint16)


@pytest.mark.parametrize("amax", [448.0, 448.5, 449.0, 224.0, 1.0, 0.875, 0.8749, 3.9,
                                  2.0 ** -20, 1e-30, 7e8, 1e30])
def test_q_split_exponent_is_the_largest_in_range(amax):
    """amax * 2^k <= 448 < amax * 2^(k+1), in exact arithmetic (clamped to
    [-32, 32])."""
    k = oracle.q_split_exponent(amax)
    a = Fraction(amax)
    two = Fraction(2)
    if -32 < k < 32:
        assert a * two ** k <= 448 < a * two ** (k + 1), (amax, k)
    else:
        assert k in (-32, 32)
        assert (a * two ** k <= 448) if k == 32 else (a * two ** k > 224)
    assert oracle.q_split_exponent(0.0) == 0


def test_q_split_is_exact_where_the_residual_fits():
    """Every bf16 value x with 2^-2 <= |x| <= 448 is hi + lo exactly (the
    residual has at most four significant bits on a 2^-9 grid); below that
    the error is at most half the smallest E4M3 step (2^-10). A row holding
    448 gets k = 0, so the codes are those of x itself."""
    e = np.arange(-20, 9)
    mant = np.arange(128)
    vals = np.array([(1 + m / 128.0) * 2.0 ** int(x) for x in e for m in mant], np.float64)
    vals = vals[vals <= 448.0]
    vals = np.concatenate([vals, -vals]).astype(np.float32)
    for start in range(0, vals.size, 575):
        chunk = vals[start:start + 575]
        row = np.zeros(576, np.float32)
        row[0] = 448.0
        row[1:1 + chunk.size] = chunk
        hi, lo, k = oracle.q_split(_bf16_bits(row))
        assert k == 0
        got = dec(hi) + dec(lo)
        x = row.astype(np.float64)
        big = np.abs(x) >= 0.25
        assert np.array_equal(got[big], x[big])
        assert np.all(np.abs(got[~big] - x[~big]) <= 2.0 ** -10)
        # hi alone is the plain E4M3 rounding of x (torch's cast)
        assert np.array_equal(dec(hi), dec(inputs.to_e4m3(row)))


@pytest.mark.parametrize("shift", [0, -5, 3])
def test_bf16_query_that_is_e4m3_reduces_to_the_e4m3_decode(shift):
    """A bf16 query whose values are E4M3 values times 2^shift, with 448 x
    2^shift in every (row, head): the split gives lo = 0 and k = -shift, so
    the decode is the E4M3 decode with q_scale = 2^shift, bit for bit."""
    case = inputs.random_case(90, B=3, H=16, W=100, N=800, counts=[100, 37, 0])
    q8 = case.q8.copy()
    q8[:, :, 5] = 0x7E  # 448
    qv = (dec(q8) * 2.0 ** shift).astype(np.float32)
    q16 = _bf16_bits(qv)
    o16, o64, lse, ks = oracle.sparse_mla_decode_bf16q(q16, case.kv8, case.indices, case.counts,
                                                       case.sm_scale, case.k_scale)
    assert np.all(ks == -shift)
    r16, r64, rlse = oracle.sparse_mla_decode(q8, case.kv8, case.indices, case.counts,
                                              case.sm_scale, 2.0 ** shift, case.k_scale)
    assert np.array_equal(o16, r16)
    assert np.array_equal(lse.view(np.uint64), rlse.view(np.uint64))


def test_bf16_query_split_removes_the_query_rounding():
    """Against a float64 reference that uses the bf16 query unrounded (and P
    unquantized): the split query's decode (P unquantized too) is within
    1e-4 of max|out|, and more than 20x closer than the per-tensor E4M3
    query's decode. A split that dropped lo would be as far off as E4M3."""
    case = inputs.random_case(91, B=2, H=16, W=300, N=3000, counts=[300, 211])
    qv = (case.q16.astype(np.uint32) << 16).view(np.float32)  # the bf16 values
    kvv = dec(case.kv8)
    lam0 = float(np.float32(case.sm_scale * case.k_scale * 1.4426950408889634))
    ref = np.zeros((case.B, case.H, 512))
    for b in range(case.B):
        n = int(case.counts[b])
        rows = kvv[case.indices[b, :n]]
        s = lam0 * (qv[b].astype(np.float64) @ rows.T)       # [H, n], base 2
        P = np.exp2(s - s.max(axis=1, keepdims=True))
        ref[b] = case.k_scale * (P @ rows[:, :512]) / P.sum(axis=1, keepdims=True)
    _, split64, _, _ = oracle.sparse_mla_decode_bf16q(case.q16, case.kv8, case.indices,
                                                      case.counts, case.sm_scale, case.k_scale,
                                                      mode=oracle.MODE_UNQUANT)
    _, e4m3_64, _ = oracle.sparse_mla_decode(case.q8, case.kv8, case.indices, case.counts,
                                             case.sm_scale, case.q_scale, case.k_scale,
                                             mode=oracle.MODE_UNQUANT)
    scale = np.abs(ref).max()
    err_split = np.abs(split64 - ref).max()
    err_e4m3 = np.abs(e4m3_64 - ref).max()
    assert err_split <= 1e-4 * scale, (err_split, scale)
    assert err_split * 20 < err_e4m3, (err_split, err_e4m3)
