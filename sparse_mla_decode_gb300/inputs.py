"""Seeded synthetic inputs for sparse MLA decode.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark. It draws random numbers and packs them into the call's input
layout; it holds none of the decode arithmetic. The only numeric step is
turning the drawn query / cache values into E4M3 bytes, which is done with
torch's own ``float8_e4m3fn`` cast (round to nearest even), after clamping to
the format's largest finite value (448).

Layouts (what the C ABI takes):
  q8       uint8 [B, H, 576]   E4M3 query codes
  q16      uint16 [B, H, 576]  the bf16 query (bits) the codes were quantized
                               from, for the bf16-query entry point
  kv8      uint8 [N, 576]      E4M3 cache rows (512 latent + 64 more QK columns)
  indices  int32 [B, W]        the first counts[b] entries of row b are its keys
  counts   int32 [B]
  sm_scale, q_scale, k_scale   python floats (exactly representable in fp32)

Workloads follow the five configurations the method is evaluated on (tiny,
latency decode, DSA decode, throughput decode, dense-as-sparse); ``random_case``
draws small shapes for sweeps.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROW = 576       # bytes per cache row: 512 latent columns + 64 QK-only columns
LATENT = 512    # columns used by PV
E4M3_MAX = 448.0


@dataclasses.dataclass
class Case:
    name: str
    q8: np.ndarray        # uint8 [B, H, 576]
    kv8: np.ndarray       # uint8 [N, 576]
    indices: np.ndarray   # int32 [B, W]
    counts: np.ndarray    # int32 [B]
    sm_scale: float
    q_scale: float
    k_scale: float
    q16: np.ndarray | None = None  # uint16 [B, H, 576]: the bf16 query q8 was quantized from

    @property
    def B(self) -> int:
        return int(self.q8.shape[0])

    @property
    def H(self) -> int:
        return int(self.q8.shape[1])

    @property
    def W(self) -> int:
        return int(self.indices.shape[1])

    @property
    def N(self) -> int:
        return int(self.kv8.shape[0])

    def clamped_counts(self) -> np.ndarray:
        return np.clip(self.counts.astype(np.int64), 0, self.W)

    def unique_rows(self) -> int:
        """Distinct cache rows referenced by the valid index entries."""
        n = self.clamped_counts()
        if self.B == 0 or n.sum() == 0:
            return 0
        mask = np.arange(self.W)[None, :] < n[:, None]
        return int(np.unique(self.indices[mask]).size)

    def gathered_rows(self) -> int:
        return int(self.clamped_counts().sum())


def _f32(x: float) -> float:
    return float(np.float32(x))


def to_e4m3(x: np.ndarray) -> np.ndarray:
    """float32 array (already scaled into range) -> E4M3 codes (uint8)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = t.clamp_(-E4M3_MAX, E4M3_MAX)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (RNE) and return them as float32."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def _normal_blocks(seed_seq: np.random.SeedSequence, rows: int, cols: int,
                   threads: int = 8, block_rows: int = 16384) -> np.ndarray:
    """float32 N(0,1) [rows, cols], filled block by block from spawned streams."""
    out = np.empty((rows, cols), np.float32)
    nblk = max(1, -(-rows // block_rows))
    kids = seed_seq.spawn(nblk)

    def fill(i: int) -> None:
        g = np.random.Generator(np.random.PCG64(kids[i]))
        lo, hi = i * block_rows, min(rows, (i + 1) * block_rows)
        if hi > lo:
            g.standard_normal(out=out[lo:hi], dtype=np.float32)

    if nblk == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def quantize_per_tensor(x: np.ndarray) -> tuple[np.ndarray, float]:
    """Per-tensor scale = amax / 448 (fp32) and the E4M3 codes of x / scale."""
    amax = float(np.max(np.abs(x))) if x.size else 1.0
    if amax == 0.0:
        amax = 1.0
    scale = _f32(np.float32(amax) / np.float32(E4M3_MAX))
    codes = to_e4m3(x / np.float32(scale))
    return codes, scale


def make_query(rng: np.random.Generator, B: int, H: int) -> tuple[np.ndarray, float, np.ndarray]:
    """The bf16 query N(0,1): its per-tensor E4M3 codes and scale, and its
    bf16 bits (for the bf16-query entry point)."""
    q = rng.standard_normal((B, H, ROW), dtype=np.float32)
    q = to_bf16_values(q)  # the model's query is bf16
    codes, scale = quantize_per_tensor(q)
    q16 = (np.ascontiguousarray(q, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return codes, scale, q16


def make_pool(seed_seq: np.random.SeedSequence, N: int, heavy_frac: float = 0.0,
              heavy_gain: float = 8.0, rng: np.random.Generator | None = None
              ) -> tuple[np.ndarray, float]:
    kv = _normal_blocks(seed_seq, N, ROW)
    if heavy_frac > 0.0 and rng is not None:
        heavy = rng.choice(N, size=max(1, int(round(heavy_frac * N))), replace=False)
        kv[heavy] *= np.float32(heavy_gain)
    return quantize_per_tensor(kv)


def _unique_uniform(rng: np.random.Generator, N: int, k: int, exclude=None) -> np.ndarray:
    if exclude is None or len(exclude) == 0:
        return rng.choice(N, size=k, replace=False).astype(np.int64)
    excl = set(int(e) for e in exclude)
    out: list[int] = []
    seen = set(excl)
    while len(out) < k:
        cand = rng.integers(0, N, size=2 * (k - len(out)) + 8)
        for c in cand.tolist():
            if c not in seen:
                seen.add(c)
                out.append(c)
                if len(out) == k:
                    break
    return np.asarray(out, np.int64)


def _fill_tail(rng: np.random.Generator, indices: np.ndarray, counts: np.ndarray, N: int) -> None:
    """Entries past a row's count get valid but unrelated pool rows: a decode
    that read them would give a wrong answer instead of an out-of-bounds read."""
    B, W = indices.shape
    for b in range(B):
        n = int(min(max(counts[b], 0), W))
        if n < W:
            indices[b, n:] = rng.integers(0, N, size=W - n)


def tiny(seed: int = 0) -> Case:
    """B=2, H=16, top-k 64, pool 4096 rows, counts {64, 37}."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    B, H, W, N = 2, 16, 64, 4096
    q8, qs, q16 = make_query(rng, B, H)
    kv8, ks = make_pool(ss.spawn(1)[0], N)
    counts = np.array([64, 37], np.int32)
    idx = np.zeros((B, W), np.int64)
    for b in range(B):
        idx[b] = rng.choice(N, size=W, replace=False)
    _fill_tail(rng, idx, counts, N)
    return Case("tiny", q8, kv8, idx.astype(np.int32), counts, _f32(192 ** -0.5), qs, ks, q16=q16)


def latency(seed: int = 1) -> Case:
    """Latency decode: B=5 verify rows, H=64, top-k 256, counts U[200,256] with
    one row of count 0, pool 65536 rows."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    B, H, W, N = 5, 64, 256, 65536
    q8, qs, q16 = make_query(rng, B, H)
    kv8, ks = make_pool(ss.spawn(1)[0], N)
    counts = rng.integers(200, 257, size=B).astype(np.int32)
    counts[rng.integers(0, B)] = 0
    idx = np.zeros((B, W), np.int64)
    for b in range(B):
        idx[b] = rng.choice(N, size=W, replace=False)
    _fill_tail(rng, idx, counts, N)
    return Case("latency", q8, kv8, idx.astype(np.int32), counts, _f32(192 ** -0.5), qs, ks, q16=q16)


def dsa(seed: int = 2) -> Case:
    """DSA decode: B=64, H=128, top-k 2048, counts U[1,2048] with 4 rows of
    count 0; half of each row's keys come from a 4096-row recent window."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    B, H, W, N, WIN = 64, 128, 2048, 262144, 4096
    q8, qs, q16 = make_query(rng, B, H)
    kv8, ks = make_pool(ss.spawn(1)[0], N)
    counts = rng.integers(1, W + 1, size=B).astype(np.int32)
    counts[rng.choice(B, size=4, replace=False)] = 0
    idx = np.zeros((B, W), np.int64)
    for b in range(B):
        start = int(rng.integers(0, N - WIN + 1))
        local = start + rng.choice(WIN, size=W // 2, replace=False)
        far = _unique_uniform(rng, N, W - W // 2, exclude=local)
        row = np.concatenate([local, far])
        rng.shuffle(row)
        idx[b] = row
    _fill_tail(rng, idx, counts, N)
    return Case("dsa", q8, kv8, idx.astype(np.int32), counts, _f32(192 ** -0.5), qs, ks, q16=q16)


def throughput(seed: int = 3) -> Case:
    """Throughput decode: B=256, H=128, top-k 2048 all full, pool 1048576 rows
    (~604 MB), 1% of the pool rows scaled x8 before quantisation."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    B, H, W, N = 256, 128, 2048, 1 << 20
    q8, qs, q16 = make_query(rng, B, H)
    kv8, ks = make_pool(ss.spawn(1)[0], N, heavy_frac=0.01, heavy_gain=8.0, rng=rng)
    counts = np.full(B, W, np.int32)
    idx = np.zeros((B, W), np.int64)
    for b in range(B):
        idx[b] = rng.choice(N, size=W, replace=False)
    return Case("throughput", q8, kv8, idx.astype(np.int32), counts, _f32(192 ** -0.5), qs, ks, q16=q16)


def dense(seed: int = 4) -> Case:
    """Dense-as-sparse: 32 requests x 4 causal query rows, L ~ U[1024,8192];
    row i of a request sees its first L-3+i cache rows, which live at
    scattered places of a shuffled 262144-row pool. H=16, top-k width 8192."""
    ss = np.random.SeedSequence(seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    R, QLEN, H, W, N = 32, 4, 16, 8192, 262144
    B = R * QLEN
    q8, qs, q16 = make_query(rng, B, H)
    kv8, ks = make_pool(ss.spawn(1)[0], N)
    perm = rng.permutation(N)
    L = rng.integers(1024, 8193, size=R)
    counts = np.zeros(B, np.int32)
    idx = np.zeros((B, W), np.int64)
    off = 0
    for r in range(R):
        tokens = perm[off:off + L[r]]
        off += int(L[r])
        for i in range(QLEN):
            b = r * QLEN + i
            n = int(L[r]) - QLEN + i + 1
            counts[b] = n
            idx[b, :n] = tokens[:n]
    _fill_tail(rng, idx, counts, N)
    return Case("dense", q8, kv8, idx.astype(np.int32), counts, _f32(192 ** -0.5), qs, ks, q16=q16)


CONFIGS = {
    "tiny": tiny,
    "latency": latency,
    "dsa": dsa,
    "throughput": throughput,
    "dense": dense,
}


def config(name: str) -> Case:
    return CONFIGS[name]()


def random_case(seed: int, B: int, H: int, W: int, N: int, counts=None,
                heavy_frac: float = 0.0, sm_scale: float | None = None,
                dup: bool = False) -> Case:
    """Small random case. ``counts`` may be a list (values may lie outside
    [0, W]: they are clamped by the call), else U[0, W]. ``dup`` draws each
    row's indices with replacement (duplicates allowed)."""
    ss = np.random.SeedSequence(1000 + seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    q8, qs, q16 = make_query(rng, B, H)
    kv8, ks = make_pool(ss.spawn(1)[0], N, heavy_frac=heavy_frac, rng=rng)
    if counts is None:
        counts = rng.integers(0, W + 1, size=B)
    counts = np.asarray(counts, np.int64).astype(np.int32)
    idx = np.zeros((B, W), np.int64)
    for b in range(B):
        if W == 0:
            continue
        if dup or W > N:
            idx[b] = rng.integers(0, N, size=W)
        else:
            idx[b] = rng.choice(N, size=W, replace=False)
    _fill_tail(rng, idx, counts, N)
    sm = _f32(192 ** -0.5) if sm_scale is None else _f32(sm_scale)
    return Case(f"random{seed}", q8, kv8, idx.astype(np.int32), counts, sm, qs, ks, q16=q16)


def grouped_case(seed: int, R: int, G: int, H: int, W: int, N: int, counts=None) -> Case:
    """R requests of G query rows that share one index list (the causal rows
    of a multi-token decode step). Every row of a request holds the request's
    whole list of W unique pool rows, of which it reads its first counts[b];
    by default row i of a request reads L - G + 1 + i, L ~ U[G, W]. ``counts``
    (R*G values, any order within a group, clamped by the call) overrides."""
    ss = np.random.SeedSequence(5000 + seed)
    rng = np.random.Generator(np.random.PCG64(ss.spawn(1)[0]))
    B = R * G
    q8, qs, q16 = make_query(rng, B, H)
    kv8, ks = make_pool(ss.spawn(1)[0], N, rng=rng)
    if counts is None:
        L = rng.integers(G, W + 1, size=R)
        counts = np.array([L[r] - G + 1 + i for r in range(R) for i in range(G)])
    counts = np.asarray(counts, np.int64).astype(np.int32)
    idx = np.zeros((B, W), np.int64)
    for r in range(R):
        lst = rng.choice(N, size=W, replace=False) if W <= N else rng.integers(0, N, size=W)
        idx[r * G:(r + 1) * G] = lst
    _fill_tail(rng, idx, counts, N)
    return Case(f"grouped{seed}", q8, kv8, idx.astype(np.int32), counts, _f32(192 ** -0.5), qs, ks, q16=q16)


def algorithmic_bytes(case: Case) -> dict:
    """Bytes a decode must move at least once: the distinct cache rows read,
    the query, the BF16 output and the FP32 LSE (index/count reads excluded)."""
    B, H = case.B, case.H
    kv = ROW * case.unique_rows()
    q = ROW * B * H
    out = 2 * LATENT * B * H + 4 * B * H
    flops = 2 * H * (ROW + LATENT) * case.gathered_rows()
    return {"kv_unique": kv, "kv_gathered": ROW * case.gathered_rows(), "q": q,
            "out": out, "total": kv + q + out, "flops": flops}


def seeded_permutation(seed: int, n: int) -> np.ndarray:
    return np.random.Generator(np.random.PCG64(seed)).permutation(n)


__all__ = ["Case", "CONFIGS", "config", "random_case", "algorithmic_bytes",
           "to_e4m3", "to_bf16_values", "ROW", "LATENT", "E4M3_MAX",
           "seeded_permutation"]


@dataclasses.dataclass
class TopkCase:
    """Inputs of the top-k select: bf16 logits (bits) [B, L] and row lengths."""
    name: str
    logits: np.ndarray    # uint16 [B, L] bf16 bits
    row_ends: np.ndarray  # int32 [B]
    K: int

    @property
    def B(self) -> int:
        return int(self.logits.shape[0])

    @property
    def L(self) -> int:
        return int(self.logits.shape[1])


def topk_case(seed: int, B: int, L: int, K: int, row_ends=None, scale: float = 1.0,
              nan_frac: float = 0.0) -> TopkCase:
    """bf16 logits N(0, scale^2) (a small scale makes many equal values), a
    fraction of NaNs at random places; row lengths uniform in [K / 2, L]
    unless given."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, L), dtype=np.float32) * np.float32(scale)
    if nan_frac > 0:
        x[rng.random((B, L)) < nan_frac] = np.nan
    bits = (np.ascontiguousarray(to_bf16_values(x), np.float32).view(np.uint32) >> 16).astype(np.uint16)
    if row_ends is None:
        ends = rng.integers(max(1, min(K // 2, L)), L + 1, size=B).astype(np.int32)
    else:
        ends = np.asarray(row_ends, np.int32)
    return TopkCase(f"topk{seed}", bits, ends, int(K))


def topk_config() -> TopkCase:
    """The indexer's select at DSA decode: 64 rows of bf16 logits over up to
    65536 cached tokens (row lengths uniform in [1024, 65536]), top-k 2048."""
    return topk_case(7, 64, 65536, 2048, scale=1.0,
                     row_ends=np.random.default_rng(8).integers(1024, 65537, size=64))
