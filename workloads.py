"""Seeded synthetic inputs for the selected-token log-probability workloads.

This module is shared by the CPU oracle's tests and the CUDA path's tests and
benchmark, and it holds none of the operator's arithmetic: it only draws
logits, targets and upstream gradients, and stores them in the element type
the operator reads (float32, or bfloat16 / float16 bit patterns in uint16).

Every random number comes from numpy's PCG64 seeded through a SeedSequence
keyed by (workload seed, stream, chunk).  Rows are drawn in chunks of
``CHUNK_ROWS`` with one independent stream per chunk, so any subset of chunks
can be regenerated on its own and chunks can be drawn in parallel threads
without changing a single byte.

The five workloads follow the shapes, distributions and structure of the
operator page's measured shapes ("Batch-Invariant LogP", "Measured results":
vocabularies up to 151936, 4096-8192 rows, bf16) and its invariance contract
("Batch-Invariance"):

  tiny      N=16, V=4096 fp32, x = 2*randn, tile 512, rows 3 and 11 ignored,
            g = 1, fp32 gradient.
  prefill   B=4 x T=1024, V=151936 bf16, x = 3*randn plus one +12 spike per
            row, row stride 155648 with -inf in the pad columns, 5% of rows
            ignored, tile 4096, forward only.
  training  B=8 x T=2048, V=151936 bf16, x = 3*randn, 70% of targets drawn from
            the row's five largest logits, g ~ N(0, 1) fp32, bf16 gradient.
  decode    a bank of 256 rows, V=151936 bf16, x = 3*randn, uniform targets.
  packed    B=2 x T=8192 rows packed from sequences of uniform length 256-4096,
            right-padded with ignore_index, V=151936 bf16, x = 3*randn.
  linear    the fused LM-head + logp ("[RFC][ROCm] End-to-end optimization of
            bitwise VIME R/R beyond native P/P", "Workstream 3"; its target
            model is Qwen3-8B: hidden size 4096, vocabulary 151936): hidden
            states [N, 4096] bf16 ~ randn, LM-head weight [151936, 4096] bf16
            ~ randn * 3/64 (so that the logits have standard deviation ~3, as
            in the other workloads), uniform targets, 5% of rows ignored.

"randn" scaled by s means a standard normal times s (s is the standard
deviation).  Values are drawn in float32 and stored with round-to-nearest-even.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK_ROWS = 256
VOCAB = 151936
PADDED_VOCAB = 155648
IGNORE_INDEX = -100
BF16_NEG_INF = 0xFF80

SEEDS = {"tiny": 0, "prefill": 1, "training": 2, "decode": 3, "packed": 4, "linear": 5}
HIDDEN = 4096


def rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest, ties to even (finite x)."""
    b = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    lsb = b >> np.uint32(16)
    lsb &= np.uint32(1)
    b += np.uint32(0x7FFF)
    b += lsb
    b >>= np.uint32(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    """Store float32 values in the element type the operator reads."""
    if dtype == "float32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bfloat16":
        return f32_to_bf16_bits(x)
    if dtype == "float16":
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)
    raise ValueError(dtype)


def stored_to_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "float32":
        return a
    if dtype == "bfloat16":
        return bf16_bits_to_f32(a)
    return a.view(np.float16).astype(np.float32)


@dataclass
class Workload:
    name: str
    logits: np.ndarray          # [N, ld] stored elements (float32, or uint16 bits)
    dtype: str                  # "float32" | "bfloat16" | "float16"
    vocab: int
    tile_v: int
    target_ids: np.ndarray      # [N] int64
    ignore_index: int = IGNORE_INDEX
    grad_logp: np.ndarray | None = None   # [N] float32, None for forward-only workloads
    dlogits_dtype: str = "bfloat16"
    meta: dict = field(default_factory=dict)

    @property
    def n_rows(self) -> int:
        return self.logits.shape[0]

    @property
    def ld(self) -> int:
        return self.logits.shape[1]


def _pool_map(fn, items, workers=None):
    items = list(items)
    workers = workers or min(16, os.cpu_count() or 1, max(1, len(items)))
    if workers <= 1 or len(items) <= 1:
        return [fn(i) for i in items]
    with ThreadPoolExecutor(workers) as ex:
        return list(ex.map(fn, items))


def _normal_chunk(seed: int, chunk: int, rows: int, vocab: int, scale: float) -> np.ndarray:
    x = rng(seed, 0, chunk).standard_normal((rows, vocab), dtype=np.float32)
    x *= np.float32(scale)
    return x


def _chunks(n_rows: int, chunks):
    total = -(-n_rows // CHUNK_ROWS)
    return range(total) if chunks is None else sorted(set(chunks))


def _fill_rows(out: np.ndarray, n_rows: int, chunks, make_chunk):
    """Run make_chunk(chunk) -> stored rows for each selected chunk, in threads."""
    def work(c):
        r0 = c * CHUNK_ROWS
        r1 = min(n_rows, r0 + CHUNK_ROWS)
        out[r0:r1, : make_chunk.width] = make_chunk(c, r1 - r0)
    _pool_map(work, _chunks(n_rows, chunks))


def tiny() -> Workload:
    seed, n, v = SEEDS["tiny"], 16, 4096
    x = _normal_chunk(seed, 0, n, v, 2.0)
    t = rng(seed, 1).integers(0, v, n, dtype=np.int64)
    t[3] = IGNORE_INDEX
    t[11] = IGNORE_INDEX
    return Workload("tiny", store(x, "float32"), "float32", v, 512, t,
                    grad_logp=np.ones(n, np.float32), dlogits_dtype="float32")


def _bf16_rows(seed, n_rows, vocab, ld, scale, chunks, pad_bits=None, spike=None):
    out = np.zeros((n_rows, ld), np.uint16)
    if pad_bits is not None and ld > vocab:
        out[:, vocab:] = pad_bits

    def make(c, rows):
        x = _normal_chunk(seed, c, rows, vocab, scale)
        if spike is not None:
            cols = rng(seed, 2, c).integers(0, vocab, rows)
            x[np.arange(rows), cols] += np.float32(spike)
        return f32_to_bf16_bits(x)
    make.width = vocab
    _fill_rows(out, n_rows, chunks, make)
    return out


def prefill(ld: int = PADDED_VOCAB, chunks=None) -> Workload:
    """B=4, T=1024; one +12 spike per row; pad columns (ld > V) hold -inf."""
    seed, n, v = SEEDS["prefill"], 4 * 1024, VOCAB
    logits = _bf16_rows(seed, n, v, ld, 3.0, chunks, pad_bits=BF16_NEG_INF, spike=12.0)
    t = rng(seed, 1).integers(0, v, n, dtype=np.int64)
    n_ignored = int(round(0.05 * n))
    t[rng(seed, 3).permutation(n)[:n_ignored]] = IGNORE_INDEX
    return Workload("prefill", logits, "bfloat16", v, 4096, t,
                    meta={"n_ignored": n_ignored, "B": 4, "T": 1024})


def _top5_target(row: np.ndarray, fifth: float, r: np.random.Generator) -> int:
    """Uniform pick among the row's five largest entries (ties -> lower index).

    `fifth` is the row's fifth largest value."""
    idx = np.flatnonzero(row >= fifth)
    order = np.lexsort((idx, -row[idx]))                # value desc, then index asc
    top5 = idx[order[:5]]
    return int(top5[r.integers(0, 5)])


def training(n_rows: int = 8 * 2048, chunks=None) -> Workload:
    """B=8, T=2048; 70% of targets from the row's top-5 columns, 30% uniform."""
    seed, v = SEEDS["training"], VOCAB
    logits = np.zeros((n_rows, v), np.uint16)
    targets = np.zeros(n_rows, np.int64)

    def make(c, rows):
        bits = f32_to_bf16_bits(_normal_chunk(seed, c, rows, v, 3.0))
        vals = bf16_bits_to_f32(bits)
        fifth = np.partition(vals, v - 5, axis=1)[:, v - 5]
        r = rng(seed, 4, c)
        pick_top = r.random(rows) < 0.7
        uniform = r.integers(0, v, rows, dtype=np.int64)
        r0 = c * CHUNK_ROWS
        for i in range(rows):
            targets[r0 + i] = _top5_target(vals[i], fifth[i], r) if pick_top[i] else uniform[i]
        return bits
    make.width = v
    _fill_rows(logits, n_rows, chunks, make)
    g = rng(seed, 5).standard_normal(n_rows, dtype=np.float32)
    return Workload("training", logits, "bfloat16", v, 4096, targets, grad_logp=g,
                    dlogits_dtype="bfloat16", meta={"B": 8, "T": n_rows // 8})


def decode_bank() -> Workload:
    seed, n, v = SEEDS["decode"], 256, VOCAB
    logits = _bf16_rows(seed, n, v, v, 3.0, None)
    t = rng(seed, 1).integers(0, v, n, dtype=np.int64)
    return Workload("decode", logits, "bfloat16", v, 4096, t)


def decode_draws(n: int, draws: int = 8):
    """Seeded row selections of the decode bank: `draws` arrays of n distinct bank rows."""
    r = rng(SEEDS["decode"], 6, n)
    return [r.permutation(256)[:n] for _ in range(draws)]


def packed_layout(B: int = 2, T: int = 8192):
    """Greedy packing of sequences of uniform length 256..4096 into B rows of T slots.

    Returns a list of (batch_row, start, length); slots after the last sequence
    of a batch row are padding."""
    r = rng(SEEDS["packed"], 1)
    seqs = []
    for b in range(B):
        pos = 0
        while True:
            length = int(r.integers(256, 4097))
            if pos + length > T:
                break
            seqs.append((b, pos, length))
            pos += length
    return seqs


def packed(B: int = 2, T: int = 8192) -> Workload:
    seed, v = SEEDS["packed"], VOCAB
    n = B * T
    logits = _bf16_rows(seed, n, v, v, 3.0, None)
    t = np.full(n, IGNORE_INDEX, np.int64)
    seqs = packed_layout(B, T)
    r = rng(seed, 2)
    for b, start, length in seqs:
        t[b * T + start: b * T + start + length] = r.integers(0, v, length, dtype=np.int64)
    return Workload("packed", logits, "bfloat16", v, 4096, t, meta={"B": B, "T": T, "seqs": seqs})


def random_rows(seed: int, n_rows: int, vocab: int, dtype: str = "bfloat16", scale: float = 3.0,
                ld: int | None = None, pad_value: float = float("nan"), tile_v: int = 4096,
                ignore_every: int = 0) -> Workload:
    """Small general-purpose workload for edge cases (odd V, row strides, dtypes).

    Pad columns (ld > vocab) hold `pad_value` (NaN by default, so that a
    kernel that reads them would show it)."""
    ld = vocab if ld is None else ld
    x = np.full((n_rows, ld), pad_value, np.float32)
    x[:, :vocab] = rng(seed, 0, 0).standard_normal((n_rows, vocab), dtype=np.float32) * np.float32(scale)
    t = rng(seed, 1).integers(0, vocab, n_rows, dtype=np.int64)
    if ignore_every:
        t[::ignore_every] = IGNORE_INDEX
    g = rng(seed, 5).standard_normal(n_rows, dtype=np.float32)
    return Workload(f"random{seed}", store(x, dtype), dtype, vocab, tile_v, t, grad_logp=g,
                    dlogits_dtype="float32")


@dataclass
class LinearWorkload:
    """Inputs of the fused LM-head + logp: hidden [N, H] and weight [V, H] as
    stored bf16 bits, targets [N], upstream gradients [N]."""
    name: str
    hidden: np.ndarray
    weight: np.ndarray
    dtype: str
    target_ids: np.ndarray
    grad_logp: np.ndarray
    ignore_index: int = IGNORE_INDEX

    @property
    def n_rows(self) -> int:
        return self.hidden.shape[0]

    @property
    def vocab(self) -> int:
        return self.weight.shape[0]

    @property
    def hidden_size(self) -> int:
        return self.hidden.shape[1]


def _normal_rows(seed: int, stream: int, n_rows: int, width: int, scale: float, chunks=None,
                 dtype: str = "bfloat16") -> np.ndarray:
    out = np.zeros((n_rows, width), np.uint16)

    def make(c, rows):
        x = rng(seed, stream, c).standard_normal((rows, width), dtype=np.float32)
        x *= np.float32(scale)
        return store(x, dtype)
    make.width = width
    _fill_rows(out, n_rows, chunks, make)
    return out


def linear_hidden(n_rows: int, hidden: int = HIDDEN, seed: int = SEEDS["linear"], chunks=None,
                  dtype: str = "bfloat16") -> np.ndarray:
    """Hidden states [n_rows, hidden] ~ randn (bf16 or fp16 bits); chunk c of 256 rows is
    stream (10, c)."""
    return _normal_rows(seed, 10, n_rows, hidden, 1.0, chunks, dtype)


def linear_weight(vocab: int = VOCAB, hidden: int = HIDDEN, seed: int = SEEDS["linear"], chunks=None,
                  dtype: str = "bfloat16") -> np.ndarray:
    """LM-head weight [vocab, hidden] ~ randn * 3 / sqrt(hidden) (bf16 or fp16 bits); chunk c
    of 256 vocabulary rows is stream (11, c)."""
    return _normal_rows(seed, 11, vocab, hidden, 3.0 / np.sqrt(hidden), chunks, dtype)


def linear(n_rows: int = 16384, hidden: int = HIDDEN, vocab: int = VOCAB, seed: int = SEEDS["linear"],
           ignore_frac: float = 0.05, dtype: str = "bfloat16") -> LinearWorkload:
    """Qwen3-8B-shaped LM head over n_rows tokens (B=8 x T=2048 by default)."""
    x = linear_hidden(n_rows, hidden, seed, dtype=dtype)
    w = linear_weight(vocab, hidden, seed, dtype=dtype)
    t = rng(seed, 1).integers(0, vocab, n_rows, dtype=np.int64)
    n_ignored = int(round(ignore_frac * n_rows))
    t[rng(seed, 3).permutation(n_rows)[:n_ignored]] = IGNORE_INDEX
    g = rng(seed, 5).standard_normal(n_rows, dtype=np.float32)
    return LinearWorkload(f"linear{n_rows}x{hidden}x{vocab}", x, w, dtype, t, g)
