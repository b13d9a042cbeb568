"""Seeded synthetic workloads for the H2O (Heavy-Hitter Oracle) decode/prefill path.

This module is the one piece of code shared by the CPU oracle's tests, the GPU
parity tests and the benchmark. It only draws inputs, rounds them to bf16 and
states workload sizes; it holds none of the eviction policy's arithmetic.

Synthetic stand-in. The pages measure on trained OPT / LLaMA / GPT-NeoX weights
and on datasets (XSUM, CNN/Daily Mail, lm-eval-harness tasks, PG-19), none of
which are used here. Instead every (layer, batch row, head) gets i.i.d. N(0,1)
queries, keys and values plus a power-law component along one shared unit
direction per head, so that a few keys attract most of the attention mass
("Accumulated attention scores follow a power-law distribution", H2O summary
page, section 3.2 Heavy-Hitters for Low Miss Rate):

    K_t += a_t * u_head,  a_t = 4 * rank_t ** (-alpha),  rank_t = pi(t) + 1
    Q_t += 2 * u_head

with pi a random permutation of the N = prompt + steps tokens of that row.
Everything is drawn in float32 and rounded once, round-to-nearest-even, to bf16.
Both the GPU path and the oracle consume the same bf16 bits.

Seeding: each (layer, b, head) row has its own numpy Generator seeded with
SeedSequence([0, cfg_id, layer, b, head]); the direction u of (layer, head) uses
SeedSequence([0, cfg_id, layer, U_STREAM, head]). Rows can therefore be drawn
one at a time, in any order, which lets a test regenerate just the rows it
samples.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

U_STREAM = 0xFFFF  # batch index reserved for the per-head direction stream


@dataclass(frozen=True)
class Workload:
    """One synthetic H2O workload: sizes, budget and power-law exponent."""

    cfg_id: int
    name: str
    layers: int
    batch: int
    heads: int
    head_dim: int
    prompt: int  # T, prompt tokens per row (uniform across the batch)
    steps: int  # S, decode steps after the prompt
    h: int  # heavy-hitter budget
    r: int  # recent-window budget
    alpha: float = 0.8  # Zipf exponent of the shared-direction magnitudes

    @property
    def k(self) -> int:
        return self.h + self.r

    @property
    def rows_per_layer(self) -> int:
        return self.batch * self.heads

    @property
    def tokens(self) -> int:
        return self.prompt + self.steps

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads the method is measured on. Sizes follow the model shapes
# the pages name (OPT-6.7B / OPT-30B at a 20 % budget, a LLaMA-7B-shaped long
# context, a large-batch case) plus a tiny case for exhaustive checking.
WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in (
        Workload(1, "tiny", 1, 1, 4, 64, 128, 64, 16, 16, 0.8),
        Workload(2, "opt-6.7b-layer", 1, 8, 32, 128, 2048, 256, 230, 230, 0.8),
        Workload(3, "opt-30b-stack", 48, 64, 56, 128, 512, 512, 102, 102, 0.8),
        Workload(4, "llama-7b-32k", 1, 4, 32, 128, 32768, 1024, 2048, 2048, 1.0),
        Workload(5, "batch-256", 1, 256, 32, 128, 1024, 1024, 205, 205, 0.8),
    )
}


# ----------------------------------------------------------------------------
# bf16 rounding (input preparation only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16, round-to-nearest-even; returns uint16 bits.

    Inputs here are finite (no NaN handling needed)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Widen bf16 bits to float32 exactly."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(u: np.ndarray) -> np.ndarray:
    """Widen bf16 bits to float64 exactly."""
    return bf16_bits_to_f32(u).astype(np.float64)


# ----------------------------------------------------------------------------
# generator
# ----------------------------------------------------------------------------
def head_direction(w: Workload, layer: int, head: int) -> np.ndarray:
    """Unit vector u of (layer, head), float32 [d]; shared by every batch row."""
    rng = np.random.default_rng(np.random.SeedSequence([0, w.cfg_id, layer, U_STREAM, head]))
    u = rng.standard_normal(w.head_dim, dtype=np.float32)
    return (u / np.float32(np.linalg.norm(u.astype(np.float64)))).astype(np.float32)


def row_tokens(w: Workload, layer: int, b: int, head: int, u: np.ndarray | None = None):
    """bf16 bits (uint16) of q, k, v for all N = prompt + steps tokens of one row.

    Returns three arrays of shape [N, d]. Tokens [0, T) form the prompt; token
    T + s is the input of decode step s."""
    n, d = w.tokens, w.head_dim
    if u is None:
        u = head_direction(w, layer, head)
    rng = np.random.default_rng(np.random.SeedSequence([0, w.cfg_id, layer, b, head]))
    x = rng.standard_normal((3, n, d), dtype=np.float32)
    perm = rng.permutation(n)
    a = (np.float32(4.0) * np.power((perm + 1).astype(np.float32), np.float32(-w.alpha))).astype(np.float32)
    x[1] += a[:, None] * u[None, :]
    x[0] += np.float32(2.0) * u[None, :]
    bits = f32_to_bf16_bits(x)
    return bits[0], bits[1], bits[2]


def stream_chunk(seed: int, chunk: int, steps: int, rows: int, d: int):
    """bf16 bits (uint16) of q, k, v for chunk `chunk` of a long decode stream:
    three arrays [steps, rows, d], the inputs of decode steps
    chunk * steps .. (chunk + 1) * steps - 1 of every row.

    For streams too long to draw at once (millions of steps): each chunk has its
    own Generator, SeedSequence([1, seed, chunk]), so any chunk can be drawn
    alone. Same construction as row_tokens with one unit direction u per stream
    (SeedSequence([1, seed, U_STREAM])), except that a key's power-law amplitude
    uses a rank drawn uniformly from 1 .. 2^20 instead of a permutation of the
    row's tokens: a_t = 4 * rank_t ** -0.8."""
    ru = np.random.default_rng(np.random.SeedSequence([1, seed, U_STREAM]))
    u = ru.standard_normal(d, dtype=np.float32)
    u = (u / np.float32(np.linalg.norm(u.astype(np.float64)))).astype(np.float32)
    rng = np.random.default_rng(np.random.SeedSequence([1, seed, chunk]))
    x = rng.standard_normal((3, steps, rows, d), dtype=np.float32)
    rank = rng.integers(1, 1 << 20, size=(steps, rows), endpoint=True).astype(np.float32)
    a = (np.float32(4.0) * np.power(rank, np.float32(-0.8))).astype(np.float32)
    x[1] += a[..., None] * u
    x[0] += np.float32(2.0) * u
    bits = f32_to_bf16_bits(x)
    return bits[0], bits[1], bits[2]


def layer_tokens(w: Workload, layer: int, rows: list[tuple[int, int]] | None = None):
    """bf16 bits of q, k, v for one layer: arrays [B, H, N, d] (uint16).

    With ``rows`` (a list of (b, head)), only those rows are drawn and the
    arrays have shape [len(rows), N, d] instead."""
    n, d = w.tokens, w.head_dim
    dirs = [head_direction(w, layer, j) for j in range(w.heads)]
    if rows is not None:
        out = np.empty((3, len(rows), n, d), dtype=np.uint16)
        for i, (b, j) in enumerate(rows):
            q, k, v = row_tokens(w, layer, b, j, dirs[j])
            out[0, i], out[1, i], out[2, i] = q, k, v
        return out[0], out[1], out[2]
    out = np.empty((3, w.batch, w.heads, n, d), dtype=np.uint16)
    for b in range(w.batch):
        for j in range(w.heads):
            q, k, v = row_tokens(w, layer, b, j, dirs[j])
            out[0, b, j], out[1, b, j], out[2, b, j] = q, k, v
    return out[0], out[1], out[2]


# ----------------------------------------------------------------------------
# sizes (bytes and flops), used for rooflines and the pages' sizing example
# ----------------------------------------------------------------------------
def kv_cache_bytes(layers: int, hidden: int, batch: int, seq: int, bytes_per_elem: int = 2) -> int:
    """Bytes of a full (un-evicted) KV cache: K and V, every layer, every token.

    The H2O summary page (section 1, Introduction) sizes a 30B model at batch
    128 and sequence 1024 at 180 GB; OPT-30B has 48 layers of hidden size 7168
    and the figure holds for 2-byte elements."""
    return 2 * layers * hidden * batch * seq * bytes_per_elem


def decode_bytes_per_row_step(k: int, d: int, kv: str = "bf16", layout: str = "slots",
                              h: int | None = None) -> int:
    """Algorithmic HBM bytes of one decode step of one (layer, b, head) row.

    Reads: the k cached K and V rows (bf16, 4kd), the k accumulated scores
    (fp32, 4k) and positions (int32, 4k), and q, k_new, v_new (bf16, 6d).
    Writes: the k updated scores (4k), the new slot's K/V (4d) with its
    position and score (8), and the fp32 output (4d).
    With an FP8 cache (kv="fp8") a slot holds E4M3 codes (2kd for K and V)
    plus two fp32 scales (8k read), and the new slot is written as 2d code
    bytes plus 8 scale bytes.
    Ring layout (layout="ring", h heavy slots): positions are read for the h
    heavy slots only (4h instead of 4k), and the token leaving the recent
    window moves into the heavy slot it displaces (4d read, 4d + 8 written;
    counted every step, an upper bound)."""
    if kv == "fp8":
        return 2 * k * d + 8 * k + 12 * k + 6 * d + 2 * d + 16 + 4 * d
    if layout == "ring":
        return 4 * k * d + 8 * k + 4 * h + 6 * d + 4 * d + 8 + 4 * d + 8 * d + 8
    return 4 * k * d + 12 * k + 6 * d + 4 * d + 8 + 4 * d


def prefill_flops_per_row(T: int, d: int) -> int:
    """Algorithmic flops of causal prefill attention for one row: QK^T and PV
    over the T(T+1)/2 causal (query, key) pairs, 2d flops each."""
    return 2 * d * T * (T + 1)


def prefill_bytes_per_row(T: int, d: int, k: int, kv: str = "bf16") -> int:
    """Algorithmic HBM bytes of the prefill of one row: the least any
    implementation moves. Reads: the prompt's Q, K and V (bf16, 6Td). Writes:
    the fp32 attention output (4Td) and the min(T, k) kept cache slots -- K and
    V (bf16 4d a slot; FP8 codes 2d plus two fp32 scales) with their position
    and accumulated score (8). The column sums and the kept positions are
    intermediates a fused design keeps on chip, so they are not counted."""
    kept = min(T, k)
    slot = 2 * d + 8 if kv == "fp8" else 4 * d
    return 6 * T * d + 4 * T * d + kept * (slot + 8)
