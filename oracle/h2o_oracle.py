"""fp64 CPU oracle of the H2O (Heavy-Hitter Oracle) KV-cache eviction policy.

TEST INFRASTRUCTURE. This package is the independent checker of the CUDA path.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
it; the library (the C-ABI shared object and its Python binding) never does, and
this file imports nothing from the library. The two share no code: the only
module both sides use is the seeded input generator (``workloads``), which holds
none of the policy's arithmetic.

Sources (cited by page title and section):
  [H2O] "H2O: Heavy-Hitter Oracle for Efficient Generative Inference of Large
        Language Models", the section-by-section summary page of arXiv
        2306.14048v3 (paperlayer.ai).
  [ABS] the H2O abstract as listed on the attentionhub.org discoveries pages.

What the policy computes (one (layer, batch row, head) row at a time; rows are
independent):
  * Each row keeps at most k = h + r cached tokens: h heavy hitters and the r
    most recent ([H2O] A, System Details: heavy-hitter region plus a
    recent-token region; [H2O] TL;DR and section 2: the cache size is fixed at
    k and at most one entry is evicted between consecutive decoding steps).
  * A token's accumulated score is the running sum of the normalised attention
    (softmax probability) it has received ([H2O] section 1 "local accumulated
    attention statistics"; section 3.2 "accumulated attention scores").
  * Prefill: full causal attention over the prompt; the accumulated score of
    prompt token j is the column sum of the causal softmax matrix; keep the r
    most recent tokens plus the top-h of the rest ([H2O] A, Pseudocode: K heavy
    hitters and K recent tokens are selected from the prompt).
  * Decode: append the new token, attend over the cached set plus the new
    token, add each probability to the token's score, then evict the token with
    the lowest score among those outside the r most recent positions ([H2O]
    section 4.1: with budget 3 the fourth decoding step evicts the token with
    the lowest accumulated score).

Readings where the pages are silent (each is listed in the design notes):
  * logits are scaled by ``scale`` (default 1/sqrt(d), the usual scaled dot
    product; the recursive attention definition of [H2O] D prints no scale);
  * ties in the accumulated score are broken by position, smaller position
    evicted first; prefill uses the same total order (drop by (score, pos)
    ascending), so among equal scores the later position is kept;
  * a prompt of T <= k tokens is kept whole; no eviction happens until the
    cache would exceed k;
  * with r = 0 the new token is itself an eviction candidate; if it has the
    lowest key it is dropped at once;
  * evicted tokens lose their score and never re-enter; prefill scores carry
    into decode.

All arithmetic is float64 on the bf16 inputs widened exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import kv_fp8

NEAR_TIE = 1e-4  # relative margin below which an eviction decision is a near-tie


def default_scale(d: int) -> float:
    return 1.0 / np.sqrt(d)


# ----------------------------------------------------------------------------
# Prefill
# ----------------------------------------------------------------------------
def prefill_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                      row_block: int | None = None):
    """Causal softmax attention over a prompt and the column sums of its
    probability matrix ([H2O] A Pseudocode; section 3.2 accumulated scores).

    For every query i: s_ij = scale * q_i . k_j for j <= i, P_i = softmax(s_i),
    O_i = sum_j P_ij v_j. The accumulated score of token j is
    colsum_j = sum_{i >= j} P_ij.

    ``row_block`` evaluates the definition for a block of query rows at a time
    (each row's softmax is still computed whole), which bounds memory for long
    prompts. Returns (O [T,d], colsum [T], lse [T]) in float64; lse_i is the
    natural log of the softmax normaliser of row i including its max."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    T = Q.shape[0]
    d = V.shape[1] if V.ndim == 2 else 0
    O = np.zeros((T, d))
    colsum = np.zeros(T)
    lse = np.zeros(T)
    if T == 0:
        return O, colsum, lse
    blk = T if row_block is None else max(1, row_block)
    for i0 in range(0, T, blk):
        i1 = min(T, i0 + blk)
        S = scale * (Q[i0:i1] @ K[:i1].T)  # [rows, keys j < i1]
        rows = np.arange(i0, i1)[:, None]
        cols = np.arange(i1)[None, :]
        S = np.where(cols <= rows, S, -np.inf)  # causal: key j visible to query i iff j <= i
        m = S.max(axis=1, keepdims=True)
        E = np.exp(S - m)
        Z = E.sum(axis=1, keepdims=True)
        P = E / Z
        O[i0:i1] = P @ V[:i1]
        colsum[:i1] += P.sum(axis=0)
        lse[i0:i1] = (m + np.log(Z))[:, 0]
    return O, colsum, lse


def prefill_select(colsum: np.ndarray, h: int, r: int):
    """Positions kept after prefill ([H2O] A Pseudocode and System Details).

    If the prompt has T <= h + r tokens, every token is kept. Otherwise the r
    most recent positions T-r .. T-1 are kept, and of the candidates 0 .. T-r-1
    the h with the largest keys (score, position) are kept: candidates are
    ordered by (score ascending, position ascending) and the first T-r-h are
    dropped.

    Returns (kept positions ascending, boundary margin). The margin is
    (s_kept_min - s_dropped_max) / s_kept_min between the smallest kept and the
    largest dropped heavy-hitter candidate (inf when nothing competes)."""
    T = colsum.shape[0]
    if T <= h + r:
        return np.arange(T, dtype=np.int64), np.inf
    n_cand = T - r
    cand = np.arange(n_cand)
    order = np.lexsort((cand, colsum[:n_cand]))  # primary: score, secondary: position
    n_drop = n_cand - h
    heavy = order[n_drop:]
    margin = np.inf
    if h > 0 and n_drop > 0:
        s_keep = colsum[order[n_drop]]
        s_drop = colsum[order[n_drop - 1]]
        margin = (s_keep - s_drop) / s_keep if s_keep > 0 else 0.0
    kept = np.sort(np.concatenate([heavy, np.arange(n_cand, T)]))
    return kept.astype(np.int64), margin


@dataclass
class RowCache:
    """Retained set of one row: positions with their K, V and accumulated score."""

    h: int
    r: int
    scale: float
    pos: np.ndarray  # int64 [n]
    K: np.ndarray  # float64 [n, d]
    V: np.ndarray  # float64 [n, d]
    score: np.ndarray  # float64 [n]
    t: int  # position of the next token to be decoded
    # With an FP8 cache (kv_fp8 module): K and V hold the dequantised tokens and
    # these arrays the stored codes [n, d] (uint8) and scales [n] (float32).
    kv_fp8: bool = False
    Kc: np.ndarray | None = None
    Ks: np.ndarray | None = None
    Vc: np.ndarray | None = None
    Vs: np.ndarray | None = None

    @property
    def k(self) -> int:
        return self.h + self.r


@dataclass
class PrefillResult:
    cache: RowCache
    O: np.ndarray
    colsum: np.ndarray
    lse: np.ndarray
    kept: np.ndarray
    margin: float


def _quantized(X: np.ndarray):
    """Codes, scales and dequantised rows of token vectors X [n, d] (kv_fp8)."""
    n, d = X.shape
    codes = np.zeros((n, d), dtype=np.uint8)
    scales = np.zeros(n, dtype=np.float32)
    for i in range(n):
        codes[i], scales[i] = kv_fp8.quantize_vector(X[i])
    deq = np.array([kv_fp8.dequantize_vector(codes[i], scales[i]) for i in range(n)]).reshape(n, d)
    return codes, scales, deq


def prefill(Q, K, V, h: int, r: int, scale: float | None = None,
            row_block: int | None = None, kv_fp8_cache: bool = False) -> PrefillResult:
    """Prefill one row: causal attention, column-sum scores, selection.

    Retained tokens carry their prefill column sums forward as their
    accumulated scores. With ``kv_fp8_cache`` the attention still runs on the
    full-precision prompt and the retained tokens are stored quantised
    (kv_fp8 module)."""
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    d = K.shape[1]
    if scale is None:
        scale = default_scale(d)
    O, colsum, lse = prefill_attention(Q, K, V, scale, row_block)
    kept, margin = prefill_select(colsum, h, r)
    cache = RowCache(h, r, scale, kept.copy(), K[kept].copy(), V[kept].copy(),
                     colsum[kept].copy(), K.shape[0])
    if kv_fp8_cache:
        cache.kv_fp8 = True
        cache.Kc, cache.Ks, cache.K = _quantized(cache.K)
        cache.Vc, cache.Vs, cache.V = _quantized(cache.V)
    return PrefillResult(cache, O, colsum, lse, kept, margin)


# ----------------------------------------------------------------------------
# Decode
# ----------------------------------------------------------------------------
@dataclass
class StepLog:
    out: np.ndarray  # [d] attention output of the new token
    p: np.ndarray  # probabilities over (previously retained tokens ..., new token)
    pos_attended: np.ndarray  # positions matching p
    evicted: int  # evicted position, -1 if none
    margin: float  # (s2 - s1) / s2 between evicted and runner-up candidate
    n_candidates: int = 0
    evicted_score: float = 0.0  # accumulated score the evicted token held when it left


def decode_step(c: RowCache, q, k_new, v_new) -> StepLog:
    """One decode step of one row, in place on ``c``.

    Order ([H2O] section 4.1 illustration; section 2 problem formulation):
      1. append the new token at position t;
      2. attend over the retained tokens plus the new one:
         p = softmax(scale * K q), out = sum_j p_j v_j;
      3. accumulate: every retained token's score += p_j; the new token's
         score is its own p;
      4. if more than k tokens are now held, evict one: among candidates with
         position <= t - r (the r most recent, t included, are never evicted),
         the smallest (score, position);
      5. the survivors form the new retained set."""
    q = np.asarray(q, dtype=np.float64)
    t = c.t
    k_new = np.asarray(k_new, dtype=np.float64)
    v_new = np.asarray(v_new, dtype=np.float64)
    if c.kv_fp8:  # the new token is stored quantised before it is attended to
        kc, ks, k_new = _quantized(k_new[None, :])
        vc, vs, v_new = _quantized(v_new[None, :])
        Kc, Ks = np.vstack([c.Kc, kc]), np.append(c.Ks, ks)
        Vc, Vs = np.vstack([c.Vc, vc]), np.append(c.Vs, vs)
        k_new, v_new = k_new[0], v_new[0]
    pos = np.append(c.pos, t)
    K = np.vstack([c.K, k_new[None, :]])
    V = np.vstack([c.V, v_new[None, :]])
    s = c.scale * (K @ q)
    e = np.exp(s - s.max())
    p = e / e.sum()
    out = p @ V
    score = np.append(c.score + p[:-1], p[-1])
    pos_attended = pos.copy()

    evicted, margin, n_cand, ev_score = -1, np.inf, 0, 0.0
    if pos.shape[0] > c.k:
        cand = np.nonzero(pos <= t - c.r)[0]
        n_cand = cand.shape[0]
        order = cand[np.lexsort((pos[cand], score[cand]))]  # (score, pos) ascending
        e_idx = order[0]
        evicted = int(pos[e_idx])
        ev_score = float(score[e_idx])
        if n_cand > 1:
            s1, s2 = score[order[0]], score[order[1]]
            margin = (s2 - s1) / s2 if s2 > 0 else 0.0
        keep = np.ones(pos.shape[0], dtype=bool)
        keep[e_idx] = False
        pos, K, V, score = pos[keep], K[keep], V[keep], score[keep]
        if c.kv_fp8:
            Kc, Ks, Vc, Vs = Kc[keep], Ks[keep], Vc[keep], Vs[keep]

    c.pos, c.K, c.V, c.score, c.t = pos, K, V, score, t + 1
    if c.kv_fp8:
        c.Kc, c.Ks, c.Vc, c.Vs = Kc, Ks, Vc, Vs
    return StepLog(out, p, pos_attended, evicted, margin, n_cand, ev_score)


# ----------------------------------------------------------------------------
# Whole row: prefill then S decode steps
# ----------------------------------------------------------------------------
@dataclass
class RowTrace:
    prefill: PrefillResult
    outs: list = field(default_factory=list)
    evicted: list = field(default_factory=list)
    margins: list = field(default_factory=list)
    kept_after: list = field(default_factory=list)
    scores_after: list = field(default_factory=list)
    evicted_scores: list = field(default_factory=list)  # score the evicted token held (0 if none)


def run_row(q_all, k_all, v_all, T: int, S: int, h: int, r: int,
            scale: float | None = None, row_block: int | None = None,
            keep_sets: bool = True, kv_fp8_cache: bool = False) -> RowTrace:
    """Prefill tokens [0, T) then decode tokens T .. T+S-1 of one row."""
    q_all = np.asarray(q_all, dtype=np.float64)
    k_all = np.asarray(k_all, dtype=np.float64)
    v_all = np.asarray(v_all, dtype=np.float64)
    pre = prefill(q_all[:T], k_all[:T], v_all[:T], h, r, scale, row_block, kv_fp8_cache)
    tr = RowTrace(pre)
    c = pre.cache
    for s in range(S):
        lg = decode_step(c, q_all[T + s], k_all[T + s], v_all[T + s])
        tr.outs.append(lg.out)
        tr.evicted.append(lg.evicted)
        tr.margins.append(lg.margin)
        tr.evicted_scores.append(lg.evicted_score)
        if keep_sets:
            tr.kept_after.append(c.pos.copy())
            tr.scores_after.append(c.score.copy())
    return tr
