"""Per-row pieces of the GPU-versus-oracle parity check (test support only).

Nothing here imports torch or touches a GPU: these functions run in spawn
worker processes next to the CPU oracle, and the CPU tests drive them with
traces of planted-mistake oracles to show that the comparison catches them.

Rules (the benchmark spec's tolerances, with the near-tie reading of the design
notes):
  * outputs within MAX_ABS max-abs and MEAN_ABS mean-abs of the fp64 oracle;
  * accumulated scores of the retained tokens within SCORE_RTOL relative of
    the oracle's;
  * retained position sets and evicted positions equal, except where the
    oracle's relative margin (s2 - s1) / s2 between its evicted key and the
    runner-up is below the near-tie threshold. Even there a differing decision
    is excused only if it is itself a near-minimal choice under the oracle's
    scores: the GPU's evicted token must be an eviction candidate the oracle
    kept, whose oracle score s_g lies within the threshold of the oracle's
    evicted score, (s_g - s1) / s_g < NEAR_TIE. At prefill every token the two
    sides disagree on must be a heavy-hitter candidate whose oracle column sum
    lies within the threshold of the boundary (the smallest kept candidate
    score). So a wrong margin can never excuse a real mismatch.

Tolerance of the scores. A retained token's score is a sum of positive
softmax probabilities (its column sum at prefill plus one probability per
decode step), so its relative error is at most the largest relative error of
its terms plus the rounding of the fp32 sums. A probability's relative error
is the absolute error of its logit (an fp32 dot product of d bf16 products,
about sqrt(d) 2^-24 sum |q_i k_i| / sqrt(d), some 1e-6 here) plus that of the
normaliser and of the hardware exp2 (2^-22). Summing n terms in fp32 adds at
most about n 2^-24 in the worst case and sqrt(n) 2^-24 typically (n = T + S,
3e-6 for 2304 terms). 1e-4 leaves a wide margin over the 3e-6 to 4e-6 these
errors produce, and is far below what any mistake in the accumulation does:
a dropped normaliser multiplies a score by the softmax denominator, a dropped
step removes a whole probability, a dropped prefill column sum removes most of
the score.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
from workloads import bf16_bits_to_f64, head_direction, row_tokens

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
SCORE_RTOL = 1e-4
NEAR_TIE = oracle.NEAR_TIE


# ----------------------------------------------------------------------------- oracle side
def trace_dict(tr) -> dict:
    """Compact per-step logs of an oracle RowTrace."""
    pre = tr.prefill
    S = len(tr.outs)
    d = pre.O.shape[1] if pre.O.ndim == 2 else 0
    return {
        "O": pre.O.astype(np.float32),
        "colsum": pre.colsum,
        "kept": pre.kept,
        "kept_scores": pre.colsum[pre.kept],
        "margin": pre.margin,
        "outs": np.array(tr.outs, dtype=np.float64).reshape(S, d),
        "evicted": np.array(tr.evicted, dtype=np.int64),
        "margins": np.array(tr.margins, dtype=np.float64),
        "evicted_scores": np.array(tr.evicted_scores, dtype=np.float64),
        "kept_after": tr.kept_after,
        "scores_after": tr.scores_after,
    }


def oracle_row(job) -> dict:
    """Pool worker: runs the oracle on one row of a workload and returns its logs.

    job = (workload, layer, b, head, row_block, fp8 cache, prompt length)."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    w, layer, b, j, row_block, fp8, prompt = job
    q, k, v = row_tokens(w, layer, b, j, head_direction(w, layer, j))
    q, k, v = bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)
    tr = oracle.run_row(q, k, v, prompt, w.steps, w.h, w.r, row_block=row_block,
                        kv_fp8_cache=fp8)
    return trace_dict(tr)


def row_bits(job):
    """Pool worker: bf16 bits [3, N, d] of one row (job = (workload, layer, b, head))."""
    w, layer, b, j = job
    return np.stack(row_tokens(w, layer, b, j, head_direction(w, layer, j)))


# ----------------------------------------------------------------------------- decisions
def eviction_excused(kept_after: np.ndarray, scores_after: np.ndarray, evicted_score: float,
                     gpu_ev: int, oracle_ev: int, t: int, r: int) -> bool:
    """Whether a GPU eviction that differs from the oracle's is a near-minimal
    choice under the oracle's scores (see the module docstring).

    kept_after / scores_after: the oracle's retained positions (ascending) and
    scores after the step; evicted_score: the score of the token the oracle
    evicted; t: the step's position; r: the recent window."""
    if gpu_ev < 0 or oracle_ev < 0 or gpu_ev > t - r:
        return False  # one side evicted nothing, or the GPU evicted a protected token
    i = int(np.searchsorted(kept_after, gpu_ev))
    if i >= len(kept_after) or kept_after[i] != gpu_ev:
        return False  # not a token the oracle held at this step
    s_g = float(scores_after[i])
    return s_g >= evicted_score and s_g > 0 and (s_g - evicted_score) / s_g < NEAR_TIE


def prefill_swap_excused(kept: np.ndarray, colsum: np.ndarray, gpu_kept: np.ndarray, T: int,
                         r: int) -> bool:
    """Whether a GPU prefill selection that differs from the oracle's swaps only
    heavy-hitter candidates lying within the near-tie band of the boundary."""
    if len(gpu_kept) != len(kept) or T <= 0:
        return False
    if len(np.unique(gpu_kept)) != len(gpu_kept) or gpu_kept.min() < 0 or gpu_kept.max() >= T:
        return False
    n_cand = T - r
    heavy = kept[kept < n_cand]
    if len(heavy) == 0:
        return False
    s_k = float(colsum[heavy].min())  # the boundary: smallest kept candidate score
    if s_k <= 0:
        return False
    only_gpu = np.setdiff1d(gpu_kept, kept)
    only_oracle = np.setdiff1d(kept, gpu_kept)
    if np.any(only_gpu >= n_cand) or np.any(only_oracle >= n_cand):
        return False  # a recent token was dropped or a non-candidate swapped in
    ok_in = all((s_k - colsum[p]) / s_k < NEAR_TIE for p in only_gpu.tolist())
    ok_out = all(colsum[p] > 0 and (colsum[p] - s_k) / colsum[p] < NEAR_TIE
                 for p in only_oracle.tolist())
    return ok_in and ok_out


def score_rel_error(ref_pos: np.ndarray, ref_scores: np.ndarray, gpu_pos_row: np.ndarray,
                    gpu_score_row: np.ndarray) -> float:
    """Largest relative error of the GPU's scores of the oracle's retained
    positions (the sets must already be known to be equal)."""
    if len(ref_pos) == 0:
        return 0.0
    occ = gpu_pos_row >= 0
    order = np.argsort(gpu_pos_row[occ], kind="stable")
    gp = gpu_pos_row[occ][order]
    gs = gpu_score_row[occ][order].astype(np.float64)
    idx = np.searchsorted(gp, ref_pos)
    got = gs[idx]
    return float(np.max(np.abs(got - ref_scores) / np.maximum(ref_scores, 1e-30)))


def kept_of(gpu_pos_row: np.ndarray) -> np.ndarray:
    return np.sort(gpu_pos_row[gpu_pos_row >= 0])


# ----------------------------------------------------------------------------- whole rows
def new_stats() -> dict:
    return {"prefill_max": 0.0, "prefill_sum": 0.0, "prefill_cnt": 0, "dec_max": 0.0,
            "dec_sum": 0.0, "dec_cnt": 0, "evict_checks": 0, "near_ties": 0, "excused": 0,
            "mismatches": [], "set_checks": 0, "score_checks": 0, "score_max_rel": 0.0,
            "diverged_at": -1, "prefill_checks": 0}


def compare_row(tr: dict, gpu: dict, T: int, r: int, snap_steps: list) -> dict:
    """Compares one row's GPU results, taken without any resynchronisation, with
    the oracle's trace ``tr`` (trace_dict).

    gpu: {"O": [T, d] prefill output or None, "pre_pos" / "pre_score": [k] slots
    after prefill, "ev": [S] evicted positions, "outs": [S, d] outputs,
    "snap_pos" / "snap_score": [len(snap_steps), k] slots after the listed
    steps}. A near-tie decision that differs (and is excused) ends the
    comparison of the row: the two caches then hold different tokens, so the
    step is recorded in "diverged_at"."""
    st = new_stats()
    if gpu.get("O") is not None and T > 0:
        e = np.abs(gpu["O"][:T].astype(np.float64) - tr["O"].astype(np.float64))
        st["prefill_max"] = float(e.max())
        st["prefill_sum"] = float(e.sum())
        st["prefill_cnt"] = int(e.size)
    st["prefill_checks"] = 1
    st["set_checks"] += 1
    near = tr["margin"] < NEAR_TIE
    st["near_ties"] += int(near)
    gk = kept_of(gpu["pre_pos"])
    if not np.array_equal(gk, tr["kept"]):
        if near and prefill_swap_excused(tr["kept"], tr["colsum"], gk, T, r):
            st["excused"] += 1
            st["diverged_at"] = 0
            return st
        st["mismatches"].append(("prefill set", gk.tolist()[:16], tr["kept"].tolist()[:16],
                                 float(tr["margin"])))
        return st
    st["score_checks"] += 1
    st["score_max_rel"] = score_rel_error(tr["kept"], tr["kept_scores"], gpu["pre_pos"],
                                          gpu["pre_score"])
    S = len(tr["evicted"])
    ev = np.asarray(gpu["ev"], dtype=np.int64)[:S]
    diff = np.nonzero(ev != tr["evicted"])[0]
    end = S if len(diff) == 0 else int(diff[0]) + 1  # steps whose outputs are comparable
    if end:
        e = np.abs(gpu["outs"][:end].astype(np.float64) - tr["outs"][:end])
        st["dec_max"] = float(e.max())
        st["dec_sum"] = float(e.sum())
        st["dec_cnt"] = int(e.size)
    st["evict_checks"] = end
    st["near_ties"] += int(np.sum(tr["margins"][:end] < NEAR_TIE))
    if len(diff):
        s = int(diff[0])
        if tr["margins"][s] < NEAR_TIE and eviction_excused(
                tr["kept_after"][s], tr["scores_after"][s], tr["evicted_scores"][s], int(ev[s]),
                int(tr["evicted"][s]), T + s, r):
            st["excused"] += 1
            st["diverged_at"] = s + 1
        else:
            st["mismatches"].append(("evicted", s, int(ev[s]), int(tr["evicted"][s]),
                                     float(tr["margins"][s])))
    for i, s in enumerate(snap_steps):
        if s >= end - (1 if len(diff) else 0):
            break  # from the first differing step on, the caches differ
        st["set_checks"] += 1
        gk = kept_of(gpu["snap_pos"][i])
        if not np.array_equal(gk, tr["kept_after"][s]):
            st["mismatches"].append(("set", s, gk.tolist()[:16], tr["kept_after"][s].tolist()[:16]))
            break
        st["score_checks"] += 1
        st["score_max_rel"] = max(st["score_max_rel"], score_rel_error(
            tr["kept_after"][s], tr["scores_after"][s], gpu["snap_pos"][i], gpu["snap_score"][i]))
    return st


def oracle_compare_row(job) -> dict:
    """Pool worker: oracle trace of one row, compared with the GPU's results.

    job = (oracle_row job, gpu dict, prompt length, r, snapshot steps)."""
    ojob, gpu, T, r, snaps = job
    st = compare_row(oracle_row(ojob), gpu, T, r, snaps)
    st["row"] = (ojob[2], ojob[3])
    return st


def merge_stats(acc: dict, st: dict) -> dict:
    """Adds one row's statistics into an accumulator (new_stats())."""
    for key in ("prefill_sum", "prefill_cnt", "dec_sum", "dec_cnt", "evict_checks", "near_ties",
                "excused", "set_checks", "score_checks", "prefill_checks"):
        acc[key] += st[key]
    for key in ("prefill_max", "dec_max", "score_max_rel"):
        acc[key] = max(acc[key], st[key])
    acc["mismatches"].extend([(st.get("row"),) + tuple(m) for m in st["mismatches"]])
    if st["diverged_at"] >= 0:
        acc.setdefault("diverged", []).append((st.get("row"), st["diverged_at"]))
    return acc
