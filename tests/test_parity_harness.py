"""The GPU-versus-oracle comparison has teeth (CPU only).

The rows of a planted-mistake oracle stand in for GPU results and go through
the same comparison the GPU parity tests use (parity_rows.compare_row and the
excusal rules). Each mistake must be reported, including when the reference's
near-tie margin is itself broken (forced to 0, so that every step would count
as a near-tie): the excusal of a differing decision rests on the oracle's
scores, not on its margin. The mistakes are planted in copies of the oracle,
on the CPU; the real oracle is untouched.
"""
import numpy as np
import pytest

import oracle
import parity_rows as pr
from test_oracle_mutations import MUTANTS, _load_mutant
from workloads import Workload, bf16_bits_to_f64, row_tokens

W = Workload(120, "harness", 1, 1, 2, 16, 24, 40, 5, 4, 0.8)
SNAPS = [9, 19, 29, 39]


def _inputs(j=0):
    q, k, v = row_tokens(W, 0, 0, j)
    return bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)


def _trace(mod, j=0):
    q, k, v = _inputs(j)
    return pr.trace_dict(mod.run_row(q, k, v, W.prompt, W.steps, W.h, W.r))


def _slots(pos, scores, k, rng):
    """A cache row as the GPU holds it: the retained tokens in shuffled slots,
    empty slots -1 / 0."""
    p = np.full(k, -1, dtype=np.int32)
    sc = np.zeros(k, dtype=np.float32)
    where = rng.permutation(k)[:len(pos)]
    p[where] = pos
    sc[where] = scores
    return p, sc


def _as_gpu(tr, seed=0):
    rng = np.random.default_rng(seed)
    k = W.k
    pre_pos, pre_score = _slots(tr["kept"], tr["kept_scores"], k, rng)
    snaps = [_slots(tr["kept_after"][s], tr["scores_after"][s], k, rng) for s in SNAPS]
    return {"O": tr["O"], "outs": tr["outs"].astype(np.float32), "ev": tr["evicted"],
            "pre_pos": pre_pos, "pre_score": pre_score,
            "snap_pos": np.stack([p for p, _ in snaps]), "snap_score": np.stack([x for _, x in snaps])}


def _bad(st):
    return (bool(st["mismatches"]) or st["score_max_rel"] > pr.SCORE_RTOL
            or st["prefill_max"] > pr.MAX_ABS or st["dec_max"] > pr.MAX_ABS)


@pytest.mark.parametrize("j", [0, 1])
def test_identical_results_pass(j):
    tr = _trace(oracle, j)
    st = pr.compare_row(tr, _as_gpu(tr), W.prompt, W.r, SNAPS)
    assert not _bad(st) and st["evict_checks"] == W.steps and st["score_checks"] == 1 + len(SNAPS)
    assert st["diverged_at"] == -1 and st["score_max_rel"] < 1e-6  # fp32 storage of the scores


SCORE_MISTAKES = {
    "accumulated scores not normalised": ("score = np.append(c.score + p[:-1], p[-1])",
                                          "score = np.append(c.score + e[:-1], e[-1])"),
    "a step's probability added twice": ("score = np.append(c.score + p[:-1], p[-1])",
                                         "score = np.append(c.score + 2 * p[:-1], p[-1])"),
    "prefill scores dropped": ("colsum[kept].copy(), K.shape[0])", "0 * colsum[kept], K.shape[0])"),
}


@pytest.mark.parametrize("name", sorted(SCORE_MISTAKES))
def test_score_mistakes_are_reported(name):
    mod = _load_mutant(name, *SCORE_MISTAKES[name])
    st = pr.compare_row(_trace(oracle), _as_gpu(_trace(mod)), W.prompt, W.r, SNAPS)
    assert _bad(st), name


@pytest.mark.parametrize("name", ["decode evicts the maximum", "candidate mask off by one",
                                  "new token left out of attention",
                                  "prefill keeps the lowest scores", "recent window shifted"])
def test_decision_mistakes_are_reported_even_with_a_broken_margin(name):
    gpu = _as_gpu(_trace(_load_mutant(name, *MUTANTS[name])))
    for ref in (oracle, _load_mutant("decode margin forced to zero",
                                     *MUTANTS["decode margin forced to zero"]),
                _load_mutant("prefill margin forced to zero",
                             *MUTANTS["prefill margin forced to zero"])):
        st = pr.compare_row(_trace(ref), gpu, W.prompt, W.r, SNAPS)
        assert _bad(st), (name, ref.__name__)


def test_eviction_excusal_needs_a_near_minimal_candidate():
    kept = np.array([0, 2, 5, 7, 8])
    scores = np.array([0.9, 0.30001, 0.5, 0.2, 0.1])  # after the step; the oracle evicted 0.3
    t, r = 8, 2
    assert pr.eviction_excused(kept, scores, 0.3, 2, 3, t, r)  # within 1e-4 of the minimum
    assert not pr.eviction_excused(kept, scores, 0.3, 5, 3, t, r)  # 0.5: far from it
    assert not pr.eviction_excused(kept, scores, 0.3, 7, 3, t, r)  # protected (> t - r)
    assert not pr.eviction_excused(kept, scores, 0.3, 4, 3, t, r)  # not held by the oracle
    assert not pr.eviction_excused(kept, scores, 0.3, -1, 3, t, r)  # GPU evicted nothing
    assert not pr.eviction_excused(kept, np.array([0.9, 0.29, 0.5, 0.2, 0.1]), 0.3, 2, 3, t, r)


def test_prefill_excusal_needs_swaps_within_the_band():
    # T = 8, r = 2, h = 3: the oracle keeps candidates 0 (1.0), 4 (2.0) and
    # 5 (0.9, the boundary) plus the recent tokens 6 and 7; candidate 2 sits
    # within 1e-4 below the boundary, candidate 3 far below it
    kept = np.array([0, 4, 5, 6, 7])
    colsum = np.array([1.0, 0.5, 0.89995, 0.8, 2.0, 0.9, 0.3, 0.4])
    assert pr.prefill_swap_excused(kept, colsum, np.array([0, 2, 4, 6, 7]), 8, 2)
    assert not pr.prefill_swap_excused(kept, colsum, np.array([0, 3, 4, 6, 7]), 8, 2)  # 0.8
    assert not pr.prefill_swap_excused(kept, colsum, np.array([0, 2, 4, 5, 7]), 8, 2)  # recent 6 gone
    assert not pr.prefill_swap_excused(kept, colsum, np.array([0, 2, 4, 5, 6, 7]), 8, 2)  # size
