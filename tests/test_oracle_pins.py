"""Pins of the CPU oracle to things other than itself (CPU only).

(a) with h + r >= T + S nothing is evicted and every output equals dense causal
    attention, computed by torch's scaled_dot_product_attention in float64;
    with V = identity the same routine returns the probability matrix itself,
    which pins the column-sum scores;
(b) with h = 0 decode equals sliding-window attention over keys [t - r, t];
(c) invariants: each step's probabilities sum to 1, scores are non-negative,
    the total accumulated mass over every token ever seen equals the number of
    query rows processed (a closed form), the set size, the protected recent
    window and the candidate count;
(d) brute force on tiny inputs: prefill keeps the max-sum subset (ties to later
    positions) and every decode eviction is the exhaustive minimum;
(e) the budget-3 illustration of the H2O summary page (section 4.1);
(f) the 180 GB sizing example of the H2O summary page (section 1);
(g) the near-tie margin that decides which eviction decisions are excused
    from bit-exact comparison: exact values on hand-built decode and prefill
    cases where a token outside the candidate set would change the answer, and
    a recomputation by plain loops over the candidates on tiny random inputs.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle as _real_oracle
from workloads import (WORKLOADS, Workload, bf16_bits_to_f64, f32_to_bf16_bits, kv_cache_bytes,
                       row_tokens)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _row(w: Workload, b=0, j=0, layer=0):
    q, k, v = row_tokens(w, layer, b, j)
    return bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)


def _sdpa(q, k, v, mask=None, causal=False, scale=None):
    tq = torch.from_numpy(q)[None, None]
    tk = torch.from_numpy(k)[None, None]
    tv = torch.from_numpy(v)[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, is_causal=causal,
                                                         scale=scale)
    return o[0, 0].numpy()


SMALL = Workload(101, "small", 1, 1, 2, 32, 40, 24, 6, 5, 0.8)


# ----------------------------------------------------------------------------- (a)
def check_a_no_eviction_equals_dense_causal_attention(oracle, d, T, S):
    w = SMALL.with_(head_dim=d, prompt=T, steps=S, h=T + S, r=0)
    q, k, v = _row(w)
    for h, r in [(T + S, 0), (0, T + S), (T, S), (T + S - 3, 3)]:
        tr = oracle.run_row(q, k, v, T, S, h, r)
        dense = _sdpa(q, k, v, causal=True)  # default scale 1/sqrt(d)
        np.testing.assert_allclose(tr.prefill.O, dense[:T], rtol=0, atol=1e-12)
        np.testing.assert_allclose(np.array(tr.outs), dense[T:], rtol=0, atol=1e-12)
        assert all(e == -1 for e in tr.evicted)


def check_a_colsum_scores_equal_probability_matrix_column_sums(oracle):
    """V = identity makes SDPA return the causal probability matrix P itself."""
    w = SMALL.with_(prompt=48, steps=16)
    q, k, v = _row(w)
    N = w.prompt + w.steps
    eye = np.eye(N)
    P = _sdpa(q, k, eye, causal=True)
    # prefill: column sums over the prompt rows only
    O, colsum, _ = oracle.prefill_attention(q[:w.prompt], k[:w.prompt], eye[:w.prompt, :w.prompt],
                                            oracle.default_scale(w.head_dim))
    np.testing.assert_allclose(O, P[:w.prompt, :w.prompt], atol=1e-12)
    np.testing.assert_allclose(colsum, P[:w.prompt, :w.prompt].sum(axis=0), atol=1e-12)
    # decode without eviction: final accumulated score of token j = sum_i P_ij over all N rows
    tr = oracle.run_row(q, k, v, w.prompt, w.steps, N, 0)
    c = tr.prefill.cache
    np.testing.assert_array_equal(c.pos, np.arange(N))
    np.testing.assert_allclose(c.score, P.sum(axis=0), atol=1e-12)


def check_a_scale_parameter_is_used(oracle):
    w = SMALL
    q, k, v = _row(w)
    tr = oracle.run_row(q, k, v, w.prompt, w.steps, 100, 100, scale=1.0)
    dense = _sdpa(q, k, v, causal=True, scale=1.0)
    np.testing.assert_allclose(np.array(tr.outs), dense[w.prompt:], atol=1e-12)


# ----------------------------------------------------------------------------- (b)
def check_b_heavy_budget_zero_is_sliding_window(oracle, r):
    w = SMALL.with_(prompt=30, steps=20)
    q, k, v = _row(w)
    T, S = w.prompt, w.steps
    tr = oracle.run_row(q, k, v, T, S, 0, r)
    dense = _sdpa(q[:T], k[:T], v[:T], causal=True)
    np.testing.assert_allclose(tr.prefill.O, dense, atol=1e-12)
    np.testing.assert_array_equal(tr.prefill.kept, np.arange(T - r, T))
    N = T + S
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    band = (j <= i) & (j >= i - r)  # query t sees keys t-r .. t (r + 1 keys)
    win = _sdpa(q, k, v, mask=band)
    np.testing.assert_allclose(np.array(tr.outs), win[T:], atol=1e-12)
    for s in range(S):
        t = T + s
        assert tr.evicted[s] == t - r
        np.testing.assert_array_equal(tr.kept_after[s], np.arange(t - r + 1, t + 1))


# ----------------------------------------------------------------------------- (c)
def check_c_invariants(oracle, h, r):
    w = SMALL.with_(prompt=33, steps=40)
    q, k, v = _row(w, j=1)
    T, S = w.prompt, w.steps
    kk = h + r
    pre = oracle.prefill(q[:T], k[:T], v[:T], h, r)
    c = pre.cache
    # every prompt query row distributes mass 1
    np.testing.assert_allclose(pre.colsum.sum(), T, atol=1e-9)
    assert (pre.colsum > 0).all()
    left = float(np.delete(pre.colsum, pre.kept).sum())  # mass held by tokens no longer cached
    ledger = {int(j): float(pre.colsum[j]) for j in range(T)}  # per-token sum of logged p
    assert len(c.pos) == min(kk, T)
    for s in range(S):
        t = T + s
        n_before = len(c.pos)
        lg = oracle.decode_step(c, q[t], k[t], v[t])
        assert abs(lg.p.sum() - 1.0) < 1e-12
        assert (lg.p >= 0).all() and (c.score >= 0).all()
        np.testing.assert_array_equal(lg.pos_attended[-1], t)
        for pos_, p_ in zip(lg.pos_attended.tolist(), lg.p.tolist()):
            ledger[pos_] = ledger.get(pos_, 0.0) + p_
        if lg.evicted >= 0:
            left += lg.evicted_score
            assert abs(lg.evicted_score - ledger[lg.evicted]) < 1e-12
        # closed form: all mass ever handed out = number of query rows so far
        np.testing.assert_allclose(c.score.sum() + left, T + s + 1, atol=1e-9)
        # each retained score equals the sum of the probabilities logged for it
        for pos_, sc in zip(c.pos.tolist(), c.score.tolist()):
            assert abs(sc - ledger[pos_]) < 1e-12
        assert len(c.pos) == min(kk, T + s + 1)
        assert len(set(c.pos.tolist())) == len(c.pos)
        if lg.evicted != t:  # the r most recent (t included) are never evicted
            assert set(range(max(0, t - r + 1), t + 1)) <= set(c.pos.tolist())
        if n_before + 1 > kk:
            assert lg.evicted >= 0 and lg.n_candidates == h + 1
        else:
            assert lg.evicted == -1


# ----------------------------------------------------------------------------- (d)
def _best_subset_brute(score, cand, h):
    """Max-sum h-subset of ``cand``; among equal sums the one with the largest
    position sum (that is, later positions kept on ties)."""
    best, best_key = None, None
    for sub in itertools.combinations(cand, h):
        key = (round(sum(score[j] for j in sub), 12), sum(sub))
        if best_key is None or key > best_key:
            best, best_key = sub, key
    return sorted(best)


def check_d_prefill_keeps_max_sum_subset(oracle, T, h, r):
    for seed in range(4):
        w = SMALL.with_(head_dim=8, prompt=T, steps=0)
        q, k, v = _row(w, b=seed)
        pre = oracle.prefill(q, k, v, h, r)
        cand = list(range(T - r))
        heavy = _best_subset_brute(pre.colsum, cand, h)
        np.testing.assert_array_equal(pre.kept, sorted(heavy + list(range(T - r, T))))


def check_d_prefill_tie_rule_keeps_later_positions(oracle):
    colsum = np.array([1.0, 0.5, 0.5, 0.5, 2.0, 0.5, 0.3, 0.9])
    for h in range(0, 6):
        kept, margin = oracle.prefill_select(colsum, h, 2)
        heavy = _best_subset_brute(colsum, list(range(6)), h)
        np.testing.assert_array_equal(kept, sorted(heavy + [6, 7]))
    kept, margin = oracle.prefill_select(colsum, 3, 2)  # boundary inside the 0.5 group
    np.testing.assert_array_equal(kept, [0, 4, 5, 6, 7])
    assert margin == 0.0


def check_d_decode_eviction_is_exhaustive_minimum_and_greedy(oracle, h, r):
    w = SMALL.with_(head_dim=8, prompt=10, steps=12)
    q, k, v = _row(w, b=2)
    T, S = w.prompt, w.steps
    c = oracle.prefill(q[:T], k[:T], v[:T], h, r).cache
    for s in range(S):
        t = T + s
        pos_before = c.pos.tolist() + [t]
        lg = oracle.decode_step(c, q[t], k[t], v[t])
        # scores after accumulation, before eviction, from the logged state
        after = dict(zip(c.pos.tolist(), c.score.tolist()))
        if lg.evicted >= 0:
            after[lg.evicted] = lg.evicted_score
        if len(pos_before) <= h + r:
            assert lg.evicted == -1
            continue
        # exhaustive scan in a plain loop: smallest score, then smallest position
        best = None
        for pj in pos_before:
            if pj <= t - r and (best is None or (after[pj], pj) < (after[best], best)):
                best = pj
        assert lg.evicted == best
        # greedy: the kept set maximises the kept score sum over every k-subset
        # of the attended set that holds the r most recent tokens
        must = set(range(t - r + 1, t + 1))
        best_sum = max(sum(after[x] for x in sub)
                       for sub in itertools.combinations(pos_before, h + r) if must <= set(sub))
        assert abs(sum(after[x] for x in c.pos.tolist()) - best_sum) < 1e-12


def check_d_decode_tie_goes_to_smallest_position(oracle):
    d = 4
    K = np.zeros((5, d))
    V = np.eye(5, d)
    c = oracle.RowCache(h=3, r=1, scale=1.0, pos=np.array([0, 1, 2, 3]), K=K[:4].copy(),
                        V=V[:4].copy(), score=np.array([0.7, 0.2, 0.2, 0.1]), t=4)
    lg = oracle.decode_step(c, np.zeros(d), K[4], V[4])  # uniform p = 0.2 each
    # candidates: positions <= 3 -> scores 0.9, 0.4, 0.4, 0.3: position 3 has the minimum
    assert lg.evicted == 3
    c = oracle.RowCache(h=3, r=1, scale=1.0, pos=np.array([0, 1, 2, 3]), K=K[:4].copy(),
                        V=V[:4].copy(), score=np.array([0.7, 0.2, 0.2, 0.3]), t=4)
    lg = oracle.decode_step(c, np.zeros(d), K[4], V[4])
    assert lg.evicted == 1 and lg.margin == 0.0  # exact tie between 1 and 2


def check_d_r_zero_can_drop_the_new_token(oracle):
    d = 2
    c = oracle.RowCache(h=2, r=0, scale=1.0, pos=np.array([0, 1]), K=np.array([[1.0, 0], [1.0, 0]]),
                        V=np.eye(2), score=np.array([5.0, 5.0]), t=2)
    lg = oracle.decode_step(c, np.array([3.0, 0.0]), np.array([-1.0, 0.0]), np.array([0.0, 0.0]))
    assert lg.evicted == 2
    np.testing.assert_array_equal(c.pos, [0, 1])


# ----------------------------------------------------------------------------- (e)
def check_e_budget_three_illustration(oracle):
    g = json.load(open(os.path.join(GOLDEN, "budget3_example.json")))
    q, k, v = (np.array(g[x], dtype=np.float64) for x in ("q", "k", "v"))
    T = g["prompt"]
    for case in g["cases"]:
        tr = oracle.run_row(q, k, v, T, 1, case["h"], case["r"], scale=g["scale"])
        assert tr.evicted[0] == case["expected_evicted_at_fourth_step"]


# ----------------------------------------------------------------------------- (f)
def check_f_kv_cache_sizing_example(oracle):
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_sizing.json")))
    m = g["model_dims"]
    b = kv_cache_bytes(m["layers"], m["hidden"], g["batch"], g["seq"], g["bytes_per_elem"])
    assert round(b / 1e9) == g["expected_gb"]


# ----------------------------------------------------------------------------- (g)
# The margin of an eviction is (s2 - s1) / s2 between the evicted key s1 and the
# runner-up s2 among the candidates (positions <= t - r); at prefill it is
# (s_keep - s_drop) / s_keep between the smallest kept and the largest dropped
# heavy-hitter candidate. Steps whose margin is below the near-tie threshold are
# the only ones whose decisions may differ from the GPU's, so the margin must be
# right: too small and real mismatches are excused, too large and none are.
def check_g_decode_margin_hand_built(oracle):
    d = 4
    K = np.zeros((5, d))
    V = np.eye(5, d)
    # zero query: every one of the 5 attended tokens gets p = 0.2
    c = oracle.RowCache(h=3, r=1, scale=1.0, pos=np.array([0, 1, 2, 3]), K=K[:4].copy(),
                        V=V[:4].copy(), score=np.array([0.7, 0.2, 0.25, 0.1]), t=4)
    lg = oracle.decode_step(c, np.zeros(d), K[4], V[4])
    # candidates (positions <= 3) after accumulation: 0.9, 0.4, 0.45, 0.3; the new
    # token (position 4, score 0.2, the smallest of all) is not a candidate
    assert lg.evicted == 3 and lg.n_candidates == 4
    assert abs(lg.evicted_score - 0.3) < 1e-15
    assert abs(lg.margin - (0.4 - 0.3) / 0.4) < 1e-12
    # with r = 2 position 3 is protected as well: candidates 0.9, 0.4, 0.45
    c = oracle.RowCache(h=2, r=2, scale=1.0, pos=np.array([0, 1, 2, 3]), K=K[:4].copy(),
                        V=V[:4].copy(), score=np.array([0.7, 0.2, 0.25, 0.1]), t=4)
    lg = oracle.decode_step(c, np.zeros(d), K[4], V[4])
    assert lg.evicted == 1 and lg.n_candidates == 3
    assert abs(lg.margin - (0.45 - 0.4) / 0.45) < 1e-12
    # a single candidate has no runner-up: no near-tie is possible
    c = oracle.RowCache(h=0, r=1, scale=1.0, pos=np.array([3]), K=K[:1].copy(), V=V[:1].copy(),
                        score=np.array([0.5]), t=4)
    lg = oracle.decode_step(c, np.zeros(d), K[4], V[4])
    assert lg.evicted == 3 and lg.margin == np.inf


def check_g_prefill_margin_hand_built(oracle):
    # T = 8, r = 2: candidates 0..5 with scores 1.0 0.5 0.8 0.6 2.0 0.9; the two
    # recent tokens (0.3, 0.4) have the smallest scores but never compete
    colsum = np.array([1.0, 0.5, 0.8, 0.6, 2.0, 0.9, 0.3, 0.4])
    kept, margin = oracle.prefill_select(colsum, 2, 2)
    np.testing.assert_array_equal(kept, [0, 4, 6, 7])
    assert abs(margin - (1.0 - 0.9) / 1.0) < 1e-12
    kept, margin = oracle.prefill_select(colsum, 3, 2)
    np.testing.assert_array_equal(kept, [0, 4, 5, 6, 7])
    assert abs(margin - (0.9 - 0.8) / 0.9) < 1e-12
    kept, margin = oracle.prefill_select(colsum, 0, 2)  # nothing kept among candidates
    assert margin == np.inf
    kept, margin = oracle.prefill_select(colsum, 6, 2)  # T <= h + r: nothing dropped
    assert margin == np.inf and len(kept) == 8


def _margin_by_loops(keys):
    """(s2 - s1) / s2 of the two smallest (score, position) keys, plain loops."""
    first = second = None
    for key in keys:
        if first is None or key < first:
            first, second = key, first
        elif second is None or key < second:
            second = key
    if second is None:
        return np.inf
    return (second[0] - first[0]) / second[0] if second[0] > 0 else 0.0


def check_g_margins_equal_recomputation_over_candidates(oracle, h, r):
    w = SMALL.with_(head_dim=8, prompt=12, steps=16)
    for seed in range(3):
        q, k, v = _row(w, b=seed)
        T, S = w.prompt, w.steps
        pre = oracle.prefill(q[:T], k[:T], v[:T], h, r)
        if T > h + r and h > 0:
            cand = range(T - r)
            kept_heavy = [j for j in cand if j in set(pre.kept.tolist())]
            dropped = [j for j in cand if j not in set(pre.kept.tolist())]
            s_keep = min(pre.colsum[j] for j in kept_heavy)
            s_drop = max(pre.colsum[j] for j in dropped)
            assert abs(pre.margin - (s_keep - s_drop) / s_keep) < 1e-12
        c = pre.cache
        for s in range(S):
            t = T + s
            lg = oracle.decode_step(c, q[t], k[t], v[t])
            if lg.evicted < 0:
                continue
            after = dict(zip(c.pos.tolist(), c.score.tolist()))
            after[lg.evicted] = lg.evicted_score
            keys = [(after[p], p) for p in lg.pos_attended.tolist() if p <= t - r]
            assert len(keys) == lg.n_candidates
            m = _margin_by_loops(keys)
            assert (m == np.inf and lg.margin == np.inf) or abs(lg.margin - m) < 1e-12


# ----------------------------------------------------------------------------- inputs
def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 7,
                        np.array([1.00390625, 1.01171875, -2.00781250, 0.0, -0.0], np.float32)])
    ours = f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(bf16_bits_to_f64(ours),
                                  torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_generator_is_row_addressable_and_deterministic():
    w = WORKLOADS["tiny"]
    a = row_tokens(w, 0, 0, 3)
    b = row_tokens(w, 0, 0, 3)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    c = row_tokens(w, 0, 0, 2)
    assert not np.array_equal(a[1], c[1])


# ----------------------------------------------------------------------------- wrappers
# Each pin is a check_* function of the oracle module, so that the mutation
# tests can run the same pins against copies of the oracle with planted mistakes.


@pytest.mark.parametrize("d,T,S", [(32, 40, 24), (64, 57, 9), (16, 1, 12)])
def test_a_no_eviction_equals_dense_causal_attention(d, T, S):
    check_a_no_eviction_equals_dense_causal_attention(_real_oracle, d, T, S)


def test_a_colsum_scores_equal_probability_matrix_column_sums():
    check_a_colsum_scores_equal_probability_matrix_column_sums(_real_oracle)


def test_a_scale_parameter_is_used():
    check_a_scale_parameter_is_used(_real_oracle)


@pytest.mark.parametrize("r", [1, 3, 8])
def test_b_heavy_budget_zero_is_sliding_window(r):
    check_b_heavy_budget_zero_is_sliding_window(_real_oracle, r)


@pytest.mark.parametrize("h,r", [(6, 5), (10, 1), (1, 10), (4, 0), (0, 4), (12, 12), (1, 0), (0, 1)])
def test_c_invariants(h, r):
    check_c_invariants(_real_oracle, h, r)


@pytest.mark.parametrize("T,h,r", [(10, 3, 3), (9, 2, 1), (8, 3, 0), (10, 1, 3), (7, 0, 2)])
def test_d_prefill_keeps_max_sum_subset(T, h, r):
    check_d_prefill_keeps_max_sum_subset(_real_oracle, T, h, r)


def test_d_prefill_tie_rule_keeps_later_positions():
    check_d_prefill_tie_rule_keeps_later_positions(_real_oracle)


@pytest.mark.parametrize("h,r", [(3, 3), (2, 1), (3, 0), (0, 2), (1, 1)])
def test_d_decode_eviction_is_exhaustive_minimum_and_greedy(h, r):
    check_d_decode_eviction_is_exhaustive_minimum_and_greedy(_real_oracle, h, r)


def test_d_decode_tie_goes_to_smallest_position():
    check_d_decode_tie_goes_to_smallest_position(_real_oracle)


def test_d_r_zero_can_drop_the_new_token():
    check_d_r_zero_can_drop_the_new_token(_real_oracle)


def test_e_budget_three_illustration():
    check_e_budget_three_illustration(_real_oracle)


def test_f_kv_cache_sizing_example():
    check_f_kv_cache_sizing_example(_real_oracle)


def test_g_decode_margin_hand_built():
    check_g_decode_margin_hand_built(_real_oracle)


def test_g_prefill_margin_hand_built():
    check_g_prefill_margin_hand_built(_real_oracle)


@pytest.mark.parametrize("h,r", [(3, 3), (4, 1), (2, 0), (1, 2)])
def test_g_margins_equal_recomputation_over_candidates(h, r):
    check_g_margins_equal_recomputation_over_candidates(_real_oracle, h, r)
