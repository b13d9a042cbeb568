"""The ring cache layout (H2O_LAYOUT_RING: heavy slots, then the recent window as
a circular queue, as in the pages' implementation) against the oracle.

The layout changes where tokens sit, not what the policy computes: outputs,
evictions and retained sets must match the oracle exactly as the default
slot-indexed layout does (tolerances and near-tie rules of test_gpu_parity).
"""
import numpy as np
import pytest
import torch

from h2o_parity import run_parity
from test_gpu_parity import _assert_ok
from workloads import Workload, head_direction, row_tokens

pytestmark = pytest.mark.gpu

RING = [
    # (name, batch, heads, d, T, S, h, r)
    ("ragged-d128", 2, 3, 128, 300, 40, 40, 24),
    ("ragged-d64", 2, 2, 64, 259, 33, 17, 9),
    ("prompt-shorter-than-budget", 1, 3, 128, 50, 40, 40, 30),   # the window fills, then moves
    ("recent-only-h0", 1, 2, 128, 200, 30, 0, 24),
    ("budget-one-recent", 1, 2, 64, 40, 12, 0, 1),
    ("single-token-prompt", 1, 2, 128, 1, 20, 4, 4),
    ("empty-prompt", 1, 2, 64, 0, 30, 6, 4),
    ("large-budget-split-rows", 1, 2, 128, 1500, 20, 300, 300),  # rows split over CTAs
    ("rows-256", 8, 32, 128, 300, 48, 40, 40),
]


@pytest.mark.parametrize("name,B,H,d,T,S,h,r", RING, ids=[c[0] for c in RING])
def test_ring_layout_matches_oracle(name, B, H, d, T, S, h, r):
    w = Workload(600 + [c[0] for c in RING].index(name), name, 1, B, H, d, T, S, h, r, 0.8)
    _assert_ok(run_parity(w, layout="ring"), name)


def test_ring_layout_multistep_call_matches_oracle():
    """h2o_decode_steps on a ring cache (one launch per step inside the call)."""
    w = Workload(622, "ring-multi", 1, 2, 2, 128, 180, 30, 20, 12, 0.8)
    _assert_ok(run_parity(w, layout="ring", decode="multi"), "ring-multi")


def test_ring_layout_ragged_batch_matches_oracle():
    lens = [300, 0, 7, 130, 257]
    w = Workload(620, "ring-ragged", 1, len(lens), 2, 128, 300, 30, 20, 12, 0.8)
    _assert_ok(run_parity(w, layout="ring", lens=lens), "ring-ragged")


def test_ring_layout_places_the_window_in_its_queue():
    """After prefill and after every decode step, recent position p sits in
    slot h + p mod r and the older kept tokens fill slots 0 .. n - 1."""
    import h2o_heavy_hitter_gb300 as h2o
    B, H, d, T, S, h, r = 1, 4, 64, 150, 25, 12, 10
    w = Workload(621, "ring-places", 1, B, H, d, T, S, h, r, 0.8)
    bits = [row_tokens(w, 0, 0, j, head_direction(w, 0, j)) for j in range(H)]
    full = [torch.from_numpy(np.stack([x[c] for x in bits]).view(np.int16)).cuda()
            .view(torch.bfloat16).reshape(B, H, T + S, d) for c in range(3)]
    ctx = h2o.h2o_create(1, B, H, d, h, r, layout="ring")
    h2o.h2o_prefill(ctx, 0, *(x[:, :, :T].contiguous() for x in full))
    for s in range(S + 1):
        t = T + s  # next position
        pos = h2o.h2o_cache_positions(ctx, 0)
        for row in pos:
            for p in range(t - r, t):
                assert row[h + p % r] == p, (s, row.tolist())
            assert np.all(row[:h] >= 0) and np.all(row[:h] < t - r)
        if s < S:
            h2o.h2o_decode_step(ctx, 0, *(x[:, :, t].contiguous() for x in full))
    ctx.close()


def test_ring_layout_rejects_unsupported_caches():
    import h2o_heavy_hitter_gb300 as h2o
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_create(1, 1, 1, 64, 4, 0, layout="ring")  # no window
    assert e.value.code == h2o.H2O_EINVAL
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_create(1, 1, 1, 64, 4, 4, kv="fp8", layout="ring")
    assert e.value.code == h2o.H2O_EINVAL
