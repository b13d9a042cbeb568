"""GPU parity of the FP8 (E4M3) KV cache (h2o_create_ex, H2O_KV_FP8) against
the oracle's FP8 mode, through the C ABI.

Same bar as the bf16 cache: retained sets and evictions equal outside
near-ties (margin < 1e-4, counted and resynchronised), outputs within 2e-2
max-abs and 2e-3 mean-abs of the fp64 oracle. In addition the codes and
scales stored on the GPU must equal the oracle's quantisation of the same
tokens bit for bit, after prefill and after the decode steps.
"""
import numpy as np
import pytest
import torch

from h2o_parity import run_parity
from test_gpu_parity import _assert_ok
from workloads import WORKLOADS, Workload

pytestmark = pytest.mark.gpu


def _assert_fp8(rep, label):
    _assert_ok(rep, label)
    print(f"[{label}] fp8 code checks={rep.code_checks} mismatches={len(rep.code_mismatches)}")
    assert rep.code_checks > 0
    assert not rep.code_mismatches, rep.code_mismatches[:5]


def test_fp8_tiny_every_row():
    _assert_fp8(run_parity(WORKLOADS["tiny"], kv="fp8"), "fp8-tiny")


FP8_EDGE = [
    # (name, batch, heads, d, T, S, h, r)
    ("fp8-ragged-d128", 2, 3, 128, 300, 40, 40, 24),
    ("fp8-ragged-d64", 2, 2, 64, 259, 33, 17, 9),
    ("fp8-heavy-only-r0", 1, 2, 128, 200, 30, 24, 0),
    ("fp8-single-token-prompt", 1, 2, 128, 1, 20, 4, 4),
    ("fp8-large-budget-split", 1, 2, 128, 1500, 20, 300, 300),
]


@pytest.mark.parametrize("name,B,H,d,T,S,h,r", FP8_EDGE, ids=[e[0] for e in FP8_EDGE])
def test_fp8_edge_shapes(name, B, H, d, T, S, h, r):
    w = Workload(300 + FP8_EDGE.index((name, B, H, d, T, S, h, r)), name, 1, B, H, d, T, S, h, r, 0.8)
    _assert_fp8(run_parity(w, kv="fp8"), name)


def test_fp8_opt_6_7b_layer_sampled_rows():
    """Full-size OPT-6.7B-shaped layer (256 rows, launch shape of the bench);
    32 seeded rows checked, repeated over the batch."""
    w = WORKLOADS["opt-6.7b-layer"]
    rows = [(b, j) for b in range(w.batch) for j in range(0, w.heads, 8)]
    _assert_fp8(run_parity(w, rows=rows, tile=True, set_check_every=32, kv="fp8"), "fp8-opt-6.7b")


def test_fp8_zero_token_has_zero_scale_and_codes():
    """A token whose key (or value) vector is all zeros is stored with scale 0
    and zero codes (the quantiser's definition), and attending to it is
    well defined."""
    import h2o_heavy_hitter_gb300 as h2o
    dev = torch.device("cuda")
    g = torch.Generator(device="cuda").manual_seed(1)
    B, H, T, d = 1, 2, 6, 128
    Q, K, V = [torch.randn(B, H, T, d, device=dev, generator=g).to(torch.bfloat16) for _ in range(3)]
    K[:, :, 2] = 0
    V[:, :, 4] = 0
    ctx = h2o.h2o_create(1, B, H, d, 4, 4, kv="fp8")
    try:
        h2o.h2o_prefill(ctx, 0, Q, K, V)
        view, sc = h2o.h2o_cache_view(ctx, 0), h2o.h2o_cache_scales(ctx, 0)
        pos = view["pos"].cpu().numpy()
        for row in range(B * H):
            s2 = int(np.nonzero(pos[row] == 2)[0][0])
            s4 = int(np.nonzero(pos[row] == 4)[0][0])
            assert sc["K"][row, s2].item() == 0.0 and int(view["K"][row, s2].abs().sum()) == 0
            assert sc["V"][row, s4].item() == 0.0 and int(view["V"][row, s4].abs().sum()) == 0
            assert sc["K"][row, s4].item() > 0.0
        out = torch.empty(B, H, d, device=dev)
        z = torch.zeros(B, H, d, device=dev, dtype=torch.bfloat16)
        h2o.h2o_decode_step(ctx, 0, Q[:, :, 0].contiguous(), z, z, out)
        h2o.h2o_sync_check(ctx)
        assert torch.isfinite(out).all()
    finally:
        ctx.close()


def test_fp8_scales_refused_for_bf16_cache():
    import h2o_heavy_hitter_gb300 as h2o
    ctx = h2o.h2o_create(1, 1, 1, 64, 2, 2)
    try:
        with pytest.raises(h2o.H2OError):
            h2o.h2o_cache_scales(ctx, 0)
    finally:
        ctx.close()
