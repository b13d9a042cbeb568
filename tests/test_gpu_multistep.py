"""Several decode steps in one launch (h2o_decode_steps) against the oracle and
against the same steps taken one launch at a time.

Tolerances and near-tie rules as in test_gpu_parity; inside one call nothing
can be resynchronised, so a row whose eviction differs from the oracle's at a
near-tie is counted and no longer compared.
"""
import numpy as np
import pytest
import torch

from h2o_parity import run_parity
from test_gpu_parity import _assert_ok
from workloads import Workload, head_direction, row_tokens

pytestmark = pytest.mark.gpu

MULTI = [
    # (name, batch, heads, d, T, S, h, r)
    ("rows-256-d128", 8, 32, 128, 300, 64, 40, 40),   # 256-thread CTAs, two batches in flight
    ("rows-640-d64", 20, 32, 64, 64, 16, 8, 8),       # many rows: 128-thread CTAs
    ("ragged-d64", 2, 2, 64, 259, 33, 17, 9),
    ("r0-new-token-competes", 1, 2, 128, 200, 30, 24, 0),
    ("h0-recent-only", 1, 2, 128, 200, 30, 0, 24),
    ("empty-prompt", 1, 2, 64, 0, 30, 6, 4),
    ("budget-over-8192-per-step-launches", 1, 1, 64, 8300, 8, 4100, 4100),
    ("few-long-rows-per-step-launches", 1, 2, 64, 1300, 12, 600, 600),  # rows split over CTAs
]


@pytest.mark.parametrize("name,B,H,d,T,S,h,r", MULTI, ids=[m[0] for m in MULTI])
def test_multistep_matches_oracle(name, B, H, d, T, S, h, r):
    w = Workload(400 + [m[0] for m in MULTI].index(name), name, 1, B, H, d, T, S, h, r, 0.8)
    rep = run_parity(w, decode="multi", row_block=1024)
    _assert_ok(rep, name)
    assert rep.evict_checks > 0


def test_multistep_ragged_batch_matches_oracle():
    lens = [180, 3, 77, 129]
    w = Workload(420, "multi-ragged", 1, len(lens), 2, 128, 180, 40, 20, 12, 0.8)
    _assert_ok(run_parity(w, decode="multi", lens=lens), "multi-ragged")


def test_multistep_fp8_cache_matches_oracle():
    w = Workload(421, "multi-fp8", 1, 2, 4, 128, 190, 40, 16, 16, 0.8)
    rep = run_parity(w, decode="multi", kv="fp8")
    _assert_ok(rep, "multi-fp8")
    assert rep.code_checks > 0 and not rep.code_mismatches, rep.code_mismatches[:5]


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_multistep_equals_single_steps_bitwise(kv):
    """256 rows (one CTA per row in both launch shapes): every output, every
    evicted position, and the final cache equal those of one launch per step."""
    import h2o_heavy_hitter_gb300 as h2o
    B, H, d, T, S, h, r = 8, 32, 128, 200, 40, 24, 24
    w = Workload(430, "multi-bitwise", 1, B, H, d, T, S, h, r, 0.8)
    rows = [(b, j) for b in range(B) for j in range(H)]
    bits = [row_tokens(w, 0, b, j, head_direction(w, 0, j)) for b, j in rows]
    full = [_bf16(np.stack([x[c] for x in bits])).reshape(B, H, T + S, d) for c in range(3)]
    pre = [x[:, :, :T].contiguous() for x in full]
    steps = [x[:, :, T:].permute(2, 0, 1, 3).contiguous() for x in full]  # [S, B, H, d]
    one = h2o.h2o_create(1, B, H, d, h, r, kv=kv)
    many = h2o.h2o_create(1, B, H, d, h, r, kv=kv)
    for c in (one, many):
        h2o.h2o_prefill(c, 0, *pre)
    out1 = torch.empty((S, B, H, d), dtype=torch.float32, device="cuda")
    ev1 = []
    for s in range(S):
        h2o.h2o_decode_step(one, 0, steps[0][s], steps[1][s], steps[2][s], out1[s])
        ev1.append(h2o.h2o_last_evicted(one, 0))
    outm = torch.empty_like(out1)
    evm = torch.empty((S, B * H), dtype=torch.int32, device="cuda")
    h2o.h2o_decode_steps(many, 0, *steps, outm, evm)
    h2o.h2o_sync_check(many)
    assert torch.equal(out1, outm)
    assert np.array_equal(np.stack(ev1), evm.cpu().numpy())
    assert (evm >= 0).any()  # evictions happened
    assert np.array_equal(h2o.h2o_cache_positions(one, 0), h2o.h2o_cache_positions(many, 0))
    v1, vm = h2o.h2o_cache_view(one, 0), h2o.h2o_cache_view(many, 0)
    for key in ("score", "meta", "K", "V"):
        assert torch.equal(v1[key], vm[key]), key
    if kv == "fp8":
        s1, sm = h2o.h2o_cache_scales(one, 0), h2o.h2o_cache_scales(many, 0)
        assert torch.equal(s1["K"], sm["K"]) and torch.equal(s1["V"], sm["V"])
    one.close()
    many.close()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("B,H,k", [(8, 32, 48), (40, 32, 48), (1, 4, 600)],
                         ids=["256-rows", "1280-rows", "4-rows-split"])
def test_back_to_back_steps_equal_synchronised_steps(kv, B, H, k):
    """A decode step is launched as a programmatic dependent of the kernel
    before it: its CTAs start (and prefetch the row's K/V into L2) while the
    previous step, or an h2o_decode_steps call, of the same layer still runs.
    Steps launched back to back after a multi-step call must equal, bit for
    bit, the same calls with the stream synchronised after every launch. Row
    shapes: 256 and 1280 rows of 48 slots (one CTA per row, 256 and 128
    threads) and 4 rows of 600 slots split over several CTAs."""
    import h2o_heavy_hitter_gb300 as h2o
    d, h = 128, k // 2
    r = k - h
    T, S1, S2 = k + 40, 6, 40
    w = Workload(440 + B + k, "pdl", 1, B, H, d, T, S1 + S2, h, r, 0.8)
    dh = [head_direction(w, 0, j) for j in range(H)]
    bits = [row_tokens(w, 0, b, j, dh[j]) for b in range(B) for j in range(H)]
    full = [_bf16(np.stack([x[c] for x in bits])).reshape(B, H, T + S1 + S2, d) for c in range(3)]
    pre = [x[:, :, :T].contiguous() for x in full]
    steps = [x[:, :, T:].permute(2, 0, 1, 3).contiguous() for x in full]  # [S1 + S2, B, H, d]
    outs, caches = [], []
    for sync in (False, True):
        ctx = h2o.h2o_create(1, B, H, d, h, r, kv=kv)
        h2o.h2o_prefill(ctx, 0, *pre)
        if sync:
            torch.cuda.synchronize()
        o = torch.zeros((S1 + S2, B, H, d), dtype=torch.float32, device="cuda")
        h2o.h2o_decode_steps(ctx, 0, *[x[:S1] for x in steps], o[:S1])
        for s in range(S1, S1 + S2):
            if sync:
                torch.cuda.synchronize()
            h2o.h2o_decode_step(ctx, 0, steps[0][s], steps[1][s], steps[2][s], o[s])
        h2o.h2o_sync_check(ctx)
        view = h2o.h2o_cache_view(ctx, 0)
        caches.append({key: view[key].clone() for key in ("score", "pos", "meta", "K", "V")})
        outs.append(o)
        ctx.close()
    assert torch.equal(outs[0], outs[1])
    for key in caches[0]:
        assert torch.equal(caches[0][key], caches[1][key]), key
    assert (caches[0]["meta"][:, 2] >= 0).any()  # evictions happened


def test_multistep_zero_steps_and_state_errors():
    import h2o_heavy_hitter_gb300 as h2o
    ctx = h2o.h2o_create(1, 1, 2, 64, 4, 4)
    x = torch.zeros((3, 1, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_decode_steps(ctx, 0, x, x, x)
    assert e.value.code == h2o.H2O_ESTATE
    e0 = torch.zeros((1, 2, 0, 64), dtype=torch.bfloat16, device="cuda")
    h2o.h2o_prefill(ctx, 0, e0, e0, e0)  # T = 0: empty cache
    h2o.h2o_decode_steps(ctx, 0, x[:0], x[:0], x[:0])  # nothing to do
    assert np.all(h2o.h2o_cache_positions(ctx, 0) == -1)
    h2o.h2o_decode_steps(ctx, 0, x, x, x)
    assert sorted(h2o.h2o_cache_positions(ctx, 0)[0][:3].tolist()) == [0, 1, 2]
    ctx.close()
