"""Ragged batches: prompts of different lengths in one prefill (h2o_prefill_ragged).

Each batch entry's prompt is right-padded with large finite garbage to the
longest length; the oracle runs every row at its own length. Tolerances and
near-tie rules as in test_gpu_parity. A ragged row must also reproduce, bit for
bit, a dense prefill of the same prompt at its own length (the padded keys
enter the tensor-core products with probability exactly 0).
"""
import numpy as np
import pytest
import torch

from h2o_parity import run_parity
from test_gpu_parity import _assert_ok
from workloads import Workload, head_direction, row_tokens

pytestmark = pytest.mark.gpu

RAGGED = [
    # (name, heads, d, T_max, S, h, r, lengths per batch entry)
    ("d128-mixed", 2, 128, 300, 24, 20, 12, [300, 0, 1, 20, 128, 129, 257]),
    ("d64-mixed", 3, 64, 259, 20, 17, 9, [259, 5, 26, 130, 200]),
    ("recent-only", 2, 128, 200, 16, 0, 24, [200, 24, 25, 3]),
]


@pytest.mark.parametrize("name,H,d,T,S,h,r,lens", RAGGED, ids=[c[0] for c in RAGGED])
def test_ragged_batch_matches_oracle(name, H, d, T, S, h, r, lens):
    w = Workload(300 + [c[0] for c in RAGGED].index(name), name, 1, len(lens), H, d, T, S, h, r,
                 0.8)
    _assert_ok(run_parity(w, lens=lens), name)


def test_ragged_batch_fp8_cache_matches_oracle():
    lens = [190, 1, 64, 150]
    w = Workload(310, "ragged-fp8", 1, len(lens), 2, 128, 190, 20, 16, 16, 0.8)
    rep = run_parity(w, lens=lens, kv="fp8")
    _assert_ok(rep, "ragged-fp8")
    assert rep.code_checks > 0 and not rep.code_mismatches, rep.code_mismatches[:5]


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def test_ragged_rows_equal_dense_prefill_bitwise():
    """Row b of a ragged batch == a dense prefill of its prompt at length
    lens[b]: outputs, cache positions and scores, then decode outputs and the
    positions kept after them."""
    import h2o_heavy_hitter_gb300 as h2o
    lens = [333, 128, 45, 200]
    B, H, d, T, S, h, r = len(lens), 2, 128, 333, 12, 24, 16
    w = Workload(320, "ragged-bitwise", 1, B, H, d, T, S, h, r, 0.8)
    bits = [[row_tokens(w, 0, b, j, head_direction(w, 0, j)) for j in range(H)] for b in range(B)]
    full = [_bf16(np.stack([np.stack([bits[b][j][c] for j in range(H)]) for b in range(B)]))
            for c in range(3)]  # [B, H, N, d]
    pad = []
    for x in full:
        y = x[:, :, :T].clone()
        for b, n in enumerate(lens):
            y[b, :, n:] = 3.0  # finite padding
        pad.append(y.contiguous())
    ctx = h2o.h2o_create(1, B, H, d, h, r)
    out = h2o.h2o_prefill(ctx, 0, *pad, lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    pos = h2o.h2o_cache_positions(ctx, 0)
    score = h2o.h2o_cache_view(ctx, 0)["score"].clone()
    tok = torch.tensor(lens, device="cuda")[None, :] + torch.arange(S, device="cuda")[:, None]
    bidx = torch.arange(B, device="cuda")[None, :].expand(S, B)
    steps = [x.permute(0, 2, 1, 3)[bidx, tok].contiguous() for x in full]  # [S, B, H, d]
    dec = torch.empty((S, B, H, d), dtype=torch.float32, device="cuda")
    for s in range(S):
        h2o.h2o_decode_step(ctx, 0, steps[0][s], steps[1][s], steps[2][s], dec[s])
    h2o.h2o_sync_check(ctx)
    for b, n in enumerate(lens):
        # a dense batch of the same shape with every prompt cut to n tokens
        # (same decode launch shape); only entry b is compared
        one = h2o.h2o_create(1, B, H, d, h, r)
        o1 = h2o.h2o_prefill(one, 0, *(x[:, :, :n].contiguous() for x in full))
        assert torch.equal(out[b, :, :n], o1[b]), b
        p1 = h2o.h2o_cache_positions(one, 0)
        s1 = h2o.h2o_cache_view(one, 0)["score"]
        rows = slice(b * H, (b + 1) * H)
        assert np.array_equal(pos[rows], p1[rows]), b
        assert torch.equal(score[rows], s1[rows]), b
        d1 = torch.empty((S, B, H, d), dtype=torch.float32, device="cuda")
        for s in range(S):
            h2o.h2o_decode_step(one, 0, *(x[:, :, n + s].contiguous() for x in full), d1[s])
        assert torch.equal(dec[:, b], d1[:, b]), b
        assert np.array_equal(h2o.h2o_cache_positions(ctx, 0)[rows],
                              h2o.h2o_cache_positions(one, 0)[rows]), b
        one.close()
    ctx.close()


def test_ragged_length_out_of_range_is_clamped_and_reported():
    """A length above T_max is clamped to T_max and one below 0 to 0; the
    device error word reports it (no access leaves the padded tensors)."""
    import h2o_heavy_hitter_gb300 as h2o
    B, H, d, T = 2, 2, 64, 130
    g = torch.Generator(device="cuda").manual_seed(7)
    Q, K, V = (torch.randn((B, H, T, d), device="cuda", generator=g).to(torch.bfloat16)
               for _ in range(3))
    ctx = h2o.h2o_create(1, B, H, d, 8, 8)
    h2o.h2o_prefill(ctx, 0, Q, K, V, lens=torch.tensor([T + 5, -1], dtype=torch.int32,
                                                        device="cuda"))
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_sync_check(ctx)
    assert e.value.code == h2o.H2O_EDEVICE and "word 0x4 " in str(e.value)
    pos = h2o.h2o_cache_positions(ctx, 0)
    meta = h2o.h2o_cache_view(ctx, 0)["meta"].cpu().numpy()
    assert np.all(pos[2:] == -1) and np.all(meta[2:, :2] == 0)  # clamped to an empty prompt
    assert np.all(meta[:2, 1] == T) and np.all(meta[:2, 0] == 16)  # clamped to T_max
    h2o.h2o_sync_check(ctx)  # the word was cleared
    ctx.close()
