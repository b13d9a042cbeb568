"""The failure path of the library's bounded device waits, made to happen on
purpose without faulting anything: a kernel waits on an mbarrier that nothing
arrives on, gives up after the wait limit, sets the device error word and
returns. The host reads the status, and the context keeps working."""
import time

import numpy as np
import pytest
import torch

from workloads import WORKLOADS, head_direction, row_tokens

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_is_reported_and_the_context_survives():
    import h2o_heavy_hitter_gb300 as h2o
    w = WORKLOADS["tiny"]
    B, H, d, T = w.batch, w.heads, w.head_dim, w.prompt
    bits = [row_tokens(w, 0, 0, j, head_direction(w, 0, j)) for j in range(H)]
    full = [torch.from_numpy(np.stack([x[c] for x in bits]).view(np.int16)).cuda()
            .view(torch.bfloat16).reshape(B, H, w.tokens, d) for c in range(3)]
    ctx = h2o.h2o_create(1, B, H, d, w.h, w.r)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    h2o.h2o_test_wait_limit(ctx)
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_sync_check(ctx)
    waited = time.perf_counter() - t0
    assert e.value.code == h2o.H2O_EDEVICE and "word 0x1 " in str(e.value)
    assert 1.5 < waited < 30, waited  # the 2 s limit, then the kernel returned
    h2o.h2o_sync_check(ctx)  # the word was cleared
    # the context still runs the hot path
    h2o.h2o_prefill(ctx, 0, *(x[:, :, :T].contiguous() for x in full))
    for s in range(4):
        h2o.h2o_decode_step(ctx, 0, *(x[:, :, T + s].contiguous() for x in full))
    h2o.h2o_sync_check(ctx)
    assert np.all(h2o.h2o_cache_positions(ctx, 0)[:, -4:] >= 0)
    ctx.close()


def _tiny_inputs():
    w = WORKLOADS["tiny"]
    bits = [row_tokens(w, 0, 0, j, head_direction(w, 0, j)) for j in range(w.heads)]
    full = [torch.from_numpy(np.stack([x[c] for x in bits]).view(np.int16)).cuda()
            .view(torch.bfloat16).reshape(w.batch, w.heads, w.tokens, w.head_dim) for c in range(3)]
    return w, full


def test_cache_free_attention_reports_a_wait_that_runs_out():
    """The cache-free prefill entry points report through the library's own
    error word (no context): a wait that runs out against it is seen by
    h2o_attention_sync_check, on the stream that ran it, and then cleared."""
    import h2o_heavy_hitter_gb300 as h2o
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    h2o.h2o_attention_sync_check(side)  # nothing reported so far
    t0 = time.perf_counter()
    h2o.h2o_attention_test_wait_limit(side)
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_attention_sync_check(side)
    assert e.value.code == h2o.H2O_EDEVICE and "word 0x1 " in str(e.value)
    assert 1.5 < time.perf_counter() - t0 < 30
    h2o.h2o_attention_sync_check(side)  # cleared
    w, full = _tiny_inputs()
    Q, K, V = (x[0].contiguous() for x in full)  # [heads, N, d]: rows of the cache-free call
    out, score = h2o.h2o_prefill_attention(Q, K, V)
    h2o.h2o_attention_sync_check()
    assert torch.isfinite(out).all() and torch.isfinite(score).all()


def test_second_prefill_needs_a_reset():
    import h2o_heavy_hitter_gb300 as h2o
    w, full = _tiny_inputs()
    T = w.prompt
    pre = [x[:, :, :T].contiguous() for x in full]
    ctx = h2o.h2o_create(2, w.batch, w.heads, w.head_dim, w.h, w.r)
    h2o.h2o_prefill(ctx, 0, *pre)
    first = h2o.h2o_cache_positions(ctx, 0)
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_prefill(ctx, 0, *pre)
    assert e.value.code == h2o.H2O_ESTATE
    assert np.array_equal(h2o.h2o_cache_positions(ctx, 0), first)  # unchanged
    h2o.h2o_prefill(ctx, 1, *pre)  # the other layer is still empty
    h2o.h2o_reset(ctx, 0)
    assert np.all(h2o.h2o_cache_positions(ctx, 0) == -1)
    x = full[0][:, :, T].contiguous()
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_decode_step(ctx, 0, x, x, x)  # empty again: decode needs a prompt first
    assert e.value.code == h2o.H2O_ESTATE
    h2o.h2o_prefill(ctx, 0, *pre)
    assert np.array_equal(h2o.h2o_cache_positions(ctx, 0), first)
    h2o.h2o_reset(ctx, -1)
    for layer in range(2):
        h2o.h2o_prefill(ctx, layer, *pre)
    h2o.h2o_sync_check(ctx)
    ctx.close()


def test_allocation_failure_is_reported_and_nothing_changes():
    """Host-side fault injection: the library's next device allocations fail as
    an exhausted allocator would. Calls that allocate return H2O_ENOMEM and
    leave the state as it was; calls that allocate nothing are unaffected."""
    import h2o_heavy_hitter_gb300 as h2o
    w, full = _tiny_inputs()
    T = w.prompt
    pre = [x[:, :, :T].contiguous() for x in full]
    try:
        h2o.h2o_test_fail_allocations(1)
        with pytest.raises(h2o.H2OError) as e:
            h2o.h2o_create(1, w.batch, w.heads, w.head_dim, w.h, w.r)
        assert e.value.code == h2o.H2O_ENOMEM
        ctx = h2o.h2o_create(1, w.batch, w.heads, w.head_dim, w.h, w.r)  # the fault was used up
        h2o.h2o_test_fail_allocations(1)
        with pytest.raises(h2o.H2OError) as e:
            h2o.h2o_prefill(ctx, 0, *pre)
        assert e.value.code == h2o.H2O_ENOMEM
        x = full[0][:, :, T].contiguous()
        with pytest.raises(h2o.H2OError) as e:
            h2o.h2o_decode_step(ctx, 0, x, x, x)  # the failed prefill left the layer empty
        assert e.value.code == h2o.H2O_ESTATE
        h2o.h2o_test_fail_allocations(1)
        Q, K, V = (t[0, :, :T].contiguous() for t in full)
        with pytest.raises(h2o.H2OError) as e:
            h2o.h2o_prefill_attention(Q, K, V)
        assert e.value.code == h2o.H2O_ENOMEM
        h2o.h2o_test_fail_allocations(0)
        h2o.h2o_prefill(ctx, 0, *pre)  # the context still works
        h2o.h2o_test_fail_allocations(1000)  # decode steps allocate nothing
        for s in range(4):
            h2o.h2o_decode_step(ctx, 0, *(t[:, :, T + s].contiguous() for t in full))
        h2o.h2o_sync_check(ctx)
        ctx.close()
    finally:
        h2o.h2o_test_fail_allocations(0)


def test_inconsistent_cache_state_is_reported_not_written_through():
    """A cache state no call of the library produces, installed through the
    cache view: the decode kernel reports it in the error word (bad state)
    instead of using it, and leaves a row with impossible counts untouched."""
    import h2o_heavy_hitter_gb300 as h2o
    w, full = _tiny_inputs()
    T, k = w.prompt, w.k
    pre = [x[:, :, :T].contiguous() for x in full]
    ctx = h2o.h2o_create(1, w.batch, w.heads, w.head_dim, w.h, w.r)
    h2o.h2o_prefill(ctx, 0, *pre)
    view = h2o.h2o_cache_view(ctx, 0)
    step = lambda s: h2o.h2o_decode_step(ctx, 0, *(t[:, :, T + s].contiguous() for t in full))
    step(0)
    h2o.h2o_sync_check(ctx)
    meta_before = view["meta"].clone()
    pos_before = view["pos"].clone()
    view["meta"][0, 0] = k + 3  # more tokens than slots
    view["meta"][1, 0] = -2  # a negative fill count
    step(1)
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_sync_check(ctx)
    assert e.value.code == h2o.H2O_EDEVICE and "word 0x2 " in str(e.value)
    assert torch.equal(view["pos"][:2], pos_before[:2])  # rows 0 and 1 untouched
    assert torch.equal(view["meta"][0, 1:], meta_before[0, 1:])
    assert torch.all(view["meta"][2:, 1] == meta_before[2:, 1] + 1)  # the others advanced
    view["meta"][:2] = meta_before[:2] + torch.tensor([0, 1, 0, 0], dtype=torch.int32,
                                                      device="cuda")  # consistent again
    view["pos"][2, 0] = T + 100  # a position the row has not reached
    step(2)
    with pytest.raises(h2o.H2OError) as e:
        h2o.h2o_sync_check(ctx)
    assert e.value.code == h2o.H2O_EDEVICE and "word 0x2 " in str(e.value)
    h2o.h2o_reset(ctx, 0)
    h2o.h2o_prefill(ctx, 0, *pre)
    step(0)
    h2o.h2o_sync_check(ctx)
    ctx.close()
