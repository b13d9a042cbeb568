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
