"""GPU test of h2o_prefill_attention_noalloc, the entry point for callers that
must not allocate device memory during a call (its scratch is a fixed array in
the library instead of an allocation).

It is called through the C ABI twice in a row, on different shapes and data,
and each time compared with h2o_prefill_attention (which allocates its scratch)
using the same tolerances as the other prefill parity tests; a third call is
compared with the CPU oracle directly, row by row. A request larger
than the fixed scratch must be refused with H2O_EINVAL, and the call must run
on the stream it is given, not on the caller's current stream. This file is
named so that pytest collects it last; it also passes when run on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from workloads import Workload, bf16_bits_to_f64, head_direction, row_tokens

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3  # output tolerance of the prefill parity tests
SCORE_RTOL, SCORE_ATOL = 2e-5, 1e-6


def _lib():
    import h2o_heavy_hitter_gb300 as h2o
    lib = h2o.load_library()
    fn = lib.h2o_prefill_attention_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 3
    return h2o, lib


def _inputs(cfg_id, rows_b, heads, d, T):
    w = Workload(cfg_id, "noalloc", 1, rows_b, heads, d, T, 0, 8, 8, 0.8)
    bits = [row_tokens(w, 0, b, j, head_direction(w, 0, j))
            for b in range(rows_b) for j in range(heads)]
    dev = torch.device("cuda")
    return [torch.from_numpy(np.stack([x[i] for x in bits]).view(np.int16)).to(dev)
            .view(torch.bfloat16) for i in range(3)]


def _call_noalloc(lib, Q, K, V):
    rows, T, d = Q.shape
    out = torch.full((rows, T, d), float("nan"), dtype=torch.float32, device=Q.device)
    score = torch.full((rows, T), float("nan"), dtype=torch.float32, device=Q.device)
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.h2o_prefill_attention_noalloc(Q.data_ptr(), K.data_ptr(), V.data_ptr(), rows, T, d,
                                           out.data_ptr(), score.data_ptr(), stream)
    assert rc == 0, lib.h2o_last_error()
    return out, score


def _compare(got, ref):
    out, score = got
    out_ref, score_ref = ref
    torch.cuda.synchronize()
    err = (out - out_ref).abs()
    assert torch.isfinite(out).all() and torch.isfinite(score).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    np.testing.assert_allclose(score.cpu().numpy(), score_ref.cpu().numpy(), rtol=SCORE_RTOL,
                               atol=SCORE_ATOL)


def test_noalloc_matches_allocating_entry_point_on_two_calls():
    h2o, lib = _lib()
    # first call: several 128-token tiles and a ragged tail, d = 128
    Q, K, V = _inputs(290, 2, 3, 128, 333)
    _compare(_call_noalloc(lib, Q, K, V), h2o.h2o_prefill_attention(Q, K, V))
    # second call: other shape, other data, d = 64; the fixed scratch still holds
    # the first call's values, which must not leak into this result
    Q, K, V = _inputs(291, 1, 4, 64, 700)
    _compare(_call_noalloc(lib, Q, K, V), h2o.h2o_prefill_attention(Q, K, V))


def test_noalloc_matches_oracle():
    """Every row's output and column sums against the fp64 oracle (the same
    bar as the allocating entry point's oracle test): 3 x 2 rows of 389 tokens,
    d = 128, three full query tiles and a ragged tail."""
    _, lib = _lib()
    w = Workload(293, "noalloc-oracle", 1, 3, 2, 128, 389, 0, 8, 8, 0.8)
    bits = [row_tokens(w, 0, b, j, head_direction(w, 0, j))
            for b in range(w.batch) for j in range(w.heads)]
    Q, K, V = _inputs(293, 3, 2, 128, 389)
    out, score = _call_noalloc(lib, Q, K, V)
    torch.cuda.synchronize()
    out, score = out.cpu().numpy(), score.cpu().numpy()
    for i, x in enumerate(bits):
        q, k, v = (bf16_bits_to_f64(y) for y in x)
        O, colsum, _ = oracle.prefill_attention(q, k, v, oracle.default_scale(w.head_dim))
        err = np.abs(out[i] - O)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (i, err.max(), err.mean())
        np.testing.assert_allclose(score[i], colsum, rtol=SCORE_RTOL, atol=SCORE_ATOL)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    _, lib = _lib()
    limit = 1 << 20  # H2O_NOALLOC_MAX_LSE floats
    rows, T = limit // 128 + 1, 128  # one row too many
    rc = lib.h2o_prefill_attention_noalloc(None, None, None, rows, T, 128, None, None, None)
    assert rc == -1
    assert b"exceeds the fixed scratch" in lib.h2o_last_error()


def test_noalloc_runs_on_the_stream_it_is_given():
    """With the current stream busy (a long spin kernel queued on it), a call
    given another stream must still finish on that stream: copies of its
    outputs queued behind it on the same stream see finished results. Had the
    kernels gone to the current stream, the copies would run first and hold
    the NaN fill."""
    h2o, lib = _lib()
    Q, K, V = _inputs(292, 1, 2, 128, 257)
    ref = h2o.h2o_prefill_attention(Q, K, V)
    rows, T, d = Q.shape
    out = torch.full((rows, T, d), float("nan"), dtype=torch.float32, device=Q.device)
    score = torch.full((rows, T), float("nan"), dtype=torch.float32, device=Q.device)
    out_c, score_c = torch.empty_like(out), torch.empty_like(score)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    torch.cuda._sleep(200_000_000)  # about 0.1 s of work on the current stream
    rc = lib.h2o_prefill_attention_noalloc(Q.data_ptr(), K.data_ptr(), V.data_ptr(), rows, T, d,
                                           out.data_ptr(), score.data_ptr(), side.cuda_stream)
    assert rc == 0, lib.h2o_last_error()
    with torch.cuda.stream(side):
        out_c.copy_(out)
        score_c.copy_(score)
    torch.cuda.synchronize()
    _compare((out_c, score_c), ref)
    h2o.h2o_attention_sync_check(side)  # no device error reported by the kernels
