"""CPU pins of the oracle's FP8 (E4M3) KV-cache mode (oracle/kv_fp8.py).

The codec is pinned to the format's definition (decode table values, exact
round trips, brute-force nearest-value search with ties to even, saturation),
the quantiser to its error bound, and the quantised decode to two facts that
do not reuse its own arithmetic: it must equal the plain oracle run on
inputs that were quantised and dequantised beforehand, and it must equal the
plain oracle exactly when every token is representable (quantisation is then
the identity).
"""
import numpy as np
import pytest

import oracle
from oracle import kv_fp8
from workloads import Workload, bf16_bits_to_f64, row_tokens

TABLE = kv_fp8.e4m3_decode(np.arange(256))
FINITE = np.nonzero(~np.isnan(TABLE))[0]


def test_decode_table_fixed_points():
    assert TABLE[0x00] == 0.0 and TABLE[0x01] == 2.0 ** -9 and TABLE[0x07] == 7 * 2.0 ** -9
    assert TABLE[0x08] == 2.0 ** -6  # smallest normal
    assert TABLE[0x38] == 1.0 and TABLE[0xB8] == -1.0
    assert TABLE[0x7E] == 448.0 and TABLE[0xFE] == -448.0
    assert np.isnan(TABLE[0x7F]) and np.isnan(TABLE[0xFF])
    assert len(FINITE) == 254
    assert np.all(np.diff(TABLE[:0x7F]) > 0)  # positive codes are ordered by value


def test_encode_round_trips_every_finite_code():
    assert np.array_equal(kv_fp8.e4m3_encode(TABLE[FINITE].astype(np.float32)), FINITE.astype(np.uint8))


def _nearest_even(x):
    """Brute force: the finite code whose value is nearest x; ties to the even code."""
    pos = FINITE[FINITE < 0x80]
    vals = TABLE[pos]
    a = abs(float(x))
    if a >= 448.0:
        c = 0x7E
    else:
        dist = np.abs(vals - a)
        best = np.nonzero(dist == dist.min())[0]
        cands = pos[best]
        c = int(cands[0]) if len(cands) == 1 else int([v for v in cands if v % 2 == 0][0])
    return c | (0x80 if np.signbit(x) else 0)


def test_encode_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(3)
    xs = np.concatenate([
        rng.standard_normal(3000) * 40, rng.standard_normal(2000) * 0.01,
        (TABLE[1:0x7E] + TABLE[2:0x7F]) / 2,  # every midpoint between neighbours
        -(TABLE[1:0x7E] + TABLE[2:0x7F]) / 2, [0.0, -0.0, 447.9, 460.0, 470.0, 1e9],
    ]).astype(np.float32)
    got = kv_fp8.e4m3_encode(xs)
    want = np.array([_nearest_even(x) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_quantize_vector_bounds_and_zero():
    codes, scale = kv_fp8.quantize_vector(np.zeros(64))
    assert scale == 0 and not codes.any()
    rng = np.random.default_rng(4)
    for _ in range(200):
        x = (rng.standard_normal(128) * rng.uniform(0.01, 30)).astype(np.float32)
        codes, scale = kv_fp8.quantize_vector(x)
        i = int(np.argmax(np.abs(x)))
        assert codes[i] & 0x7F == 0x7E  # the largest element maps to +-448
        err = np.abs(kv_fp8.dequantize_vector(codes, scale) - x.astype(np.float64))
        # half a mantissa step (1/16 relative) or half a subnormal step
        assert np.all(err <= np.abs(x) / 16 * (1 + 1e-6) + scale * 2.0 ** -10 * (1 + 1e-6))


def _row(cfg_id=7, T=24, S=30, d=32):
    w = Workload(cfg_id, "fp8pin", 1, 1, 1, d, T, S, 4, 4, 0.8)
    q, k, v = row_tokens(w, 0, 0, 0)
    return w, bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)


def test_fp8_decode_equals_plain_oracle_on_prequantised_inputs():
    w, q, k, v = _row()
    T, S = w.prompt, w.steps
    got = oracle.run_row(q, k, v, T, S, w.h, w.r, kv_fp8_cache=True)
    pre = oracle.prefill(q[:T], k[:T], v[:T], w.h, w.r)
    c = pre.cache
    c.K = np.array([kv_fp8.roundtrip(x) for x in c.K])
    c.V = np.array([kv_fp8.roundtrip(x) for x in c.V])
    for s in range(S):
        lg = oracle.decode_step(c, q[T + s], kv_fp8.roundtrip(k[T + s]), kv_fp8.roundtrip(v[T + s]))
        assert lg.evicted == got.evicted[s]
        assert np.array_equal(lg.out, got.outs[s])
        assert np.array_equal(c.pos, got.kept_after[s])
        assert np.array_equal(c.score, got.scores_after[s])


def test_fp8_equals_plain_oracle_when_tokens_are_representable():
    rng = np.random.default_rng(5)
    T, S, d = 20, 25, 32
    codes = rng.integers(0, 0x7F, size=(3, T + S, d)).astype(np.uint8)
    codes[:, :, 0] = 0x7E  # amax = 448 in every token: scale 2^-5 after the 2^-5 factor
    codes |= (rng.integers(0, 2, size=codes.shape) << 7).astype(np.uint8)
    codes[:, :, 0] &= 0x7F
    x = kv_fp8.e4m3_decode(codes) * 2.0 ** -5
    q, k, v = x
    plain = oracle.run_row(q, k, v, T, S, 4, 4)
    fp8 = oracle.run_row(q, k, v, T, S, 4, 4, kv_fp8_cache=True)
    assert plain.evicted == fp8.evicted
    for a, b in zip(plain.outs, fp8.outs):
        assert np.array_equal(a, b)


def test_fp8_cache_keeps_codes_aligned_with_positions():
    w, q, k, v = _row(cfg_id=8, T=16, S=40)
    T = w.prompt
    pre = oracle.prefill(q[:T], k[:T], v[:T], w.h, w.r, kv_fp8_cache=True)
    c = pre.cache
    for s in range(w.steps):
        oracle.decode_step(c, q[T + s], k[T + s], v[T + s])
        for i, p in enumerate(c.pos):
            kc, ks = kv_fp8.quantize_vector(k[p])
            assert np.array_equal(c.Kc[i], kc) and c.Ks[i] == ks
            assert np.array_equal(c.K[i], kv_fp8.dequantize_vector(kc, ks))
