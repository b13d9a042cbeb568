"""Host-side helpers shared by the tests and the bench (CPU only)."""
import numpy as np

from h2o_parity import _slots_of
from workloads import (bf16_bits_to_f32, decode_bytes_per_row_step, prefill_bytes_per_row,
                       prefill_flops_per_row, stream_chunk)


def test_stream_chunks_are_reproducible_and_independent():
    a = stream_chunk(7, 3, 64, 4, 64)
    b = stream_chunk(7, 3, 64, 4, 64)
    c = stream_chunk(7, 4, 64, 4, 64)
    assert all(x.shape == (64, 4, 64) and x.dtype == np.uint16 for x in a)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not any(np.array_equal(x, y) for x, y in zip(a, c))


def test_stream_chunk_queries_lean_on_one_direction():
    """Queries carry +2 u along one unit direction shared by every chunk, so
    their mean is about 2 u (2 in norm) while the values have mean about 0."""
    q0, _, v0 = (bf16_bits_to_f32(x).reshape(-1, 64) for x in stream_chunk(1, 0, 2048, 2, 64))
    q1 = bf16_bits_to_f32(stream_chunk(1, 1, 2048, 2, 64)[0]).reshape(-1, 64)
    m0, m1 = q0.mean(axis=0), q1.mean(axis=0)
    assert abs(np.linalg.norm(m0) - 2.0) < 0.1
    assert np.dot(m0, m1) / (np.linalg.norm(m0) * np.linalg.norm(m1)) > 0.99
    assert np.linalg.norm(v0.mean(axis=0)) < 0.2


def test_ring_slots_of_retained_positions():
    """Ring layout: positions before the window fill slots 0.. in order; window
    position p sits in slot h + p mod r."""
    pos = np.array([1, 5, 9, 16, 17, 18, 19])
    slots = _slots_of(pos, k=7, t_next=20, ring=(3, 4))
    assert slots.tolist() == [0, 1, 2, 3, 4, 5, 6]
    pos = np.array([2, 13, 14, 15, 16])  # window 13..16 of t_next = 17
    assert _slots_of(pos, k=7, t_next=17, ring=(3, 4)).tolist() == [0, 4, 5, 6, 3]
    assert _slots_of(pos, k=7, t_next=17, ring=None).tolist() == [0, 1, 2, 3, 4]


def test_decode_byte_model_of_the_layouts():
    k, d, h = 460, 128, 230
    slots = decode_bytes_per_row_step(k, d)
    ring = decode_bytes_per_row_step(k, d, "bf16", "ring", h)
    assert slots == 4 * k * d + 12 * k + 14 * d + 8
    # the ring layout reads h positions instead of k and moves one token (8d + 8)
    assert ring - slots == 4 * h - 4 * k + 8 * d + 8
    assert decode_bytes_per_row_step(k, d, "fp8") == 2 * k * d + 20 * k + 12 * d + 16


def test_prefill_byte_and_flop_models():
    """T = 4, d = 2, k = 3 by hand: Q, K, V read 3 * 4 * 2 * 2 = 48 bytes, fp32
    O written 4 * 2 * 4 = 32, three kept slots of K + V (2 * 2 * 2 = 8) plus
    position and score (8): 48. Causal pairs 4 * 5 / 2 = 10, 2 * 2 * 2 flops
    each (QK^T and PV)."""
    assert prefill_bytes_per_row(4, 2, 3) == 48 + 32 + 3 * (8 + 8)
    # FP8 slots: 2 code bytes per element of K and V, two fp32 scales
    assert prefill_bytes_per_row(4, 2, 3, "fp8") == 48 + 32 + 3 * (4 + 8 + 8)
    # a prompt shorter than the budget keeps every token
    assert prefill_bytes_per_row(2, 2, 3) == 24 + 16 + 2 * 16
    assert prefill_flops_per_row(4, 2) == 10 * 8
    # the OPT-6.7B-shaped layer sits above the ridge of a 1.9 PF/s, 6.8 TB/s
    # part and the 512-token prompt below it
    ai = lambda T, k: prefill_flops_per_row(T, 128) / prefill_bytes_per_row(T, 128, k)
    assert ai(2048, 460) > 1907.5 / 6.8152 > ai(512, 204)


def test_profiled_traffic_needs_the_current_source_and_scales_by_rows(tmp_path):
    """The bench takes a kernel's DRAM traffic from a committed summary only if
    the summary's source hash is that of the kernel's files now, and scales it
    from the rows the summary states to the rows of the launch."""
    import hashlib

    import bench
    csrc = tmp_path / "h2o_heavy_hitter_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "a.cu").write_bytes(b"one")
    (csrc / "b.cuh").write_bytes(b"two")
    digest = hashlib.sha256(b"onetwo").hexdigest()
    summary = tmp_path / "profiles" / "decode_kernel_w.md"
    summary.write_text(f"source_sha256 (a + b): {digest}\ndram_bytes_per_launch: 1000\n"
                       "traffic_rows: 8\n")
    files = ("a.cu", "b.cuh")
    assert bench._profiled_traffic(files, "w", 8, str(tmp_path)) == 1000
    assert bench._profiled_traffic(files, "w", 2, str(tmp_path)) == 250
    assert bench._profiled_traffic(files, "other", 8, str(tmp_path)) is None
    (csrc / "b.cuh").write_bytes(b"changed")
    assert bench._profiled_traffic(files, "w", 8, str(tmp_path)) is None


def test_clock_record_keeps_the_timed_region_and_its_throttle_reasons():
    import datetime

    import bench
    day = "2026/12/03 08:00:0"
    na = "Not Active"

    def line(sec, mhz, cap=False):
        return (f"{day}{sec}.000, {mhz}, 2070, 900.0, 0x0, {na}, {na}, {na}, "
                f"{'Active' if cap else na}")

    text = "\n".join([line(0, 1200), line(2, 2070), line(3, 2070, cap=True), line(4, 2055),
                      line(5, 2070), line(8, 1000, cap=True), "garbage,1,2"])
    t = lambda sec: datetime.datetime.strptime(f"{day}{sec}.000", "%Y/%m/%d %H:%M:%S.%f").timestamp()
    c = bench.ClockSampler(0)
    c.mark(t(2), t(5))
    rec = c.summarize(text)
    assert rec["samples_in_timed_region"] == 4 and rec["window"] == "timed region"
    assert rec["sm_mhz"] == 2070.0 and rec["sm_mhz_min"] == 2055.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"]
    # fewer than three samples in the timed region: the whole window is reported
    c.mark(t(8), t(9))
    rec = c.summarize(text)
    assert rec["window"] == "warm-up and timed region" and rec["samples"] == 6
    assert rec["sm_mhz_min"] == 1000.0 and rec["reasons"] == ["sw_power_cap"]
    assert c.summarize("") is None
