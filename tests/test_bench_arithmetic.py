"""The bench's measurement arithmetic on hand-worked examples: the
algorithmic work of an iteration, the iteration roofline, the roofline
object of a kernel class, and the steady-state window (CS349D Lecture 2,
section 5 results: steady-state throughput counts up to the iteration in
which the last request produces its first token)."""
import os
import sys
from types import SimpleNamespace

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

SHAPE = SimpleNamespace(hidden=4, n_layers=2, vocab=10)
PEAKS = {"hbm_gbs": 1.0, "bf16_tflops_sustained": 1e-3}  # 1e9 B/s and 1e9 FLOP/s: balance 1 FLOP/B


def test_iteration_work_by_hand():
    # rows: a prompt of 3 (no cache) and one decode row over 5 cached keys
    # pairs = 3*0 + 3*4/2 + 1*5 + 1*2/2 = 12; N = 4 rows, B = 2 requests
    # Linears 2*N*12*H^2*layers = 2*4*12*16*2 = 3072; LM head 2*B*H*V = 160; attention 4*H*pairs*layers = 384
    flops, kv = bench.iteration_work(SHAPE, [(3, 0), (1, 5)])
    assert flops == 3072 + 160 + 384
    # K/V: (cached + new) keys * (K and V) * H * 2 bytes * layers = 9 * 2 * 4 * 2 * 2
    assert kv == 288


def test_iteration_roofline_by_hand():
    batches = [[(3, 0), (1, 5)], [(1, 3), (1, 6)]]
    f2, kv2 = bench.iteration_work(SHAPE, batches[1])
    # second batch: N = 2, B = 2, pairs = 3 + 1 + 6 + 1 = 11 -> 2*2*12*16*2 + 160 + 4*4*11*2 = 1536 + 160 + 352
    assert f2 == 2048 and kv2 == (9 + 2) * 2 * 4 * 2 * 2
    w = 1000.0  # weight bytes
    r = bench.iteration_roofline(SHAPE, w, batches, measured_s=1e-5, peaks=PEAKS)
    t = max((w + 288) / 1e9, 3616 / 1e9) + max((w + 352) / 1e9, 2048 / 1e9)
    assert r["t_roof_ms_per_step"] == pytest.approx(1000 * t / 2)
    assert r["frac"] == pytest.approx(t / 1e-5)
    assert r["bound"] == "tensor"  # 5664 FLOP against 2640 bytes over the two iterations
    assert r["flops_per_step"] == pytest.approx((3616 + 2048) / 2)


def test_roofline_of_takes_the_bound_by_intensity():
    agg = {"gemm": {"launches": 4, "ms": 2.0, "flops": 8e9, "bytes": 1e9},
           "attn": {"launches": 2, "ms": 1.0, "flops": 1e8, "bytes": 5e8}}
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops_sustained": 2.0}  # balance 2 FLOP/B
    g = bench.roofline_of(agg, "gemm", peaks, "measured", "no-such-config")
    assert g["bound"] == "tensor" and g["unit"] == "TFLOP/s"
    assert g["achieved"] == pytest.approx(8e9 / 2e-3 / 1e12) and g["frac"] == pytest.approx(4.0 / 2.0)
    assert g["algorithmic_per_launch"] == pytest.approx(2e9) and g["ms_per_launch"] == pytest.approx(0.5)
    assert g["traffic"] is None
    a = bench.roofline_of(agg, "attn", peaks, "measured", "no-such-config")
    assert a["bound"] == "hbm" and a["achieved"] == pytest.approx(500.0) and a["frac"] == pytest.approx(0.5)
    per = bench.per_kernel_roofline(agg, peaks)
    assert per["gemm"]["frac_tensor"] == pytest.approx(2.0) and per["attn"]["frac_hbm"] == pytest.approx(0.5)


def _rec(req_ids, next_tokens, n_new, released):
    return SimpleNamespace(req_ids=req_ids, next_tokens=next_tokens, n_new=n_new, released=released)


def test_steady_state_window_by_hand():
    # request 3 arrives late and produces its first token in iteration 2; iteration 3 only drains
    recs = [_rec([1, 2], [7, 8], [4, 2], []),
            _rec([1, 2], [5, 6], [1, 1], [2]),
            _rec([1, 3], [9, 4], [1, 5], []),
            _rec([1, 3], [3, 2], [1, 1], [1, 3])]
    it_ms = [2.0, 1.0, 3.0, 1.0]
    s = bench.steady_state(recs, it_ms)
    assert s["iterations"] == 3 and s["seconds"] == pytest.approx(6e-3)
    assert s["processed_tokens_per_s"] == pytest.approx((6 + 2 + 6) / 6e-3)
    assert s["generated_tokens_per_s"] == pytest.approx(6 / 6e-3)
    assert s["completed_requests_per_s"] == pytest.approx(1 / 6e-3)
