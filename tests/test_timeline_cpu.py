"""Host logic of the device timeline (mxfp8_mlp_gqa_gb300.timeline) on synthetic records: the
launches of one step are recovered per kernel id by cutting at the largest entry-time gaps,
and the per-launch summary (entry, wait return, marks, exit, exposed time) is computed from
the right records."""
import numpy as np

from mxfp8_mlp_gqa_gb300 import timeline


def _rec(kid, block, t_enter, t_wait, t_exit, m1=0, m2=0, warp=0):
    return [kid, block, warp, t_enter, t_wait, t_exit, m1, m2]


def _step(t0):
    us = lambda x: int(t0 + x * 1000)  # noqa: E731
    r = []
    r += [_rec(3, b, us(0.0), us(0.1), us(2.0)) for b in range(4)]                       # shift (forked)
    r += [_rec(2, b, us(1.0), us(1.5), us(5.0)) for b in range(4)]                       # rmsnorm 1
    r += [_rec(17, b, us(2.0), us(6.0), us(18.0), us(11.0), us(12.0)) for b in range(4)]  # qkv
    r += [_rec(6, b, us(7.0), us(19.0), us(90.0), us(50.0), us(89.0)) for b in range(8)]  # split
    r += [_rec(7, b, us(82.0), us(91.0), us(97.0)) for b in range(8)]                    # combine
    r += [_rec(17, b, us(95.0), us(98.0), us(106.0), us(101.0), us(103.0)) for b in range(4)]  # o
    r += [_rec(2, b, us(99.0), us(106.5), us(110.0)) for b in range(4)]                  # rmsnorm 2
    r += [_rec(18, b, us(107.0), us(111.0), us(122.0), us(120.0), us(121.0)) for b in range(4)]  # gate/up
    r += [_rec(17, b, us(121.0), us(123.0), us(134.0), us(130.0), us(131.0)) for b in range(4)]  # down
    rec = np.array(r, np.int64)
    return rec[np.random.default_rng(0).permutation(len(rec))]  # buffer order is arbitrary


def test_launches_recovered_and_summarised():
    steps = [_step(1_000_000), _step(9_000_000)]
    parts = dict(timeline.split_launches(steps[0]))
    assert len(parts["qkv gemm + kv append"]) == 4 and len(parts["mlp down + residual"]) == 4
    assert parts["o gemm + residual"][:, 3].min() - steps[0][:, 3].min() == 95_000
    s = timeline.summarize(steps)
    assert s["qkv gemm + kv append"]["waited"] == 6.0
    assert s["attention split"]["mark2"] == 89.0
    assert s["attention combine"]["exposed"] == 97.0 - 90.0
    assert s["rmsnorm 1 + quant"]["exposed"] == 5.0       # first on the chain: from the step's start
    assert s["mlp down + residual"]["exit"] == 134.0
    assert np.isnan(s["prev_tokens_shift"]["exposed"])   # off the critical chain
    assert "mlp gate/up + swiglu" in timeline.format_table(s)
