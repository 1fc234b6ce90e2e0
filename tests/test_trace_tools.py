"""Host logic of the trace tools (no GPU): the steady-state summaries of
trace_attn and trace_mla on synthetic stamp arrays with known step lengths."""
import numpy as np

import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import trace_attn, trace_mla


def _attn_stamps(ntile, pipelined, period=4000, step=100):
    ev = {n: i for i, n in enumerate(gb.ATTN_TRACE_EVENTS)}
    tr = np.zeros((4, len(ev), 132), dtype=np.int64)
    clock = np.zeros((4, 4), dtype=np.int64)
    base = 1000
    order = ["wait_v", "v_seen", "p0_seen", "pv0_issued", "k_next_seen", "s0_next_issued",
             "s0_seen", "s0_loaded", "max0", "exp0", "p0_arrive"]
    if not pipelined:
        order += ["p1_seen", "pv1_issued", "s1_next_issued", "s1_seen", "s1_loaded", "max1", "exp1", "p1_arrive"]
    for j in range(ntile):
        for k, name in enumerate(order):
            tr[0, ev[name], j] = base + j * period + k * step
    clock[0] = (0, 0, 2 * (ntile * period + 10000), ntile * period + 10000)   # 2 cycles per ns
    return tr, clock


def test_attn_summary_two_tile_form():
    tr, clock = _attn_stamps(40, pipelined=False)
    sm = trace_attn.steady_state_summary(tr, clock, 0)
    assert sm["form"] == "two-tile" and sm["tiles"] == 40
    assert abs(sm["ghz"] - 2.0) < 1e-9
    assert sm["period"] == 4000
    assert sm["issuer: wait V"] == 100 and sm["issuer: wait P0"] == 100
    assert sm["softmax 0: load scores"] == 100
    # the next tile's S is seen one period after this tile's issue, less the steps between
    assert sm["softmax 0: S issued -> seen"] == 4000 + 100
    assert trace_attn.steady_state_summary(tr, clock, 1)["tiles"] == 0


def test_attn_summary_pipelined_form():
    tr, clock = _attn_stamps(24, pipelined=True)
    sm = trace_attn.steady_state_summary(tr, clock, 0)
    assert sm["form"] == "pipelined" and sm["tiles"] == 24
    assert sm["period"] == 4000
    assert sm["issuer: wait P"] == 100 and sm["issuer: issue P V"] == 100
    assert sm["softmax: arrive -> issuer sees P"] == -800      # the synthetic order stamps P seen first
    assert "softmax 1: load scores" not in sm


def test_mla_summary_reads_step_medians():
    ev = {n: i for i, n in enumerate(gb.MLA_TRACE_EVENTS)}
    tr = np.zeros((2, len(ev), 64), dtype=np.uint64)
    for c in range(2):
        for t in range(40):
            for k, name in enumerate(gb.MLA_TRACE_EVENTS):
                tr[c, ev[name], t] = 10 ** 6 + t * 1700 + k * 50 + (0 if name != "load" else -2000)
    sm = trace_mla.steady_state_summary(tr)
    assert sm["tiles_traced"] == 40
    assert abs(sm["cta0"]["tile_period"] - 1.7) < 1e-9
    assert abs(sm["cta0"]["ring_slot_cycle"] - 4 * 1.7) < 1e-9
