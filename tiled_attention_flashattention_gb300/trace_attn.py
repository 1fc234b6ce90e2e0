"""Latency trace of the prefill kernel's dense forms on the GPU (observability tool).

    python -m tiled_attention_flashattention_gb300.trace_attn [--workload NAME] [--table]

Builds the library's trace variant (``libgbattn_trace.so``: the same sources
with -DGBATTN_TRACE), runs attn_fwd on the seeded inputs of a prefill workload
(default: the 16k causal headline shape) after three warm-up calls and an L2
flush, and reads the per-key-tile cycle stamps of four CTAs
(``gbattn_attn_trace``).  For each CTA it prints the median, over the
steady-state tiles, of every step of a tile's chain: the tile period; the
issuer's waits and MMA issues (an MMA issue blocks while the tensor core's
queue is full, so its duration is tensor-core time); and per softmax warpgroup
the delay from S issued to S seen, the score load, the row maximum, the
exponentials with the P stores, the wait for the stores and the arrive, and
the delays from the arrive to the issuer seeing P and to the next S being
seen.  Cycles are converted to time with each CTA's own cycle / global-timer
ratio.  ``--table`` also prints every tile's stamps.  Launches that take the
two-tile form (long rows) and the pipelined one-tile form (short rows: one Q
tile, 64-key tiles, S of tile n + 1 issued before P V of tile n) are traced;
block-sparse launches are not.

Runs in a process of its own: the trace build and the default library export
the same symbols and are not loaded together.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import _build
from . import load_library, attn_fwd, attn_trace, check, ATTN_TRACE_EVENTS
from . import workloads as wl


def steady_state_summary(tr: np.ndarray, clock: np.ndarray, cta: int) -> dict:
    """Medians (cycles) of a traced CTA's per-tile steps over its reached tiles,
    less the first and last quarter, plus the CTA's clock (GHz) and its form
    ("two-tile" or "pipelined", from which events it stamped)."""
    ev = {n: i for i, n in enumerate(ATTN_TRACE_EVENTS)}
    x = tr[cta].astype(np.float64)
    n = int(np.sum(x[ev["v_seen"]] > 0))
    pipelined = not (x[ev["s1_seen"]] > 0).any()
    out = {"tiles": n, "form": "pipelined" if pipelined else "two-tile"}
    c0, t0, c1, t1 = (float(v) for v in clock[cta])
    out["ghz"] = (c1 - c0) / (t1 - t0) if t1 > t0 else float("nan")
    lo, hi = n // 4, n - n // 4
    if hi - lo < 4:
        return out
    r, r1 = slice(lo, hi), slice(lo + 1, hi + 1)

    def g(name, sl=r):
        return x[ev[name], sl]

    def med(v):
        return float(np.median(v))

    if pipelined:
        # issuer per tile n: K(n + 1) seen, S(n + 1) issued, V(n) seen, P(n) seen, P V(n) issued
        out.update({
            "period": med(np.diff(g("v_seen", slice(lo, hi + 1)))),
            "issuer: wait next K": med(g("k_next_seen", r1) - g("pv0_issued")),
            "issuer: issue next S": med(g("s0_next_issued") - g("k_next_seen")),
            "issuer: wait V": med(g("v_seen") - g("wait_v")),
            "issuer: wait P": med(g("p0_seen") - g("v_seen")),
            "issuer: issue P V": med(g("pv0_issued") - g("p0_seen")),
            "softmax: S issued -> seen": med(g("s0_seen", r1) - g("s0_next_issued")),
            "softmax: load scores": med(g("s0_loaded") - g("s0_seen")),
            "softmax: row max": med(g("max0") - g("s0_loaded")),
            "softmax: exp2, P stores": med(g("exp0") - g("max0")),
            "softmax: wait stores, arrive": med(g("p0_arrive") - g("exp0")),
            "softmax: arrive -> issuer sees P": med(g("p0_seen") - g("p0_arrive")),
            "softmax: arrive -> next S seen": med(g("s0_seen", r1) - g("p0_arrive")),
            "V seen - P arrive": med(g("v_seen") - g("p0_arrive")),
        })
        return out
    out.update({
        "period": med(np.diff(g("v_seen", slice(lo, hi + 1)))),
        "issuer: wait V": med(g("v_seen") - g("wait_v")),
        "issuer: wait P0": med(g("p0_seen") - g("v_seen")),
        "issuer: issue P V 0": med(g("pv0_issued") - g("p0_seen")),
        "issuer: wait next K": med(g("k_next_seen") - g("pv0_issued")),
        "issuer: issue next S 0": med(g("s0_next_issued") - g("k_next_seen")),
        "issuer: wait P1": med(g("p1_seen") - g("s0_next_issued")),
        "issuer: issue P V 1": med(g("pv1_issued") - g("p1_seen")),
        "issuer: issue next S 1": med(g("s1_next_issued") - g("pv1_issued")),
        "issuer: to next tile": med(g("wait_v", r1) - g("s1_next_issued")),
    })
    for t in (0, 1):
        nxt = "s0_next_issued" if t == 0 else "s1_next_issued"
        out.update({
            f"softmax {t}: S issued -> seen": med(g(f"s{t}_seen", r1) - g(nxt)),
            f"softmax {t}: load scores": med(g(f"s{t}_loaded") - g(f"s{t}_seen")),
            f"softmax {t}: row max": med(g(f"max{t}") - g(f"s{t}_loaded")),
            f"softmax {t}: exp2, P stores": med(g(f"exp{t}") - g(f"max{t}")),
            f"softmax {t}: wait stores, arrive": med(g(f"p{t}_arrive") - g(f"exp{t}")),
            f"softmax {t}: arrive -> issuer sees P": med(g(f"p{t}_seen") - g(f"p{t}_arrive")),
            f"softmax {t}: arrive -> next S seen": med(g(f"s{t}_seen", r1) - g(f"p{t}_arrive")),
        })
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="mha_causal_spiky_b1_h32_n16384_d128")
    ap.add_argument("--table", action="store_true", help="print every traced tile's stamps")
    args = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("trace_attn needs a GPU")
    _build.build(trace=True)
    load_library(trace=True)
    c = wl.WORKLOADS[args.workload]
    Q, K, V = (t.cuda() for t in wl.prefill_inputs(c))
    for _ in range(3):
        attn_fwd(Q, K, V, causal=c.causal, window=c.window, scale=c.softmax_scale())
    check()
    attn_trace()                                                      # clear the warm-up stamps
    torch.empty(256 << 20, dtype=torch.uint8, device="cuda").zero_()  # L2 flush
    attn_fwd(Q, K, V, causal=c.causal, window=c.window, scale=c.softmax_scale())
    check()
    tr, clock = attn_trace()
    print(f"{c.name}: trace of 4 CTAs")
    for cta in range(tr.shape[0]):
        sm = steady_state_summary(tr, clock, cta)
        if sm["tiles"] == 0:
            print(f"  CTA slot {cta}: not traced")
            continue
        ghz = sm.pop("ghz")
        print(f"  CTA slot {cta}: {sm.pop('form')} form, {sm.pop('tiles')} key tiles, SM clock {ghz:.2f} GHz")
        for k, v in sm.items():
            print(f"    {k:40s} {v:7.0f} cycles {v / ghz / 1000:6.3f} us")
        if args.table:
            x = tr[cta]
            base = clock[cta, 0]
            print("    tile " + " ".join(f"{n:>14s}" for n in ATTN_TRACE_EVENTS))
            for j in range(int(np.sum(x[1] > 0))):
                print(f"    {j:4d} " + " ".join(f"{(int(x[e, j]) - base) if x[e, j] else 0:14d}"
                                          for e in range(len(ATTN_TRACE_EVENTS))))


if __name__ == "__main__":
    main()
