"""Latency trace of the MLA decode kernel on the GPU (observability tool).

    python -m tiled_attention_flashattention_gb300.trace_mla [--table] [--B 64] [--N_kv 4096]

Builds the library's trace variant (``libgbattn_trace.so``: the same sources
with -DGBATTN_TRACE), runs mla_decode on seeded inputs of the given shape (128
heads, d_c 512, d_r 64) after three warm-up calls and an L2 flush, and reads
the per-tile event stamps of one cluster (``gbattn_mla_trace``).  It prints the
median, over the steady-state tiles, of each step of a tile's chain for both
CTAs of the cluster: the tile period, the load latency (load issued -> S
issued), the score MMA (S issued -> S read), the wait for a send buffer, the
exchange (the peer's copy issued -> this CTA's softmax has the unit), a
softmax unit, P ready -> P·V issued, and a ring slot's cycle (load of tile t ->
load of tile t + 4).  ``--table`` also prints every tile's stamps.

Runs in a process of its own: the trace build and the default library export
the same symbols and are not loaded together.
"""
from __future__ import annotations

import argparse
import math

import numpy as np
import torch

from . import _build
from . import load_library, mla_decode, mla_trace, check, MLA_TRACE_EVENTS
from . import workloads as wl


def steady_state_summary(tr: np.ndarray, ring_stages: int = 4) -> dict:
    """Medians (us) of the chain's steps over the tiles both CTAs reached, less
    the first and last quarter (start-up and drain)."""
    ev = {n: i for i, n in enumerate(MLA_TRACE_EVENTS)}
    x = tr.astype(np.float64) / 1000.0
    reached = np.all(tr > 0, axis=(0, 1))
    n = int(np.argmin(reached)) if not reached.all() else tr.shape[2]
    lo, hi = n // 4, n - n // 4
    out = {"tiles_traced": n}
    if hi - lo < 2:
        return out
    t = np.arange(lo, hi)

    def med(v):
        return float(np.median(v))

    for r in range(2):
        p = 1 - r
        d = {
            "tile_period": med(np.diff(x[r, ev["s_read"], lo:hi])),
            "load_to_s_issue": med(x[r, ev["s_issue"], t] - x[r, ev["load"], t]),
            "s_issue_to_s_read": med(x[r, ev["s_read"], t] - x[r, ev["s_issue"], t]),
            "s_read_to_send_buf_free": med(x[r, ev["send_buf0_free"], t] - x[r, ev["s_read"], t]),
            "peer_copy_to_softmax": med(x[r, ev["softmax0_in"], t] - x[p, ev["copy0_issue"], t]),
            "softmax_unit": med(x[r, ev["p0_ready"], t] - x[r, ev["softmax0_in"], t]),
            "p_ready_to_pv_issue": med(x[r, ev["pv0_issue"], t] - x[r, ev["p0_ready"], t]),
        }
        tt = t[t + ring_stages < n]
        if len(tt):
            d["ring_slot_cycle"] = med(x[r, ev["load"], tt + ring_stages] - x[r, ev["load"], tt])
        out[f"cta{r}"] = d
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--B", type=int, default=64)
    ap.add_argument("--N_kv", type=int, default=4096)
    ap.add_argument("--table", action="store_true", help="print every traced tile's stamps")
    args = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("trace_mla needs a GPU")
    _build.build(trace=True)
    load_library(trace=True)
    dev = torch.device("cuda", 0)
    Qn, Qp, KV, Kp = (t.to(dev) for t in wl.random_mla(args.B, 128, args.N_kv, 512, 64, seed=7))
    scale = 1.0 / math.sqrt(576)
    for _ in range(3):
        mla_decode(Qn, Qp, KV, Kp, scale=scale)
    check()
    mla_trace()                                             # clear the warm-up stamps
    torch.empty(256 << 20, dtype=torch.uint8, device=dev).zero_()   # L2 flush
    mla_decode(Qn, Qp, KV, Kp, scale=scale)
    check()
    tr = mla_trace()
    summary = steady_state_summary(tr)
    print(f"MLA decode B={args.B} H=128 N_kv={args.N_kv}: {summary['tiles_traced']} tiles traced")
    for r in (0, 1):
        if f"cta{r}" in summary:
            print(f"  CTA {r}: " + ", ".join(f"{k} {v:.2f} us" for k, v in summary[f"cta{r}"].items()))
    if args.table:
        t0 = tr[tr > 0].min()
        for r in range(2):
            print(f"CTA {r} (us from the first stamp): tile " + " ".join(f"{n:>14s}" for n in MLA_TRACE_EVENTS))
            for i in range(summary["tiles_traced"]):
                print(f"  {i:3d} " + " ".join(f"{(int(tr[r, e, i]) - int(t0)) / 1000:14.2f}"
                                              for e in range(len(MLA_TRACE_EVENTS))))


if __name__ == "__main__":
    main()
