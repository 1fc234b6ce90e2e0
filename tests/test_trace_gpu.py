"""The MLA decode latency trace: the trace build (-DGBATTN_TRACE) computes
bit-identical results to the default library and stamps every step of each
traced tile's chain in the order the kernel's dependencies force."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import workloads as wl
from tests._util import build_lib

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
B, N_KV, SCALE = 8, 4096, 576 ** -0.5

# Runs in a process of its own: the trace build exports the same symbols as the
# default library, which this test process has loaded.
CHILD = f"""
import sys, numpy as np, torch
sys.path.insert(0, {ROOT!r})
import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import _build, workloads as wl
_build.build(trace=True)
gb.load_library(trace=True)
x = [t.cuda() for t in wl.random_mla({B}, 128, {N_KV}, 512, 64, seed=11)]
gb.mla_decode(*x, scale={SCALE!r}); gb.check(); gb.mla_trace()
O, L = gb.mla_decode(*x, scale={SCALE!r}); gb.check()
tr = gb.mla_trace()
np.savez(sys.argv[1], O=O.view(torch.int16).cpu().numpy(), L=L.cpu().numpy(), tr=tr)
"""


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()
    gb.load_library()


def test_default_library_reports_unsupported():
    with pytest.raises(gb.GbattnError) as e:
        gb.mla_trace()
    assert e.value.code == 2


def test_trace_build_matches_and_stamps_in_order(tmp_path):
    out = str(tmp_path / "trace.npz")
    r = subprocess.run([sys.executable, "-c", CHILD, out], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    d = np.load(out)
    x = [t.cuda() for t in wl.random_mla(B, 128, N_KV, 512, 64, seed=11)]
    O, L = gb.mla_decode(*x, scale=SCALE)
    gb.check()
    assert np.array_equal(d["O"], O.view(torch.int16).cpu().numpy())
    assert np.array_equal(d["L"], L.cpu().numpy())
    tr = d["tr"].astype(np.int64)
    ev = {n: i for i, n in enumerate(gb.MLA_TRACE_EVENTS)}
    reached = np.all(tr > 0, axis=(0, 1))
    n = int(np.argmin(reached)) if not reached.all() else tr.shape[2]
    # the traced cluster's range: about B * 64 / 76 tiles, every step of each reached
    assert n >= 5
    assert not (tr[:, :, n:] > 0).any()
    for c in range(2):
        p = 1 - c
        s = lambda e: tr[c, ev[e], :n]
        assert (s("load") < s("s_issue")).all()            # S waits for the tile's data
        assert (s("s_issue") < s("s_read")).all()          # ... and is read after it completes
        assert (s("s_read") <= s("send_buf0_free")).all()
        for h in (0, 1):
            assert (s(f"send_buf{h}_free") <= s(f"copy{h}_issue")).all()
            # the softmax has a unit only after both CTAs' copies of it were issued
            assert (s(f"copy{h}_issue") <= s(f"softmax{h}_in")).all()
            assert (tr[p, ev[f"copy{h}_issue"], :n] <= s(f"softmax{h}_in")).all()
            assert (s(f"softmax{h}_in") <= s(f"p{h}_ready")).all()
            assert (s(f"p{h}_ready") <= s(f"pv{h}_issue")).all()   # P V waits for P
        assert (np.diff(s("s_issue")) > 0).all()           # tiles in order
