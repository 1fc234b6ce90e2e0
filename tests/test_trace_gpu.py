"""The latency traces of the MLA decode kernel and of the prefill kernel's
two-tile form: the trace build (-DGBATTN_TRACE) computes bit-identical results
to the default library and stamps every step of each traced tile's chain in the
order the kernel's dependencies force."""
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


# Prefill: causal, N = 4096, two heads -> the two-tile form (a 128-row query
# tile visits 16.5 key tiles on average), grid 32, traced blocks 0, 1, 10, 21.
PN, PH = 4096, 2
CHILD_ATTN = f"""
import sys, numpy as np, torch
sys.path.insert(0, {ROOT!r})
import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import _build, workloads as wl
_build.build(trace=True)
gb.load_library(trace=True)
Q, K, V = (t.cuda() for t in wl.random_prefill(1, {PH}, {PH}, {PN}, {PN}, 128, seed=12))
gb.attn_fwd(Q, K, V, causal=True, scale=0.088); gb.check(); gb.attn_trace()
O, L = gb.attn_fwd(Q, K, V, causal=True, scale=0.088); gb.check()
tr, clock = gb.attn_trace()
np.savez(sys.argv[1], O=O.view(torch.int16).cpu().numpy(), L=L.cpu().numpy(), tr=tr, clock=clock)
"""


def test_default_library_reports_unsupported_attn():
    with pytest.raises(gb.GbattnError) as e:
        gb.attn_trace()
    assert e.value.code == 2


def test_attn_trace_build_matches_and_stamps_in_order(tmp_path):
    out = str(tmp_path / "trace_attn.npz")
    r = subprocess.run([sys.executable, "-c", CHILD_ATTN, out], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    d = np.load(out)
    Q, K, V = (t.cuda() for t in wl.random_prefill(1, PH, PH, PN, PN, 128, seed=12))
    O, L = gb.attn_fwd(Q, K, V, causal=True, scale=0.088)
    gb.check()
    assert np.array_equal(d["O"], O.view(torch.int16).cpu().numpy())
    assert np.array_equal(d["L"], L.cpu().numpy())
    tr, clock = d["tr"], d["clock"]
    ev = {n: i for i, n in enumerate(gb.ATTN_TRACE_EVENTS)}
    # blocks 0 / 1 / 10 / 21 take 256-row query blocks 15 / 15 / 10 / 5 (longest
    # first over the two heads): 32 / 32 / 22 / 12 key tiles
    for cta, ntile in enumerate((32, 32, 22, 12)):
        x = tr[cta]
        assert clock[cta, 2] > clock[cta, 0] and clock[cta, 3] > clock[cta, 1]
        n = int(np.sum(x[ev["v_seen"]] > 0))
        assert n == ntile, (cta, n)
        s = lambda e, a=0, b=None: x[ev[e], a:(n if b is None else b)]
        assert (np.diff(s("v_seen")) > 0).all()              # tiles in order
        assert (s("wait_v") <= s("v_seen")).all()
        assert (s("v_seen", 0, n - 1) <= s("p0_seen", 0, n - 1)).all()
        for t in (0, 1):
            # Q tile 0 of a causal two-tile block ends one key tile before Q tile 1
            m = n - 1 if t == 0 else n
            assert (s(f"s{t}_seen", 0, m) <= s(f"s{t}_loaded", 0, m)).all()
            assert (s(f"s{t}_loaded", 0, m) <= s(f"max{t}", 0, m)).all()
            assert (s(f"max{t}", 0, m) <= s(f"exp{t}", 0, m)).all()
            assert (s(f"exp{t}", 0, m) <= s(f"p{t}_arrive", 0, m)).all()
            # the issuer sees P only after the softmax's arrive, then issues P V
            assert (s(f"p{t}_arrive", 0, m) <= s(f"p{t}_seen", 0, m)).all()
            assert (s(f"p{t}_seen", 0, m) <= s(f"pv{t}_issued", 0, m)).all()
            # the softmax sees the next tile's S only after the issuer issued it
            nxt = "s0_next_issued" if t == 0 else "s1_next_issued"
            assert (s(nxt, 0, m - 1) <= s(f"s{t}_seen", 1, m)).all()


# Prefill, pipelined one-tile form: causal N = 1024, two heads (a query tile
# visits 4.5 key tiles of 128 on average), grid 16, traced blocks 0, 1, 5, 10.
def test_attn_trace_pipelined_form_stamps_in_order(tmp_path):
    out = str(tmp_path / "trace_pipe.npz")
    child = CHILD_ATTN.replace(f"{PN}, {PN}, 128, seed=12", "1024, 1024, 128, seed=13")
    assert child != CHILD_ATTN
    r = subprocess.run([sys.executable, "-c", child, out], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    d = np.load(out)
    Q, K, V = (t.cuda() for t in wl.random_prefill(1, PH, PH, 1024, 1024, 128, seed=13))
    O, L = gb.attn_fwd(Q, K, V, causal=True, scale=0.088)
    gb.check()
    assert np.array_equal(d["O"], O.view(torch.int16).cpu().numpy())
    assert np.array_equal(d["L"], L.cpu().numpy())
    tr = d["tr"]
    ev = {n: i for i, n in enumerate(gb.ATTN_TRACE_EVENTS)}
    # blocks 0 / 1 / 5 / 10 take 128-row query blocks 7 / 7 / 5 / 2: 16 / 16 / 12 / 6
    # key tiles of 64; one Q tile, so no Q tile 1 events
    for cta, ntile in enumerate((16, 16, 12, 6)):
        x = tr[cta]
        n = int(np.sum(x[ev["v_seen"]] > 0))
        assert n == ntile, (cta, n)
        for e in ("p1_seen", "pv1_issued", "s1_next_issued", "s1_seen", "p1_arrive"):
            assert not (x[ev[e]] > 0).any()
        s = lambda e, a=0, b=None: x[ev[e], a:(n if b is None else b)]
        assert (np.diff(s("v_seen")) > 0).all()
        assert (s("wait_v") <= s("v_seen")).all()
        assert (s("s0_seen") <= s("s0_loaded")).all()
        assert (s("s0_loaded") <= s("max0")).all()
        assert (s("max0") <= s("exp0")).all()
        assert (s("exp0") <= s("p0_arrive")).all()
        assert (s("p0_arrive") <= s("p0_seen")).all()
        assert (s("p0_seen") <= s("pv0_issued")).all()
        # S of tile n + 1 is issued once its K landed and then seen by the softmax
        # (before or after P V of tile n, whichever had its inputs first)
        assert (s("k_next_seen", 0, n - 1) <= s("s0_next_issued", 0, n - 1)).all()
        assert (s("s0_next_issued", 0, n - 1) <= s("s0_seen", 1, n)).all()
        # and not before P V of tile n - 1 (it overwrites that P's buffer)
        assert (s("pv0_issued", 0, n - 2) <= s("s0_next_issued", 1, n - 1)).all()

