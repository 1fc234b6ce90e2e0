"""Bounded waits end in an error status, not a hang.

The fault is made without faulting the GPU: with injection mode 1 the prefill
kernel's producer never loads the Q tiles, so the tensor-core warp's bounded
wait for them runs out (limit set to 20 ms here); with mode 2 the SSD scan's
producer loads no chunk, so every role's wait runs out.  The kernel must stop,
free its tensor memory and return; gbattn_check() must report
GBATTN_ERR_TIMEOUT; and the next normal call must work and match the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import workloads as wl
from tests._util import build_lib, compare

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    build_lib()
    gb.load_library()
    Q, K, V = wl.random_prefill(1, 1, 1, 256, 256, 128, seed=31)   # one CTA
    Qc, Kc, Vc = Q.cuda(), K.cuda(), V.cuda()
    gb.check()
    old_timeout = gb.set_wait_timeout_ns(20_000_000)
    gb.set_fault_injection(1)
    try:
        gb.attn_fwd(Qc, Kc, Vc, causal=True)
        with pytest.raises(gb.GbattnError) as e:
            gb.check()
        assert e.value.code == 6
    finally:
        gb.set_fault_injection(0)
        gb.set_wait_timeout_ns(old_timeout)
    gb.check()                                   # status word was cleared
    O, LSE = gb.attn_fwd(Qc, Kc, Vc, causal=True)
    gb.check()
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, True, 0, 1 / math.sqrt(128))
    compare(O, LSE, O_ref, L_ref, what="after timeout")


def test_ssd_wait_timeout_is_reported_and_context_survives():
    build_lib()
    gb.load_library()
    x, dt, A, B, C, D = (t.cuda() for t in wl.random_ssd(1, 300, 2, 64, 1, 128, seed=32))
    gb.check()
    old_timeout = gb.set_wait_timeout_ns(20_000_000)
    gb.set_fault_injection(2)
    try:
        gb.ssd_scan(x, dt, A, B, C, D)
        with pytest.raises(gb.GbattnError) as e:
            gb.check()
        assert e.value.code == 6
    finally:
        gb.set_fault_injection(0)
        gb.set_wait_timeout_ns(old_timeout)
    gb.check()
    y, S = gb.ssd_scan(x, dt, A, B, C, D, want_final_state=True)
    gb.check()
    y_ref, S_ref = oracle.ssd_scan(x.cpu(), dt.cpu(), A.cpu(), B.cpu(), C.cpu(), D.cpu())
    y_abs, _ = oracle.ssd_scan(x.cpu().abs(), dt.cpu(), A.cpu(), B.cpu().abs(), C.cpu().abs(), D.cpu().abs())
    err = np.abs(y.cpu().double().numpy() - y_ref) - (2.0 ** -7 * y_abs + 1e-6)
    assert err.max() <= 0
