"""GPU checks of the host-buffer entry points (attn_fwd_host, mla_decode_host):
inputs and outputs in host memory, copies and kernels pipelined over chunks of
(batch, KV-head) units or sequences.

attn_fwd_host runs the same kernels on contiguous sub-problems, and every
query row's arithmetic is the same whatever the launch size, so its result is
bit-for-bit that of attn_fwd on device copies.  mla_decode_host splits the
batch, which changes the split-KV partition of the keys, so it is compared
with the fp64 oracle at the usual tolerances."""
import math

import pytest
import torch

import oracle
import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import workloads as wl
from tests._util import build_lib, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()
    gb.load_library()


ATTN = [
    # B, H, H_kv, N_q, N_kv, d, causal, window
    (2, 4, 2, 700, 700, 128, True, 0),
    (1, 2, 1, 300, 2100, 64, False, 0),       # one unit: a single chunk, the two-Q-tile form
    (3, 2, 2, 129, 129, 128, False, 64),      # six units over four chunks, symmetric window
    (4, 16, 16, 256, 256, 128, True, 0),
    (2, 2, 2, 200, 0, 128, False, 0),         # no keys: O = 0, LSE = -inf
]


@pytest.mark.parametrize("case", ATTN, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_attn_host_equals_device_bitwise(case, pinned):
    B, H, H_kv, N_q, N_kv, d, causal, window = case
    Q, K, V = wl.random_prefill(B, H, H_kv, N_q, N_kv, d, seed=500 + N_q + N_kv)
    scale = d ** -0.5
    O_d, L_d = gb.attn_fwd(Q.cuda(), K.cuda(), V.cuda(), causal=causal, window=window, scale=scale)
    gb.check()
    hq, hk, hv = ((t.pin_memory() if pinned else t.clone()) for t in (Q, K, V))
    O_h, L_h = gb.attn_fwd_host(hq, hk, hv, causal=causal, window=window, scale=scale)
    gb.check()
    assert O_h.device.type == "cpu" and L_h.device.type == "cpu"
    assert torch.equal(O_h.view(torch.int16), O_d.cpu().view(torch.int16))
    assert torch.equal(L_h, L_d.cpu())


def test_attn_host_matches_oracle_and_repeats():
    B, H, H_kv, N, d = 2, 8, 2, 500, 128
    Q, K, V = wl.random_prefill(B, H, H_kv, N, N, d, seed=520)
    hq, hk, hv = (t.pin_memory() for t in (Q, K, V))
    buf = torch.empty(gb.attn_fwd_host_device_bytes(B, H, H_kv, N, N, d), dtype=torch.uint8, device="cuda")
    O1, L1 = gb.attn_fwd_host(hq, hk, hv, causal=True, scale=0.1, device_buf=buf)
    gb.check()
    O1, L1 = O1.clone(), L1.clone()
    O2, L2 = gb.attn_fwd_host(hq, hk, hv, causal=True, scale=0.1, device_buf=buf)
    gb.check()
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16)) and torch.equal(L1, L2)
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, True, 0, 0.1)
    compare(O1, L1, O_ref, L_ref, what="attn_fwd_host")


@pytest.mark.parametrize("B,N_kv", [(1, 300), (5, 777), (9, 2048)])
def test_mla_host_matches_oracle(B, N_kv):
    Qn, Qp, KV, Kp = wl.random_mla(B, 128, N_kv, 512, 64, seed=530 + B)
    scale = 1 / math.sqrt(576)
    O, L = gb.mla_decode_host(*(t.pin_memory() for t in (Qn, Qp, KV, Kp)), scale=scale)
    gb.check()
    assert O.device.type == "cpu"
    O_ref, L_ref = oracle.mla_decode(Qn, Qp, KV, Kp, scale)
    compare(O, L, O_ref, L_ref, what=f"mla_decode_host B={B} N_kv={N_kv}")


def test_host_calls_wait_for_earlier_work_on_the_stream():
    # the pipeline's helper streams start only after what the caller queued before
    B, H, N, d = 1, 4, 1024, 128
    Q, K, V = wl.random_prefill(B, H, H, N, N, d, seed=540)
    hq, hk, hv = (t.pin_memory() for t in (Q, K, V))
    buf = torch.zeros(gb.attn_fwd_host_device_bytes(B, H, H, N, N, d), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(50_000_000)            # keep the stream busy (~tens of ms)
        buf.fill_(0xFF)                          # queued work that touches the device buffer
        O, L = gb.attn_fwd_host(hq, hk, hv, causal=True, scale=0.2, device_buf=buf, stream=stream)
    gb.check(stream)
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, True, 0, 0.2)
    compare(O, L, O_ref, L_ref, what="after queued work")
