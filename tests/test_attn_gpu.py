"""GPU parity of attn_fwd (through the C ABI) against the fp64 oracle.

Element-wise on small and medium shapes that span several 128-row / 128-key
tiles and ragged tails; on sampled rows at the full workload sizes, in the
same launch configuration the benchmark times.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import workloads as wl
from tests._util import build_lib, compare, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()
    gb.load_library()


def run_gpu(Q, K, V, causal, window, scale):
    O, LSE = gb.attn_fwd(Q.cuda(), K.cuda(), V.cuda(), causal=causal, window=window, scale=scale)
    gb.check()
    return O, LSE


def test_selftest_tensor_core_layouts():
    g = torch.Generator().manual_seed(5)
    A, B, P, V = (torch.randn(128, 128, generator=g).to(torch.bfloat16) for _ in range(4))
    S, O = gb.selftest_umma(A.cuda(), B.cuda(), P.cuda(), V.cuda())
    gb.check()
    S_ref = A.double() @ B.double().T
    O_ref = P.double() @ V.double()
    assert torch.allclose(S.cpu().double(), S_ref, atol=1e-3, rtol=1e-4), (S.cpu().double() - S_ref).abs().max()
    assert torch.allclose(O.cpu().double(), O_ref, atol=1e-3, rtol=1e-4), (O.cpu().double() - O_ref).abs().max()


SMALL = [
    # B, H, H_kv, N_q, N_kv, d, causal, window
    (1, 1, 1, 128, 128, 128, False, 0),
    (1, 2, 2, 128, 128, 64, False, 0),
    (1, 1, 1, 256, 256, 128, True, 0),
    (2, 4, 2, 300, 300, 128, True, 0),
    (1, 2, 1, 77, 77, 64, True, 0),
    (1, 2, 2, 200, 333, 128, False, 0),
    (1, 2, 2, 200, 333, 128, True, 0),      # bottom-right causal, N_q < N_kv
    (1, 2, 2, 333, 200, 64, True, 0),       # N_q > N_kv: the first rows see no key
    (1, 4, 1, 513, 513, 128, True, 1),
    (1, 2, 2, 700, 700, 128, True, 127),
    (1, 2, 2, 700, 700, 64, True, 128),
    (1, 2, 2, 700, 700, 128, True, 129),
    (1, 2, 2, 700, 700, 128, True, 256),
    (1, 2, 2, 650, 650, 128, True, 650),    # window = N: same as causal
    # the one-tile form runs on 64-key tiles: windows and lengths at its tile edges
    (1, 2, 2, 700, 700, 128, True, 63),
    (1, 2, 2, 700, 700, 64, True, 64),
    (1, 2, 2, 700, 700, 128, True, 65),
    (1, 2, 1, 64, 64, 128, True, 0),
    (1, 2, 2, 65, 65, 128, False, 0),
    (1, 2, 2, 191, 191, 64, False, 0),
    (1, 2, 2, 600, 600, 128, False, 63),    # symmetric
    (1, 1, 1, 1, 1, 128, False, 0),
    (1, 1, 1, 1, 1000, 64, True, 0),
    (3, 8, 8, 130, 1, 128, False, 0),
    (1, 1, 1, 1030, 1030, 128, False, 0),
    # symmetric local window (causal = 0, window > 0): |j - (i + N_kv - N_q)| <= window
    (1, 2, 2, 500, 500, 128, False, 64),
    (1, 2, 1, 333, 333, 64, False, 1),
    (1, 2, 2, 200, 700, 128, False, 100),   # N_q < N_kv
    (1, 2, 2, 700, 200, 128, False, 50),    # N_q > N_kv: the first rows see no key
    (2, 4, 2, 1030, 1030, 128, False, 300),
    (1, 2, 2, 400, 400, 64, False, 400),    # window >= N: unmasked
    # rows that visit >= 16 key tiles on average: the two-Q-tile form
    (1, 2, 2, 300, 2100, 128, False, 0),
    (1, 2, 2, 300, 2100, 64, False, 0),
    (2, 2, 1, 257, 3000, 128, True, 0),     # bottom-right causal, ragged query block
    (1, 2, 2, 2400, 2400, 128, False, 1300),  # symmetric window
    (1, 1, 1, 640, 4200, 64, True, 0),
    (1, 2, 1, 64, 16384, 128, False, 0),     # few queries, very long keys
    (1, 2, 2, 100, 9000, 128, True, 0),      # bottom-right causal: every row sees ~8900 keys
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_parity_small(case):
    B, H, H_kv, N_q, N_kv, d, causal, window = case
    Q, K, V = wl.random_prefill(B, H, H_kv, N_q, N_kv, d, seed=hash(case) & 0xffff)
    scale = 1 / math.sqrt(d)
    O, LSE = run_gpu(Q, K, V, causal, window, scale)
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, causal, window, scale)
    compare(O, LSE, O_ref, L_ref, what=str(case))


def test_large_scores_force_rescaling():
    # Keys that grow along the sequence move the running maximum on every tile.
    B, H, N, d = 1, 2, 1024, 128
    Q, K, V = wl.random_prefill(B, H, H, N, N, d, seed=77)
    ramp = torch.linspace(0.2, 6.0, N).view(1, 1, N, 1)
    K = (K.float() * ramp).to(torch.bfloat16)
    for causal in (False, True):
        O, LSE = run_gpu(Q, K, V, causal, 0, 1 / math.sqrt(d))
        O_ref, L_ref = oracle.attn_fwd(Q, K, V, causal, 0, 1 / math.sqrt(d))
        compare(O, LSE, O_ref, L_ref, what=f"ramp causal={causal}")


def test_empty_sequences():
    Q = torch.randn(1, 2, 5, 64).to(torch.bfloat16).cuda()
    K = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    O, LSE = gb.attn_fwd(Q, K, K.clone(), causal=False)
    gb.check()
    assert (O.float() == 0).all() and torch.isneginf(LSE).all()
    Q0 = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    K1 = torch.randn(1, 2, 7, 64).to(torch.bfloat16).cuda()
    O, LSE = gb.attn_fwd(Q0, K1, K1, causal=True)
    gb.check()
    assert O.numel() == 0


def test_deterministic():
    Q, K, V = wl.random_prefill(2, 4, 2, 640, 640, 128, seed=3)
    Qc, Kc, Vc = Q.cuda(), K.cuda(), V.cuda()
    O1, L1 = gb.attn_fwd(Qc, Kc, Vc, causal=True)
    O2, L2 = gb.attn_fwd(Qc, Kc, Vc, causal=True)
    gb.check()
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16)) and torch.equal(L1, L2)


def _workload_parity(name, n_random, full=False):
    c = wl.WORKLOADS[name]
    Q, K, V = wl.prefill_inputs(c)
    O, LSE = run_gpu(Q, K, V, c.causal, c.window, c.softmax_scale())
    if full:
        O_ref, L_ref = oracle.attn_fwd(Q, K, V, c.causal, c.window, c.softmax_scale())
        return compare(O, LSE, O_ref, L_ref, what=name)
    rows = sample_rows(c.B, c.H, c.N_q, n_random, seed=c.seed)
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, c.causal, c.window, c.softmax_scale(), rows=rows)
    Og = O.reshape(-1, c.d)[torch.as_tensor(rows, device=O.device)]
    Lg = LSE.reshape(-1)[torch.as_tensor(rows, device=O.device)]
    return compare(Og, Lg, O_ref, L_ref, what=name)


def test_workload_mha_small_full():
    _workload_parity("mha_b1_h2_n128_d64", 0, full=True)


def test_workload_mha_causal_2k_full():
    _workload_parity("mha_causal_b4_h16_n2048_d128", 0, full=True)


FULL_SIZE = ["gqa_causal_b2_h32_hkv8_n8192_d128",
             "gqa_window256_b2_h32_hkv8_n8192_d128",
             "gqa_swindow256_b2_h32_hkv8_n8192_d128",
             "mha_causal_spiky_b1_h32_n16384_d128"]


@pytest.mark.parametrize("name", FULL_SIZE)
def test_workload_sampled(name):
    _workload_parity(name, 160)


@pytest.mark.parametrize("name", FULL_SIZE)
def test_workload_complete_heads(name):
    # Every row of two whole (batch, head) pairs of the full-size launch: the
    # last head, whose shortest query blocks are the last CTAs of the
    # longest-first order, and one in the middle of the grid.
    c = wl.WORKLOADS[name]
    Q, K, V = wl.prefill_inputs(c)
    O, LSE = run_gpu(Q, K, V, c.causal, c.window, c.softmax_scale())
    heads = [c.B * c.H - 1, (c.B * c.H) // 2 + 1]
    rows = np.concatenate([np.arange(bh * c.N_q, (bh + 1) * c.N_q, dtype=np.int64) for bh in heads])
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, c.causal, c.window, c.softmax_scale(), rows=rows)
    idx = torch.as_tensor(rows, device=O.device)
    compare(O.reshape(-1, c.d)[idx], LSE.reshape(-1)[idx], O_ref, L_ref, what=f"{name} heads {heads}")
