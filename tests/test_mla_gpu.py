"""GPU parity of mla_decode (through the C ABI) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import workloads as wl
from tests._util import build_lib, compare

pytestmark = pytest.mark.gpu

SCALE = 1 / math.sqrt(576)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()
    gb.load_library()


def run(Qn, Qp, KV, Kp, scale=SCALE):
    O, LSE = gb.mla_decode(Qn.cuda(), Qp.cuda(), KV.cuda(), Kp.cuda(), scale=scale)
    gb.check()
    return O, LSE


@pytest.mark.parametrize("B,N_kv", [(1, 1), (1, 63), (1, 64), (1, 65), (2, 300), (3, 1000), (1, 4096),
                                    (1, 20000), (5, 777), (160, 64), (200, 130)])
def test_parity(B, N_kv):
    Qn, Qp, KV, Kp = wl.random_mla(B, 128, N_kv, 512, 64, seed=B * 100003 + N_kv)
    O, LSE = run(Qn, Qp, KV, Kp)
    O_ref, L_ref = oracle.mla_decode(Qn, Qp, KV, Kp, SCALE)
    compare(O, LSE, O_ref, L_ref, what=f"B={B} N_kv={N_kv}")


@pytest.mark.parametrize("H,B,N_kv", [(64, 3, 1000), (32, 70, 200), (16, 2, 4097), (100, 5, 777), (1, 4, 300),
                                      (64, 1, 20000)])
def test_fewer_heads(H, B, N_kv):
    # H < 128: the heads fill the first H rows of the 128-row tile, the rest read
    # as zero and are not written
    Qn, Qp, KV, Kp = wl.random_mla(B, H, N_kv, 512, 64, seed=H * 1000 + B * 7 + N_kv)
    O, LSE = run(Qn, Qp, KV, Kp)
    O_ref, L_ref = oracle.mla_decode(Qn, Qp, KV, Kp, SCALE)
    compare(O, LSE, O_ref, L_ref, what=f"H={H} B={B} N_kv={N_kv}")


def test_large_scores_force_rescaling():
    # Ramp the RoPE keys (they enter the scores only, not the values): the row
    # maximum keeps moving along the sequence while V stays N(0, 1).
    B, N_kv = 2, 2048
    Qn, Qp, KV, Kp = wl.random_mla(B, 128, N_kv, 512, 64, seed=9)
    ramp = torch.linspace(0.5, 10.0, N_kv).view(1, N_kv, 1)
    Kp = (Kp.float() * ramp).to(torch.bfloat16)
    O, LSE = run(Qn, Qp, KV, Kp)
    O_ref, L_ref = oracle.mla_decode(Qn, Qp, KV, Kp, SCALE)
    compare(O, LSE, O_ref, L_ref, what="ramp")


def test_deterministic():
    Qn, Qp, KV, Kp = (x.cuda() for x in wl.random_mla(7, 128, 999, 512, 64, seed=4))
    O1, L1 = gb.mla_decode(Qn, Qp, KV, Kp)
    O2, L2 = gb.mla_decode(Qn, Qp, KV, Kp)
    gb.check()
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16)) and torch.equal(L1, L2)


def test_workspace_too_small_is_rejected():
    Qn, Qp, KV, Kp = (x.cuda() for x in wl.random_mla(3, 128, 1000, 512, 64, seed=5))
    need = gb.mla_decode_workspace_bytes(3, 128, 1000)
    assert need > 0
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gb.GbattnError) as e:
        gb.mla_decode(Qn, Qp, KV, Kp, workspace=ws)
    assert e.value.code == 4


def test_workload_full_size_sampled():
    c = wl.WORKLOADS["mla_decode_b64_h128_nkv4096"]
    Qn, Qp, KV, Kp = wl.mla_inputs(c)
    O, LSE = run(Qn, Qp, KV, Kp, c.softmax_scale())
    g = np.random.default_rng(c.seed)
    rows = np.unique(np.concatenate([np.arange(0, 128), np.arange(63 * 128, 64 * 128),
                                     g.integers(0, 64 * 128, size=256)]))
    O_ref, L_ref = oracle.mla_decode(Qn, Qp, KV, Kp, c.softmax_scale(), rows=rows)
    idx = torch.as_tensor(rows, device=O.device)
    compare(O.reshape(-1, 512)[idx], LSE.reshape(-1)[idx], O_ref, L_ref, what=c.name)
