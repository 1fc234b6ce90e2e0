"""GPU parity of attn_fwd_sparse (block-sparse mask of 128 x 128 blocks,
through the C ABI) against the fp64 oracle: random masks with and without
causal / window, one query tile of a CTA masked out while the other is not,
empty masks, an all-ones mask against attn_fwd, determinism and a sampled long
causal GQA case."""
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


def run(Q, K, V, mask, causal, window, scale):
    O, LSE = gb.attn_fwd_sparse(Q.cuda(), K.cuda(), V.cuda(), mask.cuda(), causal=causal, window=window, scale=scale)
    gb.check()
    return O, LSE


CASES = [
    # B, H, H_kv, N_q, N_kv, d, causal, window, density
    (1, 2, 2, 512, 512, 128, False, 0, 0.5),
    (2, 4, 2, 700, 900, 128, True, 0, 0.4),
    (1, 2, 1, 1030, 1030, 64, False, 0, 0.3),
    (1, 4, 4, 640, 640, 128, True, 256, 0.6),
    (1, 2, 2, 512, 700, 128, False, 100, 0.5),     # symmetric window and blocks
    (1, 2, 2, 300, 300, 128, False, 0, 0.0),       # nothing to attend to
    (1, 1, 1, 2000, 2000, 128, True, 0, 0.15),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_parity(case):
    B, H, H_kv, N_q, N_kv, d, causal, window, density = case
    Q, K, V = wl.random_prefill(B, H, H_kv, N_q, N_kv, d, seed=hash(case[:8]) & 0xffff)
    mask = wl.random_block_mask(B, H, N_q, N_kv, density, seed=(hash(case[:8]) + 1) & 0xffff)
    scale = d ** -0.5
    O, LSE = run(Q, K, V, mask, causal, window, scale)
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, causal, window, scale, block_mask=mask)
    compare(O, LSE, O_ref, L_ref, what=str(case))


def test_one_query_tile_of_a_cta_masked_out():
    # query blocks 0/1 share a CTA (256 rows): block 0 masked out entirely, 1 dense;
    # blocks 2/3: block 3 masked out, 2 half dense
    B, H, N, d = 1, 2, 512, 128
    Q, K, V = wl.random_prefill(B, H, H, N, N, d, seed=60)
    mask = torch.ones(B, H, 4, 4, dtype=torch.uint8)
    mask[:, :, 0] = 0
    mask[:, :, 3] = 0
    mask[:, :, 2, ::2] = 0
    O, LSE = run(Q, K, V, mask, False, 0, d ** -0.5)
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, False, 0, d ** -0.5, block_mask=mask)
    compare(O, LSE, O_ref, L_ref, what="half-masked CTAs")


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_is_attn_fwd(causal):
    # An all-ones mask removes nothing: the block-sparse kernel (128-key tiles)
    # computes the dense attention.  attn_fwd runs these short rows in its
    # pipelined 64-key form, so the two round differently: each is held to the
    # oracle, and to the other within twice the bar.
    Q, K, V = wl.random_prefill(2, 4, 2, 777, 777, 128, seed=61)
    mask = torch.ones(2, 4, 7, 7, dtype=torch.uint8)
    O1, L1 = gb.attn_fwd(Q.cuda(), K.cuda(), V.cuda(), causal=causal, scale=0.1)
    gb.check()
    O2, L2 = run(Q, K, V, mask, causal, 0, 0.1)
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, causal, 0, 0.1)
    compare(O1, L1, O_ref, L_ref, what="dense")
    compare(O2, L2, O_ref, L_ref, what="all-ones mask")
    compare(O2, L2, O1.float().cpu().double().numpy(), L1.cpu().double().numpy(), o_tol=4e-2, lse_tol=2e-3,
            what="all-ones mask against dense")


def test_deterministic():
    Q, K, V = wl.random_prefill(1, 4, 2, 1500, 1500, 128, seed=62)
    mask = wl.random_block_mask(1, 4, 1500, 1500, 0.5, seed=63)
    O1, L1 = run(Q, K, V, mask, True, 0, 0.1)
    O2, L2 = run(Q, K, V, mask, True, 0, 0.1)
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L1, L2)


def test_long_causal_gqa_sampled():
    c = wl.WORKLOADS["gqa_causal_b2_h32_hkv8_n8192_d128"]
    Q, K, V = wl.prefill_inputs(c)
    mask = wl.random_block_mask(c.B, c.H, c.N_q, c.N_kv, 0.25, seed=wl.SEED_BASE + 6)
    O, LSE = run(Q, K, V, mask, True, 0, c.softmax_scale())
    rows = sample_rows(c.B, c.H, c.N_q, 120, seed=64)
    O_ref, L_ref = oracle.attn_fwd(Q, K, V, True, 0, c.softmax_scale(), rows=rows, block_mask=mask)
    idx = torch.as_tensor(rows, device=O.device)
    compare(O.reshape(-1, c.d)[idx], LSE.reshape(-1)[idx], O_ref, L_ref, what="8k causal GQA, 25 % blocks")
