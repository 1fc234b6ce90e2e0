"""Pins for the fp64 oracle, against things other than the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong mask offset, a missing
max subtraction, log base 2 instead of e) fails at least one of them:

* hand-worked cases with closed-form answers (tests/golden/*.json);
* invariants: probability rows sum to 1, constant value rows come back
  unchanged, unmasked attention is invariant to a joint permutation of keys
  and values, a per-row score shift leaves O unchanged and moves LSE by it;
* closed forms: uniform scores give the mean of the visible value rows and
  LSE = ln(count);
* reductions to library routines: torch's fp64 scaled_dot_product_attention,
  torch.logsumexp, repeat_interleave for GQA;
* structural identities of the masks (window >= N is causal, a symmetric
  window >= N is unmasked; bottom-right causal rows are the tail rows of the
  square problem); the symmetric window equals torch's fp64 attention with an
  explicit band mask;
* an independent fp64 implementation of the online (block-by-block)
  recurrence, and the exact log-sum-exp merge of two key halves.
"""
import glob
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_flashattention_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-12


def bf(x):
    return torch.tensor(x, dtype=torch.float64).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64)


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "*.json"))))
def test_golden_fixture(path):
    c = json.load(open(path))
    if c["kind"] == "attn":
        O, LSE, P = oracle.attn_fwd(bf(c["Q"]), bf(c["K"]), bf(c["V"]), c["causal"], c["window"],
                                    c["scale"], return_probs=True)
        if "expect_P" in c:
            np.testing.assert_allclose(P, np.array(c["expect_P"]), atol=TOL, rtol=0)
    else:
        O, LSE = oracle.mla_decode(bf(c["Q_nope"]), bf(c["Q_pe"]), bf(c["KV_latent"]), bf(c["K_pe"]),
                                   c["scale"])
    np.testing.assert_allclose(O, np.array(c["expect_O"]), atol=TOL, rtol=0)
    np.testing.assert_allclose(LSE, np.array(c["expect_LSE"]), atol=TOL, rtol=0)


def test_single_key_returns_its_value():
    Q, K, V = wl.random_prefill(2, 3, 3, 5, 1, 16, seed=1)
    scale = 0.37
    O, LSE = oracle.attn_fwd(Q, K, V, False, 0, scale)
    np.testing.assert_allclose(O, f64(V).expand(2, 3, 5, 16).numpy(), atol=TOL, rtol=0)
    dots = torch.einsum("bhid,bhjd->bhij", f64(Q), f64(K))[..., 0] * scale
    np.testing.assert_allclose(LSE, dots.numpy(), atol=1e-10, rtol=0)


def test_window_one_sees_only_its_own_key():
    # causal window 1 keeps key j = i only: O_i = V_i and LSE_i = scale q_i . k_i
    Q, K, V = wl.random_prefill(1, 2, 2, 9, 9, 16, seed=2)
    scale = 0.29
    O, LSE = oracle.attn_fwd(Q, K, V, True, 1, scale)
    np.testing.assert_allclose(O, f64(V).numpy(), atol=TOL, rtol=0)
    dots = torch.einsum("bhid,bhid->bhi", f64(Q), f64(K)) * scale
    np.testing.assert_allclose(LSE, dots.numpy(), atol=1e-10, rtol=0)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 3), (False, 2)])
def test_probability_rows_sum_to_one(causal, window):
    Q, K, V = wl.random_prefill(1, 2, 1, 9, 9, 8, seed=2)
    _, _, P = oracle.attn_fwd(Q, K, V, causal, window, 0.5, return_probs=True)
    np.testing.assert_allclose(P.sum(-1), 1.0, atol=TOL, rtol=0)
    assert (P >= 0).all()
    if causal:
        i, j = np.meshgrid(np.arange(9), np.arange(9), indexing="ij")
        assert (P[..., j > i] == 0).all()
        if window:
            assert (P[..., j < i - window + 1] == 0).all()
    elif window:
        i, j = np.meshgrid(np.arange(9), np.arange(9), indexing="ij")
        assert (P[..., (j < i - window) | (j > i + window)] == 0).all()
        assert (P[..., np.abs(j - i) <= window] > 0).all()


def test_constant_value_rows_come_back():
    Q, K, _ = wl.random_prefill(1, 2, 2, 7, 11, 8, seed=3)
    const = bf(np.linspace(-2, 2, 8))
    V = const.expand(1, 2, 11, 8).contiguous()
    for causal in (False, True):
        O, _ = oracle.attn_fwd(Q, K, V, causal, 0, 0.3)
        np.testing.assert_allclose(O, np.broadcast_to(f64(const).numpy(), O.shape), atol=1e-12)


def test_unmasked_permutation_invariance():
    Q, K, V = wl.random_prefill(1, 2, 2, 6, 13, 16, seed=4)
    perm = torch.randperm(13, generator=torch.Generator().manual_seed(9))
    O1, L1 = oracle.attn_fwd(Q, K, V, False, 0, 0.25)
    O2, L2 = oracle.attn_fwd(Q, K[:, :, perm].contiguous(), V[:, :, perm].contiguous(), False, 0, 0.25)
    np.testing.assert_allclose(O1, O2, atol=TOL, rtol=0)
    np.testing.assert_allclose(L1, L2, atol=TOL, rtol=0)


def test_per_row_score_shift():
    # Adding a vector u to every key adds scale * q_i.u to every score of row i:
    # O is unchanged and LSE moves by exactly that amount.  Small integers keep
    # every input and product exact.
    Q, K, V = wl.random_prefill(1, 1, 1, 4, 6, 8, seed=5, dist="int")
    u = torch.tensor([1, -1, 2, 0, 0, 1, -2, 1], dtype=torch.float32)
    K2 = (K.float() + u).to(torch.bfloat16)
    scale = 0.125
    for causal in (False, True):
        O1, L1 = oracle.attn_fwd(Q, K, V, causal, 0, scale)
        O2, L2 = oracle.attn_fwd(Q, K2, V, causal, 0, scale)
        shift = (f64(Q[0, 0]) @ f64(u)).numpy() * scale
        np.testing.assert_allclose(O1, O2, atol=1e-12)
        np.testing.assert_allclose(L2[0, 0] - L1[0, 0], shift, atol=1e-12)


@pytest.mark.parametrize("n_q,n_kv,causal,window", [(8, 8, False, 0), (8, 8, True, 0), (5, 9, True, 0),
                                                    (9, 9, True, 4), (3, 10, True, 2), (9, 9, False, 2),
                                                    (4, 11, False, 3), (10, 7, False, 4)])
def test_uniform_scores_closed_form(n_q, n_kv, causal, window):
    _, K, V = wl.random_prefill(1, 1, 1, n_q, n_kv, 8, seed=6)
    Q = torch.zeros(1, 1, n_q, 8, dtype=torch.bfloat16)
    O, LSE = oracle.attn_fwd(Q, K, V, causal, window, 0.7)
    v = f64(V[0, 0]).numpy()
    off = n_kv - n_q
    for i in range(n_q):
        if causal:
            hi = min(n_kv - 1, i + off)
            lo = max(0, i + off - window + 1) if window else 0
        elif window:        # symmetric window: |j - (i + off)| <= window
            hi = min(n_kv - 1, i + off + window)
            lo = max(0, i + off - window)
        else:
            lo, hi = 0, n_kv - 1
        np.testing.assert_allclose(O[0, 0, i], v[lo:hi + 1].mean(0), atol=1e-12)
        assert abs(LSE[0, 0, i] - math.log(hi - lo + 1)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_fp64(causal):
    Q, K, V = wl.random_prefill(2, 3, 3, 33, 33, 32, seed=7)
    scale = 1 / math.sqrt(32)
    O, LSE = oracle.attn_fwd(Q, K, V, causal, 0, scale)
    ref = torch.nn.functional.scaled_dot_product_attention(f64(Q), f64(K), f64(V), is_causal=causal,
                                                           scale=scale)
    np.testing.assert_allclose(O, ref.numpy(), atol=1e-12, rtol=0)
    s = (f64(Q) @ f64(K).transpose(-1, -2)) * scale
    if causal:
        s = s.masked_fill(torch.ones(33, 33, dtype=torch.bool).triu(1), -math.inf)
    np.testing.assert_allclose(LSE, torch.logsumexp(s, -1).numpy(), atol=1e-12, rtol=0)


def test_gqa_equals_mha_with_repeated_kv():
    Q, K, V = wl.random_prefill(2, 8, 2, 10, 12, 16, seed=8)
    O1, L1 = oracle.attn_fwd(Q, K, V, True, 0, 0.2)
    Kr, Vr = (x.repeat_interleave(4, dim=1).contiguous() for x in (K, V))
    O2, L2 = oracle.attn_fwd(Q, Kr, Vr, True, 0, 0.2)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)
    # and the group mapping is contiguous: head 5 uses kv head 1, not 5 % 2
    O3, _ = oracle.attn_fwd(Q[:, 5:6].contiguous(), K[:, 1:2].contiguous(), V[:, 1:2].contiguous(),
                            True, 0, 0.2)
    np.testing.assert_array_equal(O1[:, 5:6], O3)


def test_window_at_least_n_is_causal():
    Q, K, V = wl.random_prefill(1, 2, 2, 17, 17, 8, seed=10)
    Oc, Lc = oracle.attn_fwd(Q, K, V, True, 0, 0.3)
    for w in (17, 40):
        Ow, Lw = oracle.attn_fwd(Q, K, V, True, w, 0.3)
        np.testing.assert_array_equal(Oc, Ow)
        np.testing.assert_array_equal(Lc, Lw)


def test_symmetric_window_at_least_n_is_unmasked():
    Q, K, V = wl.random_prefill(1, 2, 2, 13, 13, 8, seed=19)
    On, Ln = oracle.attn_fwd(Q, K, V, False, 0, 0.3)
    for w in (12, 30):
        Ow, Lw = oracle.attn_fwd(Q, K, V, False, w, 0.3)
        np.testing.assert_array_equal(On, Ow)
        np.testing.assert_array_equal(Ln, Lw)
    Ow, _ = oracle.attn_fwd(Q, K, V, False, 11, 0.3)      # row 0 then misses key 12
    assert not np.array_equal(On, Ow)


@pytest.mark.parametrize("n_q,n_kv,w", [(20, 20, 3), (12, 20, 5), (20, 15, 2)])
def test_symmetric_window_matches_sdpa_with_band_mask(n_q, n_kv, w):
    Q, K, V = wl.random_prefill(2, 4, 2, n_q, n_kv, 16, seed=20)
    scale = 0.25
    O, LSE = oracle.attn_fwd(Q, K, V, False, w, scale)
    i = torch.arange(n_q)[:, None] + (n_kv - n_q)
    j = torch.arange(n_kv)[None, :]
    band = (j >= i - w) & (j <= i + w)
    Kr, Vr = (f64(x).repeat_interleave(2, dim=1) for x in (K, V))
    rows = band.any(1)                       # rows with at least one key (the others: O = 0, LSE = -inf)
    ref = torch.nn.functional.scaled_dot_product_attention(f64(Q), Kr, Vr, attn_mask=band, scale=scale)
    np.testing.assert_allclose(O[:, :, rows.numpy()], ref[:, :, rows].numpy(), atol=1e-12, rtol=0)
    s = (f64(Q) @ Kr.transpose(-1, -2)) * scale
    s = s.masked_fill(~band, -math.inf)
    np.testing.assert_allclose(LSE, torch.logsumexp(s, -1).numpy(), atol=1e-12, rtol=0)
    assert (O[:, :, ~rows.numpy()] == 0).all()


def test_bottom_right_causal_is_tail_of_square():
    Q, K, V = wl.random_prefill(1, 2, 2, 12, 12, 8, seed=11)
    O_sq, L_sq = oracle.attn_fwd(Q, K, V, True, 0, 0.4)
    O_t, L_t = oracle.attn_fwd(Q[:, :, 7:].contiguous(), K, V, True, 0, 0.4)
    np.testing.assert_array_equal(O_t, O_sq[:, :, 7:])
    np.testing.assert_array_equal(L_t, L_sq[:, :, 7:])
    O_w, _ = oracle.attn_fwd(Q[:, :, 7:].contiguous(), K, V, True, 3, 0.4)
    O_ws, _ = oracle.attn_fwd(Q, K, V, True, 3, 0.4)
    np.testing.assert_array_equal(O_w, O_ws[:, :, 7:])


def test_rows_without_keys():
    # N_q > N_kv with bottom-right causal: rows 0 and 1 see no key.
    Q, K, V = wl.random_prefill(1, 1, 1, 4, 2, 8, seed=12)
    O, LSE = oracle.attn_fwd(Q, K, V, True, 0, 0.5)
    assert (O[0, 0, :2] == 0).all() and np.isneginf(LSE[0, 0, :2]).all()
    assert np.isfinite(LSE[0, 0, 2:]).all()


def test_row_subset_is_bitwise_the_full_result():
    Q, K, V = wl.random_prefill(2, 4, 2, 9, 9, 16, seed=13)
    O, LSE = oracle.attn_fwd(Q, K, V, True, 0, 0.3)
    rows = [0, 5, 17, 71, 2 * 4 * 9 - 1]
    Os, Ls = oracle.attn_fwd(Q, K, V, True, 0, 0.3, rows=rows)
    np.testing.assert_array_equal(Os, O.reshape(-1, 16)[rows])
    np.testing.assert_array_equal(Ls, LSE.reshape(-1)[rows])


def _online_recurrence(q, k, v, scale, block):
    """fp64 block-by-block online softmax: running max m, running sum l and a
    rescaled accumulator (TileLang 学习笔记, Online Softmax 的关键), written
    independently of the oracle."""
    m = np.full(q.shape[0], -np.inf)
    l = np.zeros(q.shape[0])
    acc = np.zeros((q.shape[0], v.shape[1]))
    for j0 in range(0, k.shape[0], block):
        s = scale * q @ k[j0:j0 + block].T
        m_new = np.maximum(m, s.max(1))
        alpha = np.exp(m - m_new)
        p = np.exp(s - m_new[:, None])
        l = l * alpha + p.sum(1)
        acc = acc * alpha[:, None] + p @ v[j0:j0 + block]
        m = m_new
    return acc / l[:, None], m + np.log(l)


def test_online_recurrence_agrees_with_two_pass():
    Q, K, V = wl.random_prefill(1, 1, 1, 20, 77, 16, seed=14)
    O, LSE = oracle.attn_fwd(Q, K, V, False, 0, 0.25)
    q, k, v = (f64(x[0, 0]).numpy() for x in (Q, K, V))
    for block in (1, 8, 16, 77):
        Oo, Lo = _online_recurrence(q, k, v, 0.25, block)
        np.testing.assert_allclose(O[0, 0], Oo, atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE[0, 0], Lo, atol=1e-12, rtol=0)


def test_lse_merge_of_key_halves():
    """Exact merge of two partial results over disjoint key ranges, the step a
    split-KV decode needs: LSE = ln(e^L1 + e^L2), O = e^(L1-LSE) O1 + e^(L2-LSE) O2."""
    Q, K, V = wl.random_prefill(1, 2, 2, 6, 40, 8, seed=15)
    O, LSE = oracle.attn_fwd(Q, K, V, False, 0, 0.5)
    O1, L1 = oracle.attn_fwd(Q, K[:, :, :17].contiguous(), V[:, :, :17].contiguous(), False, 0, 0.5)
    O2, L2 = oracle.attn_fwd(Q, K[:, :, 17:].contiguous(), V[:, :, 17:].contiguous(), False, 0, 0.5)
    L = np.logaddexp(L1, L2)
    Om = np.exp(L1 - L)[..., None] * O1 + np.exp(L2 - L)[..., None] * O2
    np.testing.assert_allclose(L, LSE, atol=1e-12, rtol=0)
    np.testing.assert_allclose(Om, O, atol=1e-12, rtol=0)


def test_mla_matches_mqa_sdpa_fp64():
    Qn, Qp, KV, Kp = wl.random_mla(3, 4, 37, 32, 8, seed=16)
    scale = 1 / math.sqrt(40)
    O, LSE = oracle.mla_decode(Qn, Qp, KV, Kp, scale)
    q = torch.cat([f64(Qn), f64(Qp)], -1).unsqueeze(2)              # [B,H,1,40]
    k = torch.cat([f64(KV), f64(Kp)], -1).unsqueeze(1)              # [B,1,N,40]
    v = f64(KV).unsqueeze(1)                                        # [B,1,N,32]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k.expand(-1, 4, -1, -1),
                                                           v.expand(-1, 4, -1, -1), scale=scale)
    np.testing.assert_allclose(O, ref[:, :, 0].numpy(), atol=1e-12, rtol=0)
    s = (q @ k.transpose(-1, -2))[:, :, 0] * scale
    np.testing.assert_allclose(LSE, torch.logsumexp(s, -1).numpy(), atol=1e-12, rtol=0)


def test_mla_rows_subset():
    Qn, Qp, KV, Kp = wl.random_mla(2, 3, 9, 16, 4, seed=17)
    O, LSE = oracle.mla_decode(Qn, Qp, KV, Kp, 0.3)
    Os, Ls = oracle.mla_decode(Qn, Qp, KV, Kp, 0.3, rows=[1, 4])
    np.testing.assert_array_equal(Os, O.reshape(-1, 16)[[1, 4]])
    np.testing.assert_array_equal(Ls, LSE.reshape(-1)[[1, 4]])


def _expand_block_mask(mask, n_q, n_kv, block):
    m = mask.bool().repeat_interleave(block, 2).repeat_interleave(block, 3)
    return m[:, :, :n_q, :n_kv]


def test_block_mask_all_ones_is_dense():
    Q, K, V = wl.random_prefill(2, 4, 2, 70, 90, 16, seed=50)
    ones = torch.ones(2, 4, 3, 3, dtype=torch.uint8)
    for causal in (False, True):
        O1, L1 = oracle.attn_fwd(Q, K, V, causal, 0, 0.3)
        O2, L2 = oracle.attn_fwd(Q, K, V, causal, 0, 0.3, block_mask=ones, block=32)
        np.testing.assert_array_equal(O1, O2)
        np.testing.assert_array_equal(L1, L2)


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_matches_sdpa_with_expanded_mask(causal):
    n_q, n_kv, blk = 40, 52, 8
    Q, K, V = wl.random_prefill(2, 4, 2, n_q, n_kv, 16, seed=51)
    mask = wl.random_block_mask(2, 4, n_q, n_kv, 0.5, seed=52, block=blk)
    mask[1, 2, 3] = 0                              # query rows 24..31 of (1, 2) see no key
    O, LSE = oracle.attn_fwd(Q, K, V, causal, 0, 0.25, block_mask=mask, block=blk)
    allowed = _expand_block_mask(mask, n_q, n_kv, blk)
    if causal:
        i = torch.arange(n_q)[:, None] + (n_kv - n_q)
        allowed = allowed & (torch.arange(n_kv)[None, :] <= i)
    Kr, Vr = (f64(x).repeat_interleave(2, dim=1) for x in (K, V))
    s = (f64(Q) @ Kr.transpose(-1, -2)) * 0.25
    s = s.masked_fill(~allowed, -math.inf)
    np.testing.assert_allclose(LSE, torch.logsumexp(s, -1).numpy(), atol=1e-12, rtol=0)
    rows = allowed.any(-1)
    p = torch.softmax(s.masked_fill(~rows[..., None], 0.0), -1) * rows[..., None]
    np.testing.assert_allclose(O, (p @ Vr).numpy(), atol=1e-12, rtol=0)
    assert (~rows).any() and (O[~rows.numpy()] == 0).all() and np.isneginf(LSE[~rows.numpy()]).all()


def test_block_mask_uniform_scores_closed_form():
    n_q, n_kv, blk = 12, 16, 4
    _, K, V = wl.random_prefill(1, 1, 1, n_q, n_kv, 8, seed=53)
    Q = torch.zeros(1, 1, n_q, 8, dtype=torch.bfloat16)
    mask = torch.tensor([[[[1, 0, 1, 0], [0, 0, 0, 1], [1, 1, 1, 1]]]], dtype=torch.uint8)
    O, LSE = oracle.attn_fwd(Q, K, V, False, 0, 0.7, block_mask=mask, block=blk)
    v = f64(V[0, 0]).numpy()
    for i in range(n_q):
        keys = [j for j in range(n_kv) if mask[0, 0, i // blk, j // blk]]
        np.testing.assert_allclose(O[0, 0, i], v[keys].mean(0), atol=1e-12)
        assert abs(LSE[0, 0, i] - math.log(len(keys))) < 1e-12


def _dense_as_paged(KV, Kp, page):
    """The dense [B,N,d] caches as pages in order: sequence b owns pages b*N/page ..."""
    B, N, d_c = KV.shape
    n = N // page
    table = torch.arange(B * n, dtype=torch.int32).reshape(B, n)
    return KV.reshape(B * n, page, d_c), Kp.reshape(B * n, page, Kp.shape[-1]), table


def test_mla_paged_contiguous_pages_equal_dense():
    Qn, Qp, KV, Kp = wl.random_mla(3, 8, 256, 512, 64, seed=30)
    O, L = oracle.mla_decode(Qn, Qp, KV, Kp, 0.04)
    KVc, Kpc, table = _dense_as_paged(KV, Kp, 64)
    Op, Lp = oracle.mla_decode_paged(Qn, Qp, KVc, Kpc, table, [256] * 3, 0.04)
    np.testing.assert_array_equal(O, Op)
    np.testing.assert_array_equal(L, Lp)


def test_mla_paged_invariant_to_page_placement():
    Qn, Qp, KV, Kp, table, lens = wl.random_mla_paged(4, [130, 64, 1, 200], d_c=64, d_r=16, page=64, seed=31)
    O1, L1 = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, lens, 0.1)
    perm = torch.randperm(KV.shape[0], generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    table2 = torch.where(table >= 0, inv[table.clamp(min=0).long()].to(torch.int32), table)
    O2, L2 = oracle.mla_decode_paged(Qn, Qp, KV[perm].contiguous(), Kp[perm].contiguous(), table2, lens, 0.1)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_mla_paged_lengths_truncate_the_sequence():
    lens = [1, 63, 64, 65, 190]
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(4, lens, d_c=64, d_r=16, page=64, seed=32)
    O, LSE = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, L, 0.1)
    for b, n in enumerate(lens):
        rows = torch.arange(n)
        pages = table[b, rows // 64].long()
        kv = KV[pages, rows % 64].unsqueeze(0).contiguous()
        kp = Kp[pages, rows % 64].unsqueeze(0).contiguous()
        Od, Ld = oracle.mla_decode(Qn[b:b + 1].contiguous(), Qp[b:b + 1].contiguous(), kv, kp, 0.1)
        np.testing.assert_array_equal(O[b], Od[0])
        np.testing.assert_array_equal(LSE[b], Ld[0])


def test_mla_paged_empty_sequence():
    Qn, Qp, KV, Kp, table, lens = wl.random_mla_paged(2, [0, 70], d_c=64, d_r=16, page=64, seed=33)
    O, L = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, lens, 0.1)
    assert (O[0] == 0).all() and np.isneginf(L[0]).all()
    assert np.isfinite(L[1]).all()


def test_mla_paged_query_tokens_are_truncated_single_token_calls():
    # s_q query tokens are the last s_q positions: token t sees keys < len - (s_q - 1 - t)
    lens, s_q = [5, 70, 130, 1], 3
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(4, lens, d_c=64, d_r=16, page=64, seed=35, s_q=s_q)
    O, LSE = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, L, 0.1)
    assert O.shape == (4, s_q, 4, 64) and LSE.shape == (4, s_q, 4)
    for t in range(s_q):
        short = torch.clamp(L - (s_q - 1 - t), min=0)
        Ot, Lt = oracle.mla_decode_paged(Qn[:, t].contiguous(), Qp[:, t].contiguous(), KV, Kp, table, short, 0.1)
        np.testing.assert_array_equal(O[:, t], Ot)
        np.testing.assert_array_equal(LSE[:, t], Lt)
    assert (O[3, 0] == 0).all() and np.isneginf(LSE[3, :2]).all()    # length 1: tokens 0 and 1 see nothing


def test_mla_paged_rejects_bad_tables():
    Qn, Qp, KV, Kp, table, lens = wl.random_mla_paged(2, [70, 10], d_c=64, d_r=16, page=64, seed=34)
    with pytest.raises(ValueError):
        oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, [129, 10], 0.1)      # longer than the table
    bad = table.clone()
    bad[0, 1] = KV.shape[0]
    with pytest.raises(ValueError):
        oracle.mla_decode_paged(Qn, Qp, KV, Kp, bad, lens, 0.1)             # page out of the pool


def test_rejects_bad_arguments():
    Q, K, V = wl.random_prefill(1, 3, 2, 4, 4, 8, seed=18)  # H % H_kv != 0
    with pytest.raises(ValueError):
        oracle.attn_fwd(Q, K, V, False, 0, 1.0)
    Q, K, V = wl.random_prefill(1, 2, 2, 4, 4, 8, seed=18)
    with pytest.raises(ValueError):
        oracle.attn_fwd(Q, K, V, False, 0, 1.0, rows=[8])       # row out of range


def test_workload_inputs_are_seeded_and_spiky():
    c = wl.PrefillCase("t", 1, 2, 2, 300, 300, 8, True, spike_frac=0.01, seed=99)
    a = wl.prefill_inputs(c)
    b = wl.prefill_inputs(c)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    # exactly round(0.01*300) = 3 key rows carry the x8 spike, the same rows in every head
    g = torch.Generator().manual_seed(99)
    torch.randn(1, 2, 300, 8, generator=g)
    k_plain = torch.randn(1, 2, 300, 8, generator=g)
    ratio = a[1].float() / k_plain.to(torch.bfloat16).float()
    spiked = (ratio == 8).all(-1)
    assert ((ratio == 8) | (ratio == 1)).all()
    assert spiked.sum().item() == 2 * 3
    assert torch.equal(spiked[0, 0], spiked[0, 1])
