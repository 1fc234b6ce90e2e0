"""GPU parity of mla_decode_paged (through the C ABI) against the fp64 oracle:
per-sequence lengths, 64-key pages placed at random in the cache, empty
sequences, non-finite data past a sequence's end, and bit-equality with the
dense entry point when the pages are laid out in order."""
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


def run_paged(Qn, Qp, KV, Kp, table, lens, scale=SCALE):
    O, LSE = gb.mla_decode_paged(Qn.cuda(), Qp.cuda(), KV.cuda(), Kp.cuda(), table.cuda(), lens.cuda(), scale=scale)
    gb.check()
    return O, LSE


LENGTHS = [
    [1],
    [64],
    [65, 63],
    [0, 130, 0],                                  # empty sequences around a short one
    [4096],
    [20000],                                      # one sequence over every cluster
    [1, 63, 64, 65, 200, 0, 777, 4097, 130, 5000],
    [0, 0, 0],                                    # nothing to attend to
]


@pytest.mark.parametrize("lens", LENGTHS, ids=lambda l: "-".join(map(str, l)))
def test_parity(lens):
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(128, lens, seed=sum(lens) * 7 + len(lens))
    O, LSE = run_paged(Qn, Qp, KV, Kp, table, L)
    O_ref, L_ref = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, L, SCALE)
    compare(O, LSE, O_ref, L_ref, what=f"lens={lens}")


def test_many_short_sequences():
    # more sequences than clusters, many whole sequences inside one cluster's range
    g = torch.Generator().manual_seed(41)
    lens = torch.randint(0, 300, (300,), generator=g).tolist()
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(128, lens, seed=42)
    O, LSE = run_paged(Qn, Qp, KV, Kp, table, L)
    O_ref, L_ref = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, L, SCALE)
    compare(O, LSE, O_ref, L_ref, what="300 short sequences")


def test_non_finite_rows_past_the_end_are_ignored():
    lens = [70, 1, 129, 64, 300]
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(128, lens, seed=43)
    O_ref, L_ref = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, L, SCALE)
    KV, Kp = KV.clone(), Kp.clone()
    for b, n in enumerate(lens):
        if n % 64:
            page = int(table[b, (n - 1) // 64])
            KV[page, n % 64:] = float("nan")
            Kp[page, n % 64:] = float("inf")
    O, LSE = run_paged(Qn, Qp, KV, Kp, table, L)
    compare(O, LSE, O_ref, L_ref, what="NaN/Inf past the end")


def test_contiguous_pages_match_the_dense_entry_point_bitwise():
    B, N = 5, 777
    Qn, Qp, KV, Kp = wl.random_mla(B, 128, N, 512, 64, seed=44)
    O_d, L_d = gb.mla_decode(Qn.cuda(), Qp.cuda(), KV.cuda(), Kp.cuda(), scale=SCALE)
    n = (N + 63) // 64
    pad = n * 64 - N
    KVp = torch.cat([KV, torch.zeros(B, pad, 512, dtype=KV.dtype)], 1).reshape(B * n, 64, 512)
    Kpp = torch.cat([Kp, torch.zeros(B, pad, 64, dtype=Kp.dtype)], 1).reshape(B * n, 64, 64)
    table = torch.arange(B * n, dtype=torch.int32).reshape(B, n)
    O_p, L_p = run_paged(Qn, Qp, KVp, Kpp, table, torch.full((B,), N, dtype=torch.int32))
    assert torch.equal(O_d.view(torch.int16), O_p.view(torch.int16))
    assert torch.equal(L_d, L_p)


def test_deterministic():
    lens = [3000, 17, 999, 4500]
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(128, lens, seed=45)
    O1, L1 = run_paged(Qn, Qp, KV, Kp, table, L)
    O2, L2 = run_paged(Qn, Qp, KV, Kp, table, L)
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L1, L2)


def test_length_past_the_table_is_clamped_and_reported():
    lens = [100, 50]
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(128, lens, seed=46)
    bad = torch.tensor([table.shape[1] * 64 + 500, 50], dtype=torch.int32)
    gb.check()
    O, LSE = gb.mla_decode_paged(Qn.cuda(), Qp.cuda(), KV.cuda(), Kp.cuda(), table.cuda(), bad.cuda(), scale=SCALE)
    with pytest.raises(gb.GbattnError) as e:
        gb.check()
    assert e.value.code == 1
    # the context stays usable and a correct call matches the oracle
    O, LSE = run_paged(Qn, Qp, KV, Kp, table, L)
    O_ref, L_ref = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, L, SCALE)
    compare(O, LSE, O_ref, L_ref, what="after a clamped call")


def test_varied_lengths_full_size_sampled():
    g = torch.Generator().manual_seed(47)
    lens = torch.randint(2048, 6145, (64,), generator=g).tolist()
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(128, lens, seed=48)
    O, LSE = run_paged(Qn, Qp, KV, Kp, table, L)
    rng = np.random.default_rng(49)
    # 96 random rows plus every head of three whole sequences (the first, one in
    # the middle and the last, whose ranges end the last clusters' work)
    rows = np.unique(np.concatenate([rng.integers(0, 64 * 128, 96), np.arange(0, 128), np.arange(31 * 128, 32 * 128),
                                     np.arange(63 * 128, 64 * 128)]))
    O_ref, L_ref = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, L, SCALE, rows=rows)
    idx = torch.as_tensor(rows, device=O.device)
    compare(O.reshape(-1, 512)[idx], LSE.reshape(-1)[idx], O_ref, L_ref, what="64 varied sequences")


@pytest.mark.parametrize("s_q,lens", [(2, [5, 70, 130, 1, 4097]), (3, [2, 64, 65, 1000]), (4, [3000, 0, 129])],
                         ids=lambda v: str(v))
def test_several_query_tokens(s_q, lens):
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(128, lens, seed=70 + s_q, s_q=s_q)
    O, LSE = run_paged(Qn, Qp, KV, Kp, table, L)
    assert O.shape == (len(lens), s_q, 128, 512) and LSE.shape == (len(lens), s_q, 128)
    O_ref, L_ref = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, L, SCALE)
    compare(O.reshape(-1, 128, 512), LSE.reshape(-1, 128), O_ref.reshape(-1, 128, 512), L_ref.reshape(-1, 128),
            what=f"s_q={s_q} lens={lens}")


@pytest.mark.parametrize("H,s_q,lens", [(64, 2, [5, 70, 130, 1, 4097, 0]), (32, 4, [3, 2, 64, 65, 1000]),
                                        (16, 8, [7, 300, 4, 129]), (64, 3, [2, 64, 65, 1000, 0]),
                                        (16, 1, [1, 63, 64, 65, 5000]), (128, 2, [3, 130])])
def test_packed_query_tokens(H, s_q, lens):
    # s_q * H <= 128: all of a sequence's tokens share one 128-row tile (its keys
    # are read once), each row masked to its token's keys; H = 64 with s_q = 3
    # takes two tiles per sequence (two tokens, then one); lengths shorter than
    # s_q leave the first tokens without keys.
    Qn, Qp, KV, Kp, table, L = wl.random_mla_paged(H, lens, seed=H * 31 + s_q * 7 + len(lens), s_q=s_q)
    O, LSE = run_paged(Qn, Qp, KV, Kp, table, L)
    lead = (len(lens), s_q, H) if s_q > 1 else (len(lens), H)
    assert O.shape == (*lead, 512) and LSE.shape == lead
    O_ref, L_ref = oracle.mla_decode_paged(Qn, Qp, KV, Kp, table, L, SCALE)
    compare(O, LSE, O_ref, L_ref, what=f"H={H} s_q={s_q} lens={lens}")
