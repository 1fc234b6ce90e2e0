"""Seeded synthetic inputs for the attention workloads.

This module only draws random inputs; it holds none of the attention
arithmetic, so the CUDA path and the CPU oracle can both take their inputs from
it.  Every tensor is drawn on the CPU from ``torch.Generator('cpu')`` seeded
with ``20261202 + index``, as fp32 N(0, 1), then cast to bf16 (round to
nearest even).  Draw order: Q, K, V for prefill; Q_nope, Q_pe, KV_latent, K_pe
for MLA decode.

The long-context workload scales 1% of the key rows by 8 before the bf16 cast
(x8 is exact in bf16): the same ``round(0.01 * N_kv)`` row indices, drawn with
``randperm`` from the same generator after V, for every (batch, head).  Large
scores then appear late in a row and force the running maximum to move.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEED_BASE = 20261202


@dataclass(frozen=True)
class PrefillCase:
    name: str
    B: int
    H: int
    H_kv: int
    N_q: int
    N_kv: int
    d: int
    causal: bool
    window: int = 0
    spike_frac: float = 0.0      # fraction of key rows scaled by spike_mult
    spike_mult: float = 8.0
    seed: int = SEED_BASE
    scale: float = field(default=float("nan"))

    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d) if math.isnan(self.scale) else self.scale


@dataclass(frozen=True)
class MlaCase:
    name: str
    B: int
    H: int
    N_kv: int
    d_c: int = 512
    d_r: int = 64
    seed: int = SEED_BASE
    scale: float = field(default=float("nan"))

    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d_c + self.d_r) if math.isnan(self.scale) else self.scale


# The five named workloads (index = seed offset), plus the causal-window and
# symmetric-window variants of the GQA one, which share its inputs.
WORKLOADS = {
    "mha_b1_h2_n128_d64": PrefillCase("mha_b1_h2_n128_d64", 1, 2, 2, 128, 128, 64, False,
                                      seed=SEED_BASE + 0),
    "mha_causal_b4_h16_n2048_d128": PrefillCase("mha_causal_b4_h16_n2048_d128", 4, 16, 16, 2048,
                                                2048, 128, True, seed=SEED_BASE + 1),
    "gqa_causal_b2_h32_hkv8_n8192_d128": PrefillCase("gqa_causal_b2_h32_hkv8_n8192_d128", 2, 32, 8,
                                                     8192, 8192, 128, True, seed=SEED_BASE + 2),
    "gqa_window256_b2_h32_hkv8_n8192_d128": PrefillCase("gqa_window256_b2_h32_hkv8_n8192_d128", 2, 32,
                                                        8, 8192, 8192, 128, True, window=256,
                                                        seed=SEED_BASE + 2),
    "gqa_swindow256_b2_h32_hkv8_n8192_d128": PrefillCase("gqa_swindow256_b2_h32_hkv8_n8192_d128", 2, 32,
                                                         8, 8192, 8192, 128, False, window=256,
                                                         seed=SEED_BASE + 2),
    "mla_decode_b64_h128_nkv4096": MlaCase("mla_decode_b64_h128_nkv4096", 64, 128, 4096,
                                           seed=SEED_BASE + 3),
    "mha_causal_spiky_b1_h32_n16384_d128": PrefillCase("mha_causal_spiky_b1_h32_n16384_d128", 1, 32,
                                                       32, 16384, 16384, 128, True, spike_frac=0.01,
                                                       seed=SEED_BASE + 4),
}


@dataclass(frozen=True)
class SsdCase:
    """Mamba-2 SSD scan shape: batch, sequence length, heads, head dim P,
    B/C groups G, state dim N."""
    name: str
    Bsz: int
    L: int
    H: int
    P: int = 64
    G: int = 1
    N: int = 128
    seed: int = SEED_BASE


# A Mamba-2-sized layer (inner width 5120 = 80 heads of 64, state 128, one
# B/C group) over 8 sequences of 4096 steps.
SSD_WORKLOAD = SsdCase("ssd_b8_l4096_h80_p64_g1_n128", 8, 4096, 80, seed=SEED_BASE + 7)


def ssd_inputs(case: SsdCase):
    return random_ssd(case.Bsz, case.L, case.H, case.P, case.G, case.N, seed=case.seed)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def prefill_inputs(case: PrefillCase):
    """(Q, K, V) bf16 CPU tensors: Q [B,H,N_q,d], K/V [B,H_kv,N_kv,d]."""
    g = _gen(case.seed)
    Q = torch.randn(case.B, case.H, case.N_q, case.d, generator=g, dtype=torch.float32)
    K = torch.randn(case.B, case.H_kv, case.N_kv, case.d, generator=g, dtype=torch.float32)
    V = torch.randn(case.B, case.H_kv, case.N_kv, case.d, generator=g, dtype=torch.float32)
    if case.spike_frac > 0 and case.N_kv > 0:
        n_spike = int(round(case.spike_frac * case.N_kv))
        idx = torch.randperm(case.N_kv, generator=g)[:n_spike]
        K[:, :, idx, :] *= case.spike_mult
    return Q.to(torch.bfloat16), K.to(torch.bfloat16), V.to(torch.bfloat16)


def mla_inputs(case: MlaCase):
    """(Q_nope [B,H,d_c], Q_pe [B,H,d_r], KV_latent [B,N_kv,d_c], K_pe [B,N_kv,d_r]) bf16 CPU."""
    g = _gen(case.seed)
    Qn = torch.randn(case.B, case.H, case.d_c, generator=g, dtype=torch.float32)
    Qp = torch.randn(case.B, case.H, case.d_r, generator=g, dtype=torch.float32)
    KV = torch.randn(case.B, case.N_kv, case.d_c, generator=g, dtype=torch.float32)
    Kp = torch.randn(case.B, case.N_kv, case.d_r, generator=g, dtype=torch.float32)
    return tuple(x.to(torch.bfloat16) for x in (Qn, Qp, KV, Kp))


def random_prefill(B, H, H_kv, N_q, N_kv, d, seed, dist="normal"):
    """Small ad-hoc prefill inputs for edge-case tests (same drawing recipe)."""
    g = _gen(seed)
    shape_q, shape_kv = (B, H, N_q, d), (B, H_kv, N_kv, d)
    if dist == "normal":
        draw = lambda s: torch.randn(*s, generator=g, dtype=torch.float32)
    elif dist == "int":   # small integers: exactly representable, exact products
        draw = lambda s: torch.randint(-3, 4, s, generator=g).to(torch.float32)
    else:
        raise ValueError(dist)
    return tuple(draw(s).to(torch.bfloat16) for s in (shape_q, shape_kv, shape_kv))


def random_mla(B, H, N_kv, d_c, d_r, seed):
    g = _gen(seed)
    shapes = [(B, H, d_c), (B, H, d_r), (B, N_kv, d_c), (B, N_kv, d_r)]
    return tuple(torch.randn(*s, generator=g, dtype=torch.float32).to(torch.bfloat16)
                 for s in shapes)


def random_mla_paged(H, seqlens, d_c=512, d_r=64, page=64, spare_pages=3, seed=0, s_q=1):
    """Paged MLA decode inputs: Q_nope [B,H,d_c], Q_pe [B,H,d_r] (bf16; with
    s_q > 1 query tokens per sequence [B,s_q,H,d_c] and [B,s_q,H,d_r]),
    KV_cache [num_pages,page,d_c], K_pe_cache [num_pages,page,d_r] (bf16),
    block_table [B,max_pages] int32, seqlens [B] int32.  Each sequence gets
    ceil(len / page) pages drawn without replacement from a pool with
    `spare_pages` unused pages (random placement); unused table entries are -1.
    Same drawing recipe (torch CPU generator, N(0,1) -> bf16)."""
    g = _gen(seed)
    lens = [int(x) for x in seqlens]
    B = len(lens)
    need = [(n + page - 1) // page for n in lens]
    max_pages = max(1, max(need) if need else 1)
    num_pages = sum(need) + spare_pages
    qs = (B, s_q, H) if s_q > 1 else (B, H)
    Qn = torch.randn(*qs, d_c, generator=g, dtype=torch.float32).to(torch.bfloat16)
    Qp = torch.randn(*qs, d_r, generator=g, dtype=torch.float32).to(torch.bfloat16)
    KV = torch.randn(num_pages, page, d_c, generator=g, dtype=torch.float32).to(torch.bfloat16)
    Kp = torch.randn(num_pages, page, d_r, generator=g, dtype=torch.float32).to(torch.bfloat16)
    perm = torch.randperm(num_pages, generator=g)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n].to(torch.int32)
        k += n
    return Qn, Qp, KV, Kp, table, torch.tensor(lens, dtype=torch.int32)


def random_block_mask(B, H, N_q, N_kv, density, seed, block=128):
    """uint8 [B,H,ceil(N_q/block),ceil(N_kv/block)]: each block set with
    probability `density` (torch CPU generator)."""
    g = _gen(seed)
    shape = (B, H, -(-N_q // block), -(-N_kv // block))
    return (torch.rand(*shape, generator=g) < density).to(torch.uint8)


def random_ssd(Bsz, L, H, P, G, N, seed, with_D=True):
    """Mamba-2 SSD scan inputs (torch CPU generator): x [Bsz,L,H,P] bf16 ~ N(0,1);
    dt [Bsz,L,H] fp32 log-uniform in [0.001, 0.1]; A [H] fp32 = -exp(U[0, ln 16]);
    B, C [Bsz,L,G,N] bf16 ~ N(0,1); D [H] fp32 = 1 (or None)."""
    g = _gen(seed)
    x = torch.randn(Bsz, L, H, P, generator=g, dtype=torch.float32).to(torch.bfloat16)
    dt = torch.exp(torch.rand(Bsz, L, H, generator=g) * (math.log(0.1) - math.log(0.001)) + math.log(0.001))
    A = -torch.exp(torch.rand(H, generator=g) * math.log(16.0))
    B = torch.randn(Bsz, L, G, N, generator=g, dtype=torch.float32).to(torch.bfloat16)
    C = torch.randn(Bsz, L, G, N, generator=g, dtype=torch.float32).to(torch.bfloat16)
    D = torch.ones(H, dtype=torch.float32) if with_D else None
    return x, dt.to(torch.float32), A.to(torch.float32), B, C, D
