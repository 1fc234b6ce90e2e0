"""GPU parity of ssd_scan (Mamba-2 SSD scan, through the C ABI) against the
fp64 oracle's plain recurrence: one chunk, ragged last chunks, a single step,
several B/C groups, no D term, the final state, degenerate dt and A, and a
sampled Mamba-2-sized case.

Tolerance, from the arithmetic: the kernel takes the same bf16 inputs and sums
in fp32, but operands of its tensor-core products are rounded to bf16
(relative error at most 2^-9 per rounding): the chunk weights exp(cum_t -
cum_s) dt_s (C_t . B_s) once, the decayed rows exp(cum_end - cum_s) dt_s B_s
twice (the factor, then the product), and the carried state once.  Every term
of y is bounded by the matching term of the same recurrence run on |x|, |B|,
|C|, |D| (y_abs, by the oracle), and each term carries at most three of those
roundings, so |y - y_ref| <= 3 * 2^-9 y_abs plus fp32 noise; the test allows
2^-7 y_abs + 1e-6 (the same for the final state against S_abs).
A dropped term, a wrong sign or a shifted decay moves y by a sizeable part of
y_abs and fails it."""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import workloads as wl
from tests._util import build_lib

pytestmark = pytest.mark.gpu

REL = 2.0 ** -7


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()
    gb.load_library()


def run(x, dt, A, B, C, D, final=True):
    cu = lambda t: None if t is None else t.cuda()
    out = gb.ssd_scan(cu(x), cu(dt), cu(A), cu(B), cu(C), cu(D), want_final_state=final)
    gb.check()
    return out


def reference(x, dt, A, B, C, D):
    """(y_ref, S_ref, y_abs, S_abs): the oracle on the inputs and on their magnitudes."""
    y_ref, S_ref = oracle.ssd_scan(x, dt, A, B, C, D)
    y_abs, S_abs = oracle.ssd_scan(x.abs(), dt, A, B.abs(), C.abs(), None if D is None else D.abs())
    return y_ref, S_ref, y_abs, S_abs


def close(got, ref, bound, what):
    g = got.detach().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite"
    if not g.size:
        return
    excess = (np.abs(g - ref) - (REL * bound + 1e-6)).max()
    err = (np.abs(g - ref) / (bound + 1e-6)).max()
    assert excess <= 0, f"{what}: max |d|/bound = {err:.3e} > {REL:.3e}"


CASES = [
    # Bsz, L, H, G, with_D
    (1, 128, 2, 1, True),     # exactly one chunk
    (2, 200, 4, 2, True),     # ragged last chunk, two groups
    (1, 1, 1, 1, True),       # a single step
    (1, 1000, 8, 1, False),   # many chunks, no D
    (3, 129, 6, 6, True),     # one group per head, 1-step last chunk
    (2, 256, 4, 1, True),     # two whole chunks
    (1, 700, 4, 4, False),
    # lengths around the 128-step chunk boundary
    (1, 127, 2, 1, True),
    (1, 255, 2, 1, True),
    (2, 257, 2, 2, True),
    (1, 384, 3, 1, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_parity(case):
    Bsz, L, H, G, with_D = case
    x, dt, A, B, C, D = wl.random_ssd(Bsz, L, H, 64, G, 128, seed=900 + sum(case[:4]), with_D=with_D)
    y, S = run(x, dt, A, B, C, D)
    y_ref, S_ref, y_abs, S_abs = reference(x, dt, A, B, C, D)
    close(y, y_ref, y_abs, f"y {case}")
    close(S, S_ref, S_abs, f"final state {case}")


def test_zero_dt_leaves_only_the_skip_term():
    x, dt, A, B, C, D = wl.random_ssd(1, 300, 2, 64, 1, 128, seed=910)
    D = torch.tensor([0.5, -2.0])
    y, S = run(x, torch.zeros_like(dt), A, B, C, D)
    assert torch.equal(S.cpu(), torch.zeros_like(S.cpu()))
    assert torch.equal(y.cpu(), x.float() * D.view(1, 1, 2, 1))


def test_no_decay_is_a_running_sum():
    # A = 0: S_t is the plain sum of dt_s x_s B_s^T, the oracle's closed form
    x, dt, A, B, C, D = wl.random_ssd(1, 333, 2, 64, 1, 128, seed=911, with_D=False)
    A0 = torch.zeros_like(A)
    y, S = run(x, dt, A0, B, C, None)
    y_ref, S_ref, y_abs, S_abs = reference(x, dt, A0, B, C, None)
    close(y, y_ref, y_abs, "A = 0 y")
    close(S, S_ref, S_abs, "A = 0 final state")


def test_strong_decay_forgets_earlier_chunks():
    # dt A ~ -16 per step: the state carried over a chunk boundary is negligible
    x, dt, A, B, C, D = wl.random_ssd(1, 256, 2, 64, 1, 128, seed=912)
    dt1, A16 = torch.ones_like(dt), torch.full_like(A, -16.0)
    y, S = run(x, dt1, A16, B, C, D)
    y_ref, S_ref, y_abs, S_abs = reference(x, dt1, A16, B, C, D)
    close(y, y_ref, y_abs, "strong decay y")
    close(S, S_ref, S_abs, "strong decay final state")


def test_y_without_final_state_is_the_same():
    x, dt, A, B, C, D = wl.random_ssd(2, 500, 4, 64, 1, 128, seed=913)
    y1, _ = run(x, dt, A, B, C, D)
    y2 = run(x, dt, A, B, C, D, final=False)
    assert torch.equal(y1, y2)


def test_deterministic():
    x, dt, A, B, C, D = wl.random_ssd(2, 1000, 4, 64, 2, 128, seed=914)
    y1, S1 = run(x, dt, A, B, C, D)
    y2, S2 = run(x, dt, A, B, C, D)
    assert torch.equal(y1, y2) and torch.equal(S1, S2)


def test_mamba2_sized_sampled_heads():
    # the benchmark's shape; the oracle runs on one batch entry and a few heads
    c = wl.SSD_WORKLOAD
    x, dt, A, B, C, D = wl.ssd_inputs(c)
    y, S = run(x, dt, A, B, C, D)
    b, heads = c.Bsz - 1, [0, c.H // 2, c.H - 1]
    sel = lambda t: t[b:b + 1][:, :, heads].contiguous()
    y_ref, S_ref, y_abs, S_abs = reference(sel(x), sel(dt), A[heads].contiguous(), B[b:b + 1], C[b:b + 1],
                                           D[heads].contiguous())
    close(y[b:b + 1][:, :, heads], y_ref, y_abs, "sampled y")
    close(S[b:b + 1][:, heads], S_ref, S_abs, "sampled final state")
