"""Pins for the fp64 Mamba-2 SSD scan oracle (plain recurrence), against
things other than the recurrence itself:

* no decay (A = 0) and unit steps: the scan is causal linear attention,
  y_t = sum_{s<=t} (C_t . B_s) x_s, checked with torch matmuls and a
  lower-triangular mask;
* an impulse at t = 0 decays in closed form: y_t = exp(A sum_{0<r<=t} dt_r)
  dt_0 (B_0 . C_t) x_0;
* one step: y = dt (B . C) x + D x;
* an independent fp64 implementation of the chunked form (intra-chunk
  products with cumulative decays, inter-chunk state passing) agrees with the
  recurrence for several chunk sizes, including the final state;
* heads map to B/C groups in contiguous blocks.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_flashattention_gb300 import workloads as wl


def f64(t):
    return t.to(torch.float64)


def test_no_decay_is_causal_linear_attention():
    x, dt, A, B, C, _ = wl.random_ssd(2, 37, 3, 8, 1, 16, seed=80, with_D=False)
    dt = torch.ones_like(dt)
    A = torch.zeros_like(A)
    y, _ = oracle.ssd_scan(x, dt, A, B, C)
    Bm, Cm = f64(B[:, :, 0]), f64(C[:, :, 0])                       # [Bsz, L, N]
    W = torch.tril(Cm @ Bm.transpose(1, 2))                          # [Bsz, L(t), L(s)]
    ref = torch.einsum("bts,bshp->bthp", W, f64(x))
    np.testing.assert_allclose(y, ref.numpy(), atol=1e-10, rtol=0)


def test_impulse_decays_in_closed_form():
    x, dt, A, B, C, _ = wl.random_ssd(1, 20, 2, 4, 1, 8, seed=81, with_D=False)
    x = x.clone()
    x[:, 1:] = 0
    y, _ = oracle.ssd_scan(x, dt, A, B, C)
    for h in range(2):
        for t in range(20):
            decay = math.exp(float(A[h]) * float(dt[0, 1:t + 1, h].double().sum()))
            bc = float(f64(B[0, 0, 0]) @ f64(C[0, t, 0]))
            ref = decay * float(dt[0, 0, h]) * bc * f64(x[0, 0, h]).numpy()
            np.testing.assert_allclose(y[0, t, h], ref, atol=1e-12, rtol=1e-12)


def test_single_step():
    x, dt, A, B, C, D = wl.random_ssd(2, 1, 4, 8, 2, 16, seed=82)
    y, S = oracle.ssd_scan(x, dt, A, B, C, D)
    for b in range(2):
        for h in range(4):
            g = h // 2
            bc = float(f64(B[b, 0, g]) @ f64(C[b, 0, g]))
            ref = (float(dt[b, 0, h]) * bc + float(D[h])) * f64(x[b, 0, h]).numpy()
            np.testing.assert_allclose(y[b, 0, h], ref, atol=1e-12, rtol=1e-12)
            np.testing.assert_allclose(S[b, h], float(dt[b, 0, h]) * np.outer(f64(x[b, 0, h]).numpy(),
                                                                             f64(B[b, 0, g]).numpy()), atol=1e-12)


def chunked_reference(x, dt, A, B, C, D, Q):
    """The chunked SSD form in fp64 numpy, written independently of the
    recurrence: per chunk, intra-chunk products with cumulative decays plus the
    carried state, then the state update."""
    x, B, C = (f64(t).numpy() for t in (x, B, C))
    dt, A = dt.double().numpy(), A.double().numpy()
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros_like(x)
    S = np.zeros((Bsz, H, P, N))
    for b in range(Bsz):
        for h in range(H):
            g = h // (H // G)
            state = np.zeros((P, N))
            for c0 in range(0, L, Q):
                c1 = min(c0 + Q, L)
                a = dt[b, c0:c1, h] * A[h]
                cum = np.cumsum(a)                                    # inclusive
                Lmat = np.exp(cum[:, None] - cum[None, :]) * np.tril(np.ones((c1 - c0, c1 - c0)))
                CB = C[b, c0:c1, g] @ B[b, c0:c1, g].T                # [t, s]
                W = CB * Lmat * dt[b, c0:c1, h][None, :]
                y[b, c0:c1, h] = W @ x[b, c0:c1, h] + np.exp(cum)[:, None] * (C[b, c0:c1, g] @ state.T)
                if D is not None:
                    y[b, c0:c1, h] += float(D[h]) * x[b, c0:c1, h]
                w_end = np.exp(cum[-1] - cum) * dt[b, c0:c1, h]          # [s]
                state = np.exp(cum[-1]) * state + (x[b, c0:c1, h] * w_end[:, None]).T @ B[b, c0:c1, g]
            S[b, h] = state
    return y, S


@pytest.mark.parametrize("Q", [1, 7, 16, 64])
def test_chunked_form_agrees_with_recurrence(Q):
    x, dt, A, B, C, D = wl.random_ssd(2, 50, 4, 8, 2, 16, seed=83)
    y, S = oracle.ssd_scan(x, dt, A, B, C, D)
    yc, Sc = chunked_reference(x, dt, A, B, C, D, Q)
    np.testing.assert_allclose(y, yc, atol=1e-10, rtol=1e-10)
    np.testing.assert_allclose(S, Sc, atol=1e-10, rtol=1e-10)


def test_heads_use_contiguous_groups():
    x, dt, A, B, C, D = wl.random_ssd(1, 24, 4, 8, 2, 16, seed=84)
    y, _ = oracle.ssd_scan(x, dt, A, B, C, D)
    # heads 2, 3 use group 1
    y1, _ = oracle.ssd_scan(x[:, :, 2:].contiguous(), dt[:, :, 2:].contiguous(), A[2:].contiguous(),
                            B[:, :, 1:].contiguous(), C[:, :, 1:].contiguous(), D[2:].contiguous())
    np.testing.assert_array_equal(y[:, :, 2:], y1)
