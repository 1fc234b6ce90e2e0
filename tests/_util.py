"""Shared helpers for the test suite (parity comparison, row sampling)."""
from __future__ import annotations

import numpy as np
import torch

# Parity bar for bf16 inputs with fp32 accumulation, |O - O_ref| and |LSE - LSE_ref|.
O_TOL = 2e-2
LSE_TOL = 1e-3


def build_lib():
    from tiled_attention_flashattention_gb300 import _build
    return _build.build()


def compare(O_gpu, LSE_gpu, O_ref, LSE_ref, o_tol=O_TOL, lse_tol=LSE_TOL, what=""):
    """Element-wise comparison; -inf LSE must match exactly (rows without keys)."""
    O = O_gpu.detach().float().cpu().double().numpy()
    L = LSE_gpu.detach().float().cpu().double().numpy()
    assert O.shape == O_ref.shape, (O.shape, O_ref.shape)
    assert np.isfinite(O).all(), f"{what}: non-finite O"
    neg_ref = np.isneginf(LSE_ref)
    assert (np.isneginf(L) == neg_ref).all(), f"{what}: -inf LSE pattern differs"
    assert np.isfinite(L[~neg_ref]).all(), f"{what}: non-finite LSE"
    do = np.abs(O - O_ref).max() if O.size else 0.0
    dl = np.abs(L[~neg_ref] - LSE_ref[~neg_ref]).max() if (~neg_ref).any() else 0.0
    assert do <= o_tol, f"{what}: max|dO| = {do:.3e} > {o_tol}"
    assert dl <= lse_tol, f"{what}: max|dLSE| = {dl:.3e} > {lse_tol}"
    return do, dl


def sample_rows(B, H, N_q, n_random, seed, tile=128):
    """Flat row indices (b*H + h)*N_q + i: tile edges of a few heads plus random rows."""
    g = np.random.default_rng(seed)
    rows = set()
    heads = [(0, 0), (B - 1, H - 1), (B // 2, H // 2)]
    edges = [0, 1, tile - 1, tile, 2 * tile - 1, 2 * tile, N_q // 2, N_q - tile - 1, N_q - tile,
             N_q - 2, N_q - 1]
    for b, h in heads:
        for i in edges:
            if 0 <= i < N_q:
                rows.add((b * H + h) * N_q + i)
    total = B * H * N_q
    rows.update(int(x) for x in g.integers(0, total, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)
