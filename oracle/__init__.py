"""fp64 CPU oracle for fused attention forward (MHA/GQA prefill) and MLA decode.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (``tiled_attention_flashattention_gb300``) never imports it and
shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, one query row at a time:
full score row, explicit two-pass softmax, weighted sum of value rows).  This
module only compiles that file with gcc and marshals arguments through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, D, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_int64
            lib.oracle_attn_fwd.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, D, P, I64, I]
            lib.oracle_attn_fwd.restype = I
            lib.oracle_attn_fwd_masked.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, D, P, I, P, I64, I]
            lib.oracle_attn_fwd_masked.restype = I
            lib.oracle_ssd_scan.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I]
            lib.oracle_ssd_scan.restype = I
            lib.oracle_mla_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, D, P, I64, I]
            lib.oracle_mla_decode.restype = I
            lib.oracle_mla_decode_paged.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, D, P, I64, I]
            lib.oracle_mla_decode_paged.restype = I
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _bf16_bits(t) -> np.ndarray:
    """Contiguous uint16 view of a bf16 CPU tensor (the exact bit patterns)."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    assert t.dtype == torch.bfloat16, t.dtype
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attn_fwd(Q, K, V, causal: bool, window: int, scale: float, rows=None,
             return_probs: bool = False, threads: int | None = None, block_mask=None, block: int = 128):
    """Reference attention for bf16 Q [B,H,N_q,d], K/V [B,H_kv,N_kv,d].

    Returns (O, LSE[, P]) as float64 numpy arrays.  With ``rows`` (flat indices
    (b*H + h)*N_q + i) only those rows are computed: O is [len(rows), d] and LSE
    [len(rows)].  Without it, O is [B,H,N_q,d] and LSE [B,H,N_q].  ``block_mask``
    (uint8 [B,H,ceil(N_q/block),ceil(N_kv/block)]) removes the keys of every
    zero block from its query rows.
    """
    B, H, N_q, d = Q.shape
    _, H_kv, N_kv, _ = K.shape
    q, k, v = _bf16_bits(Q), _bf16_bits(K), _bf16_bits(V)
    if rows is None:
        n = B * H * N_q
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows_arr.shape[0]
    O = np.zeros((n, d), dtype=np.float64)
    LSE = np.zeros((n,), dtype=np.float64)
    P = np.zeros((n, N_kv), dtype=np.float64) if return_probs else None
    mask = None
    if block_mask is not None:
        mask = np.ascontiguousarray(np.asarray(block_mask, dtype=np.uint8))
        want = (B, H, -(-N_q // block), -(-N_kv // block))
        if mask.shape != want:
            raise ValueError(f"block_mask must have shape {want}, got {mask.shape}")
    rc = _load().oracle_attn_fwd_masked(
        _ptr(q), _ptr(k), _ptr(v), _ptr(O), _ptr(LSE), _ptr(P) if P is not None else None,
        B, H, H_kv, N_q, N_kv, d, int(bool(causal)), int(window), float(scale),
        _ptr(mask) if mask is not None else None, int(block),
        _ptr(rows_arr) if rows_arr is not None else None, n, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    if rows is None:
        O = O.reshape(B, H, N_q, d)
        LSE = LSE.reshape(B, H, N_q)
        if P is not None:
            P = P.reshape(B, H, N_q, N_kv)
    return (O, LSE, P) if return_probs else (O, LSE)


def mla_decode(Q_nope, Q_pe, KV_latent, K_pe, scale: float, rows=None, threads: int | None = None):
    """Reference MLA decode: Q_nope [B,H,d_c], Q_pe [B,H,d_r], KV_latent [B,N_kv,d_c],
    K_pe [B,N_kv,d_r] (bf16).  Returns (O [B,H,d_c], LSE [B,H]) float64, or the
    listed flat rows b*H + h only."""
    B, H, d_c = Q_nope.shape
    d_r = Q_pe.shape[-1]
    N_kv = KV_latent.shape[1]
    qn, qp, kv, kp = (_bf16_bits(x) for x in (Q_nope, Q_pe, KV_latent, K_pe))
    if rows is None:
        n = B * H
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows_arr.shape[0]
    O = np.zeros((n, d_c), dtype=np.float64)
    LSE = np.zeros((n,), dtype=np.float64)
    rc = _load().oracle_mla_decode(
        _ptr(qn), _ptr(qp), _ptr(kv), _ptr(kp), _ptr(O), _ptr(LSE), B, H, N_kv, d_c, d_r,
        float(scale), _ptr(rows_arr) if rows_arr is not None else None, n,
        threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_mla_decode rejected its arguments")
    if rows is None:
        O = O.reshape(B, H, d_c)
        LSE = LSE.reshape(B, H)
    return O, LSE


def mla_decode_paged(Q_nope, Q_pe, KV_cache, K_pe_cache, block_table, seqlens, scale: float, rows=None,
                     threads: int | None = None):
    """Reference MLA decode over a paged KV cache: Q_nope [B,H,d_c] or [B,s_q,H,d_c],
    Q_pe [B,(s_q,)H,d_r] (bf16), KV_cache [num_pages,page,d_c], K_pe_cache
    [num_pages,page,d_r] (bf16), block_table [B,max_pages] and seqlens [B] (int32).
    Key j of sequence b is row j % page of page block_table[b, j // page]; query
    token t of s_q sees keys j < seqlens[b] - (s_q - 1 - t).  Returns (O, LSE)
    float64 shaped like Q_nope (last dim d_c) and Q_nope without its last dim, or
    the listed flat rows (b*s_q + t)*H + h only."""
    multi = Q_nope.dim() == 4
    if multi:
        B, s_q, H, d_c = Q_nope.shape
    else:
        B, H, d_c = Q_nope.shape
        s_q = 1
    d_r = Q_pe.shape[-1]
    num_pages, page, _ = KV_cache.shape
    max_pages = block_table.shape[1]
    qn, qp, kv, kp = (_bf16_bits(x) for x in (Q_nope, Q_pe, KV_cache, K_pe_cache))
    table = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    if rows is None:
        n = B * H
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows_arr.shape[0]
    if rows is None:
        n = B * s_q * H
    O = np.zeros((n, d_c), dtype=np.float64)
    LSE = np.zeros((n,), dtype=np.float64)
    rc = _load().oracle_mla_decode_paged(
        _ptr(qn), _ptr(qp), _ptr(kv), _ptr(kp), _ptr(table), _ptr(lens), _ptr(O), _ptr(LSE), B, s_q, H,
        num_pages, max_pages, page, d_c, d_r, float(scale),
        _ptr(rows_arr) if rows_arr is not None else None, n, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_mla_decode_paged rejected its arguments")
    if rows is None:
        O = O.reshape(B, s_q, H, d_c) if multi else O.reshape(B, H, d_c)
        LSE = LSE.reshape(B, s_q, H) if multi else LSE.reshape(B, H)
    return O, LSE


def ssd_scan(x, dt, A, B, C, D=None, threads: int | None = None):
    """Reference Mamba-2 SSD scan (plain recurrence in fp64): x [Bsz,L,H,P] bf16,
    dt [Bsz,L,H] fp32, A [H] fp32, B, C [Bsz,L,G,N] bf16, D [H] fp32 or None.
    Returns (y [Bsz,L,H,P], final state [Bsz,H,P,N]) as float64 numpy arrays."""
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    xb, Bb, Cb = _bf16_bits(x), _bf16_bits(B), _bf16_bits(C)
    f32 = lambda t: np.ascontiguousarray(t.detach().cpu().to(torch.float32).numpy())
    dtn, An = f32(dt), f32(A)
    Dn = f32(D) if D is not None else None
    y = np.zeros((Bsz, L, H, P), dtype=np.float64)
    S = np.zeros((Bsz, H, P, N), dtype=np.float64)
    rc = _load().oracle_ssd_scan(_ptr(xb), _ptr(dtn), _ptr(An), _ptr(Bb), _ptr(Cb),
                                 _ptr(Dn) if Dn is not None else None, _ptr(y), _ptr(S),
                                 Bsz, L, H, P, G, N, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_ssd_scan rejected its arguments")
    return y, S
