"""GB300-native fused attention forward: tiled FlashAttention prefill and MLA decode.

A thin ctypes binding over ``libgbattn.so`` (C ABI in ``include/gbattn.h``).
The functions here only marshal arguments: they check tensor properties,
allocate outputs with torch when the caller gives none, and pass raw device
pointers and the current CUDA stream to the library.  Every arithmetic step
runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and a
missing library is an error.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = ["attn_fwd", "attn_fwd_sparse", "mla_decode", "mla_decode_workspace_bytes", "mla_decode_paged",
           "mla_decode_paged_workspace_bytes", "mla_decode_noalloc", "ssd_scan", "attn_fwd_host",
           "attn_fwd_host_device_bytes", "mla_decode_host", "mla_decode_host_device_bytes",
           "check", "selftest_umma", "mla_trace", "MLA_TRACE_EVENTS", "attn_trace", "ATTN_TRACE_EVENTS",
           "set_wait_timeout_ns", "set_fault_injection", "GbattnError", "library_path", "load_library"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libgbattn.so")
_LIB_TRACE_PATH = os.path.join(_PKG, "libgbattn_trace.so")
_lib = None
_lib_trace = False
_lock = threading.Lock()

_STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "ALIGNMENT", 4: "WORKSPACE", 5: "LAUNCH",
           6: "TIMEOUT", 7: "ARCH"}


class GbattnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"gbattn {_STATUS.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load_library(trace: bool = False):
    """Load libgbattn.so (built by ``__graft_entry__.build()``), or with
    trace=True the trace build libgbattn_trace.so (``_build.build(trace=True)``);
    one of the two per process.  Raise if it is missing."""
    global _lib, _lib_trace
    with _lock:
        if _lib is not None:
            if trace and not _lib_trace:
                raise RuntimeError("the default library is already loaded in this process; "
                                   "load the trace build first, in a process of its own")
            return _lib
        path = _LIB_TRACE_PATH if trace else _LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()'" +
                               (", then _build.build(trace=True))" if trace else ")"))
        lib = ctypes.CDLL(path)
        P, I, F, SZ, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
        lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P]
        lib.attn_fwd.restype = I
        lib.attn_fwd_sparse.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, P]
        lib.attn_fwd_sparse.restype = I
        lib.mla_decode_workspace_bytes.argtypes = [I, I, I, I]
        lib.mla_decode_workspace_bytes.restype = SZ
        lib.mla_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, P, SZ, P]
        lib.mla_decode.restype = I
        lib.mla_decode_paged_workspace_bytes.argtypes = [I, I, I, I]
        lib.mla_decode_paged_workspace_bytes.restype = SZ
        lib.mla_decode_paged.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, SZ, P]
        lib.mla_decode_paged.restype = I
        lib.ssd_scan.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P]
        lib.attn_fwd_host_device_bytes.argtypes = [I, I, I, I, I, I]
        lib.attn_fwd_host_device_bytes.restype = SZ
        lib.attn_fwd_host.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, SZ, P]
        lib.attn_fwd_host.restype = I
        lib.mla_decode_host_device_bytes.argtypes = [I, I, I, I, I]
        lib.mla_decode_host_device_bytes.restype = SZ
        lib.mla_decode_host.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, P, SZ, P]
        lib.mla_decode_host.restype = I
        lib.ssd_scan.restype = I
        lib.mla_decode_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, P]
        lib.mla_decode_noalloc.restype = I
        lib.gbattn_check.argtypes = [P]
        lib.gbattn_check.restype = I
        lib.gbattn_last_error.argtypes = []
        lib.gbattn_last_error.restype = ctypes.c_char_p
        lib.gbattn_set_wait_timeout_ns.argtypes = [U64]
        lib.gbattn_set_wait_timeout_ns.restype = U64
        lib.gbattn_set_fault_injection.argtypes = [I]
        lib.gbattn_set_fault_injection.restype = I
        lib.gbattn_selftest_umma.argtypes = [P, P, P, P, P, P, P]
        lib.gbattn_selftest_umma.restype = I
        lib.gbattn_mla_trace.argtypes = [P, SZ]
        lib.gbattn_mla_trace.restype = I
        lib.gbattn_attn_trace.argtypes = [P, SZ]
        lib.gbattn_attn_trace.restype = I
        _lib = lib
        _lib_trace = trace
        return lib


def _raise_if(rc: int):
    if rc != 0:
        msg = load_library().gbattn_last_error().decode(errors="replace")
        raise GbattnError(rc, msg)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_host(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _need(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def attn_fwd(Q, K, V, causal: bool = False, window: int = 0, scale: float | None = None,
             O=None, LSE=None, stream=None):
    """Fused attention forward.  Q [B,H,N_q,d], K/V [B,H_kv,N_kv,d] bf16 CUDA tensors.

    Returns (O [B,H,N_q,d] bf16, LSE [B,H,N_q] fp32).  With i' = i + N_kv - N_q,
    ``window > 0`` keeps keys j in [i' - window + 1, i'] when causal, and the
    symmetric band [i' - window, i' + window] when not.
    Asynchronous on ``stream`` (default: torch's current stream).
    """
    lib = load_library()
    if Q.dim() != 4 or K.dim() != 4 or V.dim() != 4:
        raise ValueError("Q, K, V must be 4-D [B, H, N, d]")
    B, H, N_q, d = Q.shape
    _, H_kv, N_kv, _ = K.shape
    _need(Q, "Q", torch.bfloat16, None)
    _need(K, "K", torch.bfloat16, (B, H_kv, N_kv, d))
    _need(V, "V", torch.bfloat16, (B, H_kv, N_kv, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if O is None:
        O = torch.empty((B, H, N_q, d), dtype=torch.bfloat16, device=Q.device)
    if LSE is None:
        LSE = torch.empty((B, H, N_q), dtype=torch.float32, device=Q.device)
    _need(O, "O", torch.bfloat16, (B, H, N_q, d))
    _need(LSE, "LSE", torch.float32, (B, H, N_q))
    rc = lib.attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, H_kv, N_q, N_kv, d,
                      int(bool(causal)), int(window), float(scale), ctypes.c_void_p(_stream_handle(stream)))
    _raise_if(rc)
    return O, LSE


def attn_fwd_sparse(Q, K, V, block_mask, causal: bool = False, window: int = 0, scale: float | None = None,
                    O=None, LSE=None, stream=None):
    """attn_fwd with a block-sparse mask: block_mask uint8 [B,H,ceil(N_q/128),ceil(N_kv/128)]
    (CUDA); a zero byte removes those 128 keys from those 128 query rows (on top
    of causal / window).  Skipped blocks are neither loaded nor computed."""
    lib = load_library()
    if Q.dim() != 4 or K.dim() != 4 or V.dim() != 4:
        raise ValueError("Q, K, V must be 4-D [B, H, N, d]")
    B, H, N_q, d = Q.shape
    _, H_kv, N_kv, _ = K.shape
    _need(Q, "Q", torch.bfloat16, None)
    _need(K, "K", torch.bfloat16, (B, H_kv, N_kv, d))
    _need(V, "V", torch.bfloat16, (B, H_kv, N_kv, d))
    _need(block_mask, "block_mask", torch.uint8, (B, H, -(-N_q // 128), -(-N_kv // 128)))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if O is None:
        O = torch.empty((B, H, N_q, d), dtype=torch.bfloat16, device=Q.device)
    if LSE is None:
        LSE = torch.empty((B, H, N_q), dtype=torch.float32, device=Q.device)
    _need(O, "O", torch.bfloat16, (B, H, N_q, d))
    _need(LSE, "LSE", torch.float32, (B, H, N_q))
    rc = lib.attn_fwd_sparse(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(block_mask), B, H, H_kv, N_q, N_kv,
                             d, int(bool(causal)), int(window), float(scale), ctypes.c_void_p(_stream_handle(stream)))
    _raise_if(rc)
    return O, LSE


def mla_decode_workspace_bytes(B: int, H: int, N_kv: int, d_c: int = 512) -> int:
    return int(load_library().mla_decode_workspace_bytes(B, H, N_kv, d_c))


def mla_decode(Q_nope, Q_pe, KV_latent, K_pe, scale: float | None = None, O=None, LSE=None,
               workspace=None, stream=None):
    """MLA decode.  Q_nope [B,H,d_c], Q_pe [B,H,d_r], KV_latent [B,N_kv,d_c], K_pe [B,N_kv,d_r] bf16.

    Returns (O [B,H,d_c] bf16, LSE [B,H] fp32).  ``workspace`` (a uint8 CUDA
    tensor of at least ``mla_decode_workspace_bytes`` bytes) is allocated when
    not given.
    """
    lib = load_library()
    B, H, d_c = Q_nope.shape
    d_r = Q_pe.shape[-1]
    N_kv = KV_latent.shape[1]
    _need(Q_nope, "Q_nope", torch.bfloat16, None)
    _need(Q_pe, "Q_pe", torch.bfloat16, (B, H, d_r))
    _need(KV_latent, "KV_latent", torch.bfloat16, (B, N_kv, d_c))
    _need(K_pe, "K_pe", torch.bfloat16, (B, N_kv, d_r))
    if scale is None:
        scale = 1.0 / math.sqrt(d_c + d_r)
    if O is None:
        O = torch.empty((B, H, d_c), dtype=torch.bfloat16, device=Q_nope.device)
    if LSE is None:
        LSE = torch.empty((B, H), dtype=torch.float32, device=Q_nope.device)
    _need(O, "O", torch.bfloat16, (B, H, d_c))
    _need(LSE, "LSE", torch.float32, (B, H))
    need = int(lib.mla_decode_workspace_bytes(B, H, N_kv, d_c))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=Q_nope.device)
    _need(workspace, "workspace", torch.uint8, None)
    rc = lib.mla_decode(_ptr(Q_nope), _ptr(Q_pe), _ptr(KV_latent), _ptr(K_pe), _ptr(O), _ptr(LSE),
                        B, H, N_kv, d_c, d_r, float(scale), _ptr(workspace), workspace.numel(),
                        ctypes.c_void_p(_stream_handle(stream)))
    _raise_if(rc)
    return O, LSE


def mla_decode_paged_workspace_bytes(B: int, s_q: int = 1, H: int = 128, d_c: int = 512) -> int:
    return int(load_library().mla_decode_paged_workspace_bytes(B, s_q, H, d_c))


def mla_decode_paged(Q_nope, Q_pe, KV_cache, K_pe_cache, block_table, cache_seqlens, scale: float | None = None,
                     O=None, LSE=None, workspace=None, stream=None):
    """MLA decode over a paged KV cache with per-sequence lengths.

    Q_nope [B,H,d_c] or [B,s_q,H,d_c], Q_pe [B,(s_q,)H,d_r], KV_cache
    [num_pages,64,d_c], K_pe_cache [num_pages,64,d_r] (bf16); block_table
    [B,max_pages] and cache_seqlens [B] (int32), all CUDA tensors.  Key j of
    sequence b is row j % 64 of page block_table[b, j // 64]; with s_q query
    tokens, token t sees keys j < len - (s_q - 1 - t).  Returns (O, LSE), O
    bf16 shaped like Q_nope with last dim d_c, LSE fp32 without it.
    """
    lib = load_library()
    multi = Q_nope.dim() == 4
    if multi:
        B, s_q, H, d_c = Q_nope.shape
    else:
        (B, H, d_c), s_q = Q_nope.shape, 1
    lead = (B, s_q, H) if multi else (B, H)
    d_r = Q_pe.shape[-1]
    num_pages, page, _ = KV_cache.shape
    max_pages = block_table.shape[1]
    _need(Q_nope, "Q_nope", torch.bfloat16, None)
    _need(Q_pe, "Q_pe", torch.bfloat16, (*lead, d_r))
    _need(KV_cache, "KV_cache", torch.bfloat16, (num_pages, page, d_c))
    _need(K_pe_cache, "K_pe_cache", torch.bfloat16, (num_pages, page, d_r))
    _need(block_table, "block_table", torch.int32, (B, max_pages))
    _need(cache_seqlens, "cache_seqlens", torch.int32, (B,))
    if scale is None:
        scale = 1.0 / math.sqrt(d_c + d_r)
    if O is None:
        O = torch.empty((*lead, d_c), dtype=torch.bfloat16, device=Q_nope.device)
    if LSE is None:
        LSE = torch.empty(lead, dtype=torch.float32, device=Q_nope.device)
    _need(O, "O", torch.bfloat16, (*lead, d_c))
    _need(LSE, "LSE", torch.float32, lead)
    need = int(lib.mla_decode_paged_workspace_bytes(B, s_q, H, d_c))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=Q_nope.device)
    _need(workspace, "workspace", torch.uint8, None)
    rc = lib.mla_decode_paged(_ptr(Q_nope), _ptr(Q_pe), _ptr(KV_cache), _ptr(K_pe_cache), _ptr(block_table),
                              _ptr(cache_seqlens), _ptr(O), _ptr(LSE), B, s_q, H, num_pages, max_pages, page, d_c,
                              d_r, float(scale), _ptr(workspace), workspace.numel(),
                              ctypes.c_void_p(_stream_handle(stream)))
    _raise_if(rc)
    return O, LSE


def attn_fwd_host_device_bytes(B: int, H: int, H_kv: int, N_q: int, N_kv: int, d: int) -> int:
    return int(load_library().attn_fwd_host_device_bytes(B, H, H_kv, N_q, N_kv, d))


def attn_fwd_host(Q, K, V, causal: bool = False, window: int = 0, scale: float | None = None, O=None, LSE=None,
                  device_buf=None, stream=None):
    """attn_fwd with host (CPU, ideally pinned) tensors; copies, kernels and copies
    back are pipelined by the library.  Returns host (O, LSE); they are valid once
    the stream reaches the call (``check()`` synchronises)."""
    lib = load_library()
    B, H, N_q, d = Q.shape
    H_kv, N_kv = K.shape[1], K.shape[2]
    _need_host(Q, "Q", torch.bfloat16, None)
    _need_host(K, "K", torch.bfloat16, (B, H_kv, N_kv, d))
    _need_host(V, "V", torch.bfloat16, (B, H_kv, N_kv, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = Q.is_pinned()
    if O is None:
        O = torch.empty((B, H, N_q, d), dtype=torch.bfloat16, pin_memory=pin)
    if LSE is None:
        LSE = torch.empty((B, H, N_q), dtype=torch.float32, pin_memory=pin)
    _need_host(O, "O", torch.bfloat16, (B, H, N_q, d))
    _need_host(LSE, "LSE", torch.float32, (B, H, N_q))
    if device_buf is None:
        device_buf = torch.empty(max(attn_fwd_host_device_bytes(B, H, H_kv, N_q, N_kv, d), 256), dtype=torch.uint8,
                                 device="cuda")
    _need(device_buf, "device_buf", torch.uint8, None)
    rc = lib.attn_fwd_host(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, H_kv, N_q, N_kv, d,
                           1 if causal else 0, int(window), float(scale), _ptr(device_buf), device_buf.numel(),
                           ctypes.c_void_p(_stream_handle(stream)))
    _raise_if(rc)
    return O, LSE


def mla_decode_host_device_bytes(B: int, H: int = 128, N_kv: int = 4096, d_c: int = 512, d_r: int = 64) -> int:
    return int(load_library().mla_decode_host_device_bytes(B, H, N_kv, d_c, d_r))


def mla_decode_host(Q_nope, Q_pe, KV_latent, K_pe, scale: float | None = None, O=None, LSE=None, device_buf=None,
                    stream=None):
    """mla_decode with host (CPU, ideally pinned) tensors, pipelined by the library.
    Returns host (O, LSE), valid once the stream reaches the call."""
    lib = load_library()
    B, H, d_c = Q_nope.shape
    d_r = Q_pe.shape[-1]
    N_kv = KV_latent.shape[1]
    _need_host(Q_nope, "Q_nope", torch.bfloat16, None)
    _need_host(Q_pe, "Q_pe", torch.bfloat16, (B, H, d_r))
    _need_host(KV_latent, "KV_latent", torch.bfloat16, (B, N_kv, d_c))
    _need_host(K_pe, "K_pe", torch.bfloat16, (B, N_kv, d_r))
    if scale is None:
        scale = 1.0 / math.sqrt(d_c + d_r)
    pin = Q_nope.is_pinned()
    if O is None:
        O = torch.empty((B, H, d_c), dtype=torch.bfloat16, pin_memory=pin)
    if LSE is None:
        LSE = torch.empty((B, H), dtype=torch.float32, pin_memory=pin)
    _need_host(O, "O", torch.bfloat16, (B, H, d_c))
    _need_host(LSE, "LSE", torch.float32, (B, H))
    if device_buf is None:
        device_buf = torch.empty(max(mla_decode_host_device_bytes(B, H, N_kv, d_c, d_r), 256), dtype=torch.uint8,
                                 device="cuda")
    _need(device_buf, "device_buf", torch.uint8, None)
    rc = lib.mla_decode_host(_ptr(Q_nope), _ptr(Q_pe), _ptr(KV_latent), _ptr(K_pe), _ptr(O), _ptr(LSE), B, H, N_kv,
                             d_c, d_r, float(scale), _ptr(device_buf), device_buf.numel(),
                             ctypes.c_void_p(_stream_handle(stream)))
    _raise_if(rc)
    return O, LSE


def ssd_scan(x, dt, A, B, C, D=None, y=None, final_state=None, want_final_state: bool = False, stream=None):
    """Mamba-2 SSD scan.  x [Bsz,L,H,P] bf16, dt [Bsz,L,H] fp32, A [H] fp32, B, C
    [Bsz,L,G,N] bf16, D [H] fp32 or None (CUDA tensors).  Returns y [Bsz,L,H,P]
    fp32, and the final state [Bsz,H,P,N] fp32 when asked for."""
    lib = load_library()
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    _need(x, "x", torch.bfloat16, None)
    _need(dt, "dt", torch.float32, (Bsz, L, H))
    _need(A, "A", torch.float32, (H,))
    _need(B, "B", torch.bfloat16, (Bsz, L, G, N))
    _need(C, "C", torch.bfloat16, (Bsz, L, G, N))
    if D is not None:
        _need(D, "D", torch.float32, (H,))
    if y is None:
        y = torch.empty((Bsz, L, H, P), dtype=torch.float32, device=x.device)
    _need(y, "y", torch.float32, (Bsz, L, H, P))
    if want_final_state and final_state is None:
        final_state = torch.empty((Bsz, H, P, N), dtype=torch.float32, device=x.device)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, (Bsz, H, P, N))
    rc = lib.ssd_scan(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D) if D is not None else None, _ptr(y),
                      _ptr(final_state) if final_state is not None else None, Bsz, L, H, P, G, N,
                      ctypes.c_void_p(_stream_handle(stream)))
    _raise_if(rc)
    return (y, final_state) if final_state is not None else y


def mla_decode_noalloc(Q_nope, Q_pe, KV_latent, K_pe, scale: float | None = None, O=None, LSE=None,
                       stream=None):
    """MLA decode through the library's built-in scratch: no workspace argument.

    For callers that cannot allocate device memory at call time (a fixed
    device-memory plan, no device synchronisation allowed).  The C call
    allocates nothing; pass preallocated O and LSE so that this wrapper does
    not allocate them with torch either.  Calls whose kernels overlap on the
    GPU race on the shared scratch, so serialise them.
    """
    lib = load_library()
    B, H, d_c = Q_nope.shape
    d_r = Q_pe.shape[-1]
    N_kv = KV_latent.shape[1]
    _need(Q_nope, "Q_nope", torch.bfloat16, None)
    _need(Q_pe, "Q_pe", torch.bfloat16, (B, H, d_r))
    _need(KV_latent, "KV_latent", torch.bfloat16, (B, N_kv, d_c))
    _need(K_pe, "K_pe", torch.bfloat16, (B, N_kv, d_r))
    if scale is None:
        scale = 1.0 / math.sqrt(d_c + d_r)
    if O is None:
        O = torch.empty((B, H, d_c), dtype=torch.bfloat16, device=Q_nope.device)
    if LSE is None:
        LSE = torch.empty((B, H), dtype=torch.float32, device=Q_nope.device)
    _need(O, "O", torch.bfloat16, (B, H, d_c))
    _need(LSE, "LSE", torch.float32, (B, H))
    rc = lib.mla_decode_noalloc(_ptr(Q_nope), _ptr(Q_pe), _ptr(KV_latent), _ptr(K_pe), _ptr(O), _ptr(LSE),
                                B, H, N_kv, d_c, d_r, float(scale), ctypes.c_void_p(_stream_handle(stream)))
    _raise_if(rc)
    return O, LSE


def check(stream=None):
    """Synchronise the stream and raise GbattnError if a kernel's bounded wait ran out."""
    _raise_if(load_library().gbattn_check(ctypes.c_void_p(_stream_handle(stream))))


def set_wait_timeout_ns(ns: int) -> int:
    return int(load_library().gbattn_set_wait_timeout_ns(int(ns)))


def set_fault_injection(mode: int) -> int:
    """Test hook: 1 makes later attn_fwd launches time out on purpose (see gbattn.h)."""
    return int(load_library().gbattn_set_fault_injection(int(mode)))


def selftest_umma(A, B, P, V, stream=None):
    """One-tile tensor-core layout check: returns (S = A B^T, O = P V) in fp32."""
    lib = load_library()
    for name, t in (("A", A), ("B", B), ("P", P), ("V", V)):
        _need(t, name, torch.bfloat16, (128, 128))
    S = torch.empty((128, 128), dtype=torch.float32, device=A.device)
    O = torch.empty((128, 128), dtype=torch.float32, device=A.device)
    rc = lib.gbattn_selftest_umma(_ptr(A), _ptr(B), _ptr(P), _ptr(V), _ptr(S), _ptr(O),
                                  ctypes.c_void_p(_stream_handle(stream)))
    _raise_if(rc)
    return S, O


# Layout of gbattn_mla_trace (include/gbattn.h): [2 CTAs][events][64 tiles] of
# global-timer ns, 0 where a step was not reached.
MLA_TRACE_EVENTS = ("load", "s_issue", "pv0_issue", "pv1_issue", "s_read", "send_buf0_free", "send_buf1_free",
                    "copy0_issue", "copy1_issue", "softmax0_in", "softmax1_in", "p0_ready", "p1_ready")
_MLA_TRACE_TILES = 64


def mla_trace():
    """Stamps of the MLA decode launches since the last call (trace build only:
    ``load_library(trace=True)``), as a uint64 numpy array [2, 13, 64]; clears them."""
    import numpy as np
    buf = np.zeros((2, len(MLA_TRACE_EVENTS), _MLA_TRACE_TILES), dtype=np.uint64)
    _raise_if(load_library().gbattn_mla_trace(ctypes.c_void_p(buf.ctypes.data), buf.nbytes))
    return buf


# Layout of gbattn_attn_trace (include/gbattn.h): int64 [4 CTAs][events][132
# tiles] of SM cycles (0 = not reached), then int64 [4 CTAs][4]: cycles and ns at
# each traced CTA's start and end.  Tile j's "k_next_seen", "s0_next_issued" and
# "s1_next_issued" refer to key tile j + 1.
ATTN_TRACE_EVENTS = ("wait_v", "v_seen", "p0_seen", "pv0_issued", "k_next_seen", "s0_next_issued", "p1_seen",
                     "pv1_issued", "s1_next_issued", "s0_seen", "s0_loaded", "max0", "exp0", "p0_arrive", "s1_seen",
                     "s1_loaded", "max1", "exp1", "p1_arrive")
_ATTN_TRACE_CTAS = 4
_ATTN_TRACE_TILES = 132


def attn_trace():
    """Stamps of the dense prefill launches since the last call (trace build
    only: ``load_library(trace=True)``): (cycles int64 [4, 19, 132], clock int64
    [4, 4]); clears them."""
    import numpy as np
    n0 = _ATTN_TRACE_CTAS * len(ATTN_TRACE_EVENTS) * _ATTN_TRACE_TILES
    buf = np.zeros(n0 + _ATTN_TRACE_CTAS * 4, dtype=np.int64)
    _raise_if(load_library().gbattn_attn_trace(ctypes.c_void_p(buf.ctypes.data), buf.nbytes))
    return (buf[:n0].reshape(_ATTN_TRACE_CTAS, len(ATTN_TRACE_EVENTS), _ATTN_TRACE_TILES),
            buf[n0:].reshape(_ATTN_TRACE_CTAS, 4))
