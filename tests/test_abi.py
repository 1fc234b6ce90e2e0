"""The C-ABI library builds, loads, exports every declared entry point, and
rejects bad arguments before touching the GPU (so these run without one).
Every call below with placeholder addresses must be rejected before a launch:
on a machine with a GPU anything else would run a kernel on them."""
import ctypes
import os
import re

import pytest

from tests._util import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbattn.h")


@pytest.fixture(scope="module")
def lib():
    path = build_lib()
    import tiled_attention_flashattention_gb300 as g
    assert os.path.samefile(path, g.library_path())
    return g.load_library()


def _gpu_present() -> bool:
    """Only argument checks that fail before any launch may run where a GPU is:
    the placeholder addresses below are not device memory."""
    import torch
    return torch.cuda.is_available()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "mla_decode", "mla_decode_workspace_bytes", "gbattn_check",
              "gbattn_last_error", "gbattn_set_wait_timeout_ns", "gbattn_selftest_umma"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"libgbattn.so does not export {n}"


def _attn(lib, Q=16, K=16, V=16, O=16, LSE=16, B=1, H=2, H_kv=2, N_q=8, N_kv=8, d=64, causal=0,
          window=0, scale=0.125):
    vp = ctypes.c_void_p
    return lib.attn_fwd(vp(Q), vp(K), vp(V), vp(O), vp(LSE), B, H, H_kv, N_q, N_kv, d, causal, window,
                        ctypes.c_float(scale), None)


def test_attn_fwd_argument_errors(lib):
    assert _attn(lib, H=3, H_kv=2) == 1                     # H % H_kv
    assert _attn(lib, B=-1) == 1
    assert _attn(lib, causal=2) == 1
    assert _attn(lib, scale=0.0) == 1
    assert _attn(lib, scale=float("nan")) == 1
    assert _attn(lib, d=96) == 2                            # unsupported head dim
    assert _attn(lib, window=4, causal=0, Q=0) == 1         # a symmetric window is accepted: the null Q is the error
    assert _attn(lib, Q=0) == 1                             # null pointer
    assert _attn(lib, K=24) == 3                            # misaligned
    assert _attn(lib, LSE=18) == 3
    assert b"16-byte" in lib.gbattn_last_error() or b"aligned" in lib.gbattn_last_error()


def test_attn_fwd_sparse_argument_errors(lib):
    vp = ctypes.c_void_p

    def sparse(mask=16, d=64, causal=0, H=2, H_kv=2, K=16):
        return lib.attn_fwd_sparse(vp(16), vp(K), vp(16), vp(16), vp(16), vp(mask), 1, H, H_kv, 8, 8, d, causal, 0,
                                   ctypes.c_float(0.125), None)
    assert sparse(mask=0) == 1                     # null mask with keys present
    assert sparse(d=96) == 2
    assert sparse(causal=3) == 1
    assert sparse(H=3, H_kv=2) == 1
    assert sparse(K=24) == 3


def test_mla_decode_argument_errors(lib):
    vp = ctypes.c_void_p

    def mla(H=128, d_c=512, d_r=64, N_kv=64, scale=0.04, Qn=16, ws=16, wsb=1 << 20):
        return lib.mla_decode(vp(Qn), vp(16), vp(16), vp(16), vp(16), vp(16), 2, H, N_kv, d_c, d_r,
                              ctypes.c_float(scale), vp(ws), wsb, None)
    assert mla(N_kv=0) == 1
    assert mla(scale=-1.0) == 1
    assert mla(H=256) == 2                         # more than one 128-row tile of heads
    assert mla(d_c=256) == 2
    assert mla(Qn=0) == 1
    assert mla(Qn=40) == 3


def test_mla_decode_paged_argument_errors(lib):
    vp = ctypes.c_void_p

    def paged(B=2, H=128, num_pages=4, max_pages=2, page=64, d_c=512, d_r=64, scale=0.04, Qn=16, table=16,
              lens=16, ws=16):
        return lib.mla_decode_paged(vp(Qn), vp(16), vp(16), vp(16), vp(table), vp(lens), vp(16), vp(16), B, 1, H,
                                    num_pages, max_pages, page, d_c, d_r, ctypes.c_float(scale), vp(ws), 1 << 20,
                                    None)
    assert paged(B=0) == 1
    assert paged(num_pages=0) == 1
    assert paged(scale=0.0) == 1
    assert paged(page=32) == 2                     # page size other than 64
    assert paged(H=256) == 2
    assert paged(table=0) == 1                     # null block table
    assert paged(lens=18) == 3                     # misaligned lengths
    assert paged(Qn=40) == 3


def test_ssd_scan_argument_errors(lib):
    vp = ctypes.c_void_p

    def ssd(Bsz=2, L=100, H=4, P=64, G=2, N=128, x=16, dt=16, D=16, y=16, fs=16):
        return lib.ssd_scan(vp(x), vp(dt), vp(16), vp(16), vp(16), vp(D), vp(y), vp(fs), Bsz, L, H, P, G, N, None)
    assert ssd(Bsz=0) == 1
    assert ssd(L=0) == 1
    assert ssd(G=3) == 1                           # H % G != 0
    assert ssd(P=128) == 2                         # head dim other than 64
    assert ssd(N=64) == 2                          # state dim other than 128
    assert ssd(x=0) == 1
    assert ssd(x=40) == 3                          # misaligned x
    assert ssd(fs=20) == 3                         # misaligned final state
    assert ssd(dt=18) == 3                         # dt not 4-byte aligned
    if not _gpu_present():
        # D and the final state may be omitted: the call passes validation and
        # fails only for want of a device.  (With a GPU present it would launch
        # the kernel on these placeholder addresses; the GPU tests cover it.)
        assert ssd(D=0, fs=0) not in (1, 3)
    assert ssd(Bsz=70000) == 2


def test_host_buffer_entry_point_argument_errors(lib):
    vp = ctypes.c_void_p

    def attn(B=1, H=2, H_kv=1, N_q=64, N_kv=64, d=128, causal=0, scale=0.1, Q=16, buf=256, nbytes=1 << 30):
        return lib.attn_fwd_host(vp(Q), vp(16), vp(16), vp(16), vp(16), B, H, H_kv, N_q, N_kv, d, causal, 0,
                                 ctypes.c_float(scale), vp(buf), nbytes, None)
    assert attn(B=0) == 1
    assert attn(H=3, H_kv=2) == 1
    assert attn(causal=2) == 1
    assert attn(scale=-1.0) == 1
    assert attn(d=96) == 2
    assert attn(Q=0) == 1
    assert attn(buf=0) == 4                        # no device buffer
    assert attn(buf=272) == 4                      # not 256-byte aligned
    assert attn(nbytes=16) == 4                    # too small
    assert lib.attn_fwd_host_device_bytes(1, 2, 1, 64, 64, 128) == 2 * 32768 + 2 * 16384 + 512
    assert lib.attn_fwd_host_device_bytes(0, 2, 1, 64, 64, 128) == 0

    def mla(B=2, H=128, N_kv=64, scale=0.04, Qn=16, buf=256, nbytes=1 << 30):
        return lib.mla_decode_host(vp(Qn), vp(16), vp(16), vp(16), vp(16), vp(16), B, H, N_kv, 512, 64,
                                   ctypes.c_float(scale), vp(buf), nbytes, None)
    assert mla(B=0) == 1
    assert mla(H=256) == 2                         # more than one 128-row tile of heads
    assert mla(scale=0.0) == 1
    assert mla(Qn=0) == 1
    assert mla(buf=0) == 4
    assert mla(nbytes=16) == 4


def test_default_library_has_no_latency_trace(lib):
    # the stamps exist only in the trace build (-DGBATTN_TRACE); the default
    # library answers UNSUPPORTED without touching the device
    assert lib.gbattn_mla_trace(None, 0) == 2
    assert b"GBATTN_TRACE" in lib.gbattn_last_error()
    assert lib.gbattn_attn_trace(None, 0) == 2
    assert b"GBATTN_TRACE" in lib.gbattn_last_error()
