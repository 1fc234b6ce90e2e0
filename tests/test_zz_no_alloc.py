"""mla_decode_noalloc: MLA decode for callers that cannot allocate device memory.

Such callers (a serving loop with a fixed device-memory plan, code that must
not synchronise the device, plain C callers without an allocator) get the same
computation through an entry point that takes no workspace and uses the
library's built-in scratch array.  This test calls it through the C ABI and
checks it against mla_decode, the entry point with a caller-provided
workspace, on two calls in a row with different inputs, so that a second call
reading stale scratch left by the first would fail.  Both entry points run the
same kernels with the same split plan, so the outputs must agree bit for bit.
It also checks the entry point's one promise: once the library is loaded, a
call changes the device's free memory by nothing.

The file name makes pytest collect it last: a run that stops at the first
failure has already run every other test.
"""
import pytest
import torch

import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import workloads as wl
from tests._util import build_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()
    gb.load_library()


def _bits(t):
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # (B, N_kv, seed): the B=64, N_kv=4096 decode shape (split sequences, so the
    # scratch is used), then a ragged one
    for B, N_kv, seed in [(64, 4096, 11), (3, 1000, 12)]:
        Qn, Qp, KV, Kp = (x.cuda() for x in wl.random_mla(B, 128, N_kv, 512, 64, seed=seed))
        O_ref, L_ref = gb.mla_decode(Qn, Qp, KV, Kp)
        O = torch.full_like(O_ref, float("nan"))
        L = torch.full_like(L_ref, float("nan"))
        gb.mla_decode_noalloc(Qn, Qp, KV, Kp, O=O, LSE=L)
        gb.check()
        assert torch.isfinite(O.float()).all() and torch.isfinite(L).all()
        assert torch.equal(_bits(O), _bits(O_ref)), (B, N_kv, (O.float() - O_ref.float()).abs().max().item())
        assert torch.equal(_bits(L), _bits(L_ref)), (B, N_kv, (L - L_ref).abs().max().item())


def test_noalloc_call_allocates_no_device_memory():
    B, N_kv = 64, 4096
    Qn, Qp, KV, Kp = (x.cuda() for x in wl.random_mla(B, 128, N_kv, 512, 64, seed=13))
    O = torch.empty(B, 128, 512, dtype=torch.bfloat16, device="cuda")
    L = torch.empty(B, 128, dtype=torch.float32, device="cuda")
    gb.mla_decode_noalloc(Qn, Qp, KV, Kp, O=O, LSE=L)     # loads the module and looks up the scratch
    gb.check()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        gb.mla_decode_noalloc(Qn, Qp, KV, Kp, O=O, LSE=L)
    gb.check()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
