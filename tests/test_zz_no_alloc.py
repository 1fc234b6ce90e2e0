"""mla_decode_noalloc: MLA decode for callers that cannot allocate device memory.

Such callers (a serving loop with a fixed device-memory plan, code that must
not synchronise the device, plain C callers without an allocator) get the same
computation through an entry point that takes no workspace and uses the
library's built-in scratch array.  This test calls it through the C ABI and
checks it against mla_decode, the entry point with a caller-provided
workspace, on two calls in a row with different inputs, so that a second call
reading stale scratch left by the first would fail.

The file name makes pytest collect it last: a run that stops at the first
failure has already run every other test.
"""
import pytest
import torch

import tiled_attention_flashattention_gb300 as gb
from tiled_attention_flashattention_gb300 import workloads as wl
from tests._util import LSE_TOL, O_TOL, build_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib()
    gb.load_library()


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # (B, N_kv, seed): the B=64, N_kv=4096 decode shape, then a ragged one
    for B, N_kv, seed in [(64, 4096, 11), (3, 1000, 12)]:
        Qn, Qp, KV, Kp = (x.cuda() for x in wl.random_mla(B, 128, N_kv, 512, 64, seed=seed))
        O_ref, L_ref = gb.mla_decode(Qn, Qp, KV, Kp)
        O = torch.empty_like(O_ref)
        L = torch.empty_like(L_ref)
        gb.mla_decode_noalloc(Qn, Qp, KV, Kp, O=O, LSE=L)
        gb.check()
        assert torch.isfinite(O.float()).all() and torch.isfinite(L).all()
        do = (O.float() - O_ref.float()).abs().max().item()
        dl = (L - L_ref).abs().max().item()
        assert do <= O_TOL and dl <= LSE_TOL, (B, N_kv, do, dl)
