"""Failure detection on the GPU without a fault: a bounded wait that runs out.

attn_selftest_timeout waits on a barrier nothing arrives at, with a short
limit; the wait gives up, records ATTN_ERR_TIMEOUT and its site in the
workspace status words, and the kernel returns.  attn_check must report it,
clear it, and the context must stay usable.
"""

import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


def test_bounded_wait_reports_timeout_and_context_survives(ea):
    from exact_attention_12_gb300 import _abi
    lib = _abi.lib()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.attn_check(ws.data_ptr(), stream) == _abi.ATTN_OK
    assert lib.attn_selftest_timeout(ws.data_ptr(), 20_000_000, stream) == _abi.ATTN_OK
    st = lib.attn_check(ws.data_ptr(), stream)
    assert st == _abi.ATTN_ERR_TIMEOUT
    assert b"wait site 99" in lib.attn_last_error()
    # read-and-clear: the next check is clean
    assert lib.attn_check(ws.data_ptr(), stream) == _abi.ATTN_OK
    # the context still runs attention correctly
    q, k, v, _ = (t.cuda() for t in workloads.random_case(1, 2, 200, 64, seed=5))
    o, lse = ea.attention_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
