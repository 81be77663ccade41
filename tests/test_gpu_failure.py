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


def _site(lib):
    msg = lib.attn_last_error().decode()
    return int(msg.rsplit("wait site", 1)[1].split()[0])


@pytest.mark.parametrize("which,d,split", [("fwd", 64, False), ("fwd", 128, False),
                                           ("bwd", 64, False), ("bwd", 128, False),
                                           ("fwd", 128, True), ("bwd", 128, True)])
def test_attention_kernel_timeout_path(ea, which, d, split):
    """A real attention kernel's bounded waits running out.

    attn_debug_stall arms a one-shot stall for the next launch: in every CTA
    one warp withholds its first "P ready" arrive, so the MMA warp's wait on
    it gives up after the armed 20 ms.  The CTA then drains its copies and
    MMAs, frees its tensor memory and returns; the call's workspace records
    ATTN_ERR_TIMEOUT with a wait site of that kernel, attn_check reports and
    clears it, and the next calls on the same context match the oracle.
    `split`: one head of 4096 keys, which the forward cuts into pieces along
    the keys and the backward along its key tiles' query tiles (the kernels
    with the pieces' code, followed by their merge kernels)."""
    import numpy as np
    from exact_attention_12_gb300 import _abi
    from oracle import attention as oracle
    from tests.helpers import GRAD_REL_L2, assert_o, max_abs, np64, rel_l2, L_MAX_ABS
    lib = _abi.lib()
    B, H, N = (1, 1, 4096) if split else (2, 3, 700)
    qc, kc, vc, doc = workloads.random_case(B, H, N, d, seed=40 + d)
    q, k, v, do = (t.cuda() for t in (qc, kc, vc, doc))
    kw = dict(scale=d ** -0.5, causal=True)
    ws = torch.zeros(1 << 26, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    o, lse = ea.attention_fwd(q, k, v, ws=ws, **kw)
    assert lib.attn_check(ws.data_ptr(), stream) == _abi.ATTN_OK
    stall = _abi.ATTN_STALL_FWD_SOFTMAX if which == "fwd" else _abi.ATTN_STALL_BWD_COMPUTE
    assert lib.attn_debug_stall(stall, 20_000_000) == _abi.ATTN_OK
    if which == "fwd":
        ea.attention_fwd(q, k, v, ws=ws, **kw)
        sites = range(1, 10)             # the forward's wait sites
    else:
        ea.attention_bwd(do, q, k, v, o, lse, ws=ws, **kw)
        sites = range(20, 29)            # the backward main kernel's wait sites
    assert lib.attn_check(ws.data_ptr(), stream) == _abi.ATTN_ERR_TIMEOUT
    assert _site(lib) in sites, lib.attn_last_error()
    assert lib.attn_check(ws.data_ptr(), stream) == _abi.ATTN_OK      # read and cleared
    # the stall was one-shot: the same calls on the same context are correct
    o, lse = ea.attention_fwd(q, k, v, ws=ws, **kw)
    dq, dk, dv = ea.attention_bwd(do, q, k, v, o, lse, ws=ws, **kw)
    assert lib.attn_check(ws.data_ptr(), stream) == _abi.ATTN_OK
    O, L, dQ, dK, dV = oracle.attention_backward(np64(qc), np64(kc), np64(vc), np64(doc), **kw)
    assert_o(np64(o.cpu()), O)
    assert max_abs(lse.cpu().numpy(), L) <= L_MAX_ABS
    for got, want in ((dq, dQ), (dk, dK), (dv, dV)):
        assert rel_l2(np64(got.cpu()), want) <= GRAD_REL_L2

