"""attn_bwd_noalloc: the backward whose scratch is built into the library.

Some callers cannot allocate device memory: a plug-in running inside an
application that owns every device allocation itself, a runtime handed a
fixed device-memory budget at start-up, or a latency-critical loop that must
not risk a cudaMalloc that synchronises the device.  For them
attn_bwd_noalloc keeps the backward's scratch in a fixed 64 MiB array inside
the library instead of a caller workspace.  These tests call it through the
C interface on two calls in a row (the array keeps the previous call's
contents, so the second call checks that nothing stale leaks through) and
require the oracle's gradients and the same gradients as attn_bwd with a
caller workspace; a time-out inside it must be visible through
attn_check(NULL, stream).

This file is collected last, so a run that stops at its first failure has
run every other test before it.
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oracle
from tests.helpers import GRAD_REL_L2, np64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


def _case(d, seed):
    B, H, N = 2, 3, 700
    q, k, v, do = workloads.random_case(B, H, N, d, seed)
    nb = (N + 127) // 128
    bm = workloads.make_block_mask(nb, 0.5, seed=seed)
    lens = torch.tensor([700, 431], dtype=torch.int32)
    kw = dict(scale=d ** -0.5, causal=True, dropout_p=0.1, seed=77, offset=2)
    return dict(cpu=(q, k, v, do), q=q.cuda(), k=k.cuda(), v=v.cuda(), do=do.cuda(),
                kw=dict(kw, key_lens=lens.cuda(), block_mask=bm.cuda()),
                okw=dict(kw, key_lens=lens.numpy(), block_mask=bm.numpy()))


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(ea, c, o, lse):
    from exact_attention_12_gb300 import _abi
    p = ea.make_params(c["q"], **c["kw"])
    dq, dk, dv = (torch.full_like(c["q"], float("nan")) for _ in range(3))
    st = _abi.lib().attn_bwd_noalloc(ctypes.byref(p), c["q"].data_ptr(), c["k"].data_ptr(),
                                     c["v"].data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     c["do"].data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                     dv.data_ptr(), _stream())
    _abi.check_status(st, "attn_bwd_noalloc")
    torch.cuda.synchronize()
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_backward_matches_the_oracle_and_the_workspace_backward(ea, d):
    from exact_attention_12_gb300 import _abi
    c = _case(d, seed=d)
    o, lse = ea.attention_fwd(c["q"], c["k"], c["v"], **c["kw"])
    ref = ea.attention_bwd(c["do"], c["q"], c["k"], c["v"], o, lse, **c["kw"])
    torch.cuda.synchronize()
    want = oracle.attention_backward(*(np64(t) for t in c["cpu"]), **c["okw"])[2:]
    for _ in range(2):
        got = _noalloc(ea, c, o, lse)
        assert _abi.lib().attn_check(None, _stream()) == _abi.ATTN_OK
        for g, r, w in zip(got, ref, want):
            assert not torch.isnan(g).any()
            assert rel_l2(np64(g), w) <= GRAD_REL_L2
            assert rel_l2(np64(g), np64(r)) <= GRAD_REL_L2


def test_noalloc_timeout_is_reported_by_attn_check_null(ea):
    from exact_attention_12_gb300 import _abi
    lib = _abi.lib()
    c = _case(128, seed=5)
    o, lse = ea.attention_fwd(c["q"], c["k"], c["v"], **c["kw"])
    # a one-shot stall in the backward main kernel: its waits give up after
    # 20 ms and record the time-out in the built-in scratch's status words
    assert lib.attn_debug_stall(_abi.ATTN_STALL_BWD_COMPUTE, 20_000_000) == _abi.ATTN_OK
    _noalloc(ea, c, o, lse)
    assert lib.attn_check(None, _stream()) == _abi.ATTN_ERR_TIMEOUT
    assert b"wait site" in lib.attn_last_error()
    assert lib.attn_check(None, _stream()) == _abi.ATTN_OK          # read and cleared
    # the next call is correct again
    got = _noalloc(ea, c, o, lse)
    assert lib.attn_check(None, _stream()) == _abi.ATTN_OK
    want = oracle.attention_backward(*(np64(t) for t in c["cpu"]), **c["okw"])[2:]
    for g, w in zip(got, want):
        assert rel_l2(np64(g), w) <= GRAD_REL_L2


def test_noalloc_rejects_problems_beyond_the_builtin_scratch(ea):
    from exact_attention_12_gb300 import _abi
    # needs ~ B*H*N*d*4 bytes of dQ accumulator: far beyond 64 MiB; nothing
    # is launched, so the tensors may be tiny placeholders
    t = torch.zeros(16, device="cuda")
    p = _abi.AttnParams()
    p.B, p.H, p.N, p.d = 8, 16, 8192, 128
    p.dtype, p.scale = _abi.ATTN_BF16, 0.1
    p.stride_b, p.stride_h, p.stride_n = 16 * 8192 * 128, 8192 * 128, 128
    ptr = t.data_ptr()
    st = _abi.lib().attn_bwd_noalloc(ctypes.byref(p), *([ptr] * 9), None)
    assert st == _abi.ATTN_ERR_WORKSPACE
    assert b"built-in scratch" in _abi.lib().attn_last_error()
    assert np.isfinite(t.sum().item())
