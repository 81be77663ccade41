"""attn_bwd_noalloc: the backward whose scratch is built into the library.

Some callers cannot allocate device memory (a plug-in inside an application
that owns every device allocation, a runtime with a fixed memory budget, a
latency-critical loop that must not risk a synchronising cudaMalloc).  For
them attn_bwd_noalloc keeps the backward's scratch in a fixed 64 MiB array
inside the library instead of a caller workspace.  These tests call it
through the C interface and require the same gradients as attn_bwd with a
caller workspace, on two calls in a row (the array keeps the previous call's
contents, so the second call checks that nothing stale leaks through).
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads
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
    return dict(q=q.cuda(), k=k.cuda(), v=v.cuda(), do=do.cuda(),
                kw=dict(scale=d ** -0.5, causal=True,
                        key_lens=torch.tensor([700, 431], dtype=torch.int32).cuda(),
                        block_mask=bm.cuda(), dropout_p=0.1, seed=77, offset=2))


def _noalloc(ea, c, o, lse):
    from exact_attention_12_gb300 import _abi
    p = ea.make_params(c["q"], **c["kw"])
    dq, dk, dv = (torch.empty_like(c["q"]) for _ in range(3))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = _abi.lib().attn_bwd_noalloc(ctypes.byref(p), c["q"].data_ptr(), c["k"].data_ptr(),
                                     c["v"].data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     c["do"].data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                     dv.data_ptr(), stream)
    _abi.check_status(st, "attn_bwd_noalloc")
    torch.cuda.synchronize()
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_backward_matches_workspace_backward(ea, d):
    c = _case(d, seed=d)
    o, lse = ea.attention_fwd(c["q"], c["k"], c["v"], **c["kw"])
    ref = ea.attention_bwd(c["do"], c["q"], c["k"], c["v"], o, lse, **c["kw"])
    torch.cuda.synchronize()
    for _ in range(2):
        got = _noalloc(ea, c, o, lse)
        for g, r in zip(got, ref):
            assert rel_l2(np64(g), np64(r)) <= GRAD_REL_L2
            assert torch.isfinite(g.float()).all()


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
