"""The library's calls can be captured in CUDA graphs and replayed.

A training or serving loop replays its step from a CUDA graph to take the
host out of the launch path, so attn_fwd, attn_bwd and attn_decode must
neither synchronise nor allocate while enqueueing, and everything a launch
depends on (tensor maps, arguments) must be fixed at capture.  Each test
captures the Python binding's calls, refills the captured input buffers
with new values, replays, and compares with the same calls made eagerly on
those values: O, L, dK, dV and the decode output bit for bit (same kernels,
fixed summation order), dQ to fp32 rounding (its key-tile contributions are
added in the order the CTAs finish), and everything against the oracle.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oracle
from tests.helpers import GRAD_REL_L2, L_MAX_ABS, O_MAX_ABS, max_abs, np64, o_err, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


def _capture(fn):
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        out = fn()
    torch.cuda.synchronize()
    return g, out


@pytest.mark.parametrize("d,causal,dropout_p", [(64, False, 0.1), (128, True, 0.0)])
def test_fwd_bwd_replay(ea, d, causal, dropout_p):
    B, H, N = 2, 4, 300
    key_lens = torch.tensor([300, 170], dtype=torch.int32).cuda()
    kw = dict(scale=d ** -0.5, causal=causal, key_lens=key_lens, dropout_p=dropout_p, seed=77,
              offset=5)
    first = [t.cuda() for t in workloads.random_case(B, H, N, d, seed=40 + d)]
    second = workloads.random_case(B, H, N, d, seed=41 + d)
    q, k, v, do = first

    def step():
        o, lse = ea.attention_fwd(q, k, v, **kw)
        return (o, lse) + ea.attention_bwd(do, q, k, v, o, lse, **kw)

    step()                      # eager warm-up: workspace and kernel attributes
    torch.cuda.synchronize()
    g, out = _capture(step)
    for dst, src in zip(first, second):
        dst.copy_(src)
    g.replay()
    torch.cuda.synchronize()
    ea.check()
    got = [t.cpu() for t in out]
    want = [t.cpu() for t in step()]
    torch.cuda.synchronize()
    ea.check()
    for i in (0, 1, 3, 4):      # O, L, dK, dV
        assert torch.equal(got[i], want[i]), i
    assert rel_l2(np64(got[2]), np64(want[2])) <= 1e-5
    oq, ok_, ov, odo = (np64(t) for t in second)
    okw = dict(scale=d ** -0.5, causal=causal, key_lens=[300, 170], dropout_p=dropout_p,
               seed=77, offset=5)
    O, L = oracle.attention_forward(oq, ok_, ov, **okw)
    _, _, dQ, dK, dV = oracle.attention_backward(oq, ok_, ov, odo, **okw)
    assert o_err(np64(got[0]), O) <= O_MAX_ABS
    assert max_abs(got[1].numpy(), L) <= L_MAX_ABS
    assert max(rel_l2(np64(a), b) for a, b in zip(got[2:], (dQ, dK, dV))) <= GRAD_REL_L2


def test_decode_replay(ea):
    B, H, H_kv, n_q, N, d = 2, 8, 2, 1, 1000, 128
    lens = torch.tensor([1000, 517], dtype=torch.int32).cuda()
    q, k, v, _ = (t.cuda() for t in workloads.random_case(B, H, N, d, seed=50, H_kv=H_kv))
    q = q[:, :, :n_q].contiguous()
    q2 = workloads.random_case(B, H, n_q, d, seed=51)[0]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, n_q), dtype=torch.float32, device=q.device)

    def step():
        return ea.attention_decode(q, k, v, lens, out=o, lse=lse)

    step()
    torch.cuda.synchronize()
    g, _ = _capture(step)
    q.copy_(q2)
    g.replay()
    torch.cuda.synchronize()
    ea.check()
    got_o, got_l = o.cpu(), lse.cpu()
    step()
    torch.cuda.synchronize()
    ea.check()
    assert torch.equal(got_o, o.cpu()) and torch.equal(got_l, lse.cpu())
    O, L = oracle.decode_forward(np64(q2), np64(k), np64(v), scale=d ** -0.5,
                                 cache_lens=[1000, 517], causal=True)
    assert o_err(np64(got_o), O) <= O_MAX_ABS
    assert max_abs(got_l.numpy(), L) <= L_MAX_ABS
