"""Concurrent calls on separate streams, each with its own workspace.

A serving or training process may run several attention problems at once on
different streams.  Each call keeps its scheduler counter, row statistics and
dQ accumulator in the workspace it is given, so calls that do not share a
workspace must not disturb one another.  The test runs two different
problems (one of them on the split-piece kernels) forward and backward on two
streams at the same time, several rounds over, and compares with the same
calls made one after another: O, L, dK and dV bit for bit (same kernels,
fixed summation order), dQ within fp32 rounding (its key-tile contributions
are added in the order the CTAs finish), and all of it against the oracle.
"""

import pytest
import torch

import workloads
from oracle import attention as oracle
from tests.helpers import GRAD_REL_L2, L_MAX_ABS, assert_o, max_abs, np64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


PROBLEMS = [
    # (B, H, H_kv, N, d, options): a many-head problem and a one-head problem
    # long enough that both passes take their split-piece kernels
    (2, 8, 4, 900, 64, dict(causal=True, dropout_p=0.1, seed=5, offset=1)),
    (1, 1, 1, 4096, 128, dict(causal=True)),
]


def _inputs(i):
    B, H, H_kv, N, d, kw = PROBLEMS[i]
    q, k, v, do = workloads.random_case(B, H, N, d, seed=70 + i, H_kv=H_kv)
    kw = dict(kw, scale=d ** -0.5)
    return (q, k, v, do), kw


def _step(ea, dev_in, kw, ws):
    q, k, v, do = dev_in
    o, lse = ea.attention_fwd(q, k, v, ws=ws, **kw)
    dq, dk, dv = ea.attention_bwd(do, q, k, v, o, lse, ws=ws, **kw)
    return o, lse, dq, dk, dv


def test_two_streams_two_workspaces(ea):
    cases = [_inputs(i) for i in range(len(PROBLEMS))]
    dev_in = [tuple(t.cuda() for t in c[0]) for c in cases]
    streams = [torch.cuda.Stream() for _ in cases]
    sizes = []
    for (inp, kw) in cases:
        p = ea.make_params(inp[0], k=inp[1], scale=kw["scale"], causal=kw.get("causal", False),
                           dropout_p=kw.get("dropout_p", 0.0))
        sizes.append(max(ea.workspace_size(p, True), ea.workspace_size(p, False)))
    ws = [torch.zeros(n, dtype=torch.uint8, device="cuda") for n in sizes]

    # one after another
    alone = []
    for i, (_, kw) in enumerate(cases):
        alone.append([t.clone() for t in _step(ea, dev_in[i], kw, ws[i])])
    torch.cuda.synchronize()
    ea.check()

    # at the same time, a few rounds
    for _ in range(3):
        together = [None] * len(cases)
        torch.cuda.synchronize()
        for i, (_, kw) in enumerate(cases):
            with torch.cuda.stream(streams[i]):
                together[i] = _step(ea, dev_in[i], kw, ws[i])
        torch.cuda.synchronize()
        for i in range(len(cases)):
            ea.check(ws[i])
            o, lse, dq, dk, dv = together[i]
            a = alone[i]
            assert torch.equal(o, a[0]) and torch.equal(lse, a[1])
            assert torch.equal(dk, a[3]) and torch.equal(dv, a[4])
            assert rel_l2(np64(dq.cpu()), np64(a[2].cpu())) <= 1e-5

    for i, ((q, k, v, do), kw) in enumerate(cases):
        O, L, dQ, dK, dV = oracle.attention_backward(np64(q), np64(k), np64(v), np64(do), **kw)
        o, lse, dq, dk, dv = (t.cpu() for t in alone[i])
        assert_o(np64(o), O, what=i)
        assert max_abs(lse.numpy(), L) <= L_MAX_ABS
        for got, want in ((dq, dQ), (dk, dK), (dv, dV)):
            assert rel_l2(np64(got), want) <= GRAD_REL_L2
