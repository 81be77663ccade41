"""Backward parity: dQ, dK, dV from the CUDA library against the fp64 oracle."""

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oracle
from tests.helpers import GRAD_REL_L2, api_kwargs, np64, oracle_kwargs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


def _run(ea, inp):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    kw = api_kwargs(inp)
    o, lse = ea.attention_fwd(q, k, v, **kw)
    dq, dk, dv = ea.attention_bwd(do, q, k, v, o, lse, **kw)
    torch.cuda.synchronize()
    ea.check()
    return o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()


def _inputs(B, H, N, d, seed, causal=False, key_lens=None, block_mask=None, dropout_p=0.0,
            std=1.0):
    q, k, v, do = workloads.random_case(B, H, N, d, seed, std=std)
    return dict(q=q, k=k, v=v, do=do,
                key_lens=None if key_lens is None else torch.tensor(key_lens, dtype=torch.int32),
                block_mask=block_mask, scale=d ** -0.5, causal=causal, dropout_p=dropout_p,
                seed=4321, offset=3)


def _check(ea, inp):
    _, _, dq, dk, dv = _run(ea, inp)
    _, _, dQ, dK, dV = oracle.attention_backward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]),
                                                 np64(inp["do"]), **oracle_kwargs(inp))
    errs = [rel_l2(np64(g), w) for g, w in ((dq, dQ), (dk, dK), (dv, dV))]
    assert max(errs) <= GRAD_REL_L2, errs
    return dq, dk, dv, (dQ, dK, dV)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_small_shapes(ea, d, N, causal):
    _check(ea, _inputs(2, 2, N, d, seed=N * 3 + d, causal=causal))


@pytest.mark.parametrize("d", [64, 128])
def test_padding_and_dropout(ea, d):
    dq, dk, dv, _ = _check(ea, _inputs(3, 2, 390, d, seed=21, key_lens=[390, 200, 129],
                                       dropout_p=0.1))
    # keys beyond the padding length get exactly zero gradients
    assert torch.all(dk[1, :, 200:] == 0) and torch.all(dv[1, :, 200:] == 0)
    assert torch.all(dk[2, :, 129:] == 0) and torch.all(dv[2, :, 129:] == 0)


def test_empty_rows_give_zero_gradients(ea):
    inp = _inputs(2, 1, 200, 64, seed=22, key_lens=[0, 150], causal=True)
    dq, dk, dv, _ = _check(ea, inp)
    assert torch.all(dq[0] == 0) and torch.all(dk[0] == 0) and torch.all(dv[0] == 0)


@pytest.mark.parametrize("per_head", [False, True])
def test_block_mask(ea, per_head):
    B, H, N = 2, 2, 600
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(8)
    shape = (B, H, nb, nb) if per_head else (nb, nb)
    bm = (torch.rand(shape, generator=g) < 0.4).to(torch.uint8)
    if per_head:
        bm[1, 0, :, 3] = 0          # a key tile no query tile visits
    else:
        bm[:, 3] = 0
    _check(ea, _inputs(B, H, N, 64, seed=23, block_mask=bm))


@pytest.mark.parametrize("d", [64, 128])
def test_everything_at_once(ea, d):
    bm = workloads.make_block_mask(5, 0.5, seed=9)
    _check(ea, _inputs(2, 2, 520, d, seed=24, block_mask=bm, causal=True, key_lens=[520, 333],
                       dropout_p=0.2))


def test_long_rows_many_query_tiles(ea):
    _check(ea, _inputs(1, 2, 1100, 128, seed=25, causal=True, std=0.5))


def test_repeatable(ea):
    # dQ uses fp32 atomics, so its low bits may vary; dK and dV must not
    inp = _inputs(1, 2, 300, 64, seed=26, causal=True)
    a = _run(ea, inp)
    b = _run(ea, inp)
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    assert rel_l2(np64(a[2]), np64(b[2])) < 1e-3


def _sample(N, seed, k=10):
    rng = np.random.default_rng(seed)
    fixed = {0, 127, 128, N // 2, N - 1}
    return np.array(sorted({x for x in fixed if 0 <= x < N} | set(rng.integers(0, N, k).tolist())))


@pytest.mark.parametrize("name", ["bert-large", "gpt2-1k", "gpt2-4k", "long-causal-4096",
                                  "long-causal-8192", "long-causal-16384", "block-sparse-64k"])
def test_full_size_workload_sampled(ea, name):
    w = workloads.get(name)
    inp = workloads.make_inputs(w)
    _, _, dq, dk, dv = _run(ea, inp)
    q, k, v, do = (np64(inp[n]) for n in ("q", "k", "v", "do"))
    kw = oracle_kwargs(inp)
    for b, h in {(0, 0), (w.B - 1, w.H - 1)}:
        rows = _sample(w.N, 7 + b * 31 + h)
        dQ = oracle.backward_rows(q, k, v, do, b, h, rows, **kw)
        dK, dV = oracle.backward_keys(q, k, v, do, b, h, rows, **kw)
        errs = (rel_l2(np64(dq[b, h, rows]), dQ), rel_l2(np64(dk[b, h, rows]), dK),
                rel_l2(np64(dv[b, h, rows]), dV))
        assert max(errs) <= GRAD_REL_L2, (name, b, h, errs)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()


def test_strided_bnhd_layout(ea):
    # [B, N, H, d] storage viewed as [B, H, N, d], backward included
    B, H, N, d = 2, 3, 300, 64
    g = torch.Generator().manual_seed(31)
    base = [torch.randn(B, N, H, d, generator=g).to(torch.bfloat16) for _ in range(4)]
    q, k, v, do = (t.transpose(1, 2) for t in base)
    kw = dict(scale=0.125, causal=True, key_lens=None, block_mask=None, dropout_p=0.1, seed=3,
              offset=1)
    qd, kd, vd, dod = (t.cuda().transpose(1, 2) for t in base)
    o, lse = ea.attention_fwd(qd, kd, vd, **kw)
    dq, dk, dv = ea.attention_bwd(dod, qd, kd, vd, o, lse, **kw)
    _, _, dQ, dK, dV = oracle.attention_backward(np64(q), np64(k), np64(v), np64(do),
                                                 **dict(kw, key_lens=None, block_mask=None))
    for got, want in ((dq, dQ), (dk, dK), (dv, dV)):
        assert rel_l2(np64(got.cpu()), want) <= GRAD_REL_L2


def _random_configs(n=14, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 4))
        N = int(rng.integers(1, 700))
        d = int(rng.choice([64, 128]))
        causal = bool(rng.integers(0, 2))
        pad = bool(rng.integers(0, 2))
        drop = float(rng.choice([0.0, 0.0, 0.15, 0.5]))
        blocks = bool(rng.integers(0, 3) == 0)
        out.append((B, H, N, d, causal, pad, drop, blocks, int(rng.integers(1 << 30))))
    return out


@pytest.mark.parametrize("cfg", _random_configs())
def test_random_configurations(ea, cfg):
    B, H, N, d, causal, pad, drop, blocks, seed = cfg
    rng = np.random.default_rng(seed)
    key_lens = [int(x) for x in rng.integers(0, N + 1, B)] if pad else None
    bm = None
    if blocks:
        nb = (N + 127) // 128
        bm = torch.from_numpy((rng.random((B, H, nb, nb)) < 0.6).astype(np.uint8))
    inp = _inputs(B, H, N, d, seed=seed % 1000, causal=causal, key_lens=key_lens, block_mask=bm,
                  dropout_p=drop)
    _check(ea, inp)
