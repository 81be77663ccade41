"""Grouped-query / multi-query attention: K, V with H_kv heads shared by groups
of H / H_kv consecutive query heads ("3.3 Hiểu sâu cơ chế Self-Attention",
§9.2-9.3).  Forward and backward from the CUDA library against the fp64
oracle, element by element on small cases and sampled at full size."""

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oracle
from tests.helpers import (GRAD_REL_L2, L_MAX_ABS, assert_o, max_abs, np64, oracle_kwargs,
                           rel_l2, tile_samples)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


def _inputs(B, H, H_kv, N, d, seed, causal=False, key_lens=None, block_mask=None,
            dropout_p=0.0, dtype=torch.bfloat16):
    q, k, v, do = workloads.random_case(B, H, N, d, seed, dtype=dtype, H_kv=H_kv)
    return dict(q=q, k=k, v=v, do=do,
                key_lens=None if key_lens is None else torch.tensor(key_lens, dtype=torch.int32),
                block_mask=block_mask, scale=d ** -0.5, causal=causal, dropout_p=dropout_p,
                seed=99, offset=5)


def _api_kw(inp):
    return dict(scale=inp["scale"], causal=inp["causal"], dropout_p=inp["dropout_p"],
                seed=inp["seed"], offset=inp["offset"],
                key_lens=None if inp["key_lens"] is None else inp["key_lens"].cuda(),
                block_mask=None if inp["block_mask"] is None else inp["block_mask"].cuda())


def _check(ea, inp, backward=True):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    kw = _api_kw(inp)
    o, lse = ea.attention_fwd(q, k, v, **kw)
    assert o.shape == q.shape
    ok = oracle_kwargs(inp)
    if backward:
        dq, dk, dv = ea.attention_bwd(do, q, k, v, o, lse, **kw)
        assert dk.shape == k.shape and dv.shape == v.shape
        torch.cuda.synchronize()
        ea.check()
        O, L, dQ, dK, dV = oracle.attention_backward(np64(inp["q"]), np64(inp["k"]),
                                                     np64(inp["v"]), np64(inp["do"]), **ok)
        errs = [rel_l2(np64(g.cpu()), w) for g, w in ((dq, dQ), (dk, dK), (dv, dV))]
        assert max(errs) <= GRAD_REL_L2, errs
    else:
        torch.cuda.synchronize()
        ea.check()
        O, L = oracle.attention_forward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), **ok)
    out_bf16 = inp["q"].dtype == torch.bfloat16
    assert_o(np64(o.cpu()), O, out_bf16)
    assert max_abs(lse.cpu().numpy(), L) <= L_MAX_ABS
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(4, 2), (6, 1), (8, 4), (3, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads(ea, d, H, H_kv, causal):
    _check(ea, _inputs(2, H, H_kv, 300, d, seed=H * 10 + H_kv + d, causal=causal))


@pytest.mark.parametrize("d", [64, 128])
def test_grouped_heads_with_padding_and_dropout(ea, d):
    inp = _inputs(3, 4, 2, 390, d, seed=5, key_lens=[390, 200, 0], dropout_p=0.1)
    _check(ea, inp)


def test_grouped_heads_with_per_head_block_mask(ea):
    # the query heads of one group visit different key tiles
    B, H, H_kv, N = 2, 4, 2, 600
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(12)
    bm = (torch.rand((B, H, nb, nb), generator=g) < 0.45).to(torch.uint8)
    bm[0, 1] = 0                   # one query head of a group attends nothing
    _check(ea, _inputs(B, H, H_kv, N, 64, seed=13, block_mask=bm, causal=True))


@pytest.mark.parametrize("d", [64, 128])
def test_grouped_heads_with_split_pairs(ea, d):
    # few heads and long rows: the forward's pairs are cut along the keys and
    # the backward's key tiles along their (query head, query tile) walks
    _check(ea, _inputs(1, 4, 1, 2048, d, seed=21 + d, causal=True, dropout_p=0.1))


def test_multi_query_fp32_forward(ea):
    _check(ea, _inputs(1, 4, 1, 200, 64, seed=3, dtype=torch.float32), backward=False)


def test_grouped_heads_bnhd_key_value_layout(ea):
    # q in [B, H, N, d] storage, k and v in [B, N, H_kv, d] storage
    B, H, H_kv, N, d = 2, 4, 2, 257, 128
    inp = _inputs(B, H, H_kv, N, d, seed=17, causal=True, dropout_p=0.2)
    q, do = inp["q"].cuda(), inp["do"].cuda()
    k = inp["k"].transpose(1, 2).contiguous().cuda().transpose(1, 2)
    v = inp["v"].transpose(1, 2).contiguous().cuda().transpose(1, 2)
    kw = _api_kw(inp)
    o, lse = ea.attention_fwd(q, k, v, **kw)
    dq, dk, dv = ea.attention_bwd(do, q, k, v, o, lse, **kw)
    assert dk.stride() == k.stride()
    O, L, dQ, dK, dV = oracle.attention_backward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]),
                                                 np64(inp["do"]), **oracle_kwargs(inp))
    assert_o(np64(o.cpu()), O)
    for got, want in ((dq, dQ), (dk, dK), (dv, dV)):
        assert rel_l2(np64(got.cpu()), want) <= GRAD_REL_L2


def test_key_value_heads_must_divide_query_heads(ea):
    q = torch.zeros(1, 3, 64, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        ea.attention_fwd(q, k, k)


def test_full_size_gqa_workload_sampled(ea):
    """gqa-4k at full size: in three query heads, O, L and dQ of one row in
    every query tile, and dK, dV of one key in every key tile of their
    key/value heads, against the oracle; every output element written (the
    outputs start as NaN)."""
    w = workloads.get("gqa-4k")
    inp = workloads.make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    kw = _api_kw(inp)
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=q.device)
    ea.attention_fwd(q, k, v, out=o, lse=lse, **kw)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    ea.attention_bwd(do, q, k, v, o, lse, dq=dq, dk=dk, dv=dv, **kw)
    torch.cuda.synchronize()
    ea.check()
    o, lse, dq, dk, dv = (t.cpu() for t in (o, lse, dq, dk, dv))
    for t in (o, lse, dq, dk, dv):
        assert not torch.isnan(t).any()
    qn, kn, vn, don = (np64(inp[n]) for n in ("q", "k", "v", "do"))
    okw = oracle_kwargs(inp)
    grp = w.H // w.kv_heads
    for b, h in sorted({(0, 0), (w.B - 1, w.H - 1), (1, 13)}):
        rows = tile_samples(w.N, 3 + b * 17 + h)
        keys = tile_samples(w.N, 500 + b * 17 + h)
        O, L = oracle.forward_rows(qn, kn, vn, b, h, rows, **okw)
        assert_o(np64(o[b, h, rows]), O, what=(b, h))
        assert max_abs(lse[b, h, rows].numpy(), L) <= L_MAX_ABS
        dQ = oracle.backward_rows(qn, kn, vn, don, b, h, rows, **okw)
        assert rel_l2(np64(dq[b, h, rows]), dQ) <= GRAD_REL_L2
        hk = h // grp
        dK, dV = oracle.backward_keys(qn, kn, vn, don, b, hk, keys, **okw)
        assert rel_l2(np64(dk[b, hk, keys]), dK) <= GRAD_REL_L2
        assert rel_l2(np64(dv[b, hk, keys]), dV) <= GRAD_REL_L2
