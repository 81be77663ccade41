"""Backward parity: dQ, dK, dV from the CUDA library against the fp64 oracle."""

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oracle
from tests.helpers import GRAD_REL_L2, api_kwargs, np64, oracle_kwargs, rel_l2, tile_samples

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


def _run(ea, inp):
    """Forward and backward; the gradients go into buffers pre-filled with
    NaN, so that an element the kernels never write shows up as NaN."""
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    kw = api_kwargs(inp)
    o, lse = ea.attention_fwd(q, k, v, **kw)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    ea.attention_bwd(do, q, k, v, o, lse, dq=dq, dk=dk, dv=dv, **kw)
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
        bm[0, 1, 2, :] = 0          # a query tile no key tile visits: dQ = 0
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


@pytest.mark.parametrize("d", [64, 128])
def test_staged_calls_match_the_oracle(ea, d):
    """attn_bwd_preprocess, attn_bwd_main and attn_bwd_dq called one by one
    on one workspace (the bench times them so) give the oracle's gradients."""
    import ctypes
    from exact_attention_12_gb300 import _abi
    inp = _inputs(2, 3, 700, d, seed=27 + d, causal=True, key_lens=[700, 433], dropout_p=0.1)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    kw = api_kwargs(inp)
    o, lse = ea.attention_fwd(q, k, v, **kw)
    p = ea.make_params(q, k=k, **kw)
    ws = torch.zeros(ea.workspace_size(p, True), dtype=torch.uint8, device="cuda")
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    lib, s = _abi.lib(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P, W = ctypes.byref(p), (ws.data_ptr(), ws.numel())
    _abi.check_status(lib.attn_bwd_preprocess(P, o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                              *W, s), "preprocess")
    _abi.check_status(lib.attn_bwd_main(P, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        do.data_ptr(), dk.data_ptr(), dv.data_ptr(), *W, s),
                      "main")
    _abi.check_status(lib.attn_bwd_dq(P, dq.data_ptr(), *W, s), "dq")
    torch.cuda.synchronize()
    ea.check(ws)
    _, _, dQ, dK, dV = oracle.attention_backward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]),
                                                 np64(inp["do"]), **oracle_kwargs(inp))
    for got, want in ((dq, dQ), (dk, dK), (dv, dV)):
        assert rel_l2(np64(got.cpu()), want) <= GRAD_REL_L2


def test_repeatable(ea):
    # dQ uses fp32 atomics, so its low bits may vary; dK and dV must not
    inp = _inputs(1, 2, 300, 64, seed=26, causal=True)
    a = _run(ea, inp)
    b = _run(ea, inp)
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    assert rel_l2(np64(a[2]), np64(b[2])) < 1e-3


@pytest.mark.parametrize("name", ["bert-large", "gpt2-1k", "gpt2-4k", "long-causal-512",
                                  "long-causal-1024", "long-causal-2048", "long-causal-4096",
                                  "long-causal-8192", "long-causal-16384", "block-sparse-64k"])
def test_full_size_workload_sampled(ea, name):
    """The bench's workloads at full size: in three heads, dQ of one row in
    every query tile and dK, dV of one key in every key tile (each key tile
    is a unit of the persistent backward, claimed by different CTAs in
    different orders) against the oracle; every gradient element written
    (the outputs start as NaN)."""
    w = workloads.get(name)
    inp = workloads.make_inputs(w)
    _, _, dq, dk, dv = _run(ea, inp)
    for t in (dq, dk, dv):
        assert not torch.isnan(t).any(), name
    q, k, v, do = (np64(inp[n]) for n in ("q", "k", "v", "do"))
    kw = oracle_kwargs(inp)
    rng = np.random.default_rng(7)
    heads = {(0, 0), (w.B - 1, w.H - 1)}
    while len(heads) < min(3, w.B * w.H):
        heads.add((int(rng.integers(w.B)), int(rng.integers(w.H))))
    for b, h in sorted(heads):
        rows = tile_samples(w.N, 7 + b * 31 + h)
        keys = tile_samples(w.N, 1000 + b * 31 + h)
        dQ = oracle.backward_rows(q, k, v, do, b, h, rows, **kw)
        dK, dV = oracle.backward_keys(q, k, v, do, b, h, keys, **kw)
        errs = (rel_l2(np64(dq[b, h, rows]), dQ), rel_l2(np64(dk[b, h, keys]), dK),
                rel_l2(np64(dv[b, h, keys]), dV))
        assert max(errs) <= GRAD_REL_L2, (name, b, h, errs)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_keep_bits_are_exact(ea, d, causal):
    """The backward's own dropout keep mask, bit-exactly through the public API.

    The backward regenerates Z by its own route (one Philox call shared by
    eight lanes, then a bit transpose), so it is checked on its own.  With
    Q = K = 0 every allowed score is 0, so P_ij = 1 / n_allowed(i), and
    dV = P~^T dO with P~_ij = Z_ij P_ij / (1 - p').  Making dO the indicator
    of query row q0 + c in column c turns dV[j, c] into P~[q0 + c, j]:
    nonzero exactly where key j is allowed for, and kept at, query q0 + c.
    One call per block of d query rows reads the whole pattern, which must
    equal the oracle's allowed mask AND keep mask element for element, with
    key padding, a block mask and (parametrised) the causal mask.
    """
    B, H, N = 2, 2, 384
    key_lens = torch.tensor([384, 250], dtype=torch.int32)
    bm = torch.tensor([[1, 0, 1], [1, 1, 0], [0, 1, 1]], dtype=torch.uint8)
    p, seed, offset = 0.25, 0xDEADBEEF12345, 9
    kw = dict(scale=0.1, causal=causal, key_lens=key_lens.cuda(), block_mask=bm.cuda(),
              dropout_p=p, seed=seed, offset=offset)
    z = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    g = torch.Generator().manual_seed(d)
    v = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).cuda()
    o, lse = ea.attention_fwd(z, z, v, **kw)
    got = np.zeros((B, H, N, N), dtype=bool)      # [b, h, query, key]
    idx = torch.arange(d)
    for q0 in range(0, N, d):
        do = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
        do[:, :, q0 + idx, idx] = 1.0
        dq, dk, dv = ea.attention_bwd(do.cuda(), z, z, v, o, lse, **kw)
        torch.cuda.synchronize()
        ea.check()
        # dv[b, h, j, c] = P~[q0 + c, j]
        got[:, :, q0:q0 + d, :] = (dv.cpu().float().numpy() != 0).transpose(0, 1, 3, 2)
        # Q = K = 0: dQ = c dS K and dK = c dS^T Q vanish
        assert not dq.any() and not dk.any()
    want = np.zeros_like(got)
    for b in range(B):
        for h in range(H):
            allowed = oracle.allowed_mask(np.arange(N), np.arange(N), causal, int(key_lens[b]),
                                          bm.numpy())
            keep = oracle.keep_mask(np.arange(N), np.arange(N), b * H + h, seed, offset, p)
            want[b, h] = allowed & keep
    assert want.any() and not want.all()
    assert np.array_equal(got, want), int((got != want).sum())


@pytest.mark.parametrize("B,H,N,d,kw", [
    (1, 1, 4096, 128, dict(causal=True)),                     # 32 key tiles, 4 pieces each
    (1, 2, 2100, 64, dict(dropout_p=0.2)),                    # a ragged last tile
    (2, 1, 2500, 128, dict(causal=True, key_lens=[2500, 0])),
    (1, 2, 2400, 64, dict(block=True)),
])
def test_split_key_tiles_match_the_oracle(ea, B, H, N, d, kw):
    """Few heads, long rows: too few key tiles to fill the GPU, so the
    backward cuts each key tile's query tiles into pieces and adds up their
    dK, dV afterwards."""
    kw = dict(kw)
    bm = workloads.make_block_mask((N + 127) // 128, 0.4, seed=N) if kw.pop("block", False) \
        else None
    inp = _inputs(B, H, N, d, seed=N + d, block_mask=bm, **kw)
    p = ea.make_params(inp["q"].cuda(), causal=inp["causal"],
                       key_lens=None if inp["key_lens"] is None else inp["key_lens"].cuda(),
                       block_mask=None if bm is None else bm.cuda())
    nb = (N + 127) // 128
    assert ea.workspace_size(p, True) > 256 + B * H * nb * 128 * 8 + B * H * N * d * 4 + (1 << 16)
    _check(ea, inp)


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
