"""Decode step: the newest n_q query positions of each sequence against its
key/value cache (attn_decode), from the CUDA library against the fp64 oracle's
decode_forward, on caches that span several split chunks, short and empty
caches, grouped heads and both cache layouts."""

import numpy as np
import pytest
import torch

from oracle import attention as oracle
from tests.helpers import L_MAX_ABS, O_MAX_ABS, max_abs, np64, o_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


def _case(B, H, H_kv, n_q, N, d, lens, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, n_q, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H_kv, N, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H_kv, N, d, generator=g).to(torch.bfloat16)
    return q, k, v, torch.tensor(lens, dtype=torch.int32)


def _check(ea, q, k, v, lens, causal, kv_dev=None):
    d = q.shape[-1]
    kd, vd = kv_dev if kv_dev is not None else (k.cuda(), v.cuda())
    o, lse = ea.attention_decode(q.cuda(), kd, vd, lens.cuda(), scale=d ** -0.5, causal=causal)
    torch.cuda.synchronize()
    ea.check()
    O, L = oracle.decode_forward(np64(q), np64(k), np64(v), scale=d ** -0.5,
                                 cache_lens=lens.numpy(), causal=causal)
    assert o_err(np64(o.cpu()), O) <= O_MAX_ABS
    assert max_abs(lse.cpu().numpy(), L) <= L_MAX_ABS
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("d", [64, 128])
# group rows (H / H_kv) * n_q: 1, 4, 32, 6, 16, 16, 24 -- both sides of the
# 16-row switch between the warp-MMA and the FMA kernels
@pytest.mark.parametrize("H,H_kv,n_q", [(8, 8, 1), (8, 2, 1), (8, 1, 4), (6, 3, 3), (16, 1, 1),
                                         (4, 1, 4), (24, 1, 1)])
@pytest.mark.parametrize("causal", [True, False])
def test_decode_small(ea, d, H, H_kv, n_q, causal):
    q, k, v, lens = _case(3, H, H_kv, n_q, 700, d, [700, 333, 2], seed=H * 7 + n_q + d)
    _check(ea, q, k, v, lens, causal)


def test_decode_empty_cache_rows(ea):
    # a sequence with no cached key gives O = 0 and L = -inf on every row
    q, k, v, lens = _case(2, 4, 2, 2, 300, 64, [0, 300], seed=3)
    o, lse = _check(ea, q, k, v, lens, True)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_decode_long_cache_many_splits(ea):
    rng = np.random.default_rng(11)
    lens = [int(x) for x in rng.integers(1, 8193, 4)]
    q, k, v, lens_t = _case(4, 16, 4, 1, 8192, 128, lens, seed=12)
    _check(ea, q, k, v, lens_t, True)


def test_decode_bnhd_cache_layout(ea):
    # caches stored [B, N, H_kv, d] and viewed as [B, H_kv, N, d]
    q, k, v, lens = _case(2, 8, 2, 1, 1000, 128, [1000, 517], seed=21)
    kd = k.transpose(1, 2).contiguous().cuda().transpose(1, 2)
    vd = v.transpose(1, 2).contiguous().cuda().transpose(1, 2)
    _check(ea, q, k, v, lens, True, kv_dev=(kd, vd))


def test_decode_rejects_unsupported_options(ea):
    import ctypes
    from exact_attention_12_gb300 import _abi
    q, k, v, lens = _case(1, 2, 1, 1, 128, 64, [128], seed=1)
    p = ea.make_params(q.cuda(), k=k.cuda(), key_lens=lens.cuda(), dropout_p=0.1)
    p.N = 128
    assert _abi.lib().attn_decode_workspace_size(ctypes.byref(p), 1) == 0
    q65 = torch.zeros(1, 65, 1, 64, dtype=torch.bfloat16, device="cuda")
    k1 = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_abi.AttnError):
        ea.attention_decode(q65, k1, k1, lens.cuda())   # 65 query rows per key/value head
