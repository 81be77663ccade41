"""FP8 (E4M3) forward: E4M3 Q, K, V with per-tensor de-scale factors, bf16 O
(the FP8 step the FlashAttention explainer's timeline names for the Hopper
successor, "FlashAttention-3").  Results of the CUDA library against the fp64
oracle on the de-scaled inputs, element by element on small cases and
sampled at full size.

Tolerance (derived from the arithmetic; the kernel rounds the unnormalised
probabilities to E4M3 for P V and normalises by the unrounded row sum):
  |O - O_exact| <= v_descale-scaled (2^-4 A + 2^-10 T) + 2^-8 |O_exact| + 2e-3
with A, T from oracle.fp8.rounding_terms (the E4M3 rounding of P), 2^-8 |O|
the bf16 rounding of O, and 2e-3 for fp32 accumulation and ex2.
  |L - L_exact| <= 1e-3 (scores from exact products, fp32 sums).
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oracle
from oracle import fp8 as oracle_fp8
from tests.helpers import L_MAX_ABS, max_abs, tile_samples

pytestmark = pytest.mark.gpu

FP8 = getattr(torch, "float8_e4m3fn", None)
SLACK = 2e-3


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


def _codes(t):
    return t.view(torch.uint8).numpy()


def _real(t, descale):
    return oracle_fp8.dequantize(_codes(t), descale)


def _bound(A, T, O):
    return 2.0 ** -4 * A + 2.0 ** -10 * T + 2.0 ** -8 * np.abs(O) + SLACK


def _run(ea, q, k, v, ds, **kw):
    """The E4M3 forward into bf16 O and fp32 L pre-filled with NaN, so that an
    element the kernel never writes shows up as NaN."""
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    ea.attention_fwd(q.cuda(), k.cuda(), v.cuda(), q_descale=ds[0], k_descale=ds[1],
                     v_descale=ds[2], out=o, lse=lse, **kw)
    torch.cuda.synchronize()
    ea.check()
    assert o.dtype == torch.bfloat16 and o.shape == q.shape
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    return o.cpu().double().numpy(), lse.cpu().numpy()


def _check_full(ea, B, H, H_kv, N, seed, causal=False, key_lens=None, block_mask=None,
                std=1.0):
    (q, qs), (k, ks), (v, vs) = workloads.random_case_fp8(B, H, N, 128, seed, std=std, H_kv=H_kv)
    kw = dict(scale=128 ** -0.5, causal=causal)
    if key_lens is not None:
        kw["key_lens"] = torch.tensor(key_lens, dtype=torch.int32).cuda()
    if block_mask is not None:
        kw["block_mask"] = block_mask.cuda()
    o, lse = _run(ea, q, k, v, (qs, ks, vs), **kw)
    okw = dict(causal=causal, key_lens=key_lens,
               block_mask=None if block_mask is None else block_mask.numpy())
    O, L = oracle_fp8.fp8_forward(_codes(q), _codes(k), _codes(v), qs, ks, vs, 128 ** -0.5, **okw)
    A, T = oracle_fp8.rounding_terms(_real(q, qs), _real(k, ks), _real(v, vs), 128 ** -0.5, **okw)
    err = np.abs(o - O)
    assert np.all(err <= _bound(A, T, O)), float((err - _bound(A, T, O)).max())
    assert max_abs(lse, L) <= L_MAX_ABS
    # the bound is a worst case; the typical error is far below it
    live = np.isfinite(L)
    if live.any():
        assert np.sqrt(np.mean(err[live] ** 2)) <= 0.25 * np.sqrt(np.mean(_bound(A, T, O)[live] ** 2))
    return o, lse


@pytest.mark.skipif(FP8 is None, reason="torch without float8_e4m3fn")
@pytest.mark.parametrize("N", [1, 100, 128, 300, 513])
@pytest.mark.parametrize("causal", [False, True])
def test_small_shapes(ea, N, causal):
    _check_full(ea, 1, 2, 2, N, seed=N + causal, causal=causal)


@pytest.mark.skipif(FP8 is None, reason="torch without float8_e4m3fn")
def test_key_padding_with_empty_and_short_rows(ea):
    _check_full(ea, 3, 2, 2, 260, seed=3, key_lens=[260, 1, 0])


@pytest.mark.skipif(FP8 is None, reason="torch without float8_e4m3fn")
def test_block_mask_and_grouped_heads(ea):
    nb = 3
    bm = workloads.make_block_mask(nb, 0.5, seed=2)
    _check_full(ea, 2, 4, 2, 300, seed=4, causal=True, block_mask=bm)


@pytest.mark.skipif(FP8 is None, reason="torch without float8_e4m3fn")
def test_multi_query_heads_and_large_scores(ea):
    # std 4 makes the scores span tens of units: the lazy rescale fires
    _check_full(ea, 1, 4, 1, 384, seed=5, causal=True, std=4.0)


@pytest.mark.skipif(FP8 is None, reason="torch without float8_e4m3fn")
def test_split_pairs_of_a_long_single_head(ea):
    # one head of 4096 keys: 16 query-tile pairs, each cut into pieces along
    # the keys whose (O, L) are merged by the logsumexp rule
    _check_full(ea, 1, 1, 1, 4096, seed=8, causal=True)


@pytest.mark.skipif(FP8 is None, reason="torch without float8_e4m3fn")
def test_descale_factors_are_applied(ea):
    (q, _), (k, _), (v, _) = workloads.random_case_fp8(1, 2, 256, 128, 6)
    o1, l1 = _run(ea, q, k, v, (0.5, 0.25, 2.0), scale=0.125)
    o2, l2 = _run(ea, q, k, v, (1.0, 1.0, 1.0), scale=0.125 * 0.125)
    # same scores; O scales with v_descale exactly (a power of two)
    assert np.array_equal(l1, l2)
    assert np.array_equal(o1, 2.0 * o2)


@pytest.mark.skipif(FP8 is None, reason="torch without float8_e4m3fn")
def test_unsupported_fp8_options_are_rejected(ea):
    (q, _), (k, _), (v, _) = workloads.random_case_fp8(1, 1, 64, 128, 7)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    with pytest.raises(Exception):
        ea.attention_fwd(q, k, v, dropout_p=0.1)
    q64 = torch.zeros((1, 1, 64, 64), dtype=FP8, device="cuda")
    with pytest.raises(Exception):
        ea.attention_fwd(q64, q64, q64)


@pytest.mark.skipif(FP8 is None, reason="torch without float8_e4m3fn")
@pytest.mark.parametrize("name", ["fp8-long-causal-4096", "fp8-long-causal-16384"])
def test_full_size_workload_sampled(ea, name):
    w = workloads.get(name)
    inp = workloads.make_inputs(w)
    ds = (inp["q_descale"], inp["k_descale"], inp["v_descale"])
    o, lse = _run(ea, inp["q"], inp["k"], inp["v"], ds, scale=w.scale, causal=True)
    q, k, v = (_real(inp[n], d) for n, d in zip("qkv", ds))
    rng = np.random.default_rng(5)
    # three heads, one row in every query tile
    for b, h in sorted({(0, 0), (0, w.H - 1), (0, int(rng.integers(1, w.H - 1)))}):
        rows = tile_samples(w.N, h)
        O, L = oracle.forward_rows(q, k, v, b, h, rows, w.scale, causal=True)
        A, T = oracle_fp8.rounding_terms_rows(q, k, v, b, h, rows, w.scale, causal=True)
        err = np.abs(o[b, h, rows] - O)
        assert np.all(err <= _bound(A, T, O)), (name, b, h, float((err - _bound(A, T, O)).max()))
        assert max_abs(lse[b, h, rows], L) <= L_MAX_ABS
