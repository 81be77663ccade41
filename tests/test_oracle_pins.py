"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

None of these tests needs a GPU.  Each checks the oracle against something
other than itself: a value printed on the pages (tests/golden/), a closed form,
an invariant, a library routine on a special case, a brute-force scalar loop
on tiny inputs, or finite differences.
"""

import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import attention as A
from oracle.blockwise import blockwise_forward
from oracle.philox import philox4x32_10, philox4x32_10_scalar

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def _fwd(q, k, v, **kw):
    """Forward on a single head given as [N, d] arrays."""
    O, L = A.attention_forward(q[None, None], k[None, None], v[None, None], **kw)
    return O[0, 0], L[0, 0]


def _bwd(q, k, v, do, **kw):
    O, L, dQ, dK, dV = A.attention_backward(q[None, None], k[None, None],
                                            v[None, None], do[None, None], **kw)
    return O[0, 0], L[0, 0], dQ[0, 0], dK[0, 0], dV[0, 0]


# ---------------------------------------------------------------- masks ----

def test_causal_mask_matches_printed_example():
    gold = np.array([[int(x) for x in r] for r in _golden_rows("causal_mask_4x4.txt")],
                    dtype=bool)
    got = A.allowed_mask(np.arange(4), np.arange(4), causal=True)
    assert np.array_equal(got, gold)


def test_block_mask_granularity_and_partial_blocks():
    N = 300                                   # 3 blocks, the last one partial
    bm = np.array([[1, 0, 1], [0, 1, 0], [1, 1, 0]], dtype=np.uint8)
    got = A.allowed_mask(np.arange(N), np.arange(N), block_mask=bm)
    for i in range(0, N, 7):
        for j in range(0, N, 5):
            assert got[i, j] == bool(bm[i // 128, j // 128])


def test_block_mask_equals_key_truncation():
    # A row whose only kept block is (0, 0) attends exactly keys 0..127:
    # identical to running the definition on the truncated key set.
    N, d = 260, 8
    q, k, v = _rand((N, d), 1), _rand((N, d), 2), _rand((N, d), 3)
    bm = np.zeros((3, 3), dtype=np.uint8)
    bm[0, 0] = 1
    bm[1, :] = 1
    bm[2, 2] = 1
    O, L = _fwd(q, k, v, scale=0.3, block_mask=bm)
    Ot, Lt = _fwd(q[:128], k[:128], v[:128], scale=0.3)
    np.testing.assert_allclose(O[:128], Ot, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L[:128], Lt, rtol=1e-12, atol=1e-12)
    # last block row attends only keys 256..259
    O2, L2 = _fwd(q[256:], k[256:], v[256:], scale=0.3)
    np.testing.assert_allclose(O[256:], O2, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- softmax / forward --

def test_probability_rows_sum_to_one():
    N, d = 37, 16
    q, k, v = _rand((N, d), 4), _rand((N, d), 5), _rand((N, d), 6)
    for kw in (dict(), dict(causal=True), dict(key_len=20)):
        hd = A._Head(q, k, v, 0.25, kw.get("causal", False), kw.get("key_len"),
                     None, 0.0, 0, 0, 0)
        _, P, _, _ = hd.chunk(np.arange(N))
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-13)


def test_constant_values_give_constant_output():
    N, d = 29, 8
    q, k = _rand((N, d), 7), _rand((N, d), 8)
    v = np.tile(np.linspace(-2, 3, d), (N, 1))
    for causal in (False, True):
        O, _ = _fwd(q, k, v, scale=0.5, causal=causal)
        np.testing.assert_allclose(O, v, rtol=0, atol=1e-13)


def test_single_key_output_is_value():
    d = 5
    q, k, v = _rand((1, d), 9), _rand((1, d), 10), _rand((1, d), 11)
    O, L = _fwd(q, k, v, scale=0.7)
    np.testing.assert_allclose(O, v, atol=1e-15)
    c = float(np.float32(0.7))
    assert L[0] == pytest.approx(c * float(q[0] @ k[0]), abs=1e-14)


def test_two_keys_closed_form():
    # softmax over two scores is a logistic function of their difference
    d = 3
    q, k, v = _rand((2, d), 12), _rand((2, d), 13), _rand((2, d), 14)
    c = float(np.float32(0.5))
    O, L = _fwd(q, k, v, scale=0.5)
    for i in range(2):
        s0 = c * sum(q[i, t] * k[0, t] for t in range(d))
        s1 = c * sum(q[i, t] * k[1, t] for t in range(d))
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        for t in range(d):
            assert O[i, t] == pytest.approx(w0 * v[0, t] + w1 * v[1, t], abs=1e-14)
        hi = max(s0, s1)
        assert L[i] == pytest.approx(hi + math.log1p(math.exp(-abs(s0 - s1))), abs=1e-14)


def test_causal_first_row_is_first_value():
    N, d = 9, 4
    q, k, v = _rand((N, d), 15), _rand((N, d), 16), _rand((N, d), 17)
    O, L = _fwd(q, k, v, scale=1.0, causal=True)
    np.testing.assert_allclose(O[0], v[0], atol=1e-15)
    assert L[0] == pytest.approx(float(q[0] @ k[0]), abs=1e-13)


def test_library_softmax_and_logsumexp():
    N, d = 23, 7
    q, k, v = _rand((N, d), 18), _rand((N, d), 19), _rand((N, d), 20)
    c = float(np.float32(0.3))
    S = c * (q @ k.T)
    O, L = _fwd(q, k, v, scale=0.3)
    np.testing.assert_allclose(L, scipy.special.logsumexp(S, axis=1), rtol=1e-13)
    np.testing.assert_allclose(O, scipy.special.softmax(S, axis=1) @ v, atol=1e-13)


def test_shift_invariance_of_scores():
    # adding u to every key adds c*q.u to each row's scores: O is unchanged,
    # L moves by exactly that amount
    N, d = 19, 6
    q, k, v = _rand((N, d), 21), _rand((N, d), 22), _rand((N, d), 23)
    u = _rand((d,), 24) * 3.0
    c = float(np.float32(0.4))
    O1, L1 = _fwd(q, k, v, scale=0.4)
    O2, L2 = _fwd(q, k + u, v, scale=0.4)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(L2 - L1, c * (q @ u), atol=1e-12)


def test_key_permutation_equivariance():
    N, d = 17, 5
    q, k, v = _rand((N, d), 25), _rand((N, d), 26), _rand((N, d), 27)
    perm = np.random.default_rng(28).permutation(N)
    O1, L1 = _fwd(q, k, v, scale=0.6)
    O2, L2 = _fwd(q, k[perm], v[perm], scale=0.6)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)


def _brute_force(q, k, v, c, causal, key_len, p, seed, offset, bh):
    """Scalar-loop restatement of the definition on a tiny head."""
    N, d = len(q), len(q[0])
    T = A.dropout_threshold(p)
    O = [[0.0] * len(v[0]) for _ in range(N)]
    L = [0.0] * N
    for i in range(N):
        s = []
        for j in range(N):
            ok = (not causal or j <= i) and (key_len is None or j < key_len)
            s.append(c * sum(q[i][t] * k[j][t] for t in range(d)) if ok else None)
        live = [x for x in s if x is not None]
        if not live:
            L[i] = -math.inf
            continue
        mx = max(live)
        tot = sum(math.exp(x - mx) for x in live)
        L[i] = mx + math.log(tot)
        for j in range(N):
            if s[j] is None:
                continue
            pij = math.exp(s[j] - L[i])
            if T:
                w = philox4x32_10_scalar((j // 8, i, bh, offset),
                                         (seed & 0xFFFFFFFF, seed >> 32))[(j % 8) // 2]
                u16 = (w >> (16 * (j % 2))) & 0xFFFF
                pij = 0.0 if u16 < T else pij / (1.0 - T / 65536.0)
            for t in range(len(v[0])):
                O[i][t] += pij * v[j][t]
    return np.array(O), np.array(L)


@pytest.mark.parametrize("causal,key_len,p", [(False, None, 0.0), (True, None, 0.0),
                                              (False, 4, 0.0), (True, 5, 0.35),
                                              (False, None, 0.5)])
def test_matches_brute_force_loops(causal, key_len, p):
    N, d = 7, 3
    q, k, v = _rand((N, d), 30), _rand((N, d), 31), _rand((N, d), 32)
    seed, offset = 0x1234_5678_9ABC_DEF0, 77
    O, L = _fwd(q, k, v, scale=0.8, causal=causal,
                key_lens=None if key_len is None else [key_len],
                dropout_p=p, seed=seed, offset=offset)
    Ob, Lb = _brute_force(q.tolist(), k.tolist(), v.tolist(),
                          float(np.float32(0.8)), causal, key_len, p, seed, offset, 0)
    np.testing.assert_allclose(O, Ob, atol=1e-13)
    np.testing.assert_allclose(L, Lb, atol=1e-13)


def test_blockwise_recurrence_matches_direct_statistics():
    # the pages' tiled online softmax reaches the direct row max and exp-sum
    # for every block size (the blockwise result equals the full softmax)
    for N in (1, 5, 17, 40):
        d = 4
        q, k, v = _rand((N, d), 40 + N), _rand((N, d), 41 + N), _rand((N, d), 42 + N)
        c = float(np.float32(0.45))
        O, L = _fwd(q, k, v, scale=0.45)
        S = c * (q @ k.T)
        for br in sorted({1, 2, 3, N // 2 or 1, N}):
            for bc in sorted({1, 4, N}):
                Ob, m, l = blockwise_forward(q, k, v, c, br, bc)
                np.testing.assert_allclose(m, S.max(axis=1), rtol=0, atol=1e-14)
                np.testing.assert_allclose(m + np.log(l), L, atol=1e-12)
                np.testing.assert_allclose(Ob, O, atol=1e-12)


@pytest.mark.parametrize("causal,p", [(False, 0.0), (True, 0.0), (True, 0.3)])
def test_key_pieces_merge_to_the_full_attention(causal, p):
    # the merge rule the split forward and decode step use (a reading of the
    # pages' running statistics): pieces of a row's keys, each with O_s
    # normalised over its keys and L_s its logsumexp, combine as
    # L = log sum_s e^{L_s} and O = sum_s e^{L_s - L} O_s, in any order.
    # Each piece here is one 128-key block column, selected by a block mask
    # in the oracle; the merge must give the unsplit attention.
    B, H, N, d = 1, 2, 300, 8
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    kw = dict(scale=0.4, causal=causal, dropout_p=p, seed=11, offset=3)
    O, L = A.attention_forward(q, k, v, **kw)
    nb = (N + 127) // 128
    parts = []
    for s in (2, 0, 1):                       # an arbitrary order
        bm = np.zeros((nb, nb), dtype=np.uint8)
        bm[:, s] = 1
        parts.append(A.attention_forward(q, k, v, block_mask=bm, **kw))
    Ls = np.stack([Lp for _, Lp in parts])                  # [pieces, B, H, N]
    Lm = np.logaddexp.reduce(Ls, axis=0)
    with np.errstate(invalid="ignore"):
        w = np.where(np.isneginf(Ls), 0.0, np.exp(Ls - Lm))
    Om = sum(w[i][..., None] * parts[i][0] for i in range(len(parts)))
    np.testing.assert_allclose(Lm, L, atol=1e-12)
    np.testing.assert_allclose(Om, O, atol=1e-12)


def test_fully_masked_row_is_zero():
    N, d = 6, 4
    q, k, v, do = (_rand((N, d), s) for s in (50, 51, 52, 53))
    O, L, dQ, dK, dV = _bwd(q, k, v, do, scale=0.5, key_lens=[0])
    assert np.all(O == 0) and np.all(np.isneginf(L))
    assert np.all(dQ == 0) and np.all(dK == 0) and np.all(dV == 0)


def test_shape_walkthrough():
    g = {r[0]: [float(x) for x in r[1:]] for r in _golden_rows("shape_walkthrough.txt")}
    B, H, N, d = (int(x) for x in g["q_heads"])
    rng = np.random.default_rng(54)
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    scale = 1.0 / g["scale_divisor"][0]
    assert math.sqrt(d) == g["scale_divisor"][0]
    O, L = A.attention_forward(q, k, v, scale)
    assert list(O.shape) == [int(x) for x in g["context_heads"]]
    assert list(L.shape) == [int(x) for x in g["scores"][:3]]
    hd = A._Head(q[0, 0], k[0, 0], v[0, 0], scale, False, None, None, 0.0, 0, 0, 0)
    _, P, _, _ = hd.chunk(np.arange(N))
    assert list(P.shape) == [int(x) for x in g["scores"][2:]]
    np.testing.assert_allclose(P.sum(axis=1), g["softmax_row_sum"][0], atol=1e-14)


def test_dot_product_standard_deviation_of_inputs():
    import torch
    import workloads
    for d_s, std_s in _golden_rows("dot_product_std.txt"):
        d, std = int(d_s), float(std_s)
        q, k, _, _ = workloads.random_case(1, 1, 20000, d, seed=d, dtype=torch.float32)
        dots = (q[0, 0].double() * k[0, 0].double()).sum(-1).numpy()
        assert abs(dots.std() - std) / std < 0.03


# ---------------------------------------------------------------- backward --

def _fd_check(kw, N=6, d=3, seed=60):
    q, k, v, do = (_rand((N, d), seed + i) for i in range(4))
    _, _, dQ, dK, dV = _bwd(q, k, v, do, **kw)

    def f(qq, kk, vv):
        O, _ = _fwd(qq, kk, vv, **kw)
        return float((O * do).sum())

    h = 1e-6
    for name, X, G in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = Xp
            fp = f(args["q"], args["k"], args["v"])
            args[name] = Xm
            fm = f(args["q"], args["k"], args["v"])
            num[idx] = (fp - fm) / (2 * h)
        err = np.linalg.norm(num - G) / max(np.linalg.norm(G), 1e-30)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("kw", [
    dict(scale=0.5),
    dict(scale=0.7, causal=True),
    dict(scale=0.3, key_lens=[4]),
    dict(scale=0.9, causal=True, key_lens=[5], dropout_p=0.3, seed=99, offset=3),
    dict(scale=0.4, dropout_p=0.5, seed=7),
])
def test_gradients_match_finite_differences(kw):
    _fd_check(kw)


def test_gradient_with_block_mask_finite_differences():
    # N spans two mask blocks so the block mask matters; only a few inputs
    # are perturbed to keep it quick
    N, d = 130, 2
    bm = np.array([[1, 0], [1, 1]], dtype=np.uint8)
    kw = dict(scale=0.5, block_mask=bm)
    q, k, v, do = (_rand((N, d), 70 + i) for i in range(4))
    _, _, dQ, dK, dV = _bwd(q, k, v, do, **kw)
    h = 1e-6
    rng = np.random.default_rng(75)
    for name, X, G in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        for _ in range(6):
            idx = (int(rng.integers(N)), int(rng.integers(d)))
            args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            args[name][idx] += h
            fp = float((_fwd(args["q"], args["k"], args["v"], **kw)[0] * do).sum())
            args[name][idx] -= 2 * h
            fm = float((_fwd(args["q"], args["k"], args["v"], **kw)[0] * do).sum())
            assert (fp - fm) / (2 * h) == pytest.approx(G[idx], rel=1e-5, abs=1e-8)


def test_D_identity_with_dropout():
    N, d = 33, 8
    q, k, v, do = (_rand((N, d), 80 + i) for i in range(4))
    hd = A._Head(q, k, v, 0.35, True, 30, None, 0.2, 5, 9, 3)
    rows = np.arange(N)
    cols, P, Zs, L = hd.chunk(rows)
    O = (P * Zs) @ v[cols]
    dP = (do @ v[cols].T) * Zs
    np.testing.assert_allclose((do * O).sum(1), (P * dP).sum(1), atol=1e-12)


def test_padded_keys_have_zero_gradients():
    N, d = 20, 4
    q, k, v, do = (_rand((N, d), 90 + i) for i in range(4))
    _, _, _, dK, dV = _bwd(q, k, v, do, scale=0.5, key_lens=[13], dropout_p=0.1, seed=1)
    assert np.all(dK[13:] == 0) and np.all(dV[13:] == 0)
    assert np.all(np.abs(dK[:13]).sum(1) > 0)


def test_sampled_helpers_match_full_evaluation():
    B, H, N, d = 2, 2, 300, 8
    rng = np.random.default_rng(100)
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    kw = dict(scale=0.35, causal=True, key_lens=[250, 300], dropout_p=0.1, seed=3,
              offset=2)
    O, L, dQ, dK, dV = A.attention_backward(q, k, v, do, **kw)
    rows = np.array([0, 5, 129, 299])
    Or, Lr = A.forward_rows(q, k, v, 1, 0, rows, **kw)
    np.testing.assert_allclose(Or, O[1, 0, rows], atol=1e-13)
    np.testing.assert_allclose(Lr, L[1, 0, rows], atol=1e-13)
    dQs = A.backward_rows(q, k, v, do, 1, 1, rows, **kw)
    np.testing.assert_allclose(dQs, dQ[1, 1, rows], atol=1e-12)
    keys = np.array([0, 127, 128, 249, 260])
    dKs, dVs = A.backward_keys(q, k, v, do, 0, 1, keys, **kw)
    np.testing.assert_allclose(dKs, dK[0, 1, keys], atol=1e-12)
    np.testing.assert_allclose(dVs, dV[0, 1, keys], atol=1e-12)


# ----------------------------------------------------------------- dropout --

def test_dropout_threshold_values():
    assert A.dropout_threshold(0.0) == 0
    assert A.dropout_threshold(0.5) == 2 ** 15
    assert A.dropout_threshold(0.25) == 2 ** 14
    assert A.dropout_threshold(0.1) == 6553                 # floor(0.1 * 65536)
    assert A.dropout_threshold(0.99999) == 65535
    assert A.dropout_threshold(1e-6) == 0 and A.keep_scale(1e-6) == 1.0
    assert A.keep_scale(0.5) == 2.0
    assert A.keep_scale(0.1) == 65536 / (65536 - 6553)


def test_keep_mask_uses_counter_word_layout():
    rows = np.array([0, 3, 511])
    cols = np.array([0, 1, 2, 3, 4, 7, 8, 9, 510])
    seed, offset, bh = (5 << 32) | 17, 11, 6
    Z = A.keep_mask(rows, cols, bh, seed, offset, 0.5)
    for a, i in enumerate(rows):
        for b, j in enumerate(cols):
            w = philox4x32_10_scalar((j // 8, i, bh, offset), (17, 5))[(j % 8) // 2]
            u16 = (w >> (16 * (j % 2))) & 0xFFFF
            assert Z[a, b] == (u16 >= 2 ** 15)


def test_keep_fraction_within_binomial_band():
    p = A.dropout_threshold(0.1) / 65536.0          # the exact drop rate
    Z = A.keep_mask(np.arange(512), np.arange(512), 3, 0, 0, 0.1)
    n = Z.size
    keep = Z.mean()
    sigma = math.sqrt(p * (1 - p) / n)
    assert abs(keep - (1 - p)) < 5 * sigma
    assert A.keep_mask(np.arange(4), np.arange(4), 0, 0, 0, 0.0).all()


def test_inverted_dropout_is_unbiased():
    N, d = 12, 3
    q, k, v = _rand((N, d), 110), _rand((N, d), 111), _rand((N, d), 112)
    p = 0.3
    O0, _ = _fwd(q, k, v, scale=0.5)
    n_seeds = 1500
    acc = np.zeros_like(O0)
    for s in range(n_seeds):
        acc += _fwd(q, k, v, scale=0.5, dropout_p=p, seed=s)[0]
    mean = acc / n_seeds
    hd = A._Head(q, k, v, 0.5, False, None, None, 0.0, 0, 0, 0)
    _, P, _, _ = hd.chunk(np.arange(N))
    pp = A.dropout_threshold(p) / 65536.0              # the exact drop rate
    var = (P ** 2) @ (v ** 2) * pp / (1 - pp)           # per-seed variance
    sigma = np.sqrt(var / n_seeds)
    assert np.all(np.abs(mean - O0) < 6 * sigma + 1e-12)


# ------------------------------------------------------------------ philox --

def test_philox_vector_matches_scalar():
    rng = np.random.default_rng(120)
    ctr = rng.integers(0, 2 ** 32, size=(64, 4), dtype=np.uint64)
    keys = rng.integers(0, 2 ** 32, size=(64, 2), dtype=np.uint64)
    for c, kk in zip(ctr, keys):
        vec = philox4x32_10(c[0], c[1], c[2], c[3], int(kk[0]), int(kk[1]))
        sca = philox4x32_10_scalar(c.tolist(), kk.tolist())
        assert tuple(int(x) for x in vec) == sca


def test_philox_output_bits_are_balanced():
    n = 1 << 14
    words = philox4x32_10(np.arange(n), 0, 0, 0, 0x1234, 0x5678)
    bits = np.unpackbits(np.stack(words).view(np.uint8))
    assert abs(bits.mean() - 0.5) < 5 * math.sqrt(0.25 / bits.size)
    # neighbouring counters differ in about half of their bits
    x = words[0][1:] ^ words[0][:-1]
    flips = np.unpackbits(x.view(np.uint8)).mean()
    assert abs(flips - 0.5) < 0.01


def _curand_host_philox(seed, nwords):
    """`nwords` 32-bit outputs of cuRAND's host-side Philox4x32-10 generator
    (CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161 in curand.h), which runs on the
    CPU without a device.  None if the library cannot be loaded."""
    import ctypes
    import ctypes.util
    names = [ctypes.util.find_library("curand"), "/usr/local/cuda/lib64/libcurand.so",
             "/usr/local/cuda/lib64/libcurand.so.10", "libcurand.so.10"]
    lib = None
    for n in names:
        if not n:
            continue
        try:
            lib = ctypes.CDLL(n)
            break
        except OSError:
            continue
    if lib is None:
        return None
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:
        return None
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        buf = (ctypes.c_uint * nwords)()
        assert lib.curandGenerate(gen, buf, ctypes.c_size_t(nwords)) == 0
        return np.array(list(buf), dtype=np.uint64)
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0, 1, 0x123456789ABCDEF0, 2 ** 64 - 1])
def test_philox_matches_an_independent_implementation(seed):
    # cuRAND's host generator implements the same published Philox4x32-10.
    # Its first 64 output blocks of four words come from counters
    # (0, 0, i, 0), i = 0..63 (the subsequence index in counter word 2), with
    # the seed's low and high 32 bits as the key.  A wrong multiplier, Weyl
    # constant, word order or round count changes every block.
    words = _curand_host_philox(seed, 4 * 64)
    if words is None:
        pytest.skip("cuRAND's host generator is not available")
    k0, k1 = seed & 0xFFFFFFFF, seed >> 32
    i = np.arange(64, dtype=np.uint64)
    got = philox4x32_10(np.zeros(64, dtype=np.uint64), 0, i, 0, k0, k1)
    assert np.array_equal(np.stack(got, axis=1).reshape(-1), words)
    assert philox4x32_10_scalar((0, 0, 5, 0), (k0, k1)) == tuple(int(x) for x in words[20:24])


# ------------------------------------------------------ grouped-query heads --
# "3.3 Hiểu sâu cơ chế Self-Attention", §9.2-9.3: groups of query heads share
# one key/value head; one group per head is MHA, a single group is MQA.

def _rand4(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_mqa_equals_every_head_attending_the_same_keys():
    # one key/value head: each query head is an ordinary single-head problem
    # against that head, computed here head by head through the MHA path
    B, H, N, d = 2, 3, 9, 4
    q = _rand4((B, H, N, d), 1)
    k, v, do = _rand4((B, 1, N, d), 2), _rand4((B, 1, N, d), 3), _rand4((B, H, N, d), 4)
    kw = dict(scale=0.6, causal=True, key_lens=[9, 5], dropout_p=0.2, seed=5, offset=1)
    O, L, dQ, dK, dV = A.attention_backward(q, k, v, do, **kw)
    dK_sum, dV_sum = np.zeros_like(k), np.zeros_like(v)
    for h in range(H):
        # the dropout counter uses the query head's b*H+h: run the single head
        # inside an H-head problem whose other heads are ignored
        qh = np.zeros_like(q)
        qh[:, h] = q[:, h]
        doh = np.zeros_like(do)
        doh[:, h] = do[:, h]
        kh, vh = np.repeat(k, H, axis=1), np.repeat(v, H, axis=1)
        o, l, dq, dk, dv = A.attention_backward(qh, kh, vh, doh, **kw)
        np.testing.assert_allclose(O[:, h], o[:, h], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(L[:, h], l[:, h], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dQ[:, h], dq[:, h], rtol=1e-12, atol=1e-12)
        dK_sum[:, 0] += dk[:, h]
        dV_sum[:, 0] += dv[:, h]
    np.testing.assert_allclose(dK, dK_sum, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dV, dV_sum, rtol=1e-11, atol=1e-12)


def test_gqa_reads_key_value_head_of_its_consecutive_group():
    # H = 6 query heads over H_kv = 2 key/value heads: heads 0-2 read kv head
    # 0, heads 3-5 kv head 1, i.e. the MHA result on K, V with each key/value
    # head repeated for its three query heads
    B, H, Hk, N, d = 1, 6, 2, 11, 3
    q, do = _rand4((B, H, N, d), 11), _rand4((B, H, N, d), 12)
    k, v = _rand4((B, Hk, N, d), 13), _rand4((B, Hk, N, d), 14)
    kw = dict(scale=0.5, causal=False, key_lens=[8])
    O, L, dQ, dK, dV = A.attention_backward(q, k, v, do, **kw)
    ke, ve = np.repeat(k, H // Hk, axis=1), np.repeat(v, H // Hk, axis=1)
    Oe, Le, dQe, dKe, dVe = A.attention_backward(q, ke, ve, do, **kw)
    np.testing.assert_allclose(O, Oe, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L, Le, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dQ, dQe, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dK, dKe.reshape(B, Hk, H // Hk, N, d).sum(axis=2),
                               rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dV, dVe.reshape(B, Hk, H // Hk, N, d).sum(axis=2),
                               rtol=1e-11, atol=1e-12)


def test_gqa_gradients_match_finite_differences():
    # the shared key/value heads' gradients, including the group sum, against
    # central differences of sum(O * dO)
    B, H, Hk, N, d = 1, 4, 2, 5, 2
    q, do = _rand4((B, H, N, d), 21), _rand4((B, H, N, d), 22)
    k, v = _rand4((B, Hk, N, d), 23), _rand4((B, Hk, N, d), 24)
    kw = dict(scale=0.8, causal=True, dropout_p=0.25, seed=3, offset=2)
    _, _, dQ, dK, dV = A.attention_backward(q, k, v, do, **kw)

    def f(qq, kk, vv):
        return float((A.attention_forward(qq, kk, vv, **kw)[0] * do).sum())

    eps = 1e-6
    for name, X, G in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            args[name][idx] += eps
            fp = f(args["q"], args["k"], args["v"])
            args[name][idx] -= 2 * eps
            fm = f(args["q"], args["k"], args["v"])
            num[idx] = (fp - fm) / (2 * eps)
        err = np.linalg.norm(num - G) / max(np.linalg.norm(G), 1e-30)
        assert err < 1e-6, (name, err)


def test_gqa_backward_keys_sums_the_group():
    B, H, Hk, N, d = 2, 4, 2, 7, 3
    q, do = _rand4((B, H, N, d), 31), _rand4((B, H, N, d), 32)
    k, v = _rand4((B, Hk, N, d), 33), _rand4((B, Hk, N, d), 34)
    kw = dict(scale=0.4, causal=True, key_lens=[7, 6], dropout_p=0.1, seed=1)
    _, _, _, dK, dV = A.attention_backward(q, k, v, do, **kw)
    keys = np.array([0, 3, 6])
    for b in range(B):
        for hk in range(Hk):
            dk, dv = A.backward_keys(q, k, v, do, b, hk, keys, **kw)
            np.testing.assert_allclose(dk, dK[b, hk, keys], rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(dv, dV[b, hk, keys], rtol=1e-11, atol=1e-12)


def test_key_value_heads_must_divide_query_heads():
    q = np.zeros((1, 3, 4, 2))
    k = np.zeros((1, 2, 4, 2))
    with pytest.raises(ValueError):
        A.attention_forward(q, k, k, scale=1.0)


# ------------------------------------------------------------ decode step --
# The newest N_q positions of each sequence against its key/value cache: the
# same attention as the last N_q rows of the square problem over the cached
# prefix, computed here through the square (already pinned) path.

@pytest.mark.parametrize("causal", [True, False])
def test_decode_equals_last_rows_of_the_square_problem(causal):
    B, H, Hk, Nq, Nkv, d = 3, 4, 2, 3, 40, 5
    q = _rand4((B, H, Nq, d), 41)
    k, v = _rand4((B, Hk, Nkv, d), 42), _rand4((B, Hk, Nkv, d), 43)
    lens = [40, 17, 2]            # the last sequence is shorter than N_q
    O, L = A.decode_forward(q, k, v, scale=0.45, cache_lens=lens, causal=causal)
    for b, n in enumerate(lens):
        # causal: query rows before the start of the sequence see no key; the
        # others are the last rows of the square causal problem over the n
        # cached positions.  Non-causal: positions do not matter, so every
        # row is a row of a square problem of N' = max(n, N_q) positions whose
        # keys beyond the cache are padding (key_lens = n).
        rows = min(n, Nq) if causal else Nq
        Np = n if causal else max(n, Nq)
        if rows:
            qs = np.zeros((1, H, Np, d))
            qs[0, :, Np - rows:] = q[b, :, Nq - rows:]
            ks, vs = np.zeros((1, Hk, Np, d)), np.zeros((1, Hk, Np, d))
            ks[0, :, :n], vs[0, :, :n] = k[b, :, :n], v[b, :, :n]
            Os, Ls = A.attention_forward(qs, ks, vs, scale=0.45, causal=causal, key_lens=[n])
            np.testing.assert_allclose(O[b, :, Nq - rows:], Os[0, :, Np - rows:], rtol=1e-12,
                                       atol=1e-12)
            np.testing.assert_allclose(L[b, :, Nq - rows:], Ls[0, :, Np - rows:], rtol=1e-12,
                                       atol=1e-12)
        if rows < Nq:
            assert np.all(O[b, :, :Nq - rows] == 0) and np.all(np.isneginf(L[b, :, :Nq - rows]))


def test_decode_single_query_is_softmax_over_the_cache():
    # one query per sequence: O = sum_j softmax_j(c q.k_j) v_j over the cached keys
    B, H, Nkv, d = 2, 2, 9, 3
    q = _rand4((B, H, 1, d), 51)
    k, v = _rand4((B, H, Nkv, d), 52), _rand4((B, H, Nkv, d), 53)
    lens = [9, 4]
    O, L = A.decode_forward(q, k, v, scale=0.7, cache_lens=lens)
    for b, n in enumerate(lens):
        for h in range(H):
            c = float(np.float32(0.7))   # the scale travels as a float32
            s = c * np.array([float(np.dot(q[b, h, 0], k[b, h, j])) for j in range(n)])
            w = scipy.special.softmax(s)
            np.testing.assert_allclose(O[b, h, 0], (w[:, None] * v[b, h, :n]).sum(axis=0),
                                       rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(L[b, h, 0], scipy.special.logsumexp(s), rtol=1e-12)


# ------------------------------------------------------------------ FP8 ----

from oracle import fp8 as F  # noqa: E402


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0),
    (0x30, 0.5), (0x08, 2.0 ** -6), (0x07, 0.875 * 2.0 ** -6), (0x01, 2.0 ** -9),
    (0x77, 240.0), (0x78, 256.0), (0x7E, 448.0), (0xB8, -1.0), (0xFE, -448.0),
    (0x81, -(2.0 ** -9)),
])
def test_e4m3_values_from_the_format_definition(code, value):
    # sign | 4-bit exponent (bias 7) | 3-bit mantissa, subnormals at exponent 0
    assert F.e4m3_value([code])[0] == value


def test_e4m3_nan_zero_and_ordering():
    vals = F.e4m3_value(np.arange(256))
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert np.isnan(vals).sum() == 2
    assert vals[0x80] == 0.0 and math.copysign(1.0, vals[0x80]) == -1.0
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0)                    # codes 0..126 increase strictly
    assert np.array_equal(vals[0x80:0xFF], -pos)       # the sign bit only negates
    assert pos.max() == F.E4M3_MAX
    # spacing: 2^-9 through the subnormals and the first normal binade, then doubling
    assert np.all(np.diff(pos[:17]) == 2.0 ** -9)
    assert np.diff(pos[0x38:0x40]).tolist() == [0.125] * 7


def test_e4m3_matches_torch_float8():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_value(np.arange(256))
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_fp8_forward_descales_each_operand():
    rng = np.random.default_rng(3)
    q8 = rng.integers(0, 0x70, (1, 2, 9, 4)).astype(np.uint8)
    k8 = rng.integers(0, 0x70, (1, 2, 9, 4)).astype(np.uint8)
    v8 = rng.integers(0x80, 0xF0, (1, 2, 9, 4)).astype(np.uint8)
    # constant V (all one code): O is that value times v_descale in every row
    vc = np.full_like(v8, 0x44)                                        # 3.0
    O, _ = F.fp8_forward(q8, k8, vc, 0.5, 0.25, 0.125, 0.5, causal=True)
    assert np.allclose(O, 0.375, rtol=0, atol=1e-14)
    # the scores see q_descale * k_descale * scale as one factor: doubling
    # q_descale and halving scale leaves O and L unchanged
    O1, L1 = F.fp8_forward(q8, k8, v8, 0.5, 0.25, 2.0, 0.5)
    O2, L2 = F.fp8_forward(q8, k8, v8, 1.0, 0.25, 2.0, 0.25)
    assert np.allclose(O1, O2, atol=1e-12) and np.allclose(L1, L2, atol=1e-12)
    # N = 1: O = V
    O, L = F.fp8_forward(q8[:, :, :1], k8[:, :, :1], v8[:, :, :1], 1.0, 1.0, 2.0, 0.5)
    assert np.array_equal(O, 2.0 * F.e4m3_value(v8[:, :, :1]))


def test_rounding_terms_special_cases():
    rng = np.random.default_rng(4)
    q, k, v = _rand((1, 1, 6, 3), 5), _rand((1, 1, 6, 3), 6), _rand((1, 1, 6, 3), 7)
    A_, T_ = F.rounding_terms(q, k, v, 0.75, causal=True)
    # row 0 attends key 0 only: A = T = |V_0|
    assert np.allclose(A_[0, 0, 0], np.abs(v[0, 0, 0])) and np.allclose(T_[0, 0, 0], np.abs(v[0, 0, 0]))
    # |O| <= A (triangle inequality); A and T against scalar loops
    O, _ = A.attention_forward(q, k, v, 0.75, causal=True)
    assert np.all(np.abs(O) <= A_ + 1e-12)
    for i in range(6):
        s = 0.75 * np.array([q[0, 0, i] @ k[0, 0, j] for j in range(i + 1)])
        w = np.exp(s - s.max())
        for c in range(3):
            a = sum(w[j] * abs(v[0, 0, j, c]) for j in range(i + 1)) / w.sum()
            t = sum(abs(v[0, 0, j, c]) for j in range(i + 1)) / w.sum()
            assert abs(A_[0, 0, i, c] - a) < 1e-12 and abs(T_[0, 0, i, c] - t) < 1e-12
    # a row with no key: both zero
    A0, T0 = F.rounding_terms(q, k, v, 0.75, key_lens=[0])
    assert not A0.any() and not T0.any()


def test_rounding_bound_holds_for_simulated_e4m3_probabilities():
    # round the unnormalised weights to the nearest E4M3 value (a brute-force
    # nearest search over the 127 non-negative codes), with a lazily kept max
    # (gamma up to 2^8), and check the error against 2^-4 A + 2^-10 T
    grid = F.e4m3_value(np.arange(0x7F))
    rng = np.random.default_rng(8)
    q, k, v = _rand((1, 1, 40, 8), 9, 1.5), _rand((1, 1, 40, 8), 10, 1.5), _rand((1, 1, 40, 8), 11)
    O, _ = A.attention_forward(q, k, v, 0.5, causal=True)
    A_, T_ = F.rounding_terms(q, k, v, 0.5, causal=True)
    for i in range(40):
        s = 0.5 * (q[0, 0, i] @ k[0, 0, : i + 1].T)
        gamma = 2.0 ** rng.uniform(0, 8)
        w = gamma * np.exp(s - s.max())
        wr = grid[np.abs(grid[None, :] - w[:, None]).argmin(axis=1)]
        o = (wr @ v[0, 0, : i + 1]) / w.sum()
        assert np.all(np.abs(o - O[0, 0, i]) <= 2.0 ** -4 * A_[0, 0, i] + 2.0 ** -10 * T_[0, 0, i] + 1e-12)


def test_rounding_terms_rows_match_the_full_evaluation():
    q, k, v = _rand((2, 4, 20, 3), 12), _rand((2, 2, 20, 3), 13), _rand((2, 2, 20, 3), 14)
    A_, T_ = F.rounding_terms(q, k, v, 0.5, causal=True, key_lens=[20, 7])
    rows = np.array([0, 6, 7, 19])
    for b, h in [(0, 3), (1, 1)]:
        a, t = F.rounding_terms_rows(q, k, v, b, h, rows, 0.5, causal=True, key_lens=[20, 7])
        assert np.allclose(a, A_[b, h, rows], atol=1e-13) and np.allclose(t, T_[b, h, rows], atol=1e-13)
