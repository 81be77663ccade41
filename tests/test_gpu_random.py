"""Seeded random configurations, forward and backward through the public API
against the fp64 oracle: shapes, head groups, layouts and every mask drawn
together, so that combinations no hand-written case names are covered too
(and likewise for the fp32 forward, the decode step and the E4M3 forward).
Outputs start as NaN (an element the kernels never write fails the check).

The draws are fixed by the seed: a failing case keeps its id from run to run.
Value std runs to 2 and dropout to 0.5, beyond the workloads' regime (std up
to 1, dropout 0.1) for which the O bar of 1e-2 is stated; there the bar widens
in proportion to |V| and 1 / (1 - p) (tests.helpers.o_magnitude_factor), the
only two things the kernel's O error scales with.  L and dV keep their bars;
dQ and dK add what forming D from the forward's bf16 O contributes (see
d_rounding_terms), which only matters where they cancel to nearly nothing.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oracle
from tests.helpers import (GRAD_REL_L2, L_MAX_ABS, assert_o, max_abs, np64,
                           o_magnitude_factor)

pytestmark = pytest.mark.gpu

N_SHORT = 120         # cases with N <= 700 (every path but the split ones)
N_LONG = 8            # few heads, N >= 2048: the forward's and backward's split paths
N_FP32 = 24           # fp32 forward (the TF32 tensor-core path)
EDGE_N = (1, 2, 63, 64, 127, 128, 129, 255, 256, 257, 383, 640, 700)


def _draw(i):
    """Case i: a dict of sizes and options, drawn from a generator seeded by i."""
    r = np.random.default_rng(1000 + i)
    long = N_SHORT <= i < N_SHORT + N_LONG
    d = int(r.choice([64, 128]))
    if long:
        B, H_kv, group = 1, 1, int(r.choice([1, 2]))
        N = int(r.integers(2048, 2600))
    else:
        B = int(r.integers(1, 4))
        H_kv = int(r.integers(1, 4))
        group = int(r.choice([1, 1, 2, 4]))
        N = int(r.choice(EDGE_N)) if r.random() < 0.4 else int(r.integers(1, 701))
    H = H_kv * group
    c = dict(B=B, H=H, H_kv=H_kv, N=N, d=d, causal=bool(r.random() < 0.5),
             std=float(r.choice([0.5, 1.0, 2.0])),
             scale=float(d ** -0.5 * r.uniform(0.5, 1.5)),
             dropout_p=float(r.choice([0.1, 0.25, 0.5])) if r.random() < 0.4 else 0.0,
             seed=int(r.integers(0, 2 ** 31)), offset=int(r.integers(0, 1000)),
             bnhd=bool(r.random() < 0.25), key_lens=None, block_mask=None,
             fp32=i >= N_SHORT + N_LONG)
    if c["fp32"]:
        c["bnhd"] = False   # the fp32 cases run in [B, H, N, d] storage
    if r.random() < 0.4:
        lens = r.integers(0, N + 1, size=B)
        if B > 1 and r.random() < 0.5:
            lens[int(r.integers(0, B))] = int(r.choice([0, N]))
        c["key_lens"] = [int(x) for x in lens]
    if not long and r.random() < 0.3:
        nb = (N + 127) // 128
        per_head = bool(r.random() < 0.5)
        shape = (B, H, nb, nb) if per_head else (nb, nb)
        c["block_mask"] = (r.random(shape) < r.uniform(0.2, 0.8)).astype(np.uint8)
    return c


def _case_id(i):
    c = _draw(i)
    parts = [f"B{c['B']}H{c['H']}/{c['H_kv']}N{c['N']}d{c['d']}"]
    parts += [n for n, on in (("causal", c["causal"]), ("pad", c["key_lens"] is not None),
                              ("drop", c["dropout_p"] > 0), ("block", c["block_mask"] is not None),
                              ("bnhd", c["bnhd"])) if on]
    return f"{i}-" + ("fp32-" if c["fp32"] else "") + "-".join(parts)


@pytest.fixture(scope="module")
def ea():
    import exact_attention_12_gb300 as ea
    from exact_attention_12_gb300 import build
    build.build()
    return ea


def _to_dev(t, bnhd):
    """t [B, H, N, d] on the GPU, stored [B, N, H, d] when bnhd (same logical view)."""
    if not bnhd:
        return t.cuda()
    return t.transpose(1, 2).contiguous().cuda().transpose(1, 2)


def d_rounding_terms(q, k, do, O, o_gpu, c, kl):
    """Norms of what the forward's O error carries into dQ and dK: the
    backward forms D = rowsum(dO * O) from the O it is given (the forward's
    bf16 output), so with e_i = rowsum(dO * (O_gpu - O)) the error of D_i,
    dS_ij changes by -P_ij e_i (P the softmax probabilities before dropout),
    dQ_i by -c e_i sum_j P_ij K_j and dK_j by -c sum_i P_ij e_i Q_i (summed
    over a key/value head's query heads)."""
    qn, kn, don = np64(q), np64(k), np64(do)
    e = (don * (o_gpu - O)).sum(-1)                            # [B, H, N]
    B, H, N, _ = qn.shape
    grp = H // c["H_kv"]
    eq = np.zeros_like(qn)
    ek = np.zeros_like(kn)
    bm = c["block_mask"]
    for b in range(B):
        for h in range(H):
            hk = h // grp
            head_bm = None if bm is None else (bm[b, h] if bm.ndim == 4 else bm)
            allowed = oracle.allowed_mask(np.arange(N), np.arange(N), c["causal"],
                                          None if kl is None else int(kl[b]), head_bm)
            S = np.where(allowed, c["scale"] * qn[b, h] @ kn[b, hk].T, -np.inf)
            m = S.max(axis=1, keepdims=True)
            P = np.where(allowed, np.exp(S - np.where(np.isfinite(m), m, 0.0)), 0.0)
            s = P.sum(axis=1, keepdims=True)
            P = np.divide(P, s, out=np.zeros_like(P), where=s > 0)
            Pe = P * e[b, h][:, None]
            eq[b, h] = c["scale"] * Pe @ kn[b, hk]
            ek[b, hk] += c["scale"] * Pe.T @ qn[b, h]
    return float(np.linalg.norm(eq)), float(np.linalg.norm(ek))


@pytest.mark.parametrize("i", range(N_SHORT + N_LONG), ids=_case_id)
def test_random_configuration(ea, i):
    c = _draw(i)
    q, k, v, do = workloads.random_case(c["B"], c["H"], c["N"], c["d"], c["seed"],
                                        std=c["std"], H_kv=c["H_kv"])
    kl = None if c["key_lens"] is None else torch.tensor(c["key_lens"], dtype=torch.int32)
    bm = None if c["block_mask"] is None else torch.from_numpy(c["block_mask"])
    kw = dict(scale=c["scale"], causal=c["causal"], dropout_p=c["dropout_p"], seed=c["seed"],
              offset=c["offset"], key_lens=None if kl is None else kl.cuda(),
              block_mask=None if bm is None else bm.cuda())
    qd, kd, vd, dod = (_to_dev(t, c["bnhd"]) for t in (q, k, v, do))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(qd.shape[:3], float("nan"), dtype=torch.float32, device=qd.device)
    ea.attention_fwd(qd, kd, vd, out=o, lse=lse, **kw)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (qd, kd, vd))
    ea.attention_bwd(dod, qd, kd, vd, o, lse, dq=dq, dk=dk, dv=dv, **kw)
    torch.cuda.synchronize()
    ea.check()

    okw = dict(scale=c["scale"], causal=c["causal"], dropout_p=c["dropout_p"],
               seed=c["seed"], offset=c["offset"],
               key_lens=None if kl is None else kl.numpy(),
               block_mask=c["block_mask"])
    O, L, dQ, dK, dV = oracle.attention_backward(np64(q), np64(k), np64(v), np64(do), **okw)
    assert_o(np64(o.cpu()), O, what=_case_id(i),
             factor=o_magnitude_factor(c["std"], c["dropout_p"]))
    assert max_abs(lse.cpu().numpy(), L) <= L_MAX_ABS
    # rel-L2 as everywhere, plus what D adds where dQ and dK cancel to
    # (nearly) nothing (one or two keys per row, say, where dS = P (dP - D)
    # is exactly 0): D = rowsum(dO * O) is formed from the forward's bf16 O,
    # so O's error (within the forward's bar) reaches dS and, through it, dQ
    # and dK (d_rounding_terms: that term, exactly, from the oracle's values
    # and the forward's O), and a floor of 1e-4 per element (x std^2) for dP
    # and D adding the same products in different orders
    eq, ek = d_rounding_terms(q, k, do, O, np64(o.cpu()), c, kl)
    floor = 1e-4 * max(1.0, c["std"] ** 2)
    for name, got, want, extra in (("dQ", dq, dQ, eq), ("dK", dk, dK, ek), ("dV", dv, dV, 0.0)):
        g = np64(got.cpu())
        assert not np.isnan(g).any(), name
        err = np.linalg.norm(g - want)
        bar = GRAD_REL_L2 * np.linalg.norm(want) + extra + floor * np.sqrt(want.size)
        assert err <= bar, (name, err, np.linalg.norm(want), extra)


@pytest.mark.parametrize("i", range(N_SHORT + N_LONG, N_SHORT + N_LONG + N_FP32), ids=_case_id)
def test_random_fp32_forward(ea, i):
    """fp32 inputs and output on the TF32 path: O within 1e-2 (fp32 output,
    nothing subtracted; widened as above beyond the workloads' regime) and,
    without dropout, within the bound of rounding P and V to TF32 (2^-11
    relative each; the scores take three TF32 passes), doubled, plus 1e-4
    for the fp32 sums; L within 1e-3."""
    from oracle import fp8 as oracle_fp8
    c = _draw(i)
    q, k, v, _ = workloads.random_case(c["B"], c["H"], c["N"], c["d"], c["seed"],
                                       dtype=torch.float32, std=c["std"], H_kv=c["H_kv"])
    kl = None if c["key_lens"] is None else torch.tensor(c["key_lens"], dtype=torch.int32)
    bm = None if c["block_mask"] is None else torch.from_numpy(c["block_mask"])
    kw = dict(scale=c["scale"], causal=c["causal"], dropout_p=c["dropout_p"], seed=c["seed"],
              offset=c["offset"], key_lens=None if kl is None else kl.cuda(),
              block_mask=None if bm is None else bm.cuda())
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(qd.shape[:3], float("nan"), dtype=torch.float32, device=qd.device)
    ea.attention_fwd(qd, kd, vd, out=o, lse=lse, **kw)
    torch.cuda.synchronize()
    ea.check()
    okw = dict(scale=c["scale"], causal=c["causal"], dropout_p=c["dropout_p"],
               seed=c["seed"], offset=c["offset"],
               key_lens=None if kl is None else kl.numpy(), block_mask=c["block_mask"])
    qn, kn, vn = np64(q), np64(k), np64(v)
    O, L = oracle.attention_forward(qn, kn, vn, **okw)
    err = np.abs(np64(o.cpu()) - O)
    assert not np.isnan(err).any()
    assert err.max() <= 1e-2 * o_magnitude_factor(c["std"], c["dropout_p"]), float(err.max())
    assert max_abs(lse.cpu().numpy(), L) <= L_MAX_ABS
    if not c["dropout_p"]:
        A, _ = oracle_fp8.rounding_terms(qn, kn, vn, c["scale"], causal=c["causal"],
                                         key_lens=okw["key_lens"], block_mask=c["block_mask"])
        assert np.all(err <= 2.0 ** -9 * A + 1e-4), float((err - 2.0 ** -9 * A).max())


N_DECODE = 40         # decode steps against random caches


def _draw_decode(i):
    r = np.random.default_rng(5000 + i)
    B = int(r.integers(1, 5))
    H_kv = int(r.integers(1, 5))
    group = int(r.choice([1, 2, 4, 8]))
    n_q = int(r.integers(1, 9))
    while group * n_q > 64:
        n_q //= 2
    N = int(r.choice([1, 63, 64, 65, 700, 2049])) if r.random() < 0.3 else int(r.integers(1, 3001))
    lens = [int(x) for x in r.integers(0, N + 1, size=B)]
    if r.random() < 0.3:
        lens[int(r.integers(0, B))] = int(r.choice([0, N]))
    return dict(B=B, H=H_kv * group, H_kv=H_kv, n_q=n_q, N=N, d=int(r.choice([64, 128])),
                lens=lens, causal=bool(r.random() < 0.7), bnhd=bool(r.random() < 0.3),
                seed=int(r.integers(0, 2 ** 31)))


def _decode_id(i):
    c = _draw_decode(i)
    return (f"{i}-B{c['B']}H{c['H']}/{c['H_kv']}q{c['n_q']}N{c['N']}d{c['d']}"
            + ("-causal" if c["causal"] else "") + ("-bnhd" if c["bnhd"] else ""))


@pytest.mark.parametrize("i", range(N_DECODE), ids=_decode_id)
def test_random_decode_step(ea, i):
    """attn_decode (the newest n_q positions of each sequence against its
    cache, split into chunks merged by the logsumexp rule) against the
    oracle's decode_forward: O within 1e-2 beyond its bf16 rounding, L within
    1e-3; sequences with an empty cache give O = 0 and L = -inf."""
    from tests.helpers import O_MAX_ABS, o_err
    c = _draw_decode(i)
    g = torch.Generator().manual_seed(c["seed"])
    q = torch.randn(c["B"], c["H"], c["n_q"], c["d"], generator=g).to(torch.bfloat16)
    k = torch.randn(c["B"], c["H_kv"], c["N"], c["d"], generator=g).to(torch.bfloat16)
    v = torch.randn(c["B"], c["H_kv"], c["N"], c["d"], generator=g).to(torch.bfloat16)
    lens = torch.tensor(c["lens"], dtype=torch.int32)
    kd, vd = (_to_dev(t, c["bnhd"]) for t in (k, v))
    scale = c["d"] ** -0.5
    o, lse = ea.attention_decode(q.cuda(), kd, vd, lens.cuda(), scale=scale, causal=c["causal"])
    torch.cuda.synchronize()
    ea.check()
    O, L = oracle.decode_forward(np64(q), np64(k), np64(v), scale=scale,
                                 cache_lens=lens.numpy(), causal=c["causal"])
    assert o_err(np64(o.cpu()), O) <= O_MAX_ABS, _decode_id(i)
    assert max_abs(lse.cpu().numpy(), L) <= L_MAX_ABS, _decode_id(i)


N_FP8 = 24            # E4M3 forwards (the last four few-head long cases on the split path)


def _draw_fp8(i):
    r = np.random.default_rng(7000 + i)
    long = i >= N_FP8 - 4
    B = 1 if long else int(r.integers(1, 4))
    H_kv = 1 if long else int(r.integers(1, 4))
    H = H_kv * (int(r.choice([1, 2])) if long else int(r.choice([1, 2, 4])))
    N = int(r.integers(2048, 2600)) if long else (
        int(r.choice(EDGE_N)) if r.random() < 0.4 else int(r.integers(1, 701)))
    c = dict(B=B, H=H, H_kv=H_kv, N=N, causal=bool(r.random() < 0.5),
             std=float(r.choice([0.5, 1.0, 2.0])), seed=int(r.integers(0, 2 ** 31)),
             key_lens=None, block_mask=None)
    if r.random() < 0.4:
        c["key_lens"] = [int(x) for x in r.integers(0, N + 1, size=B)]
    if not long and r.random() < 0.3:
        nb = (N + 127) // 128
        shape = (B, H, nb, nb) if r.random() < 0.5 else (nb, nb)
        c["block_mask"] = torch.from_numpy((r.random(shape) < r.uniform(0.2, 0.8)).astype(np.uint8))
    return c


def _fp8_id(i):
    c = _draw_fp8(i)
    return (f"{i}-B{c['B']}H{c['H']}/{c['H_kv']}N{c['N']}-std{c['std']}"
            + ("-causal" if c["causal"] else "") + ("-pad" if c["key_lens"] is not None else "")
            + ("-block" if c["block_mask"] is not None else ""))


@pytest.mark.parametrize("i", range(N_FP8), ids=_fp8_id)
def test_random_fp8_forward(ea, i):
    """The E4M3 forward (d = 128) against the oracle on the de-scaled inputs,
    under the E4M3 rounding bound of tests/test_gpu_fp8.py."""
    from tests.test_gpu_fp8 import FP8, _check_full
    if FP8 is None:
        pytest.skip("torch without float8_e4m3fn")
    c = _draw_fp8(i)
    _check_full(ea, c["B"], c["H"], c["H_kv"], c["N"], c["seed"], causal=c["causal"],
                key_lens=c["key_lens"], block_mask=c["block_mask"], std=c["std"])
