"""Shared helpers for the GPU parity tests: tolerances, conversions, oracle calls."""

import numpy as np
import torch

# Tolerances of the parity bar (bf16 I/O, fp32 accumulation):
O_MAX_ABS = 1e-2      # forward output: max |O_gpu - O_oracle| beyond the output's
                      # own bf16 rounding (see o_err)
BF16_HALF_ULP_REL = 2.0 ** -8   # one round-to-nearest into bf16, relative
L_MAX_ABS = 1e-3      # logsumexp, max |L_gpu - L_oracle|
GRAD_REL_L2 = 1e-2    # dQ, dK, dV: ||g_gpu - g_oracle|| / ||g_oracle||
# Below this magnitude half a bf16 ulp of the output (<= 2^-8 |O|) stays at
# or under half of O_MAX_ABS, so there the plain bound |O_gpu - O_oracle| <=
# O_MAX_ABS is checked as well, with nothing subtracted.
O_PLAIN_BELOW = 1.28


def np64(t):
    """Exact fp64 copy of a (bf16/fp32) tensor as numpy."""
    return t.detach().to("cpu", torch.float64).numpy()


def to_dev(x, device="cuda"):
    return None if x is None else x.to(device)


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    with np.errstate(invalid="ignore"):
        both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
        d = np.where(both_inf, 0.0, np.abs(a - b))
    return float(np.nanmax(np.where(np.isnan(d), np.inf, d)))


def o_err(got, want, out_bf16=True):
    """Max |got - want| beyond the output's own rounding.

    A bf16 output cannot be closer to the exact value than half a bf16 ulp
    (<= 2^-8 |want|), so that much is subtracted per element before taking
    the max; for fp32 outputs nothing is subtracted.
    """
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if got.size == 0:
        return 0.0
    slack = BF16_HALF_ULP_REL * np.abs(want) if out_bf16 else 0.0
    d = np.abs(got - want) - slack
    return float(np.max(np.where(np.isnan(d), np.inf, d)))


def o_plain_err(got, want, below=O_PLAIN_BELOW):
    """Max |got - want| over the elements with |want| < below (no slack)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    sel = np.abs(want) < below
    return max_abs(got[sel], want[sel]) if sel.any() else 0.0


def o_magnitude_factor(std, dropout_p):
    """How much the O bar widens for inputs beyond the workloads' regime
    (value std up to 1, dropout up to 0.1): the kernel's O error (bf16
    P~ = P Z / (1 - p) times V, fp32 accumulation) grows linearly with |V|
    and with 1 / (1 - p).  1 inside that regime."""
    return max(1.0, std) * max(1.0, 0.9 / (1.0 - dropout_p))


def assert_o(got, want, out_bf16=True, what="", factor=1.0):
    """The forward-output bar: within O_MAX_ABS beyond the output's own bf16
    rounding everywhere, and within plain O_MAX_ABS where |O| < O_PLAIN_BELOW
    (the bar times `factor`, see o_magnitude_factor; 1 for every fixed case;
    the plain check keeps the region where the output's rounding is at most
    half of the unwidened bar)."""
    bound = O_MAX_ABS * factor
    e1 = o_err(got, want, out_bf16)
    e2 = o_plain_err(got, want)
    assert e1 <= bound and e2 <= bound, (what, e1, e2, bound)
    return e1, e2


def tile_samples(N, seed, tile=128):
    """Row (or key) indices that reach every 128-row tile of a length-N
    sequence: one random index inside each tile, plus the first and last
    index of the sequence and of its first and last tiles."""
    rng = np.random.default_rng(seed)
    nb = (N + tile - 1) // tile
    idx = {min(N - 1, tile * t + int(rng.integers(tile))) for t in range(nb)}
    idx |= {0, min(tile - 1, N - 1), tile * (nb - 1), N - 1}
    return np.array(sorted(idx))


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    if nb == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def oracle_kwargs(inp):
    """Translate a workloads.make_inputs dict into oracle keyword arguments."""
    kl = inp.get("key_lens")
    bm = inp.get("block_mask")
    return dict(scale=inp["scale"], causal=inp["causal"],
                key_lens=None if kl is None else kl.numpy(),
                block_mask=None if bm is None else bm.numpy(),
                dropout_p=inp["dropout_p"], seed=inp["seed"], offset=inp["offset"])


def api_kwargs(inp, device="cuda"):
    """Translate a workloads.make_inputs dict into API keyword arguments."""
    return dict(scale=inp["scale"], causal=inp["causal"],
                key_lens=to_dev(inp.get("key_lens"), device),
                block_mask=to_dev(inp.get("block_mask"), device),
                dropout_p=inp["dropout_p"], seed=inp["seed"], offset=inp["offset"])
