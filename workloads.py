"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and builds masks; it holds none of the
attention arithmetic.  Tests (GPU path and oracle alike) and bench.py take
their inputs from here, so both sides always see the same values.

Workloads (shapes of the pages' benchmarks, data synthetic):
  single-head-fp32    B=1,  H=1,  N=256,  d=64,  fp32, forward only
  bert-large          B=16, H=16, N=512,  d=64,  bf16, key padding
                      lengths ~ U{256..512} (seed 1), dropout p=0.1
                      (Philox seed 0, offset 0), non-causal
  gpt2-1k             B=8,  H=12, N=1024, d=64,  bf16, causal
  gpt2-4k             B=2,  H=12, N=4096, d=64,  bf16, causal
  long-causal-<N>     B=1,  H=16, d=128, N in {512..16384}, entries
                      N(0, 0.5^2), causal
  block-sparse-64k    B=1,  H=8,  N=65536, d=64, 128x128 block mask with
                      the diagonal and block column 0 kept and the other
                      blocks kept with Bernoulli(q) so the density is ~0.1
  gqa-4k              B=2,  H=32 query heads over H_kv=8 key/value heads,
                      N=4096, d=128, bf16, causal (the head layout of the
                      GQA comparison on the self-attention tutorial page)
  decode-gqa-8k       decode step: B=16, one new token per sequence, H=32
                      query heads over H_kv=8 key/value heads, d=128, bf16,
                      key/value caches of capacity N=8192 holding
                      U{4096..8192} keys (seed 1), causal
  fp8-long-causal-<N> the long-context sweep's shapes with E4M3 inputs,
                      forward only

Q, K, V, dO are i.i.d. normal fp32 draws from a CPU torch.Generator seeded
with 0, in the order Q, K, V, dO, scaled by the workload's std and rounded to
the workload's dtype.  K and V have H_kv heads ([B, H_kv, N, d]).

FP8 workloads store each of Q, K, V as E4M3 codes (torch.float8_e4m3fn) with
one de-scale factor per tensor: descale = amax / 448 of the fp32 draw
(448 is the largest E4M3 value), codes = round-to-nearest(x / descale).
"""

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

BLOCK = 128
LONG_SWEEP = (512, 1024, 2048, 4096, 8192, 16384)


@dataclass
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str = "bf16"          # "bf16", "fp32" or "fp8" (E4M3 inputs, bf16 output)
    causal: bool = False
    std: float = 1.0
    key_len_range: Optional[tuple] = None   # (lo, hi) inclusive, seed 1
    dropout_p: float = 0.0
    philox_seed: int = 0
    philox_offset: int = 0
    block_density: Optional[float] = None   # block-sparse target density
    fwd_only: bool = False
    seed: int = 0
    H_kv: int = 0                # key/value heads (0 = H)
    decode_n_q: int = 0          # decode step: query rows per sequence (0 = square problem)
    extra: dict = field(default_factory=dict)

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d)

    @property
    def kv_heads(self):
        return self.H_kv or self.H

    @property
    def torch_dtype(self):
        return {"fp32": torch.float32, "fp8": torch.float8_e4m3fn}.get(self.dtype, torch.bfloat16)


def _all():
    w = {
        "single-head-fp32": Workload("single-head-fp32", 1, 1, 256, 64,
                                     dtype="fp32", fwd_only=True),
        "bert-large": Workload("bert-large", 16, 16, 512, 64,
                               key_len_range=(256, 512), dropout_p=0.1),
        "gpt2-1k": Workload("gpt2-1k", 8, 12, 1024, 64, causal=True),
        "gpt2-4k": Workload("gpt2-4k", 2, 12, 4096, 64, causal=True),
        "block-sparse-64k": Workload("block-sparse-64k", 1, 8, 65536, 64,
                                     block_density=0.1),
        "gqa-4k": Workload("gqa-4k", 2, 32, 4096, 128, causal=True, H_kv=8),
        "decode-gqa-8k": Workload("decode-gqa-8k", 16, 32, 8192, 128, causal=True, H_kv=8,
                                  key_len_range=(4096, 8192), fwd_only=True, decode_n_q=1),
    }
    for n in LONG_SWEEP:
        name = f"long-causal-{n}"
        w[name] = Workload(name, 1, 16, n, 128, causal=True, std=0.5)
        w["fp8-" + name] = Workload("fp8-" + name, 1, 16, n, 128, dtype="fp8", causal=True,
                                    std=0.5, fwd_only=True)
    return w


WORKLOADS = _all()


def get(name, **overrides):
    """A workload by name, optionally with fields replaced (e.g. a smaller N)."""
    base = WORKLOADS[name]
    if not overrides:
        return base
    kw = dict(base.__dict__)
    kw.update(overrides)
    return Workload(**kw)


def make_block_mask(nb, density, seed=0):
    """uint8 [nb, nb]: diagonal and block column 0 kept, the rest Bernoulli(q).

    q is chosen so that the expected fraction of kept blocks is `density`:
    q = (density*nb^2 - (2nb - 1)) / (nb^2 - (2nb - 1)).
    """
    g = torch.Generator().manual_seed(seed)
    forced = 2 * nb - 1 if nb > 1 else 1
    total = nb * nb
    q = max(0.0, (density * total - forced) / max(1, total - forced))
    m = (torch.rand((nb, nb), generator=g) < q)
    m |= torch.eye(nb, dtype=torch.bool)
    m[:, 0] = True
    return m.to(torch.uint8)


def make_inputs(w: Workload):
    """Draw the workload's tensors on the CPU.

    Returns a dict with q, k, v, do ([B, H, N, d] in the workload dtype; do is
    None for forward-only workloads), key_lens (int32 [B] or None),
    block_mask (uint8 [nb, nb] or None) and the scalar settings.
    """
    g = torch.Generator().manual_seed(w.seed)
    shape = (w.B, w.H, w.decode_n_q or w.N, w.d)
    kv_shape = (w.B, w.kv_heads, w.N, w.d)

    def draw(sh):
        return (torch.randn(sh, generator=g, dtype=torch.float32) * w.std
                ).to(w.torch_dtype)

    descales = {}
    if w.dtype == "fp8":
        q, k, v = [fp8_quantize(torch.randn(sh, generator=g, dtype=torch.float32) * w.std)
                   for sh in (shape, kv_shape, kv_shape)]
        descales = dict(q_descale=q[1], k_descale=k[1], v_descale=v[1])
        q, k, v = q[0], k[0], v[0]
    else:
        q, k, v = draw(shape), draw(kv_shape), draw(kv_shape)
    do = None if w.fwd_only else draw(shape)
    key_lens = None
    if w.key_len_range is not None:
        lo, hi = w.key_len_range
        gl = torch.Generator().manual_seed(1)
        key_lens = torch.randint(lo, hi + 1, (w.B,), generator=gl,
                                 dtype=torch.int64).to(torch.int32)
    block_mask = None
    if w.block_density is not None:
        nb = (w.N + BLOCK - 1) // BLOCK
        block_mask = make_block_mask(nb, w.block_density, seed=0)
    return dict(q=q, k=k, v=v, do=do, key_lens=key_lens,
                block_mask=block_mask, scale=w.scale, causal=w.causal,
                dropout_p=w.dropout_p, seed=w.philox_seed,
                offset=w.philox_offset, **descales)


def fp8_quantize(x):
    """E4M3 codes of an fp32 tensor with one de-scale factor: returns
    (codes as torch.float8_e4m3fn, descale) with descale = amax / 448 (a
    float32 value; 1 for an all-zero tensor) and codes = x / descale rounded
    to the nearest E4M3 value."""
    amax = float(x.abs().max()) if x.numel() else 0.0
    descale = float(torch.tensor(amax / 448.0 if amax > 0 else 1.0, dtype=torch.float32))
    return (x / descale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn), descale


def random_case_fp8(B, H, N, d, seed, std=1.0, H_kv=None):
    """Small E4M3 q, k, v with their de-scale factors: [(codes, descale)] * 3."""
    g = torch.Generator().manual_seed(seed)
    kv_shape = (B, H if H_kv is None else H_kv, N, d)
    return [fp8_quantize(torch.randn(sh, generator=g) * std)
            for sh in ((B, H, N, d), kv_shape, kv_shape)]


def random_case(B, H, N, d, seed, dtype=torch.bfloat16, std=1.0, H_kv=None):
    """Small i.i.d. normal q, k, v, do for edge-case tests (k, v with H_kv
    heads when given)."""
    g = torch.Generator().manual_seed(seed)
    shape = (B, H, N, d)
    kv_shape = (B, H if H_kv is None else H_kv, N, d)
    return [(torch.randn(sh, generator=g) * std).to(dtype)
            for sh in (shape, kv_shape, kv_shape, shape)]
