"""Reference oracle for fused exact attention — TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, fp64 CPU restatement of what the GPU path
computes.  It exists so that tests, the package smoke check and the bench's
CPU-baseline leg have something independent to compare against.  Nothing in
the product path (the CUDA library and its Python binding) may import it, and
it imports nothing from the product path: the two share no code.

Sources (web pages about FlashAttention, Dao et al. 2022):
  * "FlashAttention: Cơ chế Attention chính xác, nhanh và tối ưu bộ nhớ với
    nhận thức IO" (xyznot.com/vi/paper/2205.14135) — online-softmax
    statistics, block-sparse mask, stored (l, m) statistics.
  * "3.3 Hiểu sâu cơ chế Self-Attention" (infra-guide-du8.pages.dev) — the
    scaled dot-product definition (§3, §4), safe softmax (§7.2), causal mask
    (§10.2), tiling (§12.2).
  * "FlashAttention: انتباه دقيق وسريع وموفِّر للذاكرة" (azimuth.plus/paper/
    flashattention) — the step-by-step algorithm and the online-softmax update.

Modules
  attention  -- the plain definition: masked scaled scores, softmax, dropout,
                O and the per-row logsumexp L, and the chain-rule gradients.
  philox     -- Philox4x32-10 counter-based generator (Salmon et al., SC'11),
                a vectorised numpy version and an independent scalar one.
  blockwise  -- the pages' tiled online-softmax recurrence, restated; used
                only to pin the direct definition in tests.
  fp8        -- E4M3 codes with per-tensor de-scale factors as inputs (OCP
                OFP8 format), and the terms of the error bound for a kernel
                that rounds the probabilities to E4M3.

Parity status: every function is pinned by tests under tests/test_oracle_*.py;
`philox` against cuRAND's host-side Philox4x32-10 generator, an independent
implementation of the same published generator (no published known-answer
vector file is available here).
"""

from .attention import (  # noqa: F401
    allowed_mask,
    attention_forward,
    attention_backward,
    decode_forward,
    forward_rows,
    backward_keys,
    backward_rows,
    dropout_threshold,
    keep_scale,
    keep_mask,
)
from .fp8 import e4m3_value, fp8_forward, rounding_terms, rounding_terms_rows  # noqa: F401
