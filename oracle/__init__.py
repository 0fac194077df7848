"""Plain CPU oracle for the S³R paged decode-attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and its ``--impl reference`` arm) may use it.  It shares
no code, table or constant generator with the CUDA library; the two meet only
through the seeded inputs made by the ``workloads`` package.

Everything here is written from the definitions the S³R pages give (or, where
they leave a step open, from the reading stated in each docstring), in float64,
as plain loops over (sequence, head, row) with NumPy doing the inner dot
products, sums and sorts.  No blocking, fusion or reordering beyond the
definitions.

Pages cited (titles and sections, as printed):
  * [abstract]  "S³R: Fast and Faithful RL Rollouts via Self-Sparse Speculative
    Decoding", arXiv 2610.13202 listing (paperdot / space-kitty mirrors).
  * [wispaper]  wispaper.ai research summary "Can self-sparse speculative
    decoding speed up RL rollouts without changing response groups".
  * [rebas]     rebasdaily.com article on S³R (Chinese).
  * [ritwork]   rit.work blog "s3r-sparse-drafting-dense-verification" (Russian).

Parity status of each function is stated in its module header.
"""

from .bf16 import bf16_bits_to_f64
from .attention import (
    PAGE_SIZE,
    dense_decode_attn,
    sparse_draft_attn,
    verify_attn,
)
from .selection import select_draft_pages, selection_budget
from .philox import philox4x32_10, philox_uniform, STREAM_ACCEPT, STREAM_RESAMPLE, STREAM_DRAFT
from .spec_sample import spec_sample, residual_row
from .draft_sample import sample_draft_tokens
from .kv_cache import kv_append, commit_lengths
from .round import closed_round

__all__ = [
    "PAGE_SIZE",
    "bf16_bits_to_f64",
    "dense_decode_attn",
    "sparse_draft_attn",
    "verify_attn",
    "select_draft_pages",
    "selection_budget",
    "philox4x32_10",
    "philox_uniform",
    "STREAM_ACCEPT",
    "STREAM_RESAMPLE",
    "STREAM_DRAFT",
    "spec_sample",
    "residual_row",
    "sample_draft_tokens",
    "kv_append",
    "commit_lengths",
    "closed_round",
]
