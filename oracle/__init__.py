"""CPU oracle for certified sparse decode attention -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, independent restatement of the decode step of
"Certified Sparse Attention via Perturbed Retrieval" (arXiv 2610.24991).
Sources, cited by page and section in every function:
  * picx.dev summary -- "Methodology / Problem Setup", "Algorithm Components"
    1-4, "Theoretical Contributions" (Theorems 1-4);
  * readsearch.ai abstract page -- "Abstract" (one scan serves a GQA group;
    the perturbations are drawn anew for each decode step).

It shares no code with the CUDA library under
``certified_sparse_attention_gb300/``: no headers, kernels, helpers, constants
or tables.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the product path never does.

Precision: exact scores, weights, statistics and certificates are float64.
The pieces the GPU must reproduce bit for bit -- the 4-bit key quantiser, the
deterministic score bounds, the hashed perturbations and the candidate levels
-- are emulated step by step in IEEE float32 (numpy float32, no fused
multiply-add), with the operation order written out in ``bounds.py`` and
``fp32.py``.

Parity status per function (the pins live in ``tests/test_oracle_*.py``):
  * hashing / log2, quantiser (4- and 8-bit), bounds, inclusion law,
    nestedness, unbiasedness, exact special cases, the per-level sums (a
    pool summed by hand, and a per-key event formulation), the Chernoff
    interval (exact Poisson-binomial coverage, not over-wide), the G and H
    events, the Pinelis constant (the exact tail of a binomial sum near the
    bound: a log term 20% smaller or 50% larger fails), beta (the
    derivation's identity), coverage, the Theorem 2 error bound and sample
    size: pinned (closed forms, brute force, exact tails, Monte Carlo).
  * the decode step as a whole: its pieces are pinned as above, and its
    composition by exact special cases and by metamorphic relations between
    runs (monotone in eps and delta, homogeneous in the values, invariant
    to a common score shift).  The pages print no worked example, so no
    external value fixes which level a given head stops at: the readings
    the certificate rests on (the event budget, the variance proxy, the
    Bernstein form) are the pages' open choices, listed with the tests.
"""
from .fp32 import tree_sum_f32, log2_m53_f32
from .hashing import mix64, group_key, key_hashes, perturb_t
from .quantize import quantize_keys, value_sq_norms_f32, vmax_blocks
from .bounds import query_prep, key_bounds, QM_DEFAULT
from .certificate import chernoff_interval, certificate_levels
from .step import (Params, grid_J, oracle_decode_group, dense_attention,
                   GroupResult, exact_levels, level_sums, score_f32,
                   cstar_lower_f32, bound_levels_f32)

__all__ = [
    "tree_sum_f32", "log2_m53_f32", "mix64", "group_key", "key_hashes",
    "perturb_t", "quantize_keys", "value_sq_norms_f32", "vmax_blocks", "query_prep", "key_bounds",
    "QM_DEFAULT", "chernoff_interval", "certificate_levels", "Params",
    "grid_J", "oracle_decode_group", "dense_attention", "GroupResult",
    "exact_levels", "level_sums", "score_f32", "cstar_lower_f32",
    "bound_levels_f32",
]
