"""Float64 CPU oracle for speculative-decoding verification.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, deliberately unoptimised
statement of what the verification path computes, used to check the CUDA library.
Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference arm may import it.  The product (``speculative_decoding_verification_gb300``)
never imports, calls or falls back to it, and this package imports nothing from the
product.  The two share no code; only the seeded input generators in ``synth`` feed both.

Sources (cited by page title and section):
  * "Speculative Speculative Decoding" notes (SSD notes): §2.2 SD recap, §4.3 Theorem 12,
    §4.4 Theorems 15 and 19, §5.1 cache construction, §7.1 Corollary 16.
  * SSD abstract page (hyper.ai, 2603.03251), "Method": the speculation cache, the
    Theorem 12 fan-out formula, the Saguaro sampling scheme sigma_{F,C}.
  * "Accelerating LLM Decoding with Speculative Sampling (2023)" notes (SpS notes):
    §1 notation (q target, p draft), §3 modified rejection sampling, §6 checks.
  * "Mirror Speculative Decoding" notes (Mirror-SD notes): §1.1 tree drafts, §2 greedy verify,
    §3.1 top-kappa early-exit roots and branch-complete trees, §3.2-§3.3 verification vs. reuse.
  * "3-Model Speculative Decoding (PyramidSD)" notes (PyramidSD notes): "Method", the fuzzy
    (divergence-threshold) and assisted acceptance of one verification stage.

Every function works in float64 on logits already converted exactly to float64
(bf16 -> f64 and f32 -> f64 are exact).  Ties in any ranking go to the lowest token id.
"""
from .dist import (argmax_first, softmax_t, nucleus, saguaro_transform, row_distribution,  # noqa: F401
                   inverse_cdf)
from .verify import verify, draft_sample  # noqa: F401
from .saguaro import fanout, cache_keys, cache_lookup  # noqa: F401
from .mirror import topk_rows, mirror_reuse  # noqa: F401
from .fuzzy import jensen_shannon, fuzzy_verify  # noqa: F401
from .tree import tree_verify, tree_reuse  # noqa: F401
