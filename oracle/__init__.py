"""FP64 CPU oracle for deterministic selected-token log-probability.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA
library never calls it, and it shares no code, header, table or constant
generator with the CUDA library: it reads numpy arrays and returns numpy
arrays.  Inputs come from the seeded generator in ``synth`` (or from a test),
never from the GPU path.

What it computes, and where the pages define it:

* ``logprob`` -- the plain full-vocabulary definition (no tiles): LSE over the
  real vocabulary, the selected log-probability, and its gradient
  ``g * (onehot(target) - softmax)``, and the softmax's entropy; plus the
  tiled method's own steps
  (per-tile (max, sumexp) partials with the (-inf, 0) identity, merged in
  fixed tile-index order), so that the method's algebra can be pinned
  against the plain definition.
* ``lmhead`` -- the same quantities when the logits are ``hidden @ W^T``
  (the fused lm_head variant), plus the gradients of hidden and W.
* ``grpo`` -- the token-mean GRPO loss of per-token log-probabilities, with
  an optional KL term, and its gradient with respect to each logp.

Every function is FP64 and loops only where the definition does.
"""
from .logprob import (  # noqa: F401
    NEG_INF,
    active_rows,
    bf16_bits_to_f64,
    dlogits,
    entropy,
    fold_partials,
    merge_partials,
    lse_full,
    lse_of_values,
    selected_logp,
    tile_bounds,
    tile_partials,
)
from .lmhead import lmhead_logits, lmhead_forward, lmhead_grads  # noqa: F401
from .grpo import grpo_loss  # noqa: F401
