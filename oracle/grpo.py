"""FP64 oracle of the GRPO token-level loss reduction.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name a GRPO loss contract (issue #323 "[WS2][Logprob] H100
validation and reproduction guide", "Validation Boundary": the PR5 GRPO
contract tests) and KL-regularised RL runs (the H100 matrix document,
"Completed full-model matrix": KL coefficient 0.01), but print no formula.
The convention computed here, stated in full:

* N = number of active tokens of the batch (token mean); with N = 0 the loss
  and every gradient are 0.
* per active token r: the policy term -A_r * logp_r, and with a reference
  log-probability ref_r the KL term beta * k3_r with
  k3_r = exp(ref_r - logp_r) - (ref_r - logp_r) - 1 (the per-token k3
  estimator of KL(pi || pi_ref), >= 0, 0 where ref_r = logp_r);
* loss = (1/N) * sum over active r of (-A_r * logp_r + beta * k3_r);
* g_r = d loss / d logp_r = (mask_r / N) * (-A_r + beta * (1 - exp(ref_r - logp_r))),
  the upstream gradient of the backward; 0 on inactive rows.
"""
import numpy as np


def grpo_loss(logp, advantage, active, ref_logp=None, beta=0.0):
    """(loss, g, N) in FP64 for per-token logp, advantages and the active mask."""
    logp = np.asarray(logp, dtype=np.float64)
    adv = np.asarray(advantage, dtype=np.float64)
    act = np.asarray(active, dtype=bool)
    n = int(act.sum())
    if n == 0:
        return 0.0, np.zeros(len(logp)), 0
    terms = -adv * logp
    dterm = -adv
    if ref_logp is not None:
        d = np.asarray(ref_logp, dtype=np.float64) - logp
        terms = terms + beta * (np.exp(d) - d - 1.0)
        dterm = dterm + beta * (1.0 - np.exp(d))
    loss = float(terms[act].sum()) / n
    g = np.where(act, dterm / n, 0.0)
    return loss, g, n
