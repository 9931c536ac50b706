"""FP64 oracle of the fused lm_head variant: logits = hidden @ W^T, never rounded.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The fused variant computes the same selected log-probability as the
streaming path, but from hidden states [T, H] and the lm_head weight
[V_padded, H] instead of materialised logits; the optional fused kernel of
issue #323 ("Validation Boundary": "the optional PR6 fused kernel") is its
prior art.  Reading used here: the logits are the exact products
x_rc = sum_k h_rk * W_ck of the BF16 inputs (FP64 here), with no rounding to
BF16, and rows of W at c >= V_real are padding that takes no part.

Gradients of L = sum_r g_r * logp_r:
  dlogits_rc = g_r * ([c == t_r] - softmax_rc)   (0 on inactive rows, padded c)
  dhidden    = dlogits @ W
  dW         = dlogits^T @ hidden                (rows c >= V_real are 0)
The matrix products use numpy's FP64 matmul as a library step.
"""
import numpy as np

from .logprob import bf16_bits_to_f64, lse_of_values


def lmhead_logits(hidden_bits, weight_bits, v_cols=None, chunk=16384):
    """FP64 [R, v_cols] logits hidden @ W[:v_cols]^T, computed in column chunks."""
    weight_bits = np.asarray(weight_bits)
    v = weight_bits.shape[0] if v_cols is None else v_cols
    h = bf16_bits_to_f64(hidden_bits)
    out = np.empty((h.shape[0], v), dtype=np.float64)
    for c0 in range(0, v, chunk):
        c1 = min(v, c0 + chunk)
        out[:, c0:c1] = h @ bf16_bits_to_f64(weight_bits[c0:c1]).T
    return out


def lmhead_forward(hidden_bits, weight_bits, targets, active, v_real):
    """(logp, lse, x) for the given hidden rows: logp = x_t - LSE on active rows, else 0."""
    x = lmhead_logits(hidden_bits, weight_bits, v_cols=v_real)
    lse = lse_of_values(x)
    active = np.asarray(active, dtype=bool)
    targets = np.asarray(targets)
    logp = np.zeros(len(lse))
    rows = np.nonzero(active)[0]
    t = targets[rows]
    if np.any((t < 0) | (t >= v_real)):
        raise ValueError("active target outside [0, V_real)")
    logp[rows] = x[rows, t] - lse[rows]
    return logp, lse, x


def lmhead_dlogits(x, lse, targets, active, grad):
    """FP64 dlogits over the real vocabulary from the logits x and their LSE."""
    active = np.asarray(active, dtype=bool)
    d = np.zeros_like(x)
    rows = np.nonzero(active)[0]
    if len(rows):
        with np.errstate(invalid="ignore", over="ignore"):
            p = np.exp(x[rows] - lse[rows, None])
        dr = -p
        dr[np.arange(len(rows)), np.asarray(targets)[rows]] += 1.0
        d[rows] = dr * np.asarray(grad, dtype=np.float64)[rows, None]
    return d


def lmhead_grads(hidden_bits, weight_bits, targets, active, grad, v_real):
    """(dhidden [R, H], dweight [V_padded, H]) in FP64, over all given rows."""
    weight_bits = np.asarray(weight_bits)
    logp, lse, x = lmhead_forward(hidden_bits, weight_bits, targets, active, v_real)
    d = lmhead_dlogits(x, lse, targets, active, grad)
    W = bf16_bits_to_f64(weight_bits[:v_real])
    h = bf16_bits_to_f64(hidden_bits)
    dh = d @ W
    dw = np.zeros((weight_bits.shape[0], h.shape[1]))
    dw[:v_real] = d.T @ h
    return dh, dw
