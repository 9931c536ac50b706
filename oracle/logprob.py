"""FP64 oracle of selected-token log-probability over a (tiled) vocabulary.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources, by page and section:

* PR #289 "[WS2][PR4][Logp] feat: add distributed TP/CP logprob drift report",
  PR-1 commit message (the typed contract): selected-token logprob over a
  vocabulary with "padded-vs-real vocab", an active-token mask or
  ignore_index, and an FP32 (max, sumexp) merge in fixed global
  vocab-shard index order.
* Same PR, commit "docs: state that cross-TP bitwise equality needs a global
  tile-level merge structure ...": padded columns are masked to -inf before
  the local (max, sumexp) partials are formed, and the tiles are global
  (independent of the TP partitioning).
* Same PR, the "typed contract" commit: the (-inf, 0) identity partial for
  padding-only or all -inf shards; MaskMode explicit_active_mask |
  ignore_index (inactive targets need not hold ignore_index);
  LogprobOutputSpec = FP32 selected logprob and FP32 vocabulary LSE.
* Same PR, review excerpt of ``vocab_parallel_logp.py`` (the entry point):
  active targets are validated against the real vocabulary, and a
  non-finite LSE on an active row is an error.
* Same PR, PR body "Comparison contract": LSE drift covers every token row;
  selected-logprob drift covers active rows only.
* Issue #323 "[WS2][Logprob] H100 validation and reproduction guide ...",
  "H100 validation matrix": BF16 logits with FP32 accumulation, compared
  with an independent full-vocabulary oracle.

The merge of two partials is the log-sum-exp identity
``log(e^a + e^b) = m + log(e^(a-m) + e^(b-m))`` with ``m = max(a, b)``:
for (m1, s1), (m2, s2) the merged partial is
``m = max(m1, m2), s = s1 * exp(m1 - m) + s2 * exp(m2 - m)``.  The pages
do not print these formulas; they follow from the definition of a
(max, sumexp) partial.

Readings where the pages are silent (each listed in the design notes):
an operand with m = -inf contributes exactly 0 (no -inf - -inf NaN); an
all -inf row has LSE = -inf; NaN propagates; inactive rows get logp = 0 and
dlogits = 0; padded columns of dlogits are 0.
"""
import numpy as np

NEG_INF = float("-inf")


def bf16_bits_to_f64(bits):
    """Exact value of BF16 bit patterns (uint16 array) as float64.

    A BF16 number is the upper half of an IEEE binary32, so widening the bits
    by 16 zero bits gives the float32 with the same value, exactly.
    """
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to NaN
        return u.view(np.float32).astype(np.float64)


def active_rows(targets, mask, mask_mode, ignore_index):
    """Which rows are active: explicit mask (mode 0) or target != ignore_index (mode 1)."""
    if mask_mode == 0:
        return np.asarray(mask) != 0
    return np.asarray(targets) != ignore_index


def lse_full(logits_bits, v_real):
    """Plain definition: LSE_r = log sum_{c < v_real} exp(x_rc), in FP64, no tiles.

    Columns c >= v_real (padding) take no part.  Computed as M + log sum
    exp(x - M) with M the row maximum; an all -inf row gives -inf and a NaN
    anywhere in the real columns gives NaN.
    """
    return lse_of_values(bf16_bits_to_f64(np.asarray(logits_bits)[:, :v_real]))


def lse_of_values(x):
    """LSE of each row of an FP64 matrix of real-vocabulary logits (see lse_full)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        M = x.max(axis=1)
        S = np.exp(x - M[:, None]).sum(axis=1)
        lse = M + np.log(S)
    lse[M == -np.inf] = -np.inf
    return lse


def selected_logp(logits_bits, targets, active, v_real):
    """(logp, lse): logp_r = x_{r, t_r} - LSE_r on active rows, exactly 0 on inactive rows.

    LSE is returned for every row.  An inactive row's target is never used
    as an index.  An active target outside [0, v_real) raises ValueError
    (the pages validate active targets against the real vocabulary).
    """
    logits_bits = np.asarray(logits_bits)
    targets = np.asarray(targets)
    active = np.asarray(active, dtype=bool)
    lse = lse_full(logits_bits, v_real)
    logp = np.zeros(len(lse), dtype=np.float64)
    rows = np.nonzero(active)[0]
    t = targets[rows]
    if np.any((t < 0) | (t >= v_real)):
        raise ValueError("active target outside [0, V_real)")
    xt = bf16_bits_to_f64(logits_bits[rows, t])
    with np.errstate(invalid="ignore"):
        logp[rows] = xt - lse[rows]
    return logp, lse


def dlogits(logits_bits, targets, active, grad, v_real, v_padded):
    """Gradient of sum_r g_r * logp_r with respect to the logits, FP64 [R, v_padded].

    Active row r, real column c: g_r * ([c == t_r] - exp(x_rc - LSE_r)).
    Padded columns (c >= v_real) and inactive rows: exactly 0.
    """
    logits_bits = np.asarray(logits_bits)
    active = np.asarray(active, dtype=bool)
    grad = np.asarray(grad, dtype=np.float64)
    R = logits_bits.shape[0]
    out = np.zeros((R, v_padded), dtype=np.float64)
    lse = lse_full(logits_bits, v_real)
    rows = np.nonzero(active)[0]
    if len(rows) == 0:
        return out
    x = bf16_bits_to_f64(logits_bits[rows, :v_real])
    with np.errstate(invalid="ignore", over="ignore"):
        p = np.exp(x - lse[rows, None])
    d = -p
    t = np.asarray(targets)[rows]
    if np.any((t < 0) | (t >= v_real)):
        raise ValueError("active target outside [0, V_real)")
    d[np.arange(len(rows)), t] += 1.0
    out[rows, :v_real] = d * grad[rows, None]
    return out


def entropy(logits_bits, v_real):
    """Entropy of each row's softmax over the real vocabulary, FP64, no tiles.

    H_r = -sum_{c < v_real} p_rc log p_rc with p_r = softmax(x_r[:v_real]); a
    column with p = 0 adds 0.  The pages log a mean policy entropy beside the
    loss in their RL runs (the H100 matrix document, "Completed full-model
    matrix"); the formula is Shannon's definition.  A row whose LSE is not
    finite (all -inf, +inf or NaN in its real columns) has no distribution:
    NaN.
    """
    x = bf16_bits_to_f64(np.asarray(logits_bits)[:, :v_real])
    lse = lse_of_values(x)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        logp = x - lse[:, None]
        p = np.exp(logp)
        terms = np.where(p > 0, -p * logp, 0.0)
    h = terms.sum(axis=1)
    h[~np.isfinite(lse)] = np.nan
    return h


def tile_bounds(v_padded, num_tiles):
    """Column ranges [k*W, (k+1)*W) of the num_tiles global tiles, W = v_padded / num_tiles."""
    if num_tiles <= 0 or v_padded % num_tiles:
        raise ValueError("vocabulary is not tileable: num_tiles must divide V_padded")
    w = v_padded // num_tiles
    return [(k * w, (k + 1) * w) for k in range(num_tiles)]


def tile_partials(logits_bits, v_real, v_padded, num_tiles):
    """The method's per-tile partials (m_k, s_k), FP64 [R, num_tiles] each.

    Tile k covers columns [k*W, (k+1)*W).  Columns c >= v_real are -inf.
    m_k is the tile maximum and s_k = sum exp(x - m_k); a tile with
    m_k = -inf (padding only, or all -inf) is the identity (-inf, 0).
    """
    logits_bits = np.asarray(logits_bits)
    R = logits_bits.shape[0]
    m = np.full((R, num_tiles), -np.inf)
    s = np.zeros((R, num_tiles))
    for k, (c0, c1) in enumerate(tile_bounds(v_padded, num_tiles)):
        hi = min(c1, v_real)
        if hi <= c0:
            continue  # padding-only tile: identity partial
        x = bf16_bits_to_f64(logits_bits[:, c0:hi])
        with np.errstate(invalid="ignore", over="ignore"):
            mk = x.max(axis=1)
            sk = np.exp(x - mk[:, None]).sum(axis=1)
        empty = mk == -np.inf
        sk[empty] = 0.0
        m[:, k] = mk
        s[:, k] = sk
    return m, s


def merge_partials(m1, s1, m2, s2):
    """Merge two (max, sumexp) partials; an operand with m = -inf contributes 0."""
    m1, s1, m2, s2 = (np.asarray(a, dtype=np.float64) for a in (m1, s1, m2, s2))
    m = np.maximum(m1, m2)  # NaN propagates
    with np.errstate(invalid="ignore", over="ignore"):
        a = np.where(m1 == -np.inf, 0.0, s1 * np.exp(m1 - m))
        b = np.where(m2 == -np.inf, 0.0, s2 * np.exp(m2 - m))
    return m, a + b


def fold_partials(m, s):
    """Left fold of the partials over k = 0..NT-1 from the identity (-inf, 0); returns LSE.

    This is the fixed global tile-index order: the same sequence of merges
    whatever the vocabulary-parallel degree.  LSE = m + log s, -inf when
    m = -inf.
    """
    m = np.asarray(m, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    R, NT = m.shape
    acc_m = np.full(R, -np.inf)
    acc_s = np.zeros(R)
    for k in range(NT):
        acc_m, acc_s = merge_partials(acc_m, acc_s, m[:, k], s[:, k])
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = acc_m + np.log(acc_s)
    lse[acc_m == -np.inf] = -np.inf
    return lse
