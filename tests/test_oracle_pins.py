"""Pins of the FP64 oracle against what the mathematics and the pages fix.

Each test checks the oracle against something other than itself: closed
forms, a direct pure-Python summation, a library routine
(scipy.special.logsumexp), finite differences of the forward definition,
and invariants.  ``test_pins_catch_planted_mistakes`` plants plausible
mistakes in copies of the oracle's functions and shows that a pin fails
for each.
"""
import math
import random

import numpy as np
import pytest
import scipy.special

import oracle

LN = math.log


def bf16_bits(values):
    """BF16 bits of float values that are exactly representable in BF16 (checked)."""
    f = np.asarray(values, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in BF16"
    return (u >> 16).astype(np.uint16)


def rand_bf16(rng, shape, scale=3.0):
    """Random finite BF16 bits (round-to-nearest-even of scaled normals)."""
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def garbage_bits(rng, shape):
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)


# ----------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("v_real,v_padded", [(151936, 151936), (151936, 152576), (1, 8), (37, 40)])
@pytest.mark.parametrize("c", [0.0, 1.5, -3.25, 20.0])
def test_uniform_logits_closed_form(v_real, v_padded, c):
    rng = np.random.default_rng(1)
    row = np.empty((1, v_padded), dtype=np.uint16)
    row[0, :v_real] = bf16_bits([c])[0]
    row[0, v_real:] = garbage_bits(rng, v_padded - v_real)  # padding must not matter
    lse = oracle.lse_full(row, v_real)[0]
    assert abs(lse - (c + LN(v_real))) <= 1e-12 * max(1.0, abs(c) + LN(v_real) + 1)
    logp, _ = oracle.selected_logp(row, np.array([v_real // 2]), np.array([True]), v_real)
    assert abs(logp[0] - (-LN(v_real))) <= 1e-12 * (LN(v_real) + 1)


def test_uniform_closed_form_values():
    # ln 151936 and ln 152576, the real and padded Qwen3 vocabularies
    row = np.zeros((2, 152576), dtype=np.uint16)
    assert abs(oracle.lse_full(row, 151936)[0] - 11.931214658529285) < 1e-13
    assert abs(oracle.lse_full(row, 152576)[0] - 11.935418111544912) < 1e-13


@pytest.mark.parametrize("s", [1.0, 15.0, 30.0, 60.0])
def test_one_hot_spike_closed_form(s):
    v = 151936
    t = 12345
    row = np.zeros((1, v), dtype=np.uint16)
    row[0, t] = bf16_bits([s])[0]
    logp, lse = oracle.selected_logp(row, np.array([t]), np.array([True]), v)
    want = -math.log1p((v - 1) * math.exp(-s))
    assert abs(logp[0] - want) <= 1e-14 + 1e-12 * abs(want)
    assert abs(lse[0] - (s + math.log1p((v - 1) * math.exp(-s)))) <= 1e-12 * (s + 1)
    if s == 15.0:
        assert abs(want - (-0.045429541755874)) < 1e-12


def test_single_finite_column():
    row = np.full((1, 16), bf16_bits([-np.inf])[0], dtype=np.uint16)
    row[0, 5] = bf16_bits([2.5])[0]
    assert oracle.lse_full(row, 16)[0] == 2.5


# ----------------------------------------------------------------------------- brute force

def brute_lse(values):
    """Direct summation in pure Python: log of the exactly rounded sum of exp(x)."""
    return math.log(math.fsum(math.exp(v) for v in values))


def test_brute_force_tiny_vocab():
    rng = np.random.default_rng(7)
    for _ in range(200):
        v_real = int(rng.integers(1, 65))
        v_padded = v_real + int(rng.integers(0, 40))
        bits = rand_bf16(rng, (3, v_padded), scale=4.0)
        bits[:, v_real:] = garbage_bits(rng, (3, v_padded - v_real))
        lse = oracle.lse_full(bits, v_real)
        for r in range(3):
            vals = [float(x) for x in oracle.bf16_bits_to_f64(bits[r, :v_real])]
            assert abs(lse[r] - brute_lse(vals)) <= 1e-13 * max(1.0, abs(lse[r]))


def test_matches_scipy_logsumexp():
    rng = np.random.default_rng(11)
    bits = rand_bf16(rng, (8, 5000), scale=3.0)
    x = oracle.bf16_bits_to_f64(bits[:, :4321])
    np.testing.assert_allclose(oracle.lse_full(bits, 4321), scipy.special.logsumexp(x, axis=1),
                               rtol=1e-14, atol=1e-13)


def test_bf16_widening_is_exact():
    # every finite BF16 pattern round-trips through the float64 value
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_bits_to_f64(bits)
    finite = np.isfinite(v)
    back = (v[finite].astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(back, bits[finite])
    assert oracle.bf16_bits_to_f64(np.array([0x3F80], dtype=np.uint16))[0] == 1.0
    assert oracle.bf16_bits_to_f64(np.array([0xC040], dtype=np.uint16))[0] == -3.0


# ----------------------------------------------------------------------------- invariants

def test_shift_invariance():
    rng = np.random.default_rng(3)
    k = rng.integers(-120, 120, size=(4, 3000))
    x = k / 8.0                                  # exact in BF16 (8 significant bits)
    for c in (1.0, -4.0, 3.0):
        a = oracle.lse_full(bf16_bits(x), 3000)
        b = oracle.lse_full(bf16_bits(x + c), 3000)  # |x + c| < 32 stays exact
        np.testing.assert_allclose(b, a + c, rtol=0, atol=1e-12)


def test_special_values():
    v = 64
    ninf, nan, inf = (bf16_bits([-np.inf])[0], np.uint16(0x7FC0), bf16_bits([np.inf])[0])
    rows = np.zeros((4, v + 8), dtype=np.uint16)
    rows[0, :v] = ninf                  # all -inf -> -inf
    rows[1, 3] = nan                    # NaN in the real vocabulary -> NaN
    rows[2, v:] = nan                   # NaN in padding -> no effect
    rows[3, 7] = inf                    # +inf -> not finite
    lse = oracle.lse_full(rows, v)
    assert lse[0] == -np.inf
    assert np.isnan(lse[1])
    assert lse[2] == LN(v)
    assert not np.isfinite(lse[3])


# ----------------------------------------------------------------------------- masking

def test_inactive_rows_and_poison_targets():
    rng = np.random.default_rng(5)
    v_real, v_padded = 100, 104
    bits = rand_bf16(rng, (6, v_padded))
    active = np.array([1, 0, 1, 0, 1, 0], dtype=bool)
    targets = np.array([3, -7, 99, v_padded + 5, 0, 10**12])  # poison on inactive rows
    logp, lse = oracle.selected_logp(bits, targets, active, v_real)
    assert np.all(logp[~active] == 0.0) and not np.any(np.signbit(logp[~active]))
    assert np.all(np.isfinite(lse))
    d = oracle.dlogits(bits, targets, active, np.ones(6), v_real, v_padded)
    assert np.all(d[~active] == 0.0)
    assert np.all(d[:, v_real:] == 0.0)
    with pytest.raises(ValueError):
        oracle.selected_logp(bits, np.array([3, 0, 100, 0, 0, 0]), active, v_real)  # t = V_real


def test_ignore_index_mode_equals_explicit_mask():
    rng = np.random.default_rng(9)
    bits = rand_bf16(rng, (5, 50))
    tgt = np.array([1, -100, 7, -100, 49])
    act_i = oracle.active_rows(tgt, None, 1, -100)
    act_e = oracle.active_rows(None, np.array([1, 0, 1, 0, 1], dtype=np.uint8), 0, -100)
    assert np.array_equal(act_i, act_e)
    a = oracle.selected_logp(bits, tgt, act_i, 50)
    b = oracle.selected_logp(bits, np.where(act_e, tgt, 12345), act_e, 50)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ----------------------------------------------------------------------------- tiled method

def test_tiled_fold_equals_plain_definition():
    rng = random.Random(13)
    nrng = np.random.default_rng(13)
    for _ in range(150):
        nt = rng.choice([1, 2, 3, 4, 7, 8, 16, 64])
        w = rng.randint(1, 40)
        v_padded = nt * w
        v_real = rng.randint(1, v_padded)
        bits = rand_bf16(nrng, (3, v_padded), scale=3.0)
        bits[:, v_real:] = garbage_bits(nrng, (3, v_padded - v_real))
        m, s = oracle.tile_partials(bits, v_real, v_padded, nt)
        for k, (c0, c1) in enumerate(oracle.tile_bounds(v_padded, nt)):
            if c0 >= v_real:  # padding-only tile: the identity, exactly
                assert np.all(m[:, k] == -np.inf) and np.all(s[:, k] == 0.0)
        lse_t = oracle.fold_partials(m, s)
        lse_p = oracle.lse_full(bits, v_real)
        np.testing.assert_allclose(lse_t, lse_p, rtol=1e-14, atol=1e-13)


def test_tile_partial_definition():
    # one tile by hand: m = max, s = sum exp(x - m)
    x = np.array([[0.5, -1.0, 2.0, 2.0, -3.0, 1.25]])
    m, s = oracle.tile_partials(bf16_bits(x), 6, 6, 2)
    assert m[0, 0] == 2.0 and m[0, 1] == 2.0
    assert abs(s[0, 0] - (math.exp(-1.5) + math.exp(-3.0) + 1.0)) < 1e-15
    assert abs(s[0, 1] - (1.0 + math.exp(-5.0) + math.exp(-0.75))) < 1e-15


def test_merge_identity_and_order():
    m, s = oracle.merge_partials(-np.inf, 0.0, 1.5, 2.0)
    assert m == 1.5 and s == 2.0
    m, s = oracle.merge_partials(1.5, 2.0, -np.inf, 0.0)
    assert m == 1.5 and s == 2.0
    m, s = oracle.merge_partials(-np.inf, 0.0, -np.inf, 0.0)
    assert m == -np.inf and s == 0.0
    m, s = oracle.merge_partials(1.0, 1.0, 3.0, 1.0)
    assert m == 3.0 and abs(s - (1.0 + math.exp(-2.0))) < 1e-15
    with pytest.raises(ValueError):
        oracle.tile_bounds(100, 7)


def test_fold_is_tp_independent_by_construction():
    # grouping tiles into shards (virtual TP) leaves the left fold unchanged
    rng = np.random.default_rng(17)
    bits = rand_bf16(rng, (4, 64 * 30))
    m, s = oracle.tile_partials(bits, 64 * 30 - 11, 64 * 30, 64)
    ref = oracle.fold_partials(m, s)
    for vtp in (1, 2, 4, 8):
        shards = np.split(np.arange(64), vtp)
        order = np.concatenate(shards)  # gathered partials, shard by shard, in global index order
        assert np.array_equal(oracle.fold_partials(m[:, order], s[:, order]), ref)


# ----------------------------------------------------------------------------- backward

def fd_grad(x, t, h=1e-6):
    """Central differences of logp = x_t - LSE(x) with respect to every x_c."""
    out = np.empty_like(x)
    for c in range(len(x)):
        xp, xm = x.copy(), x.copy()
        xp[c] += h
        xm[c] -= h
        lp = xp[t] - oracle.lse_of_values(xp[None])[0]
        lm = xm[t] - oracle.lse_of_values(xm[None])[0]
        out[c] = (lp - lm) / (2 * h)
    return out


def test_dlogits_matches_finite_differences():
    rng = np.random.default_rng(21)
    for v_real, v_padded in [(7, 8), (31, 40), (64, 64)]:
        bits = rand_bf16(rng, (2, v_padded), scale=2.0)
        targets = np.array([3, v_real - 1])
        g = np.array([0.75, -2.0])
        d = oracle.dlogits(bits, targets, np.array([True, True]), g, v_real, v_padded)
        for r in range(2):
            x = oracle.bf16_bits_to_f64(bits[r, :v_real])
            np.testing.assert_allclose(d[r, :v_real], g[r] * fd_grad(x, targets[r]), atol=1e-7)


def test_dlogits_rows_sum_to_zero_and_bounded():
    rng = np.random.default_rng(23)
    v_real, v_padded = 151936, 152576
    bits = rand_bf16(rng, (3, v_padded), scale=3.0)
    g = np.array([1.0, -0.5, 3.0])
    d = oracle.dlogits(bits, np.array([0, 77777, v_real - 1]), np.ones(3, bool), g, v_real, v_padded)
    for r in range(3):
        assert abs(math.fsum(d[r])) <= 1e-12 * abs(g[r]) * v_real
        assert np.max(np.abs(d[r])) <= abs(g[r])


# ----------------------------------------------------------------------------- lm_head

def test_lmhead_logits_brute_force():
    rng = np.random.default_rng(29)
    h = rand_bf16(rng, (3, 5), scale=1.0)
    W = rand_bf16(rng, (7, 5), scale=0.5)
    x = oracle.lmhead_logits(h, W)
    hv, Wv = oracle.bf16_bits_to_f64(h), oracle.bf16_bits_to_f64(W)
    for r in range(3):
        for c in range(7):
            want = math.fsum(float(hv[r, k]) * float(Wv[c, k]) for k in range(5))
            assert abs(x[r, c] - want) <= 1e-14 * max(1.0, abs(want))


def test_lmhead_grads_match_finite_differences():
    rng = np.random.default_rng(31)
    R, H, V, v_real = 3, 4, 9, 7
    h = rand_bf16(rng, (R, H), scale=1.0)
    W = rand_bf16(rng, (V, H), scale=0.7)
    targets = np.array([0, 6, 123])
    active = np.array([True, True, False])
    g = np.array([1.0, -0.5, 9.0])
    dh, dw = oracle.lmhead_grads(h, W, targets, active, g, v_real)
    hv, Wv = oracle.bf16_bits_to_f64(h), oracle.bf16_bits_to_f64(W)

    def loss(hh, ww):
        x = hh @ ww[:v_real].T
        lse = oracle.lse_of_values(x)
        return sum(g[r] * (x[r, targets[r]] - lse[r]) for r in range(R) if active[r])

    eps = 1e-6
    for r in range(R):
        for k in range(H):
            hp, hm = hv.copy(), hv.copy()
            hp[r, k] += eps
            hm[r, k] -= eps
            assert abs(dh[r, k] - (loss(hp, Wv) - loss(hm, Wv)) / (2 * eps)) < 1e-7
    for c in range(V):
        for k in range(H):
            wp, wm = Wv.copy(), Wv.copy()
            wp[c, k] += eps
            wm[c, k] -= eps
            assert abs(dw[c, k] - (loss(hv, wp) - loss(hv, wm)) / (2 * eps)) < 1e-7
    assert np.all(dw[v_real:] == 0.0)
    assert np.all(dh[2] == 0.0)


def _lmhead_fwd_pins_pass(fwd):
    """Pins of the lm_head forward's logp and LSE (fwd has the signature of
    oracle.lmhead_forward); True when every pin holds.

    * Uniform logits: hidden row r = a_r e_0 and every real W row = 1.5 e_0
      give x_rc = 1.5 a_r for all real c, so LSE_r = 1.5 a_r + ln V_real and
      logp_r = -ln V_real whatever the target.
    * One-hot spike: hidden row r = s_r e_1 and W = e_1 on row t* only give
      x_{r,t*} = s_r and 0 elsewhere, so logp = -log1p((V_real - 1) e^-s_r)
      for target t*, and -log(V_real - 1 + e^s_r) for any other target.
    * Padded W rows hold NaN, +inf and random bits and take no part.
    * Inactive rows give logp = +0.0 exactly; an active target in the padding
      raises ValueError.
    """
    ok = True
    H, v_real, v_padded = 8, 37, 40
    rng = np.random.default_rng(43)
    W = np.zeros((v_padded, H), dtype=np.uint16)
    W[:v_real, 0] = bf16_bits([1.5])[0]
    W[v_real:] = garbage_bits(rng, (v_padded - v_real, H))
    W[v_real, :] = 0x7FC0   # NaN
    W[v_real + 1, :] = 0x7F80  # +inf
    a = np.array([0.5, 1.0, 2.0, 3.0])
    h = np.zeros((4, H), dtype=np.uint16)
    h[:, 0] = bf16_bits(a)
    targets = np.array([0, 36, 5, 17])
    with np.errstate(all="ignore"):
        logp, lse, _ = fwd(h, W, targets, np.ones(4, dtype=bool), v_real)
        ok &= bool(np.all(np.abs(logp + LN(v_real)) < 1e-12))
        ok &= bool(np.all(np.abs(lse - (1.5 * a + LN(v_real))) < 1e-12))
        # one-hot spike
        t_star = 11
        W2 = W.copy()
        W2[:v_real] = 0
        W2[t_star, 1] = bf16_bits([1.0])[0]
        sv = np.array([4.0, 8.0, 15.0, 30.0])
        h2 = np.zeros((4, H), dtype=np.uint16)
        h2[:, 1] = bf16_bits(sv)
        t2 = np.array([t_star, t_star, 3, t_star])
        logp2, lse2, _ = fwd(h2, W2, t2, np.ones(4, dtype=bool), v_real)
        want = np.where(t2 == t_star, -np.log1p((v_real - 1) * np.exp(-sv)), -np.log(v_real - 1 + np.exp(sv)))
        ok &= bool(np.all(np.abs(logp2 - want) < 1e-12 * np.maximum(1.0, np.abs(want))))
        ok &= bool(np.all(np.abs(lse2 - np.log(v_real - 1 + np.exp(sv))) < 1e-12 * np.maximum(1.0, sv)))
        # inactive rows: exactly +0.0, their targets never used
        act = np.array([True, False, True, False])
        logp3, _, _ = fwd(h, W, np.array([0, -7, 5, 10 ** 6]), act, v_real)
        ok &= bool(np.all(logp3[~act] == 0.0) and not np.any(np.signbit(logp3[~act])))
        ok &= bool(np.all(np.abs(logp3[act] + LN(v_real)) < 1e-12))
        # an active target in the padding is an error
        try:
            fwd(h, W, np.array([0, v_real + 1, 5, 17]), np.ones(4, dtype=bool), v_real)
            ok = False
        except ValueError:
            pass
        except Exception:
            ok = False
    return ok


def test_lmhead_forward_pins():
    assert _lmhead_fwd_pins_pass(oracle.lmhead_forward)


def test_lmhead_forward_pins_catch_planted_mistakes():
    from oracle.lmhead import lmhead_logits

    def sign_flipped(hb, wb, targets, active, v_real):
        logp, lse, x = oracle.lmhead_forward(hb, wb, targets, active, v_real)
        return -logp, lse, x

    def wrong_row(hb, wb, targets, active, v_real):
        x = lmhead_logits(hb, wb, v_cols=v_real)
        lse = oracle.lse_of_values(x)
        logp = np.zeros(len(lse))
        rows = np.nonzero(np.asarray(active))[0]
        t = np.asarray(targets)[rows]
        if np.any((t < 0) | (t >= v_real)):
            raise ValueError("active target outside [0, V_real)")
        logp[rows] = x[np.roll(rows, 1), t] - lse[rows]
        return logp, lse, x

    def padding_included(hb, wb, targets, active, v_real):
        return oracle.lmhead_forward(hb, wb, targets, active, np.asarray(wb).shape[0])

    def no_range_check(hb, wb, targets, active, v_real):
        x = lmhead_logits(hb, wb)
        lse = oracle.lse_of_values(x[:, :v_real])
        logp = np.zeros(len(lse))
        rows = np.nonzero(np.asarray(active))[0]
        logp[rows] = x[rows, np.asarray(targets)[rows]] - lse[rows]
        return logp, lse, x

    for bad in (sign_flipped, wrong_row, padding_included, no_range_check):
        assert not _lmhead_fwd_pins_pass(bad), bad.__name__


# ----------------------------------------------------------------------------- pin sensitivity

def _pins_pass(lse_fn, dlogits_fn, fold_fn):
    """Run a subset of the pins against candidate functions; True when all hold."""
    ok = True
    v_real, v_padded = 151936, 152576
    rng = np.random.default_rng(1)
    row = np.full((1, v_padded), bf16_bits([1.5])[0], dtype=np.uint16)
    row[0, v_real:] = garbage_bits(rng, v_padded - v_real)
    with np.errstate(all="ignore"):
        ok &= bool(abs(lse_fn(row, v_real)[0] - (1.5 + LN(v_real))) < 1e-9)
        bits = rand_bf16(rng, (2, 40), scale=2.0)
        x = oracle.bf16_bits_to_f64(bits[0, :31])
        d = dlogits_fn(bits, np.array([3, 0]), np.array([True, True]), np.array([0.75, 1.0]), 31, 40)
        ok &= bool(np.allclose(d[0, :31], 0.75 * fd_grad(x, 3), atol=1e-6))
        b2 = rand_bf16(rng, (2, 64 * 3), scale=3.0)
        m, s = oracle.tile_partials(b2, 64 * 3 - 5, 64 * 3, 64)
        ok &= bool(np.allclose(fold_fn(m, s), oracle.lse_full(b2, 64 * 3 - 5), rtol=1e-12))
    return ok


def test_pins_catch_planted_mistakes():
    assert _pins_pass(oracle.lse_full, oracle.dlogits, oracle.fold_partials)

    def lse_includes_padding(bits, v_real):
        return oracle.lse_of_values(oracle.bf16_bits_to_f64(np.asarray(bits)))

    def lse_drops_max(bits, v_real):       # "LSE = log sum exp(x - M)" without adding M back
        x = oracle.bf16_bits_to_f64(np.asarray(bits)[:, :v_real])
        return np.log(np.exp(x - x.max(axis=1, keepdims=True)).sum(axis=1))

    def dlogits_sign_flipped(*a):
        return -oracle.dlogits(*a)

    def dlogits_onehot_shifted(bits, targets, active, g, v_real, v_padded):
        return oracle.dlogits(bits, np.minimum(np.asarray(targets) + 1, v_real - 1), active, g,
                              v_real, v_padded)

    def fold_without_rescale(m, s):        # merge that forgets the s1 * exp(m1 - m) factor
        acc_m, acc_s = np.full(m.shape[0], -np.inf), np.zeros(m.shape[0])
        for k in range(m.shape[1]):
            new_m = np.maximum(acc_m, m[:, k])
            acc_s = acc_s + np.where(m[:, k] == -np.inf, 0.0, s[:, k] * np.exp(m[:, k] - new_m))
            acc_m = new_m
        return acc_m + np.log(acc_s)

    assert not _pins_pass(lse_includes_padding, oracle.dlogits, oracle.fold_partials)
    assert not _pins_pass(lse_drops_max, oracle.dlogits, oracle.fold_partials)
    assert not _pins_pass(oracle.lse_full, dlogits_sign_flipped, oracle.fold_partials)
    assert not _pins_pass(oracle.lse_full, dlogits_onehot_shifted, oracle.fold_partials)
    assert not _pins_pass(oracle.lse_full, oracle.dlogits, fold_without_rescale)


# ------------------------------------------------------------------ entropy

def _row(vals):
    """One row of BF16 bits from values that BF16 holds exactly."""
    v = np.asarray(vals, dtype=np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)[None, :]


def _entropy_pins_pass(fn):
    """Every entropy pin, for an entropy implementation fn(bits, v_real)."""
    import math
    try:
        for v_real, c in ((1, 0.0), (7, 3.0), (151936, -2.5)):  # uniform: log V (five padded columns)
            if abs(fn(_row([c] * (v_real + 5)), v_real)[0] - np.log(v_real)) > 1e-9 * max(1.0, np.log(v_real)):
                return False
        V = 1000
        for a in (1.0, 4.0, 16.0):  # one column at a, V-1 at 0: H = log Z - a e^a / Z
            vals = np.zeros(V, dtype=np.float32)
            vals[17] = a
            Z = np.exp(a) + (V - 1)
            if abs(fn(_row(vals), V)[0] - (np.log(Z) - a * np.exp(a) / Z)) > 1e-9:
                return False
        rng = np.random.default_rng(5)
        for V in (1, 2, 3, 9):  # direct summation
            vals = rng.integers(-12, 12, size=V).astype(np.float32) / 4.0
            ex = [math.exp(float(v)) for v in vals]
            Z = sum(ex)
            if abs(fn(_row(vals), V)[0] + sum((e / Z) * math.log(e / Z) for e in ex)) > 1e-12:
                return False
        # shift and permutation invariance, 0 <= H <= log V; values k/4 with |k| <= 64 need at
        # most 7 significant bits, also after +8: exact in BF16
        rng = np.random.default_rng(6)
        x = (rng.integers(-64, 65, size=(4, 333)) / 4.0).astype(np.float32)
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)
        h = fn(bits, 333)
        shifted = ((x + np.float32(8.0)).view(np.uint32) >> 16).astype(np.uint16)
        if not np.allclose(fn(shifted, 333), h, atol=1e-9, rtol=0):
            return False
        if not np.allclose(fn(bits[:, rng.permutation(333)], 333), h, atol=1e-12, rtol=0):
            return False
        return bool(np.all(h >= 0) and np.all(h <= np.log(333) + 1e-12))
    except (ValueError, FloatingPointError):
        return False


def test_entropy_pins():
    assert _entropy_pins_pass(oracle.entropy)


def test_entropy_pins_catch_planted_mistakes():
    def with_padding(bits, v_real):
        return oracle.entropy(bits, np.asarray(bits).shape[1])

    def sign_flipped(bits, v_real):
        return -oracle.entropy(bits, v_real)

    def log2_based(bits, v_real):
        return oracle.entropy(bits, v_real) / np.log(2.0)

    def unnormalised(bits, v_real):         # p = exp(x - max) instead of exp(x - LSE)
        x = oracle.bf16_bits_to_f64(np.asarray(bits)[:, :v_real])
        q = np.exp(x - x.max(axis=1, keepdims=True))
        with np.errstate(divide="ignore", invalid="ignore"):
            return np.where(q > 0, -q * np.log(q), 0.0).sum(axis=1)

    for mistake in (with_padding, sign_flipped, log2_based, unnormalised):
        assert not _entropy_pins_pass(mistake), mistake.__name__


def test_entropy_special_rows():
    ninf = np.float32(-np.inf)
    bits = np.concatenate([_row([ninf, ninf, 0.0, ninf]), _row([ninf] * 4), _row([np.nan, 0, 0, 0])])
    h = oracle.entropy(bits, 4)
    assert h[0] == 0.0  # a single finite column: a point mass
    assert np.isnan(h[1]) and np.isnan(h[2])


# ------------------------------------------------------------------ GRPO loss

def _grpo_pins_pass(fn):
    """Every GRPO-loss pin, for an implementation fn(logp, adv, active, ref, beta) -> (loss, g, n)."""
    rng = np.random.default_rng(31)
    T = 50
    logp = -rng.random(T) * 5
    adv = rng.standard_normal(T)
    act = rng.random(T) < 0.6
    # closed form without KL: minus the mean of A * logp over active tokens
    loss, g, n = fn(logp, adv, act, None, 0.0)
    if n != act.sum() or abs(loss + (adv * logp)[act].mean()) > 1e-12:
        return False
    if not np.allclose(g, np.where(act, -adv / act.sum(), 0.0), rtol=0, atol=1e-15):
        return False
    # KL term: zero where ref == logp, non-negative, and the gradient is the derivative
    if abs(fn(logp, adv, act, logp, 0.3)[0] - loss) > 1e-12:
        return False
    ref = logp + rng.standard_normal(T) * 0.5
    l0 = fn(logp, np.zeros(T), act, ref, 0.3)[0]
    if l0 < 0:
        return False
    loss_k, g_k, _ = fn(logp, adv, act, ref, 0.3)
    h = 1e-6
    for r in np.nonzero(act)[0][:5]:
        e = np.zeros(T)
        e[r] = h
        fd = (fn(logp + e, adv, act, ref, 0.3)[0] - fn(logp - e, adv, act, ref, 0.3)[0]) / (2 * h)
        if abs(fd - g_k[r]) > 1e-7:
            return False
    if np.any(g_k[~act] != 0):
        return False
    # no active token: loss and gradients 0
    l_empty, g_empty, n_empty = fn(logp, adv, np.zeros(T, dtype=bool), ref, 0.3)
    return l_empty == 0.0 and n_empty == 0 and not g_empty.any()


def test_grpo_loss_pins():
    assert _grpo_pins_pass(oracle.grpo_loss)


def test_grpo_pins_catch_planted_mistakes():
    def sequence_mean(logp, adv, act, ref=None, beta=0.0):  # divides by T, not the active count
        loss, g, n = oracle.grpo_loss(logp, adv, act, ref, beta)
        return loss * n / len(logp), g * n / len(logp), n

    def kl_sign(logp, adv, act, ref=None, beta=0.0):
        return oracle.grpo_loss(logp, adv, act, ref, -beta)

    def grad_sign(logp, adv, act, ref=None, beta=0.0):
        loss, g, n = oracle.grpo_loss(logp, adv, act, ref, beta)
        return loss, -g, n

    for mistake in (sequence_mean, kl_sign, grad_sign):
        assert not _grpo_pins_pass(mistake), mistake.__name__
