"""Host-side contract checks against the rules the header states, on random contracts.

rlk_logp_check_contract, rlk_logp_check_shard_contract and
rlk_logp_lmhead_workspace_size touch no device.  Each seeded case draws every
field from values around the rules' edges and checks the documented meaning
without assuming an order among the rules: the contract is accepted exactly
when it breaks none of them, and a rejected one returns the code of one of the
rules it breaks.
"""
import numpy as np
import pytest

import vocab_selected_token_tile_gb300 as rlk

OK, INVALID, UNSUPPORTED, NON_TILEABLE, MISALIGNED = (rlk.RLK_OK, rlk.RLK_ERR_INVALID_ARG, rlk.RLK_ERR_UNSUPPORTED,
                                                      rlk.RLK_ERR_NON_TILEABLE, rlk.RLK_ERR_MISALIGNED)


@pytest.fixture(scope="module", autouse=True)
def _library():
    try:
        rlk.library()
    except Exception as e:  # pragma: no cover - build() makes it
        pytest.skip(f"library not built: {e}")


def broken_rules(c):
    """Codes of the rules the contract breaks, as the header states them (a rule that needs an
    earlier one to hold, divisibility by num_tiles say, is only judged when that one holds)."""
    out = set()
    if c.T < 0:
        out.add(INVALID)
    if c.T > 1 << 40:
        out.add(UNSUPPORTED)
    if c.V_real < 1:
        out.add(INVALID)
    if c.V_padded < c.V_real:
        out.add(INVALID)
    if c.V_padded > 1 << 31:
        out.add(UNSUPPORTED)
    tiles_ok = c.num_tiles >= 1
    if not tiles_ok:
        out.add(INVALID)
    if c.num_tiles > 1024:
        out.add(UNSUPPORTED)
    divides = tiles_ok and c.V_padded % c.num_tiles == 0
    if tiles_ok and not divides:
        out.add(NON_TILEABLE)
    vtp_ok = c.virtual_tp in (1, 2, 4, 8)
    if not vtp_ok:
        out.add(UNSUPPORTED)
    if tiles_ok and vtp_ok and c.num_tiles % c.virtual_tp != 0:
        out.add(NON_TILEABLE)
    if divides and c.V_padded // c.num_tiles > 16384:
        out.add(UNSUPPORTED)
    stride = c.row_stride if c.row_stride else c.V_padded
    if stride < c.V_padded:
        out.add(INVALID)
    if stride % 8 != 0:
        out.add(MISALIGNED)
    if c.mask_mode not in (rlk.MASK_EXPLICIT, rlk.MASK_IGNORE_INDEX):
        out.add(INVALID)
    if c.validate not in (0, 1):
        out.add(INVALID)
    if c.wait_timeout_ns < 0:
        out.add(INVALID)
    return out


def draw(rng):
    pick = lambda *xs: xs[int(rng.integers(len(xs)))]  # noqa: E731
    nt = int(pick(-1, 0, 1, 2, 3, 7, 8, 64, 1000, 1024, 1025, 2048))
    w = int(pick(1, 5, 8, 16, 2384, 16383, 16384, 16385, 40000))
    vp = int(pick(nt * w, nt * w + 1, nt * w - 1, 152576, 1 << 31, (1 << 31) + 64, 0))
    vr = int(pick(vp, vp - 1, max(vp - 640, -3), 1, 0, vp + 1))
    stride = int(pick(0, 0, vp, vp + 8, vp + 3, (vp + 7) // 8 * 8, vp - 8, 16))
    return rlk.Contract(T=int(pick(0, 1, 65536, -1, (1 << 40) + 1)), V_real=vr, V_padded=vp, row_stride=stride,
                        num_tiles=nt, virtual_tp=int(pick(1, 2, 4, 8, 3, 16, 0)),
                        mask_mode=int(pick(0, 1, 2, -1)), validate=int(pick(0, 1, 2)),
                        ignore_index=-100, wait_timeout_ns=int(pick(0, 1000, -5)))


def test_check_contract_matches_the_stated_rules():
    rng = np.random.default_rng(2024)
    seen = {OK: 0, INVALID: 0, UNSUPPORTED: 0, NON_TILEABLE: 0, MISALIGNED: 0}
    for _ in range(20000):
        c = draw(rng)
        broken = broken_rules(c)
        st = rlk.rlk_logp_check_contract(c)
        if broken:
            assert st in broken, (st, broken, c.__dict__ if hasattr(c, "__dict__") else repr(c))
        else:
            assert st == OK, (st, repr(c))
        seen[st] = seen.get(st, 0) + 1
    # every outcome occurred, so the draw reaches each rule
    assert all(v > 0 for v in seen.values()), seen


def test_shard_contract_matches_the_stated_rules():
    """A shard contract is the whole problem's with row_stride that of the shard's buffer (0 -> Vs):
    valid as a whole (row_stride aside), 0 <= shard < virtual_tp, Vs = V_padded/virtual_tp a multiple
    of 8, the stride >= Vs and a multiple of 8."""
    rng = np.random.default_rng(7)
    outcomes = set()
    for _ in range(20000):
        c = draw(rng)
        shard = int(rng.choice([-1, 0, 1, 3, 7, 8]))
        whole = c.replace(row_stride=0)
        broken = broken_rules(whole)
        if not broken:
            if not 0 <= shard < c.virtual_tp:
                broken.add(INVALID)
            vs = c.V_padded // c.virtual_tp
            if vs % 8 != 0:
                broken.add(MISALIGNED)
            stride = c.row_stride if c.row_stride else vs
            if stride < vs:
                broken.add(INVALID)
            if stride % 8 != 0:
                broken.add(MISALIGNED)
        st = rlk.rlk_logp_check_shard_contract(c, shard)
        if broken:
            assert st in broken, (st, broken, shard, repr(c))
        else:
            assert st == OK, (st, shard, repr(c))
        outcomes.add(st)
    assert {OK, INVALID, MISALIGNED} <= outcomes


def test_lmhead_workspace_size_is_zero_exactly_for_unsupported_shapes():
    """0 for a contract that fails its check, H not a positive multiple of 64 or above 2^20, a tile
    width not a multiple of 16, or T above 2^31 - 128; otherwise at least the BF16 dlogits and FP32
    logits of the backward (T * V_padded * 6 bytes)."""
    rng = np.random.default_rng(11)
    nonzero = 0
    for _ in range(5000):
        c = draw(rng)
        H = int(rng.choice([0, 32, 64, 100, 128, 4096, 4160, (1 << 20), (1 << 20) + 64, -64]))
        bad = bool(broken_rules(c)) or H < 64 or H % 64 != 0 or H > 1 << 20
        if not broken_rules(c):
            bad = bad or (c.V_padded // c.num_tiles) % 16 != 0 or c.T > (1 << 31) - 128
        n = rlk.rlk_logp_lmhead_workspace_size(c, H)
        if bad:
            assert n == 0, (H, repr(c))
        else:
            assert n >= c.T * c.V_padded * 6, (n, H, repr(c))
            nonzero += 1
    assert nonzero > 0
