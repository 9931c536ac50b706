"""The GRPO step in one pass over the logits (rlk_grpo_fused_step), on the GPU.

Composed from the other calls the step is rlk_logp_fwd -> rlk_grpo_loss ->
rlk_logp_bwd with lse_in, reading the logits twice.  The fused step forms each
row's g on chip from the row's logp with the GRPO loss kernel's own FP32
operations, so its loss, g, logp, LSE and dlogits must be bitwise those of the
composition -- with and without the KL term, in both mask modes, at every
virtual TP and CTA count, in place or not.  One case is also checked directly
against the FP64 oracle: g against oracle.grpo_loss of the step's logp (a few
FP32 roundings), dlogits against oracle.dlogits with the step's g (one BF16
rounding).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import vocab_selected_token_tile_gb300 as rlk
from parity import check_dlogits, check_fwd, contract, sha, to_dev

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - the CPU suite deselects this module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

EPS32 = 2.0 ** -24


def inputs(T, vr, vp, nt, seed, mode):
    bits = synth.logits_host(0, T, vp, vp, vr, seed=seed, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, vr, seed, ignore_frac=0.3 if mode == rlk.MASK_IGNORE_INDEX else 0.0)
    rng = np.random.default_rng(seed)
    if mode == rlk.MASK_EXPLICIT:
        mask = (rng.random(T) < 0.6).astype(np.uint8)
        mask[0] = 1
        tgt = np.where(mask != 0, tgt, -7)  # never read as an index
    else:
        mask = (tgt != -100).astype(np.uint8)
    adv = rng.standard_normal(T).astype(np.float32)
    ref = (-4.0 * rng.random(T)).astype(np.float32)
    return bits, tgt, mask, adv, ref


def composition(c, logits, dt, dm, mask_u8, dadv, dref, beta):
    logp, lse = rlk.logp_fwd(c, logits, dt, dm)
    loss, g, n = rlk.grpo_loss(logp, dadv, mask_u8, dref, beta)
    dl = rlk.logp_bwd(c, logits, dt, dm, lse, g)
    return dict(logp=logp, lse=lse, grad=g, loss=loss, active_count=n, dlogits=dl)


def assert_same(got, want, vp, where):
    for k in ("logp", "lse", "grad", "loss", "active_count"):
        assert torch.equal(got[k], want[k]), (k, where)
    assert torch.equal(got["dlogits"][:, :vp], want["dlogits"][:, :vp]), ("dlogits", where)


CASES = [
    (5, 37, 40, 4),           # unaligned tiles, ragged real end
    (33, 1000, 1024, 64),     # padding-only tiles
    (40, 151936, 151936, 64),  # 2374-column tiles
    (64, 16383, 16384, 8),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T%d_V%d_P%d_NT%d" % c)
@pytest.mark.parametrize("mode", [rlk.MASK_EXPLICIT, rlk.MASK_IGNORE_INDEX], ids=["explicit", "ignore"])
@pytest.mark.parametrize("beta", [0.0, 0.01])
def test_fused_step_is_bitwise_the_composition(case, mode, beta):
    T, vr, vp, nt = case
    bits, tgt, mask, adv, ref = inputs(T, vr, vp, nt, seed=T + nt, mode=mode)
    logits = to_dev(bits)
    dt, dm_u8, dadv = (torch.from_numpy(a).cuda() for a in (tgt, mask, adv))
    dm = dm_u8 if mode == rlk.MASK_EXPLICIT else None
    dref = torch.from_numpy(ref).cuda() if beta else None
    for vtp in (v for v in (1, 2, 4, 8) if nt % v == 0):
        c = contract(T, vr, vp, nt, vtp, mode)
        want = composition(c, logits, dt, dm, dm_u8, dadv, dref, beta)
        got = rlk.grpo_fused_step(c, logits, dt, dm, dadv, dref, beta)
        torch.cuda.synchronize()
        assert_same(got, want, vp, (vtp, "out of place"))
        buf = logits.clone()
        got = rlk.grpo_fused_step(c, buf, dt, dm, dadv, dref, beta, dlogits=buf)
        torch.cuda.synchronize()
        assert_same(got, want, vp, (vtp, "in place"))


@pytest.mark.parametrize("near", [True, False], ids=["ref_near_logp", "ref_far"])
def test_fused_step_against_the_oracle(near):
    """g against oracle.grpo_loss of the step's own logp, dlogits against oracle.dlogits with the step's g.
    The FP32 difference d = ref - logp rounds by |d| 2^-24, which exp turns into a relative error of e^d, so
    the bound on g carries a |d| term (large here when ref is far from logp: |d| up to ~30, g up to ~1e7)."""
    T, vr, vp, nt, beta = 48, 3001, 3072, 64, 0.01
    bits, tgt, mask, adv, ref = inputs(T, vr, vp, nt, seed=11, mode=rlk.MASK_EXPLICIT)
    c = contract(T, vr, vp, nt, 2, rlk.MASK_EXPLICIT)
    logits = to_dev(bits)
    dt, dm, dadv = (torch.from_numpy(a).cuda() for a in (tgt, mask, adv))
    if near:  # a reference policy close to this one: its logp within a few hundredths
        lp0, _ = rlk.logp_fwd(c, logits, dt, dm)
        ref = (lp0.cpu().numpy() + 0.05 * np.random.default_rng(3).standard_normal(T)).astype(np.float32)
    got = rlk.grpo_fused_step(c, logits, dt, dm, dadv, torch.from_numpy(ref).cuda(), beta)
    torch.cuda.synchronize()
    act = mask != 0
    logp, lse = got["logp"].cpu().numpy(), got["lse"].cpu().numpy()
    check_fwd(bits, tgt, act, vr, logp, lse)
    ol, og, on = oracle.grpo_loss(logp, adv, act, ref, beta)
    g = got["grad"].cpu().numpy()
    assert float(got["active_count"].item()) == on
    d = np.abs(ref.astype(np.float64) - logp)
    e = np.exp(ref.astype(np.float64) - logp)
    assert np.all(np.abs(g - og) <= 8 * EPS32 * (np.abs(adv) + beta * (1.0 + e * (1.0 + d))) / on)
    assert np.all(g[~act].view(np.uint32) == 0)
    terms = np.abs(adv * logp) + beta * e * (1.0 + d)
    assert abs(float(got["loss"].item()) - ol) <= 8 * EPS32 * float(terms[act].sum()) / on + 2 * EPS32 * abs(ol)
    if near:  # (far from ref, g reaches ~1e7 and dlogits with it: the 1e-2 absolute bar assumes g of order 1)
        check_dlogits(bits, tgt, act, g, vr, vp, got["dlogits"].cpu().numpy().view(np.uint16))


def test_fused_step_qwen3_shape_all_virtual_tp(monkeypatch):
    """4096 rows: many rows per CTA, the skewed order wraps the ring; bitwise the composition at one and two
    CTAs per SM and every virtual TP, and the entropy bitwise rlk_logp_fwd_entropy's."""
    from synth import workloads as W
    w = W.QWEN3
    bits = W.logits_host(w)
    tgt = W.targets(w)
    mask = (tgt != w.ignore_index).astype(np.uint8)
    rng = np.random.default_rng(5)
    adv = np.repeat(rng.standard_normal(4), w.T // 4).astype(np.float32)
    ref = (-6.0 * rng.random(w.T)).astype(np.float32)
    logits = to_dev(bits)
    dt, dm_u8, dadv, dref = (torch.from_numpy(a).cuda() for a in (tgt, mask, adv, ref))
    c2 = contract(w.T, w.v_real, w.v_padded, w.num_tiles, 2, rlk.MASK_IGNORE_INDEX)
    want = composition(c2, logits, dt, None, dm_u8, dadv, dref, 0.01)
    _, _, ent = rlk.logp_fwd_entropy(c2, logits, dt)
    torch.cuda.synchronize()
    for per_sm in ("1", "2"):
        monkeypatch.setenv("RLK_CTAS_PER_SM", per_sm)
        for vtp in (1, 2, 4, 8):
            c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, vtp, rlk.MASK_IGNORE_INDEX)
            got = rlk.grpo_fused_step(c, logits, dt, None, dadv, dref, 0.01, entropy=True)
            torch.cuda.synchronize()
            assert_same(got, want, w.v_padded, (per_sm, vtp))
            assert sha(got["entropy"]) == sha(ent), (per_sm, vtp)
    monkeypatch.setenv("RLK_FUSED_SCHEDULE", "resident")
    with pytest.raises(rlk.RlkError) as ei:
        rlk.grpo_fused_step(c2, logits, dt, None, dadv, dref, 0.01)
    assert ei.value.status == rlk.RLK_ERR_UNSUPPORTED


def test_fused_step_degenerate_batches():
    """No active row (N = 0: loss 0, g and dlogits all +0.0), one active row, and an empty batch."""
    T, vr, vp, nt = 24, 1000, 1024, 8
    bits, _, _, adv, ref = inputs(T, vr, vp, nt, seed=2, mode=rlk.MASK_EXPLICIT)
    tgt = synth.targets(T, vr, 2)  # every row's target valid: any row may be the active one
    logits = to_dev(bits)
    dt, dadv, dref = (torch.from_numpy(a).cuda() for a in (tgt, adv, ref))
    c = contract(T, vr, vp, nt, 2, rlk.MASK_EXPLICIT)
    for m in (np.zeros(T, np.uint8), np.eye(1, T, 7, dtype=np.uint8)[0]):
        dm = torch.from_numpy(m).cuda()
        got = rlk.grpo_fused_step(c, logits, dt, dm, dadv, dref, 0.01)
        want = composition(c, logits, dt, dm, dm, dadv, dref, 0.01)
        torch.cuda.synchronize()
        assert_same(got, want, vp, int(m.sum()))
        if m.sum() == 0:
            assert float(got["loss"].item()) == 0.0 and float(got["active_count"].item()) == 0.0
            assert (got["grad"].view(torch.int32) == 0).all() and (got["dlogits"][:, :vp] == 0).all()
    z = contract(0, vr, vp, nt, 2, rlk.MASK_EXPLICIT)
    loss = torch.full((1,), 7.0, device="cuda")
    n = torch.full((1,), 7.0, device="cuda")
    rlk.check(rlk.rlk_grpo_fused_step(z, None, None, None, None, None, 0.01, None, None, None, None, None,
                                      loss.data_ptr(), n.data_ptr(), None, None))
    torch.cuda.synchronize()
    assert float(loss.item()) == 0.0 and float(n.item()) == 0.0
