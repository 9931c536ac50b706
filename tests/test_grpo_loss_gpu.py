"""Parity of the GRPO loss reduction (rlk_grpo_loss) with the FP64 oracle, on the GPU.

The loss is the token mean of -A_r logp_r (+ beta k3_r with a reference
logp) over the active rows; g_r its derivative in logp_r.  The kernel forms
each token's term in FP32 (the inputs' precision) and sums in FP64, so the
tolerances are a few FP32 roundings of each term: for the loss,
8 * 2^-24 * mean |term| plus one rounding of the result; for g, 8 * 2^-24 *
(|A_r| + beta (1 + e^(ref_r - logp_r))) / N.  N is exact; inactive rows get
g = +0.0 exactly; the loss is bitwise reproducible.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import vocab_selected_token_tile_gb300 as rlk
from parity import check_dlogits, check_fwd, contract, to_dev

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - the CPU suite deselects this module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

EPS32 = 2.0 ** -24


def grpo_batch(batch, seq, prompt, len_min, len_max, seed):
    """A GRPO batch: response masks after a prompt, one advantage per sequence
    broadcast over its tokens, logp in (-12, 0], a reference logp near it."""
    mask, _ = synth.response_mask(batch, seq, prompt, len_min, len_max, seed)
    rng = np.random.default_rng(seed)
    adv = np.repeat(rng.standard_normal(batch), seq).astype(np.float32)
    logp = (-12.0 * rng.random(batch * seq) ** 2).astype(np.float32)
    ref = (logp + 0.05 * rng.standard_normal(batch * seq)).astype(np.float32)
    return logp, adv, mask, ref


def run(logp, adv, mask, ref, beta):
    d = [torch.from_numpy(x).cuda() for x in (logp, adv, mask)]
    r = torch.from_numpy(ref).cuda() if ref is not None else None
    loss, g, n = rlk.grpo_loss(d[0], d[1], d[2], r, beta)
    torch.cuda.synchronize()
    return float(loss.item()), g.cpu().numpy(), float(n.item())


def check(logp, adv, mask, ref, beta):
    loss, g, n = run(logp, adv, mask, ref, beta)
    ol, og, on = oracle.grpo_loss(logp, adv, mask != 0, ref, beta)
    assert n == on
    act = mask != 0
    if on == 0:
        assert loss == 0.0 and np.array_equal(g, np.zeros_like(g))
        return loss, g
    lp, a = logp.astype(np.float64), adv.astype(np.float64)
    e = np.exp(ref.astype(np.float64) - lp) if ref is not None else np.zeros_like(lp)
    kl = beta * np.abs(e - (ref - lp) - 1.0) if ref is not None else 0.0
    mean_abs = float(np.sum((np.abs(a * lp) + kl)[act])) / on
    assert abs(loss - ol) <= 8 * EPS32 * mean_abs + 2 * EPS32 * abs(ol), (loss, ol)
    gtol = 8 * EPS32 * (np.abs(a) + beta * (1.0 + e)) / on
    assert np.all(np.abs(g - og) <= gtol)
    assert np.all(g[~act].view(np.uint32) == 0)  # +0.0 exactly
    return loss, g


@pytest.mark.parametrize("beta", [0.0, 0.01, 0.5])
@pytest.mark.parametrize("shape", [(2, 16, 8, 8, 8), (4, 1024, 128, 16, 896), (32, 2048, 256, 64, 1792)],
                         ids=["tiny", "qwen3", "grpo"])
def test_grpo_loss_matches_oracle(shape, beta):
    logp, adv, mask, ref = grpo_batch(*shape, seed=7)
    check(logp, adv, mask, ref if beta else None, beta)
    if beta == 0.0:
        check(logp, adv, mask, ref, 0.0)  # a reference with beta 0 adds nothing


def test_grpo_loss_edge_cases_and_repeatability():
    logp, adv, mask, ref = grpo_batch(3, 3000, 10, 1, 2990, seed=3)
    check(logp, adv, np.zeros_like(mask), ref, 0.01)           # N = 0
    one = np.zeros_like(mask)
    one[1234] = 1
    check(logp, adv, one, ref, 0.01)                           # N = 1
    check(logp, adv, np.ones_like(mask), ref, 0.01)            # every row active
    for T in (1, 1023, 1024, 1025, 8191, 8193):                # around a CTA's and the cluster's stride
        check(logp[:T], adv[:T], np.ones(T, np.uint8), ref[:T], 0.01)
    check(*grpo_batch(3, 33337, 100, 1, 33000, seed=5), 0.01)  # several unrolled passes, ragged end
    loss, g, n = run(logp[:0], adv[:0], mask[:0], ref[:0], 0.01)  # T = 0
    assert loss == 0.0 and n == 0.0 and g.size == 0
    a = run(logp, adv, mask, ref, 0.01)
    b = run(logp, adv, mask, ref, 0.01)
    assert np.float32(a[0]).view(np.uint32) == np.float32(b[0]).view(np.uint32)
    assert np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))
    with pytest.raises(rlk.RlkError):
        run(logp, adv, mask, ref, -1.0)


def test_grpo_step_logits_to_dlogits():
    """The whole step on one batch: logits -> logp (forward) -> loss and g
    (rlk_grpo_loss) -> dlogits (backward with that g), against the oracle's
    chain in FP64."""
    T, v_real, v_padded, nt = 48, 5003, 5120, 64
    stride = v_padded
    bits = synth.logits_host(0, T, stride, v_padded, v_real, seed=11, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, v_real, 11)
    mask, _ = synth.response_mask(3, 16, 4, 2, 12, 11)
    adv = np.repeat(np.random.default_rng(11).standard_normal(3), 16).astype(np.float32)
    c = contract(T, v_real, v_padded, nt, 2, rlk.MASK_EXPLICIT, stride=stride)
    d, dt, dm = to_dev(bits), torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda()
    logp, lse = rlk.logp_fwd(c, d, dt, dm)
    ref = (logp + 0.05 * torch.randn(T, device="cuda", generator=torch.Generator("cuda").manual_seed(11)))
    loss, g, n = rlk.grpo_loss(logp, torch.from_numpy(adv).cuda(), dm, ref, 0.01)
    dl, _, _ = rlk.logp_fwd_bwd(c, d, dt, dm, g)
    torch.cuda.synchronize()

    act = mask != 0
    check_fwd(bits, tgt, act, v_real, logp.cpu().numpy(), lse.cpu().numpy())
    o_logp, _ = oracle.selected_logp(bits, tgt, act, v_real)
    ol, og, on = oracle.grpo_loss(o_logp, adv, act, ref.cpu().numpy(), 0.01)
    assert n.item() == on
    assert abs(loss.item() - ol) <= 1e-5 * max(1.0, abs(ol))
    check_dlogits(bits, tgt, act, og, v_real, v_padded, dl.cpu().numpy().view(np.uint16))
