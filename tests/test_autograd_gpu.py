"""The torch.autograd entry point (SelectedTokenLogprob): its forward is
rlk_logp_fwd and its backward rlk_logp_bwd with the saved LSE, bit for bit,
and the gradient of a scalar loss of logp matches the FP64 oracle."""
import numpy as np
import pytest
import torch

import synth
import vocab_selected_token_tile_gb300 as rlk
from parity import check_dlogits, check_fwd, contract, to_dev
from vocab_selected_token_tile_gb300.autograd import selected_logprob

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - the CPU suite deselects this module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.mark.parametrize("explicit", [True, False], ids=["mask", "ignore_index"])
@pytest.mark.parametrize("vtp", [1, 2, 8])
def test_autograd_matches_the_c_entry_points(explicit, vtp):
    T, v_real, v_padded, nt, stride = 48, 5003, 5120, 64, 5128
    bits = synth.logits_host(0, T, stride, v_padded, v_real, seed=17, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, v_real, 17, ignore_frac=0.0 if explicit else 0.25)
    mask = (np.random.default_rng(17).random(T) < 0.7).astype(np.uint8) if explicit else None
    active = mask != 0 if explicit else tgt != -100
    w = np.random.default_rng(18).standard_normal(T).astype(np.float32)

    x16 = to_dev(bits)
    x = x16.view(torch.bfloat16).clone().requires_grad_(True)
    dt = torch.from_numpy(tgt).cuda()
    dm = torch.from_numpy(mask).cuda() if explicit else None
    logp, lse = selected_logprob(x, dt, dm, v_real=v_real, v_padded=v_padded, num_tiles=nt, virtual_tp=vtp)
    assert not lse.requires_grad and logp.requires_grad
    (logp * torch.from_numpy(w).cuda()).sum().backward()
    torch.cuda.synchronize()

    c = contract(T, v_real, v_padded, nt, vtp, rlk.MASK_EXPLICIT if explicit else rlk.MASK_IGNORE_INDEX,
                 stride=stride)
    ref_logp, ref_lse = rlk.logp_fwd(c, x16, dt, dm)
    ref_dl = rlk.logp_bwd(c, x16, dt, dm, ref_lse, torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert torch.equal(logp.detach().view(torch.int32), ref_logp.view(torch.int32))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    grad_bits = x.grad.view(torch.int16)
    assert torch.equal(grad_bits[:, :v_padded], ref_dl[:, :v_padded])
    assert not grad_bits[:, v_padded:].any()  # columns past V_padded: exactly zero

    check_fwd(bits, tgt, active, v_real, logp.detach().cpu().numpy(), lse.cpu().numpy())
    check_dlogits(bits, tgt, active, np.where(active, w, 0).astype(np.float32), v_real, v_padded,
                  grad_bits.cpu().numpy().view(np.uint16))


def test_lmhead_autograd_matches_the_c_entry_points_and_the_oracle():
    """FusedLmHeadLogprob: forward = rlk_logp_fused_lmhead, backward = rlk_logp_fused_lmhead_bwd from
    the saved LSE; the gradients of sum(w * logp) are bitwise those of the fused call with
    grad_logp = w, and within the BF16 bound of the FP64 oracle's."""
    import oracle
    from vocab_selected_token_tile_gb300.autograd import lmhead_logprob
    T, H, v_real, v_padded, nt = 130, 128, 600, 608, 2
    hb = synth.normal_bf16_host(0, T, H, 41, synth.STREAM_HIDDEN, 1.0)
    wb = synth.normal_bf16_host(0, v_padded, H, 41, synth.STREAM_WEIGHT, 0.2)
    tgt = synth.targets(T, v_real, seed=41)
    mask = (np.arange(T) % 5 != 0).astype(np.uint8)
    w = np.random.default_rng(41).standard_normal(T).astype(np.float32)
    h = torch.from_numpy(hb.view(np.int16)).cuda().view(torch.bfloat16).requires_grad_(True)
    W = torch.from_numpy(wb.view(np.int16)).cuda().view(torch.bfloat16).requires_grad_(True)
    dt, dm = torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda()
    logp, lse = lmhead_logprob(h, W, dt, dm, v_real=v_real, num_tiles=nt)
    (logp * torch.from_numpy(w).cuda()).sum().backward()
    torch.cuda.synchronize()
    c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=1)
    ref = rlk.logp_fused_lmhead(c, h.detach(), W.detach(), dt, dm,
                                grad=torch.from_numpy(np.where(mask != 0, w, 0).astype(np.float32)).cuda())
    torch.cuda.synchronize()
    assert torch.equal(logp.detach(), ref[0]) and torch.equal(lse, ref[1])
    assert torch.equal(h.grad, ref[2]) and torch.equal(W.grad, ref[3])
    from oracle.lmhead import lmhead_dlogits
    act = mask != 0
    gw = np.where(act, w, 0.0)
    ref_logp, ref_lse, x = oracle.lmhead_forward(hb, wb, tgt, act, v_real)
    assert np.max(np.abs(logp.detach().cpu().numpy() - ref_logp)) <= 1e-4
    dh_ref, dw_ref = oracle.lmhead_grads(hb, wb, tgt, act, gw, v_real)
    # BF16 dlogits (one rounding) summed in FP32, then one BF16 rounding of the result:
    # |err| <= 2^-8 (|ref| + sum |dlogits| |operand|)
    d = np.abs(lmhead_dlogits(x, ref_lse, tgt, act, gw))
    sc_dh = d @ np.abs(oracle.bf16_bits_to_f64(wb[:v_real]))
    sc_dw = d.T @ np.abs(oracle.bf16_bits_to_f64(hb))
    got_dh = h.grad.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got_dh - dh_ref) <= 2.0 ** -8 * (np.abs(dh_ref) + sc_dh) + 1e-30)
    got_dw = W.grad.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got_dw[:v_real] - dw_ref[:v_real]) <= 2.0 ** -8 * (np.abs(dw_ref[:v_real]) + sc_dw) + 1e-30)
    assert np.all(got_dw[v_real:] == 0.0)


def test_lmhead_autograd_keep_logits_is_bitwise_the_recompute_path():
    """keep_logits=True (the forward keeps its FP32 logits, the backward forms dlogits from them) gives
    bitwise the logp, LSE and gradients of keep_logits=False (the backward re-runs the GEMM)."""
    from vocab_selected_token_tile_gb300.autograd import lmhead_logprob
    T, H, v_real, v_padded, nt = 259, 192, 1000, 1024, 4
    hb = synth.normal_bf16_host(0, T, H, 43, synth.STREAM_HIDDEN, 1.0)
    wb = synth.normal_bf16_host(0, v_padded, H, 43, synth.STREAM_WEIGHT, 0.3)
    tgt = synth.targets(T, v_real, seed=43, ignore_frac=0.25)
    w = torch.from_numpy(np.random.default_rng(43).standard_normal(T).astype(np.float32)).cuda()
    dt = torch.from_numpy(tgt).cuda()
    out = []
    for keep in (False, True):
        h = torch.from_numpy(hb.view(np.int16)).cuda().view(torch.bfloat16).requires_grad_(True)
        W = torch.from_numpy(wb.view(np.int16)).cuda().view(torch.bfloat16).requires_grad_(True)
        logp, lse = lmhead_logprob(h, W, dt, None, v_real=v_real, num_tiles=nt, keep_logits=keep)
        (logp * w).sum().backward()
        torch.cuda.synchronize()
        out.append((logp.detach(), lse, h.grad, W.grad))
    for a, b in zip(*out):
        assert torch.equal(a, b)
