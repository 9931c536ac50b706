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
