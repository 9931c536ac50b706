"""The Python binding refuses tensors that cannot hold what a call touches, before any launch.

The C entry points check pointers, alignment and the device, but only the
caller knows how large each buffer is; the binding compares every tensor's
storage (from its first element) with the bytes the call reads or writes,
its dtype and its device.  Each case below raises before the library is
called, so no kernel ever sees the short buffer.  A shard read in place
from the whole row buffer (a strided view) passes, and shard_bwd then
allocates its dlogits with the shard's row stride.
"""
import numpy as np
import pytest
import torch

import synth
import vocab_selected_token_tile_gb300 as rlk
from parity import contract, to_dev

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - the CPU suite deselects this module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

T, VR, VP, NT = 33, 1000, 1024, 8


@pytest.fixture(scope="module")
def batch():
    bits = synth.logits_host(0, T, VP, VP, VR, seed=5, sigma=3.0, garbage=True)
    tgt = synth.targets(T, VR, 5)
    mask = (np.arange(T) % 3 != 0).astype(np.uint8)
    g = np.where(mask != 0, 0.5, 0.0).astype(np.float32)
    return (to_dev(bits), torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda(), torch.from_numpy(g).cuda())


def test_short_or_mistyped_tensors_raise_before_any_launch(batch):
    logits, dt, dm, dg = batch
    c = contract(T, VR, VP, NT, 2)
    lse = torch.zeros(T, dtype=torch.float32, device="cuda")
    cases = [
        lambda: rlk.logp_fwd(c, logits[:T - 1], dt, dm),                        # one row short
        lambda: rlk.logp_fwd(c, logits.view(-1)[:T * VP - 8], dt, dm),          # the last row cut
        lambda: rlk.logp_fwd(c, logits, dt[:T - 1], dm),                        # targets short
        lambda: rlk.logp_fwd(c, logits, dt.to(torch.int32), dm),                # targets not int64
        lambda: rlk.logp_fwd(c, logits, dt, dm[:T - 1]),                        # mask short
        lambda: rlk.logp_fwd(c, logits.float(), dt, dm),                        # logits not 16-bit
        lambda: rlk.logp_fwd(c, logits.cpu(), dt, dm),                          # logits on the host
        lambda: rlk.logp_bwd(c, logits, dt, dm, lse[:T - 1], dg),              # lse short
        lambda: rlk.logp_fwd_bwd(c, logits, dt, dm, dg, dlogits=logits[:T - 1]),  # dlogits short
        lambda: rlk.logp_fwd_bwd(c, logits, dt, dm, dg.double()),               # grad not FP32
        lambda: rlk.grpo_fused_step(c, logits, dt, dm, dg[:T - 1]),             # advantage short
        lambda: rlk.grpo_loss(lse, dg[:T - 1], dm),                             # advantage short
        lambda: rlk.shard_fwd(c, 0, logits[:, :VP // 2][:T - 1], dt, dm),       # shard rows short
    ]
    for i, call in enumerate(cases):
        with pytest.raises((ValueError, TypeError)):
            call()
    torch.cuda.synchronize()


def test_lmhead_shape_checks():
    Tl, H, vr, vp = 16, 64, 600, 608
    h = torch.zeros((Tl, H), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((vp, H), dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(Tl, dtype=torch.int64, device="cuda")
    c = rlk.Contract(T=Tl, V_real=vr, V_padded=vp, num_tiles=2, virtual_tp=1, mask_mode=rlk.MASK_IGNORE_INDEX)
    with pytest.raises(ValueError):
        rlk.logp_fused_lmhead(c.replace(T=Tl + 1), h, w, torch.zeros(Tl + 1, dtype=torch.int64, device="cuda"))
    with pytest.raises(ValueError):
        rlk.logp_fused_lmhead(c, h, w[:vp - 16], t)
    with pytest.raises(ValueError):
        rlk.logp_fused_lmhead(c, h[:, :H // 2], w, t)
    with pytest.raises(ValueError):  # [T, H] but transposed storage: not contiguous
        rlk.logp_fused_lmhead(c, torch.zeros((H, Tl), dtype=torch.bfloat16, device="cuda").t(), w, t)
    logp, lse, logits = rlk.logp_fused_lmhead_keep(c, h, w, t)
    g = torch.zeros(Tl, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        rlk.logp_fused_lmhead_bwd_kept(c, h, w, t, None, lse, logits[:Tl - 1], g)
    with pytest.raises(ValueError):
        rlk.logp_fused_lmhead_bwd(c, h, w, t, None, lse, g, workspace=torch.empty(64, dtype=torch.uint8,
                                                                                   device="cuda"))
    torch.cuda.synchronize()


def test_strided_shard_backward_allocates_the_shard_stride(batch):
    """shard_bwd on a shard read in place from the whole buffer (a strided view), with no dlogits given,
    is bitwise the same call on a contiguous copy of the shard."""
    logits, dt, dm, dg = batch
    c = contract(T, VR, VP, NT, 2)
    logp, lse = rlk.logp_fwd(c, logits, dt, dm)
    vs = VP // 2
    for j in range(2):
        view = logits[:, j * vs:(j + 1) * vs]
        d_view = rlk.shard_bwd(c.replace(row_stride=VP), j, view, dt, dm, lse, dg)
        d_copy = rlk.shard_bwd(c, j, view.contiguous(), dt, dm, lse, dg)
        torch.cuda.synchronize()
        assert d_view.shape == (T, VP) and torch.equal(d_view[:, :vs], d_copy[:, :vs]), j
