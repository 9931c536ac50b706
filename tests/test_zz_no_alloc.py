"""The allocation-free forward entry point, through the C ABI, on the GPU.

rlk_logp_fwd_noalloc is for callers that cannot allocate device memory while
they run (memory reserved up front, a plugin handed only a stream, a step
that must not call the synchronising cudaMalloc): its status scratch is a
static device array instead of a caller workspace.  Its outputs must equal
rlk_logp_fwd's, on two calls in a row (the second call reuses the array the
first one left behind).  This file sorts last so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import synth
import vocab_selected_token_tile_gb300 as rlk

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

TOL = 1e-4  # the LSE/logp tolerance of the parity tests


def test_noalloc_forward_matches_workspace_forward(built):
    T, v_real, v_padded, nt = 96, 151936, 152576, 64
    bits = synth.logits_host(0, T, v_padded, v_padded, v_real, seed=31, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, v_real, 31)
    mask = (np.arange(T) % 3 != 0).astype(np.uint8)
    logits = torch.from_numpy(bits.view(np.int16)).cuda()
    dt = torch.from_numpy(tgt).cuda()
    dm = torch.from_numpy(mask).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    for vtp in (1, 4):
        c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=vtp,
                         mask_mode=rlk.MASK_EXPLICIT, validate=1)
        ref_logp, ref_lse, ref_part = rlk.logp_fwd(c, logits, dt, dm, partials=True)
        for _ in range(2):
            logp = torch.full((T,), float("nan"), device="cuda")
            lse = torch.full((T,), float("nan"), device="cuda")
            part = torch.full((T, nt, 2), float("nan"), device="cuda")
            st = rlk.rlk_logp_fwd_noalloc(c, logits.data_ptr(), dt.data_ptr(), dm.data_ptr(), logp.data_ptr(),
                                          lse.data_ptr(), part.data_ptr(), stream)
            assert st == rlk.RLK_OK, rlk.rlk_last_error_message()
            torch.cuda.synchronize()
            assert (logp - ref_logp).abs().max().item() <= TOL
            assert (lse - ref_lse).abs().max().item() <= TOL
            assert torch.equal(logp, ref_logp) and torch.equal(lse, ref_lse) and torch.equal(part, ref_part)
    # a device-side condition is still reported through the static scratch (validate = 1) ...
    bad = dt.clone()
    bad[5] = v_real
    c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=2,
                     mask_mode=rlk.MASK_EXPLICIT, validate=1)
    logp = torch.empty(T, device="cuda")
    lse = torch.empty(T, device="cuda")
    assert rlk.rlk_logp_fwd_noalloc(c, logits.data_ptr(), bad.data_ptr(), dm.data_ptr(), logp.data_ptr(),
                                    lse.data_ptr(), None, stream) == rlk.RLK_ERR_TARGET_RANGE
    # ... and cleared again by the next call
    assert rlk.rlk_logp_fwd_noalloc(c, logits.data_ptr(), dt.data_ptr(), dm.data_ptr(), logp.data_ptr(),
                                    lse.data_ptr(), None, stream) == rlk.RLK_OK
