"""Every pointer an entry point receives must be device memory of the device
that holds its first operand; host memory (pinned or plain) fails closed with
RLK_ERR_INVALID_ARG before anything is launched.  The outputs keep their
sentinel values, which shows that no kernel ran."""
import ctypes

import numpy as np
import pytest
import torch

import vocab_selected_token_tile_gb300 as rlk

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def host_ptr(a):
    """Address of a plain (unregistered) host numpy buffer."""
    return a.ctypes.data_as(ctypes.c_void_p).value


def expect_invalid(st, name):
    assert st == rlk.RLK_ERR_INVALID_ARG, rlk.rlk_status_string(st)
    assert name in rlk.rlk_last_error_message()


def test_streaming_entries_reject_host_pointers(built):
    T, vr, vp, nt = 64, 1000, 1024, 4
    c = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=nt, virtual_tp=2, validate=1)
    logits = torch.zeros((T, vp), dtype=torch.int16, device="cuda")
    tgt = torch.zeros(T, dtype=torch.int64, device="cuda")
    mask = torch.ones(T, dtype=torch.uint8, device="cuda")
    g = torch.ones(T, dtype=torch.float32, device="cuda")
    logp = torch.full((T,), 7.0, device="cuda")
    lse = torch.full((T,), 7.0, device="cuda")
    dl = torch.full((T, vp), 0x7E7E, dtype=torch.int16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    pinned_tgt = torch.zeros(T, dtype=torch.int64).pin_memory()
    plain_tgt = np.zeros(T, dtype=np.int64)
    pinned_out = torch.zeros(T, dtype=torch.float32).pin_memory()
    for bad in (pinned_tgt.data_ptr(), host_ptr(plain_tgt)):
        expect_invalid(rlk.rlk_logp_fwd(c, logits.data_ptr(), bad, mask.data_ptr(), logp.data_ptr(), lse.data_ptr(),
                                        None, ws.data_ptr(), s), "targets")
        expect_invalid(rlk.rlk_logp_bwd(c, logits.data_ptr(), bad, mask.data_ptr(), None, g.data_ptr(),
                                        dl.data_ptr(), logp.data_ptr(), lse.data_ptr(), ws.data_ptr(), s), "targets")
        expect_invalid(rlk.rlk_logp_fwd_noalloc(c, logits.data_ptr(), bad, mask.data_ptr(), logp.data_ptr(),
                                                lse.data_ptr(), None, s), "targets")
    expect_invalid(rlk.rlk_logp_fwd(c, logits.data_ptr(), tgt.data_ptr(), mask.data_ptr(), pinned_out.data_ptr(),
                                    lse.data_ptr(), None, ws.data_ptr(), s), "logp")
    expect_invalid(rlk.rlk_logp_bwd(c, logits.data_ptr(), tgt.data_ptr(), mask.data_ptr(), lse.data_ptr(),
                                    pinned_out.data_ptr(), dl.data_ptr(), None, None, ws.data_ptr(), s), "grad_logp")
    ent_host = np.zeros(T, dtype=np.float32)
    expect_invalid(rlk.rlk_logp_fwd_entropy(c, logits.data_ptr(), tgt.data_ptr(), mask.data_ptr(), logp.data_ptr(),
                                            lse.data_ptr(), host_ptr(ent_host), ws.data_ptr(), s), "entropy")
    host_ws = np.zeros(256, dtype=np.uint8)
    expect_invalid(rlk.rlk_logp_fwd(c, logits.data_ptr(), tgt.data_ptr(), mask.data_ptr(), logp.data_ptr(),
                                    lse.data_ptr(), None, host_ptr(host_ws), s), "workspace")
    adv_host = np.zeros(T, dtype=np.float32)
    loss = torch.zeros(1, device="cuda")
    expect_invalid(rlk.rlk_grpo_loss(T, logp.data_ptr(), host_ptr(adv_host), mask.data_ptr(), None, 0.0,
                                     loss.data_ptr(), g.data_ptr(), None, s), "advantage")
    torch.cuda.synchronize()
    assert (logp == 7.0).all() and (lse == 7.0).all() and (dl == 0x7E7E).all()
    assert not ws.any()
    # the same call with device memory everywhere succeeds
    st = rlk.rlk_logp_fwd(c, logits.data_ptr(), tgt.data_ptr(), mask.data_ptr(), logp.data_ptr(), lse.data_ptr(),
                          None, ws.data_ptr(), s)
    assert st == rlk.RLK_OK, rlk.rlk_last_error_message()


def test_lmhead_rejects_host_targets_and_weight(built):
    T, H, vr, vp, nt = 128, 64, 256, 256, 1
    c = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=nt, virtual_tp=1, validate=1)
    hidden = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    weight = torch.zeros((vp, H), dtype=torch.int16, device="cuda")
    tgt = torch.zeros(T, dtype=torch.int64, device="cuda")
    mask = torch.ones(T, dtype=torch.uint8, device="cuda")
    g = torch.ones(T, dtype=torch.float32, device="cuda")
    logp = torch.full((T,), 7.0, device="cuda")
    lse = torch.full((T,), 7.0, device="cuda")
    dh = torch.full((T, H), 0x7E7E, dtype=torch.int16, device="cuda")
    dw = torch.full((vp, H), 0x7E7E, dtype=torch.int16, device="cuda")
    ws = torch.zeros(rlk.rlk_logp_lmhead_workspace_size(c, H), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    host_tgt = torch.zeros(T, dtype=torch.int64).pin_memory()
    host_w = torch.zeros((vp, H), dtype=torch.int16).pin_memory()
    host_dw = np.zeros((vp, H), dtype=np.float32)
    cases = [
        ((hidden, host_w.data_ptr(), tgt.data_ptr(), None, None, None), "weight"),
        ((hidden, weight.data_ptr(), host_tgt.data_ptr(), None, None, None), "targets"),
        ((hidden, weight.data_ptr(), tgt.data_ptr(), g.data_ptr(), host_ptr(host_dw), dw.data_ptr()), "dweight_f32"),
    ]
    for (hd, wp, tp, gp, dwf, dwb), name in cases:
        st = rlk.rlk_logp_fused_lmhead(c, hd.data_ptr(), H, wp, tp, mask.data_ptr(), gp, logp.data_ptr(),
                                       lse.data_ptr(), dh.data_ptr() if gp else None, dwf, dwb, ws.data_ptr(), s)
        expect_invalid(st, name)
    torch.cuda.synchronize()
    assert (logp == 7.0).all() and (lse == 7.0).all() and (dh == 0x7E7E).all() and (dw == 0x7E7E).all()
    assert not ws.any()
