"""The entry points inside a CUDA graph: a captured fused forward+backward and a captured fused
lm_head forward+backward replay with the eager calls' bits, and a replay after the inputs change
gives the new inputs' results.  The captured calls take validate = 0 (validate synchronises) and
preallocated outputs and workspace; a first eager call on the device comes before the capture."""
import numpy as np
import pytest
import torch

import synth
import vocab_selected_token_tile_gb300 as rlk

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def test_fused_step_replays_from_a_graph(built):
    T, vr, vp, nt = 300, 5003, 5120, 64
    bits = synth.logits_host(0, T, vp, vp, vr, seed=3, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, vr, seed=3)
    mask = (np.arange(T) % 4 != 0).astype(np.uint8)
    g = np.where(mask != 0, 0.5, 0.0).astype(np.float32)
    logits = torch.from_numpy(bits.view(np.int16)).cuda()
    dt, dm, dg = (torch.from_numpy(a).cuda() for a in (tgt, mask, g))
    c = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=nt, virtual_tp=4, validate=0)
    ref = rlk.logp_fwd_bwd(c, logits, dt, dm, dg)  # the eager call (also the first call on the device)
    dl = torch.empty_like(logits)
    logp = torch.empty(T, device="cuda")
    lse = torch.empty(T, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rlk.check(rlk.rlk_logp_bwd(c, logits.data_ptr(), dt.data_ptr(), dm.data_ptr(), None, dg.data_ptr(),
                                   dl.data_ptr(), logp.data_ptr(), lse.data_ptr(), ws.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(dl, ref[0]) and torch.equal(logp, ref[1]) and torch.equal(lse, ref[2])
    assert rlk.rlk_logp_workspace_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == rlk.RLK_OK
    # new inputs in the same buffers: the replay computes them
    logits.copy_(torch.flip(logits, dims=[0]))
    ref2 = rlk.logp_fwd_bwd(c, logits, dt, dm, dg)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(dl, ref2[0]) and torch.equal(logp, ref2[1]) and torch.equal(lse, ref2[2])
    assert not torch.equal(ref2[2], ref[2])


def test_lmhead_forward_backward_replays_from_a_graph(built):
    T, H, vr, vp, nt = 257, 192, 1000, 1024, 4
    hb = synth.normal_bf16_host(0, T, H, 5, synth.STREAM_HIDDEN, 1.0)
    wb = synth.normal_bf16_host(0, vp, H, 5, synth.STREAM_WEIGHT, 0.2)
    tgt = synth.targets(T, vr, seed=5)
    mask = (np.arange(T) % 5 != 1).astype(np.uint8)
    g = np.where(mask != 0, 0.25, 0.0).astype(np.float32)
    hd = torch.from_numpy(hb.view(np.int16)).cuda()
    wd = torch.from_numpy(wb.view(np.int16)).cuda()
    dt, dm, dg = (torch.from_numpy(a).cuda() for a in (tgt, mask, g))
    c = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=nt, virtual_tp=2, validate=0)
    ref = rlk.logp_fused_lmhead(c, hd, wd, dt, dm, grad=dg)
    logp = torch.empty(T, device="cuda")
    lse = torch.empty(T, device="cuda")
    dh = torch.empty_like(hd)
    dw = torch.empty_like(wd)
    ws = torch.zeros(rlk.rlk_logp_lmhead_workspace_size(c, H), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rlk.check(rlk.rlk_logp_fused_lmhead(c, hd.data_ptr(), H, wd.data_ptr(), dt.data_ptr(), dm.data_ptr(),
                                            dg.data_ptr(), logp.data_ptr(), lse.data_ptr(), dh.data_ptr(), None,
                                            dw.data_ptr(), ws.data_ptr(), torch.cuda.current_stream().cuda_stream))
    for _ in range(2):  # the tickets are cleared inside the graph, so replays repeat exactly
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(logp, ref[0]) and torch.equal(lse, ref[1])
        assert torch.equal(dh, ref[2]) and torch.equal(dw, ref[3])


def test_grpo_step_replays_from_a_graph(built):
    """The fused GRPO step (two memsets, the count, the fused pass, the loss) captured once, replayed with
    the eager call's bits, then replayed on a new advantage in the same buffer."""
    T, vr, vp, nt = 200, 3001, 3072, 64
    bits = synth.logits_host(0, T, vp, vp, vr, seed=4, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, vr, seed=4)
    mask = (np.arange(T) % 3 != 0).astype(np.uint8)
    rng = np.random.default_rng(4)
    adv_h = rng.standard_normal(T).astype(np.float32)
    logits = torch.from_numpy(bits.view(np.int16)).cuda()
    dt, dm, adv = (torch.from_numpy(a).cuda() for a in (tgt, mask, adv_h))
    c = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=nt, virtual_tp=2, validate=0)
    ref_lp = rlk.logp_fwd(c, logits, dt, dm)[0] + 0.03
    want = rlk.grpo_fused_step(c, logits, dt, dm, adv, ref_lp, 0.01)  # eager
    bufs = {k: torch.empty(T, device="cuda") for k in ("logp", "lse", "grad")}
    dl = torch.empty_like(logits)
    loss = torch.empty(1, device="cuda")
    n = torch.empty(1, device="cuda")
    ws = torch.zeros(rlk.rlk_grpo_fused_workspace_size(c), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rlk.check(rlk.rlk_grpo_fused_step(c, logits.data_ptr(), dt.data_ptr(), dm.data_ptr(), adv.data_ptr(),
                                          ref_lp.data_ptr(), 0.01, dl.data_ptr(), bufs["logp"].data_ptr(),
                                          bufs["lse"].data_ptr(), bufs["grad"].data_ptr(), None, loss.data_ptr(),
                                          n.data_ptr(), ws.data_ptr(), torch.cuda.current_stream().cuda_stream))
    graph.replay()
    torch.cuda.synchronize()
    for k in ("logp", "lse", "grad"):
        assert torch.equal(bufs[k], want[k]), k
    assert torch.equal(dl, want["dlogits"]) and torch.equal(loss, want["loss"]) and torch.equal(n, want["active_count"])
    adv.copy_(torch.flip(adv, dims=[0]))
    want2 = rlk.grpo_fused_step(c, logits, dt, dm, adv, ref_lp, 0.01)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(bufs["grad"], want2["grad"]) and torch.equal(loss, want2["loss"])
    assert torch.equal(dl, want2["dlogits"]) and not torch.equal(want2["grad"], want["grad"])
