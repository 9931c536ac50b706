"""The fused lm_head forward (tcgen05 GEMM + per-tile partials) against the FP64 oracle.

logits = hidden @ W^T are never materialised on the GPU; the oracle forms
them in FP64 from the same BF16 bits.  Tolerance: LSE and logp max abs
<= 1e-4 (FP32 accumulation over H terms stays far inside it); masking
bit-exact; outputs bitwise identical across virtual TP 1/2/4/8.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle.lmhead import lmhead_dlogits
import vocab_selected_token_tile_gb300 as rlk
from parity import report

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

TOL = 1e-4


def close(kind, got, ref):
    """Max abs error of an FP32 output against the FP64 oracle, within TOL."""
    err = float(np.max(np.abs(np.asarray(got, dtype=np.float64) - ref)))
    report("lmhead_" + kind, err)
    assert err <= TOL, f"{kind} max abs {err}"


def make(T, H, v_real, v_padded, seed, w_sigma=0.2):
    hb = synth.normal_bf16_host(0, T, H, seed, synth.STREAM_HIDDEN, 1.0)
    wb = synth.normal_bf16_host(0, v_padded, H, seed, synth.STREAM_WEIGHT, w_sigma)
    rng = np.random.default_rng(seed)
    wb[v_real:] = rng.integers(0, 1 << 16, size=(v_padded - v_real, H), dtype=np.uint16)  # padding rows: any bits
    return hb, wb


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def run(c, hb, wb, tgt, mask):
    return rlk.logp_fused_lmhead(c, dev(hb), dev(wb), torch.from_numpy(tgt).cuda(),
                                 None if mask is None else torch.from_numpy(mask).cuda())


# (T, H, V_real, V_padded, num_tiles)
CASES = [
    (128, 64, 256, 256, 1),        # one unit, one chunk, one K block
    (130, 128, 600, 608, 2),       # ragged token block, 48-column remainder chunk, padded rows
    (257, 192, 1000, 1024, 4),     # chunks of exactly 256, three token blocks
    (64, 256, 4000, 4096, 8),      # 512-column tiles: two full chunks each
    (96, 128, 2380, 2384 * 2, 2),  # the 2384-wide tile of the Qwen3 padded vocabulary (9 x 256 + 80)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T%d_H%d_V%d_P%d_NT%d" % c)
def test_lmhead_small_cases(case):
    T, H, v_real, v_padded, nt = case
    hb, wb = make(T, H, v_real, v_padded, seed=T + H)
    tgt = synth.targets(T, v_real, seed=T)
    mask = (np.arange(T) % 7 != 3).astype(np.uint8)
    tgt = np.where(mask != 0, tgt, -12345)  # inactive targets are never used as indices
    ref_logp, ref_lse, _ = oracle.lmhead_forward(hb, wb, np.where(mask != 0, tgt, 0), mask != 0, v_real)
    outs = set()
    for vtp in (v for v in (1, 2, 4, 8) if nt % v == 0):
        c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=vtp, validate=1)
        logp, lse = run(c, hb, wb, tgt, mask)
        torch.cuda.synchronize()
        lp, ls = logp.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
        close("lse", ls, ref_lse)
        close("logp", lp, ref_logp)
        assert np.all(lp[mask == 0] == 0.0) and not np.any(np.signbit(lp[mask == 0]))
        outs.add((lp.tobytes(), ls.tobytes()))
    assert len(outs) == 1, "virtual TP outputs differ"


def test_lmhead_ignore_index_and_errors():
    T, H, v_real, v_padded, nt = 140, 128, 600, 608, 2
    hb, wb = make(T, H, v_real, v_padded, seed=5)
    tgt = synth.targets(T, v_real, seed=5, ignore_frac=0.3)
    c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=2,
                     mask_mode=rlk.MASK_IGNORE_INDEX, validate=1)
    logp, lse = run(c, hb, wb, tgt, None)
    active = tgt != -100
    ref_logp, ref_lse, _ = oracle.lmhead_forward(hb, wb, np.where(active, tgt, 0), active, v_real)
    torch.cuda.synchronize()
    close("lse", lse.cpu().numpy(), ref_lse)
    close("logp", logp.cpu().numpy(), ref_logp)
    bad = tgt.copy()
    bad[np.nonzero(active)[0][0]] = v_real + 3  # an active target in the padding
    with pytest.raises(rlk.RlkError) as ei:
        run(c, hb, wb, bad, None)
    assert ei.value.status == rlk.RLK_ERR_TARGET_RANGE


def test_lmhead_rejects_unsupported_shapes():
    c = rlk.Contract(T=8, V_real=600, V_padded=600, num_tiles=2, virtual_tp=1)  # tile width 300
    assert rlk.rlk_logp_lmhead_workspace_size(c, 128) == 0
    c = rlk.Contract(T=8, V_real=608, V_padded=608, num_tiles=2, virtual_tp=1)
    assert rlk.rlk_logp_lmhead_workspace_size(c, 100) == 0                    # H not a multiple of 64
    assert rlk.rlk_logp_lmhead_workspace_size(c, 128) > 0


def test_lmhead_full_shape_sampled_rows():
    """hidden [8192, 4096] x W [152576, 4096], 64 tiles, in the bench's configuration."""
    from synth import workloads as Wl
    w = Wl.LMHEAD
    T, H, v_real, v_padded = w.T, w.hidden, w.v_real, w.v_padded
    hd = torch.empty((T, H), dtype=torch.int16, device="cuda")
    wd = torch.empty((v_padded, H), dtype=torch.int16, device="cuda")
    synth.normal_bf16_device(hd, 0, T, H, w.seed, synth.STREAM_HIDDEN, w.hidden_sigma)
    synth.normal_bf16_device(wd, 0, v_padded, H, w.seed, synth.STREAM_WEIGHT, w.weight_sigma)
    tgt = Wl.targets(w)
    mask = Wl.active_mask(w)
    dt, dm = torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda()
    res = {}
    for vtp in (1, 8):
        c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=64, virtual_tp=vtp, validate=1)
        res[vtp] = rlk.logp_fused_lmhead(c, hd, wd, dt, dm)
        torch.cuda.synchronize()
    assert torch.equal(res[1][0], res[8][0]) and torch.equal(res[1][1], res[8][1])
    rows = np.unique(np.concatenate([[0, 127, 128, T - 1], np.random.default_rng(3).choice(T, 28, replace=False)]))
    hb = np.concatenate([synth.normal_bf16_host(int(r), 1, H, w.seed, synth.STREAM_HIDDEN, w.hidden_sigma)
                         for r in rows])
    wb = synth.normal_bf16_host(0, v_padded, H, w.seed, synth.STREAM_WEIGHT, w.weight_sigma)
    assert np.array_equal(hd[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint16), hb)
    ref_logp, ref_lse, _ = oracle.lmhead_forward(hb, wb, tgt[rows], mask[rows] != 0, v_real)
    logp, lse = res[1]
    close("lse", lse.cpu().numpy()[rows], ref_lse)
    close("logp", logp.cpu().numpy()[rows], ref_logp)


def grad_bounds(hb, wb, tgt, active, g, v_real):
    """Oracle dhidden, dweight and the scale of their terms, sum |a||b|, in FP64."""
    _, lse, x = oracle.lmhead_forward(hb, wb, tgt, active, v_real)
    d = lmhead_dlogits(x, lse, tgt, active, g)
    h = oracle.bf16_bits_to_f64(hb)
    w = oracle.bf16_bits_to_f64(wb[:v_real])
    dh, dw = d @ w, d.T @ h
    return dh, dw, np.abs(d) @ np.abs(w), np.abs(d).T @ np.abs(h)


def within(got_bits, ref, scale):
    """BF16 result vs FP64: dlogits and the output are each rounded once to BF16 (2^-9
    relative); the GEMM accumulates in FP32.  Bound: 2^-8 (|ref| + sum |terms|)."""
    got = oracle.bf16_bits_to_f64(got_bits)
    return np.abs(got - ref) <= 2.0 ** -8 * (np.abs(ref) + scale) + 1e-30


@pytest.mark.parametrize("case", CASES[1:5] + [(129, 64, 300, 320, 5)], ids=lambda c: "T%d_H%d_V%d_P%d_NT%d" % c)
def test_lmhead_backward_small_cases(case):
    T, H, v_real, v_padded, nt = case
    hb, wb = make(T, H, v_real, v_padded, seed=3 * T + H)
    tgt = synth.targets(T, v_real, seed=T + 1)
    mask = (np.arange(T) % 5 != 1).astype(np.uint8)
    g = np.where(mask != 0, np.random.default_rng(T).standard_normal(T), 0.0).astype(np.float32)
    ref_dh, ref_dw, sc_dh, sc_dw = grad_bounds(hb, wb, tgt, mask != 0, g, v_real)
    ref_logp, ref_lse, _ = oracle.lmhead_forward(hb, wb, tgt, mask != 0, v_real)
    outs = set()
    for vtp in (v for v in (1, 2, 4) if nt % v == 0):
        c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=vtp, validate=1)
        logp, lse, dh, dw = rlk.logp_fused_lmhead(c, dev(hb), dev(wb), torch.from_numpy(tgt).cuda(),
                                                  torch.from_numpy(mask).cuda(), grad=torch.from_numpy(g).cuda())
        torch.cuda.synchronize()
        close("lse", lse.cpu().numpy(), ref_lse)
        close("logp", logp.cpu().numpy(), ref_logp)
        dhb = dh.cpu().numpy().view(np.uint16)
        dwb = dw.cpu().numpy().view(np.uint16)
        assert np.all(within(dhb, ref_dh, sc_dh))
        assert np.all(within(dwb[:v_real], ref_dw, sc_dw))
        assert np.all(dwb[v_real:] == 0)
        outs.add((dhb.tobytes(), dwb.tobytes()))
    assert len(outs) == 1, "virtual TP gradients differ"


def test_lmhead_backward_full_shape():
    """8192 x 4096 x 152576: dhidden on sampled rows against the oracle; dweight by properties."""
    from synth import workloads as Wl
    w = Wl.LMHEAD
    T, H, v_real, v_padded = w.T, w.hidden, w.v_real, w.v_padded
    hd = torch.empty((T, H), dtype=torch.int16, device="cuda")
    wd = torch.empty((v_padded, H), dtype=torch.int16, device="cuda")
    synth.normal_bf16_device(hd, 0, T, H, w.seed, synth.STREAM_HIDDEN, w.hidden_sigma)
    synth.normal_bf16_device(wd, 0, v_padded, H, w.seed, synth.STREAM_WEIGHT, w.weight_sigma)
    tgt = Wl.targets(w)
    mask = Wl.active_mask(w)
    g = Wl.grad(w, mask != 0)
    c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=64, virtual_tp=2, validate=1)
    logp, lse, dh, dw = rlk.logp_fused_lmhead(c, hd, wd, torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda(),
                                              grad=torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    rows = np.array([0, 1, 4095, T - 1])
    hb = np.concatenate([synth.normal_bf16_host(int(r), 1, H, w.seed, synth.STREAM_HIDDEN, w.hidden_sigma)
                         for r in rows])
    wb = synth.normal_bf16_host(0, v_padded, H, w.seed, synth.STREAM_WEIGHT, w.weight_sigma)
    _, ref_lse, x = oracle.lmhead_forward(hb, wb, tgt[rows], mask[rows] != 0, v_real)
    d = lmhead_dlogits(x, ref_lse, tgt[rows], mask[rows] != 0, g[rows])
    wv = oracle.bf16_bits_to_f64(wb[:v_real])
    ref = d @ wv
    scale = np.abs(d) @ np.abs(wv)
    got = dh[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint16)
    assert np.all(within(got, ref, scale))
    dwb = dw.view(torch.bfloat16)
    assert not dw[v_real:].any()
    # sum over the vocabulary of dW = sum_t h_t * sum_v dlogits[t, v] = 0, up to BF16 rounding
    col_sum = dwb[:v_real].float().sum(dim=0)
    col_abs = dwb[:v_real].float().abs().sum(dim=0)
    assert (col_sum.abs() <= 2.0 ** -6 * col_abs + 1e-6).all()


def test_lmhead_repeat_runs_are_bitwise_equal():
    """Units are handed out by an atomic ticket, so which CTA runs which
    (token block, tile) unit changes from run to run; every unit's arithmetic
    is fixed, so logp, LSE and both gradients are bitwise the same on every
    run.  Three token blocks and a 2384-wide tile (9 x 256 + 80 columns)."""
    T, H, v_real, v_padded, nt = 300, 128, 2380, 2384 * 2, 2
    hb, wb = make(T, H, v_real, v_padded, seed=11)
    tgt = synth.targets(T, v_real, seed=12)
    mask = (np.arange(T) % 3 != 0).astype(np.uint8)
    g = np.where(mask != 0, np.random.default_rng(13).standard_normal(T), 0.0).astype(np.float32)
    outs = set()
    for _ in range(3):
        c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=2, validate=1)
        logp, lse, dh, dw = rlk.logp_fused_lmhead(c, dev(hb), dev(wb), torch.from_numpy(tgt).cuda(),
                                                  torch.from_numpy(mask).cuda(), grad=torch.from_numpy(g).cuda())
        torch.cuda.synchronize()
        outs.add(tuple(t.cpu().numpy().tobytes() for t in (logp, lse, dh, dw)))
    assert len(outs) == 1
    ref_logp, ref_lse, _ = oracle.lmhead_forward(hb, wb, tgt, mask != 0, v_real)
    logp = np.frombuffer(next(iter(outs))[0], dtype=np.float32)
    close("logp", logp, ref_logp)


def bf16_rn_bits(x):
    """FP32 values rounded to BF16 (round to nearest even), as uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


@pytest.mark.parametrize("case", [CASES[1], CASES[4], (200, 320, 1000, 1024, 4)],
                         ids=lambda c: "T%d_H%d_V%d_P%d_NT%d" % c)
def test_lmhead_fp32_dweight(case):
    """The FP32 dweight output is the GEMM's FP32 accumulator: within the FP32
    accumulation bound of the FP64 oracle, and its BF16 rounding is bitwise
    the BF16 dweight output of the same call.  H = 320 leaves a 64-wide last
    block of the hidden dimension."""
    T, H, v_real, v_padded, nt = case
    hb, wb = make(T, H, v_real, v_padded, seed=7 * T + H)
    tgt = synth.targets(T, v_real, seed=T + 5)
    mask = (np.arange(T) % 4 != 2).astype(np.uint8)
    g = np.where(mask != 0, np.random.default_rng(T + 1).standard_normal(T), 0.0).astype(np.float32)
    ref_dh, ref_dw, sc_dh, sc_dw = grad_bounds(hb, wb, tgt, mask != 0, g, v_real)
    c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=1, validate=1)
    _, _, dh, (dwf, dwb) = rlk.logp_fused_lmhead(c, dev(hb), dev(wb), torch.from_numpy(tgt).cuda(),
                                                 torch.from_numpy(mask).cuda(), grad=torch.from_numpy(g).cuda(),
                                                 dweight_dtype="both")
    torch.cuda.synchronize()
    f = dwf.cpu().numpy().astype(np.float64)
    # dlogits are BF16 (one rounding, 2^-9 relative) and the sum is FP32
    assert np.all(np.abs(f[:v_real] - ref_dw) <= 2.0 ** -8 * (np.abs(ref_dw) + sc_dw) + 1e-30)
    assert np.all(f[v_real:] == 0.0) and not np.any(np.signbit(f[v_real:]))
    assert np.array_equal(bf16_rn_bits(dwf.cpu().numpy()), dwb.cpu().numpy().view(np.uint16))
    assert np.all(within(dh.cpu().numpy().view(np.uint16), ref_dh, sc_dh))


@pytest.mark.parametrize("case", [CASES[1], CASES[4]], ids=lambda c: "T%d_H%d_V%d_P%d_NT%d" % c)
def test_lmhead_backward_from_a_given_lse_is_bitwise_the_fused_call(case):
    """rlk_logp_fused_lmhead_bwd (recompute + gradient GEMMs from the forward's LSE) gives bitwise
    the gradients of rlk_logp_fused_lmhead with grad_logp; an out-of-range active target and a
    non-finite LSE on an active row are reported."""
    T, H, v_real, v_padded, nt = case
    hb, wb = make(T, H, v_real, v_padded, seed=5 * T + H)
    tgt = synth.targets(T, v_real, seed=T + 9)
    mask = (np.arange(T) % 6 != 4).astype(np.uint8)
    g = np.where(mask != 0, np.random.default_rng(T + 2).standard_normal(T), 0.0).astype(np.float32)
    c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=1, validate=1)
    dh_, dw_ = dev(hb), dev(wb)
    dt, dm, dg = torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda(), torch.from_numpy(g).cuda()
    logp, lse, dh, dw = rlk.logp_fused_lmhead(c, dh_, dw_, dt, dm, grad=dg, dweight_dtype="both")
    dh2, dw2 = rlk.logp_fused_lmhead_bwd(c, dh_, dw_, dt, dm, lse, dg, dweight_dtype="both")
    torch.cuda.synchronize()
    assert torch.equal(dh, dh2) and torch.equal(dw[0], dw2[0]) and torch.equal(dw[1], dw2[1])
    bad = dt.clone()
    bad[int(np.nonzero(mask)[0][0])] = v_real + 1
    with pytest.raises(rlk.RlkError) as ei:
        rlk.logp_fused_lmhead_bwd(c, dh_, dw_, bad, dm, lse, dg)
    assert ei.value.status == rlk.RLK_ERR_TARGET_RANGE
    l2 = lse.clone()
    l2[int(np.nonzero(mask)[0][1])] = float("inf")
    with pytest.raises(rlk.RlkError) as ei:
        rlk.logp_fused_lmhead_bwd(c, dh_, dw_, dt, dm, l2, dg)
    assert ei.value.status == rlk.RLK_ERR_NONFINITE_LSE


@pytest.mark.parametrize("case", [(1, 64, 200, 256, 2), (127, 64, 1000, 1024, 8), (3, 128, 2380, 2384 * 8, 8)],
                         ids=lambda c: "T%d_H%d_V%d_P%d_NT%d" % c)
def test_lmhead_degenerate_sizes(case):
    """A single token, one partial token block, one tile per shard at virtual TP 8, padded tiles:
    forward and backward against the oracle, bitwise across virtual TP."""
    T, H, v_real, v_padded, nt = case
    hb, wb = make(T, H, v_real, v_padded, seed=T + 17)
    tgt = synth.targets(T, v_real, seed=T + 18)
    mask = np.ones(T, dtype=np.uint8)
    if T > 2:
        mask[1] = 0
    g = np.where(mask != 0, np.random.default_rng(T).standard_normal(T), 0.0).astype(np.float32)
    ref_logp, ref_lse, _ = oracle.lmhead_forward(hb, wb, tgt, mask != 0, v_real)
    ref_dh, ref_dw, sc_dh, sc_dw = grad_bounds(hb, wb, tgt, mask != 0, g, v_real)
    outs = set()
    for vtp in (v for v in (1, 2, 4, 8) if nt % v == 0):
        c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=vtp, validate=1)
        logp, lse, dh, dw = rlk.logp_fused_lmhead(c, dev(hb), dev(wb), torch.from_numpy(tgt).cuda(),
                                                  torch.from_numpy(mask).cuda(), grad=torch.from_numpy(g).cuda())
        torch.cuda.synchronize()
        close("lse", lse.cpu().numpy(), ref_lse)
        close("logp", logp.cpu().numpy(), ref_logp)
        dhb, dwb = dh.cpu().numpy().view(np.uint16), dw.cpu().numpy().view(np.uint16)
        assert np.all(within(dhb, ref_dh, sc_dh))
        assert np.all(within(dwb[:v_real], ref_dw, sc_dw)) and np.all(dwb[v_real:] == 0)
        outs.add((logp.cpu().numpy().tobytes(), lse.cpu().numpy().tobytes(), dhb.tobytes(), dwb.tobytes()))
    assert len(outs) == 1


@pytest.mark.parametrize("case", [CASES[1], CASES[4], (129, 64, 300, 320, 5)], ids=lambda c: "T%d_H%d_V%d_P%d_NT%d" % c)
def test_lmhead_kept_logits_forward_and_backward(case):
    """rlk_logp_fused_lmhead_keep: logp and LSE bitwise the plain forward's; the kept FP32 logits within
    FP32 accumulation of the FP64 oracle's on the real columns, bitwise the same at every virtual TP.
    rlk_logp_fused_lmhead_bwd_kept: dHidden and dW bitwise those of the backward from the LSE and of
    the fused call, the kept logits untouched; an active target outside [0, V_real) and a non-finite
    LSE are reported."""
    T, H, v_real, v_padded, nt = case
    hb, wb = make(T, H, v_real, v_padded, seed=5 * T + H)
    tgt = synth.targets(T, v_real, seed=T + 3)
    mask = (np.arange(T) % 6 != 2).astype(np.uint8)
    g = np.where(mask != 0, np.random.default_rng(T).standard_normal(T), 0.0).astype(np.float32)
    dh_, dw_, dt, dm, dg = dev(hb), dev(wb), torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda(), \
        torch.from_numpy(g).cuda()
    c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=1, validate=1)
    logp, lse = rlk.logp_fused_lmhead(c, dh_, dw_, dt, dm)
    logp_k, lse_k, logits = rlk.logp_fused_lmhead_keep(c, dh_, dw_, dt, dm)
    torch.cuda.synchronize()
    assert torch.equal(logp, logp_k) and torch.equal(lse, lse_k)
    x = logits.cpu().numpy().astype(np.float64)[:, :v_real]
    ref = oracle.lmhead_logits(hb, wb, v_real)
    scale = np.abs(oracle.bf16_bits_to_f64(hb)) @ np.abs(oracle.bf16_bits_to_f64(wb[:v_real])).T
    # a tensor-core FP32 accumulation: a few units of 2^-24 per addition at most (2^-22 taken)
    assert np.all(np.abs(x - ref) <= H * 2.0 ** -22 * scale + 1e-30), "kept logits outside FP32 accumulation"
    for vtp in (v for v in (2, 4, 8) if nt % v == 0):
        cv = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=vtp, validate=1)
        _, _, lv = rlk.logp_fused_lmhead_keep(cv, dh_, dw_, dt, dm)
        torch.cuda.synchronize()
        assert torch.equal(lv[:, :v_real], logits[:, :v_real]), vtp
    before = logits.clone()
    dh1, dw1 = rlk.logp_fused_lmhead_bwd(c, dh_, dw_, dt, dm, lse, dg, dweight_dtype="both")
    dh2, dw2 = rlk.logp_fused_lmhead_bwd_kept(c, dh_, dw_, dt, dm, lse_k, logits, dg, dweight_dtype="both")
    _, _, dh3, dw3 = rlk.logp_fused_lmhead(c, dh_, dw_, dt, dm, grad=dg, dweight_dtype="both")
    torch.cuda.synchronize()
    assert torch.equal(logits.view(torch.int32), before.view(torch.int32))  # bits: padded columns may hold NaN
    for a, b in ((dh1, dh2), (dw1[0], dw2[0]), (dw1[1], dw2[1]), (dh3, dh2), (dw3[0], dw2[0]), (dw3[1], dw2[1])):
        assert torch.equal(a, b)
    bad = tgt.copy()
    bad[int(np.nonzero(mask)[0][0])] = v_real + 1
    with pytest.raises(rlk.RlkError) as ei:
        rlk.logp_fused_lmhead_bwd_kept(c, dh_, dw_, torch.from_numpy(bad).cuda(), dm, lse_k, logits, dg)
    assert ei.value.status == rlk.RLK_ERR_TARGET_RANGE
    l2 = lse_k.clone()
    l2[int(np.nonzero(mask)[0][1])] = float("nan")
    with pytest.raises(rlk.RlkError) as ei:
        rlk.logp_fused_lmhead_bwd_kept(c, dh_, dw_, dt, dm, l2, logits, dg)
    assert ei.value.status == rlk.RLK_ERR_NONFINITE_LSE


def test_lmhead_ragged_last_band_of_token_blocks():
    """At H = 4096 a band of the logits GEMMs' unit order is 32 token blocks (32 MB of hidden); 5000
    rows are 40 blocks, a full band and a ragged one of 8.  Forward and backward against the oracle,
    bitwise across virtual TP, in both the one-call form and the split form that keeps the logits."""
    T, H, v_real, v_padded, nt = 5000, 4096, 600, 608, 2
    hb, wb = make(T, H, v_real, v_padded, seed=61, w_sigma=0.05)
    tgt = synth.targets(T, v_real, seed=61)
    mask = (np.arange(T) % 9 != 4).astype(np.uint8)
    g = np.where(mask != 0, np.random.default_rng(61).standard_normal(T), 0.0).astype(np.float32)
    act = mask != 0
    ref_logp, ref_lse, _ = oracle.lmhead_forward(hb, wb, tgt, act, v_real)
    ref_dh, ref_dw, sc_dh, sc_dw = grad_bounds(hb, wb, tgt, act, g, v_real)
    dh_, dw_, dt, dm, dg = dev(hb), dev(wb), torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda(), \
        torch.from_numpy(g).cuda()
    outs = set()
    for vtp in (1, 2):
        c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=vtp, validate=1)
        logp, lse, dh, dw = rlk.logp_fused_lmhead(c, dh_, dw_, dt, dm, grad=dg)
        _, lse_k, logits = rlk.logp_fused_lmhead_keep(c, dh_, dw_, dt, dm)
        dh2, dw2 = rlk.logp_fused_lmhead_bwd_kept(c, dh_, dw_, dt, dm, lse_k, logits, dg)
        dh3, dw3 = rlk.logp_fused_lmhead_bwd(c, dh_, dw_, dt, dm, lse, dg)
        torch.cuda.synchronize()
        close("lse", lse.cpu().numpy(), ref_lse)
        close("logp", logp.cpu().numpy()[act], ref_logp[act])
        dhb, dwb = dh.cpu().numpy().view(np.uint16), dw.cpu().numpy().view(np.uint16)
        assert np.all(within(dhb, ref_dh, sc_dh))
        assert np.all(within(dwb[:v_real], ref_dw, sc_dw)) and np.all(dwb[v_real:] == 0)
        for a, b in ((dh, dh2), (dw, dw2), (dh, dh3), (dw, dw3), (lse, lse_k)):
            assert torch.equal(a, b), vtp
        outs.add((logp.cpu().numpy().tobytes(), lse.cpu().numpy().tobytes(), dhb.tobytes(), dwb.tobytes()))
    assert len(outs) == 1


def test_lmhead_gradient_ragged_band_of_h_blocks():
    """The gradient GEMMs take their 256-wide H blocks in bands of 8; H = 2368 is 10 blocks (the last
    64 wide), a full band and a ragged one of 2.  dHidden and dW against the oracle, bitwise across
    virtual TP."""
    T, H, v_real, v_padded, nt = 300, 2368, 1000, 1024, 4
    hb, wb = make(T, H, v_real, v_padded, seed=67, w_sigma=0.05)
    tgt = synth.targets(T, v_real, seed=67)
    mask = (np.arange(T) % 7 != 2).astype(np.uint8)
    g = np.where(mask != 0, np.random.default_rng(67).standard_normal(T), 0.0).astype(np.float32)
    act = mask != 0
    ref_dh, ref_dw, sc_dh, sc_dw = grad_bounds(hb, wb, tgt, act, g, v_real)
    dh_, dw_, dt, dm, dg = dev(hb), dev(wb), torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda(), \
        torch.from_numpy(g).cuda()
    outs = set()
    for vtp in (1, 4):
        c = rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=vtp, validate=1)
        _, _, dh, dw = rlk.logp_fused_lmhead(c, dh_, dw_, dt, dm, grad=dg, dweight_dtype="f32")
        torch.cuda.synchronize()
        dhb, dwf = dh.cpu().numpy().view(np.uint16), dw.cpu().numpy().astype(np.float64)
        assert np.all(within(dhb, ref_dh, sc_dh))
        # FP32 dW: the BF16 dlogits' rounding (2^-9) and the FP32 sum, no output rounding
        assert np.all(np.abs(dwf[:v_real] - ref_dw) <= 2.0 ** -8 * (np.abs(ref_dw) + sc_dw) + 1e-30)
        assert np.all(dwf[v_real:] == 0.0)
        outs.add((dhb.tobytes(), dwf.tobytes()))
    assert len(outs) == 1
