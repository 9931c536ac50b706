"""Full-size parity: the 65536 x 152576 rollout/GRPO batch, in bench.py's launch configuration.

The oracle computes sampled rows one by one from host-generated copies of
the same rows (first, last, inactive and seeded random rows); properties that
hold at any size are checked over the whole batch on the device.
"""
import numpy as np
import pytest
import torch

import oracle
import vocab_selected_token_tile_gb300 as rlk
from parity import check_dlogits, check_entropy, check_fwd, contract
from synth import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

BENCH_VTP = 2  # bench.py's default virtual TP for the fused step


@pytest.fixture(scope="module")
def batch():
    w = W.GRPO
    logits = torch.empty((w.T, w.v_padded), dtype=torch.int16, device="cuda")
    W.logits_device(w, logits)
    tgt = W.targets(w)
    mask = W.active_mask(w)
    active = mask != 0
    g = W.grad(w, active)
    rng = np.random.default_rng(99)
    inactive = np.nonzero(~active)[0]
    rows = np.unique(np.concatenate([[0, 1, 2, w.T - 3, w.T - 2, w.T - 1], rng.choice(w.T, 96, replace=False),
                                     rng.choice(inactive, 16, replace=False)]))
    bits = np.concatenate([W.logits_host(w, row0=int(r), nrows=1) for r in rows])
    yield dict(w=w, logits=logits, tgt=tgt, mask=mask, active=active, g=g, rows=rows, bits=bits,
               dt=torch.from_numpy(tgt).cuda(), dm=torch.from_numpy(mask).cuda(), dg=torch.from_numpy(g).cuda())
    del logits
    torch.cuda.empty_cache()


def test_sampled_rows_match_the_host_generator(batch):
    got = batch["logits"][torch.from_numpy(batch["rows"]).cuda()].cpu().numpy().view(np.uint16)
    assert np.array_equal(got, batch["bits"])


def test_rollout_forward_full_size(batch):
    w, rows = batch["w"], batch["rows"]
    for vtp in (1, 8):
        c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, vtp)
        logp, lse = rlk.logp_fwd(c, batch["logits"], batch["dt"], batch["dm"])
        torch.cuda.synchronize()
        assert torch.isfinite(lse).all()
        act = torch.from_numpy(batch["active"]).cuda()
        assert (logp[~act] == 0).all() and (logp[act] <= 0).all()
        lp, ls = logp.cpu().numpy()[rows], lse.cpu().numpy()[rows]
        check_fwd(batch["bits"], batch["tgt"][rows], batch["active"][rows], w.v_real, lp, ls)
        if vtp == 1:
            ref = (logp.clone(), lse.clone())
        else:
            assert torch.equal(ref[0], logp) and torch.equal(ref[1], lse)


def test_grpo_fused_full_size_in_bench_configuration(batch):
    w, rows = batch["w"], batch["rows"]
    c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, BENCH_VTP, validate=0)
    dl, logp, lse = rlk.logp_fwd_bwd(c, batch["logits"], batch["dt"], batch["dm"], batch["dg"])
    torch.cuda.synchronize()
    assert rlk.rlk_logp_workspace_status(rlk.workspace_for(c, dl.device).data_ptr(),
                                         torch.cuda.current_stream().cuda_stream) == rlk.RLK_OK
    # sampled rows against the oracle, element by element
    lp, ls = logp.cpu().numpy()[rows], lse.cpu().numpy()[rows]
    check_fwd(batch["bits"], batch["tgt"][rows], batch["active"][rows], w.v_real, lp, ls)
    dl_rows = dl[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint16)
    check_dlogits(batch["bits"], batch["tgt"][rows], batch["active"][rows], batch["g"][rows], w.v_real,
                  w.v_padded, dl_rows, rows=np.arange(len(rows)))
    # whole batch, in row blocks: inactive rows and padded columns exactly zero, and
    # each active row's dlogits sum to ~0 (BF16 rounding of about 2|g| of mass)
    act = torch.from_numpy(batch["active"]).cuda()
    for r0 in range(0, w.T, 4096):
        blk, a = dl[r0:r0 + 4096], act[r0:r0 + 4096]
        assert not blk[~a].any()
        assert not blk[:, w.v_real:].any()
        sums = blk[a].view(torch.bfloat16).float().sum(dim=1)
        gabs = batch["dg"][r0:r0 + 4096][a].abs()
        assert (sums.abs() <= 2.0 ** -6 * gabs + 1e-12).all()
    # the split path (fwd then bwd with lse_in) gives the same bits
    c1 = c.replace(virtual_tp=1)
    logp1, lse1 = rlk.logp_fwd(c1, batch["logits"], batch["dt"], batch["dm"])
    assert torch.equal(logp1, logp) and torch.equal(lse1, lse)
    dl1 = rlk.logp_bwd(c1, batch["logits"], batch["dt"], batch["dm"], lse1, batch["dg"])
    torch.cuda.synchronize()
    assert torch.equal(dl1, dl)
    # the fused step at virtual TP 1 and 8 (their own planner choices: two CTAs per SM with
    # no row skew, and two rows of skew) gives the same bits as the bench configuration
    for vtp in (1, 8):
        dlv, lpv, lsv = rlk.logp_fwd_bwd(c.replace(virtual_tp=vtp), batch["logits"], batch["dt"], batch["dm"],
                                         batch["dg"], dlogits=dl1)
        torch.cuda.synchronize()
        assert torch.equal(lpv, logp) and torch.equal(lsv, lse) and torch.equal(dlv, dl), vtp
    # oracle-side sanity of the sampled rows' gradient sums (pins the device property above)
    ref = oracle.dlogits(batch["bits"][:8], batch["tgt"][rows[:8]], batch["active"][rows[:8]],
                         batch["g"][rows[:8]], w.v_real, w.v_padded)
    assert np.all(np.abs(ref.sum(axis=1)) <= 1e-9 * (np.abs(batch["g"][rows[:8]]) + 1e-30) * w.v_real)


def test_grpo_step_and_entropy_full_size(batch):
    """Two more of the bench's lines at full size, virtual TP 2.  The fused GRPO step (beta 0.01, a
    reference logp, one advantage per 2048-token sequence, as bench.py draws them) is bitwise the
    composition forward -> rlk_grpo_loss -> backward from the LSE, and its loss and g are the oracle's
    on the step's own logp within FP32 rounding.  The fused forward+backward with the entropy gives the
    fused step's bits and the oracle's entropy on the sampled rows."""
    w, rows = batch["w"], batch["rows"]
    T = w.T
    c = contract(T, w.v_real, w.v_padded, w.num_tiles, BENCH_VTP, validate=0)
    rng = np.random.default_rng(1)
    adv = np.repeat(rng.standard_normal(T // 2048 or 1), 2048)[:T].astype(np.float32)
    ref = (-6.0 * rng.random(T)).astype(np.float32)
    dadv, dref = torch.from_numpy(adv).cuda(), torch.from_numpy(ref).cuda()
    dl_a, dl_b = torch.empty_like(batch["logits"]), torch.empty_like(batch["logits"])
    st = rlk.grpo_fused_step(c, batch["logits"], batch["dt"], batch["dm"], dadv, dref, 0.01, dlogits=dl_a)
    logp, lse = rlk.logp_fwd(c, batch["logits"], batch["dt"], batch["dm"])
    loss, g, n = rlk.grpo_loss(logp, dadv, batch["dm"], dref, 0.01)
    rlk.logp_bwd(c, batch["logits"], batch["dt"], batch["dm"], lse, g, dlogits=dl_b)
    torch.cuda.synchronize()
    for k, want in (("logp", logp), ("lse", lse), ("grad", g), ("loss", loss), ("active_count", n)):
        assert torch.equal(st[k], want), k
    assert torch.equal(dl_a, dl_b)
    act = batch["active"]
    lp = logp.cpu().numpy()
    ol, og, on = oracle.grpo_loss(lp, adv, act, ref, 0.01)
    assert float(n.item()) == on
    eps = 2.0 ** -24
    d = np.abs(ref.astype(np.float64) - lp)
    e = np.exp(ref.astype(np.float64) - lp)
    assert np.all(np.abs(g.cpu().numpy() - og) <= 8 * eps * (np.abs(adv) + 0.01 * (1.0 + e * (1.0 + d))) / on)
    terms = np.abs(adv * lp) + 0.01 * e * (1.0 + d)
    assert abs(float(loss.item()) - ol) <= 8 * eps * float(terms[act].sum()) / on + 2 * eps * abs(ol)
    # the entropy in the fused pass
    dl_e, lp_e, ls_e, ent = rlk.logp_fwd_bwd_entropy(c, batch["logits"], batch["dt"], batch["dm"], batch["dg"],
                                                     dlogits=dl_a)
    dl_f, lp_f, ls_f = rlk.logp_fwd_bwd(c, batch["logits"], batch["dt"], batch["dm"], batch["dg"], dlogits=dl_b)
    torch.cuda.synchronize()
    assert torch.equal(lp_e, lp_f) and torch.equal(ls_e, ls_f) and torch.equal(dl_e, dl_f)
    assert torch.isfinite(ent).all() and (ent >= -1e-4).all()
    check_entropy(batch["bits"], w.v_real, ent.cpu().numpy()[rows])
    del dl_a, dl_b, dl_e, dl_f, st
    torch.cuda.empty_cache()


def test_vocabulary_shards_full_size(batch):
    """The bench's --split vocab configuration emulated on one GPU: 8 column shards of the 65536 x
    152576 batch (19072 columns each), each through rlk_logp_shard_fwd, the partials stacked as an
    all-gather leaves them, rlk_logp_fold, then rlk_logp_shard_bwd per shard.  logp, LSE and the
    shards' dlogits side by side are bitwise the fused step's."""
    w = batch["w"]
    tp = 8
    vs = w.v_padded // tp
    c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, tp, validate=1)
    dl, logp, lse = rlk.logp_fwd_bwd(c.replace(virtual_tp=BENCH_VTP), batch["logits"], batch["dt"], batch["dm"],
                                     batch["dg"])
    parts, xts = [], []
    for j in range(tp):
        sh = batch["logits"][:, j * vs:(j + 1) * vs].contiguous()
        p, x = rlk.shard_fwd(c, j, sh, batch["dt"], batch["dm"])
        parts.append(p)
        xts.append(x)
        del sh
    logp_s, lse_s = rlk.fold_gathered(c, torch.stack(parts), torch.stack(xts), batch["dt"], batch["dm"])
    torch.cuda.synchronize()
    assert torch.equal(logp_s, logp) and torch.equal(lse_s, lse)
    del parts, xts
    for j in range(tp):
        sh = batch["logits"][:, j * vs:(j + 1) * vs].contiguous()
        d = rlk.shard_bwd(c, j, sh, batch["dt"], batch["dm"], lse_s, batch["dg"])
        torch.cuda.synchronize()
        assert torch.equal(d, dl[:, j * vs:(j + 1) * vs]), j
        del sh, d
