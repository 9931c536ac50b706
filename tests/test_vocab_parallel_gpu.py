"""Vocabulary-parallel shard calls on one GPU: tp shards emulated in one process.

Each shard j of tp is cut out of the logits into a buffer of its own
(columns [j*Vs, (j+1)*Vs)), rlk_logp_shard_fwd runs on it, the partials and
target logits are stacked shard-major (what an all-gather leaves), and
rlk_logp_fold folds them.  logp and LSE must be bitwise those of
rlk_logp_fwd on the whole vocabulary (SHA-256), the stacked partials bitwise
the whole row's, and the shards' rlk_logp_shard_bwd outputs, side by side,
bitwise rlk_logp_bwd's dlogits -- for tp = 1, 2, 4, 8.
"""
import hashlib

import numpy as np
import pytest
import torch

import oracle
import synth
import vocab_selected_token_tile_gb300 as rlk

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def sha(t):
    return hashlib.sha256(t.contiguous().cpu().numpy().tobytes()).hexdigest()


def emulate(c, logits, targets, mask, grad, lse_whole, stride_pad=0):
    """(logp, lse, stacked partials [T, NT, 2], dlogits [T, V_padded]) from tp shard calls."""
    tp = c.virtual_tp
    vs = c.V_padded // tp
    parts, xts, dls = [], [], []
    for j in range(tp):
        sh = torch.zeros((c.T, vs + stride_pad), dtype=torch.int16, device="cuda")
        sh[:, :vs] = logits[:, j * vs:(j + 1) * vs]
        cj = c.replace(row_stride=vs + stride_pad if stride_pad else 0)
        p, x = rlk.shard_fwd(cj, j, sh, targets, mask)
        parts.append(p)
        xts.append(x)
        d = torch.full_like(sh, 0x7E7E)
        rlk.shard_bwd(cj, j, sh, targets, mask, lse_whole, grad, dlogits=d)
        if stride_pad:
            assert (d[:, vs:] == 0x7E7E).all()  # columns beyond the shard are not touched
        dls.append(d[:, :vs])
    gathered = torch.stack(parts)
    gathered_xt = torch.stack(xts)
    logp, lse = rlk.fold_gathered(c, gathered, gathered_xt, targets, mask)
    return logp, lse, torch.cat(parts, dim=1), torch.cat(dls, dim=1)


def test_qwen3_shards_reproduce_the_whole_vocabulary_bitwise():
    from synth import workloads as W
    w = W.QWEN3
    bits = W.logits_host(w)
    tgt = W.targets(w)
    active = tgt != w.ignore_index
    g = W.grad(w, active)
    logits = torch.from_numpy(bits.view(np.int16)).cuda()
    dt, dg = torch.from_numpy(tgt).cuda(), torch.from_numpy(g).cuda()
    c1 = rlk.Contract(T=w.T, V_real=w.v_real, V_padded=w.v_padded, num_tiles=w.num_tiles, virtual_tp=1,
                      mask_mode=rlk.MASK_IGNORE_INDEX, validate=1)
    logp, lse, part = rlk.logp_fwd(c1, logits, dt, partials=True)
    dl = rlk.logp_bwd(c1, logits, dt, None, lse, dg)
    torch.cuda.synchronize()
    want = (sha(logp), sha(lse), sha(part), sha(dl))
    assert np.max(np.abs(lse.cpu().numpy()[:256] - oracle.lse_full(bits[:256], w.v_real))) <= 1e-4
    for tp in (1, 2, 4, 8):
        c = c1.replace(virtual_tp=tp)
        got = emulate(c, logits, dt, None, dg, lse)
        torch.cuda.synchronize()
        assert (sha(got[0]), sha(got[1]), sha(got[2]), sha(got[3])) == want, tp


# (T, V_real, V_padded, num_tiles, tp, stride_pad): ragged real tails, shards of padding only, wide tiles
CASES = [
    (37, 1000, 1024, 8, 2, 0),
    (50, 100, 1024, 8, 8, 8),      # shards 1..7 hold padding only: identity partials, zero dlogits
    (33, 5000, 2376 * 4, 8, 4, 0),  # 1188-wide tiles: tile ends not on 8-column groups
    (20, 6000, 6144, 2, 2, 16),    # one 3072-column tile per shard
    (64, 16383, 16384, 64, 8, 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T%d_V%d_P%d_NT%d_tp%d_pad%d" % c)
def test_small_shards_are_bitwise_the_whole(case):
    T, vr, vp, nt, tp, pad = case
    bits = synth.logits_host(0, T, vp, vp, vr, seed=T + tp, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, vr, seed=T)
    mask = (np.arange(T) % 5 != 2).astype(np.uint8)
    tgt = np.where(mask != 0, tgt, -12345)  # poison on inactive rows: never used as an index
    tgt[np.nonzero(mask)[0][:3]] = [0, vr - 1, vr // 2]
    g = np.where(mask != 0, np.random.default_rng(T).standard_normal(T), 0.0).astype(np.float32)
    logits = torch.from_numpy(bits.view(np.int16)).cuda()
    dt, dm, dg = (torch.from_numpy(a).cuda() for a in (tgt, mask, g))
    c1 = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=nt, virtual_tp=1, validate=1)
    logp, lse, part = rlk.logp_fwd(c1, logits, dt, dm, partials=True)
    dl = rlk.logp_bwd(c1, logits, dt, dm, lse, dg)
    torch.cuda.synchronize()
    act = mask != 0
    ref_logp, ref_lse = oracle.selected_logp(bits, np.where(act, tgt, 0), act, vr)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= 1e-4
    got = emulate(c1.replace(virtual_tp=tp), logits, dt, dm, dg, lse, stride_pad=pad)
    torch.cuda.synchronize()
    assert torch.equal(got[0], logp) and torch.equal(got[1], lse)
    assert torch.equal(got[2], part)
    assert torch.equal(got[3], dl)
    assert (got[0][~torch.from_numpy(act).cuda()] == 0).all()


def test_shard_calls_fail_closed():
    T, vr, vp = 16, 1000, 1024
    c = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=8, virtual_tp=2, validate=1)
    assert rlk.rlk_logp_check_shard_contract(c, 2) == rlk.RLK_ERR_INVALID_ARG  # shard out of range
    assert rlk.rlk_logp_check_shard_contract(c, -1) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_check_shard_contract(c.replace(row_stride=500), 0) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_check_shard_contract(c.replace(row_stride=516), 0) == rlk.RLK_ERR_MISALIGNED
    c8 = rlk.Contract(T=T, V_real=100, V_padded=8 * 20, num_tiles=8, virtual_tp=8)  # Vs = 20: not 16-byte
    assert rlk.rlk_logp_check_shard_contract(c8, 0) == rlk.RLK_ERR_MISALIGNED
    # an active target outside [0, V_real) is reported by the fold and by the shard backward
    logits = torch.zeros((T, vp), dtype=torch.int16, device="cuda")
    tgt = torch.zeros(T, dtype=torch.int64, device="cuda")
    tgt[3] = vr + 2
    m = torch.ones(T, dtype=torch.uint8, device="cuda")
    sh = logits[:, :512].contiguous()
    p0, x0 = rlk.shard_fwd(c, 0, sh, tgt, m)
    p1, x1 = rlk.shard_fwd(c, 1, logits[:, 512:].contiguous(), tgt, m)
    with pytest.raises(rlk.RlkError) as ei:
        rlk.fold_gathered(c, torch.stack([p0, p1]), torch.stack([x0, x1]), tgt, m)
    assert ei.value.status == rlk.RLK_ERR_TARGET_RANGE
    with pytest.raises(rlk.RlkError) as ei:
        rlk.shard_bwd(c, 0, sh, tgt, m, torch.zeros(T, device="cuda"), torch.ones(T, device="cuda"))
    assert ei.value.status == rlk.RLK_ERR_TARGET_RANGE


def test_layer_over_a_one_rank_nccl_group():
    """VocabParallelLogp with a real NCCL group of one rank (tp = 1): the agreement all-reduce and the
    all-gather run on the GPU, and logp, LSE and dlogits are bitwise those of rlk_logp_fwd / rlk_logp_bwd."""
    import os
    import socket

    import torch.distributed as dist
    from vocab_selected_token_tile_gb300.vocab_parallel import VocabParallelLogp
    T, vr, vp, nt = 96, 3001, 3072, 64
    bits = synth.logits_host(0, T, vp, vp, vr, seed=77, sigma=3.0, garbage=True)
    tgt = synth.targets(T, vr, seed=77)
    mask = (np.arange(T) % 3 != 0).astype(np.uint8)
    g = np.where(mask != 0, 0.5, 0.0).astype(np.float32)
    logits = torch.from_numpy(bits.view(np.int16)).cuda()
    dt, dm, dg = (torch.from_numpy(a).cuda() for a in (tgt, mask, g))
    c = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=nt, virtual_tp=1, validate=1)
    want_logp, want_lse = rlk.logp_fwd(c, logits, dt, dm)
    want_dl = rlk.logp_bwd(c, logits, dt, dm, want_lse, dg)
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        layer = VocabParallelLogp(c)
        logp, lse = layer.forward(logits, dt, dm)
        dl = layer.backward(logits, dt, dm, lse, dg)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert torch.equal(logp, want_logp) and torch.equal(lse, want_lse) and torch.equal(dl, want_dl)
