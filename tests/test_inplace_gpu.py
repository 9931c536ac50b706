"""dlogits written over the logits they come from (in place), on the GPU.

The backward may take dlogits == logits: every logit is read before its
gradient overwrites it (phase A of a row ends before the row's LSE exists,
and a tile's gradient is written after its own copy is read; halo columns a
copy shares with a neighbouring tile are read but never used).  The in-place
result must be bitwise the out-of-place one over columns [0, V_padded), for
the fused L2 schedule at one or two CTAs per SM, the resident schedule, the
split backward given the LSE, the fused step with entropy and the
vocabulary-shard backward, at every virtual TP, on ragged shapes.  Columns
beyond V_padded (the stride gap) keep the logits' bytes.  Nothing here is
compared with the oracle: the out-of-place outputs are (test_parity_gpu).
"""
import numpy as np
import pytest
import torch

import synth
import vocab_selected_token_tile_gb300 as rlk
from parity import contract, to_dev

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

# (T, V_real, V_padded, num_tiles, extra stride columns)
CASES = [
    (5, 37, 40, 4, 0),            # tile width 10: unaligned tiles, ragged real end
    (17, 3001, 3072, 64, 0),      # ragged real end inside the last tile
    (33, 1000, 1024, 64, 8),      # padding-only tiles, stride gap
    (40, 151936, 151936, 64, 0),  # 2374-column tiles: halo groups shared by neighbouring tiles
    (9, 151936, 152576, 64, 1),   # the Qwen3 padded shape with a stride gap
    (6, 32765, 32768, 2, 0),      # widest tile
    (2, 7, 7, 7, 1),              # V_padded not a multiple of 8
]


def inputs(T, vr, vp, nt, extra, seed):
    stride = ((vp + 7) // 8) * 8 + 8 * extra
    bits = synth.logits_host(0, T, stride, vp, vr, seed=seed, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, vr, seed)
    rng = np.random.default_rng(seed)
    mask = (rng.random(T) < 0.7).astype(np.uint8)
    mask[0] = 1
    tgt = np.where(mask != 0, tgt, -7)
    tgt[0] = vr - 1  # a target in the ragged real tail
    g = np.where(mask != 0, rng.standard_normal(T), 0.0).astype(np.float32)
    return stride, to_dev(bits), (torch.from_numpy(a).cuda() for a in (tgt, mask, g))


def same_grad(inplace, ref, vp):
    assert torch.equal(inplace[:, :vp], ref[:, :vp])


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T%d_V%d_P%d_NT%d_x%d" % c)
def test_inplace_equals_out_of_place(case, monkeypatch):
    T, vr, vp, nt, extra = case
    stride, logits, (dt, dm, dg) = inputs(T, vr, vp, nt, extra, seed=T * 7 + nt)
    for vtp in (v for v in (1, 2, 4, 8) if nt % v == 0):
        c = contract(T, vr, vp, nt, vtp, rlk.MASK_EXPLICIT, stride=stride)
        dl, logp, lse = rlk.logp_fwd_bwd(c, logits, dt, dm, dg)
        for per_sm in ("1", "2"):
            monkeypatch.setenv("RLK_CTAS_PER_SM", per_sm)
            buf = logits.clone()
            _, lp, ls = rlk.logp_fwd_bwd(c, buf, dt, dm, dg, dlogits=buf)
            same_grad(buf, dl, vp)
            assert torch.equal(buf[:, vp:], logits[:, vp:])  # the stride gap keeps the logits
            assert torch.equal(lp, logp) and torch.equal(ls, lse)
            buf = logits.clone()
            _, lp, ls, ent = rlk.logp_fwd_bwd_entropy(c, buf, dt, dm, dg, dlogits=buf)
            same_grad(buf, dl, vp)
            assert torch.equal(lp, logp) and torch.equal(ls, lse)
        monkeypatch.delenv("RLK_CTAS_PER_SM")
        monkeypatch.setenv("RLK_FUSED_SCHEDULE", "resident")
        buf = logits.clone()
        _, lp, ls = rlk.logp_fwd_bwd(c, buf, dt, dm, dg, dlogits=buf)
        same_grad(buf, dl, vp)
        assert torch.equal(lp, logp) and torch.equal(ls, lse)
        monkeypatch.delenv("RLK_FUSED_SCHEDULE")
        # the split backward from the forward's LSE
        buf = logits.clone()
        rlk.logp_bwd(c, buf, dt, dm, lse, dg, dlogits=buf)
        same_grad(buf, dl, vp)
    torch.cuda.synchronize()


def test_inplace_qwen3_shape_and_shards():
    """The Qwen3-shaped batch (4096 rows: many rows per CTA, the ring wraps) in place at virtual TP 1, 2
    and 8, and the tp = 4 vocabulary-shard backward in place on each shard's own buffer."""
    from synth import workloads as W
    w = W.QWEN3
    bits = W.logits_host(w)
    tgt = W.targets(w)
    g = W.grad(w, tgt != w.ignore_index)
    logits = to_dev(bits)
    dt, dg = torch.from_numpy(tgt).cuda(), torch.from_numpy(g).cuda()
    for vtp in (1, 2, 8):
        c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, vtp, rlk.MASK_IGNORE_INDEX)
        dl, logp, lse = rlk.logp_fwd_bwd(c, logits, dt, None, dg)
        buf = logits.clone()
        _, lp, ls = rlk.logp_fwd_bwd(c, buf, dt, None, dg, dlogits=buf)
        assert torch.equal(buf, dl) and torch.equal(lp, logp) and torch.equal(ls, lse), vtp
        del buf
    tp = 4
    vs = w.v_padded // tp
    cs = contract(w.T, w.v_real, w.v_padded, w.num_tiles, tp, rlk.MASK_IGNORE_INDEX)
    for j in range(tp):
        sh = logits[:, j * vs:(j + 1) * vs].contiguous()
        want = rlk.shard_bwd(cs, j, sh, dt, None, lse, dg)
        rlk.shard_bwd(cs, j, sh, dt, None, lse, dg, dlogits=sh)
        assert torch.equal(sh, want), j
        assert torch.equal(sh, dl[:, j * vs:(j + 1) * vs]), j
    torch.cuda.synchronize()
