"""The fused single-pass forward+backward with each row's entropy (rlk_logp_fwd_bwd_entropy).

Its dlogits, logp and LSE must be bitwise those of the fused step (rlk_logp_bwd with lse_in =
NULL), and its entropy bitwise that of the forward's (rlk_logp_fwd_entropy), at every virtual TP;
the entropy is also checked against the FP64 oracle.
"""
import numpy as np
import pytest
import torch

import synth
import vocab_selected_token_tile_gb300 as rlk
from parity import check_entropy, contract, to_dev
from test_parity_gpu import SMALL, make_inputs, sha, vtps

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "T%d_V%d_P%d_NT%d_x%d" % c)
def test_fused_entropy_small_cases(case):
    T, v_real, v_padded, nt, extra = case
    stride, bits, tgt, mask, active, g = make_inputs(T, v_real, v_padded, nt, extra, seed=T * 11 + nt)
    dlog = to_dev(bits)
    dt, dm, dg = torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda(), torch.from_numpy(g).cuda()
    shas = set()
    for vtp in vtps(nt):
        c = contract(T, v_real, v_padded, nt, vtp, rlk.MASK_EXPLICIT, stride)
        dl_e, logp_e, lse_e, ent = rlk.logp_fwd_bwd_entropy(c, dlog, dt, dm, dg,
                                                           dlogits=torch.full_like(dlog, 0x7E7E))
        dl, logp, lse = rlk.logp_fwd_bwd(c, dlog, dt, dm, dg, dlogits=torch.full_like(dlog, 0x7E7E))
        _, _, ent_f = rlk.logp_fwd_entropy(c, dlog, dt, dm)
        torch.cuda.synchronize()
        assert torch.equal(dl_e, dl) and torch.equal(logp_e, logp) and torch.equal(lse_e, lse)
        assert torch.equal(ent, ent_f)
        check_entropy(bits, v_real, ent.cpu().numpy())
        shas.add((sha(ent), sha(dl_e)))
    assert len(shas) == 1, "virtual TP outputs differ"


def test_fused_entropy_qwen3_shape_and_special_rows(monkeypatch):
    from synth import workloads as W
    v_real, v_padded, nt = 1000, 1024, 64
    bits = synth.logits_host(0, 5, v_padded, v_padded, v_real, seed=9, sigma=2.0)
    bits[1, :v_real] = 0xFF80          # all -inf: NaN entropy
    bits[2, :v_real] = 0xFF80
    bits[2, 500] = 0x3F80              # one finite column: entropy 0
    bits[3, 3:v_real:7] = 0xFF80       # -inf logits scattered among finite ones, in every tile
    bits[4, 640:656] = 0xFF80          # one whole tile -inf beside finite tiles
    tg = torch.full((5,), -100, dtype=torch.int64).cuda()
    for vtp in (1, 2, 8):
        c = contract(5, v_real, v_padded, nt, vtp, rlk.MASK_IGNORE_INDEX, validate=0)
        _, _, lse, ent = rlk.logp_fwd_bwd_entropy(c, to_dev(bits), tg, None, torch.zeros(5).cuda())
        _, _, e0 = rlk.logp_fwd_entropy(c, to_dev(bits), tg)
        torch.cuda.synchronize()
        e = ent.cpu().numpy()
        assert np.isnan(e[1]) and e[2] == 0.0 and np.all(np.isfinite(e[[0, 3, 4]]))
        check_entropy(bits, v_real, e)
        assert np.array_equal(e.view(np.uint32), e0.cpu().numpy().view(np.uint32)), vtp

    w = W.QWEN3
    qbits = W.logits_host(w)
    dq = to_dev(qbits)
    tgt = W.targets(w)
    dt = torch.from_numpy(tgt).cuda()
    dg = torch.from_numpy(W.grad(w, tgt != w.ignore_index)).cuda()
    ref = None
    for per_sm in ("1", "2"):
        monkeypatch.setenv("RLK_CTAS_PER_SM", per_sm)
        for vtp in (1, 2, 4, 8):
            cq = contract(w.T, w.v_real, w.v_padded, w.num_tiles, vtp, rlk.MASK_IGNORE_INDEX)
            dl, logp, lse, eq = rlk.logp_fwd_bwd_entropy(cq, dq, dt, None, dg)
            torch.cuda.synchronize()
            got = (sha(dl), sha(logp), sha(lse), sha(eq))
            if ref is None:
                ref = got
                check_entropy(qbits, w.v_real, eq.cpu().numpy(), rows=np.arange(0, w.T, 13))
                dl0, logp0, lse0 = rlk.logp_fwd_bwd(cq, dq, dt, None, dg)
                _, _, e0 = rlk.logp_fwd_entropy(cq, dq, dt)
                torch.cuda.synchronize()
                assert got == (sha(dl0), sha(logp0), sha(lse0), sha(e0))
            assert got == ref, (per_sm, vtp)
    monkeypatch.setenv("RLK_FUSED_SCHEDULE", "resident")
    with pytest.raises(rlk.RlkError) as ei:
        rlk.logp_fwd_bwd_entropy(contract(w.T, w.v_real, w.v_padded, w.num_tiles, 2, rlk.MASK_IGNORE_INDEX),
                                 dq, dt, None, dg)
    assert ei.value.status == rlk.RLK_ERR_UNSUPPORTED
