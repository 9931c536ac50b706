"""A seeded random sweep of the fused lm_head's shapes, on the GPU.

Each case draws its own tile count (1 .. 64), tile width (a multiple of 16
from 16 to 1536 columns, so one to six 256-row weight chunks a tile with a
ragged last chunk of 16 .. 240 rows), where the real vocabulary ends, the
hidden size H (64 .. 512), the token count (1 .. 600, ragged last block), the
mask mode and the fraction of inactive rows.  Every case checks logp and LSE
against the FP64 oracle and bitwise across the virtual TPs the tile count
allows; every other case also runs the backward (dHidden and dW within the
BF16 bound of the FP64 oracle, dW's padded rows exactly 0, bitwise across
virtual TP).
"""
import numpy as np
import pytest
import torch

import synth
import oracle
import vocab_selected_token_tile_gb300 as rlk
from test_lmhead_gpu import close, dev, grad_bounds, make, within

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - the CPU suite deselects this module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

NCASES = 24
MAX_FLOP = 2e9   # T x V_padded x H per case: the FP64 oracle GEMMs finish in well under a second
TILE_COUNTS = [1, 2, 3, 4, 5, 6, 8, 12, 16, 64]
HIDDEN = [64, 128, 192, 256, 320, 512]


def draw(i):
    """Case i's shape and inputs, all from default_rng(7000 + i)."""
    rng = np.random.default_rng(7000 + i)
    nt = int(rng.choice(TILE_COUNTS))
    w = 16 * int(np.exp(rng.uniform(0.0, np.log(96.0))))   # 16 .. 1536 columns
    vp = nt * w
    end = rng.integers(3)
    if end == 0:
        vr = int(rng.integers(max(1, vp - w + 1), vp + 1))
    elif end == 1:
        vr = int(rng.integers(max(1, vp - 3 * w), vp + 1))
    else:
        vr = int(rng.integers(1, vp + 1))
    H = int(rng.choice(HIDDEN))
    T = int(min(rng.integers(1, 600), max(1, MAX_FLOP // (vp * H))))
    mode = rlk.MASK_EXPLICIT if rng.random() < 0.5 else rlk.MASK_IGNORE_INDEX
    p_active = float(rng.choice([1.0, 0.7, 0.2]))
    seed = 7000 + i
    hb, wb = make(T, H, vr, vp, seed=seed, w_sigma=float(rng.choice([0.05, 0.2, 0.6])))
    tgt = synth.targets(T, vr, seed)
    active = rng.random(T) < p_active
    g = np.where(active, rng.standard_normal(T), 0.0).astype(np.float32)
    return dict(T=T, H=H, vr=vr, vp=vp, nt=nt, mode=mode, hb=hb, wb=wb, tgt=tgt, active=active, g=g,
                bwd=(i % 2 == 1))


@pytest.mark.parametrize("i", range(NCASES))
def test_random_lmhead_case(i):
    k = draw(i)
    T, H, vr, vp, nt, act = k["T"], k["H"], k["vr"], k["vp"], k["nt"], k["active"]
    if k["mode"] == rlk.MASK_EXPLICIT:
        tgt_dev = np.where(act, k["tgt"], -12345)  # never read as an index
        mask = torch.from_numpy(act.astype(np.uint8)).cuda()
    else:
        tgt_dev = np.where(act, k["tgt"], -100)
        mask = None
    tgt_or = np.where(act, k["tgt"], 0)
    ref_logp, ref_lse, _ = oracle.lmhead_forward(k["hb"], k["wb"], tgt_or, act, vr)
    if k["bwd"]:
        ref_dh, ref_dw, sc_dh, sc_dw = grad_bounds(k["hb"], k["wb"], tgt_or, act, k["g"], vr)
    dh_, dw_, dt = dev(k["hb"]), dev(k["wb"]), torch.from_numpy(tgt_dev).cuda()
    dg = torch.from_numpy(k["g"]).cuda()
    outs = set()
    for vtp in (v for v in (1, 2, 4, 8) if nt % v == 0):
        c = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=nt, virtual_tp=vtp, mask_mode=k["mode"],
                         validate=1)
        if k["bwd"]:
            logp, lse, dh, dw = rlk.logp_fused_lmhead(c, dh_, dw_, dt, mask, grad=dg)
        else:
            logp, lse = rlk.logp_fused_lmhead(c, dh_, dw_, dt, mask)
        torch.cuda.synchronize()
        lp, ls = logp.cpu().numpy(), lse.cpu().numpy()
        close("lse", ls, ref_lse)
        if act.any():
            close("logp", lp[act], ref_logp[act])
        assert np.all(lp[~act].view(np.uint32) == 0), "inactive rows must be exactly +0.0"
        key = [lp.tobytes(), ls.tobytes()]
        if k["bwd"]:
            dhb, dwb = dh.cpu().numpy().view(np.uint16), dw.cpu().numpy().view(np.uint16)
            assert np.all(within(dhb, ref_dh, sc_dh))
            assert np.all(within(dwb[:vr], ref_dw, sc_dw)) and np.all(dwb[vr:] == 0)
            key += [dhb.tobytes(), dwb.tobytes()]
        outs.add(tuple(key))
    assert len(outs) == 1, "virtual TP outputs differ"
