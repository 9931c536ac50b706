"""Many short rows: every CTA runs hundreds of rows, so the slot ring, the row
buffers, the tile rotation and (at virtual TP 8, one tile per CTA and row)
the row skip of the forward wrap around many times.  All rows of every output
are compared with the FP64 oracle; outputs are bitwise equal across virtual
TP and between the fused, split and entropy paths."""
import numpy as np
import pytest
import torch

import oracle
import synth
import vocab_selected_token_tile_gb300 as rlk
from parity import ENT_TOL, LSE_TOL, contract, f32_bits, to_dev

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - the CPU suite deselects this module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def test_many_short_rows_all_paths_all_virtual_tp():
    T, v_real, v_padded, nt = 131072 + 37, 61, 64, 8
    bits = synth.logits_host(0, T, v_padded, v_padded, v_real, seed=29, sigma=3.0, nspikes=1, garbage=True)
    tgt = synth.targets(T, v_real, 29)
    rng = np.random.default_rng(29)
    mask = (rng.random(T) < 0.6).astype(np.uint8)
    active = mask != 0
    g = np.where(active, rng.standard_normal(T), 0.0).astype(np.float32)

    ref_logp, ref_lse = oracle.selected_logp(bits, tgt, active, v_real)
    ref_ent = oracle.entropy(bits, v_real)
    ref_dl = oracle.dlogits(bits, tgt, active, g, v_real, v_padded)

    d = to_dev(bits)
    dt, dm, dg = (torch.from_numpy(a).cuda() for a in (tgt, mask, g))
    first = None
    for vtp in (1, 2, 4, 8):
        c = contract(T, v_real, v_padded, nt, vtp)
        logp, lse = rlk.logp_fwd(c, d, dt, dm)
        lp_e, ls_e, ent = rlk.logp_fwd_entropy(c, d, dt, dm)
        dl, lp_f, ls_f = rlk.logp_fwd_bwd(c, d, dt, dm, dg)
        dl_s = rlk.logp_bwd(c, d, dt, dm, lse, dg)
        torch.cuda.synchronize()
        outs = [t.cpu().numpy() for t in (logp, lse, ent, dl)]
        for a, b in ((logp, lp_e), (lse, ls_e), (logp, lp_f), (lse, ls_f), (dl, dl_s)):
            assert torch.equal(a, b), vtp
        if first is None:
            first = outs
            lp, ls, en, dlb = outs
            assert np.max(np.abs(ls - ref_lse)) <= LSE_TOL
            assert np.max(np.abs(lp[active] - ref_logp[active])) <= LSE_TOL
            assert np.all(f32_bits(lp[~active]) == 0)
            assert np.max(np.abs(en - ref_ent)) <= ENT_TOL
            got = oracle.bf16_bits_to_f64(dlb.view(np.uint16)[:, :v_padded])
            err = np.abs(got - ref_dl)
            assert np.all(err <= np.ldexp(np.abs(ref_dl), -8) + 4e-6 * np.abs(g)[:, None] + 1e-30)
            assert not dlb.view(np.uint16)[:, v_real:].any() and not dlb.view(np.uint16)[~active].any()
        else:
            for a, b in zip(first, outs):
                assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), vtp


def test_many_short_rows_every_planner_choice_gives_the_same_bits(monkeypatch):
    """The same many-row batch under every planner override (one or two CTAs per SM,
    2/4/8 row buffers, row skew 0-2, the resident fused schedule): bitwise the
    default outputs at every virtual TP."""
    T, v_real, v_padded, nt = 65536 + 11, 61, 64, 8
    bits = synth.logits_host(0, T, v_padded, v_padded, v_real, seed=31, sigma=3.0, nspikes=1, garbage=True)
    tgt = synth.targets(T, v_real, 31)
    rng = np.random.default_rng(31)
    mask = (rng.random(T) < 0.6).astype(np.uint8)
    g = np.where(mask != 0, rng.standard_normal(T), 0.0).astype(np.float32)
    d = to_dev(bits)
    dt, dm, dg = (torch.from_numpy(a).cuda() for a in (tgt, mask, g))

    def run(vtp):
        c = contract(T, v_real, v_padded, nt, vtp)
        logp, lse = rlk.logp_fwd(c, d, dt, dm)
        _, _, ent = rlk.logp_fwd_entropy(c, d, dt, dm)
        dl, lp_f, ls_f = rlk.logp_fwd_bwd(c, d, dt, dm, dg)
        dl_s = rlk.logp_bwd(c, d, dt, dm, lse, dg)
        torch.cuda.synchronize()
        return [t.cpu().numpy().view(np.uint8) for t in (logp, lse, ent, dl, lp_f, ls_f, dl_s)]

    ref = run(1)
    variants = [{"RLK_CTAS_PER_SM": "1"}, {"RLK_CTAS_PER_SM": "2"}, {"RLK_ROW_BUFS": "2"}, {"RLK_ROW_BUFS": "8"},
                {"RLK_FUSED_SKEW": "0"}, {"RLK_FUSED_SKEW": "2"}, {"RLK_FUSED_SCHEDULE": "resident"}]
    for env in [{}] + variants:
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        for vtp in (1, 2, 4, 8):
            got = run(vtp)
            for i, (a, b) in enumerate(zip(ref, got)):
                assert np.array_equal(a, b), (env, vtp, i)
        for k in env:
            monkeypatch.delenv(k)


# (T, V_real, V_padded, num_tiles): the widest tiles (16384 columns, one per copy), the most
# tiles (1024 of 8 columns, a 48 KB per-tile table), and an odd tile count
SHAPES = [(3001, 32765, 32768, 2), (16384 + 5, 8190, 8192, 1024), (20000 + 3, 6997, 7007, 7)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "T%d_V%d_P%d_NT%d" % s)
def test_many_rows_at_extreme_tile_shapes(shape):
    T, v_real, v_padded, nt = shape
    stride = (v_padded + 7) // 8 * 8
    bits = synth.logits_host(0, T, stride, v_padded, v_real, seed=37, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, v_real, 37, ignore_frac=0.2)
    active = tgt != -100
    g = np.where(active, np.random.default_rng(37).standard_normal(T), 0.0).astype(np.float32)
    d = to_dev(bits)
    dt, dg = torch.from_numpy(tgt).cuda(), torch.from_numpy(g).cuda()
    rows = np.unique(np.concatenate([np.arange(0, T, max(1, T // 600)), [T - 1]]))
    ref_logp, ref_lse = oracle.selected_logp(bits[rows], tgt[rows], active[rows], v_real)
    first = None
    for vtp in [v for v in (1, 2, 4, 8) if nt % v == 0]:
        c = contract(T, v_real, v_padded, nt, vtp, rlk.MASK_IGNORE_INDEX, stride=stride)
        logp, lse = rlk.logp_fwd(c, d, dt)
        dl, lp_f, ls_f = rlk.logp_fwd_bwd(c, d, dt, None, dg)
        dl_s = rlk.logp_bwd(c, d, dt, None, lse, dg)
        torch.cuda.synchronize()
        # columns [V_padded, row_stride) of dlogits are not written (the caller's memory)
        dl, dl_s = dl[:, :v_padded], dl_s[:, :v_padded]
        assert torch.equal(logp, lp_f) and torch.equal(lse, ls_f) and torch.equal(dl, dl_s), vtp
        out = [t.cpu().numpy() for t in (logp, lse, dl)]
        if first is None:
            first = out
            lp, ls, dlb = out
            assert np.max(np.abs(ls[rows] - ref_lse)) <= LSE_TOL
            a = active[rows]
            assert np.max(np.abs(lp[rows][a] - ref_logp[a])) <= LSE_TOL
            assert np.all(f32_bits(lp[~active]) == 0)
            sub = rows[:64]
            ref_dl = oracle.dlogits(bits[sub], tgt[sub], active[sub], g[sub], v_real, v_padded)
            got = oracle.bf16_bits_to_f64(dlb.view(np.uint16)[sub])
            assert np.all(np.abs(got - ref_dl) <= np.ldexp(np.abs(ref_dl), -8) + 4e-6 * np.abs(g[sub])[:, None] + 1e-30)
            assert not dlb.view(np.uint16)[:, v_real:v_padded].any() and not dlb.view(np.uint16)[~active].any()
        else:
            for x, y in zip(first, out):
                assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), vtp
