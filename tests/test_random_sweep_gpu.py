"""A seeded random sweep over the contract's shape space, on the GPU.

The other GPU tests pick their shapes by hand.  Here each case draws its own:
the tile count (1 .. 256, odd ones included), the tile width (1 .. 4096
columns), where the real vocabulary ends (in the last tile, a few tiles
earlier, or anywhere), a row stride gap, the mask mode and the fraction of
inactive rows, the logit scale and spikes, planted -inf columns, -inf tiles
and all -inf rows, and one planner override (CTAs per SM, row buffers and
skew, or the resident fused schedule).  Every case checks, at each virtual TP
the tile count allows:

- the forward's logp and LSE against the FP64 oracle (every row);
- the entropy against the oracle, with the forward's logp and LSE bitwise;
- the fused forward + backward's dlogits against the oracle (one BF16
  rounding), bitwise the split backward from the forward's LSE;
- the fused GRPO step bitwise the forward -> loss -> backward composition;
- where the shards start on 16-byte boundaries, each shard read in place from
  the whole buffer and the shards folded: bitwise the whole-vocabulary forward;
- every output bitwise the same across virtual TP and under the override.
"""
import numpy as np
import pytest
import torch

import synth
import vocab_selected_token_tile_gb300 as rlk
from parity import check_dlogits, check_entropy, check_fwd, contract, to_dev

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - the CPU suite deselects this module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

NCASES = 48
MAX_ELEMS = 1_500_000   # T x V_padded per case: the oracle finishes each in well under a second
NEG_INF = 0xFF80
TILE_COUNTS = [1, 2, 3, 4, 5, 6, 7, 8, 12, 16, 24, 32, 40, 64, 96, 128, 256]
OVERRIDES = [{}, {"RLK_CTAS_PER_SM": "1"}, {"RLK_CTAS_PER_SM": "2"}, {"RLK_ROW_BUFS": "2", "RLK_FUSED_SKEW": "1"},
             {"RLK_ROW_BUFS": "4", "RLK_FUSED_SKEW": "0"}, {"RLK_ROW_BUFS": "4", "RLK_FUSED_SKEW": "3"},
             {"RLK_ROW_BUFS": "8", "RLK_FUSED_SKEW": "7"}, {"RLK_FUSED_SCHEDULE": "resident"}]


def draw(i):
    """Case i's shape and inputs, all from default_rng(9000 + i)."""
    rng = np.random.default_rng(9000 + i)
    nt = int(rng.choice(TILE_COUNTS))
    w = int(np.exp(rng.uniform(0.0, np.log(4096.0))))
    while nt * w > MAX_ELEMS:
        w //= 2
    w = max(w, 1)
    vp = nt * w
    end = rng.integers(3)
    if end == 0:                                   # the real end inside the last tile
        vr = int(rng.integers(max(1, vp - w + 1), vp + 1))
    elif end == 1:                                 # a few padding-only tiles
        vr = int(rng.integers(max(1, vp - 3 * w), vp + 1))
    else:
        vr = int(rng.integers(1, vp + 1))
    T = int(min(rng.integers(1, 700), max(1, MAX_ELEMS // vp)))
    stride = (vp + 7) // 8 * 8 + 8 * int(rng.integers(3))
    mode = rlk.MASK_EXPLICIT if rng.random() < 0.5 else rlk.MASK_IGNORE_INDEX
    p_active = float(rng.choice([1.0, 0.7, 0.3, 0.05]))
    sigma = float(rng.choice([0.3, 3.0, 12.0]))
    seed = 9000 + i
    bits = synth.logits_host(0, T, stride, vp, vr, seed=seed, sigma=sigma, nspikes=int(rng.integers(4)),
                             garbage=True)
    tgt = synth.targets(T, vr, seed)
    active = rng.random(T) < p_active
    if rng.random() < 0.5 and T >= 4:              # planted -inf patterns
        r = rng.permutation(T)[:4]
        k = int(rng.integers(2, 9))
        bits[r[0], 1:vr:k] = NEG_INF               # scattered through every tile
        lo = int(rng.integers(nt)) * w
        bits[r[1], lo:min(lo + w, vr)] = NEG_INF   # one whole tile (an identity partial)
        bits[r[2], :vr] = NEG_INF                  # an all -inf row (LSE -inf), kept inactive
        active[r[2]] = False
        for rr in r[:2]:                           # the target column stays finite
            bits[rr, tgt[rr]] = 0x3F80
    if mode == rlk.MASK_EXPLICIT:
        mask = active.astype(np.uint8)
        tgt = np.where(active, tgt, -7 - np.arange(T))  # never read as an index
    else:
        tgt = np.where(active, tgt, -100)
        mask = active.astype(np.uint8)
    g = np.where(active, rng.standard_normal(T), 0.0).astype(np.float32)
    adv = rng.standard_normal(T).astype(np.float32)
    ref = (-4.0 * rng.random(T)).astype(np.float32)
    beta = float(rng.choice([0.0, 0.01]))
    env = OVERRIDES[int(rng.integers(len(OVERRIDES)))]
    return dict(T=T, vr=vr, vp=vp, nt=nt, stride=stride, mode=mode, bits=bits, tgt=tgt, mask=mask,
                active=active, g=g, adv=adv, ref=ref, beta=beta, env=env)


def run_all(k, vtp):
    """Every call of the path at one virtual TP; returns host copies, checked bitwise against each other."""
    c = contract(k["T"], k["vr"], k["vp"], k["nt"], vtp, k["mode"], stride=k["stride"])
    d, dt, dm_u8, dg, dadv = k["dev"]
    dm = dm_u8 if k["mode"] == rlk.MASK_EXPLICIT else None
    dref = k["dref"] if k["beta"] else None
    vp = k["vp"]
    logp, lse = rlk.logp_fwd(c, d, dt, dm)
    lp_e, ls_e, ent = rlk.logp_fwd_entropy(c, d, dt, dm)
    dl, lp_f, ls_f = rlk.logp_fwd_bwd(c, d, dt, dm, dg)
    dl_s = rlk.logp_bwd(c, d, dt, dm, lse, dg)
    out = dict(logp=logp, lse=lse, ent=ent, dl=dl[:, :vp])
    for a, b, what in ((logp, lp_e, "entropy logp"), (lse, ls_e, "entropy lse"), (logp, lp_f, "fused logp"),
                       (lse, ls_f, "fused lse"), (dl[:, :vp], dl_s[:, :vp], "split dlogits")):
        assert torch.equal(a, b), (what, vtp)
    if k.get("grpo", True):
        loss, gr, n = rlk.grpo_loss(logp, dadv, dm_u8, dref, k["beta"])
        dl_c = rlk.logp_bwd(c, d, dt, dm, lse, gr)
        st = rlk.grpo_fused_step(c, d, dt, dm, dadv, dref, k["beta"])
        for key, want in (("logp", logp), ("lse", lse), ("grad", gr), ("loss", loss), ("active_count", n)):
            assert torch.equal(st[key], want), ("grpo " + key, vtp)
        assert torch.equal(st["dlogits"][:, :vp], dl_c[:, :vp]), ("grpo dlogits", vtp)
        out["grpo_dl"] = dl_c[:, :vp]
    vs = vp // vtp
    if vtp > 1 and vs % 8 == 0:
        # each shard read in place from the whole buffer: a shard contract's row_stride is that of the shard's
        # buffer, here the whole row, so shard j's rows end at (T-1)*stride + vp <= T*stride elements
        cs = c.replace(row_stride=k["stride"])
        parts = [rlk.shard_fwd(cs, j, d[:, j * vs:(j + 1) * vs], dt, dm) for j in range(vtp)]
        slogp, slse = rlk.fold_gathered(c, torch.stack([p for p, _ in parts]), torch.stack([x for _, x in parts]),
                                        dt, dm)
        assert torch.equal(slogp, logp) and torch.equal(slse, lse), ("shards folded", vtp)
    torch.cuda.synchronize()
    return {key: t.cpu().numpy() for key, t in out.items()}


def same_bits(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8), np.ascontiguousarray(b).view(np.uint8))


@pytest.mark.parametrize("i", range(NCASES))
def test_random_case(i, monkeypatch):
    k = draw(i)
    T, vr, vp, nt = k["T"], k["vr"], k["vp"], k["nt"]
    k["dev"] = tuple(torch.from_numpy(a).cuda() for a in (k["tgt"], k["mask"], k["g"], k["adv"]))
    k["dev"] = (to_dev(k["bits"]),) + k["dev"]
    k["dref"] = torch.from_numpy(k["ref"]).cuda()
    vtps = [v for v in (1, 2, 4, 8) if nt % v == 0]
    first = None
    for vtp in vtps:
        got = run_all(k, vtp)
        if first is None:
            first = got
            act = k["active"]
            check_fwd(k["bits"][:, :vp], k["tgt"], act, vr, got["logp"], got["lse"])
            check_entropy(k["bits"][:, :vp], vr, got["ent"])
            check_dlogits(k["bits"][:, :vp], k["tgt"], act, k["g"], vr, vp, got["dl"].view(np.uint16))
        else:
            for key in first:
                assert same_bits(first[key], got[key]), (key, vtp)
    # the same batch under the case's planner override (the GRPO step has no resident schedule)
    for name, val in k["env"].items():
        monkeypatch.setenv(name, val)
    k["grpo"] = "RLK_FUSED_SCHEDULE" not in k["env"]
    for vtp in vtps:
        got = run_all(k, vtp)
        for key in got:
            assert same_bits(first[key], got[key]), (key, vtp, k["env"])
    assert T >= 1 and 1 <= vr <= vp
