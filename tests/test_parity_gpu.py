"""Parity of the CUDA path with the FP64 oracle, through the C ABI, on the GPU.

Small cases span several tiles, ragged real/padded edges, unaligned tile
widths, padding-only tiles and the largest supported tile and tile count;
they are compared element by element.  Tolerances: LSE and logp max abs
<= 1e-4; dlogits max abs <= 1e-2 and within one BF16 rounding of the FP64
value; masking, padding and indexing bit-exact; outputs bitwise identical
across virtual TP 1/2/4/8 and between the fused and split backward.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import vocab_selected_token_tile_gb300 as rlk
from parity import (check_dlogits, check_entropy, check_fwd, contract, f32_bits, sha, to_dev)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - the CPU suite deselects this module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

# (T, V_real, V_padded, num_tiles, extra stride columns)
SMALL = [
    (1, 1, 8, 1, 0),            # one real column
    (5, 37, 40, 4, 0),          # tile width 10: unaligned tiles, ragged real end
    (33, 1000, 1024, 64, 8),    # tile 63 is padding only; stride gap
    (17, 3001, 3072, 64, 0),    # ragged real end inside the last tile
    (64, 5003, 5120, 8, 16),
    (40, 151936, 151936, 64, 0),  # tile width 2374 (4748 B): tiles not 16-byte aligned
    (9, 151936, 152576, 64, 0),   # the Qwen3 padded shape
    (6, 32765, 32768, 2, 0),      # widest supported tile (16384 columns)
    (3, 300, 1024, 1024, 0),      # 1024 tiles of width 1, most padding only
    (7, 20, 24, 3, 0),            # three tiles of 8
    (2, 7, 7, 7, 1),              # V_padded not a multiple of 8 (stride 8)
]


def make_inputs(T, v_real, v_padded, nt, extra, seed, mode=rlk.MASK_EXPLICIT):
    stride = ((v_padded + 7) // 8) * 8 + 8 * extra
    bits = synth.logits_host(0, T, stride, v_padded, v_real, seed=seed, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, v_real, seed, ignore_frac=0.25 if mode == rlk.MASK_IGNORE_INDEX else 0.0)
    rng = np.random.default_rng(seed)
    if mode == rlk.MASK_EXPLICIT:
        mask = (rng.random(T) < 0.7).astype(np.uint8)
        if T:
            mask[0] = 1
        poison = np.array([-7, v_padded + 5, 1 << 62, -(1 << 62)])
        tgt = np.where(mask != 0, tgt, poison[np.arange(T) % 4])  # never read as indices
        active = mask != 0
    else:
        mask = None
        active = tgt != -100
    g = np.where(active, rng.standard_normal(T), 0.0).astype(np.float32)
    return stride, bits, tgt, mask, active, g


def vtps(nt):
    return [v for v in (1, 2, 4, 8) if nt % v == 0]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "T%d_V%d_P%d_NT%d" % c[:4])
@pytest.mark.parametrize("mode", [rlk.MASK_EXPLICIT, rlk.MASK_IGNORE_INDEX], ids=["explicit", "ignore"])
def test_small_cases_all_paths(case, mode):
    T, v_real, v_padded, nt, extra = case
    stride, bits, tgt, mask, active, g = make_inputs(T, v_real, v_padded, nt, extra, seed=T * 131 + nt, mode=mode)
    dlog = to_dev(bits)
    dt = torch.from_numpy(tgt).cuda()
    dm = torch.from_numpy(mask).cuda() if mask is not None else None
    dg = torch.from_numpy(g).cuda()
    m_ref, s_ref = oracle.tile_partials(bits, v_real, v_padded, nt)
    outs = {}
    for vtp in vtps(nt):
        c = contract(T, v_real, v_padded, nt, vtp, mode, stride)
        logp, lse, part = rlk.logp_fwd(c, dlog, dt, dm, partials=True)
        torch.cuda.synchronize()
        check_fwd(bits, tgt, active, v_real, logp.cpu().numpy(), lse.cpu().numpy())
        part = part.cpu().numpy().astype(np.float64)
        # tile maxima are exact; sums within 1e-5 relative
        assert np.array_equal(part[..., 0], m_ref.astype(np.float32).astype(np.float64))
        fin = np.isfinite(s_ref) & (s_ref > 0)
        assert np.all(np.abs(part[..., 1][fin] - s_ref[fin]) <= 1e-5 * s_ref[fin])
        assert np.all(part[..., 1][m_ref == -np.inf] == 0.0)
        # backward, split and fused
        sentinel = torch.full_like(dlog, 0x7E7E)
        dl_split = rlk.logp_bwd(c, dlog, dt, dm, lse, dg, dlogits=sentinel.clone())
        dl_fused, logp2, lse2 = rlk.logp_fwd_bwd(c, dlog, dt, dm, dg, dlogits=sentinel.clone())
        torch.cuda.synchronize()
        assert torch.equal(dl_split, dl_fused)
        assert torch.equal(logp2, logp) and torch.equal(lse2, lse)
        dl_bits = dl_fused.cpu().numpy().view(np.uint16)
        check_dlogits(bits, tgt, active, g, v_real, v_padded, dl_bits)
        assert np.all(dl_bits[:, v_padded:] == 0x7E7E), "columns beyond V_padded must not be written"
        outs[vtp] = (sha(logp), sha(lse), sha(dl_fused))
    assert len(set(outs.values())) == 1, "virtual TP outputs differ"


def test_ignore_index_equals_explicit_mask():
    T, v_real, v_padded, nt = 96, 151936, 152576, 64
    _, bits, tgt, _, active, _ = make_inputs(T, v_real, v_padded, nt, 0, seed=5, mode=rlk.MASK_IGNORE_INDEX)
    dlog = to_dev(bits)
    mask = active.astype(np.uint8)
    a = rlk.logp_fwd(contract(T, v_real, v_padded, nt, 4, rlk.MASK_IGNORE_INDEX), dlog,
                     torch.from_numpy(tgt).cuda())
    b = rlk.logp_fwd(contract(T, v_real, v_padded, nt, 2, rlk.MASK_EXPLICIT), dlog,
                     torch.from_numpy(np.where(active, tgt, 123)).cuda(), torch.from_numpy(mask).cuda())
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_workload_tiny():
    from synth import workloads as W
    w = W.TINY
    bits = W.logits_host(w)
    tgt = W.targets(w)
    mask = W.active_mask(w)
    active = mask != 0
    g = W.grad(w, active)
    dlog = to_dev(bits)
    dt, dm, dg = (torch.from_numpy(a).cuda() for a in (tgt, mask, g))
    shas = set()
    for vtp in (1, 2, 4, 8):
        c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, vtp)
        dl, logp, lse = rlk.logp_fwd_bwd(c, dlog, dt, dm, dg)
        torch.cuda.synchronize()
        check_fwd(bits, tgt, active, w.v_real, logp.cpu().numpy(), lse.cpu().numpy())
        check_dlogits(bits, tgt, active, g, w.v_real, w.v_padded, dl.cpu().numpy().view(np.uint16))
        shas.add((sha(logp), sha(lse)))
    assert len(shas) == 1


def test_workload_qwen3_all_rows_and_vtp_sha():
    from synth import workloads as W
    w = W.QWEN3
    bits = W.logits_host(w)
    tgt = W.targets(w)
    active = tgt != w.ignore_index
    g = W.grad(w, active)
    dlog = to_dev(bits)
    dt, dg = torch.from_numpy(tgt).cuda(), torch.from_numpy(g).cuda()
    shas = {}
    for vtp in (1, 2, 4, 8):
        c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, vtp, rlk.MASK_IGNORE_INDEX)
        logp, lse = rlk.logp_fwd(c, dlog, dt)
        torch.cuda.synchronize()
        shas[vtp] = (sha(logp), sha(lse))
        if vtp == 1:
            check_fwd(bits, tgt, active, w.v_real, logp.cpu().numpy(), lse.cpu().numpy())
            dl = rlk.logp_bwd(c, dlog, dt, None, lse, dg)
            dl_bits = dl.cpu().numpy().view(np.uint16)
            rows = np.unique(np.concatenate([np.arange(0, w.T, 17), [w.T - 1]]))
            check_dlogits(bits, tgt, active, g, w.v_real, w.v_padded, dl_bits, rows=rows)
            assert np.all(dl_bits[:, w.v_real:] == 0)
            assert np.all(dl_bits[~active] == 0)
    assert len(set(shas.values())) == 1, shas


def test_fused_schedules_agree_bitwise(monkeypatch):
    """The L2 schedule (default) and the resident schedule of the fused
    forward+backward, and the forward, at one or two CTAs per SM and row
    skews 0-2, run the
    same per-tile arithmetic on the same bytes, so their outputs are bitwise
    equal, at every virtual TP, on the Qwen3-shaped batch (13-27 rows per
    CTA: the skewed row order wraps the ring many times)."""
    from synth import workloads as W
    w = W.QWEN3
    bits = W.logits_host(w)
    tgt = W.targets(w)
    active = tgt != w.ignore_index
    g = W.grad(w, active)
    dlog = to_dev(bits)
    dt, dg = torch.from_numpy(tgt).cuda(), torch.from_numpy(g).cuda()
    ref = None
    for schedule, per_sm, skew in (("l2", "0", "-1"), ("l2", "1", "-1"), ("l2", "2", "-1"), ("l2", "2", "0"),
                                   ("l2", "1", "0"), ("l2", "2", "2"), ("resident", "0", "-1")):
        monkeypatch.setenv("RLK_FUSED_SCHEDULE", schedule)
        monkeypatch.setenv("RLK_CTAS_PER_SM", per_sm)  # 0: the planner's choice
        monkeypatch.setenv("RLK_FUSED_SKEW", skew)  # -1: the planner's choice
        for vtp in (1, 2, 4, 8):
            c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, vtp, rlk.MASK_IGNORE_INDEX)
            dl, logp, lse = rlk.logp_fwd_bwd(c, dlog, dt, None, dg)
            torch.cuda.synchronize()
            got = (sha(logp), sha(lse), sha(dl))
            if ref is None:
                ref = got
                check_fwd(bits, tgt, active, w.v_real, logp.cpu().numpy(), lse.cpu().numpy())
                rows = np.unique(np.concatenate([np.arange(0, w.T, 29), [w.T - 1]]))
                check_dlogits(bits, tgt, active, g, w.v_real, w.v_padded, dl.cpu().numpy().view(np.uint16),
                              rows=rows)
            assert got == ref, (schedule, per_sm, skew, vtp)
    # the forward at one and two CTAs per SM gives the same LSE and logp
    monkeypatch.delenv("RLK_FUSED_SCHEDULE")
    monkeypatch.delenv("RLK_FUSED_SKEW")
    for per_sm in ("1", "2"):
        monkeypatch.setenv("RLK_CTAS_PER_SM", per_sm)
        for vtp in (1, 8):
            c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, vtp, rlk.MASK_IGNORE_INDEX)
            logp, lse = rlk.logp_fwd(c, dlog, dt)
            torch.cuda.synchronize()
            assert (sha(logp), sha(lse)) == ref[:2], (per_sm, vtp)


def test_host_pipelined_call_equals_one_device_call():
    """logp_fwd_bwd_host copies ragged row chunks on a second stream while the
    previous chunk computes; rows are independent, so every output is
    bitwise that of one call on the whole batch."""
    from synth import workloads as W
    w = W.QWEN3
    bits = W.logits_host(w)
    tgt = W.targets(w)
    active = tgt != w.ignore_index
    g = W.grad(w, active)
    c = contract(w.T, w.v_real, w.v_padded, w.num_tiles, 2, rlk.MASK_IGNORE_INDEX)
    dl_ref, logp_ref, lse_ref = rlk.logp_fwd_bwd(c, to_dev(bits), torch.from_numpy(tgt).cuda(), None,
                                                 torch.from_numpy(g).cuda())
    h_logits = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).pin_memory()
    dl, logp, lse = rlk.logp_fwd_bwd_host(c, h_logits, torch.from_numpy(tgt).pin_memory(), None,
                                          torch.from_numpy(g).pin_memory(), torch.device("cuda"), chunk_rows=1000)
    torch.cuda.synchronize()
    assert torch.equal(dl, dl_ref)
    assert torch.equal(logp, logp_ref.cpu()) and torch.equal(lse, lse_ref.cpu())


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "T%d_V%d_P%d_NT%d" % c[:4])
def test_entropy_small_cases(case):
    """The forward's entropy against the FP64 oracle; logp and LSE stay bitwise
    those of rlk_logp_fwd; the entropy is bitwise identical across virtual TP."""
    T, v_real, v_padded, nt, extra = case
    stride, bits, tgt, mask, active, g = make_inputs(T, v_real, v_padded, nt, extra, seed=T * 7 + nt)
    dlog = to_dev(bits)
    dt, dm = torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda()
    shas = set()
    for vtp in vtps(nt):
        c = contract(T, v_real, v_padded, nt, vtp, rlk.MASK_EXPLICIT, stride)
        logp_e, lse_e, ent = rlk.logp_fwd_entropy(c, dlog, dt, dm)
        logp, lse = rlk.logp_fwd(c, dlog, dt, dm)
        torch.cuda.synchronize()
        assert torch.equal(logp_e, logp) and torch.equal(lse_e, lse)
        check_entropy(bits, v_real, ent.cpu().numpy())
        shas.add(sha(ent))
    assert len(shas) == 1, "virtual TP entropies differ"


def test_entropy_special_rows_and_qwen3_shape(monkeypatch):
    """Rows with one finite column (entropy 0), no finite column (NaN) and
    -inf logits scattered among finite ones (a -inf term adds 0, which the
    tile sum takes from its clamped redo); then the Qwen3-shaped batch, every
    13th row against the oracle, at one and two CTAs per SM and every virtual
    TP, bitwise equal."""
    v_real, v_padded, nt = 1000, 1024, 64
    bits = synth.logits_host(0, 5, v_padded, v_padded, v_real, seed=9, sigma=2.0)
    bits[1, :v_real] = 0xFF80          # all -inf
    bits[2, :v_real] = 0xFF80
    bits[2, 500] = 0x3F80              # one finite column (1.0)
    bits[3, 3:v_real:7] = 0xFF80       # every 7th column -inf, in every tile
    bits[4, 640:656] = 0xFF80          # one whole tile -inf (identity partial) beside finite tiles
    c = contract(5, v_real, v_padded, nt, 2, rlk.MASK_IGNORE_INDEX, validate=0)
    dbits = to_dev(bits)
    tgt5 = torch.full((5,), -100, dtype=torch.int64).cuda()
    _, lse, ent = rlk.logp_fwd_entropy(c, dbits, tgt5)
    torch.cuda.synchronize()
    e = ent.cpu().numpy()
    assert np.isnan(e[1]) and e[2] == 0.0
    assert np.all(np.isfinite(e[[0, 3, 4]]))
    check_entropy(bits, v_real, e)
    _, lse_plain = rlk.logp_fwd(c, dbits, tgt5)
    assert torch.equal(lse, lse_plain)  # the clamped redo leaves the LSE bitwise that of the plain forward

    from synth import workloads as W
    w = W.QWEN3
    qbits = W.logits_host(w)
    dq = to_dev(qbits)
    dt = torch.from_numpy(W.targets(w)).cuda()
    ref = None
    for per_sm in ("1", "2"):
        monkeypatch.setenv("RLK_CTAS_PER_SM", per_sm)
        for vtp in (1, 2, 4, 8):
            cq = contract(w.T, w.v_real, w.v_padded, w.num_tiles, vtp, rlk.MASK_IGNORE_INDEX)
            _, _, eq = rlk.logp_fwd_entropy(cq, dq, dt)
            torch.cuda.synchronize()
            if ref is None:
                ref = sha(eq)
                check_entropy(qbits, w.v_real, eq.cpu().numpy(), rows=np.arange(0, w.T, 13))
            assert sha(eq) == ref, (per_sm, vtp)


def test_outputs_are_batch_invariant():
    """A row's logp, LSE, entropy and dlogits do not depend on the rows that
    share its batch, their order, or the batch size: the same rows permuted,
    or cut into sub-batches of other sizes, give bitwise the same values per
    row (the kernels give every row the same arithmetic, whichever cluster,
    CTA, ring slot or row buffer serves it)."""
    from synth import workloads as W
    w = W.QWEN3
    bits = W.logits_host(w)[:1500]
    tgt = W.targets(w)[:1500]
    g = np.random.default_rng(21).standard_normal(1500).astype(np.float32)
    T = len(tgt)

    def run(rows):
        c = contract(len(rows), w.v_real, w.v_padded, w.num_tiles, 2, rlk.MASK_IGNORE_INDEX)
        d = to_dev(bits[rows])
        dt = torch.from_numpy(tgt[rows]).cuda()
        logp, lse, ent = rlk.logp_fwd_entropy(c, d, dt)
        dl, logp2, lse2 = rlk.logp_fwd_bwd(c, d, dt, None, torch.from_numpy(g[rows]).cuda())
        torch.cuda.synchronize()
        assert torch.equal(logp, logp2) and torch.equal(lse, lse2)
        return [t.cpu().numpy() for t in (logp, lse, ent, dl)]

    ref = run(np.arange(T))
    perm = np.random.default_rng(22).permutation(T)
    got = run(perm)
    for a, b in zip(ref, got):
        assert np.array_equal(a[perm], b, equal_nan=True)
    for lo, hi in ((0, 1), (1, 153), (153, 1000), (1000, T)):
        got = run(np.arange(lo, hi))
        for a, b in zip(ref, got):
            assert np.array_equal(a[lo:hi], b, equal_nan=True)


def test_device_generator_matches_host():
    from synth import workloads as W
    w = W.QWEN3
    dev = torch.empty((64, w.stride), dtype=torch.int16, device="cuda")
    W.logits_device(w, dev, row0=1000, nrows=64)
    host = W.logits_host(w, row0=1000, nrows=64)
    assert np.array_equal(dev.cpu().numpy().view(np.uint16), host)
    hd = torch.empty((8, 4096), dtype=torch.int16, device="cuda")
    synth.normal_bf16_device(hd, 17, 8, 4096, 4096, synth.STREAM_WEIGHT, 0.02)
    assert np.array_equal(hd.cpu().numpy().view(np.uint16),
                          synth.normal_bf16_host(17, 8, 4096, 4096, synth.STREAM_WEIGHT, 0.02))


# ------------------------------------------------------------------ statuses

def _one_row_case(v_real=1000, v_padded=1024, nt=64):
    bits = synth.logits_host(0, 4, v_padded, v_padded, v_real, seed=3, sigma=2.0)
    return bits, v_real, v_padded, nt


def test_active_target_out_of_range_is_reported():
    bits, v_real, v_padded, nt = _one_row_case()
    for bad in (v_real, v_padded - 1, -1):
        tgt = torch.tensor([1, bad, 2, 3], dtype=torch.int64, device="cuda")
        mask = torch.ones(4, dtype=torch.uint8, device="cuda")
        c = contract(4, v_real, v_padded, nt, 2)
        with pytest.raises(rlk.RlkError) as ei:
            rlk.logp_fwd(c, to_dev(bits), tgt, mask)
        assert ei.value.status == rlk.RLK_ERR_TARGET_RANGE
        logp, lse = rlk.logp_fwd(c.replace(validate=0), to_dev(bits), tgt, mask)
        torch.cuda.synchronize()
        assert torch.isnan(logp[1]) and torch.isfinite(logp[0])


def test_nonfinite_lse_on_active_row_only():
    bits, v_real, v_padded, nt = _one_row_case()
    bits = bits.copy()
    bits[1, 10] = 0x7FC0                 # NaN in a real column of row 1
    bits[2, :v_real] = 0xFF80            # row 2: all -inf
    bits[3, v_real + 3] = 0x7FC0         # NaN in padding of row 3: no effect
    tgt = torch.tensor([1, 2, 3, 4], dtype=torch.int64, device="cuda")
    c = contract(4, v_real, v_padded, nt, 1)
    mask = torch.tensor([1, 0, 0, 1], dtype=torch.uint8, device="cuda")
    logp, lse = rlk.logp_fwd(c, to_dev(bits), tgt, mask)     # non-finite only on inactive rows: OK
    torch.cuda.synchronize()
    assert torch.isnan(lse[1]) and lse[2].item() == -np.inf and torch.isfinite(lse[3])
    ref = oracle.lse_full(bits, v_real)
    assert abs(lse[3].item() - ref[3]) < 1e-4
    for bad_row in (1, 2):
        m = mask.clone()
        m[bad_row] = 1
        with pytest.raises(rlk.RlkError) as ei:
            rlk.logp_fwd(c, to_dev(bits), tgt, m)
        assert ei.value.status == rlk.RLK_ERR_NONFINITE_LSE


def test_bounded_wait_expires_with_status_and_context_survives():
    # a wait on an mbarrier that nothing arrives at must end by its deadline
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for ns in (1_000, 2_000_000):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        assert rlk.rlk_selftest_bounded_wait(ns, ws.data_ptr(), stream) == rlk.RLK_ERR_TIMEOUT
        t1.record()
        torch.cuda.synchronize()
        assert t0.elapsed_time(t1) * 1e6 >= ns
    # the product kernels take the same deadline from the contract; with a
    # generous one they finish normally, and the context is still exact
    v_real, v_padded, nt = 151936, 152576, 64
    bits = synth.logits_host(0, 64, v_padded, v_padded, v_real, seed=3, sigma=2.0)
    dlog = to_dev(bits)
    tgt = torch.zeros(64, dtype=torch.int64, device="cuda")
    mask = torch.ones(64, dtype=torch.uint8, device="cuda")
    c = contract(64, v_real, v_padded, nt, 2, wait_timeout_ns=50_000_000)
    logp, lse = rlk.logp_fwd(c, dlog, tgt, mask)
    torch.cuda.synchronize()
    check_fwd(bits, tgt.cpu().numpy(), np.ones(64, bool), v_real, logp.cpu().numpy(), lse.cpu().numpy())


def test_inactive_logp_is_positive_zero_and_f32_outputs():
    T, v_real, v_padded, nt = 24, 5003, 5120, 8
    _, bits, tgt, mask, active, g = make_inputs(T, v_real, v_padded, nt, 0, seed=77)
    logp, lse = rlk.logp_fwd(contract(T, v_real, v_padded, nt, 8, stride=((v_padded + 7) // 8) * 8),
                             to_dev(bits), torch.from_numpy(tgt).cuda(), torch.from_numpy(mask).cuda())
    assert logp.dtype == torch.float32 and lse.dtype == torch.float32
    lp = logp.cpu().numpy()
    assert np.all(f32_bits(lp[~active]) == 0)
