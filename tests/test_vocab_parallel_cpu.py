"""The vocabulary-parallel layer across processes, on CPU with gloo ranks.

vocab_selected_token_tile_gb300.vocab_parallel checks each rank's call, makes
the ranks agree before any data moves, all-gathers the partials and target
logits shard-major, and folds.  Here the per-rank computations are the FP64
oracle (the CUDA ones need a GPU; they are checked bit for bit on one GPU in
test_vocab_parallel_gpu.py), and the contract check is the C library's own
host check.  What is tested is the layer's logic:

* the gathered partials, in global tile order, are exactly the partials of
  the whole row, and the fold gives the whole row's LSE and logp (gather
  order and owner-rank resolution of the target logit);
* a rank whose call is invalid makes every rank raise, with no rank left
  waiting in a collective (the pages' review: rank-local validation failures
  can strand the other TP ranks) -- whether the layer's own check, the C
  library's contract check or the shard call's host checks reject it, in
  the forward or in the backward;
* ranks whose contracts are each valid but differ (the pages' preflight
  compares a contract fingerprint) all raise before any data moves;
* the backward returns each rank's own shard;
* token rows split over ranks cover every row once.
"""
import json
import os
import socket
import sys
from datetime import timedelta

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

T, V_REAL, V_PADDED, NT = 24, 1000, 1024, 8


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def full_inputs():
    rng = np.random.default_rng(5)
    f = (rng.standard_normal((T, V_PADDED)) * 3.0).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    bits = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    bits[:, V_REAL:] = rng.integers(0, 1 << 16, size=(T, V_PADDED - V_REAL), dtype=np.uint16)
    tgt = rng.integers(0, V_REAL, size=T).astype(np.int64)
    mask = (np.arange(T) % 4 != 1).astype(np.uint8)
    tgt[mask == 0] = -7  # never read
    return bits, tgt, mask


class OracleOps:
    """Per-rank computations in FP64 on CPU (test stand-ins for the CUDA shard calls)."""

    def __init__(self, lib_ops):
        self.lib = lib_ops

    def check(self, contract, shard):
        return self.lib.check(contract, shard)

    def shard_fwd(self, contract, shard, logits_shard, targets, mask):
        import oracle
        vs = contract.V_padded // contract.virtual_tp
        c0 = shard * vs
        vr_l = min(max(contract.V_real - c0, 0), vs)
        bits = logits_shard.numpy().view(np.uint16)
        m, s = oracle.tile_partials(bits, vr_l, vs, contract.num_tiles // contract.virtual_tp)
        t = targets.numpy()
        act = mask.numpy() != 0
        xt = np.zeros(contract.T)
        own = act & (t >= c0) & (t < c0 + vr_l)
        xt[own] = oracle.bf16_bits_to_f64(bits[own, t[own] - c0])
        return torch.from_numpy(np.stack([m, s], axis=-1)), torch.from_numpy(xt)

    def fold(self, contract, gathered, gathered_xt, targets, mask):
        import oracle
        g = gathered.numpy()  # [tp, T, NT/tp, 2]
        full = np.concatenate(list(g), axis=1)  # [T, NT, 2] in global tile order
        lse = oracle.fold_partials(full[..., 0], full[..., 1])
        vs = contract.V_padded // contract.virtual_tp
        t = targets.numpy()
        act = mask.numpy() != 0
        logp = np.zeros(contract.T)
        rows = np.nonzero(act)[0]
        logp[rows] = gathered_xt.numpy()[t[rows] // vs, rows] - lse[rows]
        return torch.from_numpy(logp), torch.from_numpy(lse), full

    def shard_bwd(self, contract, shard, logits_shard, targets, mask, lse, grad):
        # a marker of the rank that computed it (the CUDA backward is checked on the GPU)
        return torch.full(tuple(logits_shard.shape), shard, dtype=torch.int16)


class FailingOps(OracleOps):
    """The shard calls of one rank fail on the host, as the C library's pointer or device checks would."""

    def __init__(self, lib_ops, failing_rank, failing_call):
        super().__init__(lib_ops)
        self.failing_rank = failing_rank
        self.failing_call = failing_call

    def _fail(self, shard, call):
        import vocab_selected_token_tile_gb300 as rlk
        if shard == self.failing_rank and call == self.failing_call:
            raise rlk.RlkError(rlk.RLK_ERR_INVALID_ARG, "targets must be device memory (it is host memory)")

    def shard_fwd(self, contract, shard, *args):
        self._fail(shard, "fwd")
        return super().shard_fwd(contract, shard, *args)

    def shard_bwd(self, contract, shard, *args):
        self._fail(shard, "bwd")
        return super().shard_bwd(contract, shard, *args)


def _rank_main(rank, world, port, case, out_dir):
    import vocab_selected_token_tile_gb300 as rlk
    from vocab_selected_token_tile_gb300 import vocab_parallel as vp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=60))
    res = {}
    try:
        bits, tgt, mask = full_inputs()
        vs = V_PADDED // world
        c = rlk.Contract(T=T, V_real=V_REAL, V_padded=V_PADDED, num_tiles=NT, virtual_tp=world)
        shard = torch.from_numpy(np.ascontiguousarray(bits[:, rank * vs:(rank + 1) * vs]).view(np.int16))
        targets, m = torch.from_numpy(tgt), torch.from_numpy(mask)
        if case == "bad_contract" and rank == 1:
            c = c.replace(num_tiles=6)  # 6 does not divide 1024: this rank's host check fails
        if case == "bad_shape" and rank == 0:
            shard = shard[:, :-8].contiguous()
        if case == "contract_mismatch" and rank == 1:
            c = c.replace(V_real=V_REAL - 1)  # valid on its own, but not the group's contract
        ops = OracleOps(vp.KernelOps())
        if case == "fwd_call_fails":
            ops = FailingOps(vp.KernelOps(), failing_rank=1, failing_call="fwd")
        if case in ("bwd_call_fails", "bwd_ok"):
            ops = FailingOps(vp.KernelOps(), failing_rank=0 if case == "bwd_call_fails" else -1, failing_call="bwd")
        layer = vp.VocabParallelLogp(c, ops=ops)
        try:
            logp, lse, full = layer.forward(shard, targets, m)
            res["ok"] = True
            res["logp"] = logp.tolist()
            res["lse"] = lse.tolist()
            res["partials"] = full.tolist()
        except rlk.RlkError as e:
            res["ok"] = False
            res["status"] = e.status
            res["message"] = str(e)
        if case in ("bad_bwd", "bad_bwd_dtype", "bwd_call_fails", "bwd_ok"):
            lse = torch.zeros(T if rank == 0 or case != "bad_bwd" else T - 1)
            if case == "bad_bwd_dtype" and rank == 1:
                lse = lse.double()
            try:
                d = layer.backward(shard, targets, m, lse, torch.zeros(T))
                res["bwd_ok"] = True
                res["bwd_marker"] = sorted(set(d.flatten().tolist()))
                res["bwd_shape"] = list(d.shape)
            except rlk.RlkError as e:
                res["bwd_ok"] = False
                res["bwd_status"] = e.status
                res["bwd_message"] = str(e)
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


def run(world, case, tmp_path):
    mp.start_processes(_rank_main, args=(world, free_port(), case, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    return [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]


@pytest.mark.parametrize("world", [2, 4])
def test_gather_order_and_fold_give_the_whole_row(built, tmp_path, world):
    import oracle
    bits, tgt, mask = full_inputs()
    act = mask != 0
    m, s = oracle.tile_partials(bits, V_REAL, V_PADDED, NT)
    want_lse = oracle.fold_partials(m, s)
    want_logp, _ = oracle.selected_logp(bits, np.where(act, tgt, 0), act, V_REAL)
    res = run(world, "ok", tmp_path)
    for r in res:
        assert r["ok"]
        p = np.asarray(r["partials"])
        assert np.array_equal(p[..., 0], m) and np.array_equal(p[..., 1], s)  # shard-major gather = tile order
        assert np.array_equal(np.asarray(r["lse"]), want_lse)
        assert np.max(np.abs(np.asarray(r["logp"]) - want_logp)) < 1e-12
        assert all(v == 0.0 for v, a in zip(r["logp"], act) if not a)
    assert res[0]["logp"] == res[1]["logp"]


@pytest.mark.parametrize("case", ["bad_contract", "bad_shape", "fwd_call_fails", "bad_bwd", "bad_bwd_dtype",
                                  "bwd_call_fails", "contract_mismatch"])
def test_an_invalid_call_on_one_rank_fails_closed_on_every_rank(built, tmp_path, case):
    """A host check that fails on one rank -- the layer's own, the contract check, or the shard call's
    pointer checks -- makes every rank raise the same status, and no rank is left inside a collective
    (the all-gather of the forward is never entered)."""
    import vocab_selected_token_tile_gb300 as rlk
    res = run(2, case, tmp_path)
    if case.startswith("bad_bwd") or case == "bwd_call_fails":
        assert all(r["ok"] for r in res)  # the forward was valid on both ranks
        assert all(not r["bwd_ok"] for r in res)
        assert all(r["bwd_status"] == rlk.RLK_ERR_INVALID_ARG for r in res)
        bad = 0 if case == "bwd_call_fails" else 1
        assert "another rank" in res[1 - bad]["bwd_message"]
        assert "another rank" not in res[bad]["bwd_message"]
        return
    assert all(not r["ok"] for r in res)
    if case == "contract_mismatch":  # both contracts are valid: every rank names the mismatch
        assert all(r["status"] == rlk.RLK_ERR_INVALID_ARG and "different contracts" in r["message"] for r in res)
        return
    bad = 0 if case == "bad_shape" else 1
    want = rlk.RLK_ERR_NON_TILEABLE if case == "bad_contract" else rlk.RLK_ERR_INVALID_ARG
    assert res[bad]["status"] == want
    assert res[1 - bad]["status"] == want and "another rank" in res[1 - bad]["message"]
    if case == "fwd_call_fails":
        assert "device memory" in res[bad]["message"]


def test_backward_returns_each_ranks_own_shard(built, tmp_path):
    res = run(2, "bwd_ok", tmp_path)
    for rank, r in enumerate(res):
        assert r["ok"] and r["bwd_ok"]
        assert r["bwd_marker"] == [rank] and r["bwd_shape"] == [T, V_PADDED // 2]


def test_split_rows_covers_every_row_once():
    from vocab_selected_token_tile_gb300.vocab_parallel import split_rows
    for T_ in (0, 1, 7, 65536, 65537):
        for world in (1, 2, 3, 4, 8):
            spans = [split_rows(T_, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T_
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
