"""Vocabulary-parallel selected-token log-probability across GPUs, one rank per GPU.

The pages' distributed form (PR #289 "[WS2][PR4][Logp] feat: add distributed
TP/CP logprob drift report", PR-1 contract commit: tile-aligned vocabulary
shards, FP32 (max, sumexp) partials exchanged by all-gather and merged by
every rank in fixed global tile order, the target logit resolved on its
owner rank; issue #323 "[WS2][Logprob] H100 validation and reproduction
guide", "Six-Case TP/CP Matrix").  Rank j of a tensor-parallel group of tp
ranks holds columns [j*Vs, (j+1)*Vs) of every row, Vs = V_padded / tp.

Forward, on every rank:

1. the rank checks its own call on the host (the C library's contract check,
   shapes and dtypes) -- no device work;
2. ``rlk_logp_shard_fwd`` on the rank's columns, unless step 1 failed:
   partials [T, NT/tp, 2] and the target logits it owns [T];
3. the ranks agree, before any data moves: one all-reduce (MAX) of the
   status codes of steps 1 and 2 (the call's host-side pointer and device
   checks) and of a fingerprint of the contract (every field, and T) taken
   with both signs, so that MAX gives both ends of the fingerprints' range.
   If any rank's call failed, or the ranks' contracts differ, every rank
   raises the same error, so a rank-local failure never leaves the others
   waiting inside a collective (the pages' review of the vocab-parallel entry
   point raises exactly this, and their preflight compares a rank-independent
   contract fingerprint across the TP group).  One all-reduce and one host
   synchronisation per call;
4. one all-gather of each (plain device buffers);
5. ``rlk_logp_fold`` on the gathered partials, in global tile order: logp and
   LSE, replicated on every rank and bitwise those of ``rlk_logp_fwd`` on one
   GPU for every tp.

Backward: ``rlk_logp_shard_bwd`` from the replicated LSE, after the same
agreement step; it needs no exchange.

Token rows (the pages' CP axis, "not a numerical merge axis") need no
exchange at all: ``split_rows`` gives a rank its contiguous slice.

Every computation is a call into the CUDA library; this module only checks,
agrees and moves buffers.  ``ops`` lets a test substitute the per-rank
computations to exercise the agreement and gather logic on CPU ranks.
"""
import ctypes
import hashlib

import torch
import torch.distributed as dist

from . import (RLK_ERR_INVALID_ARG, RLK_OK, RlkError, fold_gathered, rlk_last_error_message,
               rlk_logp_check_shard_contract, rlk_status_string, shard_bwd, shard_fwd)


class KernelOps:
    """The per-rank computations: the CUDA library's shard entry points."""

    def check(self, contract, shard):
        st = rlk_logp_check_shard_contract(contract, shard)
        return st, ("" if st == RLK_OK else rlk_last_error_message())

    def shard_fwd(self, contract, shard, logits_shard, targets, mask):
        return shard_fwd(contract, shard, logits_shard, targets, mask)

    def fold(self, contract, gathered_partials, gathered_target_logit, targets, mask):
        return fold_gathered(contract, gathered_partials, gathered_target_logit, targets, mask)

    def shard_bwd(self, contract, shard, logits_shard, targets, mask, lse, grad):
        return shard_bwd(contract, shard, logits_shard, targets, mask, lse, grad)


def contract_fingerprint(contract):
    """A rank-independent identity of a contract: the first 62 bits of the SHA-256 of its 64 bytes."""
    raw = ctypes.string_at(ctypes.addressof(contract), ctypes.sizeof(contract))
    return int.from_bytes(hashlib.sha256(raw).digest()[:8], "little") >> 2


def split_rows(T, world, rank):
    """Rows [r0, r1) of rank `rank` when T token rows are split over `world` ranks (contiguous, sizes differ by
    at most one)."""
    base, extra = divmod(T, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


class VocabParallelLogp:
    """One rank's handle on the vocabulary-parallel path (contract.virtual_tp = the group's size)."""

    def __init__(self, contract, group=None, ops=None):
        self.contract = contract
        self.group = group
        self.ops = ops if ops is not None else KernelOps()
        self.tp = dist.get_world_size(group)
        self.rank = dist.get_rank(group)

    # -------------------------------------------------------------- checks and agreement

    def _local_check(self, logits_shard, targets, mask):
        c = self.contract
        if c.virtual_tp != self.tp:
            return RLK_ERR_INVALID_ARG, f"contract.virtual_tp = {c.virtual_tp} but the group has {self.tp} ranks"
        st, msg = self.ops.check(c, self.rank)
        if st != RLK_OK:
            return st, msg
        vs = c.V_padded // c.virtual_tp
        stride = c.row_stride or vs
        if logits_shard.dim() != 2 or logits_shard.shape[0] != c.T or logits_shard.shape[1] != stride:
            return RLK_ERR_INVALID_ARG, f"logits_shard must be [T={c.T}, {stride}], got {tuple(logits_shard.shape)}"
        if logits_shard.dtype not in (torch.int16, torch.bfloat16) or not logits_shard.is_contiguous():
            return RLK_ERR_INVALID_ARG, "logits_shard must be contiguous BF16 (bfloat16 or int16 storage)"
        if targets.dtype != torch.int64 or targets.numel() != c.T:
            return RLK_ERR_INVALID_ARG, "targets must be int64 [T]"
        if (mask is None) != (c.mask_mode == 1):
            return RLK_ERR_INVALID_ARG, "active_mask must be given in explicit mode and None in ignore_index mode"
        if mask is not None and (mask.dtype not in (torch.uint8, torch.bool) or mask.numel() != c.T):
            return RLK_ERR_INVALID_ARG, "active_mask must be uint8 [T]"
        if targets.device != logits_shard.device or (mask is not None and mask.device != logits_shard.device):
            return RLK_ERR_INVALID_ARG, "logits_shard, targets and active_mask must be on one device"
        return RLK_OK, ""

    def _call(self, fn, *args):
        """(status, message, result) of one per-rank computation; an RlkError becomes its status."""
        try:
            return RLK_OK, "", fn(*args)
        except RlkError as e:
            return e.status, str(e), None

    def _agree(self, status, message, device):
        """One all-reduce (MAX) of the ranks' status codes and of the contract fingerprint with both signs;
        every rank raises if any rank's call is invalid or the contracts differ."""
        fp = contract_fingerprint(self.contract)
        t = torch.tensor([int(status), fp, -fp], dtype=torch.int64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=self.group)
        worst, fp_max, fp_min = int(t[0].item()), int(t[1].item()), -int(t[2].item())
        if worst != RLK_OK:
            if status != RLK_OK:
                raise RlkError(status, message)
            raise RlkError(worst, f"another rank of the group rejected its call ({rlk_status_string(worst)})")
        if fp_max != fp_min:
            raise RlkError(RLK_ERR_INVALID_ARG, "the ranks of the group hold different contracts "
                                                "(T, vocabulary, tiles, virtual_tp, mask mode or stride differ)")

    def _all_gather(self, out, x):
        """out[r] = rank r's x, shard-major (out has a leading dimension of tp)."""
        if dist.get_backend(self.group) == "nccl":
            dist.all_gather_into_tensor(out.view(-1), x.contiguous().view(-1), group=self.group)
        else:
            dist.all_gather(list(out.unbind(0)), x.contiguous(), group=self.group)

    # -------------------------------------------------------------- the path

    def forward(self, logits_shard, targets, mask=None):
        """(logp, lse) of every row, replicated on every rank."""
        st, msg = self._local_check(logits_shard, targets, mask)
        out = None
        if st == RLK_OK:  # a rank whose own checks fail skips its call and still joins the agreement
            st, msg, out = self._call(self.ops.shard_fwd, self.contract, self.rank, logits_shard, targets, mask)
        self._agree(st, msg, targets.device)  # one host synchronisation per call
        part, xt = out
        gathered = torch.empty((self.tp,) + tuple(part.shape), dtype=part.dtype, device=part.device)
        gathered_xt = torch.empty((self.tp,) + tuple(xt.shape), dtype=xt.dtype, device=xt.device)
        self._all_gather(gathered, part)
        self._all_gather(gathered_xt, xt)
        return self.ops.fold(self.contract, gathered, gathered_xt, targets, mask)

    def backward(self, logits_shard, targets, mask, lse, grad):
        """BF16 dlogits of this rank's columns, from the replicated LSE; no exchange."""
        st, msg = self._local_check(logits_shard, targets, mask)
        if st == RLK_OK and any(t.dtype != torch.float32 or t.numel() != self.contract.T or
                                t.device != logits_shard.device for t in (lse, grad)):
            st, msg = RLK_ERR_INVALID_ARG, "lse and grad must be FP32 [T] on the logits' device"
        out = None
        if st == RLK_OK:
            st, msg, out = self._call(self.ops.shard_bwd, self.contract, self.rank, logits_shard, targets, mask, lse,
                                      grad)
        # no collective follows, but every rank still returns or raises together
        self._agree(st, msg, targets.device)
        return out
