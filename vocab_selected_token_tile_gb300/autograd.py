"""torch.autograd entry points of the selected-token log-probability.

Argument marshalling only: ``SelectedTokenLogprob``'s forward calls
``rlk_logp_fwd`` and its backward ``rlk_logp_bwd`` with the saved LSE;
``FusedLmHeadLogprob``'s forward calls ``rlk_logp_fused_lmhead`` (logits =
hidden @ weight^T, never materialised) and its backward
``rlk_logp_fused_lmhead_bwd`` with the saved LSE -- or, with keep_logits,
``rlk_logp_fused_lmhead_keep`` and ``rlk_logp_fused_lmhead_bwd_kept`` with the
saved FP32 logits.  Every step of the
arithmetic runs in the CUDA library.  The outputs follow the typed contract of PR #289
("[WS2][PR4][Logp] feat: add distributed TP/CP logprob drift report",
"typed contract" commit: FP32 logprob and FP32 LSE outputs); the LSE is not
differentiable.
"""
import torch

from . import (MASK_EXPLICIT, MASK_IGNORE_INDEX, Contract, logp_bwd, logp_fused_lmhead, logp_fused_lmhead_bwd,
               logp_fused_lmhead_bwd_kept, logp_fused_lmhead_keep, logp_fwd)

_LOGIT_DTYPES = (torch.bfloat16, torch.int16)  # int16: BF16 bits viewed as integers


class SelectedTokenLogprob(torch.autograd.Function):
    """(logp, lse) of BF16 logits [T, row_stride]; d logits = g (onehot - softmax) in BF16."""

    @staticmethod
    def forward(ctx, logits, targets, mask, contract):
        if logits.dtype not in _LOGIT_DTYPES or not logits.is_cuda:
            raise TypeError("logits must be a CUDA tensor of BF16 (or its int16 bits)")
        logp, lse = logp_fwd(contract, logits, targets, mask)
        ctx.save_for_backward(logits, targets, mask, lse)
        ctx.contract = contract
        ctx.mark_non_differentiable(lse)
        return logp, lse

    @staticmethod
    def backward(ctx, grad_logp, grad_lse):
        logits, targets, mask, lse = ctx.saved_tensors
        if grad_logp is None:
            return None, None, None, None
        g = grad_logp if (grad_logp.dtype == torch.float32 and grad_logp.is_contiguous()) else \
            grad_logp.to(torch.float32).contiguous()
        c = ctx.contract
        # columns [V_padded, row_stride) are not the kernel's: their gradient is zero
        out = torch.zeros_like(logits) if c.row_stride > c.V_padded else None
        dlogits = logp_bwd(c, logits, targets, mask, lse, g, dlogits=out)
        return dlogits, None, None, None


def selected_logprob(logits, targets, mask=None, v_real=None, v_padded=None, num_tiles=64, virtual_tp=1,
                     ignore_index=-100):
    """(logp, lse) with autograd; ``mask`` None selects ignore_index mode.

    ``logits`` is [T, row_stride] BF16 on the GPU; columns [v_real, v_padded)
    are padding (v_padded defaults to row_stride, v_real to v_padded).
    """
    T, stride = logits.shape
    vp = stride if v_padded is None else v_padded
    vr = vp if v_real is None else v_real
    c = Contract(T=T, V_real=vr, V_padded=vp, num_tiles=num_tiles, virtual_tp=virtual_tp,
                 mask_mode=MASK_EXPLICIT if mask is not None else MASK_IGNORE_INDEX, ignore_index=ignore_index,
                 row_stride=stride)
    return SelectedTokenLogprob.apply(logits, targets, mask, c)


class FusedLmHeadLogprob(torch.autograd.Function):
    """(logp, lse) of logits = hidden @ weight^T over a tiled vocabulary; d hidden and d weight in BF16
    (the dtype of the inputs).  hidden [T, H], weight [V_padded, H].  With keep_logits False the logits
    are never materialised and the backward re-runs the GEMM; with True the forward keeps its FP32
    logits (T * V_padded * 4 bytes, held until the backward) and the backward forms dlogits from them
    instead.  The gradients are bitwise the same either way."""

    @staticmethod
    def forward(ctx, hidden, weight, targets, mask, contract, keep_logits=False):
        for name, t in (("hidden", hidden), ("weight", weight)):
            if t.dtype not in _LOGIT_DTYPES or not t.is_cuda or not t.is_contiguous():
                raise TypeError(f"{name} must be a contiguous CUDA tensor of BF16 (or its int16 bits)")
        logits = None
        if keep_logits and (ctx.needs_input_grad[0] or ctx.needs_input_grad[1]):
            logp, lse, logits = logp_fused_lmhead_keep(contract, hidden, weight, targets, mask)
        else:
            logp, lse = logp_fused_lmhead(contract, hidden, weight, targets, mask)
        ctx.save_for_backward(hidden, weight, targets, mask, lse, logits)
        ctx.contract = contract
        ctx.mark_non_differentiable(lse)
        return logp, lse

    @staticmethod
    def backward(ctx, grad_logp, grad_lse):
        hidden, weight, targets, mask, lse, logits = ctx.saved_tensors
        if grad_logp is None:
            return None, None, None, None, None, None
        g = grad_logp if (grad_logp.dtype == torch.float32 and grad_logp.is_contiguous()) else \
            grad_logp.to(torch.float32).contiguous()
        if logits is not None:
            dh, dw = logp_fused_lmhead_bwd_kept(ctx.contract, hidden, weight, targets, mask, lse, logits, g)
        else:
            dh, dw = logp_fused_lmhead_bwd(ctx.contract, hidden, weight, targets, mask, lse, g)
        return dh, dw, None, None, None, None


def lmhead_logprob(hidden, weight, targets, mask=None, v_real=None, num_tiles=64, virtual_tp=1, ignore_index=-100,
                   keep_logits=False):
    """(logp, lse) of hidden @ weight^T with autograd; ``mask`` None selects ignore_index mode.

    ``weight`` is [V_padded, H]; rows [v_real, V_padded) are padding (v_real defaults to V_padded).
    ``keep_logits`` trades T * V_padded * 4 bytes, held from the forward to the backward, for the
    backward's recompute GEMM (a third of the forward+backward's tensor work).
    """
    T = hidden.shape[0]
    vp = weight.shape[0]
    vr = vp if v_real is None else v_real
    c = Contract(T=T, V_real=vr, V_padded=vp, num_tiles=num_tiles, virtual_tp=virtual_tp,
                 mask_mode=MASK_EXPLICIT if mask is not None else MASK_IGNORE_INDEX, ignore_index=ignore_index)
    return FusedLmHeadLogprob.apply(hidden, weight, targets, mask, c, keep_logits)
