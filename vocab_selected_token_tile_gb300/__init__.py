"""Deterministic selected-token log-probability over a tiled vocabulary (GB300, sm_103a).

A thin ctypes binding of ``librlk_logp.so`` (declared in ``include/rlk_logp.h``).
The functions named ``rlk_*`` mirror the C entry points one to one and take
raw device pointers; ``logp_fwd``, ``logp_bwd`` and ``logp_fwd_bwd`` only
marshal torch tensors (allocate outputs, pass ``data_ptr()`` and the current
stream).  Every step of the computation runs in the CUDA library: if it is
missing or fails to load, these functions raise -- there is no fallback.
"""
import ctypes
import os

from . import _build

RLK_OK = 0
RLK_ERR_INVALID_ARG = 1
RLK_ERR_UNSUPPORTED = 2
RLK_ERR_NON_TILEABLE = 3
RLK_ERR_MISALIGNED = 4
RLK_ERR_TARGET_RANGE = 5
RLK_ERR_NONFINITE_LSE = 6
RLK_ERR_TIMEOUT = 7
RLK_ERR_CUDA = 8

MASK_EXPLICIT = 0
MASK_IGNORE_INDEX = 1

EXPORTED = (
    "rlk_logp_check_contract",
    "rlk_logp_workspace_size",
    "rlk_logp_fwd",
    "rlk_logp_bwd",
    "rlk_logp_fwd_noalloc",
    "rlk_logp_fwd_entropy",
    "rlk_logp_fwd_bwd_entropy",
    "rlk_grpo_loss",
    "rlk_grpo_fused_workspace_size",
    "rlk_grpo_fused_step",
    "rlk_logp_lmhead_workspace_size",
    "rlk_logp_fused_lmhead",
    "rlk_logp_fused_lmhead_bwd",
    "rlk_logp_fused_lmhead_keep",
    "rlk_logp_fused_lmhead_bwd_kept",
    "rlk_logp_check_shard_contract",
    "rlk_logp_shard_workspace_size",
    "rlk_logp_shard_fwd",
    "rlk_logp_fold",
    "rlk_logp_shard_bwd",
    "rlk_logp_workspace_status",
    "rlk_selftest_bounded_wait",
    "rlk_status_string",
    "rlk_last_error_message",
)


class Contract(ctypes.Structure):
    """Mirror of ``rlk_logp_contract`` (64 bytes)."""
    _fields_ = [
        ("T", ctypes.c_int64),
        ("V_real", ctypes.c_int64),
        ("V_padded", ctypes.c_int64),
        ("row_stride", ctypes.c_int64),
        ("num_tiles", ctypes.c_int32),
        ("virtual_tp", ctypes.c_int32),
        ("mask_mode", ctypes.c_int32),
        ("validate", ctypes.c_int32),
        ("ignore_index", ctypes.c_int64),
        ("wait_timeout_ns", ctypes.c_int64),
    ]

    def __init__(self, T, V_real, V_padded, num_tiles=64, virtual_tp=1, mask_mode=MASK_EXPLICIT,
                 ignore_index=-100, validate=0, row_stride=0, wait_timeout_ns=0):
        super().__init__(T, V_real, V_padded, row_stride, num_tiles, virtual_tp, mask_mode, validate,
                         ignore_index, wait_timeout_ns)

    def replace(self, **kw):
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d.update(kw)
        return Contract(**d)


class RlkError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{rlk_status_string(status)}: {message}")
        self.status = status


_lib = None


def library():
    """Load librlk_logp.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"CUDA library not built: {_build.LIB} (run __graft_entry__.build())")
        lib = ctypes.CDLL(_build.LIB)
        P = ctypes.POINTER(Contract)
        vp, i = ctypes.c_void_p, ctypes.c_int
        lib.rlk_logp_check_contract.argtypes = [P]
        lib.rlk_logp_check_contract.restype = i
        lib.rlk_logp_workspace_size.argtypes = [P]
        lib.rlk_logp_workspace_size.restype = ctypes.c_size_t
        lib.rlk_logp_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_fwd.restype = i
        lib.rlk_logp_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_bwd.restype = i
        lib.rlk_logp_lmhead_workspace_size.argtypes = [P, ctypes.c_int64]
        lib.rlk_logp_lmhead_workspace_size.restype = ctypes.c_size_t
        lib.rlk_logp_fused_lmhead.argtypes = [P, vp, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_fused_lmhead.restype = i
        lib.rlk_logp_fused_lmhead_bwd.argtypes = [P, vp, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_fused_lmhead_bwd.restype = i
        lib.rlk_logp_fused_lmhead_keep.argtypes = [P, vp, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_fused_lmhead_keep.restype = i
        lib.rlk_logp_fused_lmhead_bwd_kept.argtypes = [P, vp, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                       vp, vp]
        lib.rlk_logp_fused_lmhead_bwd_kept.restype = i
        lib.rlk_logp_fwd_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_fwd_noalloc.restype = i
        lib.rlk_logp_fwd_entropy.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_fwd_entropy.restype = i
        lib.rlk_logp_fwd_bwd_entropy.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_fwd_bwd_entropy.restype = i
        lib.rlk_grpo_loss.argtypes = [ctypes.c_int64, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp]
        lib.rlk_grpo_loss.restype = i
        lib.rlk_grpo_fused_workspace_size.argtypes = [P]
        lib.rlk_grpo_fused_workspace_size.restype = ctypes.c_size_t
        lib.rlk_grpo_fused_step.argtypes = [P, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_grpo_fused_step.restype = i
        lib.rlk_logp_check_shard_contract.argtypes = [P, ctypes.c_int32]
        lib.rlk_logp_check_shard_contract.restype = i
        lib.rlk_logp_shard_workspace_size.argtypes = [P]
        lib.rlk_logp_shard_workspace_size.restype = ctypes.c_size_t
        lib.rlk_logp_shard_fwd.argtypes = [P, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_shard_fwd.restype = i
        lib.rlk_logp_fold.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_fold.restype = i
        lib.rlk_logp_shard_bwd.argtypes = [P, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logp_shard_bwd.restype = i
        lib.rlk_logp_workspace_status.argtypes = [vp, vp]
        lib.rlk_logp_workspace_status.restype = i
        lib.rlk_selftest_bounded_wait.argtypes = [ctypes.c_int64, vp, vp]
        lib.rlk_selftest_bounded_wait.restype = i
        lib.rlk_status_string.argtypes = [i]
        lib.rlk_status_string.restype = ctypes.c_char_p
        lib.rlk_last_error_message.argtypes = []
        lib.rlk_last_error_message.restype = ctypes.c_char_p
        _lib = lib
    return _lib


# ------------------------------------------------------------------ C names

def rlk_logp_check_contract(contract):
    return library().rlk_logp_check_contract(ctypes.byref(contract))


def rlk_logp_workspace_size(contract):
    return library().rlk_logp_workspace_size(ctypes.byref(contract))


def rlk_logp_fwd(contract, logits, targets, active_mask, logp, lse, partials, workspace, stream):
    return library().rlk_logp_fwd(ctypes.byref(contract), logits, targets, active_mask, logp, lse, partials,
                                  workspace, stream)


def rlk_logp_bwd(contract, logits, targets, active_mask, lse_in, grad_logp, dlogits, logp_out, lse_out,
                 workspace, stream):
    return library().rlk_logp_bwd(ctypes.byref(contract), logits, targets, active_mask, lse_in, grad_logp,
                                  dlogits, logp_out, lse_out, workspace, stream)


def rlk_logp_lmhead_workspace_size(contract, H):
    return library().rlk_logp_lmhead_workspace_size(ctypes.byref(contract), H)


def rlk_logp_fused_lmhead(contract, hidden, H, weight, targets, active_mask, grad_logp, logp, lse, dhidden,
                          dweight_f32, dweight_bf16, workspace, stream):
    return library().rlk_logp_fused_lmhead(ctypes.byref(contract), hidden, H, weight, targets, active_mask,
                                           grad_logp, logp, lse, dhidden, dweight_f32, dweight_bf16, workspace,
                                           stream)


def rlk_logp_fused_lmhead_bwd(contract, hidden, H, weight, targets, active_mask, lse_in, grad_logp, dhidden,
                              dweight_f32, dweight_bf16, workspace, stream):
    return library().rlk_logp_fused_lmhead_bwd(ctypes.byref(contract), hidden, H, weight, targets, active_mask,
                                               lse_in, grad_logp, dhidden, dweight_f32, dweight_bf16, workspace,
                                               stream)


def rlk_logp_fused_lmhead_keep(contract, hidden, H, weight, targets, active_mask, logp, lse, logits_f32, workspace,
                               stream):
    return library().rlk_logp_fused_lmhead_keep(ctypes.byref(contract), hidden, H, weight, targets, active_mask,
                                                logp, lse, logits_f32, workspace, stream)


def rlk_logp_fused_lmhead_bwd_kept(contract, hidden, H, weight, targets, active_mask, lse_in, logits_f32, grad_logp,
                                   dhidden, dweight_f32, dweight_bf16, workspace, stream):
    return library().rlk_logp_fused_lmhead_bwd_kept(ctypes.byref(contract), hidden, H, weight, targets, active_mask,
                                                    lse_in, logits_f32, grad_logp, dhidden, dweight_f32,
                                                    dweight_bf16, workspace, stream)


def rlk_logp_fwd_entropy(contract, logits, targets, active_mask, logp, lse, entropy, workspace, stream):
    return library().rlk_logp_fwd_entropy(ctypes.byref(contract), logits, targets, active_mask, logp, lse, entropy,
                                          workspace, stream)


def rlk_logp_fwd_bwd_entropy(contract, logits, targets, active_mask, grad_logp, dlogits, logp_out, lse_out,
                             entropy_out, workspace, stream):
    return library().rlk_logp_fwd_bwd_entropy(ctypes.byref(contract), logits, targets, active_mask, grad_logp,
                                              dlogits, logp_out, lse_out, entropy_out, workspace, stream)


def rlk_grpo_loss(T, logp, advantage, active_mask, ref_logp, beta, loss, grad_logp, active_count, stream):
    return library().rlk_grpo_loss(T, logp, advantage, active_mask, ref_logp, beta, loss, grad_logp, active_count,
                                   stream)


def rlk_grpo_fused_workspace_size(contract):
    return library().rlk_grpo_fused_workspace_size(ctypes.byref(contract))


def rlk_grpo_fused_step(contract, logits, targets, active_mask, advantage, ref_logp, beta, dlogits, logp_out, lse_out,
                        grad_out, entropy_out, loss, active_count, workspace, stream):
    return library().rlk_grpo_fused_step(ctypes.byref(contract), logits, targets, active_mask, advantage, ref_logp,
                                         beta, dlogits, logp_out, lse_out, grad_out, entropy_out, loss, active_count,
                                         workspace, stream)


def rlk_logp_fwd_noalloc(contract, logits, targets, active_mask, logp, lse, partials, stream):
    return library().rlk_logp_fwd_noalloc(ctypes.byref(contract), logits, targets, active_mask, logp, lse,
                                          partials, stream)


def rlk_logp_check_shard_contract(contract, shard):
    return library().rlk_logp_check_shard_contract(ctypes.byref(contract), shard)


def rlk_logp_shard_workspace_size(contract):
    return library().rlk_logp_shard_workspace_size(ctypes.byref(contract))


def rlk_logp_shard_fwd(contract, shard, logits_shard, targets, active_mask, partials_shard, target_logit, workspace,
                       stream):
    return library().rlk_logp_shard_fwd(ctypes.byref(contract), shard, logits_shard, targets, active_mask,
                                        partials_shard, target_logit, workspace, stream)


def rlk_logp_fold(contract, gathered_partials, gathered_target_logit, targets, active_mask, logp, lse, workspace,
                  stream):
    return library().rlk_logp_fold(ctypes.byref(contract), gathered_partials, gathered_target_logit, targets,
                                   active_mask, logp, lse, workspace, stream)


def rlk_logp_shard_bwd(contract, shard, logits_shard, targets, active_mask, lse_in, grad_logp, dlogits_shard,
                       workspace, stream):
    return library().rlk_logp_shard_bwd(ctypes.byref(contract), shard, logits_shard, targets, active_mask, lse_in,
                                        grad_logp, dlogits_shard, workspace, stream)


def rlk_logp_workspace_status(workspace, stream):
    return library().rlk_logp_workspace_status(workspace, stream)


def rlk_selftest_bounded_wait(timeout_ns, workspace, stream):
    return library().rlk_selftest_bounded_wait(timeout_ns, workspace, stream)


def rlk_status_string(status):
    return library().rlk_status_string(status).decode()


def rlk_last_error_message():
    return library().rlk_last_error_message().decode()


def check(status):
    if status != RLK_OK:
        raise RlkError(status, rlk_last_error_message())


# ------------------------------------------------------------------ torch marshalling

def _ptr(t):
    return None if t is None else t.data_ptr()


_BF16 = ("bfloat16", "int16", "uint16")  # BF16 logits, or their bits as 16-bit integers
_I64 = ("int64",)
_U8 = ("uint8", "bool")
_F32 = ("float32",)


def _need(t, name, nbytes, kinds, optional=False):
    """Fails before any launch when ``t`` cannot be what the call reads or writes through its pointer:
    a CUDA tensor of one of ``kinds`` whose storage holds ``nbytes`` from its first element on (so no
    access leaves it) and, when it is contiguous, whose own elements cover them (a short view of a
    larger buffer is a mistake too).  The C entry points check pointers, alignment and the device;
    only the caller knows the sizes."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    kind = str(t.dtype).replace("torch.", "")
    if kind not in kinds:
        raise TypeError(f"{name} must be {' or '.join(kinds)}, not {kind}")
    have = t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes from its first element; the call touches {nbytes}")
    if t.is_contiguous() and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} has {t.numel()} elements; the call touches {nbytes} bytes")


def _need_rows(t, name, T, stride, width, kinds):
    """A [T, stride] row buffer of 16-bit elements of which the call touches ``width`` a row; a 2-D
    view must also have those rows and that row stride (a shard read in place from the whole row
    buffer is such a view)."""
    _need(t, name, _rows(T, stride, width, 2), kinds)
    if t.dim() == 2 and T > 0 and (t.shape[0] < T or t.shape[1] < width or t.stride(1) != 1 or
                                   (T > 1 and t.stride(0) != stride)):
        raise ValueError(f"{name} is a {list(t.shape)} view with strides {list(t.stride())}; the call reads {T} "
                         f"rows of {width} elements, {stride} apart")


def _rows(T, stride, width, esize):
    """Bytes from the first element of a [T, stride] row-major buffer to the end of row T-1's width."""
    return 0 if T <= 0 else ((T - 1) * stride + width) * esize


def _dlogits_out(contract, logits, dlogits, stride=None, width=None):
    """The dlogits buffer: the given one, checked, or a new [T, row stride] one like the logits."""
    import torch
    stride = stride or contract.row_stride or contract.V_padded
    width = width or contract.V_padded
    if dlogits is None:
        return torch.empty((contract.T, stride), dtype=logits.dtype, device=logits.device)
    _need_rows(dlogits, "dlogits", contract.T, stride, width, _BF16)
    return dlogits


def _lmhead_operands(contract, hidden, weight):
    """hidden [T, H] and weight [V_padded, H], BF16, contiguous; returns H."""
    if hidden.dim() != 2 or hidden.shape[0] != contract.T:
        raise ValueError(f"hidden must be [T = {contract.T}, H], not {list(hidden.shape)}")
    H = hidden.shape[1]
    if weight.dim() != 2 or weight.shape[0] != contract.V_padded or weight.shape[1] != H:
        raise ValueError(f"weight must be [V_padded = {contract.V_padded}, H = {H}], not {list(weight.shape)}")
    for name, t in (("hidden", hidden), ("weight", weight)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        _need(t, name, 2 * t.numel(), _BF16)
    return H


def _lmhead_workspace(contract, H, dev, workspace):
    import torch
    n = rlk_logp_lmhead_workspace_size(contract, H)
    if n == 0:
        check(rlk_logp_check_contract(contract) or RLK_ERR_UNSUPPORTED)
    if workspace is None:
        return torch.empty(n, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", n, ("uint8",))
    return workspace


def _rowwise(contract, targets, mask, **f32):
    """targets int64 [T], mask uint8/bool [T] (None in ignore_index mode) and FP32 [T] vectors."""
    T = contract.T
    _need(targets, "targets", 8 * T, _I64)
    _need(mask, "mask", T, _U8, optional=True)
    for name, t in f32.items():
        _need(t, name, 4 * T, _F32)


def _stream(stream):
    import torch
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


_workspaces = {}


def workspace_for(contract, device, stream=None):
    """A per-(device, stream) status workspace; calls on one stream never overlap."""
    import torch
    key = (str(device), _stream(stream))
    n = max(rlk_logp_workspace_size(contract), 256)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < n:
        ws = torch.zeros(n, dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def logp_fwd(contract, logits, targets, mask=None, partials=False, stream=None, out=None):
    """(logp, lse[, partials]) for BF16 ``logits`` [T, row_stride] (bf16/int16 storage) on the GPU."""
    import torch
    dev = logits.device
    T = contract.T
    _need_rows(logits, "logits", contract.T, contract.row_stride or contract.V_padded, contract.V_padded, _BF16)
    logp, lse = out if out is not None else (torch.empty(T, dtype=torch.float32, device=dev),
                                             torch.empty(T, dtype=torch.float32, device=dev))
    _rowwise(contract, targets, mask, logp=logp, lse=lse)
    part = torch.empty((T, contract.num_tiles, 2), dtype=torch.float32, device=dev) if partials else None
    ws = workspace_for(contract, dev, stream)
    check(rlk_logp_fwd(contract, _ptr(logits), _ptr(targets), _ptr(mask), _ptr(logp), _ptr(lse), _ptr(part),
                       _ptr(ws), _stream(stream)))
    return (logp, lse, part) if partials else (logp, lse)


def logp_bwd(contract, logits, targets, mask, lse, grad, dlogits=None, stream=None):
    """BF16 dlogits [T, row_stride] from the forward's LSE (the logits are re-read)."""
    dev = logits.device
    _need_rows(logits, "logits", contract.T, contract.row_stride or contract.V_padded, contract.V_padded, _BF16)
    _rowwise(contract, targets, mask, lse=lse, grad=grad)
    dlogits = _dlogits_out(contract, logits, dlogits)
    ws = workspace_for(contract, dev, stream)
    check(rlk_logp_bwd(contract, _ptr(logits), _ptr(targets), _ptr(mask), _ptr(lse), _ptr(grad),
                       _ptr(dlogits), None, None, _ptr(ws), _stream(stream)))
    return dlogits


def logp_fwd_entropy(contract, logits, targets, mask=None, stream=None):
    """(logp, lse, entropy) for BF16 ``logits`` on the GPU, in one pass; entropy of each row's softmax."""
    import torch
    dev = logits.device
    T = contract.T
    _need_rows(logits, "logits", contract.T, contract.row_stride or contract.V_padded, contract.V_padded, _BF16)
    _rowwise(contract, targets, mask)
    logp, lse, ent = (torch.empty(T, dtype=torch.float32, device=dev) for _ in range(3))
    ws = workspace_for(contract, dev, stream)
    check(rlk_logp_fwd_entropy(contract, _ptr(logits), _ptr(targets), _ptr(mask), _ptr(logp), _ptr(lse), _ptr(ent),
                               _ptr(ws), _stream(stream)))
    return logp, lse, ent


def grpo_loss(logp, advantage, mask, ref_logp=None, beta=0.0, stream=None):
    """(loss, grad_logp, active_count) of the token-mean GRPO loss (GPU tensors; loss and count are 1-element)."""
    import torch
    dev = logp.device
    T = logp.numel()
    _need(logp, "logp", 4 * T, _F32)
    _need(advantage, "advantage", 4 * T, _F32)
    _need(mask, "mask", T, _U8, optional=True)
    _need(ref_logp, "ref_logp", 4 * T, _F32, optional=True)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    count = torch.empty(1, dtype=torch.float32, device=dev)
    g = torch.empty(T, dtype=torch.float32, device=dev)
    check(rlk_grpo_loss(T, _ptr(logp), _ptr(advantage), _ptr(mask), _ptr(ref_logp), float(beta), _ptr(loss),
                        _ptr(g), _ptr(count), _stream(stream)))
    return loss, g, count


def grpo_fused_step(contract, logits, targets, mask, advantage, ref_logp=None, beta=0.0, dlogits=None,
                    entropy=False, stream=None, workspace=None):
    """The GRPO step in one pass over the logits: a dict of dlogits, logp, lse, grad (g), loss and active_count
    (1-element), and entropy if asked; bitwise logp_fwd -> grpo_loss -> logp_bwd(lse, g)."""
    import torch
    dev = logits.device
    T = contract.T
    _need_rows(logits, "logits", contract.T, contract.row_stride or contract.V_padded, contract.V_padded, _BF16)
    _rowwise(contract, targets, mask, advantage=advantage)
    _need(ref_logp, "ref_logp", 4 * T, _F32, optional=True)
    dlogits = _dlogits_out(contract, logits, dlogits)
    out = {"dlogits": dlogits}
    for k in ("logp", "lse", "grad"):
        out[k] = torch.empty(T, dtype=torch.float32, device=dev)
    out["entropy"] = torch.empty(T, dtype=torch.float32, device=dev) if entropy else None
    out["loss"] = torch.empty(1, dtype=torch.float32, device=dev)
    out["active_count"] = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(rlk_grpo_fused_workspace_size(contract), 256), dtype=torch.uint8, device=dev)
    else:
        _need(workspace, "workspace", rlk_grpo_fused_workspace_size(contract), ("uint8",))
    check(rlk_grpo_fused_step(contract, _ptr(logits), _ptr(targets), _ptr(mask), _ptr(advantage), _ptr(ref_logp),
                              float(beta), _ptr(dlogits), _ptr(out["logp"]), _ptr(out["lse"]), _ptr(out["grad"]),
                              _ptr(out["entropy"]), _ptr(out["loss"]), _ptr(out["active_count"]), _ptr(workspace),
                              _stream(stream)))
    return out


def logp_fwd_bwd(contract, logits, targets, mask, grad, dlogits=None, stream=None, out=None):
    """Fused single pass: (dlogits, logp, lse); each logits row is read from HBM once."""
    import torch
    dev = logits.device
    T = contract.T
    _need_rows(logits, "logits", contract.T, contract.row_stride or contract.V_padded, contract.V_padded, _BF16)
    dlogits = _dlogits_out(contract, logits, dlogits)
    logp, lse = out if out is not None else (torch.empty(T, dtype=torch.float32, device=dev),
                                             torch.empty(T, dtype=torch.float32, device=dev))
    _rowwise(contract, targets, mask, grad=grad, logp=logp, lse=lse)
    ws = workspace_for(contract, dev, stream)
    check(rlk_logp_bwd(contract, _ptr(logits), _ptr(targets), _ptr(mask), None, _ptr(grad), _ptr(dlogits),
                       _ptr(logp), _ptr(lse), _ptr(ws), _stream(stream)))
    return dlogits, logp, lse


def logp_fwd_bwd_entropy(contract, logits, targets, mask, grad, dlogits=None, stream=None):
    """Fused single pass plus each row's entropy: (dlogits, logp, lse, entropy)."""
    import torch
    dev = logits.device
    T = contract.T
    _need_rows(logits, "logits", contract.T, contract.row_stride or contract.V_padded, contract.V_padded, _BF16)
    _rowwise(contract, targets, mask, grad=grad)
    dlogits = _dlogits_out(contract, logits, dlogits)
    logp, lse, ent = (torch.empty(T, dtype=torch.float32, device=dev) for _ in range(3))
    ws = workspace_for(contract, dev, stream)
    check(rlk_logp_fwd_bwd_entropy(contract, _ptr(logits), _ptr(targets), _ptr(mask), _ptr(grad), _ptr(dlogits),
                                   _ptr(logp), _ptr(lse), _ptr(ent), _ptr(ws), _stream(stream)))
    return dlogits, logp, lse, ent


def logp_fwd_bwd_host(contract, logits, targets, mask, grad, device, chunk_rows=8192, dlogits=None,
                      staging=None):
    """Fused forward+backward of inputs in (pinned) host memory.

    Row chunks of ``logits`` (host, [T, row_stride] bf16/int16) are copied to
    the device on a copy stream while the previous chunk computes on the
    current stream; rows are independent, so the results are bitwise those of
    one call on the whole batch.  ``targets`` int64 [T], ``mask`` uint8 [T]
    (None in ignore_index mode) and ``grad`` float32 [T] are host tensors too.
    ``staging`` (device, like ``logits``) and ``dlogits`` (device) may be
    passed to reuse allocations.  Returns (dlogits on the device, logp and LSE
    in pinned host memory); the copies back are enqueued on the current
    stream, so synchronise it before reading them.  With contract.validate the
    call synchronises and checks every chunk's status.
    """
    import torch
    T = contract.T
    stride = contract.row_stride or contract.V_padded
    if logits.dim() != 2 or logits.shape[0] < T or logits.shape[1] < stride:
        raise ValueError(f"logits must be [T >= {T}, row_stride >= {stride}], not {list(logits.shape)}")
    for name, t in (("targets", targets), ("mask", mask), ("grad", grad)):
        if t is not None and t.numel() < T:
            raise ValueError(f"{name} must hold T = {T} values")
    comp = torch.cuda.current_stream(device)
    copy = torch.cuda.Stream(device)
    d_logits = staging if staging is not None else torch.empty(logits.shape, dtype=logits.dtype, device=device)
    d_dl = dlogits if dlogits is not None else torch.empty(logits.shape, dtype=logits.dtype, device=device)
    d_tgt = torch.empty(T, dtype=torch.int64, device=device)
    d_mask = torch.empty(T, dtype=torch.uint8, device=device) if mask is not None else None
    d_g = torch.empty(T, dtype=torch.float32, device=device)
    d_logp = torch.empty(T, dtype=torch.float32, device=device)
    d_lse = torch.empty(T, dtype=torch.float32, device=device)
    h_logp = torch.empty(T, dtype=torch.float32, pin_memory=True)
    h_lse = torch.empty(T, dtype=torch.float32, pin_memory=True)
    starts = list(range(0, T, chunk_rows))
    ws = torch.zeros(max(len(starts), 1) * 256, dtype=torch.uint8, device=device)  # a status word per chunk
    copy.wait_stream(comp)  # the buffers above exist before the copy stream writes them
    with torch.cuda.stream(copy):
        d_tgt.copy_(targets, non_blocking=True)
        if mask is not None:
            d_mask.copy_(mask, non_blocking=True)
        d_g.copy_(grad, non_blocking=True)
    for i, r0 in enumerate(starts):
        r1 = min(T, r0 + chunk_rows)
        with torch.cuda.stream(copy):
            d_logits[r0:r1].copy_(logits[r0:r1], non_blocking=True)
            landed = torch.cuda.Event()
            landed.record(copy)
        comp.wait_event(landed)
        c = contract.replace(T=r1 - r0, validate=0)
        check(rlk_logp_bwd(c, d_logits[r0].data_ptr(), d_tgt[r0:].data_ptr(),
                           None if d_mask is None else d_mask[r0:].data_ptr(), None, d_g[r0:].data_ptr(),
                           d_dl[r0].data_ptr(), d_logp[r0:].data_ptr(), d_lse[r0:].data_ptr(),
                           ws[i * 256:].data_ptr(), comp.cuda_stream))
    comp.wait_stream(copy)
    h_logp.copy_(d_logp, non_blocking=True)
    h_lse.copy_(d_lse, non_blocking=True)
    if contract.validate:
        for i in range(len(starts)):
            check(rlk_logp_workspace_status(ws[i * 256:].data_ptr(), comp.cuda_stream))
    return d_dl, h_logp, h_lse


def logp_fused_lmhead(contract, hidden, weight, targets, mask=None, grad=None, stream=None, workspace=None,
                      dweight_dtype="bf16"):
    """Fused lm_head on BF16 hidden [T, H] and weight [V_padded, H] (GPU tensors).

    Forward only: returns (logp, lse).  With ``grad`` (FP32 [T]): returns
    (logp, lse, dhidden [T, H] BF16, dweight [V_padded, H]); ``dweight_dtype``
    "bf16" (default), "f32", or "both" (then dweight is a (f32, bf16) pair).
    """
    import torch
    dev = hidden.device
    H = _lmhead_operands(contract, hidden, weight)
    T = contract.T
    _rowwise(contract, targets, mask)
    _need(grad, "grad", 4 * T, _F32, optional=True)
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    dh = dwf = dwb = None
    if grad is not None:
        if dweight_dtype not in ("bf16", "f32", "both"):
            raise ValueError("dweight_dtype must be bf16, f32 or both")
        dh = torch.empty_like(hidden)
        if dweight_dtype in ("f32", "both"):
            dwf = torch.empty(weight.shape, dtype=torch.float32, device=dev)
        if dweight_dtype in ("bf16", "both"):
            dwb = torch.empty_like(weight)
    ws = _lmhead_workspace(contract, H, dev, workspace)
    check(rlk_logp_fused_lmhead(contract, _ptr(hidden), H, _ptr(weight), _ptr(targets), _ptr(mask), _ptr(grad),
                                _ptr(logp), _ptr(lse), _ptr(dh), _ptr(dwf), _ptr(dwb), _ptr(ws), _stream(stream)))
    if grad is None:
        return logp, lse
    dw = {"bf16": dwb, "f32": dwf, "both": (dwf, dwb)}[dweight_dtype]
    return logp, lse, dh, dw


def logp_fused_lmhead_bwd(contract, hidden, weight, targets, mask, lse, grad, stream=None, workspace=None,
                          dweight_dtype="bf16"):
    """(dhidden [T, H] BF16, dweight [V_padded, H]) from the forward's LSE; ``dweight_dtype`` as for
    logp_fused_lmhead."""
    import torch
    dev = hidden.device
    H = _lmhead_operands(contract, hidden, weight)
    _rowwise(contract, targets, mask, lse=lse, grad=grad)
    if dweight_dtype not in ("bf16", "f32", "both"):
        raise ValueError("dweight_dtype must be bf16, f32 or both")
    dh = torch.empty_like(hidden)
    dwf = torch.empty(weight.shape, dtype=torch.float32, device=dev) if dweight_dtype in ("f32", "both") else None
    dwb = torch.empty_like(weight) if dweight_dtype in ("bf16", "both") else None
    ws = _lmhead_workspace(contract, H, dev, workspace)
    check(rlk_logp_fused_lmhead_bwd(contract, _ptr(hidden), H, _ptr(weight), _ptr(targets), _ptr(mask), _ptr(lse),
                                    _ptr(grad), _ptr(dh), _ptr(dwf), _ptr(dwb), _ptr(ws), _stream(stream)))
    return dh, {"bf16": dwb, "f32": dwf, "both": (dwf, dwb)}[dweight_dtype]


def logp_fused_lmhead_keep(contract, hidden, weight, targets, mask=None, stream=None, workspace=None):
    """(logp, lse, logits): the fused lm_head forward that also keeps its FP32 logits [T, V_padded] for
    logp_fused_lmhead_bwd_kept (T * V_padded * 4 bytes)."""
    import torch
    dev = hidden.device
    H = _lmhead_operands(contract, hidden, weight)
    T = contract.T
    _rowwise(contract, targets, mask)
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    logits = torch.empty((T, weight.shape[0]), dtype=torch.float32, device=dev)
    ws = _lmhead_workspace(contract, H, dev, workspace)
    check(rlk_logp_fused_lmhead_keep(contract, _ptr(hidden), H, _ptr(weight), _ptr(targets), _ptr(mask), _ptr(logp),
                                     _ptr(lse), _ptr(logits), _ptr(ws), _stream(stream)))
    return logp, lse, logits


def logp_fused_lmhead_bwd_kept(contract, hidden, weight, targets, mask, lse, logits, grad, stream=None, workspace=None,
                               dweight_dtype="bf16"):
    """(dhidden, dweight) from the logits and LSE of logp_fused_lmhead_keep; bitwise logp_fused_lmhead_bwd's."""
    import torch
    dev = hidden.device
    H = _lmhead_operands(contract, hidden, weight)
    _rowwise(contract, targets, mask, lse=lse, grad=grad)
    _need(logits, "logits", 4 * contract.T * contract.V_padded, _F32)
    if dweight_dtype not in ("bf16", "f32", "both"):
        raise ValueError("dweight_dtype must be bf16, f32 or both")
    dh = torch.empty_like(hidden)
    dwf = torch.empty(weight.shape, dtype=torch.float32, device=dev) if dweight_dtype in ("f32", "both") else None
    dwb = torch.empty_like(weight) if dweight_dtype in ("bf16", "both") else None
    ws = _lmhead_workspace(contract, H, dev, workspace)
    check(rlk_logp_fused_lmhead_bwd_kept(contract, _ptr(hidden), H, _ptr(weight), _ptr(targets), _ptr(mask),
                                         _ptr(lse), _ptr(logits), _ptr(grad), _ptr(dh), _ptr(dwf), _ptr(dwb), _ptr(ws),
                                         _stream(stream)))
    return dh, {"bf16": dwb, "f32": dwf, "both": (dwf, dwb)}[dweight_dtype]


# ------------------------------------------------------------------ vocabulary shards (one rank's calls)

def shard_workspace(contract, device):
    import torch
    n = rlk_logp_shard_workspace_size(contract)
    if n == 0:
        check(rlk_logp_check_shard_contract(contract, 0) or RLK_ERR_INVALID_ARG)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def shard_fwd(contract, shard, logits_shard, targets, mask=None, stream=None, workspace=None):
    """(partials [T, num_tiles/tp, 2], target_logit [T]) of one vocabulary shard (GPU tensors)."""
    import torch
    dev = logits_shard.device
    T = contract.T
    vs = contract.V_padded // contract.virtual_tp
    _need_rows(logits_shard, "logits_shard", T, contract.row_stride or vs, vs, _BF16)
    _rowwise(contract, targets, mask)
    part = torch.empty((T, contract.num_tiles // contract.virtual_tp, 2), dtype=torch.float32, device=dev)
    xt = torch.empty(T, dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else shard_workspace(contract, dev)
    check(rlk_logp_shard_fwd(contract, shard, _ptr(logits_shard), _ptr(targets), _ptr(mask), _ptr(part), _ptr(xt),
                             _ptr(ws), _stream(stream)))
    return part, xt


def fold_gathered(contract, gathered_partials, gathered_target_logit, targets, mask=None, stream=None,
                  workspace=None):
    """(logp, lse) from every shard's partials [tp, T, num_tiles/tp, 2] and target logits [tp, T]."""
    import torch
    dev = gathered_partials.device
    T = contract.T
    _need(gathered_partials, "gathered_partials", 8 * T * contract.num_tiles, _F32)
    _need(gathered_target_logit, "gathered_target_logit", 4 * T * contract.virtual_tp, _F32)
    _rowwise(contract, targets, mask)
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    ws = workspace if workspace is not None else shard_workspace(contract, dev)
    check(rlk_logp_fold(contract, _ptr(gathered_partials), _ptr(gathered_target_logit), _ptr(targets), _ptr(mask),
                        _ptr(logp), _ptr(lse), _ptr(ws), _stream(stream)))
    return logp, lse


def shard_bwd(contract, shard, logits_shard, targets, mask, lse, grad, dlogits=None, stream=None, workspace=None):
    """BF16 dlogits of one vocabulary shard [T, row_stride] (columns [0, V_padded/tp) written)."""
    dev = logits_shard.device
    vs = contract.V_padded // contract.virtual_tp
    stride = contract.row_stride or vs
    _need_rows(logits_shard, "logits_shard", contract.T, stride, vs, _BF16)
    _rowwise(contract, targets, mask, lse=lse, grad=grad)
    dlogits = _dlogits_out(contract, logits_shard, dlogits, stride=stride, width=vs)
    ws = workspace if workspace is not None else shard_workspace(contract, dev)
    check(rlk_logp_shard_bwd(contract, shard, _ptr(logits_shard), _ptr(targets), _ptr(mask), _ptr(lse), _ptr(grad),
                             _ptr(dlogits), _ptr(ws), _stream(stream)))
    return dlogits
