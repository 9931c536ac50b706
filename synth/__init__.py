"""Seeded synthetic inputs for the selected-token log-probability path.

This module is the only code that both the CPU oracle's callers and the CUDA
path's callers share.  It holds no log-probability arithmetic: it turns
(seed, stream, counter) into BF16 logits, targets, masks and upstream
gradients, identically on the host (``*_host``) and on the GPU
(``*_device``).  See ``synth_core.h`` for the generator's definition.

The workloads it can build are in :mod:`synth.workloads`.
"""
import ctypes
import os

import numpy as np

from . import _build

_host = None
_dev = None

STREAM_ADVANTAGE = 7
STREAM_HIDDEN = 8
STREAM_WEIGHT = 9


def _load_host():
    global _host
    if _host is None:
        if not os.path.exists(_build.HOST_LIB):
            raise RuntimeError(f"synth host library missing: {_build.HOST_LIB}; run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.HOST_LIB)
        i64, u64, f32, i32, u32 = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_float,
                                   ctypes.c_int32, ctypes.c_uint32)
        vp = ctypes.c_void_p
        lib.syn_host_logits.argtypes = [vp, i64, i64, i64, i64, i64, u64, f32, i32, f32, i32, i32]
        lib.syn_host_logits.restype = None
        lib.syn_host_normal_bf16.argtypes = [vp, i64, i64, i64, u64, u32, f32, i32]
        lib.syn_host_normal_bf16.restype = None
        lib.syn_host_targets.argtypes = [vp, i64, i64, u64, u64, i64]
        lib.syn_host_targets.restype = None
        lib.syn_host_response_mask.argtypes = [vp, vp, i64, i64, i64, i64, i64, u64]
        lib.syn_host_response_mask.restype = None
        lib.syn_host_normal_f64.argtypes = [vp, i64, u64, u32]
        lib.syn_host_normal_f64.restype = None
        _host = lib
    return _host


def _load_dev():
    global _dev
    if _dev is None:
        if not os.path.exists(_build.DEV_LIB):
            raise RuntimeError(f"synth device library missing: {_build.DEV_LIB}; run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.DEV_LIB)
        i64, u64, f32, i32, u32 = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_float,
                                   ctypes.c_int32, ctypes.c_uint32)
        vp = ctypes.c_void_p
        lib.syn_dev_logits.argtypes = [vp, i64, i64, i64, i64, i64, u64, f32, i32, f32, i32, vp]
        lib.syn_dev_logits.restype = ctypes.c_int
        lib.syn_dev_normal_bf16.argtypes = [vp, i64, i64, i64, u64, u32, f32, vp]
        lib.syn_dev_normal_bf16.restype = ctypes.c_int
        _dev = lib
    return _dev


def scale_of(sigma):
    """The float32 multiplier that turns a centred IH12 integer into sigma * N(0, 1)."""
    return float(np.float32(sigma / 65536.0))


def logits_host(row0, nrows, row_stride, v_padded, v_real, seed, sigma,
                nspikes=0, spike=15.0, garbage=False, nthreads=0):
    """BF16 bits (uint16) of rows [row0, row0+nrows) of a [T, row_stride] logits buffer."""
    out = np.zeros((nrows, row_stride), dtype=np.uint16)
    if nrows:
        _load_host().syn_host_logits(out.ctypes.data, row0, nrows, row_stride, v_padded, v_real,
                                     seed, scale_of(sigma), nspikes, spike, int(garbage), nthreads)
    return out


def logits_device(dst, row0, nrows, row_stride, v_padded, v_real, seed, sigma,
                  nspikes=0, spike=15.0, garbage=False, stream=None):
    """Fill a CUDA tensor (int16/uint16/bf16 storage, nrows*row_stride elements) like logits_host."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    err = _load_dev().syn_dev_logits(dst.data_ptr(), row0, nrows, row_stride, v_padded, v_real, seed,
                                     scale_of(sigma), nspikes, spike, int(garbage), s.cuda_stream)
    if err:
        raise RuntimeError(f"syn_dev_logits failed with cudaError {err}")


def normal_bf16_host(row0, nrows, cols, seed, stream_id, sigma, nthreads=0):
    """BF16 bits of rows [row0, row0+nrows) of a dense [*, cols] sigma * N(0, 1) matrix."""
    out = np.zeros((nrows, cols), dtype=np.uint16)
    if nrows:
        _load_host().syn_host_normal_bf16(out.ctypes.data, row0, nrows, cols, seed, stream_id,
                                          scale_of(sigma), nthreads)
    return out


def normal_bf16_device(dst, row0, nrows, cols, seed, stream_id, sigma, stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    err = _load_dev().syn_dev_normal_bf16(dst.data_ptr(), row0, nrows, cols, seed, stream_id,
                                          scale_of(sigma), s.cuda_stream)
    if err:
        raise RuntimeError(f"syn_dev_normal_bf16 failed with cudaError {err}")


def targets(T, v_real, seed, ignore_frac=0.0, ignore_index=-100):
    """int64 targets uniform in [0, v_real); a fraction ignore_frac replaced by ignore_index."""
    out = np.zeros(T, dtype=np.int64)
    thresh = int(ignore_frac * 4294967296.0) if ignore_frac > 0 else 0
    if T:
        _load_host().syn_host_targets(out.ctypes.data, T, v_real, seed, thresh, ignore_index)
    return out


def response_mask(batch, seq, prompt, len_min, len_max, seed):
    """uint8 [batch*seq] mask: positions [prompt, prompt+L_b) active, L_b ~ U{len_min..len_max}."""
    out = np.zeros(batch * seq, dtype=np.uint8)
    lens = np.zeros(batch, dtype=np.int64)
    if batch * seq:
        _load_host().syn_host_response_mask(out.ctypes.data, lens.ctypes.data, batch, seq, prompt,
                                            len_min, len_max, seed)
    return out, lens


def normal_f64(n, seed, stream_id):
    """n approximately standard normal doubles (IH12 / 65536, exact)."""
    out = np.zeros(n, dtype=np.float64)
    if n:
        _load_host().syn_host_normal_f64(out.ctypes.data, n, seed, stream_id)
    return out
