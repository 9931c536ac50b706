"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle, compare.

The oracle side always gets host-generated inputs (synth host build); the
GPU side gets the same bits copied to the device, or generated there by the
synth device build (checked bit-identical in test_parity_gpu).
"""
import hashlib
import json
import os

import numpy as np
import torch

import oracle
import vocab_selected_token_tile_gb300 as rlk

LSE_TOL = 1e-4     # LSE and logp max abs error against the FP64 oracle
ENT_TOL = 1e-4     # entropy max abs error: H = LSE - T/S; FP32 rounding of T/S at |E[x]| <= 20 is ~1e-5
DL_TOL = 1e-2      # dlogits max abs error (BF16 output)


def report(kind, value):
    """Appends a measured error to the JSON-lines file named by RLK_PARITY_REPORT, if set."""
    path = os.environ.get("RLK_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                "kind": kind, "max_abs": float(value)}) + "\n")


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def sha(t):
    return hashlib.sha256(t.detach().cpu().numpy().tobytes()).hexdigest()


def f32_bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def oracle_fwd(bits, tgt, active, v_real, chunk=128):
    """Oracle (logp, lse) over row chunks (bounded host memory)."""
    R = bits.shape[0]
    logp = np.zeros(R)
    lse = np.zeros(R)
    for r0 in range(0, R, chunk):
        r1 = min(R, r0 + chunk)
        logp[r0:r1], lse[r0:r1] = oracle.selected_logp(bits[r0:r1], tgt[r0:r1], active[r0:r1], v_real)
    return logp, lse


def check_fwd(bits, tgt, active, v_real, logp, lse, tol=LSE_TOL):
    """Element-wise parity of GPU (logp, lse) with the oracle; bit-exact masking."""
    ref_logp, ref_lse = oracle_fwd(bits, tgt, active, v_real)
    logp = np.asarray(logp, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    err_lse = np.max(np.abs(lse[fin] - ref_lse[fin])) if fin.any() else 0.0
    err_logp = np.max(np.abs(logp[active & fin] - ref_logp[active & fin])) if (active & fin).any() else 0.0
    report("lse", err_lse)
    report("logp", err_logp)
    assert err_lse <= tol, f"LSE max abs {err_lse}"
    assert err_logp <= tol, f"logp max abs {err_logp}"
    # inactive rows: exactly +0.0
    assert np.all(f32_bits(logp[~active]) == 0)
    return err_lse, err_logp


def check_dlogits(bits, tgt, active, g, v_real, v_padded, dl_bits, rows=None):
    """dlogits parity: max abs <= 1e-2 and within one BF16 rounding of the FP64 value
    (2^-8 relative) plus 4e-6 |g| for the FP32 arithmetic; padding and inactive rows
    exactly 0x0000."""
    rows = np.arange(bits.shape[0]) if rows is None else rows
    worst = 0.0
    for r0 in range(0, len(rows), 64):
        rr = rows[r0:r0 + 64]
        ref = oracle.dlogits(bits[rr], tgt[rr], active[rr], g[rr], v_real, v_padded)
        got = oracle.bf16_bits_to_f64(dl_bits[rr][:, :v_padded])
        err = np.abs(got - ref)
        worst = max(worst, float(err.max()))
        bound = np.ldexp(np.abs(ref), -8) + 4e-6 * np.abs(g[rr])[:, None] + 1e-30
        assert np.all(err <= bound), f"dlogits outside the BF16 rounding bound at rows {rr[np.any(err > bound, 1)]}"
        assert np.all(dl_bits[rr][:, v_real:v_padded] == 0), "padded columns must be exactly 0"
        assert np.all(dl_bits[rr][~active[rr]][:, :v_padded] == 0), "inactive rows must be exactly 0"
    report("dlogits", worst)
    assert worst <= DL_TOL
    return worst


def contract(T, v_real, v_padded, nt, vtp=1, mode=rlk.MASK_EXPLICIT, stride=0, validate=1, **kw):
    return rlk.Contract(T=T, V_real=v_real, V_padded=v_padded, num_tiles=nt, virtual_tp=vtp, mask_mode=mode,
                        ignore_index=-100, validate=validate, row_stride=stride, **kw)


def check_entropy(bits, v_real, ent, rows=None, tol=ENT_TOL):
    """Entropy parity with the oracle: NaN exactly where the oracle's is NaN, max abs <= tol elsewhere."""
    rows = np.arange(bits.shape[0]) if rows is None else rows
    ref = oracle.entropy(bits[rows], v_real)
    got = np.asarray(ent, dtype=np.float64)[rows]
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    err = float(np.max(np.abs(got[fin] - ref[fin]))) if fin.any() else 0.0
    report("entropy", err)
    assert err <= tol, f"entropy max abs {err}"
    return err
