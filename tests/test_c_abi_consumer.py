"""The C ABI from a plain C99 program (tests/c_abi_consumer.c): no Python in the call path.

CPU: the header compiles as strict C99 (-pedantic -Werror) and the host-only
calls answer as documented.  GPU: the program copies seeded inputs into
cudaMalloc'ed buffers and runs rlk_logp_fwd and the fused rlk_logp_bwd; its
outputs match the FP64 oracle within the stated tolerances and are bitwise
those of the Python binding on the same inputs.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import vocab_selected_token_tile_gb300 as rlk

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "c_abi_consumer.c")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_consumer(out_dir, with_cuda):
    lib_dir = os.path.dirname(rlk._build.LIB)
    exe = os.path.join(out_dir, "c_abi_consumer")
    argv = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-O1", "-I", os.path.join(ROOT, "include"),
            SRC, "-o", exe, "-L", lib_dir, "-lrlk_logp", "-Wl,-rpath," + lib_dir]
    if with_cuda:  # the CUDA runtime's own headers need C11 (anonymous unions), not pedantic C99
        argv = [a for a in argv if a not in ("-pedantic", "-Werror")]
        argv[1:2] = ["-std=c11", "-DRLK_WITH_CUDA", "-I", os.path.join(CUDA_HOME, "include")]
        argv += ["-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA_HOME, "lib64")]
    r = subprocess.run(argv, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_c99_and_host_calls_answer(built, tmp_path):
    exe = compile_consumer(str(tmp_path), with_cuda=False)
    r = subprocess.run([exe, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "host ok"


@pytest.mark.gpu
def test_c_program_runs_the_path(built, tmp_path):
    import torch
    import synth
    from parity import check_dlogits, check_fwd, contract, to_dev
    if not torch.cuda.is_available():  # pragma: no cover
        pytest.skip("needs a CUDA GPU")
    T, vr, vp, nt, vtp = 70, 30001, 30016, 64, 4  # ragged real end; 469-column tiles (not 8-aligned)
    bits = synth.logits_host(0, T, vp, vp, vr, seed=5, sigma=3.0, nspikes=2, garbage=True)
    tgt = synth.targets(T, vr, 5)
    rng = np.random.default_rng(5)
    mask = (rng.random(T) < 0.75).astype(np.uint8)
    tgt = np.where(mask != 0, tgt, -7)
    g = np.where(mask != 0, rng.standard_normal(T), 0.0).astype(np.float32)
    inp, out = tmp_path / "in", tmp_path / "out"
    inp.mkdir()
    out.mkdir()
    bits.astype(np.uint16).tofile(inp / "logits.bin")
    tgt.astype(np.int64).tofile(inp / "targets.bin")
    mask.tofile(inp / "mask.bin")
    g.tofile(inp / "grad.bin")
    exe = compile_consumer(str(tmp_path), with_cuda=True)
    r = subprocess.run([exe, "run", str(T), str(vr), str(vp), str(nt), str(vtp), str(inp), str(out)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    logp = np.fromfile(out / "logp.bin", dtype=np.float32)
    lse = np.fromfile(out / "lse.bin", dtype=np.float32)
    dl = np.fromfile(out / "dlogits.bin", dtype=np.uint16).reshape(T, vp)
    active = mask != 0
    check_fwd(bits, tgt, active, vr, logp, lse)
    check_dlogits(bits, tgt, active, g, vr, vp, dl)
    assert np.array_equal(np.fromfile(out / "logp_fused.bin", dtype=np.uint32), logp.view(np.uint32))
    assert np.array_equal(np.fromfile(out / "lse_fused.bin", dtype=np.uint32), lse.view(np.uint32))
    # bitwise the binding's results on the same inputs
    c = contract(T, vr, vp, nt, vtp)
    dt, dm, dg = (torch.from_numpy(a).cuda() for a in (tgt, mask, g))
    dlt, lp, ls = rlk.logp_fwd_bwd(c, to_dev(bits), dt, dm, dg)
    torch.cuda.synchronize()
    assert np.array_equal(lp.cpu().numpy().view(np.uint32), logp.view(np.uint32))
    assert np.array_equal(ls.cpu().numpy().view(np.uint32), lse.view(np.uint32))
    assert np.array_equal(dlt.cpu().numpy().view(np.uint16), dl)
