"""The C ABI without a GPU: symbols, struct layout, host-side contract validation.

Nothing here launches work; every call either validates on the host or
returns before touching a device.
"""
import ctypes
import os
import re

import pytest

import vocab_selected_token_tile_gb300 as rlk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "rlk_logp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rlk_\w+)\s*\(", text)))


def test_library_exports_every_declared_function(built):
    lib = rlk.library()
    names = header_functions()
    assert "rlk_logp_fwd" in names and "rlk_logp_bwd" in names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in rlk_logp.h but not exported"
    assert set(names) <= set(rlk.EXPORTED) | {n for n in names if n.startswith("rlk_")}


def test_exports_are_exactly_the_c_abi(built):
    # the shared object exports only extern "C" rlk_* symbols (hidden visibility otherwise)
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", rlk._build.LIB], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert syms, out
    assert {s for s in syms if not s.startswith("rlk_")} == set(), syms
    assert set(header_functions()) <= syms


def test_contract_struct_layout():
    assert ctypes.sizeof(rlk.Contract) == 64
    assert rlk.Contract.ignore_index.offset == 48 and rlk.Contract.num_tiles.offset == 32


def ok_contract(**kw):
    base = dict(T=8, V_real=151936, V_padded=152576, num_tiles=64, virtual_tp=2)
    base.update(kw)
    return rlk.Contract(**base)


@pytest.mark.parametrize("kw,status", [
    ({}, rlk.RLK_OK),
    (dict(virtual_tp=8), rlk.RLK_OK),
    (dict(V_padded=151936, V_real=151936), rlk.RLK_OK),
    (dict(T=0), rlk.RLK_OK),
    (dict(num_tiles=7), rlk.RLK_ERR_NON_TILEABLE),          # 7 does not divide 152576
    (dict(num_tiles=2, virtual_tp=4), rlk.RLK_ERR_NON_TILEABLE),
    (dict(virtual_tp=3), rlk.RLK_ERR_UNSUPPORTED),
    (dict(virtual_tp=16), rlk.RLK_ERR_UNSUPPORTED),
    (dict(num_tiles=1, virtual_tp=1), rlk.RLK_ERR_UNSUPPORTED),  # tile wider than 16384 columns
    (dict(num_tiles=2048, V_padded=2048 * 8, V_real=2048 * 8), rlk.RLK_ERR_UNSUPPORTED),
    (dict(V_real=0), rlk.RLK_ERR_INVALID_ARG),
    (dict(V_padded=100, V_real=101, num_tiles=4, virtual_tp=1), rlk.RLK_ERR_INVALID_ARG),
    (dict(T=-1), rlk.RLK_ERR_INVALID_ARG),
    (dict(row_stride=152576 + 4), rlk.RLK_ERR_MISALIGNED),
    (dict(row_stride=152000), rlk.RLK_ERR_INVALID_ARG),
    (dict(mask_mode=2), rlk.RLK_ERR_INVALID_ARG),
    (dict(validate=2), rlk.RLK_ERR_INVALID_ARG),
    (dict(wait_timeout_ns=-5), rlk.RLK_ERR_INVALID_ARG),
])
def test_check_contract(built, kw, status):
    c = ok_contract(**kw)
    assert rlk.rlk_logp_check_contract(c) == status
    if status != rlk.RLK_OK:
        assert rlk.rlk_last_error_message() != ""
        assert rlk.rlk_logp_workspace_size(c) == 0
    else:
        assert rlk.rlk_logp_workspace_size(c) >= 4


def test_null_contract(built):
    assert rlk.library().rlk_logp_check_contract(None) == rlk.RLK_ERR_INVALID_ARG


def test_calls_fail_closed_before_any_device_work(built):
    c = ok_contract()
    # missing pointers are rejected on the host, before any CUDA call
    assert rlk.rlk_logp_fwd(c, None, None, None, None, None, None, None, None) == rlk.RLK_ERR_INVALID_ARG
    assert "logits" in rlk.rlk_last_error_message()
    assert rlk.rlk_logp_fwd(c, 0x1008, 0x2000, 0x3000, 0x4000, 0x5000, None, 0x6000, None) == rlk.RLK_ERR_MISALIGNED
    # ignore-index mode takes no mask, explicit mode needs one
    ci = ok_contract(mask_mode=rlk.MASK_IGNORE_INDEX)
    assert rlk.rlk_logp_fwd(ci, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, None, 0x6000, None) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_fwd(c, 0x1000, 0x2000, None, 0x4000, 0x5000, None, 0x6000, None) == rlk.RLK_ERR_INVALID_ARG
    # backward: lse_in excludes forward outputs; the fused form needs them
    assert rlk.rlk_logp_bwd(c, 0x1000, 0x2000, 0x3000, 0x7000, 0x8000, 0x9000, 0xA000, None, 0x6000,
                            None) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_bwd(c, 0x1000, 0x2000, 0x3000, None, 0x8000, 0x9000, None, None, 0x6000,
                            None) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_bwd(c, 0x1000, 0x2000, 0x3000, None, 0x8000, 0x9008, 0xA000, 0xB000, 0x6000,
                            None) == rlk.RLK_ERR_MISALIGNED
    # an empty batch is a no-op
    assert rlk.rlk_logp_fwd(ok_contract(T=0), None, None, None, None, None, None, None, None) == rlk.RLK_OK


def test_status_strings(built):
    for code in range(9):
        assert rlk.rlk_status_string(code).startswith("RLK_")
    assert rlk.rlk_status_string(99) == "RLK_ERR_UNKNOWN"


def test_product_path_has_no_fallback():
    # the package never imports the oracle or the generator
    import inspect
    src = inspect.getsource(rlk)
    assert "import oracle" not in src and "import synth" not in src
    csrc = os.path.join(ROOT, "vocab_selected_token_tile_gb300", "csrc")
    for f in os.listdir(csrc):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            assert "oracle" not in open(os.path.join(csrc, f)).read().lower()


@pytest.mark.parametrize("name,value", [("RLK_ROW_BUFS", "3"), ("RLK_ROW_BUFS", "16"), ("RLK_CTAS_PER_SM", "3"),
                                        ("RLK_FUSED_SKEW", "9"), ("RLK_FUSED_SKEW", "x"),
                                        ("RLK_FUSED_SCHEDULE", "fast"), ("RLK_TPS", "2"), ("RLK_MAX_SLOTS", "7"),
                                        ("RLK_LMHEAD_PAIR", "2")])
def test_off_model_planner_overrides_fail_closed(built, monkeypatch, name, value):
    """Planner overrides outside the ring shapes the protocol model replays are
    rejected on the host, before any device is touched."""
    c = rlk.Contract(T=16, V_real=1000, V_padded=1024, num_tiles=4)
    assert rlk.rlk_logp_check_contract(c) == rlk.RLK_OK
    monkeypatch.setenv(name, value)
    assert rlk.rlk_logp_check_contract(c) == rlk.RLK_ERR_UNSUPPORTED
    assert name in rlk.rlk_last_error_message()
    assert rlk.rlk_logp_workspace_size(c) == 0


@pytest.mark.parametrize("name,value", [("RLK_ROW_BUFS", "2"), ("RLK_ROW_BUFS", "8"), ("RLK_CTAS_PER_SM", "1"),
                                        ("RLK_FUSED_SKEW", "0"), ("RLK_FUSED_SKEW", "-1"),
                                        ("RLK_FUSED_SCHEDULE", "resident"), ("RLK_FUSED_SCHEDULE", "l2")])
def test_modelled_planner_overrides_are_accepted(built, monkeypatch, name, value):
    c = rlk.Contract(T=16, V_real=1000, V_padded=1024, num_tiles=4)
    monkeypatch.setenv(name, value)
    assert rlk.rlk_logp_check_contract(c) == rlk.RLK_OK


def test_new_entry_points_fail_closed_on_the_host(built):
    """The shard calls, the gathered fold and the lm_head backward check their arguments before any
    CUDA call: an empty batch is a no-op, missing or misaligned pointers and bad shard indices fail."""
    c = ok_contract(virtual_tp=8)
    z = ok_contract(T=0, virtual_tp=8)
    assert rlk.rlk_logp_shard_fwd(z, 0, None, None, None, None, None, None, None) == rlk.RLK_OK
    assert rlk.rlk_logp_fold(z, None, None, None, None, None, None, None, None) == rlk.RLK_OK
    assert rlk.rlk_logp_shard_bwd(z, 0, None, None, None, None, None, None, None, None) == rlk.RLK_OK
    assert rlk.rlk_logp_check_shard_contract(c, 7) == rlk.RLK_OK
    assert rlk.rlk_logp_check_shard_contract(c, 8) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_shard_workspace_size(c) >= 256
    assert rlk.rlk_logp_shard_fwd(c, 8, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, None) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_shard_fwd(c, 0, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, None) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_shard_fwd(c, 0, 0x1008, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, None) == rlk.RLK_ERR_MISALIGNED
    assert rlk.rlk_logp_shard_fwd(c, 0, 0x1000, 0x2000, 0x3000, None, 0x5000, 0x6000, None) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_fold(c, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, None) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_fold(c, 0x1000, 0x2000, 0x3000, 0x4000, None, 0x6000, 0x7000, None) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_shard_bwd(c, 0, 0x1000, 0x2000, 0x3000, None, 0x5000, 0x6000, 0x7000,
                                  None) == rlk.RLK_ERR_INVALID_ARG
    assert rlk.rlk_logp_shard_bwd(c, 0, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6008, 0x7000,
                                  None) == rlk.RLK_ERR_MISALIGNED
    # the lm_head backward from a given LSE
    cl = ok_contract(virtual_tp=2)
    assert rlk.rlk_logp_fused_lmhead_bwd(ok_contract(T=0), None, 128, None, None, None, None, None, None, None,
                                         None, None, None) == rlk.RLK_OK
    assert rlk.rlk_logp_fused_lmhead_bwd(cl, 0x1000, 100, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, None,
                                         0x8000, 0x9000, None) == rlk.RLK_ERR_UNSUPPORTED  # H not a multiple of 64
    assert rlk.rlk_logp_fused_lmhead_bwd(cl, 0x1000, 128, 0x2000, 0x3000, 0x4000, None, 0x6000, 0x7000, None,
                                         0x8000, 0x9000, None) == rlk.RLK_ERR_INVALID_ARG  # no lse_in
    assert rlk.rlk_logp_fused_lmhead_bwd(cl, 0x1000, 128, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, None,
                                         None, 0x9000, None) == rlk.RLK_ERR_INVALID_ARG  # no dweight output
    assert rlk.rlk_logp_fused_lmhead(cl, 0x1000, 128, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000,
                                     0x9008, None, 0xA000, None) == rlk.RLK_ERR_MISALIGNED  # FP32 dweight
    # the lm_head forward keeping its logits, and the backward from them
    assert rlk.rlk_logp_fused_lmhead_keep(ok_contract(T=0), None, 128, None, None, None, None, None, None, None,
                                          None) == rlk.RLK_OK
    assert rlk.rlk_logp_fused_lmhead_keep(cl, 0x1000, 128, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, None, 0xA000,
                                          None) == rlk.RLK_ERR_INVALID_ARG  # no logits_f32
    assert rlk.rlk_logp_fused_lmhead_keep(cl, 0x1000, 128, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7008, 0xA000,
                                          None) == rlk.RLK_ERR_MISALIGNED
    assert rlk.rlk_logp_fused_lmhead_keep(cl, 0x1000, 192, 0x2000, 0x3000, None, 0x5000, 0x6000, 0x7000, 0xA000,
                                          None) == rlk.RLK_ERR_INVALID_ARG  # explicit mask mode, no mask
    assert rlk.rlk_logp_fused_lmhead_bwd_kept(ok_contract(T=0), None, 128, None, None, None, None, None, None, None,
                                              None, None, None, None) == rlk.RLK_OK
    assert rlk.rlk_logp_fused_lmhead_bwd_kept(cl, 0x1000, 128, 0x2000, 0x3000, 0x4000, 0x5000, None, 0x6000, 0x7000,
                                              None, 0x9000, 0xA000, None) == rlk.RLK_ERR_INVALID_ARG  # no logits_f32
    assert rlk.rlk_logp_fused_lmhead_bwd_kept(cl, 0x1000, 128, 0x2000, 0x3000, 0x4000, 0x5000, 0x5008, 0x6000,
                                              0x7000, None, 0x9000, 0xA000, None) == rlk.RLK_ERR_MISALIGNED
    assert rlk.rlk_logp_fused_lmhead_bwd_kept(cl, 0x1000, 128, 0x2000, 0x3000, 0x4000, None, 0x5000, 0x6000, 0x7000,
                                              None, 0x9000, 0xA000, None) == rlk.RLK_ERR_INVALID_ARG  # no lse_in
    assert rlk.rlk_logp_fused_lmhead_bwd_kept(cl, 0x1000, 128, 0x2000, 0x3000, 0x4000, 0x5000, 0x5800, 0x6000,
                                              0x7000, None, None, 0xA000, None) == rlk.RLK_ERR_INVALID_ARG  # no dW


def test_dlogits_may_alias_logits_only_exactly(built):
    """dlogits == logits (in place) passes the host checks; a dlogits buffer that overlaps the logits at
    another address is rejected before any CUDA call; a disjoint one passes.  (Calls that pass the host
    checks stop at the device check here: there is no GPU.)"""
    c = ok_contract(T=8)  # 8 rows x 152576 BF16 = 2,441,216 bytes
    base, span = 0x10000000, 8 * 152576 * 2

    def bwd(dl):
        return rlk.rlk_logp_bwd(c, base, 0x2000, 0x3000, 0x4000, 0x5000, dl, None, None, 0x6000, None)

    def fused_ent(dl):
        return rlk.rlk_logp_fwd_bwd_entropy(c, base, 0x2000, 0x3000, 0x5000, dl, 0x7000, 0x8000, 0x9000, 0x6000,
                                            None)
    for call in (bwd, fused_ent):
        for dl in (base + 16, base + span - 16, base - span + 16):
            assert call(dl) == rlk.RLK_ERR_INVALID_ARG
            assert "overlaps logits" in rlk.rlk_last_error_message()
        for dl in (base, base + span, base - span):
            call(dl)
            assert "overlaps" not in rlk.rlk_last_error_message()
    cs = ok_contract(T=8, virtual_tp=8)  # shard buffers of 152576/8 columns
    sspan = 8 * (152576 // 8) * 2
    assert rlk.rlk_logp_shard_bwd(cs, 0, base, 0x2000, 0x3000, 0x4000, 0x5000, base + sspan - 16, 0x6000,
                                  None) == rlk.RLK_ERR_INVALID_ARG
    assert "overlaps logits" in rlk.rlk_last_error_message()
    rlk.rlk_logp_shard_bwd(cs, 0, base, 0x2000, 0x3000, 0x4000, 0x5000, base + sspan, 0x6000, None)
    assert "overlaps" not in rlk.rlk_last_error_message()


def test_grpo_fused_step_fails_closed_on_the_host(built):
    """The fused GRPO step checks its arguments before any CUDA call: a missing loss, a bad beta, a missing
    advantage or output, a misaligned or partly overlapping dlogits."""
    c = ok_contract(T=8)
    assert rlk.rlk_grpo_fused_workspace_size(c) >= 256 + 256 + 256
    assert rlk.rlk_grpo_fused_workspace_size(ok_contract(num_tiles=63)) == 0
    base = 0x10000000

    def call(**kw):
        a = dict(logits=base, targets=0x2000, mask=0x3000, adv=0x4000, ref=None, beta=0.01, dl=0x20000000,
                 logp=0x5000, lse=0x6000, grad=0x7000, ent=None, loss=0x8000, count=None, ws=0x9000)
        a.update(kw)
        return rlk.rlk_grpo_fused_step(c, a["logits"], a["targets"], a["mask"], a["adv"], a["ref"], a["beta"], a["dl"],
                                       a["logp"], a["lse"], a["grad"], a["ent"], a["loss"], a["count"], a["ws"], None)
    assert call(loss=None) == rlk.RLK_ERR_INVALID_ARG and "loss" in rlk.rlk_last_error_message()
    assert call(beta=-1.0) == rlk.RLK_ERR_INVALID_ARG and "beta" in rlk.rlk_last_error_message()
    assert call(beta=float("nan")) == rlk.RLK_ERR_INVALID_ARG
    assert call(adv=None) == rlk.RLK_ERR_INVALID_ARG and "advantage" in rlk.rlk_last_error_message()
    assert call(grad=None) == rlk.RLK_ERR_INVALID_ARG
    assert call(dl=0x20000008) == rlk.RLK_ERR_MISALIGNED
    assert call(dl=base + 16) == rlk.RLK_ERR_INVALID_ARG and "overlaps" in rlk.rlk_last_error_message()
    assert call(mask=None) == rlk.RLK_ERR_INVALID_ARG  # explicit mode needs the mask
    # everything well-formed: the call gets as far as the device check (no GPU here)
    assert call() == rlk.RLK_ERR_INVALID_ARG and "CUDA pointer" in rlk.rlk_last_error_message()
