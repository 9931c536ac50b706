"""The host planner in logp_stream.cu against its replay in test_ring_protocol.py.

The protocol-model tests run the ring with the replay's (cluster size, tiles
per copy, ring depth, row buffers, skew, CTAs per SM); this checks, on a GB300,
that the compiled planner picks exactly those at the benchmark shapes, by
reading the plan it prints with RLK_VERBOSE=1.
"""
import os
import re
import subprocess
import sys

import pytest
import torch

from ring_protocol_model import skip_condition
from test_ring_protocol import SMEM_OPTIN, consumers_for, ctas_per_sm, l2_skew, plan, row_bufs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - the CPU suite deselects this module
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

PLAN = re.compile(r"rlk stream plan: mode (\d+), (\d+) CTA\(s\)/SM, (\d+) clusters x (\d+) CTAs, (\d+) tiles/copy, "
                  r"(\d+) slots of (\d+) B, (\d+) row buffers, skew (\d+), row skip (\d+)")
MODES = {0: "fwd", 1: "bwd", 3: "fused_l2"}

SCRIPT = r"""
import sys, torch
sys.path.insert(0, {root!r})
import vocab_selected_token_tile_gb300 as rlk
T, vr, vp, nt = 1024, 151936, 152576, 64
x = torch.zeros((T, vp), dtype=torch.int16, device="cuda")
t = torch.zeros(T, dtype=torch.int64, device="cuda")
m = torch.ones(T, dtype=torch.uint8, device="cuda")
g = torch.zeros(T, dtype=torch.float32, device="cuda")
for vtp in (1, 2, 4, 8):
    c = rlk.Contract(T=T, V_real=vr, V_padded=vp, num_tiles=nt, virtual_tp=vtp, mask_mode=rlk.MASK_EXPLICIT)
    logp, lse = rlk.logp_fwd(c, x, t, m)
    rlk.logp_bwd(c, x, t, m, lse, g)
    rlk.logp_fwd_bwd(c, x, t, m, g)
torch.cuda.synchronize()
"""


def test_compiled_planner_matches_the_replay():
    prop = torch.cuda.get_device_properties(0)
    if prop.multi_processor_count != 152 or getattr(prop, "shared_memory_per_block_optin", SMEM_OPTIN) != SMEM_OPTIN:
        pytest.skip("the replay is set up for a GB300 with 152 SMs and 227 KB of opt-in shared memory")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RLK_VERBOSE="1")
    for k in ("RLK_FUSED_SCHEDULE", "RLK_CTAS_PER_SM", "RLK_ROW_BUFS", "RLK_FUSED_SKEW", "RLK_TPS", "RLK_MAX_SLOTS"):
        env.pop(k, None)
    out = subprocess.run([sys.executable, "-c", SCRIPT.format(root=root)], env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    plans = [tuple(int(v) for v in m.groups()) for m in PLAN.finditer(out.stderr)]
    assert len(plans) == 12, out.stderr[-2000:]
    for i, vtp in enumerate((1, 2, 4, 8)):
        for j, want_mode in enumerate(("fwd", "bwd", "fused_l2")):
            mode, per_sm, clusters, C, tps, ns, _, rb, skew, skip = plans[3 * i + j]
            assert MODES[mode] == want_mode
            assert (C, tps, ns) == plan(want_mode, vtp, 152576, 64), (want_mode, vtp)
            assert per_sm == ctas_per_sm(want_mode, vtp, 152576, 64), (want_mode, vtp)
            assert rb == row_bufs(want_mode, 64), (want_mode, vtp)
            if want_mode == "fused_l2":
                assert skew == l2_skew(vtp, 152576, 64), vtp
            want_skip = skip_condition(want_mode, consumers_for(want_mode, per_sm), 64 // C, rb, skew)
            assert skip == int(want_skip), (want_mode, vtp)
