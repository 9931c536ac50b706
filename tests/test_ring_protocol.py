"""The streaming kernel's slot-ring protocol, checked on the host.

The planner arithmetic below replays the host planner of logp_stream.cu
(chunk size, cluster size and ring depth for each mode) for a GB300's
227 KB of opt-in shared memory; ring_protocol_model then runs the
kernel's wait/arrive protocol with adversarial timings.  Without the
per-slot issued-item check, consumers of the forward and backward modes can
wait two phases ahead and read a slot before its copy has landed (the model
finds it); with the check, no configuration reads a stale slot or deadlocks.
"""
import pytest

from ring_protocol_model import ProtocolError, simulate

SMEM_OPTIN = 232448


def align(v, a):
    return (v + a - 1) // a * a


def layout(ns, slot_bytes, nt, rbufs=2):
    off = ns * slot_bytes + 16 * ns
    off = align(off, 16) + 36 * ns
    off = align(off, 16) + rbufs * 8 * nt + 8 * nt
    off = align(off, 16) + rbufs * 32
    off = align(off, 8) + 32 * rbufs + 16
    return align(off, 128)


def plan(mode, vtp, v_padded, nt):
    """(C, tps, NS) as the host planner picks them."""
    w = v_padded // nt
    budget = SMEM_OPTIN - 1024
    tps_target = 1 if w >= 8192 else 8192 // w

    def slot_bytes(tps):
        return align((align(tps * w, 8) + 8) * 2, 16)

    def max_slots(sb):
        best = 0
        for ns in range(1, 97):
            if layout(ns, sb, nt) <= budget:
                best = ns
        return best

    C = 1 if mode == "bwd" else vtp
    tps = tps_target
    if mode == "fused":
        while True:
            ntl = -(-nt // C)
            tps = min(tps_target, ntl)
            while tps > 1 and ntl % tps:
                tps -= 1
            ns = max_slots(slot_bytes(tps))
            if ns >= 2 * -(-ntl // tps):
                return C, tps, ns
            C *= 2
    return C, tps, max_slots(slot_bytes(tps))


def plan_l2(vtp, v_padded, nt):
    """The L2-assisted fused mode is planned like the forward: C = virtual TP, no residency."""
    return plan("fwd", vtp, v_padded, nt)


CONFIGS = [(mode, vtp) for mode in ("fwd", "bwd", "fused", "fused_l2") for vtp in (1, 2, 4, 8)
           if not (mode == "bwd" and vtp > 1)]


@pytest.mark.parametrize("mode,vtp", CONFIGS)
def test_ring_protocol_reads_only_landed_slots(mode, vtp):
    C, tps, ns = plan_l2(vtp, 152576, 64) if mode == "fused_l2" else plan(mode, vtp, 152576, 64)
    for seed in range(3):
        simulate(mode, rows=24, C=C, NT=64, tps=tps, NS=ns, W=16, seed=seed)


def test_planner_replay_matches_the_benchmark_shapes():
    assert plan("fused", 2, 152576, 64) == (4, 2, 23)
    assert plan("fwd", 1, 152576, 64) == (1, 3, 15)


@pytest.mark.parametrize("ns", [1, 2, 3, 5])
def test_l2_fused_schedule_progresses_with_tiny_rings(ns):
    # The skewed producer order A(0), A(1), B(0), A(2), ... must not need more
    # than one slot: consumers take items in the order they are issued.
    for C in (1, 2, 4):
        for tps in (1, 3):
            simulate("fused_l2", rows=7, C=C, NT=64, tps=tps, NS=ns, W=16, seed=10 * ns + C)


def test_without_the_issued_item_check_the_model_finds_stale_reads():
    C, tps, ns = plan("bwd", 1, 152576, 64)
    found = 0
    for seed in range(6):
        try:
            simulate("bwd", rows=24, C=C, NT=64, tps=tps, NS=ns, W=16, seed=seed, seqcheck=False)
        except ProtocolError:
            found += 1
    assert found > 0
