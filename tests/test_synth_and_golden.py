"""Seeded input generator (host build) and the pages' printed run parameters."""
import json
import os

import numpy as np

import synth
from synth import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def test_generator_is_deterministic_and_row_addressable(built):
    a = synth.logits_host(0, 12, 1000, 992, 990, seed=5, sigma=3.0, nspikes=4, garbage=True)
    b = synth.logits_host(0, 12, 1000, 992, 990, seed=5, sigma=3.0, nspikes=4, garbage=True, nthreads=1)
    c = synth.logits_host(7, 3, 1000, 992, 990, seed=5, sigma=3.0, nspikes=4, garbage=True)
    assert np.array_equal(a, b)
    assert np.array_equal(a[7:10], c)
    d = synth.logits_host(0, 12, 1000, 992, 990, seed=6, sigma=3.0, nspikes=4, garbage=True)
    assert not np.array_equal(a[:, :990], d[:, :990])


def test_generator_moments_and_spikes(built):
    v = 151936
    bits = synth.logits_host(0, 16, v, v, v, seed=1, sigma=3.0)
    x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 3.0) < 0.01
    assert np.abs(x).max() <= 18.0                       # Irwin-Hall(12) support: 6 sigma
    sp = synth.logits_host(0, 16, v, v, v, seed=1, sigma=3.0, nspikes=4, spike=15.0)
    xs = (sp.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    changed = (sp != bits).sum(axis=1)
    assert np.all(changed <= 4) and np.all(changed >= 1)
    assert np.all(xs.max(axis=1) > 12.0)


def test_workload_masks_and_grads(built):
    tiny = W.TINY
    m = W.active_mask(tiny)
    assert m.tolist() == ([0] * 8 + [1] * 8) * 2
    g = W.grad(tiny, m != 0)
    assert np.array_equal(g, (m != 0).astype(np.float32))
    q = W.QWEN3
    t = W.targets(q)
    frac = np.mean(t == -100)
    assert 0.08 < frac < 0.12 and np.all(t[t != -100] < q.v_real) and np.all(t[t != -100] >= 0)
    r = W.ROLLOUT
    mask, lens = synth.response_mask(r.batch, r.seq, r.prompt, r.len_min, r.len_max, r.seed)
    assert np.all((lens >= 64) & (lens <= 1792))
    assert mask.reshape(r.batch, r.seq)[:, :256].sum() == 0
    ga = W.grad(W.GRPO, mask != 0)
    assert np.all(ga[mask == 0] == 0.0)
    # token-mean normalisation: sum |g| over a sequence = |A_b| * L_b / active_count
    adv = synth.normal_f64(r.batch, r.seed, synth.STREAM_ADVANTAGE)
    per_seq = ga.reshape(r.batch, r.seq).astype(np.float64).sum(axis=1)
    np.testing.assert_allclose(per_seq, adv * lens / mask.sum(), rtol=1e-5)


def test_tiny_workload_matches_the_pages_run():
    gold = json.load(open(os.path.join(HERE, "golden", "issue323_tiny_matrix.json")))
    p = gold["parameters"]
    t = W.TINY
    assert (t.v_real, t.v_padded, t.num_tiles) == (p["real_vocab"], p["padded_vocab"], p["num_vocab_tiles"])
    assert (t.batch, t.seq, t.prompt, t.seed) == (p["batch"], p["seq"], p["prompt_tokens"], p["seed"])
    # our parity bars are inside the pages' acceptance tolerance
    assert 1e-4 < gold["acceptance"]["atol"]
    assert W.QWEN3.v_padded == 152576  # the fixed padded vocabulary of the H100 matrix document
