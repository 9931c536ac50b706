"""The synthetic workloads of the selected-token log-probability path.

Each workload fixes shapes, value distributions, the mask recipe and the
upstream gradient, as the five measured configurations describe them:

* ``tiny``    batch 2 x seq 16 (T=32), the first 8 positions of each sequence
              inactive, V_real = V_padded = 151936, 64 tiles, logits ~N(0, 2),
              seed 123, targets uniform in [0, V_real), g = 1 on active rows.
* ``qwen3``   batch 4 x seq 1024 (T=4096), V_real = 151936 padded to 152576
              (padded columns hold random bits), logits ~N(0, 3) plus +15 at
              4 uniform columns per row, 10% of targets = ignore_index -100.
* ``rollout`` batch 32 x seq 2048 (T=65536), V_padded = 152576, V_real =
              151936, logits ~N(0, 3), explicit mask: a 256-token prompt, then a
              response of length uniform in {64..1792} (the seq - prompt cap).
* ``grpo``    the rollout logits and mask; g = A_b * mask / active_count with
              A_b ~ N(0, 1) per sequence and active_count the batch's active
              tokens (token mean).
* ``lmhead``  hidden [8192, 4096] ~N(0, 1), W [152576, 4096] ~N(0, 0.02) in
              BF16, targets uniform in [0, 151936), all rows active, g = 1/T.

"~N(0, s)" is realised as s times the centred Irwin-Hall(12) variate (unit
variance, support +-6), so that host and GPU builds give identical bits.
"""
from dataclasses import dataclass, replace

import numpy as np

import synth

MASK_EXPLICIT = 0
MASK_IGNORE_INDEX = 1


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seq: int
    v_real: int
    v_padded: int
    num_tiles: int = 64
    sigma: float = 3.0
    nspikes: int = 0
    spike: float = 15.0
    garbage: bool = False         # padded columns filled with random bit patterns
    mask_mode: int = MASK_EXPLICIT
    prompt: int = 0               # explicit masks: inactive prompt length
    len_min: int = 0              # explicit masks: response length range
    len_max: int = 0
    ignore_frac: float = 0.0      # ignore-index masks: fraction of ignored targets
    ignore_index: int = -100
    grad: str = "ones"            # "ones" | "mean" | "advantage" | "inv_T"
    seed: int = 123
    row_stride: int = 0           # 0 -> v_padded
    hidden: int = 0               # lm_head workloads: hidden size H
    hidden_sigma: float = 1.0
    weight_sigma: float = 0.02

    @property
    def T(self):
        return self.batch * self.seq

    @property
    def stride(self):
        return self.row_stride or self.v_padded

    def with_(self, **kw):
        return replace(self, **kw)


TINY = Workload("tiny", batch=2, seq=16, v_real=151936, v_padded=151936, sigma=2.0,
                mask_mode=MASK_EXPLICIT, prompt=8, len_min=8, len_max=8, grad="ones", seed=123)
QWEN3 = Workload("qwen3", batch=4, seq=1024, v_real=151936, v_padded=152576, sigma=3.0,
                 nspikes=4, spike=15.0, garbage=True, mask_mode=MASK_IGNORE_INDEX,
                 ignore_frac=0.10, grad="mean", seed=1234)
ROLLOUT = Workload("rollout", batch=32, seq=2048, v_real=151936, v_padded=152576, sigma=3.0,
                   garbage=True, mask_mode=MASK_EXPLICIT, prompt=256, len_min=64, len_max=1792,
                   grad="advantage", seed=2048)
GRPO = ROLLOUT.with_(name="grpo")
LMHEAD = Workload("lmhead", batch=1, seq=8192, v_real=151936, v_padded=152576,
                  mask_mode=MASK_EXPLICIT, prompt=0, len_min=8192, len_max=8192, grad="inv_T",
                  seed=4096, hidden=4096, hidden_sigma=1.0, weight_sigma=0.02)

WORKLOADS = {w.name: w for w in (TINY, QWEN3, ROLLOUT, GRPO, LMHEAD)}


def targets(w):
    return synth.targets(w.T, w.v_real, w.seed, w.ignore_frac if w.mask_mode == MASK_IGNORE_INDEX else 0.0,
                         w.ignore_index)


def active_mask(w):
    """uint8 [T] explicit mask (explicit mode) -- in ignore mode, None."""
    if w.mask_mode != MASK_EXPLICIT:
        return None
    m, _ = synth.response_mask(w.batch, w.seq, w.prompt, w.len_min, w.len_max, w.seed)
    return m


def active_rows(w, tgt=None, mask=None):
    """Boolean [T]: which rows are active under the workload's mask mode."""
    if w.mask_mode == MASK_EXPLICIT:
        return (active_mask(w) if mask is None else mask) != 0
    t = targets(w) if tgt is None else tgt
    return t != w.ignore_index


def grad(w, active):
    """FP32 upstream gradient of each row's log-probability (0 on inactive rows)."""
    T = w.T
    act = active.astype(np.float64)
    n = max(int(act.sum()), 1)
    if w.grad == "ones":
        g = act
    elif w.grad == "mean":
        g = act / n
    elif w.grad == "inv_T":
        g = act / T
    elif w.grad == "advantage":
        adv = synth.normal_f64(w.batch, w.seed, synth.STREAM_ADVANTAGE)
        g = np.repeat(adv, w.seq) * act / n
    else:
        raise ValueError(w.grad)
    return g.astype(np.float32)


def logits_host(w, row0=0, nrows=None):
    nrows = w.T - row0 if nrows is None else nrows
    return synth.logits_host(row0, nrows, w.stride, w.v_padded, w.v_real, w.seed, w.sigma,
                             w.nspikes, w.spike, w.garbage)


def logits_device(w, dst, row0=0, nrows=None, stream=None):
    nrows = w.T - row0 if nrows is None else nrows
    synth.logits_device(dst, row0, nrows, w.stride, w.v_padded, w.v_real, w.seed, w.sigma,
                        w.nspikes, w.spike, w.garbage, stream=stream)
