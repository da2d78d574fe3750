"""Ring AllReduce cost model: predicted time per call, fitted to measurements.

The model is the one the pages give for NCCL's tuner ("NCCL 源码解析：从硬件
拓扑到集合通信选型的完整链路", §五, the decision formula, and "NCCL
原始碼解讀", ring bandwidth estimate, steps 1-3):

    time = lat * latCount + nBytes / (1000 * bw)            [us; bytes; GB/s]

with, for the ring AllReduce of N ranks (nSteps = 2 (N - 1)):

    lat = base + nSteps * hop            (the ring's latency grows linearly)
    bw  = busBw * disc * N / nSteps      (algorithm bandwidth of the ring)

where `disc` is the protocol's bandwidth discount (Simple 1, LL 0.5 for the
flag half of every 8-byte word, LL128 120/128 = 0.92 for the flag word of every
128-byte line) and latCount = 1 (one launch per call). nBytes is the per-rank
buffer B.

Here `base`, `hop` and `busBw * disc` are fitted per protocol to measured call
times on one GB300 (`fit`), by least squares on relative error; the fitted
discounts (busBw_p / busBw_Simple) can then be set beside the pages' 0.5 and
0.92, and `crossover` gives the size where one protocol stops being faster
than another.

The virtual ring adds a second form, in the same spirit (latCount = passes):
a call makes `parts` independent ring passes spread over `rings` rings that
run at once, each ring taking its passes one after another, so

    time = base + ceil(parts / rings) * (2 (N - 1) + 1) * stage
                + nBytes / (1000 * bw)

with `stage` the time of one stage of one pass and bw as above (`fit_passes`).
The pass term follows the plateaus of the measured curve (one pass per ring up
to a few MiB per rank), which a single latency cannot. A third form counts
the FIFO steps a rank warp takes one after another (`fit_steps`): the stages
of a pass that carry data, times the passes, each step costing a fixed time
and its bytes at the warp's rate.
"""
from dataclasses import dataclass

import numpy as np

# The pages' bandwidth discounts per protocol.
PAGE_DISCOUNT = {"simple": 1.0, "ll": 0.5, "ll128": 120.0 / 128.0}


@dataclass
class ProtoParams:
    base_us: float      # fixed cost per call (launch, prologue, drain)
    hop_us: float       # cost per ring step
    bus_gbs: float      # busBw * disc: bus bandwidth the protocol reaches

    def lat_us(self, n_ranks):
        return self.base_us + 2 * (n_ranks - 1) * self.hop_us

    def bw_gbs(self, n_ranks):
        """Algorithm bandwidth (B / t) of the ring at large B."""
        return self.bus_gbs * n_ranks / (2 * (n_ranks - 1))


def predict_us(p, nbytes, n_ranks):
    """Predicted time of one AllReduce of `nbytes` per rank on N ranks."""
    return p.lat_us(n_ranks) + nbytes / (1000.0 * p.bw_gbs(n_ranks))


def fit(points):
    """Fit one protocol's parameters to measured (nbytes, n_ranks, time_us)
    points: time = base + 2(N-1) hop + nbytes * 2(N-1) / (1000 N bus) is
    linear in (base, hop, 1/bus); least squares on relative error (each row
    divided by the measured time). Needs at least two ring sizes to tell base
    from hop; with one, hop is 0 and base carries the whole latency."""
    pts = np.asarray(points, dtype=np.float64)
    b, n, t = pts[:, 0], pts[:, 1], pts[:, 2]
    steps = 2.0 * (n - 1.0)
    cols = [np.ones_like(t), steps, b * steps / (1000.0 * n)]
    one_size = np.unique(n).size < 2
    if one_size:
        cols = [cols[0], cols[2]]
    a = np.stack(cols, axis=1) / t[:, None]
    x, *_ = np.linalg.lstsq(a, np.ones_like(t), rcond=None)
    if one_size:
        base, hop, inv_bus = x[0], 0.0, x[1]
    else:
        base, hop, inv_bus = x
    return ProtoParams(float(base), float(hop), float(1.0 / inv_bus) if inv_bus > 0 else float("inf"))


def crossover_bytes(p_fast_small, p_fast_large, n_ranks):
    """Per-rank size above which `p_fast_large` beats `p_fast_small` (None if
    the lines do not cross at a positive size)."""
    dl = p_fast_large.lat_us(n_ranks) - p_fast_small.lat_us(n_ranks)
    ds = 1.0 / (1000.0 * p_fast_small.bw_gbs(n_ranks)) - 1.0 / (1000.0 * p_fast_large.bw_gbs(n_ranks))
    if ds <= 0:
        return None
    x = dl / ds
    return x if x > 0 else None


def residuals(p, points):
    """Relative error (predicted / measured - 1) of every point."""
    return [predict_us(p, b, n) / t - 1.0 for b, n, t in points]


@dataclass
class PassParams:
    base_us: float      # fixed cost per call
    stage_us: float     # one stage of one ring pass
    bus_gbs: float      # bus bandwidth, as in ProtoParams

    def bw_gbs(self, n_ranks):
        return self.bus_gbs * n_ranks / (2 * (n_ranks - 1))


def passes(parts, rings):
    """Ring passes one after another: ceil(parts / rings)."""
    return -(-parts // rings) if rings else 0


def predict_passes_us(p, n_ranks, n_passes, nbytes):
    return (p.base_us + n_passes * (2 * (n_ranks - 1) + 1) * p.stage_us
            + nbytes / (1000.0 * p.bw_gbs(n_ranks)))


def fit_passes(points):
    """Fit (base, stage, bus) to measured (nbytes, n_ranks, n_passes, time_us)
    points by least squares on relative error (linear in base, stage and
    1/bus)."""
    pts = np.asarray(points, dtype=np.float64)
    b, n, k, t = pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]
    steps = 2.0 * (n - 1.0)
    cols = [np.ones_like(t), k * (steps + 1.0), b * steps / (1000.0 * n)]
    a = np.stack(cols, axis=1) / t[:, None]
    x, *_ = np.linalg.lstsq(a, np.ones_like(t), rcond=None)
    return PassParams(float(x[0]), float(x[1]), float(1.0 / x[2]) if x[2] > 0 else float("inf"))


def residuals_passes(p, points):
    return [predict_passes_us(p, n, k, b) / t - 1.0 for b, n, k, t in points]


# ---------------------------------------------------------------------------
# Third form: steps. A stage whose chunk slice is empty is skipped by both
# ends of its edge, so a pass has 2 ne - 1 stages with data, ne the chunks of
# a loop that hold any element (all N once a channel holds a whole loop of N
# chunks; fewer in a short last loop, whose chunk is alignUp(divUp(rem, N),
# 16 / e) elements: "NCCL 原始碼解讀", ch.2 §2.2-2.3). Every such stage moves
# one FIFO step of about B / (parts N) bytes per rank, and a rank warp takes
# its passes' steps one after another:
#
#     time = base + ceil(parts / rings) (2 ne - 1) (step + plen * byte)
#     plen = nBytes / (parts N)
#
# `step` is the fixed cost of one step and 1 / `byte` a rank warp's rate.
# ---------------------------------------------------------------------------
def data_stages(count, n_ranks, n_channels, chunk_bytes, elem_size):
    """2 ne - 1 for the largest channel (channel 0) of a call of `count`
    elements per rank; 0 for count 0."""
    if count <= 0:
        return 0
    align = 16 // elem_size
    per = -(-count // n_channels)
    per = -(-per // align) * align
    per = min(per, count)
    loop = n_ranks * (chunk_bytes // elem_size)
    if per >= loop:
        ne = n_ranks
    else:
        cur = -(-(-(-per // n_ranks)) // align) * align
        ne = -(-per // cur)
    return 2 * ne - 1


@dataclass
class StepParams:
    base_us: float      # fixed cost per call
    step_us: float      # fixed cost of one step of one rank warp
    byte_us: float      # cost of one byte of a step (1 / a rank warp's rate)

    def warp_gbs(self):
        return 1e-3 / self.byte_us if self.byte_us > 0 else float("inf")


def predict_steps_us(p, n_ranks, parts, rings, n_stages, nbytes):
    plen = nbytes / (parts * n_ranks) if parts else 0.0
    return p.base_us + passes(parts, rings) * n_stages * (p.step_us + plen * p.byte_us)


def fit_steps(points):
    """Fit (base, step, byte) to measured (nbytes, n_ranks, parts, rings,
    n_stages, time_us) points by least squares on relative error (linear in
    the three parameters)."""
    pts = np.asarray(points, dtype=np.float64)
    b, n, parts, rings, g, t = (pts[:, i] for i in range(6))
    k = np.ceil(parts / rings)
    plen = b / (parts * n)
    cols = [np.ones_like(t), k * g, k * g * plen]
    a = np.stack(cols, axis=1) / t[:, None]
    x, *_ = np.linalg.lstsq(a, np.ones_like(t), rcond=None)
    return StepParams(float(x[0]), float(x[1]), float(x[2]))


def residuals_steps(p, points):
    return [predict_steps_us(p, int(n), int(parts), int(rings), g, b) / t - 1.0
            for b, n, parts, rings, g, t in points]
