"""Pins of the CPU oracle to facts outside itself.

Each function raises AssertionError when the oracle library `lib` breaks a fact
the pages or the mathematics fix. test_oracle_pins.py runs them against the
real oracle; test_oracle_mutants.py runs them against deliberately broken
copies of the oracle and requires that every copy fails at least one pin.
"""
import itertools
import math
import os

import numpy as np

import oracle
from oracle.simulate import simulate, simulate_all_gather, simulate_reduce_scatter

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


def pin_m1_pairs(lib):
    """Worked example: 4 ranks holding [r, r+1] give [6, 10] on every rank."""
    rows = _read_golden("m1_four_rank_pairs.txt")
    kv = {}
    ranks = []
    expect = None
    for r in rows:
        if r.startswith("rank "):
            ranks.append([float(v) for v in r.split(":")[1].split()])
        elif r.startswith("expect:"):
            expect = [float(v) for v in r.split(":")[1].split()]
        else:
            k, v = r.split()
            kv[k] = v
    assert int(kv["n_ranks"]) == len(ranks) == 4
    xs = [np.array(v, np.float32) for v in ranks]
    for chunk in (16, 64, 512 * 1024):
        for nch in (1, 2):
            out = oracle.allreduce(xs, kv["dtype"], kv["op"], nch, chunk, lib=lib)
            assert out.tolist() == expect, (chunk, nch, out)


def pin_m2_first_element(lib, max_count=None):
    """Worked example: element 0 = r, rest 0 -> element 0 = N(N-1)/2, rest 0."""
    for row in _read_golden("m2_first_element.txt"):
        n, count, first, rest = (int(v) for v in row.split())
        if max_count is not None:
            count = min(count, max_count)
        xs = []
        for r in range(n):
            x = np.zeros(count, np.float32)
            x[0] = r
            xs.append(x)
        out = oracle.allreduce(xs, "float32", "sum", 1, 512 * 1024, nthreads=4, lib=lib)
        assert out[0] == first == n * (n - 1) // 2
        assert not np.any(out[1:] != rest)


def pin_sentinel_start_rank(lib):
    """Ring-order sentinel (N = 3, float32). For the elements of chunk c set
    x[c] = 2^24 and x[c+1] = x[c+2] = 1. Starting at rank c+1 gives
    1 + 1 + 2^24 = 2^24 + 2 exactly; starting at rank c or c+2, or walking the
    ring backwards, rounds one of the 1s away (2^24 + 1 ties to even, 2^24).
    Chunk boundaries are derived by hand from the chunk-size rule:
      count 12, chunk 1 MiB: one loop, cur = alignUp(divUp(12, 3), 4) = 4;
      count 60, chunk 16 B (4 floats): five full loops of three 4-element chunks.
    """
    big = np.float32(2 ** 24)
    for count, chunk_bytes, nloops in ((12, 1 << 20, 1), (60, 16, 5)):
        xs = [np.empty(count, np.float32) for _ in range(3)]
        for loop in range(nloops):
            for c in range(3):
                sl = slice(12 * loop + 4 * c, 12 * loop + 4 * c + 4)
                xs[c][sl] = big
                xs[(c + 1) % 3][sl] = 1
                xs[(c + 2) % 3][sl] = 1
        out = oracle.allreduce(xs, "float32", "sum", 1, chunk_bytes, lib=lib)
        assert np.all(out == np.float32(2 ** 24 + 2)), out


def _orders_result(vals, order):
    acc = np.float32(vals[order[0]])
    for k in order[1:]:
        acc = np.float32(acc + np.float32(vals[k]))
    return acc


def pin_bruteforce_order(lib, seed=1):
    """Brute force over all N! visiting orders (N = 3, 4, 5): identify from the
    oracle's own outputs which orders it can have used, and require that only
    the ring order (start at rank c+1, then c+2, ..., c) survives.

    An order is written relative to the chunk id c as the sequence of rank
    offsets (rank - c) mod N. For every element the set of relative orders whose
    float32 left-to-right sum reproduces the oracle's value is computed; the
    intersection over all elements must be exactly the ring order and its twin
    with the first two terms swapped (IEEE addition commutes, so those two give
    the same bits). Data: |x| in [1, 2) * 2^k, k in 0..3, random signs, so most
    sums round and different orders round differently."""
    rng = np.random.default_rng(seed)
    for n in (3, 4, 5):
        loops = 8
        count = 4 * n * loops          # chunk 16 B = 4 floats; loop = 4n floats
        xs = [(rng.uniform(1, 2, count) * np.exp2(rng.integers(0, 4, count))
               * rng.choice([-1.0, 1.0], count)).astype(np.float32) for _ in range(n)]
        out = oracle.allreduce(xs, "float32", "sum", 1, 16, lib=lib)
        perms = list(itertools.permutations(range(n)))
        alive = set(perms)
        for i in range(count):
            c = (i % (4 * n)) // 4
            vals = [xs[r][i] for r in range(n)]
            ok = set()
            for rel in alive:
                if _orders_result(vals, [(c + k) % n for k in rel]) == out[i]:
                    ok.add(rel)
            alive &= ok
        ring = tuple(list(range(1, n)) + [0])
        twin = (ring[1], ring[0]) + ring[2:]
        assert alive == {ring, twin}, (n, sorted(alive))


def _sum_abs_bound(xs, n, unit_roundoff):
    s = np.sum([np.abs(x.astype(np.float64)) for x in xs], axis=0)
    g = (n - 1) * unit_roundoff
    return g / (1 - g) * s


def pin_fp_error_bound(lib, seed=2):
    """Any order of N-1 rounded additions stays within gamma_{N-1} * sum|x|
    of the exact sum (the standard recursive-summation bound). Exact sums are
    taken with math.fsum."""
    rng = np.random.default_rng(seed)
    for dtype, u in (("float32", 2.0 ** -24), ("float64", 2.0 ** -53)):
        for n in (2, 5, 16):
            count = 257
            xs = [rng.uniform(-1, 1, count).astype(oracle.NP_DTYPE[dtype]) for _ in range(n)]
            out = oracle.allreduce(xs, dtype, "sum", 2, 64, lib=lib)
            exact = np.array([math.fsum(float(x[i]) for x in xs) for i in range(count)])
            bound = _sum_abs_bound(xs, n, u)
            assert np.all(np.abs(out.astype(np.float64) - exact) <= bound)
    # 16-bit formats, through the oracle's own decode of the result codes.
    import torch
    for dtype, u in (("float16", 2.0 ** -11), ("bfloat16", 2.0 ** -8)):
        n, count = 8, 129
        vals = [rng.uniform(-1, 1, count) for _ in range(n)]
        if dtype == "float16":
            xs = [v.astype(np.float16) for v in vals]
            dec = [x.astype(np.float64) for x in xs]
        else:
            ts = [torch.tensor(v, dtype=torch.float64).to(torch.bfloat16) for v in vals]
            xs = [t.view(torch.int16).numpy().view(np.uint16) for t in ts]
            dec = [t.to(torch.float64).numpy() for t in ts]
        out = oracle.allreduce(xs, dtype, "sum", 1, 32, lib=lib)
        if dtype == "float16":
            got = out.view(np.float16).astype(np.float64)
        else:
            got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
        exact = np.array([math.fsum(float(d[i]) for d in dec) for i in range(count)])
        bound = _sum_abs_bound(dec, n, u)
        assert np.all(np.abs(got - exact) <= bound)


def pin_rounding_16bit(lib, seed=3):
    """The oracle's float16 / bfloat16 rounding equals library conversions
    (numpy float64 -> float16; torch float64 -> bfloat16, both round to nearest
    even), on random values, exact ties, subnormals and the overflow edge."""
    import torch
    rng = np.random.default_rng(seed)
    vals = list(rng.standard_normal(4000) * np.exp2(rng.integers(-30, 20, 4000)))
    # float16 ties and edges
    vals += [1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -26,
             65504.0, 65519.99, 65520.0, -65520.0, 2.0 ** -14 - 2.0 ** -25, 0.0, -0.0]
    for v in vals:
        with np.errstate(over="ignore"):
            want = int(np.array([v], np.float64).astype(np.float16).view(np.uint16)[0])
            want_value = float(np.float16(v))
        got = oracle.f16_from_double(v, lib=lib)
        assert got == want, ("f16", v, hex(got), hex(want))
        assert oracle.round_to_format(v, 11, -14, 15, lib=lib) == want_value
        back = oracle.f16_decode(got, lib=lib)
        assert back == float(np.uint16(got).view(np.float16)) or (math.isinf(back))
    bvals = list(rng.standard_normal(4000) * np.exp2(rng.integers(-140, 120, 4000)))
    bvals += [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 2.0 ** -134, 3 * 2.0 ** -134,
              3.3895313892515355e38, 3.4e38, -3.39e38, 2.0 ** -126, 0.0, -0.0]
    tb = torch.tensor(bvals, dtype=torch.float64).to(torch.bfloat16).view(torch.int16)
    for v, w in zip(bvals, tb.tolist()):
        want = w & 0xFFFF
        got = oracle.bf16_from_double(v, lib=lib)
        assert got == want, ("bf16", v, hex(got), hex(want))


# The 8-bit floating types: torch's name and the largest finite value.
FP8_TORCH = {"float8_e4m3": ("float8_e4m3fn", 448.0), "float8_e5m2": ("float8_e5m2", 57344.0)}


def _fp8_codes(values, dtype):
    """Codes of `values` (clamped into the finite range) by torch's conversion."""
    import torch
    name, maxf = FP8_TORCH[dtype]
    v = np.clip(np.asarray(values, np.float32), -maxf, maxf)
    return torch.from_numpy(v).to(getattr(torch, name)).view(torch.uint8).numpy().copy()


def _fp8_values(codes, dtype):
    """Values of 8-bit codes by torch's decoding."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return t.view(getattr(torch, FP8_TORCH[dtype][0])).to(torch.float64).numpy()


def pin_rounding_fp8(lib, seed=13):
    """The 8-bit formats against torch's float8_e4m3fn / float8_e5m2: every
    code decodes to torch's value (NaN where torch has NaN); rounding equals
    torch's float32 conversion (nearest even) on random values across the
    normal and subnormal ranges, on exact ties and below the largest finite
    value; beyond it (and at infinity) the result saturates to +-448 / +-57344
    (the E4M3 code 0x7E, E5M2 0x7B, with the sign bit for negatives)."""
    import torch
    rng = np.random.default_rng(seed)
    for dtype, fmt in (("float8_e4m3", "e4m3"), ("float8_e5m2", "e5m2")):
        name, maxf = FP8_TORCH[dtype]
        want = _fp8_values(np.arange(256), dtype)
        for h in range(256):
            got = oracle.fp8_decode(h, fmt, lib=lib)
            assert (math.isnan(got) and math.isnan(want[h])) or got == want[h], (dtype, h)
        lo = -9 if fmt == "e4m3" else -16
        vals = rng.standard_normal(6000) * np.exp2(rng.integers(lo - 2, 16, 6000))
        finite = want[~np.isnan(want) & ~np.isinf(want)]
        grid = np.unique(finite)
        vals = np.concatenate([vals, (grid[1:] + grid[:-1]) / 2, grid,
                               [maxf * 1.03, -maxf * 1.03]]).astype(np.float32)
        vals = vals[np.abs(vals) <= maxf * 1.04]
        ref = _fp8_codes(vals, dtype)
        for v, w in zip(vals.tolist(), ref.tolist()):
            assert oracle.fp8_from_double(v, fmt, lib=lib) == w, (dtype, v, w)
        top = 0x7E if fmt == "e4m3" else 0x7B
        for v in (maxf * 1.2, 1e9, float("inf")):
            assert oracle.fp8_from_double(v, fmt, lib=lib) == top, (dtype, v)
            assert oracle.fp8_from_double(-v, fmt, lib=lib) == top | 0x80, (dtype, -v)
        # a sum past the largest finite value saturates; a product too
        xs = [np.array([top, top, 0x38 if fmt == "e4m3" else 0x3C], np.uint8)] * 2
        got = oracle.allreduce(xs, dtype, "sum", 1, 16, lib=lib)
        assert got.tolist() == [top, top, _fp8_codes([2.0], dtype)[0]], (dtype, got)


def pin_fp8_pairs_exhaustive(lib):
    """Every pair of finite 8-bit codes, sum and product, against torch: both
    operands decoded exactly to float32, the op in float32 (exact for E4M3
    and for every product; an E5M2 sum rounds in float32 at most once more,
    which cannot change the 8-bit result, float32 having more than 2*3+2
    significand bits), clamped to the largest finite value and converted by
    torch (nearest even). Two ranks, so each element is op(one rank's code,
    the other's); IEEE sum and product commute bit for bit, so which rank
    starts does not matter."""
    import torch
    for dtype in FP8_TORCH:
        name, maxf = FP8_TORCH[dtype]
        vals = _fp8_values(np.arange(256), dtype)
        finite = np.nonzero(np.isfinite(vals))[0].astype(np.uint8)
        a = np.repeat(finite, len(finite))
        b = np.tile(finite, len(finite))
        fa = torch.from_numpy(a).view(getattr(torch, name)).to(torch.float32)
        fb = torch.from_numpy(b).view(getattr(torch, name)).to(torch.float32)
        for op, f in (("sum", torch.add), ("prod", torch.mul)):
            want = _fp8_codes(f(fa, fb).numpy(), dtype)
            got = oracle.allreduce([a, b], dtype, op, 1, 16, lib=lib)
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, (dtype, op, bad.size, int(a[bad[0]]), int(b[bad[0]]))


def pin_chunk_map(lib):
    """Chunk boundaries worked by hand from the channel split and the chunk-size
    rule, plus the partition and 16-byte alignment properties."""
    def spans(count, n, nch, es, chunk):
        r = oracle.chunk_ranges(count, n, nch, es, chunk, lib=lib)
        return list(zip(r["channel"].tolist(), r["loop"].tolist(), r["chunk"].tolist(),
                        r["begin"].tolist(), r["end"].tolist()))

    # 65,536 float32, N=4, 1 channel, 512 KiB chunks: one loop, cur = 16,384.
    assert spans(65536, 4, 1, 4, 512 << 10) == [
        (0, 0, c, 16384 * c, 16384 * (c + 1)) for c in range(4)]
    # 64 Mi bfloat16, N=8, 16 channels, 512 KiB chunks: 4 Mi per channel, two
    # full loops of eight 256 Ki chunks.
    s = spans(64 << 20, 8, 16, 2, 512 << 10)
    assert len(s) == 16 * 2 * 8
    assert s[0] == (0, 0, 0, 0, 256 << 10)
    assert s[8] == (0, 1, 0, 2 << 20, (2 << 20) + (256 << 10))
    assert s[16] == (1, 0, 0, 4 << 20, (4 << 20) + (256 << 10))
    # 2 Mi float16, N=72, 8 channels, 64 KiB chunks: one loop per channel,
    # cur = alignUp(divUp(262144, 72), 8) = 3648; the last chunk holds 3136.
    s = spans(2 << 20, 72, 8, 2, 64 << 10)
    assert len(s) == 8 * 72
    assert s[0] == (0, 0, 0, 0, 3648)
    assert s[71] == (0, 0, 71, 71 * 3648, 262144)
    # 1000 float32, N=3, 2 channels of 500, 64 B chunks: ten full loops of 48,
    # then rem = 20, cur = alignUp(7, 4) = 8: [480,488) [488,496) [496,500).
    s = spans(1000, 3, 2, 4, 64)
    ch0 = [x for x in s if x[0] == 0]
    assert ch0[-3:] == [(0, 10, 0, 480, 488), (0, 10, 1, 488, 496), (0, 10, 2, 496, 500)]
    assert [x for x in s if x[0] == 1][0] == (1, 0, 0, 500, 516)
    # 5 float32 over 4 channels: per = alignUp(2, 4) = 4 -> [0,4) [4,5), two empty.
    assert oracle.channel_range(5, 4, 4, 0, lib=lib) == (0, 4)
    assert oracle.channel_range(5, 4, 4, 1, lib=lib) == (4, 5)
    assert oracle.channel_range(5, 4, 4, 2, lib=lib) == (5, 5)
    # Partition and alignment on a grid.
    for count, n, nch, es, chunk in itertools.product((1, 7, 100, 1023), (1, 2, 3, 5), (1, 3),
                                                      (1, 2, 4, 8), (16, 48, 256)):
        s = spans(count, n, nch, es, chunk)
        cover = np.zeros(count, np.int32)
        for ch, lp, c, b, e in s:
            assert b < e
            cover[b:e] += 1
            assert (b * es) % 16 == 0, "chunk starts are 16-byte aligned"
            assert e == count or (e * es) % 16 == 0
        assert np.all(cover == 1)


def pin_fold_equals_simulation(lib, seed=4, quick=False):
    """The closed-form fold equals a literal execution of the ring schedule on
    tiny inputs, for every element type and op."""
    rng = np.random.default_rng(seed)
    import torch
    dtypes = list(oracle.DTYPES)
    shapes = []
    counts = (0, 1, 2, 3, 5, 8, 13, 17, 33, 64)
    for n in (1, 2, 3, 4, 5):
        for count in counts:
            for chunk in range(16, 257, 16 if not quick else 48):
                for nch in (1, 2, 3):
                    shapes.append((n, count, chunk, nch))

    def draw(dtype, count):
        if dtype in ("float16", "float32", "float64"):
            v = rng.standard_normal(count) * np.exp2(rng.integers(-8, 8, count))
            return v.astype(oracle.NP_DTYPE[dtype])
        if dtype == "bfloat16":
            v = rng.standard_normal(count) * np.exp2(rng.integers(-8, 8, count))
            t = torch.tensor(v, dtype=torch.float64).to(torch.bfloat16)
            return t.view(torch.int16).numpy().view(np.uint16)
        if dtype in FP8_TORCH:
            return _fp8_codes(rng.standard_normal(count) * np.exp2(rng.integers(-8, 5, count)),
                              dtype)
        info = np.iinfo(oracle.NP_DTYPE[dtype])
        return rng.integers(info.min, info.max, count, dtype=oracle.NP_DTYPE[dtype],
                            endpoint=True)

    # fp32 sum on the whole shape grid; every dtype x op on a subset.
    for i, (n, count, chunk, nch) in enumerate(shapes):
        combos = [("float32", "sum")]
        if i % 7 == 0:
            combos = [(d, o) for d in dtypes for o in oracle.OPS]
        for dtype, op in combos:
            xs = [draw(dtype, count) for _ in range(n)]
            want = oracle.allreduce(xs, dtype, op, nch, chunk, lib=lib)
            got = simulate(xs, dtype, op, nch, chunk)
            for g in got:
                assert np.array_equal(g.view(np.uint8), want.view(np.uint8)), \
                    (dtype, op, n, count, chunk, nch)


def pin_order_free_invariants(lib, seed=5):
    """Integer sum / max / min and float max / min do not depend on order: the
    oracle must equal numpy's plain reductions (sums wrap modulo 2^bits)."""
    rng = np.random.default_rng(seed)
    for dtype in ("int8", "uint8", "int32", "uint32", "int64", "uint64"):
        info = np.iinfo(oracle.NP_DTYPE[dtype])
        n, count = 6, 301
        xs = [rng.integers(info.min, info.max, count, dtype=oracle.NP_DTYPE[dtype],
                           endpoint=True) for _ in range(n)]
        stack = np.stack(xs)
        with np.errstate(over="ignore"):
            want_sum = np.sum(stack, axis=0, dtype=oracle.NP_DTYPE[dtype])
            want_prod = np.prod(stack, axis=0, dtype=oracle.NP_DTYPE[dtype])
        assert np.array_equal(oracle.allreduce(xs, dtype, "sum", 2, 32, lib=lib), want_sum)
        assert np.array_equal(oracle.allreduce(xs, dtype, "prod", 2, 32, lib=lib), want_prod)
        assert np.array_equal(oracle.allreduce(xs, dtype, "max", 2, 32, lib=lib), stack.max(0))
        assert np.array_equal(oracle.allreduce(xs, dtype, "min", 2, 32, lib=lib), stack.min(0))
    for dtype in ("float16", "float32", "float64"):
        n, count = 5, 211
        xs = [rng.standard_normal(count).astype(oracle.NP_DTYPE[dtype]) for _ in range(n)]
        stack = np.stack(xs)
        assert np.array_equal(oracle.allreduce(xs, dtype, "max", 3, 16, lib=lib), stack.max(0))
        assert np.array_equal(oracle.allreduce(xs, dtype, "min", 3, 16, lib=lib), stack.min(0))


def pin_sampled_equals_full(lib, seed=6):
    """The per-element entry point (used to check full-size runs on sampled
    outputs) equals the full fold at every index, on ragged multi-channel,
    multi-loop shapes of every element size."""
    rng = np.random.default_rng(seed)
    for dtype, n, count, nch, chunk in (("float32", 5, 3001, 3, 64), ("bfloat16", 8, 4099, 2, 256),
                                        ("int8", 3, 777, 4, 16), ("float64", 7, 1031, 5, 48),
                                        ("float16", 72, 1500, 2, 64)):
        npd = oracle.NP_DTYPE[dtype]
        if dtype in ("float32", "float64", "float16"):
            xs = [rng.standard_normal(count).astype(npd) for _ in range(n)]
        else:
            xs = [rng.integers(0, 1 << (8 * np.dtype(npd).itemsize - 1), count).astype(npd)
                  for _ in range(n)]
        full = oracle.allreduce(xs, dtype, "sum", nch, chunk, lib=lib)
        idx = np.arange(count, dtype=np.uint64)
        vals = np.stack(xs)
        at = oracle.allreduce_at(vals, idx, count, dtype, "sum", nch, chunk, lib=lib)
        assert np.array_equal(at.view(np.uint8), full.view(np.uint8)), dtype


def pin_reduce_scatter_closed_form(lib):
    """N = 4, three elements per block, rank r holds 10r + j at position j
    (integers, exact in float32): rank b gets sum_r (10r + 3b + i) =
    60 + 4(3b + i)."""
    n, rc = 4, 3
    xs = [np.array([10 * r + j for j in range(n * rc)], np.float32) for r in range(n)]
    outs = oracle.reduce_scatter(xs, "float32", "sum", lib=lib)
    for b in range(n):
        assert outs[b].tolist() == [60 + 4 * (3 * b + i) for i in range(rc)], (b, outs[b])


def pin_reduce_scatter_order(lib, seed=7):
    """ReduceScatter's fold of block b starts at rank b+1 and ends at rank b:
    the sentinel (block b: x_b = 2^24, others 1 -> 2^24 + 2) and the brute
    force over all N! orders (N = 3, 4, 5) on order-revealing data."""
    n = 3
    xs = [np.ones(3 * 4, np.float32) for _ in range(n)]
    for b in range(n):
        xs[b][b * 4:(b + 1) * 4] = 2 ** 24
    for o in oracle.reduce_scatter(xs, "float32", "sum", lib=lib):
        assert np.all(o == np.float32(2 ** 24 + 2)), o
    rng = np.random.default_rng(seed)
    for n in (3, 4, 5):
        rc = 40
        xs = [(rng.uniform(1, 2, n * rc) * np.exp2(rng.integers(0, 4, n * rc))
               * rng.choice([-1.0, 1.0], n * rc)).astype(np.float32) for _ in range(n)]
        outs = oracle.reduce_scatter(xs, "float32", "sum", lib=lib)
        alive = set(itertools.permutations(range(n)))
        for b in range(n):
            for i in range(rc):
                vals = [xs[r][b * rc + i] for r in range(n)]
                alive = {rel for rel in alive
                         if _orders_result(vals, [(b + k) % n for k in rel]) == outs[b][i]}
        ring = tuple(list(range(1, n)) + [0])
        assert alive == {ring, (ring[1], ring[0]) + ring[2:]}, (n, sorted(alive))


def pin_reduce_scatter_is_allreduce_blocks(lib, seed=8):
    """With one channel and a chunk of exactly one block, the AllReduce chunk
    map cuts the buffer into the N blocks, so AllReduce block c equals rank
    c's ReduceScatter output bit for bit."""
    rng = np.random.default_rng(seed)
    for dtype, n, rc in (("float32", 5, 64), ("bfloat16", 4, 128), ("float16", 7, 32)):
        if dtype == "bfloat16":
            import torch
            xs = [torch.tensor(rng.standard_normal(n * rc)).to(torch.bfloat16)
                  .view(torch.int16).numpy().view(np.uint16) for _ in range(n)]
        else:
            xs = [rng.standard_normal(n * rc).astype(oracle.NP_DTYPE[dtype]) for _ in range(n)]
        es = oracle.ELEM_SIZE[dtype]
        ar = oracle.allreduce(xs, dtype, "sum", 1, rc * es, lib=lib)
        rs = oracle.reduce_scatter(xs, dtype, "sum", lib=lib)
        for c in range(n):
            assert np.array_equal(ar[c * rc:(c + 1) * rc].view(np.uint8), rs[c].view(np.uint8))


def pin_rs_ag_equal_simulation(lib, seed=9):
    """ReduceScatter and AllGather equal literal ring executions, every type
    and op."""
    rng = np.random.default_rng(seed)
    import torch
    for dtype in oracle.DTYPES:
        npd = oracle.NP_DTYPE[dtype]
        for n in (1, 2, 3, 6):
            rc = int(rng.integers(1, 20))
            if dtype in ("float16", "float32", "float64"):
                xs = [(rng.standard_normal(n * rc) * 4).astype(npd) for _ in range(n)]
            elif dtype == "bfloat16":
                xs = [torch.tensor(rng.standard_normal(n * rc)).to(torch.bfloat16)
                      .view(torch.int16).numpy().view(np.uint16) for _ in range(n)]
            elif dtype in FP8_TORCH:
                xs = [_fp8_codes(rng.standard_normal(n * rc) * 4, dtype) for _ in range(n)]
            else:
                info = np.iinfo(npd)
                xs = [rng.integers(info.min, info.max, n * rc, dtype=npd, endpoint=True)
                      for _ in range(n)]
            for op in oracle.OPS:
                want = oracle.reduce_scatter(xs, dtype, op, lib=lib)
                got = simulate_reduce_scatter(xs, dtype, op)
                for g, w in zip(got, want):
                    assert np.array_equal(np.ascontiguousarray(g).view(np.uint8), w.view(np.uint8))
            ag = oracle.all_gather(xs, dtype, lib=lib)
            for g, w in zip(simulate_all_gather(xs), ag):
                assert np.array_equal(g.view(np.uint8), w.view(np.uint8))
            for w in ag:
                assert np.array_equal(w.view(np.uint8), np.concatenate(xs).view(np.uint8))


# ---------------------------------------------------------------------------
# Double binary tree.
# ---------------------------------------------------------------------------

def _trees(lib, n):
    return [[oracle.tree_node(n, r, t, lib=lib) for r in range(n)] for t in (0, 1)]


def pin_tree_pages_examples(lib):
    """The pages' hand-worked tree facts (tests/golden/btree_pages_examples.txt)."""
    for row in _read_golden("btree_pages_examples.txt"):
        kind, *vals = row.split()
        vals = [int(v) for v in vals]
        if kind == "node":
            n, r, up, d0, d1 = vals
            assert oracle.tree_node(n, r, 0, lib=lib) == (up, d0, d1), row
        elif kind == "parent":
            n, r, up = vals
            assert oracle.tree_node(n, r, 0, lib=lib)[0] == up, row
        else:
            n, r, *kids = vals
            got = [c for c in oracle.tree_node(n, r, 0, lib=lib)[1:] if c >= 0]
            assert sorted(got) == sorted(kids), row


def pin_tree_structure(lib):
    """For every ring size 1..128, each tree is one binary tree over all
    ranks: one root, every other rank the child of its parent, every rank
    reachable from the root, height at most ceil(log2 n) + 1; the first
    tree's root is 0, the second tree's root is n - 1 (mirror, even n) or 1
    (shift, odd n); in the first tree a node's children straddle it
    (child0 < node < child1). For even n the second tree is the first
    mirrored, and the two trees' leaf sets do not meet (the pages: in the
    second tree the leaves become inner nodes)."""
    for n in range(1, 129):
        trees = _trees(lib, n)
        for t, tree in enumerate(trees):
            roots = [r for r in range(n) if tree[r][0] == -1]
            assert len(roots) == 1, (n, t, roots)
            root = roots[0]
            want_root = 0 if t == 0 or n == 1 else (n - 1 if n % 2 == 0 else 1)
            assert root == want_root, (n, t, root)
            for r, (up, d0, d1) in enumerate(tree):
                for c in (d0, d1):
                    if c >= 0:
                        assert 0 <= c < n and tree[c][0] == r, (n, t, r, c)
                if up >= 0:
                    assert r in tree[up][1:], (n, t, r, up)
                if t == 0:
                    assert d0 < 0 or d0 < r, (n, r, d0)
                    assert d1 < 0 or d1 > r, (n, r, d1)
            depth = {root: 0}
            todo = [root]
            while todo:
                r = todo.pop()
                for c in tree[r][1:]:
                    if c >= 0:
                        assert c not in depth, (n, t, c)
                        depth[c] = depth[r] + 1
                        todo.append(c)
            assert len(depth) == n, (n, t)
            assert max(depth.values()) <= max(1, math.ceil(math.log2(n))) + 1, (n, t)
        if n % 2 == 0:
            for r in range(n):
                up, d0, d1 = trees[0][n - 1 - r]
                m = lambda x: -1 if x < 0 else n - 1 - x
                assert trees[1][r] == (m(up), m(d0), m(d1)), (n, r)
            if n >= 4:
                leaves = [set(r for r in range(n) if tree[r][1] < 0 and tree[r][2] < 0)
                          for tree in trees]
                assert not (leaves[0] & leaves[1]), (n, leaves)


def pin_tree_fold_by_hand(lib, seed=10):
    """4 ranks worked out by hand from the pages' rule. Tree 0: 0 -> 2 ->
    {1, 3}; tree 1 (the mirror): 3 -> 1 -> {2, 0}. A node's value is its own
    element, then op with child0's value, then with child1's: tree 0 gives
    x0 + ((x2 + x1) + x3), tree 1 gives x3 + ((x1 + x2) + x0). 16 float32:
    the first 8 on tree 0, the rest on tree 1."""
    rng = np.random.default_rng(seed)
    f = np.float32
    for _ in range(50):
        xs = [(rng.standard_normal(16) * 10.0 ** rng.integers(-3, 4, 16)).astype(f)
              for _ in range(4)]
        got = oracle.tree_allreduce(xs, "float32", "sum", lib=lib)
        x0, x1, x2, x3 = xs
        want = np.concatenate([(x0 + ((x2 + x1) + x3))[:8], (x3 + ((x1 + x2) + x0))[8:]])
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        mx = oracle.tree_allreduce(xs, "float32", "max", lib=lib)
        assert np.array_equal(mx, np.maximum.reduce(xs))


def pin_tree_sentinel(lib):
    """3 ranks, tree 0 = 0 -> 2 -> 1: a child's subtree is reduced before its
    parent adds it, x0 + (x2 + x1); with x0 = 2^24 and x1 = x2 = 1 that is
    2^24 + 2 exactly, where any other association rounds to 2^24."""
    xs = [np.array([2.0 ** 24], np.float32), np.ones(1, np.float32), np.ones(1, np.float32)]
    got = oracle.tree_allreduce(xs, "float32", "sum", lib=lib)
    assert got[0] == 2.0 ** 24 + 2, got


def pin_tree_order_free(lib, seed=11):
    """Integer sum / max / min and float max / min do not depend on the order:
    the tree fold equals numpy's reductions, for every ring size 1..40, and the
    float32 sum lies within gamma_{2h} * sum|x| of the exact sum (h the
    height; a value meets at most two additions per level)."""
    rng = np.random.default_rng(seed)
    for n in range(1, 41):
        cnt = int(rng.integers(1, 70))
        xs = [rng.integers(-2 ** 20, 2 ** 20, cnt, dtype=np.int32) for _ in range(n)]
        assert np.array_equal(oracle.tree_allreduce(xs, "int32", "sum", lib=lib),
                              np.sum(xs, axis=0, dtype=np.int32))
        for op, fn in (("max", np.maximum), ("min", np.minimum)):
            assert np.array_equal(oracle.tree_allreduce(xs, "int32", op, lib=lib), fn.reduce(xs))
        fx = [rng.standard_normal(cnt).astype(np.float32) for _ in range(n)]
        assert np.array_equal(oracle.tree_allreduce(fx, "float32", "max", lib=lib),
                              np.maximum.reduce(fx))
        h = max(1, math.ceil(math.log2(n))) + 1
        u = 2.0 ** -24
        gam = 2 * h * u / (1 - 2 * h * u)
        got = oracle.tree_allreduce(fx, "float32", "sum", lib=lib).astype(np.float64)
        exact = np.array([math.fsum(float(x[i]) for x in fx) for i in range(cnt)])
        bound = gam * np.sum(np.abs(np.array(fx, np.float64)), axis=0)
        assert np.all(np.abs(got - exact) <= bound + 1e-300)


def pin_tree_split(lib):
    """The halves: the first alignUp(divUp(count, 2), 16/e) elements go to
    tree 0 (the pages: the first half on tree 1, the rest on tree 2; reading:
    rounded to 16 bytes like the ring's channels), capped at count."""
    assert oracle.tree_split(13, 4, lib=lib) == 8
    assert oracle.tree_split(3, 4, lib=lib) == 3
    assert oracle.tree_split(17, 2, lib=lib) == 16
    assert oracle.tree_split(100, 8, lib=lib) == 50
    assert oracle.tree_split(1, 1, lib=lib) == 1


# ---------------------------------------------------------------------------
# Average and pre-multiplied sum.
# ---------------------------------------------------------------------------

def pin_scaled_ops(lib, seed=12):
    """Pre-multiplied sum and average against facts outside the oracle:
    scaling every input by 2 scales the ring-order sum by exactly 2 (a power
    of two, no overflow); an integer pre-multiplied sum is sum(s * x) with
    wrap-around; the integer average truncates sum / N toward zero; the
    float average of inputs that are multiples of 1/4 with N = 4 is exact;
    a float16 scalar is rounded to float16 before the product (0.1 is not
    float16); the ReduceScatter versions give the same blocks."""
    rng = np.random.default_rng(seed)
    for dtype in ("float16", "bfloat16", "float32", "float64"):
        npd = oracle.NP_DTYPE[dtype]
        n, cnt = 5, 257
        if dtype == "bfloat16":
            import torch
            xs = [torch.tensor(rng.standard_normal(cnt)).to(torch.bfloat16)
                  .view(torch.int16).numpy().view(np.uint16) for _ in range(n)]
        else:
            xs = [rng.standard_normal(cnt).astype(npd) for _ in range(n)]
        plain = oracle.allreduce(xs, dtype, "sum", 3, 64, lib=lib)
        got = oracle.allreduce_scaled(xs, dtype, "premulsum", 2.0, 3, 64, lib=lib)
        if dtype == "bfloat16":
            assert [oracle.bf16_decode(g, lib=lib) for g in got] == \
                [2 * oracle.bf16_decode(p, lib=lib) for p in plain]
        else:
            assert np.array_equal(got, (2 * plain).astype(npd)), dtype
    # integer pre-multiplied sum with wrap, and the integer average
    for dtype, npd in (("int32", np.int32), ("uint8", np.uint8), ("int64", np.int64),
                       ("int8", np.int8)):
        n, cnt = 7, 301
        info = np.iinfo(npd)
        xs = [rng.integers(info.min, info.max, cnt, dtype=npd, endpoint=True) for _ in range(n)]
        got = oracle.allreduce_scaled(xs, dtype, "premulsum", 3, 2, 64, lib=lib)
        want = np.zeros(cnt, np.uint64)
        for x in xs:
            want = want + (x.astype(np.int64).astype(np.uint64) * np.uint64(3))
        assert np.array_equal(got.view(npd), want.astype(npd)), dtype
        avg = oracle.allreduce_scaled(xs, dtype, "avg", 0, 2, 64, lib=lib)
        tot = [sum(int(x[i]) for x in xs) for i in range(cnt)]
        bits = 8 * np.dtype(npd).itemsize
        def wrap(v):
            v &= (1 << bits) - 1
            return v - (1 << bits) if info.min < 0 and v >= 1 << (bits - 1) else v
        cdiv = lambda v, d: -((-v) // d) if v < 0 else v // d  # C: toward zero
        want_avg = [cdiv(wrap(t), n) for t in tot]
        assert [int(v) for v in avg] == want_avg, dtype
        rs = oracle.reduce_scatter_scaled([np.tile(x, 1)[: n * (cnt // n)] for x in xs],
                                          dtype, "avg", 0, lib=lib)
        blk = cnt // n
        for b in range(n):
            t = [wrap(sum(int(x[b * blk + i]) for x in xs)) for i in range(blk)]
            assert [int(v) for v in rs[b]] == [cdiv(v, n) for v in t], (dtype, b)
    # 8-bit floating types: doubling every input doubles the sum exactly while
    # it stays below the largest finite value (|x| <= 8, N = 5: |2 sum| <= 80)
    for dtype, fmt in (("float8_e4m3", "e4m3"), ("float8_e5m2", "e5m2")):
        xs = [_fp8_codes(rng.uniform(-8, 8, 203), dtype) for _ in range(5)]
        plain = oracle.allreduce(xs, dtype, "sum", 2, 32, lib=lib)
        got = oracle.allreduce_scaled(xs, dtype, "premulsum", 2.0, 2, 32, lib=lib)
        assert np.array_equal(_fp8_values(got, dtype), 2 * _fp8_values(plain, dtype)), dtype
    # exact float average
    xs = [(rng.integers(-64, 64, 100) / 4.0).astype(np.float32) for _ in range(4)]
    avg = oracle.allreduce_scaled(xs, "float32", "avg", 0, 1, 16, lib=lib)
    assert np.array_equal(avg, (sum(x.astype(np.float64) for x in xs) / 4).astype(np.float32))
    # the float16 scalar is rounded before the product
    xs = [np.array([1.0, 3.0, -7.5], np.float16), np.zeros(3, np.float16)]
    got = oracle.allreduce_scaled(xs, "float16", "premulsum", 0.1, 1, 16, lib=lib)
    assert np.array_equal(got, (xs[0] * np.float16(0.1)).astype(np.float16))


def pin_tree_scaled_ops(lib, seed=14):
    """The tree's average and pre-multiplied sum against facts outside the
    oracle: premul by 2 doubles the tree's sum exactly; an integer
    pre-multiplied sum is sum(s * x) with wrap-around (order-free); the
    integer average is the wrapped sum divided by N toward zero; the float
    average of multiples of 1/4 over 4 ranks is exact."""
    rng = np.random.default_rng(seed)
    for n in (1, 2, 5, 8, 13):
        xs = [rng.standard_normal(131).astype(np.float32) for _ in range(n)]
        plain = oracle.tree_allreduce(xs, "float32", "sum", lib=lib)
        got = oracle.tree_allreduce_scaled(xs, "float32", "premulsum", 2.0, lib=lib)
        assert np.array_equal(got, (2 * plain).astype(np.float32)), n
        for dtype, npd in (("int32", np.int32), ("uint8", np.uint8), ("int64", np.int64)):
            info = np.iinfo(npd)
            ix = [rng.integers(info.min, info.max, 77, dtype=npd, endpoint=True)
                  for _ in range(n)]
            bits = 8 * np.dtype(npd).itemsize
            def wrap(v):
                v &= (1 << bits) - 1
                return v - (1 << bits) if info.min < 0 and v >= 1 << (bits - 1) else v
            tot = [wrap(sum(int(x[i]) for x in ix)) for i in range(77)]
            cdiv = lambda v, d: -((-v) // d) if v < 0 else v // d
            avg = oracle.tree_allreduce_scaled(ix, dtype, "avg", 0, lib=lib)
            assert [int(v) for v in avg] == [cdiv(t, n) for t in tot], (n, dtype)
            pm = oracle.tree_allreduce_scaled(ix, dtype, "premulsum", -3, lib=lib)
            want = [wrap(sum(-3 * int(x[i]) for x in ix)) for i in range(77)]
            assert [int(v) for v in pm] == want, (n, dtype)
    xs = [(rng.integers(-64, 64, 90) / 4.0).astype(np.float32) for _ in range(4)]
    avg = oracle.tree_allreduce_scaled(xs, "float32", "avg", 0, lib=lib)
    assert np.array_equal(avg, (sum(x.astype(np.float64) for x in xs) / 4).astype(np.float32))


ALL_PINS = [pin_fp8_pairs_exhaustive, pin_tree_scaled_ops, pin_rounding_fp8, pin_reduce_scatter_closed_form, pin_reduce_scatter_order,
            pin_reduce_scatter_is_allreduce_blocks, pin_rs_ag_equal_simulation, pin_sampled_equals_full, pin_m1_pairs, pin_m2_first_element, pin_sentinel_start_rank, pin_bruteforce_order,
            pin_fp_error_bound, pin_rounding_16bit, pin_chunk_map, pin_fold_equals_simulation,
            pin_order_free_invariants, pin_tree_pages_examples, pin_tree_structure,
            pin_tree_fold_by_hand, pin_tree_sentinel, pin_tree_order_free, pin_tree_split,
            pin_scaled_ops]
