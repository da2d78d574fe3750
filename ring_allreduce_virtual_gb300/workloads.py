"""The measured workloads: virtual-rank AllReduce configurations with their
input recipes (see synthetic.py). Shared by the benchmark and the full-size
parity tests so both run exactly the same launch configuration."""
from dataclasses import dataclass

from . import synthetic


@dataclass(frozen=True)
class Workload:
    name: str
    n_ranks: int
    count: int          # elements per rank
    dtype: str
    dist: str
    op: str
    proto: str
    n_channels: int
    chunk_bytes: int
    seed: int

    @property
    def elem_size(self):
        return {"int8": 1, "uint8": 1, "float16": 2, "bfloat16": 2, "int32": 4, "uint32": 4,
                "float32": 4}.get(self.dtype, 8)

    @property
    def bytes_per_rank(self):
        return self.count * self.elem_size

    def describe(self):
        return (f"N={self.n_ranks} virtual ranks, {self.count} {self.dtype} per rank "
                f"({self.bytes_per_rank} B), {self.dist}, op={self.op}, {self.proto}, "
                f"{self.n_channels} channels, {self.chunk_bytes} B chunks")


MiB = 1 << 20
KiB = 1 << 10

# 1: 4 ranks, 65,536 float32 U[-1,1), sum, Simple, 1 channel (small case).
SMALL = Workload("n4_64Ki_f32_simple", 4, 65536, "float32", "uniform", "sum", "simple", 1,
                 512 * KiB, synthetic.SEED_BASE + 0)
# 2: 8 ranks, 64 Mi bfloat16 N(0, 0.01), sum, LL128, 16 channels, 512 KiB chunks.
BF16_LL128 = Workload("n8_64Mi_bf16_ll128", 8, 64 * MiB, "bfloat16", "normal:0.01", "sum",
                      "ll128", 16, 512 * KiB, synthetic.SEED_BASE + 1)
# 4: 72 ranks, 4 MiB float16 N(0, 1) per rank, sum, LL, 8 channels, 64 KiB chunks.
F16_LL_72 = Workload("n72_4MiB_f16_ll", 72, 2 * MiB, "float16", "normal:1", "sum", "ll", 8,
                     64 * KiB, synthetic.SEED_BASE + 3)
# 5: 16 ranks, 256 Mi float32 U[-1,1) (1 GiB per rank), sum, Simple, 32 channels, 1 MiB
# chunks: the bandwidth-bound case.
F32_SIMPLE_16 = Workload("n16_1GiB_f32_simple", 16, 256 * MiB, "float32", "uniform", "sum",
                         "simple", 32, 1 * MiB, synthetic.SEED_BASE + 4)


# Profiling stand-in of the headline workload: the same 16 ranks, float32,
# Simple protocol, 32 channels and 1 MiB chunks, at 128 MiB per rank (4 GiB in
# and out) so that an ncu capture stays small.
F32_SIMPLE_16_PROFILE = Workload("n16_128MiB_f32_simple", 16, 32 * MiB, "float32", "uniform",
                                 "sum", "simple", 32, 1 * MiB, synthetic.SEED_BASE + 4)


# The headline workload's shape on a ring of 17 ranks, a size that no cluster
# splits evenly (CTAs of 9 and 8 ranks): 17 x 1 GiB float32, Simple, 32
# channels, 1 MiB chunks.
F32_SIMPLE_17 = Workload("n17_1GiB_f32_simple", 17, 256 * MiB, "float32", "uniform", "sum",
                         "simple", 32, 1 * MiB, synthetic.SEED_BASE + 5)


# Profiling stand-in of the 17-rank workload: 128 MiB per rank (4.25 GiB in
# and out), for ncu captures.
F32_SIMPLE_17_PROFILE = Workload("n17_128MiB_f32_simple", 17, 32 * MiB, "float32", "uniform",
                                 "sum", "simple", 32, 1 * MiB, synthetic.SEED_BASE + 5)


# The LL128 gradient-bucket workload's shape (bf16 N(0, 0.01), 16 channels,
# 512 KiB chunks) on a ring of 24 ranks, which spans a cluster of 2 CTAs:
# 24 x 32 Mi bf16 (64 MiB per rank, 3 GiB in and out).
BF16_LL128_24 = Workload("n24_32Mi_bf16_ll128", 24, 32 * MiB, "bfloat16", "normal:0.01", "sum",
                         "ll128", 16, 512 * KiB, synthetic.SEED_BASE + 6)


def int32_sweep():
    """3: 8 ranks, int32 U-int[-2^20, 2^20], sum and max, per-rank size 8 B to
    256 MiB in powers of two, Simple (512 KiB chunks) and LL (64 KiB chunks),
    16 channels."""
    out = []
    for p in range(3, 29):
        count = (1 << p) // 4
        for proto, chunk in (("simple", 512 * KiB), ("ll", 64 * KiB)):
            for op in ("sum", "max"):
                out.append(Workload(f"n8_{1 << p}B_i32_{proto}_{op}", 8, count, "int32",
                                    "int:-1048576:1048576", op, proto, 16, chunk,
                                    synthetic.SEED_BASE + 2))
    return out


ALL = {w.name: w for w in [SMALL, BF16_LL128, F16_LL_72, F32_SIMPLE_16, F32_SIMPLE_16_PROFILE,
                            F32_SIMPLE_17, F32_SIMPLE_17_PROFILE, BF16_LL128_24]
       + int32_sweep()}
HEADLINE = F32_SIMPLE_16
