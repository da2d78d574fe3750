"""Seeded synthetic rank buffers for the virtual-rank AllReduce.

This module only draws inputs; it holds none of the AllReduce arithmetic. The
tests, the benchmark and the CPU oracle's callers all take their inputs from
here, so the CUDA path and the oracle always see the same bytes (GPU-drawn
inputs are copied to the host for the oracle).

Recipes (seed = 0x5EED0000 + workload index, one torch.Generator per call):
  uniform     U[-1, 1) drawn in float32, then rounded (RNE) to the dtype
  normal:S    N(0, S^2) drawn in float32, then rounded (RNE) to the dtype
  int:LO:HI   uniform integers in [LO, HI] (inclusive)
  pairs       rank r holds [r, r+1] (count must be 2): the 4-rank MPI demo of
              "NVIDIA GPU 集合通信库 NCCL 初始化流程源码级剖析" (AllReduce Sum
              demo section)
  first       rank r holds r in element 0 and zeros elsewhere: the N-GPU demo
              of "NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程", ch.1 §1.3
"""
import torch

# Unsigned 32/64-bit buffers are held in signed torch tensors of the same width
# (same bits; torch's unsigned wide types support few operations).
TORCH_DTYPE = {"int8": torch.int8, "uint8": torch.uint8, "int32": torch.int32,
               "uint32": torch.int32, "int64": torch.int64, "uint64": torch.int64,
               "float16": torch.float16, "bfloat16": torch.bfloat16,
               "float32": torch.float32, "float64": torch.float64,
               "float8_e4m3": torch.float8_e4m3fn, "float8_e5m2": torch.float8_e5m2}

SEED_BASE = 0x5EED0000


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def rank_buffers(n_ranks, count, dtype, dist, seed, device="cpu"):
    """N rank buffers of `count` elements of `dtype` (a name) drawn by `dist`."""
    tdt = TORCH_DTYPE[dtype]
    dev = torch.device(device)
    if dist == "pairs":
        if count != 2:
            raise ValueError("the pairs recipe has exactly two elements per rank")
        return [torch.tensor([r, r + 1], dtype=torch.float64).to(tdt).to(dev)
                for r in range(n_ranks)]
    if dist == "first":
        out = []
        for r in range(n_ranks):
            t = torch.zeros(count, dtype=tdt, device=dev)
            if count:
                t[0] = r
            out.append(t)
        return out
    g = _gen(seed, dev)
    out = []
    for _ in range(n_ranks):
        if dist == "uniform":
            t = torch.rand(count, generator=g, device=dev, dtype=torch.float32) * 2 - 1
            out.append(t.to(tdt))
        elif dist.startswith("normal:"):
            std = float(dist.split(":")[1])
            t = torch.randn(count, generator=g, device=dev, dtype=torch.float32) * std
            out.append(t.to(tdt))
        elif dist.startswith("int:"):
            _, lo, hi = dist.split(":")
            t = torch.randint(int(lo), int(hi) + 1, (count,), generator=g, device=dev,
                              dtype=torch.int64)
            out.append(t.to(tdt))  # unsigned values above the signed range wrap to the same bits
        else:
            raise ValueError(f"unknown recipe {dist!r}")
    return out


def to_numpy(t):
    """Host numpy view of a rank buffer; bfloat16 becomes raw uint16 codes,
    the 8-bit floating types raw uint8 codes."""
    import numpy as np
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return t.view(torch.uint8).numpy()
    return t.numpy()


def default_recipe(dtype):
    """The value distribution the tests use for an element type."""
    return {"int8": "int:-128:127", "uint8": "int:0:255", "int32": "int:-1048576:1048576",
            "uint32": "int:0:2097152", "int64": "int:-1048576:1048576",
            "uint64": "int:0:2097152"}.get(dtype, "uniform")
