"""Seeded synthetic inputs for the attention forward.

This module holds no attention arithmetic: it only draws Q, K, V.  Both the
CUDA path (tests, ``bench.py``) and the float64 oracle consume what it makes.

Recipe: a NumPy ``Generator(PCG64(seed))`` draws Q, then K, then V, each as
float32 standard normal of shape [B, H, N, D]; each is multiplied by
``input_scale`` (a power of two, so exact) and then rounded to the working
dtype (fp16 / bf16 via torch's round-to-nearest-even cast, fp32 unchanged).
The oracle upcasts the rounded values to float64, so both sides see exactly
the same numbers.

The workloads mirror the pages' benchmark shapes: "FlashAttention under the
catlass template", section "Performance data" (B=4, H=32, N=4096, D=128 fp16
``torch.randn`` inputs), plus the small, causal, bf16 and sliding-window cases
listed in :data:`WORKLOADS`.
"""

import math
from dataclasses import dataclass, field

import numpy as np
import torch

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_WINDOW = 2

_TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str          # "f16" | "bf16" | "f32"
    scale: float
    mask: int
    win_l: int = -1
    win_r: int = -1
    input_scale: float = 1.0
    seed: int = 0
    rope: str = ""            # "" (none), "half" or "interleaved": rotary embedding of Q and K first
    rope_base: float = 10000.0
    backward: bool = False    # the step is the backward pass (dQ, dK, dV) for a random upstream dO
    notes: str = field(default="", compare=False)


WORKLOADS = {
    "tiny_f32_full": Workload("tiny_f32_full", 1, 2, 128, 64, "f32", 1.0 / 8.0, MASK_NONE, seed=1001),
    "tiny_f32_causal": Workload("tiny_f32_causal", 1, 2, 128, 64, "f32", 1.0 / 8.0, MASK_CAUSAL, seed=1001),
    "f16_causal_1k": Workload("f16_causal_1k", 2, 8, 1024, 64, "f16", 0.125, MASK_CAUSAL, seed=1002),
    "f16_full_4k": Workload("f16_full_4k", 4, 32, 4096, 128, "f16", 1.0 / math.sqrt(128), MASK_NONE, seed=1003),
    "f16_causal_4k": Workload("f16_causal_4k", 4, 32, 4096, 128, "f16", 1.0 / math.sqrt(128), MASK_CAUSAL, seed=1004),
    "bf16_causal_4k": Workload("bf16_causal_4k", 4, 32, 4096, 128, "bf16", 1.0 / math.sqrt(128), MASK_CAUSAL, seed=1004),
    "bf16_full_4k": Workload("bf16_full_4k", 4, 32, 4096, 128, "bf16", 1.0 / math.sqrt(128), MASK_NONE, seed=1003),
    "bf16_window_16k": Workload("bf16_window_16k", 1, 64, 16384, 128, "bf16", 1.0 / math.sqrt(128),
                                MASK_WINDOW, 1024, 0, input_scale=0.5, seed=1005),
    # the benchmark shape with the rotary embedding of Q and K in the step
    "f16_rope_full_4k": Workload("f16_rope_full_4k", 4, 32, 4096, 128, "f16", 1.0 / math.sqrt(128), MASK_NONE,
                                 seed=1003, rope="half", rope_base=10000.0),
    # backward pass at the benchmark shape (dO drawn like Q)
    "f16_bwd_full_4k": Workload("f16_bwd_full_4k", 4, 32, 4096, 128, "f16", 1.0 / math.sqrt(128), MASK_NONE,
                                seed=1003, backward=True),
    "f16_bwd_causal_4k": Workload("f16_bwd_causal_4k", 4, 32, 4096, 128, "f16", 1.0 / math.sqrt(128),
                                  MASK_CAUSAL, seed=1004, backward=True),
    "bf16_bwd_causal_4k": Workload("bf16_bwd_causal_4k", 4, 32, 4096, 128, "bf16", 1.0 / math.sqrt(128),
                                   MASK_CAUSAL, seed=1004, backward=True),
    # causal with the 500000 rotary base of the Llama-3 models the pages run
    "bf16_rope_causal_4k": Workload("bf16_rope_causal_4k", 4, 32, 4096, 128, "bf16", 1.0 / math.sqrt(128),
                                    MASK_CAUSAL, seed=1004, rope="half", rope_base=500000.0),
}


@dataclass(frozen=True)
class DecodeWorkload:
    """Nq new queries against an Nk-entry K/V cache (query i at position Nk - Nq + i)."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    D: int
    dtype: str
    scale: float
    mask: int
    win_l: int = -1
    win_r: int = -1
    seed: int = 0
    Hkv: int = 0        # K/V heads (0: same as H)
    page_size: int = 0  # > 0: the cache is paged, its pages shuffled in memory



DECODE_WORKLOADS = {
    "bf16_decode_32k": DecodeWorkload("bf16_decode_32k", 8, 32, 1, 32768, 128, "bf16", 1.0 / math.sqrt(128),
                                      MASK_CAUSAL, seed=1101),
    "bf16_decode_gqa_32k": DecodeWorkload("bf16_decode_gqa_32k", 8, 32, 1, 32768, 128, "bf16", 1.0 / math.sqrt(128),
                                          MASK_CAUSAL, seed=1103, Hkv=8),
    "f16_decode_4k_q4": DecodeWorkload("f16_decode_4k_q4", 4, 32, 4, 4096, 128, "f16", 1.0 / math.sqrt(128),
                                       MASK_CAUSAL, seed=1102),
    # the grouped-head cache above, cut into 256-position pages at shuffled places
    "bf16_decode_paged_32k": DecodeWorkload("bf16_decode_paged_32k", 8, 32, 1, 32768, 128, "bf16",
                                            1.0 / math.sqrt(128), MASK_CAUSAL, seed=1103, Hkv=8, page_size=256),
}


def make_paged(w: DecodeWorkload, k, v):
    """Cut the contiguous cache k, v [B, H_kv, Nk, D] into page_size-position
    pages [num_pages, page_size, H_kv, D], placed by a seeded permutation;
    returns (k_cache, v_cache, block_table int32 [B, Nk / page_size])."""
    B, Hkv, Nk, D = k.shape
    ps = w.page_size
    per_seq = Nk // ps
    perm = torch.from_numpy(np.random.default_rng(w.seed + 7).permutation(B * per_seq).astype(np.int64))
    def pages(x):
        x = x.permute(0, 2, 1, 3).reshape(B * per_seq, ps, Hkv, D)   # logical page order
        out = torch.empty_like(x)
        out[perm] = x
        return out.contiguous()
    table = perm.reshape(B, per_seq).to(torch.int32)
    return pages(k), pages(v), table


def make_decode(w: DecodeWorkload):
    """Q [B, H, Nq, D] and the K, V cache [B, H, Nk, D] (K and V from their own stream)."""
    q, _, _ = make_qkv(w.B, w.H, w.Nq, w.D, w.dtype, seed=w.seed, n_k=1)
    _, k, v = make_qkv(w.B, w.Hkv or w.H, 1, w.D, w.dtype, seed=w.seed + 1, n_k=w.Nk)
    return q, k, v


def torch_dtype(name):
    return _TORCH_DTYPES[name]


def make_qkv(B, H, N, D, dtype="f16", seed=0, input_scale=1.0, n_k=None):
    """Draw Q [B,H,N,D] and K, V [B,H,n_k,D] (n_k defaults to N) on the CPU.

    Returns three contiguous CPU torch tensors of the working dtype.
    """
    n_k = N if n_k is None else n_k
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for shape in ((B, H, N, D), (B, H, n_k, D), (B, H, n_k, D)):
        x = rng.standard_normal(size=shape, dtype=np.float32)
        if input_scale != 1.0:
            x *= np.float32(input_scale)
        out.append(torch.from_numpy(x).to(_TORCH_DTYPES[dtype]).contiguous())
    return tuple(out)


def make_workload(w: Workload):
    return make_qkv(w.B, w.H, w.N, w.D, w.dtype, w.seed, w.input_scale)
