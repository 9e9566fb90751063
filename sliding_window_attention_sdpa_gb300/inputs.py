"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the attention method: it only draws random
tensors (torch.Generator on the CPU, then RNE casts to the I/O dtype) and lays
out sequence lengths and THD slots. Both the CUDA path and the CPU oracle are
fed from here.

Recipe (the workloads of the cuDNN-frontend pages: the gpt_oss dashboard shape
and the A100 study shapes):
  * Q, K, V, dO ~ N(0, 1) in fp32 from torch.Generator(seed), cast to bf16/f16;
  * sink logits ~ N(0, 1) in fp32, one per q-head;
  * THD: lengths ~ U[lo, hi] from the same seed; each sequence's slot is padded
    up to a multiple of `slot_align` tokens and gap tokens hold N(0, 1) values,
    so any leak of a gap token into a result shows.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16}


@dataclass
class Tensors:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    sink: Optional[torch.Tensor]


def randn(shape, seed: int, dtype=torch.float32, device="cpu") -> torch.Tensor:
    """N(0, 1) drawn in fp32 by torch's generator on `device`, then cast (RNE).
    A CPU and a CUDA draw with the same seed differ; each workload uses one."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=device).to(dtype)


def make_tensors(q_shape, kv_shape, h_q: int, dtype: str, seed: int, sink: bool,
                 device="cpu") -> Tensors:
    """Q, K, V, dO (I/O dtype) and optional fp32 sink logits on `device`."""
    dt = DTYPES[dtype]
    return Tensors(
        q=randn(q_shape, seed * 16 + 1, dt, device),
        k=randn(kv_shape, seed * 16 + 2, dt, device),
        v=randn(kv_shape, seed * 16 + 3, dt, device),
        do=randn(q_shape, seed * 16 + 4, dt, device),
        sink=randn((h_q,), seed * 16 + 5, torch.float32, device) if sink else None,
    )


def thd_lengths(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n sequence lengths drawn uniformly from [lo, hi]."""
    g = torch.Generator().manual_seed(int(seed) * 16 + 7)
    return torch.randint(lo, hi + 1, (n,), generator=g).numpy().astype(np.int32)


def thd_offsets(lens: np.ndarray, slot_align: int) -> np.ndarray:
    """Token offsets ([n+1], int64) of slots that hold each sequence padded up
    to a multiple of slot_align tokens."""
    slots = (np.asarray(lens, np.int64) + slot_align - 1) // slot_align * slot_align
    return np.concatenate([[0], np.cumsum(slots)]).astype(np.int64)


def padded_lengths(b: int, s_max: int, seed: int, lo: Optional[int] = None) -> np.ndarray:
    """Per-batch actual lengths in [lo, s_max] for the BSHD padding mask."""
    lo = 1 if lo is None else lo
    g = torch.Generator().manual_seed(int(seed) * 16 + 9)
    return torch.randint(lo, s_max + 1, (b,), generator=g).numpy().astype(np.int32)
