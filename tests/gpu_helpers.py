"""Shared pieces of the GPU parity tests: device fixture, oracle tiles of
generated inputs (computed on host threads), and the oracle's attention over
oracle-made records."""
from __future__ import annotations

import concurrent.futures
import os

import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_quantize_gb300 import inputs as I

T = D = 128
NTHREADS = os.cpu_count() or 4


def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_kv_cache_quantize_gb300 import build as B
    B.build()
    return "cuda"


def bits(x16: torch.Tensor) -> np.ndarray:
    """16-bit tensor (any device) -> uint16 numpy on the host."""
    return x16.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def tile_values(x16: torch.Tensor, dtype: str) -> np.ndarray:
    """[128, 128] 16-bit tile -> exact fp64."""
    return O.decode16(bits(x16), dtype)


def oracle_tiles(jobs, dtype: str, iters: int = 8, k_bits: int = 4, v_bits: int = 2):
    """jobs: list of (tile16 [128,128] tensor, is_v).  Returns oracle Tiles."""
    def one(job):
        x16, is_v = job
        return O.quantize_tile(tile_values(x16, dtype), O.levels(is_v, k_bits, v_bits), iters)
    with concurrent.futures.ThreadPoolExecutor(NTHREADS) as ex:
        return list(ex.map(one, jobs))


def oracle_attention_units(units, scale, k_bits: int = 4, v_bits: int = 2):
    """units: list of dicts with q [G,D] fp64, krec/vrec lists, ktail/vtail
    [n,D] fp64.  Folded-form oracle attention of each unit (threads)."""
    def one(u):
        return O.attention_folded(u["q"], u["krec"], u["vrec"], u["ktail"], u["vtail"], scale, k_bits, v_bits)
    with concurrent.futures.ThreadPoolExecutor(NTHREADS) as ex:
        return list(ex.map(one, units))
