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


def upload_oracle_prefill(w, c, seqs, keep_from=None, keep_to=None):
    """Quantise the closed tiles of each sequence in `seqs` (its first
    w.seq_lens[b] tokens) with the oracle on host threads and write the
    records into the GPU pool, one sequence at a time, so that the decode
    reads ORACLE records and no expected value depends on the GPU quantiser.
    The raw remainder goes into the open tile.

    Memory stays bounded by one sequence's context: only the tokens
    [keep_from[b], keep_to[b]) of each sequence (default: from the open
    tile's first token to the context's end) are kept on the host.
    Returns (recs, kept): recs[(b, t, h, kv)] = record (a view into a host
    copy of the pool); kept[b] = (k, v, first_token) with k, v [n, H, D]
    16-bit CPU tensors."""
    H, kb, vb = c.H, w.k_bits, w.v_bits
    heads = range(c.h0, c.h1)
    pool_h = c.pool.cpu().numpy()
    hr, krb, vrb = c.block_bytes // H, O.record_bytes(False, kb, vb), O.record_bytes(True, kb, vb)
    recs, kept = {}, {}
    for b in seqs:
        n = w.seq_lens[b]
        nf = n // T
        lo = nf * T if keep_from is None else keep_from[b]
        hi = n if keep_to is None else keep_to[b]
        k = I.kv_sequence(w, "k", b, max(n, hi), c.device, heads).cpu()
        v = I.kv_sequence(w, "v", b, max(n, hi), c.device, heads).cpu()
        if nf:
            first = np.array([t * T * H * D + h * D for t in range(nf) for h in range(H)], np.int64)
            for kv, src in ((0, k), (1, v)):
                rec, flags = O.quantize_batch(bits(src[:nf * T]).reshape(-1), w.dtype, first, H * D, bool(kv),
                                              nthreads=NTHREADS, k_bits=kb, v_bits=vb)
                rb = vrb if kv else krb
                for i in range(nf * H):
                    t, h = divmod(i, H)
                    off = int(c.table[b, t]) * c.block_bytes + h * hr + kv * krb
                    pool_h[off:off + rb] = rec[i]
                    recs[(b, t, h, kv)] = pool_h[off:off + rb]
        r = n - nf * T
        if r:
            c.tail[b, :, 0, :r] = k[nf * T:n].permute(1, 0, 2).to(c.device)
            c.tail[b, :, 1, :r] = v[nf * T:n].permute(1, 0, 2).to(c.device)
        kept[b] = (k[lo:hi].clone(), v[lo:hi].clone(), lo)
        del k, v
    c.pool.copy_(torch.from_numpy(pool_h))
    return recs, kept


def oracle_decode(w, units_in, scale, k_bits=4, v_bits=2):
    """Oracle attention (folded fp64 form, C threads) of many (sequence, KV
    head) units: units_in = list of (q [G, D] fp64, krecs, vrecs, ktail
    [n, D] fp64, vtail).  Returns [U, G, D]."""
    q = np.stack([u[0] for u in units_in])
    kt = np.zeros((len(units_in), T, D)); vt = np.zeros((len(units_in), T, D))
    nt = np.zeros(len(units_in), np.int32)
    for i, u in enumerate(units_in):
        m = u[3].shape[0]
        kt[i, :m] = u[3]; vt[i, :m] = u[4]; nt[i] = m
    return O.attention_batch(q, [u[1] for u in units_in], [u[2] for u in units_in], kt, vt, nt, scale,
                             nthreads=NTHREADS, k_bits=k_bits, v_bits=v_bits)
