"""Seeded synthetic inputs for the KV-cache workloads.

This module is shared by the CUDA path's tests and benchmark and by the
oracle side of the tests; it holds none of the method's arithmetic, only the
random numbers and shapes of the workloads.  Every value is a pure function
of (seed, stream, element index): a counter-based generator (SplitMix64
finaliser applied to the counter), so any element can be regenerated without
generating the rest.  Uniforms are exact 23-bit fractions; normals come from
Box-Muller in float32 and are rounded to the 16-bit storage type
(round-to-nearest-even).  The integer part is bit-identical on every device;
float32 log/cos may differ in the last bit between CPU and GPU, so a test
generates its inputs once, on one device, and hands the same bytes to both
sides.

Workloads (distributions of the page "Huawei's KVarN puts KV-cache
quantization inside vLLM's backend", section "Reported benchmarks and the
verification gap": Qwen3-4B and Qwen3-32B shapes, 16K context):
  single_tile   1 KV head, 1 query head, 128 tokens, fp16
  qwen3_4b      8 seqs x 4096 tokens, 32 q heads / 8 KV heads, bf16
  qwen3_32b     32 seqs x 16384 tokens, 64 q heads / 8 KV heads, fp16
  prefill_32b   32 seqs x 16384 tokens x 8 KV heads, bf16 (write path)
  ragged_32b    256 seqs, lengths U[128, 32768] (never a multiple of 128),
                64 decode steps, 64 q heads / 8 KV heads, fp16
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D = 128
T = 128
OUTLIER_CHANNELS = (3, 17, 64, 101)  # scaled x20 in the unrotated key index
OUTLIER_GAIN = 20.0

_M64 = (1 << 64) - 1


def _s64(x: int) -> int:
    """Unsigned 64-bit constant as the signed int64 torch stores."""
    x &= _M64
    return x - (1 << 64) if x >= (1 << 63) else x


_GOLD = _s64(0x9E3779B97F4A7C15)
_MUL1 = _s64(0xBF58476D1CE4E5B9)
_MUL2 = _s64(0x94D049BB133111EB)


def _shr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bits."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = z + _GOLD
    z = (z ^ _shr(z, 30)) * _MUL1
    z = (z ^ _shr(z, 27)) * _MUL2
    return z ^ _shr(z, 31)


def hash64(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """64 random bits (as int64) for each counter in idx."""
    key = int(_mix(torch.tensor([_s64(seed * 0x100000001B3 + stream)], dtype=torch.int64))[0])
    return _mix(idx.to(torch.int64) ^ key)


def uniform(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """U(0,1) in float32 (exact 23-bit fractions plus half a step), never 0 or 1."""
    h = _shr(hash64(seed, stream, idx), 41)
    return (h.to(torch.float32) + 0.5) * (2.0 ** -23)


def normal(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """N(0,1) in float32 (Box-Muller on two counters per value)."""
    i2 = idx.to(torch.int64) * 2
    u1 = uniform(seed, stream, i2)
    u2 = uniform(seed, stream, i2 + 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def student_t4(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """Student-t with 4 degrees of freedom: N / sqrt(chi2_4 / 4), chi2_4 =
    -2 ln(U3 U4)."""
    z = normal(seed, stream, idx)
    i2 = idx.to(torch.int64) * 2
    u3 = uniform(seed, stream + 7919, i2)
    u4 = uniform(seed, stream + 7919, i2 + 1)
    chi2 = -2.0 * (torch.log(u3) + torch.log(u4))
    return z / torch.sqrt(chi2 / 4.0)


def to16(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """float32 -> 16-bit, rounding to nearest even."""
    return x.to(torch.float32).to(dtype)


def torch_dtype(name: str) -> torch.dtype:
    return {"f16": torch.float16, "bf16": torch.bfloat16}[name]


# --------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    dtype: str                      # "f16" | "bf16"
    seq_lens: list                  # context length of each sequence before decoding
    seed: int
    v_dist: str = "normal"          # "normal" | "t4"
    k_outliers: str = "fixed"       # "fixed" (channels x20) | "random" (4 per head, U(10,30))
    decode_steps: int = 0
    max_tokens: int = 0             # token stride of the generated K/V streams
    block_perm: bool = False        # physical blocks randomly permuted
    extra: dict = field(default_factory=dict)
    k_bits: int = 4                 # key code width: 4 (kvarn_k4v2, K4/V4 presets) or 2 (K2/V2 preset)
    v_bits: int = 2                 # value code width: 2, or 4 (K4/V4 preset)

    @property
    def G(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(D)


def single_tile() -> Workload:
    return Workload("single_tile", 1, 1, 1, "f16", [128], seed=0, max_tokens=128)


def qwen3_4b() -> Workload:
    return Workload("qwen3_4b_layer", 8, 32, 8, "bf16", [4096] * 8, seed=1, v_dist="t4",
                    k_outliers="random", max_tokens=4096)


def qwen3_32b() -> Workload:
    return Workload("qwen3_32b_decode_16k", 32, 64, 8, "f16", [16384] * 32, seed=2, max_tokens=16384,
                    block_perm=True)


def prefill_32b() -> Workload:
    return Workload("prefill_32b_16k", 32, 64, 8, "bf16", [16384] * 32, seed=3, max_tokens=16384,
                    block_perm=True)


def ragged_32b(batch: int = 256, steps: int = 64, seed: int = 4) -> Workload:
    lens = ragged_lengths(seed, batch)
    return Workload("ragged_32b_serving", batch, 64, 8, "f16", lens, seed=seed, decode_steps=steps,
                    max_tokens=32768 + steps, block_perm=True)


def ragged_lengths(seed: int, batch: int, lo: int = 128, hi: int = 32768) -> list:
    """Integers U[lo, hi], redrawn while a multiple of 128 (every sequence
    then has an open tail tile)."""
    out = []
    for b in range(batch):
        k = 0
        while True:
            u = float(uniform(seed, 900, torch.tensor([b * 1000 + k]))[0])
            n = lo + int(u * (hi - lo + 1))
            if n % T != 0:
                out.append(n)
                break
            k += 1
    return out


# streams: one per tensor so K, V and queries never share random numbers
S_K, S_V, S_Q, S_OUTL, S_PERM, S_MQ = 10, 11, 12, 13, 14, 15


def outlier_gain(w: Workload, device="cpu") -> torch.Tensor:
    """[H_kv, D] float32 multiplier applied to the keys (unrotated index)."""
    gain = torch.ones(w.num_kv_heads, D, dtype=torch.float32, device=device)
    if w.k_outliers == "fixed":
        gain[:, list(OUTLIER_CHANNELS)] = OUTLIER_GAIN
    else:
        for h in range(w.num_kv_heads):
            chosen = []
            k = 0
            while len(chosen) < 4:
                c = int(uniform(w.seed, S_OUTL, torch.tensor([h * 1000 + k]))[0] * D)
                k += 1
                if c not in chosen:
                    chosen.append(c)
            for i, c in enumerate(chosen):
                f = 10.0 + 20.0 * float(uniform(w.seed, S_OUTL + 1, torch.tensor([h * 16 + i]))[0])
                gain[h, c] = f
    return gain


def kv_values(w: Workload, which: str, b: int, t0: int, n_tok: int, device="cpu",
              heads=None) -> torch.Tensor:
    """K or V of sequence b, tokens [t0, t0+n_tok), as 16-bit [n_tok, H, D]
    (H = all KV heads, or the listed ones)."""
    heads = list(range(w.num_kv_heads)) if heads is None else list(heads)
    t = torch.arange(t0, t0 + n_tok, dtype=torch.int64, device=device)
    h = torch.tensor(heads, dtype=torch.int64, device=device)
    d = torch.arange(D, dtype=torch.int64, device=device)
    idx = (((b * w.max_tokens + t)[:, None, None] * w.num_kv_heads + h[None, :, None]) * D + d[None, None, :])
    if which == "k":
        x = normal(w.seed, S_K, idx) * outlier_gain(w, device)[h][None, :, :]
    elif w.v_dist == "t4":
        x = student_t4(w.seed, S_V, idx)
    else:
        x = normal(w.seed, S_V, idx)
    return to16(x, torch_dtype(w.dtype))


def kv_sequence(w: Workload, which: str, b: int, n_tok: int, device="cpu", heads=None) -> torch.Tensor:
    """Whole context of one sequence, [n_tok, H, D] (H = all KV heads, or
    the listed ones), generated in chunks."""
    heads = list(range(w.num_kv_heads)) if heads is None else list(heads)
    out = torch.empty(n_tok, len(heads), D, dtype=torch_dtype(w.dtype), device=device)
    step = 2048
    for t0 in range(0, n_tok, step):
        n = min(step, n_tok - t0)
        out[t0:t0 + n] = kv_values(w, which, b, t0, n, device, heads)
    return out


def queries(w: Workload, step: int = 0, device="cpu") -> torch.Tensor:
    """One decode query per sequence and query head: [B, H_q, D] 16-bit."""
    n = w.batch * w.num_q_heads * D
    idx = torch.arange(n, dtype=torch.int64, device=device) + step * n
    return to16(normal(w.seed, S_Q, idx), torch_dtype(w.dtype)).reshape(w.batch, w.num_q_heads, D)


def multi_queries(w: Workload, n_queries: int, device="cpu") -> torch.Tensor:
    """n_queries new query tokens per sequence and query head, N(0, 1):
    [B, n_queries, H_q, D] 16-bit."""
    n = w.batch * n_queries * w.num_q_heads * D
    idx = torch.arange(n, dtype=torch.int64, device=device)
    return to16(normal(w.seed, S_MQ, idx), torch_dtype(w.dtype)).reshape(w.batch, n_queries, w.num_q_heads, D)


def permutation(seed: int, n: int, device="cpu") -> torch.Tensor:
    """Seeded random permutation of range(n) (argsort of 64-bit keys)."""
    keys = hash64(seed, S_PERM, torch.arange(n, dtype=torch.int64, device=device))
    return torch.argsort(keys, stable=True).to(torch.int32)


def block_tables(w: Workload, n_tokens_final=None, device="cpu"):
    """Block table [B, max_blocks] int32 and the pool size.  Sequence b gets
    ceil(n_tokens_final[b] / 128) blocks; physical ids are consecutive or a
    seeded permutation.  Unused entries are -1."""
    final = n_tokens_final or [n + w.decode_steps for n in w.seq_lens]
    nblk = [(n + T - 1) // T for n in final]
    total = sum(nblk)
    maxb = max(nblk)
    phys = permutation(w.seed, total) if w.block_perm else torch.arange(total, dtype=torch.int32)
    table = torch.full((w.batch, maxb), -1, dtype=torch.int32)
    off = 0
    for b, k in enumerate(nblk):
        table[b, :k] = phys[off:off + k]
        off += k
    return table.to(device), total
