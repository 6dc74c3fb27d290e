"""Per-token error distribution of the quantised cache, with and without the
Hadamard rotation and the variance normalisation.

"Huawei's KVarN puts KV-cache quantization inside vLLM's backend", section
"Why KV-cache quantization degrades under autoregressive decoding": the
largest 5% of per-token errors cause most of the end-to-end loss, so the
tail of the per-token error distribution is the figure of merit.  This tool
quantises synthetic K or V tiles on the GPU (``kvarn_token_errors``: quantise,
dequantise, compare, per token), once per variant:

    full      rotation + normalisation (the preset)
    no_norm   rotation only (0 normalisation iterations)
    no_rot    normalisation only (no rotation)
    plain     neither: per-token asymmetric round-to-nearest

and reports the relative per-token error e_t = |xhat_t - x_t| / |x_t| (L2
over the 128 channels): mean, percentiles, the mean of the largest 5%, and
the share of the total squared error those tokens carry.

    python -m bit_kv_cache_quantize_gb300.errors --workload qwen3_4b_layer --kv k
"""
from __future__ import annotations

import argparse
import json

import numpy as np

VARIANTS = {"full": (1, None), "no_norm": (1, 0), "no_rot": (0, None), "plain": (0, 0)}


def error_stats(err2: np.ndarray, norm2: np.ndarray, top: float = 0.05) -> dict:
    """Distribution of the relative per-token error sqrt(err2 / norm2) over
    tokens with a nonzero norm."""
    err2 = np.asarray(err2, np.float64).reshape(-1)
    norm2 = np.asarray(norm2, np.float64).reshape(-1)
    keep = norm2 > 0
    e2, n2 = err2[keep], norm2[keep]
    rel = np.sqrt(e2 / n2)
    k = max(1, int(round(top * rel.size)))
    order = np.argsort(e2)
    return {
        "tokens": int(rel.size),
        "mean": float(rel.mean()),
        "p50": float(np.percentile(rel, 50)),
        "p95": float(np.percentile(rel, 95)),
        "p99": float(np.percentile(rel, 99)),
        "max": float(rel.max()),
        "top_mean": float(np.sort(rel)[-k:].mean()),
        "top_share_sq_err": float(e2[order[-k:]].sum() / e2.sum()) if e2.sum() > 0 else 0.0,
    }


def measure(w, kv: str, rotate: int, iters, seqs=None, device="cuda"):
    """(err2, norm2) [n_tiles, H, 128] for the closed tiles of `seqs` of
    workload w, K (kv='k') or V (kv='v'), one GPU call per sequence."""
    import torch

    from . import inputs as I
    from . import kvarn as K

    seqs = list(range(w.batch)) if seqs is None else seqs
    iters = w.extra.get("iters", 8) if iters is None else iters
    cfg = K.make_config(w.num_kv_heads, w.num_q_heads, 1, w.dtype, k_bits=w.k_bits, v_bits=w.v_bits)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    e_all, n_all = [], []
    for b in seqs:
        n_tiles = w.seq_lens[b] // 128
        if n_tiles == 0:
            continue
        x = I.kv_sequence(w, kv, b, n_tiles * 128, device)
        first = torch.arange(n_tiles, dtype=torch.int64, device=device) * 128
        sb = K.kvarn_token_errors_scratch_bytes(cfg, n_tiles, kv == "v")
        scratch = torch.empty(sb, dtype=torch.uint8, device=device)
        out = torch.empty(n_tiles, w.num_kv_heads, 128, 2, dtype=torch.float32, device=device)
        K.kvarn_token_errors(cfg, x, w.num_kv_heads * 128, x.shape[0], first, n_tiles, int(kv == "v"), rotate, iters,
                             scratch, sb, out, err)
        torch.cuda.synchronize()
        if int(err.item()):
            raise RuntimeError(f"device error {int(err.item())}")
        o = out.cpu().numpy().astype(np.float64)
        e_all.append(o[..., 0])
        n_all.append(o[..., 1])
    return np.concatenate(e_all), np.concatenate(n_all)


def ablation(w, kv: str, seqs=None, device="cuda") -> dict:
    """error_stats for every variant."""
    out = {}
    for name, (rot, iters) in VARIANTS.items():
        e2, n2 = measure(w, kv, rot, iters, seqs, device)
        out[name] = error_stats(e2, n2)
    return out


def main():
    from . import build as B
    from . import inputs as I

    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="qwen3_4b_layer",
                    choices=["single_tile", "qwen3_4b_layer", "qwen3_32b_decode_16k"])
    ap.add_argument("--kv", default="k", choices=["k", "v"])
    ap.add_argument("--k-bits", type=int, default=4, choices=[4, 2])
    ap.add_argument("--v-bits", type=int, default=2, choices=[2, 4])
    ap.add_argument("--seqs", type=int, default=2, help="sequences of the workload to measure")
    args = ap.parse_args()
    B.build()
    w = {"single_tile": I.single_tile, "qwen3_4b_layer": I.qwen3_4b, "qwen3_32b_decode_16k": I.qwen3_32b}[args.workload]()
    w.k_bits, w.v_bits = args.k_bits, args.v_bits
    res = ablation(w, args.kv, seqs=list(range(min(args.seqs, w.batch))))
    print(json.dumps({"workload": w.name, "kv": args.kv, "k_bits": w.k_bits, "v_bits": w.v_bits, "variants": res}))


if __name__ == "__main__":
    main()
