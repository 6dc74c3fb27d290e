"""Decode-step path: append one token per sequence into the raw open tile,
close and quantise tiles as they fill, attend after every append."""
import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_quantize_gb300 import inputs as I
from bit_kv_cache_quantize_gb300 import kvarn as K
from bit_kv_cache_quantize_gb300.cache import PagedCache

import parity as PR
from gpu_helpers import bits, device, oracle_decode, oracle_tiles, upload_oracle_prefill

pytestmark = pytest.mark.gpu
T = D = 128
TOL = 1e-3


def run_steps(w, steps, check_seqs=None, attend_every=1, full_check_steps=()):
    """Prefill, then `steps` decode steps (append one token per sequence,
    attend).  Every tile that closes (any sequence) is compared with the
    oracle record by record; the attention of `check_seqs` (default all) is
    compared with the oracle's after every `attend_every`-th step and the
    last, and that of every sequence at the steps in `full_check_steps`.
    Sequences whose attention is checked hold oracle records only."""
    dev = device()
    c = PagedCache(w, dev)
    c.prefill()
    torch.cuda.synchronize()
    assert c.check_error() == 0
    check_seqs = list(range(w.batch)) if check_seqs is None else check_seqs
    attend_seqs = list(range(w.batch)) if full_check_steps else check_seqs
    total = [n + steps for n in w.seq_lens]
    # oracle records for the closed prefill tiles of every sequence whose
    # attention is checked; raw tokens from its open tile on are kept on the
    # host (inputs generated on the device; the oracle reads the same bytes)
    recs, kept = upload_oracle_prefill(w, c, attend_seqs, keep_to=total)
    st = PR.Stats()
    lens = torch.tensor(w.seq_lens, dtype=torch.int32)
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    worst = 0.0
    n_attended = set()
    for s in range(steps):
        pos = lens.clone()
        k_new = torch.stack([I.kv_values(w, "k", b, int(pos[b]), 1, dev)[0] for b in range(w.batch)])
        v_new = torch.stack([I.kv_values(w, "v", b, int(pos[b]), 1, dev)[0] for b in range(w.batch)])
        c.append(k_new, v_new, pos.to(dev))
        lens = pos + 1
        torch.cuda.synchronize()
        assert c.check_error() == 0
        # the raw slot holds the token bit for bit; tiles that filled are quantised
        closing = [b for b in range(w.batch) if int(pos[b]) % T == T - 1]
        for b in range(w.batch):
            slot = int(pos[b]) % T
            assert torch.equal(c.tail[b, :, 0, slot], k_new[b]) and torch.equal(c.tail[b, :, 1, slot], v_new[b])
        jobs, keys = [], []
        for b in closing:
            t = int(pos[b]) // T
            full_k = I.kv_values(w, "k", b, t * T, T, dev).cpu()
            full_v = I.kv_values(w, "v", b, t * T, T, dev).cpu()
            for h in range(w.num_kv_heads):
                jobs += [(full_k[:, h], 0), (full_v[:, h], 1)]
                keys += [(b, t, h, 0), (b, t, h, 1)]
        tiles = oracle_tiles(jobs, w.dtype, k_bits=w.k_bits, v_bits=w.v_bits)
        for (b, t, h, kv), tl in zip(keys, tiles):
            blk = int(c.table[b, t])
            PR.compare_record(c.record(blk, h, kv).cpu().numpy(), tl, bool(kv), st,
                              where=f"step {s} seq {b} closed tile {t} head {h} kv {kv}", k_bits=w.k_bits,
                              v_bits=w.v_bits)
            if b in kept:  # decode parity reads oracle records only
                rec = O.pack_record(bool(kv), tl, w.k_bits, w.v_bits)
                recs[(b, t, h, kv)] = rec
                c.set_record(blk, h, kv, torch.from_numpy(rec).to(dev))
        full = s in full_check_steps
        if not full and s % attend_every and s != steps - 1:
            continue
        q = I.queries(w, step=s + 1, device=dev).cpu()
        c.decode(q.to(dev), out, lens=lens.to(dev))
        torch.cuda.synchronize()
        assert c.check_error() == 0
        got = out.cpu().numpy().astype(np.float64)
        seqs = attend_seqs if full else check_seqs
        units, ukeys = [], []
        for b in seqs:
            n = int(lens[b])
            nf = n // T
            k, v, lo = kept[b]
            for h in range(w.num_kv_heads):
                units.append((O.decode16(bits(q[b, h * w.G:(h + 1) * w.G]), w.dtype),
                              [recs[(b, t, h, 0)] for t in range(nf)], [recs[(b, t, h, 1)] for t in range(nf)],
                              O.decode16(bits(k[nf * T - lo:n - lo, h]), w.dtype).reshape(-1, D),
                              O.decode16(bits(v[nf * T - lo:n - lo, h]), w.dtype).reshape(-1, D)))
                ukeys.append((b, h))
        want = oracle_decode(w, units, w.scale, w.k_bits, w.v_bits)
        for (b, h), o in zip(ukeys, want):
            worst = max(worst, np.abs(got[b, h * w.G:(h + 1) * w.G] - o).max())
            n_attended.add(b)
    print(w.name, PR.finish(st), f"max |gpu - oracle| = {worst:.3e} over {len(n_attended)} sequences")
    assert worst <= TOL
    return st


def test_append_close_small():
    w = I.Workload("append_small", 6, 16, 2, "f16", [125, 126, 127, 255, 300, 10], seed=41, decode_steps=4,
                   max_tokens=310, block_perm=True)
    st = run_steps(w, 4)
    assert st.tiles == 4 * 2 * 2   # seqs 0..3 close one tile each


def test_k2_append_close_small():
    w = I.Workload("append_small_k2", 6, 16, 2, "f16", [125, 126, 127, 255, 300, 10], seed=47, decode_steps=4,
                   max_tokens=310, block_perm=True, k_bits=2)
    st = run_steps(w, 4)
    assert st.tiles == 4 * 2 * 2


def test_v4_append_close_small():
    w = I.Workload("append_small_v4", 6, 16, 2, "bf16", [125, 126, 127, 255, 300, 10], seed=49, decode_steps=4,
                   max_tokens=310, block_perm=True, v_dist="t4", v_bits=4)
    st = run_steps(w, 4)
    assert st.tiles == 4 * 2 * 2


def test_append_close_bf16():
    w = I.Workload("append_bf16", 3, 8, 2, "bf16", [127, 383, 5], seed=43, decode_steps=2, max_tokens=400,
                   v_dist="t4", k_outliers="random", block_perm=True)
    run_steps(w, 2)


@pytest.mark.parametrize("k_bits,v_bits", [(4, 2), (2, 2), (4, 4)])
def test_append_every_sequence_closes(k_bits, v_bits):
    """320 sequences x 8 KV heads = 5120 (sequence, head, K|V) units, more
    than the grid's CTAs take in one pass of sixteen, and every sequence
    closes a tile on the same step: CTAs quantise up to sixteen tiles one
    after another and make two passes, in each preset.  Every closed tile
    is compared with the oracle."""
    lens = [127 + 128 * (b % 3) for b in range(320)]
    w = I.Workload(f"append_all_close_k{k_bits}v{v_bits}", len(lens), 16, 8, "bf16", lens, seed=53, decode_steps=1,
                   max_tokens=400, block_perm=True, k_bits=k_bits, v_bits=v_bits)
    st = run_steps(w, 1, check_seqs=[0, 1, 2, 319])
    assert st.tiles == 2 * 8 * len(lens)


@pytest.mark.slow
def test_ragged_serving_full_size():
    """256 sequences, lengths U[128, 32768], 64 decode steps: every tile that
    closes (any sequence) is compared with the oracle; the attention of all
    256 sequences is compared at steps 0 and 63, and that of 8 sampled
    sequences (4 of them closing a tile during the run) after every step."""
    w = I.ragged_32b()
    lens = np.array(w.seq_lens)
    closing = [b for b in range(w.batch) if (lens[b] % T) + 64 >= T][:4]
    others = [b for b in range(w.batch) if b not in closing][:4]
    run_steps(w, 64, check_seqs=closing + others, attend_every=1, full_check_steps=(0, 63))
