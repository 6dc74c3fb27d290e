"""GPU read path (packed decode attention, 16-bit comparison kernel) against
the CPU oracle.  The packed cache the GPU reads is made of ORACLE records
(uploaded), so the expected outputs never depend on the GPU quantiser."""
import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_quantize_gb300 import inputs as I
from bit_kv_cache_quantize_gb300 import kvarn as K
from bit_kv_cache_quantize_gb300.cache import PagedCache

from gpu_helpers import bits, device, oracle_attention_units, oracle_decode, oracle_tiles, upload_oracle_prefill

pytestmark = pytest.mark.gpu
T = D = 128
TOL = 1e-3


def load_oracle_records(w, c: PagedCache, seqs, ctx):
    """Quantise the closed tiles of `seqs` with the oracle, upload the
    records into the GPU pool and the raw remainder into the open tile.
    Returns per (b, h) the oracle records."""
    recs = {}
    jobs, keys = [], []
    for b in seqs:
        k, v = ctx[b]
        n_full = k.shape[0] // T
        for t in range(n_full):
            for h in range(w.num_kv_heads):
                for kv, src in ((0, k), (1, v)):
                    jobs.append((src[t * T:(t + 1) * T, h], kv))
                    keys.append((b, t, h, kv))
    tiles = oracle_tiles(jobs, w.dtype, k_bits=w.k_bits, v_bits=w.v_bits)
    for (b, t, h, kv), tl in zip(keys, tiles):
        rec = O.pack_record(bool(kv), tl, w.k_bits, w.v_bits)
        recs[(b, t, h, kv)] = rec
        c.set_record(int(c.table[b, t]), h, kv, torch.from_numpy(rec).to(c.device))
    for b in seqs:
        k, v = ctx[b]
        n_full = k.shape[0] // T
        r = k.shape[0] - n_full * T
        if r:
            c.tail[b, :, 0, :r] = k[n_full * T:].permute(1, 0, 2).to(c.device)
            c.tail[b, :, 1, :r] = v[n_full * T:].permute(1, 0, 2).to(c.device)
    return recs


def oracle_outputs(w, seqs, ctx, recs, q, lens=None):
    """Oracle attention per (b, h) over oracle records + raw tail."""
    G = w.G
    units, keys = [], []
    for b in seqs:
        k, v = ctx[b]
        n = k.shape[0] if lens is None else lens[b]
        n_full = n // T
        for h in range(w.num_kv_heads):
            units.append(dict(
                q=O.decode16(bits(q[b, h * G:(h + 1) * G]), w.dtype),
                krec=[recs[(b, t, h, 0)] for t in range(n_full)],
                vrec=[recs[(b, t, h, 1)] for t in range(n_full)],
                ktail=O.decode16(bits(k[n_full * T:n, h]), w.dtype).reshape(-1, D),
                vtail=O.decode16(bits(v[n_full * T:n, h]), w.dtype).reshape(-1, D)))
            keys.append((b, h))
    outs = oracle_attention_units(units, w.scale, w.k_bits, w.v_bits)
    return dict(zip(keys, outs))


def run_decode_case(w, seqs=None, full_gpu_prefill=False):
    dev = device()
    seqs = list(range(w.batch)) if seqs is None else seqs
    c = PagedCache(w, dev)
    # inputs generated once on the device; the oracle reads the same bytes
    ctx = {b: (I.kv_sequence(w, "k", b, w.seq_lens[b], dev).cpu(), I.kv_sequence(w, "v", b, w.seq_lens[b], dev).cpu())
           for b in seqs}
    if full_gpu_prefill:
        c.prefill()            # every sequence, GPU quantiser
    recs = load_oracle_records(w, c, seqs, ctx)
    q = I.queries(w, device=dev).cpu()
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    c.decode(q.to(dev), out)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    want = oracle_outputs(w, seqs, ctx, recs, q)
    got = out.cpu().numpy().astype(np.float64)
    worst = 0.0
    for (b, h), o in want.items():
        d = np.abs(got[b, h * w.G:(h + 1) * w.G] - o).max()
        worst = max(worst, d)
    print(f"{w.name}: max |gpu - oracle| = {worst:.3e}")
    assert worst <= TOL
    return worst


def test_single_tile():
    run_decode_case(I.single_tile())


def test_qwen3_4b_layer():
    run_decode_case(I.qwen3_4b())


def ragged_small():
    return I.Workload("ragged_small", 7, 16, 2, "f16", [1, 127, 128, 129, 700, 2200, 0], seed=21, max_tokens=2400,
                      block_perm=True)


def test_ragged_tails_and_empty_sequence():
    run_decode_case(ragged_small())


def test_k2_single_tile():
    w = I.single_tile()
    w.k_bits = 2
    run_decode_case(w)


def test_k2_qwen3_4b_layer():
    w = I.qwen3_4b()
    w.k_bits = 2
    run_decode_case(w)


def test_k2_ragged_tails_and_empty_sequence():
    w = ragged_small()
    w.k_bits = 2
    run_decode_case(w)


def test_v4_single_tile():
    w = I.single_tile()
    w.v_bits = 4
    run_decode_case(w)


def test_v4_qwen3_4b_layer():
    w = I.qwen3_4b()
    w.v_bits = 4
    run_decode_case(w)


def test_v4_ragged_tails_and_empty_sequence():
    w = ragged_small()
    w.v_bits = 4
    run_decode_case(w)


def test_64_tile_chunks_ragged():
    """120 ragged sequences of up to 8191 tokens (64 blocks), 64 q / 8 KV
    heads: 120 x 8 (sequence, head) pairs give at least three waves of CTAs
    with one 64-tile chunk each, so the call takes 64-tile chunks (partial
    ones for every sequence), beside an empty sequence, a one-token one, one
    of exactly 63 closed tiles and one ending one token short of 64."""
    lens = I.ragged_lengths(31, 116, lo=1, hi=8150) + [0, 1, 63 * T, 64 * T - 1]
    w = I.Workload("ragged_chunk64", len(lens), 64, 8, "f16", lens, seed=33, max_tokens=64 * T, block_perm=True)
    run_decode_case(w)


def test_group_sizes_bf16():
    for hq, hkv in ((2, 2), (4, 2), (6, 3)):
        w = I.Workload(f"g{hq // hkv}", 3, hq, hkv, "bf16", [300, 128, 77], seed=30 + hq, max_tokens=300,
                       v_dist="t4", k_outliers="random")
        run_decode_case(w)


@pytest.mark.slow
def test_qwen3_32b_full_size_all_sequences():
    """The 16K decode at full size (32 x 16384 tokens, 64 q / 8 KV heads,
    permuted blocks) in the launch the benchmark times: every closed tile
    holds the oracle's record, and all 32 sequences x 64 query heads are
    compared with the oracle's attention."""
    dev = device()
    w = I.qwen3_32b()
    c = PagedCache(w, dev)
    recs, _ = upload_oracle_prefill(w, c, range(w.batch))
    q = I.queries(w, device=dev)
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    c.decode(q, out)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    qh = q.cpu()
    nf = w.seq_lens[0] // T
    units = [(O.decode16(bits(qh[b, h * w.G:(h + 1) * w.G]), w.dtype),
              [recs[(b, t, h, 0)] for t in range(nf)], [recs[(b, t, h, 1)] for t in range(nf)],
              np.zeros((0, D)), np.zeros((0, D))) for b in range(w.batch) for h in range(w.num_kv_heads)]
    want = oracle_decode(w, units, w.scale).reshape(w.batch, w.num_q_heads, D)
    worst = np.abs(out.cpu().numpy().astype(np.float64) - want).max()
    print(f"{w.name}: all {w.batch} sequences, max |gpu - oracle| = {worst:.3e}")
    assert worst <= TOL


def fp16_case(w, seqs=None):
    dev = device()
    seqs = list(range(w.batch)) if seqs is None else seqs
    c = PagedCache(w, dev, fp16_pool=True)
    ctx = {}
    for b in range(w.batch):
        k = I.kv_sequence(w, "k", b, w.seq_lens[b], dev)
        v = I.kv_sequence(w, "v", b, w.seq_lens[b], dev)
        c.quantize_sequence(b, k, v)
        if b in seqs:
            ctx[b] = (k.cpu(), v.cpu())
    q = I.queries(w).to(dev)
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    c.decode_fp16(q, out)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    got = out.cpu().numpy().astype(np.float64)
    worst = 0.0
    for b in seqs:
        k, v = ctx[b]
        for h in range(w.num_kv_heads):
            want = O.attention(O.decode16(bits(q[b, h * w.G:(h + 1) * w.G]), w.dtype),
                               O.decode16(bits(k[:, h]), w.dtype), O.decode16(bits(v[:, h]), w.dtype), w.scale)
            worst = max(worst, np.abs(got[b, h * w.G:(h + 1) * w.G] - want).max())
    print(f"fp16 {w.name}: max |gpu - oracle| = {worst:.3e}")
    assert worst <= TOL


def test_fp16_baseline_ragged():
    fp16_case(ragged_small())


def test_fp16_baseline_bf16_layer():
    fp16_case(I.qwen3_4b(), seqs=[0, 5])


def test_bounded_wait_expiry_reports_timeout_and_returns():
    """A record copy that never starts: the wait on it gives up after the
    short poll limit, the kernel stores KVARN_DEV_ERR_TIMEOUT and returns,
    and the device keeps working (a normal decode afterwards matches the
    oracle)."""
    dev = device()
    # sequence 0 has closed tiles, so its first unit has a key-record copy to leave out
    w = I.Workload("wait_expiry", 3, 16, 2, "f16", [700, 129, 2200], seed=23, max_tokens=2400, block_perm=True)
    c = PagedCache(w, dev)
    ctx = {b: (I.kv_sequence(w, "k", b, w.seq_lens[b], dev).cpu(), I.kv_sequence(w, "v", b, w.seq_lens[b], dev).cpu())
           for b in range(w.batch)}
    recs = load_oracle_records(w, c, list(range(w.batch)), ctx)
    q = I.queries(w).to(dev)
    out = torch.zeros(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    lens = c.lens.clone()
    K.kvarn_test_decode_wait_expiry(c.cfg, q, c.table, c.max_blocks, lens, w.batch, c.pool, c.tail, w.scale, out,
                                    c.ws, c.ws_bytes, c.err, 64)
    torch.cuda.synchronize()                                   # the call completes
    assert c.check_error() == K.KVARN_DEV_ERR_TIMEOUT
    assert torch.isfinite(out[1:]).all()
    with pytest.raises(K.KvarnError):                          # the poll limit must be positive
        K.kvarn_test_decode_wait_expiry(c.cfg, q, c.table, c.max_blocks, lens, w.batch, c.pool, c.tail, w.scale,
                                        out, c.ws, c.ws_bytes, c.err, 0)
    c.err.zero_()
    c.decode(q, out)                                           # the device still answers, correctly
    torch.cuda.synchronize()
    assert c.check_error() == 0
    want = oracle_outputs(w, list(range(w.batch)), ctx, recs, q.cpu())
    got = out.cpu().numpy().astype(np.float64)
    worst = max(np.abs(got[b, h * w.G:(h + 1) * w.G] - o).max() for (b, h), o in want.items())
    assert worst <= TOL


def test_decode_device_errors():
    dev = device()
    w = ragged_small()
    c = PagedCache(w, dev)
    q = I.queries(w).to(dev)
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    bad = c.table.clone()
    bad[4, 2] = c.num_blocks + 5
    K.kvarn_decode_attention(c.cfg, q, bad, c.max_blocks, c.lens, w.batch, c.pool, c.tail, w.scale, out, c.ws,
                             c.ws_bytes, c.err)
    torch.cuda.synchronize()
    assert c.check_error() == K.KVARN_DEV_ERR_BLOCK_RANGE
    c.err.zero_()
    lens = c.lens.clone()
    lens[1] = T * c.max_blocks + 1
    c.decode(q, out, lens=lens)
    torch.cuda.synchronize()
    assert c.check_error() == K.KVARN_DEV_ERR_TOKEN_RANGE
    assert not out[1].any()


def degenerate_context(dtype, k_bits, v_bits):
    """One sequence per degenerate tile of the quantiser tests (1 KV head,
    8 query heads): that tile as values, a degenerate key tile (cycling
    through all but the one at the 16-bit range), then a random tile and a
    5-token open tail.  Returns the workload and {b: (k, v)} [n, 1, 128]."""
    from test_gpu_quantize import degenerate_tiles
    tiles = degenerate_tiles(dtype)[:, 0].reshape(-1, T, D)  # [n, T, D] 16-bit
    n = tiles.shape[0]
    k_ok = [i for i in range(n) if i != 4]  # index 4: values at the 16-bit range
    rng = np.random.default_rng(5)
    n_tok = 2 * T + 5
    w = I.Workload(f"degenerate_{dtype}", n, 8, 1, dtype, [n_tok] * n, seed=8, k_bits=k_bits, v_bits=v_bits)
    td = I.torch_dtype(dtype)
    ctx = {}
    for b in range(n):
        rk = torch.from_numpy(rng.standard_normal((T + 5, D)).astype(np.float32)).to(td)
        rv = torch.from_numpy(rng.standard_normal((T + 5, D)).astype(np.float32)).to(td)
        k = torch.cat([tiles[k_ok[b % len(k_ok)]], rk]).reshape(n_tok, 1, D)
        v = torch.cat([tiles[b], rv]).reshape(n_tok, 1, D)
        ctx[b] = (k, v)
    return w, ctx


@pytest.mark.parametrize("dtype,k_bits,v_bits", [("f16", 4, 2), ("bf16", 4, 2), ("f16", 2, 2), ("bf16", 4, 4)])
def test_decode_over_degenerate_tiles(dtype, k_bits, v_bits):
    """Attention over records of degenerate tiles (the quantiser's edge cases:
    zero, identical tokens, one large or saturating outlier, values at the
    16-bit range, tiny values, one live channel or token) against the oracle.
    Sequence i has degenerate value tile i and a degenerate key tile, then a
    random tile and a 5-token open tail.  Keys at the 16-bit range are left
    out: their scores reach ~1e6 and the fp32-vs-fp64 comparison would test
    the conditioning of the softmax, not the kernel.  The max-abs bound is
    1e-3 scaled by max(1, max |v|) of the sequence, since values at the
    16-bit range give outputs of that size."""
    dev = device()
    w, ctx = degenerate_context(dtype, k_bits, v_bits)
    n = w.batch
    c = PagedCache(w, dev)
    recs = load_oracle_records(w, c, list(range(n)), ctx)
    q = I.queries(w, device=dev).cpu()
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    c.decode(q.to(dev), out)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    want = oracle_outputs(w, list(range(n)), ctx, recs, q)
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    worst = 0.0
    for (b, h), o in want.items():
        scale = max(1.0, float(ctx[b][1].float().abs().max()))
        worst = max(worst, np.abs(got[b, h * w.G:(h + 1) * w.G] - o).max() / scale)
    print(f"{w.name} K{k_bits}/V{v_bits}: max |gpu - oracle| / max(1, max|v|) = {worst:.3e}")
    assert worst <= TOL


def test_shared_prefix_blocks():
    """Sequences whose block tables share physical blocks (a common prefix
    kept once, as a paged serving cache does) decode like sequences with
    private copies: sequences 1 and 2 reuse the first 3 and 5 blocks of
    sequence 0 and hold the same tokens there."""
    dev = device()
    lens = [1000, 700, 1300, 260]
    w = I.Workload("shared_prefix", len(lens), 32, 4, "bf16", lens, seed=21, block_perm=True)
    c = PagedCache(w, dev)
    ctx = {b: [I.kv_sequence(w, "k", b, n, dev).cpu(), I.kv_sequence(w, "v", b, n, dev).cpu()]
           for b, n in enumerate(lens)}
    for b, nb in ((1, 3), (2, 5)):
        for i in range(2):
            ctx[b][i][:nb * T] = ctx[0][i][:nb * T]
        c.table[b, :nb] = c.table[0, :nb]
    recs = load_oracle_records(w, c, list(range(w.batch)), ctx)
    q = I.queries(w, device=dev).cpu()
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    c.decode(q.to(dev), out)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    want = oracle_outputs(w, list(range(w.batch)), ctx, recs, q)
    got = out.cpu().numpy().astype(np.float64)
    worst = max(np.abs(got[b, h * w.G:(h + 1) * w.G] - o).max() for (b, h), o in want.items())
    print(f"shared prefix: max |gpu - oracle| = {worst:.3e}")
    assert worst <= TOL


@pytest.mark.slow
def test_long_context_128k():
    """Two sequences of ~128 K tokens (1023 closed tiles and an open tail of
    91 tokens; 1024 closed tiles): 64 split-K chunks of 16 tiles per KV head
    plus the open tile, merged by the combine.  Every closed tile holds the
    oracle's record and all 2 x 64 query heads are compared with the
    oracle's attention."""
    dev = device()
    lens = [131072 - 37, 131072]
    w = I.Workload("long_128k", 2, 64, 8, "f16", lens, seed=77, max_tokens=max(lens), block_perm=True)
    c = PagedCache(w, dev)
    recs, kept = upload_oracle_prefill(w, c, range(w.batch))
    q = I.queries(w, device=dev)
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    c.decode(q, out)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    qh = q.cpu()
    units = []
    for b in range(w.batch):
        nf = lens[b] // T
        k, v, first = kept[b]
        assert first == nf * T
        for h in range(w.num_kv_heads):
            units.append((O.decode16(bits(qh[b, h * w.G:(h + 1) * w.G]), w.dtype),
                          [recs[(b, t, h, 0)] for t in range(nf)], [recs[(b, t, h, 1)] for t in range(nf)],
                          O.decode16(bits(k[:, h]), w.dtype).reshape(-1, D),
                          O.decode16(bits(v[:, h]), w.dtype).reshape(-1, D)))
    want = oracle_decode(w, units, w.scale).reshape(w.batch, w.num_q_heads, D)
    worst = np.abs(out.cpu().numpy().astype(np.float64) - want).max()
    print(f"{w.name}: max |gpu - oracle| = {worst:.3e}")
    assert worst <= TOL


@pytest.mark.parametrize("h_kv,g", [(32, 1), (16, 2)])
def test_many_kv_heads(h_kv, g):
    """More KV heads than the workloads above: 32 heads without grouping
    (multi-head attention) and 16 heads in pairs, ragged lengths."""
    w = I.Workload(f"kv{h_kv}_g{g}", 3, h_kv * g, h_kv, "bf16", [700, 129, 1500], seed=60 + h_kv, max_tokens=1500,
                   block_perm=True, v_dist="t4", k_outliers="random")
    run_decode_case(w)
