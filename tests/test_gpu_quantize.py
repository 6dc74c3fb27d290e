"""GPU write path (quantise, dequantise) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_quantize_gb300 import inputs as I
from bit_kv_cache_quantize_gb300 import kvarn as K
from bit_kv_cache_quantize_gb300.cache import PagedCache

import parity as PR
from gpu_helpers import bits, device, oracle_tiles, tile_values

pytestmark = pytest.mark.gpu
T = D = 128


def quantize_and_compare(w, seqs, sample=None, seed=0):
    """GPU-quantise the context of `seqs`, then compare all (or `sample`
    random) records with the oracle."""
    dev = device()
    c = PagedCache(w, dev)
    ctx = {}
    for b in seqs:
        n = w.seq_lens[b]
        k = I.kv_sequence(w, "k", b, n, dev)
        v = I.kv_sequence(w, "v", b, n, dev)
        c.quantize_sequence(b, k, v)
        ctx[b] = (k, v)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    jobs = [(b, t, h, kv) for b in seqs for t in range(w.seq_lens[b] // T) for h in range(w.num_kv_heads)
            for kv in (0, 1)]
    if sample is not None and sample < len(jobs):
        rng = np.random.default_rng(seed)
        jobs = [jobs[i] for i in rng.choice(len(jobs), sample, replace=False)]
    tiles = oracle_tiles([(ctx[b][kv][t * T:(t + 1) * T, h], kv) for b, t, h, kv in jobs], w.dtype,
                         k_bits=w.k_bits, v_bits=w.v_bits)
    st = PR.Stats()
    for (b, t, h, kv), tl in zip(jobs, tiles):
        blk = int(c.table[b, t])
        rec = c.record(blk, h, kv).cpu().numpy()
        PR.compare_record(rec, tl, bool(kv), st, where=f"seq {b} tile {t} head {h} {'V' if kv else 'K'}",
                          k_bits=w.k_bits, v_bits=w.v_bits)
    print(w.name, PR.finish(st))
    return st


def test_single_tile():
    st = quantize_and_compare(I.single_tile(), [0])
    assert st.tiles == 2


def test_qwen3_4b_layer_all_tiles():
    w = I.qwen3_4b()
    quantize_and_compare(w, list(range(w.batch)))


def test_k2_single_tile():
    w = I.single_tile()
    w.k_bits = 2
    st = quantize_and_compare(w, [0])
    assert st.tiles == 2


def test_v4_single_tile():
    w = I.single_tile()
    w.v_bits = 4
    st = quantize_and_compare(w, [0])
    assert st.tiles == 2


def test_v4_qwen3_4b_layer_all_tiles():
    w = I.qwen3_4b()
    w.v_bits = 4
    quantize_and_compare(w, list(range(w.batch)))


def test_k2_qwen3_4b_layer_all_tiles():
    w = I.qwen3_4b()
    w.k_bits = 2
    quantize_and_compare(w, list(range(w.batch)))


@pytest.mark.slow
def test_prefill_32b_full_size_all_tiles():
    """All 32 x 16384 tokens x 8 heads (65536 tile jobs) in the launch the
    benchmark times; every record compared with the oracle's (the oracle
    runs on all host cores, a chunk of tiles at a time)."""
    w = I.prefill_32b()
    dev = device()
    c = PagedCache(w, dev)
    B, n = w.batch, w.seq_lens[0]
    k = torch.empty(B * n, w.num_kv_heads, D, dtype=I.torch_dtype(w.dtype), device=dev)
    v = torch.empty_like(k)
    for b in range(B):
        k[b * n:(b + 1) * n] = I.kv_sequence(w, "k", b, n, dev)
        v[b * n:(b + 1) * n] = I.kv_sequence(w, "v", b, n, dev)
    n_tiles = B * n // T
    first = torch.arange(n_tiles, dtype=torch.int64, device=dev) * T
    dst = c.table[:, : n // T].reshape(-1).contiguous()
    K.kvarn_quantize_tiles(c.cfg, k, v, w.num_kv_heads * D, B * n, first, dst, n_tiles, c.pool, c.err)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    H = w.num_kv_heads
    pool = c.pool.cpu().numpy()
    srcs = [bits(k).reshape(-1), bits(v).reshape(-1)]
    del k, v
    dsth = dst.cpu().numpy().astype(np.int64)
    st = PR.Stats()
    CH = 64                                            # tiles per chunk (x 8 heads x K|V)
    for t0 in range(0, n_tiles, CH):
        tiles = np.arange(t0, min(n_tiles, t0 + CH))
        first = (tiles[:, None] * (T * H * D) + np.arange(H)[None, :] * D).reshape(-1)
        for kv in (0, 1):
            ora = O.quantize_batch_fields(srcs[kv], w.dtype, first, H * D, O.levels(bool(kv)))
            rb = K.rec_bytes(2 if kv else 4)
            offs = (dsth[tiles][:, None] * c.block_bytes + np.arange(H)[None, :] * K.HEAD_REC + kv * K.K_REC)
            recs = pool[offs.reshape(-1)[:, None] + np.arange(rb)[None, :]]
            PR.compare_batch(recs, ora, bool(kv), st, where=f"tiles {t0}.. {'V' if kv else 'K'}")
    print(PR.finish(st))
    assert st.tiles == n_tiles * H * 2 == 65536


def degenerate_tiles(dtype):
    """[n_tiles*128, 1, 128] 16-bit: zero, identical tokens, one large
    outlier, a saturating outlier, extreme values, tiny values, random."""
    rng = np.random.default_rng(11)
    tiles = []
    tiles.append(np.zeros((T, D)))
    row = rng.standard_normal(D)
    tiles.append(np.repeat(row[None], T, axis=0))
    x = np.zeros((T, D)); x[5, 9] = 3000.0; tiles.append(x)
    x = rng.standard_normal((T, D)) * 0.1; x[77, 3] = 60000.0; tiles.append(x)
    tiles.append(np.where(rng.random((T, D)) < 0.5, -1.0, 1.0) * (65504.0 if dtype == "f16" else 1e4))
    tiles.append(rng.standard_normal((T, D)) * 1e-6)
    x = np.zeros((T, D)); x[:, 0] = rng.standard_normal(T); tiles.append(x)   # one live channel
    x = np.zeros((T, D)); x[3] = rng.standard_normal(D); tiles.append(x)      # one live token
    tiles.append(rng.standard_normal((T, D)))
    arr = np.concatenate(tiles).astype(np.float32)
    t = torch.from_numpy(arr).to(I.torch_dtype(dtype))
    return t.reshape(-1, 1, D)


@pytest.mark.parametrize("dtype,k_bits,v_bits", [("f16", 4, 2), ("bf16", 4, 2), ("f16", 2, 2), ("bf16", 4, 4)])
def test_degenerate_tiles(dtype, k_bits, v_bits):
    dev = device()
    kv = degenerate_tiles(dtype).to(dev)
    n_tiles = kv.shape[0] // T
    cfg = K.make_config(1, 1, n_tiles, dtype, k_bits=k_bits, v_bits=v_bits)
    pool = torch.zeros(n_tiles * K.kvarn_block_bytes(cfg), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    first = torch.arange(n_tiles, dtype=torch.int64, device=dev) * T
    dst = torch.arange(n_tiles, dtype=torch.int32, device=dev).flip(0).contiguous()
    K.kvarn_quantize_tiles(cfg, kv, kv, D, kv.shape[0], first, dst, n_tiles, pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    tiles = oracle_tiles([(kv[i * T:(i + 1) * T, 0], is_v) for i in range(n_tiles) for is_v in (0, 1)], dtype,
                         k_bits=k_bits, v_bits=v_bits)
    st = PR.Stats()
    bb = K.kvarn_block_bytes(cfg)
    kr = K.rec_bytes(k_bits)
    for idx, tl in enumerate(tiles):
        i, is_v = divmod(idx, 2)
        blk = int(dst[i])
        rec = pool[blk * bb + is_v * kr: blk * bb + is_v * kr + K.rec_bytes(v_bits if is_v else k_bits)]
        PR.compare_record(rec.cpu().numpy(), tl, bool(is_v), st, where=f"degenerate tile {i} {'V' if is_v else 'K'}",
                          k_bits=k_bits, v_bits=v_bits)
    print(PR.finish(st))


@pytest.mark.parametrize("iters", [0, 1, 3])
def test_other_sinkhorn_counts(iters):
    dev = device()
    w = I.single_tile()
    k = I.kv_sequence(w, "k", 0, T, dev)
    cfg = K.make_config(1, 1, 1, "f16", sinkhorn_iters=iters)
    pool = torch.zeros(K.kvarn_block_bytes(cfg), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    K.kvarn_quantize_tiles(cfg, k, k, D, T, torch.zeros(1, dtype=torch.int64, device=dev),
                           torch.zeros(1, dtype=torch.int32, device=dev), 1, pool, err)
    tl = oracle_tiles([(k[:, 0], 0), (k[:, 0], 1)], "f16", iters)
    st = PR.Stats()
    PR.compare_record(pool[:K.K_REC].cpu().numpy(), tl[0], False, st)
    PR.compare_record(pool[K.K_REC:K.K_REC + K.V_REC].cpu().numpy(), tl[1], True, st)
    PR.finish(st)


@pytest.mark.parametrize("k_bits,v_bits", [(4, 2), (2, 2), (4, 4)])
def test_dequantize_matches_oracle(k_bits, v_bits):
    """Oracle-made records uploaded; the GPU dequantiser must rebuild the
    oracle's unrotated values."""
    dev = device()
    w = I.qwen3_4b()
    k = I.kv_values(w, "k", 0, 0, 2 * T)
    v = I.kv_values(w, "v", 0, 0, 2 * T)
    H = 2
    cfg = K.make_config(H, H, 3, "bf16", k_bits=k_bits, v_bits=v_bits)
    bb = K.kvarn_block_bytes(cfg)
    pool = torch.zeros(3 * bb, dtype=torch.uint8)
    want = np.zeros((2, 2, H, T, D))
    blocks = [2, 0]
    for n, blk in enumerate(blocks):
        for h in range(H):
            for kv, src in ((0, k), (1, v)):
                tl = O.quantize_tile(tile_values(src[n * T:(n + 1) * T, h], "bf16"), O.levels(bool(kv), k_bits, v_bits))
                rec = O.pack_record(bool(kv), tl, k_bits, v_bits)
                off = blk * bb + h * K.head_rec(k_bits, v_bits) + kv * K.rec_bytes(k_bits)
                pool[off:off + rec.size] = torch.from_numpy(rec)
                want[n, kv, h] = O.dequantize_record(bool(kv), rec, k_bits, v_bits=v_bits)
    pool = pool.to(dev)
    out = torch.empty(2, 2, H, T, D, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    K.kvarn_dequantize(cfg, pool, torch.tensor(blocks, dtype=torch.int32, device=dev), 2, out, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    assert np.abs(got - want).max() <= 1e-5 * max(1.0, np.abs(want).max())


def test_device_errors_skip_units():
    dev = device()
    cfg = K.make_config(1, 1, 2, "f16")
    x = torch.randn(2 * T, 1, D, device=dev).half()
    pool = torch.zeros(2 * K.kvarn_block_bytes(cfg), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    first = torch.tensor([0, T], dtype=torch.int64, device=dev)
    K.kvarn_quantize_tiles(cfg, x, x, D, 2 * T, first, torch.tensor([0, 7], dtype=torch.int32, device=dev), 2,
                           pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == K.KVARN_DEV_ERR_BLOCK_RANGE
    assert pool[:K.K_REC].any() and not pool[K.kvarn_block_bytes(cfg):].any()
    err.zero_()
    K.kvarn_quantize_tiles(cfg, x, x, D, 2 * T, torch.tensor([0, T + 1], dtype=torch.int64, device=dev),
                           torch.tensor([0, 1], dtype=torch.int32, device=dev), 2, pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == K.KVARN_DEV_ERR_TOKEN_RANGE


@pytest.mark.parametrize("h_kv,g", [(32, 1), (16, 2)])
def test_many_kv_heads(h_kv, g):
    """32 and 16 KV heads: every closed tile of every head record by record."""
    w = I.Workload(f"q_kv{h_kv}", 2, h_kv * g, h_kv, "bf16", [640, 300], seed=80 + h_kv, max_tokens=640,
                   v_dist="t4", k_outliers="random")
    quantize_and_compare(w, list(range(w.batch)))
