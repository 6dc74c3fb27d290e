"""GPU causal multi-query attention against the CPU oracle.  As in the decode
tests, the packed cache holds ORACLE records (uploaded) and the raw open
tile, so the expected outputs never depend on the GPU quantiser."""
import concurrent.futures

import numpy as np
import pytest
import torch

import oracle as O
from bit_kv_cache_quantize_gb300 import inputs as I
from bit_kv_cache_quantize_gb300 import kvarn as K
from bit_kv_cache_quantize_gb300.cache import PagedCache

from gpu_helpers import NTHREADS, bits, device
from test_gpu_decode import degenerate_context, load_oracle_records

pytestmark = pytest.mark.gpu
T = D = 128
TOL = 1e-3


def oracle_mq(w, seqs, ctx, recs, q, Q):
    """Oracle causal attention per (sequence, KV head): [Q, G, D] each."""
    G = w.G

    def one(key):
        b, h = key
        k, v = ctx[b]
        n = k.shape[0]
        nf = n // T
        Kc, Vc = O.cache_values([recs[(b, t, h, 0)] for t in range(nf)], [recs[(b, t, h, 1)] for t in range(nf)],
                                O.decode16(bits(k[nf * T:, h]), w.dtype), O.decode16(bits(v[nf * T:, h]), w.dtype),
                                w.k_bits, w.v_bits)
        qq = O.decode16(bits(q[b, :, h * G:(h + 1) * G]), w.dtype).reshape(Q, G, D)
        return O.causal_attention(qq, Kc, Vc, w.scale)

    keys = [(b, h) for b in seqs for h in range(w.num_kv_heads)]
    with concurrent.futures.ThreadPoolExecutor(NTHREADS) as ex:
        return dict(zip(keys, ex.map(one, keys)))


def run_mq_case(w, Q, seqs=None, full_gpu_prefill=False):
    dev = device()
    seqs = list(range(w.batch)) if seqs is None else seqs
    c = PagedCache(w, dev)
    ctx = {b: (I.kv_sequence(w, "k", b, w.seq_lens[b], dev).cpu(), I.kv_sequence(w, "v", b, w.seq_lens[b], dev).cpu())
           for b in seqs}
    if full_gpu_prefill:
        c.prefill()
    recs = load_oracle_records(w, c, seqs, ctx)
    q = I.multi_queries(w, Q, device=dev).cpu()
    out = torch.full((w.batch, Q, w.num_q_heads, D), float("nan"), dtype=torch.float32, device=dev)
    c.multiquery(q.to(dev), Q, out)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    got = out.cpu().numpy().astype(np.float64)
    worst = 0.0
    for (b, h), o in oracle_mq(w, seqs, ctx, recs, q, Q).items():
        g = got[b, :, h * w.G:(h + 1) * w.G]
        assert np.isfinite(g).all(), (b, h)
        worst = max(worst, np.abs(g - o).max())
    print(f"{w.name} Q={Q} k_bits={w.k_bits}: max |gpu - oracle| = {worst:.3e}")
    assert worst <= TOL
    return worst


def test_small_ragged_group8():
    w = I.Workload("mq_small", 3, 16, 2, "f16", [300, 133, 700], seed=51, max_tokens=700, block_perm=True)
    run_mq_case(w, 4)


def test_one_full_row_block_bf16():
    """16 queries x 8 heads = exactly one 128-row block; t4 values, random outliers."""
    w = I.Workload("mq_rb1", 2, 16, 2, "bf16", [2000, 1153], seed=52, max_tokens=2000, v_dist="t4",
                   k_outliers="random", block_perm=True)
    run_mq_case(w, 16)


def test_two_row_blocks_partial():
    """20 queries x 8 heads = 160 rows: a full and a partial row block."""
    w = I.Workload("mq_rb2", 2, 16, 2, "f16", [900, 1300], seed=53, max_tokens=1300, block_perm=True)
    run_mq_case(w, 20)


def test_causal_inside_packed_tiles_group1():
    """130 queries with G = 1: query positions span closed tiles, so the
    causal mask cuts through packed tiles; two row blocks."""
    w = I.Workload("mq_g1", 2, 2, 2, "f16", [400, 260], seed=54, max_tokens=400, block_perm=True)
    run_mq_case(w, 130)


def test_whole_sequence_is_queries():
    """Every token of the sequence is a query (prefill from an empty cache)."""
    w = I.Workload("mq_all", 2, 4, 1, "bf16", [256, 200], seed=55, max_tokens=256, v_dist="t4")
    run_mq_case(w, 200)


def test_k2_keys_group4():
    w = I.Workload("mq_k2", 3, 8, 2, "f16", [700, 129, 1500], seed=56, max_tokens=1500, block_perm=True, k_bits=2)
    run_mq_case(w, 8)


def test_v4_values_group8():
    w = I.Workload("mq_v4", 2, 16, 2, "bf16", [900, 400], seed=59, max_tokens=900, block_perm=True, v_dist="t4",
                   v_bits=4)
    run_mq_case(w, 16)


def test_single_query_matches_decode_oracle():
    w = I.Workload("mq_q1", 2, 16, 2, "bf16", [1000, 513], seed=57, max_tokens=1000, block_perm=True)
    run_mq_case(w, 1)


@pytest.mark.slow
def test_qwen3_32b_16k_chunk_sampled():
    """32 x 16384 tokens quantised by the GPU, a 16-query chunk per sequence
    in the launch the benchmark times; two sequences carry oracle records."""
    w = I.qwen3_32b()
    run_mq_case(w, 16, seqs=[3, 29], full_gpu_prefill=True)


@pytest.mark.slow
def test_long_context_128k():
    """16 causal queries at the end of two ~128 K-token sequences (1023
    closed tiles and a 91-token open tail; 1024 closed tiles): 32 split-K
    chunks per (KV head, row block) plus the open tile, merged by the
    combine; all query rows against the oracle."""
    lens = [131072 - 37, 131072]
    w = I.Workload("mq_long_128k", 2, 64, 8, "f16", lens, seed=78, max_tokens=max(lens), block_perm=True)
    run_mq_case(w, 16)


def test_device_errors():
    dev = device()
    w = I.Workload("mq_err", 3, 16, 2, "f16", [300, 3, 700], seed=58, max_tokens=700)
    c = PagedCache(w, dev)
    c.prefill()
    q = I.multi_queries(w, 4, device=dev)
    out = torch.full((w.batch, 4, w.num_q_heads, D), float("nan"), dtype=torch.float32, device=dev)
    c.multiquery(q, 4, out)   # sequence 1 is shorter than the query chunk
    torch.cuda.synchronize()
    assert c.check_error() == K.KVARN_DEV_ERR_TOKEN_RANGE
    assert not out[1].any() and torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all()
    c.err.zero_()
    bad = c.table.clone()
    bad[2, 1] = c.num_blocks + 3
    lens = c.lens.clone()
    lens[1] = 4   # long enough now; only the block id of sequence 2 is wrong
    K.kvarn_multiquery_attention(c.cfg, q, 4, bad, c.max_blocks, lens, w.batch, c.pool, c.tail, w.scale, out,
                                 c.mq_ws, c.mq_ws.numel() * 4, c.err)
    torch.cuda.synchronize()
    assert c.check_error() == K.KVARN_DEV_ERR_BLOCK_RANGE
    assert torch.isfinite(out[2]).all()


@pytest.mark.parametrize("dtype,k_bits,v_bits", [("f16", 4, 2), ("bf16", 4, 2), ("f16", 2, 2), ("bf16", 4, 4)])
def test_multiquery_over_degenerate_tiles(dtype, k_bits, v_bits):
    """The last 8 tokens of each sequence as causal queries over records of
    the quantiser's degenerate tiles (the decode test's sequences); the 1e-3
    bound scaled by max(1, max |v|) of the sequence, as there."""
    dev = device()
    w, ctx = degenerate_context(dtype, k_bits, v_bits)
    Q = 8
    c = PagedCache(w, dev)
    recs = load_oracle_records(w, c, list(range(w.batch)), ctx)
    q = I.multi_queries(w, Q, device=dev).cpu()
    out = torch.full((w.batch, Q, w.num_q_heads, D), float("nan"), dtype=torch.float32, device=dev)
    c.multiquery(q.to(dev), Q, out)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    got = out.cpu().numpy().astype(np.float64)
    worst = 0.0
    for (b, h), o in oracle_mq(w, list(range(w.batch)), ctx, recs, q, Q).items():
        g = got[b, :, h * w.G:(h + 1) * w.G]
        assert np.isfinite(g).all(), (b, h)
        scale = max(1.0, float(ctx[b][1].float().abs().max()))
        worst = max(worst, np.abs(g - o).max() / scale)
    print(f"{w.name} K{k_bits}/V{v_bits} Q={Q}: max |gpu - oracle| / max(1, max|v|) = {worst:.3e}")
    assert worst <= TOL


@pytest.mark.parametrize("h_kv,g", [(32, 1), (16, 2)])
def test_many_kv_heads(h_kv, g):
    """32 KV heads without grouping and 16 in pairs: one row block per KV
    head holds the 8 query tokens' rows."""
    w = I.Workload(f"mq_kv{h_kv}_g{g}", 2, h_kv * g, h_kv, "f16", [900, 300], seed=70 + h_kv, max_tokens=900,
                   block_perm=True)
    run_mq_case(w, 8)
