"""Stray-write checks for every entry point (a stand-in for a memory
sanitizer, which this GPU pool does not offer): each device buffer a call
may write is surrounded by guard bytes of a known pattern, each buffer it
must only read is fingerprinted, and parts of a buffer that a call has no
business writing (pool blocks it was not given, workspace past the split it
uses) are pre-filled with the pattern.  After the call every guard, every
read-only buffer and every untouched region must be bit-for-bit unchanged.
Shapes are ragged (tails, an empty sequence, permuted blocks) so that edge
tiles and partial chunks run."""
import pytest
import torch

from bit_kv_cache_quantize_gb300 import inputs as I
from bit_kv_cache_quantize_gb300 import kvarn as K
from bit_kv_cache_quantize_gb300.cache import PagedCache

from gpu_helpers import device

pytestmark = pytest.mark.gpu
T = D = 128
GUARD = 4096          # bytes on each side (a multiple of 16 keeps the interior aligned)
PATTERN = 0xA5


class Guarded:
    """A device buffer of `nbytes` with GUARD pattern bytes on both sides;
    `.view(dtype)` is the interior the kernel gets."""

    def __init__(self, nbytes, dev, fill=None):
        self.n = nbytes
        self.raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=dev)
        if fill is not None:
            self.raw[GUARD:GUARD + nbytes] = fill

    def view(self, dtype=torch.uint8):
        return self.raw[GUARD:GUARD + self.n].view(dtype)

    def check(self, what):
        lo, hi = self.raw[:GUARD], self.raw[GUARD + self.n:]
        assert bool((lo == PATTERN).all()), f"{what}: bytes written below the buffer"
        assert bool((hi == PATTERN).all()), f"{what}: bytes written past the end of the buffer"


def fingerprint(t):
    return t.detach().clone()


def ragged():
    return I.Workload("canary", 5, 16, 2, "f16", [300, 1, 0, 129, 640], seed=61, max_tokens=700, block_perm=True,
                      decode_steps=3)


def test_quantize_and_append_write_only_their_blocks():
    dev = device()
    w = ragged()
    c = PagedCache(w, dev)
    pool = Guarded(c.num_blocks * c.block_bytes, dev)      # every byte of the pool starts as the pattern
    err = Guarded(4, dev, fill=0)
    k = I.kv_sequence(w, "k", 4, 640, dev)
    v = I.kv_sequence(w, "v", 4, 640, dev)
    k0, v0 = fingerprint(k), fingerprint(v)
    first = torch.arange(5, dtype=torch.int64, device=dev) * T
    dst = c.table[4, :5].contiguous()
    K.kvarn_quantize_tiles(c.cfg, k, v, w.num_kv_heads * D, 640, first, dst, 5, pool.view(), err.view(torch.int32))
    torch.cuda.synchronize()
    assert int(err.view(torch.int32)[0]) == 0
    pool.check("quantize pool"); err.check("quantize dev_err")
    assert torch.equal(k, k0) and torch.equal(v, v0), "quantize wrote its inputs"
    blocks = pool.view().view(c.num_blocks, c.block_bytes)
    written = set(int(b) for b in dst.cpu())
    for b in range(c.num_blocks):                          # the five destination blocks, nothing else
        untouched = bool((blocks[b] == PATTERN).all())
        assert untouched == (b not in written), f"block {b}"
    # append one token per sequence; the token of sequence 3 lands in slot 127 of its tile 1 and closes it, so
    # the tails and that one block are all that may change
    tail = Guarded(K.kvarn_tail_bytes(c.cfg, w.batch), dev, fill=0)
    pos = torch.tensor([300, 1, 0, 255, 640], dtype=torch.int32, device=dev)
    kn = torch.stack([I.kv_values(w, "k", b, int(pos[b]), 1, dev)[0] for b in range(w.batch)])
    vn = torch.stack([I.kv_values(w, "v", b, int(pos[b]), 1, dev)[0] for b in range(w.batch)])
    before = fingerprint(pool.view())
    K.kvarn_append_tokens(c.cfg, kn, vn, pos, c.table, c.max_blocks, w.batch, tail.view(), pool.view(),
                          err.view(torch.int32))
    torch.cuda.synchronize()
    assert int(err.view(torch.int32)[0]) == 0
    tail.check("append tail"); pool.check("append pool"); err.check("append dev_err")
    changed = (pool.view() != before).view(c.num_blocks, c.block_bytes).any(dim=1).nonzero().flatten().tolist()
    assert changed == [int(c.table[3, 1])], f"append changed blocks {changed}"
    tv = tail.view(torch.float16).view(w.batch, w.num_kv_heads, 2, T, D)
    for b in range(w.batch):                               # exactly one slot per sequence holds data
        slot = int(pos[b]) % T
        nz = tv[b].abs().sum(dim=(0, 1, 3)).nonzero().flatten().tolist()
        assert nz in ([slot], []), f"sequence {b}: tail slots {nz}"


@pytest.mark.parametrize("k_bits,v_bits", [(4, 2), (2, 2), (4, 4)])
def test_decode_writes_only_its_output_and_workspace(k_bits, v_bits):
    dev = device()
    w = ragged()
    w.k_bits, w.v_bits = k_bits, v_bits
    c = PagedCache(w, dev)
    c.prefill()
    torch.cuda.synchronize()
    q = I.queries(w, device=dev)
    ins = {n: fingerprint(t) for n, t in (("q", q), ("pool", c.pool), ("tail", c.tail), ("table", c.table),
                                          ("lens", c.lens))}
    out = Guarded(w.batch * w.num_q_heads * D * 4, dev)
    ws = Guarded(c.ws_bytes, dev)
    err = Guarded(4, dev, fill=0)
    K.kvarn_decode_attention(c.cfg, q, c.table, c.max_blocks, c.lens, w.batch, c.pool, c.tail, w.scale,
                             out.view(torch.float32), ws.view(torch.float32), c.ws_bytes, err.view(torch.int32))
    torch.cuda.synchronize()
    assert int(err.view(torch.int32)[0]) == 0
    out.check("decode out"); ws.check("decode workspace"); err.check("decode dev_err")
    assert not bool((out.view() == PATTERN).all()), "decode wrote no output"
    for n, t in (("q", q), ("pool", c.pool), ("tail", c.tail), ("table", c.table), ("lens", c.lens)):
        assert torch.equal(t, ins[n]), f"decode wrote its input {n}"
    # the no-alloc entry point: output only (its scratch is the library's own)
    out2 = Guarded(w.batch * w.num_q_heads * D * 4, dev)
    K.kvarn_decode_attention_noalloc(c.cfg, q, c.table, c.max_blocks, c.lens, w.batch, c.pool, c.tail, w.scale,
                                     out2.view(torch.float32), err.view(torch.int32))
    torch.cuda.synchronize()
    out2.check("no-alloc decode out")
    assert torch.equal(out2.view(), out.view())


def test_multiquery_writes_only_its_output_and_workspace():
    dev = device()
    w = I.Workload("canary_mq", 3, 16, 2, "f16", [300, 129, 640], seed=63, max_tokens=700, block_perm=True)
    c = PagedCache(w, dev)
    c.prefill()
    Q = 5
    q = I.multi_queries(w, Q, device=dev)
    q0, pool0 = fingerprint(q), fingerprint(c.pool)
    need = K.kvarn_multiquery_workspace_bytes(c.cfg, w.batch, c.max_blocks, Q)
    out = Guarded(w.batch * Q * w.num_q_heads * D * 4, dev)
    ws = Guarded(need, dev)
    err = Guarded(4, dev, fill=0)
    K.kvarn_multiquery_attention(c.cfg, q, Q, c.table, c.max_blocks, c.lens, w.batch, c.pool, c.tail, w.scale,
                                 out.view(torch.float32), ws.view(torch.float32), need, err.view(torch.int32))
    torch.cuda.synchronize()
    assert int(err.view(torch.int32)[0]) == 0
    out.check("multi-query out"); ws.check("multi-query workspace"); err.check("multi-query dev_err")
    assert torch.equal(q, q0) and torch.equal(c.pool, pool0)


def test_fp16_decode_dequantize_and_token_errors_stay_in_bounds():
    dev = device()
    w = ragged()
    c = PagedCache(w, dev, fp16_pool=True)
    c.prefill()
    q = I.queries(w, device=dev)
    err = Guarded(4, dev, fill=0)
    out = Guarded(w.batch * w.num_q_heads * D * 4, dev)
    ws = Guarded(c.ws_bytes, dev)
    p16 = fingerprint(c.pool16)
    K.kvarn_fp16_decode_attention(c.cfg, q, c.table, c.max_blocks, c.lens, w.batch, c.pool16, w.scale,
                                  out.view(torch.float32), ws.view(torch.float32), c.ws_bytes, err.view(torch.int32))
    torch.cuda.synchronize()
    assert int(err.view(torch.int32)[0]) == 0
    out.check("fp16 decode out"); ws.check("fp16 decode workspace")
    assert torch.equal(c.pool16, p16)
    blocks = torch.tensor([int(c.table[4, 2]), int(c.table[0, 0])], dtype=torch.int32, device=dev)
    deq = Guarded(2 * 2 * w.num_kv_heads * T * D * 4, dev)
    K.kvarn_dequantize(c.cfg, c.pool, blocks, 2, deq.view(torch.float32), err.view(torch.int32))
    torch.cuda.synchronize()
    deq.check("dequantize out")
    x = I.kv_sequence(w, "k", 4, 640, dev)
    first = torch.tensor([0, 256], dtype=torch.int64, device=dev)
    need = K.kvarn_token_errors_scratch_bytes(c.cfg, 2, 0)
    scratch = Guarded(need, dev)
    eo = Guarded(2 * w.num_kv_heads * T * 2 * 4, dev)
    for rot, it in ((1, 8), (0, 0)):
        K.kvarn_token_errors(c.cfg, x, w.num_kv_heads * D, 640, first, 2, 0, rot, it, scratch.view(), need,
                             eo.view(torch.float32), err.view(torch.int32))
        torch.cuda.synchronize()
        scratch.check("token errors scratch"); eo.check("token errors out")
    assert int(err.view(torch.int32)[0]) == 0
    err.check("dev_err")
