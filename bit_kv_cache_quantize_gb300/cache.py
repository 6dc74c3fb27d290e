"""Device-side paged KVarN cache for a workload: torch owns the memory, every
computation goes through the C ABI (``kvarn``).

A ``PagedCache`` holds the packed block pool, the per-sequence block table,
the raw open-tile buffer, the decode workspace and the device error word, and
optionally the 16-bit paged pool of the comparison kernel.  With
``heads=(h0, h1)`` it holds only KV heads h0 .. h1-1 of the workload and
their query heads (one rank's shard, see ``shard``): every buffer, the
configuration and the generated inputs are those of that head range.
"""
from __future__ import annotations

import torch

from . import inputs as I
from . import kvarn as K

T = D = 128


class PagedCache:
    def __init__(self, w: I.Workload, device="cuda", fp16_pool: bool = False, extra_blocks: int = 0,
                 heads=None):
        self.w = w
        self.device = device
        self.h0, self.h1 = (0, w.num_kv_heads) if heads is None else heads
        self.H = self.h1 - self.h0                   # KV heads held here
        self.Hq = self.H * w.G                       # their query heads
        table, total = I.block_tables(w)
        self.table = table.to(device)
        self.max_blocks = table.shape[1]
        self.num_blocks = total + extra_blocks
        self.cfg = K.make_config(self.H, self.Hq, self.num_blocks, w.dtype, k_bits=w.k_bits, v_bits=w.v_bits)
        self.block_bytes = K.kvarn_block_bytes(self.cfg)
        self.pool = torch.zeros(self.num_blocks * self.block_bytes, dtype=torch.uint8, device=device)
        self.tail = torch.zeros(w.batch, self.H, 2, T, D, dtype=I.torch_dtype(w.dtype), device=device)
        self.ws_bytes = K.kvarn_decode_workspace_bytes(self.cfg, w.batch, self.max_blocks)
        self.ws = torch.empty(self.ws_bytes // 4 + 4, dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.lens = torch.tensor(w.seq_lens, dtype=torch.int32, device=device)
        self.pool16 = None
        if fp16_pool:
            self.pool16 = torch.zeros(self.num_blocks, self.H, 2, T, D, dtype=I.torch_dtype(w.dtype), device=device)

    # ------------------------------------------------------------ write path
    def quantize_sequence(self, b: int, k: torch.Tensor, v: torch.Tensor, stream=None):
        """k, v: [n_tok, H, D] of sequence b (device; the heads held here).
        Quantises the whole tiles into the sequence's blocks and copies the
        remainder into the open tile."""
        n = k.shape[0]
        n_full = n // T
        if n_full:
            first = torch.arange(n_full, dtype=torch.int64, device=self.device) * T
            dst = self.table[b, :n_full].contiguous()
            K.kvarn_quantize_tiles(self.cfg, k, v, self.H * D, n, first, dst, n_full, self.pool, self.err, stream)
        r = n - n_full * T
        if r:
            self.tail[b, :, 0, :r] = k[n_full * T:].permute(1, 0, 2)
            self.tail[b, :, 1, :r] = v[n_full * T:].permute(1, 0, 2)
        if self.pool16 is not None:
            nb = (n + T - 1) // T
            for i in range(nb):
                blk = int(self.table[b, i])
                m = min(T, n - i * T)
                self.pool16[blk, :, 0, :m] = k[i * T:i * T + m].permute(1, 0, 2)
                self.pool16[blk, :, 1, :m] = v[i * T:i * T + m].permute(1, 0, 2)

    def prefill(self, seqs=None, stream=None):
        """Generate each sequence's context on the device and write it."""
        heads = range(self.h0, self.h1)
        for b in (range(self.w.batch) if seqs is None else seqs):
            n = self.w.seq_lens[b]
            k = I.kv_sequence(self.w, "k", b, n, self.device, heads)
            v = I.kv_sequence(self.w, "v", b, n, self.device, heads)
            self.quantize_sequence(b, k, v, stream)

    def append(self, k_new, v_new, pos, stream=None):
        K.kvarn_append_tokens(self.cfg, k_new, v_new, pos, self.table, self.max_blocks, self.w.batch, self.tail,
                              self.pool, self.err, stream)

    # ------------------------------------------------------------ read path
    def decode(self, q, out, lens=None, stream=None):
        K.kvarn_decode_attention(self.cfg, q, self.table, self.max_blocks, self.lens if lens is None else lens,
                                 self.w.batch, self.pool, self.tail, self.w.scale, out, self.ws, self.ws_bytes,
                                 self.err, stream)

    def multiquery(self, q, n_queries, out, lens=None, stream=None):
        """q [B][n_queries][Hq][D]: the last n_queries tokens of each sequence
        attend causally to the cache (workspace grown on first use)."""
        need = K.kvarn_multiquery_workspace_bytes(self.cfg, self.w.batch, self.max_blocks, n_queries)
        if getattr(self, "mq_ws", None) is None or self.mq_ws.numel() * 4 < need:
            self.mq_ws = torch.empty(need // 4 + 4, dtype=torch.float32, device=self.device)
        K.kvarn_multiquery_attention(self.cfg, q, n_queries, self.table, self.max_blocks,
                                     self.lens if lens is None else lens, self.w.batch, self.pool, self.tail,
                                     self.w.scale, out, self.mq_ws, self.mq_ws.numel() * 4, self.err, stream)

    def decode_fp16(self, q, out, lens=None, stream=None):
        K.kvarn_fp16_decode_attention(self.cfg, q, self.table, self.max_blocks, self.lens if lens is None else lens,
                                      self.w.batch, self.pool16, self.w.scale, out, self.ws, self.ws_bytes,
                                      self.err, stream)

    # ------------------------------------------------------------ access
    def record(self, blk: int, head: int, kv: int) -> torch.Tensor:
        kb, vb = self.cfg.k_bits, self.cfg.v_bits
        off = blk * self.block_bytes + head * K.head_rec(kb, vb) + kv * K.rec_bytes(kb)
        return self.pool[off:off + K.rec_bytes(vb if kv else kb)]

    def set_record(self, blk: int, head: int, kv: int, rec: torch.Tensor):
        self.record(blk, head, kv).copy_(rec)

    def check_error(self) -> int:
        return int(self.err.item())
