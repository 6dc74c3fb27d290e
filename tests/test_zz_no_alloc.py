"""kvarn_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (an engine whose memory manager has already reserved
the free device memory for its paged cache, or a decode loop where cudaMalloc
would synchronise the device).  Its split-K partials live in the library's
fixed 16 MiB device array instead of a caller workspace.

This file is collected last on purpose: it runs after every other test and
also passes alone in a fresh process.  It checks two calls in a row against
kvarn_decode_attention on the same inputs (the same kernels on the same
inputs with the same split, so the outputs must be bit-identical), and that
a request too large for the fixed array is refused without a launch."""
import pytest
import torch

from bit_kv_cache_quantize_gb300 import inputs as I
from bit_kv_cache_quantize_gb300 import kvarn as K
from bit_kv_cache_quantize_gb300.cache import PagedCache

from gpu_helpers import device

pytestmark = pytest.mark.gpu
def test_noalloc_matches_workspace_decode_twice():
    dev = device()
    w = I.Workload("noalloc_mix", 6, 32, 4, "f16", [1, 200, 128, 1000, 4100, 0], seed=77, max_tokens=4200,
                   block_perm=True)
    c = PagedCache(w, dev)
    c.prefill()
    need = K.kvarn_decode_workspace_bytes(c.cfg, w.batch, c.max_blocks)
    assert 0 < need <= K.NOALLOC_SCRATCH_BYTES
    ref = torch.empty(w.batch, w.num_q_heads, 128, dtype=torch.float32, device=dev)
    got = torch.empty_like(ref)
    for step in range(2):                      # the scratch keeps the last call's contents
        q = I.queries(w, step=step, device=dev)
        c.decode(q, ref)
        got.fill_(float("nan"))
        K.kvarn_decode_attention_noalloc(c.cfg, q, c.table, c.max_blocks, c.lens, w.batch, c.pool, c.tail, w.scale,
                                         got, c.err)
        torch.cuda.synchronize()
        assert c.check_error() == 0
        assert torch.isfinite(got).all()
        assert torch.equal(got, ref)


def test_noalloc_rejects_requests_beyond_the_fixed_scratch():
    device()
    cfg = K.make_config(8, 64, 70000, "f16")
    batch, max_blocks = 256, 257               # ragged serving mix: needs ~155 MB of partials
    assert K.kvarn_decode_workspace_bytes(cfg, batch, max_blocks) > K.NOALLOC_SCRATCH_BYTES
    st = K.kvarn_decode_attention_noalloc(cfg, 16, 16, max_blocks, 16, batch, 16, 16, 0.1, 16, 16, check=False)
    assert st == K.KVARN_ERR_UNSUPPORTED
