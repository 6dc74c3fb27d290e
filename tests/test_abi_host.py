"""C-ABI checks that need no GPU: the library loads, exports every function
include/kvarn.h declares, sizes its buffers as documented, and rejects bad
arguments on the host without launching anything."""
import ctypes
import os
import re

import pytest

from bit_kv_cache_quantize_gb300 import build as B
from bit_kv_cache_quantize_gb300 import kvarn as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvarn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvarn_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(K.EXPORTS)


def test_sizes(lib):
    cfg = K.make_config(8, 64, 100, "f16")
    assert K.kvarn_block_bytes(cfg) == 8 * 13312
    assert K.kvarn_tail_bytes(cfg, 3) == 3 * 8 * 2 * 128 * 128 * 2
    assert K.kvarn_fp16_block_bytes(cfg) == 8 * 65536
    cfg2 = K.make_config(8, 64, 100, "f16", k_bits=2)
    assert K.kvarn_block_bytes(cfg2) == 8 * 9216  # 2-bit keys: two 4608-byte records per head
    assert K.head_rec(2) == 9216 and K.head_rec(4) == 13312 and K.head_rec(4, 4) == 17408
    cfg44 = K.make_config(8, 64, 100, "f16", k_bits=4, v_bits=4)
    assert K.kvarn_block_bytes(cfg44) == 8 * 17408  # K4/V4: two 8704-byte records per head
    assert K.kvarn_block_bytes(K.make_config(8, 64, 100, "f16", k_bits=2, v_bits=4)) == 0  # not a preset
    ws = K.kvarn_decode_workspace_bytes(cfg, 32, 128)
    assert ws == 32 * 8 * (8 + 1) * 8 * 132 * 4  # the 16-bit kernel's chunks of 16 tiles + open tile bound it


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 64, K.KVARN_ERR_UNSUPPORTED), ("tile_tokens", 64, K.KVARN_ERR_UNSUPPORTED),
    ("k_bits", 3, K.KVARN_ERR_UNSUPPORTED), ("k_bits", 8, K.KVARN_ERR_UNSUPPORTED),
    ("v_bits", 3, K.KVARN_ERR_UNSUPPORTED), ("v_bits", 8, K.KVARN_ERR_UNSUPPORTED),
    ("num_q_heads", 12, K.KVARN_ERR_INVALID), ("num_q_heads", 128, K.KVARN_ERR_UNSUPPORTED),
    ("num_kv_heads", 0, K.KVARN_ERR_INVALID), ("dtype", 7, K.KVARN_ERR_INVALID),
    ("sinkhorn_iters", -1, K.KVARN_ERR_INVALID), ("sinkhorn_iters", 65, K.KVARN_ERR_INVALID),
])
def test_config_validation(lib, field, value, status):
    cfg = K.make_config(8, 64, 10)
    setattr(cfg, field, value)
    assert K.kvarn_block_bytes(cfg) == 0
    st = K.kvarn_quantize_tiles(cfg, 16, 16, 1024, 128, 16, 16, 1, 16, 16, stream=0, check=False)
    assert st == status


def test_argument_validation_is_host_side(lib):
    cfg = K.make_config(8, 64, 10)
    # no tiles: nothing to do, even with null pointers
    assert K.kvarn_quantize_tiles(cfg, None, None, 1024, 0, None, None, 0, None, None, stream=0, check=False) == 0
    bad = [
        dict(k=None), dict(k=17), dict(token_stride_elems=1020), dict(token_stride_elems=512), dict(block_pool=None),
    ]
    for b in bad:
        args = dict(k=16, v=16, token_stride_elems=1024, n_tokens=128, tile_first_token=16, tile_dst_block=16,
                    n_tiles=1, block_pool=16, dev_err=16)
        args.update(b)
        st = K.kvarn_quantize_tiles(cfg, args["k"], args["v"], args["token_stride_elems"], args["n_tokens"],
                                    args["tile_first_token"], args["tile_dst_block"], args["n_tiles"],
                                    args["block_pool"], args["dev_err"], stream=0, check=False)
        assert st == K.KVARN_ERR_INVALID, b
    ws = K.kvarn_decode_workspace_bytes(cfg, 2, 4)
    assert K.kvarn_decode_attention(cfg, 16, 16, 4, 16, 2, 16, 16, 0.1, 16, 16, ws - 4, 16, stream=0,
                                    check=False) == K.KVARN_ERR_INVALID
    assert K.kvarn_decode_attention(cfg, 16, 16, 0, 16, 2, 16, 16, 0.1, 16, 16, ws, 16, stream=0,
                                    check=False) == K.KVARN_ERR_INVALID
    assert K.kvarn_append_tokens(cfg, 16, 16, 16, 16, 4, 0, 16, 16, 16, stream=0, check=False) == 0
    assert K.kvarn_append_tokens(cfg, 8, 16, 16, 16, 4, 1, 16, 16, 16, stream=0, check=False) == K.KVARN_ERR_INVALID
    # the append walks batch x heads x (K, V) units with a 32-bit count
    big = 0x7fffffff // (2 * 8) + 1
    assert K.kvarn_append_tokens(cfg, 16, 16, 16, 16, 4, big, 16, 16, 16, stream=0,
                                 check=False) == K.KVARN_ERR_INVALID
    assert K.kvarn_dequantize(cfg, 16, 16, -1, 16, 16, stream=0, check=False) == K.KVARN_ERR_INVALID
    assert K.kvarn_status_string(K.KVARN_ERR_UNSUPPORTED) == "unsupported configuration"
    with pytest.raises(K.KvarnError):
        K.kvarn_dequantize(cfg, 16, 16, -1, 16, 16, stream=0)


def test_null_pool_is_invalid_when_the_pool_has_blocks(lib):
    """With num_blocks > 0 a NULL pool is an invalid argument, found on the
    host (every other argument of these calls is valid, so the pool is what
    stops them; nothing launches).  A pool of 0 blocks may be NULL: the
    kernels never touch it, since every block id is then out of range."""
    cfg = K.make_config(8, 64, 10)
    ws = K.kvarn_decode_workspace_bytes(cfg, 2, 4)
    assert K.kvarn_decode_attention(cfg, 16, 16, 4, 16, 2, None, 16, 0.1, 16, 16, ws, 16, stream=0,
                                    check=False) == K.KVARN_ERR_INVALID
    assert K.kvarn_quantize_tiles(cfg, 16, 16, 1024, 128, 16, 16, 1, None, 16, stream=0,
                                  check=False) == K.KVARN_ERR_INVALID
    assert K.kvarn_dequantize(cfg, None, 16, 1, 16, 16, stream=0, check=False) == K.KVARN_ERR_INVALID


def test_multiquery_sizes_and_validation(lib):
    cfg = K.make_config(8, 64, 100, "f16")
    # 16 queries x 8 heads = one row block; 2 sequences, 40 blocks -> 16-tile chunks (3 + the open tile)
    assert K.kvarn_multiquery_workspace_bytes(cfg, 2, 40, 16) == 2 * 8 * 1 * (3 + 1) * 128 * 132 * 4
    assert K.kvarn_multiquery_workspace_bytes(cfg, 2, 40, 17) == 2 * 8 * 2 * (3 + 1) * 128 * 132 * 4
    assert K.kvarn_multiquery_workspace_bytes(cfg, 2, 40, 0) == 0
    assert K.kvarn_multiquery_workspace_bytes(cfg, 2, 40, 4097) == 0
    ws = K.kvarn_multiquery_workspace_bytes(cfg, 2, 4, 3)
    mq = lambda **kw: K.kvarn_multiquery_attention(
        cfg, kw.get("q", 16), kw.get("nq", 3), 16, kw.get("mb", 4), 16, kw.get("batch", 2), 16, kw.get("tail", 16),
        0.1, 16, 16, kw.get("ws", ws), 16, stream=0, check=False)
    assert mq(batch=0, q=None) == 0                      # nothing to do
    assert mq(nq=0) == K.KVARN_ERR_INVALID
    assert mq(ws=ws - 4) == K.KVARN_ERR_INVALID
    assert mq(q=17) == K.KVARN_ERR_INVALID                # misaligned
    assert mq(tail=None) == K.KVARN_ERR_INVALID
    assert mq(mb=0) == K.KVARN_ERR_INVALID
    bad = K.make_config(8, 64, 100, "f16", k_bits=3)
    assert K.kvarn_multiquery_attention(bad, 16, 3, 16, 4, 16, 2, 16, 16, 0.1, 16, 16, ws, 16, stream=0,
                                        check=False) == K.KVARN_ERR_UNSUPPORTED
