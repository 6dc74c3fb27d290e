"""Python binding of ``libkvarn.so`` (the C ABI in ``include/kvarn.h``).

Argument marshalling only: every function has the C name, passes plain
pointers and sizes through ctypes and returns the ``kvarn_status``.  Tensors
(torch) are accepted wherever the C function takes a device pointer and are
passed by ``data_ptr()``; ``stream=None`` means torch's current CUDA stream.
The library must be built (``bit_kv_cache_quantize_gb300.build``); there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libkvarn.so")

KVARN_OK, KVARN_ERR_INVALID, KVARN_ERR_UNSUPPORTED, KVARN_ERR_CUDA = 0, 1, 2, 3
KVARN_DTYPE_F16, KVARN_DTYPE_BF16 = 0, 1
KVARN_DEV_ERR_BLOCK_RANGE, KVARN_DEV_ERR_TOKEN_RANGE, KVARN_DEV_ERR_TIMEOUT = 1, 2, 3
HEAD_REC = 13312          # kvarn_k4v2: 4-bit key record + 2-bit value record
K_REC = 8704
V_REC = 4608


def rec_bytes(bits: int) -> int:
    """Bytes of one (tile, head) record of one role: 512-byte header + codes."""
    return 512 + 128 * 128 * bits // 8


def head_rec(k_bits: int = 4, v_bits: int = 2) -> int:
    """Bytes of one head of a block: key record then value record."""
    return rec_bytes(k_bits) + rec_bytes(v_bits)

# every function declared in include/kvarn.h
EXPORTS = (
    "kvarn_block_bytes", "kvarn_tail_bytes", "kvarn_quantize_tiles", "kvarn_append_tokens",
    "kvarn_decode_workspace_bytes", "kvarn_decode_attention", "kvarn_dequantize",
    "kvarn_fp16_block_bytes", "kvarn_fp16_decode_attention", "kvarn_status_string",
    "kvarn_decode_attention_noalloc", "kvarn_multiquery_workspace_bytes", "kvarn_multiquery_attention",
    "kvarn_token_errors_scratch_bytes", "kvarn_token_errors", "kvarn_test_decode_wait_expiry",
)
NOALLOC_SCRATCH_BYTES = 16 << 20


class kvarn_config(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32),
                ("sinkhorn_iters", ctypes.c_int32), ("dtype", ctypes.c_int32)]


def make_config(num_kv_heads: int, num_q_heads: int, num_blocks: int, dtype: str = "f16",
                sinkhorn_iters: int = 8, head_dim: int = 128, tile_tokens: int = 128,
                k_bits: int = 4, v_bits: int = 2) -> kvarn_config:
    return kvarn_config(head_dim, tile_tokens, num_kv_heads, num_q_heads, num_blocks, k_bits, v_bits,
                        sinkhorn_iters, KVARN_DTYPE_BF16 if dtype == "bf16" else KVARN_DTYPE_F16)


class KvarnError(RuntimeError):
    def __init__(self, status: int, fn: str):
        super().__init__(f"{fn}: {kvarn_status_string(status)} (status {status})")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvarn.so is not built ({LIB_PATH}); run bit_kv_cache_quantize_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        C = ctypes.POINTER(kvarn_config)
        sig = {
            "kvarn_block_bytes": (sz, [C]),
            "kvarn_tail_bytes": (sz, [C, i32]),
            "kvarn_fp16_block_bytes": (sz, [C]),
            "kvarn_decode_workspace_bytes": (sz, [C, i32, i32]),
            "kvarn_quantize_tiles": (i32, [C, P, P, i64, i64, P, P, i32, P, P, P]),
            "kvarn_append_tokens": (i32, [C, P, P, P, P, i32, i32, P, P, P, P]),
            "kvarn_decode_attention": (i32, [C, P, P, i32, P, i32, P, P, f32, P, P, sz, P, P]),
            "kvarn_fp16_decode_attention": (i32, [C, P, P, i32, P, i32, P, f32, P, P, sz, P, P]),
            "kvarn_decode_attention_noalloc": (i32, [C, P, P, i32, P, i32, P, P, f32, P, P, P]),
            "kvarn_test_decode_wait_expiry": (i32, [C, P, P, i32, P, i32, P, P, f32, P, P, sz, P, i32, P]),
            "kvarn_dequantize": (i32, [C, P, P, i32, P, P, P]),
            "kvarn_multiquery_workspace_bytes": (sz, [C, i32, i32, i32]),
            "kvarn_token_errors_scratch_bytes": (sz, [C, i32, i32]),
            "kvarn_token_errors": (i32, [C, P, i64, i64, P, i32, i32, i32, i32, P, sz, P, P, P]),
            "kvarn_multiquery_attention": (i32, [C, P, i32, P, i32, P, i32, P, P, f32, P, P, sz, P, P]),
            "kvarn_status_string": (ctypes.c_char_p, [i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, fn: str, check: bool) -> int:
    if check and status != KVARN_OK:
        raise KvarnError(status, fn)
    return status


def kvarn_status_string(status: int) -> str:
    return lib().kvarn_status_string(int(status)).decode()


def kvarn_block_bytes(cfg: kvarn_config) -> int:
    return int(lib().kvarn_block_bytes(ctypes.byref(cfg)))


def kvarn_tail_bytes(cfg: kvarn_config, batch: int) -> int:
    return int(lib().kvarn_tail_bytes(ctypes.byref(cfg), batch))


def kvarn_fp16_block_bytes(cfg: kvarn_config) -> int:
    return int(lib().kvarn_fp16_block_bytes(ctypes.byref(cfg)))


def kvarn_decode_workspace_bytes(cfg: kvarn_config, batch: int, max_blocks: int) -> int:
    return int(lib().kvarn_decode_workspace_bytes(ctypes.byref(cfg), batch, max_blocks))


def kvarn_quantize_tiles(cfg, k, v, token_stride_elems, n_tokens, tile_first_token, tile_dst_block, n_tiles,
                         block_pool, dev_err, stream=None, check=True) -> int:
    st = lib().kvarn_quantize_tiles(ctypes.byref(cfg), _p(k), _p(v), int(token_stride_elems), int(n_tokens),
                                    _p(tile_first_token), _p(tile_dst_block), int(n_tiles), _p(block_pool),
                                    _p(dev_err), _s(stream))
    return _check(st, "kvarn_quantize_tiles", check)


def kvarn_append_tokens(cfg, k_new, v_new, pos, block_table, max_blocks, batch, tail_pool, block_pool, dev_err,
                        stream=None, check=True) -> int:
    st = lib().kvarn_append_tokens(ctypes.byref(cfg), _p(k_new), _p(v_new), _p(pos), _p(block_table),
                                   int(max_blocks), int(batch), _p(tail_pool), _p(block_pool), _p(dev_err),
                                   _s(stream))
    return _check(st, "kvarn_append_tokens", check)


def kvarn_decode_attention(cfg, q, block_table, max_blocks, seq_lens, batch, block_pool, tail_pool, softmax_scale,
                           out, workspace, workspace_bytes, dev_err, stream=None, check=True) -> int:
    st = lib().kvarn_decode_attention(ctypes.byref(cfg), _p(q), _p(block_table), int(max_blocks), _p(seq_lens),
                                      int(batch), _p(block_pool), _p(tail_pool), float(softmax_scale), _p(out),
                                      _p(workspace), int(workspace_bytes), _p(dev_err), _s(stream))
    return _check(st, "kvarn_decode_attention", check)


def kvarn_decode_attention_noalloc(cfg, q, block_table, max_blocks, seq_lens, batch, block_pool, tail_pool,
                                   softmax_scale, out, dev_err, stream=None, check=True) -> int:
    """Decode attention with the split-K partials in the library's fixed
    16 MiB device scratch instead of a caller workspace, for callers that
    cannot allocate device memory (see include/kvarn.h)."""
    st = lib().kvarn_decode_attention_noalloc(ctypes.byref(cfg), _p(q), _p(block_table), int(max_blocks),
                                              _p(seq_lens), int(batch), _p(block_pool), _p(tail_pool),
                                              float(softmax_scale), _p(out), _p(dev_err), _s(stream))
    return _check(st, "kvarn_decode_attention_noalloc", check)


def kvarn_test_decode_wait_expiry(cfg, q, block_table, max_blocks, seq_lens, batch, block_pool, tail_pool,
                                  softmax_scale, out, workspace, workspace_bytes, dev_err, wait_polls, stream=None,
                                  check=True) -> int:
    """Decode with one record copy left out and the copy waits limited to
    wait_polls polls: the error path of a bounded wait (see include/kvarn.h)."""
    st = lib().kvarn_test_decode_wait_expiry(ctypes.byref(cfg), _p(q), _p(block_table), int(max_blocks),
                                             _p(seq_lens), int(batch), _p(block_pool), _p(tail_pool),
                                             float(softmax_scale), _p(out), _p(workspace), int(workspace_bytes),
                                             _p(dev_err), int(wait_polls), _s(stream))
    return _check(st, "kvarn_test_decode_wait_expiry", check)


def kvarn_multiquery_workspace_bytes(cfg, batch: int, max_blocks: int, n_queries: int) -> int:
    return int(lib().kvarn_multiquery_workspace_bytes(ctypes.byref(cfg), batch, max_blocks, n_queries))


def kvarn_multiquery_attention(cfg, q, n_queries, block_table, max_blocks, seq_lens, batch, block_pool, tail_pool,
                               softmax_scale, out, workspace, workspace_bytes, dev_err, stream=None,
                               check=True) -> int:
    """Causal attention of the last n_queries tokens of every sequence over
    the packed cache + open tile (see include/kvarn.h)."""
    st = lib().kvarn_multiquery_attention(ctypes.byref(cfg), _p(q), int(n_queries), _p(block_table), int(max_blocks),
                                          _p(seq_lens), int(batch), _p(block_pool), _p(tail_pool),
                                          float(softmax_scale), _p(out), _p(workspace), int(workspace_bytes),
                                          _p(dev_err), _s(stream))
    return _check(st, "kvarn_multiquery_attention", check)


def kvarn_token_errors_scratch_bytes(cfg, n_tiles: int, is_v: int) -> int:
    return int(lib().kvarn_token_errors_scratch_bytes(ctypes.byref(cfg), n_tiles, is_v))


def kvarn_token_errors(cfg, x, token_stride_elems, n_tokens, tile_first_token, n_tiles, is_v, rotate, sinkhorn_iters,
                       scratch, scratch_bytes, out, dev_err, stream=None, check=True) -> int:
    """Per-token (squared error, squared norm) of quantise -> dequantise,
    with the rotation and the normalisation optional (see include/kvarn.h)."""
    st = lib().kvarn_token_errors(ctypes.byref(cfg), _p(x), int(token_stride_elems), int(n_tokens),
                                  _p(tile_first_token), int(n_tiles), int(is_v), int(rotate), int(sinkhorn_iters),
                                  _p(scratch), int(scratch_bytes), _p(out), _p(dev_err), _s(stream))
    return _check(st, "kvarn_token_errors", check)


def kvarn_fp16_decode_attention(cfg, q, block_table, max_blocks, seq_lens, batch, fp16_pool, softmax_scale, out,
                                workspace, workspace_bytes, dev_err, stream=None, check=True) -> int:
    st = lib().kvarn_fp16_decode_attention(ctypes.byref(cfg), _p(q), _p(block_table), int(max_blocks),
                                           _p(seq_lens), int(batch), _p(fp16_pool), float(softmax_scale), _p(out),
                                           _p(workspace), int(workspace_bytes), _p(dev_err), _s(stream))
    return _check(st, "kvarn_fp16_decode_attention", check)


def kvarn_dequantize(cfg, block_pool, blocks, n, out, dev_err, stream=None, check=True) -> int:
    st = lib().kvarn_dequantize(ctypes.byref(cfg), _p(block_pool), _p(blocks), int(n), _p(out), _p(dev_err),
                                _s(stream))
    return _check(st, "kvarn_dequantize", check)
