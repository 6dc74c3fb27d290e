"""Host logic of the per-token error tool: the distribution statistics and
the C-ABI argument checks of kvarn_token_errors (no GPU)."""
import numpy as np
import pytest

from bit_kv_cache_quantize_gb300 import errors as E
from bit_kv_cache_quantize_gb300 import kvarn as K


def test_error_stats_on_known_values():
    rel = np.arange(1, 101, dtype=np.float64) / 100.0      # 0.01 .. 1.00
    norm2 = np.full(100, 4.0)
    st = E.error_stats(rel ** 2 * norm2, norm2)
    assert st["tokens"] == 100
    assert st["mean"] == pytest.approx(rel.mean())
    assert st["p50"] == pytest.approx(np.percentile(rel, 50))
    assert st["p95"] == pytest.approx(np.percentile(rel, 95))
    assert st["max"] == pytest.approx(1.0)
    assert st["top_mean"] == pytest.approx(np.mean([0.96, 0.97, 0.98, 0.99, 1.0]))
    sq = rel ** 2
    assert st["top_share_sq_err"] == pytest.approx(sq[-5:].sum() / sq.sum())


def test_error_stats_skips_zero_tokens_and_zero_error():
    st = E.error_stats(np.zeros(10), np.r_[np.zeros(3), np.ones(7)])
    assert st["tokens"] == 7 and st["mean"] == 0.0 and st["top_share_sq_err"] == 0.0


@pytest.fixture(scope="module")
def lib():
    from bit_kv_cache_quantize_gb300 import build as B
    B.build()
    return K.lib()


def test_token_errors_validation(lib):
    cfg = K.make_config(8, 64, 1, "f16")
    assert K.kvarn_token_errors_scratch_bytes(cfg, 3, 0) == 3 * 8 * 8704
    assert K.kvarn_token_errors_scratch_bytes(cfg, 3, 1) == 3 * 8 * 4608
    sb = K.kvarn_token_errors_scratch_bytes(cfg, 2, 0)
    call = lambda **kw: K.kvarn_token_errors(
        cfg, kw.get("x", 16), kw.get("stride", 1024), 256, 16, kw.get("n", 2), kw.get("is_v", 0), kw.get("rot", 1),
        kw.get("iters", 8), 16, kw.get("sb", sb), 16, 16, stream=0, check=False)
    assert call(n=0, x=None) == 0
    assert call(rot=2) == K.KVARN_ERR_INVALID
    assert call(is_v=3) == K.KVARN_ERR_INVALID
    assert call(iters=65) == K.KVARN_ERR_INVALID
    assert call(sb=sb - 1) == K.KVARN_ERR_INVALID
    assert call(stride=1000) == K.KVARN_ERR_INVALID
    assert call(x=18) == K.KVARN_ERR_INVALID
