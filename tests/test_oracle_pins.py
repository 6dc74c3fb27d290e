"""Pins of the CPU oracle against what the pages and mathematics fix.

None of these compares the oracle with itself: each checks it against a
library routine (scipy's Sylvester Hadamard matrix, numpy's IEEE float16,
torch's float8_e4m3fn and float64 attention), a closed form, an invariant,
or brute force on tiny inputs.  The pages (KVarN write-ups) print no worked
example, so there is no page-printed value to pin except the preset's
numbers (tests/golden/pages_preset.json).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle as O
from bit_kv_cache_quantize_gb300 import inputs as I

D = T = 128
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def fwht_rows(X):
    """Independent fast Walsh-Hadamard butterfly, normalised."""
    Y = np.array(X, dtype=np.float64, copy=True)
    h = 1
    while h < D:
        for i in range(0, D, 2 * h):
            a = Y[:, i:i + h].copy()
            b = Y[:, i + h:i + 2 * h].copy()
            Y[:, i:i + h] = a + b
            Y[:, i + h:i + 2 * h] = a - b
        h *= 2
    return Y / math.sqrt(D)


def key_tile(seed=0):
    w = I.single_tile()
    w.seed = seed
    k = I.kv_values(w, "k", 0, 0, T)[:, 0, :]
    return O.decode16(k.view(torch.int16).numpy().view(np.uint16), "f16")


# ----------------------------------------------------------------- rotation
def test_hadamard_is_sylvester_orthonormal():
    H = O.hadamard_matrix()
    assert np.array_equal(H, scipy.linalg.hadamard(D) / math.sqrt(D))
    assert np.abs(H @ H.T - np.eye(D)).max() < 1e-15
    assert np.array_equal(H, H.T)


def test_rotation_equals_butterfly_and_preserves_norm():
    rng = np.random.default_rng(1)
    X = rng.standard_normal((7, D))
    R = O.rotate(X)
    assert np.abs(R - fwht_rows(X)).max() < 1e-12
    assert np.allclose(np.linalg.norm(R, axis=1), np.linalg.norm(X, axis=1), rtol=1e-14)
    e0 = np.zeros((1, D)); e0[0, 0] = 1.0
    assert np.abs(O.rotate(e0) - 1 / math.sqrt(D)).max() < 1e-16
    assert np.abs(O.rotate(R) - X).max() < 1e-12          # H is its own inverse


# ----------------------------------------------------------------- sinkhorn
@pytest.mark.parametrize("iters", [1, 2, 8])
def test_sinkhorn_closed_form(iters):
    """R = diag(alpha) M diag(beta), M_tc = (-1)^(t+c), alpha_2k = alpha_2k+1:
    the first column step gives v = ln beta + ln rms(alpha), the first row
    step u = ln alpha - ln rms(alpha); every later step is a no-op.  A row
    step taken first would give other values (beta is not alternating)."""
    rng = np.random.default_rng(2)
    alpha = np.repeat(np.exp(rng.normal(0, 0.7, T // 2)), 2)
    beta = np.exp(rng.normal(0, 0.7, D))
    M = (-1.0) ** (np.arange(T)[:, None] + np.arange(D)[None, :])
    R = alpha[:, None] * M * beta[None, :]
    u, v = O.sinkhorn(R, iters)
    rms_a = math.sqrt(np.mean(alpha ** 2))
    assert np.abs(v - (np.log(beta) + math.log(rms_a))).max() < 1e-12
    assert np.abs(u - (np.log(alpha) - math.log(rms_a))).max() < 1e-12


def test_sinkhorn_normalises_rows_and_converges_columns():
    R = O.rotate(key_tile())
    dev = []
    for n in (1, 2, 4, 8):
        u, v = O.sinkhorn(R, n)
        Z = R * np.exp(-u)[:, None] * np.exp(-v)[None, :]
        assert np.abs(Z.std(axis=1) - 1).max() < 1e-12        # last step is a row step
        dev.append(np.abs(Z.std(axis=0) - 1).max())
    assert all(b < a for a, b in zip(dev, dev[1:]))
    assert dev[-1] < 0.02


def test_sinkhorn_degenerate_tiles_keep_factors():
    u, v = O.sinkhorn(np.zeros((T, D)), 8)
    assert not u.any() and not v.any()
    row = O.rotate(np.random.default_rng(3).standard_normal((1, D)))
    same = np.repeat(row, T, axis=0)                           # every token identical
    u, v = O.sinkhorn(same, 8)
    assert not v.any()                                         # column std is 0
    assert np.allclose(u, np.log(row.std()), atol=1e-12)


# ----------------------------------------------------------------- formats
def test_e4m3_decode_matches_torch_exhaustive():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([O.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours)) and nan.sum() == 2
    assert np.array_equal(ref[~nan], ours[~nan])
    assert O.e4m3_decode(0x7E) == 448.0 and O.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encoders():
    for c in list(range(0x7F)) + list(range(0x81, 0xFF)):
        assert O.e4m3_encode_rne(O.e4m3_decode(c)) == c
    table = np.array([O.e4m3_decode(c) for c in range(0x7F)])
    rng = np.random.default_rng(4)
    xs = np.concatenate([np.exp(rng.uniform(math.log(2 ** -11), math.log(448), 3000)),
                         (table[1:] + table[:-1]) / 2])              # exact midpoints too
    xs = xs.astype(np.float32).astype(np.float64)                    # torch converts from fp32 exactly
    ref = torch.from_numpy(xs.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert all(O.e4m3_encode_rne(x) == r for x, r in zip(xs, ref))
    assert O.e4m3_encode_rne(1e6) == 0x7E and O.e4m3_encode_rne(-1e6) == 0xFE
    for x in xs:                                                     # round up = brute force
        want = int(np.nonzero(table >= x)[0][0]) if x <= 448 else 0x7E
        assert O.e4m3_encode_ru(x) == want
    assert O.e4m3_encode_ru(0.0) == 0 and O.e4m3_encode_ru(1000.0) == 0x7E


def test_f16_decode_and_encoders():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    ours = np.array([O.f16_decode(b) for b in range(65536)])
    fin = np.isfinite(ref)
    assert np.array_equal(ref[fin], ours[fin]) and np.array_equal(np.isnan(ref), np.isnan(ours))
    for b in range(0, 65536, 7):
        if fin[b] and b != 0x8000:
            assert O.f16_encode_rd(ref[b]) == b and O.f16_encode_rne(ref[b]) == b
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.uniform(-8, 4.8, 2000),
                         (ref[1:0x7BFF][:-1] + ref[2:0x7BFF]) / 2])   # midpoints
    xs = xs[np.abs(xs) < 65504.0]                                    # saturation checked below
    for x in xs:
        h = np.float16(x)                                            # numpy: correctly rounded
        assert O.f16_encode_rne(x) == int(np.array(h).view(np.uint16))
        if float(h) > x:
            h = np.nextafter(h, np.float16(-np.inf))
        assert O.f16_encode_rd(x) == int(np.array(h).view(np.uint16))
    assert O.f16_encode_rd(1e9) == 0x7BFF and O.f16_encode_rd(-1e9) == 0xFBFF


# ----------------------------------------------------------------- quantiser
E4M3 = np.array([O.e4m3_decode(c) for c in range(0x7F)])          # the non-negative finite values, ascending
F16 = np.arange(0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)   # 0 .. 65504 ascending


def check_scales_tight(Y, tl, levels):
    """The per-token zero-point and step are the tightest the formats allow
    ("Huawei's KVarN puts KV-cache quantization inside vLLM's backend",
    "The four-stage pipeline": asymmetric round-to-nearest over each
    token's range): b is the LARGEST FP16 value <= min Y and a the SMALLEST
    E4M3 value with b + L a >= max Y, checked in exact rational arithmetic
    (a step one code too high or a zero-point one ulp too low fails)."""
    from fractions import Fraction as Fr
    for t in range(T):
        lo, hi = Fr(float(Y[t].min())), Fr(float(Y[t].max()))
        b = Fr(O.f16_decode(int(tl.b16[t])))
        assert b <= lo, t
        nb = -F16[F16 < -float(b)].max() if b < 0 else F16[F16 > float(b)].min()
        assert Fr(float(nb)) > lo, t                                  # the next FP16 up is above min Y
        a = Fr(O.e4m3_decode(int(tl.a8[t])))
        assert b + levels * a >= hi, t                                # covers max Y
        i = int(np.searchsorted(E4M3, float(a)))
        if i > 1:                                                      # 2^-9 is the floor
            assert b + levels * Fr(float(E4M3[i - 1])) < hi, t       # the E4M3 value below does not


@pytest.mark.parametrize("levels,seed", [(15, 0), (3, 1), (15, 7), (3, 9)])
def test_quantize_tile_properties(levels, seed):
    X = key_tile(seed)
    if levels == 3:
        X = X / 20.0 + np.sin(np.arange(D))[None, :]
    tl = O.quantize_tile(X, levels)
    assert tl.flags == 0
    g, a, b = tl.g(), tl.a(), tl.b()
    # gauge: centred log factors; g is the E4M3 value nearest to exp(v)
    assert abs(tl.v.sum()) < 1e-10
    assert (np.abs(g - np.exp(tl.v)) <= np.abs(E4M3[None, :] - np.exp(tl.v)[:, None]).min(axis=1)).all()
    Y = tl.R / g[None, :]
    assert np.abs(tl.R - O.rotate(X)).max() < 1e-12
    check_scales_tight(Y, tl, levels)
    # codes in range, equal to the brute-force nearest level except at ties
    assert tl.code.max() <= levels
    levels_grid = a[:, None, None] * np.arange(levels + 1)[None, None, :] + b[:, None, None]
    brute = np.abs(Y[:, :, None] - levels_grid).argmin(axis=2)
    frac = tl.pre - np.floor(tl.pre)
    near_tie = np.abs(frac - 0.5) < 1e-5
    assert np.array_equal(brute[~near_tie], tl.code[~near_tie])
    # round trip within half a step, per element and per token in the original domain
    recon = a[:, None] * tl.code + b[:, None]
    assert (np.abs(Y - recon) <= a[:, None] / 2 * (1 + 1e-6)).all()
    Xh = O.dequantize_record(levels == 3, O.pack_record(levels == 3, tl))
    bound = 0.5 * np.sqrt(((g[None, :] * a[:, None]) ** 2).sum(axis=1)) * (1 + 1e-6)
    assert (np.linalg.norm(Xh - X, axis=1) <= bound).all()


def test_scale_pins_reject_loose_scales():
    """The tightness pin fails on the plausible mistakes it is there for: a
    per-token step one E4M3 code too high, a zero-point one FP16 ulp too low."""
    X = key_tile(3)
    tl = O.quantize_tile(X, 15)
    Y = tl.R / tl.g()[None, :]
    check_scales_tight(Y, tl, 15)
    loose_a = O.Tile(tl.g8, tl.a8.copy(), tl.b16, tl.code, tl.pre, tl.R, tl.v, 0)
    loose_a.a8[17] += 1
    with pytest.raises(AssertionError):
        check_scales_tight(Y, loose_a, 15)
    low_b = O.Tile(tl.g8, tl.a8, tl.b16.copy(), tl.code, tl.pre, tl.R, tl.v, 0)
    b = low_b.b16[40]
    low_b.b16[40] = b + 1 if b & 0x8000 else b - 1                   # one ulp towards -inf
    with pytest.raises(AssertionError):
        check_scales_tight(Y, low_b, 15)


def test_quantize_degenerate_tiles():
    z = O.quantize_tile(np.zeros((T, D)), 15)
    assert (z.g8 == 0x38).all() and (z.a8 == 0x01).all() and (z.b16 == 0).all() and not z.code.any()
    same = np.repeat(key_tile()[:1], T, axis=0)
    s = O.quantize_tile(same, 3)
    assert (s.g8 == 0x38).all()                                      # no column information: g = 1
    assert (s.code == s.code[0]).all()
    big = np.zeros((T, D)); big[5, 9] = 3000.0                      # one huge outlier
    bt = O.quantize_tile(big, 15)
    assert bt.flags == 0
    Xh = O.dequantize_record(False, O.pack_record(False, bt))
    g, a = bt.g(), bt.a()
    bound = 0.5 * np.sqrt(((g[None, :] * a[:, None]) ** 2).sum(axis=1)) * (1 + 1e-6)
    assert (np.linalg.norm(Xh - big, axis=1) <= bound).all()
    # beyond the format: a per-token step above 448 (the largest E4M3 value)
    # saturates and the codes clamp; the oracle flags it
    big[5, 9] = 60000.0
    sat = O.quantize_tile(big, 15)
    assert sat.flags & O.FLAG_STEP_SAT and sat.flags & O.FLAG_CLAMPED
    assert sat.a8[5] == 0x7E and sat.code.max() <= 15


# ----------------------------------------------------------------- layout
def test_record_layout_bytes():
    tl = O.Tile(np.arange(D, dtype=np.uint8), (np.arange(T) * 3 % 256).astype(np.uint8),
                (np.arange(T) * 517).astype(np.uint16),
                ((np.arange(T)[:, None] + 3 * np.arange(D)[None, :]) % 16).astype(np.uint8),
                None, None, None, 0)
    rk = O.pack_record(False, tl)
    assert rk.size == 8704 and O.record_bytes(False) == 8704
    assert rk[5] == 5 and rk[128 + 7] == 21 and rk[256 + 2 * 9] == (9 * 517) & 0xFF
    assert rk[257 + 2 * 9] == (9 * 517) >> 8
    t, i = 11, 13                                                    # byte i of token t
    assert rk[512 + t * 64 + i] == tl.code[t, 2 * i] | (tl.code[t, 2 * i + 1] << 4)
    tl.code = tl.code % 4
    rv = O.pack_record(True, tl)
    assert rv.size == 4608
    c, w = 77, 5                                                     # word w of channel c
    word = int.from_bytes(bytes(rv[512 + c * 32 + 4 * w: 512 + c * 32 + 4 * w + 4]), "little")
    even = sum(int(tl.code[16 * w + u, c]) << u for u in range(0, 16, 2))        # low half
    odd = sum(int(tl.code[16 * w + u, c]) << (15 + u) for u in range(1, 16, 2))  # high half
    assert word == even | odd
    g8, a8, b16, code = O.unpack_record(True, rv)
    assert np.array_equal(code, tl.code) and np.array_equal(b16, tl.b16)


def test_k2_record_layout_bytes():
    """K2/V2 preset: 2-bit key codes token-major, 32 B per token, four
    codes per byte with channel 4i+k at bits 2k of byte i."""
    tl = O.Tile((np.arange(D) % 120).astype(np.uint8), (np.arange(T) * 5 % 120).astype(np.uint8),
                (np.arange(T) * 301 % 30000).astype(np.uint16),
                ((np.arange(T)[:, None] * 7 + np.arange(D)[None, :]) % 4).astype(np.uint8),
                None, None, None, 0)
    rk = O.pack_record(False, tl, k_bits=2)
    assert rk.size == 4608 and O.record_bytes(False, 2) == 4608 and O.levels(False, 2) == 3
    assert rk[7] == 7 and rk[128 + 3] == 15 and rk[256 + 2 * 5] == (5 * 301) & 0xFF  # header as for 4-bit keys
    t, i = 41, 19
    assert rk[512 + t * 32 + i] == sum(int(tl.code[t, 4 * i + k]) << (2 * k) for k in range(4))
    g8, a8, b16, code = O.unpack_record(False, rk, k_bits=2)
    assert np.array_equal(code, tl.code) and np.array_equal(g8, tl.g8) and np.array_equal(a8, tl.a8)
    # the same codes in the 4-bit key layout dequantise to the same values
    rk4 = O.pack_record(False, tl, k_bits=4)
    assert np.array_equal(O.dequantize_record(False, rk, 2), O.dequantize_record(False, rk4, 4))
    assert (O.record_bytes(False, 2) * 8 / (T * D), O.record_bytes(True) * 8 / (T * D)) == (2.25, 2.25)


def test_v4_record_layout_bytes():
    """K4/V4 preset: 4-bit value codes channel-major, 64 B per channel as 16
    little-endian words of 8 tokens, even tokens in the low half-word and odd
    tokens in the high half-word (token 8w + u at bit 2u or 14 + 2u)."""
    tl = O.Tile((np.arange(D) % 120).astype(np.uint8), (np.arange(T) * 5 % 120).astype(np.uint8),
                (np.arange(T) * 301 % 30000).astype(np.uint16),
                ((np.arange(T)[:, None] * 7 + np.arange(D)[None, :] * 3) % 16).astype(np.uint8),
                None, None, None, 0)
    rv = O.pack_record(True, tl, v_bits=4)
    assert rv.size == 8704 and O.record_bytes(True, 4, 4) == 8704 and O.levels(True, 4, 4) == 15
    assert rv[7] == 7 and rv[128 + 3] == 15
    c, w = 37, 11
    word = int.from_bytes(rv[512 + c * 64 + 4 * w: 512 + c * 64 + 4 * w + 4].tobytes(), "little")
    for u in range(8):
        bit = 14 + 2 * u if u & 1 else 2 * u
        assert (word >> bit) & 15 == tl.code[8 * w + u, c]
    g8, a8, b16, code = O.unpack_record(True, rv, v_bits=4)
    assert np.array_equal(code, tl.code) and np.array_equal(b16, tl.b16)
    assert O.record_bytes(True, 4, 4) * 8 / (T * D) == 4.25


def test_bits_per_element_against_pages():
    """The pages give ~2.3 bits/element including the dual FP8 scales and
    FP16 zero-points, for 4-bit keys / 2-bit values per 128-token tile."""
    with open(os.path.join(GOLDEN, "pages_preset.json")) as f:
        p = json.load(f)
    assert p["tile_tokens"] == T and p["k_bits"] == 4 and p["v_bits"] == 2
    k_bits = O.record_bytes(False) * 8 / (T * D)
    v_bits = O.record_bytes(True) * 8 / (T * D)
    assert (k_bits, v_bits) == (4.25, 2.25)
    assert abs(v_bits - p["effective_bits_per_element"]) < 0.1        # the V side matches ~2.3
    assert 3 <= 16 / ((k_bits + v_bits) / 2) <= 5                    # "3-5x" capacity


# ----------------------------------------------------------------- attention
def test_attention_closed_forms():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((3, D))
    k1, v1 = rng.standard_normal((1, D)), rng.standard_normal((1, D))
    assert np.abs(O.attention(q, k1, v1, 0.1) - v1).max() < 1e-15      # one token: o = v
    K = np.repeat(k1, 9, axis=0); V = rng.standard_normal((9, D))
    assert np.abs(O.attention(q, K, V, 0.1) - V.mean(0)).max() < 1e-14  # equal keys: mean
    assert not O.attention(q, np.zeros((0, D)), np.zeros((0, D)), 0.1).any()


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((4, D)); K = rng.standard_normal((37, D)) * 3; V = rng.standard_normal((37, D))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], scale=0.3)[0]
    assert np.abs(O.attention(q, K, V, 0.3) - ref.numpy()).max() < 1e-13


@pytest.mark.parametrize("k_bits,v_bits", [(4, 2), (2, 2), (4, 4)])
@pytest.mark.parametrize("n_tiles,n_tail", [(1, 0), (2, 37), (0, 5), (3, 127)])
def test_folded_attention_equals_plain(n_tiles, n_tail, k_bits, v_bits):
    rng = np.random.default_rng(10 + n_tiles)
    krec, vrec, Ks, Vs = [], [], [], []
    for i in range(n_tiles):
        Xk = key_tile(20 + i); Xv = rng.standard_normal((T, D))
        krec.append(O.pack_record(False, O.quantize_tile(Xk, O.levels(False, k_bits)), k_bits))
        vrec.append(O.pack_record(True, O.quantize_tile(Xv, O.levels(True, v_bits=v_bits)), v_bits=v_bits))
        Ks.append(O.dequantize_record(False, krec[-1], k_bits))
        Vs.append(O.dequantize_record(True, vrec[-1], v_bits=v_bits))
    kt = rng.standard_normal((n_tail, D)); vt = rng.standard_normal((n_tail, D))
    q = rng.standard_normal((8, D))
    K = np.concatenate(Ks + [kt]); V = np.concatenate(Vs + [vt])
    plain = O.attention(q, K, V, 1 / math.sqrt(D))
    folded = O.attention_folded(q, krec, vrec, kt, vt, 1 / math.sqrt(D), k_bits, v_bits)
    assert np.abs(plain - folded).max() < 1e-9


def test_batch_drivers_agree_with_single_calls():
    w = I.qwen3_4b()
    k = I.kv_values(w, "k", 0, 0, 2 * T).view(torch.int16).numpy().view(np.uint16)   # [256, 8, 128]
    first = np.array([0 * D, 3 * D, T * 8 * D + 5 * D], np.int64)                     # (tile, head)
    rec, flags = O.quantize_batch(k, "bf16", first, 8 * D, False, nthreads=2)
    flat = k.reshape(-1)
    for i, f in enumerate(first):
        X = O.decode16(np.stack([flat[f + r * 8 * D: f + r * 8 * D + D] for r in range(T)]), "bf16")
        assert np.array_equal(rec[i], O.pack_record(False, O.quantize_tile(X, 15)))
    assert not flags.any()


# ---------------------------------------------------------------- causal multi-query attention
def _cache(n_tiles, n_tail, seed, k_bits=4):
    rng = np.random.default_rng(seed)
    krec = [O.pack_record(False, O.quantize_tile(key_tile(40 + seed + i), O.levels(False, k_bits)), k_bits)
            for i in range(n_tiles)]
    vrec = [O.pack_record(True, O.quantize_tile(rng.standard_normal((T, D)), 3)) for _ in range(n_tiles)]
    return krec, vrec, rng.standard_normal((n_tail, D)), rng.standard_normal((n_tail, D)), rng


def test_causal_attention_matches_torch_causal_sdpa():
    """Against torch's scaled_dot_product_attention with an explicit causal
    mask over the last Q positions (fp64)."""
    krec, vrec, kt, vt, rng = _cache(2, 45, 3)
    K, V = O.cache_values(krec, vrec, kt, vt)
    n, Q, G = K.shape[0], 7, 3
    q = rng.standard_normal((Q, G, D))
    want = O.causal_attention(q, K, V, 1 / math.sqrt(D))
    pos = torch.arange(n - Q, n)[:, None]
    mask = torch.arange(n)[None, :] <= pos                              # [Q, n]
    qt = torch.from_numpy(q).permute(1, 0, 2)                            # [G, Q, D]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, torch.from_numpy(K)[None].expand(G, n, D), torch.from_numpy(V)[None].expand(G, n, D),
        attn_mask=mask[None].expand(G, Q, n)).permute(1, 0, 2).numpy()
    assert np.abs(want - ref).max() < 1e-12


def test_causal_attention_ignores_later_tokens():
    """Query i must not change when any token after its position changes."""
    krec, vrec, kt, vt, rng = _cache(1, 60, 4)
    K, V = O.cache_values(krec, vrec, kt, vt)
    n, Q = K.shape[0], 5
    q = rng.standard_normal((Q, 2, D))
    base = O.causal_attention(q, K, V, 0.1)
    for i in range(Q - 1):
        K2, V2 = K.copy(), V.copy()
        K2[n - Q + i + 1:] *= 50.0
        V2[n - Q + i + 1:] += 7.0
        assert np.array_equal(O.causal_attention(q, K2, V2, 0.1)[:i + 1], base[:i + 1])
        # the next query sees that token: with a zero query (uniform weights
        # over its prefix of n - Q + i + 2 tokens) the output moves by 7 / prefix
        q0 = q.copy()
        q0[i + 1] = 0.0
        V3 = V.copy()
        V3[n - Q + i + 1] += 7.0
        moved = O.causal_attention(q0, K, V3, 0.1)[i + 1] - O.causal_attention(q0, K, V, 0.1)[i + 1]
        assert np.abs(moved - 7.0 / (n - Q + i + 2)).max() < 1e-12


@pytest.mark.parametrize("k_bits", [4, 2])
def test_causal_attention_last_query_equals_decode_form(k_bits):
    """The last query sees the whole cache: the folded decode form."""
    krec, vrec, kt, vt, rng = _cache(3, 17, 5, k_bits)
    K, V = O.cache_values(krec, vrec, kt, vt, k_bits)
    q = rng.standard_normal((4, 8, D))
    got = O.causal_attention(q, K, V, 1 / math.sqrt(D))
    want = O.attention_folded(q[-1], krec, vrec, kt, vt, 1 / math.sqrt(D), k_bits)
    assert np.abs(got[-1] - want).max() < 1e-9


# ---------------------------------------------------------------- per-token error ablations
@pytest.mark.parametrize("levels,seed", [(15, 2), (3, 3)])
def test_unrotated_quantize_properties(levels, seed):
    """Without the rotation the record describes X itself: codes are the
    nearest level (brute force) except exact ties, and every value is within
    half a step of its reconstruction."""
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, D)) * (1 + 5 * (np.arange(D) % 17 == 0))
    tl = O.quantize_tile(X, levels, 8, rotate=False)
    g = np.array([O.e4m3_decode(c) for c in tl.g8]); a = np.array([O.e4m3_decode(c) for c in tl.a8])
    b = np.array([O.f16_decode(c) for c in tl.b16])
    Y = X / g[None, :]
    lv = a[:, None, None] * np.arange(levels + 1)[None, None, :] + b[:, None, None]
    best = np.abs(Y[:, :, None] - lv).argmin(axis=2)
    tie = np.abs(tl.pre - np.floor(tl.pre) - 0.5) < 1e-9
    assert np.array_equal(best[~tie], tl.code[~tie])
    Xh = O.dequantize_record(levels == 3, O.pack_record(levels == 3, tl), rotate=False)
    assert (np.abs(Xh - X) <= 0.5 * a[:, None] * g[None, :] * (1 + 1e-9)).all()


def test_plain_rtn_is_per_token_min_max():
    """No rotation and no normalisation: unit channel scales (g = 1), and each
    token's zero-point / step cover its own min / max (b <= min, b + L a >= max)."""
    rng = np.random.default_rng(7)
    X = rng.standard_normal((T, D))
    tl = O.quantize_tile(X, 15, 0, rotate=False)
    assert (tl.g8 == O.e4m3_encode_rne(1.0)).all()
    check_scales_tight(X, tl, 15)


def test_token_errors_definition_and_rotation_benefit():
    """err2 / norm2 are the plain sums of the reconstruction; on keys with
    outlier channels the rotation + normalisation shrink the largest token
    errors relative to plain per-token RTN (the pages' claim, checked on
    synthetic tiles)."""
    X = key_tile(11)
    e_full, n_full = O.token_errors(X, False)
    tl = O.quantize_tile(X, 15)
    Xh = O.dequantize_record(False, O.pack_record(False, tl))
    assert np.allclose(e_full, ((Xh - X) ** 2).sum(1), rtol=0, atol=1e-12)
    assert np.allclose(n_full, (X ** 2).sum(1), rtol=0, atol=1e-9)
    e_plain, _ = O.token_errors(X, False, iters=0, rotate=False)
    rel_full, rel_plain = np.sqrt(e_full / n_full), np.sqrt(e_plain / n_full)
    top = lambda r: np.sort(r)[-max(1, len(r) // 20):].mean()
    assert top(rel_full) < top(rel_plain)
