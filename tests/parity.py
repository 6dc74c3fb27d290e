"""Comparison of GPU-packed records with the oracle's, under the parity rule:

* scales: every FP8 per-channel scale g within one code of the oracle's
  (adjacent values).  The per-token zero-point b and step a follow from the
  channel scales (b = FP16_rd(min_c R/g), a = E4M3_ru((max_c R/g - b)/L)),
  so they must be within one code of that definition applied to the GPU's
  own g (computed here in fp64 from the oracle's rotated tile); where the
  GPU's g equal the oracle's this is the oracle's b and a.  (A channel scale
  that flips at an E4M3 rounding boundary can move the zero-point of a token
  whose minimum sits in that channel by many FP16 codes, legitimately.)  The
  number of differing scales is reported;
* codes: where g[c], a[t] and b[t] all equal the oracle's, every code is
  bit-exact except where the oracle's fp64 pre-rounding value (Y - b)/a lies
  within 1e-5 of a .5 boundary; there it may differ by one level, in at most
  0.01% of the codes;
* where a scale differs (both values are then valid quantisations), the GPU
  code must still be the nearest level of its own scales: rint((Y - b)/a)
  computed here in fp64 from the oracle's rotated tile, same tie rule.

The GPU bytes are decoded here with numpy/torch, not with the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

T = D = 128


def e4m3(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def f16(bits: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def f16_order(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns -> integers ordered like the values."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


E4M3_TABLE = e4m3(np.arange(0x7F, dtype=np.uint8))                 # non-negative finite values, ascending


def f16_rd_bits(x: np.ndarray) -> np.ndarray:
    """Largest FP16 value <= x (fp64 array), as FP16 bits."""
    h = x.astype(np.float16)
    h = np.where(h.astype(np.float64) > x, np.nextafter(h, np.float16(-np.inf)), h).astype(np.float16)
    return h.view(np.uint16)


def token_scales_for(R: np.ndarray, g8: np.ndarray, b16: np.ndarray, L: int):
    """The per-token zero-points and steps the definition gives for channel
    scales g8 (and, for the step, zero-points b16): ([T] FP16 bits,
    [T] E4M3 codes), from the fp64 rotated tile R [T, D]."""
    Y = R / e4m3(g8)[None, :]
    b_exp = f16_rd_bits(Y.min(axis=1))
    step = (Y.max(axis=1) - f16(b16)) / L
    a_exp = np.minimum(np.searchsorted(E4M3_TABLE, step, side="left"), 0x7E)
    return b_exp, np.maximum(a_exp, 1).astype(np.uint8)


def unpack(rec: np.ndarray, is_v: bool, k_bits: int = 4, v_bits: int = 2):
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    g8 = rec[:128].copy()
    a8 = rec[128:256].copy()
    b16 = rec[256:512].view(np.uint16).copy()
    body = rec[512:]
    if not is_v and k_bits == 2:
        by = body.reshape(T, 32)                      # [token][byte]: channels 4i .. 4i+3 at bits 2k
        code = np.stack([(by >> (2 * k)) & 3 for k in range(4)], axis=-1).reshape(T, D).astype(np.uint8)
    elif not is_v:
        by = body.reshape(T, 64)
        code = np.empty((T, D), np.uint8)
        code[:, 0::2] = by & 15
        code[:, 1::2] = by >> 4
    elif v_bits == 4:
        words = body.view("<u4").reshape(D, T // 8)   # [channel][word]: tokens 8w .. 8w+7
        pos = np.array([2 * u if u % 2 == 0 else 14 + 2 * u for u in range(8)], dtype=np.uint32)
        nib = (words[:, :, None] >> pos[None, None, :]) & 15  # [c][w][u] -> token 8w+u
        code = nib.reshape(D, T).T.astype(np.uint8).copy()
    else:
        words = body.view("<u4").reshape(D, T // 16)  # [channel][word]: tokens 16w .. 16w+15
        pos = np.array([u if u % 2 == 0 else 15 + u for u in range(16)], dtype=np.uint32)
        crumbs = (words[:, :, None] >> pos[None, None, :]) & 3  # [c][w][u] -> token 16w+u
        code = crumbs.reshape(D, T).T.astype(np.uint8).copy()
    return g8, a8, b16, code


class Stats:
    def __init__(self):
        self.tiles = self.codes = 0
        self.g_flip = self.a_flip = self.b_flip = 0
        self.tie_diff = self.valid_checked = 0

    def __repr__(self):
        return (f"tiles={self.tiles} codes={self.codes} g_flip={self.g_flip} a_flip={self.a_flip} "
                f"b_flip={self.b_flip} tie_diff={self.tie_diff} checked_vs_own_scales={self.valid_checked}")


def compare_record(gpu_rec: np.ndarray, tile, is_v: bool, st: Stats, where: str = "", k_bits: int = 4,
                   v_bits: int = 2):
    """tile: oracle.Tile of the same input."""
    L = 15 if (v_bits if is_v else k_bits) == 4 else 3
    g8, a8, b16, code = unpack(gpu_rec, is_v, k_bits, v_bits)
    st.tiles += 1
    st.codes += code.size
    assert code.max() <= L, where
    dg = np.abs(g8.astype(int) - tile.g8.astype(int))
    assert dg.max() <= 1, f"{where}: channel scale off by more than one code"
    b_ref, a_ref = (tile.b16, tile.a8) if not dg.any() else token_scales_for(tile.R, g8, b16, L)
    da = np.abs(a8.astype(int) - a_ref.astype(int))
    db = np.abs(f16_order(b16) - f16_order(b_ref))
    assert da.max() <= 1 and db.max() <= 1, f"{where}: token scale off by more than one code"
    da = np.abs(a8.astype(int) - tile.a8.astype(int))
    db = np.abs(f16_order(b16) - f16_order(tile.b16))
    st.g_flip += int((dg > 0).sum()); st.a_flip += int((da > 0).sum()); st.b_flip += int((db > 0).sum())
    same = (dg == 0)[None, :] & (da == 0)[:, None] & (db == 0)[:, None]
    frac = tile.pre - np.floor(tile.pre)
    near = np.abs(frac - 0.5) < 1e-5
    mism = code != tile.code
    bad = mism & same & ~near
    assert not bad.any(), f"{where}: {int(bad.sum())} codes differ with identical scales (first {np.argwhere(bad)[:3]})"
    tie = mism & same & near
    assert (np.abs(code.astype(int) - tile.code.astype(int))[tie] <= 1).all(), where
    st.tie_diff += int(tie.sum())
    if not same.all():
        g, a, b = e4m3(g8), e4m3(a8), f16(b16)
        t = (tile.R / g[None, :] - b[:, None]) / a[:, None]
        want = np.clip(np.rint(t), 0, L)
        near2 = np.abs((t - np.floor(t)) - 0.5) < 1e-5
        chk = ~same
        badv = chk & (code != want) & ~(near2 & (np.abs(code - want) <= 1))
        assert not badv.any(), f"{where}: {int(badv.sum())} codes are not the nearest level of their own scales"
        st.valid_checked += int(chk.sum())


def unpack_batch(recs: np.ndarray, is_v: bool, k_bits: int = 4, v_bits: int = 2):
    """unpack() of n records at once: recs [n, record bytes] ->
    g8 [n,128], a8 [n,128], b16 [n,128], code [n,128,128] (token-major)."""
    recs = np.ascontiguousarray(recs, dtype=np.uint8)
    n = recs.shape[0]
    g8, a8 = recs[:, :128].copy(), recs[:, 128:256].copy()
    b16 = recs[:, 256:512].copy().view(np.uint16)
    body = recs[:, 512:]
    if not is_v and k_bits == 2:
        by = body.reshape(n, T, 32)
        code = np.stack([(by >> (2 * k)) & 3 for k in range(4)], axis=-1).reshape(n, T, D)
    elif not is_v:
        by = body.reshape(n, T, 64)
        code = np.empty((n, T, D), np.uint8)
        code[:, :, 0::2] = by & 15
        code[:, :, 1::2] = by >> 4
    elif v_bits == 4:
        words = body.copy().view("<u4").reshape(n, D, T // 8)
        pos = np.array([2 * u if u % 2 == 0 else 14 + 2 * u for u in range(8)], dtype=np.uint32)
        nib = (words[..., None] >> pos) & 15                     # [n][c][w][u] -> token 8w+u
        code = nib.reshape(n, D, T).transpose(0, 2, 1)
    else:
        words = body.copy().view("<u4").reshape(n, D, T // 16)
        pos = np.array([u if u % 2 == 0 else 15 + u for u in range(16)], dtype=np.uint32)
        crumbs = (words[..., None] >> pos) & 3                   # [n][c][w][u] -> token 16w+u
        code = crumbs.reshape(n, D, T).transpose(0, 2, 1)
    return g8, a8, b16, np.ascontiguousarray(code, dtype=np.uint8)


def compare_batch(gpu_recs: np.ndarray, ora: dict, is_v: bool, st: Stats, where: str = "", k_bits: int = 4,
                  v_bits: int = 2):
    """compare_record() over n tiles at once.  ora: the oracle's fields of the
    same inputs (oracle.quantize_batch_fields with pre and R)."""
    L = 15 if (v_bits if is_v else k_bits) == 4 else 3
    g8, a8, b16, code = unpack_batch(gpu_recs, is_v, k_bits, v_bits)
    n = code.shape[0]
    st.tiles += n
    st.codes += code.size
    assert code.max() <= L, where
    dg = np.abs(g8.astype(int) - ora["g8"].astype(int))
    assert dg.max() <= 1, f"{where}: channel scale off by more than one code (tile {np.argwhere(dg > 1)[0]})"
    b_ref, a_ref = ora["b16"].copy(), ora["a8"].copy()
    for i in np.nonzero(dg.any(axis=1))[0]:      # a channel scale flipped: the token scales its g imply
        b_ref[i], a_ref[i] = token_scales_for(ora["R"][i], g8[i], b16[i], L)
    da = np.abs(a8.astype(int) - a_ref.astype(int))
    db = np.abs(f16_order(b16) - f16_order(b_ref))
    if not (da.max() <= 1 and db.max() <= 1):
        msg = []
        for name, d, gpu, want in (("a", da, a8, a_ref), ("b", db, b16, b_ref)):
            for i, j in np.argwhere(d > 1)[:4]:
                msg.append(f"{name}[tile {i}][{j}] gpu {gpu[i, j]:#x} expected {want[i, j]:#x} (g flips in tile: "
                           f"{int((dg[i] > 0).sum())})")
        raise AssertionError(f"{where}: token scale off by more than one code: " + "; ".join(msg))
    da = np.abs(a8.astype(int) - ora["a8"].astype(int))
    db = np.abs(f16_order(b16) - f16_order(ora["b16"]))
    st.g_flip += int((dg > 0).sum()); st.a_flip += int((da > 0).sum()); st.b_flip += int((db > 0).sum())
    same = (dg == 0)[:, None, :] & (da == 0)[:, :, None] & (db == 0)[:, :, None]
    pre = ora["pre"]
    near = np.abs(pre - np.floor(pre) - 0.5) < 1e-5
    mism = code != ora["code"]
    bad = mism & same & ~near
    assert not bad.any(), f"{where}: {int(bad.sum())} codes differ with identical scales (first {np.argwhere(bad)[:3]})"
    tie = mism & same & near
    assert (np.abs(code.astype(int) - ora["code"].astype(int))[tie] <= 1).all(), where
    st.tie_diff += int(tie.sum())
    diff_tiles = np.nonzero(~same.reshape(n, -1).all(axis=1))[0]
    for i in diff_tiles:                     # a scale differs: the GPU code is the nearest level of its own scales
        g, a, b = e4m3(g8[i]), e4m3(a8[i]), f16(b16[i])
        t = (ora["R"][i] / g[None, :] - b[:, None]) / a[:, None]
        want = np.clip(np.rint(t), 0, L)
        near2 = np.abs((t - np.floor(t)) - 0.5) < 1e-5
        chk = ~same[i]
        badv = chk & (code[i] != want) & ~(near2 & (np.abs(code[i] - want) <= 1))
        assert not badv.any(), f"{where} tile {i}: {int(badv.sum())} codes are not the nearest level of their own scales"
        st.valid_checked += int(chk.sum())


def finish(st: Stats):
    assert st.tie_diff <= 1e-4 * max(st.codes, 1), f"too many boundary flips: {st}"
    return st
