"""ctypes front end of the plain CPU oracle (``kvarn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
CPU-baseline leg of ``bench.py`` use it; the product path never imports it.
It shares no code with the CUDA library.  Every function works on numpy
arrays and is fp64 inside; see the C file for the definitions and sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvarn_oracle.c")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libkvarn_oracle.so")

D = 128
T = 128
K_LEVELS = 15
V_LEVELS = 3
FLAG_CLAMPED = 1
FLAG_STEP_SAT = 2


_build_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with plain IEEE semantics (no FMA contraction, which
    gcc enables by default on aarch64).  Safe to call from several threads
    (one compiles, the others wait) and processes (each writes its own
    temporary file and renames it into place)."""
    with _build_lock:
        os.makedirs(BUILD, exist_ok=True)
        if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            tmp = LIB + f".{os.getpid()}.{threading.get_ident()}.tmp"
            subprocess.check_call(
                ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                 "-shared", "-Wall", "-o", tmp, SRC, "-lm", "-lpthread"])
            os.replace(tmp, LIB)
        return LIB


_lib = None
_lib_lock = threading.Lock()


def lib():
    global _lib
    if _lib is not None:
        return _lib
    with _lib_lock:
        return _load()


def _load():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl, u8, u16 = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_uint8, ctypes.c_uint16
        L.ora_e4m3_decode.restype = dbl; L.ora_e4m3_decode.argtypes = [u8]
        L.ora_e4m3_encode_rne.restype = u8; L.ora_e4m3_encode_rne.argtypes = [dbl]
        L.ora_e4m3_encode_ru.restype = u8; L.ora_e4m3_encode_ru.argtypes = [dbl]
        L.ora_f16_decode.restype = dbl; L.ora_f16_decode.argtypes = [u16]
        L.ora_f16_encode_rd.restype = u16; L.ora_f16_encode_rd.argtypes = [dbl]
        L.ora_f16_encode_rne.restype = u16; L.ora_f16_encode_rne.argtypes = [dbl]
        L.ora_bf16_decode.restype = dbl; L.ora_bf16_decode.argtypes = [u16]
        L.ora_hadamard_matrix.argtypes = [P]
        L.ora_rotate.argtypes = [P, i32, P]
        L.ora_sinkhorn.argtypes = [P, i32, P, P]
        L.ora_quantize_tile.restype = i32
        L.ora_quantize_tile.argtypes = [P, i32, i32, P, P, P, P, P, P, P]
        L.ora_record_bytes.restype = i32; L.ora_record_bytes.argtypes = [i32]
        L.ora_pack_record.argtypes = [i32, P, P, P, P, P]
        L.ora_unpack_record.argtypes = [i32, P, P, P, P, P]
        L.ora_dequantize_record.argtypes = [i32, P, P]
        L.ora_quantize_tile_ex.restype = i32
        L.ora_quantize_tile_ex.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, P]
        L.ora_dequantize_record_ex.argtypes = [i32, P, i32, P]
        L.ora_attention.argtypes = [P, i32, P, P, i32, dbl, P]
        L.ora_attention_folded.argtypes = [P, i32, P, P, i32, P, P, i32, dbl, i32, i32, P]
        L.ora_quantize_batch.argtypes = [P, i32, P, i64, i32, i32, i32, P, P, i32]
        L.ora_attention_batch.argtypes = [P, i32, P, P, P, P, P, P, P, dbl, i32, i32, i32, P, i32]
        L.ora_quantize_batch_fields.argtypes = [P, i32, P, i64, i32, i32, i32, P, P, P, P, P, P, P, i32]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- formats
def e4m3_decode(code: int) -> float:
    return lib().ora_e4m3_decode(int(code))


def e4m3_encode_rne(x: float) -> int:
    return int(lib().ora_e4m3_encode_rne(float(x)))


def e4m3_encode_ru(x: float) -> int:
    return int(lib().ora_e4m3_encode_ru(float(x)))


def f16_decode(bits: int) -> float:
    return lib().ora_f16_decode(int(bits))


def f16_encode_rd(x: float) -> int:
    return int(lib().ora_f16_encode_rd(float(x)))


def f16_encode_rne(x: float) -> int:
    return int(lib().ora_f16_encode_rne(float(x)))


def decode16(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of 16-bit storage (dtype 'f16' or 'bf16')."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- rotation
def hadamard_matrix() -> np.ndarray:
    H = np.empty((D, D), np.float64)
    lib().ora_hadamard_matrix(_p(H))
    return H


def rotate(X: np.ndarray) -> np.ndarray:
    X = np.ascontiguousarray(X, dtype=np.float64).reshape(-1, D)
    Y = np.empty_like(X)
    lib().ora_rotate(_p(X), X.shape[0], _p(Y))
    return Y


def sinkhorn(R: np.ndarray, iters: int = 8):
    """Returns (u[T], v[D]) log-factors (v not yet centred)."""
    R = np.ascontiguousarray(R, dtype=np.float64)
    assert R.shape == (T, D)
    u = np.empty(T); v = np.empty(D)
    lib().ora_sinkhorn(_p(R), iters, _p(u), _p(v))
    return u, v


# ---------------------------------------------------------------- tiles
class Tile:
    """Quantised tile as the oracle computes it."""

    def __init__(self, g8, a8, b16, code, pre, R, v, flags):
        self.g8, self.a8, self.b16, self.code = g8, a8, b16, code
        self.pre, self.R, self.v, self.flags = pre, R, v, flags

    def g(self):
        return np.array([e4m3_decode(c) for c in self.g8])

    def a(self):
        return np.array([e4m3_decode(c) for c in self.a8])

    def b(self):
        return self.b16.view(np.float16).astype(np.float64)


def quantize_tile(X: np.ndarray, levels: int, iters: int = 8, rotate: bool = True) -> Tile:
    """rotate=False quantises X itself (the no-rotation ablation)."""
    X = np.ascontiguousarray(X, dtype=np.float64)
    assert X.shape == (T, D)
    g8 = np.empty(D, np.uint8); a8 = np.empty(T, np.uint8); b16 = np.empty(T, np.uint16)
    code = np.empty((T, D), np.uint8); pre = np.empty((T, D)); R = np.empty((T, D)); v = np.empty(D)
    f = lib().ora_quantize_tile_ex(_p(X), levels, iters, 1 if rotate else 0, _p(g8), _p(a8), _p(b16), _p(code),
                                   _p(pre), _p(R), _p(v))
    return Tile(g8, a8, b16, code, pre, R, v, f)


# Record kinds: 4-bit keys (the kvarn_k4v2 preset), 2-bit values, 2-bit keys
# (the K2/V2 preset), 4-bit values (the K4/V4 preset).  Functions take is_v
# and the key and value widths.
K4, V2, K2, V4 = 0, 1, 2, 3


def kind(is_v: bool, k_bits: int = 4, v_bits: int = 2) -> int:
    assert k_bits in (2, 4) and v_bits in (2, 4)
    if is_v:
        return V2 if v_bits == 2 else V4
    return K4 if k_bits == 4 else K2


def levels(is_v: bool, k_bits: int = 4, v_bits: int = 2) -> int:
    return 15 if (v_bits if is_v else k_bits) == 4 else 3


def record_bytes(is_v: bool, k_bits: int = 4, v_bits: int = 2) -> int:
    return int(lib().ora_record_bytes(kind(is_v, k_bits, v_bits)))


def pack_record(is_v: bool, tile: Tile, k_bits: int = 4, v_bits: int = 2) -> np.ndarray:
    rec = np.zeros(record_bytes(is_v, k_bits, v_bits), np.uint8)
    lib().ora_pack_record(kind(is_v, k_bits, v_bits), _p(tile.g8), _p(tile.a8), _p(tile.b16),
                          _p(np.ascontiguousarray(tile.code)), _p(rec))
    return rec


def unpack_record(is_v: bool, rec: np.ndarray, k_bits: int = 4, v_bits: int = 2):
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    g8 = np.empty(D, np.uint8); a8 = np.empty(T, np.uint8); b16 = np.empty(T, np.uint16)
    code = np.empty((T, D), np.uint8)
    lib().ora_unpack_record(kind(is_v, k_bits, v_bits), _p(rec), _p(g8), _p(a8), _p(b16), _p(code))
    return g8, a8, b16, code


def dequantize_record(is_v: bool, rec: np.ndarray, k_bits: int = 4, rotate: bool = True,
                      v_bits: int = 2) -> np.ndarray:
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    out = np.empty((T, D))
    lib().ora_dequantize_record_ex(kind(is_v, k_bits, v_bits), _p(rec), 1 if rotate else 0, _p(out))
    return out


def token_errors(X: np.ndarray, is_v: bool, k_bits: int = 4, iters: int = 8, rotate: bool = True,
                 v_bits: int = 2):
    """Per-token reconstruction error of one tile ("Huawei's KVarN puts
    KV-cache quantization inside vLLM's backend", section "Why KV-cache
    quantization degrades under autoregressive decoding": per-token errors):
    quantise, pack, dequantise, then for each token t
      err2[t] = sum_c (Xhat[t][c] - X[t][c])^2,  norm2[t] = sum_c X[t][c]^2."""
    X = np.ascontiguousarray(X, dtype=np.float64)
    tl = quantize_tile(X, levels(is_v, k_bits, v_bits), iters, rotate)
    Xh = dequantize_record(is_v, pack_record(is_v, tl, k_bits, v_bits), k_bits, rotate, v_bits)
    return ((Xh - X) ** 2).sum(axis=1), (X ** 2).sum(axis=1)


# ---------------------------------------------------------------- attention
def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float64).reshape(-1, D)
    K = np.ascontiguousarray(K, dtype=np.float64).reshape(-1, D)
    V = np.ascontiguousarray(V, dtype=np.float64).reshape(-1, D)
    out = np.empty_like(q)
    lib().ora_attention(_p(q), q.shape[0], _p(K), _p(V), K.shape[0], float(scale), _p(out))
    return out


def _ptr_array(recs):
    arr = (ctypes.c_void_p * max(1, len(recs)))()
    for i, r in enumerate(recs):
        arr[i] = r.ctypes.data
    return arr


def attention_folded(q, krecs, vrecs, ktail, vtail, scale, k_bits: int = 4, v_bits: int = 2) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float64).reshape(-1, D)
    krecs = [np.ascontiguousarray(r, dtype=np.uint8) for r in krecs]
    vrecs = [np.ascontiguousarray(r, dtype=np.uint8) for r in vrecs]
    ktail = np.ascontiguousarray(ktail, dtype=np.float64).reshape(-1, D)
    vtail = np.ascontiguousarray(vtail, dtype=np.float64).reshape(-1, D)
    out = np.empty_like(q)
    ka, va = _ptr_array(krecs), _ptr_array(vrecs)
    lib().ora_attention_folded(_p(q), q.shape[0], ka, va, len(krecs), _p(ktail), _p(vtail),
                               ktail.shape[0], float(scale), kind(False, k_bits), kind(True, k_bits, v_bits),
                               _p(out))
    return out


def cache_values(krecs, vrecs, ktail, vtail, k_bits: int = 4, v_bits: int = 2):
    """The cache as attention reads it ("Huawei's KVarN puts KV-cache
    quantization inside vLLM's backend", section "The four-stage pipeline":
    dequantisation at read time): the dequantised closed tiles in order, then
    the raw open-tile tokens.  Returns K, V as [n, D] fp64."""
    ks = [dequantize_record(False, r, k_bits) for r in krecs] + [np.asarray(ktail, np.float64).reshape(-1, D)]
    vs = [dequantize_record(True, r, k_bits, v_bits=v_bits) for r in vrecs] + [np.asarray(vtail, np.float64).reshape(-1, D)]
    return np.concatenate(ks), np.concatenate(vs)


def causal_attention(q, K, V, scale) -> np.ndarray:
    """Several new query tokens over a cache of n tokens: q [Q, G, D] holds
    the G heads of each of the last Q positions n - Q .. n - 1 of K, V
    ([n, D]); query i attends to positions 0 .. n - Q + i.  Plain softmax
    attention (``attention``) over each prefix; returns [Q, G, D]."""
    q = np.asarray(q, np.float64)
    n, Q = K.shape[0], q.shape[0]
    assert n >= Q
    return np.stack([attention(q[i], K[:n - Q + i + 1], V[:n - Q + i + 1], scale) for i in range(Q)])


def quantize_batch(src_bits: np.ndarray, dtype: str, first: np.ndarray, row_stride: int, is_v: bool,
                   iters: int = 8, nthreads: int | None = None, k_bits: int = 4, v_bits: int = 2):
    """Quantise len(first) tiles read from flat 16-bit storage; returns
    (records [n, record_bytes], flags [n])."""
    src_bits = np.ascontiguousarray(src_bits, dtype=np.uint16).reshape(-1)
    first = np.ascontiguousarray(first, dtype=np.int64)
    n = first.shape[0]
    rec = np.zeros((n, record_bytes(is_v, k_bits, v_bits)), np.uint8)
    flags = np.zeros(n, np.int32)
    nthreads = nthreads or os.cpu_count() or 1
    lib().ora_quantize_batch(_p(src_bits), 1 if dtype == "bf16" else 0, _p(first), int(row_stride), n,
                             kind(is_v, k_bits, v_bits), iters, _p(rec), _p(flags), int(nthreads))
    return rec, flags


def quantize_batch_fields(src_bits: np.ndarray, dtype: str, first: np.ndarray, row_stride: int, levels: int,
                          iters: int = 8, nthreads: int | None = None, with_pre: bool = True, with_R: bool = True):
    """Quantise len(first) tiles read from flat 16-bit storage (as
    quantize_batch) and return every field unpacked: dict of g8 [n,128],
    a8 [n,128], b16 [n,128], code [n,128,128], flags [n], and optionally the
    pre-rounding values pre [n,128,128] and the rotated tiles R [n,128,128]."""
    src_bits = np.ascontiguousarray(src_bits, dtype=np.uint16).reshape(-1)
    first = np.ascontiguousarray(first, dtype=np.int64)
    n = first.shape[0]
    out = dict(g8=np.empty((n, D), np.uint8), a8=np.empty((n, T), np.uint8), b16=np.empty((n, T), np.uint16),
               code=np.empty((n, T, D), np.uint8), flags=np.zeros(n, np.int32),
               pre=np.empty((n, T, D)) if with_pre else None, R=np.empty((n, T, D)) if with_R else None)
    nthreads = nthreads or os.cpu_count() or 1
    lib().ora_quantize_batch_fields(_p(src_bits), 1 if dtype == "bf16" else 0, _p(first), int(row_stride), n,
                                    int(levels), int(iters), _p(out["g8"]), _p(out["a8"]), _p(out["b16"]),
                                    _p(out["code"]), _p(out["pre"]) if with_pre else None,
                                    _p(out["R"]) if with_R else None, _p(out["flags"]), int(nthreads))
    return out


def attention_batch(q, krec_lists, vrec_lists, ktails, vtails, n_tail, scale, nthreads=None, k_bits: int = 4,
                    v_bits: int = 2):
    """q [U, G, D]; krec_lists/vrec_lists: per unit a list of records;
    ktails/vtails [U, T, D] fp64 (rows beyond n_tail[u] ignored)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    U, G = q.shape[0], q.shape[1]
    flatk = [np.ascontiguousarray(r, dtype=np.uint8) for lst in krec_lists for r in lst]
    flatv = [np.ascontiguousarray(r, dtype=np.uint8) for lst in vrec_lists for r in lst]
    n_tiles = np.array([len(lst) for lst in krec_lists], np.int32)
    off = np.zeros(U, np.int64)
    off[1:] = np.cumsum(n_tiles)[:-1]
    ktails = np.ascontiguousarray(ktails, dtype=np.float64)
    vtails = np.ascontiguousarray(vtails, dtype=np.float64)
    n_tail = np.ascontiguousarray(n_tail, dtype=np.int32)
    out = np.empty((U, G, D))
    nthreads = nthreads or os.cpu_count() or 1
    lib().ora_attention_batch(_p(q), G, _ptr_array(flatk), _ptr_array(flatv), _p(off), _p(n_tiles),
                              _p(ktails), _p(vtails), _p(n_tail), float(scale), kind(False, k_bits),
                              kind(True, k_bits, v_bits), U, _p(out),
                              int(nthreads))
    return out
