"""The checked (debug) build, libkvarn_check.so (compiled with KVARN_CHECK):
every global store, every split-K partial read and every bulk-copy source
is first tested against the extent of its buffer, and an access outside it
would be skipped and reported as KVARN_DEV_ERR_BOUNDS.  On ragged workloads
of every entry point it must report nothing and produce bit-for-bit the
results of the normal library (the checks change no arithmetic)."""
import contextlib

import pytest
import torch

from bit_kv_cache_quantize_gb300 import build as B
from bit_kv_cache_quantize_gb300 import inputs as I
from bit_kv_cache_quantize_gb300 import kvarn as K
from bit_kv_cache_quantize_gb300.cache import PagedCache

from gpu_helpers import device

pytestmark = pytest.mark.gpu
T = D = 128


@contextlib.contextmanager
def library(path):
    saved_lib, saved_path = K._lib, K.LIB_PATH
    K._lib, K.LIB_PATH = None, path
    try:
        K.lib()
        yield
    finally:
        K._lib, K.LIB_PATH = saved_lib, saved_path


@pytest.fixture(scope="module")
def libs():
    device()
    return B.LIB, B.build_checked()


def ragged(k_bits=4, v_bits=2):
    w = I.Workload("checked", 5, 16, 2, "f16", [300, 1, 0, 129, 640], seed=71, max_tokens=700, block_perm=True,
                   decode_steps=3)
    w.k_bits, w.v_bits = k_bits, v_bits
    return w


def run_all(w, dev):
    """Prefill, three append+decode steps, a multi-query call, the 16-bit
    decode, a dequantisation and the error tool; returns every output."""
    outs = {}
    c = PagedCache(w, dev, fp16_pool=True)
    c.prefill()
    lens = c.lens.clone()
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    for s in range(3):
        pos = lens.clone()
        kn = torch.stack([I.kv_values(w, "k", b, int(pos[b]), 1, dev)[0] for b in range(w.batch)])
        vn = torch.stack([I.kv_values(w, "v", b, int(pos[b]), 1, dev)[0] for b in range(w.batch)])
        c.append(kn, vn, pos)
        lens = pos + 1
        c.decode(I.queries(w, step=s + 1, device=dev), out, lens=lens)
        outs[f"decode{s}"] = out.clone()
    outs["pool"], outs["tail"] = c.pool.clone(), c.tail.clone()
    Q = 1
    qm = I.multi_queries(w, Q, device=dev)
    om = torch.empty(w.batch, Q, w.num_q_heads, D, dtype=torch.float32, device=dev)
    c.multiquery(qm, Q, om, lens=lens)
    outs["mq"] = om.clone()
    c.decode_fp16(I.queries(w, device=dev), out)
    outs["fp16"] = out.clone()
    blocks = torch.tensor([int(c.table[4, 1]), int(c.table[0, 0])], dtype=torch.int32, device=dev)
    dq = torch.empty(2, 2, w.num_kv_heads, T, D, dtype=torch.float32, device=dev)
    K.kvarn_dequantize(c.cfg, c.pool, blocks, 2, dq, c.err)
    outs["dequant"] = dq
    x = I.kv_sequence(w, "v", 4, 640, dev)
    first = torch.tensor([0, 384], dtype=torch.int64, device=dev)
    need = K.kvarn_token_errors_scratch_bytes(c.cfg, 2, 1)
    scratch = torch.zeros(need, dtype=torch.uint8, device=dev)
    eo = torch.empty(2, w.num_kv_heads, T, 2, dtype=torch.float32, device=dev)
    K.kvarn_token_errors(c.cfg, x, w.num_kv_heads * D, 640, first, 2, 1, 1, 8, scratch, need, eo, c.err)
    outs["errors"] = eo
    torch.cuda.synchronize()
    outs["err"] = c.check_error()
    return outs


@pytest.mark.parametrize("k_bits,v_bits", [(4, 2), (2, 2), (4, 4)])
def test_checked_build_reports_nothing_and_matches(libs, k_bits, v_bits):
    dev = device()
    normal, checked = libs
    with library(normal):
        want = run_all(ragged(k_bits, v_bits), dev)
    with library(checked):
        got = run_all(ragged(k_bits, v_bits), dev)
    assert want["err"] == 0
    assert got["err"] == 0, f"checked build stored device error {got['err']}"
    for name, t in want.items():
        if name != "err":
            assert torch.equal(got[name], t), f"{name} differs between the checked and the normal build"
