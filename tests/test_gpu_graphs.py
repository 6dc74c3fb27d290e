"""The entry points capture into a CUDA graph, as a serving engine records its
decode step once and replays it: one step (append one token per sequence,
two of which close a tile, then the decode and a multi-query call) recorded
after a direct run replays to the same bytes.  The combines are launched as
programmatic dependents of their split-K kernels, which the capture keeps."""
import pytest
import torch

from bit_kv_cache_quantize_gb300 import inputs as I
from bit_kv_cache_quantize_gb300.cache import PagedCache

from gpu_helpers import device

pytestmark = pytest.mark.gpu
T = D = 128


def test_serving_step_replays_from_a_graph():
    dev = device()
    lens0 = [1000, 127, 700, 2047]  # sequences 1 and 3 close a tile with this token
    w = I.Workload("graph_step", len(lens0), 32, 4, "bf16", lens0, seed=90, max_tokens=2048 + 8, block_perm=True,
                   decode_steps=1)
    c = PagedCache(w, dev)
    c.prefill()
    pos = torch.tensor(lens0, dtype=torch.int32, device=dev)
    k_new = torch.stack([I.kv_values(w, "k", b, lens0[b], 1, dev)[0] for b in range(w.batch)])
    v_new = torch.stack([I.kv_values(w, "v", b, lens0[b], 1, dev)[0] for b in range(w.batch)])
    lens = pos + 1
    q = I.queries(w, device=dev)
    Q = 3
    qm = I.multi_queries(w, Q, device=dev)
    out = torch.empty(w.batch, w.num_q_heads, D, dtype=torch.float32, device=dev)
    outm = torch.empty(w.batch, Q, w.num_q_heads, D, dtype=torch.float32, device=dev)

    def step():
        c.append(k_new, v_new, pos)
        c.decode(q, out, lens=lens)
        c.multiquery(qm, Q, outm, lens=lens)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # direct run (also fills the first-use caches and the workspaces)
    torch.cuda.synchronize()
    assert c.check_error() == 0
    ref, refm, pool = out.clone(), outm.clone(), c.pool.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    out.fill_(float("nan"))
    outm.fill_(float("nan"))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert c.check_error() == 0
    assert torch.equal(c.pool, pool)  # the re-closed tiles quantise to the same records
    assert torch.equal(out, ref) and torch.equal(outm, refm)
