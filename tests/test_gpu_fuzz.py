"""Seeded random configurations against the oracle: head counts, group sizes,
dtypes, presets, value distributions, outlier patterns and ragged lengths
(empty, one token, tile edges, long) drawn from one generator, so that
combinations no hand-written case names still meet the parity bar.  Every
case quantises all closed tiles on the GPU and compares them record by
record, decodes over oracle records (plus the raw open tile), and runs the
multi-query attention for a random number of query tokens."""
import numpy as np
import pytest

from bit_kv_cache_quantize_gb300 import inputs as I

from test_gpu_append import run_steps
from test_gpu_decode import run_decode_case
from test_gpu_multiquery import run_mq_case
from test_gpu_quantize import quantize_and_compare

pytestmark = pytest.mark.gpu
T = 128
N_CASES = 32
EDGES = [0, 1, 127, 128, 129, 255, 256, 383]


def random_workload(i, min_len=0):
    rng = np.random.default_rng(9000 + i)
    h_kv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    batch = int(rng.integers(1, 6))
    k_bits, v_bits = [(4, 2), (2, 2), (4, 4)][int(rng.integers(0, 3))]
    lens = []
    for _ in range(batch):
        n = int(rng.choice(EDGES)) if rng.random() < 0.5 else int(rng.integers(1, 1600))
        lens.append(max(n, min_len))
    if max(lens) < T:  # the ABI takes max_blocks >= 1: keep one closed tile in the batch
        lens[0] = T + 1
    w = I.Workload(f"fuzz{i}", batch, g * h_kv, h_kv, str(rng.choice(["f16", "bf16"])), lens, seed=700 + i,
                   v_dist=str(rng.choice(["normal", "t4"])), k_outliers=str(rng.choice(["fixed", "random"])),
                   max_tokens=max(max(lens), T), block_perm=True, k_bits=k_bits, v_bits=v_bits)
    return w, rng


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i):
    w, rng = random_workload(i)
    print(f"{w.name}: B={w.batch} H_kv={w.num_kv_heads} G={w.G} {w.dtype} K{w.k_bits}/V{w.v_bits} "
          f"v={w.v_dist} outliers={w.k_outliers} lens={w.seq_lens}")
    if any(n >= T for n in w.seq_lens):
        quantize_and_compare(w, list(range(w.batch)))
    run_decode_case(w)
    q_tokens = int(rng.integers(1, 21))
    wm, _ = random_workload(i, min_len=q_tokens)
    run_mq_case(wm, q_tokens)


@pytest.mark.parametrize("i", range(8))
def test_random_append_steps(i):
    """Random decode steps: append one token per sequence (closing tiles on
    the way), attend after every step; every closed tile and every step's
    attention against the oracle."""
    w, rng = random_workload(100 + i)
    steps = int(rng.integers(2, 6))
    # start some sequences a few tokens short of a tile edge so that tiles close during the run
    w.seq_lens = [n - (n % T) + T - int(rng.integers(1, steps + 1)) if rng.random() < 0.5 else n for n in w.seq_lens]
    w.decode_steps = steps
    w.max_tokens = max(w.seq_lens) + steps
    print(f"{w.name}: B={w.batch} H_kv={w.num_kv_heads} G={w.G} {w.dtype} K{w.k_bits}/V{w.v_bits} "
          f"lens={w.seq_lens} steps={steps}")
    run_steps(w, steps)
