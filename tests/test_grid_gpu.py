"""GPU parity over the whole ragged-varlen stress grid: {64/8, 32/4} heads x
head dim {64, 128, 256} x window {1, 15, 64, 127, 128, 129, 4096, none} x
sinks {none, per-head, smooth_softmax} x {fp16, bf16} -- 288 cells.

Each cell is a reduced ragged batch of its own (6 sequences, prefixes drawn
uniformly in [0, 2048], extends in [1, 700], seeded per cell), generated on
the GPU, run through the C ABI, and checked against the oracle on sampled
rows of every sequence: the first and last rows, rows on both sides of a
128-position boundary, and a seeded random draw."""
import numpy as np
import pytest
import torch

from gqa_flash_attention_prefill_gb300 import workloads as W
from parity_util import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

HEADS = [(64, 8), (32, 4)]
DIMS = [64, 128, 256]
WINDOWS = [1, 15, 64, 127, 128, 129, 4096, 0]
SINKS = ["none", "head", "smooth"]
DTYPES = ["f16", "bf16"]


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__
    __graft_entry__.build()
    import gqa_flash_attention_prefill_gb300 as pkg
    pkg.load()
    pkg.force_block_n(0)
    pkg.force_q_tiles(0)
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkg


def _cell_seed(hq, d, window, sink, dtype):
    return (hq * 131 + d * 7 + window * 3 + SINKS.index(sink) * 100003
            + DTYPES.index(dtype) * 7919)


def _rows(batch, seed, per_seq=6):
    rng = np.random.default_rng(seed)
    cu = batch.cu_seqlens_q.tolist()
    rows = []
    for b in range(batch.num_seqs):
        e = cu[b + 1] - cu[b]
        cand = {0, e - 1, 127, 128}
        cand.update(int(x) for x in rng.integers(0, e, size=per_seq))
        rows.extend(cu[b] + i for i in cand if 0 <= i < e)
    return np.array(sorted(set(rows)), dtype=np.int64)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("sink", SINKS)
@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("d", DIMS)
@pytest.mark.parametrize("hq,hkv", HEADS)
def test_ragged_grid_cell(pkg, hq, hkv, d, window, sink, dtype):
    seed = _cell_seed(hq, d, window, sink, dtype)
    gen = torch.Generator().manual_seed(seed)
    pre = torch.randint(0, 2048 + 1, (6,), generator=gen).tolist()
    ext = torch.randint(1, 700 + 1, (6,), generator=gen).tolist()
    dev = W.make_batch(pre, ext, hq, hkv, d, dtype, window=window, sink_mode=sink,
                       seed=seed, device="cuda",
                       name=f"grid {hq}/{hkv} d{d} w{window} {sink} {dtype}")
    cpu = dev.to("cpu")
    out, lse = run_gpu(pkg, cpu)
    rows = _rows(cpu, seed)
    ref, ref_lse = run_oracle(cpu, rows=rows)
    compare(out, lse, ref, ref_lse, rows=rows, label=cpu.name)
    # rows not sampled were written too, with finite values
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
