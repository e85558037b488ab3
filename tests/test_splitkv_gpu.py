"""Split-KV through the C ABI: each unit's key tiles divided over several
CTAs, fp32 partials merged by log-sum-exp, compared with the CPU oracle on the
same seeded inputs (and with the unsplit kernel)."""
import numpy as np
import pytest
import torch

from gqa_flash_attention_prefill_gb300 import workloads as W
from parity_util import compare, run_oracle, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__
    __graft_entry__.build()
    import gqa_flash_attention_prefill_gb300 as pkg
    pkg.load()
    pkg.force_block_n(0)
    pkg.force_q_tiles(0)
    return pkg


def run_split(pkg, batch_cpu, num_splits):
    dev = batch_cpu.to("cuda")
    out = torch.full_like(dev.q, float("nan"))
    lse = torch.full(dev.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    pkg.prefill_splitkv(dev, num_splits=num_splits, out=out, lse=lse)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    return out.cpu(), lse.cpu()


def check(pkg, b, num_splits, rows=None, label=""):
    out, lse = run_split(pkg, b, num_splits)
    ref, ref_lse = run_oracle(b, rows=rows)
    return compare(out, lse, ref, ref_lse, rows=rows, label=label or f"{b.name}/S{num_splits}")


@pytest.mark.parametrize("num_splits", [2, 3, 16])
@pytest.mark.parametrize("window", [0, 1, 100])
@pytest.mark.parametrize("sink_mode,dtype", [("head", "bf16"), ("smooth", "f16"), ("none", "bf16")])
def test_split_ragged_small(pkg, num_splits, window, sink_mode, dtype):
    """Ragged batch with prefixes; 16 splits leave most short units' splits
    empty."""
    b = W.make_batch([0, 400, 3, 1500], [200, 77, 129, 40], 16, 2, 64, dtype, window=window,
                     sink_mode=sink_mode, seed=7 * num_splits + window)
    check(pkg, b, num_splits)


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("window", [0, 100])
def test_split_head_dims(pkg, d, window):
    b = W.make_batch([300, 0], [90, 200], 16, 2, d, "bf16", window=window, sink_mode="head",
                     seed=d + window)
    check(pkg, b, 4)


@pytest.mark.parametrize("d,dtype,sink_mode", [(128, "f16", "smooth"), (256, "bf16", "head")])
@pytest.mark.parametrize("num_splits", [7, 16])
@pytest.mark.parametrize("window", [0, 37])
def test_split_wide_heads_many_splits(pkg, d, dtype, sink_mode, num_splits, window):
    """Head dims whose merge spreads a row over 8 or 16 column groups, with
    more splits than some units have tiles (empty splits)."""
    b = W.make_batch([900, 0, 64], [40, 150, 9], 16, 4, d, dtype, window=window,
                     sink_mode=sink_mode, seed=d + num_splits + window)
    check(pkg, b, num_splits)


def test_split_short_chunk_long_prefix_auto(pkg):
    """The case split-KV exists for: a 48-query chunk over a 5000-token prefix
    (24 units on a GPU with hundreds of CTA slots)."""
    b = W.make_batch([5000], [48], 64, 8, 64, "bf16", window=0, sink_mode="head", seed=11)
    used, nbytes = pkg.splitkv_workspace(b.num_seqs, b.total_q, b.max_seqlen_q, b.hq, b.hkv,
                                         b.d, "bf16", b.window, 0)
    assert used > 1 and nbytes > 0
    check(pkg, b, 0, label="auto split")


def test_split_long_window_chunk(pkg):
    b = W.make_batch([6000, 2000], [64, 30], 64, 8, 64, "bf16", window=128, sink_mode="head",
                     seed=12)
    check(pkg, b, 8)


def test_split_two_query_tiles(pkg):
    b = W.make_batch([700, 0], [300, 257], 16, 2, 64, "bf16", window=0, sink_mode="smooth",
                     seed=13)
    pkg.force_q_tiles(2)
    try:
        check(pkg, b, 3, label="two query tiles, 3 splits")
    finally:
        pkg.force_q_tiles(0)


def test_split_one_is_the_unsplit_kernel_bitwise(pkg):
    b = W.make_batch([100, 0], [300, 65], 16, 2, 64, "bf16", window=0, sink_mode="head", seed=14)
    dev = b.to("cuda")
    a_out, a_lse = pkg.prefill(dev)
    s_out, s_lse = pkg.prefill_splitkv(dev, num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(a_out, s_out) and torch.equal(a_lse, s_lse)


def test_split_matches_unsplit_and_is_deterministic(pkg):
    b = W.make_batch([3000], [128], 64, 8, 64, "bf16", window=0, sink_mode="head", seed=15)
    dev = b.to("cuda")
    ref_out, ref_lse = pkg.prefill(dev)
    o1, l1 = pkg.prefill_splitkv(dev, num_splits=5)
    o2, l2 = pkg.prefill_splitkv(dev, num_splits=5)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    rel = float((o1.float() - ref_out.float()).norm() / ref_out.float().norm())
    assert rel < 3e-3, rel
    assert float((l1 - ref_lse).abs().max()) < 1e-3


def test_split_chunked_prefix_full_size_sampled(pkg):
    full = W.chunked_prefix(num_seqs=2, prefix=8192, extend=512, window=0, seed=16)
    rows = sample_rows(full, per_seq=24, seed=17)
    check(pkg, full, 0, rows=rows, label="chunked prefix, auto split")


def test_split_workspace_checks(pkg):
    b = W.make_batch([2000], [32], 16, 2, 64, "bf16", window=0, sink_mode="head", seed=18)
    dev = b.to("cuda")
    used, nbytes = pkg.splitkv_workspace(1, 32, 32, 16, 2, 64, "bf16", 0, 4)
    assert used == 4 and nbytes > 0
    small = torch.empty(nbytes - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.GQAError):
        pkg.prefill_splitkv(dev, num_splits=4, workspace=small)
    with pytest.raises(pkg.GQAError):
        pkg.gqa_flash_prefill_splitkv(dev.q, dev.k, dev.v, dev.cu_seqlens_q, dev.prefix_lens,
                                      dev.kv_indptr, dev.scale, None, num_splits=4,
                                      out=torch.empty_like(dev.q))
    with pytest.raises(pkg.GQAError):  # more than 16 splits
        pkg.splitkv_workspace(1, 32, 32, 16, 2, 64, "bf16", 0, 17)
    assert pkg.splitkv_workspace(1, 32, 32, 16, 2, 64, "bf16", 0, 1) == (1, 0)


def test_split_bad_metadata_writes_nothing(pkg):
    b = W.make_batch([10], [40], 8, 2, 64, "bf16", window=0, sink_mode="none", seed=19)
    dev = b.to("cuda")
    bad_kv = dev.kv_indptr.clone()
    bad_kv[1] += 3  # kv span no longer prefix + extend
    out = torch.full_like(dev.q, 7.0)
    used, nbytes = pkg.splitkv_workspace(1, 40, 40, 8, 2, 64, "bf16", 0, 4)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    pkg.gqa_flash_prefill_splitkv(dev.q, dev.k, dev.v, dev.cu_seqlens_q, dev.prefix_lens,
                                  bad_kv, dev.scale, ws, num_splits=4, out=out)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == pkg.GQA_DEV_BAD_METADATA
    assert bool((out == 7.0).all())


def test_split_decode_few_sequences_long_prefix(pkg):
    """Decode of a few sequences over long full-attention prefixes: a handful
    of units, so the library splits."""
    b = W.decode(num_seqs=4, min_prefix=4000, max_prefix=6000, window=0, sink_mode="head",
                 seed=43)
    used, _ = pkg.splitkv_workspace(b.num_seqs, b.total_q, b.max_seqlen_q, b.hq, b.hkv, b.d,
                                    "bf16", 0, 0)
    assert used > 1
    check(pkg, b, 0, label="decode, auto split")
