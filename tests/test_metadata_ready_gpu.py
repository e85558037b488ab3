"""GQA_FLAG_METADATA_READY (gqa_prefill_set_call_flags): with the flag the
kernels read and check the metadata before waiting on the previous kernel in
the stream.  The metadata below is uploaded before any call, so the flag's
guarantee holds; every kind of call must give bit-identical results with and
without it, back to back on one stream (programmatic dependent launch)."""
import numpy as np
import pytest
import torch

from gqa_flash_attention_prefill_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__
    __graft_entry__.build()
    import gqa_flash_attention_prefill_gb300 as pkg
    pkg.load()
    pkg.force_block_n(0)
    pkg.force_q_tiles(0)
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield pkg
    pkg.set_call_flags(0)


def _batches():
    rng = np.random.default_rng(11)
    pre = rng.integers(0, 3000, size=600).tolist()
    ext = rng.integers(1, 24, size=600).tolist()
    return [
        W.make_batch([0, 400, 3, 1500], [200, 77, 129, 40], 16, 2, 64, "bf16", window=0,
                     sink_mode="head", seed=1),
        W.make_batch([0, 400, 3, 1500], [200, 77, 129, 40], 16, 2, 64, "f16", window=100,
                     sink_mode="smooth", seed=2),
        W.make_batch([2000, 0], [512, 300], 64, 8, 128, "bf16", window=0, sink_mode="head",
                     seed=3),
        W.make_batch(pre, ext, 16, 2, 64, "bf16", window=128, sink_mode="head", seed=4),
    ]


def _run_all(pkg, devs, kinds):
    outs = []
    for dev in devs:
        for kind in kinds:
            out = torch.full_like(dev.q, float("nan"))
            lse = torch.full(dev.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
            if kind == "plain":
                pkg.prefill(dev, out=out, lse=lse)
            elif kind == "balanced":
                pkg.prefill_splitkv(dev, num_splits=pkg.SPLITS_BALANCED, out=out, lse=lse)
            elif kind == "split4":
                pkg.prefill_splitkv(dev, num_splits=4, out=out, lse=lse)
            outs.append((out, lse))
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    return outs


def test_metadata_ready_is_bit_identical(pkg):
    devs = [b.to("cuda") for b in _batches()]
    kinds = ["plain", "balanced", "split4"]
    pkg.set_call_flags(0)
    ref = _run_all(pkg, devs, kinds)
    pkg.set_call_flags(pkg.FLAG_METADATA_READY)
    try:
        for _ in range(2):
            got = _run_all(pkg, devs, kinds)
            for (o, l), (ro, rl) in zip(got, ref):
                assert torch.equal(o.view(torch.int16), ro.view(torch.int16))
                assert torch.equal(l, rl)
    finally:
        pkg.set_call_flags(0)


def test_metadata_ready_paged_and_masked(pkg):
    b = W.make_batch([300, 0, 900], [129, 64, 40], 16, 2, 64, "bf16", window=64,
                     sink_mode="head", seed=5)
    pb = W.paged(b, 16, seed=1).to("cuda")
    keep = W.random_custom_mask(b.extend_lens, density=0.6, seed=2)
    words, indptr = W.pack_custom_mask(keep)
    dev = b.to("cuda")
    words, indptr = words.cuda(), indptr.cuda()

    def both():
        o1, l1 = pkg.prefill_paged(pb)
        o2, l2 = pkg.prefill_masked(dev, words, indptr)
        torch.cuda.synchronize()
        assert pkg.get_device_status() == 0
        return o1, l1, o2, l2

    pkg.set_call_flags(0)
    ref = both()
    pkg.set_call_flags(pkg.FLAG_METADATA_READY)
    try:
        got = both()
    finally:
        pkg.set_call_flags(0)
    for a, r in zip(got, ref):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           r.view(torch.int32) if r.dtype == torch.float32 else r.view(torch.int16))


def test_metadata_ready_bad_metadata_still_reported(pkg):
    """Bad metadata read before the wait is still reported through the status
    word, and the output is left untouched."""
    b = W.make_batch([5, 6], [20, 40], 8, 2, 64, "bf16", window=0, sink_mode="none", seed=6)
    dev = b.to("cuda")
    bad = dev.kv_indptr.clone()
    bad[1] += 1  # sequence 0 claims one key row too many
    out = torch.full_like(dev.q, 7.0)
    pkg.set_call_flags(pkg.FLAG_METADATA_READY)
    try:
        pkg.gqa_flash_prefill(dev.q, dev.k, dev.v, dev.cu_seqlens_q, dev.prefix_lens, bad,
                              dev.scale, out=out)
        torch.cuda.synchronize()
    finally:
        pkg.set_call_flags(0)
    assert pkg.get_device_status() == pkg.GQA_DEV_BAD_METADATA
    assert bool((out == 7.0).all())
