"""Runtime behaviour on the GPU: the bounded-wait self-test, the configuration
cache's tuning sweep, CUDA-graph capture of calls, and non-default streams."""
import pytest
import torch

from gqa_flash_attention_prefill_gb300 import workloads as W
from parity_util import compare, run_gpu, run_oracle

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


def test_bounded_wait_times_out_and_context_survives(pkg):
    assert pkg.get_device_status() == 0
    assert pkg.selftest_timeout(50) == pkg.GQA_DEV_TIMEOUT
    assert pkg.get_device_status() == 0  # read-and-clear
    b = W.make_batch([5], [40], 8, 2, 64, "bf16", window=9, sink_mode="head", seed=3)
    out, lse = run_gpu(pkg, b)
    ref, ref_lse = run_oracle(b)
    compare(out, lse, ref, ref_lse, label="after timeout self-test")


def test_tuning_sweep_fills_the_cache(pkg):
    pkg.clear_config_cache()
    pkg.set_tuning(True)
    try:
        b = W.make_batch([0], [1024], 64, 8, 64, "bf16", window=0, sink_mode="head", seed=8)
        assert pkg.config_block_n(b.total_q, b.max_seqlen_q, 64, 8, 64, "bf16", 0) == (0, 0, False)
        out, lse = run_gpu(pkg, b)
        bn, qt, tuned = pkg.config_block_n(b.total_q, b.max_seqlen_q, 64, 8, 64, "bf16", 0)
        assert tuned and bn in (64, 96, 128) and qt in (1, 2)
        ref, ref_lse = run_oracle(b, rows=list(range(0, 1024, 37)))
        rows = list(range(0, 1024, 37))
        compare(out, lse, ref, ref_lse, rows=rows, label="tuned")
        # the key ignores the KV length: a longer prefix reuses the entry
        b2 = W.make_batch([3000], [1000], 64, 8, 64, "bf16", window=0, sink_mode="head", seed=9)
        assert pkg.config_block_n(b2.total_q, b2.max_seqlen_q, 64, 8, 64, "bf16", 0) == \
            (bn, qt, True)
    finally:
        pkg.set_tuning(False)
        pkg.clear_config_cache()


def test_cuda_graph_capture_replays_identically(pkg):
    layers = [b.to("cuda") for b in W.layer_pair(seq=512, seed=21)]
    outs = [torch.empty_like(b.q) for b in layers]
    lses = [torch.empty(b.q.shape[:2], dtype=torch.float32, device="cuda") for b in layers]
    for b, o, l in zip(layers, outs, lses):  # direct calls (also fills the config cache)
        pkg.prefill(b, out=o, lse=l)
    torch.cuda.synchronize()
    direct = [o.clone() for o in outs]
    for o in outs:
        o.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for b, o, l in zip(layers, outs, lses):
            pkg.prefill(b, out=o, lse=l, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    for o, d in zip(outs, direct):
        assert torch.equal(o.view(torch.int16), d.view(torch.int16))


def test_non_default_stream(pkg):
    b = W.make_batch([7, 0], [90, 33], 16, 2, 64, "f16", window=20, sink_mode="smooth", seed=4)
    dev = b.to("cuda")
    out = torch.full_like(dev.q, float("nan"))
    lse = torch.empty(dev.q.shape[:2], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkg.prefill(dev, out=out, lse=lse, stream=s)
    s.synchronize()
    ref, ref_lse = run_oracle(b)
    compare(out.cpu(), lse.cpu(), ref, ref_lse, label="side stream")


def test_stream_status_reads_one_stream_only(pkg):
    """gqa_prefill_get_stream_status waits for its own stream only: a bad-
    metadata call on a side stream is reported while another stream is still
    busy with a long kernel, and the read clears the bit."""
    import time
    assert pkg.get_device_status() == 0
    b = W.make_batch([5, 6], [20, 30], 8, 2, 64, "bf16", window=0, sink_mode="none", seed=3)
    dev = b.to("cuda")
    bad_kv = dev.kv_indptr.clone()
    bad_kv[1] += 1
    out = torch.full_like(dev.q, 7.0)
    torch.cuda.synchronize()
    busy, side = torch.cuda.Stream(), torch.cuda.Stream()
    # load everything the timed part launches (kernels load at first use)
    with torch.cuda.stream(side):
        pkg.gqa_flash_prefill(dev.q, dev.k, dev.v, dev.cu_seqlens_q, dev.prefix_lens,
                              dev.kv_indptr, dev.scale, out=torch.empty_like(dev.q), stream=side)
    assert pkg.get_stream_status(side) == 0
    with torch.cuda.stream(busy):
        torch.cuda._sleep(3_000_000_000)  # about 1.5 s of spinning at 2 GHz
    with torch.cuda.stream(side):
        pkg.gqa_flash_prefill(dev.q, dev.k, dev.v, dev.cu_seqlens_q, dev.prefix_lens, bad_kv,
                              dev.scale, out=out, stream=side)
    t0 = time.perf_counter()
    st = pkg.get_stream_status(side)
    waited = time.perf_counter() - t0
    assert st == pkg.GQA_DEV_BAD_METADATA
    assert waited < 0.75, waited  # returned long before the busy stream's kernel ended
    assert not busy.query()
    busy.synchronize()
    assert pkg.get_stream_status(side) == 0  # cleared by the read
    assert bool((out == 7.0).all())

