"""The balanced split (num_splits = GQA_SPLITS_BALANCED) through the C ABI:
equal shares of all key tiles per resident CTA, units cut by a share boundary
merged in-kernel by log-sum-exp (the partial-result combine of SGLang PR
#34468's context-parallel path), compared with the CPU oracle on the same
seeded inputs."""
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
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return pkg


def run_balanced(pkg, dev, workspace=None):
    out = torch.full_like(dev.q, float("nan"))
    lse = torch.full(dev.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    pkg.prefill_splitkv(dev, num_splits=pkg.SPLITS_BALANCED, workspace=workspace, out=out,
                        lse=lse)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    return out, lse


def check(pkg, b, rows=None, label=""):
    out, lse = run_balanced(pkg, b.to("cuda"))
    ref, ref_lse = run_oracle(b, rows=rows)
    return compare(out.cpu(), lse.cpu(), ref, ref_lse, rows=rows,
                   label=label or f"balanced {b.name}")


def test_workspace_query(pkg):
    used, nbytes = pkg.splitkv_workspace(1, 512, 512, 64, 8, 64, "bf16", 0,
                                         pkg.SPLITS_BALANCED)
    assert used == pkg.SPLITS_BALANCED
    assert nbytes > 0


@pytest.mark.parametrize("window", [0, 1, 15, 100, 129])
@pytest.mark.parametrize("sink_mode,dtype", [("head", "bf16"), ("smooth", "f16"), ("none", "bf16")])
def test_balanced_ragged_small(pkg, window, sink_mode, dtype):
    """Few units on hundreds of CTAs: most units run as many pieces, some
    pieces hold only window-edge tiles (rows with no key in the piece)."""
    b = W.make_batch([0, 400, 3, 1500], [200, 77, 129, 40], 16, 2, 64, dtype, window=window,
                     sink_mode=sink_mode, seed=9100 + window)
    check(pkg, b)


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("window", [0, 100])
@pytest.mark.parametrize("sink_mode,dtype", [("head", "bf16"), ("smooth", "f16")])
def test_balanced_head_dims(pkg, d, window, sink_mode, dtype):
    b = W.make_batch([300, 0, 2000], [90, 200, 33], 16, 2, d, dtype, window=window,
                     sink_mode=sink_mode, seed=9200 + d + window)
    check(pkg, b)


@pytest.mark.parametrize("hq,hkv", [(64, 8), (32, 4), (8, 8)])
def test_balanced_group_sizes(pkg, hq, hkv):
    b = W.make_batch([700, 0], [333, 129], hq, hkv, 64, "bf16", window=0, sink_mode="head",
                     seed=9300 + hq)
    check(pkg, b)


@pytest.mark.parametrize("window", [0, 128])
def test_balanced_oss20b_chunk(pkg, window):
    """The 16k prefill's last chunk: 512 queries over 15,872 cached tokens,
    64/8 heads, d 64: 256 units on the resident CTAs, each cut in two or three
    pieces.  Sampled rows against the oracle."""
    b = W.make_batch([15872], [512], 64, 8, 64, "bf16", window=window, sink_mode="head",
                     seed=9400 + window)
    rows = sample_rows(b, per_seq=64)
    check(pkg, b, rows=rows, label=f"balanced oss20b chunk31 w{window}")


def test_balanced_many_units(pkg):
    """More units than CTAs (several pieces per share, most of them whole
    units), ragged lengths and prefixes."""
    b = W.make_batch([0, 5000, 100, 0, 2500], [3000, 700, 1800, 9, 1200], 32, 4, 64, "bf16",
                     window=0, sink_mode="head", seed=9500)
    rows = sample_rows(b, per_seq=48)
    check(pkg, b, rows=rows)


def test_balanced_matches_unsplit_closely(pkg):
    """Against the unsplit kernel on a full-causal chunk: the two differ only
    by the rounding of the merge (fp32 partials, one 16-bit rounding)."""
    b = W.make_batch([4096], [512], 64, 8, 64, "f16", window=0, sink_mode="head", seed=9600)
    dev = b.to("cuda")
    out, lse = run_balanced(pkg, dev)
    ref_out, ref_lse = pkg.prefill(dev)
    torch.cuda.synchronize()
    diff = (out.float() - ref_out.float()).abs().max().item()
    assert diff <= 2e-3, diff
    assert (lse - ref_lse).abs().max().item() <= 1e-4


def test_balanced_run_to_run_bitwise(pkg):
    """Whichever piece of a cut unit finishes last, the merge sums the pieces
    in share order: repeated calls give identical bits."""
    b = W.make_batch([15872], [512], 64, 8, 64, "bf16", window=0, sink_mode="head", seed=9700)
    dev = b.to("cuda")
    first = run_balanced(pkg, dev)
    for _ in range(3):
        again = run_balanced(pkg, dev)
        assert torch.equal(first[0].view(torch.int16), again[0].view(torch.int16))
        assert torch.equal(first[1], again[1])


def test_balanced_garbage_workspace(pkg):
    """The workspace needs no initialisation: filled with random bytes, and
    with the count words an earlier launch left, the result is the same."""
    b = W.make_batch([2000, 100], [300, 500], 64, 8, 64, "bf16", window=0, sink_mode="head",
                     seed=9800)
    dev = b.to("cuda")
    _, nbytes = pkg.splitkv_workspace(b.num_seqs, b.total_q, b.max_seqlen_q, b.hq, b.hkv, b.d,
                                      "bf16", b.window, pkg.SPLITS_BALANCED)
    clean = run_balanced(pkg, dev)
    g = torch.Generator(device="cuda").manual_seed(5)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
    dirty = run_balanced(pkg, dev, workspace=ws)
    assert torch.equal(clean[0].view(torch.int16), dirty[0].view(torch.int16))
    again = run_balanced(pkg, dev, workspace=ws)  # the words the first call left behind
    assert torch.equal(clean[0].view(torch.int16), again[0].view(torch.int16))


def test_balanced_graph_replay(pkg):
    """A captured call replays with the same launch tag: each merging warp
    zeroes its count, so every replay starts from zero and matches eager."""
    b = W.make_batch([3000], [512], 64, 8, 64, "bf16", window=0, sink_mode="head", seed=9900)
    dev = b.to("cuda")
    eager = run_balanced(pkg, dev)
    _, nbytes = pkg.splitkv_workspace(b.num_seqs, b.total_q, b.max_seqlen_q, b.hq, b.hkv, b.d,
                                      "bf16", b.window, pkg.SPLITS_BALANCED)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev.q)
    lse = torch.empty(dev.q.shape[:2], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # warm-up (first-call set-up stays outside the capture)
        pkg.prefill_splitkv(dev, num_splits=pkg.SPLITS_BALANCED, workspace=ws, out=out, lse=lse,
                            stream=s.cuda_stream)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pkg.prefill_splitkv(dev, num_splits=pkg.SPLITS_BALANCED, workspace=ws, out=out, lse=lse,
                            stream=s.cuda_stream)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pkg.get_device_status() == 0
        assert torch.equal(out.view(torch.int16), eager[0].view(torch.int16))
        assert torch.equal(lse, eager[1])


def test_balanced_noalloc(pkg):
    """The balanced split through the no-alloc entry point (library scratch)."""
    b = W.make_batch([1500, 0], [256, 700], 64, 8, 64, "bf16", window=128, sink_mode="head",
                     seed=9950)
    dev = b.to("cuda")
    eager = run_balanced(pkg, dev)
    out = torch.full_like(dev.q, float("nan"))
    lse = torch.full(dev.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    pkg.prefill_splitkv_noalloc(dev, num_splits=pkg.SPLITS_BALANCED, out=out, lse=lse)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    assert torch.equal(out.view(torch.int16), eager[0].view(torch.int16))


def test_balanced_many_sequences(pkg):
    """More sequences than one launch takes (600: two launches of the same
    workspace, each with its own launch tag)."""
    rng = np.random.default_rng(3)
    pre = rng.integers(0, 300, size=600).tolist()
    ext = rng.integers(1, 40, size=600).tolist()
    b = W.make_batch(pre, ext, 16, 2, 64, "bf16", window=0, sink_mode="head", seed=9990)
    rows = np.sort(rng.choice(b.total_q, size=400, replace=False))
    check(pkg, b, rows=rows, label="balanced 600 sequences")
