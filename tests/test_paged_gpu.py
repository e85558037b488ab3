"""Paged KV through the C ABI: K/V in a shuffled page pool addressed by a
page table.  Same keys in the same order as the contiguous layout, so the
result must equal the contiguous kernel's bit for bit, and the oracle's within
the parity tolerance."""
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


def run_paged(pkg, pb_cpu):
    pb = pb_cpu.to("cuda")
    out = torch.full_like(pb.batch.q, float("nan"))
    lse = torch.full(pb.batch.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    pkg.prefill_paged(pb, out=out, lse=lse)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("page_size", [8, 16, 64, 128, 256])
@pytest.mark.parametrize("window", [0, 100])
@pytest.mark.parametrize("sink_mode,dtype", [("head", "bf16"), ("smooth", "f16")])
def test_paged_equals_contiguous_bitwise(pkg, page_size, window, sink_mode, dtype):
    b = W.make_batch([0, 300, 1000, 37], [200, 129, 64, 300], 16, 2, 64, dtype, window=window,
                     sink_mode=sink_mode, seed=page_size + window)
    c_out, c_lse = run_gpu(pkg, b)
    p_out, p_lse = run_paged(pkg, W.paged(b, page_size, seed=page_size))
    assert torch.equal(c_out, p_out) and torch.equal(c_lse, p_lse)


@pytest.mark.parametrize("d", [128, 256])
def test_paged_head_dims_against_oracle(pkg, d):
    b = W.make_batch([500, 0], [100, 140], 16, 2, d, "bf16", window=64, sink_mode="head",
                     seed=d)
    out, lse = run_paged(pkg, W.paged(b, 32, seed=d))
    ref, ref_lse = run_oracle(b)
    compare(out, lse, ref, ref_lse, label=f"paged d{d}")


def test_paged_decode_window_bounded_table(pkg):
    """A decode step whose page table holds only each sequence's last
    min(prefix, window) prefix keys (a window-bounded table) gives the
    full-prefix result."""
    full = W.decode(num_seqs=24, min_prefix=0, max_prefix=4000, window=128, seed=50)
    bounded = W.window_bounded(full, 128)
    out, lse = run_paged(pkg, W.paged(bounded, 16, seed=51))
    ref, ref_lse = run_oracle(full)
    compare(out, lse, ref, ref_lse, label="paged decode, window-bounded table")


def test_paged_page_count_mismatch_writes_nothing(pkg):
    b = W.make_batch([100], [60], 8, 2, 64, "bf16", window=0, sink_mode="none", seed=52)
    pb = W.paged(b, 16, seed=52).to("cuda")
    bad_indptr = pb.page_indptr.clone()
    bad_indptr[1] -= 1  # one page short of ceil((P + E) / page_size)
    out = torch.full_like(pb.batch.q, 7.0)
    pkg.gqa_flash_prefill_paged(pb.batch.q, pb.k_pages, pb.v_pages, pb.batch.cu_seqlens_q,
                                pb.batch.prefix_lens, bad_indptr, pb.page_indices,
                                pb.batch.scale, out=out)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == pkg.GQA_DEV_BAD_METADATA
    assert bool((out == 7.0).all())


def test_paged_page_outside_pool_is_reported(pkg):
    b = W.make_batch([100], [60], 8, 2, 64, "bf16", window=0, sink_mode="none", seed=53)
    pb = W.paged(b, 16, seed=53).to("cuda")
    bad = pb.page_indices.clone()
    bad[2] = pb.k_pages.shape[0] + 5
    out = torch.empty_like(pb.batch.q)
    pkg.gqa_flash_prefill_paged(pb.batch.q, pb.k_pages, pb.v_pages, pb.batch.cu_seqlens_q,
                                pb.batch.prefix_lens, pb.page_indptr, bad, pb.batch.scale,
                                out=out)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == pkg.GQA_DEV_BAD_METADATA


def test_paged_rejects_page_sizes(pkg):
    b = W.make_batch([40], [24], 8, 2, 64, "bf16", window=0, sink_mode="none", seed=54)
    for page_size, code in ((24, -2), (12, -1), (4, -1)):  # 24 tiles no key tile; 12, 4 not x8
        pb = W.paged(b, page_size, seed=54).to("cuda")
        with pytest.raises(pkg.GQAError) as e:
            pkg.prefill_paged(pb)
        assert e.value.code == code, page_size
