"""GPU parity of gqa_flash_prefill_masked: the custom mask ANDed with the
causal and window conditions (SGLang PR #34468 "gfx950 SWA prefix trim":
the custom mask with a sliding window, the EAGLE target-verify route),
against the oracle's masked definition."""
import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_prefill_gb300 import workloads as W
from parity_util import compare

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


def _run(pkg, b, keep, poison=True):
    words, indptr = W.pack_custom_mask(keep)
    dev = b.to("cuda")
    out = torch.empty_like(dev.q)
    lse = torch.empty(dev.q.shape[:2], dtype=torch.float32, device="cuda")
    if poison:
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
    pkg.prefill_masked(dev, words.cuda(), indptr.cuda(), out=out, lse=lse)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    return out.cpu(), lse.cpu(), words, indptr


def _oracle(b, words, indptr, rows=None):
    return oracle.prefill(b.q, b.k, b.v, b.cu_seqlens_q, b.prefix_lens, b.kv_indptr, b.scale,
                          b.window, sinks=b.sinks, smooth_softmax=b.smooth, rows=rows,
                          custom_mask=words, mask_indptr=indptr)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("window", [0, 1, 15, 64, 100, 129])
@pytest.mark.parametrize("sink_mode,dtype", [("head", "bf16"), ("smooth", "f16"), ("none", "bf16")])
def test_masked_ragged_against_oracle(pkg, d, window, sink_mode, dtype):
    """Ragged sequences whose extends straddle 32-bit mask words and key
    tiles, over cached prefixes; random masks with the diagonal kept."""
    b = W.make_batch([0, 37, 200, 5], [1, 150, 77, 33], 16, 2, d, dtype, window=window,
                     sink_mode=sink_mode, seed=3000 + d + window)
    keep = W.random_custom_mask(b.extend_lens, density=0.6, seed=window + d)
    out, lse, words, indptr = _run(pkg, b, keep)
    ref, ref_lse = _oracle(b, words, indptr)
    compare(out, lse, ref, ref_lse, label=f"masked d{d} w{window} {sink_mode} {dtype}")


def test_masked_rows_with_no_key(pkg):
    """Rows whose mask keeps nothing and that have no prefix get out = 0 and
    lse = -inf; the other rows match the oracle."""
    b = W.make_batch([0, 0, 64], [40, 70, 90], 16, 2, 64, "bf16", window=0, sink_mode="head",
                     seed=3100)
    keep = W.random_custom_mask(b.extend_lens, density=0.3, seed=7, diagonal=False)
    keep[0][:5] = False
    keep[1][10] = False
    out, lse, words, indptr = _run(pkg, b, keep)
    ref, ref_lse = _oracle(b, words, indptr)
    assert np.all(out[:5].float().numpy() == 0) and np.all(np.isneginf(lse[:5].numpy()))
    assert np.all(np.isneginf(ref_lse[:5]))
    finite = np.isfinite(ref_lse).all(axis=1)
    compare(out[finite], lse[finite], ref[finite], ref_lse[finite], label="masked, empty rows")


def test_all_ones_mask_equals_unmasked_kernel(pkg):
    """An all-ones mask keeps every key the causal/window mask keeps: the
    masked kernel's output is bit-identical to gqa_flash_prefill's."""
    for window in (0, 128):
        b = W.make_batch([300, 0, 4000], [257, 129, 64], 64, 8, 64, "bf16", window=window,
                         sink_mode="head", seed=3200 + window)
        keep = [np.ones((e, e), dtype=bool) for e in b.extend_lens]
        out, lse, _, _ = _run(pkg, b, keep)
        dev = b.to("cuda")
        ref_out, ref_lse = pkg.prefill(dev)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.cpu().view(torch.int16))
        assert torch.equal(lse, ref_lse.cpu())


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("window", [0, 20, 100])
def test_masked_counting_probe_exact_key_sets(pkg, dtype, window):
    """q = 0 and v[j, c] = [j mod 64 == c]: lse = ln(n) and out * n count the
    kept keys of each residue class, so every row's key set under the custom
    mask is recovered exactly."""
    b = W.make_batch([0, 300, 1000, 63], [200, 129, 64, 70], 16, 2, 64, dtype, window=window,
                     sink_mode="none", seed=window + 1)
    b.q.zero_()
    j = torch.arange(b.total_kv) - torch.repeat_interleave(b.kv_indptr[:-1],
                                                         torch.diff(b.kv_indptr))
    b.v.zero_()
    b.v[torch.arange(b.total_kv), :, j % 64] = 1.0
    keep = W.random_custom_mask(b.extend_lens, density=0.5, seed=window + 5)
    out, lse, _, _ = _run(pkg, b, keep)
    n = torch.exp(lse.double()).round().long()
    counts = (out.double() * n[..., None]).round().long()
    cu, pre = b.cu_seqlens_q.tolist(), b.prefix_lens.tolist()
    for s in range(b.num_seqs):
        for i in range(cu[s + 1] - cu[s]):
            pos = pre[s] + i
            lo = 0 if window <= 0 else max(0, pos - window + 1)
            keys = [jj for jj in range(lo, pos + 1)
                    if jj < pre[s] or keep[s][i, jj - pre[s]]]
            want = torch.bincount(torch.tensor(keys) % 64, minlength=64)
            row = cu[s] + i
            assert bool((n[row] == len(keys)).all()), (s, i)
            assert bool((counts[row] == want).all()), (s, i)


def test_tree_verify_over_long_prefix_sampled(pkg):
    """The target-verify shape: 8 sequences with 8192 cached tokens each and
    64 draft tokens whose mask is a random tree (each token sees its
    ancestors), window 128 and full attention, in both KV layouts."""
    rng = np.random.default_rng(5)
    keep = []
    for _ in range(8):
        parent = [-1] + [int(rng.integers(0, t)) for t in range(1, 64)]
        m = np.zeros((64, 64), dtype=bool)
        for t in range(64):
            a = t
            while a >= 0:
                m[t, a] = True
                a = parent[a]
        keep.append(m)
    for window in (128, 0):
        full = W.make_batch([8192] * 8, [64] * 8, 64, 8, 64, "bf16", window=window,
                            sink_mode="head", seed=3300 + window)
        layouts = [full] + ([W.window_bounded(full, window)] if window > 0 else [])
        words, indptr = W.pack_custom_mask(keep)
        rows = np.arange(0, full.total_q, 3)
        ref, ref_lse = _oracle(full, words, indptr, rows=rows)
        for b in layouts:
            out, lse, _, _ = _run(pkg, b, keep)
            compare(out, lse, ref, ref_lse, rows=rows, label=f"tree verify w{window} {b.name}")


def test_masked_metadata_checked(pkg):
    """A mask_indptr whose spans do not match E * ceil(E / 32) raises
    GQA_DEV_BAD_METADATA and leaves the output untouched."""
    b = W.make_batch([5, 6], [20, 40], 8, 2, 64, "bf16", window=0, sink_mode="none", seed=3400)
    keep = W.random_custom_mask(b.extend_lens, seed=1)
    words, indptr = W.pack_custom_mask(keep)
    bad = indptr.clone()
    bad[1] -= 1
    dev = b.to("cuda")
    out = torch.full_like(dev.q, 7.0)
    pkg.gqa_flash_prefill_masked(dev.q, dev.k, dev.v, dev.cu_seqlens_q, dev.prefix_lens,
                                 dev.kv_indptr, dev.scale, words.cuda(), bad.cuda(), out=out)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == pkg.GQA_DEV_BAD_METADATA
    assert bool((out == 7.0).all())
