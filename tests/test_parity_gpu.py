"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Full outputs on sizes the oracle finishes quickly (several
tiles plus ragged tails); sampled rows at the full workload sizes, in the same
launch configuration the benchmark uses."""
import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_prefill_gb300 import workloads as W
from parity_util import (compare, run_gpu, run_oracle, sample_rows, sub_batch)

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


def _check_full(pkg, batch, label=None):
    out, lse = run_gpu(pkg, batch)
    ref, ref_lse = run_oracle(batch)
    return compare(out, lse, ref, ref_lse, label=label or batch.name)


def _check_sampled(pkg, batch, rows, label=None):
    out, lse = run_gpu(pkg, batch)
    ref, ref_lse = run_oracle(batch, rows=rows)
    return compare(out, lse, ref, ref_lse, rows=rows, label=label or batch.name)


# ------------------------------------------------------------- small, full output

def test_tiny_config(pkg):
    _check_full(pkg, W.tiny(seed=0))


SMALL_WINDOWS = [0, 1, 15, 64, 100, 129]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("window", SMALL_WINDOWS)
@pytest.mark.parametrize("sink_mode", ["none", "head", "smooth"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_small_ragged_grid(pkg, d, window, sink_mode, dtype):
    b = W.make_batch([0, 37, 200, 5], [1, 150, 77, 33], 16, 2, d, dtype,
                     window=window, sink_mode=sink_mode,
                     seed=1000 + d + window * 7 + len(sink_mode))
    _check_full(pkg, b)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (8, 2), (64, 8), (32, 4), (128, 1)])
def test_group_sizes(pkg, hq, hkv):
    b = W.make_batch([3, 130], [70, 129], hq, hkv, 64, "bf16", window=33,
                     sink_mode="head", seed=hq * 31 + hkv)
    _check_full(pkg, b)


@pytest.mark.parametrize("d,block_n", [(64, 64), (64, 96), (64, 128), (128, 64), (128, 128), (256, 64)])
@pytest.mark.parametrize("window", [0, 100])
def test_block_n_variants(pkg, d, block_n, window):
    pkg.force_block_n(block_n)
    try:
        b = W.make_batch([0, 190], [300, 257], 16, 2, d, "bf16", window=window,
                         sink_mode="head", seed=d + block_n + window)
        _check_full(pkg, b, label=f"d{d}/bn{block_n}/w{window}")
    finally:
        pkg.force_block_n(0)


class _Variant:
    """Pins the key-tile size and/or query tiles per unit for a block."""
    def __init__(self, pkg, block_n=0, q_tiles=0):
        self.pkg, self.bn, self.qt = pkg, block_n, q_tiles

    def __enter__(self):
        self.pkg.force_block_n(self.bn)
        self.pkg.force_q_tiles(self.qt)

    def __exit__(self, *exc):
        self.pkg.force_block_n(0)
        self.pkg.force_q_tiles(0)


@pytest.mark.parametrize("d,block_n", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("window", [0, 1, 15, 100, 129])
@pytest.mark.parametrize("sink_mode,dtype", [("head", "bf16"), ("smooth", "f16"), ("none", "bf16")])
def test_two_query_tiles_per_unit(pkg, d, block_n, window, sink_mode, dtype):
    """Two 128-row query tiles walking the same key tiles: ragged sequences
    whose last unit has a partial or an empty second tile."""
    b = W.make_batch([0, 190, 3, 1000], [300, 257, 129, 17], 16, 2, d, dtype, window=window,
                     sink_mode=sink_mode, seed=5 * d + block_n + window)
    with _Variant(pkg, block_n, 2):
        _check_full(pkg, b, label=f"2 tiles d{d}/bn{block_n}/w{window}/{sink_mode}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (64, 8), (128, 1), (16, 16)])
def test_two_query_tiles_group_sizes(pkg, hq, hkv):
    b = W.make_batch([3, 130, 0], [70, 300, 1], hq, hkv, 64, "bf16", window=33,
                     sink_mode="head", seed=hq * 37 + hkv)
    with _Variant(pkg, 0, 2):
        _check_full(pkg, b)


@pytest.mark.parametrize("q_tiles", [1, 2])
def test_layer_pair_small_both_unit_sizes(pkg, q_tiles):
    with _Variant(pkg, 0, q_tiles):
        for b in W.layer_pair(seq=640, seed=4):
            _check_full(pkg, b, label=f"{b.name}/{q_tiles} tiles")


def test_layer_pair_small_full_output(pkg):
    for b in W.layer_pair(seq=640, seed=1):
        _check_full(pkg, b)


def test_chunked_prefix_small_both_layouts(pkg):
    full = W.chunked_prefix(num_seqs=2, prefix=300, extend=200, window=128, seed=2)
    bounded = W.window_bounded(full, 128)
    a_out, a_lse = run_gpu(pkg, full)
    b_out, b_lse = run_gpu(pkg, bounded)
    ref, ref_lse = run_oracle(full)
    compare(a_out, a_lse, ref, ref_lse, label="full-prefix layout")
    compare(b_out, b_lse, ref, ref_lse, label="window-bounded layout")


def test_chunked_equals_one_shot(pkg):
    one = W.make_batch([0], [700], 64, 8, 64, "bf16", window=0, sink_mode="head", seed=5)
    ref_out, ref_lse = run_gpu(pkg, one)
    for a, c in [(0, 130), (130, 131), (131, 512), (512, 700)]:
        chunk = W.Batch(one.q[a:c], one.k[:c], one.v[:c],
                        torch.tensor([0, c - a], dtype=torch.int32),
                        torch.tensor([a], dtype=torch.int32),
                        torch.tensor([0, c], dtype=torch.int32), one.hq, one.hkv,
                        one.d, one.window, one.sinks, one.smooth, one.scale)
        out, lse = run_gpu(pkg, chunk)
        compare(out, lse, ref_out[a:c].double().numpy(), ref_lse[a:c].double().numpy(),
                label=f"chunk {a}:{c}")


def test_padding_rows_untouched_and_empty_sequences(pkg):
    b = W.make_batch([10, 0, 50], [40, 0, 25], 8, 2, 64, "f16", window=20,
                     sink_mode="smooth", seed=77)
    # 9 trailing q rows that belong to no sequence
    pad = torch.randn(9, 8, 64).to(torch.float16)
    padded = W.Batch(torch.cat([b.q, pad]), b.k, b.v, b.cu_seqlens_q, b.prefix_lens,
                     b.kv_indptr, b.hq, b.hkv, b.d, b.window, b.sinks, b.smooth, b.scale)
    out, lse = run_gpu(pkg, padded)
    assert torch.isnan(out[65:].float()).all() and torch.isnan(lse[65:]).all()
    ref, ref_lse = run_oracle(b)
    compare(out[:65], lse[:65], ref, ref_lse, label="padded")


def test_run_to_run_bitwise(pkg):
    b = W.make_batch([100, 0], [333, 129], 64, 8, 64, "bf16", window=128,
                     sink_mode="head", seed=9)
    o1, l1 = run_gpu(pkg, b)
    o2, l2 = run_gpu(pkg, b)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_bad_metadata_is_reported(pkg):
    b = W.make_batch([5, 6], [20, 30], 8, 2, 64, "bf16", window=0, sink_mode="none", seed=3)
    dev = b.to("cuda")
    bad_kv = dev.kv_indptr.clone()
    bad_kv[1] += 1  # spans no longer equal prefix + extend
    out = torch.full_like(dev.q, 7.0)
    pkg.gqa_flash_prefill(dev.q, dev.k, dev.v, dev.cu_seqlens_q, dev.prefix_lens, bad_kv,
                          dev.scale, out=out)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == pkg.GQA_DEV_BAD_METADATA
    assert bool((out == 7.0).all())
    assert pkg.get_device_status() == 0  # cleared by the read


# ------------------------------------------------------------- tile bookkeeping

def _bookkeeping(pkg, batch):
    p = pkg.plan(batch.num_seqs, batch.total_q, batch.max_seqlen_q, batch.hq, batch.hkv,
                 batch.d, batch.dtype_name, batch.window)
    log = torch.full((p["max_units"], 8), -1, dtype=torch.int32, device="cuda")
    run_gpu(pkg, batch, debug_log=log)
    log = log.cpu().numpy()
    used = log[log[:, 0] >= 0]
    want = oracle.tile_census(batch.cu_seqlens_q, batch.prefix_lens, batch.hkv,
                              p["rows_per_unit"], p["block_n"], batch.window)
    got = used[np.lexsort((used[:, 2], used[:, 1], used[:, 0]))][:, :6]
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.array_equal(got, want)
    # every unit ran exactly once, on some CTA, in that CTA's order
    assert len(used) == len(want)
    return p, used


@pytest.mark.parametrize("q_tiles", [1, 2])
@pytest.mark.parametrize("window", [0, 1, 15, 100, 128, 129, 4096])
def test_bookkeeping_bit_exact_ragged(pkg, window, q_tiles):
    b = W.make_batch([0, 37, 5000, 129, 64], [1, 300, 700, 128, 129], 64, 8, 64, "bf16",
                     window=window, sink_mode="head", seed=window + 1)
    with _Variant(pkg, 0, q_tiles):
        _bookkeeping(pkg, b)


def test_bookkeeping_full_size_layer_pair(pkg):
    for b in W.layer_pair(seq=4096, seed=1):
        _bookkeeping(pkg, b)


def test_window_cost_flat_in_prefix(pkg):
    """Tiles walked per unit stop growing with the prefix once the window is
    filled (hip-ep PR #622 window commit; SGLang PR #34468 commit 1)."""
    per_unit = []
    for prefix in (0, 512, 8192, 16384):
        b = W.make_batch([prefix], [512], 64, 8, 64, "bf16", window=128,
                         sink_mode="head", seed=prefix + 1)
        p, used = _bookkeeping(pkg, b)
        per_unit.append(int(used[:, 4].max()))
    bound = -(-(128 + p["rows_per_unit"] - 1) // p["block_n"]) + 1
    assert max(per_unit) <= bound, (per_unit, bound)
    assert per_unit[1:] == [per_unit[1]] * 3


# ------------------------------------------------------------- full sizes, sampled rows

def test_layer_pair_full_size_sampled(pkg):
    for b in W.layer_pair(seq=4096, seed=1):
        _check_sampled(pkg, b, sample_rows(b, per_seq=160, seed=1))


@pytest.mark.parametrize("layout", ["window-bounded", "full-prefix"])
def test_chunked_prefix_full_size_sampled(pkg, layout):
    full = W.chunked_prefix(num_seqs=8, prefix=8192, extend=8192, window=128, seed=2)
    b = W.window_bounded(full, 128) if layout == "window-bounded" else full
    out, lse = run_gpu(pkg, b)
    seqs = [0, 5]
    sb = sub_batch(b, seqs)
    rows_sb = sample_rows(sb, per_seq=40, seed=3)
    ref, ref_lse = run_oracle(sb, rows=rows_sb)
    cu = b.cu_seqlens_q.tolist()
    # map sub-batch rows back to the full batch's rows
    scu = sb.cu_seqlens_q.tolist()
    back = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])
    compare(out[back], lse[back], ref, ref_lse, rows=rows_sb, label=layout)


@pytest.mark.parametrize("layer", [0, 1])
@pytest.mark.parametrize("chunk", [0, 1, 17, 31])
def test_oss20b_chunks_sampled(pkg, layer, chunk):
    b = W.oss20b_chunk(layer, chunk)
    _check_sampled(pkg, b, sample_rows(b, per_seq=48, seed=chunk))


RAGGED_CELLS = [
    (64, 8, 64, 128, "head", "bf16"),
    (32, 4, 128, 0, "smooth", "f16"),
    (64, 8, 256, 1, "none", "bf16"),
    (32, 4, 64, 4096, "head", "f16"),
    (64, 8, 128, 127, "head", "bf16"),
    (32, 4, 256, 129, "smooth", "bf16"),
]


@pytest.mark.parametrize("hq,hkv,d,window,sink,dtype", RAGGED_CELLS)
def test_ragged_full_size_sampled(pkg, hq, hkv, d, window, sink, dtype):
    b = W.ragged(hq=hq, hkv=hkv, d=d, dtype=dtype, window=window, sink_mode=sink,
                 seed=4)
    out, lse = run_gpu(pkg, b)
    seqs = [0, 7, 15]
    sb = sub_batch(b, seqs)
    rows_sb = sample_rows(sb, per_seq=12, seed=5)
    ref, ref_lse = run_oracle(sb, rows=rows_sb)
    cu = b.cu_seqlens_q.tolist()
    back = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])
    compare(out[back], lse[back], ref, ref_lse, rows=rows_sb, label=b.name)
    # every row of every sequence was written with finite values
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------- exact key sets

@pytest.mark.parametrize("q_tiles", [1, 2])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("window", [0, 1, 15, 64, 100, 129])
def test_counting_probe_exact_key_sets(pkg, dtype, window, q_tiles):
    """q = 0 makes every kept probability exactly 1, so lse = ln(n) and, with
    v[j, c] = [j mod 64 == c], out[c] * n counts the kept keys in each residue
    class: integers recovered exactly pin every row's key set."""
    b = W.make_batch([0, 300, 1000, 63], [200, 129, 64, 70], 16, 2, 64, dtype,
                     window=window, sink_mode="none", seed=window)
    b.q.zero_()
    j = torch.arange(b.total_kv) - torch.repeat_interleave(
        b.kv_indptr[:-1], torch.diff(b.kv_indptr))
    b.v.zero_()
    b.v[torch.arange(b.total_kv), :, j % 64] = 1.0
    with _Variant(pkg, 0, q_tiles):
        out, lse = run_gpu(pkg, b)
    n = torch.exp(lse.double()).round().long()
    counts = (out.double() * n[..., None]).round().long()
    cu, pre = b.cu_seqlens_q.tolist(), b.prefix_lens.tolist()
    for s in range(b.num_seqs):
        for i in range(cu[s + 1] - cu[s]):
            pos = pre[s] + i
            lo = 0 if window <= 0 else max(0, pos - window + 1)
            want_n = pos - lo + 1
            want = torch.bincount(torch.arange(lo, pos + 1) % 64, minlength=64)
            row = cu[s] + i
            assert bool((n[row] == want_n).all()), (s, i, n[row], want_n)
            assert bool((counts[row] == want).all()), (s, i)


# ------------------------------------------------------------- decode (one token per sequence)

@pytest.mark.parametrize("window", [1, 64, 128, 129, 0])
@pytest.mark.parametrize("sink_mode", ["head", "smooth", "none"])
def test_decode_full_output(pkg, window, sink_mode):
    """One new token per sequence over cached prefixes (full-prefix layout)."""
    b = W.decode(num_seqs=24, min_prefix=0, max_prefix=3000, window=window,
                 sink_mode=sink_mode, seed=40 + window)
    _check_full(pkg, b)


def test_decode_layouts_agree(pkg):
    full = W.decode(num_seqs=32, min_prefix=100, max_prefix=5000, window=128, seed=41)
    bounded = W.window_bounded(full, 128)
    a_out, a_lse = run_gpu(pkg, full)
    b_out, b_lse = run_gpu(pkg, bounded)
    ref, ref_lse = run_oracle(full)
    compare(a_out, a_lse, ref, ref_lse, label="decode full-prefix layout")
    compare(b_out, b_lse, ref, ref_lse, label="decode window-bounded layout")


def test_decode_tiles_bounded_by_window(pkg):
    """Each decode unit walks at most ceil(w / BN) + 1 key tiles whatever its
    prefix (bit-exact bookkeeping against the oracle census)."""
    b = W.decode(num_seqs=16, min_prefix=0, max_prefix=20000, window=128, seed=42)
    p, used = _bookkeeping(pkg, b)
    assert int(used[:, 4].max()) <= -(-128 // p["block_n"]) + 1


# ------------------------------------------------------------- the bf16 error budget

def _bf16(x):
    """fp64 -> fp32 -> bf16 (round to nearest even at each step) -> fp64, the
    rounding path of the kernel's fp32 values."""
    return torch.from_numpy(np.ascontiguousarray(x)).float().to(torch.bfloat16).double().numpy()


def _two_roundings_model(batch):
    """The exact attention of a one-sequence batch with the two roundings a
    bf16 kernel must make: the probabilities rounded to bf16 before the
    P.V product (the tensor-core product takes both operands in one 16-bit
    type), and the output rounded to bf16.  The denominator keeps the
    unrounded probabilities (the kernel sums them in fp32).  Test-side only:
    a model of the error, not a reference result."""
    q = batch.q.double().numpy()
    k = batch.k.double().numpy()
    v = batch.v.double().numpy()
    e, hq, d = q.shape
    g = hq // batch.hkv
    p0 = int(batch.prefix_lens[0])
    out = np.empty((e, hq, d))
    pos = p0 + np.arange(e)[:, None]
    j = np.arange(k.shape[0])[None, :]
    keep = j <= pos
    if batch.window > 0:
        keep &= j >= pos - batch.window + 1
    log2e = 1.0 / np.log(2.0)
    for h in range(hq):
        s = (q[:, h, :] @ k[:, h // g, :].T) * batch.scale * log2e
        s = np.where(keep, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp2(s - m)
        den = p.sum(axis=1)
        if batch.sinks is not None:
            den = den + np.exp2(float(batch.sinks[h]) * log2e - m[:, 0])
        out[:, h, :] = (_bf16(p) @ v[:, h // g, :]) / den[:, None]
    return _bf16(out)


def test_bf16_error_is_the_two_roundings(pkg):
    """For bf16 the GPU's relL2 against the oracle is what rounding P and the
    output to bf16 costs: it stays within 10% of the two-roundings model's
    own relL2 (and under the parity bound 1e-3 + qf)."""
    for b in W.layer_pair(seq=512, seed=11):
        out, lse = run_gpu(pkg, b)
        ref, ref_lse = run_oracle(b)
        rel, _, _ = compare(out, lse, ref, ref_lse, label=b.name + " (error budget)")
        model = _two_roundings_model(b)
        e_model = float(np.linalg.norm(model - ref) / np.linalg.norm(ref))
        e_out = float(np.linalg.norm(_bf16(ref) - ref) / np.linalg.norm(ref))
        print(f"{b.name}: GPU relL2 {rel:.3e}; two-roundings model {e_model:.3e}; "
              f"output rounding alone {e_out:.3e}")
        assert rel <= 1.1 * e_model, (rel, e_model)
        assert e_model > e_out  # the P rounding is a real second term


# ------------------------------------------------------------- more sequences than one launch holds

@pytest.mark.parametrize("window", [128, 0])
def test_decode_2048_sequences(pkg, window):
    """A decode step of 2048 sequences (one new token each) runs as four
    launches of 512 sequences; every row is checked against the oracle."""
    gen = torch.Generator().manual_seed(2048 + window)
    pre = torch.randint(0, 400, (2048,), generator=gen).tolist()
    b = W.make_batch(pre, [1] * 2048, 16, 2, 64, "bf16", window=window, sink_mode="head",
                     seed=2048 + window, name=f"decode-2048-w{window}")
    _check_full(pkg, b)


def test_ragged_600_sequences_and_bookkeeping(pkg):
    """600 ragged sequences (two launches, several units per sequence):
    full output against the oracle, and every unit's tile bookkeeping
    bit-exact against the oracle census across both launches."""
    gen = torch.Generator().manual_seed(600)
    pre = torch.randint(0, 300, (600,), generator=gen).tolist()
    ext = torch.randint(1, 40, (600,), generator=gen).tolist()
    b = W.make_batch(pre, ext, 16, 2, 64, "f16", window=50, sink_mode="smooth", seed=600,
                     name="ragged-600")
    _check_full(pkg, b)
    p = pkg.plan(b.num_seqs, b.total_q, b.max_seqlen_q, b.hq, b.hkv, b.d, b.dtype_name,
                 b.window)
    groups = -(-b.num_seqs // 512)
    per_launch = p["max_units"] // groups
    log = torch.full((p["max_units"], 8), -1, dtype=torch.int32, device="cuda")
    run_gpu(pkg, b, debug_log=log)
    log = log.cpu().numpy()
    idx = np.nonzero(log[:, 0] >= 0)[0]
    used = log[idx].copy()
    used[:, 0] += 512 * (idx // per_launch)  # records count b from their launch's first sequence
    want = oracle.tile_census(b.cu_seqlens_q, b.prefix_lens, b.hkv, p["rows_per_unit"],
                              p["block_n"], b.window)
    got = used[np.lexsort((used[:, 2], used[:, 1], used[:, 0]))][:, :6]
    assert np.array_equal(got, want)


def test_splitkv_and_paged_over_600_sequences(pkg):
    """Split-KV (forced 3 splits) and paged KV on a 600-sequence decode step:
    the launch groups share one workspace in stream order."""
    gen = torch.Generator().manual_seed(601)
    pre = torch.randint(0, 500, (600,), generator=gen).tolist()
    b = W.make_batch(pre, [1] * 600, 16, 2, 64, "bf16", window=0, sink_mode="head",
                     seed=601, name="decode-600")
    ref, ref_lse = run_oracle(b)
    dev = b.to("cuda")
    out, lse = pkg.prefill_splitkv(dev, num_splits=3)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    compare(out.cpu(), lse.cpu(), ref, ref_lse, label="split-KV, 600 sequences")
    pb = W.paged(b, 16, seed=3).to("cuda")
    out, lse = pkg.prefill_paged(pb)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    compare(out.cpu(), lse.cpu(), ref, ref_lse, label="paged, 600 sequences")


def _decode_batch_300():
    gen = torch.Generator().manual_seed(300)
    pre = torch.randint(0, 6000, (300,), generator=gen).tolist()
    return W.make_batch(pre, [1] * 300, 16, 2, 64, "bf16", window=0, sink_mode="head", seed=300)


@pytest.mark.parametrize("which", ["ragged6", "decode300"])
def test_units_dealt_costliest_first_across_the_batch(pkg, which):
    """The unit records' (CTA, position) give each unit's place in the deal;
    in that order the sequences come by decreasing cost of their costliest
    unit (ties by index), each sequence's units by decreasing query position,
    and every unit appears once: a 6-sequence ragged prefill and a
    300-sequence decode step with prefixes U[0, 6000)."""
    if which == "ragged6":
        b = W.make_batch([0, 37, 5000, 129, 64, 3000], [1, 300, 700, 128, 129, 2000], 64, 8, 64,
                         "bf16", window=0, sink_mode="head", seed=77)
    else:
        b = _decode_batch_300()
    p, used = _bookkeeping(pkg, b)
    grid = p["grid"]
    cta, k = used[:, 6].astype(np.int64), used[:, 7].astype(np.int64)
    u = k * grid + np.where(k % 2 == 1, grid - 1 - cta, cta)
    assert len(np.unique(u)) == len(u)
    rec = used[np.argsort(u)]
    census = oracle.tile_census(b.cu_seqlens_q, b.prefix_lens, b.hkv, p["rows_per_unit"],
                                p["block_n"], b.window)
    key = {}
    for s in range(b.num_seqs):
        mine = census[census[:, 0] == s]
        key[s] = int(mine[np.argmax(mine[:, 2]), 4])
    seqs = [int(x) for x in rec[:, 0]]
    order = [s for i, s in enumerate(seqs) if i == 0 or s != seqs[i - 1]]
    assert len(order) == len(set(order)), order  # each sequence dealt as one block
    assert order == sorted(order, key=lambda s: (-key[s], s)), (order, key)
    for s in order:
        q0 = rec[rec[:, 0] == s][:, 2]
        assert np.all(np.diff(q0) <= 0)  # KV heads fastest, positions decreasing


# ------------------------------------------------------------- large sizes

def test_long_single_sequence_sampled(pkg):
    """One 32768-token prefill (16384 units at G = 8), full causal: the last
    rows see 32768 keys; sampled rows against the oracle."""
    b = W.make_batch([0], [32768], 64, 8, 64, "bf16", window=0, sink_mode="head", seed=32768,
                     name="single-32k")
    rows = np.array([0, 1, 127, 128, 4095, 16383, 16384, 30000, 32766, 32767], dtype=np.int64)
    _check_sampled(pkg, b, rows)


def test_window_over_a_256k_prefix(pkg):
    """A 512-token chunk over a 262144-token cached prefix, window 128, the
    whole prefix handed over: the kernel's loop floor skips to the window;
    checked against the oracle on the window-bounded layout (the same result,
    an oracle pin), every row."""
    full = W.make_batch([262144], [512], 64, 8, 64, "bf16", window=128, sink_mode="head",
                        seed=262144, name="chunk-over-256k")
    out, lse = run_gpu(pkg, full)
    ref, ref_lse = run_oracle(W.window_bounded(full, 128))
    compare(out, lse, ref, ref_lse, label=full.name)
