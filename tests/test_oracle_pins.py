"""Pins for the CPU oracle: each check ties it to something other than itself
(a library routine, a closed form, brute force, or numbers the pages print).

Every ``pin_*`` function takes the loaded oracle library so the planted-mistake
suite (tests/test_oracle_mutations.py) can run the same checks against edited
copies of the oracle and require that each edit fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_prefill_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _seq_slices(batch):
    cu = batch.cu_seqlens_q.tolist()
    kvp = batch.kv_indptr.tolist()
    pre = batch.prefix_lens.tolist()
    for b in range(batch.num_seqs):
        yield b, cu[b], cu[b + 1], kvp[b], kvp[b + 1], pre[b]


def _library_reference(batch, window):
    """torch float64 softmax attention with a band mask built by tril/triu
    (a library construction, not the oracle's predicate).  A sink is an extra
    score column whose probability mass is dropped after the softmax."""
    g = batch.hq // batch.hkv
    q = batch.q.to(torch.float64)
    k = batch.k.to(torch.float64)
    v = batch.v.to(torch.float64)
    out = torch.zeros_like(q)
    lse = torch.zeros(q.shape[:2], dtype=torch.float64)
    for b, q0, q1, k0, k1, p in _seq_slices(batch):
        e, L = q1 - q0, k1 - k0
        ones = torch.ones(e, L, dtype=torch.bool)
        band = torch.tril(ones, diagonal=p)
        if window > 0:
            band = band & torch.triu(ones, diagonal=p - window + 1)
        for h in range(batch.hq):
            s = batch.scale * q[q0:q1, h] @ k[k0:k1, h // g].T
            s = s.masked_fill(~band, float("-inf"))
            if batch.sinks is not None or batch.smooth:
                x = 0.0 if batch.smooth else float(batch.sinks[h])
                s = torch.cat([s, torch.full((e, 1), x, dtype=torch.float64)], 1)
                pr = torch.softmax(s, dim=1)[:, :L]
            else:
                pr = torch.softmax(s, dim=1)
            out[q0:q1, h] = pr @ v[k0:k1, h // g]
            lse[q0:q1, h] = torch.logsumexp(s, dim=1)
    return out.numpy(), lse.numpy()


def _small_ragged(window, sink_mode, seed=11, hq=4, hkv=2, d=16, dtype="f16"):
    return W.make_batch([0, 37, 5], [23, 9, 40], hq, hkv, d, dtype,
                        window=window, sink_mode=sink_mode, seed=seed)


def _run(lib, batch, window=None, **kw):
    return oracle.prefill(batch.q, batch.k, batch.v, batch.cu_seqlens_q,
                          batch.prefix_lens, batch.kv_indptr, batch.scale,
                          batch.window if window is None else window,
                          sinks=kw.get("sinks", batch.sinks),
                          smooth_softmax=kw.get("smooth", batch.smooth),
                          rows=kw.get("rows"), lib=lib)


# ----------------------------------------------------------------- the pins

def pin_plain_causal_is_library_softmax(lib):
    b = _small_ragged(0, "none")
    out, lse = _run(lib, b)
    ref, ref_lse = _library_reference(b, 0)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def pin_sinks_are_a_dropped_softmax_column(lib):
    b = _small_ragged(0, "head", seed=12)
    out, lse = _run(lib, b)
    ref, ref_lse = _library_reference(b, 0)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def pin_window_is_library_band(lib):
    for w, mode in [(1, "none"), (7, "head"), (16, "smooth"), (30, "head")]:
        b = _small_ragged(w, mode, seed=13 + w)
        out, lse = _run(lib, b)
        ref, ref_lse = _library_reference(b, w)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def pin_window_one_closed_form(lib):
    """window = 1: each row sees only its own key, so with sink s
    out_i = v_i * e^x / (e^x + e^s), x = scale * <q_i, k_i>; without a sink
    out_i = v_i exactly."""
    b = W.make_batch([6, 0], [10, 12], 4, 2, 16, "bf16", window=1,
                     sink_mode="head", seed=21)
    out, _ = _run(lib, b)
    out_ns, _ = _run(lib, b, sinks=None)
    g = b.hq // b.hkv
    for bb, q0, q1, k0, k1, p in _seq_slices(b):
        for i in range(q1 - q0):
            for h in range(b.hq):
                qi = b.q[q0 + i, h].double().numpy()
                ki = b.k[k0 + p + i, h // g].double().numpy()
                vi = b.v[k0 + p + i, h // g].double().numpy()
                x = b.scale * float(qi @ ki)
                s = float(b.sinks[h])
                want = vi * (1.0 / (1.0 + np.exp(s - x)))
                np.testing.assert_allclose(out[q0 + i, h], want, rtol=1e-12, atol=1e-14)
                assert np.array_equal(out_ns[q0 + i, h], vi)


def pin_wide_window_equals_no_window(lib):
    b = _small_ragged(0, "head", seed=31)
    full, lse_full = _run(lib, b, window=0)
    for w in (77, 78, 1000):  # >= P+E of every sequence (max 77)
        wide, lse_wide = _run(lib, b, window=w)
        assert np.array_equal(full, wide) and np.array_equal(lse_full, lse_wide)
    neg, _ = _run(lib, b, window=-5)
    assert np.array_equal(full, neg)


def pin_smooth_equals_zero_sinks(lib):
    b = _small_ragged(9, "smooth", seed=41)
    sm, lse_sm = _run(lib, b, sinks=None, smooth=True)
    zs, lse_zs = _run(lib, b, sinks=torch.zeros(b.hq), smooth=False)
    assert np.array_equal(sm, zs) and np.array_equal(lse_sm, lse_zs)
    plain, _ = _run(lib, b, sinks=None, smooth=False)
    assert not np.allclose(sm, plain)  # the +1 really is there


def pin_counting_probe(lib):
    """q = 0 makes every kept score 0, so with v[j] = (1, j, j^2, 0...) and
    sink s the output is (n, sum j, sum j^2) / (n + e^s) over the kept keys:
    this recovers the exact key set [pos-n+1, pos] of every row."""
    for w in (0, 1, 5, 16, 33):
        for p, e in ((0, 20), (13, 17), (40, 3)):
            L = p + e
            b = W.make_batch([p], [e], 2, 1, 8, "f16", window=w,
                             sink_mode="head", seed=51)
            b.q.zero_()
            j = torch.arange(L, dtype=torch.float64)
            b.v.zero_()
            b.v[:, 0, 0] = 1.0
            b.v[:, 0, 1] = j.to(b.v.dtype)
            b.v[:, 0, 2] = (j * j).to(b.v.dtype)
            out, lse = _run(lib, b)
            for h in range(2):
                es = np.exp(float(b.sinks[h]))
                for i in range(e):
                    pos = p + i
                    n = pos + 1 if w <= 0 else min(pos + 1, w)
                    keys = np.arange(pos - n + 1, pos + 1, dtype=np.float64)
                    den = n + es
                    np.testing.assert_allclose(
                        out[i, h, :3], [n / den, keys.sum() / den,
                                        (keys ** 2).sum() / den], rtol=1e-12)
                    np.testing.assert_allclose(lse[i, h], np.log(den), rtol=1e-12)


def pin_chunked_equals_one_shot(lib):
    """Splitting a sequence into chunks whose earlier tokens become the cached
    prefix leaves every row bit-identical."""
    one = W.make_batch([5], [60], 4, 2, 16, "bf16", window=11, sink_mode="head",
                       seed=61)
    ref, ref_lse = _run(lib, one)
    cuts = [0, 17, 18, 40, 60]
    for a, c in zip(cuts[:-1], cuts[1:]):
        chunk = W.Batch(one.q[a:c], one.k[:5 + c], one.v[:5 + c],
                        torch.tensor([0, c - a], dtype=torch.int32),
                        torch.tensor([5 + a], dtype=torch.int32),
                        torch.tensor([0, 5 + c], dtype=torch.int32), one.hq,
                        one.hkv, one.d, one.window, one.sinks, one.smooth,
                        one.scale)
        out, lse = _run(lib, chunk)
        assert np.array_equal(out, ref[a:c]) and np.array_equal(lse, ref_lse[a:c])


def pin_window_bounded_layout_equals_full(lib):
    full = W.make_batch([50, 3, 20], [12, 30, 7], 4, 2, 16, "f16", window=20,
                        sink_mode="head", seed=71)
    bounded = W.window_bounded(full, 20)
    assert bounded.prefix_lens.tolist() == [20, 3, 20]
    a, la = _run(lib, full)
    b, lb = _run(lib, bounded)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def pin_row_selection_is_exact(lib):
    b = _small_ragged(0, "head", seed=81)
    full, lf = _run(lib, b)
    rows = [0, 5, 22, 23, 30, 71]
    part, lp = _run(lib, b, rows=rows)
    assert np.array_equal(part[rows], full[rows])
    others = np.setdiff1d(np.arange(b.total_q), rows)
    assert np.isnan(part[others]).all()


def _brute_census(prefix, extend, rows, block_n, window):
    """Element-level enumeration of the mask (band from tril/triu) per unit."""
    L = prefix + extend
    keep = torch.tril(torch.ones(extend, L, dtype=torch.bool), diagonal=prefix)
    if window > 0:
        keep &= torch.triu(torch.ones(extend, L, dtype=torch.bool),
                           diagonal=prefix - window + 1)
    n_key_tiles = -(-L // block_n)
    pad = torch.zeros(extend, n_key_tiles * block_n, dtype=torch.bool)
    pad[:, :L] = keep                      # keys past L are never kept
    recs = []
    for q0 in range(0, extend, rows):
        blk = pad[q0:q0 + rows].reshape(-1, n_key_tiles, block_n)
        live = blk.any(dim=2).any(dim=0)
        has_masked = (~blk).any(dim=2).any(dim=0)
        idx = torch.nonzero(live).flatten().tolist()
        first, last = idx[0], idx[-1]
        recs.append((q0, first * block_n, last - first + 1,
                     int(has_masked[first:last + 1].sum())))
    return recs


def pin_tile_census_brute_force(lib):
    tilings = [(16, 64), (32, 32), (32, 64), (64, 64), (16, 128), (128, 64),
               (3, 5), (8, 16)]
    windows = [1, 15, 16, 63, 64, 65, 100, 127, 128, 129, 0]
    for rows, bn in tilings:
        for w in windows:
            for p in (0, 1, bn - 1, bn, 2 * bn + 1, 131):
                for e in (1, rows - 1 if rows > 1 else 1, rows, rows + 1, 70):
                    got = oracle.tile_census([0, e], [p], 1, rows, bn, w, lib=lib)
                    want = _brute_census(p, e, rows, bn, w)
                    assert [tuple(r[2:]) for r in got.tolist()] == want, \
                        (rows, bn, w, p, e)


def pin_sglang_tile_count_example(lib):
    """382 -> 256 iterated tiles per (sequence, head) on the SGLang page."""
    with open(os.path.join(GOLDEN, "sglang_tile_counts.json")) as f:
        g = json.load(f)
    bm, bn, P, E, w = g["block_m"], g["block_n"], g["prefix"], g["extend"], g["window"]
    rec = oracle.tile_census([0, E], [P], 1, bm, bn, w, lib=lib)
    assert int(rec[:, 4].sum()) == g["tiles_after"]
    # Before the change: stage 1 walked every prefix tile; stage 2 walked the
    # extend keys from its own floor to the causal end, tiles counted from
    # the extend start.  Enumerated from the extend-only mask.
    before = 0
    for m0 in range(0, E, bm):
        before += -(-P // bn)
        ext_only = oracle.tile_census([0, min(bm, E - m0)], [m0], 1, bm, bn, w,
                                      lib=lib)
        before += int(ext_only[0, 4])
    assert before == g["tiles_before"]


def _run_masked(lib, batch, keep_rows, window=None):
    words, indptr = W.pack_custom_mask(keep_rows)
    return oracle.prefill(batch.q, batch.k, batch.v, batch.cu_seqlens_q, batch.prefix_lens,
                          batch.kv_indptr, batch.scale,
                          batch.window if window is None else window, sinks=batch.sinks,
                          smooth_softmax=batch.smooth, lib=lib, custom_mask=words,
                          mask_indptr=indptr)


def _masked_library_reference(batch, keep_rows):
    """torch float64 softmax over scores with an explicit boolean keep matrix
    per sequence: the tril/triu band of the causal/window mask, with its
    extend columns ANDed with the custom keep matrix (the prefix columns
    untouched); a sink is a dropped extra column."""
    g = batch.hq // batch.hkv
    q, k, v = (batch.q.to(torch.float64), batch.k.to(torch.float64),
               batch.v.to(torch.float64))
    out = torch.zeros_like(q)
    lse = torch.zeros(q.shape[:2], dtype=torch.float64)
    w = batch.window
    for b, q0, q1, k0, k1, p in _seq_slices(batch):
        e, L = q1 - q0, k1 - k0
        ones = torch.ones(e, L, dtype=torch.bool)
        keep = torch.tril(ones, diagonal=p)
        if w > 0:
            keep = keep & torch.triu(ones, diagonal=p - w + 1)
        keep[:, p:] &= torch.from_numpy(np.asarray(keep_rows[b], dtype=bool))
        for h in range(batch.hq):
            s = batch.scale * q[q0:q1, h] @ k[k0:k1, h // g].T
            s = s.masked_fill(~keep, float("-inf"))
            if batch.sinks is not None or batch.smooth:
                x = 0.0 if batch.smooth else float(batch.sinks[h])
                s = torch.cat([s, torch.full((e, 1), x, dtype=torch.float64)], 1)
            pr = torch.softmax(s, dim=1)[:, :L]
            out[q0:q1, h] = pr @ v[k0:k1, h // g]
            lse[q0:q1, h] = torch.logsumexp(s, dim=1)
    return out.numpy(), lse.numpy()


def pin_custom_mask_is_library_masked_softmax(lib):
    """A random custom mask ANDed into the causal/window mask, against the
    library softmax over an explicit keep matrix (packed by numpy, so the
    oracle's bit layout is checked too); widths across the 32-bit words."""
    for w, mode in ((0, "head"), (9, "none"), (25, "smooth")):
        b = W.make_batch([0, 37, 5], [23, 45, 70], 4, 2, 16, "bf16", window=w,
                         sink_mode=mode, seed=91 + w)
        keep = W.random_custom_mask(b.extend_lens, density=0.6, seed=w)
        out, lse = _run_masked(lib, b, keep)
        ref, ref_lse = _masked_library_reference(b, keep)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def pin_custom_mask_full_or_causal_is_no_mask(lib):
    """All-ones and lower-triangular custom masks change nothing (causality
    already removes every key above the diagonal): bit-identical."""
    b = _small_ragged(11, "head", seed=92)
    ref, ref_lse = _run(lib, b)
    for keep in ([np.ones((e, e), bool) for e in b.extend_lens],
                 [np.tril(np.ones((e, e), bool)) for e in b.extend_lens]):
        out, lse = _run_masked(lib, b, keep)
        assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def pin_custom_mask_diagonal_is_window_one(lib):
    """Without a prefix, a custom mask keeping only the diagonal leaves each
    row its own key: the window = 1 result, bit for bit."""
    b = W.make_batch([0, 0], [33, 20], 4, 2, 16, "f16", window=0, sink_mode="head", seed=93)
    out, lse = _run_masked(lib, b, [np.eye(e, dtype=bool) for e in b.extend_lens])
    ref, ref_lse = _run(lib, b, window=1)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def pin_custom_mask_counting_probe(lib):
    """q = 0 and v[j] = (1, j, j^2): each row's output recovers the exact set
    of keys it kept -- every prefix key inside the window, plus the extend
    keys whose bit is set, at or below the row, inside the window."""
    for w in (0, 7, 40):
        p, e = 13, 50
        b = W.make_batch([p], [e], 2, 1, 8, "f16", window=w, sink_mode="head", seed=94)
        b.q.zero_()
        L = p + e
        j = torch.arange(L, dtype=torch.float64)
        b.v.zero_()
        b.v[:, 0, 0] = 1.0
        b.v[:, 0, 1] = j.to(b.v.dtype)
        b.v[:, 0, 2] = (j * j).to(b.v.dtype)
        keep = W.random_custom_mask([e], density=0.5, seed=95 + w, diagonal=False)
        out, lse = _run_masked(lib, b, keep)
        for h in range(2):
            es = np.exp(float(b.sinks[h]))
            for i in range(e):
                pos = p + i
                lo = 0 if w <= 0 else max(0, pos - w + 1)
                keys = [jj for jj in range(lo, pos + 1) if jj < p or keep[0][i, jj - p]]
                n = len(keys)
                if n == 0:
                    assert np.all(out[i, h] == 0) and lse[i, h] == -np.inf
                    continue
                den = n + es
                vs = b.v[keys, 0, :3].double().numpy()  # j^2 as stored (fp16-rounded past 2048)
                np.testing.assert_allclose(out[i, h, :3], vs.sum(axis=0) / den, rtol=1e-12)
                np.testing.assert_allclose(lse[i, h], np.log(den), rtol=1e-12)


PINS = [pin_plain_causal_is_library_softmax, pin_sinks_are_a_dropped_softmax_column,
        pin_window_is_library_band, pin_window_one_closed_form,
        pin_wide_window_equals_no_window, pin_smooth_equals_zero_sinks,
        pin_counting_probe, pin_chunked_equals_one_shot,
        pin_window_bounded_layout_equals_full, pin_row_selection_is_exact,
        pin_tile_census_brute_force, pin_sglang_tile_count_example,
        pin_custom_mask_is_library_masked_softmax, pin_custom_mask_full_or_causal_is_no_mask,
        pin_custom_mask_diagonal_is_window_one, pin_custom_mask_counting_probe]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)
