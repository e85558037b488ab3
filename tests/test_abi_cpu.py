"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/gqa_prefill.h declares, and rejects invalid host arguments
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_prefill.h")


@pytest.fixture(scope="module")
def lib():
    from gqa_flash_attention_prefill_gb300 import build
    path = build.build()
    import gqa_flash_attention_prefill_gb300 as pkg
    return pkg.load(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    import gqa_flash_attention_prefill_gb300 as pkg
    assert names == sorted(pkg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.gqa_prefill_version().decode().count(".") == 2
    for code in (0, -1, -2, -3):
        assert lib.gqa_prefill_status_string(code)


FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced


def _call(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, cu=FAKE, pre=FAKE, kvi=FAKE, B=1, total_q=16,
             total_kv=16, max_q=16, hq=8, hkv=2, d=64, dtype=1, scale=0.125, window=0,
             sinks=None, smooth=0, out=FAKE, lse=None, stream=None)
    a.update(over)
    return lib.gqa_flash_prefill(a["q"], a["k"], a["v"], a["cu"], a["pre"], a["kvi"], a["B"],
                                 a["total_q"], a["total_kv"], a["max_q"], a["hq"], a["hkv"],
                                 a["d"], a["dtype"], a["scale"], a["window"], a["sinks"],
                                 a["smooth"], a["out"], a["lse"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(hq=6, hkv=4), -1),            # Hq % Hkv != 0
    (dict(hkv=0), -1),
    (dict(d=0), -1),
    (dict(dtype=7), -1),
    (dict(scale=0.0), -1),
    (dict(scale=-1.0), -1),
    (dict(scale=float("inf")), -1),
    (dict(scale=float("nan")), -1),
    (dict(sinks=FAKE, smooth=1), -1),   # the sink modes are exclusive
    (dict(B=-1), -1),
    (dict(total_q=-5), -1),
    (dict(q=None), -1),
    (dict(out=None), -1),
    (dict(cu=None), -1),
    (dict(kvi=None), -1),
    (dict(q=FAKE + 8), -1),             # misaligned base
    (dict(out=FAKE + 2), -1),
    (dict(total_kv=0), -1),
    (dict(d=96), -2),                   # declined: head dim not implemented
    (dict(hq=24, hkv=1), -2),           # declined: G does not divide 128
    (dict(B=1 << 22, total_q=1 << 22), -2),  # declined: unit records overflow
])
def test_invalid_arguments_are_rejected_before_launch(lib, over, code):
    assert _call(lib, **over) == code


def test_empty_work_is_ok_without_launch(lib):
    assert _call(lib, B=0) == 0
    assert _call(lib, total_q=0) == 0
    assert _call(lib, B=0, q=None, k=None, v=None, out=None) == 0


def _call_noalloc(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, cu=FAKE, pre=FAKE, kvi=FAKE, B=1, total_q=16,
             total_kv=16, max_q=16, hq=8, hkv=2, d=64, dtype=1, scale=0.125, window=0,
             sinks=None, smooth=0, out=FAKE, lse=None, splits=2, stream=None)
    a.update(over)
    return lib.gqa_flash_prefill_splitkv_noalloc(
        a["q"], a["k"], a["v"], a["cu"], a["pre"], a["kvi"], a["B"], a["total_q"],
        a["total_kv"], a["max_q"], a["hq"], a["hkv"], a["d"], a["dtype"], a["scale"],
        a["window"], a["sinks"], a["smooth"], a["out"], a["lse"], a["splits"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(hq=6, hkv=4), -1),
    (dict(dtype=7), -1),
    (dict(scale=0.0), -1),
    (dict(sinks=FAKE, smooth=1), -1),
    (dict(splits=17), -1),
    (dict(splits=-2), -1),
    (dict(q=None), -1),
    (dict(d=96), -2),
    # arguments are checked before the empty-work early return
    (dict(B=0, hq=6, hkv=4), -1),
    (dict(total_q=0, dtype=7), -1),
    (dict(total_q=0, sinks=FAKE, smooth=1), -1),
    (dict(B=0, scale=float("nan")), -1),
    (dict(B=0), 0),
    (dict(total_q=0), 0),
])
def test_noalloc_entry_validates_like_the_others(lib, over, code):
    assert _call_noalloc(lib, **over) == code


def test_plan_is_host_only(lib):
    import gqa_flash_attention_prefill_gb300 as pkg
    p = pkg.plan(1, 4096, 4096, 64, 8, 64, "bf16", 0)
    assert p["rows_per_unit"] == 16 * p["q_tiles"] and p["block_n"] in (64, 128)
    assert p["max_units"] == 8 * (4096 // p["rows_per_unit"] + 1)
    assert p["grid"] >= 1
    p = pkg.plan(1, 256, 256, 4, 1, 64, "f16", 32)
    assert p["rows_per_unit"] == 32 * p["q_tiles"]
    with pytest.raises(pkg.GQAError):
        pkg.plan(1, 10, 10, 8, 2, 80, "bf16", 0)


def test_force_block_n_validates(lib):
    assert lib.gqa_prefill_force_block_n(80) == -1
    assert lib.gqa_prefill_force_block_n(64) == 0
    assert lib.gqa_prefill_force_block_n(0) == 0


def test_force_q_tiles_validates_and_shapes_plan(lib):
    import gqa_flash_attention_prefill_gb300 as pkg
    for bad in (-1, 3, 4):
        assert lib.gqa_prefill_force_q_tiles(bad) == -1
    try:
        pkg.force_q_tiles(2)
        p = pkg.plan(1, 4096, 4096, 64, 8, 64, "bf16", 0)
        assert p["q_tiles"] == 2 and p["rows_per_unit"] == 32
        assert p["max_units"] == 8 * (4096 // 32 + 1)
        assert p["ctas_per_sm"] == 1
        pkg.force_block_n(96)  # no two-tile kernel for 96-key tiles: declined
        with pytest.raises(pkg.GQAError):
            pkg.plan(1, 4096, 4096, 64, 8, 64, "bf16", 0)
        pkg.force_block_n(0)
        with pytest.raises(pkg.GQAError):  # d = 256: two tiles exceed tensor memory
            pkg.plan(1, 4096, 4096, 16, 2, 256, "bf16", 0)
        pkg.force_q_tiles(1)
        p = pkg.plan(1, 4096, 4096, 64, 8, 64, "bf16", 0)
        assert p["q_tiles"] == 1 and p["rows_per_unit"] == 16
    finally:
        pkg.force_block_n(0)
        pkg.force_q_tiles(0)
    assert pkg.plan(1, 4096, 4096, 64, 8, 64, "bf16", 0)["q_tiles"] in (1, 2)


def test_binding_refuses_to_run_without_library(tmp_path):
    import gqa_flash_attention_prefill_gb300 as pkg
    with pytest.raises(RuntimeError, match="missing"):
        pkg.load(str(tmp_path / "nope.so"))


def test_split_count_choice_is_host_only(lib):
    """The library's split-KV choice, from shapes alone (no device access):
    no split when the units fill the GPU (a 4096-token prefill, a decode step
    of 128 sequences), splits when they cannot (two 64-token chunks, a
    four-sequence decode step); explicit counts are honoured up to 16."""
    import gqa_flash_attention_prefill_gb300 as pkg
    assert pkg.splitkv_workspace(1, 4096, 4096, 64, 8, 64, "bf16", 0, 0) == (1, 0)
    assert pkg.splitkv_workspace(128, 128, 1, 64, 8, 64, "bf16", 128, 0) == (1, 0)
    used, nbytes = pkg.splitkv_workspace(2, 128, 64, 64, 8, 64, "bf16", 0, 0)
    assert used > 1 and nbytes > 0
    used, nbytes = pkg.splitkv_workspace(4, 4, 1, 64, 8, 64, "bf16", 0, 0)
    assert used > 1 and nbytes > 0
    used, nbytes = pkg.splitkv_workspace(1, 64, 64, 64, 8, 64, "bf16", 0, 16)
    assert used == 16 and nbytes > 0


def test_balanced_split_workspace_is_host_only(lib):
    """The balanced split's workspace from shapes alone: two partial tiles
    per resident CTA plus four count words per unit; a launch with more query
    tiles than the kernel's shared-memory scratch holds is declined; split
    counts below GQA_SPLITS_BALANCED are invalid."""
    import gqa_flash_attention_prefill_gb300 as pkg
    used, nbytes = pkg.splitkv_workspace(1, 512, 512, 64, 8, 64, "bf16", 0, pkg.SPLITS_BALANCED)
    p = pkg.plan(1, 512, 512, 64, 8, 64, "bf16", 0)
    slots = p["grid"] if p["grid"] < p["max_units"] else None
    assert used == pkg.SPLITS_BALANCED and nbytes >= 2 * 128 * 64 * 4 * 2
    if slots is not None:
        assert nbytes >= 2 * slots * 128 * 64 * 4
    used2, nbytes2 = pkg.splitkv_workspace(2, 4096, 2048, 64, 8, 64, "bf16", 0,
                                           pkg.SPLITS_BALANCED)
    assert used2 == pkg.SPLITS_BALANCED and nbytes2 > nbytes  # more units, more count words
    with pytest.raises(pkg.GQAError):  # 2^20 queries: 65,536 query tiles per launch
        pkg.splitkv_workspace(1, 1 << 20, 1 << 20, 64, 8, 64, "bf16", 0, pkg.SPLITS_BALANCED)
    with pytest.raises(pkg.GQAError):
        pkg.splitkv_workspace(1, 512, 512, 64, 8, 64, "bf16", 0, -2)


def _call_masked(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, cu=FAKE, pre=FAKE, kvi=FAKE, B=1, total_q=16,
             total_kv=16, max_q=16, hq=8, hkv=2, d=64, dtype=1, scale=0.125, window=0,
             sinks=None, smooth=0, mask=FAKE, mip=FAKE, words=16, out=FAKE, lse=None,
             stream=None)
    a.update(over)
    return lib.gqa_flash_prefill_masked(
        a["q"], a["k"], a["v"], a["cu"], a["pre"], a["kvi"], a["B"], a["total_q"],
        a["total_kv"], a["max_q"], a["hq"], a["hkv"], a["d"], a["dtype"], a["scale"],
        a["window"], a["sinks"], a["smooth"], a["mask"], a["mip"], a["words"], a["out"],
        a["lse"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(mask=None), -1),
    (dict(mip=None), -1),
    (dict(mask=FAKE + 2), -1),          # words must be 4-byte aligned
    (dict(words=-1), -1),
    (dict(hq=6, hkv=4), -1),
    (dict(sinks=FAKE, smooth=1), -1),
    (dict(d=96), -2),
    (dict(B=0), 0),
    (dict(B=0, dtype=7), -1),
])
def test_masked_entry_validates_before_launch(lib, over, code):
    assert _call_masked(lib, **over) == code


def test_call_flags_are_per_thread_and_checked(lib):
    """gqa_prefill_set_call_flags: known bits only, and the flags belong to
    the calling host thread (another thread starts at 0)."""
    import threading
    import gqa_flash_attention_prefill_gb300 as pkg
    assert lib.gqa_prefill_get_call_flags() == 0
    assert lib.gqa_prefill_set_call_flags(2) == -1
    assert lib.gqa_prefill_set_call_flags(pkg.FLAG_METADATA_READY) == 0
    try:
        assert lib.gqa_prefill_get_call_flags() == pkg.FLAG_METADATA_READY
        seen = []
        t = threading.Thread(target=lambda: seen.append(lib.gqa_prefill_get_call_flags()))
        t.start()
        t.join()
        assert seen == [0]
    finally:
        assert lib.gqa_prefill_set_call_flags(0) == 0
    assert lib.gqa_prefill_get_call_flags() == 0
