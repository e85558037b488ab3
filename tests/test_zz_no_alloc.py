"""gqa_flash_prefill_splitkv_noalloc: split-KV with the library's file-scope
scratch instead of a caller workspace.  Compared bit for bit with the
workspace entry point (same kernels, same split count) over calls in a row,
so the second call runs on scratch the first one left behind."""
import ctypes

import pytest

from gqa_flash_attention_prefill_gb300 import workloads as W


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__
    __graft_entry__.build()
    import gqa_flash_attention_prefill_gb300 as pkg
    pkg.load()
    pkg.force_block_n(0)
    pkg.force_q_tiles(0)
    return pkg


def _both(pkg, b):
    import torch
    dev = b.to("cuda")
    used, nbytes = pkg.splitkv_workspace(dev.num_seqs, dev.total_q, dev.max_seqlen_q, dev.hq,
                                         dev.hkv, dev.d, dev.dtype_name, dev.window, 0)
    assert used > 1 and 0 < nbytes <= pkg.NOALLOC_SCRATCH_BYTES, (used, nbytes)
    ref_out, ref_lse = pkg.prefill_splitkv(dev, num_splits=0)
    out = torch.full_like(dev.q, float("nan"))
    lse = torch.full(dev.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    pkg.prefill_splitkv_noalloc(dev, num_splits=0, out=out, lse=lse)
    torch.cuda.synchronize()
    assert pkg.get_device_status() == 0
    return (out, lse), (ref_out, ref_lse)


@pytest.mark.gpu
def test_noalloc_equals_workspace_entry_over_calls_in_a_row(pkg):
    import torch
    batches = [
        W.make_batch([3000], [64], 64, 8, 64, "bf16", window=0, sink_mode="head", seed=31),
        W.make_batch([5000, 100], [48, 33], 64, 8, 64, "f16", window=128, sink_mode="smooth",
                     seed=32),
    ]
    for b in batches + batches[:1]:  # the third call reuses scratch the second one wrote
        (out, lse), (ref_out, ref_lse) = _both(pkg, b)
        assert torch.equal(out, ref_out), b.name
        assert torch.equal(lse, ref_lse), b.name


_DECLINE_SCRIPT = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1])
import gqa_flash_attention_prefill_gb300 as pkg
lib = pkg.load()
fake = 1 << 20
used, nbytes = pkg.splitkv_workspace(1, 4096, 4096, 64, 8, 64, "bf16", 0, 16)
assert used == 16 and nbytes > pkg.NOALLOC_SCRATCH_BYTES, (used, nbytes)
rc = lib.gqa_flash_prefill_splitkv_noalloc(fake, fake, fake, fake, fake, fake, 1, 4096, 4096,
                                           4096, 64, 8, 64, pkg.GQA_BF16, ctypes.c_float(0.125),
                                           0, None, 0, fake, None, 16, None)
print("rc", rc)
"""


def test_noalloc_declines_oversize_before_launch(pkg):
    """4096 tokens x 8 KV heads in 16 splits needs ~1 GB of partials: declined
    (GQA_ERR_UNSUPPORTED) before any device access.  The call passes fake
    addresses, so it runs in a child process that sees no GPU: were the
    decline ever to slip, the launch would fail there with GQA_ERR_CUDA
    instead of touching a device."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _DECLINE_SCRIPT, root], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "rc -2" in r.stdout, r.stdout
