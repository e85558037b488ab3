"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
from gqa_flash_attention_prefill_gb300 import workloads as W

# Tolerances for 16-bit inputs with fp32 accumulation: relL2 <= 1e-3 and
# max_abs <= 2e-2, lse within 1e-3.  For bf16 outputs the relL2 bound adds the
# quantisation floor of the dtype itself, once: rounding the EXACT result to
# bf16 already costs qf = relL2(bf16(ref), ref) ~ 1.6e-3 on N(0,1) inputs, so
# no bf16 output can meet 1e-3.  bf16 uses 1e-3 + qf, with qf measured on the
# case's own oracle output.
REL_L2 = 1e-3
MAX_ABS = 2e-2
LSE_ABS = 1e-3

# Every comparison made in this process: (label, dtype, relL2, bound,
# max_abs, lse error).  tests/conftest.py prints a summary at the end of the
# run, so each bf16 case's margin is visible in the log.
RESULTS = []


def quant_floor(ref, dtype):
    """relL2 between the exact result and the exact result rounded to dtype."""
    r = torch.from_numpy(np.ascontiguousarray(ref)).to(dtype).double().numpy()
    return float(np.linalg.norm(r - ref) / max(np.linalg.norm(ref), 1e-30))


def run_gpu(pkg, batch_cpu, poison=True, debug_log=None):
    """Returns (out, lse) as CPU tensors; out/lse are pre-filled with NaN so
    that rows the kernel fails to write show up."""
    dev = batch_cpu.to("cuda")
    out = torch.empty_like(dev.q)
    lse = torch.empty(dev.q.shape[:2], dtype=torch.float32, device="cuda")
    if poison:
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
    args = (dev.q, dev.k, dev.v, dev.cu_seqlens_q, dev.prefix_lens, dev.kv_indptr,
            dev.scale)
    kw = dict(window=dev.window, sinks=dev.sinks, smooth_softmax=dev.smooth,
              out=out, lse=lse, max_seqlen_q=dev.max_seqlen_q)
    if debug_log is not None:
        pkg.gqa_flash_prefill_debug(*args, debug_log, **kw)
    else:
        pkg.gqa_flash_prefill(*args, **kw)
    torch.cuda.synchronize()
    status = pkg.get_device_status()
    assert status == 0, f"device status word raised: {status}"
    return out.cpu(), lse.cpu()


def sub_batch(batch, seqs):
    """The sequences `seqs` of a batch as a batch of their own (same values)."""
    cu = batch.cu_seqlens_q.tolist()
    kvp = batch.kv_indptr.tolist()
    pre = batch.prefix_lens.tolist()
    qs, ks, vs, ncu, nkv, npre = [], [], [], [0], [0], []
    for b in seqs:
        qs.append(batch.q[cu[b]:cu[b + 1]])
        ks.append(batch.k[kvp[b]:kvp[b + 1]])
        vs.append(batch.v[kvp[b]:kvp[b + 1]])
        ncu.append(ncu[-1] + cu[b + 1] - cu[b])
        nkv.append(nkv[-1] + kvp[b + 1] - kvp[b])
        npre.append(pre[b])
    return W.Batch(torch.cat(qs), torch.cat(ks), torch.cat(vs),
                   torch.tensor(ncu, dtype=torch.int32),
                   torch.tensor(npre, dtype=torch.int32),
                   torch.tensor(nkv, dtype=torch.int32), batch.hq, batch.hkv,
                   batch.d, batch.window, batch.sinks, batch.smooth, batch.scale,
                   batch.name + "/sub")


def run_oracle(batch, rows=None):
    return oracle.prefill(batch.q, batch.k, batch.v, batch.cu_seqlens_q,
                          batch.prefix_lens, batch.kv_indptr, batch.scale,
                          batch.window, sinks=batch.sinks,
                          smooth_softmax=batch.smooth, rows=rows)


def compare(out, lse, ref, ref_lse, rows=None, label=""):
    """relL2 <= 1e-3 and max_abs <= 2e-2 on out, |dlse| <= 1e-3, over the
    given token rows (default all rows that belong to a sequence)."""
    dtype = out.dtype
    got = out.float().numpy().astype(np.float64)
    gl = lse.numpy().astype(np.float64)
    if rows is not None:
        got, ref, gl, ref_lse = got[rows], ref[rows], gl[rows], ref_lse[rows]
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    err = got - ref
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30))
    mx = float(np.abs(err).max()) if err.size else 0.0
    lerr = float(np.abs(gl - ref_lse).max()) if gl.size else 0.0
    tol = REL_L2
    if dtype == torch.bfloat16:
        tol = REL_L2 + quant_floor(ref, torch.bfloat16)
    RESULTS.append((label, "bf16" if dtype == torch.bfloat16 else "f16", rel, tol, mx, lerr))
    assert rel <= tol and mx <= MAX_ABS, \
        f"{label}: relL2={rel:.3e} (tol {tol:.3e}) max_abs={mx:.3e}"
    assert lerr <= LSE_ABS, f"{label}: lse max_abs={lerr:.3e}"
    return rel, mx, lerr


def sample_rows(batch, per_seq=24, rows_per_unit=16, seed=0):
    """Token rows to check at full size: the first and last rows of each
    sequence, rows on both sides of unit and 128-position boundaries, and a
    seeded random draw."""
    rng = np.random.default_rng(seed)
    cu = batch.cu_seqlens_q.tolist()
    out = []
    for b in range(batch.num_seqs):
        e = cu[b + 1] - cu[b]
        if e == 0:
            continue
        cand = {0, 1, e - 1, e - 2}
        for edge in (rows_per_unit, 128, 4 * rows_per_unit):
            for mult in rng.integers(1, max(2, e // edge + 1), size=3):
                for off in (-1, 0):
                    cand.add(int(mult) * edge + off)
        cand.update(int(x) for x in rng.integers(0, e, size=per_seq))
        out.extend(cu[b] + i for i in sorted(cand) if 0 <= i < e)
    return np.array(sorted(set(out)), dtype=np.int64)
