"""GPU-side helpers for the parity tests: run the library, run the oracle on
host copies of the same inputs, compare with the stated tolerances.

Tolerances: the norm within 1e-5 relative of the oracle's; fp32 outputs
within 2 ulp, fp16/bf16 within 1 ulp; the nonfinite flag and the clip
decision identical; on SKIP every output bit-identical to its input.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import global_l2_norm_gb300 as g
import oracle
from _helpers import storage_bits, to_oracle, ulp_distance

NORM_RTOL = 1e-5
ULP_TOL = {"f32": 2, "f16": 1, "bf16": 1}


def gpu_clip(tensors, max_norm, inv_scale=1.0, variant="split", stream=None):
    """Clip `tensors` (CUDA, in place) through the C ABI; return the record."""
    with g.GradClipper(tensors, variant=variant) as c:
        norm, flag = c.clip_(max_norm, inv_scale, stream=stream)
        rec = c.result(stream=stream)
        rec["out_norm"] = float(norm.item())
        rec["out_flag"] = int(flag.item())
    return rec


def compare(inputs_host, outs_gpu, rec, max_norm, inv_scale, name=""):
    """inputs_host: oracle tensors taken before the clip; outs_gpu: torch
    tensors after it.  Returns a dict of the worst deviations."""
    want, r = oracle.clip(inputs_host, max_norm, inv_scale)
    assert bool(rec["nonfinite"]) == r.nonfinite, (name, rec, r)
    assert rec["out_flag"] == int(r.nonfinite)
    assert rec["decision"] == r.decision, (name, rec["decision"], r.decision, r.norm)
    if r.nonfinite:
        assert not math.isfinite(rec["norm"])
    else:
        rel = abs(rec["norm"] - r.norm) / r.norm if r.norm else abs(rec["norm"])
        assert rel <= NORM_RTOL, (name, rec["norm"], r.norm, rel)
    assert rec["out_norm"] == rec["norm"] or (math.isnan(rec["norm"]) and math.isnan(rec["out_norm"]))
    worst = {"f32": 0, "f16": 0, "bf16": 0}
    for i, (w, o) in enumerate(zip(want, outs_gpu)):
        got = to_oracle(o)
        if r.decision == oracle.SKIP:
            assert np.array_equal(storage_bits(got), storage_bits(inputs_host[i])), (name, i)
            continue
        if got.data.size == 0:
            continue
        d = int(ulp_distance(got, w).max())
        worst[w.dtype] = max(worst[w.dtype], d)
        assert d <= ULP_TOL[w.dtype], (name, i, w.dtype, d)
    rel_norm = 0.0
    if not r.nonfinite and r.norm:
        rel_norm = abs(rec["norm"] - r.norm) / r.norm
    return {"oracle": r, "worst_ulp": worst, "norm_rel": rel_norm}


def host_copies(tensors):
    return [to_oracle(t) for t in tensors]


def clone_all(tensors):
    return [t.clone() for t in tensors]


def restore(dst, src):
    for d, s in zip(dst, src):
        d.copy_(s)
    torch.cuda.synchronize()
