"""Out-of-place clip into fp32 buffers on the GPU against the oracle.

Tolerance as for the in-place fp32 clip: each output is x times the
float-float multiplier rounded once, so within 2 ulp of the oracle's
correctly rounded value (exact when the multiplier is a power of two); the
gradients must be left bit-identical, and nothing written on SKIP.
"""
import math

import numpy as np
import pytest
import torch

import global_l2_norm_gb300 as g
import oracle
from _helpers import storage_bits, to_oracle
from oracle import OracleTensor
from workloads import make_gradset

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    g.build()


def dev():
    return torch.device("cuda", 0)


def ulps32(a, b):
    ia = a.view(np.int32).astype(np.int64)
    ib = b.view(np.int32).astype(np.int64)
    oa = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ob = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(oa - ob)


def run(tensors, max_norm, inv_scale, misalign=False):
    keep = []
    if misalign:
        outs = []
        for t in tensors:
            b = torch.full((t.numel() + 1,), 7.0, device=dev())
            keep.append(b)
            outs.append(b[1:])
    else:
        outs = [torch.full((t.numel(),), 7.0, device=dev()) for t in tensors]
    before = [to_oracle(t) for t in tensors]
    with g.GradClipper(tensors) as c:
        c.attach_f32_out(outs)
        norm, flag = c.clip_to_f32_(max_norm, inv_scale)
        rec = c.result()
    want, r = oracle.default().clip_to_f32(before, max_norm, inv_scale, fill=7.0)
    assert rec["decision"] == r.decision and bool(rec["nonfinite"]) == r.nonfinite
    if not r.nonfinite:
        assert abs(rec["norm"] - r.norm) <= 1e-5 * r.norm
    worst = 0
    for b, t, o, w_ in zip(before, tensors, outs, want):
        assert np.array_equal(storage_bits(b), storage_bits(to_oracle(t)))   # only read
        got = o.cpu().numpy()
        d = int(ulps32(got, w_).max()) if got.size else 0
        assert d <= 2, d
        worst = max(worst, d)
    return r, worst


def test_fp16_unscale_is_exact():
    gs = make_gradset("andrea120m_fp16", device=dev())
    r, worst = run(gs.tensors, gs.max_norm, gs.inv_scale)
    assert r.decision == oracle.PASS and worst == 0


@pytest.mark.parametrize("name", ["tiny", "andrea120m", "andrea120m_bf16"])
def test_clip_into_f32(name):
    gs = make_gradset(name, device=dev())
    r, _ = run(gs.tensors, gs.max_norm, gs.inv_scale)
    assert r.decision == oracle.CLIP


def test_fp32_out_equals_in_place():
    """Same arithmetic as the in-place clip: the fp32 outputs are its bits."""
    gs = make_gradset("andrea14m", device=dev())
    for t in gs.tensors:
        t.mul_(40.0)
    outs = [torch.empty(t.numel(), device=dev()) for t in gs.tensors]
    with g.GradClipper(gs.tensors) as c:
        c.attach_f32_out(outs)
        c.clip_to_f32_(1.0, 0.75)
        c.clip_(1.0, 0.75)
    for o, t in zip(outs, gs.tensors):
        assert torch.equal(o.view(torch.int32), t.reshape(-1).view(torch.int32))


def test_misaligned_outputs_and_pass_with_unit_multiplier():
    gs = make_gradset("andrea14m", device=dev())
    r, worst = run(gs.tensors, 1.0, 1.0, misalign=True)
    assert r.decision == oracle.PASS and worst == 0    # a copy, written even at multiplier 1


def test_nonfinite_writes_nothing():
    gs = make_gradset("tiny", device=dev())
    gs.tensors[0].view(-1)[5] = -math.inf
    r, _ = run(gs.tensors, 1.0, 1.0)
    assert r.decision == oracle.SKIP


def test_attach_rejects_overlap_and_wrong_count():
    x = torch.ones(64, device=dev())
    with g.GradClipper([x[:32], x[32:]]) as c:
        with pytest.raises(g.GclipError):
            c.attach_f32_out([x[:32], torch.empty(32, device=dev())])   # output = a gradient
        with pytest.raises(g.GclipError):
            c.attach_f32_out([torch.empty(32, device=dev())])           # one of two
        with pytest.raises(g.GclipError):
            c.clip_to_f32_(1.0)                                         # nothing attached
