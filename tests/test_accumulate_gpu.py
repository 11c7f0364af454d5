"""The last microbatch's accumulation folded into the clip, on the GPU,
against the oracle.

Tolerances as for the in-place clip: the norm within 1e-5 relative of the
oracle's, fp32 outputs within 2 ulp and fp16/bf16 within 1 ulp of the
oracle's, the flag and the decision identical.  On SKIP the gradients must
hold exactly the sums the format's own addition gives (a NaN sum as any
NaN), and the addends are never modified.  Beyond the oracle: the fused call
must give, bit for bit, what torch's addition followed by clip_grad_norm
gives on the same tensors.
"""
import math

import numpy as np
import pytest
import torch

import global_l2_norm_gb300 as g
import oracle
from _helpers import as_float64, storage_bits, to_oracle, ulp_distance
from workloads import make_gradset

pytestmark = pytest.mark.gpu

NORM_RTOL = 1e-5
ULP_TOL = {"f32": 2, "f16": 1, "bf16": 1}


@pytest.fixture(scope="module", autouse=True)
def built():
    g.build()


def dev():
    return torch.device("cuda", 0)


def fused(tensors, addends, max_norm, inv_scale):
    with g.GradClipper(tensors) as c:
        c.attach_addend(addends)
        norm, flag = c.clip_accumulate_(max_norm, inv_scale)
        rec = c.result()
        rec["out_norm"] = float(norm.item())
        rec["out_flag"] = int(flag.item())
    return rec


def run(tensors, addends, max_norm, inv_scale=1.0):
    """Fused accumulate + clip on the GPU against the oracle on host copies
    of the same inputs; returns the oracle's result and the worst ulps."""
    before = [to_oracle(t) for t in tensors]
    adds = [to_oracle(a) for a in addends]
    rec = fused(tensors, addends, max_norm, inv_scale)
    want, r = oracle.default().clip_accumulate(before, adds, max_norm, inv_scale)
    assert rec["decision"] == r.decision, (rec["decision"], r.decision, r.norm)
    assert bool(rec["nonfinite"]) == r.nonfinite and rec["out_flag"] == int(r.nonfinite)
    if r.nonfinite:
        assert not math.isfinite(rec["norm"])
    else:
        rel = abs(rec["norm"] - r.norm) / r.norm if r.norm else abs(rec["norm"])
        assert rel <= NORM_RTOL, (rec["norm"], r.norm)
        assert rec["out_norm"] == rec["norm"]
    worst = {"f32": 0, "f16": 0, "bf16": 0}
    for i, (w_, t) in enumerate(zip(want, tensors)):
        got = to_oracle(t)
        if got.data.size == 0:
            continue
        nan = np.isnan(as_float64(w_))
        if nan.any():   # a NaN sum: any NaN encoding (the GPU's is canonical)
            assert np.isnan(as_float64(got)[nan]).all(), i
            got.data[nan] = w_.data[nan]
        d = int(ulp_distance(got, w_).max())
        tol = 0 if r.decision == oracle.SKIP else ULP_TOL[w_.dtype]
        assert d <= tol, (i, w_.dtype, d)
        worst[w_.dtype] = max(worst[w_.dtype], d)
    for a_host, a in zip(adds, addends):      # the addends are only read
        assert np.array_equal(storage_bits(a_host), storage_bits(to_oracle(a)))
    return r, worst


@pytest.mark.parametrize("dt", [torch.float32, torch.float16, torch.bfloat16])
def test_worked_example(dt):
    """[2, 3] + [4, 5] = [6, 8], clipped at 5 to [3, 4] exactly."""
    x = torch.tensor([2.0, 3.0], dtype=dt, device=dev())
    a = torch.tensor([4.0, 5.0], dtype=dt, device=dev())
    rec = fused([x], [a], 5.0, 1.0)
    assert rec["decision"] == g.GCLIP_DECISION_CLIP and rec["norm"] == 10.0
    assert x.tolist() == [3.0, 4.0]


@pytest.mark.parametrize("name,decision", [
    ("tiny", oracle.CLIP), ("andrea14m", oracle.PASS), ("andrea120m", oracle.CLIP),
    ("andrea120m_fp16", oracle.PASS), ("andrea120m_bf16", oracle.CLIP)])
def test_workloads(name, decision):
    gs = make_gradset(name, device=dev())
    last = make_gradset(name, seed=4321, device=dev())
    r, _ = run(gs.tensors, last.tensors, gs.max_norm, gs.inv_scale)
    assert r.decision == decision


@pytest.mark.parametrize("name,mul", [("andrea14m", 40.0), ("andrea120m_fp16", 1.0),
                                      ("andrea120m_bf16", 1.0)])
def test_equals_separate_add_then_clip(name, mul):
    gs = make_gradset(name, device=dev())
    last = make_gradset(name, seed=4321, device=dev())
    for t in gs.tensors:
        t.mul_(mul)
    other = [t.clone() for t in gs.tensors]
    rec = fused(gs.tensors, last.tensors, gs.max_norm, gs.inv_scale)
    for t, a in zip(other, last.tensors):
        t.add_(a)
    with g.GradClipper(other) as c:
        c.clip_(gs.max_norm, gs.inv_scale)
        ref = c.result()
    assert rec["norm"] == ref["norm"] and rec["decision"] == ref["decision"]
    assert (rec["sumsq_hi"], rec["sumsq_lo"]) == (ref["sumsq_hi"], ref["sumsq_lo"])
    iv = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}
    for t, o in zip(gs.tensors, other):
        assert torch.equal(t.view(iv[t.dtype]), o.view(iv[o.dtype]))


@pytest.mark.parametrize("dt", [torch.float32, torch.float16, torch.bfloat16])
def test_ragged_and_misaligned(dt):
    """Sizes around the 16-byte vectors and the 32 KiB chunks, gradients and
    addends at element offsets that differ within 16 bytes (the addend then
    takes the element-by-element path), and empty tensors."""
    gen = torch.Generator(device=dev())
    gen.manual_seed(11)
    sizes = [0, 1, 3, 7, 8191, 8193, 16384 + 5, 33000, 70001]
    gbuf = torch.randn(sum(sizes) + 64, generator=gen, device=dev()).to(dt)
    abuf = torch.randn(sum(sizes) + 64, generator=gen, device=dev()).to(dt)
    grads, adds, go, ao = [], [], 1, 3
    for n in sizes:
        grads.append(gbuf[go:go + n])
        adds.append(abuf[ao:ao + n])
        go += n + 1
        ao += n + 2
    for max_norm in (1.0, 1e4):
        r, _ = run(grads, adds, max_norm, 0.5)
        assert r.decision == (oracle.CLIP if max_norm == 1.0 else oracle.PASS)


def test_aligned_and_element_paths_agree():
    gs = make_gradset("andrea14m", device=dev())
    last = make_gradset("andrea14m", seed=4321, device=dev())
    copy = [t.clone() for t in gs.tensors]
    shifted = []
    for a in last.tensors:       # same values, one element off the 16-byte grid
        b = torch.empty(a.numel() + 1, device=dev())
        b[1:] = a.reshape(-1)
        shifted.append(b[1:])
    r1 = fused(gs.tensors, last.tensors, 0.1, 1.0)
    r2 = fused(copy, shifted, 0.1, 1.0)
    assert r1["norm"] == r2["norm"] and r1["decision"] == g.GCLIP_DECISION_CLIP
    for x, y in zip(gs.tensors, copy):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_nonfinite_addend_keeps_the_sums():
    gs = make_gradset("tiny", device=dev())
    last = make_gradset("tiny", seed=4321, device=dev())
    last.tensors[2].view(-1)[17] = math.nan
    r, _ = run(gs.tensors, last.tensors, 1.0, 0.25)
    assert r.decision == oracle.SKIP


def test_fp16_sum_overflows_to_inf():
    x = torch.full((1000,), 60000.0, dtype=torch.float16, device=dev())
    a = torch.full((1000,), 10000.0, dtype=torch.float16, device=dev())
    r, _ = run([x], [a], 1.0)
    assert r.decision == oracle.SKIP and torch.isinf(x).all()


def test_no_tensors():
    with g.GradClipper([]) as c:
        c.attach_addend([])
        norm, flag = c.clip_accumulate_(1.0)
        assert float(norm.item()) == 0.0 and int(flag.item()) == 0


def test_attach_rejects_bad_addends():
    x = torch.ones(64, device=dev())
    with g.GradClipper([x[:32], x[32:]]) as c:
        with pytest.raises(g.GclipError):
            c.clip_accumulate_(1.0)                                       # nothing attached
        with pytest.raises(g.GclipError):
            c.attach_addend([x[:32], torch.empty(32, device=dev())])      # addend = a gradient
        with pytest.raises(g.GclipError):
            c.attach_addend([torch.empty(32, device=dev())])              # one of two
        with pytest.raises(ValueError):
            c.attach_addend([torch.empty(32, device=dev(), dtype=torch.float16)] * 2)
        y = torch.empty(64, device=dev())
        with pytest.raises(g.GclipError):
            c.attach_addend([y[:32], y[16:48]])                           # addends overlap


def test_twenty_thousand_small_tensors():
    gen = torch.Generator(device="cpu").manual_seed(7)
    sizes = torch.randint(0, 10, (20000,), generator=gen).tolist()
    for i in range(0, 20000, 1000):
        sizes[i] = 3000 + i
    gbuf = torch.randn(sum(sizes) + 20000, generator=gen).to(dev())
    abuf = torch.randn(sum(sizes) + 40000, generator=gen).to(dev())
    grads, adds, go, ao = [], [], 0, 1
    for k in sizes:
        grads.append(gbuf[go:go + k])
        adds.append(abuf[ao:ao + k])
        go += k + 1
        ao += k + 2
    r, _ = run(grads, adds, 10.0, 0.5)
    assert r.decision == oracle.CLIP
