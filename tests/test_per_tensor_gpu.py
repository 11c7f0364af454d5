"""Per-tensor clipping on the GPU against the oracle, tensor by tensor.

Same tolerances as the global clip (tests/_gpu.py): each tensor's norm within
1e-5 relative, fp32 outputs within 2 ulp, fp16/bf16 within 1 ulp, decision
and flag identical, a skipped tensor bit-identical to its input.
"""
import math

import numpy as np
import pytest
import torch

import global_l2_norm_gb300 as g
import oracle
from _gpu import NORM_RTOL, ULP_TOL
from _helpers import storage_bits, to_oracle, ulp_distance
from workloads import make_gradset

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    g.build()


def dev():
    return torch.device("cuda", 0)


def check(tensors, max_norm, inv_scale=1.0):
    before = [to_oracle(t) for t in tensors]
    with g.GradClipper(tensors) as c:
        norms, flags = c.clip_per_tensor_(max_norm, inv_scale)
        recs = c.per_tensor_results()
        norms, flags = norms.cpu().numpy(), flags.cpu().numpy()
    want, rs = oracle.default().clip_per_tensor(before, max_norm, inv_scale)
    decisions = []
    for i, (b, t, w, r, rec) in enumerate(zip(before, tensors, want, rs, recs)):
        assert rec["decision"] == r.decision and bool(rec["nonfinite"]) == r.nonfinite, i
        assert flags[i] == int(r.nonfinite) and norms[i] == rec["norm"] or math.isnan(norms[i])
        if r.nonfinite:
            assert not math.isfinite(rec["norm"])
            assert np.array_equal(storage_bits(b), storage_bits(to_oracle(t)))
        else:
            tol = NORM_RTOL * r.norm if r.norm else 0.0
            assert abs(rec["norm"] - r.norm) <= tol, (i, rec["norm"], r.norm)
            got = to_oracle(t)
            if got.data.size:
                assert int(ulp_distance(got, w).max()) <= ULP_TOL[w.dtype], i
        decisions.append(r.decision)
    return decisions


def test_andrea120m_only_the_spike_clips():
    gs = make_gradset("andrea120m", device=dev())
    d = check(gs.tensors, gs.max_norm)
    spiked = [s.name for s in gs.workload.layout].index(gs.spiked[0])
    assert d[spiked] == oracle.CLIP
    assert d.count(oracle.CLIP) == 1 and d.count(oracle.PASS) == len(d) - 1


def test_many_tensors_clip_with_unscale():
    gs = make_gradset("andrea14m", device=dev())
    d = check(gs.tensors, 0.01, 0.5)
    assert oracle.CLIP in d and oracle.PASS in d


def test_fp16_and_bf16():
    for name in ("andrea120m_fp16", "andrea120m_bf16"):
        gs = make_gradset(name, device=dev())
        check(gs.tensors, 0.02, gs.inv_scale)


def test_ragged_mixed_with_a_nan_and_empties():
    gen = torch.Generator(device="cpu").manual_seed(4)
    sizes = [0, 1, 3, 17, 8191, 8193, 0, 16385, 100003, 5]
    dts = [torch.float32, torch.float16, torch.bfloat16]
    ts = []
    for i, n in enumerate(sizes):
        v = torch.randn(n, generator=gen) * (0.5 if i % 2 else 0.001)
        ts.append(v.to(dts[i % 3]).to(dev()))
    ts[4].view(-1)[100] = float("nan")
    d = check(ts, 0.8)
    assert d[4] == oracle.SKIP and d[0] == d[6] == oracle.PASS


def test_no_tensors():
    with g.GradClipper([]) as c:
        c.clip_per_tensor_(1.0)
        assert c.per_tensor_results() == []


def test_repeated_calls_reuse_the_write_list():
    """Calls on one clipper: everything rewritten (unscale), then nothing
    (every tensor passes at multiplier 1), then a few tensors clip."""
    gs = make_gradset("andrea14m", device=dev())
    with g.GradClipper(gs.tensors) as c:
        for max_norm, inv_scale, expect_writes in ((1e6, 0.5, True), (1e6, 1.0, False),
                                                    (0.02, 1.0, True)):
            before = [to_oracle(t) for t in gs.tensors]
            c.clip_per_tensor_(max_norm, inv_scale)
            recs = c.per_tensor_results()
            want, rs = oracle.default().clip_per_tensor(before, max_norm, inv_scale)
            wrote = False
            for b, t, w, r, rec in zip(before, gs.tensors, want, rs, recs):
                assert rec["decision"] == r.decision
                got = to_oracle(t)
                assert int(ulp_distance(got, w).max()) <= ULP_TOL[w.dtype]
                wrote |= not np.array_equal(storage_bits(got), storage_bits(b))
            assert wrote == expect_writes, (max_norm, inv_scale)


def test_only_empty_tensors():
    ts = [torch.empty(0, device=dev()), torch.empty(0, device=dev(), dtype=torch.float16)]
    with g.GradClipper(ts) as c:
        norms, flags = c.clip_per_tensor_(1.0, 0.5)
        assert norms.tolist() == [0.0, 0.0] and flags.tolist() == [0, 0]


def test_twenty_thousand_small_tensors():
    gen = torch.Generator(device="cpu").manual_seed(6)
    sizes = torch.randint(0, 10, (20000,), generator=gen).tolist()
    for i in range(0, 20000, 1000):
        sizes[i] = 3000 + i
    buf = torch.randn(sum(sizes) + 20000, generator=gen).to(dev())
    ts, pos = [], 0
    for k in sizes:
        ts.append(buf[pos:pos + k])
        pos += k + 1
    d = check(ts, 2.0, 0.5)
    assert oracle.CLIP in d and oracle.PASS in d
