"""Parity at gradient magnitudes whose fp32 squares underflow.

The norm is defined over every element ("Grow a language model: gradient
clipping", section "Mathematics"), however small.  The device squares in
fp32, where |y| < 2^-63 would give a subnormal or zero square; the library
sums such elements in a second, power-of-two-scaled bin.  These cases put
every element (or every element of some tensors, or a random mix inside
vectors) at 1e-20, 1e-22 and 1e-25 (fp32 and bf16), at fp32 subnormal values,
and at fp16 values unscaled by 2^-100, and compare with the oracle (double
arithmetic, no underflow at these sizes) with the usual tolerances: the norm
within 1e-5, identical decisions, outputs within 2 ulp (fp32) or 1 ulp
(fp16/bf16).  Each case is clipped twice: with a threshold below the norm
(CLIP) and above it (PASS).
"""
import numpy as np
import pytest
import torch

import global_l2_norm_gb300 as g
import oracle
from _gpu import compare, gpu_clip, host_copies

pytestmark = pytest.mark.gpu

VARIANTS = ["split", "persistent", "split_tma", "persistent_tma", "split_wave", "three_kernel"]
TD = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
SIZES = [1_000_003, 40_961, 4_099, 257, 3]


@pytest.fixture(scope="module", autouse=True)
def built():
    g.build()


def carve(values, dt, seed):
    """One CUDA tensor per array of `values`, each starting at a seeded
    element offset inside its own allocation (ragged heads and tails)."""
    rng = np.random.default_rng(seed)
    out = []
    for v in values:
        off = int(rng.integers(0, 8))
        store = torch.empty(v.size + off, dtype=TD[dt], device="cuda")
        t = store[off:]
        t.copy_(torch.from_numpy(v).to(TD[dt]))
        out.append(t)
    return out


def uniform(sigma, dt, seed):
    rng = np.random.default_rng(seed)
    return carve([rng.standard_normal(n) * sigma for n in SIZES], dt, seed)


def mixed(dt, seed):
    """Every element's magnitude drawn from {1e-20, 1e-22, 1e-25}, so most
    16-byte vectors mix elements of different magnitudes; one tensor at a
    single magnitude of each."""
    rng = np.random.default_rng(seed)
    mags = np.array([1e-20, 1e-22, 1e-25])
    vals = [rng.standard_normal(n) * mags[rng.integers(0, 3, n)] for n in SIZES]
    vals += [rng.standard_normal(5000) * m for m in mags]
    return carve(vals, dt, seed)


def norm_of(ts, inv_scale):
    _, r = oracle.clip(host_copies(ts), 1.0, inv_scale)
    return r.norm


def clip_both_ways(ts, inv_scale, variant, name):
    """Clip a copy at half the oracle norm and the original at twice it."""
    norm = norm_of(ts, inv_scale)
    assert 0.0 < norm < 1e-10, norm
    copies = [t.clone() for t in ts]
    for tensors, factor, want in ((copies, 0.5, oracle.CLIP), (ts, 2.0, oracle.PASS)):
        max_norm = float(np.float32(norm * factor))
        before = host_copies(tensors)
        rec = gpu_clip(tensors, max_norm, inv_scale, variant)
        res = compare(before, tensors, rec, max_norm, inv_scale, name)
        assert res["oracle"].decision == want, (name, factor)
        assert res["norm_rel"] <= 1e-6, (name, res["norm_rel"])


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("sigma", [1e-20, 1e-22, 1e-25])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_uniform_tiny(variant, sigma, dt):
    clip_both_ways(uniform(sigma, dt, 7), 1.0, variant, f"{dt}:{sigma}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_mixed_tiny(variant, dt):
    clip_both_ways(mixed(dt, 11), 1.0, variant, f"mixed:{dt}")


@pytest.mark.parametrize("variant", ["split", "three_kernel", "split_tma"])
def test_fp32_subnormal_elements(variant):
    """Elements of magnitude ~1e-40, below fp32's normal range themselves;
    the norm (~1e-37) is a normal fp32 number."""
    clip_both_ways(uniform(1e-40, "f32", 13), 1.0, variant, "subnormal")


@pytest.mark.parametrize("variant", ["split", "three_kernel", "persistent"])
def test_fp16_unscaled_far_down(variant):
    """fp16 gradients of ordinary size under an inv_scale of 2^-100: the
    unscaled values (~1e-31) exist only inside the computation."""
    clip_both_ways(uniform(0.5, "f16", 17), 2.0 ** -100, variant, "f16-unscaled")


def test_tiny_mixed_with_ordinary_tensors():
    """Tiny tensors beside ordinary ones: the tiny bin still counts, and the
    two bins combine in one norm."""
    rng = np.random.default_rng(19)
    vals = [rng.standard_normal(300_001) * 1e-25, rng.standard_normal(70_001) * 3e-5,
            rng.standard_normal(9_999) * 1e-22]
    ts = carve(vals, "f32", 19)
    before = host_copies(ts)
    rec = gpu_clip(ts, 1e-4, 1.0, "split")
    res = compare(before, ts, rec, 1e-4, 1.0, "tiny+ordinary")
    assert res["oracle"].decision == oracle.CLIP


def test_per_tensor_tiny():
    ts = mixed("f32", 23)
    norms = [norm_of([t], 1.0) for t in ts]
    before = host_copies(ts)
    max_norm = float(np.float32(np.median(norms)))
    want, recs = oracle.default().clip_per_tensor(before, max_norm, 1.0)
    with g.GradClipper(ts) as c:
        c.clip_per_tensor_(max_norm, 1.0)
        got = c.per_tensor_results()
    for i, (r, gr) in enumerate(zip(recs, got)):
        assert gr["decision"] == r.decision, i
        assert abs(gr["norm"] - r.norm) <= 1e-5 * r.norm, (i, gr["norm"], r.norm)
    assert {r.decision for r in recs} == {oracle.CLIP, oracle.PASS}


def test_accumulate_tiny():
    """The accumulation epilogue's squares go through the same two bins."""
    rng = np.random.default_rng(29)
    xs = carve([rng.standard_normal(n) * 1e-22 for n in SIZES], "f32", 29)
    adds = [torch.from_numpy(rng.standard_normal(t.numel()) * 1e-22).float().cuda() for t in xs]
    sums = [x + a for x, a in zip(xs, adds)]          # torch's own fp32 addition
    norm = norm_of(sums, 1.0)
    max_norm = float(np.float32(norm / 2))
    before = host_copies(sums)
    with g.GradClipper(xs) as c:
        c.attach_addend(adds)
        c.clip_accumulate_(max_norm, 1.0)
        rec = c.result()
        rec["out_norm"], rec["out_flag"] = float(c.norm.item()), int(c.flag.item())
    res = compare(before, xs, rec, max_norm, 1.0, "accumulate-tiny")
    assert res["oracle"].decision == oracle.CLIP
