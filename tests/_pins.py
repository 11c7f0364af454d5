"""Pins for the oracle: facts fixed by the pages or by mathematics.

Each pin takes an `oracle.Oracle` and raises AssertionError when the oracle
disagrees with the fact.  `test_oracle_pins.py` runs them on the oracle as
built; `test_oracle_mutants.py` runs them on builds with planted mistakes and
requires every mistake to be caught by at least one pin.
"""
from __future__ import annotations

import math
import random
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch

from oracle import CLIP, PASS, SKIP, OracleTensor
from _helpers import as_float64, golden, make, ordered, storage_bits

DTYPES = ("f32", "f16", "bf16")


def _vals(t: OracleTensor) -> list:
    return list(as_float64(t))


# -- the pages' worked examples ---------------------------------------------

def pin_worked_example(o):
    """[6, 8] at threshold 5 gives [3, 4] (glossary page); exact in every
    storage format because 3, 4, 6, 8 and the factor 1/2 are exact."""
    g = golden("worked_example.txt")
    for dt in DTYPES:
        outs, r = o.clip([make(g["input"], dt)], g["threshold"])
        assert r.norm == g["norm"], (dt, r.norm)
        assert r.decision == CLIP, (dt, r.decision)
        assert _vals(outs[0]) == g["output"], (dt, _vals(outs[0]))


def pin_boundary_passthrough(o):
    """norm == max_norm and norm < max_norm both pass unchanged (strict '>' in
    the glossary's piecewise equation and the clipping page's Mathematics)."""
    g = golden("boundary_passthrough.txt")
    for dt in DTYPES:
        x = make(g["input"], dt)
        for c in (g["threshold_boundary"], g["threshold_above"]):
            outs, r = o.clip([x], c)
            assert r.decision == PASS, (dt, c, r.decision)
            assert np.array_equal(storage_bits(outs[0]), storage_bits(x)), (dt, c)
        # just below the boundary the clip fires
        _, r = o.clip([x], np.nextafter(g["threshold_boundary"], 0.0))
        assert r.decision == CLIP, (dt, r.decision)


def pin_per_coordinate_contrast(o):
    """Clamping coordinates to [-5, 5] gives [5, 5] with length ~7.07, while the
    norm clip gives [3, 4] (glossary page, 'Shorten the arrow')."""
    g = golden("per_coordinate_contrast.txt")
    v = o.value_clip(g["input"], g["interval"])
    assert list(v) == g["output"], v
    assert abs(float(np.hypot(*v)) - g["norm_about"]) < 0.005
    outs, _ = o.clip([make(g["input"], "f32")], g["interval"])
    assert _vals(outs[0]) != g["output"]
    # direction: the norm clip keeps the ratio 6:8, the clamp does not
    a = _vals(outs[0])
    assert a[0] * 8 == a[1] * 6 and v[0] * 8 != v[1] * 6


def pin_accumulation_order(o):
    """10 and -9 summed then clipped to [-5, 5] give 1; clipped separately then
    summed give 0 (glossary page, 'Order changes the result').  In one
    dimension the norm clip at threshold c is the clamp to [-c, c], so the
    global-norm clip shows the same counterexample."""
    g = golden("accumulation_order.txt")
    a, b = g["contributions"]
    c = g["interval"]
    assert o.value_clip([a + b], c)[0] == g["clip_of_sum"]
    assert sum(o.value_clip([a, b], c)) == g["sum_of_clips"]
    out_sum, r = o.clip([make([a + b], "f32")], c)
    assert _vals(out_sum[0]) == [g["clip_of_sum"]] and r.decision == PASS
    oa, _ = o.clip([make([a], "f32")], c)
    ob, _ = o.clip([make([b], "f32")], c)
    assert _vals(oa[0])[0] + _vals(ob[0])[0] == g["sum_of_clips"]


def pin_sgd_step_length(o):
    """SGD at lr 0.1: step length 0.5 clipped, 1 unclipped (glossary page)."""
    g = golden("sgd_step_length.txt")
    outs, _ = o.clip([make(g["input"], "f32")], g["threshold"])
    step = np.asarray(_vals(outs[0])) * g["lr"]
    assert abs(np.linalg.norm(step) - g["step_length_clipped"]) < 1e-15
    unclipped = np.asarray(g["input"]) * g["lr"]
    assert abs(np.linalg.norm(unclipped) - g["step_length_unclipped"]) < 1e-15


# -- global semantics ---------------------------------------------------------

def pin_global_not_per_tensor(o):
    """Global clipping scales every tensor by one factor and keeps their
    relative sizes; per-tensor clipping does not (clipping page, 'Per-Tensor
    or Global')."""
    big = make([6.0, 8.0], "f32")        # norm 10
    small = make([0.375, 0.5], "f32")    # norm 0.625
    outs, r = o.clip([big, small], 5.0)
    assert r.decision == CLIP
    # sum of squares 100 + 0.390625 exactly
    assert r.sumsq == 100.390625, r.sumsq
    ob, os_ = (as_float64(t) for t in outs)
    ratio = np.linalg.norm(ob) / np.linalg.norm(os_)
    assert abs(ratio - 16.0) < 1e-5, ratio                  # 10 / 0.625
    pt, prs = o.clip_per_tensor([big, small], 5.0)
    assert [p.decision for p in prs] == [CLIP, PASS]
    assert list(as_float64(pt[0])) == [3.0, 4.0]
    assert list(as_float64(pt[1])) == [0.375, 0.5]           # ratio now 8
    assert not np.array_equal(as_float64(pt[0]), ob)


def pin_per_tensor_isolation(o):
    """Per-tensor clipping treats each tensor alone (clipping page, "Per-Tensor
    or Global"): a NaN in one tensor skips only that tensor, and each of the
    others is scaled by its own max_norm / norm."""
    a = make([6.0, 8.0], "f32")            # norm 10 -> [3, 4] at 5
    b = make([1.0, math.nan], "f16")        # skipped, untouched
    c = make([0.6, 0.8], "bf16")           # norm ~1 < 5: passes unchanged
    outs, rs = o.clip_per_tensor([a, b, c], 5.0)
    assert [r.decision for r in rs] == [CLIP, SKIP, PASS]
    assert list(as_float64(outs[0])) == [3.0, 4.0]
    assert np.array_equal(storage_bits(outs[1]), storage_bits(b))
    assert np.array_equal(storage_bits(outs[2]), storage_bits(c))
    assert rs[0].norm == 10.0 and not math.isfinite(rs[1].norm)


def pin_post_clip_norm(o):
    """After a clip the new norm equals max_norm (clipping page, Mathematics);
    in fp32 storage, up to the rounding of each element."""
    rng = np.random.default_rng(7)
    ts = [make(rng.normal(0, 1, n), "f32") for n in (17, 256, 3)]
    outs, r = o.clip(ts, 2.5)
    assert r.decision == CLIP
    new = np.linalg.norm(np.concatenate([as_float64(t) for t in outs]))
    assert abs(new / 2.5 - 1.0) < 1e-6, new


def pin_direction_kept(o):
    """One common factor k in (0, 1] multiplies every element, so signs and
    ratios are kept (glossary page, 'Shorten the arrow, keep the direction')."""
    rng = np.random.default_rng(11)
    ts = [make(rng.normal(0, 3, n), "f32") for n in (64, 5)]
    outs, r = o.clip(ts, 1.0)
    x = np.concatenate([as_float64(t) for t in ts])
    y = np.concatenate([as_float64(t) for t in outs])
    nz = x != 0
    k = y[nz] / x[nz]
    assert np.all(k > 0) and np.all(k <= 1)
    assert np.max(np.abs(k / r.coef - 1)) < 2 ** -23, (k.min(), k.max(), r.coef)


def pin_unscale_before_clip(o):
    """With loss scaling the threshold applies to the unscaled gradients
    (glossary page, 'Order changes the result'): raw fp16 [768, 1024] under
    inv_scale 2^-10 is [0.75, 1.0] with norm 1.25."""
    raw = make([768.0, 1024.0], "f16")
    s = 2.0 ** -10
    outs, r = o.clip([raw], 2.0, s)           # scaled norm 1280 > 2, true 1.25
    assert r.decision == PASS, r.decision
    assert r.norm == 1.25
    assert list(as_float64(outs[0])) == [0.75, 1.0]   # unscale is written
    outs, r = o.clip([raw], 1.0, s)
    assert r.decision == CLIP and r.norm == 1.25
    want = make([0.6, 0.8], "f16")                    # 0.75*0.8, 1.0*0.8
    assert np.array_equal(storage_bits(outs[0]), storage_bits(want))


def pin_power_of_two_homogeneity(o):
    """For a power-of-two inv_scale the unscale is exact, so clipping raw
    gradients with inv_scale 2^-k equals clipping pre-divided ones with 1."""
    rng = np.random.default_rng(3)
    raw = [make(rng.normal(0, 64, n), "f32") for n in (33, 7)]
    pre = [make(as_float64(t) * 2.0 ** -6, "f32") for t in raw]
    a, ra = o.clip(raw, 3.0, 2.0 ** -6)
    b, rb = o.clip(pre, 3.0, 1.0)
    assert ra.sumsq == rb.sumsq and ra.decision == rb.decision == CLIP
    for x, y in zip(a, b):
        assert np.array_equal(storage_bits(x), storage_bits(y))


def pin_closed_form_constant(o):
    """||a * 1_n|| = |a| sqrt(n): exactly 16 for a = 0.5, n = 1024."""
    _, r = o.clip([make(np.full(1024, -0.5), "f32")], 100.0)
    assert r.norm == 16.0 and r.decision == PASS
    _, r = o.clip([make(np.full(7, 3.0), "bf16")], 100.0)
    assert abs(r.norm - 3 * math.sqrt(7)) <= 1e-15 * r.norm


def pin_closed_form_tiny_magnitudes(o):
    """||a * 1_n|| = |a| sqrt(n) where the squares lie far below fp32's range:
    a = 2^-80 (fp32), 2^-140 (an fp32 subnormal), 2^-100 (bf16), and fp16
    ones unscaled by 2^-100.  Every value is a power of two, so the norm and
    the clipped outputs are exact; the clip at half the norm halves them
    (and the fp16 result, 2^-102, is below fp16's range: +0)."""
    cases = [(2.0 ** -80, 1024, "f32", 1.0, 2.0 ** -75, 2.0 ** -81),
             (2.0 ** -140, 4096, "f32", 1.0, 2.0 ** -134, 2.0 ** -141),
             (-(2.0 ** -100), 16, "bf16", 1.0, 2.0 ** -98, -(2.0 ** -101)),
             (0.5, 256, "f16", 2.0 ** -100, 2.0 ** -97, 0.0)]
    for a, n, dt, inv, norm, out in cases:
        x = make(np.full(n, a), dt)
        _, r = o.clip([x], 1.0, inv)
        assert r.norm == norm and r.decision == PASS, (a, dt, r.norm)
        outs, r = o.clip([x], norm / 2, inv)
        assert r.decision == CLIP and r.coef == 0.5, (a, dt)
        assert np.all(as_float64(outs[0]) == out), (a, dt)


def pin_nonfinite(o):
    """NaN or +-inf raises the flag and leaves every gradient as it was
    (glossary page: a nonfinite value needs diagnosis and a stopped update)."""
    for bad in (math.inf, -math.inf, math.nan):
        for dt in DTYPES:
            x = make([1.0, bad, 2.0], dt)
            y = make([30.0, 40.0], dt)
            outs, r = o.clip([y, x], 1.0)
            assert r.nonfinite and r.decision == SKIP, (bad, dt)
            assert not math.isfinite(r.norm)
            assert np.array_equal(storage_bits(outs[1]), storage_bits(x))
            assert np.array_equal(storage_bits(outs[0]), storage_bits(y))


def pin_overflow_counts_as_nonfinite(o):
    """Finite elements whose squares sum past the largest fp32 value raise the
    flag (the sum is held in fp32 on the device)."""
    outs, r = o.clip([make([2e19, 1.0], "f32")], 1.0)       # 4e38 > FLT_MAX
    assert r.nonfinite and r.decision == SKIP
    _, r = o.clip([make([1.5e19], "bf16")], 1.0)            # ~2.25e38 < FLT_MAX
    assert not r.nonfinite and r.decision == CLIP


def pin_empty(o):
    """No tensors: norm 0, nothing to do.  Empty tensors change nothing."""
    _, r = o.clip([], 1.0)
    assert r.norm == 0.0 and r.decision == PASS and not r.nonfinite
    x = make([6.0, 8.0], "f32")
    e = OracleTensor(np.zeros(0, np.float32), "f32")
    outs, r = o.clip([e, x, e], 5.0)
    assert r.norm == 10.0 and list(as_float64(outs[1])) == [3.0, 4.0]


def pin_rejects_bad_arguments(o):
    x = make([1.0], "f32")
    for c, s in ((0.0, 1.0), (-1.0, 1.0), (math.nan, 1.0), (math.inf, 1.0),
                 (1.0, 0.0), (1.0, -2.0), (1.0, math.nan)):
        try:
            o.clip([x], c, s)
        except ValueError:
            continue
        raise AssertionError(f"accepted max_norm={c} inv_scale={s}")


# -- brute force with exact arithmetic ---------------------------------------

_FMT = {"f32": (np.float32, np.int32, 32), "f16": (np.float16, np.int16, 16)}


def _neighbours(t: OracleTensor, i: int):
    """The stored value at i and the two adjacent values of its format."""
    width = 32 if t.dtype == "f32" else 16
    k = int(ordered(storage_bits(t)[i:i + 1], width)[0])
    out = []
    for kk in (k - 1, k, k + 1):
        bits = kk if kk >= 0 else ((1 << (width - 1)) | (-kk))
        if t.dtype == "f32":
            v = np.array([bits], np.uint32).view(np.float32)[0]
        elif t.dtype == "f16":
            v = np.array([bits], np.uint16).view(np.float16)[0]
        else:
            v = np.array([bits << 16], np.uint32).view(np.float32)[0]
        out.append(Fraction(float(v)))
    return out


def pin_bruteforce_exact(o):
    """Tiny mixed sets against exact rationals: the sum of squares exactly,
    the norm to 50 digits, and every output the nearest value of its format
    to the exact clipped value."""
    getcontext().prec = 60
    rng = random.Random(2024)
    for trial in range(40):
        ts = []
        for _ in range(rng.randint(1, 4)):
            dt = rng.choice(DTYPES)
            n = rng.randint(0, 6)
            ts.append(make([rng.gauss(0, 2) for _ in range(n)], dt))
        inv_scale = rng.choice([1.0, 0.25, 0.3, 3.0])
        exact = sum((Fraction(float(v)) * Fraction(inv_scale)) ** 2
                    for t in ts for v in as_float64(t))
        norm = (Decimal(exact.numerator) / Decimal(exact.denominator)).sqrt()
        c = float(norm) * rng.choice([0.5, 0.9, 1.5])
        if c <= 0:
            c = 1.0
        outs, r = o.clip(ts, c, inv_scale)
        # sum of squares: double accumulation of a handful of terms
        assert abs(Fraction(r.sumsq) - exact) <= exact / 2 ** 48, trial
        assert abs(Decimal(r.norm) - norm) <= norm * Decimal(2) ** -50, trial
        clip = norm > Decimal(c)
        assert r.decision == (CLIP if clip else PASS), trial
        k = (Decimal(c) / norm) if clip else Decimal(1)
        for t_in, t_out in zip(ts, outs):
            for i, v in enumerate(as_float64(t_in)):
                want = Decimal(float(v)) * Decimal(inv_scale) * k
                wf = Fraction(want)
                lo, mid, hi = _neighbours(t_out, i)
                d = abs(mid - wf)
                slack = Fraction(1, 2 ** 40) * abs(wf)
                assert d <= abs(lo - wf) + slack and d <= abs(hi - wf) + slack, \
                    (trial, t_out.dtype, float(mid), float(wf))


# -- the storage-format conversions the oracle uses ---------------------------

def pin_f16_conversions(o):
    """Decoding every fp16 pattern, and encoding doubles, agree with numpy's
    IEEE binary16 conversions (a library routine)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    t = OracleTensor(bits.view(np.float16), "f16")
    dec = o.decode(t)
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(dec), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(dec[ok], ref[ok])
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.normal(0, 1, 2000) * 2.0 ** rng.integers(-30, 17, 2000),
        (np.arange(-2048, 2048) + 0.5) * 2.0 ** -24,              # subnormal ties
        (np.arange(1024, 2048) + 0.5) * 2.0 ** -10,               # normal ties
        [65504.0, 65519.0, 65520.0, 65536.0, 1e6, -1e6, 0.0, -0.0, 2.0 ** -25,
         2.0 ** -25 * 1.0000001, 6.1e-5]])
    enc = o.encode(v, "f16")
    with np.errstate(over="ignore"):
        want = v.astype(np.float16)
    assert np.array_equal(enc.data.view(np.uint16), want.view(np.uint16))


def pin_bf16_conversions(o):
    """bf16 decoding of every pattern and encoding of fp32 values agree with
    torch's bfloat16 conversions; a few hand-made ties with more than fp32
    precision check the direct rounding from double."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    t = OracleTensor(bits, "bf16")
    dec = o.decode(t)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(dec), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(dec[ok], ref[ok])
    rng = np.random.default_rng(6)
    with np.errstate(over="ignore"):
        big = (rng.normal(0, 1, 3000) * 2.0 ** rng.integers(-140, 127, 3000)).astype(np.float32)
    f = np.concatenate([
        big,
        ((np.arange(128, 256) + 0.5) * 2.0 ** -7).astype(np.float32),   # ties
        ((np.arange(0, 128) + 0.5) * 2.0 ** -133).astype(np.float32),   # subnormal ties
        np.array([3.3895314e38, 3.40e38, -3.40e38, 0.0], np.float32)])
    enc = o.encode(f.astype(np.float64), "bf16")
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(enc.data, want)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even significand wins (1);
    # the same plus 2^-40 is above the tie and rounds up.
    e = o.encode([1 + 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -40, 1 + 3 * 2.0 ** -8], "bf16")
    assert list(as_float64(e)) == [1.0, 1 + 2.0 ** -7, 1 + 2.0 ** -6]


def pin_round_grid_matches_c_cast(o):
    """The oracle's grid rounding with binary32 parameters agrees bit for bit
    with C's double-to-float conversion (numpy float32 cast)."""
    rng = np.random.default_rng(8)
    v = np.concatenate([
        rng.normal(0, 1, 3000) * 2.0 ** rng.integers(-150, 128, 3000),
        (np.arange(2 ** 23, 2 ** 23 + 200) + 0.5) * 2.0 ** -23,
        (np.arange(0, 200) + 0.5) * 2.0 ** -149,
        [3.4028235677973366e38, 3.4028235e38 * 1.0000001, 1e39, -0.0]])
    got = np.array([o.round_grid_f32_bits(float(x)) for x in v], np.uint32)
    with np.errstate(over="ignore"):
        want = v.astype(np.float32).view(np.uint32)
    assert np.array_equal(got, want)


def pin_sampled_outputs_match_full_clip(o):
    """The sampled-output entry point returns, at every chosen element, the
    bits the full clip writes there, and the same decision."""
    rng = np.random.default_rng(12)
    ts = [make(rng.normal(0, 1, n), dt) for n, dt in ((40, "f32"), (33, "f16"), (9, "bf16"))]
    for c, s in ((2.0, 1.0), (50.0, 0.5), (0.1, 2.0 ** -4)):
        outs, r = o.clip(ts, c, s)
        ti = np.repeat(np.arange(3), [40, 33, 9])
        ei = np.concatenate([np.arange(40), np.arange(33), np.arange(9)])
        slots, rs = o.clip_sample(ts, c, s, ti, ei)
        assert rs.decision == r.decision and rs.norm == r.norm
        got = np.concatenate([slots[:40], slots[40:73] & 0xFFFF, slots[73:] & 0xFFFF])
        want = np.concatenate([outs[0].data.view(np.uint32), outs[1].data.view(np.uint16),
                               outs[2].data]).astype(np.uint32)
        assert np.array_equal(got, want)


# -- out-of-place fp32 output ---------------------------------------------------

def pin_to_f32_matches_in_place_for_fp32(o):
    """For fp32 gradients the out-of-place fp32 result is the in-place result
    bit for bit (same decision, one rounding into the same format)."""
    rng = np.random.default_rng(31)
    ts = [make(rng.normal(0, 1, n), "f32") for n in (50, 3, 17)]
    for c, s_ in ((2.0, 1.0), (100.0, 0.25), (0.5, 0.3)):
        a, ra = o.clip(ts, c, s_)
        b, rb = o.clip_to_f32(ts, c, s_)
        assert ra.decision == rb.decision and ra.norm == rb.norm
        for x, y in zip(a, b):
            assert np.array_equal(x.data.view(np.int32), y.view(np.int32))


def pin_to_f32_keeps_what_fp16_loses(o):
    """Unscaling fp16 gradients by 2^-18 lands in the fp16 subnormal range:
    in place, 0x3fff (1.999...) x 2^-18 must round to 128 x 2^-24; the fp32
    output holds the exact value.  Both sides agree on the decision."""
    raw = OracleTensor(np.array([0x3FFF, 0x3C00, 0xBFFF], np.uint16).view(np.float16), "f16")
    s_ = 2.0 ** -18
    inplace, r1 = o.clip([raw], 1.0, s_)
    out, r2 = o.clip_to_f32([raw], 1.0, s_)
    assert r1.decision == r2.decision == PASS
    exact = as_float64(raw) * s_
    assert np.array_equal(out[0].astype(np.float64), exact)
    assert as_float64(inplace[0])[0] == 128 * 2.0 ** -24 != exact[0]


def pin_to_f32_skip_writes_nothing(o):
    out, r = o.clip_to_f32([make([1.0, math.inf], "bf16")], 1.0, fill=7.0)
    assert r.decision == SKIP and np.all(out[0] == 7.0)


# -- clip, then AdamW (the clipping page, "Order matters: Pre-Adam") ----------

def _adamw_case(seed, sizes=(37, 5), dt="f32", scale=1e-3):
    rng = np.random.default_rng(seed)
    grads = [make(rng.normal(0, scale, n), dt) for n in sizes]
    states = [(rng.normal(0, 0.02, n).astype(np.float32),
               rng.normal(0, 1e-4, n).astype(np.float32),
               np.abs(rng.normal(0, 1e-8, n)).astype(np.float32)) for n in sizes]
    return grads, states


def pin_adamw_matches_torch(o):
    """The AdamW step of the oracle equals torch.optim.AdamW (float64, one
    step, the same clipped gradient and state) after rounding to fp32."""
    for step, wd, dt in ((1, 0.0, "f32"), (1, 0.1, "f16"), (7, 0.1, "f32"), (200, 0.01, "bf16")):
        grads, states = _adamw_case(step, dt=dt)
        c, s_inv = 1e-3, 0.5                    # norm ~3e-3: the clip fires
        hp = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=wd, step=step)
        _, new, r = o.clip_adamw(grads, states, c, s_inv, **hp)
        assert r.decision == CLIP
        for gt, (w, m, v), (w1, m1, v1) in zip(grads, states, new):
            param = torch.tensor(w, dtype=torch.float64, requires_grad=True)
            opt = torch.optim.AdamW([param], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]),
                                    eps=hp["eps"], weight_decay=wd, foreach=False)
            opt.state[param] = {"step": torch.tensor(float(step - 1)),
                                "exp_avg": torch.tensor(m, dtype=torch.float64),
                                "exp_avg_sq": torch.tensor(v, dtype=torch.float64)}
            param.grad = torch.tensor(as_float64(gt) * s_inv * r.coef, dtype=torch.float64)
            opt.step()
            st = opt.state[param]
            for ours, theirs in ((w1, param.detach()), (m1, st["exp_avg"]), (v1, st["exp_avg_sq"])):
                ref = theirs.numpy().astype(np.float32)
                d = np.abs(ours.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
                assert d.max() <= 1, (step, dt, d.max())


def pin_adamw_first_step_closed_form(o):
    """From m = v = 0 at step 1 the bias-corrected moments are g^ and g^^2,
    so w' = w (1 - lr wd) - lr g^ / (|g^| + eps)."""
    x = np.array([3e-3, -4e-3, 1e-6, 0.0], np.float32)
    w = np.array([0.5, -0.25, 1e-3, 2.0], np.float32)
    z = np.zeros(4, np.float32)
    lr, wd, eps = 1e-3, 0.05, 1e-8
    _, new, r = o.clip_adamw([make(x, "f32")], [(w, z, z)], 1.0, 1.0, lr=lr, beta1=0.9,
                             beta2=0.999, eps=eps, weight_decay=wd, step=1)
    assert r.decision == PASS
    gh = x.astype(np.float64)
    want = w.astype(np.float64) * (1 - lr * wd) - lr * gh / (np.abs(gh) + eps)
    assert np.array_equal(new[0][0], want.astype(np.float32))
    assert np.array_equal(new[0][1], (0.1 * gh).astype(np.float32))
    assert np.array_equal(new[0][2], (0.001 * gh * gh).astype(np.float32))


def pin_adamw_update_bound(o):
    """The clipping page, "Adjacent activities": with warm-up lr 1.5e-7 and
    max_norm 1 the worst-case first-step change of a parameter is
    lr x max_norm = 1.5e-7, even under a 50x spike."""
    rng = np.random.default_rng(21)
    x = rng.normal(0, 3e-5, 5000)
    x[100:600] *= 50.0
    w = rng.normal(0, 1e-4, 5000).astype(np.float32)
    z = np.zeros(5000, np.float32)
    _, new, r = o.clip_adamw([make(x, "f32")], [(w, z, z)], 1.0, 1.0, lr=1.5e-7, step=1)
    dw = np.abs(new[0][0].astype(np.float64) - w.astype(np.float64))
    # plus the rounding of the stored fp32 weight
    assert np.all(dw <= 1.5e-7 + np.spacing(np.abs(new[0][0])).astype(np.float64)), dw.max()


def pin_adamw_pre_adam(o):
    """Pre-Adam order: the first moment sees the clipped gradient, so a spike
    enters m at max_norm / norm of its size."""
    x = np.array([600.0, 800.0], np.float32)        # norm 1000
    z = np.zeros(2, np.float32)
    _, new, r = o.clip_adamw([make(x, "f32")], [(z, z, z)], 1.0, 1.0, lr=1e-3, beta1=0.9,
                             step=1)
    assert r.decision == CLIP and r.coef == 1e-3
    assert np.array_equal(new[0][1], np.array([0.06, 0.08], np.float32))   # 0.1 * [0.6, 0.8]


def pin_adamw_skip_and_zero_grads(o):
    """A nonfinite gradient stops the update: w, m, v and the gradients stay
    as they were.  Otherwise zero_grads leaves every gradient at +0."""
    grads, states = _adamw_case(3)
    bad = [grads[0], make([1.0, math.nan], "f32")]
    sts = [states[0], (np.ones(2, np.float32),) * 3]
    g2, new, r = o.clip_adamw(bad, sts, 1.0, lr=1e-3, zero_grads=True)
    assert r.decision == SKIP
    for (a, b), (c, d) in zip(zip(sts, new), zip(bad, g2)):
        for x, y in zip(a, b):
            assert np.array_equal(x.view(np.int32), y.view(np.int32))
        assert np.array_equal(storage_bits(c), storage_bits(d))
    g3, _, r = o.clip_adamw(grads, states, 1e-6, lr=1e-3, zero_grads=True)
    assert r.decision == CLIP
    for t in g3:
        assert not storage_bits(t).any()


# -- the last microbatch's accumulation folded into the clip ------------------

def _ieee_sum(a: OracleTensor, b: OracleTensor) -> OracleTensor:
    """The sum of two stored tensors by numpy (fp32, fp16) or torch (bf16),
    whose additions round the exact sum once to nearest even."""
    with np.errstate(over="ignore"):        # a sum past the largest finite is inf
        if a.dtype == "f32":
            return OracleTensor((a.data + b.data).astype(np.float32), "f32")
        if a.dtype == "f16":
            return OracleTensor((a.data + b.data).astype(np.float16), "f16")
    ta = torch.from_numpy(a.data.view(np.int16).copy()).view(torch.bfloat16)
    tb = torch.from_numpy(b.data.view(np.int16).copy()).view(torch.bfloat16)
    return OracleTensor((ta + tb).view(torch.int16).numpy().view(np.uint16).copy(), "bf16")


def pin_accumulate_is_the_ieee_sum(o):
    """Each accumulated element is the stored sum the format's own addition
    gives (backprop page, 'Accumulation across microbatches': the backward
    kernels add into the buffer), including overflow to infinity, subnormal
    sums and the signs of zero."""
    rng = np.random.default_rng(77)
    for dt in DTYPES:
        big = {"f32": 3e38, "f16": 6e4, "bf16": 3e38}[dt]
        tiny = {"f32": 1e-45, "f16": 6e-8, "bf16": 1e-40}[dt]
        vals_a = np.concatenate([rng.normal(0, 1, 200), rng.normal(0, 1e-3, 50),
                                 [big, -big, tiny, -tiny, 0.0, -0.0, 0.0, 1.0]])
        vals_b = np.concatenate([rng.normal(0, 1, 200), rng.normal(0, 1, 50) * 1e3,
                                 [big, -big, tiny, tiny, -0.0, -0.0, 0.0, -1.0]])
        a, b = make(vals_a, dt), make(vals_b, dt)
        got = o.accumulate([a], [b])[0]
        want = _ieee_sum(a, b)
        assert np.array_equal(storage_bits(got), storage_bits(want)), dt
        # the inputs are left alone
        assert np.array_equal(storage_bits(a), storage_bits(make(vals_a, dt)))


def pin_accumulate_then_clip_worked_example(o):
    """Contributions [2, 3] and [4, 5] accumulate to the glossary's [6, 8],
    which the clip at threshold 5 turns into [3, 4]; contributions that cancel
    leave a zero gradient that passes."""
    g = golden("worked_example.txt")
    for dt in DTYPES:
        outs, r = o.clip_accumulate([make([2, 3], dt)], [make([4, 5], dt)], g["threshold"])
        assert r.decision == CLIP and r.norm == g["norm"], (dt, r)
        assert _vals(outs[0]) == g["output"], (dt, _vals(outs[0]))
        outs, r = o.clip_accumulate([make(g["input"], dt)],
                                    [make([-v for v in g["input"]], dt)], g["threshold"])
        assert r.decision == PASS and r.norm == 0.0, (dt, r)


def pin_accumulate_before_clip(o):
    """The clip acts on the accumulated sum, not on each contribution
    (glossary page, 'Order changes the result'): 10 and -9 accumulate to 1,
    which a threshold of 5 keeps; clipping the contributions first would give
    5 - 9 = -4 or 0."""
    g = golden("accumulation_order.txt")
    a, b = g["contributions"]
    for dt in DTYPES:
        outs, r = o.clip_accumulate([make([a], dt)], [make([b], dt)], g["interval"])
        assert r.decision == PASS, (dt, r.decision)
        assert _vals(outs[0]) == [g["clip_of_sum"]], (dt, _vals(outs[0]))


def pin_accumulate_bruteforce_exact(o):
    """Tiny mixed sets: the norm is that of the rounded sums (computed here
    with exact rationals from the IEEE sums), and every output is the nearest
    value of its format to the exact clipped sum."""
    getcontext().prec = 60
    rng = random.Random(99)
    for trial in range(30):
        acc, add = [], []
        for _ in range(rng.randint(1, 3)):
            dt = rng.choice(DTYPES)
            n = rng.randint(0, 5)
            acc.append(make([rng.gauss(0, 1) for _ in range(n)], dt))
            add.append(make([rng.gauss(0, 1) for _ in range(n)], dt))
        sums = [_ieee_sum(a, b) for a, b in zip(acc, add)]
        inv_scale = rng.choice([1.0, 0.5, 0.3])
        exact = sum((Fraction(float(v)) * Fraction(inv_scale)) ** 2
                    for t in sums for v in as_float64(t))
        norm = (Decimal(exact.numerator) / Decimal(exact.denominator)).sqrt()
        c = max(float(norm) * rng.choice([0.5, 1.5]), 1e-3)
        outs, r = o.clip_accumulate(acc, add, c, inv_scale)
        assert abs(Fraction(r.sumsq) - exact) <= exact / 2 ** 48, trial
        clip = norm > Decimal(c)
        assert r.decision == (CLIP if clip else PASS), trial
        k = (Decimal(c) / norm) if clip else Decimal(1)
        for t_sum, t_out in zip(sums, outs):
            for i, v in enumerate(as_float64(t_sum)):
                wf = Fraction(Decimal(float(v)) * Decimal(inv_scale) * k)
                lo, mid, hi = _neighbours(t_out, i)
                d = abs(mid - wf)
                slack = Fraction(1, 2 ** 40) * abs(wf)
                assert d <= abs(lo - wf) + slack and d <= abs(hi - wf) + slack, trial


def pin_accumulate_skip_keeps_the_sums(o):
    """A nonfinite contribution stops the update but not the accumulation:
    the buffer holds the sums (with the infinity), unscaled and unclipped."""
    acc = [make([1.0, 2.0], "f32"), make([3.0], "bf16")]
    add = [make([0.5, math.inf], "f32"), make([1.0], "bf16")]
    outs, r = o.clip_accumulate(acc, add, 1.0, 0.5)
    assert r.decision == SKIP and r.nonfinite
    assert _vals(outs[0]) == [1.5, math.inf] and _vals(outs[1]) == [4.0]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
