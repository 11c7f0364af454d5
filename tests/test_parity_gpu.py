"""Parity of the CUDA path with the oracle, through the C ABI, on the GPU."""
import math

import numpy as np
import pytest
import torch

import global_l2_norm_gb300 as g
import oracle
from _gpu import clone_all, compare, gpu_clip, host_copies, restore
from _helpers import golden, storage_bits, to_oracle, ulp_distance
from oracle import OracleTensor
from workloads import WORKLOADS, make_gradset

pytestmark = pytest.mark.gpu

VARIANTS = ["split", "persistent", "split_tma", "persistent_tma", "split_wave", "three_kernel"]
TD = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def built():
    g.build()


def dev():
    return torch.device("cuda", 0)


# -- the pages' worked example -----------------------------------------------

@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_worked_example(variant, dt):
    ex = golden("worked_example.txt")
    x = torch.tensor(ex["input"], dtype=TD[dt], device=dev())
    rec = gpu_clip([x], ex["threshold"], variant=variant)
    assert rec["norm"] == ex["norm"] and rec["decision"] == g.GCLIP_DECISION_CLIP
    assert x.double().cpu().tolist() == ex["output"]


@pytest.mark.parametrize("variant", VARIANTS)
def test_boundary_passes_without_writing(variant):
    ex = golden("boundary_passthrough.txt")
    for c in (ex["threshold_boundary"], ex["threshold_above"]):
        x = torch.tensor(ex["input"], dtype=torch.float32, device=dev())
        rec = gpu_clip([x], c, variant=variant)
        assert rec["decision"] == g.GCLIP_DECISION_PASS
        assert x.cpu().tolist() == ex["output"]
        assert rec["coef_hi"] == 1.0 and rec["coef_lo"] == 0.0


# -- seeded workloads ----------------------------------------------------------

@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["tiny", "andrea14m"])
def test_small_workloads(variant, name):
    gs = make_gradset(name, device=dev())
    before = host_copies(gs.tensors)
    rec = gpu_clip(gs.tensors, gs.max_norm, gs.inv_scale, variant)
    res = compare(before, gs.tensors, rec, gs.max_norm, gs.inv_scale, name)
    expect = {"tiny": oracle.CLIP, "andrea14m": oracle.PASS}[name]
    assert res["oracle"].decision == expect


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["andrea120m", "andrea120m_fp16", "andrea120m_fp16_inf",
                                  "andrea120m_bf16"])
def test_andrea120m(variant, name):
    gs = make_gradset(name, device=dev())
    before = host_copies(gs.tensors)
    rec = gpu_clip(gs.tensors, gs.max_norm, gs.inv_scale, variant)
    res = compare(before, gs.tensors, rec, gs.max_norm, gs.inv_scale, name)
    expect = {"andrea120m": oracle.CLIP, "andrea120m_bf16": oracle.CLIP,
              "andrea120m_fp16": oracle.PASS, "andrea120m_fp16_inf": oracle.SKIP}[name]
    assert res["oracle"].decision == expect
    if name == "andrea120m_fp16":
        # the unscale by 2^-18 is exact before the final rounding: bit-exact
        assert res["worst_ulp"]["f16"] == 0


@pytest.mark.parametrize("variant", ["split", "persistent", "split_tma", "three_kernel"])
def test_andrea1p2b(variant):
    gs = make_gradset("andrea1p2b", device=dev())
    before = host_copies(gs.tensors)
    rec = gpu_clip(gs.tensors, gs.max_norm, gs.inv_scale, variant)
    res = compare(before, gs.tensors, rec, gs.max_norm, gs.inv_scale, "andrea1p2b")
    assert res["oracle"].decision == oracle.CLIP


# -- ragged, misaligned, mixed, guarded ----------------------------------------

SIZES = [0, 1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 33, 255, 256, 257, 1023, 2047, 4095,
         8191, 8192, 8193, 16383, 16384, 16385, 100003]
GUARD = 64  # bytes of sentinel on each side of every tensor


def carve(sizes, dtypes, offsets, seed):
    """Tensors cut from one byte buffer at the given element offsets, with
    sentinel bands between them."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    layout, pos = [], 0
    for n, dt, off in zip(sizes, dtypes, offsets):
        es = 4 if dt == "f32" else 2
        pos += GUARD
        pos = (pos + 15) // 16 * 16 + off * es
        layout.append((pos, n, dt))
        pos += n * es
    pos += GUARD
    buf = torch.full((pos,), 0xA5, dtype=torch.uint8, device=dev())
    tensors = []
    for p, n, dt in layout:
        es = 4 if dt == "f32" else 2
        t = buf[p:p + n * es].view(TD[dt])
        vals = torch.randn(n, generator=gen) * 0.5
        t.copy_(vals.to(TD[dt]).to(dev()))
        tensors.append(t)
    return buf, layout, tensors


def guards_intact(buf, layout):
    mask = torch.ones(buf.numel(), dtype=torch.bool, device=buf.device)
    for p, n, dt in layout:
        es = 4 if dt == "f32" else 2
        mask[p:p + n * es] = False
    return bool((buf[mask] == 0xA5).all())


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("max_norm,inv_scale", [(1.0, 1.0), (1e6, 1.0), (2.0, 2.0 ** -10),
                                                (1e6, 2.0 ** -3), (0.5, 0.3)])
def test_ragged_mixed_guarded(variant, max_norm, inv_scale):
    rng = np.random.default_rng(17)
    dts = [str(rng.choice(["f32", "f16", "bf16"])) for _ in SIZES]
    offs = [int(rng.integers(0, 8)) for _ in SIZES]
    buf, layout, ts = carve(SIZES, dts, [o % (4 if d == "f32" else 8) for o, d in zip(offs, dts)], 5)
    before = host_copies(ts)
    inv = float(np.float32(inv_scale))
    rec = gpu_clip(ts, max_norm, inv, variant)
    compare(before, ts, rec, max_norm, inv, "ragged")
    assert guards_intact(buf, layout)


@pytest.mark.parametrize("variant", VARIANTS)
def test_every_size_alone(variant):
    """Each ragged size as a one-tensor set at every misalignment."""
    for n in [1, 3, 5, 17, 257, 8191, 8193, 16385]:
        for dt in ("f32", "f16", "bf16"):
            per = 4 if dt == "f32" else 8
            for off in range(per):
                buf, layout, ts = carve([n], [dt], [off], n * 31 + off)
                before = host_copies(ts)
                rec = gpu_clip(ts, 0.25, 1.0, variant)
                compare(before, ts, rec, 0.25, 1.0, f"{dt}:{n}:{off}")
                assert guards_intact(buf, layout)


# -- edge cases -------------------------------------------------------------------

@pytest.mark.parametrize("variant", VARIANTS)
def test_empty_sets(variant):
    rec = gpu_clip([], 1.0, variant=variant)
    assert rec["norm"] == 0.0 and rec["decision"] == g.GCLIP_DECISION_PASS
    e = torch.empty(0, device=dev())
    rec = gpu_clip([e, e.clone()], 1.0, variant=variant)
    assert rec["norm"] == 0.0 and rec["nonfinite"] == 0


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("bad", [math.inf, -math.inf, math.nan])
def test_nonfinite_leaves_everything(variant, bad):
    gs = make_gradset("andrea14m", device=dev())
    gs.tensors[5].view(-1)[1234] = bad
    before = host_copies(gs.tensors)
    rec = gpu_clip(gs.tensors, 1e-3, 1.0, variant)
    assert rec["nonfinite"] == 1 and rec["decision"] == g.GCLIP_DECISION_SKIP
    compare(before, gs.tensors, rec, 1e-3, 1.0, "nonfinite")


@pytest.mark.parametrize("variant", VARIANTS)
def test_overflow_counts_as_nonfinite(variant):
    x = torch.tensor([2e19, 1.0, 3.0], device=dev())
    before = host_copies([x])
    rec = gpu_clip([x], 1.0, 1.0, variant)
    assert rec["nonfinite"] == 1
    compare(before, [x], rec, 1.0, 1.0, "overflow")


@pytest.mark.parametrize("variant", VARIANTS)
def test_sum_of_squares_exactly_at_flt_max(variant):
    """A set whose fp32 sum of squares rounds to exactly FLT_MAX: (2^64 (1 -
    2^-24))^2 rounds to 2^128 (1 - 2^-23), plus (2^52)^2 is FLT_MAX.  The sum
    is finite on the device, so the norm must be sqrt(FLT_MAX) and the clip
    must scale, not produce a NaN (the exact sum lies one ulp above FLT_MAX,
    inside the band around that threshold where the device's fp32 sum and
    the oracle's exact one may decide differently, so this case is checked
    for consistency rather than against the oracle)."""
    x = torch.tensor([2.0 ** 64 * (1 - 2.0 ** -24), 2.0 ** 52, 0.0, 0.0], device=dev())
    assert x.data_ptr() % 16 == 0
    orig = x.double().cpu()
    rec = gpu_clip([x], 1.0, 1.0, variant)
    norm = float(np.float32(math.sqrt(float(np.finfo(np.float32).max))))
    assert rec["nonfinite"] == 0 and rec["decision"] == g.GCLIP_DECISION_CLIP, rec
    assert rec["norm"] == norm, (rec["norm"], norm)
    want = (orig / math.sqrt(float(np.finfo(np.float32).max))).float()
    got = x.cpu()
    d = ulp_distance(OracleTensor(got.numpy(), "f32"), OracleTensor(want.numpy(), "f32"))
    assert int(d.max()) <= 2, (got, want)


def test_largest_tensor_64bit_offsets():
    """One fp16 tensor of 2^31 + 37 elements (4.3 GB): chunk addresses past
    2^32 bytes; the norm against the oracle, outputs on a sample (both ends
    and 4096 random elements) that the oracle computes one by one."""
    n = 2 ** 31 + 37
    x = torch.empty(n, dtype=torch.float16, device=dev())
    gen = torch.Generator(device=dev()).manual_seed(99)
    x.normal_(0.0, 1.0, generator=gen)
    host = to_oracle(x)
    with g.GradClipper([x]) as c:
        c.clip_(100.0, 1.0)
        rec = c.result()
    idx = np.concatenate([np.arange(0, 64), np.arange(n - 64, n),
                          np.random.default_rng(1).integers(0, n, 4096)])
    slots, r = oracle.default().clip_sample([host], 100.0, 1.0, np.zeros(idx.size), idx)
    assert rec["decision"] == r.decision == oracle.CLIP
    assert abs(rec["norm"] - r.norm) / r.norm < 1e-5
    got = x[torch.from_numpy(idx).to(dev())].cpu().numpy()
    want = (slots & 0xFFFF).astype(np.uint16).view(np.float16)
    d = ulp_distance(OracleTensor(got, "f16"), OracleTensor(want, "f16"))
    assert d.max() <= 1


@pytest.mark.parametrize("variant", VARIANTS)
def test_null_outputs_and_side_stream(variant):
    gs = make_gradset("tiny", device=dev())
    before = host_copies(gs.tensors)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with g.GradClipper(gs.tensors, variant=variant) as c:
        L = g.load()
        assert L.clip_grad_norm(c._h, 1.0, 1.0, None, None, s.cuda_stream) == 0
        rec = c.result(stream=s)
    rec["out_norm"], rec["out_flag"] = rec["norm"], rec["nonfinite"]
    compare(before, gs.tensors, rec, 1.0, 1.0, "stream")


def test_scalar_arguments_rejected():
    x = torch.ones(8, device=dev())
    with g.GradClipper([x]) as c:
        L = g.load()
        for m, s in ((0.0, 1.0), (-1.0, 1.0), (math.nan, 1.0), (math.inf, 1.0),
                     (1.0, 0.0), (1.0, -1.0), (1.0, math.inf)):
            assert L.clip_grad_norm(c._h, m, s, None, None, None) == g._abi.GCLIP_ERR_INVALID_ARG
        assert L.clip_set_variant(c._h, 7) == g._abi.GCLIP_ERR_INVALID_ARG
    assert x.cpu().tolist() == [1.0] * 8


def test_rejects_host_memory_descriptor():
    """Host tensors are not device memory; the library must not be handed
    them (the binding refuses before the C call)."""
    with pytest.raises(ValueError):
        g.GradClipper([torch.ones(4)])


# -- determinism ----------------------------------------------------------------

@pytest.mark.parametrize("pair", [("split", "persistent"), ("split_tma", "persistent_tma"),
                                  ("split", "split_wave"), ("three_kernel", "three_kernel")])
def test_bit_identical_runs_and_variants(pair):
    """100 runs alternating the two variants of one engine: the same norm,
    sum of squares and multiplier bit for bit, and the same outputs."""
    gs = make_gradset("andrea120m", device=dev())
    pristine = clone_all(gs.tensors)
    records, outs = [], []
    with g.GradClipper(gs.tensors) as c:
        for i in range(100):
            c.set_variant(pair[i % 2])
            restore(gs.tensors, pristine)
            c.clip_(gs.max_norm, gs.inv_scale)
            r = c.result()
            records.append((r["norm"], r["sumsq_hi"], r["sumsq_lo"], r["coef_hi"], r["coef_lo"]))
            if i < 2:
                outs.append([storage_bits(to_oracle(t)) for t in gs.tensors[:6]])
    assert len(set(records)) == 1, set(records)
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)


def test_split_scaling_follows_the_last_decision():
    """SPLIT chooses its scaling launch (one block per chunk, or one claiming
    wave) from the decision of the last call that has completed on the
    handle.  Alternating clipping and no-write calls makes every guess wrong,
    repeated decisions make them right; every call matches the oracle."""
    gs = make_gradset("andrea14m", device=dev())          # norm ~0.378
    pristine = clone_all(gs.tensors)
    with g.GradClipper(gs.tensors) as c:
        for i, m in enumerate([1.0, 0.1, 1.0, 0.1, 0.1, 1.0, 1.0, 0.1, 0.1]):
            restore(gs.tensors, pristine)
            before = host_copies(gs.tensors)
            c.clip_(m, 1.0)
            rec = c.result()
            rec["out_norm"], rec["out_flag"] = float(c.norm.item()), int(c.flag.item())
            res = compare(before, gs.tensors, rec, m, 1.0, f"call {i}")
            assert res["oracle"].decision == (oracle.CLIP if m < 0.3 else oracle.PASS)


def test_clip_twice_is_stable():
    """After a clip the norm is max_norm: a second call sees norm ~= 1."""
    gs = make_gradset("andrea14m", device=dev())
    for t in gs.tensors:
        t.mul_(100.0)
    with g.GradClipper(gs.tensors) as c:
        c.clip_(1.0)
        first = c.result()
        c.clip_(1.0)
        second = c.result()
    assert first["decision"] == g.GCLIP_DECISION_CLIP
    assert abs(second["norm"] - 1.0) < 1e-6


@pytest.mark.parametrize("name", ["andrea14m", "andrea120m"])
def test_back_to_back_writing_calls_see_each_other(name):
    """Calls enqueued back to back with no host wait, each halving every
    element (inv_scale 1/2, no clip): each call's scaling pass reads what the
    previous call's scaling pass wrote, although its first blocks load before
    its decision is out and the calls overlap through programmatic dependent
    launch.  Power-of-two scaling of normal fp32 values is exact, so after k
    calls every element is x / 2^k bit for bit, and the last call's norm is
    the first call's / 2^(k-1) (sums of squares scale exactly by 4^-j)."""
    gs = make_gradset(name, device=dev())
    before = [t.clone() for t in gs.tensors]
    with g.GradClipper([t.clone() for t in before], variant="split") as c1:
        c1.clip_(1e30, 0.5)
        first = c1.result()["norm"]
    k = 6
    with g.GradClipper(gs.tensors, variant="split") as c:
        for _ in range(k):
            c.clip_(1e30, 0.5)
        torch.cuda.synchronize()
        rec = c.result()
    assert rec["decision"] == g.GCLIP_DECISION_PASS and rec["nonfinite"] == 0
    for t, b in zip(gs.tensors, before):
        assert torch.equal(t, b * 2.0 ** -k)
    assert rec["norm"] == first * 2.0 ** -(k - 1), (rec["norm"], first)


@pytest.mark.parametrize("name", ["andrea120m", "andrea120m_fp16"])
def test_pool_back_to_back_as_the_bench_runs_it(name):
    """The bench's timed loop: a pool of distinct sets, each with its own
    handle, clipped back to back on one stream with no host wait, so that
    each clip's launches are chained to the previous clip's (another set) by
    programmatic dependent launch.  Pass 1 writes (clip, or the fp16 unscale)
    and matches the oracle set by set.  Passes 2 and 3 write nothing (pass 2
    launches the one-block-per-chunk scaling pass, whose first wave loads
    before the decision; pass 3 the claiming wave) and leave every bit as it
    was.  Pass 4 clips again after a no-write call and matches the oracle."""
    sets = [make_gradset(name, seed=1234 + 7 * k, device=dev(), flat=True) for k in range(4)]
    clippers = [g.GradClipper(s.tensors, variant="split") for s in sets]

    def run_pass(max_norm, inv_scale):
        for c in clippers:
            c.clip_(max_norm, inv_scale)
        torch.cuda.synchronize()
        recs = []
        for c in clippers:
            rec = c.result()
            rec["out_norm"], rec["out_flag"] = float(c.norm.item()), int(c.flag.item())
            recs.append(rec)
        return recs

    try:
        before = [host_copies(s.tensors) for s in sets]
        recs = run_pass(sets[0].max_norm, sets[0].inv_scale)
        for k, (b, s, rec) in enumerate(zip(before, sets, recs)):
            compare(b, s.tensors, rec, s.max_norm, s.inv_scale, f"{name} pass 1 set {k}")
        after = [clone_all(s.tensors) for s in sets]
        for p in (2, 3):
            recs = run_pass(2.0, 1.0)
            for k, (s, a, rec) in enumerate(zip(sets, after, recs)):
                assert rec["decision"] == g.GCLIP_DECISION_PASS, (p, k, rec)
                assert all(torch.equal(x, y) for x, y in zip(s.tensors, a)), (p, k)
        before = [host_copies(s.tensors) for s in sets]
        norms = [r["norm"] for r in recs]
        recs = run_pass(0.5 * min(norms), 1.0)
        for k, (b, s, rec) in enumerate(zip(before, sets, recs)):
            res = compare(b, s.tensors, rec, 0.5 * min(norms), 1.0, f"{name} pass 4 set {k}")
            assert res["oracle"].decision == oracle.CLIP
    finally:
        for c in clippers:
            c.close()


# -- the single-launch variant's bounded barrier --------------------------------

@pytest.mark.parametrize("variant", ["persistent", "persistent_tma"])
def test_barrier_timeout_reports_and_writes_nothing(variant):
    gs = make_gradset("andrea14m", device=dev())
    before = host_copies(gs.tensors)
    with g.GradClipper(gs.tensors, variant=variant) as c:
        c.debug_barrier(1, 20_000_000)     # one arrival that never comes; 20 ms
        c.clip_(1e-3)
        status = c.last_status()
        rec = c.result()
        assert rec["status"] == g.GCLIP_STATUS_TIMEOUT
        assert int(status.item()) == g.GCLIP_STATUS_TIMEOUT
        for b, t in zip(before, gs.tensors):
            assert np.array_equal(storage_bits(b), storage_bits(to_oracle(t)))
        c.debug_barrier(0)
        c.reset()
        c.clip_(1e-3)
        status = c.last_status()
        rec = c.result()
        assert rec["status"] == g.GCLIP_STATUS_OK
        assert int(status.item()) == g.GCLIP_STATUS_OK
        assert rec["decision"] == g.GCLIP_DECISION_CLIP
    rec["out_norm"], rec["out_flag"] = rec["norm"], rec["nonfinite"]
    compare(before, gs.tensors, rec, 1e-3, 1.0, "after-timeout")


# -- CUDA graph capture ------------------------------------------------------------

@pytest.mark.parametrize("variant", VARIANTS)
def test_captured_in_a_cuda_graph(variant):
    """clip_grad_norm enqueues launches only (no sync, no allocation), so it
    can be captured; replays of the graph clip the same buffers."""
    gs = make_gradset("andrea14m", device=dev())
    for t in gs.tensors:
        t.mul_(40.0)                                   # the clip fires
    pristine = clone_all(gs.tensors)
    before = host_copies(gs.tensors)
    with g.GradClipper(gs.tensors, variant=variant) as c:
        c.clip_(1.0, 0.5)                              # first call outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            c.clip_(1.0, 0.5)
        for _ in range(2):
            restore(gs.tensors, pristine)
            graph.replay()
            torch.cuda.synchronize()
            rec = c.result()
            rec["out_norm"], rec["out_flag"] = float(c.norm.item()), int(c.flag.item())
            compare(before, gs.tensors, rec, 1.0, 0.5, "graph")


def test_graph_captured_after_a_no_write_call():
    """A SPLIT clip captured right after a call that wrote nothing keeps the
    claiming-wave scaling it chose then; replayed on gradients that clip, it
    must still write every element correctly."""
    gs = make_gradset("andrea14m", device=dev())          # norm ~0.378: no write at 1.0
    pristine = clone_all(gs.tensors)
    before = host_copies(gs.tensors)
    with g.GradClipper(gs.tensors) as c:
        c.clip_(1.0)
        assert c.result()["decision"] == g.GCLIP_DECISION_PASS   # synchronises: the hint is set
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            c.clip_(0.1, 0.5)
        for _ in range(2):
            restore(gs.tensors, pristine)
            graph.replay()
            torch.cuda.synchronize()
            rec = c.result()
            rec["out_norm"], rec["out_flag"] = float(c.norm.item()), int(c.flag.item())
            res = compare(before, gs.tensors, rec, 0.1, 0.5, "graph-after-pass")
            assert res["oracle"].decision == oracle.CLIP


# -- accuracy of the norm -------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "andrea14m", "andrea120m", "andrea120m_fp16",
                                  "andrea120m_bf16"])
def test_norm_is_the_rounded_exact_norm(name):
    """The float-float sum is good to ~2^-44, so the reported fp32 norm is the
    oracle's (exact up to fp64 rounding) norm rounded to fp32 - at most one
    ulp away in the rare case that the exact value sits next to a rounding
    boundary.  A plain fp32 tree sum would drift several ulp at 92M terms."""
    gs = make_gradset(name, device=dev())
    before = host_copies(gs.tensors)
    with g.GradClipper(gs.tensors) as c:
        c.clip_(gs.max_norm, gs.inv_scale)
        got = np.float32(c.result()["norm"])
    _, r = oracle.default().clip(before, gs.max_norm, gs.inv_scale)
    want = np.float32(r.norm)
    ulps = abs(int(np.array([got]).view(np.int32)[0]) - int(np.array([want]).view(np.int32)[0]))
    assert ulps <= 1, (float(got), float(want), ulps)


# -- many small tensors -------------------------------------------------------------

def many_small(seed, n=20000, dt=torch.float32):
    """n tensors of 0..9 elements (plus every 1000th of a few thousand), cut
    out of one buffer at odd element offsets: most chunks are only a head or
    a tail, with no vector body."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    sizes = torch.randint(0, 10, (n,), generator=gen).tolist()
    for i in range(0, n, 1000):
        sizes[i] = 3000 + i
    buf = torch.randn(sum(sizes) + n, generator=gen).to(dt).to(dev())
    ts, pos = [], 0
    for k in sizes:
        ts.append(buf[pos:pos + k])
        pos += k + 1
    return ts


@pytest.mark.parametrize("variant", ["split", "persistent", "split_tma", "three_kernel"])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_twenty_thousand_small_tensors(variant, dt):
    ts = many_small(5, dt=dt)
    before = host_copies(ts)
    rec = gpu_clip(ts, 10.0, 0.5, variant)
    compare(before, ts, rec, 10.0, 0.5, f"many-{variant}")
    assert rec["decision"] == g.GCLIP_DECISION_CLIP


# -- cache hints change timing only ---------------------------------------------------

@pytest.mark.parametrize("name", ["andrea14m", "andrea120m"])
def test_l2_hints_do_not_change_results(name):
    """The 14M set is read with the normal L2 policy, the 120M set with
    evict_first plus the next-chunk prefetch; an evict_last keep region on
    top changes neither the record nor a single output bit."""
    gs = make_gradset(name, device=dev())
    for t in gs.tensors:
        t.mul_(30.0)                                   # the clip fires on both sets
    other = [t.clone() for t in gs.tensors]
    recs = []
    for ts, keep in ((gs.tensors, 0), (other, 64 << 20)):
        with g.GradClipper(ts) as c:
            c.set_l2_keep(keep)
            c.clip_(1.0, 0.5)
            r = c.result()
            recs.append((r["norm"], r["sumsq_hi"], r["sumsq_lo"], r["coef_hi"], r["coef_lo"]))
    assert recs[0] == recs[1]
    for a, b in zip(gs.tensors, other):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
