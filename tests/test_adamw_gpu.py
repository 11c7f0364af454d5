"""Fused clip + AdamW on the GPU against the oracle (clip, then AdamW in fp64).

Tolerances, from the fp32 arithmetic of the kernel (every operation rounds
once, eps = 2^-24 relative; the hyperparameters reach both sides as the same
fp32 values, and the device's 1 - beta, 1 / (1 - beta^t) and 1 - lr * wd are
each rounded once more):
  m' = beta1 m + (1 - beta1) g^  within 8 eps (beta1 |m| + (1 - beta1) |g^|)
  v' = beta2 v + (1 - beta2) g^2 within 8 eps (beta2 v + (1 - beta2) g^2)
  w' within 2 eps (|w| + |w'|) + lr (tol_m / bc1 / denom
                                   + |upd| (8 eps + tol_v / (2 v')))
The bounds scale with the terms, not the result, because m' and w' can
cancel.  The decision, the flag and the norm are checked as for the clip.
"""
import math

import numpy as np
import pytest
import torch

import global_l2_norm_gb300 as g
import oracle
from _helpers import as_float64, storage_bits, to_oracle
from workloads import make_gradset

pytestmark = pytest.mark.gpu
EPS = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def built():
    g.build()


def dev():
    return torch.device("cuda", 0)


def f32(x):
    return float(np.float32(x))


def make_states(tensors, seed, fresh=False, misalign=False):
    gen = torch.Generator(device=dev()).manual_seed(seed)
    out, keep = [], []
    for t in tensors:
        n = t.numel()
        if misalign:          # views one element into a larger buffer: no vector access
            bufs = [torch.empty(n + 1, device=dev()) for _ in range(3)]
            w, m, v = (b[1:] for b in bufs)
            keep += bufs
        else:
            w, m, v = (torch.empty(n, device=dev()) for _ in range(3))
        w.normal_(0.0, 0.02, generator=gen)
        if fresh:
            m.zero_()
            v.zero_()
        else:
            m.normal_(0.0, 1e-4, generator=gen)
            v.normal_(0.0, 1e-8, generator=gen).abs_()
        out.append((w, m, v))
    return out, keep


def check(tensors, states, max_norm, inv_scale, hp, step, zero_grads=False, name="", alone=False):
    """alone: clip_adamw_step (the AdamW step with the gradients as they
    are), against the oracle's clip + AdamW at a threshold no norm reaches and
    inv_scale 1 (multiplier 1)."""
    hp = {k: f32(v) for k, v in hp.items()}
    max_norm, inv_scale = f32(max_norm), f32(inv_scale)
    g_host = [to_oracle(t) for t in tensors]
    s_host = [tuple(a.detach().cpu().numpy().copy() for a in st) for st in states]
    with g.GradClipper(tensors) as c:
        c.attach_adamw(states)
        if alone:
            c.adamw_step_(step=step, zero_grads=zero_grads, **hp)
            torch.cuda.synchronize()
        else:
            norm, flag = c.clip_adamw_(max_norm, inv_scale, step=step, zero_grads=zero_grads, **hp)
            rec = c.result()
    grads_want, new, r = oracle.default().clip_adamw(g_host, s_host, max_norm, inv_scale,
                                                     step=step, zero_grads=zero_grads, **hp)
    if alone:
        assert r.decision == oracle.PASS and r.coef == 1.0 and inv_scale == 1.0, (name, r.norm)
    else:
        assert rec["decision"] == r.decision and bool(rec["nonfinite"]) == r.nonfinite, name
        assert int(flag.item()) == int(r.nonfinite)
        if not r.nonfinite:
            assert abs(rec["norm"] - r.norm) <= 1e-5 * r.norm, (name, rec["norm"], r.norm)
    bc1 = 1 - hp["beta1"] ** step
    bc2 = 1 - hp["beta2"] ** step
    worst = 0.0
    for gt, (w0, m0, v0), (w1, m1, v1), st, gw, gnow in zip(g_host, s_host, new, states, grads_want,
                                                           tensors):
        gw_, gm_, gv_ = (a.detach().cpu().numpy() for a in st)
        if r.decision == oracle.SKIP:
            for a, b in ((w0, gw_), (m0, gm_), (v0, gv_)):
                assert np.array_equal(a.view(np.int32), b.view(np.int32)), name
            assert np.array_equal(storage_bits(gt), storage_bits(to_oracle(gnow)))
            continue
        gh = as_float64(gt) * inv_scale * r.coef
        w0d, m0d, v0d = (a.astype(np.float64) for a in (w0, m0, v0))
        m1d, v1d, w1d = (a.astype(np.float64) for a in (m1, v1, w1))
        tol_m = 8 * EPS * (hp["beta1"] * np.abs(m0d) + (1 - hp["beta1"]) * np.abs(gh)) + 1e-45
        tol_v = 8 * EPS * (hp["beta2"] * v0d + (1 - hp["beta2"]) * gh * gh) + 1e-45
        denom = np.sqrt(v1d / bc2) + hp["eps"]
        upd = m1d / bc1 / denom
        rel_v = np.where(v1d > 0, tol_v / (2 * np.maximum(v1d, 1e-45)), 0.0)
        tol_w = (2 * EPS * (np.abs(w0d) + np.abs(w1d))
                 + hp["lr"] * (tol_m / bc1 / denom + np.abs(upd) * (8 * EPS + np.minimum(rel_v, 1))))
        for got, want, tol, what in ((gm_, m1d, tol_m, "m"), (gv_, v1d, tol_v, "v"),
                                     (gw_, w1d, tol_w, "w")):
            err = np.abs(got.astype(np.float64) - want)
            assert np.all(err <= tol), (name, what, float(err.max()), float((err / tol).max()))
            worst = max(worst, float((err / tol).max()) if err.size else 0.0)
        if zero_grads:
            assert not storage_bits(to_oracle(gnow)).any(), name
        else:
            assert np.array_equal(storage_bits(gt), storage_bits(to_oracle(gnow))), name
    return worst


HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


@pytest.mark.parametrize("name,step,fresh", [("tiny", 1, True), ("andrea14m", 3, False),
                                             ("andrea120m", 1, True), ("andrea120m", 50, False),
                                             ("andrea120m_fp16", 2, False),
                                             ("andrea120m_bf16", 9, False)])
def test_fused_matches_oracle(name, step, fresh):
    gs = make_gradset(name, device=dev())
    states, _ = make_states(gs.tensors, 7, fresh=fresh)
    check(gs.tensors, states, gs.max_norm, gs.inv_scale, HP, step, name=name)


@pytest.mark.parametrize("name,step", [("tiny", 1), ("andrea14m", 4), ("andrea120m_bf16", 2)])
def test_step_alone_matches_oracle(name, step):
    """clip_adamw_step: AdamW with the gradients as they are."""
    gs = make_gradset(name, device=dev())
    states, _ = make_states(gs.tensors, 13)
    check(gs.tensors, states, 3.0e38, 1.0, HP, step, name=name, alone=True)


def test_step_alone_zero_grads_and_misaligned_state():
    gs = make_gradset("andrea14m", device=dev())
    states, keep = make_states(gs.tensors, 17, misalign=True)
    check(gs.tensors, states, 3.0e38, 1.0, HP, 3, zero_grads=True, name="alone zero+misaligned",
          alone=True)


@pytest.mark.parametrize("name", ["andrea120m", "andrea14m"])
def test_clip_then_step_equals_fused(name):
    """For fp32 gradients, clip_grad_norm followed by clip_adamw_step leaves
    w, m and v bit for bit where clip_grad_norm_adamw does: the in-place clip
    stores exactly the fp32 value the fused pass forms in registers."""
    gs = make_gradset(name, device=dev())
    grads_a = [t.clone() for t in gs.tensors]
    grads_b = [t.clone() for t in gs.tensors]
    states_a, _ = make_states(gs.tensors, 19)
    states_b = [tuple(a.clone() for a in st) for st in states_a]
    with g.GradClipper(grads_a) as ca, g.GradClipper(grads_b) as cb:
        ca.attach_adamw(states_a)
        cb.attach_adamw(states_b)
        for step in (1, 2):
            ca.clip_adamw_(gs.max_norm, gs.inv_scale, step=step, **HP)
            for t, o in zip(grads_b, gs.tensors):    # the fused call only reads its gradients
                t.copy_(o)
            cb.clip_(gs.max_norm, gs.inv_scale)
            cb.adamw_step_(step=step, **HP)
            torch.cuda.synchronize()
            assert ca.result()["decision"] == cb.result()["decision"]
            assert ca.result()["norm"] == cb.result()["norm"]
        for sa, sb in zip(states_a, states_b):
            for a, b in zip(sa, sb):
                assert torch.equal(a, b)


def test_zero_grads_and_misaligned_state():
    gs = make_gradset("andrea14m", device=dev())
    for t in gs.tensors:
        t.mul_(100.0)                              # the clip fires
    states, keep = make_states(gs.tensors, 3, misalign=True)
    check(gs.tensors, states, 1.0, 1.0, HP, 4, zero_grads=True, name="zero+misaligned")


def test_nonfinite_updates_nothing():
    gs = make_gradset("tiny", device=dev())
    gs.tensors[2].view(-1)[17] = float("nan")
    states, _ = make_states(gs.tensors, 5)
    check(gs.tensors, states, 1.0, 1.0, HP, 2, zero_grads=True, name="nan")


def test_warmup_bound_on_device():
    """The clipping page, "Adjacent activities": at warm-up lr 1.5e-7 and
    max_norm 1, no parameter moves more than 1.5e-7 in the first step, even
    with a 50x spike (plus the fp32 rounding of the stored weight)."""
    gs = make_gradset("andrea120m", device=dev())
    states, _ = make_states(gs.tensors, 11, fresh=True)
    before = [st[0].clone() for st in states]
    with g.GradClipper(gs.tensors) as c:
        c.attach_adamw(states)
        c.clip_adamw_(1.0, lr=1.5e-7, beta1=0.9, beta2=0.95, eps=1e-8, step=1)
        assert c.result()["decision"] == g.GCLIP_DECISION_CLIP
    for b, (w, _, _) in zip(before, states):
        dw = (w.double() - b.double()).abs()
        assert bool((dw <= 1.5e-7 + torch.abs(w).double() * 2.0 ** -23).all())


def test_argument_checks():
    x = torch.ones(8, device=dev())
    w, m, v = (torch.zeros(8, device=dev()) for _ in range(3))
    with g.GradClipper([x]) as c:
        L = g.load()
        p = g._abi.clip_adamw_params_t(1e-3, 0.9, 0.999, 1e-8, 0.0, 0)
        assert L.clip_grad_norm_adamw(c._h, 1.0, 1.0, p, 1, None, None, None) == \
            g._abi.GCLIP_ERR_INVALID_ARG               # no state attached
        with pytest.raises(g.GclipError):
            c.attach_adamw([(w, m, w)])                # overlapping state
        c.attach_adamw([(w, m, v)])
        for bad in (dict(lr=-1.0), dict(beta1=1.0), dict(beta2=-0.1), dict(eps=0.0),
                    dict(weight_decay=-1.0), dict(lr=math.inf)):
            kw = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
            kw.update(bad)
            with pytest.raises(g.GclipError):
                c.clip_adamw_(1.0, **kw)
        with pytest.raises(g.GclipError):
            c.clip_adamw_(1.0, lr=1e-3, step=0)
        for bad in (dict(lr=-1.0), dict(beta1=1.0), dict(eps=0.0), dict(step=0)):
            kw = dict(lr=1e-3, step=1)
            kw.update(bad)
            with pytest.raises(g.GclipError):
                c.adamw_step_(**kw)
        assert L.clip_adamw_step(None, p, 1, None) == g._abi.GCLIP_ERR_INVALID_ARG
        assert L.clip_adamw_step(c._h, None, 1, None) == g._abi.GCLIP_ERR_INVALID_ARG
    with g.GradClipper([x]) as c:
        L = g.load()
        p = g._abi.clip_adamw_params_t(1e-3, 0.9, 0.999, 1e-8, 0.0, 0)
        assert L.clip_adamw_step(c._h, p, 1, None) == g._abi.GCLIP_ERR_INVALID_ARG  # no state
    assert x.cpu().tolist() == [1.0] * 8
