"""The fused and alternative entry points captured in a CUDA graph.

Every call of the library only enqueues launches (no host synchronisation,
no allocation), so it can be captured.  Each test runs a call eagerly on one
copy of the inputs and replays a captured graph of the same call, twice, on
another copy restored before each replay: the results must be bit-identical
(the eager results themselves are checked against the oracle in each path's
own test file).
"""
import pytest
import torch

import global_l2_norm_gb300 as g
from workloads import make_gradset

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    g.build()


def dev():
    return torch.device("cuda", 0)


def bits(t):
    return t.reshape(-1).view(torch.int32 if t.element_size() == 4 else torch.int16)


def same(xs, ys):
    return all(torch.equal(bits(x), bits(y)) for x, y in zip(xs, ys))


def capture(fn):
    fn()                                    # one call outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


def scaled_set(name, mul):
    gs = make_gradset(name, device=dev())
    for t in gs.tensors:
        t.mul_(mul)
    return gs


@pytest.mark.parametrize("name,mul", [("andrea14m", 30.0), ("andrea120m_bf16", 1.0)])
def test_per_tensor(name, mul):
    gs = scaled_set(name, mul)
    pristine = [t.clone() for t in gs.tensors]
    eager = [t.clone() for t in pristine]
    with g.GradClipper(eager) as c:
        n_e, f_e = (x.clone() for x in c.clip_per_tensor_(1.0, 0.5))
    work = [t.clone() for t in pristine]
    with g.GradClipper(work) as c:
        graph = capture(lambda: c.clip_per_tensor_(1.0, 0.5))
        for _ in range(2):
            for w, p in zip(work, pristine):
                w.copy_(p)
            graph.replay()
            torch.cuda.synchronize()
            assert same(work, eager)
            assert torch.equal(c._pt_norms[:len(work)], n_e) and torch.equal(c._pt_flags[:len(work)], f_e)


@pytest.mark.parametrize("variant", ["split", "split_wave"])
def test_accumulate(variant):
    gs = scaled_set("andrea14m", 20.0)
    last = make_gradset("andrea14m", seed=4321, device=dev())
    pristine = [t.clone() for t in gs.tensors]
    eager = [t.clone() for t in pristine]
    with g.GradClipper(eager, variant=variant) as c:
        c.attach_addend(last.tensors)
        c.clip_accumulate_(1.0)
        rec_e = c.result()
    work = [t.clone() for t in pristine]
    with g.GradClipper(work, variant=variant) as c:
        c.attach_addend(last.tensors)
        graph = capture(lambda: c.clip_accumulate_(1.0))
        for _ in range(2):
            for w, p in zip(work, pristine):
                w.copy_(p)
            graph.replay()
            torch.cuda.synchronize()
            assert same(work, eager)
            assert c.result()["norm"] == rec_e["norm"]


def test_to_f32():
    gs = make_gradset("andrea120m_fp16", device=dev())
    outs_e = [torch.empty(t.numel(), device=dev()) for t in gs.tensors]
    outs_g = [torch.empty(t.numel(), device=dev()) for t in gs.tensors]
    with g.GradClipper(gs.tensors) as c:
        c.attach_f32_out(outs_e)
        c.clip_to_f32_(1.0, gs.inv_scale)
        c.attach_f32_out(outs_g)
        graph = capture(lambda: c.clip_to_f32_(1.0, gs.inv_scale))
        for _ in range(2):
            for o in outs_g:
                o.fill_(7.0)
            graph.replay()
            torch.cuda.synchronize()
            assert same(outs_g, outs_e)


def test_adamw():
    gs = make_gradset("andrea14m", device=dev())
    gen = torch.Generator(device=dev()).manual_seed(3)
    states0 = []
    for t in gs.tensors:
        w = torch.empty(t.numel(), device=dev()).normal_(0, 0.02, generator=gen)
        m = torch.empty(t.numel(), device=dev()).normal_(0, 1e-4, generator=gen)
        v = torch.empty(t.numel(), device=dev()).normal_(0, 1e-8, generator=gen).abs_()
        states0.append((w, m, v))
    hp = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=7)
    eager = [tuple(a.clone() for a in st) for st in states0]
    with g.GradClipper(gs.tensors) as c:
        c.attach_adamw(eager)
        c.clip_adamw_(0.1, **hp)
    work = [tuple(a.clone() for a in st) for st in states0]
    with g.GradClipper(gs.tensors) as c:
        c.attach_adamw(work)
        graph = capture(lambda: c.clip_adamw_(0.1, **hp))
        for _ in range(2):
            for ws, s0 in zip(work, states0):
                for a, b in zip(ws, s0):
                    a.copy_(b)
            graph.replay()
            torch.cuda.synchronize()
            for ws, es in zip(work, eager):
                assert same(ws, es)
