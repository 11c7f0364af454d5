"""Seeded synthetic gradient sets shaped like the pages' ANDREA models.

This module is shared by the tests, the benchmark and the smoke check.  It
only decides shapes, value distributions and which tensor is spiked; it holds
none of the clipping arithmetic, and neither the oracle nor the CUDA library
imports it.

Shapes follow "Grow a language model: backprop" (unhomeschool.com,
Vietnamese), section "Where gradients live": per transformer block the
gradients of W_Q, W_K, W_V, W_O [d, d], W_1 [d, 4d], W_2 [4d, d] and the
gamma/beta of two layer norms [d], plus the token and position embeddings and
a final layer norm; the output head is tied to the token embedding (section
"Forward pass"), so it has no gradient tensor of its own.  The vocabulary
(8449) is the embedding shape named in the gradient-clipping page, section
"Why computing the grad norm needs three kernels"; the context (1024) is the
sequence length of the backprop page's activation-memory example.
"""
from __future__ import annotations

import random
from dataclasses import dataclass, field

import torch

VOCAB = 8449
CONTEXT = 1024
SEED = 1234


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


def andrea_layout(d: int, n_layers: int, final_ln: bool = True) -> list[TensorSpec]:
    """Gradient tensors of an ANDREA-style decoder with width d."""
    specs = [TensorSpec("tok_embed", (VOCAB, d)), TensorSpec("pos_embed", (CONTEXT, d))]
    for i in range(n_layers):
        p = f"block{i}."
        specs += [TensorSpec(p + "W_Q", (d, d)), TensorSpec(p + "W_K", (d, d)),
                  TensorSpec(p + "W_V", (d, d)), TensorSpec(p + "W_O", (d, d)),
                  TensorSpec(p + "W_1", (d, 4 * d)), TensorSpec(p + "W_2", (4 * d, d)),
                  TensorSpec(p + "LN1.gamma", (d,)), TensorSpec(p + "LN1.beta", (d,)),
                  TensorSpec(p + "LN2.gamma", (d,)), TensorSpec(p + "LN2.beta", (d,))]
    if final_ln:
        specs += [TensorSpec("LN_f.gamma", (d,)), TensorSpec("LN_f.beta", (d,))]
    return specs


TINY_LAYOUT = [TensorSpec("a", (64, 32)), TensorSpec("b", (32,)),
               TensorSpec("c", (32, 64)), TensorSpec("d", (16,))]


@dataclass(frozen=True)
class Workload:
    """One named gradient set: layout, value recipe and clip arguments."""
    name: str
    layout: tuple
    std: float                 # standard deviation of the N(0, std) values
    dtype: str                 # "f32" | "f16" | "bf16"
    max_norm: float
    inv_scale: float
    spikes: int = 0            # number of 2-D tensors multiplied by spike_factor
    spike_factor: float = 1.0
    inject_inf: bool = False   # one +inf at a seeded position
    description: str = ""

    @property
    def numel(self) -> int:
        return sum(s.numel for s in self.layout)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS = {
    "tiny": Workload(
        "tiny", tuple(TINY_LAYOUT), 0.1, "f32", 1.0, 1.0,
        description="tiny fp32 set [64,32],[32],[32,64],[16], N(0,0.1), max_norm 1"),
    "andrea14m": Workload(
        "andrea14m", tuple(andrea_layout(384, 6)), 1e-4, "f32", 1.0, 1.0,
        description="ANDREA-14M fp32 grads, N(0,1e-4), max_norm 1 (no clip)"),
    "andrea120m": Workload(
        "andrea120m", tuple(andrea_layout(768, 12)), 3e-5, "f32", 1.0, 1.0,
        spikes=1, spike_factor=50.0,
        description="ANDREA-120M fp32 grads, N(0,3e-5), one matrix x50, max_norm 1"),
    "andrea120m_noclip": Workload(
        "andrea120m_noclip", tuple(andrea_layout(768, 12)), 3e-5, "f32", 1.0, 1.0,
        description="ANDREA-120M fp32 grads, N(0,3e-5), no spike, max_norm 1 (no clip)"),
    # 4 accumulated microbatches under loss scale 65536: the stored values are
    # the scaled sums, the clip unscales by 1/(65536*4) = 2^-18.
    "andrea120m_fp16": Workload(
        "andrea120m_fp16", tuple(andrea_layout(768, 12)), 3e-5 * 65536.0 * 4.0, "f16",
        1.0, 2.0 ** -18,
        description="ANDREA-120M fp16 grads, loss scale 65536 x 4 microbatches, "
                    "inv_scale 2^-18, max_norm 1"),
    "andrea120m_fp16_inf": Workload(
        "andrea120m_fp16_inf", tuple(andrea_layout(768, 12)), 3e-5 * 65536.0 * 4.0,
        "f16", 1.0, 2.0 ** -18, inject_inf=True,
        description="as andrea120m_fp16 with one +inf injected"),
    "andrea120m_bf16": Workload(
        "andrea120m_bf16", tuple(andrea_layout(768, 12)), 3e-5, "bf16", 1.0, 1.0,
        spikes=1, spike_factor=50.0,
        description="ANDREA-120M bf16 grads, N(0,3e-5), one matrix x50, max_norm 1"),
    "andrea1p2b": Workload(
        "andrea1p2b", tuple(andrea_layout(2048, 24, final_ln=False)), 1e-5, "f32",
        1.0, 1.0, spikes=3, spike_factor=100.0,
        description="ANDREA-1.2B fp32 grads, N(0,1e-5), three matrices x100, max_norm 1"),
}

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class GradSet:
    workload: Workload
    tensors: list
    spiked: list = field(default_factory=list)   # names of the spiked tensors
    inf_at: tuple | None = None                  # (tensor index, flat index)
    flat: object = None                          # the single buffer, if flat

    @property
    def max_norm(self) -> float:
        return self.workload.max_norm

    @property
    def inv_scale(self) -> float:
        return self.workload.inv_scale


def _choices(seed: int, layout, w: Workload):
    """Which tensors are spiked and where the +inf goes: a pure function of the
    seed and the layout, identical on every machine and device."""
    rng = random.Random(seed)
    mats = [i for i, s in enumerate(layout) if len(s.shape) == 2]
    spiked = sorted(rng.sample(mats, w.spikes)) if w.spikes else []
    inf_at = None
    if w.inject_inf:
        t = rng.randrange(len(layout))
        inf_at = (t, rng.randrange(layout[t].numel))
    return spiked, inf_at


def make_gradset(name_or_workload, seed: int = SEED, device="cpu", flat: bool = False) -> GradSet:
    """Allocate and fill one gradient set.  Values come from torch's generator
    on `device` seeded with `seed`, so a set is reproducible on a given kind of
    device; parity tests hand the oracle a host copy of the very tensors the
    GPU sees.  With flat=True every tensor is a view into one buffer (each
    starting on a 256-byte boundary, as the caching allocator would place
    them), kept as `GradSet.flat`, so that a whole set can be copied at once."""
    w = WORKLOADS[name_or_workload] if isinstance(name_or_workload, str) else name_or_workload
    layout = list(w.layout)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    spiked, inf_at = _choices(seed, layout, w)
    dt = TORCH_DTYPES[w.dtype]
    flat_buf, views = None, None
    if flat:
        es = w.elem_bytes
        offs, pos = [], 0
        for spec in layout:
            offs.append(pos)
            pos += (spec.numel * es + 255) // 256 * 256
        flat_buf = torch.zeros(pos // es, dtype=dt, device=device)
        views = [flat_buf[o // es:o // es + spec.numel].view(spec.shape)
                 for o, spec in zip(offs, layout)]
    tensors = []
    for i, spec in enumerate(layout):
        t = torch.randn(spec.shape, generator=gen, device=device, dtype=torch.float32)
        t.mul_(w.std * (w.spike_factor if i in spiked else 1.0))
        if views is not None:
            views[i].copy_(t)
            tensors.append(views[i])
        else:
            tensors.append(t.to(dt))
    if inf_at is not None:
        tensors[inf_at[0]].view(-1)[inf_at[1]] = float("inf")
    gs = GradSet(w, tensors, [layout[i].name for i in spiked], inf_at)
    gs.flat = flat_buf
    return gs


def fill_gradset_(gs: GradSet, seed: int = SEED) -> None:
    """Refill an existing set in place with the values make_gradset would give
    for `seed` (same allocations, so a library handle built on them stays
    valid)."""
    w = gs.workload
    device = gs.tensors[0].device
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    spiked, inf_at = _choices(seed, list(w.layout), w)
    for i, t in enumerate(gs.tensors):
        v = torch.randn(t.shape, generator=gen, device=device, dtype=torch.float32)
        v.mul_(w.std * (w.spike_factor if i in spiked else 1.0))
        t.copy_(v)
    if inf_at is not None:
        gs.tensors[inf_at[0]].view(-1)[inf_at[1]] = float("inf")
