"""The no-allocation entry point, through the C ABI.

clip_grad_norm_flat_noalloc serves callers that cannot allocate device memory
or keep a handle: code whose device memory all belongs to another allocator
(a caching allocator, or an arena sized at start-up, where a driver
allocation in the middle of a run can fail or stall), and plug-in interfaces
that only receive a buffer and a stream.  Its scratch is a fixed array inside
the library, shared by every call.

Each case runs it on a fresh copy of a gradient buffer and checks it three
ways: against the oracle (the norm within 1e-5, the flag, every output within
2 ulp for fp32 and 1 ulp for fp16/bf16, SKIP outputs untouched); bit for bit
against clip_grad_norm with GCLIP_VARIANT_THREE_KERNEL on a one-tensor handle
over an identical copy (the same chunks, kernels and order); and, with the
same tolerances, against the default variant, which sums the chunks in
another fixed order.  The calls come in a row, the second on a smaller buffer
so that stale partial sums of the first sit past its last chunk.  This file
is collected last.
"""
import numpy as np
import pytest
import torch

import global_l2_norm_gb300 as g
import oracle
from _helpers import storage_bits, to_oracle, ulp_distance
from global_l2_norm_gb300 import _abi

pytestmark = pytest.mark.gpu

TD = {_abi.GCLIP_F32: torch.float32, _abi.GCLIP_F16: torch.float16,
      _abi.GCLIP_BF16: torch.bfloat16}
ULP = {"f32": 2, "f16": 1, "bf16": 1}


def make_buffer(numel, dtype, offset, seed, std, spike=True):
    """`numel` elements starting `offset` elements into a fresh allocation,
    N(0, std) values, one stretch spiked x50 (so that the clip fires)."""
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(seed)
    store = torch.empty(numel + offset, dtype=TD[dtype], device=dev)
    x = store[offset:]
    v = torch.randn(numel, generator=gen, device=dev) * std
    if spike and numel:
        v[numel // 3: numel // 3 + min(600_000, numel // 3)] *= 50.0
    x.copy_(v)
    return store, x


def noalloc(x, dtype, max_norm, inv_scale):
    """One call of the entry point on `x` (in place); returns (norm, flag)."""
    L = _abi.load()
    norm = torch.full((1,), -1.0, device="cuda")
    flag = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = L.clip_grad_norm_flat_noalloc(x.data_ptr() if x.numel() else None, x.numel(), dtype,
                                       max_norm, inv_scale, norm.data_ptr(), flag.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == _abi.GCLIP_OK, L.clip_status_string(rc)
    torch.cuda.synchronize()
    return float(norm.item()), int(flag.item())


def handle(x, variant, max_norm, inv_scale):
    with g.GradClipper([x], variant=variant) as c:
        norm, flag = c.clip_(max_norm, inv_scale)
        rec = c.result()
        rec["out_norm"], rec["out_flag"] = float(norm.item()), int(flag.item())
    return rec


def check_case(numel, dtype, offset, seed, std, max_norm, inv_scale, spike=True, inject=None):
    """Returns the oracle's decision after checking the three comparisons."""
    store, x = make_buffer(numel, dtype, offset, seed, std, spike)
    if inject is not None:
        x[inject[0]] = inject[1]
    before = to_oracle(x)
    three = store.clone()[offset:]
    default = store.clone()[offset:]

    norm, flag = noalloc(x, dtype, max_norm, inv_scale)

    # the oracle
    want, r = oracle.clip([before], max_norm, inv_scale)
    assert flag == int(r.nonfinite)
    if r.nonfinite:
        assert not np.isfinite(norm)
        assert np.array_equal(storage_bits(to_oracle(x)), storage_bits(before))
    else:
        assert abs(norm - r.norm) <= 1e-5 * r.norm if r.norm else norm == 0.0, (norm, r.norm)
        if numel:
            assert int(ulp_distance(to_oracle(x), want[0]).max()) <= ULP[want[0].dtype]

    # the three-kernel handle path: bit for bit
    rec = handle(three, "three_kernel", max_norm, inv_scale)
    assert rec["out_flag"] == flag
    assert np.array_equal(np.float32(rec["out_norm"]).view(np.int32),
                          np.float32(norm).view(np.int32)), (rec["out_norm"], norm)
    assert torch.equal(three.view(torch.uint8), x.view(torch.uint8))

    # the default variant: within the tolerances
    rec = handle(default, "split", max_norm, inv_scale)
    assert rec["out_flag"] == flag and rec["decision"] == r.decision
    if not r.nonfinite and r.norm:
        assert abs(rec["out_norm"] - norm) <= 1e-5 * r.norm
    if numel:
        assert int(ulp_distance(to_oracle(default), to_oracle(x)).max()) <= ULP[want[0].dtype]
    return r.decision


def test_noalloc_two_calls_against_oracle_and_handle():
    g.build()
    # first call: 40M fp32 elements at a 16-byte-misaligned start (4,883 chunks)
    d1 = check_case(40_000_003, _abi.GCLIP_F32, 1, 11, 3e-5, 1.0, 1.0)
    assert d1 == oracle.CLIP
    # second call right after: a smaller fp16 buffer under an unscale, so the
    # first call's partial sums beyond its chunks remain in the scratch
    d2 = check_case(3_000_001, _abi.GCLIP_F16, 3, 12, 0.5, 1.0, 2.0 ** -4)
    assert d2 == oracle.CLIP


def test_noalloc_edge_cases():
    g.build()
    # a +inf element: SKIP, flag raised, nothing written
    assert check_case(1_000_001, _abi.GCLIP_F32, 2, 21, 1.0, 1.0, 1.0,
                      inject=(777_777, float("inf"))) == oracle.SKIP
    # PASS with inv_scale 1: the multiplier is 1, nothing is written
    assert check_case(500_000, _abi.GCLIP_F32, 0, 22, 1e-4, 10.0, 1.0,
                      spike=False) == oracle.PASS
    # bf16, clipped
    assert check_case(2_000_003, _abi.GCLIP_BF16, 5, 23, 1e-2, 1.0, 1.0) == oracle.CLIP
    # no elements: norm 0, flag 0, written through the output pointers
    norm, flag = noalloc(torch.empty(0, device="cuda"), _abi.GCLIP_F32, 1.0, 1.0)
    assert norm == 0.0 and flag == 0


def test_noalloc_largest_buffer():
    """Exactly GCLIP_NOALLOC_MAX_CHUNKS chunks (2 GiB of fp32, aligned start):
    accepted, the norm against the oracle, outputs on a sample the oracle
    computes one by one, and bit for bit against the three-kernel handle."""
    g.build()
    per = _abi.GCLIP_CHUNK_BYTES // 4
    n = _abi.GCLIP_NOALLOC_MAX_CHUNKS * per
    x = torch.empty(n, device="cuda")
    assert x.data_ptr() % 16 == 0
    gen = torch.Generator(device="cuda").manual_seed(31)
    x.normal_(0.0, 1e-4, generator=gen)
    x[n // 2: n // 2 + 1000] *= 1e4
    host = to_oracle(x)
    three = x.clone()
    norm, flag = noalloc(x, _abi.GCLIP_F32, 1.0, 1.0)
    idx = np.concatenate([np.arange(0, 64), np.arange(n - 64, n), np.arange(n // 2, n // 2 + 64),
                          np.random.default_rng(2).integers(0, n, 4096)])
    slots, r = oracle.default().clip_sample([host], 1.0, 1.0, np.zeros(idx.size), idx)
    assert flag == 0 and r.decision == oracle.CLIP
    assert abs(norm - r.norm) <= 1e-5 * r.norm, (norm, r.norm)
    got = x[torch.from_numpy(idx).cuda()].cpu().numpy()
    want = (slots & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    assert int(ulp_distance(oracle.OracleTensor(got, "f32"), oracle.OracleTensor(want, "f32")).max()) <= 2
    del host
    rec = handle(three, "three_kernel", 1.0, 1.0)
    assert np.float32(rec["out_norm"]).view(np.int32) == np.float32(norm).view(np.int32)
    assert torch.equal(three, x)


def test_noalloc_rejects_oversized_and_bad_arguments():
    L = _abi.load()
    x = torch.ones(8, device="cuda")
    per = _abi.GCLIP_CHUNK_BYTES // 4
    too_many = _abi.GCLIP_NOALLOC_MAX_CHUNKS * per + 1   # aligned start: no head
    assert x.data_ptr() % 16 == 0
    assert L.clip_grad_norm_flat_noalloc(x.data_ptr(), too_many, _abi.GCLIP_F32, 1.0, 1.0,
                                         None, None, None) == _abi.GCLIP_ERR_TOO_LARGE
    assert L.clip_status_string(_abi.GCLIP_ERR_TOO_LARGE) != b"unknown status"
    assert L.clip_grad_norm_flat_noalloc(x.data_ptr(), 8, 7, 1.0, 1.0, None, None,
                                         None) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_grad_norm_flat_noalloc(x.data_ptr() + 2, 4, _abi.GCLIP_F32, 1.0, 1.0, None,
                                         None, None) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_grad_norm_flat_noalloc(x.data_ptr(), 8, _abi.GCLIP_F32, 0.0, 1.0, None,
                                         None, None) == _abi.GCLIP_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert x.tolist() == [1.0] * 8
