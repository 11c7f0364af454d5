"""The no-allocation entry point against the handle-based clip.

clip_grad_norm_flat_noalloc serves callers that cannot allocate device memory
or keep a handle (code whose device memory belongs to another allocator, and
plug-in interfaces that only get a buffer and a stream).  Its scratch is a
fixed array inside the library, shared by every call.  This test calls it
through the C ABI twice in a row, each time on a fresh copy of a gradient
buffer, and checks the result against clip_grad_norm on a one-tensor handle
over an identical copy, with the tolerances of the other parity tests (the
two are expected to agree bit for bit: same chunks, same arithmetic).  The
second call uses a smaller buffer, so stale partial sums from the first call
sit past its last chunk and must not be read.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import global_l2_norm_gb300 as g
from global_l2_norm_gb300 import _abi

pytestmark = pytest.mark.gpu

TD = {_abi.GCLIP_F32: torch.float32, _abi.GCLIP_F16: torch.float16,
      _abi.GCLIP_BF16: torch.bfloat16}
ULP = {_abi.GCLIP_F32: 2, _abi.GCLIP_F16: 1, _abi.GCLIP_BF16: 1}


def ulps(a: torch.Tensor, b: torch.Tensor) -> int:
    it = torch.int32 if a.dtype == torch.float32 else torch.int16
    width = 32 if a.dtype == torch.float32 else 16
    ia = a.view(it).cpu().numpy().astype(np.int64)
    ib = b.view(it).cpu().numpy().astype(np.int64)
    sign = 1 << (width - 1)
    oa = np.where(ia < 0, -(ia & (sign - 1)), ia)
    ob = np.where(ib < 0, -(ib & (sign - 1)), ib)
    return int(np.abs(oa - ob).max()) if oa.size else 0


def make_buffer(numel, dtype, offset, seed, std):
    """`numel` elements starting `offset` elements into a fresh allocation,
    N(0, std) values with one stretch spiked x50 so that the clip fires."""
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(seed)
    store = torch.empty(numel + offset, dtype=TD[dtype], device=dev)
    x = store[offset:]
    v = torch.randn(numel, generator=gen, device=dev) * std
    v[numel // 3: numel // 3 + 600_000] *= 50.0
    x.copy_(v)
    return store, x


def run_pair(numel, dtype, offset, seed, std, max_norm, inv_scale):
    store_a, a = make_buffer(numel, dtype, offset, seed, std)
    store_b = store_a.clone()
    b = store_b[offset:]
    # the existing entry point, on a handle made of this one tensor
    with g.GradClipper([a]) as c:
        c.clip_(max_norm, inv_scale)
        want = c.result()
    # the no-allocation entry point on an identical copy
    L = _abi.load()
    norm = torch.full((1,), -1.0, device=b.device)
    flag = torch.full((1,), -1, dtype=torch.int32, device=b.device)
    s = torch.cuda.current_stream()
    rc = L.clip_grad_norm_flat_noalloc(b.data_ptr(), numel, dtype, max_norm, inv_scale,
                                       norm.data_ptr(), flag.data_ptr(), s.cuda_stream)
    assert rc == _abi.GCLIP_OK, L.clip_status_string(rc)
    torch.cuda.synchronize()
    assert int(flag.item()) == want["nonfinite"] == 0
    assert abs(float(norm.item()) - want["norm"]) <= 1e-5 * want["norm"]
    assert ulps(a, b) <= ULP[dtype]
    return float(norm.item()), want


def test_noalloc_matches_handle_path_two_calls():
    g.build()
    # first call: 40M fp32 elements at a 16-byte-misaligned start (4,883 chunks)
    n1, w1 = run_pair(40_000_003, _abi.GCLIP_F32, 1, 11, 3e-5, 1.0, 1.0)
    assert w1["decision"] == _abi.GCLIP_DECISION_CLIP
    # second call right after: a smaller fp16 buffer under an unscale, so the
    # first call's partial sums beyond its chunks remain in the scratch
    n2, w2 = run_pair(3_000_001, _abi.GCLIP_F16, 3, 12, 0.5, 1.0, 2.0 ** -4)
    assert w2["decision"] == _abi.GCLIP_DECISION_CLIP
    assert n1 != n2


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
