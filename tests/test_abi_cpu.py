"""The C ABI on a machine without a GPU: the library loads, exports every
function the header declares, plans chunk tables and rejects bad arguments
before touching a device."""
import ctypes
import os
import re

import pytest

import global_l2_norm_gb300 as g
from global_l2_norm_gb300 import _abi
from workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gclip.h")


@pytest.fixture(scope="module")
def L():
    g.build()
    return _abi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(clip_\w+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("clip_create", "clip_grad_norm", "clip_destroy"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_header_constants_match_binding():
    text = open(HEADER).read()
    for name, val in re.findall(r"#define[ \t]+(GCLIP_\w+)[ \t]+(\(?[0-9x< ]+\)?)[ \t]*(?:/\*|\n)", text):
        assert getattr(_abi, name) == eval(val), name


def _descs(specs):
    arr = (_abi.clip_tensor_desc_t * max(1, len(specs)))()
    for i, (ptr, numel, dtype) in enumerate(specs):
        arr[i].ptr = ptr
        arr[i].numel = numel
        arr[i].dtype = dtype
        arr[i].reserved = 0
    return arr


def _plan(specs):
    return g.plan(_descs(specs), len(specs))


ES = {0: 4, 1: 2, 2: 2}


def check_cover(specs, chunks):
    """Every element of every non-empty tensor in exactly one chunk, in
    tensor order, each chunk within its size bound, every chunk after a
    tensor's first on a 16-byte boundary."""
    it = iter(chunks)
    for t, (ptr, numel, dtype) in enumerate(specs):
        if numel == 0:
            continue
        es = ES[dtype]
        done = 0
        first = True
        while done < numel:
            addr, n, meta = next(it)
            assert meta & 0xFF == dtype and meta >> 8 == t
            assert addr == ptr + done * es
            assert n > 0
            head = ((16 - ptr % 16) % 16) // es if first else 0
            assert n <= head + _abi.GCLIP_CHUNK_BYTES // es
            if not first:
                assert addr % 16 == 0
            done += n
            first = False
        assert done == numel
    assert next(it, None) is None


BASE = 1 << 40


@pytest.mark.parametrize("name", ["tiny", "andrea14m", "andrea120m", "andrea120m_fp16", "andrea1p2b"])
def test_plan_covers_workload_layouts(L, name):
    w = WORKLOADS[name]
    dt = {"f32": 0, "f16": 1, "bf16": 2}[w.dtype]
    specs, addr = [], BASE
    for s in w.layout:
        specs.append((addr, s.numel, dt))
        addr += (s.numel * w.elem_bytes + 511) // 512 * 512
    chunks = _plan(specs)
    check_cover(specs, chunks)
    es = w.elem_bytes
    # chunk count: ceil(bytes / chunk) per tensor when every base is aligned
    want = sum(-(-s.numel * es // _abi.GCLIP_CHUNK_BYTES) for s in w.layout)
    assert len(chunks) == want


def test_plan_ragged_and_misaligned(L):
    specs = [(BASE + 4, 3, 0), (BASE + 64, 0, 0), (BASE + 1000, 8195, 0),
             (BASE + 80002, 1, 1), (BASE + 80006, 17000, 2), (BASE + 200004, 8192 * 3 + 1, 0),
             (BASE + 400000, 16385, 1)]
    check_cover(specs, _plan(specs))


def test_plan_empty(L):
    assert _plan([]) == []
    assert _plan([(0, 0, 0), (None, 0, 1)]) == []


@pytest.mark.parametrize("specs", [
    [(0, 5, 0)],                          # NULL with elements
    [(BASE + 2, 5, 0)],                   # fp32 at a 2-byte address
    [(BASE + 1, 5, 1)],                   # fp16 at an odd address
    [(BASE, 5, 3)],                       # unknown dtype
    [(BASE, -1, 0)],                      # negative numel
    [(BASE, 100, 0), (BASE + 396, 4, 0)],  # overlap
    [(BASE + 396, 4, 0), (BASE, 100, 0)],  # overlap, reversed order
], ids=["null", "misaligned32", "misaligned16", "dtype", "negative", "overlap", "overlap_rev"])
def test_invalid_descriptors_rejected(L, specs):
    d = _descs(specs)
    n = ctypes.c_int64()
    assert L.clip_plan(d, len(specs), None, 0, ctypes.byref(n)) == _abi.GCLIP_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert L.clip_create(d, len(specs), ctypes.byref(h)) == _abi.GCLIP_ERR_INVALID_ARG
    assert h.value is None


def test_reserved_must_be_zero(L):
    d = _descs([(BASE, 4, 0)])
    d[0].reserved = 1
    n = ctypes.c_int64()
    assert L.clip_plan(d, 1, None, 0, ctypes.byref(n)) == _abi.GCLIP_ERR_INVALID_ARG


def test_adjacent_tensors_are_not_overlap(L):
    specs = [(BASE, 100, 0), (BASE + 400, 4, 0)]
    check_cover(specs, _plan(specs))


def test_bad_counts_and_nulls(L):
    h = ctypes.c_void_p()
    n = ctypes.c_int64()
    assert L.clip_create(None, 1, ctypes.byref(h)) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_create(_descs([]), -1, ctypes.byref(h)) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_create(_descs([]), _abi.GCLIP_MAX_TENSORS + 1, ctypes.byref(h)) == \
        _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_create(_descs([]), 0, None) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_plan(_descs([]), 0, None, 0, None) == _abi.GCLIP_ERR_INVALID_ARG
    table = (_abi.clip_chunk_t * 1)()
    assert L.clip_plan(_descs([(BASE, 100000, 0)]), 1, table, 1, ctypes.byref(n)) == \
        _abi.GCLIP_ERR_INVALID_ARG
    assert n.value == 13


def test_null_handle_calls(L):
    assert L.clip_grad_norm(None, 1.0, 1.0, None, None, None) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_destroy(None) == _abi.GCLIP_OK
    assert L.clip_set_variant(None, 0) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_get_variant(None) == -1
    assert L.clip_num_chunks(None) == -1
    assert L.clip_persistent_grid(None) == -1
    assert L.clip_result_device(None) is None
    assert L.clip_read_result(None, None, None) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_reset(None, None) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_debug_barrier(None, 1, 0) == _abi.GCLIP_ERR_INVALID_ARG
    assert L.clip_set_l2_keep(None, 0) == _abi.GCLIP_ERR_INVALID_ARG


def test_status_strings(L):
    for code in range(6):
        s = L.clip_status_string(code)
        assert s and s != b"unknown status"
    assert L.clip_status_string(99) == b"unknown status"


def test_record_layout_matches_header():
    assert ctypes.sizeof(_abi.clip_result_t) == 40
    assert ctypes.sizeof(_abi.clip_chunk_t) == 16
    assert ctypes.sizeof(_abi.clip_tensor_desc_t) == 24
