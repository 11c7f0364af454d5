"""CPU oracle for global L2-norm gradient clipping.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library under
``global_l2_norm_gb300/`` never does, and shares no code with it.

The arithmetic lives in ``gclip_oracle.c`` (plain C, fp64), which states the
passages of the pages it follows.  This module builds it with gcc and exposes
it over ctypes with numpy arrays.

Tensors are passed as ``OracleTensor(data, dtype)`` where ``data`` is a
contiguous numpy array holding the storage: float32 for ``"f32"``, float16 for
``"f16"`` and uint16 bit patterns for ``"bf16"`` (numpy has no bfloat16).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gclip_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}

PASS, CLIP, SKIP = 0, 1, 2
DECISION_NAMES = {PASS: "pass", CLIP: "clip", SKIP: "skip"}


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("numel", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("pad", ctypes.c_int32)]


class _AdamwParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("step", ctypes.c_int64), ("zero_grads", ctypes.c_int32), ("pad", ctypes.c_int32)]


class _AdamwState(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p)]


class _Result(ctypes.Structure):
    _fields_ = [("sumsq", ctypes.c_double), ("norm", ctypes.c_double),
                ("coef", ctypes.c_double), ("nonfinite", ctypes.c_int32),
                ("decision", ctypes.c_int32)]


@dataclass
class OracleTensor:
    data: np.ndarray
    dtype: str

    def __post_init__(self):
        if self.dtype not in DTYPES:
            raise ValueError(f"unknown dtype {self.dtype!r}")
        want = _STORAGE[self.dtype]
        if self.data.dtype != want:
            raise TypeError(f"{self.dtype} storage must be {np.dtype(want)}, "
                            f"got {self.data.dtype}")
        self.data = np.ascontiguousarray(self.data).reshape(-1)


@dataclass
class OracleResult:
    sumsq: float
    norm: float
    coef: float
    nonfinite: bool
    decision: int

    @property
    def decision_name(self) -> str:
        return DECISION_NAMES[self.decision]


def build(mutant: int = 0, outdir: str | None = None) -> str:
    """Compile the oracle into a shared library and return its path.

    ``mutant`` > 0 compiles one of the planted mistakes the mutation tests use
    to show that the pins catch it; the default build plants none.
    """
    outdir = outdir or _BUILD
    os.makedirs(outdir, exist_ok=True)
    name = "liboracle.so" if mutant == 0 else f"liboracle_m{mutant}.so"
    out = os.path.join(outdir, name)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp,
           "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """One loaded build of the oracle (the default, or a planted mutant)."""

    def __init__(self, mutant: int = 0, outdir: str | None = None):
        self.mutant = mutant
        self._lib = ctypes.CDLL(build(mutant, outdir))
        L = self._lib
        L.oracle_clip.argtypes = [ctypes.POINTER(_Tensor), ctypes.POINTER(_Tensor),
                                  ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                                  ctypes.POINTER(_Result)]
        L.oracle_clip.restype = ctypes.c_int
        L.oracle_clip_per_tensor.argtypes = L.oracle_clip.argtypes
        L.oracle_clip_per_tensor.restype = ctypes.c_int
        L.oracle_clip_sample.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_int32,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.POINTER(_Result)]
        L.oracle_clip_sample.restype = ctypes.c_int
        L.oracle_clip_adamw.argtypes = [ctypes.POINTER(_Tensor), ctypes.POINTER(_AdamwState),
                                        ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                                        ctypes.POINTER(_AdamwParams), ctypes.POINTER(_Result)]
        L.oracle_clip_adamw.restype = ctypes.c_int
        L.oracle_clip_to_f32.argtypes = [ctypes.POINTER(_Tensor), ctypes.POINTER(ctypes.c_void_p),
                                         ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                                         ctypes.POINTER(_Result)]
        L.oracle_clip_to_f32.restype = ctypes.c_int
        L.oracle_accumulate.argtypes = [ctypes.POINTER(_Tensor), ctypes.POINTER(_Tensor),
                                        ctypes.c_int32]
        L.oracle_accumulate.restype = ctypes.c_int
        L.oracle_clip_accumulate.argtypes = L.oracle_clip.argtypes
        L.oracle_clip_accumulate.restype = ctypes.c_int
        L.oracle_sumsq.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_int32,
                                   ctypes.c_double, ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_int32)]
        L.oracle_sumsq.restype = ctypes.c_int
        L.oracle_value_clip.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.c_double, ctypes.c_void_p]
        L.oracle_value_clip.restype = None
        L.oracle_decode.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32]
        L.oracle_decode.restype = ctypes.c_double
        L.oracle_encode.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                    ctypes.c_double]
        L.oracle_encode.restype = None
        L.oracle_round_grid_f32_bits.argtypes = [ctypes.c_double]
        L.oracle_round_grid_f32_bits.restype = ctypes.c_uint32

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _descs(ts):
        arr = (_Tensor * max(1, len(ts)))()
        for i, t in enumerate(ts):
            arr[i].data = t.data.ctypes.data if t.data.size else None
            arr[i].numel = t.data.size
            arr[i].dtype = DTYPES[t.dtype]
        return arr

    # -- the method ------------------------------------------------------
    def clip(self, tensors, max_norm: float, inv_scale: float = 1.0):
        """Return (clipped copies, OracleResult); the inputs are not modified."""
        outs = [OracleTensor(t.data.copy(), t.dtype) for t in tensors]
        res = _Result()
        rc = self._lib.oracle_clip(self._descs(tensors), self._descs(outs),
                                   len(tensors), float(max_norm), float(inv_scale),
                                   ctypes.byref(res))
        if rc != 0:
            raise ValueError("oracle_clip rejected its arguments")
        return outs, OracleResult(res.sumsq, res.norm, res.coef,
                                  bool(res.nonfinite), res.decision)

    def clip_sample(self, tensors, max_norm: float, inv_scale, tensor_idx, elem_idx):
        """The clip of the whole set, with the outputs of only the chosen
        elements: returns (list of storage arrays, one value per sample in its
        tensor's format, OracleResult)."""
        ti = np.ascontiguousarray(tensor_idx, dtype=np.int32)
        ei = np.ascontiguousarray(elem_idx, dtype=np.int64)
        slots = np.zeros(ti.size, dtype=np.uint32)
        res = _Result()
        rc = self._lib.oracle_clip_sample(self._descs(tensors), len(tensors), float(max_norm),
                                          float(inv_scale), ti.ctypes.data, ei.ctypes.data,
                                          ti.size, slots.ctypes.data, ctypes.byref(res))
        if rc != 0:
            raise ValueError("oracle_clip_sample rejected its arguments")
        return slots, OracleResult(res.sumsq, res.norm, res.coef, bool(res.nonfinite),
                                   res.decision)

    def accumulate(self, tensors, addends):
        """Return copies of `tensors` with `addends` added element by element,
        each sum rounded once to its format; the inputs are not modified."""
        outs = [OracleTensor(t.data.copy(), t.dtype) for t in tensors]
        if len(addends) != len(tensors):
            raise ValueError("one addend per tensor")
        rc = self._lib.oracle_accumulate(self._descs(outs), self._descs(addends), len(outs))
        if rc != 0:
            raise ValueError("oracle_accumulate rejected its arguments")
        return outs

    def clip_accumulate(self, tensors, addends, max_norm: float, inv_scale: float = 1.0):
        """The last microbatch's accumulation, then the clip of the sums:
        returns (new copies of `tensors`, OracleResult); inputs unmodified."""
        outs = [OracleTensor(t.data.copy(), t.dtype) for t in tensors]
        if len(addends) != len(tensors):
            raise ValueError("one addend per tensor")
        res = _Result()
        rc = self._lib.oracle_clip_accumulate(self._descs(outs), self._descs(addends), len(outs),
                                              float(max_norm), float(inv_scale),
                                              ctypes.byref(res))
        if rc != 0:
            raise ValueError("oracle_clip_accumulate rejected its arguments")
        return outs, OracleResult(res.sumsq, res.norm, res.coef, bool(res.nonfinite),
                                  res.decision)

    def clip_to_f32(self, tensors, max_norm: float, inv_scale: float = 1.0, fill=np.nan):
        """Out-of-place clip into new float32 arrays (left at `fill` on
        SKIP); returns (outputs, OracleResult)."""
        outs = [np.full(t.data.size, fill, dtype=np.float32) for t in tensors]
        ptrs = (ctypes.c_void_p * max(1, len(outs)))(*[o.ctypes.data if o.size else None
                                                        for o in outs])
        res = _Result()
        rc = self._lib.oracle_clip_to_f32(self._descs(tensors), ptrs, len(tensors),
                                          float(max_norm), float(inv_scale), ctypes.byref(res))
        if rc != 0:
            raise ValueError("oracle_clip_to_f32 rejected its arguments")
        return outs, OracleResult(res.sumsq, res.norm, res.coef, bool(res.nonfinite),
                                  res.decision)

    def clip_adamw(self, tensors, states, max_norm: float, inv_scale: float = 1.0, *,
                   lr: float, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                   weight_decay: float = 0.0, step: int = 1, zero_grads: bool = False):
        """Clip, then one AdamW step.  `states` is a list of (w, m, v) float32
        arrays; returns (new gradients, [(w, m, v)], OracleResult); the inputs
        are not modified."""
        grads = [OracleTensor(t.data.copy(), t.dtype) for t in tensors]
        new = [tuple(np.ascontiguousarray(a, dtype=np.float32).reshape(-1).copy() for a in st)
               for st in states]
        for t, (w, m, v) in zip(tensors, new):
            if not (w.size == m.size == v.size == t.data.size):
                raise ValueError("state arrays must match their gradient tensor")
        sts = (_AdamwState * max(1, len(new)))()
        for i, (w, m, v) in enumerate(new):
            sts[i].w, sts[i].m, sts[i].v = (a.ctypes.data if a.size else None for a in (w, m, v))
        p = _AdamwParams(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                         int(step), int(bool(zero_grads)), 0)
        res = _Result()
        rc = self._lib.oracle_clip_adamw(self._descs(grads), sts, len(grads), float(max_norm),
                                         float(inv_scale), ctypes.byref(p), ctypes.byref(res))
        if rc != 0:
            raise ValueError("oracle_clip_adamw rejected its arguments")
        return grads, new, OracleResult(res.sumsq, res.norm, res.coef, bool(res.nonfinite),
                                        res.decision)

    def clip_per_tensor(self, tensors, max_norm: float, inv_scale: float = 1.0):
        outs = [OracleTensor(t.data.copy(), t.dtype) for t in tensors]
        res = (_Result * max(1, len(tensors)))()
        rc = self._lib.oracle_clip_per_tensor(self._descs(tensors), self._descs(outs),
                                              len(tensors), float(max_norm),
                                              float(inv_scale), res)
        if rc != 0:
            raise ValueError("oracle_clip_per_tensor rejected its arguments")
        return outs, [OracleResult(r.sumsq, r.norm, r.coef, bool(r.nonfinite),
                                   r.decision) for r in res[:len(tensors)]]

    def sumsq(self, tensors, inv_scale: float = 1.0):
        s = ctypes.c_double()
        nf = ctypes.c_int32()
        rc = self._lib.oracle_sumsq(self._descs(tensors), len(tensors),
                                    float(inv_scale), ctypes.byref(s), ctypes.byref(nf))
        if rc != 0:
            raise ValueError("oracle_sumsq rejected its arguments")
        return s.value, bool(nf.value)

    def value_clip(self, x, c: float) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty_like(x)
        self._lib.oracle_value_clip(x.ctypes.data, x.size, float(c), out.ctypes.data)
        return out

    # -- storage-format conversions (exposed so the tests can pin them) ---
    def decode(self, t: OracleTensor) -> np.ndarray:
        out = np.empty(t.data.size, dtype=np.float64)
        for i in range(t.data.size):
            out[i] = self._lib.oracle_decode(t.data.ctypes.data, i, DTYPES[t.dtype])
        return out

    def encode(self, values, dtype: str) -> OracleTensor:
        v = np.ascontiguousarray(values, dtype=np.float64).reshape(-1)
        data = np.zeros(v.size, dtype=_STORAGE[dtype])
        for i in range(v.size):
            self._lib.oracle_encode(data.ctypes.data, i, DTYPES[dtype], float(v[i]))
        return OracleTensor(data, dtype)

    def round_grid_f32_bits(self, v: float) -> int:
        return int(self._lib.oracle_round_grid_f32_bits(float(v)))


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    """The oracle as built from source with no planted mistake."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(0)
    return _DEFAULT


def clip(tensors, max_norm, inv_scale=1.0):
    return default().clip(tensors, max_norm, inv_scale)


def sumsq(tensors, inv_scale=1.0):
    return default().sumsq(tensors, inv_scale)


if __name__ == "__main__":  # pragma: no cover - manual build step
    print(build(int(sys.argv[1]) if len(sys.argv) > 1 else 0))
