"""Global L2-norm gradient clipping on one GB300 GPU.

A thin Python face of the C ABI in ``include/gclip.h`` (library
``libgclip.so``, built by :func:`build`).  PyTorch supplies device memory and
streams; every step of the clip runs in the library's CUDA kernels.

    clipper = GradClipper([p.grad for p in model.parameters()])
    norm, flag = clipper.clip_(max_norm=1.0, inv_scale=1.0 / (loss_scale * n_micro))

The clip follows "Grow a language model: gradient clipping" (unhomeschool.com),
section "Mathematics", and "Gradient Clipping" (paweldubiel.com glossary),
section "Mechanism and details": norm = sqrt(sum of squares over every
element), elements scaled by max_norm / norm when norm > max_norm.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import (GCLIP_BF16, GCLIP_DECISION_CLIP, GCLIP_DECISION_PASS,
                   GCLIP_DECISION_SKIP, GCLIP_F16, GCLIP_F32, GCLIP_STATUS_OK,
                   GCLIP_STATUS_TIMEOUT, GCLIP_VARIANT_PERSISTENT,
                   GCLIP_VARIANT_SPLIT, GclipError, clip_chunk_t,
                   clip_result_t, clip_tensor_desc_t, check, load)
from ._build import build as _build_lib

__all__ = ["build", "load", "GradClipper", "GclipError", "plan", "descs_for",
           "GCLIP_F32", "GCLIP_F16", "GCLIP_BF16", "GCLIP_VARIANT_SPLIT",
           "GCLIP_VARIANT_PERSISTENT", "GCLIP_DECISION_PASS", "GCLIP_DECISION_CLIP",
           "GCLIP_DECISION_SKIP", "GCLIP_STATUS_OK", "GCLIP_STATUS_TIMEOUT"]

DTYPE_CODES = {torch.float32: GCLIP_F32, torch.float16: GCLIP_F16,
               torch.bfloat16: GCLIP_BF16}
VARIANTS = {"split": GCLIP_VARIANT_SPLIT,
            "persistent": GCLIP_VARIANT_PERSISTENT,
            "split_tma": _abi.GCLIP_VARIANT_SPLIT_TMA,
            "persistent_tma": _abi.GCLIP_VARIANT_PERSISTENT_TMA,
            "split_wave": _abi.GCLIP_VARIANT_SPLIT_WAVE,
            "three_kernel": _abi.GCLIP_VARIANT_THREE_KERNEL}


def build(force: bool = False) -> str:
    """Compile libgclip.so for sm_103a (in-tree) and load it."""
    path = _build_lib(force=force)
    load()
    return path


def descs_for(tensors) -> ctypes.Array:
    """C descriptors for a list of contiguous tensors (any device; the
    library only accepts CUDA memory at clip_create)."""
    arr = (clip_tensor_desc_t * max(1, len(tensors)))()
    for i, t in enumerate(tensors):
        if t.dtype not in DTYPE_CODES:
            raise TypeError(f"unsupported gradient dtype {t.dtype}")
        if not t.is_contiguous():
            raise ValueError("gradient tensors must be contiguous")
        arr[i].ptr = t.data_ptr() if t.numel() else None
        arr[i].numel = t.numel()
        arr[i].dtype = DTYPE_CODES[t.dtype]
        arr[i].reserved = 0
    return arr


def plan(descs, n: int):
    """Host-only chunk table for `n` descriptors (no device needed)."""
    L = load()
    count = ctypes.c_int64()
    check("clip_plan", L.clip_plan(descs, n, None, 0, ctypes.byref(count)))
    table = (clip_chunk_t * max(1, count.value))()
    check("clip_plan", L.clip_plan(descs, n, table, count.value, ctypes.byref(count)))
    return [(table[i].addr, table[i].numel, table[i].meta) for i in range(count.value)]


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


class GradClipper:
    """One planned clip of a fixed set of CUDA gradient tensors.

    The tensors must stay allocated (same storage) for the clipper's life;
    they are clipped in place.  Calls on one clipper must not overlap on the
    device.
    """

    def __init__(self, tensors, variant: str | int | None = None):
        self.tensors = list(tensors)
        devs = {t.device for t in self.tensors}
        if any(d.type != "cuda" for d in devs) or len(devs) > 1:
            raise ValueError("all gradient tensors must be on one CUDA device")
        self.device = next(iter(devs)) if devs else torch.device("cuda", torch.cuda.current_device())
        self._lib = load()
        descs = descs_for(self.tensors)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            check("clip_create", self._lib.clip_create(descs, len(self.tensors), ctypes.byref(h)))
        self._h = h
        self.norm = torch.zeros(1, dtype=torch.float32, device=self.device)
        self.flag = torch.zeros(1, dtype=torch.int32, device=self.device)
        n = max(1, len(self.tensors))
        self._pt_norms = torch.zeros(n, dtype=torch.float32, device=self.device)
        self._pt_flags = torch.zeros(n, dtype=torch.int32, device=self.device)
        if variant is not None:
            self.set_variant(variant)

    # -- the hot path -----------------------------------------------------
    def clip_(self, max_norm: float, inv_scale: float = 1.0, stream=None,
              out_norm: torch.Tensor | None = None, out_flag: torch.Tensor | None = None):
        """Clip in place on `stream` (default: the current stream); returns the
        device tensors receiving the norm (float32[1]) and the nonfinite flag
        (int32[1]).  Nothing is synchronised."""
        out_norm = self.norm if out_norm is None else out_norm
        out_flag = self.flag if out_flag is None else out_flag
        check("clip_grad_norm", self._lib.clip_grad_norm(
            self._h, float(max_norm), float(inv_scale), out_norm.data_ptr(),
            out_flag.data_ptr(), _stream_handle(stream, self.device)))
        return out_norm, out_flag

    # -- per-tensor clipping ---------------------------------------------------
    def clip_per_tensor_(self, max_norm: float, inv_scale: float = 1.0, stream=None):
        """Clip every tensor by its own norm, in place.  Returns device tensors
        of the per-tensor norms (float32[n]) and nonfinite flags (int32[n])."""
        n = len(self.tensors)
        check("clip_grad_norm_per_tensor", self._lib.clip_grad_norm_per_tensor(
            self._h, float(max_norm), float(inv_scale), self._pt_norms.data_ptr(),
            self._pt_flags.data_ptr(), _stream_handle(stream, self.device)))
        return self._pt_norms[:n], self._pt_flags[:n]

    def per_tensor_results(self, stream=None) -> list:
        n = len(self.tensors)
        recs = (clip_result_t * max(1, n))()
        check("clip_read_per_tensor", self._lib.clip_read_per_tensor(
            self._h, recs, n, _stream_handle(stream, self.device)))
        return [{k: getattr(r, k) for k, _ in clip_result_t._fields_ if k != "reserved"}
                for r in recs[:n]]

    # -- out-of-place fp32 output ---------------------------------------------
    def attach_f32_out(self, outs) -> None:
        """Attach fp32 CUDA tensors, one per gradient tensor (same numel), to
        receive clip_to_f32_'s results.  They stay owned by the caller."""
        outs = list(outs)
        arr = (ctypes.c_void_p * max(1, len(outs)))()
        for i, o in enumerate(outs):
            if o.dtype != torch.float32 or not o.is_contiguous() or o.device != self.device:
                raise ValueError("outputs must be contiguous fp32 on the gradients' device")
            arr[i] = o.data_ptr() if o.numel() else None
        self._outs = outs
        check("clip_attach_f32_out", self._lib.clip_attach_f32_out(self._h, arr, len(outs)))

    def clip_to_f32_(self, max_norm: float, inv_scale: float = 1.0, stream=None):
        """Clip into the attached fp32 outputs; the gradients are only read.
        Returns (norm, flag) device tensors."""
        check("clip_grad_norm_to_f32", self._lib.clip_grad_norm_to_f32(
            self._h, float(max_norm), float(inv_scale), self.norm.data_ptr(),
            self.flag.data_ptr(), _stream_handle(stream, self.device)))
        return self.norm, self.flag

    # -- the last microbatch's accumulation folded into the clip -------------
    def attach_addend(self, addends) -> None:
        """Attach CUDA tensors, one per gradient tensor (same numel and dtype),
        that clip_accumulate_ adds into the gradients.  They stay owned by the
        caller and are only read."""
        addends = list(addends)
        arr = (ctypes.c_void_p * max(1, len(addends)))()
        for i, (a, g) in enumerate(zip(addends, self.tensors)):
            if a.dtype != g.dtype or not a.is_contiguous() or a.device != self.device:
                raise ValueError("addends must be contiguous, of the gradient's dtype and device")
            arr[i] = a.data_ptr() if a.numel() else None
        self._addends = addends
        check("clip_attach_addend", self._lib.clip_attach_addend(self._h, arr, len(addends)))

    def clip_accumulate_(self, max_norm: float, inv_scale: float = 1.0, stream=None):
        """Add the attached addends into the gradients, then clip the sums in
        place (see clip_grad_norm_accumulate in include/gclip.h).  Returns
        (norm, flag) device tensors."""
        check("clip_grad_norm_accumulate", self._lib.clip_grad_norm_accumulate(
            self._h, float(max_norm), float(inv_scale), self.norm.data_ptr(),
            self.flag.data_ptr(), _stream_handle(stream, self.device)))
        return self.norm, self.flag

    # -- fused clip + AdamW --------------------------------------------------
    def attach_adamw(self, states) -> None:
        """Attach fp32 (w, m, v) CUDA tensors, one triple per gradient tensor
        (same numel), for clip_adamw_.  They stay owned by the caller."""
        states = list(states)
        arr = (_abi.clip_adamw_state_t * max(1, len(states)))()
        for i, (w, m, v) in enumerate(states):
            for a in (w, m, v):
                if a.dtype != torch.float32 or not a.is_contiguous() or a.device != self.device:
                    raise ValueError("AdamW state must be contiguous fp32 on the gradients' device")
            arr[i].w, arr[i].m, arr[i].v = (a.data_ptr() if a.numel() else None for a in (w, m, v))
        self._states = states
        check("clip_attach_adamw", self._lib.clip_attach_adamw(self._h, arr, len(states)))

    def clip_adamw_(self, max_norm: float, inv_scale: float = 1.0, *, lr: float,
                    beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                    weight_decay: float = 0.0, step: int = 1, zero_grads: bool = False,
                    stream=None):
        """Clip, then one AdamW step on the attached state (see
        clip_grad_norm_adamw in include/gclip.h).  Returns (norm, flag)."""
        p = _abi.clip_adamw_params_t(float(lr), float(beta1), float(beta2), float(eps),
                                     float(weight_decay), int(bool(zero_grads)))
        check("clip_grad_norm_adamw", self._lib.clip_grad_norm_adamw(
            self._h, float(max_norm), float(inv_scale), ctypes.byref(p), int(step),
            self.norm.data_ptr(), self.flag.data_ptr(), _stream_handle(stream, self.device)))
        return self.norm, self.flag

    def adamw_step_(self, *, lr: float, beta1: float = 0.9, beta2: float = 0.999,
                    eps: float = 1e-8, weight_decay: float = 0.0, step: int = 1,
                    zero_grads: bool = False, stream=None) -> None:
        """One AdamW step on the attached state with the gradients as they
        are, no clip (see clip_adamw_step in include/gclip.h)."""
        p = _abi.clip_adamw_params_t(float(lr), float(beta1), float(beta2), float(eps),
                                     float(weight_decay), int(bool(zero_grads)))
        check("clip_adamw_step", self._lib.clip_adamw_step(
            self._h, ctypes.byref(p), int(step), _stream_handle(stream, self.device)))

    # -- configuration and inspection -----------------------------------
    def set_variant(self, variant) -> None:
        v = VARIANTS[variant] if isinstance(variant, str) else int(variant)
        check("clip_set_variant", self._lib.clip_set_variant(self._h, v))

    @property
    def variant(self) -> int:
        return int(self._lib.clip_get_variant(self._h))

    @property
    def num_chunks(self) -> int:
        return int(self._lib.clip_num_chunks(self._h))

    @property
    def tma_grid(self) -> int:
        return int(self._lib.clip_tma_grid(self._h))

    @property
    def persistent_grid(self) -> int:
        return int(self._lib.clip_persistent_grid(self._h))

    def result(self, stream=None) -> dict:
        """The device record of the last call (synchronises `stream`)."""
        r = clip_result_t()
        check("clip_read_result", self._lib.clip_read_result(
            self._h, ctypes.byref(r), _stream_handle(stream, self.device)))
        return {k: getattr(r, k) for k, _ in clip_result_t._fields_ if k != "reserved"}

    def last_status(self, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Enqueue a copy of the record's status word (GCLIP_STATUS_*) into
        the device int32 tensor `out` (a new one if None); no sync."""
        if out is None:
            out = torch.empty(1, dtype=torch.int32, device=self.device)
        if out.dtype != torch.int32 or out.device != self.device:
            raise ValueError("out must be an int32 tensor on the gradients' device")
        check("clip_last_status", self._lib.clip_last_status(
            self._h, out.data_ptr(), _stream_handle(stream, self.device)))
        return out

    def reset(self, stream=None) -> None:
        check("clip_reset", self._lib.clip_reset(self._h, _stream_handle(stream, self.device)))

    def set_l2_keep(self, nbytes: int) -> None:
        check("clip_set_l2_keep", self._lib.clip_set_l2_keep(self._h, int(nbytes)))

    def debug_barrier(self, extra_arrivals: int, timeout_ns: int = 0) -> None:
        check("clip_debug_barrier", self._lib.clip_debug_barrier(
            self._h, int(extra_arrivals), int(timeout_ns)))

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            check("clip_destroy", self._lib.clip_destroy(self._h))
            self._h = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
