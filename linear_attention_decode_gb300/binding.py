"""ctypes binding of libgdnreplay.so — argument marshalling only.

Each function has the name of the C entry point it calls (declared in
``include/gdnreplay.h``).  It checks that the torch tensors it is given have the
shapes, dtypes and device the C call expects (the C layer cannot see tensor
sizes), packs their device pointers into the C structs, calls the library on
the current CUDA stream (or the one given) and raises ``GdnError`` on a
non-OK status.  There is no fallback: if the library is missing, loading it
raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgdnreplay.so")

from .constants import (BF16, DEV_BAD_ACCEPTED, DEV_BAD_SLOT, DEV_BAD_WRITE_POS, DEV_INTERNAL, DEV_TIMEOUT,  # noqa: F401
                        F16, F32, GATE_PER_K, GATE_SCALAR, GDN_DTYPE, RECON_FFMA, RECON_OUTPUT, RECON_TENSOR,
                        STEP_OVERLAP_PREVIOUS, STEP_PERSISTENT_KERNEL, TORCH_DTYPE)


class GdnError(RuntimeError):
    pass


class LayerDesc(ctypes.Structure):
    _fields_ = [("num_slots", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("num_k_heads", ctypes.c_int32), ("k_dim", ctypes.c_int32),
                ("v_dim", ctypes.c_int32), ("ring_len", ctypes.c_int32),
                ("gate", ctypes.c_int32), ("state_dtype", ctypes.c_int32),
                ("ring_dtype", ctypes.c_int32)]


class _Cache(ctypes.Structure):
    _fields_ = [("state", ctypes.c_void_p), ("ring_d", ctypes.c_void_p),
                ("ring_k", ctypes.c_void_p), ("ring_g", ctypes.c_void_p)]


class _SpecStep(ctypes.Structure):
    _fields_ = [("mixed_qkv", ctypes.c_void_p), ("qkv_dtype", ctypes.c_int32),
                ("qkv_row_stride", ctypes.c_int64), ("g", ctypes.c_void_p),
                ("beta", ctypes.c_void_p), ("ssm_state_indices", ctypes.c_void_p),
                ("batch", ctypes.c_int32), ("window", ctypes.c_int32), ("q_scale", ctypes.c_float),
                ("qk_l2norm", ctypes.c_int32), ("out", ctypes.c_void_p),
                ("out_dtype", ctypes.c_int32)]


class _Step(ctypes.Structure):
    _fields_ = [("mixed_qkv", ctypes.c_void_p), ("qkv_dtype", ctypes.c_int32),
                ("qkv_row_stride", ctypes.c_int64), ("g", ctypes.c_void_p),
                ("beta", ctypes.c_void_p), ("ssm_state_indices", ctypes.c_void_p),
                ("batch", ctypes.c_int32), ("q_scale", ctypes.c_float),
                ("qk_l2norm", ctypes.c_int32), ("out", ctypes.c_void_p),
                ("out_dtype", ctypes.c_int32), ("flags", ctypes.c_uint32)]


def layer_desc(num_slots, num_v_heads, num_k_heads, k_dim, v_dim, ring_len,
               gate=GATE_SCALAR, ring_dtype=F16, state_dtype=F32) -> LayerDesc:
    return LayerDesc(num_slots, num_v_heads, num_k_heads, k_dim, v_dim, ring_len,
                     gate, state_dtype, ring_dtype)


@dataclass
class Cache:
    """One layer's cache tensors (device)."""
    state: torch.Tensor                     # [N, HV, V, K] fp32
    ring_d: Optional[torch.Tensor] = None   # [N, HV, L, V] ring dtype
    ring_k: Optional[torch.Tensor] = None   # [N, HK, L, K] ring dtype
    ring_g: Optional[torch.Tensor] = None   # [N, HV, L] or [N, HV, L, K] fp32


@dataclass
class Step:
    """One decode step's inputs and output (device)."""
    mixed_qkv: torch.Tensor          # [B, >= 2*HK*K + HV*V], unit inner stride
    g: torch.Tensor                  # [B, HV] or [B, HV, K] fp32
    beta: torch.Tensor               # [B, HV] fp32
    ssm_state_indices: torch.Tensor  # [B] int32
    out: torch.Tensor                # [B, HV, V]
    q_scale: float = 1.0
    qk_l2norm: bool = False
    flags: int = 0                   # STEP_* bits (STEP_OVERLAP_PREVIOUS, STEP_PERSISTENT_KERNEL)


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libgdnreplay.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise GdnError(f"{path} is missing: build it with linear_attention_decode_gb300.build")
        lib = ctypes.CDLL(path)
        vp, i32, u32p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p
        dp = ctypes.POINTER(LayerDesc)
        cp, sp = ctypes.POINTER(_Cache), ctypes.POINTER(_Step)
        lib.gdn_packed_decode.argtypes = [dp, vp, sp, u32p, vp]
        lib.gdn_replayssm_decode.argtypes = [dp, cp, vp, vp, sp, i32, vp, u32p, vp]
        lib.gdn_replayssm_decode_advance.argtypes = [dp, cp, vp, vp, sp, i32, vp, vp, u32p, vp]
        lib.gdn_replayssm_decode_advance_noalloc.argtypes = [dp, cp, vp, vp, sp, i32, vp, u32p, vp]
        lib.gdn_replayssm_advance.argtypes = [vp, i32, vp, i32, i32, vp, u32p, vp]
        lib.gdn_replayssm_spec_verify.argtypes = [dp, cp, vp, ctypes.POINTER(_SpecStep), i32, u32p, vp]
        lib.gdn_replayssm_spec_commit.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, u32p, vp]
        lib.gdn_replayssm_flush.argtypes = [dp, cp, vp, vp, i32, u32p, vp]
        lib.gdn_replayssm_reset_slots.argtypes = [vp, i32, vp, i32, u32p, vp]
        lib.gdn_lossless_verify.argtypes = [dp, vp, ctypes.POINTER(_SpecStep), vp, vp, vp, u32p, vp]
        lib.gdn_lossless_commit.argtypes = [dp, vp, vp, vp, vp, i32, i32, vp, vp, vp, u32p, vp]
        lib.gdn_selftest_wait_timeout.argtypes = [u32p, ctypes.c_uint32, vp]
        lib.gdn_noalloc_scratch_peek.argtypes = [vp, i32]
        lib.gdn_replayssm_decode_kernel.argtypes = [dp, cp, sp, i32, vp]
        for f in ("gdn_packed_decode", "gdn_replayssm_decode", "gdn_replayssm_decode_advance",
                  "gdn_replayssm_decode_advance_noalloc", "gdn_replayssm_advance", "gdn_replayssm_flush",
                  "gdn_replayssm_reset_slots", "gdn_replayssm_spec_verify", "gdn_replayssm_spec_commit",
                  "gdn_lossless_verify", "gdn_lossless_commit", "gdn_selftest_wait_timeout",
                  "gdn_noalloc_scratch_peek", "gdn_replayssm_decode_kernel"):
            getattr(lib, f).restype = ctypes.c_int
        lib.gdn_status_str.argtypes = [ctypes.c_int]
        lib.gdn_status_str.restype = ctypes.c_char_p
        lib.gdn_last_error.argtypes = []
        lib.gdn_last_error.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _check(status: int, fn: str) -> None:
    if status != 0:
        lib = load_library()
        raise GdnError(f"{fn}: {lib.gdn_status_str(status).decode()}: {lib.gdn_last_error().decode()}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: Optional[torch.Tensor], name: str, shape=None, dtype=None, optional=False):
    if t is None:
        if optional:
            return None
        raise GdnError(f"{name} is required")
    if not t.is_cuda:
        raise GdnError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise GdnError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise GdnError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise GdnError(f"{name} must be contiguous")
    return t.data_ptr()


def _status_ptr(dev_status):
    return _dev(dev_status, "dev_status", (1,), torch.int32, optional=True)


def _pack_step(d: LayerDesc, s: Step) -> _Step:
    B = s.ssm_state_indices.shape[0]
    HV, HK, K, V = d.num_v_heads, d.num_k_heads, d.k_dim, d.v_dim
    q = s.mixed_qkv
    if not q.is_cuda or q.dim() != 2 or q.shape[0] != B or q.stride(1) != 1:
        raise GdnError("mixed_qkv must be a CUDA [B, row] tensor with unit inner stride")
    if q.shape[1] < 2 * HK * K + HV * V:
        raise GdnError("mixed_qkv rows are shorter than 2*HK*K + HV*V")
    if q.dtype not in GDN_DTYPE:
        raise GdnError("mixed_qkv must be fp32, bf16 or fp16")
    gshape = (B, HV, K) if d.gate == GATE_PER_K else (B, HV)
    if s.out.dtype not in GDN_DTYPE:
        raise GdnError("out must be fp32, bf16 or fp16")
    return _Step(q.data_ptr() if B else None, GDN_DTYPE[q.dtype], q.stride(0) if B > 1 else q.shape[1],
                 _dev(s.g, "g", gshape, torch.float32),
                 _dev(s.beta, "beta", (B, HV), torch.float32),
                 _dev(s.ssm_state_indices, "ssm_state_indices", (B,), torch.int32),
                 B, float(s.q_scale), int(bool(s.qk_l2norm)),
                 _dev(s.out, "out", (B, HV, V)), GDN_DTYPE[s.out.dtype], int(s.flags))


def _pack_cache(d: LayerDesc, c: Cache) -> _Cache:
    N, HV, HK, K, V, L = d.num_slots, d.num_v_heads, d.num_k_heads, d.k_dim, d.v_dim, d.ring_len
    rdt = TORCH_DTYPE[d.ring_dtype]
    st = _dev(c.state, "state", (N, HV, V, K), torch.float32)
    opt = L == 1
    gshape = (N, HV, L, K) if d.gate == GATE_PER_K else (N, HV, L)
    return _Cache(st, _dev(c.ring_d, "ring_d", (N, HV, L, V), rdt, opt),
                  _dev(c.ring_k, "ring_k", (N, HK, L, K), rdt, opt),
                  _dev(c.ring_g, "ring_g", gshape, torch.float32, opt))


def gdn_packed_decode(desc: LayerDesc, state: torch.Tensor, step: Step,
                      dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    st = _dev(state, "state", (desc.num_slots, desc.num_v_heads, desc.v_dim, desc.k_dim), torch.float32)
    s = _pack_step(desc, step)
    _check(load_library().gdn_packed_decode(ctypes.byref(desc), st, ctypes.byref(s),
                                            _status_ptr(dev_status), _stream(stream)),
           "gdn_packed_decode")


def gdn_replayssm_decode(desc: LayerDesc, cache: Cache, write_pos: torch.Tensor,
                         force_flush: Optional[torch.Tensor], step: Step,
                         recon: int = RECON_TENSOR, flushed_out: Optional[torch.Tensor] = None,
                         dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    B = step.ssm_state_indices.shape[0]
    c = _pack_cache(desc, cache)
    s = _pack_step(desc, step)
    _check(load_library().gdn_replayssm_decode(
        ctypes.byref(desc), ctypes.byref(c),
        _dev(write_pos, "write_pos", (desc.num_slots,), torch.int32),
        _dev(force_flush, "force_flush", (B,), torch.uint8, optional=True),
        ctypes.byref(s), int(recon),
        _dev(flushed_out, "flushed_out", (B,), torch.uint8, optional=True),
        _status_ptr(dev_status), _stream(stream)), "gdn_replayssm_decode")


# gdn_replayssm_decode_kernel results
KERNEL_PERSISTENT_TC, KERNEL_PER_HEAD_TC, KERNEL_CUDA_CORE, KERNEL_SMALL_BATCH = 0, 1, 2, 3


def gdn_replayssm_decode_kernel(desc: LayerDesc, cache: Cache, step: Step, recon: int = RECON_TENSOR) -> int:
    """Which decode kernel a call with these arguments would launch (host only)."""
    c = _pack_cache(desc, cache)
    s = _pack_step(desc, step)
    out = ctypes.c_int32(-1)
    _check(load_library().gdn_replayssm_decode_kernel(ctypes.byref(desc), ctypes.byref(c), ctypes.byref(s),
                                                      int(recon), ctypes.byref(out)), "gdn_replayssm_decode_kernel")
    return int(out.value)


DECODE_ADVANCE_WORKSPACE_BYTES = 4


def decode_advance_workspace(device=None) -> torch.Tensor:
    """A zeroed workspace for gdn_replayssm_decode_advance (each call leaves it zero)."""
    return torch.zeros(DECODE_ADVANCE_WORKSPACE_BYTES // 4, dtype=torch.int32, device=device or "cuda")


def gdn_replayssm_decode_advance(desc: LayerDesc, cache: Cache, write_pos: torch.Tensor,
                                 force_flush: Optional[torch.Tensor], step: Step, workspace: torch.Tensor,
                                 recon: int = RECON_TENSOR, flushed_out: Optional[torch.Tensor] = None,
                                 dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    B = step.ssm_state_indices.shape[0]
    c = _pack_cache(desc, cache)
    s = _pack_step(desc, step)
    _check(load_library().gdn_replayssm_decode_advance(
        ctypes.byref(desc), ctypes.byref(c),
        _dev(write_pos, "write_pos", (desc.num_slots,), torch.int32),
        _dev(force_flush, "force_flush", (B,), torch.uint8, optional=True),
        ctypes.byref(s), int(recon),
        _dev(flushed_out, "flushed_out", (B,), torch.uint8, optional=True),
        _dev(workspace, "workspace", (DECODE_ADVANCE_WORKSPACE_BYTES // 4,), torch.int32),
        _status_ptr(dev_status), _stream(stream)), "gdn_replayssm_decode_advance")


class PreparedCall:
    """One decode call's arguments checked and packed once, for a loop that
    calls it again and again with the same tensors (the buffers of a serving
    step: the caller refills them in place, keeps them alive and keeps their
    shapes, dtypes and addresses).  ``run()`` is then a single foreign call:
    what a Python loop pays per launch at small batch, where the kernels take a
    few microseconds.  Built by ``prepare_packed_decode`` and
    ``prepare_replayssm_decode``."""

    def __init__(self, fn, args, keep, name):
        self._fn, self._args, self._keep, self._name = fn, args, keep, name

    def run(self, stream=None) -> None:
        """The call on `stream` (a torch stream or a raw handle; default: the
        current stream)."""
        status = self._fn(*self._args, _stream(stream))
        if status != 0:
            _check(status, self._name)


def prepare_packed_decode(desc: LayerDesc, state: torch.Tensor, step: Step,
                          dev_status: Optional[torch.Tensor] = None) -> PreparedCall:
    """gdn_packed_decode with its arguments checked and packed once."""
    st = _dev(state, "state", (desc.num_slots, desc.num_v_heads, desc.v_dim, desc.k_dim), torch.float32)
    d = LayerDesc.from_buffer_copy(desc)
    s = _pack_step(desc, step)
    lib = load_library()
    return PreparedCall(lib.gdn_packed_decode, (ctypes.byref(d), st, ctypes.byref(s), _status_ptr(dev_status)),
                        (d, s, state, step, dev_status), "gdn_packed_decode")


def prepare_replayssm_decode(desc: LayerDesc, cache: Cache, write_pos: torch.Tensor,
                             force_flush: Optional[torch.Tensor], step: Step,
                             recon: int = RECON_TENSOR, workspace: Optional[torch.Tensor] = None,
                             flushed_out: Optional[torch.Tensor] = None,
                             dev_status: Optional[torch.Tensor] = None) -> PreparedCall:
    """gdn_replayssm_decode (or, with a workspace, gdn_replayssm_decode_advance)
    with its arguments checked and packed once."""
    B = step.ssm_state_indices.shape[0]
    d = LayerDesc.from_buffer_copy(desc)
    c = _pack_cache(desc, cache)
    s = _pack_step(desc, step)
    common = (ctypes.byref(d), ctypes.byref(c), _dev(write_pos, "write_pos", (desc.num_slots,), torch.int32),
              _dev(force_flush, "force_flush", (B,), torch.uint8, optional=True), ctypes.byref(s), int(recon),
              _dev(flushed_out, "flushed_out", (B,), torch.uint8, optional=True))
    keep = (d, c, s, cache, write_pos, force_flush, step, workspace, flushed_out, dev_status)
    lib = load_library()
    if workspace is None:
        return PreparedCall(lib.gdn_replayssm_decode, common + (_status_ptr(dev_status),), keep,
                            "gdn_replayssm_decode")
    ws = _dev(workspace, "workspace", (DECODE_ADVANCE_WORKSPACE_BYTES // 4,), torch.int32)
    return PreparedCall(lib.gdn_replayssm_decode_advance, common + (ws, _status_ptr(dev_status)), keep,
                        "gdn_replayssm_decode_advance")


def gdn_replayssm_decode_advance_noalloc(desc: LayerDesc, cache: Cache, write_pos: torch.Tensor,
                                         force_flush: Optional[torch.Tensor], step: Step,
                                         recon: int = RECON_TENSOR, flushed_out: Optional[torch.Tensor] = None,
                                         dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """gdn_replayssm_decode_advance with the library's own scratch: for callers
    that cannot allocate device memory (see the C declaration)."""
    B = step.ssm_state_indices.shape[0]
    c = _pack_cache(desc, cache)
    s = _pack_step(desc, step)
    _check(load_library().gdn_replayssm_decode_advance_noalloc(
        ctypes.byref(desc), ctypes.byref(c),
        _dev(write_pos, "write_pos", (desc.num_slots,), torch.int32),
        _dev(force_flush, "force_flush", (B,), torch.uint8, optional=True),
        ctypes.byref(s), int(recon),
        _dev(flushed_out, "flushed_out", (B,), torch.uint8, optional=True),
        _status_ptr(dev_status), _stream(stream)), "gdn_replayssm_decode_advance_noalloc")


def gdn_noalloc_scratch_peek(n: int = 1):
    """The first n 32-bit words of the no-alloc entry point's scratch array on
    the current device (a blocking copy; for tests and diagnostics)."""
    buf = (ctypes.c_uint32 * n)()
    _check(load_library().gdn_noalloc_scratch_peek(ctypes.cast(buf, ctypes.c_void_p), int(n)),
           "gdn_noalloc_scratch_peek")
    return list(buf)


def _pack_spec_step(desc: LayerDesc, T: int, step: Step) -> _SpecStep:
    B = step.ssm_state_indices.shape[0]
    HV, HK, K, V = desc.num_v_heads, desc.num_k_heads, desc.k_dim, desc.v_dim
    q = step.mixed_qkv
    if not q.is_cuda or q.dim() != 2 or q.shape[0] != B * T or q.stride(1) != 1:
        raise GdnError("mixed_qkv must be a CUDA [B*T, row] tensor with unit inner stride")
    if q.shape[1] < 2 * HK * K + HV * V:
        raise GdnError("mixed_qkv rows are shorter than 2*HK*K + HV*V")
    if q.dtype not in GDN_DTYPE or step.out.dtype not in GDN_DTYPE:
        raise GdnError("mixed_qkv and out must be fp32, bf16 or fp16")
    gshape = (B * T, HV, K) if desc.gate == GATE_PER_K else (B * T, HV)
    return _SpecStep(q.data_ptr() if B else None, GDN_DTYPE[q.dtype], q.stride(0) if B * T > 1 else q.shape[1],
                     _dev(step.g, "g", gshape, torch.float32), _dev(step.beta, "beta", (B * T, HV), torch.float32),
                     _dev(step.ssm_state_indices, "ssm_state_indices", (B,), torch.int32), B, T,
                     float(step.q_scale), int(bool(step.qk_l2norm)),
                     _dev(step.out, "out", (B * T, HV, V)), GDN_DTYPE[step.out.dtype])


def tuple_shapes(desc: LayerDesc, batch: int, window: int):
    """Shapes of the lossless verify's fp32 tuple buffers (u, k, g)."""
    B, T, HV, HK, K, V = batch, window, desc.num_v_heads, desc.num_k_heads, desc.k_dim, desc.v_dim
    return ((B, T, HV, V), (B, T, HK, K), (B, T, HV, K) if desc.gate == GATE_PER_K else (B, T, HV))


def gdn_lossless_verify(desc: LayerDesc, state: torch.Tensor, window: int, step: Step, tup_u: torch.Tensor,
                        tup_k: torch.Tensor, tup_g: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    """Lossless verify: `step` holds B*T token rows (token t of row b at row
    b*T + t); out is [B*T, HV, V]; the fp32 tuples have tuple_shapes(desc, B, T)."""
    T = int(window)
    B = step.ssm_state_indices.shape[0]
    su, sk, sg = tuple_shapes(desc, B, T)
    s = _pack_spec_step(desc, T, step)
    _check(load_library().gdn_lossless_verify(
        ctypes.byref(desc), _dev(state, "state", (desc.num_slots, desc.num_v_heads, desc.v_dim, desc.k_dim),
                                 torch.float32),
        ctypes.byref(s), _dev(tup_u, "tup_u", su, torch.float32), _dev(tup_k, "tup_k", sk, torch.float32),
        _dev(tup_g, "tup_g", sg, torch.float32), _status_ptr(dev_status), _stream(stream)), "gdn_lossless_verify")


def gdn_lossless_commit(desc: LayerDesc, state: torch.Tensor, ssm_state_indices: torch.Tensor,
                        accepted: torch.Tensor, window: int, tup_u: torch.Tensor, tup_k: torch.Tensor,
                        tup_g: torch.Tensor, dst_indices: Optional[torch.Tensor] = None,
                        dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Exact-order commit of each row's accepted tuples into state (in place,
    or into dst_indices[b] when given)."""
    T = int(window)
    B = ssm_state_indices.shape[0]
    su, sk, sg = tuple_shapes(desc, B, T)
    _check(load_library().gdn_lossless_commit(
        ctypes.byref(desc), _dev(state, "state", (desc.num_slots, desc.num_v_heads, desc.v_dim, desc.k_dim),
                                 torch.float32),
        _dev(ssm_state_indices, "ssm_state_indices", (B,), torch.int32),
        _dev(dst_indices, "dst_indices", (B,), torch.int32, optional=True),
        _dev(accepted, "accepted", (B,), torch.int32), B, T,
        _dev(tup_u, "tup_u", su, torch.float32), _dev(tup_k, "tup_k", sk, torch.float32),
        _dev(tup_g, "tup_g", sg, torch.float32), _status_ptr(dev_status), _stream(stream)), "gdn_lossless_commit")


def gdn_replayssm_spec_verify(desc: LayerDesc, cache: Cache, write_pos: torch.Tensor, window: int,
                              step: Step, recon: int = RECON_TENSOR, dev_status: Optional[torch.Tensor] = None,
                              stream=None) -> None:
    """Speculative verify window: `step` holds B*T token rows (token t of row b
    at row b*T + t) and ssm_state_indices [B]; out is [B*T, HV, V]."""
    T = int(window)
    B = step.ssm_state_indices.shape[0]
    HV, HK, K, V = desc.num_v_heads, desc.num_k_heads, desc.k_dim, desc.v_dim
    q = step.mixed_qkv
    if not q.is_cuda or q.dim() != 2 or q.shape[0] != B * T or q.stride(1) != 1:
        raise GdnError("mixed_qkv must be a CUDA [B*T, row] tensor with unit inner stride")
    if q.shape[1] < 2 * HK * K + HV * V:
        raise GdnError("mixed_qkv rows are shorter than 2*HK*K + HV*V")
    if q.dtype not in GDN_DTYPE or step.out.dtype not in GDN_DTYPE:
        raise GdnError("mixed_qkv and out must be fp32, bf16 or fp16")
    gshape = (B * T, HV, K) if desc.gate == GATE_PER_K else (B * T, HV)
    s = _SpecStep(q.data_ptr() if B else None, GDN_DTYPE[q.dtype], q.stride(0) if B * T > 1 else q.shape[1],
                  _dev(step.g, "g", gshape, torch.float32), _dev(step.beta, "beta", (B * T, HV), torch.float32),
                  _dev(step.ssm_state_indices, "ssm_state_indices", (B,), torch.int32), B, T,
                  float(step.q_scale), int(bool(step.qk_l2norm)),
                  _dev(step.out, "out", (B * T, HV, V)), GDN_DTYPE[step.out.dtype])
    c = _pack_cache(desc, cache)
    _check(load_library().gdn_replayssm_spec_verify(
        ctypes.byref(desc), ctypes.byref(c), _dev(write_pos, "write_pos", (desc.num_slots,), torch.int32),
        ctypes.byref(s), int(recon), _status_ptr(dev_status), _stream(stream)), "gdn_replayssm_spec_verify")


def gdn_replayssm_spec_commit(ssm_state_indices: torch.Tensor, accepted: torch.Tensor, window: int,
                              num_slots: int, ring_len: int, write_pos: torch.Tensor, flush_slots: torch.Tensor,
                              dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    B = ssm_state_indices.shape[0]
    _check(load_library().gdn_replayssm_spec_commit(
        _dev(ssm_state_indices, "ssm_state_indices", (B,), torch.int32),
        _dev(accepted, "accepted", (B,), torch.int32), B, int(window), int(num_slots), int(ring_len),
        _dev(write_pos, "write_pos", (num_slots,), torch.int32),
        _dev(flush_slots, "flush_slots", (B,), torch.int32), _status_ptr(dev_status), _stream(stream)),
        "gdn_replayssm_spec_commit")


def gdn_replayssm_advance(ssm_state_indices: torch.Tensor, force_flush: Optional[torch.Tensor],
                          num_slots: int, ring_len: int, write_pos: torch.Tensor,
                          dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    B = ssm_state_indices.shape[0]
    _check(load_library().gdn_replayssm_advance(
        _dev(ssm_state_indices, "ssm_state_indices", (B,), torch.int32), B,
        _dev(force_flush, "force_flush", (B,), torch.uint8, optional=True),
        int(num_slots), int(ring_len), _dev(write_pos, "write_pos", (num_slots,), torch.int32),
        _status_ptr(dev_status), _stream(stream)), "gdn_replayssm_advance")


def gdn_replayssm_flush(desc: LayerDesc, cache: Cache, write_pos: torch.Tensor,
                        slots: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    n = slots.shape[0]
    c = _pack_cache(desc, cache)
    _check(load_library().gdn_replayssm_flush(
        ctypes.byref(desc), ctypes.byref(c),
        _dev(write_pos, "write_pos", (desc.num_slots,), torch.int32),
        _dev(slots, "slots", (n,), torch.int32), n, _status_ptr(dev_status), _stream(stream)),
        "gdn_replayssm_flush")


def gdn_replayssm_reset_slots(write_pos: torch.Tensor, slots: torch.Tensor,
                              dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    n = slots.shape[0]
    N = write_pos.shape[0]
    _check(load_library().gdn_replayssm_reset_slots(
        _dev(write_pos, "write_pos", (N,), torch.int32), N,
        _dev(slots, "slots", (n,), torch.int32), n, _status_ptr(dev_status), _stream(stream)),
        "gdn_replayssm_reset_slots")


def gdn_selftest_wait_timeout(dev_status: torch.Tensor, limit_us: int = 2000, stream=None) -> None:
    """One block waits, with the decode kernels' bounded wait, on a barrier
    nothing completes; dev_status ([1] int32) gets DEV_TIMEOUT."""
    _check(load_library().gdn_selftest_wait_timeout(_status_ptr(dev_status), int(limit_us), _stream(stream)),
           "gdn_selftest_wait_timeout")


def gdn_status_str(status: int) -> str:
    return load_library().gdn_status_str(int(status)).decode()


def gdn_last_error() -> str:
    return load_library().gdn_last_error().decode()
