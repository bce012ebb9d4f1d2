"""CPU oracle for GDN / KDA ReplaySSM decode (test infrastructure only).

A plain double-precision C model (``gdn_oracle.c``) of what the decode path
computes, loaded with ctypes.  It shares nothing with the CUDA library and the
product never imports it: only the tests, the smoke check and the benchmark's
CPU-baseline leg do.

Every function here is argument marshalling around one C function; the
arithmetic and its citations live in ``gdn_oracle.c``.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")

F64, F32, F16, BF16 = 0, 1, 2, 3
GATE_SCALAR, GATE_PER_K = 0, 1
BAD_SLOT, BAD_WRITE_POS, BAD_ACCEPTED = 1, 2, 16


def compile_source(src: str, out: str) -> str:
    """Compiles one oracle source with gcc (no FMA contraction, so x86 and Arm agree)."""
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                    "-I", _HERE, src, "-o", out, "-lm"], check=True)
    return out


def build(force: bool = False) -> str:
    """Compiles the oracle library if it is missing or older than its sources."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "gdn_oracle.h"))
    ):
        tmp = _SO + f".tmp{os.getpid()}"
        compile_source(_SRC, tmp)
        os.replace(tmp, _SO)
    return _SO


_lib_handle = None


def _configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    dp, ip = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)
    up, bp = ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_ubyte)
    gp = ctypes.POINTER(Geom)
    lib.oracle_round.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.oracle_round.restype = ctypes.c_double
    lib.oracle_round_array.argtypes = [dp, ctypes.c_long, ctypes.c_int]
    lib.oracle_gdn_step.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, dp, dp,
                                    ctypes.c_double, ctypes.c_double, dp, dp]
    lib.oracle_kda_step.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp,
                                    ctypes.c_double, dp, dp]
    lib.oracle_packed_decode.argtypes = [gp, dp, ctypes.c_int, ip, dp, dp, dp,
                                         ctypes.c_double, ctypes.c_int, dp, up]
    lib.oracle_replay_state.argtypes = [gp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, dp]
    lib.oracle_replay_decode.argtypes = [gp, dp, dp, dp, dp, ip, ctypes.c_int, ip, bp,
                                         dp, dp, dp, ctypes.c_double, ctypes.c_int,
                                         dp, bp, up]
    lib.oracle_replay_advance.argtypes = [ctypes.c_int, ctypes.c_int, ip, bp,
                                          ctypes.c_int, ip, up]
    lib.oracle_replay_fold.argtypes = [gp, dp, dp, dp, dp, ip, ctypes.c_int, ip, up]
    lib.oracle_spec_verify.argtypes = [gp, dp, dp, dp, dp, ip, ctypes.c_int, ctypes.c_int, ip,
                                       dp, dp, dp, ctypes.c_double, ctypes.c_int, dp, up]
    lib.oracle_spec_commit.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ip, ip,
                                       ip, ip, up]
    fp = ctypes.POINTER(ctypes.c_float)
    lib.oracle_step_f32.argtypes = [ctypes.c_int, ctypes.c_int, fp, fp, fp, fp, ctypes.c_float, fp,
                                    ctypes.c_float, fp, fp]
    lib.oracle_lossless_verify.argtypes = [gp, dp, ctypes.c_int, ctypes.c_int, ip, dp, dp, dp,
                                           ctypes.c_double, ctypes.c_int, dp, dp, dp, dp, up]
    lib.oracle_lossless_commit.argtypes = [gp, fp, ctypes.c_int, ctypes.c_int, ip, ip, ip, fp, fp, fp, up]
    return lib


def _lib():
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _configure(ctypes.CDLL(build()))
    return _lib_handle


@contextlib.contextmanager
def using_library(path: str):
    """Temporarily routes every oracle call to another build of the oracle
    source (the mutation tests plant a mistake in a copy and load it here)."""
    global _lib_handle
    saved = _lib()
    _lib_handle = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib_handle = saved


class Geom(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("N", "HV", "HK", "K", "V", "L", "gate", "state_dtype", "ring_dtype")]


def geom(N, HV, HK, K, V, L=1, gate=GATE_SCALAR, state_dtype=F32, ring_dtype=F32) -> Geom:
    if HV % HK:
        raise ValueError("HV must be a multiple of HK")
    return Geom(N, HV, HK, K, V, L, gate, state_dtype, ring_dtype)


def _d(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous, "oracle arrays are C-contiguous float64"
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i(a: np.ndarray):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _b(a):
    if a is None:
        return None
    assert a.dtype == np.uint8 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))


def f64(a) -> np.ndarray:
    """Exact conversion of any numeric array (torch or numpy) to C-contiguous float64."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def round_to(x, dtype: int) -> np.ndarray:
    """Round every element to the storage type (IEEE round-to-nearest-even)."""
    out = f64(x).copy()
    _lib().oracle_round_array(_d(out), out.size, dtype)
    return out


def gdn_step(S: np.ndarray, q, k, v, g: float, beta: float):
    """One sequential GDN step on one head; S ([V][K]) is updated in place. Returns (y, u)."""
    V, K = S.shape
    q, k, v = f64(q), f64(k), f64(v)
    y, u = np.zeros(V), np.zeros(V)
    _lib().oracle_gdn_step(K, V, _d(S), _d(q), _d(k), _d(v), float(g), float(beta), _d(y), _d(u))
    return y, u


def kda_step(S: np.ndarray, q, k, v, g, beta: float):
    """One sequential KDA step (per-key-channel gate g[K]) on one head; S updated in place."""
    V, K = S.shape
    q, k, v, g = f64(q), f64(k), f64(v), f64(g)
    y, u = np.zeros(V), np.zeros(V)
    _lib().oracle_kda_step(K, V, _d(S), _d(q), _d(k), _d(v), _d(g), float(beta), _d(y), _d(u))
    return y, u


@dataclass
class Cache:
    """One layer's ReplaySSM cache held in double (values already at their storage type)."""
    state: np.ndarray   # [N, HV, V, K]
    ring_d: np.ndarray  # [N, HV, L, V]
    ring_k: np.ndarray  # [N, HK, L, K]
    ring_g: np.ndarray  # [N, HV, L] or [N, HV, L, K]

    @staticmethod
    def from_arrays(state, ring_d, ring_k, ring_g) -> "Cache":
        return Cache(f64(state).copy(), f64(ring_d).copy(), f64(ring_k).copy(), f64(ring_g).copy())

    def copy(self) -> "Cache":
        return Cache(self.state.copy(), self.ring_d.copy(), self.ring_k.copy(), self.ring_g.copy())


def packed_decode(G: Geom, state: np.ndarray, indices, mixed_qkv, g, beta,
                  q_scale: float = 1.0, qk_l2norm: int = 0):
    """Read + write baseline over one batch; state updated in place. Returns (o, status)."""
    idx = np.ascontiguousarray(np.asarray(indices, dtype=np.int32))
    qkv, gg, bb = f64(mixed_qkv), f64(g), f64(beta)
    B = idx.shape[0]
    o = np.zeros((B, G.HV, G.V))
    st = ctypes.c_uint(0)
    _lib().oracle_packed_decode(ctypes.byref(G), _d(state), B, _i(idx), _d(qkv), _d(gg), _d(bb),
                                float(q_scale), int(qk_l2norm), _d(o), ctypes.byref(st))
    return o, st.value


def replay_state(G: Geom, cache: Cache, slot: int, hv: int, p: int) -> np.ndarray:
    """Pre-token state of (slot, hv) rebuilt from the checkpoint and p ring entries."""
    S = np.zeros((G.V, G.K))
    _lib().oracle_replay_state(ctypes.byref(G), _d(cache.state), _d(cache.ring_d),
                               _d(cache.ring_k), _d(cache.ring_g), slot, hv, p, _d(S))
    return S


def replay_decode(G: Geom, cache: Cache, write_pos, indices, force_flush, mixed_qkv, g, beta,
                  q_scale: float = 1.0, qk_l2norm: int = 0):
    """One ReplaySSM decode launch; cache updated in place. Returns (o, flushed, status)."""
    wp = np.ascontiguousarray(np.asarray(write_pos, dtype=np.int32))
    idx = np.ascontiguousarray(np.asarray(indices, dtype=np.int32))
    ff = None if force_flush is None else np.ascontiguousarray(np.asarray(force_flush, dtype=np.uint8))
    qkv, gg, bb = f64(mixed_qkv), f64(g), f64(beta)
    B = idx.shape[0]
    o = np.zeros((B, G.HV, G.V))
    flushed = np.zeros(B, dtype=np.uint8)
    st = ctypes.c_uint(0)
    _lib().oracle_replay_decode(ctypes.byref(G), _d(cache.state), _d(cache.ring_d),
                                _d(cache.ring_k), _d(cache.ring_g), _i(wp), B, _i(idx), _b(ff),
                                _d(qkv), _d(gg), _d(bb), float(q_scale), int(qk_l2norm), _d(o),
                                _b(flushed), ctypes.byref(st))
    return o, flushed, st.value


def replay_advance(N: int, indices, force_flush, L: int, write_pos: np.ndarray) -> int:
    """Cursor advance once per forward; write_pos (int32) updated in place. Returns status."""
    idx = np.ascontiguousarray(np.asarray(indices, dtype=np.int32))
    ff = None if force_flush is None else np.ascontiguousarray(np.asarray(force_flush, dtype=np.uint8))
    st = ctypes.c_uint(0)
    _lib().oracle_replay_advance(N, idx.shape[0], _i(idx), _b(ff), L, _i(write_pos), ctypes.byref(st))
    return st.value


def replay_fold(G: Geom, cache: Cache, write_pos, slots) -> int:
    """Fold each listed slot's ring into its checkpoint (cursor untouched). Returns status."""
    wp = np.ascontiguousarray(np.asarray(write_pos, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int32))
    st = ctypes.c_uint(0)
    _lib().oracle_replay_fold(ctypes.byref(G), _d(cache.state), _d(cache.ring_d), _d(cache.ring_k),
                              _d(cache.ring_g), _i(wp), sl.shape[0], _i(sl), ctypes.byref(st))
    return st.value


def spec_verify(G: Geom, cache: Cache, write_pos, indices, T: int, mixed_qkv, g, beta,
                q_scale: float = 1.0, qk_l2norm: int = 0):
    """Verify window of T tokens per row (token t of row b at row b*T + t of the
    inputs); the ring gets the window's entries, checkpoint and cursors stay.
    Returns (o [B*T, HV, V], status)."""
    wp = np.ascontiguousarray(np.asarray(write_pos, dtype=np.int32))
    idx = np.ascontiguousarray(np.asarray(indices, dtype=np.int32))
    qkv, gg, bb = f64(mixed_qkv), f64(g), f64(beta)
    B = idx.shape[0]
    o = np.zeros((B * T, G.HV, G.V))
    st = ctypes.c_uint(0)
    _lib().oracle_spec_verify(ctypes.byref(G), _d(cache.state), _d(cache.ring_d), _d(cache.ring_k),
                              _d(cache.ring_g), _i(wp), B, int(T), _i(idx), _d(qkv), _d(gg), _d(bb),
                              float(q_scale), int(qk_l2norm), _d(o), ctypes.byref(st))
    return o, st.value


def spec_commit(N: int, L: int, T: int, indices, accepted, write_pos: np.ndarray):
    """Move the cursors over the accepted tokens; write_pos (int32) updated in
    place. Returns (flush_slots [B], status)."""
    idx = np.ascontiguousarray(np.asarray(indices, dtype=np.int32))
    acc = np.ascontiguousarray(np.asarray(accepted, dtype=np.int32))
    fs = np.zeros(idx.shape[0], dtype=np.int32)
    st = ctypes.c_uint(0)
    _lib().oracle_spec_commit(N, L, int(T), idx.shape[0], _i(idx), _i(acc), _i(write_pos), _i(fs),
                              ctypes.byref(st))
    return fs, st.value


def _f(a: np.ndarray):
    assert a.dtype == np.float32 and a.flags.c_contiguous, "binary32 oracle arrays are C-contiguous float32"
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def f32(a) -> np.ndarray:
    """Exact (or RNE) conversion of any numeric array to C-contiguous float32."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def step_f32(h: np.ndarray, q, k, v, g: float, beta: float, gk=None):
    """One binary32 step of the sequential recurrence (decayed state formed once,
    update as one fma); h ([V][K] float32) updated in place. Returns (y, u)."""
    V, K = h.shape
    q, k, v = f32(q), f32(k), f32(v)
    gkk = None if gk is None else f32(gk)
    y, u = np.zeros(V, dtype=np.float32), np.zeros(V, dtype=np.float32)
    _lib().oracle_step_f32(K, V, _f(h), _f(q), _f(k), _f(v), float(g), None if gkk is None else _f(gkk),
                           float(beta), _f(y), _f(u))
    return y, u


def lossless_verify(G: Geom, state: np.ndarray, indices, T: int, mixed_qkv, g, beta,
                    q_scale: float = 1.0, qk_l2norm: int = 0):
    """Verify of T tokens per row without a state update. Returns
    (o [B*T, HV, V], tup_u [B, T, HV, V], tup_k [B, T, HK, K], tup_g [B, T, HV(, K)], status);
    tuples are fp32 values held in float64."""
    idx = np.ascontiguousarray(np.asarray(indices, dtype=np.int32))
    qkv, gg, bb = f64(mixed_qkv), f64(g), f64(beta)
    B = idx.shape[0]
    o = np.zeros((B * T, G.HV, G.V))
    tu = np.zeros((B, T, G.HV, G.V))
    tk = np.zeros((B, T, G.HK, G.K))
    tg = np.zeros((B, T, G.HV, G.K) if G.gate == GATE_PER_K else (B, T, G.HV))
    st = ctypes.c_uint(0)
    _lib().oracle_lossless_verify(ctypes.byref(G), _d(state), B, int(T), _i(idx), _d(qkv), _d(gg), _d(bb),
                                  float(q_scale), int(qk_l2norm), _d(o), _d(tu), _d(tk), _d(tg),
                                  ctypes.byref(st))
    return o, tu, tk, tg, st.value


def lossless_commit(G: Geom, state: np.ndarray, T: int, src, accepted, tup_u, tup_k, tup_g, dst=None) -> int:
    """Exact-order (binary32) replay of each row's accepted tuples into state
    (float32 [N, HV, V, K], updated in place). Returns status."""
    s_ = np.ascontiguousarray(np.asarray(src, dtype=np.int32))
    a_ = np.ascontiguousarray(np.asarray(accepted, dtype=np.int32))
    d_ = None if dst is None else np.ascontiguousarray(np.asarray(dst, dtype=np.int32))
    u, k, g = f32(tup_u), f32(tup_k), f32(tup_g)
    st = ctypes.c_uint(0)
    _lib().oracle_lossless_commit(ctypes.byref(G), _f(state), s_.shape[0], int(T), _i(s_),
                                  None if d_ is None else _i(d_), _i(a_), _f(u), _f(k), _f(g), ctypes.byref(st))
    return st.value
