"""Shared driver for the GPU parity tests: runs the CUDA path (through the C ABI
binding) and the CPU oracle on the same seeded inputs, step by step, and
compares everything a step produces."""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Callable, Optional

import numpy as np
import torch

import oracle as O
from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import inputs as I

# gdn_dtype_t -> oracle storage type
ORACLE_DT = {Bd.F32: O.F32, Bd.F16: O.F16, Bd.BF16: O.BF16}

# Error bounds, as a fraction of max|reference| over one launch's tensor:
# fp32 ring + CUDA-core replay; any fp16/bf16 ring or tensor-core replay.
TOL_FFMA_F32 = 1e-5
TOL_TC = 2e-3


# The tensor-core recon runs two ways in the parity tests: as a caller gets it
# (a batch with few (row, head) items takes the small-batch kernel) and, as
# TCP, forced onto the persistent tensor-core kernel (STEP_PERSISTENT_KERNEL).
TCP = 1000


def recon_and_flags(recon: int):
    """The C recon value and the extra step flags of a test's recon id."""
    return (Bd.RECON_TENSOR, Bd.STEP_PERSISTENT_KERNEL) if recon == TCP else (recon, 0)


def decode(desc, cache, write_pos, force_flush, step, recon=Bd.RECON_TENSOR, *args, **kw):
    """gdn_replayssm_decode with a test recon id (TCP included)."""
    r, f = recon_and_flags(recon)
    return Bd.gdn_replayssm_decode(desc, cache, write_pos, force_flush, replace(step, flags=step.flags | f), r,
                                   *args, **kw)


def tolerance(w: I.Workload, recon: int) -> float:
    recon, _ = recon_and_flags(recon)
    if recon in (Bd.RECON_FFMA, Bd.RECON_OUTPUT) and w.ring_dtype == Bd.F32:
        return TOL_FFMA_F32
    if w.ring_dtype == Bd.BF16:
        # Both sides round nearly equal corrections d to bf16 on their own; a
        # pair that straddles a rounding boundary lands one bf16 ulp (2^-7 of
        # the entry) apart, and the replay carries that into later outputs and
        # checkpoints with weight w_j |k_j| <= 1.  The bound gets that ulp.
        return TOL_TC + 2.0 ** -7
    return TOL_TC


# A value stored at a narrower type is round(x_gpu) on one side and round(x_ref)
# on the other: the two can sit one unit in the last place apart even when x_gpu
# and x_ref are within the bound, so stored ring values get one ulp on top
# (2^-7 of the value for bf16, 2^-10 for fp16, 2^-23 for fp32).
STORAGE_ULP = {Bd.BF16: 2.0 ** -7, Bd.F16: 2.0 ** -10, Bd.F32: 2.0 ** -23}


# Guard bands: every device tensor a parity run hands the library sits between
# two 4 KiB bands of a known bit pattern (a NaN pattern for float views), checked
# bitwise after each step, so a write just outside a tensor cannot go unseen.
GUARD_BYTES = 4096
GUARD_WORD = 0x7FA5A5A5


class Guarded:
    """A device copy of a tensor between two guard bands; the body starts
    `offset` bytes past a 16-byte boundary (a multiple of the element size)."""

    def __init__(self, t: torch.Tensor, offset: int = 0):
        self.nbytes = t.numel() * t.element_size()
        assert offset % t.element_size() == 0 and 0 <= offset < 16
        self.start = GUARD_BYTES + offset
        total = 2 * GUARD_BYTES + ((offset + self.nbytes + 15) // 16) * 16
        self.raw = torch.full((total // 4,), GUARD_WORD, dtype=torch.int32, device="cuda")
        u8 = self.raw.view(torch.uint8)
        self.body = u8[self.start:self.start + self.nbytes].view(t.dtype).view(t.shape)
        self.body.copy_(t.to("cuda"))
        self.bands = torch.cat([u8[:self.start], u8[self.start + self.nbytes:]]).clone()

    def check(self, what: str) -> None:
        u8 = self.raw.view(torch.uint8)
        now = torch.cat([u8[:self.start], u8[self.start + self.nbytes:]])
        assert torch.equal(now, self.bands), f"{what}: a write landed in the guard band around the tensor"


def guarded(t: torch.Tensor, keep: list, offset: int = 0) -> torch.Tensor:
    """Device tensor with t's contents inside guard bands; its checker goes to keep."""
    g = Guarded(t, offset)
    keep.append(g)
    return g.body


def check_guards(keep: list, what: str) -> None:
    for g in keep:
        g.check(what)


def ring_tolerance(w: I.Workload, tol: float) -> float:
    return tol + STORAGE_ULP[w.ring_dtype]


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return err / scale if scale > 0 else err


def oracle_geom(w: I.Workload):
    return O.geom(w.N, w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, state_dtype=O.F32,
                  ring_dtype=ORACLE_DT[w.ring_dtype])


@dataclass
class Layer:
    """One layer's device cache plus the oracle's copy of it."""
    w: I.Workload
    dev: Bd.Cache
    ora: O.Cache
    init: I.CacheTensors  # CPU copy of the initial cache (for untouched checks)
    guards: list = field(default_factory=list)

    @staticmethod
    def make(w: I.Workload, gen, wp_cpu: torch.Tensor, ring_g_offset: int = 0) -> "Layer":
        c = I.cache(gen, w, wp_cpu, "cpu")
        g: list = []
        dev = Bd.Cache(guarded(c.state, g), guarded(c.ring_d, g), guarded(c.ring_k, g),
                       guarded(c.ring_g, g, ring_g_offset))
        return Layer(w, dev, O.Cache.from_arrays(c.state, c.ring_d, c.ring_k, c.ring_g), c, g)


@dataclass
class StepReport:
    o_err: float = 0.0
    state_err: float = 0.0
    ring_d_err: float = 0.0
    flushes: int = 0
    appends: int = 0


@dataclass
class RunReport:
    steps: list = field(default_factory=list)

    @property
    def max_o(self):
        return max(s.o_err for s in self.steps)

    @property
    def max_state(self):
        return max(s.state_err for s in self.steps)


def desc_of(w: I.Workload) -> Bd.LayerDesc:
    return Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, ring_dtype=w.ring_dtype)


def run_parity(w: I.Workload, recon: int, steps: Optional[int] = None,
               force: Optional[Callable[[int, int], np.ndarray]] = None,
               out_dtype=torch.float32, layers: int = 1, tol: Optional[float] = None,
               check_untouched: bool = True, q_scale: float = 1.0, qk_l2norm: bool = False,
               tweak: Optional[Callable[[int, "I.StepInputs"], None]] = None, overlap: bool = False,
               outputs: Optional[list] = None, ring_g_offset: int = 0, qkv_offset: int = 0) -> RunReport:
    """Runs `steps` decode steps of `layers` layers sharing one cursor array
    on both sides and asserts parity after every step.  overlap: every layer
    but the first is launched with STEP_OVERLAP_PREVIOUS (the launch before it
    touches neither its cache nor the cursors).  outputs: if given, receives
    each step's outputs (float64, [rows, HV, V]) of every layer.  ring_g_offset:
    the g ring starts that many bytes past a 16-byte boundary (the ABI asks
    only for float alignment there).  qkv_offset: mixed_qkv is a view that
    starts that many elements into a wider buffer (rows neither 16-byte aligned
    nor a multiple of 16 bytes apart)."""
    steps = w.steps if steps is None else steps
    tol = tolerance(w, recon) if tol is None else tol
    gen = I.generator(w.seed, "cpu")
    wp = I.write_pos(gen, w, "cpu")
    Ls = [Layer.make(w, gen, wp, ring_g_offset) for _ in range(layers)]
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu")
    rows = idx.shape[0]
    live = idx.numpy() >= 0
    io_guards: list = []
    wp_dev = guarded(wp, io_guards)
    wp_ora = wp.numpy().astype(np.int32).copy()
    idx_dev = guarded(idx, io_guards)
    desc = desc_of(w)
    G = oracle_geom(w)
    status = guarded(torch.zeros(1, dtype=torch.int32), io_guards)
    flushed = guarded(torch.zeros(rows, dtype=torch.uint8), io_guards)
    report = RunReport()
    for t in range(steps):
        ff = None if force is None else force(t, rows)
        ff_dev = None if ff is None else torch.from_numpy(ff).cuda()
        wp_before = wp_ora.copy()
        rep = StepReport()
        for li, layer in enumerate(Ls):
            si = I.step_inputs(gen, w, "cpu")
            if tweak is not None:
                tweak(t, si)
            step_guards: list = []
            out = guarded(torch.full((rows, w.HV, w.V), float("nan"), dtype=out_dtype), step_guards)
            flags = Bd.STEP_OVERLAP_PREVIOUS if (overlap and li > 0) else 0
            qkv = guarded(si.mixed_qkv, step_guards)
            if qkv_offset:
                row = si.mixed_qkv.shape[1]
                wide = torch.zeros((rows, row + qkv_offset + 6), dtype=si.mixed_qkv.dtype)
                wide[:, qkv_offset:qkv_offset + row] = si.mixed_qkv
                qkv = guarded(wide, step_guards)[:, qkv_offset:qkv_offset + row]
            step = Bd.Step(qkv, guarded(si.g, step_guards),
                           guarded(si.beta, step_guards), idx_dev, out, q_scale=q_scale, qk_l2norm=qk_l2norm,
                           flags=flags)
            decode(desc, layer.dev, wp_dev, ff_dev, step, recon, flushed, status)
            o_ref, fl_ref, st_ref = O.replay_decode(G, layer.ora, wp_ora, idx.numpy(), ff,
                                                    si.mixed_qkv, si.g, si.beta, q_scale, int(qk_l2norm))
            torch.cuda.synchronize()
            assert st_ref == 0 and int(status.item()) == 0, f"status gpu={status.item()} oracle={st_ref}"
            assert np.array_equal(flushed.cpu().numpy(), fl_ref), f"flush flags differ at step {t}"
            o = out.float().cpu().numpy()
            if outputs is not None:
                outputs.append(o.astype(np.float64))
            assert np.all(o[~live] == 0.0), "padding rows must be exactly zero"
            ref = o_ref
            if out_dtype != torch.float32:
                ref = torch.from_numpy(o_ref).to(out_dtype).double().numpy()
            rep.o_err = max(rep.o_err, rel_err(o[live], ref[live]))
            assert rep.o_err <= tol, f"step {t} layer {li}: out rel err {rep.o_err:.3e} > {tol:.1e}"
            _compare_cache(layer, w, idx.numpy(), wp_before, fl_ref, tol, rep, t, exact_k=not qk_l2norm)
            check_guards(step_guards + layer.guards, f"step {t} layer {li}")
        Bd.gdn_replayssm_advance(idx_dev, ff_dev, w.N, w.L, wp_dev, status)
        torch.cuda.synchronize()
        check_guards(io_guards, f"step {t} cursors")
        O.replay_advance(w.N, idx.numpy(), ff, w.L, wp_ora)
        assert np.array_equal(wp_dev.cpu().numpy(), wp_ora), f"write_pos differs after step {t}"
        report.steps.append(rep)
    if check_untouched:
        unused = torch.from_numpy(np.setdiff1d(np.arange(w.N), idx.numpy()[live]))
        for layer in Ls:
            for name in ("state", "ring_d", "ring_k", "ring_g"):
                a = getattr(layer.dev, name).cpu()[unused]
                b = getattr(layer.init, name)[unused]
                assert torch.equal(_bits(a), _bits(b)), f"{name} of a slot no row names was modified"
    return report


def _bits(t: torch.Tensor) -> torch.Tensor:
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _compare_cache(layer: Layer, w: I.Workload, idx, wp_before, flushed, tol, rep: StepReport, t,
                   exact_k: bool = True):
    """Flushed rows: the whole checkpoint within tolerance.  Appending rows: the
    new ring entry (k and g bit-exact, d within tolerance).  Small caches are
    also compared whole, NaN-filled stale positions included, so a write to a
    wrong slot, head or position cannot hide.  With the in-kernel L2 norm the
    cached key is computed, not copied, and is compared within the bound."""
    for b, slot in enumerate(idx):
        if slot < 0:
            continue
        p = int(wp_before[slot])
        if flushed[b]:
            rep.flushes += 1
            e = rel_err(layer.dev.state[slot].cpu().numpy(), layer.ora.state[slot])
            rep.state_err = max(rep.state_err, e)
            assert e <= tol, f"step {t}: flushed checkpoint rel err {e:.3e} > {tol:.1e}"
        else:
            rep.appends += 1
            gk = layer.dev.ring_k[slot, :, p].double().cpu().numpy()
            if exact_k:
                assert np.array_equal(gk, layer.ora.ring_k[slot, :, p]), f"step {t}: ring k entry differs"
            else:
                assert rel_err(gk, layer.ora.ring_k[slot, :, p]) <= ring_tolerance(w, tol)
            gg = layer.dev.ring_g[slot, :, p].double().cpu().numpy()
            assert np.array_equal(gg, layer.ora.ring_g[slot, :, p]), f"step {t}: ring g entry differs"
            e = rel_err(layer.dev.ring_d[slot, :, p].double().cpu().numpy(), layer.ora.ring_d[slot, :, p])
            rep.ring_d_err = max(rep.ring_d_err, e)
            assert e <= ring_tolerance(w, tol), f"step {t}: ring d rel err {e:.3e}"
    if layer.dev.state.numel() <= (1 << 23):
        rk = layer.dev.ring_k.double().cpu().numpy()
        if exact_k:
            assert np.array_equal(rk, layer.ora.ring_k, equal_nan=True), f"step {t}: ring k tensor differs"
        else:
            assert np.array_equal(np.isnan(rk), np.isnan(layer.ora.ring_k)), f"step {t}: stale ring k written"
        rg = layer.dev.ring_g.double().cpu().numpy()
        assert np.array_equal(rg, layer.ora.ring_g, equal_nan=True), f"step {t}: ring g tensor differs"
        rd = layer.dev.ring_d.double().cpu().numpy()
        nan = np.isnan(layer.ora.ring_d)
        assert np.array_equal(np.isnan(rd), nan), f"step {t}: ring d written at a stale position"
        assert rel_err(rd[~nan], layer.ora.ring_d[~nan]) <= ring_tolerance(w, tol)
        e = rel_err(layer.dev.state.cpu().numpy(), layer.ora.state)
        assert e <= tol, f"step {t}: checkpoint tensor rel err {e:.3e}"


def run_sampled(w: I.Workload, recon: int, steps: int = 2, samples: int = 6) -> RunReport:
    """Full-size launch on the GPU (inputs generated there); the oracle
    recomputes a seeded sample of rows one by one from copies of their slots."""
    tol = tolerance(w, recon)
    gen = I.generator(w.seed, "cuda")
    wp = I.write_pos(gen, w, "cuda")
    c = I.cache(gen, w, wp, "cuda")
    dev = Bd.Cache(c.state, c.ring_d, c.ring_k, c.ring_g)
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cuda")
    rows = idx.shape[0]
    desc = desc_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flushed = torch.empty(rows, dtype=torch.uint8, device="cuda")
    pick = np.random.default_rng(w.seed)
    report = RunReport()
    for t in range(steps):
        si = I.step_inputs(gen, w, "cuda")
        idx_h = idx.cpu().numpy()
        live_rows = np.nonzero(idx_h >= 0)[0]
        chosen = np.sort(pick.choice(live_rows, size=min(samples, live_rows.size), replace=False))
        slots = idx_h[chosen]
        wp_h = wp.cpu().numpy()
        # the sampled slots' cache before the step, as a small oracle pool
        sl = torch.as_tensor(slots, dtype=torch.long, device="cuda")
        ch = torch.as_tensor(chosen, dtype=torch.long, device="cuda")
        mini = O.Cache.from_arrays(dev.state[sl], dev.ring_d[sl], dev.ring_k[sl], dev.ring_g[sl])
        out = torch.full((rows, w.HV, w.V), float("nan"), dtype=torch.float32, device="cuda")
        step = Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out)
        decode(desc, dev, wp, None, step, recon, flushed, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        Gm = O.geom(len(slots), w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, state_dtype=O.F32,
                    ring_dtype=ORACLE_DT[w.ring_dtype])
        o_ref, fl_ref, st = O.replay_decode(Gm, mini, wp_h[slots].astype(np.int32), np.arange(len(slots)),
                                            None, si.mixed_qkv[ch], si.g[ch], si.beta[ch])
        assert st == 0
        rep = StepReport()
        o = out.cpu().numpy()
        assert np.all(o[idx_h < 0] == 0.0)
        rep.o_err = rel_err(o[chosen], o_ref)
        assert rep.o_err <= tol, f"step {t}: sampled out rel err {rep.o_err:.3e}"
        assert np.array_equal(flushed.cpu().numpy()[chosen], fl_ref)
        fl_all = flushed.cpu().numpy()[live_rows]
        p_all = wp_h[idx_h[live_rows]]
        assert np.array_equal(fl_all, (p_all == w.L - 1).astype(np.uint8)), "flush flags"
        for i, (b, slot) in enumerate(zip(chosen, slots)):
            p = int(wp_h[slot])
            if fl_ref[i]:
                rep.flushes += 1
                e = rel_err(dev.state[slot].cpu().numpy(), mini.state[i])
                rep.state_err = max(rep.state_err, e)
                assert e <= tol, f"step {t}: flushed checkpoint rel err {e:.3e}"
            else:
                rep.appends += 1
                assert np.array_equal(dev.ring_k[slot, :, p].double().cpu().numpy(), mini.ring_k[i, :, p])
                assert np.array_equal(dev.ring_g[slot, :, p].double().cpu().numpy(), mini.ring_g[i, :, p])
                e = rel_err(dev.ring_d[slot, :, p].double().cpu().numpy(), mini.ring_d[i, :, p])
                assert e <= ring_tolerance(w, tol)
        Bd.gdn_replayssm_advance(idx, None, w.N, w.L, wp, status)
        wp_ref = wp_h.copy()
        O.replay_advance(w.N, idx_h, None, w.L, wp_ref)
        assert np.array_equal(wp.cpu().numpy(), wp_ref)
        report.steps.append(rep)
    return report
