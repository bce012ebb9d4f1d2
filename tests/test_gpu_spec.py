"""The speculative verify window and its commit (gdn_replayssm_spec_verify,
gdn_replayssm_spec_commit) against the oracle's window and commit, on the same
seeded inputs, window after window: outputs of every token, the ring entries the
window caches (k and g bit for bit, d within the bound), cursors and fold lists
bit for bit, and the checkpoints the folds write.  Rejected drafts stay in the
ring past the cursor on both sides, so the whole ring is compared too.

The windows of a run cross several folds (the commit lists a slot once its next
window would not fit), and the acceptance counts are drawn at random in
[0, T], so both the all-rejected and the all-accepted commits occur."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_harness import ORACLE_DT, TOL_TC, _bits, desc_of, oracle_geom, rel_err, ring_tolerance, tolerance
from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu

FF, TC = Bd.RECON_FFMA, Bd.RECON_TENSOR

CASES = {
    # fp32 ring: the CUDA-core bound; GQA 2:1, padding rows, several windows per fold
    "gdn_f32_T3": (I.Workload("spec f32", N=12, B=5, n_pad=2, HV=4, HK=2, K=128, L=9, ring_dtype=Bd.F32,
                              qkv_dtype=Bd.BF16, steps=10, seed=41), 3),
    "gdn_f16_T4": (I.Workload("spec f16", N=12, B=6, n_pad=1, HV=8, HK=4, K=128, L=16, ring_dtype=Bd.F16,
                              qkv_dtype=Bd.BF16, steps=10, seed=42), 4),
    "gdn_bf16_T2_k64": (I.Workload("spec bf16 K=64", N=10, B=4, n_pad=1, HV=4, HK=4, K=64, L=6,
                                   ring_dtype=Bd.BF16, qkv_dtype=Bd.F16, steps=10, seed=43), 2),
    "kda_f32_T3": (I.Workload("spec kda f32", N=8, B=3, n_pad=1, HV=4, HK=4, K=128, L=8, ring_dtype=Bd.F32,
                              qkv_dtype=Bd.BF16, gate=Bd.GATE_PER_K, steps=10, seed=44), 3),
    "kda_f16_T5_k64": (I.Workload("spec kda f16 K=64", N=8, B=4, n_pad=0, HV=4, HK=2, K=64, L=12,
                                  ring_dtype=Bd.F16, qkv_dtype=Bd.BF16, gate=Bd.GATE_PER_K, steps=8, seed=45), 5),
    # window of one token: a commit is a plain decode step that may be rejected
    "gdn_f32_T1": (I.Workload("spec T=1", N=8, B=4, n_pad=1, HV=4, HK=2, K=128, L=4, ring_dtype=Bd.F32,
                              qkv_dtype=Bd.F32, steps=8, seed=46), 1),
    # the largest window the ring allows: every commit folds
    "gdn_f16_T_max": (I.Workload("spec T=L-1", N=8, B=3, n_pad=1, HV=4, HK=2, K=128, L=8, ring_dtype=Bd.F16,
                                 qkv_dtype=Bd.BF16, steps=5, seed=47), 7),
}


def _cursors(gen, w: I.Workload, T: int) -> torch.Tensor:
    """Cursors uniform over the positions a window of T fits at (p + T <= L - 1)."""
    return torch.randint(0, w.L - T, (w.N,), generator=gen, dtype=torch.int32)


def _compare_window(dev: Bd.Cache, ora: O.Cache, w: I.Workload, idx, wp_before, T: int, tol: float, tag: str):
    """Ring entries p .. p+T-1 of every live row, then the whole ring."""
    for slot in idx[idx >= 0]:
        p = int(wp_before[slot])
        hk_rows = dev.ring_k[slot, :, p:p + T].double().cpu().numpy()
        assert np.array_equal(hk_rows, ora.ring_k[slot, :, p:p + T]), f"{tag}: cached k differs"
        gg = dev.ring_g[slot, :, p:p + T].double().cpu().numpy()
        assert np.array_equal(gg, ora.ring_g[slot, :, p:p + T]), f"{tag}: cached g differs"
        e = rel_err(dev.ring_d[slot, :, p:p + T].double().cpu().numpy(), ora.ring_d[slot, :, p:p + T])
        assert e <= ring_tolerance(w, tol), f"{tag}: cached d rel err {e:.3e}"
    rk = dev.ring_k.double().cpu().numpy()
    assert np.array_equal(rk, ora.ring_k, equal_nan=True), f"{tag}: ring k tensor differs"
    rg = dev.ring_g.double().cpu().numpy()
    assert np.array_equal(rg, ora.ring_g, equal_nan=True), f"{tag}: ring g tensor differs"
    rd = dev.ring_d.double().cpu().numpy()
    nan = np.isnan(ora.ring_d)
    assert np.array_equal(np.isnan(rd), nan), f"{tag}: ring d written at a position the oracle did not write"
    assert rel_err(rd[~nan], ora.ring_d[~nan]) <= ring_tolerance(w, tol), f"{tag}: ring d tensor"


@pytest.mark.parametrize("recon", [TC, FF], ids=["tensor", "ffma"])
@pytest.mark.parametrize("name", list(CASES))
def test_spec_windows_match_the_oracle(gdnlib, name, recon):
    w, T = CASES[name]
    tol = tolerance(w, recon)
    gen = I.generator(w.seed, "cpu")
    wp = _cursors(gen, w, T)
    c = I.cache(gen, w, wp, "cpu")
    dev = Bd.Cache(c.state.cuda(), c.ring_d.cuda(), c.ring_k.cuda(), c.ring_g.cuda())
    ora = O.Cache.from_arrays(c.state, c.ring_d, c.ring_k, c.ring_g)
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu")
    idx_h = idx.numpy()
    live = idx_h >= 0
    rows = idx_h.shape[0]
    idx_dev = idx.cuda()
    wp_dev = wp.cuda()
    wp_ora = wp.numpy().astype(np.int32).copy()
    desc = desc_of(w)
    G = oracle_geom(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush_dev = torch.empty(rows, dtype=torch.int32, device="cuda")
    acc_rng = np.random.default_rng(w.seed)
    folds = accepted_total = 0
    for win in range(w.steps):
        si = I.step_inputs(gen, w, "cpu", rows=rows * T)
        out = torch.full((rows * T, w.HV, w.V), float("nan"), device="cuda")
        Bd.gdn_replayssm_spec_verify(desc, dev, wp_dev, T,
                                     Bd.Step(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda(), idx_dev, out),
                                     recon, status)
        wp_before = wp_ora.copy()
        o_ref, st = O.spec_verify(G, ora, wp_ora, idx_h, T, si.mixed_qkv, si.g, si.beta)
        torch.cuda.synchronize()
        assert st == 0 and int(status.item()) == 0, f"window {win}: status gpu={status.item()} oracle={st}"
        assert np.array_equal(wp_dev.cpu().numpy(), wp_ora), f"window {win}: verify moved a cursor"
        o = out.cpu().numpy().reshape(rows, T, w.HV, w.V)
        o_ref = o_ref.reshape(rows, T, w.HV, w.V)
        assert np.all(o[~live] == 0.0), "padding rows must be exactly zero"
        e = rel_err(o[live], o_ref[live])
        assert e <= tol, f"window {win}: out rel err {e:.3e} > {tol:.1e}"
        _compare_window(dev, ora, w, idx_h, wp_before, T, tol, f"window {win}")

        acc = acc_rng.integers(0, T + 1, size=rows).astype(np.int32)
        accepted_total += int(acc[live].sum())
        Bd.gdn_replayssm_spec_commit(idx_dev, torch.from_numpy(acc).cuda(), T, w.N, w.L, wp_dev, flush_dev,
                                     status)
        fs_ref, st = O.spec_commit(w.N, w.L, T, idx_h, acc, wp_ora)
        torch.cuda.synchronize()
        assert st == 0 and int(status.item()) == 0
        assert np.array_equal(wp_dev.cpu().numpy(), wp_ora), f"window {win}: cursors differ after the commit"
        assert np.array_equal(flush_dev.cpu().numpy(), fs_ref), f"window {win}: fold lists differ"
        if np.any(fs_ref >= 0):
            folds += int((fs_ref >= 0).sum())
            Bd.gdn_replayssm_flush(desc, dev, wp_dev, flush_dev, status)
            Bd.gdn_replayssm_reset_slots(wp_dev, flush_dev, status)
            assert O.replay_fold(G, ora, wp_ora, fs_ref) == 0
            wp_ora[fs_ref[fs_ref >= 0]] = 0
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert np.array_equal(wp_dev.cpu().numpy(), wp_ora)
            for s in fs_ref[fs_ref >= 0]:
                e = rel_err(dev.state[s].cpu().numpy(), ora.state[s])
                assert e <= tol, f"window {win}: folded checkpoint rel err {e:.3e}"
    assert folds >= 2, "the run should cross several folds"
    assert accepted_total > 0
    e = rel_err(dev.state.cpu().numpy(), ora.state)
    assert e <= tol, f"checkpoint tensor rel err {e:.3e}"
    unused = torch.from_numpy(np.setdiff1d(np.arange(w.N), idx_h[live]))
    for name_ in ("state", "ring_d", "ring_k", "ring_g"):
        a = getattr(dev, name_).cpu()[unused]
        b = getattr(c, name_)[unused]
        assert torch.equal(_bits(a), _bits(b)), f"{name_} of a slot no row names was modified"


def test_tensor_core_decode_reads_what_the_windows_cached(gdnlib):
    """Windows, commits and folds, then plain decode steps through the
    tensor-core kernel: the ring the windows left (rejected drafts included)
    must decode as the oracle's does."""
    w, T = I.Workload("spec then decode", N=16, B=8, n_pad=1, HV=8, HK=4, K=128, L=16, ring_dtype=Bd.F16,
                      qkv_dtype=Bd.BF16, steps=4, seed=48), 4
    gen = I.generator(w.seed, "cpu")
    wp = _cursors(gen, w, T)
    c = I.cache(gen, w, wp, "cpu")
    dev = Bd.Cache(c.state.cuda(), c.ring_d.cuda(), c.ring_k.cuda(), c.ring_g.cuda())
    ora = O.Cache.from_arrays(c.state, c.ring_d, c.ring_k, c.ring_g)
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu")
    idx_h = idx.numpy()
    live = idx_h >= 0
    rows = idx_h.shape[0]
    idx_dev, wp_dev = idx.cuda(), wp.cuda()
    wp_ora = wp.numpy().astype(np.int32).copy()
    desc, G = desc_of(w), oracle_geom(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush_dev = torch.empty(rows, dtype=torch.int32, device="cuda")
    acc_rng = np.random.default_rng(w.seed)
    for win in range(w.steps):
        si = I.step_inputs(gen, w, "cpu", rows=rows * T)
        out = torch.empty((rows * T, w.HV, w.V), device="cuda")
        Bd.gdn_replayssm_spec_verify(desc, dev, wp_dev, T,
                                     Bd.Step(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda(), idx_dev, out),
                                     TC, status)
        O.spec_verify(G, ora, wp_ora, idx_h, T, si.mixed_qkv, si.g, si.beta)
        acc = acc_rng.integers(0, T + 1, size=rows).astype(np.int32)
        Bd.gdn_replayssm_spec_commit(idx_dev, torch.from_numpy(acc).cuda(), T, w.N, w.L, wp_dev, flush_dev,
                                     status)
        fs_ref, _ = O.spec_commit(w.N, w.L, T, idx_h, acc, wp_ora)
        Bd.gdn_replayssm_flush(desc, dev, wp_dev, flush_dev, status)
        Bd.gdn_replayssm_reset_slots(wp_dev, flush_dev, status)
        O.replay_fold(G, ora, wp_ora, fs_ref)
        wp_ora[fs_ref[fs_ref >= 0]] = 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(wp_dev.cpu().numpy(), wp_ora)
    ws = Bd.decode_advance_workspace()
    flushed = torch.empty(rows, dtype=torch.uint8, device="cuda")
    for t in range(2 * w.L):  # every slot crosses a flush
        si = I.step_inputs(gen, w, "cpu")
        out = torch.empty((rows, w.HV, w.V), device="cuda")
        Bd.gdn_replayssm_decode_advance(desc, dev, wp_dev, None,
                                        Bd.Step(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda(), idx_dev, out),
                                        ws, Bd.RECON_TENSOR, flushed, status)
        o_ref, fl_ref, st = O.replay_decode(G, ora, wp_ora, idx_h, None, si.mixed_qkv, si.g, si.beta)
        O.replay_advance(w.N, idx_h, None, w.L, wp_ora)
        torch.cuda.synchronize()
        assert st == 0 and int(status.item()) == 0
        assert np.array_equal(flushed.cpu().numpy(), fl_ref)
        assert np.array_equal(wp_dev.cpu().numpy(), wp_ora)
        e = rel_err(out.cpu().numpy()[live], o_ref[live])
        assert e <= TOL_TC, f"decode step {t}: out rel err {e:.3e}"
    e = rel_err(dev.state.cpu().numpy(), ora.state)
    assert e <= TOL_TC, f"checkpoint rel err {e:.3e}"


def test_spec_bad_rows_report_and_touch_nothing(gdnlib):
    """A window that does not fit (p + T > L - 1) and a slot past the pool give
    zeros and a status bit; a bad acceptance count leaves the cursor; the oracle
    reports the same bits."""
    w, T = I.Workload("spec bad rows", N=6, B=3, HV=4, HK=2, K=128, L=8, ring_dtype=Bd.F32,
                      qkv_dtype=Bd.F32, seed=49), 3
    gen = I.generator(w.seed, "cpu")
    wp = torch.tensor([0, 5, 2, 4, 1, 0], dtype=torch.int32)  # slot 1: 5 + 3 > 7
    c = I.cache(gen, w, wp, "cpu")
    dev = Bd.Cache(c.state.cuda(), c.ring_d.cuda(), c.ring_k.cuda(), c.ring_g.cuda())
    ora = O.Cache.from_arrays(c.state, c.ring_d, c.ring_k, c.ring_g)
    desc, G = desc_of(w), oracle_geom(w)
    for (rows_idx, want), recon in [(c, r) for c in (([1], Bd.DEV_BAD_WRITE_POS), ([9], Bd.DEV_BAD_SLOT))
                                    for r in (TC, FF)]:
        idx = torch.tensor(rows_idx, dtype=torch.int32)
        si = I.step_inputs(gen, w, "cpu", rows=T)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full((T, w.HV, w.V), float("nan"), device="cuda")
        Bd.gdn_replayssm_spec_verify(desc, dev, wp.cuda(), T,
                                     Bd.Step(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda(), idx.cuda(), out),
                                     recon, status)
        o_ref, st = O.spec_verify(G, ora, wp.numpy().copy(), idx.numpy(), T, si.mixed_qkv, si.g, si.beta)
        torch.cuda.synchronize()
        assert int(status.item()) == want == st
        assert torch.all(out == 0.0) and np.all(o_ref == 0.0)
    for name in ("state", "ring_d", "ring_k", "ring_g"):
        assert torch.equal(_bits(getattr(dev, name).cpu()), _bits(getattr(c, name))), f"{name} was modified"
    # commit: accepted above T, below 0, a cursor whose window did not fit, a bad slot, a padding row
    idx = np.array([0, 2, 1, 9, -1, 3], dtype=np.int32)
    acc = np.array([T + 1, -1, 1, 1, 2, 2], dtype=np.int32)
    wp_dev = wp.cuda()
    wp_ora = wp.numpy().copy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fs = torch.empty(idx.shape[0], dtype=torch.int32, device="cuda")
    Bd.gdn_replayssm_spec_commit(torch.from_numpy(idx).cuda(), torch.from_numpy(acc).cuda(), T, w.N, w.L, wp_dev,
                                 fs, status)
    fs_ref, st = O.spec_commit(w.N, w.L, T, idx, acc, wp_ora)
    torch.cuda.synchronize()
    assert int(status.item()) == st == (Bd.DEV_BAD_ACCEPTED | Bd.DEV_BAD_WRITE_POS | Bd.DEV_BAD_SLOT)
    assert np.array_equal(wp_dev.cpu().numpy(), wp_ora)
    assert np.array_equal(fs.cpu().numpy(), fs_ref)
    assert list(wp_ora) == [0, 5, 2, 6, 1, 0], "only slot 3 (row 5, accepted 2) moves"


def test_spec_headline_sizes_sampled(gdnlib):
    """One window of 4 tokens at the benchmark's layer size (HV=32, HK=16,
    K=V=128, L=16, fp16 ring, 256 rows of a 512-slot pool); the oracle
    recomputes a seeded sample of rows from copies of their slots."""
    w, T = I.with_(I.HEADLINE, n_pad=3, seed=50), 4
    gen = I.generator(w.seed, "cuda")
    wp = torch.randint(0, w.L - T, (w.N,), generator=gen, device="cuda", dtype=torch.int32)
    c = I.cache(gen, w, wp, "cuda")
    dev = Bd.Cache(c.state, c.ring_d, c.ring_k, c.ring_g)
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cuda")
    rows = idx.shape[0]
    si = I.step_inputs(gen, w, "cuda", rows=rows * T)
    idx_h, wp_h = idx.cpu().numpy(), wp.cpu().numpy()
    pick = np.random.default_rng(w.seed)
    chosen = np.sort(pick.choice(np.nonzero(idx_h >= 0)[0], size=4, replace=False))
    slots = idx_h[chosen]
    sl = torch.as_tensor(slots, dtype=torch.long, device="cuda")
    mini = O.Cache.from_arrays(dev.state[sl], dev.ring_d[sl], dev.ring_k[sl], dev.ring_g[sl])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((rows * T, w.HV, w.V), float("nan"), dtype=torch.bfloat16, device="cuda")
    Bd.gdn_replayssm_spec_verify(desc_of(w), dev, wp, T, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out), TC,
                                 status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tok = torch.as_tensor((chosen[:, None] * T + np.arange(T)[None, :]).reshape(-1), device="cuda")
    Gm = O.geom(len(slots), w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, state_dtype=O.F32,
                ring_dtype=ORACLE_DT[w.ring_dtype])
    wp_m = wp_h[slots].astype(np.int32)
    o_ref, st = O.spec_verify(Gm, mini, wp_m.copy(), np.arange(len(slots)), T, si.mixed_qkv[tok], si.g[tok],
                              si.beta[tok])
    assert st == 0
    o = out.float().cpu().numpy().reshape(rows, T, w.HV, w.V)
    ref = torch.from_numpy(o_ref).to(torch.bfloat16).double().numpy().reshape(len(slots), T, w.HV, w.V)
    e = rel_err(o[chosen], ref)
    assert e <= TOL_TC, f"sampled out rel err {e:.3e}"
    assert np.all(o[idx_h < 0] == 0.0)
    for i, slot in enumerate(slots):
        p = int(wp_m[i])
        got = dev.ring_d[slot, :, p:p + T].double().cpu().numpy()
        assert rel_err(got, mini.ring_d[i, :, p:p + T]) <= ring_tolerance(w, TOL_TC)
        assert np.array_equal(dev.ring_k[slot, :, p:p + T].double().cpu().numpy(), mini.ring_k[i, :, p:p + T])
        assert np.array_equal(dev.ring_g[slot, :, p:p + T].double().cpu().numpy(), mini.ring_g[i, :, p:p + T])
    assert np.array_equal(wp.cpu().numpy(), wp_h), "verify moved a cursor"
