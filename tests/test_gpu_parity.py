"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Bounds: max|err| <= tau * max|ref| per launch tensor, tau = 1e-5 for an fp32
ring with the CUDA-core replay, 2e-3 for tensor-core replay or an fp16/bf16
ring.  Integer and index results (cursors, flush flags, padding rows, k/g ring
entries, untouched slots) are compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_harness import (TCP, TOL_TC, Layer, decode, desc_of, guarded, oracle_geom, recon_and_flags, rel_err,
                         run_parity, run_sampled)
from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TC, FF, OUT = Bd.RECON_TENSOR, Bd.RECON_FFMA, Bd.RECON_OUTPUT

# Several CTAs per launch, a ragged batch with padding rows, mixed flush and
# append rows (staggered cursors) and GQA 2:1, at the pages' head size.
RAGGED = I.Workload("ragged", N=16, B=5, n_pad=2, HV=8, HK=4, K=128, L=16, ring_dtype=Bd.F16,
                    qkv_dtype=Bd.BF16, steps=34, staggered=True, seed=11)
KDA_SMALL = I.Workload("kda small", N=8, B=3, n_pad=1, HV=4, HK=4, K=128, L=16, ring_dtype=Bd.F16,
                       qkv_dtype=Bd.BF16, gate=Bd.GATE_PER_K, steps=34, staggered=True, seed=12)


@pytest.fixture(autouse=True)
def _lib(gdnlib):
    yield


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
def test_tiny_fp32(recon):
    rep = run_parity(I.TINY, recon)
    assert sum(s.flushes for s in rep.steps) == 8 * I.TINY.B  # 32 steps, L = 4


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
@pytest.mark.parametrize("ring", [Bd.F16, Bd.BF16, Bd.F32], ids=["f16", "bf16", "f32"])
def test_ragged_staggered(recon, ring):
    rep = run_parity(I.with_(RAGGED, ring_dtype=ring), recon)
    assert sum(s.flushes for s in rep.steps) > 0 and sum(s.appends for s in rep.steps) > 0


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
def test_kda(recon):
    run_parity(KDA_SMALL, recon)


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
@pytest.mark.parametrize("gate,L", [(Bd.GATE_SCALAR, 8), (Bd.GATE_PER_K, 8), (Bd.GATE_PER_K, 24)],
                         ids=["gdn_L8", "kda_L8", "kda_L24"])
def test_head_dim_64(recon, gate, L):
    w = I.Workload("k64", N=6, B=4, HV=4, HK=1 if gate == Bd.GATE_SCALAR else 4, K=64, L=L,
                   ring_dtype=Bd.F16, qkv_dtype=Bd.F16, gate=gate, steps=L + 10, staggered=True, seed=13)
    run_parity(w, recon)


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
@pytest.mark.parametrize("ring", [Bd.F16, Bd.F32], ids=["f16", "f32"])
@pytest.mark.parametrize("gate", [Bd.GATE_SCALAR, Bd.GATE_PER_K], ids=["gdn", "kda"])
def test_longest_ring(recon, ring, gate):
    """L = 64: the replay runs in up to four chunks of 16 ring entries on the
    persistent tensor-core kernel (the first chunk landed by bulk copy, the
    others loaded from the ring directly), each contracted into the same
    accumulator; 70 steps from an empty ring take p through 0 .. 63.  A KDA
    layer with an fp32 ring replays in chunks of 8 entries (its landing slots
    carry the per-channel gates as well), up to eight of them."""
    w = I.Workload("L64", N=3, B=2, HV=2, HK=1 if gate == Bd.GATE_SCALAR else 2, K=128, L=64,
                   ring_dtype=ring, qkv_dtype=Bd.BF16, gate=gate, steps=70, seed=14)
    if recon == TCP:
        assert _kernel_for(w, recon) == Bd.KERNEL_PERSISTENT_TC
    elif recon == TC:
        assert _kernel_for(w, recon) == Bd.KERNEL_SMALL_BATCH
    rep = run_parity(w, recon)
    assert sum(s.flushes for s in rep.steps) == 2


def _kernel_for(w: I.Workload, recon: int, ring_g_offset: int = 0) -> int:
    """The decode kernel the library picks for the workload's shapes (device
    buffers laid out as the parity harness lays them out; ring_g_offset as in
    run_parity)."""
    gen = I.generator(w.seed, "cuda")
    wp = I.write_pos(gen, w, "cuda")
    c = I.cache(gen, w, wp, "cuda")
    keep: list = []
    if ring_g_offset:
        c = I.CacheTensors(c.state, c.ring_d, c.ring_k, guarded(c.ring_g, keep, ring_g_offset))
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cuda")
    si = I.step_inputs(gen, w, "cuda")
    out = torch.empty((idx.shape[0], w.HV, w.V), device="cuda")
    r, f = recon_and_flags(recon)
    return Bd.gdn_replayssm_decode_kernel(desc_of(w), Bd.Cache(c.state, c.ring_d, c.ring_k, c.ring_g),
                                          Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out, flags=f), r)


@pytest.mark.parametrize("ring", [Bd.F16, Bd.BF16, Bd.F32], ids=["f16", "bf16", "f32"])
@pytest.mark.parametrize("L", [24, 34])
def test_chunked_replay_boundaries(ring, L):
    """Staggered cursors put replay depths on both sides of 16 and 32 in one
    launch, on the persistent kernel: L = 24 replays up to 23 entries in one
    contraction (16-bit rings) or in chunks of 16 (fp32 ring); L = 34 chunks
    every ring type (p = 15, 16, 17, 31, 32, 33 all occur)."""
    w = I.Workload(f"L{L}", N=40, B=24, n_pad=2, HV=4, HK=2, K=128, L=L, ring_dtype=ring,
                   qkv_dtype=Bd.BF16, steps=L + 6, staggered=True, seed=15)
    assert _kernel_for(w, TCP) == Bd.KERNEL_PERSISTENT_TC
    rep = run_parity(w, TCP)
    assert sum(s.flushes for s in rep.steps) > 0


@pytest.mark.parametrize("ring", [Bd.F16, Bd.F32], ids=["f16", "f32"])
@pytest.mark.parametrize("L", [10, 24, 34])
def test_chunked_replay_boundaries_kda(ring, L):
    """The same depths with per-channel gates (KDA: the decays fold onto each
    chunk's keys), on the persistent kernel.  An fp32 KDA ring replays in
    chunks of 8 entries (p = 7, 8, 9, 15, 16, 17, ... all occur; L = 10 is the
    shortest ring that chunks); 16-bit rings in chunks of 16 from L = 34."""
    w = I.Workload(f"kda L{L}", N=24, B=12, n_pad=1, HV=4, HK=4, K=128, L=L, ring_dtype=ring,
                   qkv_dtype=Bd.BF16, gate=Bd.GATE_PER_K, steps=L + 4, staggered=True, seed=16)
    assert _kernel_for(w, TCP) == Bd.KERNEL_PERSISTENT_TC
    rep = run_parity(w, TCP)
    assert sum(s.flushes for s in rep.steps) > 0


@pytest.mark.parametrize("ring", [Bd.F16, Bd.F32], ids=["f16", "f32"])
def test_per_head_kernel_on_unaligned_gate_ring(ring):
    """A KDA g ring that starts 4 bytes past a 16-byte boundary (the ABI asks
    only for float alignment there) cannot be bulk-copied, so the one-block-
    per-head tensor-core kernel takes the launch; it must match the oracle
    with the same guard bands, padding rows and flushes."""
    w = I.Workload("kda unaligned g", N=24, B=12, n_pad=1, HV=4, HK=4, K=128, L=24, ring_dtype=ring,
                   qkv_dtype=Bd.BF16, gate=Bd.GATE_PER_K, steps=28, staggered=True, seed=17)
    assert _kernel_for(w, TCP) == Bd.KERNEL_PERSISTENT_TC
    assert _kernel_for(w, TCP, ring_g_offset=4) == Bd.KERNEL_PER_HEAD_TC
    rep = run_parity(w, TCP, ring_g_offset=4)
    assert sum(s.flushes for s in rep.steps) > 0 and sum(s.appends for s in rep.steps) > 0


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
def test_forced_flush_mid_ring(recon):
    sched = lambda t, rows: (np.arange(rows) % 3 == t % 3).astype(np.uint8) if t % 5 == 2 else np.zeros(rows, np.uint8)
    rep = run_parity(I.with_(RAGGED, steps=20), recon, force=sched)
    assert sum(s.flushes for s in rep.steps) > 0


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
def test_three_layer_stack_shared_cursor(recon):
    run_parity(I.with_(RAGGED, steps=18), recon, layers=3)


@pytest.mark.parametrize("recon", [TC, TCP], ids=["small_batch", "persistent"])
def test_two_layers_second_overlaps_previous(recon):
    """Two layers per forward sharing one cursor array, the second launched
    with STEP_OVERLAP_PREVIOUS (its rows, cursors and checkpoints may be read
    before the first layer's launch has finished): parity with the oracle,
    flush flags and status included."""
    rep = run_parity(I.with_(RAGGED, steps=18), recon, layers=2, overlap=True)
    assert sum(s.flushes for s in rep.steps) > 0


def test_two_layers_kda_second_overlaps_previous():
    """The same with per-channel gates (KDA), on the persistent kernel."""
    rep = run_parity(I.with_(KDA_SMALL, steps=18), TCP, layers=2, overlap=True)
    assert sum(s.flushes for s in rep.steps) > 0


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
@pytest.mark.parametrize("l2norm", [False, True], ids=["raw", "l2norm"])
def test_unaligned_qkv_rows(recon, l2norm):
    """mixed_qkv one element into a wider buffer: its rows start off any 16-byte
    boundary and lie an odd number of elements apart, so the persistent kernel
    loads q, k and v per thread instead of by bulk copy (the ABI asks only for
    element alignment there)."""
    rep = run_parity(I.with_(RAGGED, steps=12), recon, qkv_offset=1, qk_l2norm=l2norm, q_scale=0.75)
    assert sum(s.flushes for s in rep.steps) > 0


def test_bf16_output():
    # bf16 rounding of the output alone can be 2^-8 relative: one bf16 ulp on top of the bound
    run_parity(I.with_(RAGGED, steps=10), TC, out_dtype=torch.bfloat16, tol=TOL_TC + 2.0 ** -8)


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
def test_in_kernel_l2norm_and_scale(recon):
    run_parity(I.with_(RAGGED, steps=6), recon, q_scale=0.37, qk_l2norm=True)


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
def test_beta0_g0_leaves_checkpoint_bit_identical(recon):
    """beta = 0 and g = 0 at every step: d = 0 and alpha = 1, so after a full
    ring cycle the flushed checkpoint equals S0 bit for bit."""
    w = I.with_(RAGGED, steps=16, staggered=False)

    def zero_gates(t, si):
        si.g.zero_()
        si.beta.zero_()

    gen = I.generator(w.seed, "cpu")
    wp = I.write_pos(gen, w, "cpu")
    S0 = I.cache(gen, w, wp, "cpu").state
    rep = run_parity(w, recon, tweak=zero_gates, check_untouched=False)
    assert rep.steps[-1].flushes == w.B
    # re-run to get the device state after the last (flush) step
    gen = I.generator(w.seed, "cpu")
    wp = I.write_pos(gen, w, "cpu")
    layer = Layer.make(w, gen, wp)
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu").cuda()
    wpd = wp.cuda()
    for t in range(w.steps):
        si = I.step_inputs(gen, w, "cpu")
        zero_gates(t, si)
        out = torch.empty((idx.shape[0], w.HV, w.V), device="cuda")
        decode(desc_of(w), layer.dev, wpd, None,
                                Bd.Step(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda(), idx, out), recon)
        Bd.gdn_replayssm_advance(idx, None, w.N, w.L, wpd)
    assert torch.equal(layer.dev.state.cpu().view(torch.int32), S0.view(torch.int32))


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
def test_erased_history_closed_form(recon):
    """g = -1e4 makes alpha underflow to 0: out = beta v (k^T q) whatever the history."""
    w = I.with_(RAGGED, steps=1)
    gen = I.generator(w.seed, "cpu")
    wp = I.write_pos(gen, w, "cpu")
    layer = Layer.make(w, gen, wp)
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu")
    si = I.step_inputs(gen, w, "cpu")
    si.g.fill_(-1e4)
    out = torch.empty((idx.shape[0], w.HV, w.V), device="cuda")
    decode(desc_of(w), layer.dev, wp.cuda(), None,
                            Bd.Step(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda(), idx.cuda(), out), recon)
    x = si.mixed_qkv.double()
    R = x.shape[0]
    q = x[:, : w.HK * w.K].reshape(R, w.HK, w.K)
    k = x[:, w.HK * w.K: 2 * w.HK * w.K].reshape(R, w.HK, w.K)
    v = x[:, 2 * w.HK * w.K:].reshape(R, w.HV, w.V)
    kq = (q * k).sum(-1).repeat_interleave(w.HV // w.HK, dim=1)  # [R, HV]
    ref = si.beta.double()[..., None] * v * kq[..., None]
    live = idx >= 0
    assert rel_err(out.cpu()[live].numpy(), ref[live].numpy()) <= 1e-5
    assert torch.all(out.cpu()[~live] == 0)


def test_l1_replay_is_packed_decode_bitwise():
    """L = 1: the CUDA-core replay decode and the packed decode give identical bits."""
    w = I.Workload("L1", N=6, B=4, n_pad=1, HV=8, HK=4, K=128, L=1, ring_dtype=Bd.F32,
                   qkv_dtype=Bd.BF16, steps=5, seed=15)
    gen = I.generator(w.seed, "cpu")
    S0 = I.state(gen, w.N, w.HV, w.V, w.K, "cpu").cuda()
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu").cuda()
    sa, sb = S0.clone(), S0.clone()
    wp = torch.zeros(w.N, dtype=torch.int32, device="cuda")
    flushed = torch.empty(idx.shape[0], dtype=torch.uint8, device="cuda")
    d = desc_of(w)
    for _ in range(w.steps):
        si = I.step_inputs(gen, w, "cuda")
        oa = torch.empty((idx.shape[0], w.HV, w.V), device="cuda")
        ob = torch.empty_like(oa)
        decode(d, Bd.Cache(sa), wp, None, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, oa), FF, flushed)
        Bd.gdn_packed_decode(d, sb, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, ob))
        Bd.gdn_replayssm_advance(idx, None, w.N, 1, wp)
        assert torch.equal(oa, ob) and torch.equal(sa, sb)
        assert torch.equal(flushed.cpu(), (idx.cpu() >= 0).to(torch.uint8))
    assert torch.all(wp == 0)


@pytest.mark.parametrize("recon", [TC, TCP], ids=["default", "persistent"])
def test_l1_tensor_path_matches_packed(recon):
    """L = 1: a tensor-core call runs the CUDA-core replay kernel (the ring is
    empty, so the decode is the packed decode: identical bits) unless the step
    asks for the persistent tensor-core kernel (then within 1e-5)."""
    w = I.Workload("L1", N=6, B=4, HV=8, HK=4, K=128, L=1, ring_dtype=Bd.F16, qkv_dtype=Bd.BF16,
                   steps=4, seed=16)
    assert _kernel_for(w, recon) == (Bd.KERNEL_CUDA_CORE if recon == TC else Bd.KERNEL_PERSISTENT_TC)
    gen = I.generator(w.seed, "cpu")
    S0 = I.state(gen, w.N, w.HV, w.V, w.K, "cpu").cuda()
    idx = I.indices(gen, w.B, w.N, 0, "cpu").cuda()
    sa, sb = S0.clone(), S0.clone()
    wp = torch.zeros(w.N, dtype=torch.int32, device="cuda")
    d = desc_of(w)
    for _ in range(w.steps):
        si = I.step_inputs(gen, w, "cuda")
        oa = torch.empty((w.B, w.HV, w.V), device="cuda")
        ob = torch.empty_like(oa)
        decode(d, Bd.Cache(sa), wp, None, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, oa), recon)
        Bd.gdn_packed_decode(d, sb, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, ob))
        if recon == TC:
            assert torch.equal(oa, ob) and torch.equal(sa, sb)
        assert rel_err(oa.cpu().numpy(), ob.cpu().numpy()) <= 1e-5
        assert rel_err(sa.cpu().numpy(), sb.cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("gate", [Bd.GATE_SCALAR, Bd.GATE_PER_K], ids=["gdn", "kda"])
def test_packed_decode_vs_oracle(gate):
    w = I.Workload("packed", N=10, B=6, n_pad=2, HV=4, HK=2 if gate == Bd.GATE_SCALAR else 4, K=128, L=1,
                   ring_dtype=Bd.F32, qkv_dtype=Bd.F32, gate=gate, steps=6, seed=17)
    gen = I.generator(w.seed, "cpu")
    S0 = I.state(gen, w.N, w.HV, w.V, w.K, "cpu")
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu")
    dev = S0.cuda()
    ora = O.f64(S0).copy()
    G = O.geom(w.N, w.HV, w.HK, w.K, w.V, 1, gate=gate, state_dtype=O.F32)
    for _ in range(w.steps):
        si = I.step_inputs(gen, w, "cpu")
        out = torch.empty((idx.shape[0], w.HV, w.V), device="cuda")
        Bd.gdn_packed_decode(desc_of(w), dev, Bd.Step(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda(), idx.cuda(), out))
        o_ref, st = O.packed_decode(G, ora, idx.numpy(), si.mixed_qkv, si.g, si.beta)
        assert st == 0
        live = idx.numpy() >= 0
        assert rel_err(out.cpu().numpy()[live], o_ref[live]) <= 1e-5
        assert np.all(out.cpu().numpy()[~live] == 0)
        assert rel_err(dev.cpu().numpy(), ora) <= 1e-5


@pytest.mark.parametrize("recon", [FF, TC, TCP, OUT], ids=["ffma", "tensor", "tensor_persistent", "output"])
def test_bad_rows_set_status_and_touch_nothing(recon):
    w = I.with_(RAGGED, steps=1)
    gen = I.generator(w.seed, "cpu")
    wp = I.write_pos(gen, w, "cpu")
    layer = Layer.make(w, gen, wp)
    wp[3] = w.L + 2                                         # cursor out of range
    idx = torch.tensor([-1, w.N + 5, 3, 1], dtype=torch.int32)  # padding, bad slot, bad cursor, good
    si = I.step_inputs(gen, w, "cpu", rows=4)
    out = torch.full((4, w.HV, w.V), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flushed = torch.full((4,), 7, dtype=torch.uint8, device="cuda")
    before = layer.dev.state.clone()
    decode(desc_of(w), layer.dev, wp.cuda(), None,
                            Bd.Step(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda(), idx.cuda(), out),
                            recon, flushed, status)
    torch.cuda.synchronize()
    assert int(status.item()) == (Bd.DEV_BAD_SLOT | Bd.DEV_BAD_WRITE_POS)
    o = out.cpu()
    assert torch.all(o[:3] == 0) and torch.all(torch.isfinite(o[3]))
    assert flushed.cpu()[:3].tolist() == [0, 0, 0]
    assert torch.equal(layer.dev.state[3], before[3])
    status.zero_()
    wpd = wp.cuda()
    Bd.gdn_replayssm_advance(idx.cuda(), None, w.N, w.L, wpd, status)
    torch.cuda.synchronize()
    assert int(status.item()) == (Bd.DEV_BAD_SLOT | Bd.DEV_BAD_WRITE_POS)
    assert int(wpd[3].item()) == w.L + 2


def test_empty_and_all_padding_batches():
    w = I.with_(RAGGED, steps=1)
    gen = I.generator(w.seed, "cpu")
    wp = I.write_pos(gen, w, "cpu")
    layer = Layer.make(w, gen, wp)
    before = [t.clone() for t in (layer.dev.state, layer.dev.ring_d, layer.dev.ring_k, layer.dev.ring_g)]
    for rows in (0, 3):
        idx = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        si = I.step_inputs(gen, w, "cuda", rows=rows)
        out = torch.full((rows, w.HV, w.V), float("nan"), device="cuda")
        for recon in (FF, TC, TCP, OUT):
            decode(desc_of(w), layer.dev, wp.cuda(), None,
                                    Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out), recon)
        Bd.gdn_packed_decode(desc_of(w), layer.dev.state, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out))
        torch.cuda.synchronize()
        assert torch.all(out == 0)
    after = (layer.dev.state, layer.dev.ring_d, layer.dev.ring_k, layer.dev.ring_g)
    for a, b in zip(after, before):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("gate", [Bd.GATE_SCALAR, Bd.GATE_PER_K], ids=["gdn", "kda"])
def test_fold_then_reset(gate):
    """gdn_replayssm_flush folds the ring into the checkpoint (oracle replay_fold);
    gdn_replayssm_reset_slots zeroes the cursors; decoding then continues."""
    w = I.with_(KDA_SMALL if gate == Bd.GATE_PER_K else RAGGED, steps=1)
    w = I.with_(w, ring_dtype=Bd.F32)
    gen = I.generator(w.seed, "cpu")
    wp = I.write_pos(gen, w, "cpu")
    layer = Layer.make(w, gen, wp)
    slots = torch.tensor([1, -1, 4, 2], dtype=torch.int32)
    wpd = wp.cuda()
    Bd.gdn_replayssm_flush(desc_of(w), layer.dev, wpd, slots.cuda())
    O.replay_fold(oracle_geom(w), layer.ora, wp.numpy(), slots.numpy())
    assert rel_err(layer.dev.state.cpu().numpy(), layer.ora.state) <= 1e-5
    Bd.gdn_replayssm_reset_slots(wpd, slots.cuda())
    expect = wp.clone()
    expect[[1, 4, 2]] = 0
    assert torch.equal(wpd.cpu(), expect)


def test_host_side_rejects_bad_arguments():
    w = I.with_(RAGGED, steps=1)
    gen = I.generator(w.seed, "cpu")
    wp = I.write_pos(gen, w, "cpu")
    layer = Layer.make(w, gen, wp)
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu").cuda()
    si = I.step_inputs(gen, w, "cuda")
    out = torch.empty((idx.shape[0], w.HV, w.V), device="cuda")
    step = Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out)
    bad = [desc_of(I.with_(w, K=96)), Bd.layer_desc(w.N, 6, 4, 128, 128, 16),
           Bd.layer_desc(w.N, w.HV, w.HK, 128, 128, 65)]
    for d in bad:
        with pytest.raises(Bd.GdnError):
            decode(d, layer.dev, wp.cuda(), None, step, TC)
    with pytest.raises(Bd.GdnError):
        decode(desc_of(w), layer.dev, wp.cuda(), None, step, 7)


@pytest.mark.parametrize("w", [I.QWEN3NEXT_LAYER, I.HEADLINE, I.KDA_LAYER],
                         ids=["qwen3next_layer", "headline_B256_L16", "kda_layer"])
def test_full_size_sampled(w):
    """The launch configuration the benchmark times, checked on sampled rows."""
    run_sampled(w, TC, steps=3)


def test_full_size_sampled_long_fp32_ring():
    """B = 256, L = 32 with an fp32 ring (tf32 operands), the launch the sweep
    times: two replay chunks per long item, on the persistent kernel."""
    w = I.sweep_point(256, 32, Bd.F32)
    assert _kernel_for(w, TC) == Bd.KERNEL_PERSISTENT_TC
    run_sampled(w, TC, steps=3)


def test_full_size_sampled_kda_long_fp32_ring():
    """The KDA layer (B = 128, HV = HK = 32, K = V = 128) with an fp32 ring at
    L = 64, the launch `bench.py --workload kda_layer:64:f32` times: up to eight
    8-entry replay chunks per item on the persistent kernel; sampled rows."""
    import bench
    w = bench.pick_workload("kda_layer:64:f32")
    assert _kernel_for(w, TC) == Bd.KERNEL_PERSISTENT_TC
    run_sampled(w, TC, steps=3)


@pytest.mark.parametrize("B,ring,kernel", [(1, Bd.F16, Bd.KERNEL_SMALL_BATCH), (2, Bd.F32, Bd.KERNEL_SMALL_BATCH),
                                           (8, Bd.F16, Bd.KERNEL_PERSISTENT_TC)],
                         ids=["B1_f16", "B2_f32", "B8_f16"])
def test_full_size_sampled_small_batches(B, ring, kernel):
    """The pages' head shapes (HV=32, HK=16, K=V=128, L=16) at batch 1, 2 and
    8, staggered cursors: B <= 2 runs the small-batch kernel, B = 8 the
    persistent one; sampled rows against the oracle."""
    w = I.sweep_point(B, 16, ring)
    assert _kernel_for(w, TC) == kernel
    run_sampled(w, TC, steps=4)


@pytest.mark.parametrize("B,L,ring", [(4, 8, Bd.F16), (8, 4, Bd.F32), (8, 8, Bd.F16)],
                         ids=["B4_L8_f16", "B8_L4_f32", "B8_L8_f16"])
def test_full_size_sampled_small_batch_wide_slices(B, L, ring):
    """GDN batches of 128 and 256 (row, head) items with short rings run the
    small-batch kernel with slices of 32 and 64 state rows; sampled rows
    against the oracle over two ring cycles."""
    w = I.sweep_point(B, L, ring)
    assert _kernel_for(w, TC) == Bd.KERNEL_SMALL_BATCH
    run_sampled(w, TC, steps=2 * L)


@pytest.mark.parametrize("B,L", [(3, 4), (7, 8)], ids=["128_items_L4", "256_items_L8"])
def test_small_batch_wide_slices_every_row(B, L):
    """The same kernel with 32- and 64-row slices (one padding row besides the
    B live ones: 128 and 256 items) checked on every row, padding rows and
    flushes included (32 value heads, a small slot pool)."""
    w = I.Workload(f"wide slices B{B}", N=2 * B + 4, B=B, n_pad=1, HV=32, HK=16, K=128, L=L,
                   ring_dtype=Bd.F16, qkv_dtype=Bd.BF16, steps=2 * L + 2, staggered=True, seed=18)
    assert _kernel_for(w, TC) == Bd.KERNEL_SMALL_BATCH
    rep = run_parity(w, TC)
    assert sum(s.flushes for s in rep.steps) > 0 and sum(s.appends for s in rep.steps) > 0


def test_full_size_sampled_output_only():
    """The output-only readout at the benchmark's layer size, sampled rows."""
    run_sampled(I.HEADLINE, OUT, steps=3)


@pytest.mark.parametrize("ring", [Bd.F16, Bd.F32], ids=["f16_ring", "f32_ring"])
def test_drift_after_four_rings(ring):
    """4L steps (four full rings, four flushes per slot) of the tensor-core
    path.  Parity with the oracle that rounds what it stores as the cache does
    holds at every step (run_parity).  The drift is the distance of the GPU
    outputs to the unrounded recurrence (the oracle with double storage), per
    ring of L steps: it must stay within 4 x 2^-11 of max|ref| (fp16 storage
    and f16 / tf32 operands carry 2^-11 relative per stored or multiplied
    value; d k products and the decayed sums add a few of those) and must not
    grow from the first ring to the last by more than the bound of one ring."""
    import json
    import os

    w = I.with_(RAGGED, staggered=False, steps=64, n_pad=0, ring_dtype=ring)
    outs: list = []
    rep = run_parity(w, TCP, outputs=outs)  # the tensor-core arithmetic
    # the same seeded draws as run_parity: cursors, cache, rows, then each step's inputs
    gen = I.generator(w.seed, "cpu")
    wp = I.write_pos(gen, w, "cpu")
    c = I.cache(gen, w, wp, "cpu")
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu").numpy()
    Gp = O.geom(w.N, w.HV, w.HK, w.K, w.V, w.L, state_dtype=O.F64, ring_dtype=O.F64)
    pure = O.Cache.from_arrays(c.state, c.ring_d, c.ring_k, c.ring_g)
    wpp = wp.numpy().copy()
    per_ring = [0.0] * (w.steps // w.L)
    for t in range(w.steps):
        si = I.step_inputs(gen, w, "cpu")
        op, _, _ = O.replay_decode(Gp, pure, wpp, idx, None, si.mixed_qkv, si.g, si.beta)
        O.replay_advance(w.N, idx, None, w.L, wpp)
        per_ring[t // w.L] = max(per_ring[t // w.L], rel_err(outs[t], op))
    bound = 4 * 2.0 ** -11
    record = {"ring": {Bd.F16: "f16", Bd.F32: "f32"}[ring], "L": w.L, "steps": w.steps,
              "gpu_vs_oracle_with_storage_rounding": {"out": rep.max_o, "checkpoint": rep.max_state},
              "gpu_vs_unrounded_recurrence_per_ring": per_ring, "bound": bound}
    print("\n[drift 4L] " + json.dumps(record))
    rec_dir = os.environ.get("GDN_TEST_RECORD_DIR")
    if rec_dir:
        os.makedirs(rec_dir, exist_ok=True)
        with open(os.path.join(rec_dir, f"drift_after_four_rings_{record['ring']}.json"), "w") as f:
            json.dump(record, f)
    assert rep.max_o <= TOL_TC
    assert max(per_ring) <= bound, f"drift {per_ring} above {bound:.2e}"
    assert per_ring[-1] <= per_ring[0] + bound / 4, f"drift grows across rings: {per_ring}"
