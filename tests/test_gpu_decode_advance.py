"""gdn_replayssm_decode_advance against gdn_replayssm_decode followed by
gdn_replayssm_advance, on identical inputs and caches.

The decode arithmetic is the same kernel in both, so outputs, checkpoints,
rings, flush flags and cursors must agree bit for bit after every step; only
where the cursors are advanced differs (in the decode launch, by the last block
to finish, or in a second launch).  The workspace must be back at zero after
every call."""
import numpy as np
import pytest
import torch

from gpu_harness import desc_of
from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TC, FF = Bd.RECON_TENSOR, Bd.RECON_FFMA

CASES = {
    # several blocks, padding rows, GQA 2:1, flush and append rows mixed
    "ragged": (I.Workload("ragged", N=16, B=5, n_pad=2, HV=8, HK=4, K=128, L=16, ring_dtype=Bd.F16,
                          qkv_dtype=Bd.BF16, steps=20, staggered=True, seed=21), TC, False),
    # the benchmark's launch configuration (one block per SM, persistent)
    "headline": (I.with_(I.HEADLINE, steps=3), TC, False),
    # more rows than the kernel has threads: the cursors are read again at the end
    "rows_beyond_one_pass": (I.Workload("600 rows", N=700, B=600, n_pad=3, HV=2, HK=1, K=64, L=4,
                                        ring_dtype=Bd.F16, qkv_dtype=Bd.BF16, steps=6, staggered=True,
                                        seed=22), TC, False),
    "kda": (I.Workload("kda", N=8, B=3, n_pad=1, HV=4, HK=4, K=128, L=16, ring_dtype=Bd.F16,
                       qkv_dtype=Bd.BF16, gate=Bd.GATE_PER_K, steps=18, staggered=True, seed=23), TC, False),
    "forced_flushes": (I.Workload("forced", N=16, B=6, n_pad=1, HV=8, HK=4, K=128, L=8, ring_dtype=Bd.F16,
                                  qkv_dtype=Bd.BF16, steps=12, staggered=True, seed=24), TC, True),
    # CUDA-core replay: decode and advance are two launches inside the call
    "ffma": (I.Workload("ffma", N=16, B=5, n_pad=2, HV=8, HK=4, K=128, L=16, ring_dtype=Bd.F32,
                        qkv_dtype=Bd.BF16, steps=18, staggered=True, seed=25), FF, False),
    # output-only readout: also two launches
    "output_only": (I.Workload("output", N=16, B=5, n_pad=2, HV=8, HK=4, K=128, L=16, ring_dtype=Bd.F16,
                               qkv_dtype=Bd.BF16, steps=18, staggered=True, seed=28), Bd.RECON_OUTPUT, True),
    "ring_len_1": (I.Workload("L=1", N=16, B=5, n_pad=2, HV=8, HK=4, K=128, L=1, ring_dtype=Bd.F16,
                              qkv_dtype=Bd.BF16, steps=3, seed=26), TC, False),
}


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    if a.element_size() == 2:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)


@pytest.mark.parametrize("persistent", [False, True], ids=["default", "persistent"])
@pytest.mark.parametrize("name", list(CASES))
def test_decode_advance_matches_decode_then_advance(gdnlib, name, persistent):
    """Small batches run the small-batch kernel by default; `persistent` forces
    the tensor-core recon onto the persistent kernel (STEP_PERSISTENT_KERNEL),
    whose fused advance counts its blocks differently."""
    w, recon, forced = CASES[name]
    flags = Bd.STEP_PERSISTENT_KERNEL if persistent else 0
    gen = I.generator(w.seed, "cuda")
    wp0 = I.write_pos(gen, w, "cuda")
    c0 = I.cache(gen, w, wp0, "cuda")
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cuda")
    rows = idx.shape[0]
    two = Bd.Cache(c0.state.clone(), c0.ring_d.clone(), c0.ring_k.clone(), c0.ring_g.clone())
    one = Bd.Cache(c0.state, c0.ring_d, c0.ring_k, c0.ring_g)
    wp_two, wp_one = wp0.clone(), wp0.clone()
    desc = desc_of(w)
    ws = Bd.decode_advance_workspace()
    st_two = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_one = torch.zeros(1, dtype=torch.int32, device="cuda")
    fl_two = torch.empty(rows, dtype=torch.uint8, device="cuda")
    fl_one = torch.empty(rows, dtype=torch.uint8, device="cuda")
    for t in range(w.steps):
        si = I.step_inputs(gen, w, "cuda")
        ff = (torch.rand(rows, generator=gen, device="cuda") < 0.3).to(torch.uint8) if forced else None
        out_two = torch.full((rows, w.HV, w.V), float("nan"), device="cuda")
        out_one = torch.full((rows, w.HV, w.V), float("nan"), device="cuda")
        Bd.gdn_replayssm_decode(desc, two, wp_two, ff,
                                Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out_two, flags=flags), recon, fl_two, st_two)
        Bd.gdn_replayssm_advance(idx, ff, w.N, w.L, wp_two, st_two)
        Bd.gdn_replayssm_decode_advance(desc, one, wp_one, ff,
                                        Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out_one, flags=flags),
                                        ws, recon, fl_one, st_one)
        torch.cuda.synchronize()
        assert _same_bits(out_one, out_two), f"step {t}: outputs differ"
        assert torch.equal(fl_one, fl_two), f"step {t}: flush flags differ"
        assert torch.equal(wp_one, wp_two), f"step {t}: cursors differ"
        assert int(ws.item()) == 0, f"step {t}: workspace not left at zero"
    assert int(st_one.item()) == 0 and int(st_two.item()) == 0
    for a, b, what in ((one.state, two.state, "checkpoint"), (one.ring_d, two.ring_d, "d ring"),
                       (one.ring_k, two.ring_k, "k ring"), (one.ring_g, two.ring_g, "g ring")):
        assert _same_bits(a, b), f"{what} differs"


def test_decode_advance_stack_shares_one_cursor_array(gdnlib):
    """Three layers per forward sharing one cursor array: decode on the first
    two, decode + advance on the last, against three decodes and an advance."""
    w = I.Workload("stack", N=16, B=6, n_pad=1, HV=8, HK=4, K=128, L=8, ring_dtype=Bd.F16,
                   qkv_dtype=Bd.BF16, steps=10, staggered=True, seed=27)
    gen = I.generator(w.seed, "cuda")
    wp0 = I.write_pos(gen, w, "cuda")
    caches = [I.cache(gen, w, wp0, "cuda") for _ in range(3)]
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cuda")
    rows = idx.shape[0]
    ref = [Bd.Cache(c.state.clone(), c.ring_d.clone(), c.ring_k.clone(), c.ring_g.clone()) for c in caches]
    got = [Bd.Cache(c.state, c.ring_d, c.ring_k, c.ring_g) for c in caches]
    wp_ref, wp_got = wp0.clone(), wp0.clone()
    desc = desc_of(w)
    ws = Bd.decode_advance_workspace()
    for t in range(w.steps):
        for layer in range(3):
            si = I.step_inputs(gen, w, "cuda")
            o_ref = torch.empty((rows, w.HV, w.V), device="cuda")
            o_got = torch.empty((rows, w.HV, w.V), device="cuda")
            Bd.gdn_replayssm_decode(desc, ref[layer], wp_ref, None, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, o_ref))
            step = Bd.Step(si.mixed_qkv, si.g, si.beta, idx, o_got)
            if layer < 2:
                Bd.gdn_replayssm_decode(desc, got[layer], wp_got, None, step)
            else:
                Bd.gdn_replayssm_decode_advance(desc, got[layer], wp_got, None, step, ws)
            torch.cuda.synchronize()
            assert _same_bits(o_got, o_ref), f"step {t} layer {layer}: outputs differ"
        Bd.gdn_replayssm_advance(idx, None, w.N, w.L, wp_ref)
        torch.cuda.synchronize()
        assert torch.equal(wp_got, wp_ref), f"step {t}: cursors differ"
    assert int(ws.item()) == 0


OVERLAP_CASES = {
    # few items: the small-batch kernel (one block per 16 state rows)
    "small_batch": I.Workload("overlap small", N=24, B=6, n_pad=2, HV=8, HK=4, K=128, L=8, ring_dtype=Bd.F16,
                              qkv_dtype=Bd.BF16, steps=10, staggered=True, seed=43),
    # more items than SMs, so consecutive launches really share the GPU
    "persistent": I.Workload("overlap", N=96, B=48, n_pad=3, HV=8, HK=4, K=128, L=8, ring_dtype=Bd.F16,
                             qkv_dtype=Bd.BF16, steps=10, staggered=True, seed=41),
    # more rows than threads: block 0 reads the rows again for their flush flags
    "rows_beyond_one_pass": I.Workload("overlap 600", N=700, B=600, n_pad=3, HV=2, HK=1, K=64, L=4,
                                       ring_dtype=Bd.F16, qkv_dtype=Bd.BF16, steps=6, staggered=True, seed=42),
}


@pytest.mark.parametrize("name", list(OVERLAP_CASES))
def test_overlap_flag_back_to_back_is_bitwise_the_same(gdnlib, name):
    """Three layers per forward launched back to back with no host sync, the
    last also advancing the cursors: with STEP_OVERLAP_PREVIOUS on the second
    and third layer (their launches may start, read rows and cursors and stream
    checkpoints while the previous layer's launch is still running) every
    output, flush flag, cache and cursor equals the run without the flag bit
    for bit, and the workspace ends at zero."""
    w = OVERLAP_CASES[name]
    layers = 3
    gen = I.generator(w.seed, "cuda")
    wp0 = I.write_pos(gen, w, "cuda")
    c0 = [I.cache(gen, w, wp0, "cuda") for _ in range(layers)]
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cuda")
    rows = idx.shape[0]
    inputs = [[I.step_inputs(gen, w, "cuda") for _ in range(layers)] for _ in range(w.steps)]
    desc = desc_of(w)

    def run(flagged: bool):
        caches = [Bd.Cache(c.state.clone(), c.ring_d.clone(), c.ring_k.clone(), c.ring_g.clone()) for c in c0]
        wp = wp0.clone()
        ws = Bd.decode_advance_workspace()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs = torch.full((w.steps, layers, rows, w.HV, w.V), float("nan"), device="cuda")
        fls = torch.full((w.steps, layers, rows), 7, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        for t in range(w.steps):
            for layer in range(layers):
                si = inputs[t][layer]
                flags = Bd.STEP_OVERLAP_PREVIOUS if (flagged and layer > 0) else 0
                step = Bd.Step(si.mixed_qkv, si.g, si.beta, idx, outs[t, layer], flags=flags)
                if layer < layers - 1:
                    Bd.gdn_replayssm_decode(desc, caches[layer], wp, None, step, TC, fls[t, layer], st)
                else:
                    Bd.gdn_replayssm_decode_advance(desc, caches[layer], wp, None, step, ws, TC, fls[t, layer], st)
        torch.cuda.synchronize()
        return caches, wp, outs, fls, int(ws.item()), int(st.item())

    ref = run(False)
    got = run(True)
    assert ref[4] == 0 and got[4] == 0, "workspace not left at zero"
    assert ref[5] == 0 and got[5] == 0, "status"
    assert torch.equal(got[1], ref[1]), "cursors differ"
    assert torch.equal(got[3], ref[3]), "flush flags differ"
    assert int((ref[3] == 1).sum()) > 0, "the run should include flushing rows"
    assert _same_bits(got[2], ref[2]), "outputs differ"
    for layer in range(layers):
        for name_ in ("state", "ring_d", "ring_k", "ring_g"):
            assert _same_bits(getattr(got[0][layer], name_), getattr(ref[0][layer], name_)), \
                f"layer {layer} {name_} differs"
