"""Prepared calls (arguments checked and packed once, then one foreign call per
launch) launch exactly what the direct calls launch: a few steps of a two-layer
stack (decode, then decode + advance) and of the packed decode, run both ways
from the same starting buffers, agree bit for bit in every output, cache tensor
and cursor."""
import pytest
import torch

from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int32) if t.element_size() == 4 else t.contiguous().view(torch.int16)


@pytest.mark.parametrize("B", [1, 6], ids=["small_batch", "persistent"])
def test_prepared_calls_match_direct_calls(gdnlib, B):
    w = I.Workload("prep", N=16, B=B, n_pad=1, HV=8, HK=4, K=128, L=8, ring_dtype=Bd.F16, qkv_dtype=Bd.BF16,
                   staggered=True, seed=96)
    gen = I.generator(w.seed, "cuda")
    wp0 = I.write_pos(gen, w, "cuda")
    c0 = [I.cache(gen, w, wp0, "cuda") for _ in range(2)]
    p0 = I.state(gen, w.N, w.HV, w.V, w.K, "cuda")
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cuda")
    rows = idx.shape[0]
    ins = I.step_inputs(gen, w, "cuda")
    desc = Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, w.L, ring_dtype=w.ring_dtype)

    def setup():
        caches = [Bd.Cache(c.state.clone(), c.ring_d.clone(), c.ring_k.clone(), c.ring_g.clone()) for c in c0]
        outs = [torch.empty((rows, w.HV, w.V), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        return caches, wp0.clone(), outs, Bd.decode_advance_workspace(), p0.clone()

    def steps(outs):
        first = Bd.Step(ins.mixed_qkv, ins.g, ins.beta, idx, outs[0])
        second = Bd.Step(ins.mixed_qkv, ins.g, ins.beta, idx, outs[1], flags=Bd.STEP_OVERLAP_PREVIOUS)
        packed = Bd.Step(ins.mixed_qkv, ins.g, ins.beta, idx, outs[2])
        return first, second, packed

    # direct calls, three steps
    d_caches, d_wp, d_outs, d_ws, d_pst = setup()
    first, second, packed = steps(d_outs)
    for _ in range(3):
        Bd.gdn_replayssm_decode(desc, d_caches[0], d_wp, None, first)
        Bd.gdn_replayssm_decode_advance(desc, d_caches[1], d_wp, None, second, d_ws)
        Bd.gdn_packed_decode(desc, d_pst, packed)
    torch.cuda.synchronize()

    # the same through prepared calls
    p_caches, p_wp, p_outs, p_ws, p_pst = setup()
    first, second, packed = steps(p_outs)
    calls = [Bd.prepare_replayssm_decode(desc, p_caches[0], p_wp, None, first),
             Bd.prepare_replayssm_decode(desc, p_caches[1], p_wp, None, second, workspace=p_ws),
             Bd.prepare_packed_decode(desc, p_pst, packed)]
    for _ in range(3):
        for call in calls:
            call.run()
    torch.cuda.synchronize()

    assert torch.equal(p_wp, d_wp), "cursors differ"
    assert int(p_ws.item()) == 0
    for a, b in zip(p_outs, d_outs):
        assert torch.equal(_bits(a), _bits(b)), "outputs differ"
    for pc, dc in zip(p_caches, d_caches):
        for name in ("state", "ring_d", "ring_k", "ring_g"):
            assert torch.equal(_bits(getattr(pc, name)), _bits(getattr(dc, name))), f"{name} differs"
    assert torch.equal(_bits(p_pst), _bits(d_pst)), "packed state differs"


def test_prepared_call_reports_errors(gdnlib):
    """A prepared call raises on a non-OK status like the direct call does."""
    desc = Bd.layer_desc(4, 4, 2, 64, 64, 4)
    bad = Bd.layer_desc(4, 4, 2, 64, 64, 0)  # ring_len 0: the library rejects it at every call
    gen = I.generator(1, "cuda")
    st = I.state(gen, 4, 4, 64, 64, "cuda")
    w = I.Workload("e", N=4, B=2, n_pad=0, HV=4, HK=2, K=64, L=4, ring_dtype=Bd.F32, qkv_dtype=Bd.F32, seed=1)
    si = I.step_inputs(gen, w, "cuda")
    idx = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    out = torch.empty((2, 4, 64), dtype=torch.float32, device="cuda")
    Bd.prepare_packed_decode(desc, st, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out)).run()
    call = Bd.prepare_packed_decode(bad, st, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out))
    with pytest.raises(Bd.GdnError):
        call.run()
