"""The library allocates nothing and never synchronises, so its calls can be
captured in a CUDA graph: a few fused decode + advance steps captured once and
replayed give, bit for bit, what the same launches give run one by one."""
import pytest
import torch

from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int32) if t.element_size() == 4 else t.contiguous().view(torch.int16)


@pytest.mark.parametrize("recon", [Bd.RECON_TENSOR, Bd.RECON_FFMA], ids=["tensor", "ffma"])
def test_captured_steps_match_eager_steps(gdnlib, recon):
    w = I.Workload("graph", N=16, B=5, n_pad=1, HV=8, HK=4, K=128, L=8, ring_dtype=Bd.F16, qkv_dtype=Bd.BF16,
                   staggered=True, seed=95)
    gen = I.generator(w.seed, "cuda")
    wp0 = I.write_pos(gen, w, "cuda")
    c0 = I.cache(gen, w, wp0, "cuda")
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cuda")
    rows = idx.shape[0]
    steps = [I.step_inputs(gen, w, "cuda") for _ in range(3)]
    desc = Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, w.L, ring_dtype=w.ring_dtype)

    def setup():
        cache = Bd.Cache(c0.state.clone(), c0.ring_d.clone(), c0.ring_k.clone(), c0.ring_g.clone())
        outs = [torch.empty((rows, w.HV, w.V), dtype=torch.bfloat16, device="cuda") for _ in steps]
        return cache, wp0.clone(), outs, Bd.decode_advance_workspace()

    def run(cache, wp, outs, ws, stream=None):
        for si, out in zip(steps, outs):
            Bd.gdn_replayssm_decode_advance(desc, cache, wp, None, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out),
                                            ws, recon, None, None, stream)

    # eager: the three steps twice
    e_cache, e_wp, e_outs, e_ws = setup()
    run(e_cache, e_wp, e_outs, e_ws)
    run(e_cache, e_wp, e_outs, e_ws)
    torch.cuda.synchronize()

    # graph: the three steps captured once (after one eager pass on scratch
    # buffers so every lazily set-up host state exists), replayed twice
    g_cache, g_wp, g_outs, g_ws = setup()
    s_cache, s_wp, s_outs, s_ws = setup()
    run(s_cache, s_wp, s_outs, s_ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    with torch.cuda.stream(cs):
        with torch.cuda.graph(graph, stream=cs):
            run(g_cache, g_wp, g_outs, g_ws, torch.cuda.current_stream())
    # capture records, it does not run: the buffers are still the initial ones
    torch.cuda.synchronize()
    assert torch.equal(g_wp, wp0)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()

    assert torch.equal(g_wp, e_wp), "cursors differ"
    assert int(g_ws.item()) == 0
    for a, b in zip(g_outs, e_outs):
        assert torch.equal(_bits(a), _bits(b)), "outputs differ"
    for name in ("state", "ring_d", "ring_k", "ring_g"):
        assert torch.equal(_bits(getattr(g_cache, name)), _bits(getattr(e_cache, name))), f"{name} differs"
