"""gdn_replayssm_decode_advance_noalloc, the entry point for callers that cannot
allocate device memory (an engine that reserved the whole device for its own
pools, a plugin whose host owns every allocation): its scratch comes from an
array inside the library instead of a caller workspace.

Two calls in a row through the C ABI must give what the workspace entry point
gives on the same inputs and cache: outputs within the tensor-core bound (the
arithmetic is the same kernel, so in practice bit for bit), and identical
cursors and flush flags.  After every call the library's counter must be back
at zero.  Both the one-row-per-thread launch (the cursors advance right after
the rows are dealt) and the launch with more rows than the kernel has threads
(the cursors advance at the end) are covered.  This file is collected last,
and it must pass both alone in a fresh process (the first call sets the
scratch up) and after the other tests."""
import pytest
import torch

from gpu_harness import TOL_TC, desc_of, rel_err
from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu

CASES = {
    # several blocks, padding rows, GQA 2:1, flush and append rows mixed in a launch
    "one_pass": I.Workload("no-alloc", N=24, B=9, n_pad=2, HV=8, HK=4, K=128, L=4, ring_dtype=Bd.F16,
                           qkv_dtype=Bd.BF16, steps=2, staggered=True, seed=31),
    # more rows than threads: the last block to finish advances the cursors
    "rows_beyond_one_pass": I.Workload("no-alloc 600", N=700, B=600, n_pad=3, HV=2, HK=1, K=64, L=4,
                                       ring_dtype=Bd.F16, qkv_dtype=Bd.BF16, steps=2, staggered=True, seed=32),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_the_workspace_entry_point(gdnlib, name):
    W = CASES[name]
    gen = I.generator(W.seed, "cuda")
    wp0 = I.write_pos(gen, W, "cuda")
    c0 = I.cache(gen, W, wp0, "cuda")
    idx = I.indices(gen, W.B, W.N, W.n_pad, "cuda")
    rows = idx.shape[0]
    ref = Bd.Cache(c0.state.clone(), c0.ring_d.clone(), c0.ring_k.clone(), c0.ring_g.clone())
    got = Bd.Cache(c0.state, c0.ring_d, c0.ring_k, c0.ring_g)
    wp_ref, wp_got = wp0.clone(), wp0.clone()
    desc = desc_of(W)
    ws = Bd.decode_advance_workspace()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flushes = 0
    for call in range(2):  # two calls in a row share the library's scratch
        si = I.step_inputs(gen, W, "cuda")
        o_ref = torch.empty((rows, W.HV, W.V), device="cuda")
        o_got = torch.empty((rows, W.HV, W.V), device="cuda")
        fl_ref = torch.empty(rows, dtype=torch.uint8, device="cuda")
        fl_got = torch.empty(rows, dtype=torch.uint8, device="cuda")
        Bd.gdn_replayssm_decode_advance(desc, ref, wp_ref, None, Bd.Step(si.mixed_qkv, si.g, si.beta, idx, o_ref),
                                        ws, Bd.RECON_TENSOR, fl_ref)
        Bd.gdn_replayssm_decode_advance_noalloc(desc, got, wp_got, None,
                                                Bd.Step(si.mixed_qkv, si.g, si.beta, idx, o_got),
                                                Bd.RECON_TENSOR, fl_got, status)
        torch.cuda.synchronize()
        err = rel_err(o_got.cpu().numpy(), o_ref.cpu().numpy())
        assert err <= TOL_TC, f"call {call}: output rel err {err:.3e} > {TOL_TC}"
        assert torch.equal(wp_got, wp_ref), f"call {call}: cursors differ"
        assert torch.equal(fl_got, fl_ref), f"call {call}: flush flags differ"
        assert Bd.gdn_noalloc_scratch_peek(1) == [0], f"call {call}: the scratch counter is not back at zero"
        flushes += int(fl_got.sum().item())
    assert int(status.item()) == 0
    assert flushes > 0, "the two calls should include flushing rows"
    assert rel_err(got.state.cpu().numpy(), ref.state.cpu().numpy()) <= TOL_TC
