"""Lossless verify and its exact-order commit (sglang #42388: The idea;
Modifications, Verify kernel and Commit) on the GPU.

The defining property is bit-identity with the sequential kernel: the verify's
outputs equal, bit for bit, those of T successive gdn_packed_decode calls on the
same inputs, and committing a accepted tuples leaves exactly the state a
successive packed decodes leave.  Both are checked on the GPU against
gdn_packed_decode (torch.equal on the raw bits).  Against the CPU oracle:
outputs and u tuples within 1e-5 (fp32 arithmetic, independent rounding), k and
g tuples bit-exact (copies of the inputs), and the commit of the oracle's own
tuples bit-exact wherever exp(g) is exact on both sides (g = 0, g = -1e4),
within 1e-6 otherwise (the two sides' expf may differ in the last place)."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_harness import check_guards, guarded
from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _bits(x: torch.Tensor) -> torch.Tensor:
    return x.contiguous().view(torch.int32) if x.dtype == torch.float32 else x.contiguous().view(torch.int16)


def _same_bits(a, b) -> bool:
    return torch.equal(_bits(a), _bits(b))


def _rel(a, b) -> float:
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30)) if a.size else 0.0


def _desc(w):
    return Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, 1, gate=w.gate)


def _setup(w, T, seed):
    gen = I.generator(seed, "cpu")
    S0 = I.state(gen, w.N, w.HV, w.V, w.K, "cpu")
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu")
    R = idx.shape[0]
    si = I.step_inputs(gen, w, "cpu", rows=R * T)
    return gen, S0, idx, si


def _token_rows(R, T, t):
    return torch.arange(R) * T + t


def _packed_sequence(w, S0_dev, idx_dev, si_dev, T, out_dtype, accepted=None, q_scale=1.0, l2=False):
    """T successive packed decodes on a copy of the state; returns per-token
    outputs [R*T, HV, V] and the states after each prefix length (if accepted
    is given: the state where row b stopped after accepted[b] tokens)."""
    R = idx_dev.shape[0]
    st = S0_dev.clone()
    outs = torch.empty((R * T, w.HV, w.V), dtype=out_dtype, device="cuda")
    d = _desc(w)
    for t in range(T):
        rows = _token_rows(R, T, t).cuda()
        idx_t = idx_dev.clone()
        if accepted is not None:
            idx_t[accepted.cuda() <= t] = -1  # this row has stopped: its state stays
        o = torch.empty((R, w.HV, w.V), dtype=out_dtype, device="cuda")
        Bd.gdn_packed_decode(d, st, Bd.Step(si_dev.mixed_qkv[rows].contiguous(), si_dev.g[rows].contiguous(),
                                            si_dev.beta[rows].contiguous(), idx_t, o, q_scale, l2))
        outs[rows] = o
    return outs, st


def _dev_inputs(si):
    return I.StepInputs(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda())


def _verify(w, S_dev, idx_dev, si_dev, T, out_dtype, status=None, q_scale=1.0, l2=False, guards=None):
    """The verify into NaN-filled tuple and output buffers, each between guard
    bands (checked here after the launch; the bands' owners go to `guards`)."""
    R = idx_dev.shape[0]
    su, sk, sg = Bd.tuple_shapes(_desc(w), R, T)
    g = [] if guards is None else guards
    tu = guarded(torch.full(su, float("nan")), g)
    tk = guarded(torch.full(sk, float("nan")), g)
    tg = guarded(torch.full(sg, float("nan")), g)
    out = guarded(torch.full((R * T, w.HV, w.V), float("nan"), dtype=out_dtype), g)
    Bd.gdn_lossless_verify(_desc(w), S_dev, T, Bd.Step(si_dev.mixed_qkv, si_dev.g, si_dev.beta, idx_dev, out,
                                                       q_scale, l2),
                           tu, tk, tg, status)
    torch.cuda.synchronize()
    check_guards(g, "lossless verify")
    return out, tu, tk, tg


CASES = {
    # name: (workload, T, out dtype)
    "gdn_k128_T4": (I.Workload("l", N=10, B=5, n_pad=2, HV=8, HK=4, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.BF16, seed=60), 4,
                    torch.float32),
    "gdn_k128_T16_bf16out": (I.Workload("l", N=10, B=4, n_pad=1, HV=4, HK=2, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.BF16,
                                        seed=61), 16, torch.bfloat16),
    "gdn_k64_T1": (I.Workload("l", N=6, B=3, n_pad=1, HV=4, HK=4, K=64, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.F32, seed=62), 1,
                   torch.float32),
    "gdn_k64_T32_fp32qkv": (I.Workload("l", N=6, B=3, n_pad=0, HV=4, HK=1, K=64, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.F32,
                                       seed=63), 32, torch.float32),
    "kda_k128_T8": (I.Workload("l", N=8, B=4, n_pad=1, HV=8, HK=4, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.BF16,
                               gate=Bd.GATE_PER_K, seed=64), 8, torch.float32),
    # the longest window: the staged checkpoint and 32 tokens' vectors in one block's shared memory
    "gdn_k128_T32": (I.Workload("l", N=6, B=3, n_pad=1, HV=4, HK=2, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.BF16,
                                seed=66), 32, torch.float32),
    "kda_k128_T32_f16out": (I.Workload("l", N=6, B=3, n_pad=0, HV=4, HK=2, K=128, L=1, ring_dtype=Bd.F32,
                                       qkv_dtype=Bd.F16, gate=Bd.GATE_PER_K, seed=67), 32, torch.float16),
    # one-token window, and the largest staging (a 32-token KDA window of fp32 inputs, 210 KB)
    "gdn_k128_T1": (I.Workload("l", N=6, B=4, n_pad=1, HV=4, HK=2, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.BF16,
                               seed=69), 1, torch.float32),
    "kda_k128_T32_fp32qkv": (I.Workload("l", N=4, B=2, n_pad=0, HV=4, HK=4, K=128, L=1, ring_dtype=Bd.F32,
                                        qkv_dtype=Bd.F32, gate=Bd.GATE_PER_K, seed=70), 32, torch.float32),
    # several items per block of the persistent verify, padding rows among them
    "gdn_k128_many_items_padded": (I.Workload("l", N=64, B=48, n_pad=8, HV=32, HK=16, K=128, L=1,
                                              ring_dtype=Bd.F32, qkv_dtype=Bd.BF16, seed=71), 3, torch.bfloat16),
    # HV not a multiple of 4: the gate and beta tiles cannot be mapped, the 8-lane form runs
    "gdn_k128_hv6_T5": (I.Workload("l", N=6, B=3, n_pad=1, HV=6, HK=3, K=128, L=1, ring_dtype=Bd.F32,
                                   qkv_dtype=Bd.BF16, seed=68), 5, torch.float32),
    "kda_k64_T3": (I.Workload("l", N=8, B=4, n_pad=1, HV=4, HK=4, K=64, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.F32,
                              gate=Bd.GATE_PER_K, seed=65), 3, torch.float32),
}


# cases whose inputs go through the in-kernel L2 norm and q_scale
NORMED = {"gdn_k128_T4", "kda_k64_T3"}


@pytest.mark.parametrize("name", list(CASES) + [n + "_l2norm" for n in sorted(NORMED)])
def test_verify_and_commit_are_bit_identical_to_packed_decode(gdnlib, name):
    normed = name.endswith("_l2norm")
    w, T, out_dtype = CASES[name[: -len("_l2norm")] if normed else name]
    gen, S0, idx, si = _setup(w, T, w.seed)
    if normed:  # unnormalised q, k: the kernels normalise and scale them
        si = I.StepInputs(si.mixed_qkv * 3.0, si.g, si.beta)
    q_scale, l2 = (0.37, True) if normed else (1.0, False)
    R = idx.shape[0]
    S_dev, idx_dev, si_dev = S0.cuda(), idx.cuda(), _dev_inputs(si)
    out, tu, tk, tg = _verify(w, S_dev, idx_dev, si_dev, T, out_dtype, q_scale=q_scale, l2=l2)
    ref_out, _ = _packed_sequence(w, S_dev, idx_dev, si_dev, T, out_dtype, q_scale=q_scale, l2=l2)
    torch.cuda.synchronize()
    assert torch.equal(S_dev.cpu(), S0), "verify wrote the state"
    assert _same_bits(out, ref_out), "verify outputs differ from successive packed decodes"

    # commit a random accepted prefix per row, in place
    acc = torch.randint(0, T + 1, (R,), generator=gen, dtype=torch.int32)
    acc[idx < 0] = -1
    cg: list = []
    st = guarded(S_dev, cg)
    Bd.gdn_lossless_commit(_desc(w), st, idx_dev, acc.cuda(), T, tu, tk, tg)
    torch.cuda.synchronize()
    check_guards(cg, "lossless commit")
    _, ref_st = _packed_sequence(w, S_dev, idx_dev, si_dev, T, out_dtype, accepted=acc.clamp(min=0),
                                 q_scale=q_scale, l2=l2)
    torch.cuda.synchronize()
    assert _same_bits(st, ref_st), "committed state differs from the packed decodes' state"

    # the oracle: outputs and corrections within 1e-5, key and gate tuples exact
    G = O.geom(w.N, w.HV, w.HK, w.K, w.V, gate=w.gate, state_dtype=O.F64)
    o_ref, tu_ref, tk_ref, tg_ref, status = O.lossless_verify(G, O.f64(S0), idx.numpy(), T, si.mixed_qkv,
                                                              si.g, si.beta, q_scale, int(l2))
    assert status == 0
    live = np.repeat(idx.numpy() >= 0, T)
    o = out.float().cpu().numpy()
    tol_o = TOL if out_dtype == torch.float32 else TOL + 2.0 ** -8
    assert _rel(o[live], o_ref[live]) <= tol_o
    assert np.all(o[~live] == 0.0), "padding rows must be zero"
    lb = idx.numpy() >= 0
    assert _rel(tu.cpu().numpy()[lb], tu_ref[lb]) <= TOL
    if normed:  # the normalised keys: fp32 on the GPU, double in the oracle
        assert _rel(tk.cpu().numpy()[lb], tk_ref[lb]) <= TOL
    else:  # copies of the inputs
        assert np.array_equal(tk.cpu().numpy()[lb], tk_ref[lb])
    assert np.array_equal(tg.cpu().numpy()[lb], tg_ref[lb])
    assert torch.all(torch.isnan(tu[torch.from_numpy(~lb).cuda()])), "padding rows' tuples must stay untouched"


@pytest.mark.parametrize("gate", [Bd.GATE_SCALAR, Bd.GATE_PER_K], ids=["gdn", "kda"])
@pytest.mark.parametrize("gmode", ["zero", "erase", "random"])
def test_commit_against_the_oracle(gdnlib, gate, gmode):
    """The commit fed the oracle's tuples: bit-exact where exp(g) is exact on
    both sides, within 1e-6 elsewhere."""
    w = I.Workload("c", N=7, B=4, n_pad=1, HV=4, HK=2, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.F32, gate=gate, seed=70)
    T = 5
    gen, S0, idx, si = _setup(w, T, w.seed)
    G = O.geom(w.N, w.HV, w.HK, w.K, w.V, gate=gate, state_dtype=O.F64)
    _, tu, tk, tg, st = O.lossless_verify(G, O.f64(S0), idx.numpy(), T, si.mixed_qkv, si.g, si.beta)
    assert st == 0
    if gmode == "zero":
        tg[:] = 0.0
    elif gmode == "erase":
        tg[:] = -1e4
    R = idx.shape[0]
    acc = torch.randint(0, T + 1, (R,), generator=gen, dtype=torch.int32)
    dst = idx.clone()
    ref = S0.numpy().astype(np.float32).copy()
    assert O.lossless_commit(G, ref, T, idx.numpy(), acc.numpy(), tu, tk, tg) == 0
    got = S0.cuda()
    Bd.gdn_lossless_commit(_desc(w), got, idx.cuda(), acc.cuda(), T, torch.from_numpy(tu).float().cuda(),
                           torch.from_numpy(tk).float().cuda(), torch.from_numpy(tg).float().cuda(),
                           dst_indices=dst.cuda())
    g = got.cpu().numpy()
    if gmode == "random":
        assert _rel(g, ref) <= 1e-6
    else:
        assert np.array_equal(g.view(np.uint32), ref.view(np.uint32))


def test_track_commit_before_in_place(gdnlib):
    """#42388 Commit, "Order matters": the track state (m tokens, into another
    slot) is committed first, then the accepted state in place; the other order
    gives a wrong track state."""
    w = I.Workload("t", N=8, B=2, n_pad=0, HV=4, HK=2, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.BF16, seed=71)
    T = 6
    gen, S0, idx, si = _setup(w, T, w.seed)
    S_dev, idx_dev, si_dev = S0.cuda(), idx.cuda(), _dev_inputs(si)
    _, tu, tk, tg = _verify(w, S_dev, idx_dev, si_dev, T, torch.float32)
    m = torch.tensor([2, 1], dtype=torch.int32)
    a = torch.tensor([5, 4], dtype=torch.int32)
    free = [s for s in range(w.N) if s not in idx.tolist()][:2]
    track = torch.tensor(free, dtype=torch.int32)
    _, st_m = _packed_sequence(w, S_dev, idx_dev, si_dev, T, torch.float32, accepted=m)
    _, st_a = _packed_sequence(w, S_dev, idx_dev, si_dev, T, torch.float32, accepted=a)
    d = _desc(w)
    st = S_dev.clone()
    Bd.gdn_lossless_commit(d, st, idx_dev, m.cuda(), T, tu, tk, tg, dst_indices=track.cuda())
    Bd.gdn_lossless_commit(d, st, idx_dev, a.cuda(), T, tu, tk, tg)
    for b in range(2):
        s = int(idx[b])
        assert _same_bits(st[track[b]], st_m[s]), "track state"
        assert _same_bits(st[s], st_a[s]), "accepted state"
    st = S_dev.clone()
    Bd.gdn_lossless_commit(d, st, idx_dev, a.cuda(), T, tu, tk, tg)
    Bd.gdn_lossless_commit(d, st, idx_dev, m.cuda(), T, tu, tk, tg, dst_indices=track.cuda())
    assert not _same_bits(st[track[0]], st_m[int(idx[0])]), "the wrong order must be visible"


def test_bad_rows_are_reported_and_touch_nothing(gdnlib):
    w = I.Workload("b", N=6, B=3, n_pad=0, HV=4, HK=2, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.BF16, seed=72)
    T = 3
    gen, S0, idx, si = _setup(w, T, w.seed)
    S_dev, si_dev = S0.cuda(), _dev_inputs(si)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_idx = torch.tensor([w.N + 3, -1, 2], dtype=torch.int32, device="cuda")
    out, tu, tk, tg = _verify(w, S_dev, bad_idx, si_dev, T, torch.float32, status)
    torch.cuda.synchronize()
    assert int(status.item()) == Bd.DEV_BAD_SLOT
    assert torch.all(out[: 2 * T] == 0) and torch.all(torch.isnan(tu[:2]))
    d = _desc(w)
    for src, acc, dst, bits in (([w.N], [1], None, Bd.DEV_BAD_SLOT), ([2], [T + 1], None, Bd.DEV_BAD_ACCEPTED),
                                ([2], [1], [w.N + 1], Bd.DEV_BAD_SLOT), ([-1], [1], None, 0), ([2], [-1], None, 0),
                                ([2], [1], [-1], 0), ([2], [0], None, 0)):
        st = S_dev.clone()
        status.zero_()
        dd = None if dst is None else torch.tensor(dst, dtype=torch.int32, device="cuda")
        Bd.gdn_lossless_commit(d, st, torch.tensor(src, dtype=torch.int32, device="cuda"),
                               torch.tensor(acc, dtype=torch.int32, device="cuda"), T, tu[2:3].contiguous(),
                               tk[2:3].contiguous(), tg[2:3].contiguous(), dst_indices=dd, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == bits, (src, acc, dst)
        assert _same_bits(st, S_dev), (src, acc, dst)


@pytest.mark.parametrize("T", [4, 8])
def test_layer_size_bit_identical(gdnlib, T):
    """One Qwen3-Next-like layer (HV=32, HK=16, K=V=128) at B=256 and a 4- or
    8-token window: verify outputs and the committed states against the packed
    decodes, bit for bit, over the whole batch."""
    w = I.Workload("layer", N=256, B=256, n_pad=0, HV=32, HK=16, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.BF16, seed=73)
    gen = I.generator(w.seed, "cuda")
    S_dev = I.state(gen, w.N, w.HV, w.V, w.K, "cuda")
    idx_dev = I.indices(gen, w.B, w.N, 0, "cuda")
    si_dev = I.step_inputs(gen, w, "cuda", rows=w.B * T)
    out, tu, tk, tg = _verify(w, S_dev, idx_dev, si_dev, T, torch.bfloat16)
    ref_out, _ = _packed_sequence(w, S_dev, idx_dev, si_dev, T, torch.bfloat16)
    assert _same_bits(out, ref_out)
    acc = torch.randint(0, T + 1, (w.B,), generator=gen, device="cuda", dtype=torch.int32)
    st = S_dev.clone()
    Bd.gdn_lossless_commit(_desc(w), st, idx_dev, acc, T, tu, tk, tg)
    _, ref_st = _packed_sequence(w, S_dev, idx_dev, si_dev, T, torch.bfloat16, accepted=acc.cpu())
    torch.cuda.synchronize()
    assert _same_bits(st, ref_st)
