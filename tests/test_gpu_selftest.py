"""The on-chip wait bound, exercised without anything being stuck.

A block waits, with the same bounded wait the decode kernels use, on a
shared-memory barrier that no thread ever arrives on; the wait must run out,
report GDN_DEV_TIMEOUT in the status word and return, and the context must stay
usable (a packed decode afterwards still matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle as O
from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_reports(gdnlib):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    Bd.gdn_selftest_wait_timeout(status, limit_us=2000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == Bd.DEV_TIMEOUT
    assert 0.002 <= elapsed < 5.0, f"the wait took {elapsed:.4f} s"

    # the context is still usable
    w = I.Workload("after", N=6, B=3, n_pad=1, HV=4, HK=2, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.F32, seed=90)
    gen = I.generator(w.seed, "cpu")
    S0 = I.state(gen, w.N, w.HV, w.V, w.K, "cpu")
    idx = I.indices(gen, w.B, w.N, w.n_pad, "cpu")
    si = I.step_inputs(gen, w, "cpu")
    out = torch.empty((idx.shape[0], w.HV, w.V), device="cuda")
    st = S0.cuda()
    Bd.gdn_packed_decode(Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, 1), st,
                         Bd.Step(si.mixed_qkv.cuda(), si.g.cuda(), si.beta.cuda(), idx.cuda(), out))
    o_ref, _ = O.packed_decode(O.geom(w.N, w.HV, w.HK, w.K, w.V), O.f64(S0), idx.numpy(), si.mixed_qkv, si.g, si.beta)
    err = np.max(np.abs(out.cpu().numpy() - o_ref)) / np.max(np.abs(o_ref))
    assert err <= 1e-5
