"""Pins of the CPU oracle.

Each pin checks the oracle against something other than itself: a value the
pages print (the L = 4 cursor table), a closed form, an invariant of the
recurrence, a reduction to a simpler case, or a library routine (numpy / torch
float conversion).  A pin is a plain function that raises AssertionError on a
mismatch.  test_oracle_pins runs them all; test_oracle_mutations plants
mistakes in copies of the oracle source and checks that each is caught.

Page references (title, section):
  sglang #28451 "ReplaySSM decode": Modifications; Design 1, 3, 5, 7.
  "ReplaySSM" explainer (llm.rainlin.net): 1, 2.1, 2.2, 3.1, 3.3.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def _unit(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x)


def _close(a, b, tol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 0.0)
    assert a.shape == b.shape and err <= tol * scale, f"{what}: max err {err:.3e} (tol {tol:.1e})"


# ---------------------------------------------------------------------------
# Storage rounding against library conversions.
# ---------------------------------------------------------------------------

def pin_round_f16_f32_match_numpy():
    r = _rng(0)
    x = r.standard_normal(4000) * 10.0 ** r.integers(-9, 6, 4000)
    special = [2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -14, 65504.0, 65519.99, 65520.0,
               1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 1 + 2.0 ** -24, 1 + 3 * 2.0 ** -24, -0.0, 1e-30,
               -5.96e-8, 1e39]
    x = np.concatenate([x, special, -np.asarray(special)])
    with np.errstate(over="ignore"):
        for dt, npdt in ((O.F16, np.float16), (O.F32, np.float32)):
            want = x.astype(npdt).astype(np.float64)
            got = O.round_to(x, dt)
            assert np.array_equal(got, want), f"rounding to {npdt.__name__} differs from numpy"


def pin_round_bf16_matches_torch():
    r = _rng(1)
    x32 = (r.standard_normal(4000) * 10.0 ** r.integers(-40, 38, 4000)).astype(np.float32)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 2.0 ** -133, 3 * 2.0 ** -134], dtype=np.float32)
    x32 = np.concatenate([x32, ties, -ties])
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_to(x32.astype(np.float64), O.BF16)
    assert np.array_equal(got, want), "rounding to bf16 differs from torch"


# ---------------------------------------------------------------------------
# The sequential recurrence (explainer section 1; #28451 Design 7).
# K != V everywhere so a transposed operand cannot pass.
# ---------------------------------------------------------------------------

K5, V3 = 5, 3


def pin_gdn_retrieval():
    """beta = 1, |k| = 1: the new state maps k to v exactly, and y = S_t k = v."""
    r = _rng(2)
    S = r.standard_normal((V3, K5))
    k = _unit(r.standard_normal(K5))
    v = r.standard_normal(V3)
    y, _ = O.gdn_step(S, k, k, v, -0.7, 1.0)
    _close(S @ k, v, 1e-13, "S_t k")
    _close(y, v, 1e-13, "y with q = k")


def pin_gdn_decay_only():
    """beta = 0: S_t = exp(g) S, y = exp(g) S q, no correction."""
    r = _rng(3)
    S0 = r.standard_normal((V3, K5))
    S = S0.copy()
    q, k, v = r.standard_normal(K5), r.standard_normal(K5), r.standard_normal(V3)
    y, u = O.gdn_step(S, q, k, v, -0.3, 0.0)
    _close(S, np.exp(-0.3) * S0, 1e-15, "decayed state")
    _close(y, np.exp(-0.3) * (S0 @ q), 1e-14, "decayed output")
    assert np.all(u == 0.0)


def pin_gdn_identity_step():
    """beta = 0 and g = 0 leave the state bit-identical; y = S q."""
    r = _rng(4)
    S0 = r.standard_normal((V3, K5))
    S = S0.copy()
    q = r.standard_normal(K5)
    y, _ = O.gdn_step(S, q, r.standard_normal(K5), r.standard_normal(V3), 0.0, 0.0)
    assert np.array_equal(S, S0)
    _close(y, S0 @ q, 1e-14, "y")


def pin_gdn_other_directions_only_decay():
    """beta = 1, |k| = 1: a direction x orthogonal to k sees only the decay."""
    r = _rng(5)
    S0 = r.standard_normal((V3, K5))
    S = S0.copy()
    k = _unit(r.standard_normal(K5))
    x = r.standard_normal(K5)
    x -= (x @ k) * k
    O.gdn_step(S, r.standard_normal(K5), k, r.standard_normal(V3), -0.4, 1.0)
    _close(S @ x, np.exp(-0.4) * (S0 @ x), 1e-13, "S_t x")


def pin_gdn_erase_history():
    """g = -1e4 underflows alpha to 0: S_t = beta v k^T, y = beta v (k^T q)."""
    r = _rng(6)
    S = r.standard_normal((V3, K5))
    q, k, v = r.standard_normal(K5), r.standard_normal(K5), r.standard_normal(V3)
    y, u = O.gdn_step(S, q, k, v, -1e4, 0.6)
    _close(S, 0.6 * np.outer(v, k), 1e-15, "state")
    _close(y, 0.6 * v * (k @ q), 1e-14, "y")
    _close(u, 0.6 * v, 1e-15, "u")


def pin_gdn_correction_vanishes_when_retrieved():
    """If v already equals the decayed retrieval exp(g) S k, the correction u is 0."""
    r = _rng(7)
    S0 = r.standard_normal((V3, K5))
    k, q = r.standard_normal(K5), r.standard_normal(K5)
    v = np.exp(-0.2) * (S0 @ k)
    S = S0.copy()
    y, u = O.gdn_step(S, q, k, v, -0.2, 0.9)
    _close(u, np.zeros(V3), 1e-14, "u")
    _close(S, np.exp(-0.2) * S0, 1e-14, "state")


def pin_kda_equal_channels_is_gdn():
    """A per-channel gate with every channel equal reduces KDA to GDN."""
    r = _rng(8)
    S0 = r.standard_normal((V3, K5))
    q, k, v = r.standard_normal(K5), r.standard_normal(K5), r.standard_normal(V3)
    Sa, Sb = S0.copy(), S0.copy()
    ya, ua = O.gdn_step(Sa, q, k, v, -0.45, 0.7)
    yb, ub = O.kda_step(Sb, q, k, v, np.full(K5, -0.45), 0.7)
    _close(Sb, Sa, 1e-14, "state")
    _close(yb, ya, 1e-14, "y")


def pin_kda_decay_is_per_key_column():
    """KDA with beta = 0: column c of the state (key channel c) decays by exp(g[c])."""
    r = _rng(9)
    S0 = r.standard_normal((V3, K5))
    g = -r.random(K5)
    q = r.standard_normal(K5)
    S = S0.copy()
    y, _ = O.kda_step(S, q, r.standard_normal(K5), r.standard_normal(V3), g, 0.0)
    _close(S, S0 * np.exp(g)[None, :], 1e-15, "state")
    _close(y, S0 @ (np.exp(g) * q), 1e-14, "y")


def pin_kda_retrieval():
    r = _rng(10)
    S = r.standard_normal((V3, K5))
    k = _unit(r.standard_normal(K5))
    v = r.standard_normal(V3)
    y, _ = O.kda_step(S, k, k, v, -r.random(K5), 1.0)
    _close(S @ k, v, 1e-13, "S_t k")
    _close(y, v, 1e-13, "y")


def pin_scalar_head_closed_form():
    """K = V = 1: the recurrence is the scalar s <- a s + b (v - a s k) k with
    y = s q (a = exp g); the sequential step and the whole replay state machine
    (ring of 3, natural flushes, cursor advance) must follow it, for GDN and
    for KDA (one channel: its gate is the head's gate)."""
    r = _rng(600)
    steps = 10
    q, k, v = r.standard_normal(steps), r.standard_normal(steps), r.standard_normal(steps)
    g = -np.log1p(np.exp(r.standard_normal(steps)))
    b = 1 / (1 + np.exp(-r.standard_normal(steps)))
    s0 = 0.7
    want, s = [], s0
    for t in range(steps):
        a = np.exp(g[t])
        s = a * s + b[t] * (v[t] - a * s * k[t]) * k[t]
        want.append(s * q[t])
    for gate in (O.GATE_SCALAR, O.GATE_PER_K):
        S = np.array([[s0]])
        for t in range(steps):
            fn = O.kda_step if gate else O.gdn_step
            y, _ = fn(S, [q[t]], [k[t]], [v[t]], [g[t]] if gate else g[t], b[t])
            _close(y, [want[t]], 1e-14, f"scalar step {t} (gate {gate})")
        G = O.geom(1, 1, 1, 1, 1, 3, gate=gate, state_dtype=O.F64, ring_dtype=O.F64)
        gk = (1,) if gate else ()
        cache = O.Cache(np.full((1, 1, 1, 1), s0), np.full((1, 1, 3, 1), np.nan), np.full((1, 1, 3, 1), np.nan),
                        np.full((1, 1, 3) + gk, np.nan))
        wp = np.zeros(1, dtype=np.int32)
        for t in range(steps):
            gt = np.array([[[g[t]]]]) if gate else np.array([[g[t]]])
            o, _, st = O.replay_decode(G, cache, wp, [0], None, np.array([[q[t], k[t], v[t]]]), gt, np.array([[b[t]]]))
            assert st == 0 and O.replay_advance(1, [0], None, 3, wp) == 0
            _close(o[0, 0], [want[t]], 1e-13, f"scalar replay step {t} (gate {gate})")


# ---------------------------------------------------------------------------
# The replay state machine (explainer 2.1, 3.1-3.3; #28451 Design 1/3/5/7).
# ---------------------------------------------------------------------------

def _packed_row(q_heads, k_heads, v_heads):
    return np.concatenate([np.ravel(q_heads), np.ravel(k_heads), np.ravel(v_heads)])


class _Seq:
    """Random per-step inputs for one slot; HV value heads sharing HK key heads."""

    def __init__(self, seed, steps, HV, HK, K, V, gate):
        r = _rng(seed)
        self.q = np.stack([[_unit(r.standard_normal(K)) / np.sqrt(K) for _ in range(HK)] for _ in range(steps)])
        self.k = np.stack([[_unit(r.standard_normal(K)) for _ in range(HK)] for _ in range(steps)])
        self.v = r.standard_normal((steps, HV, V))
        self.g = -np.log1p(np.exp(r.standard_normal((steps, HV, K) if gate else (steps, HV))))
        self.beta = 1 / (1 + np.exp(-r.standard_normal((steps, HV))))
        self.HV, self.HK = HV, HK

    def row(self, t):
        return _packed_row(self.q[t], self.k[t], self.v[t])[None, :]


def _run_replay(G, S0, seq, steps, force=None, slot=0, fold_at=None):
    """Drives the oracle's replay decode over `steps` tokens for one slot.
    Returns per-step outputs, flushed flags, write_pos before each step, caches."""
    N, HV, HK, K, V, L = G.N, G.HV, G.HK, G.K, G.V, G.L
    gk = (K,) if G.gate == O.GATE_PER_K else ()
    cache = O.Cache(np.zeros((N, HV, V, K)), np.full((N, HV, L, V), np.nan),
                    np.full((N, HK, L, K), np.nan), np.full((N, HV, L) + gk, np.nan))
    cache.state[slot] = S0
    wp = np.zeros(N, dtype=np.int32)
    outs, flags, cursors = [], [], []
    for t in range(steps):
        if fold_at is not None and t == fold_at:
            assert O.replay_fold(G, cache, wp, [slot]) == 0
            wp[slot] = 0
        ff = None if force is None else np.array([force[t]], dtype=np.uint8)
        cursors.append(int(wp[slot]))
        o, fl, st = O.replay_decode(G, cache, wp, [slot], ff, seq.row(t), seq.g[t][None], seq.beta[t][None])
        assert st == 0
        assert O.replay_advance(N, [slot], ff, L, wp) == 0
        outs.append(o[0])
        flags.append(int(fl[0]))
    return np.array(outs), flags, cursors, cache, wp


def _run_sequential(S0, seq, steps, gate):
    """O1 per value head from the same checkpoint."""
    HV, HK = seq.HV, seq.HK
    S = [S0[h].copy() for h in range(HV)]
    ys, us = [], []
    for t in range(steps):
        yt, ut = [], []
        for h in range(HV):
            hk = h // (HV // HK)
            fn = O.kda_step if gate else O.gdn_step
            y, u = fn(S[h], seq.q[t][hk], seq.k[t][hk], seq.v[t][h], seq.g[t][h], seq.beta[t][h])
            yt.append(y)
            ut.append(u)
        ys.append(yt)
        us.append(ut)
    return np.array(ys), np.array(us), np.array(S)


def _replay_matches_sequential(gate):
    HV, HK, K, V, L, steps = 4, 2, K5, V3, 8, 19
    G = O.geom(2, HV, HK, K, V, L, gate=gate, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(20 + gate)
    S0 = r.standard_normal((HV, V, K)) * 0.3
    seq = _Seq(30 + gate, steps, HV, HK, K, V, gate)
    outs, flags, cursors, cache, wp = _run_replay(G, S0, seq, steps, slot=1)
    ys, us, S_seq = _run_sequential(S0, seq, steps, gate)
    _close(outs, ys, 1e-12, "replay outputs vs the sequential recurrence")
    # natural flush every L steps: cursor 0..L-1 then back to 0
    assert cursors == [t % L for t in range(steps)]
    assert flags == [int(t % L == L - 1) for t in range(steps)]
    # the state rebuilt from checkpoint + ring after the last step equals S_t
    for h in range(HV):
        _close(O.replay_state(G, cache, 1, h, int(wp[1])), S_seq[h], 1e-12, "replayed state")
    # the cached corrections are the recurrence's u_t for the steps since the flush
    last_flush = max(t for t in range(steps) if flags[t])
    for j, t in enumerate(range(last_flush + 1, steps)):
        _close(cache.ring_d[1, :, j], us[t], 1e-12, "ring d")
    # slot 0 was never named by a row: untouched
    assert np.all(cache.state[0] == 0.0) and np.all(np.isnan(cache.ring_d[0]))


def pin_replay_identity_gdn():
    """S_{c+h} = P_h S_c + sum_j w_{j,h} u_j k_j^T matches the step-by-step recurrence."""
    _replay_matches_sequential(O.GATE_SCALAR)


def pin_replay_identity_kda():
    _replay_matches_sequential(O.GATE_PER_K)


def pin_l1_is_packed_decode():
    """L = 1: every step flushes and the replay decode is the packed decode."""
    HV, HK, K, V, steps = 2, 1, 4, 6, 5
    G = O.geom(1, HV, HK, K, V, 1, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(40)
    S0 = r.standard_normal((HV, V, K))
    seq = _Seq(41, steps, HV, HK, K, V, 0)
    outs, flags, cursors, cache, _ = _run_replay(G, S0, seq, steps)
    state = S0[None].copy()
    for t in range(steps):
        o, st = O.packed_decode(G, state, [0], seq.row(t), seq.g[t][None], seq.beta[t][None])
        _close(outs[t], o[0], 1e-13, f"step {t}")
    assert flags == [1] * steps and cursors == [0] * steps
    _close(cache.state, state, 1e-13, "checkpoint")


def _factored_readout(gate):
    """The replayed state's readout S x, where S = A S0 + sum_j w_j d_j k_j^T
    (KDA: S0 Diag(A) + sum_j d_j (w_j o k_j)^T), equals the factored form
    A (S0 x) + sum_j w_j d_j (k_j . x) (KDA: S0 (A o x) + sum_j d_j ((w_j o k_j) . x))
    that never forms S ([P1] Design 1 "output-only"; [P2] 3.2): the algebra the
    output-only readout and the verify window's checkpoint products rely on."""
    HV, HK, K, V, L, p = 2, 1, K5, V3, 8, 5
    G = O.geom(1, HV, HK, K, V, L, gate=gate, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(610 + gate)
    gk = (K,) if gate else ()
    cache = O.Cache(r.standard_normal((1, HV, V, K)), r.standard_normal((1, HV, L, V)),
                    r.standard_normal((1, HK, L, K)), -np.abs(r.standard_normal((1, HV, L) + gk)))
    x = r.standard_normal(K)
    for hv in range(HV):
        S = O.replay_state(G, cache, 0, hv, p)
        S0, g = cache.state[0, hv], cache.ring_g[0, hv]
        d, k = cache.ring_d[0, hv], cache.ring_k[0, 0]
        if gate:
            A = np.exp(g[:p].sum(axis=0))
            y = S0 @ (A * x)
            for j in range(p):
                w = np.exp(g[j + 1:p].sum(axis=0))
                y = y + d[j] * np.dot(w * k[j], x)
        else:
            A = np.exp(g[:p].sum())
            y = A * (S0 @ x)
            for j in range(p):
                y = y + np.exp(g[j + 1:p].sum()) * d[j] * np.dot(k[j], x)
        _close(S @ x, y, 1e-12, f"factored readout, head {hv}")


def pin_factored_readout_gdn():
    _factored_readout(O.GATE_SCALAR)


def pin_factored_readout_kda():
    _factored_readout(O.GATE_PER_K)


def pin_walkthrough_L4():
    """The explainer's L = 4 table (section 3.3): checkpoint before each step,
    valid entries before each step, and the action taken."""
    rows = []
    with open(os.path.join(GOLDEN, "replay_walkthrough_L4.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                step, ckpt, valid, action = line.split()
                rows.append((int(step), ckpt, [] if valid == "-" else [int(x) for x in valid.split(",")], action))
    HV, HK, K, V, L = 1, 1, 4, 4, 4
    G = O.geom(1, HV, HK, K, V, L, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(50)
    S0 = r.standard_normal((HV, V, K))
    seq = _Seq(51, len(rows), HV, HK, K, V, 0)
    _, _, S4 = _run_sequential(S0, seq, 4, 0)
    cache = O.Cache(S0[None].copy(), np.full((1, HV, L, V), np.nan), np.full((1, HK, L, K), np.nan),
                    np.full((1, HV, L), np.nan))
    wp = np.zeros(1, dtype=np.int32)
    for step, ckpt, valid, action in rows:
        want_ckpt = S0 if ckpt == "S0" else S4
        _close(cache.state[0], want_ckpt, 1e-13, f"checkpoint before step {step}")
        # the valid entries are the tokens since the last flush, numbered from 1
        first = step - int(wp[0])
        assert list(range(first, step)) == valid, f"valid entries before step {step}"
        _, fl, st = O.replay_decode(G, cache, wp, [0], None, seq.row(step - 1), seq.g[step - 1][None],
                                    seq.beta[step - 1][None])
        assert st == 0
        assert ("flush" if fl[0] else "append") == action, f"action at step {step}"
        O.replay_advance(1, [0], None, L, wp)


def pin_forced_flush_mid_ring():
    """force_flush at a cursor below L-1 folds the valid entries and the current
    token into the checkpoint and restarts the ring (#28451 Design 5)."""
    HV, HK, K, V, L, steps = 2, 2, K5, V3, 6, 9
    G = O.geom(1, HV, HK, K, V, L, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(60)
    S0 = r.standard_normal((HV, V, K))
    seq = _Seq(61, steps, HV, HK, K, V, 0)
    force = [0, 0, 1, 0, 0, 0, 0, 0, 0]
    outs, flags, cursors, cache, wp = _run_replay(G, S0, seq, steps, force=force)
    ys, _, S_seq = _run_sequential(S0, seq, steps, 0)
    _close(outs, ys, 1e-12, "outputs")
    assert cursors == [0, 1, 2, 0, 1, 2, 3, 4, 5]
    assert flags == [0, 0, 1, 0, 0, 0, 0, 0, 1]
    _close(cache.state[0], S_seq, 1e-12, "checkpoint after the natural flush")


def pin_fold_then_reset():
    """Folding the ring into the checkpoint and resetting the cursor changes no output."""
    HV, HK, K, V, L, steps = 2, 1, K5, V3, 8, 7
    G = O.geom(1, HV, HK, K, V, L, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(70)
    S0 = r.standard_normal((HV, V, K))
    seq = _Seq(71, steps, HV, HK, K, V, 0)
    outs, _, cursors, cache, _ = _run_replay(G, S0, seq, steps, fold_at=4)
    ys, _, _ = _run_sequential(S0, seq, steps, 0)
    _close(outs, ys, 1e-12, "outputs across a fold")
    assert cursors == [0, 1, 2, 3, 0, 1, 2]
    _, _, S_at4 = _run_sequential(S0, seq, 4, 0)
    _, _, S_at7 = _run_sequential(S0, seq, 7, 0)
    # the fold made the checkpoint the state after 4 tokens; 3 more are in the ring
    _close(np.array([O.replay_state(G, cache, 0, h, 0) for h in range(HV)]), S_at4, 1e-12, "folded checkpoint")
    _close(np.array([O.replay_state(G, cache, 0, h, 3) for h in range(HV)]), S_at7, 1e-12, "replayed")


def pin_packed_layout_and_gqa():
    """mixed_qkv = q | k | v with key head hv // (HV/HK): from a zero state one
    step gives o = beta v_hv (k_hk . q_hk) and appends (beta v_hv, k_hk, g)."""
    HV, HK, K, V, L = 4, 2, K5, V3, 4
    G = O.geom(3, HV, HK, K, V, L, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(80)
    q = r.standard_normal((HK, K))
    k = r.standard_normal((HK, K))
    v = r.standard_normal((HV, V))
    g = -r.random(HV)
    beta = r.random(HV)
    cache = O.Cache(np.zeros((3, HV, V, K)), np.full((3, HV, L, V), np.nan), np.full((3, HK, L, K), np.nan),
                    np.full((3, HV, L), np.nan))
    wp = np.zeros(3, dtype=np.int32)
    o, fl, st = O.replay_decode(G, cache, wp, [2], None, _packed_row(q, k, v)[None], g[None], beta[None])
    assert st == 0 and fl[0] == 0
    for h in range(HV):
        hk = h // 2
        _close(o[0, h], beta[h] * v[h] * (k[hk] @ q[hk]), 1e-14, f"o head {h}")
        _close(cache.ring_d[2, h, 0], beta[h] * v[h], 1e-15, "ring d")
        assert cache.ring_g[2, h, 0] == g[h]
    for hk in range(HK):
        assert np.array_equal(cache.ring_k[2, hk, 0], k[hk])
    assert np.all(np.isnan(cache.ring_d[2, :, 1:])) and np.all(np.isnan(cache.ring_d[:2]))


def pin_padding_and_bad_rows():
    """Negative slots emit zeros and touch nothing; a slot >= N or a cursor
    outside [0, L) sets a status bit and is treated as padding."""
    HV, HK, K, V, L = 2, 1, 4, 4, 4
    G = O.geom(2, HV, HK, K, V, L, ring_dtype=O.F16)
    r = _rng(90)
    cache = O.Cache(r.standard_normal((2, HV, V, K)), np.full((2, HV, L, V), np.nan),
                    np.full((2, HK, L, K), np.nan), np.full((2, HV, L), np.nan))
    before = cache.copy()
    row = r.standard_normal((3, 2 * HK * K + HV * V))
    wp = np.array([0, 7], dtype=np.int32)
    o, fl, st = O.replay_decode(G, cache, wp, [-1, 5, 1], None, row, -r.random((3, HV)), r.random((3, HV)))
    assert np.all(o == 0.0) and list(fl) == [0, 0, 0]
    assert st == (O.BAD_SLOT | O.BAD_WRITE_POS)
    for a, b in ((cache.state, before.state), (cache.ring_d, before.ring_d), (cache.ring_k, before.ring_k)):
        assert np.array_equal(a, b, equal_nan=True)
    wp2 = wp.copy()
    assert O.replay_advance(2, [-1, 5, 1], None, L, wp2) == (O.BAD_SLOT | O.BAD_WRITE_POS)
    assert np.array_equal(wp2, wp)


def pin_storage_rounding():
    """Ring d and k are stored at the ring type (fp16 here), g exactly, and a
    flushed checkpoint at fp32."""
    HV, HK, K, V, L = 2, 1, 8, 8, 2
    G = O.geom(1, HV, HK, K, V, L, state_dtype=O.F32, ring_dtype=O.F16)
    r = _rng(100)
    seq = _Seq(101, 2, HV, HK, K, V, 0)
    cache = O.Cache(O.round_to(r.standard_normal((1, HV, V, K)), O.F32), np.full((1, HV, L, V), np.nan),
                    np.full((1, HK, L, K), np.nan), np.full((1, HV, L), np.nan))
    wp = np.zeros(1, dtype=np.int32)
    O.replay_decode(G, cache, wp, [0], None, seq.row(0), seq.g[0][None], seq.beta[0][None])
    assert np.array_equal(cache.ring_k[0, 0, 0], seq.k[0][0].astype(np.float16).astype(np.float64))
    d = cache.ring_d[0, :, 0]
    assert np.array_equal(d, d.astype(np.float16).astype(np.float64))
    assert np.array_equal(cache.ring_g[0, :, 0], seq.g[0])
    O.replay_advance(1, [0], None, L, wp)
    O.replay_decode(G, cache, wp, [0], None, seq.row(1), seq.g[1][None], seq.beta[1][None])
    s = cache.state[0]
    assert np.array_equal(s, s.astype(np.float32).astype(np.float64))


def pin_superposition():
    """With exact storage the outputs are jointly linear in (S0, v) for fixed q, k, g, beta."""
    HV, HK, K, V, L, steps = 2, 1, K5, V3, 4, 9
    G = O.geom(1, HV, HK, K, V, L, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(110)
    Sa, Sb = r.standard_normal((HV, V, K)), r.standard_normal((HV, V, K))
    sa = _Seq(111, steps, HV, HK, K, V, 0)
    sb = _Seq(111, steps, HV, HK, K, V, 0)
    sb.v = r.standard_normal(sb.v.shape)
    sab = _Seq(111, steps, HV, HK, K, V, 0)
    sab.v = sa.v + sb.v
    oa = _run_replay(G, Sa, sa, steps)[0]
    ob = _run_replay(G, Sb, sb, steps)[0]
    oab = _run_replay(G, Sa + Sb, sab, steps)[0]
    _close(oab, oa + ob, 1e-12, "superposition")


def pin_q_scale_is_linear_and_l2norm_scale_free():
    """out = alpha S q + d (k^T q) with d independent of q: the output is exactly
    linear in q_scale.  With the in-kernel L2 norm on, rescaling the raw q and k
    of a row by positive factors leaves every output unchanged (up to the norm's
    epsilon)."""
    HV, HK, K, V, L = 2, 1, 6, 4, 4
    G = O.geom(1, HV, HK, K, V, L, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(120)
    seq = _Seq(121, 3, HV, HK, K, V, 0)
    S0 = r.standard_normal((HV, V, K))

    def run(scale, l2, qmul=1.0, kmul=1.0):
        cache = O.Cache(S0[None].copy(), np.full((1, HV, L, V), np.nan), np.full((1, HK, L, K), np.nan),
                        np.full((1, HV, L), np.nan))
        wp = np.zeros(1, dtype=np.int32)
        outs = []
        for t in range(3):
            row = seq.row(t).copy()
            row[0, :HK * K] *= qmul
            row[0, HK * K:2 * HK * K] *= kmul
            o, _, _ = O.replay_decode(G, cache, wp, [0], None, row, seq.g[t][None], seq.beta[t][None], scale, l2)
            O.replay_advance(1, [0], None, L, wp)
            outs.append(o)
        return np.array(outs)

    base = run(1.0, 0)
    _close(run(0.37, 0)[0], 0.37 * base[0], 1e-14, "first step linear in q_scale")
    a = run(0.5, 1, qmul=10.0, kmul=10.0)
    b = run(0.5, 1, qmul=70.0, kmul=30.0)
    _close(b, a, 1e-6, "L2 norm makes the output independent of q, k magnitudes")
    assert np.max(np.abs(a - base)) > 1e-3  # the norm does change un-normalised inputs


# ---------------------------------------------------------------------------
# Speculative verify window and commit (vLLM #49887 "ReplaySSM: cache SSM
# inputs for faster Gated DeltaNet speculative decode": Core concept, Design
# notes).  Checked against the sequential recurrence run from the committed
# state: every window token's output, every cached correction, the cursor move
# and the fold that follows.
# ---------------------------------------------------------------------------

def _spec_matches_recurrence(gate):
    HV, HK, K, V, L, T, windows = 4, 2, K5, V3, 9, 3, 12
    N, slot = 2, 1
    G = O.geom(N, HV, HK, K, V, L, gate=gate, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(200 + gate)
    S0 = r.standard_normal((HV, V, K)) * 0.3
    gk = (K,) if gate else ()
    cache = O.Cache(np.zeros((N, HV, V, K)), np.full((N, HV, L, V), np.nan),
                    np.full((N, HK, L, K), np.nan), np.full((N, HV, L) + gk, np.nan))
    cache.state[slot] = S0
    wp = np.zeros(N, dtype=np.int32)
    S_ref = [S0[h].copy() for h in range(HV)]  # the committed state, by the recurrence
    flushes = 0
    for w in range(windows):
        seq = _Seq(300 + 10 * gate + w, T, HV, HK, K, V, gate)
        p = int(wp[slot])
        rows = np.concatenate([seq.row(t) for t in range(T)])
        o, st = O.spec_verify(G, cache, wp, [slot], T, rows, seq.g, seq.beta)
        assert st == 0 and int(wp[slot]) == p, "verify moved the cursor"
        # reference: the window decoded one token at a time from the committed state
        S_win = [S_ref[h].copy() for h in range(HV)]
        for t in range(T):
            for h in range(HV):
                hk = h // (HV // HK)
                fn = O.kda_step if gate else O.gdn_step
                y, u = fn(S_win[h], seq.q[t][hk], seq.k[t][hk], seq.v[t][h], seq.g[t][h], seq.beta[t][h])
                _close(o[t, h], y, 1e-12, f"window {w} token {t} head {h} output")
                _close(cache.ring_d[slot, h, p + t], u, 1e-12, f"window {w} token {t} cached correction")
        accepted = int(r.integers(0, T + 1))
        fs, st = O.spec_commit(N, L, T, [slot], [accepted], wp)
        assert st == 0 and int(wp[slot]) == p + accepted
        assert int(fs[0]) == (slot if p + accepted + T > L - 1 else -1)
        # the committed state moves over the accepted tokens only
        S_acc = [S_ref[h].copy() for h in range(HV)]
        for t in range(accepted):
            for h in range(HV):
                hk = h // (HV // HK)
                fn = O.kda_step if gate else O.gdn_step
                fn(S_acc[h], seq.q[t][hk], seq.k[t][hk], seq.v[t][h], seq.g[t][h], seq.beta[t][h])
        S_ref = S_acc
        for h in range(HV):
            _close(O.replay_state(G, cache, slot, h, int(wp[slot])), S_ref[h], 1e-12,
                   f"window {w}: committed state rebuilt from checkpoint + ring")
        if fs[0] >= 0:  # the fold the commit asked for, then the cursor reset
            assert O.replay_fold(G, cache, wp, fs) == 0
            wp[slot] = 0
            flushes += 1
            for h in range(HV):
                _close(cache.state[slot, h], S_ref[h], 1e-12, f"window {w}: folded checkpoint")
    assert flushes >= 2, "the sequence should cross several folds"
    assert np.all(cache.state[0] == 0.0) and np.all(np.isnan(cache.ring_d[0])), "slot 0 was touched"


def pin_spec_window_is_the_recurrence_gdn():
    _spec_matches_recurrence(O.GATE_SCALAR)


def pin_spec_window_is_the_recurrence_kda():
    _spec_matches_recurrence(O.GATE_PER_K)


def pin_spec_bad_rows():
    """Padding rows give zeros and touch nothing; a window that does not fit
    the ring (p + T > L - 1), a slot past the pool and an accepted count outside
    [0, T] are reported and touch nothing."""
    HV, HK, K, V, L, T = 2, 1, 4, 3, 6, 3
    N = 3
    G = O.geom(N, HV, HK, K, V, L, state_dtype=O.F64, ring_dtype=O.F64)
    r = _rng(400)
    cache = O.Cache(r.standard_normal((N, HV, V, K)), np.full((N, HV, L, V), np.nan),
                    np.full((N, HK, L, K), np.nan), np.full((N, HV, L), np.nan))
    before = cache.copy()
    seq = _Seq(401, T, HV, HK, K, V, 0)
    rows = np.concatenate([seq.row(t) for t in range(T)])
    wp = np.array([0, 3, 0], dtype=np.int32)  # slot 1: 3 + 3 > 5
    for idx, want in (([-1], 0), ([7], O.BAD_SLOT), ([1], O.BAD_WRITE_POS)):
        o, st = O.spec_verify(G, cache, wp, idx, T, rows, seq.g, seq.beta)
        assert st == want and np.all(o == 0.0), f"rows {idx}"
    assert np.array_equal(cache.state, before.state) and np.all(np.isnan(cache.ring_d))
    fs, st = O.spec_commit(N, L, T, [0, -1, 2], [T + 1, 1, -1], wp)
    assert st == O.BAD_ACCEPTED and list(fs) == [-1, -1, -1] and list(wp) == [0, 3, 0]


# ---------------------------------------------------------------------------
# Lossless verify and its exact-order commit (sglang #42388: "The idea";
# Modifications, "Verify kernel" and "Commit"; the tests it lists).  The commit
# replays fp32 (u, k, g) tuples with one rounded multiply (the decayed state)
# and one fma (the update) per element, so its state must equal, bit for bit,
# the state a binary32 sequential step with that rounding reaches.
# ---------------------------------------------------------------------------

def _f32_sequence(gate, seed, T, HV, HK, K, V, h0):
    """Runs oracle_step_f32 T times per value head from h0 [HV][V][K] (float32).
    Returns the states after every token [T + 1][HV][V][K], outputs, and the
    tuples (u [T][HV][V], k [T][HK][K], g [T][HV](, K)) in float32."""
    seq = _Seq(seed, T, HV, HK, K, V, gate)
    h = h0.copy()
    states, ys = [h.copy()], np.zeros((T, HV, V), dtype=np.float32)
    tu = np.zeros((T, HV, V), dtype=np.float32)
    tk = seq.k.astype(np.float32)
    tg = seq.g.astype(np.float32)
    for t in range(T):
        for hv in range(HV):
            hk = hv // (HV // HK)
            gk = tg[t, hv] if gate else None
            y, u = O.step_f32(h[hv], seq.q[t][hk], tk[t, hk], seq.v[t][hv],
                              0.0 if gate else tg[t, hv], seq.beta[t][hv], gk=gk)
            ys[t, hv], tu[t, hv] = y, u
        states.append(h.copy())
    return seq, states, ys, tu, tk, tg


def _bits_equal(a, b):
    return np.array_equal(np.asarray(a, dtype=np.float32).view(np.uint32),
                          np.asarray(b, dtype=np.float32).view(np.uint32))


def _lossless_commit_bit_identical(gate):
    HV, HK, K, V, T, N = 4, 2, K5, V3, 6, 3
    G = O.geom(N, HV, HK, K, V, gate=gate)
    r = _rng(500 + gate)
    pool = (r.standard_normal((N, HV, V, K)) * 0.3).astype(np.float32)
    slots = [2, 0]
    runs = [_f32_sequence(gate, 510 + 10 * gate + i, T, HV, HK, K, V, pool[s]) for i, s in enumerate(slots)]
    tup_u = np.stack([run[3] for run in runs])
    tup_k = np.stack([run[4] for run in runs])
    tup_g = np.stack([run[5] for run in runs])
    # the binary32 step follows the recurrence (O1, double) to fp32 accuracy
    for (seq, states, ys, _, _, _), s in zip(runs, slots):
        S = [pool[s, hv].astype(np.float64) for hv in range(HV)]
        for t in range(T):
            for hv in range(HV):
                hk = hv // (HV // HK)
                fn = O.kda_step if gate else O.gdn_step
                y, _ = fn(S[hv], seq.q[t][hk], seq.k[t][hk], seq.v[t][hv], seq.g[t][hv], seq.beta[t][hv])
                _close(ys[t, hv], y, 2e-6, "binary32 step output vs the recurrence")
                _close(states[t + 1][hv], S[hv], 2e-6, "binary32 step state vs the recurrence")
    for a0 in range(T + 1):
        a1 = T - a0
        st = pool.copy()
        assert O.lossless_commit(G, st, T, slots, [a0, a1], tup_u, tup_k, tup_g) == 0
        assert _bits_equal(st[2], runs[0][1][a0]), f"{a0} accepted: committed state is not bit-identical"
        assert _bits_equal(st[0], runs[1][1][a1]), f"{a1} accepted: committed state is not bit-identical"
        assert _bits_equal(st[1], pool[1]), "a slot no row names was touched"


def pin_lossless_commit_is_bit_identical_gdn():
    _lossless_commit_bit_identical(O.GATE_SCALAR)


def pin_lossless_commit_is_bit_identical_kda():
    _lossless_commit_bit_identical(O.GATE_PER_K)


def _lossless_verify_is_sequential(gate):
    HV, HK, K, V, T, N = 4, 2, K5, V3, 5, 4
    G = O.geom(N, HV, HK, K, V, gate=gate, state_dtype=O.F64)
    r = _rng(520 + gate)
    state = r.standard_normal((N, HV, V, K)) * 0.3
    before = state.copy()
    idx = [3, -1, 1]
    seqs = [_Seq(530 + 10 * gate + b, T, HV, HK, K, V, gate) for b in range(len(idx))]
    rows = np.concatenate([np.concatenate([sq.row(t) for t in range(T)]) for sq in seqs])
    g = np.concatenate([sq.g for sq in seqs])
    beta = np.concatenate([sq.beta for sq in seqs])
    o, tu, tk, tg, st = O.lossless_verify(G, state, idx, T, rows, g, beta)
    assert st == 0 and np.array_equal(state, before), "verify changed the checkpoint"
    for b, (slot, sq) in enumerate(zip(idx, seqs)):
        if slot < 0:
            assert np.all(o[b * T:(b + 1) * T] == 0.0) and np.all(tu[b] == 0.0), "padding row"
            continue
        ref = state.copy()  # T packed decodes (which do write the state) on a copy
        for t in range(T):
            ob, st2 = O.packed_decode(G, ref, [slot], sq.row(t), sq.g[t][None], sq.beta[t][None])
            _close(o[b * T + t], ob[0], 1e-13, f"row {b} token {t} output vs packed decode")
        _, us, _ = _run_sequential(state[slot], sq, T, gate)
        assert np.array_equal(tu[b], O.round_to(us, O.F32)), "u tuples are not the recurrence's corrections"
        assert np.array_equal(tk[b], O.round_to(sq.k, O.F32)), "k tuples are not the keys"
        assert np.array_equal(tg[b], O.round_to(sq.g, O.F32)), "g tuples are not the log-gates"
        # committing all T tuples (binary32) lands on the recurrence's state
        f = state.astype(np.float32)
        assert O.lossless_commit(G, f, T, [slot], [T], tu[b:b + 1], tk[b:b + 1], tg[b:b + 1]) == 0
        _close(f[slot], ref[slot], 2e-6, "commit of the verify's tuples vs the packed decodes' state")
    o, tu, tk, tg, st = O.lossless_verify(G, state, [N + 2], T, rows[:T], g[:T], beta[:T])
    assert st == O.BAD_SLOT and np.all(o == 0.0)


def pin_lossless_verify_is_sequential_gdn():
    _lossless_verify_is_sequential(O.GATE_SCALAR)


def pin_lossless_verify_is_sequential_kda():
    _lossless_verify_is_sequential(O.GATE_PER_K)


def pin_lossless_commit_special_cases():
    """No accepted token or a zero update leaves the state's bits alone; an
    erased history (exp underflows to 0) leaves exactly fl32(k u); bad rows are
    reported and touch nothing; negative entries are skipped."""
    HV, HK, K, V, T, N = 2, 1, 4, 3, 3, 3
    G = O.geom(N, HV, HK, K, V)
    r = _rng(540)
    pool = r.standard_normal((N, HV, V, K)).astype(np.float32)
    tu = r.standard_normal((1, T, HV, V)).astype(np.float32)
    tk = r.standard_normal((1, T, HK, K)).astype(np.float32)
    tg = (-r.random((1, T, HV))).astype(np.float32)
    st = pool.copy()
    assert O.lossless_commit(G, st, T, [1], [0], tu, tk, tg) == 0 and _bits_equal(st, pool)
    st = pool.copy()
    assert O.lossless_commit(G, st, T, [1], [T], np.zeros_like(tu), tk, np.zeros_like(tg)) == 0
    assert _bits_equal(st, pool), "g = 0, u = 0 must leave the state's bits unchanged"
    st = pool.copy()
    assert O.lossless_commit(G, st, T, [1], [1], tu, tk, np.full_like(tg, -1e4)) == 0
    want = tu[0, 0, :, :, None] * tk[0, 0, 0][None, None, :]  # float32 products, rounded once
    assert _bits_equal(st[1], want), "an erased history must leave fl32(k u)"
    for src, acc, dst, code in (([N], [1], None, O.BAD_SLOT), ([0], [T + 1], None, O.BAD_ACCEPTED),
                                ([0], [1], [N + 1], O.BAD_SLOT), ([-1], [1], None, 0), ([0], [-1], None, 0),
                                ([0], [1], [-1], 0)):
        st = pool.copy()
        assert O.lossless_commit(G, st, T, src, acc, tu, tk, tg, dst=dst) == code, (src, acc, dst)
        assert _bits_equal(st, pool), (src, acc, dst)


def pin_lossless_track_commit_before_in_place():
    """#42388 Commit, "Order matters": the prefix-cache track state (m tokens,
    written to another slot) must be replayed before the in-place replay of the
    accepted state, because both start from the pre-verify state."""
    HV, HK, K, V, T, N = 2, 1, K5, V3, 5, 4
    G = O.geom(N, HV, HK, K, V)
    r = _rng(550)
    pool = (r.standard_normal((N, HV, V, K)) * 0.3).astype(np.float32)
    _, states, _, tu, tk, tg = _f32_sequence(0, 551, T, HV, HK, K, V, pool[0])
    m, a, track = 2, 4, 3
    st = pool.copy()
    assert O.lossless_commit(G, st, T, [0], [m], tu[None], tk[None], tg[None], dst=[track]) == 0
    assert O.lossless_commit(G, st, T, [0], [a], tu[None], tk[None], tg[None]) == 0
    assert _bits_equal(st[track], states[m]) and _bits_equal(st[0], states[a])
    st = pool.copy()  # the wrong order: the track replay starts from the advanced state
    assert O.lossless_commit(G, st, T, [0], [a], tu[None], tk[None], tg[None]) == 0
    assert O.lossless_commit(G, st, T, [0], [m], tu[None], tk[None], tg[None], dst=[track]) == 0
    assert not _bits_equal(st[track], states[m])


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
