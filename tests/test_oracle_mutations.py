"""Control test for the oracle pins: each plausible mistake, planted in a copy of
the oracle source compiled on the CPU, must make at least one pin fail.  If a
planted mistake passes every pin, the pins are too weak to trust the oracle."""
import os
import tempfile

import pytest

import oracle as O
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(O.__file__), "gdn_oracle.c")

# (name, exact text in gdn_oracle.c, planted replacement)
MUTATIONS = [
    ("no_decay_before_correction",
     "for (size_t i = 0; i < (size_t)V * K; i++) S[i] *= alpha;       /* S~ = alpha S  */",
     "/* decay dropped */"),
    ("correction_sign",
     "for (int r = 0; r < V; r++) u[r] = beta * (v[r] - Sk[r]);        /* u             */",
     "for (int r = 0; r < V; r++) u[r] = beta * (v[r] + Sk[r]);"),
    ("update_transposed",
     "for (int c = 0; c < K; c++) S[(size_t)r * K + c] += u[r] * k[c];\n    matvec(V, K, S, q, y);                                           /* y = S_t q     */",
     "for (int c = 0; c < K; c++) S[(size_t)r * K + c] += u[r % V] * k[(c + r) % K];\n    matvec(V, K, S, q, y);"),
    ("output_from_old_state",
     "for (int c = 0; c < K; c++) S[(size_t)r * K + c] += u[r] * k[c];\n    matvec(V, K, S, q, y);                                           /* y = S_t q     */",
     "for (int c = 0; c < K; c++) S[(size_t)r * K + c] += 0.0;\n    matvec(V, K, S, q, y);\n"
     "    for (int r = 0; r < V; r++) for (int c = 0; c < K; c++) S[(size_t)r * K + c] += u[r] * k[c];"),
    ("kda_decay_on_rows",
     "for (int c = 0; c < K; c++) S[(size_t)r * K + c] *= exp(g[c]);",
     "for (int c = 0; c < K; c++) S[(size_t)r * K + c] *= exp(g[r % K]);"),
    ("gqa_map_modulo",
     "    int hk = hv / group;",
     "    int hk = hv % G->HK;"),
    ("q_k_swapped",
     "const double *qs = row + (size_t)hk * G->K;\n    const double *ks = row + (size_t)G->HK * G->K + (size_t)hk * G->K;",
     "const double *ks = row + (size_t)hk * G->K;\n    const double *qs = row + (size_t)G->HK * G->K + (size_t)hk * G->K;"),
    ("replay_weight_includes_own_gate",
     "for (int i = j + 1; i < p; i++) w *= exp(gr[i]);",
     "for (int i = j; i < p; i++) w *= exp(gr[i]);"),
    ("total_decay_one_short",
     "for (int j = 0; j < p; j++) A *= exp(gr[j]);",
     "for (int j = 1; j < p; j++) A *= exp(gr[j]);"),
    ("kda_replay_weight_index",
     "for (int i = j + 1; i < p; i++) w *= exp(gr[(size_t)i * K + c]);",
     "for (int i = j + 1; i <= p && i < L; i++) w *= exp(gr[(size_t)i * K + c]);"),
    ("readout_missing_decay",
     "for (int r = 0; r < V; r++) { Sq[r] *= alpha; Sk[r] *= alpha; }",
     "for (int r = 0; r < V; r++) { Sk[r] *= alpha; }"),
    ("output_drops_current_token",
     "ob[r] = Sq[r] + d[r] * kq;",
     "ob[r] = Sq[r];"),
    ("flush_without_decay",
     ": exp(gc[0]) * S[(size_t)r * K + c];",
     ": S[(size_t)r * K + c];"),
    ("append_at_next_position",
     "double *dr = ring_d + (((size_t)slot * HV + hv) * L + p) * V;",
     "double *dr = ring_d + (((size_t)slot * HV + hv) * L + (p + 1) % L) * V;"),
    ("advance_off_by_one",
     "write_pos[slot] = (p == L - 1 || ff) ? 0 : p + 1;",
     "write_pos[slot] = (p == L - 2 || ff) ? 0 : p + 1;"),
    ("q_scale_ignored",
     "for (int c = 0; c < K; c++) q[c] *= q_scale;",
     "for (int c = 0; c < K; c++) q[c] *= 1.0;"),
    ("l2norm_of_q_only",
     "for (int c = 0; c < K; c++) { q[c] /= nq; k[c] /= nk; }",
     "for (int c = 0; c < K; c++) { q[c] /= nq; }"),
    ("f16_mantissa_width",
     "case ORACLE_F16:  return round_binary(x, 10, -14, 15);",
     "case ORACLE_F16:  return round_binary(x, 11, -14, 15);"),
    ("spec_window_ignores_own_tokens",
     "cursor[slot] = p + t;",
     "cursor[slot] = p;"),
    ("spec_commit_moves_over_rejected",
     "write_pos[slot] = p + a;",
     "write_pos[slot] = p + T;"),
    ("spec_fold_rule_one_late",
     "if (p + a + T > L - 1) flush_slots[b] = slot;",
     "if (p + a + T > L) flush_slots[b] = slot;"),
    ("commit_update_not_fused",
     "h[(size_t)r * K + c] = fmaf(kt[c], ut[r], decayed);",
     "h[(size_t)r * K + c] = kt[c] * ut[r] + decayed;"),
    ("commit_other_contraction",
     "h[(size_t)r * K + c] = fmaf(kt[c], ut[r], decayed);",
     "h[(size_t)r * K + c] = fmaf(h[(size_t)r * K + c], at, kt[c] * ut[r]);"),
    ("commit_one_token_too_many",
     "for (int t = 0; t < a; t++) {\n                size_t row = (size_t)b * T + t;\n                const float *ut",
     "for (int t = 0; t <= a && t < T; t++) {\n                size_t row = (size_t)b * T + t;\n                const float *ut"),
    ("commit_gate_of_next_token",
     ": expf(tup_g[row * HV + hv]);",
     ": expf(tup_g[(row + (t + 1 < a)) * HV + hv]);"),
    ("commit_writes_source_slot",
     "memcpy(state + ((size_t)d * HV + hv) * V * K, h, sizeof(float) * (size_t)V * K);",
     "memcpy(state + ((size_t)s * HV + hv) * V * K, h, sizeof(float) * (size_t)V * K);"),
    ("verify_u_tuple_of_other_head",
     "for (int r = 0; r < V; r++) tup_u[(row * HV + hv) * V + r] = oracle_round(u[r], ORACLE_F32);",
     "for (int r = 0; r < V; r++) tup_u[(row * HV + (hv ^ 1)) * V + r] = oracle_round(u[r], ORACLE_F32);"),
    ("spec_capacity_one_more",
     "if (ok && (p < 0 || p + T > G->L - 1)) { *status |= ORACLE_BAD_WRITE_POS; ok = 0; }",
     "if (ok && (p < 0 || p + T > G->L)) { *status |= ORACLE_BAD_WRITE_POS; ok = 0; }"),
]


def _failing_pins():
    failed = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "gdn_oracle_mutated.c"
    mutated.write_text(src.replace(old, new))
    lib = O.compile_source(str(mutated), str(tmp_path / "liboracle_mutated.so"))
    with O.using_library(lib):
        failed = _failing_pins()
    assert failed, f"planted mistake '{name}' passed every pin"


def test_unmutated_copy_passes():
    with tempfile.TemporaryDirectory() as d:
        lib = O.compile_source(SRC, os.path.join(d, "liboracle_copy.so"))
        with O.using_library(lib):
            assert _failing_pins() == []
