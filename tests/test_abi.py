"""The C ABI library without a GPU: it loads, exports every entry point that
include/*.h declares, and its host-side argument checks reject bad calls
before any CUDA call is made."""
import ctypes
import glob
import os
import re

import pytest

from linear_attention_decode_gb300 import binding as Bd
from linear_attention_decode_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names += re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", open(h).read())
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return Bd.load_library()


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("gdn_packed_decode", "gdn_replayssm_decode", "gdn_replayssm_decode_advance", "gdn_replayssm_advance",
              "gdn_replayssm_flush", "gdn_replayssm_reset_slots", "gdn_status_str", "gdn_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_entry_points():
        assert hasattr(lib, n), f"{n} is declared in include/ but not exported"


def _step(batch=4, row=2 * 16 * 128 + 32 * 128, flags=0):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: every case below fails a host check
    return Bd._Step(fake, Bd.BF16, row, fake, fake, fake, batch, 1.0, 0, fake, Bd.F32, flags)


def _desc(**kw):
    d = dict(num_slots=8, num_v_heads=32, num_k_heads=16, k_dim=128, v_dim=128, ring_len=16)
    d.update(kw)
    return Bd.layer_desc(**d)


CASES = [
    ("hv_not_multiple_of_hk", _desc(num_k_heads=5), 1),
    ("k_dim_96", _desc(k_dim=96, v_dim=96), 2),
    ("k_ne_v", _desc(v_dim=64), 2),
    ("ring_len_65", _desc(ring_len=65), 2),
    ("ring_len_0", _desc(ring_len=0), 1),
    ("bf16_state", Bd.layer_desc(8, 32, 16, 128, 128, 16, state_dtype=Bd.BF16), 2),
    ("bad_gate", Bd.layer_desc(8, 32, 16, 128, 128, 16, gate=7), 1),
]


@pytest.mark.parametrize("name,desc,code", CASES, ids=[c[0] for c in CASES])
def test_decode_rejects_bad_descriptors(lib, name, desc, code):
    cache = Bd._Cache(0x1000, 0x1000, 0x1000, 0x1000)
    st = lib.gdn_replayssm_decode(ctypes.byref(desc), ctypes.byref(cache), 0x1000, None,
                                  ctypes.byref(_step()), 0, None, None, None)
    assert st == code, lib.gdn_last_error().decode()
    st = lib.gdn_packed_decode(ctypes.byref(desc), 0x1000, ctypes.byref(_step()), None, None)
    assert st == code


def test_decode_rejects_bad_pointers_and_sizes(lib):
    d = _desc()
    good = Bd._Cache(0x1000, 0x1000, 0x1000, 0x1000)
    calls = [
        (Bd._Cache(0x1004, 0x1000, 0x1000, 0x1000), _step(), 0x1000, 0),   # misaligned state
        (Bd._Cache(0x1000, None, 0x1000, 0x1000), _step(), 0x1000, 0),     # missing ring
        (good, _step(row=100), 0x1000, 0),                                  # short qkv row
        (good, _step(batch=-1), 0x1000, 0),                                 # negative batch
        (good, _step(), None, 0),                                           # no write_pos
        (good, _step(), 0x1000, 5),                                         # unknown recon
        (good, _step(flags=4), 0x1000, 0),                                  # unknown step flag
    ]
    for cache, step, wp, recon in calls:
        st = lib.gdn_replayssm_decode(ctypes.byref(d), ctypes.byref(cache), wp, None, ctypes.byref(step),
                                      recon, None, None, None)
        assert st == 1, lib.gdn_last_error().decode()
        assert lib.gdn_last_error().decode() != ""


def test_empty_calls_are_no_ops(lib):
    d = _desc()
    cache = Bd._Cache(0x1000, 0x1000, 0x1000, 0x1000)
    assert lib.gdn_replayssm_decode(ctypes.byref(d), ctypes.byref(cache), 0x1000, None,
                                    ctypes.byref(_step(batch=0)), 0, None, None, None) == 0
    assert lib.gdn_replayssm_advance(None, 0, None, 8, 16, None, None, None) == 0
    assert lib.gdn_replayssm_flush(ctypes.byref(d), ctypes.byref(cache), None, None, 0, None, None) == 0
    assert lib.gdn_replayssm_reset_slots(0x1000, 8, None, 0, None, None) == 0
    assert lib.gdn_replayssm_advance(None, 4, None, 8, 16, None, None, None) == 1
    assert lib.gdn_replayssm_reset_slots(None, 8, 0x1000, 3, None, None) == 1


def test_status_strings(lib):
    assert lib.gdn_status_str(0).decode() == "ok"
    assert "invalid" in lib.gdn_status_str(1).decode()


def test_decode_advance_checks_its_workspace(lib):
    d = _desc()
    cache = Bd._Cache(0x1000, 0x1000, 0x1000, 0x1000)
    f = lib.gdn_replayssm_decode_advance
    # no workspace, misaligned workspace, no write_pos, unknown recon: rejected before any launch
    for wp, ws, recon in ((0x1000, None, 0), (0x1000, 0x1002, 0), (None, 0x1000, 0), (0x1000, 0x1000, 9)):
        assert f(ctypes.byref(d), ctypes.byref(cache), wp, None, ctypes.byref(_step()), recon, None, ws,
                 None, None) == 1, lib.gdn_last_error().decode()
    assert f(ctypes.byref(_desc(k_dim=96, v_dim=96)), ctypes.byref(cache), 0x1000, None, ctypes.byref(_step()),
             0, None, 0x1000, None, None) == 2
    assert f(ctypes.byref(d), ctypes.byref(cache), 0x1000, None, ctypes.byref(_step(batch=0)), 0, None, 0x1000,
             None, None) == 0


def test_workspace_size_constant_matches_the_header():
    text = open(os.path.join(ROOT, "include", "gdnreplay.h")).read()
    m = re.search(r"#define GDN_DECODE_ADVANCE_WORKSPACE_BYTES (\d+)", text)
    assert m and int(m.group(1)) == Bd.DECODE_ADVANCE_WORKSPACE_BYTES


def _spec_step(batch=4, window=3, row=2 * 16 * 128 + 32 * 128):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: every case below fails a host check
    return Bd._SpecStep(fake, Bd.BF16, row, fake, fake, fake, batch, window, 1.0, 0, fake, Bd.F32)


def test_spec_verify_and_commit_check_their_arguments(lib):
    d = _desc()
    cache = Bd._Cache(0x1000, 0x1000, 0x1000, 0x1000)
    v = lib.gdn_replayssm_spec_verify
    # window 0, window = ring_len, short row, negative batch, no write_pos: rejected before any launch
    for step, wp in ((_spec_step(window=0), 0x1000), (_spec_step(window=16), 0x1000),
                     (_spec_step(row=100), 0x1000), (_spec_step(batch=-1), 0x1000), (_spec_step(), None)):
        assert v(ctypes.byref(d), ctypes.byref(cache), wp, ctypes.byref(step), 0, None, None) == 1, \
            lib.gdn_last_error().decode()
    assert v(ctypes.byref(d), ctypes.byref(cache), 0x1000, ctypes.byref(_spec_step()), 7, None, None) == 1
    assert v(ctypes.byref(_desc(ring_len=64)), ctypes.byref(cache), 0x1000, ctypes.byref(_spec_step(window=33)),
             0, None, None) == 2
    assert v(ctypes.byref(d), ctypes.byref(cache), 0x1000, ctypes.byref(_spec_step(batch=0)), 0, None, None) == 0
    c = lib.gdn_replayssm_spec_commit
    assert c(None, None, 0, 3, 8, 16, None, None, None, None) == 0           # empty
    assert c(0x1000, 0x1000, 4, 3, 8, 16, 0x1000, None, None, None) == 1     # no flush_slots
    assert c(0x1000, 0x1000, 4, 16, 8, 16, 0x1000, 0x1000, None, None) == 1  # window does not fit the ring
    assert c(0x1000, 0x1000, 4, 3, 8, 1, 0x1000, 0x1000, None, None) == 1    # ring of one entry


def test_status_bits_match_the_header():
    text = open(os.path.join(ROOT, "include", "gdnreplay.h")).read()
    bits = {n: int(v) for n, v in re.findall(r"#define GDN_(DEV_\w+)\s+(\d+)u", text)}
    for n in ("DEV_BAD_SLOT", "DEV_BAD_WRITE_POS", "DEV_TIMEOUT", "DEV_INTERNAL", "DEV_BAD_ACCEPTED"):
        assert bits[n] == getattr(Bd, n), n


def test_lossless_verify_and_commit_check_their_arguments(lib):
    d = _desc()
    v = lib.gdn_lossless_verify
    # window 0, window 33, short row, negative batch, no state, misaligned state, no tuples:
    # rejected before any launch
    cases = ((_spec_step(window=0), 0x1000, 0x1000, 1), (_spec_step(window=33), 0x1000, 0x1000, 2),
             (_spec_step(row=100), 0x1000, 0x1000, 1), (_spec_step(batch=-1), 0x1000, 0x1000, 1),
             (_spec_step(), None, 0x1000, 1), (_spec_step(), 0x1004, 0x1000, 1), (_spec_step(), 0x1000, None, 1))
    for step, state, tup, code in cases:
        assert v(ctypes.byref(d), state, ctypes.byref(step), tup, 0x1000, 0x1000, None, None) == code, \
            lib.gdn_last_error().decode()
    # the lossless path keeps no ring: a window longer than ring_len is fine (checked, not launched: batch 0)
    assert v(ctypes.byref(_desc(ring_len=1)), 0x1000, ctypes.byref(_spec_step(batch=0, window=8)),
             0x1000, 0x1000, 0x1000, None, None) == 0
    c = lib.gdn_lossless_commit
    assert c(ctypes.byref(d), None, None, None, None, 0, 4, None, None, None, None, None) == 0   # empty
    assert c(ctypes.byref(d), 0x1000, 0x1000, None, None, 4, 4, 0x1000, 0x1000, 0x1000, None, None) == 1  # no accepted
    assert c(ctypes.byref(d), 0x1000, 0x1000, None, 0x1000, 4, 0, 0x1000, 0x1000, 0x1000, None, None) == 1  # window 0
    assert c(ctypes.byref(d), 0x1000, 0x1000, None, 0x1000, 4, 33, 0x1000, 0x1000, 0x1000, None, None) == 2
    assert c(ctypes.byref(d), 0x1008, 0x1000, None, 0x1000, 4, 4, 0x1000, 0x1000, 0x1000, None, None) == 1  # misaligned
    assert c(ctypes.byref(_desc(num_k_heads=5)), 0x1000, 0x1000, None, 0x1000, 4, 4, 0x1000, 0x1000, 0x1000,
             None, None) == 1


def test_wait_selftest_checks_its_arguments(lib):
    f = lib.gdn_selftest_wait_timeout
    assert f(None, 10, None) == 1         # no status word
    assert f(0x1000, 0, None) == 1        # limit below 1 us
    assert f(0x1000, 100001, None) == 1   # limit above 100 ms


def test_step_flag_constants_match_the_header():
    text = open(os.path.join(ROOT, "include", "gdnreplay.h")).read()
    m = re.search(r"#define GDN_STEP_OVERLAP_PREVIOUS\s+(\d+)u", text)
    assert m and int(m.group(1)) == Bd.STEP_OVERLAP_PREVIOUS
    m = re.search(r"#define GDN_STEP_PERSISTENT_KERNEL\s+(\d+)u", text)
    assert m and int(m.group(1)) == Bd.STEP_PERSISTENT_KERNEL
    m = re.search(r"#define GDN_STEP_KNOWN_FLAGS\s+(\d+)u", text)
    assert m and int(m.group(1)) == Bd.STEP_OVERLAP_PREVIOUS | Bd.STEP_PERSISTENT_KERNEL
    for name, val in (("PERSISTENT_TC", Bd.KERNEL_PERSISTENT_TC), ("PER_HEAD_TC", Bd.KERNEL_PER_HEAD_TC),
                      ("CUDA_CORE", Bd.KERNEL_CUDA_CORE), ("SMALL_BATCH", Bd.KERNEL_SMALL_BATCH)):
        m = re.search(r"#define GDN_KERNEL_%s\s+(\d+)" % name, text)
        assert m and int(m.group(1)) == val


def test_scratch_peek_checks_its_arguments(lib):
    buf = (ctypes.c_uint32 * 64)()
    for n in (0, -1, 65):
        assert lib.gdn_noalloc_scratch_peek(ctypes.cast(buf, ctypes.c_void_p), n) == 1
    assert lib.gdn_noalloc_scratch_peek(None, 1) == 1


def test_decode_kernel_query_checks_arguments_and_reports_cuda_core_recons(lib):
    d = _desc()
    cache = Bd._Cache(0x1000, 0x1000, 0x1000, 0x1000)
    out = ctypes.c_int32(-1)
    f = lib.gdn_replayssm_decode_kernel
    assert f(ctypes.byref(d), ctypes.byref(cache), ctypes.byref(_step()), 0, None) == 1
    assert f(ctypes.byref(d), ctypes.byref(cache), ctypes.byref(_step()), 7, ctypes.byref(out)) == 1
    assert f(ctypes.byref(_desc(k_dim=96, v_dim=96)), ctypes.byref(cache), ctypes.byref(_step()), 0,
             ctypes.byref(out)) == 2
    for recon in (Bd.RECON_FFMA, Bd.RECON_OUTPUT):  # decided without looking at the device
        assert f(ctypes.byref(d), ctypes.byref(cache), ctypes.byref(_step()), recon, ctypes.byref(out)) == 0
        assert out.value == Bd.KERNEL_CUDA_CORE
