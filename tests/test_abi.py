"""The C-ABI boundary without a GPU: the library builds and loads, exports every
function include/wkv7.h declares, and its host-side logic (slot table,
argument checks that return before any launch) behaves as documented.

A pool created over a caller-supplied buffer makes no CUDA call, so these
tests give it a fake, never-dereferenced device address.
"""
import ctypes
import os
import re

import pytest

from rwkv_wkv_gb300 import build as wbuild
from rwkv_wkv_gb300 import wkv7

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE_DEVICE_ADDR = 0x7F0000000000  # 256-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    wbuild.build()
    return wkv7.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "wkv7.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(wkv7_[a-z0-9_]+)\s*\(", src)))


def test_header_declarations_are_all_exported(lib):
    declared = _declared_functions()
    assert len(declared) >= 25
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in wkv7.h but not exported"
    assert set(declared) == set(wkv7.exported_symbols())


def test_wait_timeout_test_hook_is_host_only(lib):
    """The bounded-wait test hook only sets a process-wide flag (no CUDA call)."""
    assert lib.wkv7_test_force_wait_timeout(1) == 0
    assert lib.wkv7_test_force_wait_timeout(0) == 0


def test_version_and_strings(lib):
    assert lib.wkv7_version() == 1
    assert lib.wkv7_status_string(0) == b"ok"
    assert lib.wkv7_status_string(4) == b"not enough free slots"


def _desc(**kw):
    d = dict(n_layers=2, n_heads=3, head_size=64, n_slots=8, n_snapshots=4, state_dtype=0, out_dtype=0)
    d.update(kw)
    return wkv7.PoolDesc(d["n_layers"], d["n_heads"], d["head_size"], d["n_slots"],
                         d["n_snapshots"], None, 0, d["state_dtype"], d["out_dtype"])


def _fake_pool(lib, **kw):
    desc = _desc(**kw)
    nbytes = lib.wkv7_pool_required_bytes(ctypes.byref(desc))
    desc.device_buffer = FAKE_DEVICE_ADDR
    desc.buffer_bytes = nbytes
    h = ctypes.c_void_p()
    st = lib.wkv7_pool_create(ctypes.byref(desc), ctypes.byref(h))
    return st, h


def test_required_bytes(lib):
    d = _desc()
    # header + slots + snapshots + the validation bitmap (max(8, 4) bits -> 256 bytes)
    assert lib.wkv7_pool_required_bytes(ctypes.byref(d)) == 256 + (8 + 4) * 2 * 3 * 64 * 64 * 4 + 256
    big = _desc(n_slots=70000, n_snapshots=3)   # 70000 bits = 8750 bytes -> 8960
    assert (lib.wkv7_pool_required_bytes(ctypes.byref(big))
            == 256 + 70003 * 2 * 3 * 64 * 64 * 4 + 8960)
    bad = _desc(n_slots=0)
    assert lib.wkv7_pool_required_bytes(ctypes.byref(bad)) == 0


def test_create_rejects_bad_descriptions(lib):
    h = ctypes.c_void_p()
    d = _desc(head_size=32)
    d.device_buffer, d.buffer_bytes = FAKE_DEVICE_ADDR, 1 << 30
    assert lib.wkv7_pool_create(ctypes.byref(d), ctypes.byref(h)) == 7  # UNSUPPORTED
    d = _desc(n_layers=0)
    assert lib.wkv7_pool_create(ctypes.byref(d), ctypes.byref(h)) == 1
    d = _desc()
    d.device_buffer, d.buffer_bytes = FAKE_DEVICE_ADDR, 100  # too small
    assert lib.wkv7_pool_create(ctypes.byref(d), ctypes.byref(h)) == 1
    d = _desc()
    d.device_buffer, d.buffer_bytes = FAKE_DEVICE_ADDR + 16, 1 << 30  # misaligned
    assert lib.wkv7_pool_create(ctypes.byref(d), ctypes.byref(h)) == 1


def test_slot_table(lib):
    st, h = _fake_pool(lib)
    assert st == 0
    try:
        assert lib.wkv7_slot_count_free(h) == 8
        ids = (ctypes.c_int32 * 8)()
        assert lib.wkv7_slot_alloc(h, 5, ids) == 0
        got = list(ids[:5])
        assert len(set(got)) == 5 and all(0 <= i < 8 for i in got)
        assert lib.wkv7_slot_count_free(h) == 3
        assert lib.wkv7_slot_alloc(h, 4, ids) == 4          # POOL_FULL, all or nothing
        assert lib.wkv7_slot_count_free(h) == 3
        flag = ctypes.c_int32()
        assert lib.wkv7_slot_is_allocated(h, got[0], ctypes.byref(flag)) == 0 and flag.value == 1
        assert lib.wkv7_slot_is_allocated(h, 99, ctypes.byref(flag)) == 2
        dup = (ctypes.c_int32 * 2)(got[0], got[0])
        assert lib.wkv7_slot_free(h, 2, dup) == 3            # DUP_SLOT
        free_ids = [i for i in range(8) if i not in got]
        notalloc = (ctypes.c_int32 * 2)(got[0], free_ids[0])
        assert lib.wkv7_slot_free(h, 2, notalloc) == 2       # BAD_SLOT, nothing freed
        assert lib.wkv7_slot_count_free(h) == 3
        back = (ctypes.c_int32 * 2)(got[0], got[1])
        assert lib.wkv7_slot_free(h, 2, back) == 0
        assert lib.wkv7_slot_count_free(h) == 5
        assert lib.wkv7_slot_is_allocated(h, got[0], ctypes.byref(flag)) == 0 and flag.value == 0
        # snapshot ids are a separate table
        assert lib.wkv7_snapshot_count_free(h) == 4
        assert lib.wkv7_snapshot_alloc(h, 4, ids) == 0
        assert lib.wkv7_snapshot_alloc(h, 1, ids) == 4
    finally:
        assert lib.wkv7_pool_destroy(h) == 0


def test_state_pointers(lib):
    st, h = _fake_pool(lib)
    assert st == 0
    try:
        p = ctypes.c_void_p()
        assert lib.wkv7_pool_state_ptr(h, 0, 0, ctypes.byref(p)) == 0
        assert p.value == FAKE_DEVICE_ADDR + 256
        slot_bytes = lib.wkv7_slot_bytes(h)
        assert slot_bytes == 2 * 3 * 64 * 64 * 4
        assert lib.wkv7_pool_state_ptr(h, 3, 1, ctypes.byref(p)) == 0
        assert p.value == FAKE_DEVICE_ADDR + 256 + 3 * slot_bytes + 3 * 64 * 64 * 4
        assert lib.wkv7_pool_snapshot_ptr(h, 1, 0, ctypes.byref(p)) == 0
        assert p.value == FAKE_DEVICE_ADDR + 256 + (8 + 1) * slot_bytes
        assert lib.wkv7_pool_state_ptr(h, 8, 0, ctypes.byref(p)) == 2
        assert lib.wkv7_pool_state_ptr(h, 0, 2, ctypes.byref(p)) == 1
    finally:
        lib.wkv7_pool_destroy(h)


def test_host_checks_return_before_launch(lib):
    """Each call below has one host-checkable fault; it must be reported
    without reaching the GPU (there is none here)."""
    st, h = _fake_pool(lib)
    assert st == 0
    x = ctypes.c_void_p(FAKE_DEVICE_ADDR)
    ins = [x] * 6
    try:
        # decode: layer out of range, n > n_slots, NULL ids, bad dtype, n < 0
        assert lib.wkv7_decode_step(h, 2, x, 1, 1, *ins, x, None) == 1
        assert lib.wkv7_decode_step(h, 0, x, 9, 1, *ins, x, None) == 1
        assert lib.wkv7_decode_step(h, 0, None, 1, 1, *ins, x, None) == 1
        assert lib.wkv7_decode_step(h, 0, x, 1, 5, *ins, x, None) == 1
        assert lib.wkv7_decode_step(h, 0, x, -1, 1, *ins, x, None) == 1
        assert lib.wkv7_decode_step(h, 0, x, 1, 1, x, x, x, x, x, None, x, None) == 1
        assert lib.wkv7_decode_step(h, 0, x, 0, 1, *ins, x, None) == 0  # empty: no-op
        # prefill: the chunked path takes bf16 only; inconsistent sizes
        assert lib.wkv7_prefill(h, 0, x, x, 1, 10, 10, 0, *ins, x, None) == 7
        assert lib.wkv7_prefill(h, 0, x, x, 1, 10, 11, 1, *ins, x, None) == 5
        assert lib.wkv7_prefill(h, 0, x, None, 1, 10, 10, 1, *ins, x, None) == 1
        assert lib.wkv7_prefill(h, 0, x, x, 9, 10, 10, 1, *ins, x, None) == 1
        assert lib.wkv7_prefill(h, 0, x, x, 0, 0, 0, 1, *ins, x, None) == 0
        assert lib.wkv7_prefill_sequential(h, 3, x, x, 1, 10, 10, 0, *ins, x, None) == 1
        # every input base and o 16-byte aligned, on every recurrence call
        odd = ctypes.c_void_p(FAKE_DEVICE_ADDR + 8)
        for bad in range(7):
            args = [odd if i == bad else x for i in range(7)]
            assert lib.wkv7_decode_step(h, 0, x, 1, 1, *args, None) == 7
            assert lib.wkv7_decode_multi(h, 0, x, 1, 2, 1, *args, None, None) == 7
            assert lib.wkv7_prefill(h, 0, x, x, 1, 10, 10, 1, *args, None) == 7
            assert lib.wkv7_prefill_sequential(h, 0, x, x, 1, 10, 10, 0, *args, None) == 7
        assert lib.wkv7_prefill(h, 0, x, x, 0, 0, 0, 1, *ins, odd, None) == 0  # nothing to write
        # verbs
        assert lib.wkv7_slot_fork(h, None, x, 1, None) == 1
        assert lib.wkv7_slot_snapshot(h, x, x, -1, None) == 1
        assert lib.wkv7_slot_restore(h, x, x, 0, None) == 0
        assert lib.wkv7_slot_snapshot(h, x, x, 5, None) == 1  # more than the 4 snapshots
        assert lib.wkv7_slot_fork(h, x, x, 9, None) == 1       # more than the 8 slots
        # hibernate / resume: NULL ids or host buffer, n < 0, a host buffer too small
        sb = lib.wkv7_slot_bytes(h)
        assert lib.wkv7_slot_hibernate(h, None, 1, x, sb, None) == 1
        assert lib.wkv7_slot_hibernate(h, x, 1, None, sb, None) == 1
        assert lib.wkv7_slot_hibernate(h, x, -1, x, sb, None) == 1
        assert lib.wkv7_slot_hibernate(h, x, 2, x, 2 * sb - 1, None) == 1
        assert lib.wkv7_slot_hibernate(h, x, 0, None, 0, None) == 0  # empty: no-op
        assert lib.wkv7_slot_resume(h, None, sb, x, 1, None) == 1
        assert lib.wkv7_slot_resume(h, x, sb, None, 1, None) == 1
        assert lib.wkv7_slot_resume(h, x, sb - 16, x, 1, None) == 1
        assert lib.wkv7_slot_resume(h, x, 0, x, 0, None) == 0
        ids = (ctypes.c_int32 * 9)()
        assert lib.wkv7_slot_create(h, 9, ids, None) == 4     # POOL_FULL, nothing allocated
        assert lib.wkv7_slot_count_free(h) == 8
        assert lib.wkv7_get_device_status(h, None, 10, None) == 1
        # id validation: unknown table, negative counts, NULL arrays with ids; empty is a no-op
        assert lib.wkv7_validate_ids(h, 2, x, 1, None, 0, None) == 1
        assert lib.wkv7_validate_ids(h, 0, x, -1, None, 0, None) == 1
        assert lib.wkv7_validate_ids(h, 0, x, 1, x, -2, None) == 1
        assert lib.wkv7_validate_ids(h, 0, None, 1, None, 0, None) == 1
        assert lib.wkv7_validate_ids(h, 1, x, 0, None, 3, None) == 1
        assert lib.wkv7_validate_ids(None, 0, x, 1, None, 0, None) == 1
        assert lib.wkv7_validate_ids(h, 0, None, 0, None, 0, None) == 0
    finally:
        lib.wkv7_pool_destroy(h)


def test_snapshot_verbs_need_a_snapshot_store(lib):
    st, h = _fake_pool(lib, n_snapshots=0)
    assert st == 0
    x = ctypes.c_void_p(FAKE_DEVICE_ADDR)
    try:
        assert lib.wkv7_slot_snapshot(h, x, x, 1, None) == 1
        assert lib.wkv7_slot_restore(h, x, x, 1, None) == 1
    finally:
        lib.wkv7_pool_destroy(h)


def test_bf16_state_pool(lib):
    """A bf16-state pool: half the bytes per slot, state pointers step in bf16,
    and every call is offered."""
    d16 = _desc(state_dtype=1)
    d32 = _desc()
    body32 = lib.wkv7_pool_required_bytes(ctypes.byref(d32)) - 512   # header, bitmap
    assert lib.wkv7_pool_required_bytes(ctypes.byref(d16)) - 512 == body32 // 2
    assert lib.wkv7_pool_required_bytes(ctypes.byref(_desc(state_dtype=2))) == 0
    st, h = _fake_pool(lib, state_dtype=1)
    assert st == 0
    x = ctypes.c_void_p(FAKE_DEVICE_ADDR)
    ins = [x] * 6
    try:
        sb = lib.wkv7_slot_bytes(h)
        assert sb == 2 * 3 * 64 * 64 * 2
        p00, p21 = ctypes.c_void_p(), ctypes.c_void_p()
        assert lib.wkv7_pool_state_ptr(h, 0, 0, ctypes.byref(p00)) == 0
        assert lib.wkv7_pool_state_ptr(h, 2, 1, ctypes.byref(p21)) == 0
        assert p00.value == FAKE_DEVICE_ADDR + 256
        assert p21.value - p00.value == 2 * sb + 3 * 64 * 64 * 2
        # every recurrence call is offered (empty calls: no-ops) and host-checked as usual
        assert lib.wkv7_prefill(h, 0, x, x, 0, 0, 0, 1, *ins, x, None) == 0
        assert lib.wkv7_prefill_sequential(h, 0, x, x, 0, 0, 0, 1, *ins, x, None) == 0
        assert lib.wkv7_decode_multi(h, 0, x, 0, 2, 1, *ins, x, None, None) == 0
        assert lib.wkv7_decode_step(h, 0, x, 0, 1, *ins, x, None) == 0
        assert lib.wkv7_prefill(h, 2, x, x, 1, 10, 10, 1, *ins, x, None) == 1
        assert lib.wkv7_decode_multi(h, 0, x, 1, 0, 1, *ins, x, None, None) == 1
        desc = wkv7.PoolDesc()
        assert lib.wkv7_pool_get_desc(h, ctypes.byref(desc)) == 0 and desc.state_dtype == 1
    finally:
        lib.wkv7_pool_destroy(h)


def test_bf16_output_pool(lib):
    """out_dtype: float32 (0) or bf16 (1), nothing else; it changes no byte count
    and every recurrence call is offered on such a pool."""
    base = lib.wkv7_pool_required_bytes(ctypes.byref(_desc()))
    assert lib.wkv7_pool_required_bytes(ctypes.byref(_desc(out_dtype=1))) == base
    assert lib.wkv7_pool_required_bytes(ctypes.byref(_desc(out_dtype=2))) == 0
    assert lib.wkv7_pool_required_bytes(ctypes.byref(_desc(out_dtype=-1))) == 0
    st, h = _fake_pool(lib, out_dtype=1)
    assert st == 0
    x = ctypes.c_void_p(FAKE_DEVICE_ADDR)
    ins = [x] * 6
    try:
        assert lib.wkv7_prefill(h, 0, x, x, 0, 0, 0, 1, *ins, x, None) == 0
        assert lib.wkv7_decode_step(h, 0, x, 0, 1, *ins, x, None) == 0
        assert lib.wkv7_decode_multi(h, 0, x, 0, 2, 1, *ins, x, None, None) == 0
        # o is checked like every other base: missing -> INVALID_ARG, misaligned -> UNSUPPORTED
        assert lib.wkv7_decode_step(h, 0, x, 1, 1, *ins, None, None) == 1
        assert lib.wkv7_decode_step(h, 0, x, 1, 1, *ins, ctypes.c_void_p(FAKE_DEVICE_ADDR + 2), None) == 7
        desc = wkv7.PoolDesc()
        assert lib.wkv7_pool_get_desc(h, ctypes.byref(desc)) == 0 and desc.out_dtype == 1
    finally:
        lib.wkv7_pool_destroy(h)
