"""GPU: the debug validation pass over device id arrays (wkv7_validate_ids).

It must report a repeated id (within one list, or shared by the two lists of a
mixed step: the decode and the prefill slot sets) as WKV7_DEV_DUP_SLOT and an id
outside the table as WKV7_DEV_BAD_SLOT, pass clean lists, and touch no state.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import i32
from rwkv_wkv_gb300 import DEV_BAD_SLOT, DEV_DUP_SLOT, Pool, load_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    with Pool(1, 2, 4096, n_snapshots=64) as p:
        g = torch.Generator(device="cuda").manual_seed(5)
        p.states.normal_(0.0, 0.1, generator=g)
        p.snapshots.normal_(0.0, 0.1, generator=g)
        yield p


def _mixed_step_ids(seed=4):
    perm = np.random.default_rng(seed).permutation(4096)
    return perm[:1024], perm[1024:1088]  # decode slots, prefill slots: disjoint


def test_clean_lists_pass_and_nothing_is_written(pool):
    before = pool.buffer.clone()
    dec, pre = _mixed_step_ids()
    pool.validate_ids(i32(dec), i32(pre))
    assert pool.device_status() == 0
    pool.validate_ids(i32(np.arange(64)), table="snapshots")
    assert pool.device_status() == 0
    pool.validate_ids(i32(np.arange(4096)))           # every id once
    assert pool.device_status() == 0
    n_state = (pool.n_slots + pool.n_snapshots) * pool.slot_bytes
    assert torch.equal(pool.buffer[256:256 + n_state], before[256:256 + n_state])


def test_repeat_within_one_list(pool):
    before = pool.states.clone()
    dec, _ = _mixed_step_ids()
    dup = dec.copy()
    dup[-1] = dup[3]
    pool.validate_ids(i32(dup))
    assert pool.device_status() == DEV_DUP_SLOT
    assert torch.equal(pool.states, before)
    pool.validate_ids(i32(dec))                       # the bitmap starts clean every call
    assert pool.device_status() == 0


def test_overlap_between_decode_and_prefill_sets(pool):
    dec, pre = _mixed_step_ids()
    pre = pre.copy()
    pre[10] = dec[500]
    pool.validate_ids(i32(dec), i32(pre))
    assert pool.device_status() == DEV_DUP_SLOT
    pool.validate_ids(i32(pre), i32(dec))             # either order
    assert pool.device_status() == DEV_DUP_SLOT


def test_out_of_range_ids(pool):
    pool.validate_ids(i32([0, 1, 4096]))
    assert pool.device_status() == DEV_BAD_SLOT
    pool.validate_ids(i32([-1]))
    assert pool.device_status() == DEV_BAD_SLOT
    pool.validate_ids(i32([5, 64]), table="snapshots")  # snapshot table holds 64
    assert pool.device_status() == DEV_BAD_SLOT
    pool.validate_ids(i32([5, 63]), table="snapshots")
    assert pool.device_status() == 0


def test_many_ids_one_repeat_far_apart():
    """70,000 slots: a permutation passes; the same list with its first id
    repeated at the end is caught (the ids span thousands of bitmap words and
    several CTAs)."""
    n = 70000
    with Pool(1, 1, n) as p:
        perm = np.random.default_rng(9).permutation(n)
        p.validate_ids(i32(perm))
        assert p.device_status() == 0
        bad = np.concatenate([perm, perm[:1]])
        p.validate_ids(i32(bad[: n // 2]), i32(bad[n // 2:]))
        assert p.device_status() == DEV_DUP_SLOT


def test_status_call_returns_the_dup_error():
    """Through the C-ABI: wkv7_get_device_status returns WKV7_ERR_DUP_SLOT (3) with
    the code WKV7_DEV_DUP_SLOT, and clears the word."""
    lib = load_library()
    with Pool(1, 1, 16) as p:
        ids = i32([1, 2, 3, 2])
        stream = torch.cuda.current_stream().cuda_stream
        assert lib.wkv7_validate_ids(p._h, 0, ids.data_ptr(), 4, None, 0, stream) == 0
        code = ctypes.c_int32(-1)
        assert lib.wkv7_get_device_status(p._h, stream, 10000, ctypes.byref(code)) == 3
        assert code.value == DEV_DUP_SLOT
        assert lib.wkv7_get_device_status(p._h, stream, 10000, ctypes.byref(code)) == 0
        assert code.value == 0
