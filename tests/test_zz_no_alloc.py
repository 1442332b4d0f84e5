"""GPU: the allocation-free id check (wkv7_validate_ids_noalloc) against the
pool-based one (wkv7_validate_ids).

Some callers cannot allocate device memory at all -- their device memory is
already handed out to another allocator, or their serving loop forbids
allocation once it runs -- so the library offers one check whose scratch is a
static array built into the library.  This file is collected last, so that a
run stopping at its first failure has run every other test before it; it also
passes alone in a fresh process (its first call does the per-device set-up).

Every case is run twice in a row through the C-ABI: the second call must see
the array cleared by the call itself, not the first call's marks.  The verdict
is an integer code, compared exactly with the pool-based pass's.
"""
import ctypes

import numpy as np
import pytest
import torch

from rwkv_wkv_gb300 import DEV_BAD_SLOT, DEV_DUP_SLOT, Pool, load_library

pytestmark = pytest.mark.gpu

N_TABLE = 4096


def _cases():
    perm = np.random.default_rng(21).permutation(N_TABLE)
    dec, pre = perm[:1024], perm[1024:1088]
    dup = dec.copy()
    dup[-1] = dup[7]
    over = pre.copy()
    over[3] = dec[900]
    return [("clean", dec, pre, 0), ("repeat", dup, None, DEV_DUP_SLOT),
            ("overlap", dec, over, DEV_DUP_SLOT), ("range", np.array([1, N_TABLE]), None, DEV_BAD_SLOT),
            ("clean again", dec, pre, 0), ("every id once", perm, None, 0)]


def _dev(x):
    return None if x is None else torch.as_tensor(np.asarray(x, dtype=np.int32), device="cuda")


def test_no_alloc_check_matches_the_pool_check():
    lib = load_library()
    stream = torch.cuda.current_stream().cuda_stream
    result = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    with Pool(1, 1, N_TABLE) as pool:
        for name, a, b, want in _cases():
            ta, tb = _dev(a), _dev(b)
            na, nb = ta.numel(), 0 if tb is None else tb.numel()
            pa, pb = ta.data_ptr(), None if tb is None else tb.data_ptr()
            # the existing entry point, through its pool's status word
            assert lib.wkv7_validate_ids(pool._h, 0, pa, na, pb, nb, stream) == 0
            ref = pool.device_status()
            assert ref == want, name
            for call in range(2):  # two calls in a row
                result.fill_(-1)
                st = lib.wkv7_validate_ids_noalloc(N_TABLE, pa, na, pb, nb, result.data_ptr(), stream)
                assert st == 0, (name, call, st)
                torch.cuda.synchronize()
                assert int(result.item()) == ref, (name, call)


def test_no_alloc_check_host_errors():
    lib = load_library()
    stream = torch.cuda.current_stream().cuda_stream
    result = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = _dev([0, 1])
    assert lib.wkv7_validate_ids_noalloc(-1, ids.data_ptr(), 2, None, 0, result.data_ptr(), stream) == 1
    assert lib.wkv7_validate_ids_noalloc(8, ids.data_ptr(), 2, None, 0, None, stream) == 1
    assert lib.wkv7_validate_ids_noalloc(8, None, 2, None, 0, result.data_ptr(), stream) == 1
    assert lib.wkv7_validate_ids_noalloc(8, ids.data_ptr(), 2, None, 1, result.data_ptr(), stream) == 1
    # above the built-in maximum of 2^20 ids: refused, nothing launched
    assert lib.wkv7_validate_ids_noalloc((1 << 20) + 1, ids.data_ptr(), 2, None, 0, result.data_ptr(),
                                         stream) == 7
    # at the maximum: accepted (the whole array is cleared); an empty list is clean
    result.fill_(-1)
    assert lib.wkv7_validate_ids_noalloc(1 << 20, ids.data_ptr(), 2, None, 0, result.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    assert int(result.item()) == 0
    result.fill_(-1)
    assert lib.wkv7_validate_ids_noalloc(0, None, 0, None, 0, result.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    assert int(result.item()) == 0
