"""Hibernate and resume on the GPU: slots go to pinned host memory and come back
bit for bit, into the same or other slots, through the C-ABI; a run that is
hibernated, disturbed and resumed continues bit-identically; bad ids are
flagged and skipped; host memory that the device cannot address is refused
before any launch."""
import ctypes

import pytest
import torch

import workloads as wl
from gpu_helpers import dev_inputs, i32
from rwkv_wkv_gb300 import DEV_BAD_SLOT, Pool, Wkv7Error

pytestmark = pytest.mark.gpu

L, H, N = 2, 4, 64


def _fill_random(pool, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    pool.states.normal_(0.0, 0.1, generator=g)


def _pinned(n_slots, pool, fill=0):
    host = torch.empty(n_slots * pool.slot_bytes, dtype=torch.uint8, pin_memory=True)
    host.fill_(fill)
    return host


def test_hibernate_then_resume_is_bit_exact():
    with Pool(L, H, 16) as pool:
        _fill_random(pool, 11)
        before = pool.states.clone()
        ids = [13, 2, 7, 0, 9]
        host = _pinned(len(ids), pool, fill=0xAB)
        pool.hibernate(i32(ids), host)
        torch.cuda.synchronize()
        packed = host.view(torch.float32).view(len(ids), L, H, N, N)
        assert torch.equal(packed, before[ids].cpu())  # packed in call order
        pool.states[ids] = 5.0  # the slots are reused meanwhile
        pool.resume(host, i32(ids))
        assert torch.equal(pool.states, before)
        assert pool.device_status() == 0


def test_resume_into_other_slots_and_partial_buffers():
    with Pool(L, H, 16) as pool:
        _fill_random(pool, 12)
        before = pool.states.clone()
        host = _pinned(6, pool)  # larger than needed
        pool.hibernate(i32([1, 4, 5]), host)
        pool.resume(host, i32([10, 11, 12]))  # a migration through host memory
        for s, d in zip([1, 4, 5], [10, 11, 12]):
            assert torch.equal(pool.states[d], before[s])
        untouched = [s for s in range(16) if s not in (10, 11, 12)]
        assert torch.equal(pool.states[untouched], before[untouched])
        # resume only the first image
        pool.states[3] = 0.0
        pool.resume(host, i32([3]))
        assert torch.equal(pool.states[3], before[1])
        assert pool.device_status() == 0


def test_hibernated_run_continues_bit_identically():
    """Run A: 4 decode steps.  Run B: 2 steps, hibernate, 2 steps with other inputs
    on the same slot, resume, then the same last 2 steps.  Outputs and states
    of the last 2 steps are equal bit for bit."""
    steps = [wl.token_inputs(21, f"hib/step{i}", 3, H, N, dtype="bf16") for i in range(4)]
    noise = [wl.token_inputs(21, f"hib/noise{i}", 3, H, N, dtype="bf16") for i in range(2)]

    def run(disturb):
        with Pool(1, H, 8) as pool:
            _fill_random(pool, 13)
            ids = i32([6, 1, 4])
            for x in steps[:2]:
                pool.decode_step(0, ids, *dev_inputs(x, "bf16"))
            if disturb:
                host = _pinned(3, pool)
                pool.hibernate(ids, host)
                for x in noise:
                    pool.decode_step(0, ids, *dev_inputs(x, "bf16"))
                pool.resume(host, ids)
            outs = [pool.decode_step(0, ids, *dev_inputs(x, "bf16")).clone() for x in steps[2:]]
            assert pool.device_status() == 0
            return torch.stack(outs).cpu(), pool.states.cpu()

    oa, sa = run(False)
    ob, sb = run(True)
    assert torch.equal(oa, ob)
    assert torch.equal(sa, sb)


def test_out_of_range_ids_are_flagged_and_skipped():
    with Pool(1, H, 8) as pool:
        _fill_random(pool, 14)
        before = pool.states.clone()
        host = _pinned(2, pool, fill=0)
        pool.hibernate(i32([3, 8]), host)
        assert pool.device_status() == DEV_BAD_SLOT
        packed = host.view(torch.float32).view(2, 1, H, N, N)
        assert torch.equal(packed[0], before[3].cpu())
        assert bool((packed[1] == 0).all())  # the bad id's image is not written
        pool.resume(host, i32([-1, 5]))
        assert pool.device_status() == DEV_BAD_SLOT
        assert torch.equal(pool.states[5], packed[1].cuda())
        assert torch.equal(pool.states[[0, 1, 2, 3, 4, 6, 7]], before[[0, 1, 2, 3, 4, 6, 7]])


def test_memory_the_device_cannot_address_is_refused():
    with Pool(1, H, 8) as pool:
        _fill_random(pool, 15)
        before = pool.states.clone()
        pageable = torch.empty(2 * pool.slot_bytes, dtype=torch.uint8)  # not page-locked
        with pytest.raises(Wkv7Error) as err:
            pool.hibernate(i32([0, 1]), pageable)
        assert err.value.name == "ERR_INVALID_ARG"
        with pytest.raises(Wkv7Error):
            pool.resume(pageable, i32([0, 1]))
        host = _pinned(2, pool)
        lib = pool._lib
        ids = i32([0, 1])
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        # too small for two slots; misaligned by 4 bytes
        assert lib.wkv7_slot_hibernate(pool._h, ids.data_ptr(), 2, host.data_ptr(),
                                       2 * pool.slot_bytes - 1, stream) == 1
        assert lib.wkv7_slot_hibernate(pool._h, ids.data_ptr(), 1, host.data_ptr() + 4,
                                       pool.slot_bytes, stream) == 1
        assert lib.wkv7_slot_resume(pool._h, host.data_ptr() + 4, pool.slot_bytes,
                                    ids.data_ptr(), 1, stream) == 1
        torch.cuda.synchronize()
        assert torch.equal(pool.states, before)
        assert pool.device_status() == 0
