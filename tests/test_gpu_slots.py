"""Slot verbs on the GPU: create zeroes, snapshot/restore/fork copy bit for bit,
and a run that is snapshotted, disturbed and restored continues bit-identically
to an uninterrupted run."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_helpers import dev_inputs, i32
from rwkv_wkv_gb300 import DEV_BAD_SLOT, Pool

pytestmark = pytest.mark.gpu

L, H, N = 2, 4, 64


def _fill_random(pool, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    pool.states.normal_(0.0, 0.1, generator=g)
    if pool.n_snapshots:
        pool.snapshots.normal_(0.0, 0.1, generator=g)


def test_create_zeroes_only_the_new_slots():
    with Pool(L, H, 16) as pool:
        _fill_random(pool)
        before = pool.states.clone()
        ids = pool.create(5)
        assert pool.device_status() == 0
        for s in range(16):
            if s in ids:
                assert bool((pool.states[s] == 0).all())
            else:
                assert torch.equal(pool.states[s], before[s])
        assert pool.n_free() == 11


def test_snapshot_restore_fork_are_bit_exact():
    with Pool(L, H, 16, n_snapshots=8) as pool:
        _fill_random(pool, 1)
        before = pool.states.clone()
        src = pool.alloc(6)
        snaps = pool.snapshot_alloc(6)
        pool.snapshot(i32(src), i32(snaps))
        for s, p in zip(src, snaps):
            assert torch.equal(pool.snapshots[p], before[s])
        dst = pool.alloc(6)
        pool.fork(i32(src), i32(dst))
        for s, d in zip(src, dst):
            assert torch.equal(pool.states[d], before[s])
        pool.states[src[0]].fill_(9.0)
        pool.restore(i32(snaps[:1]), i32(src[:1]))
        assert torch.equal(pool.states[src[0]], before[src[0]])
        untouched = [s for s in range(16) if s not in dst]
        assert torch.equal(pool.states[untouched], before[untouched])
        assert pool.device_status() == 0


def test_out_of_range_ids_are_flagged_and_skipped():
    with Pool(1, H, 8, n_snapshots=2) as pool:
        _fill_random(pool, 2)
        before = pool.states.clone()
        pool.fork(i32([1, 2]), i32([3, 40]))
        assert pool.device_status() == DEV_BAD_SLOT
        assert torch.equal(pool.states[3], before[1])
        assert torch.equal(pool.states[[0, 1, 2, 4, 5, 6, 7]], before[[0, 1, 2, 4, 5, 6, 7]])
        pool.snapshot(i32([0]), i32([5]))
        assert pool.device_status() == DEV_BAD_SLOT
        pool.reset(i32([-1, 6]))
        assert pool.device_status() == DEV_BAD_SLOT
        assert bool((pool.states[6] == 0).all())


def test_fork_then_identical_inputs_give_identical_states():
    ins = wl.token_inputs(3, "fork", 2, H, N, dtype="bf16")
    with Pool(1, H, 8) as pool:
        _fill_random(pool, 3)
        pool.fork(i32([2]), i32([5]))
        step = {k: np.concatenate([v[:1], v[:1]]) for k, v in ins.items()}
        o = pool.decode_step(0, i32([2, 5]), *dev_inputs(step, "bf16"))
        assert torch.equal(o[0], o[1])
        assert torch.equal(pool.states[2], pool.states[5])


def test_restore_undoes_a_step_exactly():
    ins = wl.token_inputs(4, "undo", 3, H, N, dtype="bf16")
    with Pool(1, H, 8, n_snapshots=3) as pool:
        _fill_random(pool, 4)
        before = pool.states.clone()
        pool.snapshot(i32([0, 3, 6]), i32([0, 1, 2]))
        pool.decode_step(0, i32([0, 3, 6]), *dev_inputs(ins, "bf16"))
        assert not torch.equal(pool.states[3], before[3])
        pool.restore(i32([0, 1, 2]), i32([0, 3, 6]))
        assert torch.equal(pool.states, before)


@pytest.mark.parametrize("sequential", [False, True])
def test_snapshot_and_resume_is_bit_identical(sequential):
    """Run A: prefill 200 tokens, then 5 decode steps.  Run B: the same prefill,
    snapshot, 3 decode steps with other inputs and a fork over the slot,
    restore, then the same 5 decode steps.  Outputs and states are equal bit
    for bit."""
    pre = wl.token_inputs(6, "resume/prefill", 200, H, N, dtype="bf16")
    steps = [wl.token_inputs(6, f"resume/step{i}", 1, H, N, dtype="bf16") for i in range(5)]
    noise = [wl.token_inputs(6, f"resume/noise{i}", 1, H, N, dtype="bf16") for i in range(3)]
    cu = i32([0, 200])

    def run(disturb):
        with Pool(1, H, 4, n_snapshots=1) as pool:
            slot = pool.create(1)
            ids = i32(slot)
            pool.prefill(0, ids, cu, *dev_inputs(pre, "bf16"), max_seqlen=200,
                         sequential=sequential)
            if disturb:
                pool.snapshot(ids, i32([0]))
                for x in noise:
                    pool.decode_step(0, ids, *dev_inputs(x, "bf16"))
                other = pool.create(1)
                pool.fork(i32(other), ids)
                pool.restore(i32([0]), ids)
            outs = [pool.decode_step(0, ids, *dev_inputs(x, "bf16")).clone() for x in steps]
            assert pool.device_status() == 0
            return torch.stack(outs).cpu(), pool.states[slot[0]].cpu()

    oa, sa = run(False)
    ob, sb = run(True)
    assert torch.equal(oa, ob)
    assert torch.equal(sa, sb)


def test_verbs_past_one_launch():
    """More ids than one launch covers: create zeroes from host ids 512 at a time,
    fork and reset take device ids 65535 per launch."""
    n, half = 140000, 70000
    with Pool(1, 1, n) as pool:
        _fill_random(pool, 7)
        before = pool.states.clone()
        created = pool.create(600)
        assert pool.device_status() == 0
        c = torch.as_tensor(created, dtype=torch.long, device="cuda")
        assert bool((pool.states[c] == 0).all())
        others = torch.ones(n, dtype=torch.bool, device="cuda")
        others[c] = False
        assert torch.equal(pool.states[others], before[others])

        perm = torch.as_tensor(np.random.default_rng(3).permutation(n).astype(np.int32), device="cuda")
        src, dst = perm[:half], perm[half:]
        mid = pool.states.clone()
        pool.fork(src, dst)
        assert pool.device_status() == 0
        assert torch.equal(pool.states[dst.long()], mid[src.long()])
        assert torch.equal(pool.states[src.long()], mid[src.long()])

        pool.reset(dst)
        assert pool.device_status() == 0
        assert bool((pool.states[dst.long()] == 0).all())
        assert torch.equal(pool.states[src.long()], mid[src.long()])
