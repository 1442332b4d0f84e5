"""GPU parity of decode on a bf16-state pool against the oracle.

Contract (one step from a stored bf16 state): the output o, read from the
unrounded new state, within normwise relative error 1e-4 of the oracle's
float64 step; the stored new state within one bf16 spacing of the oracle's
float64 step rounded to bf16 (the float32 and float64 results round to
different neighbours only when they straddle a rounding boundary), plus the
float32 arithmetic error of the step (2^-18 of the head's largest state
entry, which matters only where an entry nearly cancels), with at least 99% of
the elements identical.  Over many steps the bf16 state drifts
from the float32 recurrence; that drift is reported against the unrounded
oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import check_bf16_state_step, dev_inputs, host_inputs, i32, rel
from rwkv_wkv_gb300 import DEV_BAD_SLOT, Pool

pytestmark = pytest.mark.gpu

W = wl.DECODE_12L  # 12 layers x 12 heads x 64, 1024-slot pool
B = 256


_check_step = check_bf16_state_step


@pytest.fixture(scope="module")
def setup():
    slots = wl.distinct_slots(W.seed, "bf16state/slots", B, W.n_slots)
    S0 = oracle.round_bf16(wl.slot_states(W.seed, "bf16state/state", slots, 2, W.H, W.N))
    ins = [wl.token_inputs(W.seed, f"bf16state/step{t}", B, W.H, W.N, dtype="bf16")
           for t in range(4)]
    return slots, S0, ins


def _pool_with(slots, S0, n_layers=2):
    pool = Pool(n_layers, W.H, W.n_slots, state_dtype="bf16")
    pool.states.fill_(7.0)  # inactive slots: sentinel
    pool.states[torch.as_tensor(slots, dtype=torch.long)] = torch.from_numpy(S0).cuda().to(torch.bfloat16)
    return pool


def test_single_step_parity(setup):
    slots, S0, ins = setup
    with _pool_with(slots, S0) as pool:
        ids = i32(slots)
        o = pool.decode_step(1, ids, *dev_inputs(ins[0], "bf16")).cpu().numpy()
        assert pool.device_status() == 0
        S_gpu = pool.states[torch.as_tensor(slots, dtype=torch.long), 1].double().cpu().numpy()
        inactive = np.setdiff1d(np.arange(W.n_slots), slots)
        assert bool((pool.states[torch.as_tensor(inactive, dtype=torch.long)] == 7.0).all())
        S_l0 = pool.states[torch.as_tensor(slots, dtype=torch.long), 0].double().cpu().numpy()
    assert np.array_equal(S_l0, S0[:, 0])  # the other layer is untouched
    o_ref, S_ref = oracle.decode_step_bf16_state(S0[:, 1], *host_inputs(ins[0]), n_threads=8)
    _check_step(o, S_gpu, o_ref, S_ref)


def test_float32_inputs():
    slots = wl.distinct_slots(W.seed, "bf16state/f32slots", 32, W.n_slots)
    S0 = oracle.round_bf16(wl.slot_states(W.seed, "bf16state/f32state", slots, 1, W.H, W.N))
    x = wl.token_inputs(W.seed, "bf16state/f32in", 32, W.H, W.N, dtype="f32")
    with _pool_with(slots, S0, n_layers=1) as pool:
        o = pool.decode_step(0, i32(slots), *dev_inputs(x, "f32")).cpu().numpy()
        S_gpu = pool.states[torch.as_tensor(slots, dtype=torch.long), 0].double().cpu().numpy()
        assert pool.device_status() == 0
    o_ref, S_ref = oracle.decode_step_bf16_state(S0[:, 0], *host_inputs(x), n_threads=8)
    _check_step(o, S_gpu, o_ref, S_ref)


def test_every_step_of_a_run_and_the_drift(setup):
    """Each of four steps meets the one-step contract from the GPU's own stored
    state; after them the bf16 state stays close to the unrounded recurrence."""
    slots, S0, ins = setup
    S_exact = S0[:, 1].copy()
    with _pool_with(slots, S0) as pool:
        ids = i32(slots)
        sel = torch.as_tensor(slots, dtype=torch.long)
        for x in ins:
            S_prev = pool.states[sel, 1].double().cpu().numpy()
            o = pool.decode_step(1, ids, *dev_inputs(x, "bf16")).cpu().numpy()
            S_gpu = pool.states[sel, 1].double().cpu().numpy()
            o_ref, S_ref = oracle.decode_step_bf16_state(S_prev, *host_inputs(x), n_threads=8)
            _check_step(o, S_gpu, o_ref, S_ref)
            _, S_exact = oracle.decode_step(S_exact, *host_inputs(x), n_threads=8)
        assert pool.device_status() == 0
    drift = rel(S_gpu, S_exact)
    assert drift < 1e-2, drift  # four bf16 roundings of a contracting state


def test_batch_order_invariance(setup):
    slots, S0, ins = setup
    perm = np.random.default_rng(1).permutation(B)
    res = []
    for order in (np.arange(B), perm):
        with _pool_with(slots, S0) as pool:
            x = {k: v[order] for k, v in ins[0].items()}
            o = pool.decode_step(1, i32(np.asarray(slots)[order]), *dev_inputs(x, "bf16"))
            inv = np.argsort(order)
            res.append((o.cpu()[inv], pool.states.cpu()))
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])


def test_verbs_on_a_bf16_pool():
    with Pool(2, 4, 8, n_snapshots=2, state_dtype="bf16") as pool:
        g = torch.Generator(device="cuda").manual_seed(5)
        pool.states.copy_(torch.randn(pool.states.shape, generator=g, device="cuda").to(torch.bfloat16))
        before = pool.states.clone()
        assert pool.slot_bytes == 2 * 4 * 64 * 64 * 2
        pool.snapshot(i32([1, 2]), i32([0, 1]))
        pool.fork(i32([1]), i32([6]))
        assert torch.equal(pool.snapshots[0], before[1]) and torch.equal(pool.states[6], before[1])
        host = torch.empty(2 * pool.slot_bytes, dtype=torch.uint8, pin_memory=True)
        pool.hibernate(i32([3, 4]), host)
        pool.states[3] = 0
        pool.resume(host, i32([3, 4]))
        assert torch.equal(pool.states[3], before[3])
        pool.reset(i32([5]))
        assert bool((pool.states[5] == 0).all())
        pool.decode_step(0, i32([0, 9]), *[torch.zeros(2, 4, 64, dtype=torch.bfloat16, device="cuda")] * 6)
        assert pool.device_status() == DEV_BAD_SLOT
