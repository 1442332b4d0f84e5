"""GPU parity of the batched decode step (wkv7_decode_step) against the oracle.

Tolerance: normwise-max relative error 1e-4 on outputs and states (float32
path).  Per-slot results must not depend on the batch composition (bitwise).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import DECODE_TOL, check_parity, dev_inputs, host_inputs, i32, rel
from rwkv_wkv_gb300 import DEV_BAD_SLOT, Pool

pytestmark = pytest.mark.gpu


def test_single_layer_64_sequential_decode_calls_fp32():
    """1 layer, 4 heads, 2 slots, 64 tokens as 64 decode calls, fp32 inputs,
    zero initial state (created slots)."""
    W = wl.SINGLE_LAYER
    T = 64
    ins = wl.token_inputs(W.seed, "tokens", T * W.n_slots, W.H, W.N, dtype="f32")
    ins = {k: v.reshape(T, W.n_slots, W.H, W.N) for k, v in ins.items()}
    with Pool(W.n_layers, W.H, W.n_slots) as pool:
        slots = pool.create(W.n_slots)
        ids = i32(slots)
        outs = []
        for t in range(T):
            step = {k: v[t] for k, v in ins.items()}
            outs.append(pool.decode_step(0, ids, *dev_inputs(step, "f32")).cpu().numpy())
        assert pool.device_status() == 0
        o_gpu = np.stack(outs)                                  # [T, B, H, N]
        S_gpu = pool.states[slots, 0].cpu().numpy()             # [B, H, N, N]
    S = np.zeros((W.n_slots, W.H, W.N, W.N))
    o_ref = []
    for t in range(T):
        o, S = oracle.decode_step(S, *[x[t] for x in host_inputs(ins)])
        o_ref.append(o)
    o_ref = np.stack(o_ref)
    check_parity(o_gpu, o_ref, DECODE_TOL, lead=3, elementwise=True, what="o")   # [T, B, H]
    check_parity(S_gpu, S, DECODE_TOL, lead=2, elementwise=True, what="S")       # [B, H]


@pytest.fixture(scope="module")
def decode12():
    """12 layers x 12 heads, 256 active slots of a 1024-slot pool at random ids,
    N(0, 0.1) states, bf16 inputs: one decode step per layer."""
    W = wl.DECODE_12L
    B = 256
    slots = wl.distinct_slots(W.seed, "decode/slots", B, W.n_slots)
    S0 = wl.slot_states(W.seed, "state", slots, W.n_layers, W.H, W.N)   # [B, L, H, N, N]
    ins = [wl.token_inputs(W.seed, f"layer{l}", B, W.H, W.N, dtype="bf16")
           for l in range(W.n_layers)]
    return W, B, slots, S0, ins


def test_decode_12_layers_full_size(decode12):
    W, B, slots, S0, ins = decode12
    with Pool(W.n_layers, W.H, W.n_slots) as pool:
        pool.states.fill_(7.0)                       # inactive slots: sentinel
        pool.states[torch.as_tensor(slots, dtype=torch.long)] = torch.from_numpy(S0).cuda()
        ids = i32(slots)
        o_gpu = [pool.decode_step(l, ids, *dev_inputs(ins[l], "bf16")).cpu().numpy()
                 for l in range(W.n_layers)]
        assert pool.device_status() == 0
        S_gpu = pool.states[torch.as_tensor(slots, dtype=torch.long)].cpu().numpy()
        inactive = np.setdiff1d(np.arange(W.n_slots), slots)
        assert bool((pool.states[torch.as_tensor(inactive, dtype=torch.long)] == 7.0).all())
    for l in range(W.n_layers):
        o_ref, S_ref = oracle.decode_step(S0[:, l], *host_inputs(ins[l]), n_threads=8)
        check_parity(o_gpu[l], o_ref, DECODE_TOL, lead=2, elementwise=True, what=f"o{l}")
        check_parity(S_gpu[:, l], S_ref, DECODE_TOL, lead=2, elementwise=True, what=f"S{l}")


def test_decode_batch_order_invariance_and_determinism(decode12):
    """Shuffling the batch order gives bitwise the same per-slot results, and
    running twice from the same state gives bitwise the same bits."""
    W, B, slots, S0, ins = decode12
    perm = np.random.default_rng(0).permutation(B)
    results = []
    with Pool(1, W.H, W.n_slots) as pool:
        for order in (np.arange(B), perm, np.arange(B)):
            pool.states[torch.as_tensor(slots, dtype=torch.long), 0] = torch.from_numpy(S0[:, 0]).cuda()
            step = {k: v[order] for k, v in ins[0].items()}
            o = pool.decode_step(0, i32(slots[order]), *dev_inputs(step, "bf16"))
            o_by_slot = torch.empty_like(o)
            o_by_slot[torch.as_tensor(order, dtype=torch.long)] = o
            results.append((o_by_slot.cpu(), pool.states[torch.as_tensor(slots, dtype=torch.long), 0].cpu()))
    for o, S in results[1:]:
        assert torch.equal(o, results[0][0])
        assert torch.equal(S, results[0][1])


def test_decode_out_of_range_slot_is_flagged_and_skipped():
    H, N, n_slots = 2, 64, 8
    ins = wl.token_inputs(11, "bad", 3, H, N, dtype="bf16")
    S0 = wl.slot_states(11, "state", range(n_slots), 1, H, N)[:, 0]
    with Pool(1, H, n_slots) as pool:
        pool.states[:, 0] = torch.from_numpy(S0).cuda()
        o = torch.full((3, H, N), -3.0, device="cuda")
        pool.decode_step(0, i32([1, n_slots + 5, 4]), *dev_inputs(ins, "bf16"), o=o)
        assert pool.device_status() == DEV_BAD_SLOT
        assert pool.device_status() == 0                      # read clears the word
        S_gpu = pool.states[:, 0].cpu().numpy()
        o = o.cpu().numpy()
    assert np.all(o[1] == -3.0)                               # skipped row untouched
    o_ref, S_ref = oracle.decode_step(S0[[1, 4]], *[x[[0, 2]] for x in host_inputs(ins)])
    assert rel(o[[0, 2]], o_ref) < DECODE_TOL
    assert rel(S_gpu[[1, 4]], S_ref) < DECODE_TOL
    others = [0, 2, 3, 5, 6, 7]
    np.testing.assert_array_equal(S_gpu[others], S0[others])


@pytest.mark.parametrize("B", [1, 4096])
def test_decode_sweep_32_layers_64_heads_sampled(B):
    """32 layers x 64 heads x 64 over a 4096-slot pool (128 GiB of float32
    state), layers invoked back to back as the benchmark times them.  Inputs of
    rows outside the sample come from torch's device generator; the sampled
    rows and slots carry seeded host values that the oracle also sees."""
    W = wl.SWEEP_32L
    slots = wl.distinct_slots(W.seed, f"sweep/slots{B}", B, W.n_slots)
    sample_rows = np.unique(np.linspace(0, B - 1, min(B, 6)).astype(int))
    layers_checked = (0, W.n_layers - 1)
    pool = Pool(W.n_layers, W.H, W.n_slots)
    try:
        gen = torch.Generator(device="cuda").manual_seed(W.seed)
        pool.states.normal_(0.0, 0.1, generator=gen)
        S0 = {}
        for rix in sample_rows:
            st = wl.slot_states(W.seed, "state", [slots[rix]], W.n_layers, W.H, W.N,
                                layers=layers_checked)[0]
            for li, l in enumerate(layers_checked):
                pool.states[int(slots[rix]), l] = torch.from_numpy(st[li]).cuda()
                S0[(rix, l)] = st[li]
        dev_ins = [torch.randn(B, W.H, W.N, device="cuda", generator=gen).to(torch.bfloat16)
                   for _ in range(6)]
        dev_ins[1] = torch.exp(-torch.exp(-0.6 + 0.3 * dev_ins[1].float())).to(torch.bfloat16)
        host = {}
        for l in layers_checked:
            ins = wl.token_inputs(W.seed, f"sweep/layer{l}", len(sample_rows), W.H, W.N, "bf16")
            host[l] = ins
        ids = i32(slots)
        o_keep = {}
        for l in range(W.n_layers):
            if l in host:
                for n, name in enumerate(wl.INPUT_NAMES):
                    dev_ins[n][torch.as_tensor(sample_rows, dtype=torch.long)] = \
                        torch.from_numpy(host[l][name]).cuda().to(torch.bfloat16)
            o = pool.decode_step(l, ids, *dev_ins)
            if l in host:
                o_keep[l] = o[torch.as_tensor(sample_rows, dtype=torch.long)].cpu().numpy()
        assert pool.device_status() == 0
        for l in layers_checked:
            St = np.stack([S0[(rix, l)] for rix in sample_rows])
            o_ref, S_ref = oracle.decode_step(St, *host_inputs(host[l]))
            S_gpu = pool.states[torch.as_tensor(slots[sample_rows], dtype=torch.long), l].cpu().numpy()
            assert rel(o_keep[l], o_ref) < DECODE_TOL
            assert rel(S_gpu, S_ref) < DECODE_TOL
    finally:
        pool.close()
        del pool
        torch.cuda.empty_cache()


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_dependent_calls_without_host_sync(state_dtype):
    """Eight decode steps on the same slots, each launched right after the
    previous one with no host synchronisation (each kernel may begin launching
    while the previous one drains and must still read the state it wrote), then
    a snapshot, a fork and a prefill that read those states; compared with the
    oracle's chained steps."""
    H, N, B, T = 8, 64, 64, 8
    ins = wl.token_inputs(45, "chain", T * B, H, N, dtype="bf16")
    ins = {k: v.reshape(T, B, H, N) for k, v in ins.items()}
    dev = [[torch.from_numpy(ins[n][t]).cuda().to(torch.bfloat16) for n in wl.INPUT_NAMES]
           for t in range(T)]
    S0 = wl.slot_states(45, "chain/s0", range(B), 1, H, N)[:, 0]
    if state_dtype == "bf16":
        S0 = oracle.round_bf16(S0)
    pre = wl.token_inputs(46, "chain/pre", 100, H, N, dtype="bf16")
    tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    with Pool(1, H, 2 * B, n_snapshots=B, state_dtype=state_dtype) as pool:
        pool.states[:B, 0] = torch.from_numpy(S0).cuda().to(tdt)
        ids, fork_dst, pre_slot, pre_cu = i32(range(B)), i32(range(B, 2 * B)), i32([B]), i32([0, 100])
        pre_dev = dev_inputs(pre, "bf16")
        torch.cuda.synchronize()
        outs = [pool.decode_step(0, ids, *dev[t]) for t in range(T)]
        pool.snapshot(ids, ids)
        pool.fork(ids, fork_dst)
        o_pre = pool.prefill(0, pre_slot, pre_cu, *pre_dev, max_seqlen=100)
        torch.cuda.synchronize()
        assert pool.device_status() == 0
        o_gpu = torch.stack(outs).cpu().numpy()
        S_gpu = pool.states[:B, 0].double().cpu().numpy()
        assert torch.equal(pool.snapshots[:, 0], pool.states[:B, 0])
        assert torch.equal(pool.states[B + 1:2 * B, 0], pool.states[1:B, 0])
        S_pre = pool.states[B, 0].double().cpu().numpy()
    S = S0.astype(np.float64)
    step = oracle.decode_step_bf16_state if state_dtype == "bf16" else oracle.decode_step
    for t in range(T):
        o, S = step(S, *[x[t] for x in host_inputs(ins)], n_threads=8)
        assert rel(o_gpu[t], o) < (DECODE_TOL if state_dtype == "f32" else 1e-2), t
    assert rel(S_gpu, S) < (DECODE_TOL if state_dtype == "f32" else 1e-2)
    o_ref, S_ref = oracle.prefill(S_gpu[:1], np.array([0, 100]), *host_inputs(pre))
    assert rel(o_pre.cpu().numpy(), o_ref) < 2e-2
    if state_dtype == "bf16":
        S_ref = oracle.round_bf16(S_ref)
    assert rel(S_pre, S_ref[0]) < 2e-2
