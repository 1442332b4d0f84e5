"""GPU parity of multi-token decode with per-token rollback states
(wkv7_decode_multi).

K consecutive tokens per slot in one call, the verify pass of speculative
decoding (the rvLLM README, "Speculative decoding (GPU, shipped)"), with the
state after every token kept in a snapshot so that the slot can be rolled back
to the last accepted token (the fork/restore verbs of "wkvm: state-slot
inference for RWKV, GDN and Mamba hybrids").  Tolerance 1e-4 against the
oracle; K single-token calls and rollback-then-continue must agree bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import DECODE_TOL, NAMES, i32, rel
from rwkv_wkv_gb300 import DEV_BAD_SLOT, Pool

pytestmark = pytest.mark.gpu


def _inputs(seed, B, K, H, N, dtype):
    ins = wl.token_inputs(seed, "multi", B * K, H, N, dtype=dtype)
    host = {n: ins[n].reshape(B, K, H, N) for n in NAMES}
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = [torch.from_numpy(np.ascontiguousarray(host[n])).cuda().to(tdt) for n in NAMES]
    return host, dev


@pytest.mark.parametrize("K", [1, 3, 8, 13])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("snaps", [False, True])
def test_decode_multi_matches_oracle(K, dtype, snaps):
    H, N, B, pool_n = 4, 64, 12, 40
    host, dev = _inputs(50 + K, B, K, H, N, dtype)
    ids = wl.distinct_slots(51, "ids", B, pool_n)
    S0 = wl.slot_states(52, "state", range(pool_n), 1, H, N)[:, 0]
    with Pool(1, H, pool_n, n_snapshots=B * K if snaps else 0) as pool:
        pool.states[:, 0] = torch.from_numpy(S0).cuda()
        step = i32(np.arange(B * K)[::-1].copy()) if snaps else None
        o = pool.decode_multi(0, i32(ids), *dev, step_snap_ids=step)
        assert pool.device_status() == 0
        o_gpu = o.cpu().numpy()
        S_gpu = pool.states[torch.as_tensor(ids), 0].cpu().numpy()
        snap_gpu = pool.snapshots[:, 0].cpu().numpy() if snaps else None
        untouched = np.setdiff1d(np.arange(pool_n), ids)
        assert torch.equal(pool.states[torch.as_tensor(untouched), 0].cpu(),
                           torch.from_numpy(S0[untouched]))
    o_ref, S_ref, per_tok = oracle.decode_multi(
        S0[ids].astype(np.float64), *[host[n].astype(np.float64) for n in NAMES], n_threads=8)
    assert rel(o_gpu, o_ref) < DECODE_TOL
    assert rel(S_gpu, S_ref) < DECODE_TOL
    if snaps:
        order = np.arange(B * K)[::-1]  # row b, token k -> snapshot order[b*K + k]
        got = snap_gpu[order].reshape(B, K, H, N, N)
        assert rel(got, per_tok) < DECODE_TOL


def test_k_single_steps_and_k1_are_bit_identical():
    """decode_multi over K tokens equals K decode_step calls bit for bit, and
    K = 1 equals one decode_step."""
    H, N, B, K = 4, 64, 16, 5
    host, dev = _inputs(60, B, K, H, N, "bf16")
    S0 = torch.from_numpy(wl.slot_states(61, "state", range(B), 1, H, N)[:, 0]).cuda()
    ids = i32(np.arange(B))
    with Pool(1, H, B) as pool:
        pool.states[:, 0] = S0
        o_multi = pool.decode_multi(0, ids, *dev).clone()
        S_multi = pool.states.clone()
        pool.states[:, 0] = S0
        for t in range(K):
            o_t = pool.decode_step(0, ids, *[x[:, t].contiguous() for x in dev])
            assert torch.equal(o_t, o_multi[:, t])
        assert torch.equal(pool.states, S_multi)
        pool.states[:, 0] = S0
        o1 = pool.decode_multi(0, ids, *[x[:, :1].contiguous() for x in dev])
        S1 = pool.states.clone()
        pool.states[:, 0] = S0
        o2 = pool.decode_step(0, ids, *[x[:, 0].contiguous() for x in dev])
        assert torch.equal(o1[:, 0], o2) and torch.equal(pool.states, S1)
        assert pool.device_status() == 0


def test_rollback_to_an_accepted_token_then_continue():
    """Verify K drafted tokens, accept the first j, restore the state after
    token j-1 and decode on: identical to having decoded only those tokens."""
    H, N, B, K = 2, 64, 4, 6
    host, dev = _inputs(70, B, K, H, N, "bf16")
    _, dev2 = _inputs(71, B, 1, H, N, "bf16")   # the token after the accepted prefix
    S0 = torch.from_numpy(wl.slot_states(72, "state", range(B), 1, H, N)[:, 0]).cuda()
    ids = i32(np.arange(B))
    accept = [0, 2, 5, 1]  # per row: index of the last accepted token
    with Pool(1, H, 2 * B, n_snapshots=B * K) as pool:
        pool.states[:B, 0] = S0
        o_ver = pool.decode_multi(0, ids, *dev, step_snap_ids=i32(np.arange(B * K)))
        pool.restore(i32([b * K + accept[b] for b in range(B)]), ids)
        o_next = pool.decode_step(0, ids, *[x[:, 0].contiguous() for x in dev2]).clone()
        S_next = pool.states[:B].clone()
        # reference: only the accepted tokens, then the next one, on fresh slots
        ref_ids = i32(np.arange(B, 2 * B))
        pool.states[B:, 0] = S0
        for b in range(B):
            sub = [x[b:b + 1, :accept[b] + 1].contiguous() for x in dev]
            o_acc = pool.decode_multi(0, ref_ids[b:b + 1], *sub)
            assert torch.equal(o_acc[0], o_ver[b, :accept[b] + 1])
        o_ref = pool.decode_step(0, ref_ids, *[x[:, 0].contiguous() for x in dev2])
        assert torch.equal(o_ref, o_next)
        assert torch.equal(pool.states[B:], S_next)
        assert pool.device_status() == 0


def test_bad_snapshot_id_is_flagged_and_skipped():
    H, N, B, K = 2, 64, 2, 3
    host, dev = _inputs(80, B, K, H, N, "bf16")
    with Pool(1, H, B, n_snapshots=B * K) as pool:
        pool.snapshots.fill_(-1.0)
        pool.decode_multi(0, i32([0, 1]), *dev, step_snap_ids=i32([0, 1, 2, 3, 77, 5]))
        assert pool.device_status() == DEV_BAD_SLOT
        assert bool((pool.snapshots[4] == -1.0).all())
        for s in (0, 1, 2, 3, 5):
            assert not bool((pool.snapshots[s] == -1.0).all())
