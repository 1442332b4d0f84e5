"""GPU parity of the chunk-boundary state checkpoints of prefill.

wkv7_prefill_checkpointed keeps the state after every 64th token of each
sequence in caller-named snapshots (xLLM, "Virtual Memory for KV Cache and Model
Weights", prefix caching: a hybrid model resumes a cached prefix from a stored
linear-attention state).  Checked against the oracle's segment-by-segment
recurrence, and by restoring a checkpoint and prefilling the rest of the
sequence, which must reproduce the uninterrupted run bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import PREFILL_TOL, SEQ_PREFILL_TOL, dev_inputs, host_inputs, i32, rel
from rwkv_wkv_gb300 import DEV_BAD_SEQLENS, DEV_BAD_SLOT, Pool

pytestmark = pytest.mark.gpu

PATHS = [("chunked", False, PREFILL_TOL), ("sequential", True, SEQ_PREFILL_TOL)]
LENGTHS = [1, 63, 64, 65, 129, 0, 200, 256]


def _layout(lengths):
    """cu_ckpt and snapshot ids 0.. for len // 64 checkpoints per sequence."""
    cu = np.concatenate([[0], np.cumsum([n // 64 for n in lengths])]).astype(np.int32)
    return cu, np.arange(cu[-1], dtype=np.int32)


@pytest.mark.parametrize("name,sequential,tol", PATHS)
def test_checkpoints_match_oracle(name, sequential, tol):
    H, N = 2, 64
    cu = wl.cu_seqlens(LENGTHS)
    ins = wl.token_inputs(41, "ckpt", int(cu[-1]), H, N, dtype="bf16")
    S0 = wl.slot_states(41, "state", range(len(LENGTHS)), 1, H, N)[:, 0]
    cuc, ids = _layout(LENGTHS)
    slots = [5, 0, 7, 2, 9, 1, 3, 11]
    with Pool(1, H, 12, n_snapshots=int(cuc[-1])) as pool:
        pool.states[torch.as_tensor(slots), 0] = torch.from_numpy(S0).cuda()
        o = pool.prefill(0, i32(slots), i32(cu), *dev_inputs(ins, "bf16"),
                         max_seqlen=max(LENGTHS), sequential=sequential,
                         cu_ckpt=i32(cuc), ckpt_ids=i32(ids))
        assert pool.device_status() == 0
        o_gpu = o.cpu().numpy()
        S_gpu = pool.states[torch.as_tensor(slots), 0].cpu().numpy()
        ck_gpu = pool.snapshots[:, 0].cpu().numpy()
    o_ref, S_ref, ck_ref = oracle.prefill_checkpoints(S0.astype(np.float64), cu, *host_inputs(ins),
                                                      n_threads=8)
    assert rel(o_gpu, o_ref) < tol
    assert rel(S_gpu, S_ref) < tol
    for s, states in enumerate(ck_ref):
        assert len(states) == LENGTHS[s] // 64
        for m, ref in enumerate(states):
            assert rel(ck_gpu[cuc[s] + m], ref) < tol, (s, m)


@pytest.mark.parametrize("name,sequential,tol", PATHS)
def test_resume_from_checkpoint_is_bit_identical(name, sequential, tol):
    """Restore the checkpoint after token 64 m into another slot and prefill the
    remaining tokens: outputs and final state equal the uninterrupted run."""
    H, N, L = 3, 64, 230
    ins = wl.token_inputs(43, "resume", L, H, N, dtype="bf16")
    dev = dev_inputs(ins, "bf16")
    S0 = torch.from_numpy(wl.slot_states(43, "state", [0], 1, H, N)[0, 0]).cuda()
    with Pool(1, H, 4, n_snapshots=3) as pool:
        pool.states[0, 0] = S0
        o_full = pool.prefill(0, i32([0]), i32([0, L]), *dev, max_seqlen=L, sequential=sequential,
                              cu_ckpt=i32([0, 3]), ckpt_ids=i32([0, 1, 2])).clone()
        S_full = pool.states[0].clone()
        assert pool.device_status() == 0
        for m in (1, 2, 3):
            pool.restore(i32([m - 1]), i32([1]))
            rest = [x[64 * m:] for x in dev]
            o_rest = pool.prefill(0, i32([1]), i32([0, L - 64 * m]), *rest, max_seqlen=L - 64 * m,
                                  sequential=sequential)
            assert pool.device_status() == 0
            assert torch.equal(o_rest, o_full[64 * m:]), m
            assert torch.equal(pool.states[1], S_full), m


@pytest.mark.parametrize("sequential", [False, True])
def test_wrong_count_skips_the_sequence_and_bad_ids_are_flagged(sequential):
    H, N = 2, 64
    lengths = [128, 70]
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(47, "ckbad", int(cu[-1]), H, N, dtype="bf16")
    dev = dev_inputs(ins, "bf16")
    with Pool(1, H, 4, n_snapshots=4) as pool:
        pool.states.fill_(0.5)
        pool.snapshots.fill_(-1.0)
        # sequence 1 declares 2 checkpoints but has 70 // 64 = 1: it is skipped
        pool.prefill(0, i32([0, 1]), i32(cu), *dev, max_seqlen=128, sequential=sequential,
                     cu_ckpt=i32([0, 2, 4]), ckpt_ids=i32([0, 1, 2, 3]))
        assert pool.device_status() == DEV_BAD_SEQLENS
        assert bool((pool.states[1] == 0.5).all())
        assert bool((pool.snapshots[2:] == -1.0).all())
        assert not bool((pool.states[0] == 0.5).all())
        assert not bool((pool.snapshots[0] == -1.0).all())
        # an out-of-range id: that checkpoint is not written, the rest is
        pool.snapshots.fill_(-1.0)
        pool.prefill(0, i32([0, 1]), i32(cu), *dev, max_seqlen=128, sequential=sequential,
                     cu_ckpt=i32([0, 2, 3]), ckpt_ids=i32([0, 99, 3]))
        assert pool.device_status() == DEV_BAD_SLOT
        assert not bool((pool.snapshots[0] == -1.0).all())
        assert not bool((pool.snapshots[3] == -1.0).all())
        assert bool((pool.snapshots[1:3] == -1.0).all())
