"""GPU checks of the recurrence calls on a bf16-state pool beyond single-token
decode: both prefill paths (with and without chunk-boundary checkpoints) and
multi-token decode.

Contract: every call computes in float32 and rounds what it stores to bf16
(nearest even).  A prefill reads the bf16 start state exactly, carries float32
inside a sequence, rounds the final state and every checkpoint, and at a
checkpoint continues from the rounded value (so it equals the same sequence
prefilled in 64-token calls, each storing its state).  Multi-token decode is K
single steps, rounded after every token.  Checked bit for bit against runs on
a float32 pool that round at the same points, and against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import (NAMES, PREFILL_TOL, SEQ_PREFILL_TOL, bf16_spacing, check_bf16_state_step,
                         dev_inputs, host_inputs, i32, rel)
from rwkv_wkv_gb300 import Pool

pytestmark = pytest.mark.gpu

PATHS = [("chunked", False, PREFILL_TOL), ("sequential", True, SEQ_PREFILL_TOL)]
H, N = 3, 64


def _bf16(x):
    return x.to(torch.bfloat16)


def _start_states(seed, n):
    return oracle.round_bf16(wl.slot_states(seed, "bf16paths/s0", range(n), 1, H, N)[:, 0])


def _run_prefill(state_dtype, S0, lengths, dev, sequential, ckpt=False):
    """Prefill every sequence from S0 on a pool of the given state dtype; returns
    (o, final states as stored, checkpoints as stored or None)."""
    cu = wl.cu_seqlens(lengths)
    n = len(lengths)
    n_ck = sum(L // 64 for L in lengths)
    tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    with Pool(1, H, n, n_snapshots=max(n_ck, 1), state_dtype=state_dtype) as pool:
        pool.states[:, 0] = torch.from_numpy(S0).cuda().to(tdt)
        kw = {}
        if ckpt:
            cuc = np.concatenate([[0], np.cumsum([L // 64 for L in lengths])]).astype(np.int32)
            kw = dict(cu_ckpt=i32(cuc), ckpt_ids=i32(np.arange(n_ck)))
        o = pool.prefill(0, i32(range(n)), i32(cu), *dev, max_seqlen=max(lengths),
                         sequential=sequential, **kw).clone()
        assert pool.device_status() == 0
        ck = pool.snapshots[:n_ck, 0].clone() if ckpt else None
        return o, pool.states[:, 0].clone(), ck


def _pieces_on_f32_pool(S0, lengths, dev, sequential):
    """Each sequence prefilled in 64-token calls on a float32 pool, the state
    rounded to bf16 after every full piece (a checkpoint) and at the end."""
    cu = wl.cu_seqlens(lengths)
    outs, finals, cks = [], [], []
    with Pool(1, H, 1) as pool:
        for s, L in enumerate(lengths):
            pool.states[0, 0] = torch.from_numpy(S0[s]).cuda().float()
            for p0 in range(0, L, 64):
                n = min(64, L - p0)
                piece = [x[cu[s] + p0:cu[s] + p0 + n] for x in dev]
                outs.append(pool.prefill(0, i32([0]), i32([0, n]), *piece, max_seqlen=n,
                                         sequential=sequential).clone())
                if n == 64:
                    pool.states[0, 0] = _bf16(pool.states[0, 0]).float()
                    cks.append(_bf16(pool.states[0, 0]))
            assert pool.device_status() == 0
            finals.append(_bf16(pool.states[0, 0]))
    return torch.cat(outs), torch.stack(finals), (torch.stack(cks) if cks else None)


def _oracle_pieces(S0, lengths, host):
    """The oracle's recurrence with the same rounding points as _pieces_on_f32_pool."""
    cu = wl.cu_seqlens(lengths)
    outs, finals, cks = [], [], []
    for s, L in enumerate(lengths):
        S = S0[s][None].astype(np.float64)
        for p0 in range(0, L, 64):
            n = min(64, L - p0)
            piece = [x[cu[s] + p0:cu[s] + p0 + n] for x in host]
            o, S = oracle.prefill(S, np.array([0, n]), *piece)
            outs.append(o)
            if n == 64:
                S = oracle.round_bf16(S)
                cks.append(S[0])
        finals.append(oracle.round_bf16(S)[0])
    return np.concatenate(outs), np.stack(finals), (np.stack(cks) if cks else None)


def _close_bf16(got, ref, tol):
    """Stored bf16 states: within one bf16 spacing plus tol of the head's largest entry."""
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    head_max = np.abs(ref).max(axis=(-2, -1), keepdims=True)
    allow = bf16_spacing(np.maximum(np.abs(got), np.abs(ref))) + tol * head_max
    assert bool((np.abs(got - ref) <= allow).all())


@pytest.mark.parametrize("name,sequential,tol", PATHS)
def test_prefill_equals_float32_pool_rounded(name, sequential, tol):
    lengths = [130, 64, 7, 1, 200]
    ins = wl.token_inputs(61, "bf16paths/pre", sum(lengths), H, N, dtype="bf16")
    dev = dev_inputs(ins, "bf16")
    S0 = _start_states(61, len(lengths))
    o16, S16, _ = _run_prefill("bf16", S0, lengths, dev, sequential)
    o32, S32, _ = _run_prefill("f32", S0, lengths, dev, sequential)
    assert S16.dtype == torch.bfloat16
    assert torch.equal(o16, o32)
    assert torch.equal(S16, _bf16(S32))
    o_ref, S_ref = oracle.prefill(S0.astype(np.float64), wl.cu_seqlens(lengths), *host_inputs(ins))
    assert rel(o16.cpu().numpy(), o_ref) < tol
    _close_bf16(S16, oracle.round_bf16(S_ref), tol)


@pytest.mark.parametrize("name,sequential,tol", PATHS)
def test_checkpointed_prefill_equals_64_token_calls(name, sequential, tol):
    lengths = [1, 63, 64, 65, 129, 200, 256]
    ins = wl.token_inputs(62, "bf16paths/ck", sum(lengths), H, N, dtype="bf16")
    dev = dev_inputs(ins, "bf16")
    S0 = _start_states(62, len(lengths))
    o, S, ck = _run_prefill("bf16", S0, lengths, dev, sequential, ckpt=True)
    o_p, S_p, ck_p = _pieces_on_f32_pool(S0, lengths, dev, sequential)
    assert torch.equal(o, o_p)
    assert torch.equal(S, S_p)
    assert torch.equal(ck, ck_p)
    # the oracle with the same rounding points; where a float32 carry and the
    # float64 one round to different bf16 neighbours, the later results differ by
    # that one spacing's effect, hence 2e-3 rather than 1e-4 on the float32 path
    tol = max(tol, 2e-3)
    o_ref, S_ref, ck_ref = _oracle_pieces(S0, lengths, host_inputs(ins))
    assert rel(o.cpu().numpy(), o_ref) < tol
    _close_bf16(S, S_ref, tol)
    _close_bf16(ck, ck_ref, tol)


@pytest.mark.parametrize("name,sequential,tol", PATHS)
def test_resume_from_bf16_checkpoint_is_bit_identical(name, sequential, tol):
    """Restore the checkpoint after token 64 m and prefill the rest (itself
    checkpointed): outputs, later checkpoints and final state equal the
    uninterrupted run."""
    L = 230
    ins = wl.token_inputs(63, "bf16paths/resume", L, H, N, dtype="bf16")
    dev = dev_inputs(ins, "bf16")
    S0 = _start_states(63, 1)
    with Pool(1, H, 2, n_snapshots=6, state_dtype="bf16") as pool:
        pool.states[0, 0] = torch.from_numpy(S0[0]).cuda().to(torch.bfloat16)
        o_full = pool.prefill(0, i32([0]), i32([0, L]), *dev, max_seqlen=L, sequential=sequential,
                              cu_ckpt=i32([0, 3]), ckpt_ids=i32([0, 1, 2])).clone()
        S_full = pool.states[0].clone()
        ck_full = pool.snapshots[:3].clone()
        for m in (1, 2, 3):
            pool.restore(i32([m - 1]), i32([1]))
            rest = [x[64 * m:] for x in dev]
            o_rest = pool.prefill(0, i32([1]), i32([0, L - 64 * m]), *rest, max_seqlen=L - 64 * m,
                                  sequential=sequential, cu_ckpt=i32([0, 3 - m]),
                                  ckpt_ids=i32(np.arange(3, 6 - m)))
            assert pool.device_status() == 0
            assert torch.equal(o_rest, o_full[64 * m:]), m
            assert torch.equal(pool.states[1], S_full), m
            assert torch.equal(pool.snapshots[3:6 - m], ck_full[m:]), m


def _token_inputs(seed, B, K, dtype="bf16"):
    ins = wl.token_inputs(seed, "bf16paths/multi", B * K, H, N, dtype=dtype)
    host = {n: ins[n].reshape(B, K, H, N) for n in NAMES}
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = [torch.from_numpy(np.ascontiguousarray(host[n])).cuda().to(tdt) for n in NAMES]
    return host, dev


@pytest.mark.parametrize("in_dtype", ["bf16", "f32"])
def test_decode_multi_is_k_rounded_steps(in_dtype):
    """Each token meets the one-step bf16 contract from the state stored after
    the previous token (its rollback snapshot); the call equals K one-token calls
    bit for bit; rolling back to token k and continuing reproduces the rest."""
    B, K, pool_n = 10, 4, 24
    host, dev = _token_inputs(64, B, K, in_dtype)
    ids = wl.distinct_slots(64, "bf16paths/ids", B, pool_n)
    S0 = oracle.round_bf16(wl.slot_states(64, "bf16paths/multi/s0", range(pool_n), 1, H, N)[:, 0])
    sel = torch.as_tensor(ids, dtype=torch.long)
    with Pool(1, H, pool_n, n_snapshots=B * K, state_dtype="bf16") as pool:
        init = torch.from_numpy(S0).cuda().to(torch.bfloat16)
        pool.states[:, 0] = init
        step = i32(np.arange(B * K))  # row b, token k -> snapshot b*K + k
        o = pool.decode_multi(0, i32(ids), *dev, step_snap_ids=step).clone()
        assert pool.device_status() == 0
        S_end = pool.states[sel, 0].clone()
        snaps = pool.snapshots[:, 0].clone().view(B, K, H, N, N)
        assert torch.equal(snaps[:, K - 1], S_end)
        untouched = torch.as_tensor(np.setdiff1d(np.arange(pool_n), ids), dtype=torch.long)
        assert torch.equal(pool.states[untouched, 0], init[untouched])

        # K one-token calls
        pool.states[:, 0] = init
        for k in range(K):
            o1 = pool.decode_multi(0, i32(ids), *[x[:, k:k + 1].contiguous() for x in dev])
            assert torch.equal(o1[:, 0], o[:, k]), k
            assert torch.equal(pool.states[sel, 0], snaps[:, k]), k

        # roll back to the state after token 1 and continue with tokens 2..K-1
        pool.states[sel, 0] = snaps[:, 1]
        o2 = pool.decode_multi(0, i32(ids), *[x[:, 2:].contiguous() for x in dev])
        assert torch.equal(o2, o[:, 2:]) and torch.equal(pool.states[sel, 0], S_end)
        assert pool.device_status() == 0

    prev = S0[ids].astype(np.float64)
    snaps_np = snaps.double().cpu().numpy()
    o_np = o.cpu().numpy()
    for k in range(K):
        o_ref, S_ref = oracle.decode_step_bf16_state(
            prev, *[host[n][:, k].astype(np.float64) for n in NAMES], n_threads=8)
        check_bf16_state_step(o_np[:, k], snaps_np[:, k], o_ref, S_ref)
        prev = snaps_np[:, k]
