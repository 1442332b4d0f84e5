"""GPU checks of bf16 outputs (a pool created with out_dtype = bf16).

Contract: the calls compute exactly as on a float32-output pool and round each
float32 readout to bf16 (nearest even) as they store it; states, checkpoints
and rollback snapshots are unchanged.  Checked bit for bit against the same
call on a float32-output pool (its o rounded by torch, which rounds to nearest
even), and against the oracle within the path's tolerance plus half a bf16
unit (2^-8 of the largest magnitude).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import (DECODE_TOL, NAMES, PREFILL_TOL, SEQ_PREFILL_TOL, dev_inputs, host_inputs,
                         i32, rel)
from rwkv_wkv_gb300 import Pool

pytestmark = pytest.mark.gpu

H, N = 3, 64
HALF_ULP = 2.0 ** -8  # bf16 keeps 8 significant bits: half a unit is 2^-8 relative


def _pools(state_dtype, n_slots, n_snapshots, S0):
    """A float32-output and a bf16-output pool holding the same start states."""
    out = []
    for od in ("f32", "bf16"):
        p = Pool(1, H, n_slots, n_snapshots=n_snapshots, state_dtype=state_dtype, out_dtype=od)
        p.states[:, 0] = torch.from_numpy(S0).cuda().to(p.states.dtype)
        out.append(p)
    return out


def _same_storage(p32, p16, snapshots_written):
    assert torch.equal(p32.states, p16.states)
    if snapshots_written:  # else the snapshot store holds whatever the allocation held
        assert torch.equal(p32.snapshots, p16.snapshots)


def _check_rounding(o32, o16):
    assert o32.dtype == torch.float32 and o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("in_dtype", ["bf16", "f32"])
def test_decode_step_bf16_out(state_dtype, in_dtype):
    pool_n, B = 16, 11
    ins = wl.token_inputs(70, "bf16out/dec", B, H, N, dtype=in_dtype)
    S0 = wl.slot_states(71, "bf16out/s", range(pool_n), 1, H, N)[:, 0]
    if state_dtype == "bf16":
        S0 = oracle.round_bf16(S0)
    ids = wl.distinct_slots(72, "bf16out/ids", B, pool_n)
    dev = dev_inputs(ins, in_dtype)
    p32, p16 = _pools(state_dtype, pool_n, 0, S0)
    try:
        o32 = p32.decode_step(0, i32(ids), *dev)
        o16 = p16.decode_step(0, i32(ids), *dev)
        assert p32.device_status() == 0 and p16.device_status() == 0
        _check_rounding(o32, o16)
        _same_storage(p32, p16, False)
    finally:
        p32.close(), p16.close()
    step = oracle.decode_step_bf16_state if state_dtype == "bf16" else oracle.decode_step
    o_ref, _ = step(S0[ids], *host_inputs(ins))
    assert rel(o16.float().cpu().numpy(), o_ref) < DECODE_TOL + HALF_ULP


@pytest.mark.parametrize("snaps", [False, True])
def test_decode_multi_bf16_out(snaps):
    pool_n, B, K = 20, 7, 5
    ins = wl.token_inputs(73, "bf16out/multi", B * K, H, N, dtype="bf16")
    host = [ins[n].reshape(B, K, H, N).astype(np.float64) for n in NAMES]
    dev = [torch.from_numpy(np.ascontiguousarray(ins[n].reshape(B, K, H, N))).cuda().to(torch.bfloat16)
           for n in NAMES]
    S0 = wl.slot_states(74, "bf16out/ms", range(pool_n), 1, H, N)[:, 0]
    ids = wl.distinct_slots(75, "bf16out/mids", B, pool_n)
    p32, p16 = _pools("f32", pool_n, B * K if snaps else 0, S0)
    try:
        kw = dict(step_snap_ids=i32(np.arange(B * K))) if snaps else {}
        o32 = p32.decode_multi(0, i32(ids), *dev, **kw)
        o16 = p16.decode_multi(0, i32(ids), *dev, **kw)
        assert p32.device_status() == 0 and p16.device_status() == 0
        _check_rounding(o32, o16)
        _same_storage(p32, p16, snaps)
    finally:
        p32.close(), p16.close()
    o_ref, _, _ = oracle.decode_multi(S0[ids], *host)
    assert rel(o16.float().cpu().numpy(), o_ref) < DECODE_TOL + HALF_ULP


@pytest.mark.parametrize("path,sequential,tol", [("chunked", False, PREFILL_TOL),
                                                  ("sequential", True, SEQ_PREFILL_TOL)])
@pytest.mark.parametrize("ckpt", [False, True])
def test_prefill_bf16_out(path, sequential, tol, ckpt):
    lengths = [1, 63, 64, 65, 129, 0, 200]
    cu = wl.cu_seqlens(lengths)
    n = len(lengths)
    n_ck = sum(L // 64 for L in lengths)
    ins = wl.token_inputs(76, "bf16out/pf", int(cu[-1]), H, N, dtype="bf16")
    dev = dev_inputs(ins, "bf16")
    S0 = wl.slot_states(77, "bf16out/ps", range(n), 1, H, N)[:, 0]
    p32, p16 = _pools("f32", n, max(n_ck, 1), S0)
    try:
        kw = {}
        if ckpt:
            cuc = np.concatenate([[0], np.cumsum([L // 64 for L in lengths])]).astype(np.int32)
            kw = dict(cu_ckpt=i32(cuc), ckpt_ids=i32(np.arange(n_ck)))
        o32 = p32.prefill(0, i32(range(n)), i32(cu), *dev, max_seqlen=max(lengths),
                          sequential=sequential, **kw)
        o16 = p16.prefill(0, i32(range(n)), i32(cu), *dev, max_seqlen=max(lengths),
                          sequential=sequential, **kw)
        assert p32.device_status() == 0 and p16.device_status() == 0
        _check_rounding(o32, o16)
        _same_storage(p32, p16, ckpt)
    finally:
        p32.close(), p16.close()
    o_ref, _ = oracle.prefill(S0, cu, *host_inputs(ins), n_threads=8)
    assert rel(o16.float().cpu().numpy(), o_ref) < tol + HALF_ULP


def test_bf16_out_rejects_a_float32_o():
    with Pool(1, H, 2, out_dtype="bf16") as pool:
        assert pool.out_dtype == "bf16"
        ins = wl.token_inputs(78, "bf16out/rej", 2, H, N, dtype="bf16")
        dev = dev_inputs(ins, "bf16")
        with pytest.raises(ValueError):
            pool.decode_step(0, i32([0, 1]), *dev, o=torch.empty(2, H, N, device="cuda"))
