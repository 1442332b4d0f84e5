"""The mixed serving step at full size, in the benchmark's call order, against the
oracle: on a 4096-slot pool of 32 heads, create the 64 prefill slots, snapshot
64 decode slots, decode 1024 slots at permuted ids, prefill 64 ragged sequences
(lengths uniform on 1..2048) into the created slots, fork 64 decode slots into
free slots, restore the 64 snapshots.

Checked on sampled heads against the oracle: decode outputs and states (1e-4),
prefill outputs and final states (2e-2); bit for bit: the forks equal their
sources after the decode, the restored slots equal their states before it, and
every slot the step does not touch is unchanged.  The same step on a pool with
bf16 state storage: decode meets the one-step bf16 contract, prefill's final
states are the oracle's rounded to bf16 (2e-2).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import (DECODE_TOL, PREFILL_TOL, check_bf16_state_step, host_inputs, i32, rel,
                         sampled_head_inputs)
from rwkv_wkv_gb300 import Pool

pytestmark = pytest.mark.gpu

HEADS = [0, 19, 31]


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_mixed_serving_step_full_size(state_dtype):
    W = wl.MIXED
    plan = wl.mixed_plan()
    dec, pre, fsrc, fdst, ssrc = (plan[k] for k in ("decode", "prefill", "fork_src", "fork_dst",
                                                    "snap_src"))
    lengths = plan["lengths"]
    cu = wl.cu_seqlens(lengths)
    B = len(dec)
    dec_dev, dec_host = sampled_head_inputs(W.seed, "mixed/decode", B, W.H, W.N, HEADS)
    pre_dev, pre_host = sampled_head_inputs(W.seed, "mixed/prefill", int(cu[-1]), W.H, W.N, HEADS)
    L = lambda ids: torch.as_tensor(np.asarray(ids), dtype=torch.long, device="cuda")  # noqa: E731

    with Pool(1, W.H, W.n_slots, n_snapshots=wl.MIXED_VERB_N, state_dtype=state_dtype) as pool:
        g = torch.Generator(device="cuda").manual_seed(W.seed)
        pool.states.normal_(0.0, 0.1, generator=g)
        pool.alloc(W.n_slots)
        pool.free(list(pre[::-1]))           # the prefill targets are created by the step
        before = pool.states.clone()
        snaps = pool.snapshot_alloc(wl.MIXED_VERB_N)

        created = pool.create(len(pre))
        assert created == [int(x) for x in pre]
        pool.snapshot(i32(ssrc), i32(snaps))
        o_dec = pool.decode_step(0, i32(dec), *dec_dev)
        after_decode = pool.states[L(dec)].clone()
        o_pre = pool.prefill(0, i32(pre), i32(cu), *pre_dev, max_seqlen=int(np.max(lengths)))
        pool.fork(i32(fsrc), i32(fdst))
        pool.restore(i32(snaps), i32(ssrc))
        assert pool.device_status() == 0
        final = pool.states.clone()

    S_dec0 = before[L(dec), 0][:, HEADS].double().cpu().numpy()
    S_dec1 = after_decode[:, 0][:, HEADS].double().cpu().numpy()
    if state_dtype == "f32":
        o_ref, S_ref = oracle.decode_step(S_dec0, *host_inputs(dec_host), n_threads=8)
        assert rel(o_dec[:, HEADS].cpu().numpy(), o_ref) < DECODE_TOL
        assert rel(S_dec1, S_ref) < DECODE_TOL
    else:
        o_ref, S_ref = oracle.decode_step_bf16_state(S_dec0, *host_inputs(dec_host), n_threads=8)
        check_bf16_state_step(o_dec[:, HEADS].cpu().numpy(), S_dec1, o_ref, S_ref)

    o_ref, S_ref = oracle.prefill(np.zeros((len(pre), len(HEADS), W.N, W.N)), cu,
                                  *host_inputs(pre_host), n_threads=8)
    if state_dtype == "bf16":
        S_ref = oracle.round_bf16(S_ref)
    assert rel(o_pre[:, HEADS].cpu().numpy(), o_ref) < PREFILL_TOL
    assert rel(final[L(pre), 0][:, HEADS].double().cpu().numpy(), S_ref) < PREFILL_TOL

    pos = {int(s): i for i, s in enumerate(dec)}
    assert torch.equal(final[L(fdst)], after_decode[L([pos[int(s)] for s in fsrc])])
    assert torch.equal(final[L(ssrc)], before[L(ssrc)])
    kept = [i for i, s in enumerate(dec) if int(s) not in set(int(x) for x in ssrc)]
    assert torch.equal(final[L(np.asarray(dec)[kept])], after_decode[L(kept)])
    touched = set(int(x) for x in np.concatenate([dec, pre, fdst]))
    untouched = [s for s in range(W.n_slots) if s not in touched]
    assert torch.equal(final[L(untouched)], before[L(untouched)])
