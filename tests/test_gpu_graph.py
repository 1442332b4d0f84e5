"""Calls captured in a CUDA graph replay to the same bits as eager calls.

The library's launches (programmatic dependent launch, tensor maps built on the
host at call time) must capture like ordinary ones: decode steps, a
multi-token decode with rollback states and a chunked prefill, captured once
and replayed, equal the same calls run eagerly from the same start states.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_helpers import dev_inputs, i32
from rwkv_wkv_gb300 import Pool

pytestmark = pytest.mark.gpu

H, N = 4, 64


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_graph_replay_equals_eager(state_dtype):
    B, T, K = 16, 3, 4
    lengths = [130, 64, 5]
    cu = wl.cu_seqlens(lengths)
    steps = [dev_inputs(wl.token_inputs(48, f"graph/step{t}", B, H, N, dtype="bf16"), "bf16")
             for t in range(T)]
    multi = [x.view(B, K, H, N) for x in
             dev_inputs(wl.token_inputs(48, "graph/multi", B * K, H, N, dtype="bf16"), "bf16")]
    pre = dev_inputs(wl.token_inputs(48, "graph/pre", int(cu[-1]), H, N, dtype="bf16"), "bf16")
    S0 = wl.slot_states(48, "graph/s0", range(B + len(lengths)), 1, H, N)
    tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    ids, pre_ids, cu_d = i32(range(B)), i32(range(B, B + len(lengths))), i32(cu)
    snaps = i32(np.arange(B * K))
    outs = {}
    with Pool(1, H, B + len(lengths), n_snapshots=B * K, state_dtype=state_dtype) as pool:
        o_dec = [torch.empty(B, H, N, device="cuda") for _ in range(T)]
        o_multi = torch.empty(B, K, H, N, device="cuda")
        o_pre = torch.empty(int(cu[-1]), H, N, device="cuda")

        def calls():
            for t in range(T):
                pool.decode_step(0, ids, *steps[t], o=o_dec[t])
            pool.decode_multi(0, ids, *multi, o=o_multi, step_snap_ids=snaps)
            pool.prefill(0, pre_ids, cu_d, *pre, o=o_pre, max_seqlen=max(lengths))

        for mode in ("eager", "graph"):
            pool.states.copy_(torch.from_numpy(S0).to(tdt))
            pool.snapshots.zero_()
            if mode == "eager":
                calls()
            else:
                g = torch.cuda.CUDAGraph()  # the eager pass above warmed every path up
                with torch.cuda.graph(g):
                    calls()
                pool.states.copy_(torch.from_numpy(S0).to(tdt))  # the capture ran nothing
                pool.snapshots.zero_()
                g.replay()
            torch.cuda.synchronize()
            assert pool.device_status() == 0
            outs[mode] = [x.clone() for x in o_dec] + [o_multi.clone(), o_pre.clone(),
                                                        pool.states.clone(), pool.snapshots.clone()]
    for a, b in zip(outs["eager"], outs["graph"]):
        assert torch.equal(a, b)
