"""Sequences of one prefill call are independent: non-finite inputs in one
sequence (NaN and inf in v, k and w) leave every other sequence's outputs and
final state bit-identical to a run without them, on both prefill paths.  The
chunked path loads 64-token boxes that run past a sequence's end into its
neighbour; those tokens must never reach the arithmetic."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_helpers import NAMES, dev_inputs, i32
from rwkv_wkv_gb300 import Pool

pytestmark = pytest.mark.gpu

H, N = 3, 64


@pytest.mark.parametrize("sequential", [False, True])
def test_poisoned_neighbour_changes_nothing_else(sequential):
    lengths = [70, 50, 90, 1, 64]
    poisoned = 1
    cu = wl.cu_seqlens(lengths)
    n = len(lengths)
    ins = wl.token_inputs(90, "isolation", int(cu[-1]), H, N, dtype="bf16")
    S0 = wl.slot_states(91, "isolation/s0", range(n), 1, H, N)[:, 0]
    bad = {name: np.array(ins[name], copy=True) for name in NAMES}
    t0, t1 = int(cu[poisoned]), int(cu[poisoned + 1])
    bad["v"][t0:t1:3] = np.nan
    bad["k"][t0 + 1:t1:5] = np.inf
    bad["w"][t0 + 2:t1:7] = np.nan
    results = []
    for x in (ins, bad):
        dev = dev_inputs(x, "bf16")
        with Pool(1, H, n) as pool:
            pool.states[:, 0] = torch.from_numpy(S0).cuda()
            o = pool.prefill(0, i32(range(n)), i32(cu), *dev, max_seqlen=max(lengths),
                             sequential=sequential)
            assert pool.device_status() == 0
            results.append((o.clone(), pool.states[:, 0].clone()))
    (o_a, s_a), (o_b, s_b) = results
    for s in range(n):
        if s == poisoned:
            continue
        a, b = int(cu[s]), int(cu[s + 1])
        assert torch.equal(o_a[a:b], o_b[a:b]), s
        assert torch.equal(s_a[s], s_b[s]), s
    assert not torch.isfinite(o_b[t0:t1]).all()  # the poisoned sequence itself is not clean
