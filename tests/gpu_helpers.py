"""Shared plumbing for the GPU parity tests: move seeded inputs to the device and
gather what the oracle needs.  Nothing here computes the recurrence."""
import numpy as np
import torch

import workloads as wl

NAMES = wl.INPUT_NAMES  # r, w, k, v, a, b

DECODE_TOL = 1e-4    # float32 decode path, normwise-max relative error
PREFILL_TOL = 2e-2   # chunked prefill with bf16 tensor-core operands
SEQ_PREFILL_TOL = 1e-4  # float32 token-by-token prefill


def dev_inputs(ins: dict, dtype: str, device="cuda"):
    """Seeded float32 arrays (exact in dtype) -> list of device tensors r..b."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return [torch.from_numpy(np.ascontiguousarray(ins[n])).to(device).to(tdt) for n in NAMES]


def host_inputs(ins: dict):
    return [np.asarray(ins[n], dtype=np.float64) for n in NAMES]


def i32(x, device="cuda"):
    return torch.as_tensor(np.asarray(x, dtype=np.int32), device=device)


def rel(x, ref):
    import oracle
    return oracle.rel_err(np.asarray(x, dtype=np.float64), ref)


# Per-slice checks floor each slice's denominator at 1% of the median slice
# scale: a slice whose result cancels (k . r near 0 for a one-token sequence
# from a zero state, say) keeps the float32 rounding of summands of typical
# size, far above the tolerance times its own tiny magnitude.
SLICE_FLOOR = 1e-2

# Elementwise companion of the normwise bound: its median must stay under the
# path's tolerance and its 99.9th percentile under 100 times it.  Entries near
# zero are judged against a floor of 1e-6 of the tensor's largest magnitude, so
# the upper percentiles are those entries' rounding, not a wrong element.
ELEM_P999_FACTOR = 100.0


def check_parity(x, ref, tol, lead=0, cu=None, elementwise=False, what=""):
    """Assert x against the oracle's ref: the normwise-max error of the whole
    tensor and of every slice (each over the first `lead` axes, or, with cu,
    each (sequence, head) of a packed [tokens][heads][...] tensor) below tol;
    with `elementwise`, the median elementwise error below tol and its 99.9th
    percentile below ELEM_P999_FACTOR * tol.  Returns the figures."""
    import oracle
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    out = {"normwise": oracle.rel_err(x, ref)}
    assert out["normwise"] < tol, (what, out)
    if cu is not None:
        out["worst_slice"] = float(oracle.rel_err_segments(x, ref, cu, floor_frac=SLICE_FLOOR).max())
    elif lead:
        out["worst_slice"] = float(oracle.rel_err_slices(x, ref, lead, floor_frac=SLICE_FLOOR).max())
    if "worst_slice" in out:
        assert out["worst_slice"] < tol, (what, out)
    if elementwise:
        e = oracle.elementwise_rel(x, ref)
        out["elem_median"] = float(np.median(e))
        out["elem_p999"] = float(np.quantile(e, 0.999))
        assert out["elem_median"] < tol and out["elem_p999"] < ELEM_P999_FACTOR * tol, (what, out)
    return out


def sampled_head_inputs(seed: int, tag: str, n_tok: int, H: int, N: int, heads,
                        device="cuda"):
    """Full-size bf16 device inputs whose `heads` carry seeded host values (also
    returned, [n_tok, len(heads), N], for the oracle); the other heads are
    drawn with torch's device generator from the same recipe."""
    dev = wl.token_inputs_device(seed, n_tok, H, N, device)
    host = wl.token_inputs(seed, tag, n_tok, H, N, dtype="bf16", heads=heads)
    hidx = torch.as_tensor(list(heads), dtype=torch.long, device=device)
    for t, name in zip(dev, NAMES):
        t[:, hidx] = torch.from_numpy(host[name]).to(device).to(torch.bfloat16)
    return dev, host


def bf16_spacing(x):
    """Spacing of bf16 values at |x| (at least the subnormal spacing 2^-133)."""
    ax = np.maximum(np.abs(x), 2.0**-126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def check_bf16_state_step(o_gpu, S_gpu, o_ref, S_ref):
    """One step from a stored bf16 state: o within DECODE_TOL of the oracle's
    float64 step; the stored new state within one bf16 spacing of the oracle's
    float64 step rounded to bf16 (the float32 and float64 results round to
    different neighbours only when they straddle a rounding boundary), plus the
    float32 arithmetic error of the step (2^-18 of the head's largest entry,
    which matters only where an entry nearly cancels); at least 99% of the
    entries identical."""
    assert rel(o_gpu, o_ref) < DECODE_TOL
    diff = np.abs(S_gpu - S_ref)
    head_max = np.abs(S_ref).max(axis=(-2, -1), keepdims=True)
    allow = bf16_spacing(np.maximum(np.abs(S_gpu), np.abs(S_ref))) + head_max * 2.0**-18
    assert bool((diff <= allow).all()), float((diff / allow).max())
    assert float((diff == 0).mean()) >= 0.99
