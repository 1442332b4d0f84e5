"""GPU parity of the prefill paths against the oracle.

wkv7_prefill (chunked, bf16 tensor-core operands, float32 carry): normwise-max
relative error <= 2e-2 on outputs and final states.  wkv7_prefill_sequential
(float32 token by token): <= 1e-4.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import (PREFILL_TOL, SEQ_PREFILL_TOL, check_parity, dev_inputs, host_inputs, i32,
                         rel, sampled_head_inputs)
from rwkv_wkv_gb300 import DEV_BAD_SEQLENS, DEV_BAD_SLOT, DEV_WAIT_TIMEOUT, Pool, load_library

pytestmark = pytest.mark.gpu

PATHS = [("chunked", False, PREFILL_TOL), ("sequential", True, SEQ_PREFILL_TOL)]


def _run(pool, slots, cu, ins, sequential, layer=0):
    dev = ins if isinstance(ins, list) else dev_inputs(ins, "bf16")
    o = pool.prefill(layer, i32(slots), i32(cu), *dev,
                     max_seqlen=int(np.max(np.diff(cu))) if len(cu) > 1 else 0,
                     sequential=sequential)
    code = pool.device_status()
    return o.cpu().numpy(), code


def _check(pool, slots, cu, ins, S0, sequential, tol, heads=None, host=None):
    """ins: host dict (all heads) or a list of device tensors with `host`
    holding the seeded values of `heads` only."""
    o_gpu, code = _run(pool, slots, cu, ins, sequential)
    assert code == 0
    S_gpu = pool.states[torch.as_tensor(slots, dtype=torch.long), 0].cpu().numpy()
    H = S0.shape[1]
    heads = list(range(H)) if heads is None else heads
    if host is None:
        sub = [x[:, heads] for x in host_inputs(ins)]
    else:
        sub = host_inputs(host)
    o_ref, S_ref = oracle.prefill(S0[:, heads], cu, *sub, n_threads=8)
    exact = sequential  # the float32 path is also held element by element
    e_o = check_parity(o_gpu[:, heads], o_ref, tol, cu=cu, elementwise=exact, what="o")["normwise"]
    e_s = check_parity(S_gpu[:, heads], S_ref, tol, lead=2, elementwise=exact, what="S")["normwise"]
    return e_o, e_s


@pytest.mark.parametrize("name,sequential,tol", PATHS)
def test_single_layer_as_one_prefill(name, sequential, tol):
    """1 layer, 4 heads, 2 slots, T = 64 per slot, zero start (bf16-rounded
    copy of the decode inputs)."""
    W = wl.SINGLE_LAYER
    T = 64
    ins = wl.token_inputs(W.seed, "tokens", T * W.n_slots, W.H, W.N, dtype="bf16")
    # token-major [T][slot] -> sequence-major [slot][T]
    ins = {k: np.ascontiguousarray(v.reshape(T, W.n_slots, W.H, W.N).transpose(1, 0, 2, 3)
                                   .reshape(T * W.n_slots, W.H, W.N)) for k, v in ins.items()}
    cu = wl.cu_seqlens([T] * W.n_slots)
    with Pool(1, W.H, W.n_slots) as pool:
        slots = pool.create(W.n_slots)
        _check(pool, slots, cu, ins, np.zeros((W.n_slots, W.H, W.N, W.N)), sequential, tol)


@pytest.mark.parametrize("name,sequential,tol", PATHS)
def test_ragged_lengths_around_chunk_boundaries(name, sequential, tol):
    """Lengths 1, 63, 64, 65, 129, 0 (empty), 200 from N(0, 0.1) start states."""
    H, N = 3, 64
    lengths = [1, 63, 64, 65, 129, 0, 200]
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(21, "ragged", int(cu[-1]), H, N, dtype="bf16")
    S0 = wl.slot_states(21, "state", range(len(lengths)), 1, H, N)[:, 0]
    with Pool(1, H, 16) as pool:
        slots = [3, 0, 9, 15, 7, 2, 11]
        pool.states[torch.as_tensor(slots, dtype=torch.long), 0] = torch.from_numpy(S0).cuda()
        _check(pool, slots, cu, ins, S0.astype(np.float64), sequential, tol)


@pytest.mark.parametrize("name,sequential,tol", PATHS)
def test_prefill_8x4096_32_heads_sampled_heads(name, sequential, tol):
    """8 sequences x 4096 tokens, 32 heads, zero start state, chunk 64; every
    output and final state of heads 0, 7, 19, 31 checked against the oracle."""
    W = wl.PREFILL_8x4096
    T = 4096
    cu = wl.cu_seqlens([T] * 8)
    heads = [0, 7, 19, 31]
    dev, host = sampled_head_inputs(W.seed, "tokens", T * 8, W.H, W.N, heads)
    with Pool(1, W.H, W.n_slots) as pool:
        slots = pool.create(8)
        _check(pool, slots, cu, dev, np.zeros((8, W.H, W.N, W.N)), sequential, tol,
               heads=heads, host=host)


@pytest.mark.parametrize("name,sequential,tol", PATHS)
def test_prefill_ragged_64_sequences_sampled(name, sequential, tol):
    """64 sequences with lengths uniform on 1..2048, 32 heads, into created
    slots of a 4096-slot pool; heads 0, 13, 31 checked."""
    W = wl.MIXED
    plan = wl.mixed_plan()
    lengths = plan["lengths"]
    cu = wl.cu_seqlens(lengths)
    heads = [0, 13, 31]
    dev, host = sampled_head_inputs(W.seed, "prefill", int(cu[-1]), W.H, W.N, heads)
    with Pool(1, W.H, W.n_slots) as pool:
        slots = pool.create(len(lengths))
        _check(pool, slots, cu, dev, np.zeros((len(lengths), W.H, W.N, W.N)), sequential, tol,
               heads=heads, host=host)


@pytest.mark.parametrize("sequential", [False, True])
def test_bad_sequence_metadata_is_flagged(sequential):
    H, N = 2, 64
    ins = wl.token_inputs(5, "bad", 10, H, N, dtype="bf16")
    with Pool(1, H, 4) as pool:
        pool.states.fill_(1.5)
        # second sequence runs backwards: skipped and flagged
        o = pool.prefill(0, i32([0, 1]), i32([0, 6, 4]), *dev_inputs(ins, "bf16"),
                         max_seqlen=10, sequential=sequential)
        assert pool.device_status() == DEV_BAD_SEQLENS
        assert bool((pool.states[1] == 1.5).all())
        # slot id out of range
        pool.prefill(0, i32([2, 99]), i32([0, 5, 10]), *dev_inputs(ins, "bf16"),
                     max_seqlen=5, sequential=sequential)
        assert pool.device_status() == DEV_BAD_SLOT
        # a sequence longer than max_seqlen
        pool.prefill(0, i32([3]), i32([0, 10]), *dev_inputs(ins, "bf16"), max_seqlen=4,
                     sequential=sequential)
        assert pool.device_status() == DEV_BAD_SEQLENS
        assert bool((pool.states[3] == 1.5).all())
        del o


def test_chunked_and_sequential_agree():
    """The two GPU paths on the same inputs (ragged, random start states)."""
    H, N = 4, 64
    lengths = [300, 64, 5, 1000]
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(8, "agree", int(cu[-1]), H, N, dtype="bf16")
    S0 = torch.from_numpy(wl.slot_states(8, "state", range(4), 1, H, N)[:, 0]).cuda()
    outs = []
    with Pool(1, H, 4) as pool:
        for sequential in (False, True):
            pool.states[:, 0] = S0
            o, code = _run(pool, [0, 1, 2, 3], cu, ins, sequential)
            assert code == 0
            outs.append((o, pool.states[:, 0].cpu().numpy()))
    assert rel(outs[0][0], outs[1][0]) < PREFILL_TOL
    assert rel(outs[0][1], outs[1][1]) < PREFILL_TOL


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decay_beyond_the_chunk_factorisation(state_dtype):
    """A channel whose decay over half a chunk exceeds 2^120 (w = 2^-8 for 40
    tokens, or an exact w = 0) cannot be factorised in chunks; wkv7_prefill then
    runs that (sequence, head) token by token in float32 in the same call, and
    every unit -- those and their neighbours on the chunked path -- matches the
    oracle.  Nothing is flagged."""
    H, N = 3, 64
    lengths = [40, 150, 64, 200]
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(31, "decay", int(cu[-1]), H, N, dtype="bf16")
    ins["w"] = ins["w"].copy()
    ins["w"][0:40, 1, 5] = 2.0 ** -8                      # sequence 0, head 1
    ins["w"][cu[1] + 70:cu[1] + 110, 2, 60] = 2.0 ** -9   # sequence 1, head 2, its second chunk
    ins["w"][cu[3] + 130, 0, 7] = 0.0                     # sequence 3, head 0: w = 0 once
    S0 = oracle.round_bf16(wl.slot_states(31, "decay/s0", range(len(lengths)), 1, H, N)[:, 0])
    tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    with Pool(1, H, len(lengths), state_dtype=state_dtype) as pool:
        pool.states[:, 0] = torch.from_numpy(S0).cuda().to(tdt)
        o, code = _run(pool, list(range(len(lengths))), cu, ins, sequential=False)
        assert code == 0
        S_gpu = pool.states[:, 0].float().cpu().numpy()
    o_ref, S_ref = oracle.prefill(S0.astype(np.float64), cu, *host_inputs(ins))
    if state_dtype == "bf16":
        S_ref = oracle.round_bf16(S_ref)
    check_parity(o, o_ref, PREFILL_TOL, cu=cu, what="o")
    check_parity(S_gpu, S_ref, PREFILL_TOL, lead=2, what="S")
    # the units that left the chunked path are exact to float32 (bf16 storage aside)
    per = oracle.rel_err_segments(o, o_ref, cu)
    assert per[0, 1] < 1e-4 and per[1, 2] < 1e-4 and per[3, 0] < 1e-4, per


def test_decay_beyond_the_chunk_factorisation_with_checkpoints():
    """The token-by-token route also writes every 64-token checkpoint of the unit."""
    H, N = 2, 64
    lengths = [130, 64]
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(32, "decay/ck", int(cu[-1]), H, N, dtype="bf16")
    ins["w"] = ins["w"].copy()
    ins["w"][80:120, 0, 11] = 2.0 ** -8                   # sequence 0, head 0, second chunk
    n_ck = [x // 64 for x in lengths]
    cu_ck = np.concatenate([[0], np.cumsum(n_ck)]).astype(np.int32)
    with Pool(1, H, len(lengths), n_snapshots=int(cu_ck[-1])) as pool:
        slots = pool.create(len(lengths))
        o = pool.prefill(0, i32(slots), i32(cu), *dev_inputs(ins, "bf16"), max_seqlen=max(lengths),
                         cu_ckpt=i32(cu_ck), ckpt_ids=i32(np.arange(cu_ck[-1])))
        assert pool.device_status() == 0
        ck = pool.snapshots[:, 0].cpu().numpy()
        S_gpu = pool.states[torch.as_tensor(slots), 0].cpu().numpy()
    o_ref, S_ref, ck_ref = oracle.prefill_checkpoints(np.zeros((2, H, N, N)), cu, *host_inputs(ins))
    check_parity(o.cpu().numpy(), o_ref, PREFILL_TOL, cu=cu, what="o")
    check_parity(S_gpu, S_ref, PREFILL_TOL, lead=2, what="S")
    ck_ref = np.stack([c for seq in ck_ref for c in seq])
    check_parity(ck, ck_ref, PREFILL_TOL, lead=2, what="checkpoints")
    assert oracle.rel_err(ck[:2, 0], ck_ref[:2, 0]) < 1e-4  # the token-by-token unit's checkpoints


@pytest.mark.parametrize("sequential", [False, True])
def test_all_sequences_empty(sequential):
    H, N = 2, 64
    ins = wl.token_inputs(2, "empty", 1, H, N, dtype="bf16")
    with Pool(1, H, 4) as pool:
        pool.states.fill_(0.25)
        dev = [x[:0] for x in dev_inputs(ins, "bf16")]
        o = pool.prefill(0, i32([1, 3]), i32([0, 0, 0]), *dev, max_seqlen=0,
                         sequential=sequential)
        assert o.shape == (0, H, N)
        assert pool.device_status() == 0
        assert bool((pool.states == 0.25).all())


def test_chunked_prefill_is_deterministic():
    """Same inputs and start states -> the same bits (no atomics, fixed order)."""
    H, N = 4, 64
    lengths = [777, 64, 1, 130]
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(12, "det", int(cu[-1]), H, N, dtype="bf16")
    S0 = torch.from_numpy(wl.slot_states(12, "state", range(4), 1, H, N)[:, 0]).cuda()
    runs = []
    with Pool(1, H, 4) as pool:
        for _ in range(2):
            pool.states[:, 0] = S0
            o, code = _run(pool, [2, 0, 3, 1], cu, ins, sequential=False)
            assert code == 0
            runs.append((o, pool.states.cpu().numpy()))
    np.testing.assert_array_equal(runs[0][0], runs[1][0])
    np.testing.assert_array_equal(runs[0][1], runs[1][1])


def test_output_alignment_does_not_change_results():
    """o 32-byte aligned takes 32-byte stores, o only 16-byte aligned 16-byte
    ones; both write the same bits."""
    H = 4
    lengths = [130, 64, 7]
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(41, "prefill/align", int(cu[-1]), H, 64, dtype="bf16")
    S0 = wl.slot_states(41, "prefill/align/s0", range(3), 1, H, 64)[:, 0]
    dev = dev_inputs(ins, "bf16")
    outs, states = [], []
    for shift in (0, 4):  # floats: 0 -> 256-byte aligned, 4 -> 16 bytes past it
        buf = torch.full((int(cu[-1]) * H * 64 + 8,), float("nan"), device="cuda")
        o = buf[shift:shift + int(cu[-1]) * H * 64].view(int(cu[-1]), H, 64)
        assert o.data_ptr() % 32 == (0 if shift == 0 else 16)
        with Pool(1, H, 3) as pool:
            pool.states[:, 0] = torch.from_numpy(S0).cuda()
            pool.prefill(0, i32([0, 1, 2]), i32(cu), *dev, o=o, max_seqlen=max(lengths))
            assert pool.device_status() == 0
            states.append(pool.states.clone())
        outs.append(o.clone())
        assert bool(torch.isnan(buf[:shift]).all()) and bool(torch.isnan(buf[shift + o.numel():]).all())
    assert torch.equal(outs[0], outs[1]) and torch.equal(states[0], states[1])
    o_ref, _ = oracle.prefill(S0.astype(np.float64), cu, *host_inputs(ins))
    assert rel(outs[1].cpu().numpy(), o_ref) < PREFILL_TOL


@functools.lru_cache(maxsize=2)
def _many(n_seqs, max_len, H):
    """Seeded inputs, start states and slot order of the many-sequence case."""
    N = 64
    rng = np.random.default_rng(n_seqs)
    lengths = rng.integers(1, max_len + 1, n_seqs)
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(44, f"many/{n_seqs}", int(cu[-1]), H, N, dtype="bf16")
    S0 = (wl.slot_states(44, f"many/{n_seqs}/s0", range(n_seqs), 1, H, N)[:, 0] if n_seqs <= 5000
          else np.zeros((n_seqs, H, N, N)))  # created slots
    return cu, ins, S0, rng.permutation(n_seqs)


@pytest.mark.parametrize("name,sequential,tol", PATHS)
@pytest.mark.parametrize("n_seqs,max_len,H", [(5000, 40, 2), (70000, 1, 1)])
def test_many_sequences(name, sequential, tol, n_seqs, max_len, H):
    """More sequences than the chunked kernel orders longest-first (4096; then
    index order) and than one grid dimension holds (65535; the ranks are split
    over two): every sequence still gets its own result."""
    cu, ins, S0, slots = _many(n_seqs, max_len, H)
    with Pool(1, H, n_seqs) as pool:
        pool.states[torch.as_tensor(slots), 0] = torch.from_numpy(S0).cuda().float()
        o, code = _run(pool, slots, cu, ins, sequential)
        assert code == 0
        S_gpu = pool.states[torch.as_tensor(slots), 0].cpu().numpy()
    o_ref, S_ref = oracle.prefill(S0.astype(np.float64), cu, *host_inputs(ins), n_threads=8)
    check_parity(o, o_ref, tol, cu=cu, what="o")
    check_parity(S_gpu, S_ref, tol, lead=2, what="S")


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """With the test hook on, the chunked prefill's first input load is never
    issued: every wait for it gives up (about 50 ms), the CTAs release their
    tensor memory and exit, the call reports WKV7_DEV_WAIT_TIMEOUT and leaves
    the slots' states alone.  The same call then runs normally."""
    lib = load_library()
    H, N = 2, 64
    lengths = [100, 7]
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(47, "timeout", int(cu[-1]), H, N, dtype="bf16")
    S0 = wl.slot_states(47, "timeout/s0", range(2), 1, H, N)[:, 0]
    dev = dev_inputs(ins, "bf16")
    with Pool(1, H, 2) as pool:
        pool.states[:, 0] = torch.from_numpy(S0).cuda()
        before = pool.states.clone()
        assert lib.wkv7_test_force_wait_timeout(1) == 0
        try:
            pool.prefill(0, i32([0, 1]), i32(cu), *dev, max_seqlen=max(lengths))
            assert pool.device_status() == DEV_WAIT_TIMEOUT
        finally:
            lib.wkv7_test_force_wait_timeout(0)
        assert torch.equal(pool.states, before)
        o = pool.prefill(0, i32([0, 1]), i32(cu), *dev, max_seqlen=max(lengths))
        assert pool.device_status() == 0
        S_gpu = pool.states[:, 0].cpu().numpy()
    o_ref, S_ref = oracle.prefill(S0.astype(np.float64), cu, *host_inputs(ins))
    assert rel(o.cpu().numpy(), o_ref) < PREFILL_TOL
    assert rel(S_gpu, S_ref) < PREFILL_TOL


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_sequential_prefill_float32_inputs(state_dtype):
    """wkv7_prefill_sequential also takes float32 inputs: against the oracle at the
    float32 tolerance, and on a bf16-state pool equal to the float32-pool run with
    the final state rounded."""
    H, N = 3, 64
    lengths = [70, 64, 1, 9]
    cu = wl.cu_seqlens(lengths)
    ins = wl.token_inputs(49, "seq/f32", int(cu[-1]), H, N, dtype="f32")
    dev = dev_inputs(ins, "f32")
    assert dev[0].dtype == torch.float32
    S0 = oracle.round_bf16(wl.slot_states(49, "seq/f32/s0", range(len(lengths)), 1, H, N)[:, 0])
    runs = {}
    for sd, tdt in (("f32", torch.float32), (state_dtype, torch.bfloat16 if state_dtype == "bf16" else torch.float32)):
        with Pool(1, H, len(lengths), state_dtype=sd) as pool:
            pool.states[:, 0] = torch.from_numpy(S0).cuda().to(tdt)
            o = pool.prefill(0, i32(range(len(lengths))), i32(cu), *dev, max_seqlen=max(lengths),
                             sequential=True)
            assert pool.device_status() == 0
            runs[sd] = (o.clone(), pool.states[:, 0].clone())
    o_ref, S_ref = oracle.prefill(S0.astype(np.float64), cu, *host_inputs(ins))
    check_parity(runs["f32"][0].cpu().numpy(), o_ref, SEQ_PREFILL_TOL, cu=cu, elementwise=True)
    check_parity(runs["f32"][1].cpu().numpy(), S_ref, SEQ_PREFILL_TOL, lead=2, elementwise=True)
    if state_dtype == "bf16":
        assert torch.equal(runs["bf16"][0], runs["f32"][0])
        assert torch.equal(runs["bf16"][1], runs["f32"][1].to(torch.bfloat16))


def test_long_sequence_error_does_not_grow_with_length():
    """One 65,536-token sequence (1,024 chunks), 2 heads, from N(0, 0.1) start
    states: the chunked path's float32 carry with the bf16 hi/lo state split
    keeps the error of the last 4,096 tokens' outputs and of the final state
    within the tolerance, and not far above the first 4,096 tokens' error."""
    H, N, T = 2, 64, 65536
    cu = wl.cu_seqlens([T])
    ins = wl.token_inputs(31, "long", T, H, N, dtype="bf16")
    S0 = wl.slot_states(31, "long/s0", [0], 1, H, N)[:, 0]
    with Pool(1, H, 1) as pool:
        pool.states[:, 0] = torch.from_numpy(S0).cuda()
        o_gpu, code = _run(pool, [0], cu, ins, sequential=False)
        assert code == 0
        S_gpu = pool.states[:, 0].cpu().numpy()
    o_ref, S_ref = oracle.prefill(S0.astype(np.float64), cu, *host_inputs(ins), n_threads=2)
    head = rel(o_gpu[:4096], o_ref[:4096])
    tail = rel(o_gpu[-4096:], o_ref[-4096:])
    assert tail < PREFILL_TOL and rel(S_gpu, S_ref) < PREFILL_TOL, (head, tail)
    assert tail < 4 * max(head, 1e-3), (head, tail)
