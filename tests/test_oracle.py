"""Pins for the CPU oracle, independent of the oracle's own code.

The operation (RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta Rule)"),
per head:  h = S a ;  S <- S diag(w) + h b^T + v k^T ;  o = S r.

Each test fixes the oracle against something other than itself: a hand-worked
example, a closed form, a textbook routine (the LMS/delta rule, a first-order
IIR filter, a causal linear-attention product), an invariant, or the agreement
of the three independently written forms on tiny inputs.  A dropped term, a
wrong sign, a transposed operand or an off-by-one in the decay index breaks at
least one of them (test_pins_catch_planted_mistakes plants such mistakes in a
copy of the recurrence and checks that the pins reject them).
"""
import os

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def _rand_inputs(T, N, rng, contractive=True):
    r = rng.standard_normal((T, N))
    k = rng.standard_normal((T, N))
    v = rng.standard_normal((T, N))
    if contractive:
        w = np.exp(-np.exp(rng.normal(-0.6, 0.3, (T, N))))
        khat = k / np.linalg.norm(k, axis=1, keepdims=True)
        a = -khat
        b = khat / (1 + np.exp(-rng.standard_normal((T, N))))
    else:  # arbitrary values, including growth
        w = rng.uniform(0.2, 1.3, (T, N))
        a = rng.standard_normal((T, N)) * 0.7
        b = rng.standard_normal((T, N)) * 0.7
    return r, w, k, v, a, b


# ---------------------------------------------------------------- hand example

def _golden(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "wkv7_two_tokens_n2.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(x) for x in nums])
    return vals


@pytest.mark.parametrize("form", ["sequential", "chunked", "matprod"])
def test_hand_worked_two_tokens(golden_dir, form):
    g = _golden(golden_dir)
    S0 = np.stack([g["S0_0"], g["S0_1"]])
    ins = [np.stack([g[f"{n}_t1"], g[f"{n}_t2"]]) for n in ("r", "w", "k", "v", "a", "b")]
    fn = getattr(oracle, form)
    # one token: o1 and S1
    o1, S1 = fn(S0, *[x[:1] for x in ins])
    np.testing.assert_array_equal(o1[0], g["o_t1"])
    np.testing.assert_array_equal(S1, np.stack([g["S1_0"], g["S1_1"]]))
    # two tokens: o1, o2, S2
    o, S2 = fn(S0, *ins)
    np.testing.assert_array_equal(o, np.stack([g["o_t1"], g["o_t2"]]))
    np.testing.assert_array_equal(S2, np.stack([g["S2_0"], g["S2_1"]]))


# ---------------------------------------------------------------- closed forms

def test_linear_attention_closed_form():
    """w = 1, a = b = 0, S0 = 0: S_t = sum_{s<=t} v_s k_s^T, so
    o_t = sum_{s<=t} v_s (k_s . r_t): the causal linear-attention product
    O = tril(R K^T) V."""
    T, N = 23, 8
    r, _, k, v, _, _ = _rand_inputs(T, N, RNG)
    ones, zeros = np.ones((T, N)), np.zeros((T, N))
    o, S = oracle.sequential(np.zeros((N, N)), r, ones, k, v, zeros, zeros)
    O_ref = np.tril(r @ k.T) @ v
    np.testing.assert_allclose(o, O_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, v.T @ k, rtol=1e-12, atol=1e-12)


def test_decay_closed_form_direct_sum():
    """a = b = 0: S_t[i][j] = S0[i][j] D(0,t][j] + sum_s v_s[i] k_s[j] D(s,t][j]
    with D(s,t] = prod_{s<u<=t} w_u, evaluated as a direct O(T^2) sum."""
    T, N = 19, 6
    r, w, k, v, _, _ = _rand_inputs(T, N, RNG)
    S0 = RNG.standard_normal((N, N))
    zeros = np.zeros((T, N))
    o, S = oracle.sequential(S0, r, w, k, v, zeros, zeros)

    def D(s, t):  # tokens numbered 1..T
        return np.prod(w[s:t], axis=0) if t > s else np.ones(N)

    for t in range(1, T + 1):
        St = S0 * D(0, t)[None, :]
        for s in range(1, t + 1):
            St = St + np.outer(v[s - 1], k[s - 1] * D(s, t))
        np.testing.assert_allclose(o[t - 1], St @ r[t - 1], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(S, St, rtol=1e-11, atol=1e-11)


def test_constant_decay_is_first_order_iir_filter():
    """a = b = 0 and a constant decay lambda_j per key channel: every state
    element follows y_t = lambda_j y_{t-1} + v_t[i] k_t[j], a first-order IIR
    filter (scipy.signal.lfilter with a = [1, -lambda_j]) with initial value
    S0[i][j]."""
    signal = pytest.importorskip("scipy.signal")
    T, N = 31, 5
    r, _, k, v, _, _ = _rand_inputs(T, N, RNG)
    lam = RNG.uniform(0.3, 0.99, N)
    S0 = RNG.standard_normal((N, N))
    zeros = np.zeros((T, N))
    _, S = oracle.sequential(S0, r, np.tile(lam, (T, 1)), k, v, zeros, zeros)
    for i in range(N):
        for j in range(N):
            x = v[:, i] * k[:, j]
            zi = signal.lfiltic([1.0], [1.0, -lam[j]], y=[S0[i, j]])
            y, _ = signal.lfilter([1.0], [1.0, -lam[j]], x, zi=zi)
            assert abs(y[-1] - S[i, j]) <= 1e-11 * max(1.0, abs(y[-1]))


def test_delta_rule_is_lms_step():
    """w = 1, a = -khat, b = beta*khat, write key k = beta*khat (unit khat):
    S_t = S_{t-1} - beta (S_{t-1} khat - v) khat^T, the delta (Widrow-Hoff /
    LMS) update on the loss 1/2 ||S khat - v||^2 with step beta."""
    T, N = 17, 7
    S = RNG.standard_normal((N, N))
    S0 = S.copy()
    khat = RNG.standard_normal((T, N))
    khat /= np.linalg.norm(khat, axis=1, keepdims=True)
    beta = RNG.uniform(0.1, 1.0, (T, 1))
    v = RNG.standard_normal((T, N))
    r = RNG.standard_normal((T, N))
    o, S_or = oracle.sequential(S0, r, np.ones((T, N)), beta * khat, v, -khat, beta * khat)
    for t in range(T):
        grad = np.outer(S @ khat[t] - v[t], khat[t])
        S = S - beta[t, 0] * grad
        np.testing.assert_allclose(o[t], S @ r[t], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(S_or, S, rtol=1e-11, atol=1e-11)


def test_delta_rule_projection_invariant():
    """w = 1, a = -khat, b = khat, write key k = khat, ||khat|| = 1: right after
    each write S_t khat_t = v_t, and S_t x = S_{t-1} x for every x orthogonal
    to khat_t."""
    T, N = 12, 8
    khat = RNG.standard_normal((T, N))
    khat /= np.linalg.norm(khat, axis=1, keepdims=True)
    v = RNG.standard_normal((T, N))
    S_prev = RNG.standard_normal((N, N))
    ones = np.ones((1, N))
    for t in range(T):
        # read the state back through o = S r with r = khat_t and r = x
        _, S_t = oracle.sequential(S_prev, khat[t:t + 1], ones, khat[t:t + 1], v[t:t + 1],
                                   -khat[t:t + 1], khat[t:t + 1])
        np.testing.assert_allclose(S_t @ khat[t], v[t], rtol=1e-12, atol=1e-12)
        x = RNG.standard_normal(N)
        x -= (x @ khat[t]) * khat[t]
        np.testing.assert_allclose(S_t @ x, S_prev @ x, rtol=1e-11, atol=1e-11)
        S_prev = S_t


def test_linearity_in_state_and_values():
    """For fixed r, w, k, a, b the map (S0, v) -> (o, S_T) is linear."""
    T, N = 9, 6
    r, w, k, v1, a, b = _rand_inputs(T, N, RNG, contractive=False)
    v2 = RNG.standard_normal((T, N))
    S1, S2 = RNG.standard_normal((N, N)), RNG.standard_normal((N, N))
    o1, F1 = oracle.sequential(S1, r, w, k, v1, a, b)
    o2, F2 = oracle.sequential(S2, r, w, k, v2, a, b)
    o3, F3 = oracle.sequential(2 * S1 - S2, r, w, k, 2 * v1 - v2, a, b)
    np.testing.assert_allclose(o3, 2 * o1 - o2, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(F3, 2 * F1 - F2, rtol=1e-10, atol=1e-10)


def test_zero_tokens_leaves_state():
    N = 4
    S0 = RNG.standard_normal((N, N))
    empty = np.zeros((0, N))
    for fn in (oracle.sequential, oracle.chunked, oracle.matprod):
        o, S = fn(S0, empty, empty, empty, empty, empty, empty)
        assert o.shape == (0, N)
        np.testing.assert_array_equal(S, S0)


# ---------------------------------------------------------------- three forms agree

@pytest.mark.parametrize("N", [2, 4, 8])
@pytest.mark.parametrize("L", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("contractive", [True, False])
def test_three_forms_agree(N, L, contractive):
    rng = np.random.default_rng(N * 100 + L * 7 + int(contractive))
    for T in (1, 4, 11, 17):
        r, w, k, v, a, b = _rand_inputs(T, N, rng, contractive)
        S0 = rng.standard_normal((N, N))
        o_s, S_s = oracle.sequential(S0, r, w, k, v, a, b)
        o_c, S_c = oracle.chunked(S0, r, w, k, v, a, b, L=L)
        scale = max(1.0, np.max(np.abs(o_s)), np.max(np.abs(S_s)))
        np.testing.assert_allclose(o_c, o_s, rtol=0, atol=1e-11 * scale)
        np.testing.assert_allclose(S_c, S_s, rtol=0, atol=1e-11 * scale)
        if L == 1:  # matprod is O(T^2 N^3): run it once per (N, contractive)
            o_m, S_m = oracle.matprod(S0, r, w, k, v, a, b)
            np.testing.assert_allclose(o_m, o_s, rtol=0, atol=1e-11 * scale)
            np.testing.assert_allclose(S_m, S_s, rtol=0, atol=1e-11 * scale)


def test_chunked_at_head_size_64_across_chunk_boundaries():
    """The kernel-sized case: N = 64, chunk 64, lengths around the boundary."""
    rng = np.random.default_rng(77)
    N = 64
    for T in (1, 63, 64, 65, 130):
        r, w, k, v, a, b = _rand_inputs(T, N, rng)
        S0 = 0.1 * rng.standard_normal((N, N))
        o_s, S_s = oracle.sequential(S0, r, w, k, v, a, b)
        o_c, S_c = oracle.chunked(S0, r, w, k, v, a, b, L=64)
        assert oracle.rel_err(o_c, o_s) < 1e-12
        assert oracle.rel_err(S_c, S_s) < 1e-12


def test_batched_units_match_single_head_calls():
    """run_units (the threaded batch entry) equals per-head calls."""
    rng = np.random.default_rng(5)
    H, N = 3, 8
    lens = [5, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    Ttot = cu[-1]
    ins = [rng.standard_normal((Ttot, H, N)) for _ in range(6)]
    ins[1] = np.exp(-np.exp(rng.normal(-0.6, 0.3, (Ttot, H, N))))
    S0 = rng.standard_normal((len(lens), H, N, N))
    o, S = oracle.prefill(S0, cu, *ins, n_threads=3)
    for s in range(len(lens)):
        for h in range(H):
            sl = slice(cu[s], cu[s + 1])
            o1, S1 = oracle.sequential(S0[s, h], *[x[sl, h] for x in ins])
            np.testing.assert_array_equal(o[sl, h], o1)
            np.testing.assert_array_equal(S[s, h], S1)


def test_checkpoints_match_matrix_product_of_the_prefix():
    """Chunk-boundary checkpoints (xLLM, "Virtual Memory for KV Cache and Model
    Weights", prefix caching): the state recorded after token every*m of a
    sequence equals the matrix-product form (an independent closed form) over
    that prefix, and a sequence whose length is a multiple of the spacing ends
    on its final state."""
    rng = np.random.default_rng(17)
    H, N, every = 2, 4, 8
    lens = [20, 8, 3, 0, 16]
    cu = np.concatenate([[0], np.cumsum(lens)])
    Ttot = int(cu[-1])
    ins = [rng.standard_normal((Ttot, H, N)) * 0.5 for _ in range(6)]
    ins[1] = rng.uniform(0.3, 1.1, (Ttot, H, N))  # non-contractive steps too
    S0 = rng.standard_normal((len(lens), H, N, N))
    o, S, ck = oracle.prefill_checkpoints(S0, cu, *ins, every=every)
    o_ref, S_ref = oracle.prefill(S0, cu, *ins)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(S, S_ref)
    assert [len(c) for c in ck] == [n // every for n in lens]
    for s_, n in enumerate(lens):
        for m, c in enumerate(ck[s_]):
            sl = slice(cu[s_], cu[s_] + every * (m + 1))
            for h in range(H):
                _, Sm = oracle.matprod(S0[s_, h], *[x[sl, h] for x in ins])
                np.testing.assert_allclose(c[h], Sm, rtol=1e-10, atol=1e-10)
        if n and n % every == 0:
            np.testing.assert_array_equal(ck[s_][-1], S[s_])


def test_multi_token_decode_states_match_matrix_product():
    """K tokens per row: per-token states equal the matrix-product form over the
    row's first k+1 tokens, outputs equal K successive single-token steps."""
    rng = np.random.default_rng(19)
    B, K, H, N = 3, 5, 2, 4
    ins = [rng.standard_normal((B, K, H, N)) * 0.5 for _ in range(6)]
    ins[1] = rng.uniform(0.3, 1.1, (B, K, H, N))
    S0 = rng.standard_normal((B, H, N, N))
    o, S, per_tok = oracle.decode_multi(S0, *ins)
    assert o.shape == (B, K, H, N) and per_tok.shape == (B, K, H, N, N)
    np.testing.assert_array_equal(per_tok[:, -1], S)
    cur = S0.copy()
    for t in range(K):
        o1, cur = oracle.decode_step(cur, *[x[:, t] for x in ins])
        np.testing.assert_array_equal(o[:, t], o1)
        np.testing.assert_array_equal(per_tok[:, t], cur)
    for bi in range(B):
        for h in range(H):
            for t in range(K):
                _, Sm = oracle.matprod(S0[bi, h], *[x[bi, :t + 1, h] for x in ins])
                np.testing.assert_allclose(per_tok[bi, t, h], Sm, rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------- the pins bite

def _planted(S0, r, w, k, v, a, b, mistake):
    """A copy of the recurrence with one deliberate mistake, for checking that
    the pins above reject it."""
    S = np.array(S0, dtype=np.float64)
    outs = []
    for t in range(r.shape[0]):
        h = S @ a[t]
        if mistake == "transposed_read":
            h = S.T @ a[t]
        if mistake == "decay_on_rows":
            Sd = w[t][:, None] * S
        elif mistake == "decay_prev_token" and t > 0:
            Sd = S * w[t - 1][None, :]
        else:
            Sd = S * w[t][None, :]
        delta = np.outer(h, b[t])
        if mistake == "dropped_delta":
            delta = 0 * delta
        if mistake == "delta_sign":
            delta = -delta
        if mistake == "swapped_kv":
            kv = np.outer(k[t], v[t])
        else:
            kv = np.outer(v[t], k[t])
        S_new = Sd + delta + kv
        o = (S if mistake == "read_before_update" else S_new) @ r[t]
        S = S_new
        outs.append(o)
    return np.array(outs), S


@pytest.mark.parametrize("mistake", ["transposed_read", "decay_on_rows", "decay_prev_token",
                                     "dropped_delta", "delta_sign", "swapped_kv",
                                     "read_before_update"])
def test_pins_catch_planted_mistakes(golden_dir, mistake):
    g = _golden(golden_dir)
    S0 = np.stack([g["S0_0"], g["S0_1"]])
    ins = [np.stack([g[f"{n}_t1"], g[f"{n}_t2"]]) for n in ("r", "w", "k", "v", "a", "b")]
    o, S2 = _planted(S0, *ins, mistake)
    expected_o = np.stack([g["o_t1"], g["o_t2"]])
    expected_S = np.stack([g["S2_0"], g["S2_1"]])
    assert not (np.array_equal(o, expected_o) and np.array_equal(S2, expected_S))


# ------------------------------------------------ bf16 state storage (rounding)
def test_round_bf16_hand_values():
    """Values worked out from the bfloat16 format (8 significant bits, float32
    exponent range): ties go to the even significand, the subnormal spacing is
    2^-133, overflow goes to inf, and a value just above a tie rounds up even
    where a detour through float32 would first land it on the tie."""
    cases = [
        (1.0, 1.0),
        (1 + 2**-8, 1.0),                   # tie between 1 and 1 + 2^-7: even is 1
        (1 + 3 * 2**-8, 1 + 2**-6),         # tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
        (1 + 2**-8 + 2**-30, 1 + 2**-7),    # above the tie (float32 would round to the tie)
        (-(1 + 5 * 2**-9), -(1 + 2**-7)),   # 1.009765625 -> nearest is 1 + 2^-7
        (1.5 * 2**-130, 1.5 * 2**-130),     # subnormal, a multiple of 2^-133
        (2**-134, 0.0),                     # half the smallest subnormal: tie, to even (0)
        (3 * 2**-134, 2 * 2**-133),         # tie between 2^-133 (odd) and 2^-132 (even)
        (3.4e38, np.inf),
        (-3.0e38, -(2**127) * (226 / 128)),  # 3.0e38 / 2^127 * 128 = 225.7 -> 226
        (0.0, 0.0),
    ]
    x = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases])
    got = oracle.round_bf16(x)
    assert np.array_equal(got, want), list(zip(x, got, want))
    assert np.isnan(oracle.round_bf16(np.array([np.nan]))[0])


def test_round_bf16_matches_the_library_conversion_on_float32_values():
    """On values that are exact in float32 the one-step rounding must equal the
    library's float32 -> bfloat16 conversion (round to nearest even)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-60, 60, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), ref)


def test_bf16_state_decode_is_the_float64_step_then_rounding():
    """The bf16-state step reads o from the unrounded state and stores the rounded
    state: with w = 1, a = b = 0 and bf16 inputs whose products are exact in
    8 bits, nothing needs rounding and it equals the plain step."""
    rng = np.random.default_rng(3)
    B, H, N = 2, 2, 8
    S0 = oracle.round_bf16(rng.standard_normal((B, H, N, N)) * 0.25)
    small = lambda: rng.integers(-3, 4, (B, H, N)).astype(np.float64)  # noqa: E731
    r, k, v = small(), small(), small() * 0.0  # v = 0: S keeps its bf16 values
    w = np.ones((B, H, N))
    a = b = np.zeros((B, H, N))
    o1, S1 = oracle.decode_step_bf16_state(S0, r, w, k, v, a, b)
    o2, S2 = oracle.decode_step(S0, r, w, k, v, a, b)
    assert np.array_equal(S1, S2) and np.array_equal(S1, S0)
    assert np.allclose(o1, o2, rtol=0, atol=0)
    # with rounding needed, the stored state is the rounded plain step and o is unrounded
    v = rng.standard_normal((B, H, N))
    o1, S1 = oracle.decode_step_bf16_state(S0, r, w, k, v, a, b)
    o2, S2 = oracle.decode_step(S0, r, w, k, v, a, b)
    assert np.array_equal(o1, o2)
    assert np.array_equal(S1, oracle.round_bf16(S2)) and not np.array_equal(S1, S2)


# ------------------------------------------------- the other order (reading B)

def test_decay_first_reading_hand_worked(golden_dir):
    """The oracle's switch for the decay-first order of the RWKV-X pseudo-code
    reproduces its own hand-worked example, and the shared example tells the two
    readings apart at the first token (the default stays reading A)."""
    g = _golden(golden_dir)
    gb = {}
    with open(os.path.join(golden_dir, "wkv7_two_tokens_n2_decay_first.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *nums = line.split()
                gb[key] = np.array([float(x) for x in nums])
    S0 = np.stack([g["S0_0"], g["S0_1"]])
    ins = [np.stack([g[f"{n}_t1"], g[f"{n}_t2"]]) for n in ("r", "w", "k", "v", "a", "b")]
    o1, S1 = oracle.sequential(S0, *[x[:1] for x in ins], reading="B")
    np.testing.assert_array_equal(o1[0], gb["o_t1"])
    np.testing.assert_array_equal(S1, np.stack([gb["S1_0"], gb["S1_1"]]))
    o, S2 = oracle.sequential(S0, *ins, reading="B")
    np.testing.assert_array_equal(o, np.stack([gb["o_t1"], gb["o_t2"]]))
    np.testing.assert_array_equal(S2, np.stack([gb["S2_0"], gb["S2_1"]]))
    oa, _ = oracle.sequential(S0, *ins)
    np.testing.assert_array_equal(oa, np.stack([g["o_t1"], g["o_t2"]]))
    assert not np.array_equal(oa[0], o[0])
    with pytest.raises(ValueError):
        oracle.sequential(S0, *ins, reading="C")


def test_decay_first_reading_agrees_where_the_orders_coincide():
    """With w = 1 (no decay) the two orders are the same map, so the closed forms
    that cannot tell them apart hold for both; with a generic decay they differ."""
    rng = np.random.default_rng(7)
    N, T = 6, 9
    r, w, k, v, a, b = _rand_inputs(T, N, rng)
    S0 = rng.standard_normal((N, N))
    ones = np.ones_like(w)
    oa, Sa = oracle.sequential(S0, r, ones, k, v, a, b)
    ob, Sb = oracle.sequential(S0, r, ones, k, v, a, b, reading="B")
    np.testing.assert_allclose(ob, oa, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(Sb, Sa, rtol=1e-13, atol=1e-13)
    oa, _ = oracle.sequential(S0, r, w, k, v, a, b)
    ob, _ = oracle.sequential(S0, r, w, k, v, a, b, reading="B")
    assert np.max(np.abs(oa - ob)) > 1e-3
