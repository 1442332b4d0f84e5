"""The seeded input generator: determinism, counter addressing, rounding."""
import numpy as np
import pytest

import workloads as wl


def test_counter_stream_is_addressable():
    full = wl.normals(7, "x", 1000)
    part = wl.normals(7, "x", 100, start=450)
    np.testing.assert_array_equal(full[450:550], part)
    assert not np.array_equal(wl.normals(7, "y", 10), full[:10])
    assert not np.array_equal(wl.normals(8, "x", 10), full[:10])


def test_normal_moments():
    x = wl.normals(3, "moments", 400_000, mean=-0.6, std=0.3)
    assert abs(x.mean() + 0.6) < 0.003
    assert abs(x.std() - 0.3) < 0.003


def test_bf16_round_to_nearest_even():
    one = np.float32(1.0)
    cases = {
        1.0: 0x3F80,
        1.0 + 2.0 ** -8: 0x3F80,           # tie -> even (mantissa 0)
        1.0 + 3 * 2.0 ** -8: 0x3F82,       # tie -> even (mantissa 2)
        1.0 + 2.0 ** -8 + 2.0 ** -20: 0x3F81,
        -2.5: 0xC020,
        0.0: 0x0000,
    }
    for val, bits in cases.items():
        assert int(wl.bf16_bits(np.array([val]))[0]) == bits, val
    assert wl.bf16_to_f32(np.array([0x3F80], dtype=np.uint16))[0] == one


def test_bf16_rounding_is_one_step_from_float64():
    """A float64 value just above a bf16 tie rounds up; a detour through float32
    would first round it onto the tie and then to even (down)."""
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40        # 1 + half a bf16 spacing + a little
    assert np.float32(x) == np.float32(1.0 + 2.0 ** -8)  # float32 lands on the tie
    assert int(wl.bf16_bits(np.array([x]))[0]) == 0x3F81
    # subnormal spacing 2^-133, overflow to inf, signs, zero
    assert int(wl.bf16_bits(np.array([2.0 ** -133]))[0]) == 0x0001
    assert int(wl.bf16_bits(np.array([1.5 * 2.0 ** -133]))[0]) == 0x0002   # tie -> even
    assert int(wl.bf16_bits(np.array([-2.0 ** -134]))[0]) == 0x8000        # tie -> even (zero)
    assert int(wl.bf16_bits(np.array([3.4e38]))[0]) == 0x7F80              # inf
    assert int(wl.bf16_bits(np.array([-0.0]))[0]) == 0x8000
    # agrees with torch's float32 -> bf16 conversion (nearest even) on float32 inputs
    torch = pytest.importorskip("torch")
    f = np.random.default_rng(3).standard_normal(100_000).astype(np.float32) * 3.0
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(wl.bf16_bits(f), want)


def test_token_inputs_recipe():
    ins = wl.token_inputs(1, "t", 16, 3, 64, dtype="f32")
    k = ins["k"].astype(np.float64)
    khat = k / np.linalg.norm(k, axis=-1, keepdims=True)
    np.testing.assert_allclose(ins["a"], -khat, rtol=1e-6, atol=1e-7)
    gate = ins["b"] / khat
    assert np.all((gate > 0) & (gate < 1))
    assert np.all((ins["w"] > 0) & (ins["w"] < 1))
    bf = wl.token_inputs(1, "t", 16, 3, 64, dtype="bf16")
    for name in wl.INPUT_NAMES:   # bf16 values are exact in bf16
        np.testing.assert_array_equal(wl.bf16_to_f32(wl.bf16_bits(bf[name])), bf[name])


def test_slot_states_depend_only_on_slot():
    a = wl.slot_states(2, "s", [5, 9], 2, 2, 8)
    b = wl.slot_states(2, "s", [9], 2, 2, 8)
    np.testing.assert_array_equal(a[1], b[0])
    assert abs(float(a.std()) - 0.1) < 0.02


def test_mixed_plan_sets_are_disjoint():
    p = wl.mixed_plan()
    dec, pre, dst = set(p["decode"]), set(p["prefill"]), set(p["fork_dst"])
    assert len(dec) == wl.MIXED_DECODE_B and len(pre) == 64 and len(dst) == 64
    assert not (dec & pre) and not (dec & dst) and not (pre & dst)
    assert set(p["snap_src"]) <= dec and set(p["fork_src"]) <= dec
    assert not (set(p["snap_src"]) & set(p["fork_src"]))
    assert p["lengths"].min() >= 1 and p["lengths"].max() <= 2048
