"""Seeded synthetic inputs for the WKV-7 state-slot workloads.

This module is shared by the tests, the benchmark and the smoke check.  It
holds the random-number generator and the input recipes only; none of the
recurrence's arithmetic lives here.

Generator (a counter-based stream, so any element can be produced on its own):
  * splitmix64 finaliser  mix(z) = z ^ (z>>30) * 0xBF58476D1CE4E5B9 ;
    z ^ (z>>27) * 0x94D049BB133111EB ; z ^ (z>>31)   (all mod 2^64);
  * a stream is keyed by (seed, tag): key = mix(seed * G ^ fnv1a64(tag)) with
    G = 0x9E3779B97F4A7C15, and its i-th 64-bit word is mix(key + (i+1) * G);
  * a uniform in (0, 1] is ((word >> 11) + 1) * 2^-53;
  * a normal is Box-Muller on the uniforms of words 2i and 2i+1:
    sqrt(-2 ln u1) * cos(2 pi u2), evaluated in float64.

Input recipe per (token, head), in float64, then rounded once to the
arithmetic type the kernel consumes (round-to-nearest-even for bf16):
  r, k, v ~ N(0, 1);  khat = k / ||k|| (L2 over the N channels of that token
  and head);  a = -khat;  b = khat * sigmoid(N(0, 1)) (an independent draw per
  element);  w = exp(-exp(N(-0.6, 0.3)));  the write key is the raw k.
Initial slot states ~ N(0, 0.1) in float32 (second parameter = std).
The recipe follows the workload descriptions of the WKV-7 state-slot engine:
a single layer of 4 heads (T = 64), a 12-layer x 12-head batched decode over
a 1024-slot pool, an 8 x 4096-token chunked prefill with 32 heads, a mixed
serving step on a 4096-slot pool and a 32-layer x 64-head decode sweep.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _fnv1a64(tag: str) -> int:
    h = 0xCBF29CE484222325
    for ch in tag.encode("utf-8"):
        h ^= ch
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def stream_key(seed: int, tag: str) -> np.uint64:
    z = np.array([((int(seed) * 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF) ^ _fnv1a64(tag)],
                 dtype=np.uint64)
    return _mix(z)[0]


def words(key: np.uint64, start: int, n: int) -> np.ndarray:
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + i * _G)


def words_at(key: np.uint64, idx: np.ndarray) -> np.ndarray:
    """Words at arbitrary stream positions idx (same values as words())."""
    i = np.asarray(idx, dtype=np.uint64) + np.uint64(1)
    with np.errstate(over="ignore"):
        return _mix(key + i * _G)


def uniforms(key: np.uint64, start: int, n: int) -> np.ndarray:
    wds = words(key, start, n)
    return ((wds >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normals(seed: int, tag: str, n: int, mean: float = 0.0, std: float = 1.0,
            start: int = 0) -> np.ndarray:
    """n normals of stream (seed, tag), elements start..start+n-1, float64."""
    key = stream_key(seed, tag)
    out = np.empty(n, dtype=np.float64)
    for b0 in range(0, n, _BLOCK):
        m = min(_BLOCK, n - b0)
        u = uniforms(key, 2 * (start + b0), 2 * m)
        u1, u2 = u[0::2], u[1::2]
        out[b0:b0 + m] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return mean + std * out


def normals_at(seed: int, tag: str, idx: np.ndarray, mean: float = 0.0,
               std: float = 1.0) -> np.ndarray:
    """Normals of stream (seed, tag) at element positions idx (any shape);
    normals_at(s, t, arange(a, b)) == normals(s, t, b - a, start=a)."""
    key = stream_key(seed, tag)
    idx = np.asarray(idx, dtype=np.int64)
    flat = idx.reshape(-1)
    out = np.empty(flat.size, dtype=np.float64)
    for b0 in range(0, flat.size, _BLOCK):
        e = flat[b0:b0 + _BLOCK].astype(np.uint64)
        w1 = words_at(key, 2 * e)
        w2 = words_at(key, 2 * e + np.uint64(1))
        u1 = ((w1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = ((w2 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        out[b0:b0 + e.size] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return (mean + std * out).reshape(idx.shape)


# --------------------------------------------------------------------------
# rounding helpers
# --------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round values to bf16 in one step (nearest, ties to even) and return the
    uint16 bit patterns.  The input is taken as float64 (float32 values widen
    exactly), so a float64 draw is rounded once, with no float32 stop on the way.

    A finite x = m 2^e (frexp: 0.5 <= |m| < 1) is a multiple of 2^(e-8) once it
    is rounded to bf16's 8 significant bits; below 2^-126 the bf16 spacing stays
    2^-133.  Scaling by a power of two and np.rint (ties to even) are exact, and
    the rounded value is exactly a float32 whose upper 16 bits are the bf16
    pattern.  Magnitudes that round past the largest finite bf16 become inf."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = v.copy()
    fin = np.isfinite(v) & (v != 0.0)
    xf = v[fin]
    _, e = np.frexp(xf)
    spacing = np.ldexp(1.0, np.maximum(e - 8, -133))
    y = np.rint(xf / spacing) * spacing
    y = np.where(np.abs(y) > 3.3895313892515355e38, np.copysign(np.inf, y), y)
    out[fin] = y
    f = out.astype(np.float32)  # exact: every bf16 value is a float32 value
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round to the kernel's input type; returns float32 values exactly equal
    to what the kernel sees."""
    if dtype == "bf16":
        return bf16_to_f32(bf16_bits(x))
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# recipes
# --------------------------------------------------------------------------

INPUT_NAMES = ("r", "w", "k", "v", "a", "b")


def token_inputs(seed: int, tag: str, n_tok: int, H: int, N: int,
                 dtype: str = "bf16", heads=None) -> dict:
    """Inputs r, w, k, v, a, b of shape [n_tok, H, N] as float32 arrays whose
    values are exactly representable in `dtype` ("bf16" or "f32").  With
    `heads`, only those heads are produced ([n_tok, len(heads), N]), with the
    same values they have in the full tensor."""
    if heads is None:
        shape = (n_tok, H, N)
        n = n_tok * H * N

        def draw(t, mean=0.0, std=1.0):
            return normals(seed, tag + t, n, mean=mean, std=std).reshape(shape)
    else:
        hs = np.asarray(list(heads), dtype=np.int64)
        idx = ((np.arange(n_tok, dtype=np.int64)[:, None, None] * H + hs[None, :, None]) * N
               + np.arange(N, dtype=np.int64)[None, None, :])

        def draw(t, mean=0.0, std=1.0):
            return normals_at(seed, tag + t, idx, mean=mean, std=std)
    r = draw("/r")
    k = draw("/k")
    v = draw("/v")
    g = draw("/b_gate")
    x = draw("/w", mean=-0.6, std=0.3)
    norm = np.sqrt(np.sum(k * k, axis=-1, keepdims=True))
    norm = np.where(norm > 0.0, norm, 1.0)
    khat = k / norm
    a = -khat
    b = khat * (1.0 / (1.0 + np.exp(-g)))
    w = np.exp(-np.exp(x))
    vals = {"r": r, "w": w, "k": k, "v": v, "a": a, "b": b}
    return {name: round_to(vals[name], dtype) for name in INPUT_NAMES}


def slot_states(seed: int, tag: str, slot_ids, n_layers: int, H: int, N: int,
                layers=None, std: float = 0.1) -> np.ndarray:
    """Initial fp32 states of the given slots, [len(slot_ids), L, H, N, N].
    The values of a slot depend only on (seed, tag, slot id, layer), not on
    which other slots are requested."""
    layers = range(n_layers) if layers is None else layers
    per = H * N * N
    out = np.empty((len(slot_ids), len(layers), H, N, N), dtype=np.float32)
    for li, layer in enumerate(layers):
        for si, slot in enumerate(slot_ids):
            out[si, li] = normals(seed, f"{tag}/layer{layer}", per, std=std,
                                  start=int(slot) * per).astype(np.float32).reshape(H, N, N)
    return out


def distinct_slots(seed: int, tag: str, n: int, pool: int) -> np.ndarray:
    """n distinct slot ids drawn uniformly from [0, pool) (a seeded permutation
    prefix: sort pool uniforms, take the first n indices)."""
    u = uniforms(stream_key(seed, tag), 0, pool)
    return np.argsort(u, kind="stable")[:n].astype(np.int32)


def ragged_lengths(seed: int, tag: str, n: int, lo: int, hi: int) -> np.ndarray:
    """n lengths uniform on the integers lo..hi."""
    u = uniforms(stream_key(seed, tag), 0, n)
    return (lo + np.floor(u * (hi - lo + 1) - 1e-12)).astype(np.int64).clip(lo, hi)


def cu_seqlens(lengths) -> np.ndarray:
    out = np.zeros(len(lengths) + 1, dtype=np.int32)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return out


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    n_layers: int
    H: int
    N: int
    n_slots: int
    description: str


SINGLE_LAYER = Workload("single_layer_4h_T64", 1, 1, 4, 64, 2,
                        "1 layer, 4 heads x 64, 2 slots, T=64 sequential tokens, fp32 "
                        "inputs, zero initial state")
DECODE_12L = Workload("decode_12L_12H_B256_pool1024", 2, 12, 12, 64, 1024,
                      "batched decode: 12 layers x 12 heads x 64, 256 active slots "
                      "of a 1024-slot pool at random ids, N(0,0.1) states, bf16 inputs")
PREFILL_8x4096 = Workload("prefill_8x4096_32H", 3, 1, 32, 64, 8,
                          "chunked prefill: 8 sequences x 4096 tokens, 32 heads x 64, "
                          "1 layer, bf16 inputs, zero start state, chunk 64")
MIXED = Workload("mixed_serving_pool4096_32H", 4, 1, 32, 64, 4096,
                 "mixed serving step: 4096-slot pool, 32 heads x 64, 1 layer; "
                 "decode 1024 slots + ragged prefill of 64 sequences U[1,2048] into "
                 "freshly created slots + fork 64 + snapshot/restore 64")
SWEEP_32L = Workload("decode_sweep_32L_64H", 5, 32, 64, 64, 4096,
                     "decode sweep: 32 layers x 64 heads x 64, batch 1/64/512/2048/4096, "
                     "fp32 state 1 MiB per slot-layer")

MIXED_DECODE_B = 1024
MIXED_PREFILL_SEQS = 64
MIXED_MAX_LEN = 2048
MIXED_VERB_N = 64


def mixed_plan(seed: int = MIXED.seed, n_slots: int = MIXED.n_slots,
               decode_b: int = MIXED_DECODE_B, n_seqs: int = MIXED_PREFILL_SEQS,
               max_len: int = MIXED_MAX_LEN, verb_n: int = MIXED_VERB_N) -> dict:
    """Slot sets of the mixed serving step, all disjoint:
    decode slots (decode_b), snapshot/restore slots (verb_n, a subset of the
    decode slots), fork sources (verb_n decode slots) -> fork targets (verb_n
    free slots), prefill targets (n_seqs free slots), and the prefill lengths."""
    perm = distinct_slots(seed, "mixed/perm", decode_b + n_seqs + verb_n, n_slots)
    decode = perm[:decode_b]
    prefill = perm[decode_b:decode_b + n_seqs]
    fork_dst = perm[decode_b + n_seqs:decode_b + n_seqs + verb_n]
    snap_src = decode[:verb_n]
    fork_src = decode[verb_n:2 * verb_n]
    lengths = ragged_lengths(seed, "mixed/lengths", n_seqs, 1, max_len)
    return {"decode": decode, "prefill": prefill, "fork_src": fork_src,
            "fork_dst": fork_dst, "snap_src": snap_src, "lengths": lengths}


def token_inputs_device(seed: int, n_tok: int, H: int, N: int, device, dtype=None,
                        generator_offset: int = 0):
    """The same recipe drawn with torch's seeded device generator (Philox), for
    inputs too large to draw on the host.  Values differ from token_inputs();
    only shapes and distributions match.  Returns [r, w, k, v, a, b] tensors
    [n_tok, H, N] of `dtype` (default bfloat16) on `device`."""
    import torch
    dtype = torch.bfloat16 if dtype is None else dtype
    g = torch.Generator(device=device).manual_seed(int(seed) * 1000003 + generator_offset)
    shape = (n_tok, H, N)
    r = torch.randn(shape, device=device, generator=g)
    k = torch.randn(shape, device=device, generator=g)
    v = torch.randn(shape, device=device, generator=g)
    gate = torch.randn(shape, device=device, generator=g)
    x = torch.randn(shape, device=device, generator=g) * 0.3 - 0.6
    khat = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    a = -khat
    b = khat * torch.sigmoid(gate)
    w = torch.exp(-torch.exp(x))
    return [t.to(dtype).contiguous() for t in (r, w, k, v, a, b)]
