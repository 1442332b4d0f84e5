"""WKV-7 oracle: the plain double-precision CPU reference.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's ``smoke()`` check and
the benchmark's CPU-baseline leg may import this package.  The product path
(``rwkv_wkv_gb300`` and its C-ABI library) never imports, links or calls it,
and the two share no code: this side is plain C in ``wkv7_oracle.c`` plus the
array plumbing below.

The recurrence (RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta Rule)"),
per head with state S[i][j] (i value index, j key index):

    h = S a ;  S <- S diag(w) + h b^T + v k^T ;  o = S r

Pool-level helpers follow the state-slot model of "wkvm: state-slot inference
for RWKV, GDN and Mamba hybrids" ("The allocation unit wkvm changes"): a slot is
a fixed-size block holding one state per (layer, head); decode advances each
listed slot by one token, prefill advances each listed slot by its sequence.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wkv7_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile wkv7_oracle.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ll = ctypes.c_longlong
            for name in ("wkv7_oracle_sequential", "wkv7_oracle_matprod",
                         "wkv7_oracle_sequential_decay_first"):
                f = getattr(lib, name)
                f.restype = ctypes.c_int
                f.argtypes = [ctypes.c_int, ctypes.c_int, dp, ll, ll] + [dp] * 7
            f = lib.wkv7_oracle_chunked
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, ll, ll] + [dp] * 7
            f = lib.wkv7_oracle_sequential_batch
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_int, ctypes.c_int, dp, ctypes.POINTER(ll),
                          ctypes.POINTER(ctypes.c_int), ll] + [dp] * 7 + [ctypes.c_int]
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x: np.ndarray):
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _one_head(fn_name, S0, r, w, k, v, a, b, extra=()):
    """Run one head over T tokens; inputs are [T, N], S0 is [N, N]."""
    S = _f64(S0).copy()
    ins = [_f64(x) for x in (r, w, k, v, a, b)]
    T, N = ins[0].shape
    for x in ins:
        if x.shape != (T, N):
            raise ValueError("inputs must all be [T, N]")
    if S.shape != (N, N):
        raise ValueError("state must be [N, N]")
    o = np.zeros((T, N), dtype=np.float64)
    fn = getattr(_load(), fn_name)
    args = [N, T] + list(extra) + [_ptr(S), 0, N] + [_ptr(x) for x in ins] + [_ptr(o)]
    rc = fn(*args)
    if rc:
        raise RuntimeError(f"{fn_name} failed with code {rc}")
    return o, S


def sequential(S0, r, w, k, v, a, b, reading: str = "A"):
    """Sequential recurrence on one head. Returns (o [T,N], S_T [N,N]).

    reading "A" (the default, the one the build follows): h = S a is read on the
    state before the decay.  reading "B": the order of the RWKV-X pseudo-code
    ("WKV-7 Kernel (Generalized Delta Rule)"), which decays the state first and
    then reads h = (S diag(w)) a.  "B" exists only to measure how far the two
    readings lie apart; nothing else uses it."""
    if reading == "A":
        return _one_head("wkv7_oracle_sequential", S0, r, w, k, v, a, b)
    if reading == "B":
        return _one_head("wkv7_oracle_sequential_decay_first", S0, r, w, k, v, a, b)
    raise ValueError(f"reading must be 'A' or 'B', not {reading!r}")


def matprod(S0, r, w, k, v, a, b):
    """Matrix-product form on one head (tiny inputs only). Returns (o, S_T)."""
    return _one_head("wkv7_oracle_matprod", S0, r, w, k, v, a, b)


def chunked(S0, r, w, k, v, a, b, L: int = 64):
    """Chunked WY/UT form on one head, chunks of L from the first token."""
    fn = _load().wkv7_oracle_chunked
    S = _f64(S0).copy()
    ins = [_f64(x) for x in (r, w, k, v, a, b)]
    T, N = ins[0].shape
    o = np.zeros((T, N), dtype=np.float64)
    rc = fn(N, T, int(L), _ptr(S), 0, N, *[_ptr(x) for x in ins], _ptr(o))
    if rc:
        raise RuntimeError(f"wkv7_oracle_chunked failed with code {rc}")
    return o, S


def run_units(S, base, T, tok_stride, inputs, n_threads: int = 1):
    """Sequential recurrence on many independent heads at once.

    S: [n_units, N, N] float64, updated in place.  base[u], T[u]: first element
    offset and token count of unit u; token t of unit u, channel j is at
    x[base[u] + t*tok_stride + j] for every x in inputs = (r, w, k, v, a, b)
    (flat float64 arrays).  Returns o with the same flat layout as the inputs.
    """
    S = np.ascontiguousarray(S, dtype=np.float64)
    n_units, N, _ = S.shape
    base = np.ascontiguousarray(base, dtype=np.int64)
    T = np.ascontiguousarray(T, dtype=np.int32)
    ins = [_f64(x).reshape(-1) for x in inputs]
    o = np.zeros_like(ins[0])
    rc = _load().wkv7_oracle_sequential_batch(
        N, n_units, _ptr(S), base.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
        T.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), int(tok_stride),
        *[_ptr(x) for x in ins], _ptr(o), int(n_threads))
    if rc:
        raise RuntimeError(f"wkv7_oracle_sequential_batch failed with code {rc}")
    return o, S


def decode_step(states, r, w, k, v, a, b, n_threads: int = 1):
    """One decode token for B rows of H heads.

    states: [B, H, N, N] (the gathered slot states of one layer); inputs
    [B, H, N].  Returns (o [B, H, N], new states [B, H, N, N]) in float64.
    """
    st = _f64(states)
    B, H, N, _ = st.shape
    S = st.reshape(B * H, N, N).copy()
    base = np.arange(B * H, dtype=np.int64) * N
    T = np.ones(B * H, dtype=np.int32)
    o, S = run_units(S, base, T, N, (r, w, k, v, a, b), n_threads)
    return o.reshape(B, H, N), S.reshape(B, H, N, N)


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even, in one
    step (no intermediate float32 rounding).  bfloat16 keeps the float32
    exponent range with 8 significant bits: a finite x with 2^e <= |x| < 2^(e+1)
    is a multiple of 2^(e-7); below 2^-126 the spacing stays 2^-133 (subnormal
    values); magnitudes that round past the largest finite value become inf."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x) & (x != 0.0)
    xf = x[fin]
    e = np.floor(np.log2(np.abs(xf)))
    # log2 can misplace exact powers of two by one ulp: fix e so 2^e <= |x| < 2^(e+1)
    e = np.where(np.abs(xf) < np.exp2(e), e - 1, e)
    e = np.where(np.abs(xf) >= np.exp2(e + 1), e + 1, e)
    q = np.exp2(np.maximum(e - 7, -133.0))   # spacing of bf16 values around x
    y = np.rint(xf / q) * q                   # rint: nearest, ties to even
    big = np.abs(y) > 3.3895313892515355e38   # (2 - 2^-7) * 2^127, the largest finite
    y = np.where(big, np.copysign(np.inf, y), y)
    out[fin] = y
    return out


def decode_step_bf16_state(states, r, w, k, v, a, b, n_threads: int = 1):
    """One decode token for a pool whose states are stored in bfloat16: the step
    runs in float64 from the (exactly widened) stored state, o is read from the
    unrounded new state, and the new state is stored rounded to bfloat16.
    Returns (o [B, H, N], new stored states [B, H, N, N]) in float64."""
    o, S = decode_step(states, r, w, k, v, a, b, n_threads)
    return o, round_bf16(S)


def prefill(states, cu_seqlens, r, w, k, v, a, b, n_threads: int = 1):
    """Ragged prefill: sequence s covers tokens cu_seqlens[s]..cu_seqlens[s+1].

    states: [S, H, N, N] start states; inputs [Ttot, H, N].
    Returns (o [Ttot, H, N], final states [S, H, N, N]) in float64.
    """
    st = _f64(states)
    nS, H, N, _ = st.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    S = st.reshape(nS * H, N, N).copy()
    base = np.empty(nS * H, dtype=np.int64)
    T = np.empty(nS * H, dtype=np.int32)
    for s in range(nS):
        for h in range(H):
            base[s * H + h] = cu[s] * H * N + h * N
            T[s * H + h] = cu[s + 1] - cu[s]
    o, S = run_units(S, base, T, H * N, (r, w, k, v, a, b), n_threads)
    Ttot = np.asarray(r).shape[0]
    return o.reshape(Ttot, H, N), S.reshape(nS, H, N, N)


def prefill_checkpoints(states, cu_seqlens, r, w, k, v, a, b, n_threads: int = 1,
                        every: int = 64):
    """Ragged prefill that also returns the state after every `every`-th token.

    The sequential recurrence is run segment by segment (segment m of sequence
    s covers its tokens every*m .. every*(m+1)-1) with the state carried from
    one segment to the next, so each recorded state is the recurrence's state
    after that token (the stored linear-state checkpoint of a chunked prefill:
    xLLM, "Virtual Memory for KV Cache and Model Weights", prefix caching).
    Returns (o [Ttot, H, N], final states [S, H, N, N], checkpoints) where
    checkpoints[s] is a list of len_s // every arrays [H, N, N].
    """
    st = _f64(states)
    nS, H, N, _ = st.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = np.diff(cu)
    S = st.reshape(nS * H, N, N).copy()
    Ttot = np.asarray(r).shape[0]
    o = np.zeros(Ttot * H * N)
    ckpts = [[] for _ in range(nS)]
    n_seg = int((lens.max() + every - 1) // every) if nS else 0
    for m in range(n_seg):
        base = np.empty(nS * H, dtype=np.int64)
        T = np.empty(nS * H, dtype=np.int32)
        for s_ in range(nS):
            t_seg = int(max(0, min(every, lens[s_] - every * m)))
            for h in range(H):
                base[s_ * H + h] = (cu[s_] + every * m) * H * N + h * N
                T[s_ * H + h] = t_seg
        o_seg, S = run_units(S, base, T, H * N, (r, w, k, v, a, b), n_threads)
        o += o_seg  # each token is written by exactly one segment
        for s_ in range(nS):
            if lens[s_] >= every * (m + 1):
                ckpts[s_].append(S.reshape(nS, H, N, N)[s_].copy())
    return o.reshape(Ttot, H, N), S.reshape(nS, H, N, N), ckpts


def decode_multi(states, r, w, k, v, a, b, n_threads: int = 1):
    """K consecutive tokens on each of B rows (the verify pass of speculative
    decoding: rvLLM README, "Speculative decoding").

    states: [B, H, N, N]; inputs [B, K, H, N].  Returns (o [B, K, H, N], final
    states [B, H, N, N], per-token states [B, K, H, N, N]) in float64, where
    per-token state k is the state right after token k.
    """
    st = _f64(states)
    B, H, N, _ = st.shape
    K = np.asarray(r).shape[1]
    flat = [_f64(x).reshape(B * K, H, N) for x in (r, w, k, v, a, b)]
    cu = np.arange(B + 1, dtype=np.int64) * K
    o, S, ck = prefill_checkpoints(st, cu, *flat, n_threads=n_threads, every=1)
    per_tok = np.stack([np.stack(c) for c in ck]) if B and K else np.zeros((B, K, H, N, N))
    return o.reshape(B, K, H, N), S, per_tok


def rel_err(x, ref) -> float:
    """Normwise-max relative error of one tensor: max|x - ref| / max|ref|, taken
    over all entries (the plain absolute max when ref is all zero).  The shapes
    must match exactly: no broadcasting."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.shape != ref.shape:
        raise ValueError(f"rel_err: shape {x.shape} against reference shape {ref.shape}")
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(x - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


def rel_err_slices(x, ref, lead: int, floor_frac: float = 0.0) -> np.ndarray:
    """rel_err of every slice over the first `lead` axes: for x, ref of shape
    [d0, .., d_{lead-1}, ...] the array [d0, .., d_{lead-1}] of normwise-max
    errors of x[i0, .., i_{lead-1}] against ref[i0, .., i_{lead-1}], so that a
    slice whose values are small is judged against its own scale.

    With floor_frac > 0 a slice's denominator is at least floor_frac times the
    median over slices of max|ref slice|: a slice whose result nearly cancels
    (an output o = v (k . r) with k . r close to 0, say) carries the rounding of
    its summands, which are of the typical size, not of its own tiny size."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.shape != ref.shape:
        raise ValueError(f"rel_err_slices: shape {x.shape} against reference shape {ref.shape}")
    if lead < 0 or lead > ref.ndim:
        raise ValueError(f"rel_err_slices: lead {lead} for {ref.ndim} axes")
    out_shape = ref.shape[:lead]
    xf = x.reshape(int(np.prod(out_shape, dtype=np.int64)), -1)
    rf = ref.reshape(xf.shape)
    if rf.shape[1] == 0:
        return np.zeros(out_shape)
    num = np.max(np.abs(xf - rf), axis=1)
    den = np.max(np.abs(rf), axis=1)
    if floor_frac > 0.0:
        den = np.maximum(den, floor_frac * float(np.median(den)))
    res = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
    return res.reshape(out_shape)


def rel_err_segments(x, ref, cu, floor_frac: float = 0.0) -> np.ndarray:
    """rel_err of every (sequence, head) of packed [tokens][heads][...] arrays:
    sequence q covers tokens cu[q] .. cu[q+1]-1.  Returns [n_seqs, heads]
    (0 for an empty sequence); floor_frac as in rel_err_slices, the median
    taken over the non-empty (sequence, head) slices."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.shape != ref.shape:
        raise ValueError(f"rel_err_segments: shape {x.shape} against reference shape {ref.shape}")
    cu = np.asarray(cu, dtype=np.int64)
    n, H = len(cu) - 1, ref.shape[1]
    if n < 0 or (n > 0 and (cu[0] != 0 or cu[-1] != ref.shape[0] or np.any(np.diff(cu) < 0))):
        raise ValueError("rel_err_segments: cu must run from 0 to the token count, non-decreasing")
    num = np.zeros((n, H))
    den = np.zeros((n, H))
    filled = np.diff(cu) > 0
    axes = tuple(i for i in range(ref.ndim) if i != 1)
    for q in np.nonzero(filled)[0]:
        a, b = int(cu[q]), int(cu[q + 1])
        num[q] = np.max(np.abs(x[a:b] - ref[a:b]), axis=axes)
        den[q] = np.max(np.abs(ref[a:b]), axis=axes)
    if floor_frac > 0.0 and filled.any():
        den = np.maximum(den, floor_frac * float(np.median(den[filled])))
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)


def elementwise_rel(x, ref, floor: float = 1e-6) -> np.ndarray:
    """Elementwise relative error |x - ref| / (|ref| + floor * max|ref|): the
    per-entry companion of rel_err.  The floor (relative to the tensor's largest
    entry) keeps entries that are zero, or nearly, from dividing by zero."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.shape != ref.shape:
        raise ValueError(f"elementwise_rel: shape {x.shape} against reference shape {ref.shape}")
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    den = np.abs(ref) + floor * scale
    diff = np.abs(x - ref)
    return np.where(den > 0, diff / np.where(den > 0, den, 1.0), diff)
