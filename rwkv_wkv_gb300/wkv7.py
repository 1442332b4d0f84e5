"""Python binding of libwkv7 (ctypes).  Argument marshalling only: every step
of the recurrence and of the slot verbs runs in the library's CUDA kernels.
PyTorch supplies device memory (the pool buffer, the caller's tensors) and the
current CUDA stream; nothing here computes.

The C contract (layouts, ownership, errors) is documented in include/wkv7.h.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libwkv7.so")

F32, BF16 = 0, 1
DEV_OK, DEV_BAD_SLOT, DEV_BAD_SEQLENS, DEV_WAIT_TIMEOUT, DEV_DECAY_RANGE, DEV_DUP_SLOT = 0, 1, 2, 3, 4, 5
TABLE_SLOTS, TABLE_SNAPSHOTS = 0, 1
HEAD_SIZE = 64
_HEADER_BYTES = 256

STATUS_NAMES = {
    0: "OK", 1: "ERR_INVALID_ARG", 2: "ERR_BAD_SLOT", 3: "ERR_DUP_SLOT", 4: "ERR_POOL_FULL",
    5: "ERR_BAD_SEQLENS", 6: "ERR_CUDA", 7: "ERR_UNSUPPORTED", 8: "ERR_DEVICE_STATUS",
    9: "ERR_TIMEOUT", 10: "ERR_NO_MEMORY",
}


class Wkv7Error(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        msg = f"{what}: {self.name}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class PoolDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_size", ctypes.c_int32), ("n_slots", ctypes.c_int32),
                ("n_snapshots", ctypes.c_int32), ("device_buffer", ctypes.c_void_p),
                ("buffer_bytes", ctypes.c_size_t), ("state_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32)]


# name -> (restype, argtypes)
_P, _I32, _VP = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)
_SIGS = {
    "wkv7_pool_required_bytes": (ctypes.c_size_t, [ctypes.POINTER(PoolDesc)]),
    "wkv7_pool_create": (ctypes.c_int, [ctypes.POINTER(PoolDesc), ctypes.POINTER(ctypes.c_void_p)]),
    "wkv7_pool_destroy": (ctypes.c_int, [_P]),
    "wkv7_pool_get_desc": (ctypes.c_int, [_P, ctypes.POINTER(PoolDesc)]),
    "wkv7_slot_bytes": (ctypes.c_size_t, [_P]),
    "wkv7_pool_state_ptr": (ctypes.c_int, [_P, _I32, _I32, ctypes.POINTER(ctypes.c_void_p)]),
    "wkv7_pool_snapshot_ptr": (ctypes.c_int, [_P, _I32, _I32, ctypes.POINTER(ctypes.c_void_p)]),
    "wkv7_slot_alloc": (ctypes.c_int, [_P, _I32, _I32P]),
    "wkv7_slot_free": (ctypes.c_int, [_P, _I32, _I32P]),
    "wkv7_snapshot_alloc": (ctypes.c_int, [_P, _I32, _I32P]),
    "wkv7_snapshot_free": (ctypes.c_int, [_P, _I32, _I32P]),
    "wkv7_slot_count_free": (ctypes.c_int32, [_P]),
    "wkv7_snapshot_count_free": (ctypes.c_int32, [_P]),
    "wkv7_slot_is_allocated": (ctypes.c_int, [_P, _I32, _I32P]),
    "wkv7_slot_create": (ctypes.c_int, [_P, _I32, _I32P, _VP]),
    "wkv7_slot_reset": (ctypes.c_int, [_P, _VP, _I32, _VP]),
    "wkv7_slot_snapshot": (ctypes.c_int, [_P, _VP, _VP, _I32, _VP]),
    "wkv7_slot_restore": (ctypes.c_int, [_P, _VP, _VP, _I32, _VP]),
    "wkv7_slot_fork": (ctypes.c_int, [_P, _VP, _VP, _I32, _VP]),
    "wkv7_slot_hibernate": (ctypes.c_int, [_P, _VP, _I32, _VP, ctypes.c_size_t, _VP]),
    "wkv7_slot_resume": (ctypes.c_int, [_P, _VP, ctypes.c_size_t, _VP, _I32, _VP]),
    "wkv7_decode_step": (ctypes.c_int, [_P, _I32, _VP, _I32, ctypes.c_int] + [_VP] * 7 + [_VP]),
    "wkv7_prefill": (ctypes.c_int, [_P, _I32, _VP, _VP, _I32, _I32, _I32, ctypes.c_int]
                     + [_VP] * 7 + [_VP]),
    "wkv7_prefill_sequential": (ctypes.c_int, [_P, _I32, _VP, _VP, _I32, _I32, _I32, ctypes.c_int]
                                + [_VP] * 7 + [_VP]),
    "wkv7_decode_multi": (ctypes.c_int, [_P, _I32, _VP, _I32, _I32, ctypes.c_int] + [_VP] * 7
                          + [_VP, _VP]),
    "wkv7_prefill_checkpointed": (ctypes.c_int, [_P, _I32, _VP, _VP, _I32, _I32, _I32, ctypes.c_int]
                                  + [_VP] * 7 + [_VP, _VP, _I32, _VP]),
    "wkv7_validate_ids": (ctypes.c_int, [_P, _I32, _VP, _I32, _VP, _I32, _VP]),
    "wkv7_validate_ids_noalloc": (ctypes.c_int, [_I32, _VP, _I32, _VP, _I32, _VP, _VP]),
    "wkv7_get_device_status": (ctypes.c_int, [_P, _VP, _I32, _I32P]),
    "wkv7_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "wkv7_last_error": (ctypes.c_char_p, []),
    "wkv7_launch_count": (ctypes.c_uint64, []),
    "wkv7_version": (ctypes.c_int32, []),
    "wkv7_test_force_wait_timeout": (ctypes.c_int, [_I32]),
}

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libwkv7.so; raises if it has not been built.  There is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m rwkv_wkv_gb300.build` "
                          "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def exported_symbols() -> list[str]:
    return list(_SIGS)


def _check(status: int, what: str):
    if status != 0:
        detail = ""
        if status == 6:
            detail = load_library().wkv7_last_error().decode(errors="replace")
        raise Wkv7Error(status, what, detail)


def launch_count() -> int:
    return int(load_library().wkv7_launch_count())


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _ids_host(ids) -> ctypes.Array:
    vals = [int(x) for x in ids]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals), len(vals)


def _dev_i32(t: torch.Tensor, name: str, device) -> int:
    if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or not t.is_cuda:
        raise TypeError(f"{name} must be an int32 CUDA tensor")
    if t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous on {device}")
    return t.data_ptr()


class Pool:
    """A pool of fixed-size WKV-7 state slots on one GPU.

    States live in one torch-allocated device buffer: ``states`` is a float32
    (or, with state_dtype="bf16", bfloat16) view [n_slots, n_layers, n_heads,
    64, 64] and ``snapshots`` the same for the parked copies (S[i][j]: i =
    value row, j = key column).  Outputs o are float32, or bfloat16 with
    out_dtype="bf16" (the float32 readout rounded to nearest even).
    """

    def __init__(self, n_layers: int, n_heads: int, n_slots: int, n_snapshots: int = 0,
                 head_size: int = HEAD_SIZE, device=None, state_dtype: str = "f32",
                 out_dtype: str = "f32"):
        self._lib = load_library()
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        self.n_layers, self.n_heads, self.head_size = n_layers, n_heads, head_size
        self.n_slots, self.n_snapshots = n_slots, n_snapshots
        if state_dtype not in ("f32", "bf16"):
            raise ValueError("state_dtype must be 'f32' or 'bf16'")
        if out_dtype not in ("f32", "bf16"):
            raise ValueError("out_dtype must be 'f32' or 'bf16'")
        self.state_dtype, self.out_dtype = state_dtype, out_dtype
        self.o_torch_dtype = torch.bfloat16 if out_dtype == "bf16" else torch.float32
        desc = PoolDesc(n_layers, n_heads, head_size, n_slots, n_snapshots, None, 0,
                        BF16 if state_dtype == "bf16" else F32, BF16 if out_dtype == "bf16" else F32)
        nbytes = self._lib.wkv7_pool_required_bytes(ctypes.byref(desc))
        if nbytes == 0:
            raise Wkv7Error(1, "Pool", "invalid description")
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.buffer[:_HEADER_BYTES].zero_()
        desc.device_buffer = self.buffer.data_ptr()
        desc.buffer_bytes = nbytes
        handle = ctypes.c_void_p()
        _check(self._lib.wkv7_pool_create(ctypes.byref(desc), ctypes.byref(handle)), "pool_create")
        self._h = handle
        self.slot_bytes = int(self._lib.wkv7_slot_bytes(self._h))
        tdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
        per_slot = self.slot_bytes // tdt.itemsize
        body = self.buffer[_HEADER_BYTES:].view(tdt)
        shape = (n_layers, n_heads, head_size, head_size)
        self.states = body[: n_slots * per_slot].view(n_slots, *shape)
        self.snapshots = body[n_slots * per_slot:(n_slots + n_snapshots) * per_slot].view(
            n_snapshots, *shape)

    # -------------------------------------------------------------- lifetime
    def close(self):
        if getattr(self, "_h", None):
            _check(self._lib.wkv7_pool_destroy(self._h), "pool_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ------------------------------------------------------------ slot table
    def alloc(self, n: int) -> list[int]:
        arr = (ctypes.c_int32 * max(1, n))()
        _check(self._lib.wkv7_slot_alloc(self._h, n, arr), "slot_alloc")
        return list(arr[:n])

    def free(self, ids) -> None:
        arr, n = _ids_host(ids)
        _check(self._lib.wkv7_slot_free(self._h, n, arr), "slot_free")

    def snapshot_alloc(self, n: int) -> list[int]:
        arr = (ctypes.c_int32 * max(1, n))()
        _check(self._lib.wkv7_snapshot_alloc(self._h, n, arr), "snapshot_alloc")
        return list(arr[:n])

    def snapshot_free(self, ids) -> None:
        arr, n = _ids_host(ids)
        _check(self._lib.wkv7_snapshot_free(self._h, n, arr), "snapshot_free")

    def n_free(self) -> int:
        return int(self._lib.wkv7_slot_count_free(self._h))

    def n_snapshots_free(self) -> int:
        return int(self._lib.wkv7_snapshot_count_free(self._h))

    def is_allocated(self, slot: int) -> bool:
        out = ctypes.c_int32()
        _check(self._lib.wkv7_slot_is_allocated(self._h, slot, ctypes.byref(out)), "is_allocated")
        return bool(out.value)

    def state_ptr(self, slot: int, layer: int) -> int:
        p = ctypes.c_void_p()
        _check(self._lib.wkv7_pool_state_ptr(self._h, slot, layer, ctypes.byref(p)), "state_ptr")
        return int(p.value)

    # ----------------------------------------------------------------- verbs
    def create(self, n: int, stream=None) -> list[int]:
        arr = (ctypes.c_int32 * max(1, n))()
        _check(self._lib.wkv7_slot_create(self._h, n, arr, _stream_handle(stream, self.device)),
               "slot_create")
        return list(arr[:n])

    def reset(self, slot_ids: torch.Tensor, stream=None) -> None:
        _check(self._lib.wkv7_slot_reset(self._h, _dev_i32(slot_ids, "slot_ids", self.device),
                                         slot_ids.numel(), _stream_handle(stream, self.device)),
               "slot_reset")

    def snapshot(self, slot_ids: torch.Tensor, snap_ids: torch.Tensor, stream=None) -> None:
        self._pairs("wkv7_slot_snapshot", slot_ids, snap_ids, stream)

    def restore(self, snap_ids: torch.Tensor, slot_ids: torch.Tensor, stream=None) -> None:
        self._pairs("wkv7_slot_restore", snap_ids, slot_ids, stream)

    def fork(self, src_ids: torch.Tensor, dst_ids: torch.Tensor, stream=None) -> None:
        self._pairs("wkv7_slot_fork", src_ids, dst_ids, stream)

    def _host_buffer(self, host: torch.Tensor, n: int) -> tuple[int, int]:
        if not isinstance(host, torch.Tensor) or host.is_cuda or not host.is_contiguous():
            raise TypeError("host buffer must be a contiguous CPU tensor (pinned memory)")
        nbytes = host.numel() * host.element_size()
        if nbytes < n * self.slot_bytes:
            raise ValueError(f"host buffer holds {nbytes} bytes, {n} slots need {n * self.slot_bytes}")
        return host.data_ptr(), nbytes

    def hibernate(self, slot_ids: torch.Tensor, host: torch.Tensor, stream=None) -> None:
        """Copy the slots slot_ids[i] into pinned host memory `host`, packed slot after slot
        (asynchronous on the stream; see wkv7_slot_hibernate)."""
        n = slot_ids.numel()
        ptr, nbytes = self._host_buffer(host, n)
        _check(self._lib.wkv7_slot_hibernate(self._h, _dev_i32(slot_ids, "slot_ids", self.device), n,
                                             ptr, nbytes, _stream_handle(stream, self.device)),
               "slot_hibernate")

    def resume(self, host: torch.Tensor, slot_ids: torch.Tensor, stream=None) -> None:
        """Copy packed slot images from pinned host memory `host` into the slots slot_ids[i]."""
        n = slot_ids.numel()
        ptr, nbytes = self._host_buffer(host, n)
        _check(self._lib.wkv7_slot_resume(self._h, ptr, nbytes,
                                          _dev_i32(slot_ids, "slot_ids", self.device), n,
                                          _stream_handle(stream, self.device)), "slot_resume")

    def _pairs(self, fn, first, second, stream):
        if first.numel() != second.numel():
            raise ValueError("id arrays differ in length")
        _check(getattr(self._lib, fn)(self._h, _dev_i32(first, "ids", self.device),
                                      _dev_i32(second, "ids", self.device), first.numel(),
                                      _stream_handle(stream, self.device)), fn)

    # ------------------------------------------------------------ recurrence
    def _inputs(self, xs, rows):
        dt = xs[0].dtype
        if dt not in (torch.float32, torch.bfloat16):
            raise TypeError("inputs must be float32 or bfloat16")
        for x in xs:
            if x.dtype != dt or x.device != self.device or not x.is_contiguous():
                raise ValueError("inputs must share one dtype and be contiguous on the pool device")
            if tuple(x.shape) != (rows, self.n_heads, self.head_size):
                raise ValueError(f"inputs must be [{rows}, {self.n_heads}, {self.head_size}]")
        return (BF16 if dt == torch.bfloat16 else F32), [x.data_ptr() for x in xs]

    def _out(self, o, rows):
        if o is None:
            return torch.empty(rows, self.n_heads, self.head_size, dtype=self.o_torch_dtype,
                               device=self.device)
        if (o.dtype != self.o_torch_dtype or o.device != self.device or not o.is_contiguous()
                or tuple(o.shape) != (rows, self.n_heads, self.head_size)):
            raise ValueError(f"o must be a contiguous {self.o_torch_dtype} [rows, n_heads, 64] tensor")
        return o

    def decode_step(self, layer: int, slot_ids: torch.Tensor, r, w, k, v, a, b, o=None,
                    stream=None) -> torch.Tensor:
        n = slot_ids.numel()
        dt, ptrs = self._inputs((r, w, k, v, a, b), n)
        o = self._out(o, n)
        _check(self._lib.wkv7_decode_step(self._h, layer, _dev_i32(slot_ids, "slot_ids", self.device),
                                          n, dt, *ptrs, o.data_ptr(),
                                          _stream_handle(stream, self.device)), "decode_step")
        return o

    def decode_multi(self, layer: int, slot_ids: torch.Tensor, r, w, k, v, a, b, o=None,
                     step_snap_ids: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """K consecutive tokens per slot: inputs [n, K, n_heads, 64] (one dtype), o the
        same shape in the pool's output dtype; with step_snap_ids ([n, K] device int32) the state after
        every token also goes to those snapshot ids (this layer)."""
        n = slot_ids.numel()
        if r.dim() != 4 or r.shape[0] != n:
            raise ValueError("decode_multi inputs must be [n, K, n_heads, 64]")
        K = int(r.shape[1])
        dt, ptrs = self._inputs(tuple(x.reshape(n * K, *x.shape[2:]) if x.dim() == 4 and
                                      tuple(x.shape[:2]) == (n, K) else x
                                      for x in (r, w, k, v, a, b)), n * K)
        if o is None:
            o = torch.empty(n, K, self.n_heads, self.head_size, dtype=self.o_torch_dtype,
                            device=self.device)
        self._out(o.reshape(n * K, *o.shape[2:]) if o.dim() == 4 else o, n * K)
        snaps = None
        if step_snap_ids is not None:
            if step_snap_ids.numel() != n * K:
                raise ValueError("step_snap_ids must hold n * K ids")
            snaps = _dev_i32(step_snap_ids, "step_snap_ids", self.device)
        _check(self._lib.wkv7_decode_multi(self._h, layer, _dev_i32(slot_ids, "slot_ids", self.device),
                                           n, K, dt, *ptrs, o.data_ptr(), snaps,
                                           _stream_handle(stream, self.device)), "decode_multi")
        return o

    def prefill(self, layer: int, slot_ids: torch.Tensor, cu_seqlens: torch.Tensor, r, w, k, v,
                a, b, o=None, max_seqlen: int | None = None, stream=None,
                sequential: bool = False, cu_ckpt: torch.Tensor | None = None,
                ckpt_ids: torch.Tensor | None = None) -> torch.Tensor:
        """Prefill; with cu_ckpt / ckpt_ids (device int32), also the state at every
        64-token boundary of each sequence into those snapshot ids (this layer)."""
        total = r.shape[0]
        dt, ptrs = self._inputs((r, w, k, v, a, b), total)
        o = self._out(o, total)
        if cu_seqlens.numel() != slot_ids.numel() + 1:
            raise ValueError("cu_seqlens must have n_seqs + 1 entries")
        if (cu_ckpt is None) != (ckpt_ids is None):
            raise ValueError("cu_ckpt and ckpt_ids go together")
        if cu_ckpt is not None:
            if cu_ckpt.numel() != slot_ids.numel() + 1:
                raise ValueError("cu_ckpt must have n_seqs + 1 entries")
            ids_ptr = _dev_i32(ckpt_ids, "ckpt_ids", self.device) if ckpt_ids.numel() else None
            if ids_ptr is None:  # no boundary anywhere: any non-null pointer will do
                ids_ptr = _dev_i32(cu_ckpt, "cu_ckpt", self.device)
            _check(self._lib.wkv7_prefill_checkpointed(
                self._h, layer, _dev_i32(slot_ids, "slot_ids", self.device),
                _dev_i32(cu_seqlens, "cu_seqlens", self.device), slot_ids.numel(), total,
                total if max_seqlen is None else int(max_seqlen), dt, *ptrs, o.data_ptr(),
                _dev_i32(cu_ckpt, "cu_ckpt", self.device), ids_ptr, int(bool(sequential)),
                _stream_handle(stream, self.device)), "prefill_checkpointed")
            return o
        fn = self._lib.wkv7_prefill_sequential if sequential else self._lib.wkv7_prefill
        _check(fn(self._h, layer, _dev_i32(slot_ids, "slot_ids", self.device),
                  _dev_i32(cu_seqlens, "cu_seqlens", self.device), slot_ids.numel(), total,
                  total if max_seqlen is None else int(max_seqlen), dt, *ptrs, o.data_ptr(),
                  _stream_handle(stream, self.device)),
               "prefill_sequential" if sequential else "prefill")
        return o

    # ------------------------------------------------------------ validation
    def validate_ids(self, ids_a: torch.Tensor, ids_b: torch.Tensor | None = None,
                     table: str = "slots", stream=None) -> None:
        """Debug pass (wkv7_validate_ids): every id of ids_a and ids_b (device int32)
        in the table and none twice; the verdict lands in the device status word
        (DEV_DUP_SLOT, DEV_BAD_SLOT), read with device_status()."""
        if table not in ("slots", "snapshots"):
            raise ValueError("table must be 'slots' or 'snapshots'")
        nb = 0 if ids_b is None else ids_b.numel()
        pb = _dev_i32(ids_b, "ids_b", self.device) if nb else None
        na = ids_a.numel()
        pa = _dev_i32(ids_a, "ids_a", self.device) if na else None
        _check(self._lib.wkv7_validate_ids(self._h, TABLE_SLOTS if table == "slots" else TABLE_SNAPSHOTS,
                                           pa, na, pb, nb, _stream_handle(stream, self.device)),
               "validate_ids")

    # ---------------------------------------------------------------- status
    def device_status(self, stream=None, timeout_ms: int = 10000) -> int:
        """Read and clear the device status word (a DEV_* code; 0 when clean)."""
        code = ctypes.c_int32()
        st = self._lib.wkv7_get_device_status(self._h, _stream_handle(stream, self.device),
                                              timeout_ms, ctypes.byref(code))
        if st not in (0, 3, 8):  # OK, ERR_DUP_SLOT and ERR_DEVICE_STATUS carry the code
            _check(st, "get_device_status")
        return int(code.value)
