"""ctypes binding of libtri (include/tri.h), same entry-point names.

Argument marshalling only: every step of the compression path runs in the CUDA
kernels of libtri.so.  PyTorch supplies device memory and the current stream.
There is no fallback: if libtri.so is missing or cannot be loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtri.so")

TRI_OK, TRI_ERR_INVALID, TRI_ERR_CUDA, TRI_ERR_UNSUPPORTED, TRI_ERR_WORKSPACE, TRI_ERR_TIMEOUT, TRI_ERR_BOUNDS = range(7)
TRI_F32, TRI_BF16 = 0, 1
TRI_PAIR_HALF, TRI_PAIR_INTERLEAVED = 0, 1
TRI_COMPACT_ORDERED, TRI_COMPACT_HOLEFILL = 0, 1
_COMPACT = {"ordered": TRI_COMPACT_ORDERED, "holefill": TRI_COMPACT_HOLEFILL}

EXPORTED = ("tri_calibrate_stats", "tri_workspace_bytes", "tri_score", "tri_select_topb",
            "tri_compact_kv", "tri_compress_step", "tri_get_device_status",
            "tri_clear_device_status", "tri_status_string", "tri_version",
            "tri_compress_step_static_scratch")


class TriError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        msg = f"{fn}: {status_string(status)} (status {status})"
        super().__init__(msg + (f": {detail}" if detail else ""))


class tri_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int),
                ("L", ctypes.c_int), ("S", ctypes.c_int), ("Hkv", ctypes.c_int), ("d", ctypes.c_int),
                ("cap", ctypes.c_int64), ("seq_len", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("max_blocks", ctypes.c_int), ("block", ctypes.c_int), ("nblocks", ctypes.c_int64)]


class tri_stats(ctypes.Structure):
    _fields_ = [("center", ctypes.c_void_p), ("R", ctypes.c_void_p), ("mag", ctypes.c_void_p),
                ("Hq", ctypes.c_int)]


class tri_params(ctypes.Structure):
    _fields_ = [("theta", ctypes.c_double), ("pairing", ctypes.c_int), ("t", ctypes.c_void_p),
                ("offsets", ctypes.POINTER(ctypes.c_int32)), ("n_offsets", ctypes.c_int),
                ("budget", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libtri.so (raises if it is missing: build it first)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtri.so not found at {LIB_PATH}; build it with "
                               "`python -m kv_cache_compression_06_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "tri_calibrate_stats": [P, I, I64, I, I, I, I, P, P, P, P],
            "tri_workspace_bytes": [P, P, P, ctypes.POINTER(SZ)],
            "tri_score": [P, P, P, P, P, P, SZ, P],
            "tri_select_topb": [P, P, I, P, P, SZ, P],
            "tri_compact_kv": [P, P, I, I, P, P],
            "tri_compress_step": [P, P, P, I, P, P, P, SZ, P],
            "tri_compress_step_static_scratch": [P, P, P, I, P, P, P],
            "tri_get_device_status": [P, ctypes.POINTER(ctypes.c_int32)],
            "tri_clear_device_status": [P],
            "tri_status_string": [I],
            "tri_version": [],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_char_p if name == "tri_status_string" else ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().tri_status_string(int(status)).decode()


def _check(fn: str, st: int) -> None:
    if st != TRI_OK:
        raise TriError(fn, st)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---------------------------------------------------------------- descriptions
@dataclasses.dataclass
class KVCache:
    """Device KV cache.  Dense: k, v [L][S][Hkv][cap][d].  Paged: k, v pools
    [L][nblocks][block][Hkv][d] plus block_table [S][max_blocks] int32."""
    k: torch.Tensor
    v: torch.Tensor
    seq_len: torch.Tensor
    Hkv: int
    block_table: Optional[torch.Tensor] = None
    block: int = 16

    @property
    def paged(self) -> bool:
        return self.block_table is not None

    @property
    def L(self) -> int:
        return self.k.shape[0]

    @property
    def S(self) -> int:
        return self.seq_len.shape[0]

    @property
    def d(self) -> int:
        return self.k.shape[-1]

    @property
    def cap(self) -> int:
        return self.block_table.shape[1] * self.block if self.paged else self.k.shape[3]

    def to_c(self) -> tri_cache:
        for t in (self.k, self.v):
            if t is not None and not t.is_contiguous():
                raise ValueError("cache tensors must be contiguous")
        if self.k.dtype == torch.bfloat16:
            dt = TRI_BF16
        elif self.k.dtype == torch.float32:
            dt = TRI_F32
        else:
            raise ValueError(f"unsupported cache dtype {self.k.dtype}")
        c = tri_cache()
        c.k, c.v = _ptr(self.k), _ptr(self.v)
        c.dtype = dt
        c.L, c.S, c.Hkv, c.d = self.L, self.S, self.Hkv, self.d
        c.cap = self.cap
        c.seq_len = _ptr(self.seq_len)
        if self.paged:
            c.block_table = _ptr(self.block_table)
            c.max_blocks = self.block_table.shape[1]
            c.block = self.block
            c.nblocks = self.k.shape[1]
        return c


@dataclasses.dataclass
class Stats:
    center: torch.Tensor   # [L][Hq][F][2] f32
    R: torch.Tensor        # [L][Hq][F] f32
    mag: torch.Tensor      # [L][Hq][F] f32

    @property
    def Hq(self) -> int:
        return self.R.shape[1]

    def to_c(self) -> tri_stats:
        s = tri_stats()
        s.center, s.R, s.mag, s.Hq = _ptr(self.center), _ptr(self.R), _ptr(self.mag), self.Hq
        return s


@dataclasses.dataclass
class Params:
    theta: float
    t: torch.Tensor                 # [S] int32, device
    offsets: Sequence[int]
    budget: int
    pairing: str = "half"

    def to_c(self):
        arr = (ctypes.c_int32 * len(self.offsets))(*[int(o) for o in self.offsets])
        p = tri_params()
        p.theta = float(self.theta)
        p.pairing = TRI_PAIR_HALF if self.pairing == "half" else TRI_PAIR_INTERLEAVED
        p.t = _ptr(self.t)
        p.offsets = arr
        p.n_offsets = len(self.offsets)
        p.budget = int(self.budget)
        return p, arr   # keep the host offsets array alive during the call


# ---------------------------------------------------------------- entry points
def tri_calibrate_stats(q_pre: torch.Tensor, pairing: str = "half", out: Optional[Stats] = None,
                        stream=None) -> Stats:
    """q_pre [L][n][Hq][d] (f32 or bf16) -> Stats (center, R, mag)."""
    L, n, Hq, d = q_pre.shape
    if out is None:
        dev = q_pre.device
        out = Stats(torch.empty((L, Hq, d // 2, 2), dtype=torch.float32, device=dev),
                    torch.empty((L, Hq, d // 2), dtype=torch.float32, device=dev),
                    torch.empty((L, Hq, d // 2), dtype=torch.float32, device=dev))
    dt = TRI_BF16 if q_pre.dtype == torch.bfloat16 else TRI_F32
    st = lib().tri_calibrate_stats(_ptr(q_pre.contiguous()), dt, n, L, Hq, d,
                                   TRI_PAIR_HALF if pairing == "half" else TRI_PAIR_INTERLEAVED,
                                   _ptr(out.center), _ptr(out.R), _ptr(out.mag), _stream(stream))
    _check("tri_calibrate_stats", st)
    return out


def tri_workspace_bytes(cache: KVCache, stats: Stats, params: Params) -> int:
    c, s = cache.to_c(), stats.to_c()
    p, _keep = params.to_c()
    n = ctypes.c_size_t(0)
    _check("tri_workspace_bytes", lib().tri_workspace_bytes(ctypes.byref(c), ctypes.byref(s),
                                                            ctypes.byref(p), ctypes.byref(n)))
    return int(n.value)


def workspace(cache: KVCache, stats: Stats, params: Params) -> Optional[torch.Tensor]:
    """A device buffer of tri_workspace_bytes bytes (None when 0)."""
    n = tri_workspace_bytes(cache, stats, params)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=cache.k.device)


def tri_score(cache: KVCache, stats: Stats, params: Params, agg: Optional[torch.Tensor] = None,
              raw: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None):
    """Per-unit aggregated scores agg [L][S][Hkv][cap] (and per-head raw scores
    [L][S][Hq][cap] when `raw` is given)."""
    if agg is None:
        agg = torch.zeros((cache.L, cache.S, cache.Hkv, cache.cap), dtype=torch.float32, device=cache.k.device)
    if ws is None:
        ws = workspace(cache, stats, params)
    c, s = cache.to_c(), stats.to_c()
    p, _keep = params.to_c()
    st = lib().tri_score(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), _ptr(agg), _ptr(raw),
                         _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream))
    _check("tri_score", st)
    return agg


def tri_select_topb(cache: KVCache, agg: torch.Tensor, budget: int, idx: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """Kept slots idx [L][S][Hkv][budget] (ascending; -1 padding when N < budget)."""
    if idx is None:
        idx = torch.empty((cache.L, cache.S, cache.Hkv, budget), dtype=torch.int32, device=agg.device)
    c = cache.to_c()
    st = lib().tri_select_topb(ctypes.byref(c), _ptr(agg), int(budget), _ptr(idx), None, 0, _stream(stream))
    _check("tri_select_topb", st)
    return idx


def tri_compact_kv(cache: KVCache, idx: torch.Tensor, budget: int, new_len: Optional[torch.Tensor] = None,
                   stream=None, compact: str = "ordered") -> Optional[torch.Tensor]:
    """In-place compaction of K and V to the kept slots idx (per unit, ascending);
    compact = 'ordered' or 'holefill' (layout, see include/tri.h)."""
    c = cache.to_c()
    st = lib().tri_compact_kv(ctypes.byref(c), _ptr(idx), int(budget), _COMPACT[compact], _ptr(new_len),
                              _stream(stream))
    _check("tri_compact_kv", st)
    return new_len


def tri_compress_step(cache: KVCache, stats: Stats, params: Params, idx_out: Optional[torch.Tensor] = None,
                      new_len: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                      stream=None, compact: str = "ordered"):
    """The fused step (score -> z/max -> top-B -> compact) on every unit with N > B;
    compact = 'ordered' or 'holefill' (layout, see include/tri.h)."""
    if ws is None:
        ws = workspace(cache, stats, params)
    c, s = cache.to_c(), stats.to_c()
    p, _keep = params.to_c()
    st = lib().tri_compress_step(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), _COMPACT[compact],
                                 _ptr(idx_out), _ptr(new_len), _ptr(ws), 0 if ws is None else ws.numel(),
                                 _stream(stream))
    _check("tri_compress_step", st)
    return idx_out, new_len


TRI_STATIC_SCRATCH_BYTES = 32 << 20


def tri_compress_step_static_scratch(cache: KVCache, stats: Stats, params: Params,
                                     idx_out: Optional[torch.Tensor] = None,
                                     new_len: Optional[torch.Tensor] = None, stream=None):
    """tri_compress_step without a caller workspace, for callers that cannot
    allocate device memory (e.g. an engine that reserved all of it for its
    KV-cache pool).  Long units use the library's built-in scratch of
    TRI_STATIC_SCRATCH_BYTES bytes, shared by every call on the device: calls
    that overlap on the GPU race.  Make the first call on a device before any
    stream capture (it looks up the scratch address)."""
    c, s = cache.to_c(), stats.to_c()
    p, _keep = params.to_c()
    st = lib().tri_compress_step_static_scratch(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p),
                                                TRI_COMPACT_ORDERED, _ptr(idx_out), _ptr(new_len),
                                                _stream(stream))
    if st == TRI_ERR_WORKSPACE:
        need = tri_workspace_bytes(cache, stats, params)
        raise TriError("tri_compress_step_static_scratch", st,
                       f"needs {need} bytes of scratch; the built-in scratch holds {TRI_STATIC_SCRATCH_BYTES}")
    _check("tri_compress_step_static_scratch", st)
    return idx_out, new_len


def tri_get_device_status(stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("tri_get_device_status", lib().tri_get_device_status(_stream(stream), ctypes.byref(out)))
    return int(out.value)


def tri_clear_device_status(stream=None) -> None:
    _check("tri_clear_device_status", lib().tri_clear_device_status(_stream(stream)))


def tri_version() -> int:
    return int(lib().tri_version())
