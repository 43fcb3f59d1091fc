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
            "tri_compress_step_static_scratch", "tri_calib_reset", "tri_calib_accumulate",
            "tri_calib_merge", "tri_calib_finalize", "tri_distance_curves", "tri_check_bounded_wait",
            "tri_append_kv", "tri_decode_workspace_bytes", "tri_decode_attention")
TRI_CALIB_ACC_DOUBLES = 8


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
            "tri_calib_reset": [P, I, I, I, P],
            "tri_calib_accumulate": [P, I, I64, I, I, I, I, I64, I64, P, P],
            "tri_calib_merge": [P, P, I, I, I, P],
            "tri_calib_finalize": [P, I, I, I, P, P, P, P],
            "tri_distance_curves": [P, P, P, P, I, I64, I, I, I, I, ctypes.c_double, I, I, P, P, P, P],
            "tri_check_bounded_wait": [ctypes.c_uint32, P],
            "tri_append_kv": [P, P, P, P, ctypes.c_double, I, P, P, P],
            "tri_decode_workspace_bytes": [P, I, ctypes.POINTER(SZ)],
            "tri_decode_attention": [P, P, I, P, ctypes.c_double, I, ctypes.c_float, P, P, SZ, P],
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


def _pairing(pairing: str) -> int:
    if pairing not in ("half", "interleaved"):
        raise ValueError(pairing)
    return TRI_PAIR_HALF if pairing == "half" else TRI_PAIR_INTERLEAVED


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return TRI_BF16
    if t.dtype == torch.float32:
        return TRI_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def calib_accumulator(L: int, H: int, d: int, device) -> torch.Tensor:
    """A zeroed fp64 accumulator [L][H][d/2][TRI_CALIB_ACC_DOUBLES] for the
    streamed calibration (allocated by torch; tri_calib_reset zeroes it on the GPU)."""
    acc = torch.empty((L, H, d // 2, TRI_CALIB_ACC_DOUBLES), dtype=torch.float64, device=device)
    tri_calib_reset(acc, stream=None)
    return acc


def tri_calib_reset(acc: torch.Tensor, stream=None) -> None:
    L, H, F, _ = acc.shape
    _check("tri_calib_reset", lib().tri_calib_reset(_ptr(acc), L, H, 2 * F, _stream(stream)))


def tri_calib_accumulate(q: torch.Tensor, acc: torch.Tensor, pairing: str = "half", stream=None) -> None:
    """Adds the samples of q to acc.  q is [L][n][H][d], or a strided view of
    one (the sample and layer strides are passed through; the last two
    dimensions must be contiguous), e.g. the query slice of a fused QKV
    activation."""
    L, n, H, d = q.shape
    if q.stride(3) != 1 or q.stride(2) != d:
        raise ValueError("the head and element dimensions of q must be contiguous")
    if tuple(acc.shape) != (L, H, d // 2, TRI_CALIB_ACC_DOUBLES) or acc.dtype != torch.float64:
        raise ValueError("acc does not match q")
    st = lib().tri_calib_accumulate(_ptr(q), _dtype(q), n, L, H, d, _pairing(pairing), q.stride(1),
                                    q.stride(0) if L > 1 else 0, _ptr(acc), _stream(stream))
    _check("tri_calib_accumulate", st)


def tri_calib_merge(acc: torch.Tensor, other: torch.Tensor, stream=None) -> None:
    if acc.shape != other.shape:
        raise ValueError("accumulators differ in shape")
    L, H, F, _ = acc.shape
    _check("tri_calib_merge", lib().tri_calib_merge(_ptr(acc), _ptr(other), L, H, 2 * F, _stream(stream)))


def tri_calib_finalize(acc: torch.Tensor, out: Optional["Stats"] = None, stream=None) -> "Stats":
    L, H, F, _ = acc.shape
    if out is None:
        dev = acc.device
        out = Stats(torch.empty((L, H, F, 2), dtype=torch.float32, device=dev),
                    torch.empty((L, H, F), dtype=torch.float32, device=dev),
                    torch.empty((L, H, F), dtype=torch.float32, device=dev))
    st = lib().tri_calib_finalize(_ptr(acc), L, H, 2 * F, _ptr(out.center), _ptr(out.R), _ptr(out.mag),
                                  _stream(stream))
    _check("tri_calib_finalize", st)
    return out


def tri_distance_curves(q_center: torch.Tensor, k_center: torch.Tensor, q_seq: Optional[torch.Tensor],
                        k_seq: Optional[torch.Tensor], theta: float, n_delta: int, pairing: str = "half",
                        stream=None):
    """Distance-preference curves: (center_curve [L][Hq][n_delta], logit_curve
    [L][Hq][n_delta] or None, corr [L][Hq] or None).  q_center [L][Hq][F][2],
    k_center [L][Hkv][F][2]; q_seq [L][n][Hq][d], k_seq [L][n][Hkv][d] pre-RoPE
    samples of one sequence (None: center curve only)."""
    L, Hq, F, _ = q_center.shape
    Hkv = k_center.shape[1]
    d = 2 * F
    dev = q_center.device
    cc = torch.empty((L, Hq, n_delta), dtype=torch.float32, device=dev)
    lc = corr = None
    n, dt = 1, TRI_F32
    if q_seq is not None:
        q_seq, k_seq = q_seq.contiguous(), k_seq.contiguous()
        n, dt = q_seq.shape[1], _dtype(q_seq)
        lc = torch.empty_like(cc)
        corr = torch.empty((L, Hq), dtype=torch.float32, device=dev)
    st = lib().tri_distance_curves(_ptr(q_center.contiguous()), _ptr(k_center.contiguous()), _ptr(q_seq),
                                   _ptr(k_seq), dt, n, L, Hq, Hkv, d, float(theta), _pairing(pairing),
                                   int(n_delta), _ptr(cc), _ptr(lc), _ptr(corr), _stream(stream))
    _check("tri_distance_curves", st)
    return cc, lc, corr


def tri_check_bounded_wait(limit_us: int = 1000, stream=None) -> None:
    """Runs the bounded-wait health check (see include/tri.h): afterwards the
    device status reads TRI_ERR_TIMEOUT until cleared."""
    _check("tri_check_bounded_wait", lib().tri_check_bounded_wait(int(limit_us), _stream(stream)))


def tri_append_kv(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, pos: torch.Tensor, theta: float,
                  seq_len_out: torch.Tensor, pos_out: Optional[torch.Tensor] = None, pairing: str = "half",
                  stream=None) -> None:
    """Appends one token per unit: k_new, v_new [L][S][Hkv][d] (pre-RoPE key,
    value) into slot seq_len[s]; seq_len_out = seq_len + 1, pos_out = pos + 1."""
    c = cache.to_c()
    st = lib().tri_append_kv(ctypes.byref(c), _ptr(k_new.contiguous()), _ptr(v_new.contiguous()), _ptr(pos),
                             float(theta), _pairing(pairing), _ptr(seq_len_out), _ptr(pos_out), _stream(stream))
    _check("tri_append_kv", st)


def tri_decode_workspace_bytes(cache: KVCache, Hq: int) -> int:
    c = cache.to_c()
    n = ctypes.c_size_t(0)
    _check("tri_decode_workspace_bytes", lib().tri_decode_workspace_bytes(ctypes.byref(c), int(Hq), ctypes.byref(n)))
    return int(n.value)


def tri_decode_attention(cache: KVCache, q: torch.Tensor, pos: torch.Tensor, theta: float,
                         scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                         ws: Optional[torch.Tensor] = None, pairing: str = "half", stream=None) -> torch.Tensor:
    """Single-query attention of q [L][S][Hq][d] (bf16, pre-RoPE, rotated to pos
    inside) over every unit's cached keys; returns out [L][S][Hq][d] fp32."""
    L, S, Hq, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((L, S, Hq, d), dtype=torch.float32, device=q.device)
    if ws is None:
        n = tri_decode_workspace_bytes(cache, Hq)
        ws = None if n == 0 else torch.empty(n, dtype=torch.uint8, device=q.device)
    c = cache.to_c()
    st = lib().tri_decode_attention(ctypes.byref(c), _ptr(q.contiguous()), Hq, _ptr(pos), float(theta),
                                    _pairing(pairing), float(scale), _ptr(out), _ptr(ws),
                                    0 if ws is None else ws.numel(), _stream(stream))
    _check("tri_decode_attention", st)
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
                                     new_len: Optional[torch.Tensor] = None, stream=None,
                                     compact: str = "ordered"):
    """tri_compress_step without a caller workspace, for callers that cannot
    allocate device memory (e.g. an engine that reserved all of it for its
    KV-cache pool).  Long units use the library's built-in scratch of
    TRI_STATIC_SCRATCH_BYTES bytes, shared by every call on the device: calls
    that overlap on the GPU race.  Make the first call on a device before any
    stream capture (it looks up the scratch address).  compact = 'ordered' or
    'holefill', as for tri_compress_step."""
    c, s = cache.to_c(), stats.to_c()
    p, _keep = params.to_c()
    st = lib().tri_compress_step_static_scratch(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p),
                                                _COMPACT[compact], _ptr(idx_out), _ptr(new_len),
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
