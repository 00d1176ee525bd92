"""Python binding of libdms.so (the C ABI in include/dms.h).

Argument marshalling only: tensors are checked (dtype, device, shape,
contiguity) and passed as raw device pointers with the current CUDA stream.
Every step of the method runs in the library's CUDA kernels.  If libdms.so is
missing this module raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from .build import LIB_PATH

DMS_OK = 0
DMS_ERR_INVALID_ARG = -1
DMS_ERR_CUDA = -2
DMS_ERR_CAPACITY = -3
DMS_ERR_BAD_HANDLE = -4
DMS_ERR_TIMEOUT = -5
DMS_ERR_EMPTY = -6
DMS_ERR_SCRATCH_LIMIT = -7
DMS_MAX_GROUP = 8
DMS_KV_BF16 = 0
DMS_KV_FP8_E4M3 = 1
KV_FORMATS = {"bf16": DMS_KV_BF16, "fp8": DMS_KV_FP8_E4M3}

# Entry points declared in include/dms.h: name -> (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "dms_cache_create": (_P, [_I, _I, _I, _I, _I]),
    "dms_cache_create_ex": (_P, [_I, _I, _I, _I, _I, _I]),
    "dms_cache_kv_format": (_I, [_P]),
    "dms_cache_export_scales": (_I, [_P, _P, _P, _P]),
    "dms_step_graph_create": (_P, [_P, _I, _P, _P, _P, _P, _P, ctypes.c_float, _I]),
    "dms_step_graph_launch": (_I, [_P, _P]),
    "dms_step_graph_destroy": (None, [_P]),
    "dms_last_error": (_I, []),
    "dms_cache_destroy": (None, [_P]),
    "dms_append": (_I, [_P, _P, _P, _P, _P]),
    "dms_append_chunk": (_I, [_P, _P, _P, _P, _I, _P]),
    "dms_decode_attention": (_I, [_P, _P, _P, ctypes.c_float, _I, _P]),
    "dms_prefill": (_I, [_P, _P, _P, _P, _P, _I, _P, ctypes.c_float, _I, _P]),
    "dms_step": (_I, [_P, _P, _P, _P, _P, _P, ctypes.c_float, _I, _P]),
    "dms_step_host": (_I, [_P, _P, _P, _P, _P, _P, ctypes.c_float, _I, _P]),
    "dms_step_host_join": (_I, [_P, _P]),
    "dms_cache_lengths": (_I, [_P, _P, _P]),
    "dms_cache_slot_positions": (_I, [_P, _P, _P]),
    "dms_cache_export_kv": (_I, [_P, _P, _P, _P]),
    "dms_cache_status": (_I, [_P, _P]),
    "dms_cache_selftest_wait": (_I, [_P, _P]),
    "dms_cache_position": (ctypes.c_int64, [_P]),
    "dms_error_string": (ctypes.c_char_p, [_I]),
    "dms_decode_attention_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, ctypes.c_float, _I, _P]),
}

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdms.so (built in-tree) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m learned_kv_cache_eviction_b300.build` "
            "(the DMS kernels have no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class DmsError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = load_library().dms_error_string(code).decode()
        super().__init__(f"{what}: {msg} ({code})" if what else f"{msg} ({code})")


def _check(code: int, what: str) -> None:
    if code != DMS_OK:
        raise DmsError(code, what)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t: torch.Tensor, name: str, dtype, shape, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class DmsCache:
    """A DMS compacted KV cache for one attention layer (all device state is
    owned by libdms.so)."""

    def __init__(self, batch: int, kv_heads: int, capacity: int, head_dim: int, window: int = 16,
                 device=None, kv_format: str = "bf16"):
        """kv_format: "bf16" (rows stored as given) or "fp8" (E4M3 codes with a
        float32 scale per row; see dms_cache_create_ex)."""
        self._lib = load_library()
        if kv_format not in KV_FORMATS:
            raise ValueError(f"kv_format must be one of {sorted(KV_FORMATS)}")
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index or 0)
        with torch.cuda.device(self.device):
            h = self._lib.dms_cache_create_ex(batch, kv_heads, capacity, head_dim, window, KV_FORMATS[kv_format])
        if not h:
            raise DmsError(self._lib.dms_last_error(), "dms_cache_create_ex")
        self._h = ctypes.c_void_p(h)
        self.batch, self.kv_heads, self.capacity, self.head_dim, self.window = (
            batch, kv_heads, capacity, head_dim, window)
        self.kv_format = kv_format

    # -- lifetime -----------------------------------------------------------
    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.dms_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise DmsError(DMS_ERR_BAD_HANDLE, "cache is closed")
        return self._h

    @property
    def position(self) -> int:
        return int(self._lib.dms_cache_position(self.handle))

    # -- hot path ------------------------------------------------------------
    def append(self, k: torch.Tensor, v: torch.Tensor, evict_logit: torch.Tensor, stream=None) -> None:
        B, H, D = self.batch, self.kv_heads, self.head_dim
        _need(k, "k", torch.bfloat16, (B, H, D), self.device)
        _need(v, "v", torch.bfloat16, (B, H, D), self.device)
        _need(evict_logit, "evict_logit", torch.float32, (B, H), self.device)
        _check(self._lib.dms_append(self.handle, k.data_ptr(), v.data_ptr(), evict_logit.data_ptr(),
                                    _stream_handle(stream)), "dms_append")

    def append_chunk(self, k: torch.Tensor, v: torch.Tensor, logits: torch.Tensor, stream=None) -> None:
        B, H, D = self.batch, self.kv_heads, self.head_dim
        C = k.shape[2] if k.dim() == 4 else -1
        _need(k, "k", torch.bfloat16, (B, H, C, D), self.device)
        _need(v, "v", torch.bfloat16, (B, H, C, D), self.device)
        _need(logits, "logits", torch.float32, (B, H, C), self.device)
        _check(self._lib.dms_append_chunk(self.handle, k.data_ptr(), v.data_ptr(), logits.data_ptr(), C,
                                          _stream_handle(stream)), "dms_append_chunk")

    def prefill(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, logits: torch.Tensor,
                out: torch.Tensor | None = None, scale: float | None = None, stream=None) -> torch.Tensor:
        """Attention of a chunk of C tokens over the cache and the chunk itself,
        then the chunk's append (dms_prefill).  q [B][Hq][C][D] bf16, k/v
        [B][Hkv][C][D] bf16, logits [B][Hkv][C] fp32 -> out [B][Hq][C][D] fp32."""
        B, H, D = self.batch, self.kv_heads, self.head_dim
        if q.dim() != 4:
            raise ValueError("q must be [batch][q_heads][chunk][head_dim]")
        Hq, C = q.shape[1], q.shape[2]
        _need(q, "q", torch.bfloat16, (B, Hq, C, D), self.device)
        _need(k, "k", torch.bfloat16, (B, H, C, D), self.device)
        _need(v, "v", torch.bfloat16, (B, H, C, D), self.device)
        _need(logits, "logits", torch.float32, (B, H, C), self.device)
        if out is None:
            out = torch.empty((B, Hq, C, D), dtype=torch.float32, device=self.device)
        _need(out, "out", torch.float32, (B, Hq, C, D), self.device)
        scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
        _check(self._lib.dms_prefill(self.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), logits.data_ptr(), C,
                                     out.data_ptr(), scale, Hq, _stream_handle(stream)), "dms_prefill")
        return out

    def step(self, k: torch.Tensor, v: torch.Tensor, evict_logit: torch.Tensor, q: torch.Tensor,
             out: torch.Tensor, scale: float | None = None, stream=None) -> torch.Tensor:
        """Append one token and decode its query in one library call (dms_step).
        k, v [B][Hkv][D] bf16, evict_logit [B][Hkv] fp32, q [B][Hq][D] bf16,
        out [B][Hq][D] fp32 (preallocated)."""
        B, H, D = self.batch, self.kv_heads, self.head_dim
        Hq = q.shape[1] if q.dim() == 3 else -1
        _need(k, "k", torch.bfloat16, (B, H, D), self.device)
        _need(v, "v", torch.bfloat16, (B, H, D), self.device)
        _need(evict_logit, "evict_logit", torch.float32, (B, H), self.device)
        _need(q, "q", torch.bfloat16, (B, Hq, D), self.device)
        _need(out, "out", torch.float32, (B, Hq, D), self.device)
        scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
        _check(self._lib.dms_step(self.handle, k.data_ptr(), v.data_ptr(), evict_logit.data_ptr(), q.data_ptr(),
                                  out.data_ptr(), scale, Hq, _stream_handle(stream)), "dms_step")
        return out

    def step_host(self, k: torch.Tensor, v: torch.Tensor, evict_logit: torch.Tensor, q: torch.Tensor,
                  out: torch.Tensor, scale: float | None = None, stream=None) -> torch.Tensor:
        """dms_step with host tensors (dms_step_host): k, v [B][Hkv][D] bf16,
        evict_logit [B][Hkv] fp32, q [B][Hq][D] bf16 and out [B][Hq][D] fp32,
        all on the CPU (pinned memory lets the copies overlap the steps).
        Asynchronous: `out` holds the result once host_join(stream) has been
        called and the stream synchronized; until then the input tensors must
        stay alive and unchanged (the copies read them later)."""
        B, H, D = self.batch, self.kv_heads, self.head_dim
        Hq = q.shape[1] if q.dim() == 3 else -1
        cpu = torch.device("cpu")
        _need(k, "k", torch.bfloat16, (B, H, D), cpu)
        _need(v, "v", torch.bfloat16, (B, H, D), cpu)
        _need(evict_logit, "evict_logit", torch.float32, (B, H), cpu)
        _need(q, "q", torch.bfloat16, (B, Hq, D), cpu)
        _need(out, "out", torch.float32, (B, Hq, D), cpu)
        scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
        _check(self._lib.dms_step_host(self.handle, k.data_ptr(), v.data_ptr(), evict_logit.data_ptr(),
                                       q.data_ptr(), out.data_ptr(), scale, Hq, _stream_handle(stream)),
               "dms_step_host")
        return out

    def host_join(self, stream=None) -> None:
        """Make `stream` wait for every output copy of step_host so far."""
        _check(self._lib.dms_step_host_join(self.handle, _stream_handle(stream)), "dms_step_host_join")

    def decode_attention(self, q: torch.Tensor, out: torch.Tensor | None = None, scale: float | None = None,
                         stream=None) -> torch.Tensor:
        B, D = self.batch, self.head_dim
        if q.dim() != 3:
            raise ValueError("q must be [batch][q_heads][head_dim]")
        Hq = q.shape[1]
        _need(q, "q", torch.bfloat16, (B, Hq, D), self.device)
        if out is None:
            out = torch.empty((B, Hq, D), dtype=torch.float32, device=self.device)
        _need(out, "out", torch.float32, (B, Hq, D), self.device)
        scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
        _check(self._lib.dms_decode_attention(self.handle, q.data_ptr(), out.data_ptr(), scale, Hq,
                                              _stream_handle(stream)), "dms_decode_attention")
        return out

    # -- state export ----------------------------------------------------------
    def lengths(self, stream=None) -> torch.Tensor:
        out = torch.empty((self.batch, self.kv_heads), dtype=torch.int32, device=self.device)
        _check(self._lib.dms_cache_lengths(self.handle, out.data_ptr(), _stream_handle(stream)), "dms_cache_lengths")
        return out

    def slot_positions(self, stream=None) -> torch.Tensor:
        out = torch.empty((self.batch, self.kv_heads, self.capacity), dtype=torch.int32, device=self.device)
        _check(self._lib.dms_cache_slot_positions(self.handle, out.data_ptr(), _stream_handle(stream)),
               "dms_cache_slot_positions")
        return out

    def export_kv(self, stream=None):
        """K and V pools in logical order: bf16 rows, or for an fp8 cache the
        uint8 E4M3 codes (scales: export_scales)."""
        shp = (self.batch, self.kv_heads, self.capacity, self.head_dim)
        dt = torch.uint8 if self.kv_format == "fp8" else torch.bfloat16
        k = torch.empty(shp, dtype=dt, device=self.device)
        v = torch.empty(shp, dtype=dt, device=self.device)
        _check(self._lib.dms_cache_export_kv(self.handle, k.data_ptr(), v.data_ptr(), _stream_handle(stream)),
               "dms_cache_export_kv")
        return k, v

    def export_scales(self, stream=None):
        """fp8 caches: the float32 K and V scales of every slot, [B][Hkv][cap] each."""
        shp = (self.batch, self.kv_heads, self.capacity)
        k = torch.empty(shp, dtype=torch.float32, device=self.device)
        v = torch.empty(shp, dtype=torch.float32, device=self.device)
        _check(self._lib.dms_cache_export_scales(self.handle, k.data_ptr(), v.data_ptr(), _stream_handle(stream)),
               "dms_cache_export_scales")
        return k, v

    def status(self, stream=None) -> int:
        """Synchronize the stream and return the sticky device status code."""
        return int(self._lib.dms_cache_status(self.handle, _stream_handle(stream)))


class DmsStepGraph:
    """A decode step over several caches (e.g. a model's layers) captured into
    a CUDA graph (dms_step_graph_create).  The tensors are bound by address:
    write each step's inputs into them, call launch(), read `out`."""

    def __init__(self, caches, k, v, evict_logit, q, out, scale: float):
        self._lib = load_library()
        n = len(caches)
        if not (n == len(k) == len(v) == len(evict_logit) == len(q) == len(out)) or n == 0:
            raise ValueError("one k, v, evict_logit, q, out per cache")
        q_heads = q[0].shape[1]
        for c, ki, vi, li, qi, oi in zip(caches, k, v, evict_logit, q, out):
            B, H, D = c.batch, c.kv_heads, c.head_dim
            _need(ki, "k", torch.bfloat16, (B, H, D), c.device)
            _need(vi, "v", torch.bfloat16, (B, H, D), c.device)
            _need(li, "evict_logit", torch.float32, (B, H), c.device)
            _need(qi, "q", torch.bfloat16, (B, q_heads, D), c.device)
            _need(oi, "out", torch.float32, (B, q_heads, D), c.device)

        def arr(ts):
            return (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])

        handles = (ctypes.c_void_p * n)(*[c.handle.value for c in caches])
        self._keep = (caches, k, v, evict_logit, q, out)
        with torch.cuda.device(caches[0].device):
            h = self._lib.dms_step_graph_create(handles, n, arr(k), arr(v), arr(evict_logit), arr(q), arr(out),
                                                float(scale), q_heads)
        if not h:
            raise DmsError(self._lib.dms_last_error(), "dms_step_graph_create")
        self._h = ctypes.c_void_p(h)

    def launch(self, stream=None) -> None:
        _check(self._lib.dms_step_graph_launch(self._h, _stream_handle(stream)), "dms_step_graph_launch")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.dms_step_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# Module-level aliases carrying the C entry-point names.
def dms_cache_create(batch, kv_heads, capacity, head_dim, window=16, device=None) -> DmsCache:
    return DmsCache(batch, kv_heads, capacity, head_dim, window, device)


def dms_cache_create_ex(batch, kv_heads, capacity, head_dim, window=16, kv_format="bf16", device=None) -> DmsCache:
    return DmsCache(batch, kv_heads, capacity, head_dim, window, device, kv_format)


def dms_append(cache: DmsCache, k, v, evict_logit, stream=None) -> None:
    cache.append(k, v, evict_logit, stream)


def dms_append_chunk(cache: DmsCache, k, v, logits, stream=None) -> None:
    cache.append_chunk(k, v, logits, stream)


def dms_prefill(cache: DmsCache, q, k, v, logits, out=None, scale=None, stream=None):
    return cache.prefill(q, k, v, logits, out, scale, stream)


def dms_decode_attention(cache: DmsCache, q, out=None, scale=None, stream=None):
    return cache.decode_attention(q, out, scale, stream)


def dms_step(cache: DmsCache, k, v, evict_logit, q, out, scale=None, stream=None):
    return cache.step(k, v, evict_logit, q, out, scale, stream)


def dms_step_host(cache: DmsCache, k, v, evict_logit, q, out, scale=None, stream=None):
    return cache.step_host(k, v, evict_logit, q, out, scale, stream)


def dms_step_host_join(cache: DmsCache, stream=None) -> None:
    cache.host_join(stream)


def dms_step_graph_create(caches, k, v, evict_logit, q, out, scale) -> DmsStepGraph:
    return DmsStepGraph(caches, k, v, evict_logit, q, out, scale)


def dms_step_graph_launch(graph: DmsStepGraph, stream=None) -> None:
    graph.launch(stream)


def dms_step_graph_destroy(graph: DmsStepGraph) -> None:
    graph.close()


def dms_decode_attention_noalloc(k_pool: torch.Tensor, v_pool: torch.Tensor, lengths: torch.Tensor, q: torch.Tensor,
                                 out: torch.Tensor, scale: float | None = None, stream=None) -> torch.Tensor:
    """Decode attention over caller-owned pools with no device allocation
    (dms_decode_attention_noalloc).  k_pool, v_pool bf16 [B][Hkv][cap][D] (K in
    the library's chunk-permuted row layout), lengths int32 [B][Hkv], q bf16
    [B][Hq][D], out fp32 [B][Hq][D] (preallocated)."""
    lib = load_library()
    if k_pool.dim() != 4:
        raise ValueError("k_pool must be [batch][kv_heads][capacity][head_dim]")
    B, H, cap, D = k_pool.shape
    dev = k_pool.device
    Hq = q.shape[1] if q.dim() == 3 else -1
    _need(k_pool, "k_pool", torch.bfloat16, (B, H, cap, D), dev)
    _need(v_pool, "v_pool", torch.bfloat16, (B, H, cap, D), dev)
    _need(lengths, "lengths", torch.int32, (B, H), dev)
    _need(q, "q", torch.bfloat16, (B, Hq, D), dev)
    _need(out, "out", torch.float32, (B, Hq, D), dev)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib.dms_decode_attention_noalloc(k_pool.data_ptr(), v_pool.data_ptr(), lengths.data_ptr(), B, H, cap, D,
                                            q.data_ptr(), out.data_ptr(), scale, Hq, _stream_handle(stream)),
           "dms_decode_attention_noalloc")
    return out


def dms_cache_lengths(cache: DmsCache, stream=None):
    return cache.lengths(stream)


def dms_cache_slot_positions(cache: DmsCache, stream=None):
    return cache.slot_positions(stream)


def dms_cache_status(cache: DmsCache, stream=None) -> int:
    return cache.status(stream)


def dms_cache_destroy(cache: DmsCache) -> None:
    cache.close()
