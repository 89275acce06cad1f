"""Python binding of the GB300 multi-LoRA segmented linear (C ABI in include/lora.h).

Argument marshalling only: every step of the path runs in the CUDA library
``_lib/liblora_gb300.so``.  PyTorch supplies device memory and streams.  There is no
CPU or PyTorch fallback: the library is mapped on the first call into it (or by
``load_library()``), and if it is missing or fails to load, that call raises ImportError.
Importing the package alone maps nothing, so host-only users of the package (the seeded
input generators in ``workloads``) do not load the CUDA library.

Same names as the C ABI (the ``EXPORTED`` tuple: pool, segment, linear, grouped-linear and
host-tier cache entry points), plus small ``LoraPool`` and ``LoraCache`` convenience wrappers;
``LoraPool`` owns the pool's device buffer.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "liblora_gb300.so")

LORA_F32, LORA_F16, LORA_BF16 = 0, 1, 2
LORA_OK, LORA_EINVAL, LORA_ESLOT, LORA_EBUSY, LORA_ERANK = 0, -1, -2, -3, -4
LORA_ENOSPACE, LORA_EIDX, LORA_ECUDA, LORA_EUNSUP, LORA_ETIMEOUT = -5, -6, -7, -8, -9
LORA_VARIANT_AUTO, LORA_VARIANT_FUSED, LORA_VARIANT_SEPARATE, LORA_VARIANT_CUDA_CORE = 0, 1, 2, 3

TORCH_TO_LORA = {torch.float32: LORA_F32, torch.float16: LORA_F16, torch.bfloat16: LORA_BF16}

EXPORTED = (
    "lora_pool_bytes", "lora_pool_create", "lora_pool_destroy", "lora_pool_load_slot", "lora_pool_unload_slot",
    "lora_segment_workspace_bytes", "lora_segment", "lora_segment_status", "lora_linear_workspace_bytes",
    "lora_linear_fwd", "lora_linear_policy", "lora_last_error", "lora_kernel_launch_count",
    "lora_set_timing_events", "lora_linear_fwd_static_ws", "lora_linear_fwd_ex", "lora_pool_load_slots",
    "lora_linear_group_workspace_bytes", "lora_linear_fwd_group", "lora_linear_group_policy",
    "lora_cache_create", "lora_cache_destroy", "lora_cache_register", "lora_cache_unregister", "lora_cache_map",
    "lora_cache_slot_of", "lora_cache_stats", "lora_wait_selftest", "lora_set_kernel_stamps", "lora_set_aux_stamps",
    "lora_loader_create", "lora_loader_destroy", "lora_loader_mount", "lora_loader_acquire", "lora_loader_release",
    "lora_loader_stats",
)


class LoraError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class lora_pool_desc(ctypes.Structure):
    _fields_ = [("h_in", ctypes.c_int32), ("h_out", ctypes.c_int32), ("r_max", ctypes.c_int32),
                ("n_slots", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class lora_segments(ctypes.Structure):
    _fields_ = [("perm_dev", ctypes.c_void_p), ("seg_start_dev", ctypes.c_void_p), ("seg_slot_dev", ctypes.c_void_p),
                ("nseg_dev", ctypes.c_void_p), ("status_dev", ctypes.c_void_p), ("idx_dev", ctypes.c_void_p),
                ("items_dev", ctypes.c_void_p), ("n_tokens", ctypes.c_int32), ("n_slots", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
                          " (there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    P = ctypes.POINTER
    sig = {
        "lora_pool_bytes": [P(lora_pool_desc), P(sz)],
        "lora_pool_create": [P(lora_pool_desc), vp, sz, vp, P(vp)],
        "lora_pool_destroy": [vp],
        "lora_pool_load_slot": [vp, i32, vp, vp, i32, ctypes.c_float, vp],
        "lora_pool_unload_slot": [vp, i32, vp],
        "lora_pool_load_slots": [vp, i32, P(i32), P(vp), P(vp), P(i32), P(ctypes.c_float), vp],
        "lora_segment_workspace_bytes": [i32, i32, P(sz)],
        "lora_segment": [vp, i32, vp, vp, sz, P(lora_segments), vp],
        "lora_segment_status": [P(lora_segments), vp, P(i32)],
        "lora_linear_workspace_bytes": [vp, i32, P(sz)],
        "lora_linear_fwd": [vp, vp, vp, vp, P(lora_segments), i32, vp, sz, vp],
        "lora_linear_policy": [vp, i32, P(i32)],
        "lora_set_timing_events": [vp, vp, vp],
        "lora_linear_fwd_static_ws": [vp, vp, vp, vp, P(lora_segments), i32, vp],
        "lora_linear_fwd_ex": [vp, vp, vp, vp, P(lora_segments), i32, vp, sz, vp, sz, vp],
        "lora_linear_group_workspace_bytes": [i32, P(vp), i32, P(sz)],
        "lora_linear_fwd_group": [i32, P(vp), vp, vp, vp, P(lora_segments), i32, vp, sz, vp],
        "lora_linear_group_policy": [i32, P(vp), i32, P(i32)],
        "lora_cache_create": [i32, P(vp), P(vp)],
        "lora_cache_destroy": [vp],
        "lora_cache_register": [vp, ctypes.c_int64, P(vp), P(vp), P(i32), P(ctypes.c_float)],
        "lora_cache_unregister": [vp, ctypes.c_int64, vp],
        "lora_cache_map": [vp, P(ctypes.c_int64), i32, P(ctypes.c_int32), P(i32), vp],
        "lora_cache_slot_of": [vp, ctypes.c_int64, P(i32)],
        "lora_cache_stats": [vp, P(ctypes.c_uint64), P(ctypes.c_uint64), P(ctypes.c_uint64)],
        "lora_wait_selftest": [vp, vp, i32, i32, ctypes.c_uint64, vp],
        "lora_set_kernel_stamps": [vp, i32],
        "lora_set_aux_stamps": [vp, i32],
        "lora_loader_create": [i32, P(vp), vp, P(vp)],
        "lora_loader_destroy": [vp],
        "lora_loader_mount": [vp, i32, P(i32), P(vp), P(vp), P(i32), P(ctypes.c_float)],
        "lora_loader_acquire": [vp, i32, P(i32), vp],
        "lora_loader_release": [vp, i32, P(i32), vp],
        "lora_loader_stats": [vp, P(ctypes.c_uint64), P(ctypes.c_uint64)],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.lora_last_error.argtypes = []
    lib.lora_last_error.restype = ctypes.c_char_p
    lib.lora_kernel_launch_count.argtypes = []
    lib.lora_kernel_launch_count.restype = ctypes.c_uint64
    return lib


class _LazyLibrary:
    """The CDLL, mapped on first attribute access; a missing library raises there."""

    _cdll: Optional[ctypes.CDLL] = None

    def __getattr__(self, name):
        if _LazyLibrary._cdll is None:
            _LazyLibrary._cdll = _load()
        return getattr(_LazyLibrary._cdll, name)


_lib = _LazyLibrary()


def load_library() -> ctypes.CDLL:
    """Map the CUDA library now (ImportError if it is missing or broken) and return it."""
    _lib.lora_last_error  # noqa: B018  (attribute access maps the library)
    return _LazyLibrary._cdll


def lora_last_error() -> str:
    return _lib.lora_last_error().decode()


def lora_kernel_launch_count() -> int:
    return int(_lib.lora_kernel_launch_count())


def lora_set_timing_events(before_shrink=None, before_gemm=None, after_gemm=None) -> None:
    """Events (torch.cuda.Event, already recorded once so they exist) recorded around the
    kernels of every following lora_linear_fwd; call with no arguments to disable."""
    def h(e):
        return ctypes.c_void_p(0 if e is None else e.cuda_event)

    _check(_lib.lora_set_timing_events(h(before_shrink), h(before_gemm), h(after_gemm)))


def lora_set_kernel_stamps(stamps: Optional[torch.Tensor] = None) -> None:
    """While set (a device int64 tensor [pairs, 2]), every base-GEMM launch records the
    %globaltimer of its first CTA's start and last CTA's end into the next pair (round robin);
    initialise pairs to (-1, 0) (unsigned: UINT64_MAX, 0).  No argument disables."""
    if stamps is None:
        _check(_lib.lora_set_kernel_stamps(ctypes.c_void_p(0), 0))
        return
    if stamps.dtype != torch.int64 or stamps.dim() != 2 or stamps.shape[1] != 2 or not stamps.is_contiguous():
        raise ValueError("stamps must be a contiguous int64 tensor of shape [pairs, 2]")
    _check(_lib.lora_set_kernel_stamps(_ptr(_dev(stamps, "stamps")), int(stamps.shape[0])))


def lora_set_aux_stamps(stamps: Optional[torch.Tensor] = None) -> None:
    """While set (a device int64 tensor [triples, 3]), every shrink / segmented-expand launch of
    the decode path records {first CTA start, first grid-dependency wait return, last CTA end}
    (%globaltimer ns) into the next triple; initialise to (-1, -1, 0).  No argument disables."""
    if stamps is None:
        _check(_lib.lora_set_aux_stamps(ctypes.c_void_p(0), 0))
        return
    if stamps.dtype != torch.int64 or stamps.dim() != 2 or stamps.shape[1] != 3 or not stamps.is_contiguous():
        raise ValueError("stamps must be a contiguous int64 tensor of shape [triples, 3]")
    _check(_lib.lora_set_aux_stamps(_ptr(_dev(stamps, "stamps")), int(stamps.shape[0])))


def lora_wait_selftest(status: torch.Tensor, out: torch.Tensor, arrive: bool, limit_ns: int, stream=None) -> None:
    """Run the library's bounded pipeline wait on a barrier that completes only if ``arrive``:
    a wait that gives up sets status (device int32 [1]) to LORA_ETIMEOUT and leaves out
    (device float32) unwritten; otherwise out is filled with 1.0."""
    if status.dtype != torch.int32 or out.dtype != torch.float32:
        raise ValueError("status must be int32 and out float32")
    _check(_lib.lora_wait_selftest(_ptr(_dev(status, "status")), _ptr(_dev(out, "out")), out.numel(),
                                   1 if arrive else 0, int(limit_ns), _stream(stream)))


def _check(rc: int) -> None:
    if rc != LORA_OK:
        raise LoraError(rc, lora_last_error())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dev(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ---- same-named wrappers of the C ABI ------------------------------------------------------

def lora_pool_bytes(h_in: int, h_out: int, r_max: int, n_slots: int, dtype: torch.dtype) -> int:
    d = lora_pool_desc(h_in, h_out, r_max, n_slots, TORCH_TO_LORA[dtype])
    out = ctypes.c_size_t()
    _check(_lib.lora_pool_bytes(ctypes.byref(d), ctypes.byref(out)))
    return out.value


def lora_pool_create(h_in: int, h_out: int, r_max: int, n_slots: int, dtype: torch.dtype, dev_mem: torch.Tensor,
                     stream=None) -> ctypes.c_void_p:
    d = lora_pool_desc(h_in, h_out, r_max, n_slots, TORCH_TO_LORA[dtype])
    h = ctypes.c_void_p()
    _check(_lib.lora_pool_create(ctypes.byref(d), _ptr(_dev(dev_mem, "dev_mem")),
                                 dev_mem.numel() * dev_mem.element_size(), _stream(stream), ctypes.byref(h)))
    return h


def lora_pool_destroy(handle) -> None:
    _check(_lib.lora_pool_destroy(handle))


def _dev_or_pinned(t: torch.Tensor, name: str) -> torch.Tensor:
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def lora_pool_load_slot(handle, slot: int, A: torch.Tensor, B: torch.Tensor, rank: int, alpha: float,
                        stream=None) -> None:
    """A and B: device tensors or pinned host tensors (read by the mounting kernel directly)."""
    _check(_lib.lora_pool_load_slot(handle, slot, _ptr(_dev_or_pinned(A, "A")), _ptr(_dev_or_pinned(B, "B")), rank,
                                    float(alpha), _stream(stream)))


def lora_pool_load_slots(handle, slots, As, Bs, alphas, stream=None) -> None:
    """Mount len(slots) adapters with one call (As[i], Bs[i]: device or pinned host tensors)."""
    n = len(slots)
    if not (len(As) == len(Bs) == len(alphas) == n):
        raise ValueError("slots, As, Bs and alphas must have the same length")
    As = [_dev_or_pinned(a, "A") for a in As]
    Bs = [_dev_or_pinned(b, "B") for b in Bs]
    arr_i = (ctypes.c_int32 * max(n, 1))
    arr_p = (ctypes.c_void_p * max(n, 1))
    arr_f = (ctypes.c_float * max(n, 1))
    _check(_lib.lora_pool_load_slots(handle, n, arr_i(*[int(s) for s in slots]), arr_p(*[a.data_ptr() for a in As]),
                                     arr_p(*[b.data_ptr() for b in Bs]), arr_i(*[int(a.shape[0]) for a in As]),
                                     arr_f(*[float(x) for x in alphas]), _stream(stream)))


def lora_pool_unload_slot(handle, slot: int, stream=None) -> None:
    _check(_lib.lora_pool_unload_slot(handle, slot, _stream(stream)))


def lora_segment_workspace_bytes(n_tokens: int, n_slots: int) -> int:
    out = ctypes.c_size_t()
    _check(_lib.lora_segment_workspace_bytes(n_tokens, n_slots, ctypes.byref(out)))
    return out.value


def lora_segment(idx: torch.Tensor, pool_handle, ws: torch.Tensor, stream=None) -> lora_segments:
    if idx.dtype != torch.int32:
        raise ValueError("idx must be int32")
    seg = lora_segments()
    _check(_lib.lora_segment(_ptr(_dev(idx, "idx")) if idx.numel() else ctypes.c_void_p(0), idx.numel(), pool_handle,
                             _ptr(_dev(ws, "ws")), ws.numel() * ws.element_size(), ctypes.byref(seg),
                             _stream(stream)))
    return seg


def lora_segment_status(seg: lora_segments, stream=None) -> int:
    out = ctypes.c_int()
    _check(_lib.lora_segment_status(ctypes.byref(seg), _stream(stream), ctypes.byref(out)))
    return out.value


def lora_linear_workspace_bytes(pool_handle, n_tokens: int) -> int:
    out = ctypes.c_size_t()
    _check(_lib.lora_linear_workspace_bytes(pool_handle, n_tokens, ctypes.byref(out)))
    return out.value


def lora_linear_fwd_ex(pool_handle, W: torch.Tensor, x: torch.Tensor, y: torch.Tensor, seg: lora_segments,
                       ws: torch.Tensor, variant: int = LORA_VARIANT_AUTO, prefetch: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """lora_linear_fwd with an L2 prefetch hint: `prefetch` (e.g. the next linear's weight) is
    streamed into L2 while this call's epilogue runs.  Results are identical without it."""
    pf = _ptr(_dev(prefetch, "prefetch")) if prefetch is not None else ctypes.c_void_p(0)
    pf_bytes = prefetch.numel() * prefetch.element_size() if prefetch is not None else 0
    _check(_lib.lora_linear_fwd_ex(pool_handle, _ptr(_dev(W, "W")), _ptr(_dev(x, "x")), _ptr(_dev(y, "y")),
                                   ctypes.byref(seg), variant, _ptr(_dev(ws, "ws")), ws.numel() * ws.element_size(),
                                   pf, pf_bytes, _stream(stream)))
    return y


def lora_linear_fwd_static_ws(pool_handle, W: torch.Tensor, x: torch.Tensor, y: torch.Tensor, seg: lora_segments,
                              variant: int = LORA_VARIANT_AUTO, stream=None) -> torch.Tensor:
    """lora_linear_fwd for callers that cannot allocate a workspace: the library's own fixed
    4 MiB device array holds the shrink output (LORA_ENOSPACE beyond it).  The pool's device
    must be current.  Calls that may overlap on the GPU share the array and race; the first
    call on a device (which looks the array up) must come before any stream capture."""
    _check(_lib.lora_linear_fwd_static_ws(pool_handle, _ptr(_dev(W, "W")), _ptr(_dev(x, "x")), _ptr(_dev(y, "y")),
                                          ctypes.byref(seg), variant, _stream(stream)))
    return y


def lora_linear_policy(pool_handle, n_tokens: int) -> int:
    out = ctypes.c_int()
    _check(_lib.lora_linear_policy(pool_handle, n_tokens, ctypes.byref(out)))
    return out.value


def lora_linear_fwd(pool_handle, W: torch.Tensor, x: torch.Tensor, y: torch.Tensor, seg: lora_segments,
                    ws: torch.Tensor, variant: int = LORA_VARIANT_AUTO, stream=None) -> torch.Tensor:
    _check(_lib.lora_linear_fwd(pool_handle, _ptr(_dev(W, "W")), _ptr(_dev(x, "x")), _ptr(_dev(y, "y")),
                                ctypes.byref(seg), variant, _ptr(_dev(ws, "ws")), ws.numel() * ws.element_size(),
                                _stream(stream)))
    return y


def _handles(pool_handles) -> tuple:
    hs = list(pool_handles)
    arr = (ctypes.c_void_p * max(1, len(hs)))(*[h.value if isinstance(h, ctypes.c_void_p) else h for h in hs])
    return len(hs), arr


def lora_linear_group_workspace_bytes(pool_handles, n_tokens: int) -> int:
    count, arr = _handles(pool_handles)
    out = ctypes.c_size_t()
    _check(_lib.lora_linear_group_workspace_bytes(count, arr, n_tokens, ctypes.byref(out)))
    return out.value


def lora_linear_group_policy(pool_handles, n_tokens: int) -> int:
    count, arr = _handles(pool_handles)
    out = ctypes.c_int()
    _check(_lib.lora_linear_group_policy(count, arr, n_tokens, ctypes.byref(out)))
    return out.value


def lora_linear_fwd_group(pool_handles, W: torch.Tensor, x: torch.Tensor, y: torch.Tensor, seg: lora_segments,
                          ws: torch.Tensor, variant: int = LORA_VARIANT_AUTO, stream=None) -> torch.Tensor:
    """Projections sharing x and segments as one linear: W [sum h_out_q, h_in] (slices stacked
    row-wise, slice q's adapters in pool_handles[q]), y [n, sum h_out_q] (slice q = its column
    range)."""
    count, arr = _handles(pool_handles)
    _check(_lib.lora_linear_fwd_group(count, arr, _ptr(_dev(W, "W")), _ptr(_dev(x, "x")), _ptr(_dev(y, "y")),
                                      ctypes.byref(seg), variant, _ptr(_dev(ws, "ws")),
                                      ws.numel() * ws.element_size(), _stream(stream)))
    return y


def lora_cache_create(pool_handles) -> ctypes.c_void_p:
    count, arr = _handles(pool_handles)
    h = ctypes.c_void_p()
    _check(_lib.lora_cache_create(count, arr, ctypes.byref(h)))
    return h


def lora_cache_destroy(handle) -> None:
    _check(_lib.lora_cache_destroy(handle))


def lora_cache_register(handle, adapter_id: int, As, Bs, alphas) -> None:
    """As[p], Bs[p]: pinned host tensors of pool p ([rank, h_in], [h_out, rank]); kept alive by
    the caller until the adapter is unregistered."""
    for t in list(As) + list(Bs):
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError("adapter tensors of the host tier must be contiguous pinned host memory")
    n = len(As)
    Ap = (ctypes.c_void_p * n)(*[a.data_ptr() for a in As])
    Bp = (ctypes.c_void_p * n)(*[b.data_ptr() for b in Bs])
    ranks = (ctypes.c_int * n)(*[int(a.shape[0]) for a in As])
    al = (ctypes.c_float * n)(*[float(x) for x in alphas])
    _check(_lib.lora_cache_register(handle, int(adapter_id), Ap, Bp, ranks, al))


def lora_cache_unregister(handle, adapter_id: int, stream=None) -> None:
    _check(_lib.lora_cache_unregister(handle, int(adapter_id), _stream(stream)))


def lora_cache_map(handle, ids, stream=None):
    """ids: adapter id per token (-1 = base only).  Returns (idx int32 CPU tensor, mounts)."""
    ids = torch.as_tensor(ids, dtype=torch.int64).contiguous()
    n = int(ids.numel())
    idx = torch.empty(n, dtype=torch.int32)
    mounts = ctypes.c_int()
    _check(_lib.lora_cache_map(handle, ctypes.cast(ids.data_ptr(), ctypes.POINTER(ctypes.c_int64)), n,
                               ctypes.cast(idx.data_ptr(), ctypes.POINTER(ctypes.c_int32)), ctypes.byref(mounts),
                               _stream(stream)))
    return idx, mounts.value


def lora_cache_slot_of(handle, adapter_id: int) -> int:
    out = ctypes.c_int()
    _check(_lib.lora_cache_slot_of(handle, int(adapter_id), ctypes.byref(out)))
    return out.value


def lora_cache_stats(handle) -> dict:
    h, m, e = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
    _check(_lib.lora_cache_stats(handle, ctypes.byref(h), ctypes.byref(m), ctypes.byref(e)))
    return {"hits": h.value, "misses": m.value, "evictions": e.value}


class LoraCache:
    """Host-tier adapter cache over pools (``LoraPool`` objects) with the same slot count."""

    def __init__(self, pools):
        self.pools = list(pools)
        self.handle = lora_cache_create([p.handle for p in self.pools])
        self._host = {}

    def register(self, adapter_id: int, As, Bs, alphas) -> None:
        lora_cache_register(self.handle, adapter_id, As, Bs, alphas)
        self._host[int(adapter_id)] = (list(As), list(Bs))  # the host tier must stay alive

    def unregister(self, adapter_id: int, stream=None) -> None:
        lora_cache_unregister(self.handle, adapter_id, stream)
        self._host.pop(int(adapter_id), None)

    def map(self, ids, stream=None):
        return lora_cache_map(self.handle, ids, stream)

    def slot_of(self, adapter_id: int) -> int:
        return lora_cache_slot_of(self.handle, adapter_id)

    def stats(self) -> dict:
        return lora_cache_stats(self.handle)

    def close(self) -> None:
        if self.handle is not None:
            lora_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _slot_array(slots):
    slots = [int(s) for s in slots]
    return len(slots), (ctypes.c_int * max(1, len(slots)))(*slots)


def lora_loader_create(pool_handles, copy_stream) -> ctypes.c_void_p:
    count, arr = _handles(pool_handles)
    h = ctypes.c_void_p()
    _check(_lib.lora_loader_create(count, arr, _stream(copy_stream), ctypes.byref(h)))
    return h


def lora_loader_destroy(handle) -> None:
    _check(_lib.lora_loader_destroy(handle))


def lora_loader_mount(handle, slots, As, Bs, alphas) -> None:
    """As[p][i], Bs[p][i]: pinned host tensors of slot slots[i]'s adapter for pool p; alphas[i]
    its alpha (the same for every pool).  The caller keeps the tensors alive until the copy
    stream has passed the mount."""
    count, sl = _slot_array(slots)
    npools = len(As)
    flatA = [a for per_pool in As for a in per_pool]
    flatB = [b for per_pool in Bs for b in per_pool]
    for t in flatA + flatB:
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError("loader mounts read contiguous pinned host memory")
    Ap = (ctypes.c_void_p * max(1, len(flatA)))(*[a.data_ptr() for a in flatA])
    Bp = (ctypes.c_void_p * max(1, len(flatB)))(*[b.data_ptr() for b in flatB])
    ranks = (ctypes.c_int * max(1, len(flatA)))(*[int(a.shape[0]) for a in flatA])
    al = (ctypes.c_float * max(1, npools * count))(*[float(alphas[i]) for _ in range(npools) for i in range(count)])
    _check(_lib.lora_loader_mount(handle, count, sl, Ap, Bp, ranks, al))


def lora_loader_acquire(handle, slots, stream=None) -> None:
    count, sl = _slot_array(slots)
    _check(_lib.lora_loader_acquire(handle, count, sl, _stream(stream)))


def lora_loader_release(handle, slots, stream=None) -> None:
    count, sl = _slot_array(slots)
    _check(_lib.lora_loader_release(handle, count, sl, _stream(stream)))


def lora_loader_stats(handle) -> dict:
    m, d = ctypes.c_uint64(), ctypes.c_uint64()
    _check(_lib.lora_loader_stats(handle, ctypes.byref(m), ctypes.byref(d)))
    return {"mounts": m.value, "drained_fences": d.value}


class LoraLoader:
    """Background mounts into ``LoraPool`` objects (same slot count) on a copy stream, with
    acquire/release fences for the compute streams (see include/lora.h)."""

    def __init__(self, pools, copy_stream):
        self.pools = list(pools)
        self.copy_stream = copy_stream
        self.handle = lora_loader_create([p.handle for p in self.pools], copy_stream)
        self._keep = {}

    def mount(self, slots, As, Bs, alphas) -> None:
        lora_loader_mount(self.handle, slots, As, Bs, alphas)
        for t in [a for per_pool in As for a in per_pool] + [b for per_pool in Bs for b in per_pool]:
            self._keep[t.data_ptr()] = t  # host sources stay alive while the copy stream may read them

    def acquire(self, slots, stream=None) -> None:
        lora_loader_acquire(self.handle, slots, stream)

    def release(self, slots, stream=None) -> None:
        lora_loader_release(self.handle, slots, stream)

    def stats(self) -> dict:
        return lora_loader_stats(self.handle)

    def close(self) -> None:
        if self.handle is not None:
            lora_loader_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def segment_arrays(seg: lora_segments) -> dict:
    """Views (int32 device tensors) of the segment outputs inside the workspace ``seg._ws``."""
    ws = seg._ws
    base = ws.data_ptr()
    n, S = int(seg.n_tokens), int(seg.n_slots)

    def view(ptr, count):
        off = int(ptr) - base
        return ws[off:off + 4 * count].view(torch.int32)

    return {"perm": view(seg.perm_dev, n), "seg_start": view(seg.seg_start_dev, S + 2),
            "seg_slot": view(seg.seg_slot_dev, S + 1), "nseg": view(seg.nseg_dev, 4),
            "status": view(seg.status_dev, 1), "idx": view(seg.idx_dev, n), "items": view(seg.items_dev, 8 * n)}


# ---- convenience ----------------------------------------------------------------------------

def _device_bytes(nbytes: int, device) -> torch.Tensor:
    """A 256-byte aligned, zero-filled device byte buffer (torch's allocator aligns to 512)."""
    t = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
    assert t.data_ptr() % 256 == 0
    return t


class LoraPool:
    """One adapter pool (one linear layer) in a device buffer this object owns."""

    def __init__(self, h_in: int, h_out: int, r_max: int, n_slots: int, dtype: torch.dtype, device="cuda",
                 stream=None):
        self.h_in, self.h_out, self.r_max, self.n_slots, self.dtype = h_in, h_out, r_max, n_slots, dtype
        self.nbytes = lora_pool_bytes(h_in, h_out, r_max, n_slots, dtype)
        self.mem = _device_bytes(self.nbytes, device)
        self.handle = lora_pool_create(h_in, h_out, r_max, n_slots, dtype, self.mem, stream)
        self._ws = {}

    def load_slot(self, slot: int, A: torch.Tensor, B: torch.Tensor, alpha: float, stream=None) -> None:
        lora_pool_load_slot(self.handle, slot, A, B, int(A.shape[0]), alpha, stream)

    def load_slots(self, slots, As, Bs, alphas, stream=None) -> None:
        lora_pool_load_slots(self.handle, slots, As, Bs, alphas, stream)

    def unload_slot(self, slot: int, stream=None) -> None:
        lora_pool_unload_slot(self.handle, slot, stream)

    def segment_workspace(self, n_tokens: int, device="cuda") -> torch.Tensor:
        return _device_bytes(lora_segment_workspace_bytes(n_tokens, self.n_slots), device)

    def linear_workspace(self, n_tokens: int, device="cuda") -> torch.Tensor:
        return _device_bytes(lora_linear_workspace_bytes(self.handle, n_tokens), device)

    def segment(self, idx: torch.Tensor, ws: Optional[torch.Tensor] = None, stream=None):
        if ws is None:
            ws = self.segment_workspace(idx.numel(), idx.device)
        seg = lora_segment(idx, self.handle, ws, stream)
        seg._ws = ws  # keep the workspace alive with the segments
        return seg

    def linear(self, W: torch.Tensor, x: torch.Tensor, seg, variant: int = LORA_VARIANT_AUTO,
               y: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        n = int(seg.n_tokens)
        if y is None:
            y = torch.empty((n, self.h_out), dtype=self.dtype, device=x.device)
        if ws is None:
            key = (n, x.device)
            if key not in self._ws:
                self._ws[key] = self.linear_workspace(n, x.device)
            ws = self._ws[key]
        return lora_linear_fwd(self.handle, W, x, y, seg, ws, variant, stream)

    def close(self) -> None:
        if self.handle is not None:
            lora_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
