"""Python binding of ``libmoe_gb300.so`` (the C ABI of include/moe.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (PyTorch supplies device memory and streams).
The library must have been built (``routed_expert_prefill_gb300.build`` or
``__graft_entry__.build()``); there is no fallback of any kind.

Names mirror the C entry points:

* ``moe_route_topk(x, wr, k, rbias=None, want_logits=False)`` -> ``(idx, w[, logits])``
* ``moe_build_csr(idx, w, E, ws=None)`` -> ``Csr(offsets, rows, weights, slot_of)``
* ``moe_experts_fwd(x, csr, experts, shared, dims, flags=0, out=None, ws=None)`` -> ``out``
"""

from __future__ import annotations

import ctypes
import os
from typing import NamedTuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_DETERMINISTIC = 0x1
MOE_FORCE_SMALL_T = 0x2
MOE_FORCE_LARGE_T = 0x4
MOE_SIMPLE_KERNELS = 0x8
MOE_PACKED_WEIGHTS = 0x10
MOE_FUSED_DECODE = 0x20
MOE_STALL_WEIGHT_COPIES = 0x1
MOE_STALL_GRID_BARRIER = 0x2

# Every symbol include/moe.h declares.
EXPORTS = (
    "moe_last_error",
    "moe_status_string",
    "moe_route_topk",
    "moe_build_csr",
    "moe_route_csr",
    "moe_experts_fwd",
    "moe_workspace_bytes",
    "moe_clear_device_status",
    "moe_read_device_status",
    "moe_profile_enable",
    "moe_profile_read",
    "moe_packed_bytes",
    "moe_pack_experts",
    "moe_build_csr_noalloc",
    "moe_noalloc_read_status",
    "moe_forward",
    "moe_debug_stall",
    "moe_plan_residency",
    "moe_stream_slot_bytes",
    "moe_streamer_create",
    "moe_streamer_destroy",
    "moe_streamer_pool",
    "moe_forward_streamed",
)


class MoeDims(ctypes.Structure):
    _fields_ = [("t", ctypes.c_int32), ("h", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("shared_inter", ctypes.c_int32),
                ("bits", ctypes.c_int32)]


class MoeCsr(ctypes.Structure):
    _fields_ = [("offsets", ctypes.c_void_p), ("rows", ctypes.c_void_p),
                ("weights", ctypes.c_void_p), ("slot_of", ctypes.c_void_p)]


class MoeQWeights(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p)]


class MoeShared(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("gate", ctypes.c_void_p)]


class MoeProfileEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_double)]


class MoeStreamCfg(ctypes.Structure):
    _fields_ = [("pool_slots", ctypes.c_int32), ("ring_slots", ctypes.c_int32), ("group", ctypes.c_int32),
                ("miss_bits", ctypes.c_int32)]


class MoeResidencyPlan(ctypes.Structure):
    _fields_ = [("pool_expert", ctypes.c_void_p), ("pool_last", ctypes.c_void_p), ("rec", ctypes.c_void_p),
                ("batch", ctypes.c_void_p), ("copy_expert", ctypes.c_void_p), ("copy_slot", ctypes.c_void_p),
                ("wait_for", ctypes.c_void_p), ("n_copies", ctypes.c_int32), ("n_batches", ctypes.c_int32)]


class MoeStreamStats(ctypes.Structure):
    _fields_ = [("resident", ctypes.c_int32), ("filled", ctypes.c_int32), ("streamed", ctypes.c_int32),
                ("batches", ctypes.c_int32), ("bytes", ctypes.c_int64), ("prefetched", ctypes.c_int32),
                ("prefetch_used", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) and return the library; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first (python -m routed_expert_prefill_gb300.build "
            "or __graft_entry__.build()); the routed-MoE path has no fallback")
    lib = ctypes.CDLL(path)
    vp, i32, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
    lib.moe_last_error.restype = ctypes.c_char_p
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_route_topk.restype = ctypes.c_int
    lib.moe_route_topk.argtypes = [vp, vp, vp, ctypes.POINTER(MoeDims), vp, vp, vp, vp, sz, vp]
    lib.moe_build_csr.restype = ctypes.c_int
    lib.moe_build_csr.argtypes = [vp, vp, ctypes.POINTER(MoeDims), ctypes.POINTER(MoeCsr), vp, sz, vp]
    lib.moe_route_csr.restype = ctypes.c_int
    lib.moe_route_csr.argtypes = [vp, vp, vp, ctypes.POINTER(MoeDims), vp, vp, ctypes.POINTER(MoeCsr), vp, sz, vp]
    lib.moe_experts_fwd.restype = ctypes.c_int
    lib.moe_experts_fwd.argtypes = [vp, ctypes.POINTER(MoeCsr), ctypes.POINTER(MoeQWeights),
                                    ctypes.POINTER(MoeShared), vp, ctypes.POINTER(MoeDims), u32, vp, sz, vp]
    lib.moe_workspace_bytes.restype = sz
    lib.moe_workspace_bytes.argtypes = [ctypes.POINTER(MoeDims), u32]
    lib.moe_clear_device_status.restype = ctypes.c_int
    lib.moe_clear_device_status.argtypes = [vp, vp]
    lib.moe_read_device_status.restype = ctypes.c_int
    lib.moe_read_device_status.argtypes = [vp, vp]
    lib.moe_noalloc_read_status.restype = ctypes.c_int
    lib.moe_noalloc_read_status.argtypes = [vp]
    lib.moe_debug_stall.restype = ctypes.c_int
    lib.moe_debug_stall.argtypes = [vp, u32, vp]
    lib.moe_profile_enable.restype = ctypes.c_int
    lib.moe_profile_enable.argtypes = [ctypes.c_int]
    lib.moe_profile_read.restype = ctypes.c_int
    lib.moe_profile_read.argtypes = [ctypes.POINTER(MoeProfileEntry), ctypes.c_int]
    lib.moe_packed_bytes.restype = sz
    lib.moe_packed_bytes.argtypes = [ctypes.POINTER(MoeDims), ctypes.c_int]
    lib.moe_build_csr_noalloc.restype = ctypes.c_int
    lib.moe_build_csr_noalloc.argtypes = [vp, vp, ctypes.POINTER(MoeDims), ctypes.POINTER(MoeCsr), vp]
    lib.moe_forward.restype = ctypes.c_int
    lib.moe_forward.argtypes = [vp, vp, vp, ctypes.POINTER(MoeQWeights), ctypes.POINTER(MoeShared),
                                ctypes.POINTER(MoeDims), u32, vp, vp, ctypes.POINTER(MoeCsr), vp, vp, sz, vp]
    lib.moe_plan_residency.restype = ctypes.c_int
    lib.moe_plan_residency.argtypes = [vp, i32, ctypes.POINTER(MoeStreamCfg), ctypes.c_int64,
                                       ctypes.POINTER(MoeResidencyPlan)]
    lib.moe_stream_slot_bytes.restype = sz
    lib.moe_stream_slot_bytes.argtypes = [ctypes.POINTER(MoeDims), ctypes.POINTER(MoeStreamCfg)]
    lib.moe_streamer_create.restype = ctypes.c_int
    lib.moe_streamer_create.argtypes = [ctypes.POINTER(MoeDims), ctypes.POINTER(MoeStreamCfg),
                                        ctypes.POINTER(ctypes.c_void_p)]
    lib.moe_streamer_destroy.restype = ctypes.c_int
    lib.moe_streamer_destroy.argtypes = [vp]
    lib.moe_streamer_pool.restype = ctypes.c_int
    lib.moe_streamer_pool.argtypes = [vp, vp, i32]
    lib.moe_forward_streamed.restype = ctypes.c_int
    lib.moe_forward_streamed.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.POINTER(MoeShared), ctypes.POINTER(MoeDims), u32,
                                         vp, vp, ctypes.POINTER(MoeCsr), vp, vp, sz, vp, vp,
                                         ctypes.POINTER(MoeStreamStats)]
    lib.moe_pack_experts.restype = ctypes.c_int
    lib.moe_pack_experts.argtypes = [ctypes.POINTER(MoeQWeights), ctypes.POINTER(MoeDims), ctypes.c_int, vp, sz, vp]
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        lib = load_library()
        raise MoeError(status, f"{lib.moe_status_string(status).decode()}: {lib.moe_last_error().decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def dims_of(t: int, h: int, inter: int, E: int, k: int, shared_inter: int, bits: int = 4) -> MoeDims:
    return MoeDims(t, h, inter, E, k, shared_inter, bits)


def _code_bits(dims: MoeDims) -> int:
    return dims.bits or 4


class Csr(NamedTuple):
    offsets: torch.Tensor
    rows: torch.Tensor
    weights: torch.Tensor
    slot_of: torch.Tensor

    def c(self) -> MoeCsr:
        return MoeCsr(self.offsets.data_ptr(), self.rows.data_ptr(), self.weights.data_ptr(),
                      self.slot_of.data_ptr())


def workspace_bytes(dims: MoeDims, flags: int = 0) -> int:
    n = load_library().moe_workspace_bytes(ctypes.byref(dims), flags)
    if n == 0:
        raise MoeError(-2, "bad dims for moe_workspace_bytes")
    return n


def new_workspace(dims: MoeDims, flags: int = 0, device=None, stream=None) -> torch.Tensor:
    """A workspace tensor for ``dims``/``flags`` with cleared device status."""
    ws = torch.empty(workspace_bytes(dims, flags), dtype=torch.uint8, device=device or "cuda")
    _check(load_library().moe_clear_device_status(_ptr(ws), _stream(stream)))
    return ws


def _u16(t: torch.Tensor) -> torch.Tensor:
    if t.dtype not in (torch.bfloat16, torch.float16, torch.int16, torch.uint16):
        raise TypeError(f"expected a 16-bit tensor, got {t.dtype}")
    return t


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)  # bf16 values or their bit patterns
_F16 = (torch.float16, torch.int16, torch.uint16)


def _need(t, name: str, dtypes, shape=None, min_numel=None):
    """Check what the C ABI cannot see: dtype, layout, size and device.

    The library receives bare pointers, so a wrong dtype, a strided view,
    a short buffer or a tensor on another GPU would otherwise turn into
    out-of-bounds accesses on the device."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs at least {min_numel}")
    return t


def _on_current_device(**named):
    """Every tensor must live on the current CUDA device (the library launches there)."""
    cur = None
    for name, t in named.items():
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be on a CUDA device, got {t.device}")
        if cur is None:
            cur = torch.cuda.current_device()
        if t.device.index != cur:
            raise ValueError(f"{name} is on {t.device} but the current device is cuda:{cur}")


def _need_csr(c: "Csr", name: str, E: int, n: int):
    _need(c.offsets, f"{name}.offsets", (torch.int32,), min_numel=E + 1)
    _need(c.rows, f"{name}.rows", (torch.int32,), min_numel=n)
    _need(c.weights, f"{name}.weights", (torch.float32,), min_numel=n)
    _need(c.slot_of, f"{name}.slot_of", (torch.int32,), min_numel=n)
    return c


def _csr_named(c, name: str) -> dict:
    if c is None:
        return {}
    return {f"{name}.{f}": getattr(c, f) for f in ("offsets", "rows", "weights", "slot_of")}


def _need_ws(ws, dims: "MoeDims", flags: int):
    return _need(ws, "ws", (torch.uint8,), min_numel=workspace_bytes(dims, flags))


def moe_route_topk(x: torch.Tensor, wr: torch.Tensor, k: int, rbias: torch.Tensor | None = None,
                   want_logits: bool = False, out=None, ws: torch.Tensor | None = None, exact_pass: bool = False,
                   stream=None):
    """Router: x bf16 [t, h], wr bf16 [E, h] -> idx int32 [t, k], w fp32 [t, k] (, logits).

    Takes the tensor-core scoring path with exact refinement unless logits
    are wanted or ``exact_pass`` asks for the single fixed-order pass; both
    give the same idx and w.
    """
    lib = load_library()
    if x.dim() != 2 or wr.dim() != 2:
        raise ValueError("x must be [t, h] and wr [E, h]")
    t, h = x.shape
    E = wr.shape[0]
    _need(x, "x", _BF16)
    _need(wr, "wr", _BF16, shape=(E, h))
    if rbias is not None:
        _need(rbias, "rbias", (torch.float32,), shape=(E,))
    dims = MoeDims(t, h, 128, E, k, 0)
    if out is None:
        idx = torch.empty((t, k), dtype=torch.int32, device=x.device)
        w = torch.empty((t, k), dtype=torch.float32, device=x.device)
    else:
        idx, w = out
        _need(idx, "idx", (torch.int32,), shape=(t, k))
        _need(w, "w", (torch.float32,), shape=(t, k))
    logits = torch.empty((t, E), dtype=torch.float32, device=x.device) if want_logits else None
    use_ws = not (want_logits or exact_pass)
    if use_ws and ws is not None:
        _need_ws(ws, dims, 0)
    _on_current_device(x=x, wr=wr, rbias=rbias, idx=idx, w=w, ws=ws if use_ws else None)
    if use_ws and ws is None:
        ws = new_workspace(dims, 0, x.device, stream)
    wsp, wsn = (_ptr(ws), ws.numel()) if use_ws else (None, 0)
    _check(lib.moe_route_topk(_ptr(_u16(x)), _ptr(_u16(wr)), _ptr(rbias), ctypes.byref(dims), _ptr(idx),
                              _ptr(w), _ptr(logits), wsp, wsn, _stream(stream)))
    return (idx, w, logits) if want_logits else (idx, w)


def moe_build_csr(idx: torch.Tensor, w: torch.Tensor, E: int, ws: torch.Tensor | None = None,
                  out: Csr | None = None, stream=None) -> Csr:
    """Group (row, slot) pairs by expert: offsets [E+1], rows/weights/slot_of [t*k]."""
    lib = load_library()
    if idx.dim() != 2:
        raise ValueError("idx must be [t, k]")
    t, k = idx.shape
    _need(idx, "idx", (torch.int32,))
    _need(w, "w", (torch.float32,), shape=(t, k))
    dims = MoeDims(t, 128, 128, E, k, 0)
    if ws is not None:
        _need_ws(ws, dims, 0)
    if out is not None:
        _need_csr(out, "out", E, t * k)
    _on_current_device(idx=idx, w=w, ws=ws, **_csr_named(out, "out"))
    if ws is None:
        ws = new_workspace(dims, 0, idx.device, stream)
    if out is None:
        dev = idx.device
        out = Csr(torch.empty(E + 1, dtype=torch.int32, device=dev),
                  torch.empty(t * k, dtype=torch.int32, device=dev),
                  torch.empty(t * k, dtype=torch.float32, device=dev),
                  torch.empty(t * k, dtype=torch.int32, device=dev))
    c = out.c()
    _check(lib.moe_build_csr(_ptr(idx), _ptr(w), ctypes.byref(dims), ctypes.byref(c), _ptr(ws), ws.numel(),
                             _stream(stream)))
    return out


def moe_route_csr(x: torch.Tensor, wr: torch.Tensor, k: int, rbias: torch.Tensor | None = None,
                  ws: torch.Tensor | None = None, out_route=None, out_csr: Csr | None = None, stream=None):
    """Router and grouping in one call: the idx, w and Csr of moe_route_topk
    (tensor-core path) followed by moe_build_csr, with one launch fewer for
    t <= 16 rows."""
    lib = load_library()
    if x.dim() != 2 or wr.dim() != 2:
        raise ValueError("x must be [t, h] and wr [E, h]")
    t, h = x.shape
    E = wr.shape[0]
    _need(x, "x", _BF16)
    _need(wr, "wr", _BF16, shape=(E, h))
    if rbias is not None:
        _need(rbias, "rbias", (torch.float32,), shape=(E,))
    dims = MoeDims(t, h, 128, E, k, 0)
    dev = x.device
    idx = w = None
    if out_route is not None:
        idx, w = out_route
        _need(idx, "idx", (torch.int32,), shape=(t, k))
        _need(w, "w", (torch.float32,), shape=(t, k))
    if out_csr is not None:
        _need_csr(out_csr, "out_csr", E, t * k)
    if ws is not None:
        _need_ws(ws, dims, 0)
    _on_current_device(x=x, wr=wr, rbias=rbias, idx=idx, w=w, ws=ws, **_csr_named(out_csr, "out_csr"))
    if out_route is None:
        idx = torch.empty((t, k), dtype=torch.int32, device=dev)
        w = torch.empty((t, k), dtype=torch.float32, device=dev)
    if out_csr is None:
        out_csr = Csr(torch.empty(E + 1, dtype=torch.int32, device=dev),
                      torch.empty(t * k, dtype=torch.int32, device=dev),
                      torch.empty(t * k, dtype=torch.float32, device=dev),
                      torch.empty(t * k, dtype=torch.int32, device=dev))
    if ws is None:
        ws = new_workspace(dims, 0, dev, stream)
    c = out_csr.c()
    _check(lib.moe_route_csr(_ptr(_u16(x)), _ptr(_u16(wr)), _ptr(rbias), ctypes.byref(dims), _ptr(idx), _ptr(w),
                             ctypes.byref(c), _ptr(ws), ws.numel(), _stream(stream)))
    return idx, w, out_csr


def moe_build_csr_noalloc(idx: torch.Tensor, w: torch.Tensor, E: int, out: Csr | None = None,
                          stream=None) -> Csr:
    """moe_build_csr with the library's fixed scratch instead of a workspace
    (for callers that may not allocate; at most MOE_NOALLOC_MAX_PAIRS = 65536
    (row, slot) pairs).  Only the output tensors are the caller's."""
    lib = load_library()
    if idx.dim() != 2:
        raise ValueError("idx must be [t, k]")
    t, k = idx.shape
    _need(idx, "idx", (torch.int32,))
    _need(w, "w", (torch.float32,), shape=(t, k))
    dims = MoeDims(t, 128, 128, E, k, 0)
    if out is not None:
        _need_csr(out, "out", E, t * k)
    _on_current_device(idx=idx, w=w, **_csr_named(out, "out"))
    if out is None:
        dev = idx.device
        out = Csr(torch.empty(E + 1, dtype=torch.int32, device=dev),
                  torch.empty(t * k, dtype=torch.int32, device=dev),
                  torch.empty(t * k, dtype=torch.float32, device=dev),
                  torch.empty(t * k, dtype=torch.int32, device=dev))
    c = out.c()
    _check(lib.moe_build_csr_noalloc(_ptr(idx), _ptr(w), ctypes.byref(dims), ctypes.byref(c), _stream(stream)))
    return out


def noalloc_read_status(stream=None) -> int:
    """Synchronise and return the status of moe_build_csr_noalloc's scratch on
    the current device (0 = clean, MOE_EDEVICE = an id out of range was
    dropped since the last read); clears it."""
    return load_library().moe_noalloc_read_status(_stream(stream))


def moe_experts_fwd(x: torch.Tensor, csr: Csr, experts: tuple, shared: tuple | None, dims: MoeDims,
                    flags: int = 0, out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Expert FFNs.  experts = (codes u8 [E, rec], scales f16 [E, g], biases f16 [E, g]);
    shared = (codes, scales, biases, gate-or-None) or None."""
    lib = load_library()
    t, h, I, Is, E, k = dims.t, dims.h, dims.inter, dims.shared_inter, dims.E, dims.k
    _need(x, "x", _BF16, shape=(t, h))
    _need_csr(csr, "csr", E, t * k)
    packed = bool(flags & MOE_PACKED_WEIGHTS)

    def need_record(rec, name, n_rec, inter):
        if packed:
            nbytes = lib.moe_packed_bytes(ctypes.byref(MoeDims(t, h, I, E, k, Is, dims.bits)),
                                          1 if name == "shared" else 0)
            _need(rec[0], f"{name} codes", (torch.uint8,), min_numel=nbytes)
        else:
            _need(rec[0], f"{name} codes", (torch.uint8,), min_numel=n_rec * 3 * inter * h * _code_bits(dims) // 8)
            _need(rec[1], f"{name} scales", _F16, min_numel=n_rec * 3 * inter * h // 64)
            _need(rec[2], f"{name} biases", _F16, min_numel=n_rec * 3 * inter * h // 64)

    need_record(experts, "experts", E, I)
    if Is > 0:
        if shared is None:
            raise ValueError("dims.shared_inter > 0 but no shared expert given")
        need_record(shared, "shared", 1, Is)
        if shared[3] is not None:
            _need(shared[3], "shared gate", _BF16, shape=(h,))
    if ws is not None:
        _need_ws(ws, dims, flags)
    if out is not None:
        _need(out, "out", _BF16, shape=(t, h))
    recs = {f"experts[{i}]": experts[i] for i in range(3)}
    if Is > 0:
        recs.update({f"shared[{i}]": shared[i] for i in range(4)})
    _on_current_device(x=x, ws=ws, out=out, **_csr_named(csr, "csr"), **recs)
    if ws is None:
        ws = new_workspace(dims, flags, x.device, stream)
    if out is None:
        out = torch.empty((dims.t, dims.h), dtype=torch.bfloat16, device=x.device)
    dp = lambda t_: None if t_ is None else t_.data_ptr()  # noqa: E731
    q = MoeQWeights(dp(experts[0]), dp(experts[1]), dp(experts[2]))
    sh = None
    if shared is not None:
        sh = MoeShared(dp(shared[0]), dp(shared[1]), dp(shared[2]), dp(shared[3]))
    c = csr.c()
    _check(lib.moe_experts_fwd(_ptr(_u16(x)), ctypes.byref(c), ctypes.byref(q),
                               ctypes.byref(sh) if sh is not None else None, _ptr(out), ctypes.byref(dims),
                               flags, _ptr(ws), ws.numel(), _stream(stream)))
    return out


def profile_enable(on: bool) -> None:
    """Start (clearing old records) or stop per-launch accounting in the library."""
    _check(load_library().moe_profile_enable(1 if on else 0))


def profile_read() -> dict:
    """{kernel name: (launches, total ms)} recorded since profile_enable(True)."""
    buf = (MoeProfileEntry * 64)()
    n = load_library().moe_profile_read(buf, 64)
    if n < 0:
        _check(n)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n)}


def pack_experts(codes: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor, dims: MoeDims,
                 shared: bool = False, stream=None) -> torch.Tensor:
    """Tile-contiguous packed copy of the routed (or shared) expert records."""
    lib = load_library()
    n = lib.moe_packed_bytes(ctypes.byref(dims), 1 if shared else 0)
    if n == 0:
        raise MoeError(-2, "nothing to pack for these dims")
    n_rec, inter = (1, dims.shared_inter) if shared else (dims.E, dims.inter)
    _need(codes, "codes", (torch.uint8,), min_numel=n_rec * 3 * inter * dims.h * _code_bits(dims) // 8)
    _need(scales, "scales", _F16, min_numel=n_rec * 3 * inter * dims.h // 64)
    _need(biases, "biases", _F16, min_numel=n_rec * 3 * inter * dims.h // 64)
    _on_current_device(codes=codes, scales=scales, biases=biases)
    dst = torch.empty(n, dtype=torch.uint8, device=codes.device)
    q = MoeQWeights(codes.data_ptr(), scales.data_ptr(), biases.data_ptr())
    _check(lib.moe_pack_experts(ctypes.byref(q), ctypes.byref(dims), 1 if shared else 0, _ptr(dst), n,
                                _stream(stream)))
    return dst


def debug_stall(ws: torch.Tensor, what: int, stream=None) -> None:
    """Test hook: make one kind of bounded device wait run out on the calls
    that use ``ws`` until read_device_status clears it (MOE_STALL_* bits)."""
    _need(ws, "ws", (torch.uint8,))
    _check(load_library().moe_debug_stall(_ptr(ws), what, _stream(stream)))


def read_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise and return the device-side status (0 = clean); clears it."""
    return load_library().moe_read_device_status(_ptr(ws), _stream(stream))


# ---------------------------------------------------------------------------
# Convenience: host inputs (routed_expert_prefill_gb300.synth layout) -> device,
# and the three calls chained on one stream.
# ---------------------------------------------------------------------------

def upload_inputs(inp: dict, device="cuda") -> dict:
    """Copy the numpy inputs of ``synth.make_inputs`` to device tensors."""
    import numpy as np

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    def f16(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    d = dict(
        x=bf(inp["x"]), wr=bf(inp["wr"]),
        rbias=None if inp.get("rbias") is None else torch.from_numpy(inp["rbias"]).to(device),
        codes=torch.from_numpy(inp["codes"]).to(device), scales=f16(inp["scales"]), biases=f16(inp["biases"]),
        shared_codes=torch.from_numpy(inp["shared_codes"]).to(device),
        shared_scales=f16(inp["shared_scales"]), shared_biases=f16(inp["shared_biases"]),
        shared_gate=None if inp.get("shared_gate") is None else bf(inp["shared_gate"]),
    )
    return d


def add_packed(dev: dict, dims: MoeDims, stream=None) -> dict:
    """Add packed weight records (dev["packed"], dev["shared_packed"]) to uploaded inputs."""
    dev["packed"] = pack_experts(dev["codes"], dev["scales"], dev["biases"], dims, False, stream)
    if dims.shared_inter > 0:
        dev["shared_packed"] = pack_experts(dev["shared_codes"], dev["shared_scales"], dev["shared_biases"], dims,
                                            True, stream)
    return dev


def moe_forward(dev: dict, dims: MoeDims, flags: int = MOE_PACKED_WEIGHTS, ws: torch.Tensor | None = None,
                out: torch.Tensor | None = None, stream=None, bufs: dict | None = None) -> dict:
    """The whole block through the C entry point moe_forward (router, grouping
    and expert FFNs in one call; one launch for decode-shaped chunks);
    returns the intermediate tensors too.

    By default (MOE_PACKED_WEIGHTS in `flags`) the packed records of
    add_packed() are used, made on the first call when absent; flags without
    it run the row-major records as uploaded."""
    if flags & MOE_PACKED_WEIGHTS and "packed" not in dev:
        add_packed(dev, dims, stream)
    lib = load_library()
    x, wr, rbias = dev["x"], dev["wr"], dev.get("rbias")
    t, h, I, Is, E, k = dims.t, dims.h, dims.inter, dims.shared_inter, dims.E, dims.k
    _need(x, "x", _BF16, shape=(t, h))
    _need(wr, "wr", _BF16, shape=(E, h))
    if rbias is not None:
        _need(rbias, "rbias", (torch.float32,), shape=(E,))
    packed = bool(flags & MOE_PACKED_WEIGHTS)
    if packed:
        experts = (dev["packed"], None, None)
        shared = (dev["shared_packed"], None, None, dev.get("shared_gate")) if Is > 0 else None
    else:
        experts = (dev["codes"], dev["scales"], dev["biases"])
        shared = ((dev["shared_codes"], dev["shared_scales"], dev["shared_biases"], dev.get("shared_gate"))
                  if Is > 0 else None)
    b = bufs or {}
    dev_ = x.device
    idx, w = b.get("route") or (torch.empty((t, k), dtype=torch.int32, device=dev_),
                                torch.empty((t, k), dtype=torch.float32, device=dev_))
    csr = b.get("csr") or Csr(torch.empty(E + 1, dtype=torch.int32, device=dev_),
                              torch.empty(t * k, dtype=torch.int32, device=dev_),
                              torch.empty(t * k, dtype=torch.float32, device=dev_),
                              torch.empty(t * k, dtype=torch.int32, device=dev_))
    _need(idx, "idx", (torch.int32,), shape=(t, k))
    _need(w, "w", (torch.float32,), shape=(t, k))
    _need_csr(csr, "csr", E, t * k)
    for i, name in enumerate(("codes", "scales", "biases")):
        if experts[i] is not None:
            _need(experts[i], f"experts {name}", (torch.uint8,) if i == 0 else _F16)
    if ws is None:
        ws = new_workspace(dims, flags, dev_, stream)
    else:
        _need_ws(ws, dims, flags)
    if out is None:
        out = torch.empty((t, h), dtype=torch.bfloat16, device=dev_)
    else:
        _need(out, "out", _BF16, shape=(t, h))
    recs = {f"experts[{i}]": experts[i] for i in range(3)}
    if shared is not None:
        recs.update({f"shared[{i}]": shared[i] for i in range(4)})
    _on_current_device(x=x, wr=wr, rbias=rbias, idx=idx, w=w, ws=ws, out=out, **_csr_named(csr, "csr"), **recs)
    dp = lambda t_: None if t_ is None else t_.data_ptr()  # noqa: E731
    q = MoeQWeights(dp(experts[0]), dp(experts[1]), dp(experts[2]))
    sh = MoeShared(dp(shared[0]), dp(shared[1]), dp(shared[2]), dp(shared[3])) if shared is not None else None
    c = csr.c()
    _check(lib.moe_forward(_ptr(x), _ptr(wr), _ptr(rbias), ctypes.byref(q), ctypes.byref(sh) if sh else None,
                           ctypes.byref(dims), flags, _ptr(idx), _ptr(w), ctypes.byref(c), _ptr(out), _ptr(ws),
                           ws.numel(), _stream(stream)))
    return dict(idx=idx, w=w, csr=csr, out=out, ws=ws)


# ---------------------------------------------------------------------------
# Streamed experts: records in host memory, a device pool and ring of slots.
# ---------------------------------------------------------------------------

def plan_residency(counts, pool_expert, pool_last, call: int, ring: int, group: int) -> dict:
    """One chunk's residency plan (host code of the library, no GPU).

    counts int [E]; pool_expert int [P] and pool_last int [P] are the pool
    table before the chunk.  Returns the plan with the updated table, in
    the keys rec, batch, copies [(expert, slot)], n_batches, wait_for,
    pool_expert, pool_last."""
    import numpy as np

    lib = load_library()
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    E = counts.size
    pe = np.array(pool_expert, dtype=np.int32)
    pl_ = np.array(pool_last, dtype=np.int64)
    rec = np.empty(E, np.int32)
    batch = np.empty(E, np.int32)
    ce = np.empty(E, np.int32)
    cs = np.empty(E, np.int32)
    wf = np.empty(E + 1, np.int32)
    cfg = MoeStreamCfg(pe.size, ring, group, 0)
    addr = lambda a: a.ctypes.data if a.size else None  # noqa: E731
    plan = MoeResidencyPlan(addr(pe), addr(pl_), rec.ctypes.data, batch.ctypes.data, ce.ctypes.data,
                            cs.ctypes.data, wf.ctypes.data, 0, 0)
    _check(lib.moe_plan_residency(counts.ctypes.data, E, ctypes.byref(cfg), call, ctypes.byref(plan)))
    nc, nb = plan.n_copies, plan.n_batches
    return dict(rec=rec.tolist(), batch=batch.tolist(), copies=list(zip(ce[:nc].tolist(), cs[:nc].tolist())),
                n_batches=nb, wait_for=wf[:nb].tolist(), pool_expert=pe.tolist(), pool_last=pl_.tolist())


class Streamer:
    """The library's streaming context (moe_streamer) with the device slot
    buffer and the host copies of the packed routed records it streams from.

    host_records: uint8 tensor of the E packed records in page-locked host
    memory (``packed.cpu().pin_memory()``).  host_miss_records: the miss
    store, the E records packed at ``miss_bits`` (needed when miss_bits is
    not 0 and differs from dims.bits), read for every ring slot.  The slot
    buffer is allocated on the current device: pool_slots records at
    dims.bits, then ring_slots records at the miss width."""

    def __init__(self, dims: MoeDims, pool_slots: int, ring_slots: int, group: int, host_records: torch.Tensor,
                 device=None, host_miss_records: torch.Tensor | None = None, miss_bits: int = 0):
        lib = load_library()
        n = lib.moe_packed_bytes(ctypes.byref(dims), 0)
        if n == 0:
            raise MoeError(-2, "bad dims for a streamer")
        self.cfg = MoeStreamCfg(pool_slots, ring_slots, group, miss_bits)
        self.split = miss_bits not in (0, _code_bits(dims))
        for name, t, bits in (("host_records", host_records, _code_bits(dims)),
                              ("host_miss_records", host_miss_records if self.split else None, miss_bits)):
            if t is None:
                if name == "host_records" or self.split:
                    raise ValueError(f"{name} is required")
                continue
            nb = lib.moe_packed_bytes(ctypes.byref(MoeDims(dims.t, dims.h, dims.inter, dims.E, dims.k,
                                                           dims.shared_inter, bits)), 0)
            _need(t, name, (torch.uint8,), min_numel=nb)
            if t.device.type != "cpu":
                raise ValueError(f"{name} must be a host (CPU) tensor")
        self.dims = MoeDims(*(getattr(dims, f) for f, _ in MoeDims._fields_))
        self.rec_bytes = n // dims.E
        self.miss_rec_bytes = self.rec_bytes
        if self.split:
            self.miss_rec_bytes = lib.moe_packed_bytes(ctypes.byref(MoeDims(
                dims.t, dims.h, dims.inter, dims.E, dims.k, dims.shared_inter, miss_bits)), 0) // dims.E
        self.host_records = host_records
        self.host_miss_records = host_miss_records if self.split else None
        nslot = lib.moe_stream_slot_bytes(ctypes.byref(self.dims), ctypes.byref(self.cfg))
        if nslot == 0:
            raise MoeError(-1, "bad streaming configuration")
        self.slots = torch.empty(nslot, dtype=torch.uint8, device=device or "cuda")
        h = ctypes.c_void_p()
        _check(lib.moe_streamer_create(ctypes.byref(self.dims), ctypes.byref(self.cfg), ctypes.byref(h)))
        self._h = h

    def pool(self) -> list:
        import numpy as np

        out = np.empty(max(self.cfg.pool_slots, 1), np.int32)
        m = load_library().moe_streamer_pool(self._h, out.ctypes.data, self.cfg.pool_slots)
        if m < 0:
            _check(m)
        return out[:m].tolist()

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load_library().moe_streamer_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_forward_streamed(dev: dict, dims: MoeDims, st: Streamer, flags: int = MOE_PACKED_WEIGHTS,
                         ws: torch.Tensor | None = None, out: torch.Tensor | None = None, stream=None,
                         bufs: dict | None = None) -> dict:
    """The whole block through moe_forward_streamed: the routed records come
    from ``st.host_records`` through the streamer's pool and ring; the
    shared record (dev["shared_packed"]) stays on the device.  Returns the
    intermediate tensors and the streaming statistics."""
    lib = load_library()
    flags |= MOE_PACKED_WEIGHTS
    x, wr, rbias = dev["x"], dev["wr"], dev.get("rbias")
    t, h, E, k, Is = dims.t, dims.h, dims.E, dims.k, dims.shared_inter
    _need(x, "x", _BF16, shape=(t, h))
    _need(wr, "wr", _BF16, shape=(E, h))
    if rbias is not None:
        _need(rbias, "rbias", (torch.float32,), shape=(E,))
    shared = None
    if Is > 0:
        sp = dev["shared_packed"]
        _need(sp, "shared_packed", (torch.uint8,), min_numel=lib.moe_packed_bytes(ctypes.byref(dims), 1))
        g = dev.get("shared_gate")
        if g is not None:
            _need(g, "shared gate", _BF16, shape=(h,))
        shared = MoeShared(sp.data_ptr(), None, None, None if g is None else g.data_ptr())
    b = bufs or {}
    d = x.device
    idx, w = b.get("route") or (torch.empty((t, k), dtype=torch.int32, device=d),
                                torch.empty((t, k), dtype=torch.float32, device=d))
    csr = b.get("csr") or Csr(torch.empty(E + 1, dtype=torch.int32, device=d),
                              torch.empty(t * k, dtype=torch.int32, device=d),
                              torch.empty(t * k, dtype=torch.float32, device=d),
                              torch.empty(t * k, dtype=torch.int32, device=d))
    _need(idx, "idx", (torch.int32,), shape=(t, k))
    _need(w, "w", (torch.float32,), shape=(t, k))
    _need_csr(csr, "csr", E, t * k)
    if ws is None:
        ws = new_workspace(dims, flags, d, stream)
    else:
        _need_ws(ws, dims, flags)
    if out is None:
        out = torch.empty((t, h), dtype=torch.bfloat16, device=d)
    else:
        _need(out, "out", _BF16, shape=(t, h))
    _on_current_device(x=x, wr=wr, rbias=rbias, idx=idx, w=w, ws=ws, out=out, slots=st.slots,
                       shared_packed=dev.get("shared_packed") if Is > 0 else None, **_csr_named(csr, "csr"))
    stats = MoeStreamStats()
    c = csr.c()
    miss = st.host_miss_records.data_ptr() if st.host_miss_records is not None else None
    _check(lib.moe_forward_streamed(_ptr(x), _ptr(wr), _ptr(rbias), st.host_records.data_ptr(), miss, _ptr(st.slots),
                                    ctypes.byref(shared) if shared is not None else None, ctypes.byref(dims), flags,
                                    _ptr(idx), _ptr(w), ctypes.byref(c), _ptr(out), _ptr(ws), ws.numel(),
                                    st._h, _stream(stream), ctypes.byref(stats)))
    return dict(idx=idx, w=w, csr=csr, out=out, ws=ws,
                stats=dict(resident=stats.resident, filled=stats.filled, streamed=stats.streamed,
                           batches=stats.batches, bytes=stats.bytes, prefetched=stats.prefetched,
                           prefetch_used=stats.prefetch_used))
