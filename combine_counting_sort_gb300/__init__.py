"""Python binding of libmoe.so: the single-GPU MoE stage1 + combine path.

Argument marshalling only.  Every step of the path runs in the library's CUDA
kernels; PyTorch supplies device memory and the current stream.  The functions
carry the C entry points' names (include/moe.h) and take torch tensors.  There
is no fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import inputs  # noqa: F401  (seeded generators; no method arithmetic)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_EXPERT_ID, MOE_ERR_TIMEOUT = range(6)
MOE_BLOCK_M = 128
MOE_FLAGS_PER_TILE, MOE_FLAGS_PER_EXPERT = 0, 1
MOE_SCHED_EXPERT_MAJOR, MOE_SCHED_READY_FIRST = 0, 1

EXPORTS = [
    "moe_status_string", "moe_layout_sizes", "moe_route_layout", "moe_dispatch_quant",
    "moe_grouped_gemm1", "moe_combine", "moe_stage1", "moe_router_topk", "moe_quant_weights",
    "moe_dequant_rows", "moe_device_sm_count", "moe_route_layout_noalloc",
    "moe_dispatch_quant_mx", "moe_quant_weights_mx", "moe_grouped_gemm1_mx", "moe_route_layout_noplan",
    "moe_grouped_gemm1_combine", "moe_send_layout", "moe_dispatch_quant_runs", "moe_grouped_gemm1_gather",
    "moe_grouped_gemm1_pair",
]


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


class LayoutSizes(ctypes.Structure):
    _fields_ = [("pairs", ctypes.c_int64), ("max_tiles", ctypes.c_int64), ("rowmap_len", ctypes.c_int64),
                ("layout_ws_bytes", ctypes.c_size_t), ("stage1_ws_bytes", ctypes.c_size_t),
                ("gemm_combine_ws_bytes", ctypes.c_size_t), ("max_send_rows", ctypes.c_int64),
                ("send_ws_bytes", ctypes.c_size_t)]


_TABLES = ["count", "expert_offset", "expert_tile_offset", "group_offset", "ready_tokens", "pair_row",
           "row_pair", "row_weight", "rowmap", "tile_expert", "tile_row_begin", "tile_rows", "num_tiles",
           "token_order"]


class LayoutC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "k", "E", "G", "block_m", "max_tiles")] + \
               [(n, ctypes.c_void_p) for n in _TABLES]


_SEND_TABLES = ["run_offset", "send_token", "send_row", "run_ready", "gather_row"]


class SendRunsC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _SEND_TABLES]


class Stage1Opts(ctypes.Structure):
    _fields_ = [("comm_sms", ctypes.c_int32), ("flags", ctypes.c_int32), ("schedule", ctypes.c_int32),
                ("producers_join", ctypes.c_int32), ("timeout_ns", ctypes.c_int64),
                ("withhold_tile", ctypes.c_int32), ("trace", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i32]
        L.moe_layout_sizes.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(LayoutSizes)]
        L.moe_route_layout.argtypes = [vp, vp, ctypes.POINTER(LayoutC), vp, sz, vp, vp]
        L.moe_dispatch_quant.argtypes = [vp, i32, ctypes.POINTER(LayoutC), vp, vp, vp, vp]
        L.moe_grouped_gemm1.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.POINTER(LayoutC), vp, vp, vp]
        L.moe_grouped_gemm1_pair.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.POINTER(LayoutC), vp, vp, vp]
        L.moe_combine.argtypes = [vp, i32, ctypes.POINTER(LayoutC), vp, vp, vp]
        L.moe_stage1.argtypes = [vp, i32, ctypes.POINTER(LayoutC), vp, vp, i32, ctypes.POINTER(Stage1Opts),
                                 vp, vp, vp, vp, sz, vp, vp]
        L.moe_router_topk.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.moe_quant_weights.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.moe_dequant_rows.argtypes = [vp, vp, i32, ctypes.POINTER(LayoutC), vp, vp]
        L.moe_device_sm_count.argtypes = []
        L.moe_route_layout_noalloc.argtypes = [vp, vp, ctypes.POINTER(LayoutC), vp, vp]
        L.moe_send_layout.argtypes = [vp, ctypes.POINTER(LayoutC), ctypes.POINTER(SendRunsC), vp, sz, vp, vp]
        L.moe_dispatch_quant_runs.argtypes = [vp, i32, ctypes.POINTER(LayoutC), ctypes.POINTER(SendRunsC), vp, vp,
                                              vp, vp]
        L.moe_grouped_gemm1_gather.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.POINTER(LayoutC), vp,
                                               ctypes.c_longlong, vp, vp, vp]
        L.moe_grouped_gemm1_combine.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.POINTER(LayoutC), vp, vp, vp, sz,
                                                vp, vp]
        L.moe_route_layout_noplan.argtypes = [vp, vp, ctypes.POINTER(LayoutC), vp, vp]
        L.moe_dispatch_quant_mx.argtypes = [vp, i32, ctypes.POINTER(LayoutC), vp, vp, vp, vp]
        L.moe_quant_weights_mx.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.moe_grouped_gemm1_mx.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.POINTER(LayoutC), vp, vp, vp]
        for n in EXPORTS:
            if n != "moe_status_string":
                getattr(L, n).restype = i32
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _check(fn: str, rc: int):
    if rc != MOE_OK:
        raise MoEError(fn, rc)


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _shape(t: Optional[torch.Tensor], want, name: str):
    """Refuse a tensor whose shape is not the one the call's sizes imply: the C
    entry points take bare device pointers, so a short buffer would be overrun
    on the device instead of failing here."""
    if t is not None and tuple(t.shape) != tuple(int(v) for v in want):
        raise ValueError(f"{name} must have shape {tuple(int(v) for v in want)}, got {tuple(t.shape)}")


def _status(t: torch.Tensor):
    if t.numel() < 1:
        raise ValueError("status must hold one int32")


def _dims(t: torch.Tensor, n: int, name: str):
    if t.dim() != n:
        raise ValueError(f"{name} must have {n} dimensions, got {t.dim()}")
    return tuple(t.shape)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def moe_layout_sizes(T: int, k: int, E: int, G: int, block_m: int = MOE_BLOCK_M) -> LayoutSizes:
    out = LayoutSizes()
    _check("moe_layout_sizes", lib().moe_layout_sizes(T, k, E, G, block_m, ctypes.byref(out)))
    return out


class Layout:
    """Device tables of one routing layout (torch-allocated) and their C struct."""

    def __init__(self, T: int, k: int, E: int, G: int, device="cuda", block_m: int = MOE_BLOCK_M):
        s = moe_layout_sizes(T, k, E, G, block_m)
        self.T, self.k, self.E, self.G, self.block_m = T, k, E, G, block_m
        self.max_tiles = int(s.max_tiles)
        self.sizes = s
        i32 = dict(dtype=torch.int32, device=device)
        R = T * k
        self.t = {
            "count": torch.empty(E, **i32), "expert_offset": torch.empty(E + 1, **i32),
            "expert_tile_offset": torch.empty(E + 1, **i32), "group_offset": torch.empty(G + 1, **i32),
            "ready_tokens": torch.empty(E, **i32), "pair_row": torch.empty(R, **i32),
            "row_pair": torch.empty(R, **i32), "row_weight": torch.empty(R, dtype=torch.float32, device=device),
            "rowmap": torch.empty(self.max_tiles * block_m, **i32), "tile_expert": torch.empty(self.max_tiles, **i32),
            "tile_row_begin": torch.empty(self.max_tiles, **i32), "tile_rows": torch.empty(self.max_tiles, **i32),
            "num_tiles": torch.empty(1, **i32), "token_order": torch.empty(T, **i32),
        }
        self.ws = torch.empty(int(s.layout_ws_bytes), dtype=torch.uint8, device=device)
        self.c = LayoutC(T, k, E, G, block_m, self.max_tiles, *[self.t[n].data_ptr() for n in _TABLES])

    def __getitem__(self, name):
        return self.t[name]

    def numpy(self) -> dict:
        return {n: v.cpu().numpy() for n, v in self.t.items()}


def moe_route_layout(topk_ids: torch.Tensor, topk_w: torch.Tensor, layout: Layout, status: torch.Tensor,
                     stream=None):
    _shape(topk_ids, (layout.T, layout.k), "topk_ids")
    _shape(topk_w, (layout.T, layout.k), "topk_w")
    _status(status)
    _check("moe_route_layout", lib().moe_route_layout(
        _ptr(topk_ids, torch.int32, "topk_ids"), _ptr(topk_w, torch.float32, "topk_w"), ctypes.byref(layout.c),
        _ptr(layout.ws), layout.ws.numel(), _ptr(status, torch.int32, "status"), _stream(stream)))


def moe_route_layout_noalloc(topk_ids: torch.Tensor, topk_w: torch.Tensor, layout: Layout, status: torch.Tensor,
                             stream=None):
    """moe_route_layout without a workspace: for callers that cannot allocate
    device memory, the scratch is a fixed array inside the library (E <= 256).
    Calls that can overlap on the GPU share that array and must be ordered."""
    _shape(topk_ids, (layout.T, layout.k), "topk_ids")
    _shape(topk_w, (layout.T, layout.k), "topk_w")
    _status(status)
    _check("moe_route_layout_noalloc", lib().moe_route_layout_noalloc(
        _ptr(topk_ids, torch.int32, "topk_ids"), _ptr(topk_w, torch.float32, "topk_w"), ctypes.byref(layout.c),
        _ptr(status, torch.int32, "status"), _stream(stream)))


MOE_NOPLAN_MAX_PAIRS = 16384


def moe_route_layout_noplan(topk_ids: torch.Tensor, topk_w: torch.Tensor, layout: Layout, status: torch.Tensor,
                            stream=None):
    """The small-batch layout without the counting sort (T*k <= 16384): the
    same tables as moe_route_layout except that rows within an expert (and
    tokens within a first-expert group) come in reservation order."""
    _shape(topk_ids, (layout.T, layout.k), "topk_ids")
    _shape(topk_w, (layout.T, layout.k), "topk_w")
    _status(status)
    _check("moe_route_layout_noplan", lib().moe_route_layout_noplan(
        _ptr(topk_ids, torch.int32, "topk_ids"), _ptr(topk_w, torch.float32, "topk_w"), ctypes.byref(layout.c),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def moe_dispatch_quant(x: torch.Tensor, layout: Layout, A: torch.Tensor, A_scale: torch.Tensor,
                       status: torch.Tensor, stream=None):
    T, H = _dims(x, 2, "x")
    R = layout.T * layout.k
    _shape(x, (layout.T, H), "x")
    _shape(A, (R, H), "A")
    _shape(A_scale, (H // 128, R), "A_scale")
    _status(status)
    _check("moe_dispatch_quant", lib().moe_dispatch_quant(
        _ptr(x, torch.bfloat16, "x"), x.shape[1], ctypes.byref(layout.c), _ptr(A, torch.uint8, "A"),
        _ptr(A_scale, torch.float32, "A_scale"), _ptr(status, torch.int32, "status"), _stream(stream)))


def moe_grouped_gemm1(A: torch.Tensor, A_scale: torch.Tensor, W: torch.Tensor, W_scale: torch.Tensor,
                      layout: Layout, Y: torch.Tensor, status: torch.Tensor, stream=None, pair: bool = False):
    """GEMM1 over the layout's M-tiles; pair=True runs it on CTA pairs
    (moe_grouped_gemm1_pair: M = 256 MMAs over two SMs, same Y)."""
    E, N, H = _dims(W, 3, "W")
    R = layout.T * layout.k
    _shape(W, (layout.E, N, H), "W")
    _shape(W_scale, (layout.E, N // 128, H // 128), "W_scale")
    _shape(A, (R, H), "A")
    _shape(A_scale, (H // 128, R), "A_scale")
    _shape(Y, (R, N), "Y")
    _status(status)
    name = "moe_grouped_gemm1_pair" if pair else "moe_grouped_gemm1"
    _check(name, getattr(lib(), name)(
        _ptr(A, torch.uint8, "A"), _ptr(A_scale, torch.float32, "A_scale"), _ptr(W, torch.uint8, "W"),
        _ptr(W_scale, torch.float32, "W_scale"), N, H, ctypes.byref(layout.c), _ptr(Y, torch.bfloat16, "Y"),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def moe_grouped_gemm1_combine(A: torch.Tensor, A_scale: torch.Tensor, W: torch.Tensor, W_scale: torch.Tensor,
                              layout: Layout, Y: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                              status: torch.Tensor, stream=None):
    """GEMM1 and the combine in one launch, each token combined once its k
    expert outputs are stored (ws: layout.sizes.gemm_combine_ws_bytes bytes)."""
    E, N, H = _dims(W, 3, "W")
    R = layout.T * layout.k
    _shape(W, (layout.E, N, H), "W")
    _shape(W_scale, (layout.E, N // 128, H // 128), "W_scale")
    _shape(A, (R, H), "A")
    _shape(A_scale, (H // 128, R), "A_scale")
    _shape(Y, (R, N), "Y")
    _shape(out, (layout.T, N), "out")
    _status(status)
    _check("moe_grouped_gemm1_combine", lib().moe_grouped_gemm1_combine(
        _ptr(A, torch.uint8, "A"), _ptr(A_scale, torch.float32, "A_scale"), _ptr(W, torch.uint8, "W"),
        _ptr(W_scale, torch.float32, "W_scale"), N, H, ctypes.byref(layout.c), _ptr(Y, torch.bfloat16, "Y"),
        _ptr(out, torch.bfloat16, "out"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def gemm_combine_trace(ws: torch.Tensor) -> dict:
    """Trace of the last moe_grouped_gemm1_combine call on workspace ws
    (synchronises): microseconds from the kernel start."""
    v = ws[64:64 + 56].view(torch.int64).cpu().tolist()
    t0 = v[0]
    return {"gemm_first_done_us": (v[1] - t0) / 1e3, "gemm_last_done_us": (v[2] - t0) / 1e3,
            "end_us": (v[3] - t0) / 1e3, "last_push_us": (v[4] - t0) / 1e3,
            "combine_wait_us_total": v[5] / 1e3, "combine_work_us_total": v[6] / 1e3}


def moe_combine(Y: torch.Tensor, layout: Layout, out: torch.Tensor, status: torch.Tensor, stream=None):
    _, D = _dims(Y, 2, "Y")
    _shape(Y, (layout.T * layout.k, D), "Y")
    _shape(out, (layout.T, D), "out")
    _status(status)
    _check("moe_combine", lib().moe_combine(
        _ptr(Y, torch.bfloat16, "Y"), Y.shape[1], ctypes.byref(layout.c), _ptr(out, torch.bfloat16, "out"),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def stage1_opts(comm_sms=0, flags=MOE_FLAGS_PER_TILE, schedule=MOE_SCHED_EXPERT_MAJOR, producers_join=1,
                timeout_ns=0, withhold_tile=-1, trace=0) -> Stage1Opts:
    return Stage1Opts(comm_sms, flags, schedule, producers_join, timeout_ns, withhold_tile, trace)


TRACE_SLOTS = ["start", "produced", "wait_ns", "waited_units", "end", "joined_units", "units"]


def stage1_trace(ws: torch.Tensor) -> dict:
    """Trace slots of a stage1 workspace after a call with trace=1 (synchronises):
    times in microseconds from the kernel start, counters as integers."""
    v = ws[64:64 + 8 * len(TRACE_SLOTS)].view(torch.int64).cpu().tolist()
    d = dict(zip(TRACE_SLOTS, v))
    t0 = d["start"]
    return {"produced_us": (d["produced"] - t0) / 1e3, "end_us": (d["end"] - t0) / 1e3,
            "wait_us_total": d["wait_ns"] / 1e3, "waited_units": d["waited_units"],
            "joined_units": d["joined_units"], "units": d["units"]}


def moe_stage1(x: torch.Tensor, layout: Layout, W: torch.Tensor, W_scale: torch.Tensor, A: torch.Tensor,
               A_scale: torch.Tensor, Y: torch.Tensor, ws: torch.Tensor, status: torch.Tensor,
               opts: Optional[Stage1Opts] = None, stream=None):
    E, N, H = _dims(W, 3, "W")
    R = layout.T * layout.k
    _shape(x, (layout.T, H), "x")
    _shape(W, (layout.E, N, H), "W")
    _shape(W_scale, (layout.E, N // 128, H // 128), "W_scale")
    _shape(A, (R, H), "A")
    _shape(A_scale, (H // 128, R), "A_scale")
    _shape(Y, (R, N), "Y")
    _status(status)
    opts = stage1_opts() if opts is None else opts
    _check("moe_stage1", lib().moe_stage1(
        _ptr(x, torch.bfloat16, "x"), H, ctypes.byref(layout.c), _ptr(W, torch.uint8, "W"),
        _ptr(W_scale, torch.float32, "W_scale"), N, ctypes.byref(opts), _ptr(A, torch.uint8, "A"),
        _ptr(A_scale, torch.float32, "A_scale"), _ptr(Y, torch.bfloat16, "Y"), _ptr(ws, torch.uint8, "ws"),
        ws.numel(), _ptr(status, torch.int32, "status"), _stream(stream)))


def moe_router_topk(logits: torch.Tensor, k: int, topk_ids: torch.Tensor, topk_w: torch.Tensor, stream=None):
    T, E = _dims(logits, 2, "logits")
    _shape(topk_ids, (T, k), "topk_ids")
    _shape(topk_w, (T, k), "topk_w")
    _check("moe_router_topk", lib().moe_router_topk(
        _ptr(logits, torch.float32, "logits"), T, E, k, _ptr(topk_ids, torch.int32, "topk_ids"),
        _ptr(topk_w, torch.float32, "topk_w"), _stream(stream)))


def moe_quant_weights(W: torch.Tensor, Wq: torch.Tensor, W_scale: torch.Tensor, stream=None):
    E, N, H = _dims(W, 3, "W")
    _shape(Wq, (E, N, H), "Wq")
    _shape(W_scale, (E, N // 128, H // 128), "W_scale")
    _check("moe_quant_weights", lib().moe_quant_weights(
        _ptr(W, torch.bfloat16, "W"), E, N, H, _ptr(Wq, torch.uint8, "Wq"),
        _ptr(W_scale, torch.float32, "W_scale"), _stream(stream)))


def moe_dequant_rows(A: torch.Tensor, A_scale: torch.Tensor, layout: Layout, Y: torch.Tensor, stream=None):
    _, H = _dims(A, 2, "A")
    R = layout.T * layout.k
    _shape(A, (R, H), "A")
    _shape(A_scale, (H // 128, R), "A_scale")
    _shape(Y, (R, H), "Y")
    _check("moe_dequant_rows", lib().moe_dequant_rows(
        _ptr(A, torch.uint8, "A"), _ptr(A_scale, torch.float32, "A_scale"), A.shape[1], ctypes.byref(layout.c),
        _ptr(Y, torch.bfloat16, "Y"), _stream(stream)))


def moe_device_sm_count() -> int:
    return int(lib().moe_device_sm_count())


# ---------------------------------------------------------------- MXFP8 variant

def mx_sf_a_shape(layout: Layout, H: int):
    """Shape of the activation scale-factor buffer A_sf: [max_tiles, H/128, 512] bytes."""
    return (layout.max_tiles, H // 128, 512)


def mx_sf_w_shape(E: int, N: int, H: int):
    """Shape of the weight scale-factor buffer W_sf: [E, H/128, N/128, 512] bytes."""
    return (E, H // 128, N // 128, 512)


def moe_dispatch_quant_mx(x: torch.Tensor, layout: Layout, A: torch.Tensor, A_sf: torch.Tensor,
                          status: torch.Tensor, stream=None):
    T, H = _dims(x, 2, "x")
    R = layout.T * layout.k
    _shape(x, (layout.T, H), "x")
    _shape(A, (R, H), "A")
    _shape(A_sf, mx_sf_a_shape(layout, H), "A_sf")
    _status(status)
    _check("moe_dispatch_quant_mx", lib().moe_dispatch_quant_mx(
        _ptr(x, torch.bfloat16, "x"), H, ctypes.byref(layout.c), _ptr(A, torch.uint8, "A"),
        _ptr(A_sf, torch.uint8, "A_sf"), _ptr(status, torch.int32, "status"), _stream(stream)))


def moe_quant_weights_mx(W: torch.Tensor, Wq: torch.Tensor, W_sf: torch.Tensor, stream=None):
    E, N, H = _dims(W, 3, "W")
    _shape(Wq, (E, N, H), "Wq")
    _shape(W_sf, mx_sf_w_shape(E, N, H), "W_sf")
    _check("moe_quant_weights_mx", lib().moe_quant_weights_mx(
        _ptr(W, torch.bfloat16, "W"), E, N, H, _ptr(Wq, torch.uint8, "Wq"), _ptr(W_sf, torch.uint8, "W_sf"),
        _stream(stream)))


def moe_grouped_gemm1_mx(A: torch.Tensor, A_sf: torch.Tensor, W: torch.Tensor, W_sf: torch.Tensor,
                         layout: Layout, Y: torch.Tensor, status: torch.Tensor, stream=None):
    E, N, H = _dims(W, 3, "W")
    R = layout.T * layout.k
    _shape(W, (layout.E, N, H), "W")
    _shape(W_sf, mx_sf_w_shape(layout.E, N, H), "W_sf")
    _shape(A, (R, H), "A")
    _shape(A_sf, mx_sf_a_shape(layout, H), "A_sf")
    _shape(Y, (R, N), "Y")
    _status(status)
    _check("moe_grouped_gemm1_mx", lib().moe_grouped_gemm1_mx(
        _ptr(A, torch.uint8, "A"), _ptr(A_sf, torch.uint8, "A_sf"), _ptr(W, torch.uint8, "W"),
        _ptr(W_sf, torch.uint8, "W_sf"), N, H, ctypes.byref(layout.c), _ptr(Y, torch.bfloat16, "Y"),
        _ptr(status, torch.int32, "status"), _stream(stream)))


# ---------------------------------------------------------------- per-(token, group) send runs

class SendRuns:
    """Device tables of the send runs of one layout (torch-allocated), their C struct and workspace."""

    def __init__(self, layout: Layout, device="cuda"):
        T, k, E, G = layout.T, layout.k, layout.E, layout.G
        s = layout.sizes
        self.max_rows = int(s.max_send_rows)
        i32 = dict(dtype=torch.int32, device=device)
        self.t = {"run_offset": torch.empty(G + 1, **i32), "send_token": torch.empty(self.max_rows, **i32),
                  "send_row": torch.empty(T * G, **i32), "run_ready": torch.empty(E, **i32),
                  "gather_row": torch.empty(T * k, **i32)}
        self.ws = torch.empty(int(s.send_ws_bytes) + 256, dtype=torch.uint8, device=device)
        off = (-self.ws.data_ptr()) % 256            # the workspace must be 256-byte aligned
        self.ws_view = self.ws[off:off + int(s.send_ws_bytes)]
        self.c = SendRunsC(*[self.t[n].data_ptr() for n in _SEND_TABLES])

    def __getitem__(self, name):
        return self.t[name]

    def numpy(self) -> dict:
        return {n: v.cpu().numpy() for n, v in self.t.items()}


def moe_send_layout(topk_ids: torch.Tensor, layout: Layout, runs: SendRuns, status: torch.Tensor, stream=None):
    _shape(topk_ids, (layout.T, layout.k), "topk_ids")
    _status(status)
    _check("moe_send_layout", lib().moe_send_layout(
        _ptr(topk_ids, torch.int32, "topk_ids"), ctypes.byref(layout.c), ctypes.byref(runs.c),
        ctypes.c_void_p(runs.ws_view.data_ptr()), runs.ws_view.numel(), _ptr(status, torch.int32, "status"),
        _stream(stream)))


def moe_dispatch_quant_runs(x: torch.Tensor, layout: Layout, runs: SendRuns, A_send: torch.Tensor,
                            A_send_scale: torch.Tensor, status: torch.Tensor, stream=None):
    T, H = _dims(x, 2, "x")
    _shape(x, (layout.T, H), "x")
    _shape(A_send, (runs.max_rows, H), "A_send")
    _shape(A_send_scale, (H // 128, runs.max_rows), "A_send_scale")
    _status(status)
    _check("moe_dispatch_quant_runs", lib().moe_dispatch_quant_runs(
        _ptr(x, torch.bfloat16, "x"), H, ctypes.byref(layout.c), ctypes.byref(runs.c),
        _ptr(A_send, torch.uint8, "A_send"), _ptr(A_send_scale, torch.float32, "A_send_scale"),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def moe_grouped_gemm1_gather(A_send: torch.Tensor, A_send_scale: torch.Tensor, W: torch.Tensor,
                             W_scale: torch.Tensor, layout: Layout, runs: SendRuns, Y: torch.Tensor,
                             status: torch.Tensor, stream=None):
    E, N, H = _dims(W, 3, "W")
    R = layout.T * layout.k
    _shape(W, (layout.E, N, H), "W")
    _shape(W_scale, (layout.E, N // 128, H // 128), "W_scale")
    _shape(A_send, (runs.max_rows, H), "A_send")
    _shape(A_send_scale, (H // 128, runs.max_rows), "A_send_scale")
    _shape(Y, (R, N), "Y")
    _status(status)
    _check("moe_grouped_gemm1_gather", lib().moe_grouped_gemm1_gather(
        _ptr(A_send, torch.uint8, "A_send"), _ptr(A_send_scale, torch.float32, "A_send_scale"),
        _ptr(W, torch.uint8, "W"), _ptr(W_scale, torch.float32, "W_scale"), N, H, ctypes.byref(layout.c),
        _ptr(runs["gather_row"], torch.int32, "gather_row"), runs.max_rows, _ptr(Y, torch.bfloat16, "Y"),
        _ptr(status, torch.int32, "status"), _stream(stream)))
