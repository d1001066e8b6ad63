"""GB300 (sm_103a) MoE expert layer with tile-level overlapped return copy.

Thin ctypes binding of libmoe (C ABI in include/moe.h): argument marshalling only. Every step of
the layer runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and every call
raises if the library cannot be loaded. PyTorch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe.so")

MOE_OK = 0
MOE_ERR_ARG = -1
MOE_ERR_WORKSPACE = -2
MOE_ERR_CUDA = -3
MOE_ERR_TIMEOUT = -4
MOE_ERR_DEVICE = -5
MOE_ERR_PLAN = -6

MOE_PLAN_SKIP_PERMUTE = 0x1
MOE_TAIL_ASSIST = 0x2
MOE_COPY_WARPS = 0x4
MOE_PAIR_UMMA = 0x8
MOE_DIRECT_TAIL = 0x10
MOE_FUSED_DISPATCH = 0x20
MOE_FUSED_GEMMS = 0x40
MOE_PDL = 0x80
MOE_TEST_STALL_CONSUMER = 0x100
MOE_TEST_PLAN_FAIL = 0x200
MOE_ADAPTIVE_CONSUMERS = 0x1000
MOE_TEST_STALL_LAYOUT = 0x2000
MOE_TEST_STALL_PIPE0 = 0x400
MOE_TEST_STALL_PIPE1 = 0x800

TRACE_GEMM2_START, TRACE_GEMM2_END, TRACE_COPY_START, TRACE_COPY_END = 0, 1, 2, 3
TRACE_BAND_DONE, TRACE_LAST_ACQUIRE, TRACE_LAST_LOAD, TRACE_LAST_DRAIN = 4, 5, 6, 7
TRACE_UP_CYCLES, TRACE_UP_NS, TRACE_DOWN_CYCLES, TRACE_DOWN_NS = 8, 9, 10, 11

# names of the C entry points (each declared in include/moe.h)
EXPORTS = ("moe_workspace_size", "moe_workspace_layout", "moe_plan", "moe_forward", "moe_forward_sequential",
           "moe_forward_ex", "moe_forward_host", "moe_forward_host_pipelined", "moe_copy_only", "moe_dma_host_bytes",
           "moe_forward_dma", "moe_status", "moe_device_info", "moe_route_static", "moe_last_error")

# stage events of moe_forward_ex
EV_BEGIN, EV_PLANNED, EV_UP, EV_DOWN, EV_COPIED, EV_END, EV_COUNT = range(7)


class MoEError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"libmoe error {code}: {message}")
        self.code = code


class _Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "d", "ffn", "E", "topk", "R", "tile_M", "consumer_ctas", "mgb")] + [
        ("flags", ctypes.c_uint32), ("timeout_us", ctypes.c_uint32), ("tail_window", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 4)]


_LAYOUT_INTS = ("P_max", "MT_max", "n_chunks", "chunk_tokens", "n_tiles_n2", "block_n2", "rows_per_unit",
                "units_per_band", "PC_max", "IU_max")
LAYOUT_REGIONS = ("idx", "gate", "rank", "chunk_cnt", "chunk_base", "counts", "offsets", "ret_off", "tiles",
                  "tile_ret", "sched", "order", "seg", "experts", "items_up", "items_down", "slot", "cslot", "ret_slot", "yrow",
                  "tile_crow", "band_item", "tok_of", "xrows", "xready", "meta", "flags", "bands", "trace", "Xc", "Hc", "Yp", "Ret", "in_logits", "in_x", "out")


class _Layout(ctypes.Structure):
    _fields_ = [("bytes", ctypes.c_size_t)] + [(n, ctypes.c_int32) for n in _LAYOUT_INTS] + [
        (n, ctypes.c_size_t) for n in LAYOUT_REGIONS]


@dataclasses.dataclass
class Config:
    """Problem and knobs of one MoE layer call (mirrors moe_config)."""

    T: int
    d: int
    ffn: int
    E: int
    topk: int
    R: int
    tile_M: int = 128
    consumer_ctas: int = 8
    mgb: int = 1
    flags: int = 0
    timeout_us: int = 0
    tail_window: int = 0

    def to_c(self) -> _Config:
        c = _Config()
        for f in dataclasses.fields(self):
            setattr(c, f.name, int(getattr(self, f.name)))
        return c

    @classmethod
    def from_workload(cls, w, **kw) -> "Config":
        return cls(T=w.T, d=w.d, ffn=w.ffn, E=w.E, topk=w.topk, R=w.R, tile_M=w.tile_M, **kw)


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmoe; raises if it has not been built for this machine."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe is not built ({LIB_PATH} missing): run tile_level_copy_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int32)
        cfgp = ctypes.POINTER(_Config)
        L.moe_workspace_size.argtypes = [cfgp, ctypes.POINTER(sz)]
        L.moe_workspace_layout.argtypes = [cfgp, ctypes.POINTER(_Layout)]
        L.moe_plan.argtypes = [cfgp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_forward.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_forward_sequential.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_forward_ex.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, sz, ctypes.c_int, ctypes.POINTER(vp), vp]
        L.moe_forward_host.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, sz, ctypes.c_int, vp]
        L.moe_forward_host_pipelined.argtypes = [cfgp, ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, vp,
                                                 vp, ctypes.POINTER(vp), vp, sz, ctypes.c_int, vp]
        L.moe_copy_only.argtypes = [cfgp, vp, sz, ctypes.c_int, vp]
        L.moe_dma_host_bytes.argtypes = [cfgp, ctypes.POINTER(sz)]
        L.moe_forward_dma.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp, sz, ctypes.POINTER(vp), vp]
        L.moe_status.argtypes = [cfgp, vp, vp, i32p]
        L.moe_device_info.argtypes = [i32p, i32p]
        L.moe_route_static.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_last_error.restype = ctypes.c_char_p
        for n in EXPORTS[:-1]:
            getattr(L, n).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != MOE_OK:
        raise MoEError(rc, lib().moe_last_error().decode())


def workspace_size(cfg: Config) -> int:
    n = ctypes.c_size_t()
    c = cfg.to_c()
    _check(lib().moe_workspace_size(ctypes.byref(c), ctypes.byref(n)))
    return n.value


def workspace_layout(cfg: Config) -> dict:
    L = _Layout()
    c = cfg.to_c()
    _check(lib().moe_workspace_layout(ctypes.byref(c), ctypes.byref(L)))
    return {name: getattr(L, name) for name, _ in _Layout._fields_}


def _ptr(t: Optional[torch.Tensor], dtype=None, device=None, name="tensor"):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device == "cuda" and not t.is_cuda:
        raise ValueError(f"{name} must be on the GPU")
    if device == "cpu" and t.is_cuda:
        raise ValueError(f"{name} must be in host memory")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Workspace:
    """Device workspace of one config (a torch uint8 buffer) with typed views of its regions."""

    _DT = {"idx": (torch.int32, "TK"), "gate": (torch.float32, "TK"), "rank": (torch.int32, "TK"),
           "slot": (torch.int32, "TK"), "cslot": (torch.int32, "TK"), "ret_slot": (torch.int32, "TK"),
           "counts": (torch.int32, "ER"), "yrow": (torch.int32, "PC"), "tile_crow": (torch.int32, "MT"),
           "band_item": (torch.int32, "MT"), "tok_of": (torch.int32, "PC"), "xrows": (torch.int32, "E"),
           "xready": (torch.int32, "E"),
           "offsets": (torch.int32, "G1"), "ret_off": (torch.int32, "RE1"), "tiles": (torch.int32, "MT4"),
           "tile_ret": (torch.int32, "MT"), "sched": (torch.int32, "MT"), "order": (torch.int32, "MT"),
           "seg": (torch.int32, "MT2"),
           "experts": (torch.int32, "E8"), "items_up": (torch.int32, "IU2"),
           "items_down": (torch.int32, "MT2"), "meta": (torch.int32, "META"), "flags": (torch.int32, "FL"),
           "bands": (torch.int32, "MT"),
           "trace": (torch.int64, "TR"), "Xc": (torch.bfloat16, "PCd"), "Hc": (torch.bfloat16, "PCF"),
           "Yp": (torch.bfloat16, "Pd"), "Ret": (torch.bfloat16, "TKd")}

    def __init__(self, cfg: Config, device="cuda"):
        self.cfg = cfg
        self.layout = workspace_layout(cfg)
        self.nbytes = self.layout["bytes"]
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)

    def view(self, name: str) -> torch.Tensor:
        c, L = self.cfg, self.layout
        dt, kind = self._DT[name]
        TK = c.T * c.topk
        shape = {"TK": (c.T, c.topk), "ER": (c.E, c.R), "G1": (c.E * c.R + 1,), "RE1": (c.R, c.E + 1),
                 "MT4": (L["MT_max"], 4), "MT": (L["MT_max"],), "MT2": (L["MT_max"], 2), "E8": (c.E, 8),
                 "META": (64,), "FL": (L["MT_max"], L["n_tiles_n2"]), "TR": (16,), "Pd": (L["P_max"], c.d),
                 "PCd": (L["PC_max"], c.d), "PC": (L["PC_max"],), "E": (c.E,), "PCF": (L["PC_max"], c.ffn), "IU2": (L["IU_max"], 2),
                 "TKd": (TK, c.d)}[kind]
        n = 1
        for s in shape:
            n *= s
        esz = torch.empty((), dtype=dt).element_size()
        off = L[name]
        return self.buf[off:off + n * esz].view(dt).view(shape)

    @property
    def ptr(self) -> ctypes.c_void_p:
        return ctypes.c_void_p(self.buf.data_ptr())


def plan(cfg: Config, logits: torch.Tensor, x: Optional[torch.Tensor], ws: Workspace,
         topk_idx: Optional[torch.Tensor] = None, topk_w: Optional[torch.Tensor] = None, stream=None) -> None:
    c = cfg.to_c()
    _check(lib().moe_plan(ctypes.byref(c), _ptr(logits, torch.float32, "cuda", "logits"),
                          _ptr(x, torch.bfloat16, "cuda", "x"), _ptr(topk_idx, torch.int32, "cuda", "topk_idx"),
                          _ptr(topk_w, torch.float32, "cuda", "topk_w"), ws.ptr, ws.nbytes, _stream(stream)))


def forward(cfg: Config, logits: torch.Tensor, x: torch.Tensor, W1: torch.Tensor, W3: torch.Tensor,
            W2: torch.Tensor, out: torch.Tensor, ws: Workspace, sequential: bool = False, stream=None,
            events=None) -> None:
    """moe_forward (tile-level overlapped return copy) or moe_forward_sequential.

    events: optional list of EV_COUNT recorded-once torch.cuda.Event (or None entries); the library
    records them between its launches (moe_forward_ex).
    """
    c = cfg.to_c()
    bf = torch.bfloat16
    args = (ctypes.byref(c), _ptr(logits, torch.float32, "cuda", "logits"), _ptr(x, bf, "cuda", "x"),
            _ptr(W1, bf, "cuda", "W1"), _ptr(W3, bf, "cuda", "W3"), _ptr(W2, bf, "cuda", "W2"),
            _ptr(out, torch.float32, "cuda", "out"), ws.ptr, ws.nbytes)
    if events is None:
        fn = lib().moe_forward_sequential if sequential else lib().moe_forward
        _check(fn(*args, _stream(stream)))
        return
    arr = (ctypes.c_void_p * EV_COUNT)(*[None if e is None else ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib().moe_forward_ex(*args, 1 if sequential else 0, arr, _stream(stream)))


def stage_events(n: int = EV_COUNT):
    """Timing events usable by forward(events=...): created and recorded once so they own a handle."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()
    return evs


def forward_host(cfg: Config, logits_h: torch.Tensor, x_h: torch.Tensor, W1: torch.Tensor, W3: torch.Tensor,
                 W2: torch.Tensor, out_h: torch.Tensor, ws: Workspace, sequential: bool = False, stream=None) -> None:
    """moe_forward_host: host logits / x in, host out; weights on the device."""
    c = cfg.to_c()
    bf = torch.bfloat16
    _check(lib().moe_forward_host(ctypes.byref(c), _ptr(logits_h, torch.float32, "cpu", "logits_h"),
                                  _ptr(x_h, bf, "cpu", "x_h"), _ptr(W1, bf, "cuda", "W1"),
                                  _ptr(W3, bf, "cuda", "W3"), _ptr(W2, bf, "cuda", "W2"),
                                  _ptr(out_h, torch.float32, "cpu", "out_h"), ws.ptr, ws.nbytes,
                                  1 if sequential else 0, _stream(stream)))


def forward_host_pipelined(cfg: Config, logits_h, x_h, W1: torch.Tensor, W3: torch.Tensor, W2: torch.Tensor,
                           out_h, ws: Workspace, sequential: bool = False, stream=None) -> None:
    """moe_forward_host_pipelined: len(out_h) batches, host inputs / outputs given as lists of pinned
    tensors (one per batch), transfers of neighbouring batches overlapped with the layer."""
    c = cfg.to_c()
    bf = torch.bfloat16
    n = len(out_h)
    if len(logits_h) != n or len(x_h) != n:
        raise ValueError("logits_h, x_h and out_h must have one entry per batch")
    arr = ctypes.c_void_p * max(n, 1)
    pl = arr(*[_ptr(t, torch.float32, "cpu", "logits_h") for t in logits_h])
    px = arr(*[_ptr(t, bf, "cpu", "x_h") for t in x_h])
    po = arr(*[_ptr(t, torch.float32, "cpu", "out_h") for t in out_h])
    _check(lib().moe_forward_host_pipelined(ctypes.byref(c), n, pl, px, _ptr(W1, bf, "cuda", "W1"),
                                            _ptr(W3, bf, "cuda", "W3"), _ptr(W2, bf, "cuda", "W2"), po, ws.ptr,
                                            ws.nbytes, 1 if sequential else 0, _stream(stream)))


def dma_host_bytes(cfg: Config) -> int:
    n = ctypes.c_size_t()
    c = cfg.to_c()
    _check(lib().moe_dma_host_bytes(ctypes.byref(c), ctypes.byref(n)))
    return n.value


def forward_dma(cfg: Config, logits: torch.Tensor, x: torch.Tensor, W1: torch.Tensor, W3: torch.Tensor,
                W2: torch.Tensor, out: torch.Tensor, ws: Workspace, host_rec: torch.Tensor, stream=None,
                events=None) -> None:
    """moe_forward_dma: the return copy on the copy engines. host_rec: a pinned host tensor of at least
    dma_host_bytes(cfg) bytes. Blocks until the down-projection has finished on the GPU."""
    c = cfg.to_c()
    bf = torch.bfloat16
    if not host_rec.is_pinned():
        raise ValueError("host_rec must be pinned host memory")
    arr = None if events is None else (ctypes.c_void_p * EV_COUNT)(
        *[None if e is None else ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib().moe_forward_dma(ctypes.byref(c), _ptr(logits, torch.float32, "cuda", "logits"), _ptr(x, bf, "cuda", "x"),
                                 _ptr(W1, bf, "cuda", "W1"), _ptr(W3, bf, "cuda", "W3"), _ptr(W2, bf, "cuda", "W2"),
                                 _ptr(out, torch.float32, "cuda", "out"), ws.ptr, ws.nbytes,
                                 _ptr(host_rec, None, "cpu", "host_rec"), host_rec.numel() * host_rec.element_size(),
                                 arr, _stream(stream)))


def copy_only(cfg: Config, ws: Workspace, ctas: int, stream=None) -> None:
    """moe_copy_only: the return copy of the last forward on ws, alone, on `ctas` SMs."""
    c = cfg.to_c()
    _check(lib().moe_copy_only(ctypes.byref(c), ws.ptr, ws.nbytes, int(ctas), _stream(stream)))


def status(cfg: Config, ws: Optional[Workspace], stream=None):
    """(return code, detail) of the last call on ws (ws None: of the last moe_route_static call on this
    device); synchronises the stream."""
    c = cfg.to_c()
    detail = ctypes.c_int32()
    rc = lib().moe_status(ctypes.byref(c), None if ws is None else ws.ptr, _stream(stream), ctypes.byref(detail))
    return rc, detail.value


def route_static(cfg: Config, logits: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                 slot: torch.Tensor, ret_slot: torch.Tensor, offsets: torch.Tensor, stream=None) -> None:
    """moe_route_static: routing and row layout with the library's own static scratch (no workspace)."""
    c = cfg.to_c()
    i32 = torch.int32
    _check(lib().moe_route_static(ctypes.byref(c), _ptr(logits, torch.float32, "cuda", "logits"),
                                  _ptr(topk_idx, i32, "cuda", "topk_idx"), _ptr(topk_w, torch.float32, "cuda", "topk_w"),
                                  _ptr(slot, i32, "cuda", "slot"), _ptr(ret_slot, i32, "cuda", "ret_slot"),
                                  _ptr(offsets, i32, "cuda", "offsets"), _stream(stream)))


def device_info():
    sms, ok = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().moe_device_info(ctypes.byref(sms), ctypes.byref(ok)))
    return sms.value, bool(ok.value)
