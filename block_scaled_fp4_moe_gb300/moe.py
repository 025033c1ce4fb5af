"""Python binding of libmoe_fp4.so: the C-ABI calls under the same names.

Argument marshalling only: tensors are passed as device pointers, the stream
is torch's current stream unless one is given, and a nonzero status raises
MoEError.  Every computation runs in the library's CUDA kernels; if the
library is not built or cannot be loaded, every call raises.
"""
from __future__ import annotations

import contextlib
import ctypes as C
import dataclasses
import os
import threading

import torch

from . import _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_MISALIGNED = 3
MOE_ERR_WORKSPACE_TOO_SMALL = 4
MOE_ERR_CUDA = 5
MOE_ERR_DEVICE_TIMEOUT = 6
MOE_ERR_DEVICE_ASSERT = 7
MOE_ERR_UNSUPPORTED_DEVICE = 8


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")


class _Bank(C.Structure):
    _fields_ = [("w13", C.c_void_p), ("s13", C.c_void_p), ("w2", C.c_void_p), ("s2", C.c_void_p),
                ("packed", C.c_void_p), ("num_experts", C.c_int32), ("has_shared", C.c_int32),
                ("hidden", C.c_int32), ("inter", C.c_int32)]


_libs: dict[bool, C.CDLL] = {}
_lock = threading.Lock()
_debug = False


def library_path() -> str:
    return _build.DEBUG_LIB_PATH if _debug else _build.LIB_PATH


@contextlib.contextmanager
def debug_bounds():
    """Route the calls below to libmoe_fp4_debug.so, the build with device-side
    range checks (MOE_DEBUG_BOUNDS), for the duration of the block."""
    global _debug
    old, _debug = _debug, True
    try:
        yield lib()
    finally:
        _debug = old


def lib() -> C.CDLL:
    """The loaded CUDA library (the debug build inside debug_bounds()); raises
    if it has not been built."""
    debug = _debug
    if debug not in _libs:
        with _lock:
            if debug not in _libs:
                path = _build.DEBUG_LIB_PATH if debug else _build.LIB_PATH
                if not os.path.exists(path):
                    raise RuntimeError(f"CUDA library {path} is missing: run __graft_entry__.build() "
                                       "(or python -m block_scaled_fp4_moe_gb300._build)")
                L = C.CDLL(path)
                p, i, f, s = C.c_void_p, C.c_int, C.c_float, C.c_size_t
                sig = {
                    "moe_workspace_size": (s, [i, i, i, i, i, i]),
                    "moe_workspace_offset": (s, [i, i, i, i, i, i, C.c_char_p]),
                    "moe_workspace_init": (i, [p, s, p]),
                    "moe_packed_bank_size": (s, [i, i, i, i]),
                    "moe_pack_bank": (i, [C.POINTER(_Bank), p, s, p]),
                    "moe_route_topk": (i, [p, p, p, i, i, i, i, i, f, p, p, p, s, p]),
                    "moe_group_tokens": (i, [p, i, i, i, p, p, p, p, p, p, s, p]),
                    "moe_expert_ffn_mxfp4": (i, [p, p, p, i, i, C.POINTER(_Bank), p, p, s, p]),
                    "moe_layer_forward": (i, [p, p, p, i, i, C.POINTER(_Bank), f, p, p, p, p, s, p]),
                    "moe_layer_forward_hostio": (i, [p, p, p, i, i, C.POINTER(_Bank), f, p, p, s, p]),
                    "moe_layer_forward_noalloc": (i, [p, p, p, i, i, C.POINTER(_Bank), f, p, p, p, p]),
                    "moe_layer_forward_next": (i, [p, p, p, i, i, C.POINTER(_Bank), f, p, p, p, p, s, p,
                                                   C.POINTER(_Bank), p]),
                    "moe_layer_forward_mxfp8": (i, [p, p, p, i, i, C.POINTER(_Bank), p, f, p, p, p, p, s, p]),
                    "moe_layer_forward_mxfp8_profiled": (i, [p, p, p, i, i, C.POINTER(_Bank), p, f, p, p, s, p, i,
                                                             p]),
                    "moe_packed_mx_bank_size": (s, [i, i, i, i]),
                    "moe_pack_bank_mx": (i, [C.POINTER(_Bank), p, s, p]),
                    "moe_layer_forward_profiled": (i, [p, p, p, i, i, C.POINTER(_Bank), f, p, p, s, p, i, p]),
                    "moe_check_device_status": (i, [p, p]),
                    "moe_layer_launches": (i, [i, i, i, i, i, i]),
                    "moe_read_phase_times": (i, [p, p, i, p]),
                    "moe_selftest_wait_timeout": (i, [p, s, p]),
                    "moe_selftest_decode_e2m1": (i, [p, p, i, p]),
                    "moe_status_string": (C.c_char_p, [i]),
                }
                for name, (res, args) in sig.items():
                    fn = getattr(L, name)
                    fn.restype = res
                    fn.argtypes = args
                _libs[debug] = L
    return _libs[debug]


def exported_symbols() -> list[str]:
    return ["moe_workspace_size", "moe_workspace_offset", "moe_workspace_init", "moe_packed_bank_size", "moe_pack_bank", "moe_packed_mx_bank_size", "moe_pack_bank_mx", "moe_route_topk", "moe_group_tokens", "moe_expert_ffn_mxfp4",
            "moe_layer_forward", "moe_layer_forward_hostio", "moe_layer_forward_mxfp8", "moe_layer_forward_mxfp8_profiled",
            "moe_layer_forward_next",
            "moe_layer_forward_noalloc", "moe_layer_forward_profiled",
            "moe_layer_launches", "moe_read_phase_times", "moe_check_device_status", "moe_selftest_decode_e2m1", "moe_selftest_wait_timeout",
            "moe_status_string"]


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoEError(status, where)


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor | None, dtype=None, name: str = "") -> C.c_void_p | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    return C.c_void_p(t.data_ptr())


@dataclasses.dataclass
class MXFP4Bank:
    """Device-resident MXFP4 expert bank (expert E is the shared expert).

    ``packed`` is the repacked copy the expert-FFN kernels read; the canonical
    arrays (w13 [E+S, 2I, H/2], s13 [E+S, 2I, H/32], w2 [E+S, H, I/2],
    s2 [E+S, H, I/32]) are only needed to build it and may be dropped.
    """
    num_experts: int
    has_shared: int
    hidden: int
    inter: int
    packed: torch.Tensor | None = None
    w13: torch.Tensor | None = None
    s13: torch.Tensor | None = None
    w2: torch.Tensor | None = None
    s2: torch.Tensor | None = None
    packed_mx: torch.Tensor | None = None     # the MXFP8 variant's bank (canonical arrays, aligned sections)

    def c_struct(self) -> _Bank:
        ptrs = []
        for name in ("w13", "s13", "w2", "s2", "packed"):
            t = getattr(self, name)
            ptrs.append(None if t is None else _ptr(t, torch.uint8, name).value)
        return _Bank(*ptrs, self.num_experts, self.has_shared, self.hidden, self.inter)

    def pack(self, stream=None) -> "MXFP4Bank":
        """Fill ``packed`` from the canonical arrays (moe_pack_bank)."""
        n = moe_packed_bank_size(self.hidden, self.inter, self.num_experts, self.has_shared)
        if self.packed is None or self.packed.numel() < n:
            self.packed = torch.empty(n, dtype=torch.uint8, device=self.w13.device)
        b = self.c_struct()
        _check(lib().moe_pack_bank(C.byref(b), _ptr(self.packed, torch.uint8, "packed"), self.packed.numel(),
                                   _stream(stream)), "moe_pack_bank")
        return self

    def pack_mx(self, stream=None) -> "MXFP4Bank":
        """Fill ``packed_mx`` from the canonical arrays (moe_pack_bank_mx)."""
        n = int(lib().moe_packed_mx_bank_size(self.hidden, self.inter, self.num_experts, self.has_shared))
        if n == 0:
            raise MoEError(MOE_ERR_UNSUPPORTED_SHAPE, "moe_packed_mx_bank_size")
        if self.packed_mx is None or self.packed_mx.numel() < n:
            self.packed_mx = torch.empty(n, dtype=torch.uint8, device=self.w13.device)
        b = self.c_struct()
        _check(lib().moe_pack_bank_mx(C.byref(b), _ptr(self.packed_mx, torch.uint8, "packed_mx"),
                                      self.packed_mx.numel(), _stream(stream)), "moe_pack_bank_mx")
        return self

    def drop_canonical(self) -> "MXFP4Bank":
        self.w13 = self.s13 = self.w2 = self.s2 = None
        return self

    def clone_packed(self) -> "MXFP4Bank":
        mx = None if self.packed_mx is None else self.packed_mx.clone()
        return MXFP4Bank(self.num_experts, self.has_shared, self.hidden, self.inter, packed=self.packed.clone(),
                         packed_mx=mx)

    @staticmethod
    def from_host(arrays: dict, num_experts: int, has_shared: int, device="cuda",
                  keep_canonical: bool = False, with_mx: bool = False) -> "MXFP4Bank":
        t = {k: torch.from_numpy(arrays[k]).to(device) for k in ("w13", "s13", "w2", "s2")}
        hidden = t["w2"].shape[1]
        inter = t["w13"].shape[1] // 2
        bank = MXFP4Bank(num_experts, has_shared, hidden, inter, **t)
        with torch.cuda.device(t["w13"].device):
            bank.pack()
            if with_mx:
                bank.pack_mx()
        if not keep_canonical:
            torch.cuda.current_stream(t["w13"].device).synchronize()
            bank.drop_canonical()
        return bank


def moe_packed_bank_size(H: int, I: int, E: int, has_shared: int) -> int:
    return int(lib().moe_packed_bank_size(H, I, E, has_shared))


def moe_workspace_offset(T: int, H: int, I: int, E: int, top_k: int, has_shared: int, region: str) -> int:
    off = int(lib().moe_workspace_offset(T, H, I, E, top_k, has_shared, region.encode()))
    if off == (1 << 64) - 1:
        raise KeyError(region)
    return off


def moe_workspace_size(T: int, H: int, I: int, E: int, top_k: int, has_shared: int) -> int:
    return int(lib().moe_workspace_size(T, H, I, E, top_k, has_shared))


def moe_workspace_init(ws, stream=None) -> None:
    _check(lib().moe_workspace_init(_ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "moe_workspace_init")


def alloc_workspace(T: int, bank: MXFP4Bank, top_k: int, device="cuda") -> torch.Tensor:
    """Device workspace for T tokens, header initialised."""
    n = moe_workspace_size(T, bank.hidden, bank.inter, bank.num_experts, top_k, bank.has_shared)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    with torch.cuda.device(ws.device):
        moe_workspace_init(ws)
    return ws


def moe_route_topk(x, router_w, logit_bias, top_k, has_shared, shared_weight, topk_ids, topk_w, ws, stream=None):
    T, H = x.shape
    E = router_w.shape[1]
    _check(lib().moe_route_topk(_ptr(x, torch.bfloat16, "x"), _ptr(router_w, torch.float32, "router_w"),
                                _ptr(logit_bias, torch.float32, "logit_bias"), T, H, E, top_k, has_shared,
                                float(shared_weight), _ptr(topk_ids, torch.int32, "topk_ids"),
                                _ptr(topk_w, torch.float32, "topk_w"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                _stream(stream)), "moe_route_topk")


def moe_group_tokens(topk_ids, n_experts_total, expert_offsets, sorted_tok, sorted_slot, active_experts,
                     num_active, ws, stream=None):
    T, kps = topk_ids.shape
    i32 = torch.int32
    _check(lib().moe_group_tokens(_ptr(topk_ids, i32, "topk_ids"), T, kps, n_experts_total,
                                  _ptr(expert_offsets, i32, "expert_offsets"), _ptr(sorted_tok, i32, "sorted_tok"),
                                  _ptr(sorted_slot, i32, "sorted_slot"), _ptr(active_experts, i32, "active"),
                                  _ptr(num_active, i32, "num_active"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                  _stream(stream)), "moe_group_tokens")


def moe_expert_ffn_mxfp4(x, topk_ids, topk_w, top_k, bank: MXFP4Bank, y, ws, stream=None):
    T = x.shape[0]
    b = bank.c_struct()
    _check(lib().moe_expert_ffn_mxfp4(_ptr(x, torch.bfloat16, "x"), _ptr(topk_ids, torch.int32, "topk_ids"),
                                      _ptr(topk_w, torch.float32, "topk_w"), T, top_k, C.byref(b),
                                      _ptr(y, torch.bfloat16, "y"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                      _stream(stream)), "moe_expert_ffn_mxfp4")


def moe_layer_forward(x, router_w, logit_bias, top_k, bank: MXFP4Bank, shared_weight, y, topk_ids_out=None,
                      topk_w_out=None, ws=None, stream=None):
    T = x.shape[0]
    b = bank.c_struct()
    _check(lib().moe_layer_forward(_ptr(x, torch.bfloat16, "x"), _ptr(router_w, torch.float32, "router_w"),
                                   _ptr(logit_bias, torch.float32, "logit_bias"), T, top_k, C.byref(b),
                                   float(shared_weight), _ptr(y, torch.bfloat16, "y"),
                                   _ptr(topk_ids_out, torch.int32, "topk_ids_out"),
                                   _ptr(topk_w_out, torch.float32, "topk_w_out"), _ptr(ws, torch.uint8, "ws"),
                                   ws.numel(), _stream(stream)), "moe_layer_forward")


def moe_layer_forward_next(x, router_w, logit_bias, top_k, bank: MXFP4Bank, shared_weight, y, topk_ids_out=None,
                           topk_w_out=None, ws=None, next_router_w=None, next_bank: "MXFP4Bank | None" = None,
                           stream=None):
    """moe_layer_forward plus the next layer's router weights and bank as an L2 prefetch hint."""
    T = x.shape[0]
    b = bank.c_struct()
    nb = next_bank.c_struct() if next_bank is not None else None
    _check(lib().moe_layer_forward_next(_ptr(x, torch.bfloat16, "x"), _ptr(router_w, torch.float32, "router_w"),
                                        _ptr(logit_bias, torch.float32, "logit_bias"), T, top_k, C.byref(b),
                                        float(shared_weight), _ptr(y, torch.bfloat16, "y"),
                                        _ptr(topk_ids_out, torch.int32, "topk_ids_out"),
                                        _ptr(topk_w_out, torch.float32, "topk_w_out"), _ptr(ws, torch.uint8, "ws"),
                                        ws.numel(), _ptr(next_router_w, torch.float32, "next_router_w"),
                                        C.byref(nb) if nb is not None else None, _stream(stream)),
           "moe_layer_forward_next")


def moe_layer_forward_mxfp8(x, router_w, logit_bias, top_k, bank: MXFP4Bank, shared_weight, y, topk_ids_out=None,
                            topk_w_out=None, ws=None, stream=None):
    """The MXFP8 live-activation-quantisation variant (needs ``bank.packed_mx``: from_host(with_mx=True))."""
    T = x.shape[0]
    b = bank.c_struct()
    _check(lib().moe_layer_forward_mxfp8(_ptr(x, torch.bfloat16, "x"), _ptr(router_w, torch.float32, "router_w"),
                                         _ptr(logit_bias, torch.float32, "logit_bias"), T, top_k, C.byref(b),
                                         _ptr(bank.packed_mx, torch.uint8, "packed_mx"), float(shared_weight), _ptr(y, torch.bfloat16, "y"),
                                         _ptr(topk_ids_out, torch.int32, "topk_ids_out"),
                                         _ptr(topk_w_out, torch.float32, "topk_w_out"), _ptr(ws, torch.uint8, "ws"),
                                         ws.numel(), _stream(stream)), "moe_layer_forward_mxfp8")


def moe_layer_forward_noalloc(x, router_w, logit_bias, top_k, bank: MXFP4Bank, shared_weight, y, topk_ids_out=None,
                              topk_w_out=None, stream=None):
    """The whole layer on the library's built-in scratch (no workspace argument)."""
    T = x.shape[0]
    b = bank.c_struct()
    _check(lib().moe_layer_forward_noalloc(_ptr(x, torch.bfloat16, "x"), _ptr(router_w, torch.float32, "router_w"),
                                           _ptr(logit_bias, torch.float32, "logit_bias"), T, top_k, C.byref(b),
                                           float(shared_weight), _ptr(y, torch.bfloat16, "y"),
                                           _ptr(topk_ids_out, torch.int32, "topk_ids_out"),
                                           _ptr(topk_w_out, torch.float32, "topk_w_out"), _stream(stream)),
           "moe_layer_forward_noalloc")


def moe_layer_forward_profiled(x, router_w, logit_bias, top_k, bank: MXFP4Bank, shared_weight, y, ws, events,
                               stream=None):
    T = x.shape[0]
    b = bank.c_struct()
    ev = (C.c_void_p * 5)(*[e.cuda_event for e in events])
    _check(lib().moe_layer_forward_profiled(_ptr(x, torch.bfloat16, "x"), _ptr(router_w, torch.float32, "router_w"),
                                            _ptr(logit_bias, torch.float32, "logit_bias"), T, top_k, C.byref(b),
                                            float(shared_weight), _ptr(y, torch.bfloat16, "y"),
                                            _ptr(ws, torch.uint8, "ws"), ws.numel(), ev, 5, _stream(stream)),
           "moe_layer_forward_profiled")


def moe_layer_forward_mxfp8_profiled(x, router_w, logit_bias, top_k, bank: MXFP4Bank, shared_weight, y, ws, events,
                                     stream=None):
    T = x.shape[0]
    b = bank.c_struct()
    ev = (C.c_void_p * 5)(*[e.cuda_event for e in events])
    _check(lib().moe_layer_forward_mxfp8_profiled(_ptr(x, torch.bfloat16, "x"),
                                                  _ptr(router_w, torch.float32, "router_w"),
                                                  _ptr(logit_bias, torch.float32, "logit_bias"), T, top_k,
                                                  C.byref(b), _ptr(bank.packed_mx, torch.uint8, "packed_mx"),
                                                  float(shared_weight), _ptr(y, torch.bfloat16, "y"),
                                                  _ptr(ws, torch.uint8, "ws"), ws.numel(), ev, 5, _stream(stream)),
           "moe_layer_forward_mxfp8_profiled")


def moe_layer_forward_hostio(x_host, router_w, logit_bias, top_k, bank: MXFP4Bank, shared_weight, y_host, ws,
                             stream=None):
    """x_host / y_host: CPU bf16 tensors (pinned for asynchronous copies)."""
    for name, t in (("x_host", x_host), ("y_host", y_host)):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{name}: expected a contiguous CPU bf16 tensor")
    T = x_host.shape[0]
    b = bank.c_struct()
    _check(lib().moe_layer_forward_hostio(C.c_void_p(x_host.data_ptr()), _ptr(router_w, torch.float32, "router_w"),
                                          _ptr(logit_bias, torch.float32, "logit_bias"), T, top_k, C.byref(b),
                                          float(shared_weight), C.c_void_p(y_host.data_ptr()),
                                          _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)),
           "moe_layer_forward_hostio")


def moe_layer_launches(T, bank: MXFP4Bank, top_k) -> int:
    """Kernel launches one moe_layer_forward call makes (1: single launch)."""
    return int(lib().moe_layer_launches(T, bank.hidden, bank.inter, bank.num_experts, top_k, bank.has_shared))


PHASE_NAMES = ("router", "wait1", "route", "gateup", "wait2", "down_combine", "tail", "total")


def moe_read_phase_times(ws, stream=None) -> dict:
    """Phase durations (us) of the last single-launch call on `ws`."""
    out = (C.c_float * 8)()
    _check(lib().moe_read_phase_times(_ptr(ws, torch.uint8, "ws"), C.cast(out, C.c_void_p), 8, _stream(stream)),
           "moe_read_phase_times")
    return dict(zip(PHASE_NAMES, [float(v) for v in out]))


def moe_check_device_status(ws, stream=None) -> int:
    return int(lib().moe_check_device_status(_ptr(ws, torch.uint8, "ws"), _stream(stream)))


def moe_selftest_wait_timeout(ws, stream=None) -> None:
    _check(lib().moe_selftest_wait_timeout(_ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_selftest_decode_e2m1(codes, out, stream=None) -> None:
    _check(lib().moe_selftest_decode_e2m1(_ptr(codes, torch.uint8, "codes"), _ptr(out, torch.int16, "out"),
                                          codes.numel(), _stream(stream)), "moe_selftest_decode_e2m1")
