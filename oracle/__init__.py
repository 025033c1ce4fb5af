"""ctypes front end of the FP64 CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE.  Only tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference legs of ``bench.py`` may import this package.  It
shares no code with the CUDA library and the library never imports it.

The arithmetic lives in ``moe_oracle.c``; this module only compiles it
(``build()``), marshals numpy arrays and chains the C steps.  Parity pins:
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes as C
import os
import shutil
import subprocess
import sysconfig
from typing import Callable, Mapping

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so (OpenMP when the compiler has it)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc") or sysconfig.get_config_var("CC")
    base = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB_PATH)
        d, i, p = C.c_double, C.c_int, C.c_void_p
        L.oracle_e2m1_value.restype = d
        L.oracle_e2m1_value.argtypes = [i]
        L.oracle_e8m0_value.restype = d
        L.oracle_e8m0_value.argtypes = [i]
        L.oracle_bf16_value.restype = d
        L.oracle_bf16_value.argtypes = [C.c_uint16]
        L.oracle_bf16_round.restype = C.c_uint16
        L.oracle_bf16_round.argtypes = [d]
        L.oracle_decode_row.restype = None
        L.oracle_decode_row.argtypes = [p, p, i, p]
        L.oracle_route.restype = None
        L.oracle_route.argtypes = [p, p, p, i, i, i, i, i, d, p, p, p, p, p]
        L.oracle_group.restype = i
        L.oracle_group.argtypes = [p, i, i, i, p, p, p, p, p]
        L.oracle_expert_token.restype = None
        L.oracle_expert_token.argtypes = [p, p, p, p, i, i, p, p, p]
        L.oracle_moe_tokens.restype = None
        L.oracle_moe_tokens.argtypes = [p, i, i, i, p, p, p, p, p, p, p, i, p, p, p]
        L.oracle_moe_tokens_act.restype = None
        L.oracle_moe_tokens_act.argtypes = [p, i, i, i, p, p, p, p, p, p, p, i, p, p, p, i]
        L.oracle_e4m3_value.restype = d
        L.oracle_e4m3_value.argtypes = [i]
        L.oracle_e4m3_round.restype = i
        L.oracle_e4m3_round.argtypes = [d]
        L.oracle_mxfp8_quantize.restype = None
        L.oracle_mxfp8_quantize.argtypes = [p, i, p, p, p]
        L.oracle_num_threads.restype = i
        L.oracle_num_threads.argtypes = []
        L.oracle_bf16_round_array.restype = None
        L.oracle_bf16_round_array.argtypes = [p, C.c_size_t, p]
        _lib = L
    return _lib


def num_threads() -> int:
    """Threads the oracle's parallel loops use on this host."""
    return int(lib().oracle_num_threads())


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e8m0_value(s: int) -> float:
    return lib().oracle_e8m0_value(int(s))


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(int(bits))


def bf16_round(v: float) -> int:
    return int(lib().oracle_bf16_round(float(v)))


def bf16_round_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_bf16_round_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(int(code))


def e4m3_round(v: float) -> int:
    return int(lib().oracle_e4m3_round(float(v)))


def mxfp8_quantize(v: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """MXFP8 (OCP MX v1.0) of a vector whose length is a multiple of 32:
    (E4M3 codes, E8M0 scale bytes, dequantised values)."""
    v = np.ascontiguousarray(v, dtype=np.float64).ravel()
    assert v.size % 32 == 0
    codes = np.empty(v.size, dtype=np.uint8)
    scales = np.empty(v.size // 32, dtype=np.uint8)
    deq = np.empty(v.size, dtype=np.float64)
    lib().oracle_mxfp8_quantize(_ptr(v), v.size, _ptr(codes), _ptr(scales), _ptr(deq))
    return codes, scales, deq


def decode_row(codes: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty(K, dtype=np.float64)
    lib().oracle_decode_row(_ptr(codes), _ptr(scales), K, _ptr(out))
    return out


def route(x: np.ndarray, wr: np.ndarray, bias: np.ndarray | None, top_k: int,
          has_shared: int = 1, shared_weight: float = 1.0) -> dict[str, np.ndarray]:
    """Router logits (FP64), top-k, softmax weights and the shared slot."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    wr = np.ascontiguousarray(wr, dtype=np.float32)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    T, H = x.shape
    E = wr.shape[1]
    assert wr.shape[0] == H and 1 <= top_k <= E
    kps = top_k + has_shared
    ids = np.empty((T, kps), dtype=np.int32)
    w = np.empty((T, kps), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    abs_sum = np.empty((T, E), dtype=np.float64)
    gap = np.empty(T, dtype=np.float64)
    lib().oracle_route(_ptr(x), _ptr(wr), _ptr(bias), T, H, E, top_k, has_shared, shared_weight,
                       _ptr(ids), _ptr(w), _ptr(logits), _ptr(abs_sum), _ptr(gap))
    # margin of the ordering relative to the magnitude of the dot products
    scale = abs_sum.max(axis=1) if E else np.ones(T)
    return {"ids": ids, "w": w, "logits": logits, "abs_sum": abs_sum, "gap": gap,
            "rel_gap": gap / np.maximum(scale, 1e-300)}


def group(ids: np.ndarray, n_experts_total: int) -> dict[str, np.ndarray]:
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, kps = ids.shape
    offsets = np.empty(n_experts_total + 1, dtype=np.int32)
    sorted_tok = np.empty(T * kps, dtype=np.int32)
    sorted_slot = np.empty(T * kps, dtype=np.int32)
    active = np.empty(n_experts_total, dtype=np.int32)
    num_active = np.zeros(1, dtype=np.int32)
    rc = lib().oracle_group(_ptr(ids), T, kps, n_experts_total, _ptr(offsets), _ptr(sorted_tok),
                            _ptr(sorted_slot), _ptr(active), _ptr(num_active))
    if rc != 0:
        raise ValueError("expert id out of range")
    na = int(num_active[0])
    return {"offsets": offsets, "sorted_tok": sorted_tok, "sorted_slot": sorted_slot,
            "active": active[:na].copy(), "num_active": na}


def expert_token(expert: Mapping[str, np.ndarray], x_row: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """One expert on one token (x_row as float64 [H]); returns (h [I], Y [H])."""
    w13 = np.ascontiguousarray(expert["w13"])
    I2, Hh = w13.shape
    H, I = 2 * Hh, I2 // 2
    x_row = np.ascontiguousarray(x_row, dtype=np.float64)
    h = np.empty(I, dtype=np.float64)
    y = np.empty(H, dtype=np.float64)
    arrs = [np.ascontiguousarray(expert[k]) for k in ("w13", "s13", "w2", "s2")]
    lib().oracle_expert_token(*[_ptr(a) for a in arrs], H, I, _ptr(x_row), _ptr(h), _ptr(y))
    return h, y


ExpertSource = Callable[[int], Mapping[str, np.ndarray]]


ACTIVATIONS = ("exact", "mxfp8")


def moe_tokens(x: np.ndarray, ids: np.ndarray, w: np.ndarray, experts: ExpertSource,
               tokens=None, want_h: bool = False, want_slots: bool = False,
               act: str = "exact") -> dict[str, np.ndarray]:
    """Expert FFNs + weighted combine for the listed tokens (default: all).

    ``experts(e)`` returns expert e's packed arrays; only experts that the
    listed tokens select are requested.  ``act="mxfp8"``: x and h enter
    their projections MXFP8-quantised (the live-quantisation variant).
    """
    assert act in ACTIVATIONS
    x = np.ascontiguousarray(x, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    T, H = x.shape
    kps = ids.shape[1]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    needed = sorted({int(e) for e in ids[tokens].ravel()})
    n_tot = int(ids.max()) + 1
    held = {e: {k: np.ascontiguousarray(v) for k, v in experts(e).items()} for e in needed}
    I = held[needed[0]]["w13"].shape[0] // 2
    ptrs = {}
    for key in ("w13", "s13", "w2", "s2"):
        arr = (C.c_void_p * n_tot)()
        for e in needed:
            arr[e] = held[e][key].ctypes.data
        ptrs[key] = arr
    n = len(tokens)
    y = np.empty((n, H), dtype=np.float64)
    hs = np.empty((n, kps, I), dtype=np.float64) if want_h else None
    ys = np.empty((n, kps, H), dtype=np.float64) if want_slots else None
    lib().oracle_moe_tokens_act(_ptr(x), H, I, kps, _ptr(ids), _ptr(w), ptrs["w13"], ptrs["s13"],
                                ptrs["w2"], ptrs["s2"], _ptr(tokens), n, _ptr(y), _ptr(hs), _ptr(ys),
                                1 if act == "mxfp8" else 0)
    out = {"y": y, "tokens": tokens}
    if want_h:
        out["h"] = hs
    if want_slots:
        out["y_slots"] = ys
    return out


def layer_forward(x: np.ndarray, wr: np.ndarray, bias: np.ndarray | None, top_k: int,
                  experts: ExpertSource, has_shared: int = 1, shared_weight: float = 1.0,
                  tokens=None, want_h: bool = False, want_slots: bool = False,
                  act: str = "exact") -> dict[str, np.ndarray]:
    """Whole layer: routing for all tokens, FFNs + combine for ``tokens``."""
    r = route(x, wr, bias, top_k, has_shared, shared_weight)
    out = moe_tokens(x, r["ids"], r["w"], experts, tokens, want_h, want_slots, act)
    out.update(r)
    out["y_bf16"] = bf16_round_array(out["y"])
    return out
