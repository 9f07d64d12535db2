"""Python front of the plain CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()`` and by the
CPU-baseline leg of ``bench.py``; never by the library.  This wrapper only marshals
arguments and calls the C steps in the order the layer defines; all arithmetic is in
``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

F32, F16 = 0, 1
_P = ctypes.c_void_p
_I = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile the oracle: plain C, -O2, no fused contraction, no fast-math, OpenMP."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        subprocess.check_call(["gcc", "-std=gnu11", "-O2", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", SRC, "-o", LIB, "-lm"])
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_half_to_double.restype = ctypes.c_double
        L.oracle_gate_logits.argtypes = [_P, _I, _P, _I, _I, _I, _P]
        L.oracle_gate_logits.restype = None
        L.oracle_softmax_topk.argtypes = [_P, _I, _I, _I, _P, _P, _P]
        L.oracle_softmax_topk.restype = None
        L.oracle_capacity.argtypes = [_I, _I, ctypes.c_double]
        L.oracle_capacity.restype = _I
        L.oracle_dispatch.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P]
        L.oracle_dispatch.restype = _I
        L.oracle_dispatch_shard.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]
        L.oracle_dispatch_shard.restype = _I
        L.oracle_gelu.argtypes = [ctypes.c_double]
        L.oracle_gelu.restype = ctypes.c_double
        L.oracle_expert_ffn.argtypes = [_P, _I, _P, _P, _I, _I, _I, _P]
        L.oracle_expert_ffn.restype = None
        L.oracle_combine_rows.argtypes = [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P,
                                          _I, _P, _I, _P]
        L.oracle_combine_rows.restype = _I
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = _I
        L.oracle_set_num_threads.argtypes = [_I]
        L.oracle_set_num_threads.restype = None
        _lib = L
    return _lib


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float16:
        return F16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"unsupported dtype {a.dtype}")


def _c(a, dtype=None):
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
    return a


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(bits)


def gelu(x: float) -> float:
    return lib().oracle_gelu(float(x))


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Threads of later oracle calls (OpenMP); results do not depend on it."""
    lib().oracle_set_num_threads(int(n))


def gate_logits(x: np.ndarray, Wg: np.ndarray) -> np.ndarray:
    x = _c(x)
    Wg = _c(Wg, np.float32)
    T, d = x.shape
    E = Wg.shape[1]
    out = np.empty((T, E), np.float32)
    lib().oracle_gate_logits(x.ctypes.data, _dt(x), Wg.ctypes.data, T, d, E, out.ctypes.data)
    return out


def softmax_topk(logits: np.ndarray, k: int):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    probs = np.empty((T, E), np.float64)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().oracle_softmax_topk(logits.ctypes.data, T, E, k, probs.ctypes.data, idx.ctypes.data,
                              w.ctypes.data)
    return probs, idx, w


def capacity(T: int, E: int, cf: float) -> int:
    return lib().oracle_capacity(T, E, float(cf))


@dataclass
class Dispatch:
    C: int
    counts_raw: np.ndarray
    kept: np.ndarray
    offsets: np.ndarray
    perm: np.ndarray
    slot_of: np.ndarray

    @property
    def S(self) -> int:
        return int(self.offsets[-1])


def dispatch(topk_idx: np.ndarray, E: int, C: int) -> Dispatch:
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    kept = np.empty(E, np.int32)
    offs = np.empty(E + 1, np.int32)
    perm = np.full(max(1, min(T * k, E * C)), -1, np.int32)
    slot_of = np.empty((T, k), np.int32)
    S = lib().oracle_dispatch(idx.ctypes.data, T, E, k, C, counts.ctypes.data, kept.ctypes.data,
                              offs.ctypes.data, perm.ctypes.data, slot_of.ctypes.data)
    return Dispatch(C, counts, kept, offs, perm[:S].copy(), slot_of)


def shard_bases(counts_per_shard: np.ndarray) -> np.ndarray:
    """base[r, e] = assignments to expert e in shards 0 .. r-1 (shards in token order)."""
    counts = np.asarray(counts_per_shard, np.int64)
    base = np.zeros_like(counts)
    for r in range(1, counts.shape[0]):
        base[r] = base[r - 1] + counts[r - 1]
    return base.astype(np.int32)


def dispatch_shard(topk_idx: np.ndarray, E: int, C: int, base: np.ndarray) -> Dispatch:
    """Dispatch of one shard of a token-sharded batch; C is the whole batch's capacity."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    b = _c(base, np.int32)
    counts = np.empty(E, np.int32)
    kept = np.empty(E, np.int32)
    offs = np.empty(E + 1, np.int32)
    perm = np.full(max(1, T * k), -1, np.int32)
    slot_of = np.empty((T, k), np.int32)
    S = lib().oracle_dispatch_shard(idx.ctypes.data, T, E, k, C, b.ctypes.data, counts.ctypes.data,
                                    kept.ctypes.data, offs.ctypes.data, perm.ctypes.data,
                                    slot_of.ctypes.data)
    return Dispatch(C, counts, kept, offs, perm[:S].copy(), slot_of)


def expert_ffn(x_row: np.ndarray, W1e: np.ndarray, W2e: np.ndarray) -> np.ndarray:
    x_row = _c(x_row)
    W1e = _c(W1e)
    W2e = _c(W2e)
    d, f = W1e.shape
    y = np.empty(d, np.float64)
    lib().oracle_expert_ffn(x_row.ctypes.data, _dt(x_row), W1e.ctypes.data, W2e.ctypes.data,
                            _dt(W1e), d, f, y.ctypes.data)
    return y


@dataclass
class Routing:
    logits: np.ndarray
    probs: np.ndarray
    topk_idx: np.ndarray
    topk_w: np.ndarray
    disp: Dispatch


def route(x: np.ndarray, Wg: np.ndarray, k: int, cf: float, logits_in=None) -> Routing:
    """Steps 1-3: logits (or the given ones), softmax/top-k, capacity, dispatch."""
    T = x.shape[0]
    E = Wg.shape[1]
    logits = gate_logits(x, Wg) if logits_in is None else _c(logits_in, np.float32)
    probs, idx, w = softmax_topk(logits, k)
    C = capacity(T, E, cf)
    return Routing(logits, probs, idx, w, dispatch(idx, E, C))


def combine_rows(x, routing: Routing, W1, W2, Wr1=None, Wr2=None, rows=None) -> np.ndarray:
    """Steps 4-5 for the listed token rows (all rows when None), in double.

    W1 / W2: either full [E,d,f] / [E,f,d] arrays or dicts {expert: [d,f] / [f,d]} holding at
    least the experts the listed rows use.
    """
    x = _c(x)
    T, d = x.shape
    k = routing.topk_idx.shape[1]
    if isinstance(W1, dict):
        E = routing.probs.shape[1]
        keep = []
        w1p = (ctypes.c_void_p * E)()
        w2p = (ctypes.c_void_p * E)()
        for e, a in W1.items():
            a = _c(a)
            b = _c(W2[e])
            keep += [a, b]
            w1p[e] = a.ctypes.data
            w2p[e] = b.ctypes.data
        wdt = _dt(keep[0]) if keep else F16
        f = keep[0].shape[1] if keep else 1
    else:
        W1 = _c(W1)
        W2 = _c(W2)
        E, _, f = W1.shape
        keep = [W1, W2]
        w1p = (ctypes.c_void_p * E)(*[W1.ctypes.data + e * W1[0].nbytes for e in range(E)])
        w2p = (ctypes.c_void_p * E)(*[W2.ctypes.data + e * W2[0].nbytes for e in range(E)])
        wdt = _dt(W1)
    f_res = 0
    if Wr1 is not None:
        Wr1 = _c(Wr1)
        Wr2 = _c(Wr2)
        f_res = Wr1.shape[1]
    if rows is None:
        rows_a = np.arange(T, dtype=np.int32)
    else:
        rows_a = _c(np.asarray(rows), np.int32)
    out = np.empty((rows_a.size, d), np.float64)
    idx = _c(routing.topk_idx, np.int32)
    w = _c(routing.topk_w, np.float64)
    so = _c(routing.disp.slot_of, np.int32)
    rc = lib().oracle_combine_rows(
        x.ctypes.data, _dt(x), T, d, f, k, idx.ctypes.data, w.ctypes.data, so.ctypes.data,
        w1p, w2p, wdt, Wr1.ctypes.data if Wr1 is not None else None,
        Wr2.ctypes.data if Wr2 is not None else None, f_res, rows_a.ctypes.data, rows_a.size,
        out.ctypes.data)
    if rc != 0:
        raise ValueError("combine_rows: a listed row needs an expert whose weights were not given")
    return out


def layer_forward(x, Wg, W1, W2, k, cf, Wr1=None, Wr2=None, logits_in=None, rows=None):
    """The whole layer: returns (out [rows, d] float64, Routing)."""
    r = route(x, Wg, k, cf, logits_in)
    return combine_rows(x, r, W1, W2, Wr1, Wr2, rows), r


def stack_forward(x, layers, k, cf):
    """Layers chained in order (a PR-MoE style stack, DeepSpeed-MoE review, "PR-MoE: Pyramid-
    Residual-MoE"): layer l's output, rounded once to the activation dtype of x, is layer
    l+1's input.  layers: sequence of dicts with Wg, W1, W2 and, for residual layers, Wr1,
    Wr2.  Returns (list of per-layer outputs in float64, list of per-layer inputs, list of
    Routing)."""
    h = _c(x)
    outs, ins, routings = [], [], []
    for L in layers:
        ins.append(h)
        out, r = layer_forward(h, L["Wg"], L["W1"], L["W2"], k, cf, L.get("Wr1"), L.get("Wr2"))
        outs.append(out)
        routings.append(r)
        h = out.astype(x.dtype)
    return outs, ins, routings
