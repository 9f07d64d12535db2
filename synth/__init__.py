"""Seeded synthetic inputs for the MoE FFN layer.

This module draws random numbers and designs the gate-weight skew; it holds
none of the layer's arithmetic.  Both the oracle-side tests and the CUDA-side
tests and benchmark take their inputs from here.

Element draw (identical in ``synth_host.c`` and ``synth_cuda.cu``):
SplitMix64 (Vigna) used as a counter-based generator; twelve 24-bit uniforms
per element summed and centred (Irwin-Hall n=12: mean 0, variance 1, exact in
double); one rounded double multiply by the column scale; one rounding to the
storage type.

Tensor ids keep the streams of different tensors apart; token batch b uses
``TID_TOKENS + (b << 8)`` so that distinct batches can be cycled.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .configs import CONFIGS, STACKS, LayerConfig, layer_seed, workload  # noqa: F401

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libsynth_host.so")
CUDA_LIB = os.path.join(HERE, "libsynth_cuda.so")

TID_TOKENS, TID_WG, TID_W1, TID_W2, TID_WR1, TID_WR2, TID_PERM = 1, 2, 3, 4, 5, 6, 7
F32, F16 = 0, 1

_MASK = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15


def splitmix64(x: int) -> int:
    """Vigna's SplitMix64 step on a Python int (the reference for the C versions)."""
    z = (x + _GOLDEN) & _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def stream_key(seed: int, tid: int) -> int:
    return splitmix64(splitmix64(seed) ^ ((tid * _GOLDEN) & _MASK))


def draw_z_py(seed: int, tid: int, i: int) -> float:
    """Pure-Python draw of element i (slow; used to check the C generators)."""
    key = stream_key(seed, tid)
    acc = sum(splitmix64((key + 12 * i + j) & _MASK) >> 40 for j in range(12))
    return (acc - 6 * (1 << 24)) / float(1 << 24)


def build_host(force: bool = False) -> str:
    src = os.path.join(HERE, "synth_host.c")
    if force or not os.path.exists(HOST_LIB) or os.path.getmtime(HOST_LIB) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               src, "-o", HOST_LIB, "-lm"])
    return HOST_LIB


def build_cuda_cmd() -> list[str]:
    src = os.path.join(HERE, "synth_cuda.cu")
    return ["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-Xcompiler", "-fPIC",
            "-shared", src, "-o", CUDA_LIB]


_host = None


def _hostlib():
    global _host
    if _host is None:
        build_host()
        lib = ctypes.CDLL(HOST_LIB)
        lib.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                   ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                   ctypes.c_void_p, ctypes.c_uint64]
        lib.synth_fill.restype = None
        lib.synth_draw_z.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_draw_z.restype = ctypes.c_double
        lib.synth_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_stream_key.restype = ctypes.c_uint64
        lib.synth_double_to_half.argtypes = [ctypes.c_double]
        lib.synth_double_to_half.restype = ctypes.c_uint16
        _host = lib
    return _host


def fill(shape, dtype: int, seed: int, tid: int, sigma: float = 1.0, col_scale=None,
         first: int = 0) -> np.ndarray:
    """Host draw of a row-major tensor (or of a run of it starting at flat index ``first``).

    Returns float32, or float16 for dtype F16.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32 if dtype == F32 else np.float16)
    sc = None
    ncols = 0
    if col_scale is not None:
        sc = np.ascontiguousarray(col_scale, dtype=np.float64)
        ncols = sc.size
    _hostlib().synth_fill(out.ctypes.data, dtype, first, n, seed, tid, float(sigma),
                          sc.ctypes.data if sc is not None else None, ncols)
    return out.reshape(shape)


def draw_unit(n: int, seed: int, tid: int, first: int = 0) -> np.ndarray:
    """The exact unit draws z (float64) of elements first..first+n-1."""
    lib = _hostlib()
    key = lib.synth_stream_key(seed, tid)
    return np.array([lib.synth_draw_z(key, first + q) for q in range(n)], dtype=np.float64)


# ----------------------------------------------------------------------------------------
# Gate-weight skew.  Logits l_e = x . Wg[:, e] of N(0,1) tokens are close to independent
# centred Gaussians with standard deviation ||Wg[:, e]||, so the share of tokens whose
# argmax is e is P_e = int phi(y/s_e)/s_e prod_{e' != e} Phi(y/s_e') dy.  The column norms
# s_e are solved by fixed-point iteration on that integral (trapezoid quadrature) so that
# P matches a Zipf(s) target; no token is routed to design them.
# ----------------------------------------------------------------------------------------

def zipf_targets(E: int, s: float) -> np.ndarray:
    r = np.arange(1, E + 1, dtype=np.float64)
    q = r ** (-s)
    return q / q.sum()


def _argmax_shares(sd: np.ndarray, n_grid: int = 2001) -> np.ndarray:
    from scipy.special import log_ndtr
    lim = 9.0 * sd.max()
    y = np.linspace(-lim, lim, n_grid)
    logphi = log_ndtr(y[None, :] / sd[:, None])               # [E, n]
    total = logphi.sum(axis=0)                                  # [n]
    logdens = -0.5 * (y[None, :] / sd[:, None]) ** 2 - np.log(np.sqrt(2 * np.pi) * sd[:, None])
    integrand = np.exp(logdens + total[None, :] - logphi)
    dy = y[1] - y[0]
    return dy * (integrand.sum(axis=1) - 0.5 * (integrand[:, 0] + integrand[:, -1]))


def zipf_column_norms(E: int, s: float, iters: int = 400, tol: float = 1e-4) -> np.ndarray:
    """Relative column norms (rank order, hottest first) whose argmax shares follow Zipf(s).

    Damped fixed point in log space: log s_e += 0.25 (log q_e - log P_e), then re-centred.
    """
    q = zipf_targets(E, s)
    ls = np.zeros(E)
    for _ in range(iters):
        p = _argmax_shares(np.exp(ls))
        if np.abs(p - q).sum() < tol:
            break
        ls += 0.25 * (np.log(q) - np.log(np.maximum(p, 1e-300)))
        ls -= ls.mean()
    return np.exp(ls)


def seeded_permutation(n: int, seed: int, tid: int = TID_PERM) -> np.ndarray:
    """Fisher-Yates shuffle driven by the SplitMix64 stream (rank -> index map)."""
    perm = list(range(n))
    key = stream_key(seed, tid)
    for i in range(n - 1, 0, -1):
        j = splitmix64((key + i) & _MASK) % (i + 1)
        perm[i], perm[j] = perm[j], perm[i]
    return np.array(perm, dtype=np.int64)


def gate_col_scale(cfg: "LayerConfig", seed: int) -> np.ndarray | None:
    """Per-column scale of Wg[d, E]: None for i.i.d. N(0, sigma_w) (uniform routing)."""
    if cfg.zipf is None:
        return None
    sd_rank = zipf_column_norms(cfg.E, cfg.zipf)
    perm = seeded_permutation(cfg.E, seed)
    sd = np.empty(cfg.E)
    sd[perm] = sd_rank                         # rank r lives at expert perm[r]
    # compensate the realised norms of the unit draws so that ||Wg[:, e]|| ~ sd_e
    z = fill((cfg.d, cfg.E), F32, seed, TID_WG, sigma=1.0).astype(np.float64)
    norms = np.sqrt((z * z).sum(axis=0))
    return cfg.w_sigma * np.sqrt(cfg.d) * sd / norms


def host_inputs(cfg: "LayerConfig", T: int, seed: int = 0, batch: int = 0, with_experts=True):
    """All inputs of one layer call as host arrays (small configurations only).

    Returns a dict with tokens [T,d], Wg [d,E] (float32), W1 [E,d,f], W2 [E,f,d] and, for the
    residual variant, Wr1 [d,f_res], Wr2 [f_res,d]; activations and weights in cfg.dtype.
    """
    dt = F32 if cfg.dtype == "f32" else F16
    out = {"tokens": fill((T, cfg.d), dt, seed, TID_TOKENS + (batch << 8), cfg.tok_sigma)}
    cs = gate_col_scale(cfg, seed)
    out["Wg"] = fill((cfg.d, cfg.E), F32, seed, TID_WG, cfg.w_sigma, col_scale=cs)
    out["gate_col_scale"] = cs
    if with_experts:
        out["W1"] = fill((cfg.E, cfg.d, cfg.f), dt, seed, TID_W1, cfg.w_sigma)
        out["W2"] = fill((cfg.E, cfg.f, cfg.d), dt, seed, TID_W2, cfg.w_sigma)
        if cfg.residual:
            out["Wr1"] = fill((cfg.d, cfg.f_res), dt, seed, TID_WR1, cfg.w_sigma)
            out["Wr2"] = fill((cfg.f_res, cfg.d), dt, seed, TID_WR2, cfg.w_sigma)
    return out


def expert_slices(cfg: "LayerConfig", experts, seed: int = 0):
    """Host draws of W1[e], W2[e] for selected experts only (for sampled checks of big layers)."""
    dt = F32 if cfg.dtype == "f32" else F16
    w1, w2 = {}, {}
    for e in experts:
        e = int(e)
        w1[e] = fill((cfg.d, cfg.f), dt, seed, TID_W1, cfg.w_sigma, first=e * cfg.d * cfg.f)
        w2[e] = fill((cfg.f, cfg.d), dt, seed, TID_W2, cfg.w_sigma, first=e * cfg.f * cfg.d)
    return w1, w2


# ----------------------------------------------------------------------------------------
# GPU draws (same numbers) into torch device tensors.
# ----------------------------------------------------------------------------------------
_cuda = None


def _cudalib():
    global _cuda
    if _cuda is None:
        if not os.path.exists(CUDA_LIB):
            subprocess.check_call(build_cuda_cmd())
        lib = ctypes.CDLL(CUDA_LIB)
        lib.synth_cuda_fill.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                        ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_double, ctypes.c_void_p, ctypes.c_uint64,
                                        ctypes.c_void_p]
        lib.synth_cuda_fill.restype = ctypes.c_int
        _cuda = lib
    return _cuda


def fill_cuda(t, seed: int, tid: int, sigma: float = 1.0, col_scale=None, first: int = 0):
    """Draw into an existing contiguous torch CUDA tensor (float32 or float16)."""
    import torch
    assert t.is_cuda and t.is_contiguous()
    dt = F32 if t.dtype == torch.float32 else F16
    sc = None
    ncols = 0
    if col_scale is not None:
        sc = torch.as_tensor(np.ascontiguousarray(col_scale, dtype=np.float64), device=t.device)
        ncols = sc.numel()
    rc = _cudalib().synth_cuda_fill(t.data_ptr(), dt, first, t.numel(), seed, tid, float(sigma),
                                    sc.data_ptr() if sc is not None else None, ncols,
                                    torch.cuda.current_stream(t.device).cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_cuda_fill failed ({rc})")
    if sc is not None:
        torch.cuda.current_stream(t.device).synchronize()
    return t
