"""Python binding of libmoe.so, the GB300 gated Mixture-of-Experts FFN layer (forward).

Argument marshalling only: each function takes torch tensors (device memory owned by the
caller), passes their pointers and the current CUDA stream through the C ABI of
``include/moe.h`` and raises ``MoeError`` on a non-OK status.  Every step of the layer runs in
the library's CUDA kernels; there is no fallback.  The first call fails loudly when
the library has not been built (``python sparse_expert_ffn_layer_gb300/_build.py``).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_BOUNDS = 4, 5, 6
MOE_F32, MOE_F16 = 0, 1
MOE_MLP_STANDARD, MOE_MLP_RESIDUAL = 0, 1

EXPORTED = ("moe_capacity", "moe_workspace_size", "moe_gate_topk", "moe_dispatch",
            "moe_expert_ffn", "moe_combine", "moe_layer_forward", "moe_status_read",
            "moe_status_string", "moe_selftest_wait", "moe_set_stage_events",
            "moe_expert_ffn_noalloc", "moe_dispatch_sharded", "moe_kernel_launches")

_lib = None
MOE_STAGE_EVENTS = 7
STAGES = ("gate_logits", "softmax_topk", "dispatch", "expert_gemm1_gelu", "expert_gemm2_combine",
          "finalize")


def get_lib():
    """Load libmoe.so (once) and declare its signatures; raises if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python sparse_expert_ffn_layer_gb300/_build.py`"
                          " (or __graft_entry__.build())")
    L = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "moe_capacity": ([I, I, F], I),
        "moe_workspace_size": ([I, I, I, I, I, F, I, I, I, ctypes.POINTER(S)], I),
        "moe_gate_topk": ([P, I, P, P, I, I, I, I, P, P, P, P, P], I),
        "moe_dispatch": ([P, I, I, I, F, P, P, P, P, P, P], I),
        "moe_expert_ffn": ([P, P, P, P, P, I, I, I, I, I, I, P, P, S, P], I),
        "moe_combine": ([P, P, P, P, I, I, I, I, P, P], I),
        "moe_layer_forward": ([P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, P, P, P, S, P], I),
        "moe_status_read": ([P, P], I),
        "moe_status_string": ([I], ctypes.c_char_p),
        "moe_selftest_wait": ([P, ctypes.c_uint64, P], I),
        "moe_set_stage_events": ([P, I], I),
        "moe_expert_ffn_noalloc": ([P, P, P, P, P, I, I, I, I, I, I, P, P], I),
        "moe_dispatch_sharded": ([P, I, I, I, F, I, P, I, I, P, P, P, P, P, P], I),
        "moe_kernel_launches": ([], ctypes.c_ulonglong),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def __getattr__(name):
    if name == "lib":
        return get_lib()
    raise AttributeError(name)


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {get_lib().moe_status_string(code).decode()}")


def _check(code: int, where: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return MOE_F16
    if t.dtype == torch.float32:
        return MOE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def moe_kernel_launches() -> int:
    return get_lib().moe_kernel_launches()


def moe_capacity(T: int, E: int, capacity_factor: float) -> int:
    return get_lib().moe_capacity(T, E, capacity_factor)


def moe_workspace_size(T, d, f, E, k, capacity_factor, mlp_type, f_res, dtype) -> int:
    n = ctypes.c_size_t(0)
    _check(get_lib().moe_workspace_size(T, d, f, E, k, capacity_factor, mlp_type, f_res, dtype,
                                  ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_gate_topk(tokens, Wg, k, topk_idx, topk_w, logits_out=None, probs_out=None,
                  logits_in=None, stream=None):
    if logits_in is not None:
        T, E = logits_in.shape
        d = tokens.shape[1] if tokens is not None else 1
        dt = _dtype(tokens) if tokens is not None else MOE_F32
    else:
        T, d = tokens.shape
        E = Wg.shape[1]
        dt = _dtype(tokens)
    _check(get_lib().moe_gate_topk(_ptr(tokens), dt, _ptr(Wg), _ptr(logits_in), T, d, E, k,
                             _ptr(logits_out), _ptr(probs_out), _ptr(topk_idx), _ptr(topk_w),
                             _stream(stream)), "moe_gate_topk")


def moe_dispatch(topk_idx, E, capacity_factor, counts_raw, kept, offsets, perm, slot_of,
                 stream=None):
    T, k = topk_idx.shape
    _check(get_lib().moe_dispatch(_ptr(topk_idx), T, E, k, capacity_factor, _ptr(counts_raw), _ptr(kept),
                            _ptr(offsets), _ptr(perm), _ptr(slot_of), _stream(stream)),
           "moe_dispatch")


def moe_dispatch_sharded(topk_idx, E, capacity_factor, T_global, counts_all, rank, counts_raw, kept,
                         offsets, perm, slot_of, stream=None):
    T, k = topk_idx.shape
    n_ranks = counts_all.shape[0] if counts_all is not None else 1
    _check(get_lib().moe_dispatch_sharded(_ptr(topk_idx), T, E, k, capacity_factor, T_global,
                                          _ptr(counts_all), n_ranks, rank, _ptr(counts_raw),
                                          _ptr(kept), _ptr(offsets), _ptr(perm), _ptr(slot_of),
                                          _stream(stream)), "moe_dispatch_sharded")


def moe_expert_ffn(tokens, perm, offsets, W1, W2, S_max, expert_out, workspace, stream=None):
    T, d = tokens.shape
    E, _, f = W1.shape
    _check(get_lib().moe_expert_ffn(_ptr(tokens), _ptr(perm), _ptr(offsets), _ptr(W1), _ptr(W2),
                              _dtype(tokens), T, d, f, E, S_max, _ptr(expert_out), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_expert_ffn")


def moe_combine(expert_out, slot_of, topk_w, out, residual_in=None, stream=None):
    T, k = slot_of.shape
    d = out.shape[1]
    _check(get_lib().moe_combine(_ptr(expert_out), _ptr(slot_of), _ptr(topk_w), _ptr(residual_in),
                           _dtype(out), T, d, k, _ptr(out), _stream(stream)), "moe_combine")


def moe_layer_forward(tokens, Wg, W1, W2, k, capacity_factor, out, workspace, mlp_type=0,
                      Wr1=None, Wr2=None, topk_idx_out=None, slot_of_out=None, stream=None):
    T, d = tokens.shape
    E, _, f = W1.shape
    f_res = Wr1.shape[1] if Wr1 is not None else 0
    _check(get_lib().moe_layer_forward(_ptr(tokens), _ptr(Wg), _ptr(W1), _ptr(W2), _ptr(Wr1), _ptr(Wr2),
                                 _dtype(tokens), T, d, f, E, k, capacity_factor, mlp_type, f_res,
                                 _ptr(out), _ptr(topk_idx_out), _ptr(slot_of_out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_layer_forward")


def moe_status_read(workspace, stream=None) -> int:
    return get_lib().moe_status_read(_ptr(workspace), _stream(stream))


def moe_status_string(code: int) -> str:
    return get_lib().moe_status_string(code).decode()


def moe_selftest_wait(workspace, timeout_ns: int, stream=None):
    _check(get_lib().moe_selftest_wait(_ptr(workspace), timeout_ns, _stream(stream)), "moe_selftest_wait")


def moe_set_stage_events(events=None):
    """Record the given 7 torch.cuda.Event objects at the stage boundaries of this thread's next
    moe_layer_forward calls (None stops recording)."""
    if events is None:
        _check(get_lib().moe_set_stage_events(None, 0), "moe_set_stage_events")
        return
    handles = [e.cuda_event for e in events]
    if len(handles) != MOE_STAGE_EVENTS or not all(handles):
        raise ValueError("moe_set_stage_events needs 7 created events (record each once first)")
    arr = (ctypes.c_void_p * MOE_STAGE_EVENTS)(*[ctypes.c_void_p(h) for h in handles])
    _check(get_lib().moe_set_stage_events(arr, MOE_STAGE_EVENTS), "moe_set_stage_events")


def moe_expert_ffn_noalloc(tokens, perm, offsets, W1, W2, S_max, expert_out, stream=None):
    """moe_expert_ffn with the library's fixed scratch instead of a workspace (no allocation)."""
    T, d = tokens.shape
    E, _, f = W1.shape
    _check(get_lib().moe_expert_ffn_noalloc(_ptr(tokens), _ptr(perm), _ptr(offsets), _ptr(W1),
                                            _ptr(W2), _dtype(tokens), T, d, f, E, S_max,
                                            _ptr(expert_out), _stream(stream)),
           "moe_expert_ffn_noalloc")
