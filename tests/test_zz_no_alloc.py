"""The allocation-free expert FFN (moe_expert_ffn_noalloc), through the C ABI.

It serves callers that cannot allocate device memory where they run the layer (a plugin
inside a framework that owns all device memory, a serving loop that forbids cudaMalloc after
start-up); its scratch is a fixed array inside the library.  Its results must equal those of
moe_expert_ffn with a caller workspace, call after call, although every call reuses the same
scratch.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
from moe_cases import Case, lib, within_tol

pytestmark = pytest.mark.gpu


def _dispatched(m, case):
    cfg, T = case.cfg, case.T
    idx = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.k), dtype=torch.float32, device="cuda")
    lo = torch.empty((T, cfg.E), dtype=torch.float32, device="cuda")
    m.moe_gate_topk(case.d_tokens, case.d_Wg, cfg.k, idx, w, logits_out=lo)
    C = m.moe_capacity(T, cfg.E, cfg.cf)
    S_max = min(T * cfg.k, cfg.E * C)
    z = lambda n: torch.empty(n, dtype=torch.int32, device="cuda")  # noqa: E731
    counts, kept, offs, perm = z(cfg.E), z(cfg.E), z(cfg.E + 1), z(S_max)
    slot = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    m.moe_dispatch(idx, cfg.E, cfg.cf, counts, kept, offs, perm, slot)
    return perm, offs, S_max


def test_noalloc_matches_workspace_variant_on_consecutive_calls():
    m = lib()
    # three calls in a row on the shared scratch: the second is smaller than the first, so a
    # stale tail of the first call's hidden activations must not leak into it
    for name, T, seed in (("moe350m_e128", 512, 1), ("moe350m_e128", 64, 2), ("tiny_fp32", 128, 3)):
        case = Case(synth.CONFIGS[name], T, seed=seed)
        perm, offs, S_max = _dispatched(m, case)
        d = case.cfg.d
        ref = torch.zeros((S_max, d), dtype=case.d_W1.dtype, device="cuda")
        m.moe_expert_ffn(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max, ref,
                         case.workspace(m))
        got = torch.full((S_max, d), float("nan"), dtype=case.d_W1.dtype, device="cuda")
        m.moe_expert_ffn_noalloc(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max, got)
        torch.cuda.synchronize()
        S = int(offs[-1].item())
        r = ref[:S].float().cpu().numpy().astype(np.float64)
        g = got[:S].float().cpu().numpy()
        ok, err, bound = within_tol(g, r)
        assert ok, f"{name} T={T}: max err {err:.3e} > {bound:.3e}"
        assert np.array_equal(g, r), "same kernels on the same inputs should agree exactly"
        del case
        torch.cuda.empty_cache()


def _at_the_limit_case(E=8):
    """350M+MoE-128 expert shape (d 1024, f 4096) with S_max rows of H filling the 64 MiB
    scratch exactly: every token in one slot, E equal expert groups."""
    cfg = synth.CONFIGS["moe350m_e128"].at(E=E)
    S_max = (64 << 20) // (cfg.f * 2)
    case = Case(cfg, S_max, seed=9)
    perm = torch.arange(S_max, dtype=torch.int32, device="cuda")
    offs = torch.arange(0, S_max + 1, S_max // E, dtype=torch.int32, device="cuda")
    return case, perm, offs, S_max


def test_noalloc_at_its_limit_and_rejects_beyond():
    m = lib()
    case, perm, offs, S_max = _at_the_limit_case()
    d = case.cfg.d
    ref = torch.zeros((S_max, d), dtype=torch.float16, device="cuda")
    m.moe_expert_ffn(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max, ref, case.workspace(m))
    got = torch.full((S_max, d), float("nan"), dtype=torch.float16, device="cuda")
    m.moe_expert_ffn_noalloc(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max, got)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    # one row more than the scratch holds: rejected before anything runs
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_ffn_noalloc(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max + 1, got)
    assert ei.value.code == m.MOE_ERR_WORKSPACE


def test_noalloc_allocates_no_device_memory():
    """The device's free memory (cudaMemGetInfo, which also sees allocations outside torch's
    allocator) is the same before and after a run of calls; one call first so that lazily
    loaded kernels and the scratch array are resident before the first reading."""
    m = lib()
    case, perm, offs, S_max = _at_the_limit_case()
    out = torch.empty((S_max, case.cfg.d), dtype=torch.float16, device="cuda")
    m.moe_expert_ffn_noalloc(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max, out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        m.moe_expert_ffn_noalloc(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_never_writes_rows_beyond_s_max():
    """offsets that run past S_max: the rows below S_max are computed, none at or beyond it is
    written (the output buffer's tail keeps its sentinel), and the shared scratch is not
    overrun (a following in-range call still matches the workspace variant)."""
    m = lib()
    cfg = synth.CONFIGS["moe350m_e128"].at(E=4)
    T = 96
    case = Case(cfg, T, seed=10)
    perm = torch.arange(T, dtype=torch.int32, device="cuda")
    offs = torch.tensor([0, 24, 48, 72, 96], dtype=torch.int32, device="cuda")
    S_max = 40                                      # offsets[E] = 96 > S_max
    got = torch.full((T, cfg.d), 7.0, dtype=torch.float16, device="cuda")
    m.moe_expert_ffn_noalloc(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max, got)
    ref = torch.zeros((T, cfg.d), dtype=torch.float16, device="cuda")
    m.moe_expert_ffn(case.d_tokens, perm, offs, case.d_W1, case.d_W2, T, ref, case.workspace(m))
    torch.cuda.synchronize()
    assert torch.all(got[S_max:] == 7.0)
    ok, err, bound = within_tol(got[:S_max].float().cpu().numpy(),
                                ref[:S_max].float().cpu().numpy().astype(np.float64))
    assert ok, f"max err {err:.3e} > {bound:.3e}"
    again = torch.zeros((T, cfg.d), dtype=torch.float16, device="cuda")
    m.moe_expert_ffn_noalloc(case.d_tokens, perm, offs, case.d_W1, case.d_W2, T, again)
    torch.cuda.synchronize()
    assert torch.equal(again, ref)
