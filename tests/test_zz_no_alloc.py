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


def test_noalloc_rejects_sizes_beyond_its_scratch():
    m = lib()
    cfg = synth.CONFIGS["moe350m_e128"]
    tok = torch.zeros((8, cfg.d), dtype=torch.float16, device="cuda")
    w1 = torch.zeros((1, cfg.d, cfg.f), dtype=torch.float16, device="cuda")
    w2 = torch.zeros((1, cfg.f, cfg.d), dtype=torch.float16, device="cuda")
    i32 = torch.zeros(16, dtype=torch.int32, device="cuda")
    out = torch.zeros((16, cfg.d), dtype=torch.float16, device="cuda")
    too_many = (64 << 20) // (cfg.f * 2)            # rows of H that no longer fit with the status
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_ffn_noalloc(tok, i32, i32, w1, w2, too_many, out)
    assert ei.value.code == m.MOE_ERR_WORKSPACE
