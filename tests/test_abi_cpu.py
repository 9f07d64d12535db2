"""C-ABI library on the CPU: it loads, exports every declared entry point, and its host-side
logic (capacity, workspace sizing, argument checks) behaves as documented.  No call here
reaches the GPU: every call returns before any CUDA work is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from sparse_expert_ffn_layer_gb300 import _build
    _build.build()
    import sparse_expert_ffn_layer_gb300 as m
    return m


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(moe):
    names = declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(moe.lib, n), n
    assert set(names) == set(moe.EXPORTED)


def test_capacity_matches_oracle(moe, oracle_mod):
    import numpy as np
    # the C ABI takes the capacity factor as a binary32 value: the oracle gets that value
    for T in (1, 8, 64, 100, 4096, 16384):
        for E in (1, 4, 64, 128, 1000):
            for cf in (0.5, 1.0, 1.25, 2.0, 3.7):
                assert moe.moe_capacity(T, E, cf) == oracle_mod.capacity(T, E, float(np.float32(cf)))
    assert moe.moe_capacity(0, 8, 1.0) == 0
    for bad in ((-1, 4, 1.0), (4, 0, 1.0), (4, 4, 0.0), (4, 4, -2.0), (4, 4, float("-inf")),
                (4, 4, float("nan"))):
        assert moe.moe_capacity(*bad) == -1
    for T, E in ((1, 4), (4096, 128), (16384, 128)):             # dropless
        assert moe.moe_capacity(T, E, float("inf")) == T == oracle_mod.capacity(T, E, float("inf"))
    # dropless workspace: S_max = T k slots of H
    ws_drop = moe.moe_workspace_size(4096, 1024, 4096, 128, 2, float("inf"), 0, 0, 1)
    ws_cap = moe.moe_workspace_size(4096, 1024, 4096, 128, 2, 1.0, 0, 0, 1)
    assert ws_drop - ws_cap >= (2 * 4096 - 128 * 32) * 4096 * 2


def test_workspace_size(moe):
    ws = moe.moe_workspace_size(4096, 1024, 4096, 128, 1, 1.25, moe.MOE_MLP_STANDARD, 0, moe.MOE_F16)
    C = 40
    h_bytes = min(4096, 128 * C) * 4096 * 2
    assert ws >= h_bytes + 4096 * 128 * 4
    assert ws % 256 == 0
    ws_res = moe.moe_workspace_size(2048, 2048, 8192, 64, 1, 1.0, moe.MOE_MLP_RESIDUAL, 8192,
                                    moe.MOE_F16)
    assert ws_res >= 2048 * 8192 * 2 + 2 * 2048 * 2048 * 4
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(64, 1000, 4096, 8, 1, 1.0, 0, 0, moe.MOE_F16)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(64, 1024, 4096, 8, 3, 1.0, 0, 0, moe.MOE_F16)
    assert ei.value.code == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(64, 1024, 4096, 2048, 1, 1.0, 0, 0, moe.MOE_F16)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(64, 1024, 4096, 8, 1, 1.0, moe.MOE_MLP_RESIDUAL, 0, moe.MOE_F16)
    assert ei.value.code == moe.MOE_ERR_INVALID_ARG


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_argument_errors_return_before_any_launch(moe):
    L = moe.lib
    P = _fake(0x10000)     # never dereferenced: every call below fails its host checks
    s = ctypes.c_void_p(0)
    # gate: bad k, k > E, bad dtype, missing outputs, unaligned pointer
    assert L.moe_gate_topk(P, 1, P, None, 8, 128, 4, 3, P, None, P, P, s) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gate_topk(P, 1, P, None, 8, 128, 1, 2, P, None, P, P, s) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gate_topk(P, 7, P, None, 8, 128, 4, 1, P, None, P, P, s) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gate_topk(P, 1, P, None, 8, 128, 4, 1, P, None, None, P, s) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gate_topk(P, 1, P, None, 8, 128, 4, 1, None, None, P, P, s) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gate_topk(_fake(0x10002), 1, P, None, 8, 128, 4, 1, P, None, P, P, s) == \
        moe.MOE_ERR_UNSUPPORTED
    # empty batch: valid, nothing enqueued
    assert L.moe_gate_topk(P, 1, P, None, 0, 128, 4, 1, P, None, P, P, s) == moe.MOE_OK
    # dispatch
    assert L.moe_dispatch(P, 8, 4, 1, 0.0, P, P, P, P, P, s) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch(P, 8, 4, 1, 1.0, None, P, P, P, P, s) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch(P, 8, 2000, 1, 1.0, P, P, P, P, P, s) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_dispatch(P, 0, 4, 1, 1.0, P, P, P, P, P, s) == moe.MOE_OK
    # sharded dispatch: batch smaller than the shard, rank outside the ranks, counts missing
    assert L.moe_dispatch_sharded(P, 8, 4, 1, 1.0, 4, P, 2, 0, P, P, P, P, P, s) == \
        moe.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch_sharded(P, 8, 4, 1, 1.0, 16, P, 2, 2, P, P, P, P, P, s) == \
        moe.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch_sharded(P, 8, 4, 1, 1.0, 16, None, 2, 1, P, P, P, P, P, s) == \
        moe.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch_sharded(P, 8, 2000, 1, 1.0, 16, P, 2, 1, P, P, P, P, P, s) == \
        moe.MOE_ERR_UNSUPPORTED
    assert L.moe_dispatch_sharded(P, 0, 4, 1, 1.0, 16, P, 2, 1, P, P, P, P, P, s) == moe.MOE_OK
    # expert ffn: unsupported shape, small workspace
    assert L.moe_expert_ffn(P, P, P, P, P, 1, 8, 100, 256, 4, 8, P, P, 1 << 20, s) == \
        moe.MOE_ERR_UNSUPPORTED
    assert L.moe_expert_ffn(P, P, P, P, P, 1, 8, 128, 256, 4, 8, P, P, 1024, s) == \
        moe.MOE_ERR_WORKSPACE
    assert L.moe_expert_ffn(P, P, P, P, P, 1, 8, 128, 256, 4, -1, P, P, 1 << 20, s) == \
        moe.MOE_ERR_INVALID_ARG
    # combine
    assert L.moe_combine(P, P, P, None, 1, 8, 128, 3, P, s) == moe.MOE_ERR_INVALID_ARG
    # layer: residual without weights, bad mlp type, small workspace, bad capacity factor
    lf = L.moe_layer_forward
    assert lf(P, P, P, P, None, None, 1, 8, 128, 256, 4, 1, 1.0, 1, 256, P, None, None, P, 1 << 30, s) \
        == moe.MOE_ERR_INVALID_ARG
    assert lf(P, P, P, P, None, None, 1, 8, 128, 256, 4, 1, 1.0, 5, 0, P, None, None, P, 1 << 30, s) \
        == moe.MOE_ERR_INVALID_ARG
    assert lf(P, P, P, P, None, None, 1, 8, 128, 256, 4, 1, 1.0, 0, 0, P, None, None, P, 64, s) \
        == moe.MOE_ERR_WORKSPACE
    assert lf(P, P, P, P, None, None, 1, 8, 128, 256, 4, 1, -1.0, 0, 0, P, None, None, P, 1 << 30, s) \
        == moe.MOE_ERR_INVALID_ARG
    assert lf(P, P, P, P, P, P, 1, 8, 128, 256, 4, 1, 1.0, 1, 200, P, None, None, P, 1 << 30, s) \
        == moe.MOE_ERR_UNSUPPORTED
    assert lf(P, P, P, P, None, None, 1, 0, 128, 256, 4, 1, 1.0, 0, 0, P, None, None, P, 0, s) \
        == moe.MOE_OK
    # status helpers
    assert L.moe_status_read(None, s) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_wait(P, 0, s) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_status_string(moe.MOE_ERR_TIMEOUT) == "MOE_ERR_TIMEOUT"
    assert moe.moe_status_string(42) == "MOE_ERR_UNKNOWN"
    assert L.moe_set_stage_events(None, 3) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_set_stage_events(None, 0) == moe.MOE_OK
