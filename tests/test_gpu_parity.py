"""GPU parity: every stage of the CUDA path, called through the C ABI, against the CPU oracle
on the same seeded inputs.  Routing (logits, experts, counts, slots) must match bit for bit;
layer outputs within max|err| <= 2e-2 max|ref| + 1e-3."""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_cases import Case, lib, sample_rows, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    oracle.build()
    return lib()


def _gate(m, tokens, Wg, k, logits_in=None):
    T = tokens.shape[0] if tokens is not None else logits_in.shape[0]
    E = Wg.shape[1] if Wg is not None else logits_in.shape[1]
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    lo = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    pr = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    m.moe_gate_topk(None if tokens is None else torch.from_numpy(tokens).cuda(),
                    None if Wg is None else torch.from_numpy(Wg).cuda(), k, idx, w, logits_out=lo,
                    probs_out=pr,
                    logits_in=None if logits_in is None else torch.from_numpy(logits_in).cuda())
    torch.cuda.synchronize()
    return lo.cpu().numpy(), pr.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


# ------------------------------------------------------------------------------ gate
# every gate kernel the launcher picks: the lane-per-expert kernel (one and two tokens per
# warp), the 32 x 64 warp tiles of large batches (ragged last tile), the 4 x 4 tiled kernel
# (E not a multiple of 64) and the tiny fp32 layer
@pytest.mark.parametrize("name,T,E", [("tiny_fp32", 128, None), ("moe350m_e128", 1, None),
                                      ("moe350m_e128", 777, None), ("moe1p3b_e128_zipf", 256, None),
                                      ("moe2p4b_e128_top2", 1024, None),
                                      ("moe2p4b_e128_top2_zipf", 333, None),
                                      ("moe350m_e128", 2000, None), ("moe350m_e128", 4100, None),
                                      ("prmoe_e64", 1500, None), ("prmoe_e64", 2500, None),
                                      ("moe2p4b_e128_top2", 16384, None), ("moe350m_e128", 3000, 96),
                                      ("moe350m_e128", 3001, 36)])
def test_gate_bit_exact(m, name, T, E):
    cfg = synth.CONFIGS[name] if E is None else synth.CONFIGS[name].at(E=E)
    inp = synth.host_inputs(cfg, T, seed=3, with_experts=False)
    lo, pr, idx, w = _gate(m, inp["tokens"], inp["Wg"], cfg.k)
    ref_lo = oracle.gate_logits(inp["tokens"], inp["Wg"])
    assert np.array_equal(lo.view(np.uint32), ref_lo.view(np.uint32)), "logits differ in bits"
    probs, ridx, rw = oracle.softmax_topk(ref_lo, cfg.k)
    assert np.array_equal(idx, ridx)
    assert np.allclose(w, rw, rtol=2e-6, atol=1e-7)
    assert np.allclose(pr, probs, rtol=2e-6, atol=1e-8)


@pytest.mark.parametrize("k", [1, 2])
def test_gate_given_logits_with_ties(m, k):
    rng = np.random.default_rng(11)
    T, E = 500, 64
    logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)      # heavy exact ties
    logits[7] = 0.0                                                     # all equal
    logits[8, :] = -np.float32(1e-30)
    logits[8, 40] = np.float32(1e-30)                                   # near tie, one winner
    lo, pr, idx, w = _gate(m, None, None, k, logits_in=logits)
    probs, ridx, rw = oracle.softmax_topk(logits, k)
    assert np.array_equal(lo, logits)
    assert np.array_equal(idx, ridx)
    assert idx[7, 0] == 0 and (k == 1 or idx[7, 1] == 1)
    assert idx[8, 0] == 40
    assert np.allclose(w, rw, rtol=2e-6, atol=1e-7)


# ------------------------------------------------------------------------------ dispatch
def _dispatch(m, idx, E, cf):
    T, k = idx.shape
    C = m.moe_capacity(T, E, cf)
    S_cap = max(1, min(T * k, E * C))
    d_idx = torch.from_numpy(idx.astype(np.int32)).cuda()
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    kept = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    perm = torch.full((S_cap,), -1, dtype=torch.int32, device="cuda")
    slot = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    m.moe_dispatch(d_idx, E, cf, counts, kept, offs, perm, slot)
    torch.cuda.synchronize()
    return C, counts.cpu().numpy(), kept.cpu().numpy(), offs.cpu().numpy(), perm.cpu().numpy(), \
        slot.cpu().numpy()


@pytest.mark.parametrize("T,E,k,cf,skew", [(1, 128, 1, 1.25, 0), (8, 128, 1, 1.25, 0),
                                           (4096, 128, 1, 1.25, 0), (3000, 16, 2, 1.0, 1),
                                           (16384, 128, 2, 1.25, 0), (16384, 128, 2, 1.25, 1),
                                           (999, 1024, 2, 2.0, 1), (777, 3, 1, 0.5, 0),
                                           (513, 1, 1, 1.0, 0), (40000, 64, 1, 1.0, 1)])
def test_dispatch_bit_exact(m, T, E, k, cf, skew):
    rng = np.random.default_rng(T + E + k)
    p = np.ones(E) if not skew else 1.0 / np.arange(1, E + 1) ** 1.2
    p /= p.sum()
    if k == 1:
        idx = rng.choice(E, size=(T, 1), p=p)
    else:
        idx = np.array([rng.choice(E, 2, replace=False, p=p) for _ in range(T)])
    idx = idx.astype(np.int32)
    C, counts, kept, offs, perm, slot = _dispatch(m, idx, E, cf)
    ref = oracle.dispatch(idx, E, oracle.capacity(T, E, float(np.float32(cf))))
    assert C == ref.C
    assert np.array_equal(counts, ref.counts_raw)
    assert np.array_equal(kept, ref.kept)
    assert np.array_equal(offs, ref.offsets)
    assert np.array_equal(perm[:ref.S], ref.perm)
    assert np.all(perm[ref.S:] == -1)                     # entries past S untouched
    assert np.array_equal(slot, ref.slot_of)


def test_dispatch_all_to_one_expert(m):
    T, E = 2048, 8
    idx = np.full((T, 1), 5, np.int32)
    C, counts, kept, offs, perm, slot = _dispatch(m, idx, E, 1.0)
    assert counts[5] == T and kept[5] == C == 256
    assert np.array_equal(perm[:C], np.arange(C))
    assert np.all(slot[C:, 0] == -1) and np.array_equal(slot[:C, 0], np.arange(C))


@pytest.mark.parametrize("T,E,k,cf,cuts", [(4096, 128, 1, 1.25, (0, 1000, 1000, 2500, 4096)),
                                           (16384, 128, 2, 1.25, (0, 8192, 16384)),
                                           (3000, 16, 2, 1.0, (0, 1, 1500, 2999, 3000)),
                                           (999, 1024, 2, 2.0, (0, 333, 999))])
def test_dispatch_sharded_bit_exact(m, T, E, k, cf, cuts):
    """Token-sharded routing: each shard dispatched with the earlier shards' counts keeps
    exactly what the whole batch keeps.  The ranks are emulated one after another on this GPU
    (independent launches that never wait on one another); the counts exchange is a stack of
    the shards' counts_raw."""
    rng = np.random.default_rng(T + E)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    if k == 1:
        idx = rng.choice(E, size=(T, 1), p=p)
    else:
        idx = np.array([rng.choice(E, 2, replace=False, p=p) for _ in range(T)])
    idx = idx.astype(np.int32)
    R = len(cuts) - 1
    shards = [torch.from_numpy(idx[cuts[r]:cuts[r + 1]].copy()).cuda() for r in range(R)]
    counts = []
    for r in range(R):
        Tr = cuts[r + 1] - cuts[r]
        c = torch.zeros(E, dtype=torch.int32, device="cuda")
        if Tr:
            z = lambda n: torch.empty(n, dtype=torch.int32, device="cuda")  # noqa: E731
            m.moe_dispatch(shards[r], E, cf, c, z(E), z(E + 1), z(Tr * k),
                           torch.empty((Tr, k), dtype=torch.int32, device="cuda"))
        counts.append(c)
    counts_all = torch.stack(counts).contiguous()
    C = oracle.capacity(T, E, float(np.float32(cf)))
    whole = oracle.dispatch(idx, E, C)
    bases = oracle.shard_bases(counts_all.cpu().numpy())
    assert np.array_equal(counts_all.cpu().numpy().sum(0), whole.counts_raw)
    for r in range(R):
        lo, hi = cuts[r], cuts[r + 1]
        Tr = hi - lo
        cnt = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        kept = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        offs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
        perm = torch.full((max(1, Tr * k),), -1, dtype=torch.int32, device="cuda")
        slot = torch.full((Tr, k), -9, dtype=torch.int32, device="cuda")
        m.moe_dispatch_sharded(shards[r], E, cf, T, counts_all, r, cnt, kept, offs, perm, slot)
        torch.cuda.synchronize()
        if Tr == 0:
            continue
        ref = oracle.dispatch_shard(idx[lo:hi], E, C, bases[r])
        assert np.array_equal(cnt.cpu().numpy(), ref.counts_raw)
        assert np.array_equal(kept.cpu().numpy(), ref.kept)
        assert np.array_equal(offs.cpu().numpy(), ref.offsets)
        assert np.array_equal(perm.cpu().numpy()[:ref.S], ref.perm)
        assert np.array_equal(slot.cpu().numpy(), ref.slot_of)
        assert np.array_equal(ref.slot_of >= 0, whole.slot_of[lo:hi] >= 0)


# ------------------------------------------------------------------------------ whole layer
# (layer, T, rows): rows None compares every row, an int n compares sample_rows with n
# random rows besides the first / last, dropped and per-expert boundary rows
LAYER_CASES = [
    ("tiny_fp32", 128, None), ("tiny_fp32", 1, None), ("tiny_fp32", 37, None),
    ("moe350m_e128", 1, None), ("moe350m_e128", 8, None), ("moe350m_e128", 64, None),
    ("moe350m_e128", 512, None),
    ("moe1p3b_e128_zipf", 16, None), ("moe1p3b_e128_zipf", 256, None),
    ("prmoe_e64", 64, None), ("prmoe_e128", 64, None),
    ("moe2p4b_e128_top2", 1, None), ("moe2p4b_e128_top2", 32, None),
    ("moe2p4b_e128_top2_zipf", 32, None),
    ("top2_e64", 64, None), ("top2_e128", 2048, 512),
    # decode batches whose slots plus residual rows fit the split-K path (residual group split)
    ("prmoe_e64", 16, None), ("tiny_prmoe_e8", 24, None),
]


@pytest.mark.parametrize("name,T,n_rows", LAYER_CASES)
def test_layer_forward(m, name, T, n_rows):
    cfg = synth.CONFIGS[name]
    case = Case(cfg, T, seed=1)
    out, idx, slot = case.forward(m)
    r = case.routing()
    assert np.array_equal(idx, r.topk_idx)
    assert np.array_equal(slot, r.disp.slot_of)
    rows = np.arange(T, dtype=np.int32) if n_rows is None else sample_rows(r, T, n_rows)
    ref = case.reference_rows(rows)
    ok, err, bound = within_tol(out[rows], ref)
    assert np.isfinite(out).all()
    assert ok, f"max err {err:.3e} > bound {bound:.3e}"
    del case
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,T,cf", [("moe1p3b_e128_zipf", 256, 2.0), ("moe1p3b_e128_zipf", 8192, 1.0),
                                       ("moe1p3b_e128_zipf", 8192, 2.0),
                                       ("prmoe_e128", 2048, 1.0), ("prmoe_e64", 2048, 1.25)])
def test_layer_forward_capacity_and_residual(m, name, T, cf):
    cfg = synth.CONFIGS[name].at(cf=cf)
    case = Case(cfg, T, seed=2)
    out, idx, slot = case.forward(m)
    r = case.routing()
    assert np.array_equal(idx, r.topk_idx) and np.array_equal(slot, r.disp.slot_of)
    rows = sample_rows(r, T)
    ok, err, bound = within_tol(out[rows], case.reference_rows(rows))
    assert ok, f"max err {err:.3e} > bound {bound:.3e}"
    del case
    torch.cuda.empty_cache()


# Output modes that no configured layer reaches, every row: top-2 with the residual MLP (three
# addends per output: fp32 accumulators and the finalize pass), through the split-K decode path
# and the full-size path; the fp32 layer with top-2, with the residual MLP, and with both
# (the CUDA-core path's in-place sums and fp32 accumulators)
@pytest.mark.parametrize("name,T,over", [
    ("prmoe_e64", 16, {"k": 2}), ("prmoe_e64", 200, {"k": 2}),
    ("tiny_fp32", 96, {"k": 2}), ("tiny_fp32", 96, {"residual": True, "f_res": 128}),
    ("tiny_fp32", 96, {"k": 2, "residual": True, "f_res": 192})])
def test_layer_output_modes(m, name, T, over):
    cfg = synth.CONFIGS[name].at(**over)
    case = Case(cfg, T, seed=12)
    out, idx, slot = case.forward(m)
    r = case.routing()
    assert np.array_equal(idx, r.topk_idx) and np.array_equal(slot, r.disp.slot_of)
    rows = np.arange(T, dtype=np.int32)
    ok, err, bound = within_tol(out[rows], case.reference_rows(rows))
    assert ok, f"max err {err:.3e} > bound {bound:.3e}"
    b, _, _ = case.forward(m)
    assert np.array_equal(out.view(np.uint32), b.view(np.uint32))     # deterministic
    del case
    torch.cuda.empty_cache()


def test_layer_350m_every_row(m):
    """350M+MoE-128 layer, T = 4096, top-1, cf 1.25: every row against the oracle."""
    cfg = synth.CONFIGS["moe350m_e128"]
    case = Case(cfg, 4096, seed=0)
    out, idx, slot = case.forward(m)
    r = case.routing()
    assert np.array_equal(idx, r.topk_idx) and np.array_equal(slot, r.disp.slot_of)
    assert np.isfinite(out).all()
    dropped = np.where(slot[:, 0] < 0)[0]
    assert np.all(out[dropped] == 0.0)              # top-1 drops give exact zeros
    rows = np.arange(4096, dtype=np.int32)
    ok, err, bound = within_tol(out[rows], case.reference_rows(rows))
    assert ok, f"max err {err:.3e} > bound {bound:.3e}"


@pytest.mark.parametrize("name,T", [("moe2p4b_e128_top2", 16384), ("moe2p4b_e128_top2", 1024),
                                    ("moe2p4b_e128_top2_zipf", 16384),
                                    ("moe2p4b_e128_top2_zipf", 1024)])
def test_layer_forward_largest(m, name, T):
    """The 2.4B+MoE-128 top-2 layer (26 GB of experts), uniform and Zipf(1.2) routing; the
    uniform T = 16384 batch is the benchmark's workload."""
    cfg = synth.CONFIGS[name]
    case = Case(cfg, T, seed=0)
    out, idx, slot = case.forward(m)
    r = case.routing()
    assert np.array_equal(idx, r.topk_idx) and np.array_equal(slot, r.disp.slot_of)
    assert np.isfinite(out).all()
    rows = sample_rows(r, T)
    ok, err, bound = within_tol(out[rows], case.reference_rows(rows))
    assert ok, f"max err {err:.3e} > bound {bound:.3e}"
    del case
    torch.cuda.empty_cache()


def test_layer_graph_replay_matches_direct_call(m):
    """The benchmark times the layer as a CUDA graph replayed back to back over several token
    batches; at the benchmark's workload (2.4B+MoE-128, top-2, T = 16384) every replay must
    give the direct call's output bit for bit, whatever batch ran before it."""
    cfg = synth.CONFIGS["moe2p4b_e128_top2"]
    T = 16384
    case = Case(cfg, T, seed=0)
    other = torch.from_numpy(synth.fill((T, cfg.d), synth.F16, 0, synth.TID_TOKENS + (1 << 8),
                                        cfg.tok_sigma)).cuda()
    want, _, _ = case.forward(m)
    ws = case.workspace(m)
    outs = [torch.empty((T, cfg.d), dtype=torch.float16, device="cuda") for _ in range(2)]
    srcs = [case.d_tokens, other]
    cap = torch.cuda.Stream()
    graphs = []
    for b in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            m.moe_layer_forward(srcs[b], case.d_Wg, case.d_W1, case.d_W2, cfg.k, cfg.cf, outs[b],
                                ws)
        graphs.append(g)
    for rep in range(3):
        graphs[1].replay()
        graphs[0].replay()
        torch.cuda.synchronize()
        assert m.moe_status_read(ws) == m.MOE_OK
        got = outs[0].float().cpu().numpy()
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), rep
    del case
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,T", [("moe350m_e128", 512), ("moe1p3b_e128_zipf", 2048),
                                    ("moe2p4b_e128_top2_zipf", 16384)])
def test_layer_forward_dropless(m, name, T):
    """Capacity factor +inf: nothing is dropped, and the hot experts' rows (thousands at the
    Zipf(1.2) top-2 shape) spread over as many row tiles as they need."""
    cfg = synth.CONFIGS[name].at(cf=float("inf"))
    case = Case(cfg, T, seed=3)
    out, idx, slot = case.forward(m)
    r = case.routing()
    assert r.disp.C == T and r.disp.S == T * cfg.k
    assert np.all(slot >= 0)
    assert np.array_equal(idx, r.topk_idx) and np.array_equal(slot, r.disp.slot_of)
    hot = int(np.argmax(r.disp.kept))
    hot_tokens = r.disp.perm[r.disp.offsets[hot]:r.disp.offsets[hot + 1]]
    rows = np.unique(np.concatenate([sample_rows(r, T, 128),
                                     hot_tokens[[0, len(hot_tokens) // 2, -1]]])).astype(np.int32)
    ok, err, bound = within_tol(out[rows], case.reference_rows(rows))
    assert ok, f"max err {err:.3e} > bound {bound:.3e}"
    del case
    torch.cuda.empty_cache()


# ------------------------------------------------------------------------------ split path
@pytest.mark.parametrize("name,T", [("tiny_fp32", 128), ("moe350m_e128", 300), ("prmoe_e64", 64),
                                    ("moe2p4b_e128_top2", 8)])
def test_split_stages_match_fused(m, name, T):
    cfg = synth.CONFIGS[name]
    case = Case(cfg, T, seed=4)
    k, E, d = cfg.k, cfg.E, cfg.d
    tdt = case.d_W1.dtype
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    lo = torch.empty((T, E), dtype=torch.float32, device="cuda")
    m.moe_gate_topk(case.d_tokens, case.d_Wg, k, idx, w, logits_out=lo)
    C = m.moe_capacity(T, E, cfg.cf)
    S_max = min(T * k, E * C)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    kept = torch.empty(E, dtype=torch.int32, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(S_max, dtype=torch.int32, device="cuda")
    slot = torch.empty((T, k), dtype=torch.int32, device="cuda")
    m.moe_dispatch(idx, E, cfg.cf, counts, kept, offs, perm, slot)
    eo = torch.empty((S_max, d), dtype=tdt, device="cuda")
    ws = case.workspace(m)
    m.moe_expert_ffn(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max, eo, ws)
    assert m.moe_status_read(ws) == m.MOE_OK
    res = None
    if cfg.residual:
        # the residual MLP through the same entry point: one expert, identity routing
        r_perm = torch.arange(T, dtype=torch.int32, device="cuda")
        r_offs = torch.tensor([0, T], dtype=torch.int32, device="cuda")
        res = torch.empty((T, d), dtype=tdt, device="cuda")
        m.moe_expert_ffn(case.d_tokens, r_perm, r_offs, case.d_Wr1.unsqueeze(0),
                         case.d_Wr2.unsqueeze(0), T, res, ws)
    out = torch.empty((T, d), dtype=tdt, device="cuda")
    m.moe_combine(eo, slot, w, out, residual_in=res)
    torch.cuda.synchronize()
    r = case.routing()
    assert np.array_equal(idx.cpu().numpy(), r.topk_idx)
    assert np.array_equal(perm.cpu().numpy()[:r.disp.S], r.disp.perm)
    ref = case.reference_rows(np.arange(T))
    ok, err, bound = within_tol(out.float().cpu().numpy(), ref)
    assert ok, f"max err {err:.3e} > bound {bound:.3e}"
    fused, _, _ = case.forward(m)
    ok, err, bound = within_tol(fused, out.float().cpu().numpy().astype(np.float64))
    assert ok


# ------------------------------------------------------------------------------ properties
def test_deterministic_repeats(m):
    for name, T in (("moe350m_e128", 512), ("moe2p4b_e128_top2", 64), ("prmoe_e64", 64)):
        case = Case(synth.CONFIGS[name], T, seed=5)
        a, _, _ = case.forward(m)
        b, _, _ = case.forward(m)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), name
        del case
        torch.cuda.empty_cache()


def test_closed_form_zero_gate_and_zero_tokens(m):
    cfg = synth.CONFIGS["moe350m_e128"]
    T = 300
    case = Case(cfg, T, seed=6, Wg=np.zeros((cfg.d, cfg.E), np.float32))
    out, idx, slot = case.forward(m)
    C = m.moe_capacity(T, cfg.E, cfg.cf)
    assert np.all(idx[:, 0] == 0)
    assert np.array_equal(slot[:C, 0], np.arange(C)) and np.all(slot[C:, 0] == -1)
    assert np.all(out[C:] == 0.0)
    w1, w2 = synth.expert_slices(cfg, [0], 6)
    for t in (0, 1, C - 1):
        want = oracle.expert_ffn(case.tokens[t], w1[0], w2[0]) / cfg.E
        ok, err, bound = within_tol(out[t:t + 1], want[None, :])
        assert ok, (t, err, bound)
    zero = Case(cfg, 64, seed=6, tokens=np.zeros((64, cfg.d), np.float16))
    out0, _, _ = zero.forward(m)
    assert np.all(out0 == 0.0)


@pytest.mark.parametrize("k", [1, 2])
def test_layer_routing_with_tied_gate_columns(m, k):
    """Experts whose gate columns are identical tie exactly on every token (the tiled gate's
    fp32 chains give them bit-identical logits): the tie must go to the lower index, as in
    the oracle (top-2: the expert and its duplicate)."""
    cfg = synth.CONFIGS["moe350m_e128"].at(k=k)
    T = 256
    Wg = synth.fill((cfg.d, cfg.E), synth.F32, 7, synth.TID_WG, cfg.w_sigma)
    Wg[:, 64:] = Wg[:, :64]                        # expert e + 64 duplicates expert e
    case = Case(cfg, T, seed=7, Wg=Wg)
    out, idx, slot = case.forward(m)
    r = case.routing()
    assert np.array_equal(idx, r.topk_idx) and np.array_equal(slot, r.disp.slot_of)
    assert np.all(idx[:, 0] < 64)
    if k == 2:
        assert np.array_equal(idx[:, 1], idx[:, 0] + 64)
    rows = np.arange(T, dtype=np.int32)
    ok, err, bound = within_tol(out[rows], case.reference_rows(rows))
    assert ok, f"max err {err:.3e} > bound {bound:.3e}"


@pytest.mark.parametrize("name", ["moe350m_e128", "tiny_fp32"])
def test_expert_ffn_index_checks(m, name):
    """Caller-supplied offsets that run past S_max, or a perm entry outside [0, T): no row at
    or beyond S_max is written, the context stays usable, and the status word reads
    MOE_ERR_DEVICE_BOUNDS; in-range indices read MOE_OK."""
    cfg = synth.CONFIGS[name].at(E=4)
    T = 96
    case = Case(cfg, T, seed=11)
    ws = case.workspace(m)
    perm = torch.arange(T, dtype=torch.int32, device="cuda")
    offs = torch.tensor([0, 24, 48, 72, 96], dtype=torch.int32, device="cuda")
    tdt = case.d_W1.dtype
    ref = torch.zeros((T, cfg.d), dtype=tdt, device="cuda")
    m.moe_expert_ffn(case.d_tokens, perm, offs, case.d_W1, case.d_W2, T, ref, ws)
    assert m.moe_status_read(ws) == m.MOE_OK
    S_max = 40
    got = torch.full((T, cfg.d), 7.0, dtype=tdt, device="cuda")
    m.moe_expert_ffn(case.d_tokens, perm, offs, case.d_W1, case.d_W2, S_max, got, ws)
    assert m.moe_status_read(ws) == m.MOE_ERR_DEVICE_BOUNDS
    assert torch.all(got[S_max:] == 7.0)
    ok, err, bound = within_tol(got[:S_max].float().cpu().numpy(),
                                ref[:S_max].float().cpu().numpy().astype(np.float64))
    assert ok, f"max err {err:.3e} > {bound:.3e}"
    bad = perm.clone()
    bad[5] = T + 1000
    bad[6] = -3
    m.moe_expert_ffn(case.d_tokens, bad, offs, case.d_W1, case.d_W2, T, got, ws)
    assert m.moe_status_read(ws) == m.MOE_ERR_DEVICE_BOUNDS
    assert torch.isfinite(got.float()).all()
    m.moe_expert_ffn(case.d_tokens, perm, offs, case.d_W1, case.d_W2, T, got, ws)
    assert m.moe_status_read(ws) == m.MOE_OK
    assert torch.equal(got, ref)


def test_empty_batch_is_a_no_op(m):
    cfg = synth.CONFIGS["moe350m_e128"]
    case = Case(cfg, 4, seed=0)
    out = torch.zeros((0, cfg.d), dtype=torch.float16, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    m.moe_layer_forward(case.d_tokens[:0], case.d_Wg, case.d_W1, case.d_W2, 1, 1.25, out, ws)
    idx = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    w = torch.zeros((0, 1), dtype=torch.float32, device="cuda")
    m.moe_gate_topk(case.d_tokens[:0], case.d_Wg, 1, idx, w, logits_out=None)
    e = torch.zeros(cfg.E, dtype=torch.int32, device="cuda")
    m.moe_dispatch(idx, cfg.E, 1.25, e, e, torch.zeros(cfg.E + 1, dtype=torch.int32, device="cuda"),
                   idx, idx)
    torch.cuda.synchronize()


def test_bounded_wait_times_out_and_context_survives(m):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    m.moe_selftest_wait(ws, 20_000_000)               # 20 ms; nothing ever arrives
    assert m.moe_status_read(ws) == m.MOE_ERR_TIMEOUT
    case = Case(synth.CONFIGS["tiny_fp32"], 16, seed=0)
    out, _, _ = case.forward(m)                          # the context still works
    assert np.isfinite(out).all()


def test_synth_gpu_draws_match_host():
    t = torch.empty((3, 1000), dtype=torch.float16, device="cuda")
    synth.fill_cuda(t, 7, synth.TID_W1, 0.02, first=12345)
    host = synth.fill((3, 1000), synth.F16, 7, synth.TID_W1, 0.02, first=12345)
    assert np.array_equal(t.cpu().numpy().view(np.uint16), host.view(np.uint16))
    cs = np.linspace(0.5, 2.0, 64)
    g = torch.empty((32, 64), dtype=torch.float32, device="cuda")
    synth.fill_cuda(g, 1, synth.TID_WG, col_scale=cs)
    assert np.array_equal(g.cpu().numpy(), synth.fill((32, 64), synth.F32, 1, synth.TID_WG, col_scale=cs))
