"""Pins of the CPU oracle against things other than itself (CPU only).

Each test checks one part of the oracle against exact arithmetic, a brute force of a
different shape, a closed form, an identity, or a library routine, chosen so that a
plausible slip (a dropped term, a wrong sign or index, a transposed operand, a changed
summation order or tie rule) fails at least one of them.
"""
from fractions import Fraction
import itertools
import math

import numpy as np
import pytest

import synth


# ---------------------------------------------------------------- exact fp32 replay helpers
def f32_round(q: Fraction) -> float:
    """Round an exact rational to the nearest binary32 value, ties to even (no double step)."""
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                       # subnormal spacing below 2^-126
    ulp = Fraction(2) ** (e - 23)
    n = a / ulp
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = float(fl * ulp)
    assert abs(v) < 3.5e38
    return sign * float(np.float32(v))


def fma_chain(xrow, wcol) -> float:
    acc = Fraction(0)
    accf = 0.0
    for xi, wi in zip(xrow, wcol):
        accf = f32_round(Fraction(float(np.float32(xi))) * Fraction(float(wi)) + acc)
        acc = Fraction(accf)
    return accf


# ---------------------------------------------------------------- half conversion
def test_half_to_double_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zero kept
    assert math.copysign(1.0, oracle_mod.half_to_double(0x8000)) == -1.0


# ---------------------------------------------------------------- gate logits: the fp32 FMA chain
def test_gate_chain_exact_replay_random(oracle_mod):
    rng = np.random.default_rng(1)
    for dtype in (np.float16, np.float32):
        T, d, E = 3, 37, 5
        x = (rng.standard_normal((T, d)) * 3).astype(dtype)
        Wg = (rng.standard_normal((d, E)) * 0.02).astype(np.float32)
        got = oracle_mod.gate_logits(x, Wg)
        for t in range(T):
            for e in range(E):
                assert got[t, e] == np.float32(fma_chain(x[t], Wg[:, e])), (dtype, t, e)


def test_gate_chain_order_and_fusion_matter(oracle_mod):
    # ascending order: 2^24 (+1 lost to ties-to-even) - 2^24 = 0; descending order gives 1
    x = np.array([[1.0, 1.0, -1.0]], np.float32)
    Wg = np.array([[2.0 ** 24], [1.0], [2.0 ** 24]], np.float32)
    assert oracle_mod.gate_logits(x, Wg)[0, 0] == 0.0
    # fused: -1 + (1+2^-12)^2 keeps the 2^-24 term that a rounded product would drop
    x = np.array([[-1.0, 1.0 + 2.0 ** -12]], np.float32)
    Wg = np.array([[1.0], [1.0 + 2.0 ** -12]], np.float32)
    assert oracle_mod.gate_logits(x, Wg)[0, 0] == np.float32(2.0 ** -11 + 2.0 ** -24)


def test_gate_logits_error_bound(oracle_mod):
    # |fp32 chain - exact| <= gamma_d * sum |x w| (standard dot-product bound)
    rng = np.random.default_rng(2)
    T, d, E = 4, 512, 6
    x = rng.standard_normal((T, d)).astype(np.float16)
    Wg = (rng.standard_normal((d, E)) * 0.02).astype(np.float32)
    got = oracle_mod.gate_logits(x, Wg).astype(np.float64)
    ex = x.astype(np.float64) @ Wg.astype(np.float64)
    bound = (d * 2.0 ** -24 / (1 - d * 2.0 ** -24)) * (np.abs(x.astype(np.float64)) @ np.abs(Wg))
    assert np.all(np.abs(got - ex) <= bound)


# ---------------------------------------------------------------- softmax / top-k
def _topk_bruteforce(logits, k):
    T, E = logits.shape
    idx = np.empty((T, k), np.int64)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))  # logit desc, index asc
        idx[t] = order[:k]
    return idx


@pytest.mark.parametrize("k", [1, 2])
def test_topk_ties_and_weights(oracle_mod, k):
    rng = np.random.default_rng(3)
    T, E = 64, 8
    logits = rng.integers(-3, 4, size=(T, E)).astype(np.float32)   # many exact ties
    probs, idx, w = oracle_mod.softmax_topk(logits, k)
    assert np.array_equal(idx, _topk_bruteforce(logits, k))
    l64 = logits.astype(np.float64)
    p_ref = np.exp(l64 - l64.max(1, keepdims=True))
    p_ref /= p_ref.sum(1, keepdims=True)
    assert np.allclose(probs, p_ref, rtol=1e-14, atol=0)
    assert np.all(np.abs(probs.sum(1) - 1.0) <= E * 2.0 ** -52)
    if k == 1:
        assert np.allclose(w[:, 0], p_ref[np.arange(T), idx[:, 0]], rtol=1e-14)
    else:
        assert np.allclose(w.sum(1), 1.0, rtol=0, atol=4e-16)
        l1 = logits[np.arange(T), idx[:, 0]].astype(np.float64)
        l2 = logits[np.arange(T), idx[:, 1]].astype(np.float64)
        assert np.allclose(w[:, 0], 1.0 / (1.0 + np.exp(l2 - l1)), rtol=1e-14)
        assert np.all(idx[:, 0] != idx[:, 1])


# ---------------------------------------------------------------- capacity
def test_capacity_closed_form(oracle_mod):
    for T in (1, 7, 8, 64, 513, 4096, 16384):
        for E in (1, 4, 64, 128):
            for cf in (0.5, 1.0, 1.25, 2.0):
                q = Fraction(cf) * T / E
                assert oracle_mod.capacity(T, E, cf) == math.ceil(q)
    assert oracle_mod.capacity(4096, 128, 1.25) == 40
    assert oracle_mod.capacity(16384, 128, 1.25) == 160
    for bad in ((0, 4, 1.0), (4, 0, 1.0), (4, 4, 0.0), (4, 4, -1.0), (4, 4, float("-inf")),
                (4, 4, float("nan"))):
        assert oracle_mod.capacity(*bad) == -1
    # dropless (cf = +inf): C = T, so every assignment is kept however skewed the routing
    for T, E in ((1, 4), (7, 3), (4096, 128)):
        assert oracle_mod.capacity(T, E, float("inf")) == T
    rng = np.random.default_rng(8)
    for k in (1, 2):
        T, E = 500, 6
        idx = np.array([rng.choice(E, k, replace=False, p=[.7, .1, .1, .05, .03, .02])
                        for _ in range(T)], np.int32)
        dsp = oracle_mod.dispatch(idx, E, oracle_mod.capacity(T, E, float("inf")))
        assert np.all(dsp.slot_of >= 0) and dsp.S == T * k
        assert np.array_equal(dsp.kept, dsp.counts_raw)


# ---------------------------------------------------------------- dispatch
def _dispatch_bruteforce(idx, E, C):
    """Stable sort of the token-major assignment list by expert; rank = position in the run."""
    T, k = idx.shape
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E)
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    rank = np.empty_like(flat)
    for pos, a in enumerate(order):
        rank[a] = pos - starts[flat[a]]
    kept = np.minimum(counts, C)
    offs = np.concatenate([[0], np.cumsum(kept)])
    slot = np.where(rank < C, offs[flat] + rank, -1)
    perm = np.full(offs[-1], -1)
    for a in range(flat.size):
        if slot[a] >= 0:
            perm[slot[a]] = a // k
    return counts, kept, offs, perm, slot.reshape(T, k)


def _check_dispatch(oracle_mod, idx, E, C):
    got = oracle_mod.dispatch(idx, E, C)
    counts, kept, offs, perm, slot = _dispatch_bruteforce(idx, E, C)
    assert np.array_equal(got.counts_raw, counts)
    assert np.array_equal(got.kept, kept)
    assert np.array_equal(got.offsets, offs)
    assert np.array_equal(got.perm, perm)
    assert np.array_equal(got.slot_of, slot)
    return got


def test_dispatch_exhaustive_top1(oracle_mod):
    for T in range(1, 7):
        for E in (1, 2, 3):
            for cf in (0.5, 1.0, 1.25, 2.0):
                C = oracle_mod.capacity(T, E, cf)
                for combo in itertools.product(range(E), repeat=T):
                    _check_dispatch(oracle_mod, np.array(combo, np.int32).reshape(T, 1), E, C)


def test_dispatch_random_top2(oracle_mod):
    rng = np.random.default_rng(4)
    for _ in range(300):
        T = int(rng.integers(1, 9))
        E = int(rng.integers(2, 5))
        idx = np.array([rng.choice(E, 2, replace=False) for _ in range(T)], np.int32)
        cf = float(rng.choice([0.5, 1.0, 1.25, 2.0]))
        _check_dispatch(oracle_mod, idx, E, oracle_mod.capacity(T, E, cf))


def test_dispatch_invariants(oracle_mod):
    rng = np.random.default_rng(5)
    for k in (1, 2):
        T, E = 777, 16
        logits = rng.standard_normal((T, E)).astype(np.float32)
        logits[:, 3] += 1.5                                          # a hot expert
        _, idx, w = oracle_mod.softmax_topk(logits, k)
        C = oracle_mod.capacity(T, E, 1.25)
        dsp = oracle_mod.dispatch(idx, E, C)
        assert dsp.counts_raw.sum() == T * k
        assert np.all(dsp.kept <= C) and np.all(dsp.kept == np.minimum(dsp.counts_raw, C))
        assert dsp.S == dsp.kept.sum() == (dsp.slot_of >= 0).sum()
        for e in range(E):
            seg = dsp.perm[dsp.offsets[e]:dsp.offsets[e + 1]]
            assert np.all(np.diff(seg) > 0)                         # token order inside an expert
            dropped_t = [t for t in range(T) for j in range(k)
                         if idx[t, j] == e and dsp.slot_of[t, j] < 0]
            if dropped_t and seg.size:
                assert min(dropped_t) > seg.max()                    # drops are the last arrivals
        for t in range(T):
            for j in range(k):
                s = dsp.slot_of[t, j]
                if s >= 0:
                    assert dsp.perm[s] == t
                    assert dsp.offsets[idx[t, j]] <= s < dsp.offsets[idx[t, j] + 1]


def _shard_cuts(rng, T, R):
    """Token ranges of R shards in token order (some may be empty)."""
    return np.concatenate([[0], np.sort(rng.integers(0, T + 1, R - 1)), [T]]).astype(int)


def test_dispatch_shard_equals_whole_batch(oracle_mod):
    """A batch split over ranks in token order: with each shard's bases = the earlier shards'
    counts, the kept / dropped decisions and every expert's token order equal those of the
    whole batch (pinned by the stable-sort brute force)."""
    rng = np.random.default_rng(6)
    for trial in range(300):
        T = int(rng.integers(1, 40))
        E = int(rng.integers(1, 6))
        k = 1 if E == 1 else int(rng.integers(1, 3))
        idx = np.array([rng.choice(E, k, replace=False) for _ in range(T)], np.int32).reshape(T, k)
        if trial % 3 == 0:
            idx[:, 0] = rng.integers(0, min(E, 2), T)       # skewed first choices
            if k == 2:
                idx[:, 1] = (idx[:, 0] + 1 + rng.integers(0, E - 1, T)) % E
        cf = float(rng.choice([0.5, 1.0, 1.25, 2.0]))
        C = oracle_mod.capacity(T, E, cf)
        counts, kept, offs, perm, slot = _dispatch_bruteforce(idx, E, C)
        R = int(rng.integers(1, 5))
        cuts = _shard_cuts(rng, T, R)
        per = np.array([np.bincount(idx[cuts[r]:cuts[r + 1]].reshape(-1), minlength=E)
                        for r in range(R)])
        bases = oracle_mod.shard_bases(per)
        assert np.array_equal(bases[0], np.zeros(E))
        kept_sum = np.zeros(E, np.int64)
        for r in range(R):
            lo, hi = cuts[r], cuts[r + 1]
            got = oracle_mod.dispatch_shard(idx[lo:hi], E, C, bases[r])
            assert np.array_equal(got.counts_raw, per[r])
            kept_sum += got.kept
            assert np.array_equal(got.slot_of >= 0, slot[lo:hi] >= 0)
            for e in range(E):
                mine = got.perm[got.offsets[e]:got.offsets[e + 1]] + lo
                whole = perm[offs[e]:offs[e + 1]]
                assert np.array_equal(mine, whole[(whole >= lo) & (whole < hi)])
            for t in range(hi - lo):
                for j in range(k):
                    if got.slot_of[t, j] >= 0:
                        assert got.perm[got.slot_of[t, j]] == t
        assert np.array_equal(kept_sum, kept)


def test_dispatch_single_shard_is_plain_dispatch(oracle_mod):
    rng = np.random.default_rng(7)
    for _ in range(50):
        T, E = int(rng.integers(1, 50)), int(rng.integers(2, 9))
        idx = np.array([rng.choice(E, 2, replace=False) for _ in range(T)], np.int32)
        C = oracle_mod.capacity(T, E, float(rng.choice([0.5, 1.0, 1.25])))
        a = oracle_mod.dispatch(idx, E, C)
        b = oracle_mod.dispatch_shard(idx, E, C, np.zeros(E, np.int32))
        for f in ("counts_raw", "kept", "offsets", "perm", "slot_of"):
            assert np.array_equal(getattr(a, f), getattr(b, f)), f


# ---------------------------------------------------------------- GeLU and the MLP
def test_gelu_identities_and_library(oracle_mod):
    import torch
    xs = np.linspace(-8, 8, 161)
    got = np.array([oracle_mod.gelu(v) for v in xs])
    assert oracle_mod.gelu(0.0) == 0.0
    assert np.allclose(got - np.array([oracle_mod.gelu(-v) for v in xs]), xs, rtol=0, atol=1e-14)
    ref = torch.nn.functional.gelu(torch.tensor(xs, dtype=torch.float64), approximate="tanh")
    assert np.allclose(got, ref.numpy(), rtol=1e-14, atol=1e-15)
    assert abs(oracle_mod.gelu(40.0) - 40.0) < 1e-12 and abs(oracle_mod.gelu(-40.0)) < 1e-12


def _np_gelu(x):
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def _dense_bruteforce(x, W1, W2, logits, k, cf, Wr1=None, Wr2=None):
    """Every expert on every token (numpy float64), then a mask from the stable-sort dispatch."""
    T, d = x.shape
    E = W1.shape[0]
    xd = x.astype(np.float64)
    Y = np.stack([_np_gelu(xd @ W1[e].astype(np.float64)) @ W2[e].astype(np.float64)
                  for e in range(E)])                                # [E, T, d]
    l = logits.astype(np.float64)
    idx = _topk_bruteforce(logits, k)
    p = np.exp(l - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    pk = p[np.arange(T)[:, None], idx]
    w = pk if k == 1 else pk / pk.sum(1, keepdims=True)
    C = math.ceil(Fraction(cf) * T / E)
    _, _, _, _, slot = _dispatch_bruteforce(idx, E, C)
    out = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            if slot[t, j] >= 0:
                out[t] += w[t, j] * Y[idx[t, j], t]
    if Wr1 is not None:
        out += _np_gelu(xd @ Wr1.astype(np.float64)) @ Wr2.astype(np.float64)
    return out


@pytest.mark.parametrize("k,residual,dtype", [(1, False, np.float32), (2, False, np.float16),
                                              (1, True, np.float16), (2, True, np.float32)])
def test_layer_matches_dense_bruteforce(oracle_mod, k, residual, dtype):
    rng = np.random.default_rng(6 + k)
    T, d, f, E, cf = 24, 16, 32, 4, 1.0
    x = rng.standard_normal((T, d)).astype(dtype)
    Wg = (rng.standard_normal((d, E)) * 0.3).astype(np.float32)
    W1 = (rng.standard_normal((E, d, f)) * 0.2).astype(dtype)
    W2 = (rng.standard_normal((E, f, d)) * 0.2).astype(dtype)
    Wr1 = (rng.standard_normal((d, 24)) * 0.2).astype(dtype) if residual else None
    Wr2 = (rng.standard_normal((24, d)) * 0.2).astype(dtype) if residual else None
    out, r = oracle_mod.layer_forward(x, Wg, W1, W2, k, cf, Wr1, Wr2)
    ref = _dense_bruteforce(x, W1, W2, r.logits, k, cf, Wr1, Wr2)
    assert (r.disp.slot_of < 0).any()                                # some drops happen
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)
    # a subset of rows gives the same rows
    rows = np.array([5, 0, 23], np.int32)
    sub = oracle_mod.combine_rows(x, r, W1, W2, Wr1, Wr2, rows=rows)
    assert np.array_equal(sub, out[rows])


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("k", [1, 2])
def test_closed_form_zero_gate(oracle_mod, k):
    rng = np.random.default_rng(8)
    T, d, f, E, cf = 20, 8, 16, 4, 1.0
    x = rng.standard_normal((T, d)).astype(np.float16)
    W1 = (rng.standard_normal((E, d, f)) * 0.5).astype(np.float16)
    W2 = (rng.standard_normal((E, f, d)) * 0.5).astype(np.float16)
    out, r = oracle_mod.layer_forward(x, np.zeros((d, E), np.float32), W1, W2, k, cf)
    C = math.ceil(cf * T / E)
    assert np.all(r.probs == 1.0 / E)
    assert np.array_equal(r.topk_idx[:, 0], np.zeros(T))
    assert r.disp.kept[0] == min(T, C)
    xd = x.astype(np.float64)
    for t in range(T):
        if k == 1:
            want = (1.0 / E) * (_np_gelu(xd[t] @ W1[0].astype(np.float64)) @ W2[0].astype(np.float64))
        else:
            assert r.topk_idx[t, 1] == 1 and np.all(r.topk_w[t] == 0.5)
            want = sum(0.5 * (_np_gelu(xd[t] @ W1[e].astype(np.float64)) @ W2[e].astype(np.float64))
                       for e in (0, 1))
        if t >= C:
            want = np.zeros(d)
        assert np.allclose(out[t], want, rtol=1e-12, atol=1e-15)


def test_closed_form_constant_token_and_zero_input(oracle_mod):
    rng = np.random.default_rng(9)
    T, d, f, E, cf, fr = 16, 8, 16, 4, 1.25, 12
    x1 = rng.standard_normal(d).astype(np.float32)
    x = np.tile(x1, (T, 1))
    Wg = rng.standard_normal((d, E)).astype(np.float32)
    W1 = rng.standard_normal((E, d, f)).astype(np.float32)
    W2 = rng.standard_normal((E, f, d)).astype(np.float32)
    Wr1 = rng.standard_normal((d, fr)).astype(np.float32)
    Wr2 = rng.standard_normal((fr, d)).astype(np.float32)
    out, r = oracle_mod.layer_forward(x, Wg, W1, W2, 1, cf, Wr1, Wr2)
    l = x1.astype(np.float64) @ Wg.astype(np.float64)
    es = int(np.argmax(l))
    assert np.all(r.topk_idx[:, 0] == es)
    assert np.all(r.logits == r.logits[0])              # identical tokens, identical logits
    lf = r.logits[0].astype(np.float64)                 # the fp32 chain (pinned above)
    w = 1.0 / np.exp(lf - lf[es]).sum()
    C = math.ceil(cf * T / E)
    ffn = _np_gelu(x1.astype(np.float64) @ W1[es].astype(np.float64)) @ W2[es].astype(np.float64)
    res = _np_gelu(x1.astype(np.float64) @ Wr1.astype(np.float64)) @ Wr2.astype(np.float64)
    for t in range(T):
        want = (w * ffn if t < C else 0.0) + res
        assert np.allclose(out[t], want, rtol=1e-9, atol=1e-12)
    out0, _ = oracle_mod.layer_forward(np.zeros((T, d), np.float16), Wg, W1.astype(np.float16),
                                       W2.astype(np.float16), 2, cf, Wr1.astype(np.float16),
                                       Wr2.astype(np.float16))
    assert np.all(out0 == 0.0)


def test_single_expert_reduces_to_mlp(oracle_mod):
    import torch
    rng = np.random.default_rng(10)
    T, d, f = 33, 24, 40
    x = rng.standard_normal((T, d)).astype(np.float16)
    W1 = (rng.standard_normal((1, d, f)) * 0.3).astype(np.float16)
    W2 = (rng.standard_normal((1, f, d)) * 0.3).astype(np.float16)
    Wg = rng.standard_normal((d, 1)).astype(np.float32)
    out, r = oracle_mod.layer_forward(x, Wg, W1, W2, 1, 1.0)
    assert np.all(r.probs == 1.0) and (r.disp.slot_of >= 0).all()
    xt = torch.tensor(x.astype(np.float64))
    h = torch.nn.functional.gelu(xt @ torch.tensor(W1[0].astype(np.float64)), approximate="tanh")
    ref = (h @ torch.tensor(W2[0].astype(np.float64))).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_expert_ffn_single_row(oracle_mod, dtype):
    """The one-row expert FFN (the reference of the standalone expert-FFN checks) against
    torch float64 (library matmuls and torch's own tanh GeLU), with d != f so that a swapped
    or transposed W1 / W2 cannot pass; then the same row through the one-expert, weight-1
    combine, and the output's linearity in W2."""
    import torch
    rng = np.random.default_rng(21)
    d, f = 24, 56
    W1 = (rng.standard_normal((d, f)) * 0.3).astype(dtype)
    W2 = (rng.standard_normal((f, d)) * 0.3).astype(dtype)
    xs = rng.standard_normal((5, d)).astype(dtype)
    for x in xs:
        y = oracle_mod.expert_ffn(x, W1, W2)
        assert y.shape == (d,) and y.dtype == np.float64
        xt = torch.tensor(x.astype(np.float64))[None, :]
        h = torch.nn.functional.gelu(xt @ torch.tensor(W1.astype(np.float64)), approximate="tanh")
        ref = (h @ torch.tensor(W2.astype(np.float64))).numpy()[0]
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
        # a scaled W2 scales the output (exact: powers of two)
        y4 = oracle_mod.expert_ffn(x, W1, (W2.astype(np.float64) * 4).astype(dtype))
        assert np.array_equal(y4, 4 * y)
    assert np.all(oracle_mod.expert_ffn(np.zeros(d, dtype), W1, W2) == 0.0)
    # the same rows through the layer's combine with one expert and weight 1
    T = xs.shape[0]
    r = oracle_mod.Routing(logits=np.zeros((T, 1), np.float32), probs=np.ones((T, 1)),
                           topk_idx=np.zeros((T, 1), np.int32), topk_w=np.ones((T, 1)),
                           disp=oracle_mod.dispatch(np.zeros((T, 1), np.int32), 1, T))
    out = oracle_mod.combine_rows(xs, r, W1[None], W2[None])
    for t in range(T):
        assert np.array_equal(out[t], oracle_mod.expert_ffn(xs[t], W1, W2))


def test_stack_of_single_expert_layers_is_an_mlp_chain(oracle_mod):
    """A stack of E = 1 layers (one with a residual MLP) is the plain chain of MLPs, with each
    layer's output rounded to fp16 before the next layer; checked against torch float64."""
    import torch
    rng = np.random.default_rng(12)
    T, d, f = 17, 16, 24
    x = rng.standard_normal((T, d)).astype(np.float16)
    layers = []
    for l in range(3):
        L = dict(Wg=rng.standard_normal((d, 1)).astype(np.float32),
                 W1=(rng.standard_normal((1, d, f)) * 0.3).astype(np.float16),
                 W2=(rng.standard_normal((1, f, d)) * 0.3).astype(np.float16))
        if l == 1:
            L["Wr1"] = (rng.standard_normal((d, f)) * 0.3).astype(np.float16)
            L["Wr2"] = (rng.standard_normal((f, d)) * 0.3).astype(np.float16)
        layers.append(L)
    outs, ins, routings = oracle_mod.stack_forward(x, layers, 1, 1.0)
    assert len(outs) == 3 and all((r.disp.slot_of >= 0).all() for r in routings)

    def mlp(h, A, B):
        g = torch.nn.functional.gelu(h @ torch.tensor(A.astype(np.float64)), approximate="tanh")
        return g @ torch.tensor(B.astype(np.float64))

    h = torch.tensor(x.astype(np.float64))
    for l, L in enumerate(layers):
        y = mlp(h, L["W1"][0], L["W2"][0])
        if "Wr1" in L:
            y = y + mlp(h, L["Wr1"], L["Wr2"])
        assert np.allclose(outs[l], y.numpy(), rtol=1e-12, atol=1e-13), l
        assert np.array_equal(ins[l], h.numpy().astype(np.float16))
        h = torch.tensor(y.numpy().astype(np.float16).astype(np.float64))


# ---------------------------------------------------------------- stored regression fixture
def test_golden_tiny_fp32(oracle_mod):
    """Fixture written by tests/golden/make_golden.py (which calls only oracle/ and synth/)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_fp32_T128_seed0.txt")
    data = {}
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        key, val = line.split(":", 1)
        data[key.strip()] = val.split()
    cfg = synth.CONFIGS["tiny_fp32"]
    inp = synth.host_inputs(cfg, 128, seed=0)
    out, r = oracle_mod.layer_forward(inp["tokens"], inp["Wg"], inp["W1"], inp["W2"], cfg.k, cfg.cf)
    assert [int(v) for v in data["topk_idx"]] == r.topk_idx.reshape(-1).tolist()
    assert [int(v) for v in data["slot_of"]] == r.disp.slot_of.reshape(-1).tolist()
    assert [int(v) for v in data["counts_raw"]] == r.disp.counts_raw.tolist()
    assert [float.fromhex(v) for v in data["logits_row0"]] == r.logits[0].astype(np.float64).tolist()
    ref = np.array([float(v) for v in data["out_rows_0_1_127"]]).reshape(3, -1)
    assert np.allclose(out[[0, 1, 127]], ref, rtol=1e-13, atol=1e-17)


# ---------------------------------------------------------------- thread count
def test_layer_independent_of_thread_count(oracle_mod):
    """The oracle's results do not depend on how many host threads run it (each token's
    chain and FFN run in one thread, in a fixed order), so the one-core and all-core timings
    of the CPU baseline time the same computation."""
    rng = np.random.default_rng(11)
    T, d, f, E, cf = 40, 32, 64, 8, 1.25
    x = rng.standard_normal((T, d)).astype(np.float16)
    Wg = (rng.standard_normal((d, E)) * 0.3).astype(np.float32)
    W1 = (rng.standard_normal((E, d, f)) * 0.2).astype(np.float16)
    W2 = (rng.standard_normal((E, f, d)) * 0.2).astype(np.float16)
    Wr1 = (rng.standard_normal((d, 48)) * 0.2).astype(np.float16)
    Wr2 = (rng.standard_normal((48, d)) * 0.2).astype(np.float16)
    threads = oracle_mod.num_threads()
    try:
        oracle_mod.set_num_threads(1)
        assert oracle_mod.num_threads() == 1
        one, r1 = oracle_mod.layer_forward(x, Wg, W1, W2, 2, cf, Wr1, Wr2)
    finally:
        oracle_mod.set_num_threads(threads)
    assert oracle_mod.num_threads() == threads
    many, rn = oracle_mod.layer_forward(x, Wg, W1, W2, 2, cf, Wr1, Wr2)
    assert np.array_equal(r1.logits.view(np.uint32), rn.logits.view(np.uint32))
    assert np.array_equal(r1.disp.slot_of, rn.disp.slot_of)
    assert np.array_equal(one.view(np.uint64), many.view(np.uint64))
