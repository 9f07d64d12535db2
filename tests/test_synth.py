"""The seeded input generator (CPU): C draws equal the Python definition, roundings match numpy."""
import numpy as np

import synth


def test_host_draws_match_python_definition():
    for tid in (synth.TID_TOKENS, synth.TID_W1, synth.TID_WG + (3 << 8)):
        z = synth.draw_unit(7, seed=0, tid=tid, first=1000)
        assert z.tolist() == [synth.draw_z_py(0, tid, 1000 + q) for q in range(7)]
    a = synth.fill((5, 7), synth.F32, 3, synth.TID_W2, sigma=0.5, first=11)
    z = synth.draw_unit(35, 3, synth.TID_W2, first=11)
    assert np.array_equal(a.reshape(-1), (z * 0.5).astype(np.float32))


def test_half_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(20000) * s for s in (1e-7, 1e-5, 0.02, 1, 300, 6e4)])
    vals = np.concatenate([vals, [0.0, -0.0, 65504.0, 65519.9, 65520.0, 2.0 ** -24, 2.0 ** -25,
                                  3 * 2.0 ** -26, 2.0 ** -14 - 2.0 ** -26]])
    lib = synth._hostlib()
    got = np.array([lib.synth_double_to_half(float(v)) for v in vals], np.uint16)
    with np.errstate(over="ignore"):       # values past 65520 round to infinity, as intended
        want = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_fill_col_scale_and_runs():
    sc = np.array([0.5, 2.0, 1.0])
    a = synth.fill((4, 3), synth.F16, 1, synth.TID_WG, col_scale=sc)
    z = synth.draw_unit(12, 1, synth.TID_WG).reshape(4, 3)
    assert np.array_equal(a, (z * sc[None, :]).astype(np.float16))
    full = synth.fill((6, 5), synth.F16, 2, synth.TID_W1, 0.02)
    part = synth.fill((2, 5), synth.F16, 2, synth.TID_W1, 0.02, first=3 * 5)
    assert np.array_equal(full[3:5], part)


def test_draw_moments():
    z = synth.fill((200000,), synth.F32, 0, synth.TID_TOKENS, 1.0).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01


def test_zipf_design_shares():
    sd = synth.zipf_column_norms(128, 1.2)
    p = synth._argmax_shares(sd, 8001)
    assert np.abs(p - synth.zipf_targets(128, 1.2)).sum() < 2e-3
    perm = synth.seeded_permutation(128, 0)
    assert sorted(perm.tolist()) == list(range(128)) and perm[0] != 0
