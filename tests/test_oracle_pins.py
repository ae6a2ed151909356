"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks one oracle function against something it cannot agree with
by construction: numbers printed on the pages (golden fixtures), closed forms,
brute-force enumeration on tiny inputs, or a library routine (numpy/scipy)
for a special case. No test retypes the oracle's own loop.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bf16(vals):
    return synth.to_bf16_bits(np.asarray(vals, dtype=np.float64))


def f32(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ counts


def test_counts_round_to_nearest():
    # The single-layer d_ff=1024 workload states beta = 205 for a 20% dynamic
    # ratio (0.2 * 1024 = 204.8), so counts round to nearest, not down.
    assert oracle.cnt(0.2, 1024) == 205
    assert oracle.cnt(0.4, 1024) - oracle.cnt(0.2, 1024) == 205
    assert oracle.cnt(0.7, 1024) == 717
    assert oracle.cnt(0.5, 3) == 2          # x.5 rounds up
    assert oracle.cnt(0.0, 100) == 0 and oracle.cnt(1.0, 100) == 100


def test_table1_layer_range(golden_dir):
    """Table 1: selection starts at layer 5 ("First layer 5") and skips the
    last two ("Last layer -2 (skip last 2)"); the other layers stay dense."""
    g = json.load(open(os.path.join(golden_dir, "selectinfer_table1.json")))
    first, last = g["first_layer"], g["last_layer"]
    for L in (16, 28, 36, 8):          # Llama3.2-1B, -3B, Qwen2.5-3B depths, a shallow stack
        m = oracle.sparse_layers(L, first, last)
        assert m.shape == (L,)
        assert not m[:5].any()          # layers 0..4 keep the dense FFN
        assert not m[-2:].any()         # so do the last two
        assert m[5:L - 2].all()         # and every layer in between selects
        assert int(m.sum()) == L - 7
    assert oracle.sparse_layers(16, 0, 0).all()                 # skip the last 0: the whole stack
    assert oracle.sparse_layers(16, 2, 10).sum() == 8           # a positive end is a layer index
    assert not oracle.sparse_layers(6, 5, -2).any()             # too shallow for the range
    with pytest.raises(ValueError):
        oracle.sparse_layers(16, -1, -2)


def test_table1_fractions(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "selectinfer_table1.json")))
    # static + dynamic = computed (phi = delta + epsilon), base + secondary = loaded
    assert g["static_pct"] + g["dynamic_pct"] == g["computed_pct"]
    assert g["static_pct"] + g["secondary_pct"] == g["loaded_pct"]
    # the oracle's loading and selection realise exactly those fractions
    N = 1000
    rng = np.random.default_rng(1)
    sc = rng.random(N).astype(np.float32)
    loaded, st = oracle.rank_loaded(sc, sc, g["loaded_pct"] / 100, g["static_pct"] / 100)
    assert len(loaded) == oracle.cnt(0.7, N) == 700
    assert int(st.sum()) == oracle.cnt(0.3, N) == 300
    A = synth.lognormal_absact(3, 8, len(loaded))
    n_sel = oracle.cnt(g["computed_pct"] / 100, N)
    S = oracle.select(A, 8, 1, len(loaded), st, 50, n_sel)
    assert S.shape == (1, 400)
    assert int(st[S[0]].sum()) == 300        # all static neurons are computed
    assert len(S[0]) - 300 == 100            # dynamic = 10% of N


def test_eq2_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "selectinfer_eq2.json")))
    # Eq. (2) with the printed numbers gives the printed 0.945 GB
    dm = g["n_ffn_params"] * (1 - g["r_load"]) * g["r_layer"] * g["bytes_per_param"]
    assert abs(dm / 1e9 - g["delta_m_gb"]) < 1e-9
    # the oracle's byte accounting of selective loading on the real shape
    s = g["llama32_3b_shape"]
    d, N, L = s["d"], s["d_ff"], s["layers"]
    n_ffn = 3 * d * N * L
    assert abs(n_ffn / 2.1e9 - 1) < 0.01      # "N_ffn ~ 2.1B"
    applied = round(g["r_layer"] * L)
    full = 3 * d * N * g["bytes_per_param"]
    kept = oracle.loaded_bytes(d, oracle.cnt(g["r_load"], N), g["bytes_per_param"])
    saved = applied * (full - kept)
    assert abs(saved / 1e9 - g["delta_m_gb"]) / g["delta_m_gb"] < 0.01


# ------------------------------------------------------------- activations

SILU2 = 1.0 + math.tanh(1.0)       # silu(2) = 2 * sigmoid(2), sigmoid(x) = (1 + tanh(x/2)) / 2
SILUM2 = -(1.0 - math.tanh(1.0))   # silu(-2)
SILU3 = 1.5 * (1.0 + math.tanh(1.5))


def test_profile_closed_form():
    # d = 2; tokens e1, -e1, e2. Neuron 0: g = 2*x0, u = x0; neuron 1: g = 2*x0, u = -x0;
    # neuron 2: g = 3*x1, u = 0.5*x1; neuron 3: g = 0 (silu(0) = 0), u = 7*x0.
    Wg = bf16([[2, 0], [2, 0], [0, 3], [0, 0]])
    Wu = bf16([[1, 0], [-1, 0], [0, 0.5], [7, 0]])
    X = bf16([[1, 0], [-1, 0], [0, 1]])
    s = oracle.profile_scores(Wg, Wu, X)
    # neuron 0: |silu(2)*1| + |silu(-2)*(-1)| + 0 = (1 + tanh 1) + (1 - tanh 1) = 2
    assert s[0] == pytest.approx(2.0, rel=1e-15)
    assert s[1] == pytest.approx(2.0, rel=1e-15)          # |a| keeps negative activations
    assert s[2] == pytest.approx(0.5 * SILU3, rel=1e-15)
    assert s[3] == 0.0
    # accumulation over calls (scores are running sums)
    s2 = oracle.profile_scores(Wg, Wu, X, scores=s.copy())
    assert np.allclose(s2, 2 * s, rtol=1e-15)


def _np_act(Wg, Wu, X):
    g = f32(X) @ f32(Wg).T
    u = f32(X) @ f32(Wu).T
    return g * expit(g) * u


def test_profile_vs_library():
    Wg, Wu, _ = synth.layer_weights(7, 0, 64, 48)
    X = synth.tokens(7, 0, synth.T_CALIB, 20, 64)
    s = oracle.profile_scores(Wg, Wu, X)
    ref = np.abs(_np_act(Wg, Wu, X)).sum(axis=0)
    assert np.allclose(s, ref, rtol=1e-12, atol=0)


def test_absact_and_dense_act_vs_library():
    Wg, Wu, _ = synth.layer_weights(8, 0, 40, 30, sigma=1.5)
    X = synth.tokens(8, 0, synth.T_PROMPT, 5, 40)
    loaded = np.array([0, 3, 4, 9, 10, 29], np.int32)
    A = oracle.absact(Wg, Wu, loaded, X)
    ref = np.abs(_np_act(Wg, Wu, X))[:, loaded]
    assert np.allclose(A, ref, rtol=1e-12, atol=1e-300)
    a = oracle.dense_act(Wg, Wu, X[2])
    assert np.allclose(a, _np_act(Wg, Wu, X[2:3])[0], rtol=1e-12)


def test_silu_special_values():
    Wg = bf16([[2], [-2], [3]])
    Wu = bf16([[1], [1], [1]])
    a = oracle.dense_act(Wg, Wu, bf16([1]))
    assert a == pytest.approx([SILU2, SILUM2, SILU3], rel=1e-15)


# ------------------------------------------------------------- sparse FFN


def test_sparse_ffn_all_neurons_is_dense_ffn():
    # gamma = phi = 1: no neuron is skipped, so the output is the dense SwiGLU FFN
    d, N = 24, 40                       # d != N catches a transposed down matrix
    Wg, Wu, Wd = synth.layer_weights(9, 0, d, N)
    x = synth.tokens(9, 0, synth.T_DECODE, 1, d)[0]
    loaded = np.arange(N, dtype=np.int32)
    y = oracle.sparse_ffn(Wg, Wu, Wd, loaded, loaded, x)
    ref = f32(Wd) @ _np_act(Wg, Wu, x[None, :])[0]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)


def test_sparse_ffn_subset_is_masked_dense():
    d, N = 16, 50
    Wg, Wu, Wd = synth.layer_weights(10, 0, d, N)
    x = synth.tokens(10, 0, synth.T_DECODE, 1, d)[0]
    loaded = np.array(sorted(np.random.default_rng(0).choice(N, 30, replace=False)), np.int32)
    S = np.array([0, 2, 3, 7, 11, 29], np.int32)          # packed positions
    y = oracle.sparse_ffn(Wg, Wu, Wd, loaded, S, x)
    keep = loaded[S]
    a = _np_act(Wg, Wu, x[None, :])[0]
    ref = f32(Wd)[:, keep] @ a[keep]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------- top-k


def _brute_topk(vals, k):
    """The unique k-subset whose members all precede every non-member in the
    order (value desc, index asc), found by enumeration."""
    n = len(vals)

    def before(i, j):
        return vals[i] > vals[j] or (vals[i] == vals[j] and i < j)

    found = []
    for sub in itertools.combinations(range(n), k):
        s = set(sub)
        if all(before(i, j) for i in s for j in range(n) if j not in s):
            found.append(s)
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("seed", range(6))
def test_topk_rows_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 9))
    rows = 4
    A = (rng.integers(0, 3, size=(rows, n)) / 2).astype(np.float32)   # many ties
    for k in range(0, n + 1):
        sel = oracle.topk_rows(A, k)
        for r in range(rows):
            assert set(np.nonzero(sel[r])[0]) == (_brute_topk(list(A[r]), k) if k else set())


def test_topk_uses_magnitude_and_ld():
    A = np.array([[-5.0, 1.0, 2.0, 99.0]], np.float32)   # column 3 outside n
    sel = oracle.topk_rows(A, 1, n=3)
    assert list(sel[0]) == [1, 0, 0]


@pytest.mark.parametrize("seed", range(5))
def test_select_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    n_loaded = int(rng.integers(3, 8))
    T, B = int(rng.integers(1, 5)), int(rng.integers(1, 3))
    st = np.zeros(n_loaded, np.uint8)
    st[rng.choice(n_loaded, int(rng.integers(0, n_loaded)), replace=False)] = 1
    n_static = int(st.sum())
    alpha = int(rng.integers(1, n_loaded + 1))
    n_sel = int(rng.integers(n_static, n_loaded + 1))
    A = (rng.integers(0, 4, size=(B * T, n_loaded)) / 4).astype(np.float32)
    S, counts, sel = oracle.select(A, T, B, n_loaded, st, alpha, n_sel, want_counts=True, want_sel=True)
    for b in range(B):
        lists = [_brute_topk(list(A[b * T + t]), alpha) for t in range(T)]
        for t in range(T):
            assert set(np.nonzero(sel[b * T + t])[0]) == lists[t]
        ref_cnt = np.bincount([p for l in lists for p in l], minlength=n_loaded)
        assert np.array_equal(counts[b], ref_cnt)
        cand = [p for p in range(n_loaded) if not st[p]]
        beta = n_sel - n_static
        # top-beta of the counts among non-static positions, by enumeration
        cv = [float(ref_cnt[p]) for p in cand]
        dyn = {cand[i] for i in _brute_topk(cv, beta)} if beta else set()
        expect = sorted(set(np.nonzero(st)[0]) | dyn)
        assert list(S[b]) == expect


def test_select_zero_counts_fill_by_lower_index():
    # one token, alpha=1: only position 4 gets a count; beta=3 takes 4 then 0, 1
    A = np.array([[0, 0, 0, 0, 9, 0]], np.float32)
    st = np.zeros(6, np.uint8)
    S = oracle.select(A, 1, 1, 6, st, 1, 3)
    assert list(S[0]) == [0, 1, 4]


# --------------------------------------------------------------- loading


@pytest.mark.parametrize("seed", range(5))
def test_rank_loaded_brute_force(seed):
    rng = np.random.default_rng(200 + seed)
    N = int(rng.integers(2, 9))
    task = (rng.integers(0, 4, N) / 2).astype(np.float32)
    model = (rng.integers(0, 4, N) / 2).astype(np.float32)
    gamma = float(rng.integers(1, N + 1)) / N
    delta = float(rng.integers(0, int(round(gamma * N)) + 1)) / N
    loaded, st = oracle.rank_loaded(task, model, gamma, delta)
    nb, nl = oracle.cnt(delta, N), oracle.cnt(gamma, N)
    base = _brute_topk(list(task), nb) if nb else set()
    rest = [n for n in range(N) if n not in base]
    sec = {rest[i] for i in _brute_topk([float(model[n]) for n in rest], nl - nb)} if nl > nb else set()
    assert list(loaded) == sorted(base | sec)
    assert {int(loaded[p]) for p in range(len(loaded)) if st[p]} == base


def test_rank_loaded_single_file_is_top_gamma():
    rng = np.random.default_rng(5)
    s = rng.random(300).astype(np.float32)
    loaded, st = oracle.rank_loaded(s, s, 0.7, 0.2)
    assert set(loaded) == set(np.argsort(-s, kind="stable")[:210])
    assert set(loaded[st == 1]) == set(np.argsort(-s, kind="stable")[:60])


def test_merge_scores_hand_computed():
    # file 1: scores (2, 4) over 2 tokens; file 2: (9, 3) over 3 tokens
    out = oracle.merge_scores([np.array([2, 4], np.float32), np.array([9, 3], np.float32)], [2, 3])
    assert list(out) == [4.0, 3.0]
    out1 = oracle.merge_scores([np.array([6, 1.5], np.float32)], [3])
    assert list(out1) == [2.0, 0.5]


# ------------------------------------------------------------------ SpAx


def test_spax_encode_bound_and_layout():
    d, N = 256, 6
    _, _, Wd = synth.layer_weights(11, 0, d, N)
    codes, params = oracle.spax_encode(Wd, 4, 128)
    w = f32(Wd)
    for n in range(N):
        q = np.zeros(d, np.int64)
        q[0::2] = codes[n] & 0xF
        q[1::2] = codes[n] >> 4
        for g in range(d // 128):
            scale, mn = params[n, g]
            grp = w[g * 128:(g + 1) * 128, n]
            assert mn == grp.min()
            assert scale == pytest.approx((grp.max() - grp.min()) / 15, rel=1e-6)
            rec = mn + q[g * 128:(g + 1) * 128] * float(scale)
            assert np.all(np.abs(rec - grp) <= float(scale) / 2 * (1 + 1e-5) + 1e-12)


def test_spax_encode_constant_and_ramp_groups():
    d, N = 256, 2
    W = np.zeros((d, N))
    W[:128, 0] = 0.375                      # constant group: scale 0, codes 0, exact
    W[128:, 0] = np.arange(128) % 16 * 0.5  # ramp 0..7.5: min 0, scale 0.5, codes = ramp
    W[:, 1] = -1.25
    Wd = bf16(W)
    codes, params = oracle.spax_encode(Wd, 4, 128)
    assert params[0, 0, 0] == 0.0 and params[0, 0, 1] == np.float32(0.375)
    assert np.all(codes[0, :64] == 0)
    assert params[0, 1, 0] == np.float32(0.5) and params[0, 1, 1] == 0.0
    ramp = np.arange(128) % 16
    assert np.array_equal(codes[0, 64:], (ramp[0::2] | (ramp[1::2] << 4)).astype(np.uint8))
    assert codes[0, 64] == 0x10             # element 2i in the low nibble
    assert np.all(params[1, :, 0] == 0.0) and np.all(params[1, :, 1] == np.float32(-1.25))


def _codes_of(codes, d, bits):
    # element i of a column: bits i*bits .. i*bits+bits-1 of the column's
    # little-endian bit stream, read through a Python integer
    out = np.zeros((codes.shape[0], d), np.int64)
    for n in range(codes.shape[0]):
        stream = int.from_bytes(bytes(codes[n]), "little")
        for i in range(d):
            out[n, i] = (stream >> (i * bits)) & ((1 << bits) - 1)
    return out


def test_spax_encode_other_widths():
    d, N = 128, 3
    _, _, Wd = synth.layer_weights(12, 0, d, N)
    for bits in (2, 3, 8):
        codes, params = oracle.spax_encode(Wd, bits, 64)
        assert codes.shape == (N, d * bits // 8)
        w = f32(Wd)
        q = _codes_of(codes, d, bits)
        for n in range(N):
            for g in range(2):
                scale, mn = params[n, g]
                rec = mn + q[n, g * 64:(g + 1) * 64] * float(scale)
                assert np.all(np.abs(rec - w[g * 64:(g + 1) * 64, n]) <= float(scale) / 2 * (1 + 1e-5) + 1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_spax_tiers_brute_force(seed):
    rng = np.random.default_rng(300 + seed)
    N = int(rng.integers(2, 9))
    a = ((rng.integers(0, 5, N) - 2) / 2).astype(np.float32)   # signs and ties
    k_top = int(rng.integers(0, N + 1))
    k_mid = int(rng.integers(0, N - k_top + 1))
    top, mid = oracle.spax_tiers(a, k_top, k_mid)
    mag = list(np.abs(a))
    t = _brute_topk(mag, k_top) if k_top else set()
    tm = _brute_topk(mag, k_top + k_mid) if k_top + k_mid else set()
    assert list(top) == sorted(t)
    assert list(mid) == sorted(tm - t)


def test_spax_down_limits():
    d, N = 256, 40
    _, _, Wd = synth.layer_weights(13, 0, d, N)
    a = synth.normal(13, 0, synth.T_SPAX_A, N).astype(np.float32)
    codes, params = oracle.spax_encode(Wd, 4, 128)
    allc = np.arange(N, dtype=np.int32)
    none = np.zeros(0, np.int32)
    # top = 100%: the dense down projection
    y = oracle.spax_down(a, Wd, codes, params, allc, none)
    assert np.allclose(y, f32(Wd) @ a.astype(np.float64), rtol=1e-12, atol=1e-14)
    # mid = 100%: within the quantisation error bound of the dense result
    y2 = oracle.spax_down(a, Wd, codes, params, none, allc)
    bound = (np.abs(a.astype(np.float64))[None, :] * np.repeat(params[:, :, 0].T, 128, axis=0) / 2).sum(axis=1)
    assert np.all(np.abs(y2 - f32(Wd) @ a.astype(np.float64)) <= bound * (1 + 1e-5) + 1e-12)
    # nothing selected: zero
    assert np.all(oracle.spax_down(a, Wd, codes, params, none, none) == 0)


def test_down_norms():
    """Weight norms of the salience |a_n| * ||Wd[:, n]||_2: closed forms on
    constant and one-hot columns, and numpy's norm on random bf16 columns."""
    d, N = 64, 5
    Wd = np.zeros((d, N))
    Wd[:, 0] = 1.0                 # sqrt(d)
    Wd[:, 1] = -0.5                # 0.5 sqrt(d)
    Wd[7, 2] = 3.0                 # one-hot: |3|
    Wd[:, 4] = 2.0                 # sqrt(4 d)
    got = oracle.down_norms(bf16(Wd), np.array([4, 0, 2, 1, 3], np.int32))
    assert np.allclose(got, [2 * np.sqrt(d), np.sqrt(d), 3.0, 0.5 * np.sqrt(d), 0.0], rtol=0, atol=1e-12)
    Wr = bf16(np.random.default_rng(5).standard_normal((256, 40)) * 0.1)
    loaded = np.array([39, 0, 17, 5], np.int32)
    ref = np.linalg.norm(f32(Wr)[:, loaded], axis=0)
    assert np.allclose(oracle.down_norms(Wr, loaded), ref, rtol=1e-12, atol=0)


def test_expand_clusters():
    """Cluster-granular selection: whole clusters of contiguous neuron indices
    come in when any of their neurons is selected."""
    # loaded neurons (positions 0..7) and clusters of 4 neuron indices
    loaded = np.array([0, 2, 3, 5, 6, 9, 12, 13], np.int32)
    # select position 1 (neuron 2, cluster 0) and position 6 (neuron 12, cluster 3)
    got = oracle.expand_clusters(loaded, np.array([1, 6], np.int32), 16, 4)
    assert got.tolist() == [0, 1, 2, 6, 7]           # neurons 0, 2, 3 and 12, 13
    # position 3 (neuron 5, cluster 1) brings neuron 6 too; cluster 2 holds only neuron 9
    assert oracle.expand_clusters(loaded, np.array([3], np.int32), 16, 4).tolist() == [3, 4]
    assert oracle.expand_clusters(loaded, np.array([5], np.int32), 16, 4).tolist() == [5]
    # clusters of one neuron change nothing; an empty selection stays empty
    S = np.array([0, 3, 7], np.int32)
    assert np.array_equal(oracle.expand_clusters(loaded, S, 16, 1), S)
    assert oracle.expand_clusters(loaded, np.zeros(0, np.int32), 16, 8).size == 0
    # brute force on random sets: the result is the positions whose cluster meets S
    rng = np.random.default_rng(11)
    for _ in range(20):
        N = int(rng.integers(8, 200))
        loaded = np.sort(rng.choice(N, int(rng.integers(1, N)), replace=False)).astype(np.int32)
        S = np.sort(rng.choice(len(loaded), int(rng.integers(0, len(loaded) + 1)), replace=False)).astype(np.int32)
        c = int(rng.choice([1, 2, 3, 32, 64]))
        hit = {int(loaded[s]) // c for s in S}
        ref = [p for p in range(len(loaded)) if int(loaded[p]) // c in hit]
        got = oracle.expand_clusters(loaded, S, N, c)
        assert got.tolist() == ref
        assert set(S.tolist()) <= set(got.tolist())
    with pytest.raises(ValueError):
        oracle.expand_clusters(loaded, S, N, 0)


def test_swiglu_closed_form():
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0])
    u = np.array([5.0, 2.0, 2.0, 1.0, 1.0])
    got = oracle.swiglu(g, u)
    ref = [0.0, 2.0 / (1 + np.exp(-1.0)), -2.0 / (1 + np.exp(1.0)), 30.0 / (1 + np.exp(-30.0)),
           -30.0 / (1 + np.exp(30.0))]
    assert np.allclose(got, ref, rtol=1e-15, atol=1e-300)


def test_spax_gate_up_special_cases():
    """Tiers on gate/up by |x|: every channel in the top tier is the dense
    activation pass; no channel at all gives silu(0) * 0 = 0; the tiers rank
    the input channels by |x|."""
    d, N = 256, 256                 # groups of 128 along the neuron axis
    Wg, Wu, _ = synth.layer_weights(71, 0, d, N)
    x = synth.tokens(72, 0, synth.T_DECODE, 1, d)[0]
    a, top, mid = oracle.spax_gate_up(x, Wg, Wu, 1.0, 0.0)
    assert len(top) == d and len(mid) == 0
    assert np.allclose(a, oracle.dense_act(Wg, Wu, x), rtol=1e-12, atol=1e-15)
    a0, top0, mid0 = oracle.spax_gate_up(x, Wg, Wu, 0.0, 0.0)
    assert len(top0) == 0 and len(mid0) == 0 and not a0.any()
    _, t, m = oracle.spax_gate_up(x, Wg, Wu, 0.25, 0.25)
    ax = np.abs(f32(x))
    assert ax[t].min() >= ax[m].max() and len(t) == len(m) == 64
    # a middle tier rebuilt from 8-bit codes stays close to the dense pass
    a8, _, _ = oracle.spax_gate_up(x, Wg, Wu, 0.0, 1.0, bits=8)
    ref = oracle.dense_act(Wg, Wu, x)
    assert np.abs(a8 - ref).max() <= 0.05 * np.abs(ref).max()


# --------------------------------------------------------- bf16 rounding


def _bf16_of(bits16):
    return float((np.asarray([bits16], np.uint32) << 16).view(np.float32)[0])


def test_bf16_round_fixed_cases():
    one = 0x3F800000
    f = lambda u: np.asarray([u], np.uint32).view(np.float32)[0]
    cases = [
        (one, 0x3F80),                 # exact
        (one + 0x8000, 0x3F80),        # 1 + 2^-8: a tie, the kept bit is 0 -> stays
        (one + 0x18000, 0x3F82),       # 1 + 3 * 2^-8: a tie, the kept bit is 1 -> up
        (one + 0x8001, 0x3F81),        # just above the tie -> up
        (one + 0x7FFF, 0x3F80),        # just below the tie -> down
        (0x3FFF8000, 0x4000),          # a tie that carries into the exponent (-> 2.0)
        (0xBF808000, 0xBF80),          # negative tie to even
        (0xBF818000, 0xBF82),          # negative tie, odd -> away from zero
        (0x7F800000, 0x7F80),          # inf
        (0xFF800000, 0xFF80),          # -inf
        (0x00000001, 0x0000),          # the smallest subnormal -> +0
        (0x00018000, 0x0002),          # subnormal tie, odd -> up
    ]
    for u, want in cases:
        got = int(oracle.bf16_round(np.array([f(u)], np.float32))[0])
        assert got == want, (hex(u), hex(got), hex(want))
    nan = oracle.bf16_round(np.array([np.nan], np.float32))[0]
    assert math.isnan(_bf16_of(nan))


def test_bf16_round_is_the_nearest_bf16():
    # every finite float32 rounds to the nearer of the two bf16 values around
    # it (distances in float64), an exact tie to the one with an even last bit
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]
    f = bits.view(np.float32)
    got = oracle.bf16_round(f).astype(np.uint32)
    lo = bits >> 16
    hi = lo + 1
    vf = f.astype(np.float64)
    vlo = (lo << 16).view(np.float32).astype(np.float64)
    vhi = (hi << 16).view(np.float32).astype(np.float64)
    dlo, dhi = np.abs(vf - vlo), np.abs(vhi - vf)
    want = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    # a value above the largest finite bf16 that is nearer to it stays finite;
    # one at or past the midpoint to 2^128 rounds to inf (hi = 0x7F80 there)
    assert np.array_equal(got, want)


# -------------------------------------------------------- decode stack


def _tiny_layer():
    one = int(synth.to_bf16_bits(np.array([1.0], np.float32))[0])
    Wg = np.array([[one, 0]], np.uint16)      # g = x0
    Wu = np.array([[0, one]], np.uint16)      # u = x1
    Wd = np.array([[one], [0]], np.uint16)    # the output goes to h0 only
    return Wg, Wu, Wd, np.array([0], np.int32), np.array([0], np.int32)


def _silu(z):
    return z * (1.0 + math.tanh(z / 2.0)) / 2.0     # z * sigmoid(z) by the tanh identity


def test_sparse_ffn_stack_two_layers_closed_form():
    # d = 2, one neuron: g = x0, u = x1, the output goes to h0 only.
    # Each layer reads x = bf16(float32(h / sqrt(mean(h^2) + 1e-5))).
    lay = _tiny_layer()
    h, xs = oracle.sparse_ffn_stack(np.array([2.0, 1.0]), [lay, lay])
    h0 = [2.0, 1.0]
    want_x = []
    for _ in range(2):
        r = 1.0 / math.sqrt((h0[0] ** 2 + h0[1] ** 2) / 2.0 + 1e-5)
        xb = synth.to_bf16_bits(np.array([h0[0] * r, h0[1] * r]))
        want_x.append([int(v) for v in xb])
        xf = synth.bf16_bits_to_f32(xb).astype(np.float64)
        h0 = [h0[0] + _silu(xf[0]) * xf[1], h0[1]]
    assert [[int(v) for v in row] for row in xs] == want_x
    # the first input by hand: r = 1/sqrt(2.50001) = 0.632454..., 2r = 1.264908
    # lies between the bf16 values 1.265625 (0x3FA2) and 1.2578125 (0x3FA1),
    # nearer the first; r lies between 0.6328125 (0x3F22) and 0.62890625
    # (0x3F21), nearer the first
    assert want_x[0] == [0x3FA2, 0x3F22]
    assert abs(h[0] - h0[0]) <= 1e-12 and h[1] == 1.0
    # an oracle that skipped the bf16 rounding of the second layer's input
    # (or its normalisation) would land measurably elsewhere
    x1 = synth.bf16_bits_to_f32(np.array(want_x[0], np.uint16)).astype(np.float64)
    h1 = 2.0 + _silu(x1[0]) * x1[1]
    r1 = 1.0 / math.sqrt((h1 ** 2 + 1.0) / 2.0 + 1e-5)
    assert abs(h1 + _silu(h1 * r1) * r1 - h[0]) > 1e-4
    assert abs(h1 + _silu(h1) * 1.0 - h[0]) > 1e-2


def test_sparse_ffn_stack_reduces_to_one_layer_and_composes():
    d, N = 96, 160
    rng_layers = []
    for l in range(3):
        Wg, Wu, Wd = synth.layer_weights(70, l, d, N)
        s = synth.lognormal_absact(70 + l, 1, N)[0]
        loaded, st = oracle.rank_loaded(s, s, 0.8, 0.2)
        S = oracle.select(synth.lognormal_absact(80 + l, 8, len(loaded)), 8, 1, len(loaded), st, 16,
                          oracle.cnt(0.5, N))[0]
        rng_layers.append((Wg, Wu, Wd, loaded, S))
    h0 = synth.normal(71, 0, 0, d)
    # one layer: h + FFN(bf16(h / rms(h)))
    h1, xs = oracle.sparse_ffn_stack(h0, rng_layers[:1])
    x0 = synth.to_bf16_bits(h0 / np.sqrt(np.mean(h0 ** 2) + 1e-5))
    assert np.array_equal(xs[0], x0)
    Wg, Wu, Wd, loaded, S = rng_layers[0]
    assert np.allclose(h1, h0 + oracle.sparse_ffn(Wg, Wu, Wd, loaded, S, x0), rtol=0, atol=1e-12)
    # three layers = one, then the other two on its output
    h3, xs3 = oracle.sparse_ffn_stack(h0, rng_layers)
    h3b, xs3b = oracle.sparse_ffn_stack(h1, rng_layers[1:])
    assert np.array_equal(h3, h3b) and np.array_equal(xs3[1:], xs3b)
    # the layers do not commute (each reads the stream the previous one wrote)
    h3r, _ = oracle.sparse_ffn_stack(h0, rng_layers[::-1])
    assert np.max(np.abs(h3r - h3)) > 1e-6


def test_sparse_ffn_stack_empty_sets_leave_h():
    d, N = 64, 80
    Wg, Wu, Wd = synth.layer_weights(72, 0, d, N)
    loaded = np.arange(N, dtype=np.int32)
    h0 = synth.normal(73, 0, 0, d)
    h, xs = oracle.sparse_ffn_stack(h0, [(Wg, Wu, Wd, loaded, np.zeros(0, np.int32))] * 4)
    assert np.array_equal(h, h0)
    x0 = synth.to_bf16_bits(h0 / np.sqrt(np.mean(h0 ** 2) + 1e-5))
    assert all(np.array_equal(x, x0) for x in xs)


def test_rms_norm_input_scale_invariance():
    # the layer input does not change when h is scaled by a power of two
    # (the 1e-5 epsilon aside, which a large stream makes negligible)
    h = synth.normal(74, 0, 0, 512) * 100.0
    assert np.array_equal(oracle.rms_norm_bf16(h), oracle.rms_norm_bf16(h * 4.0))
    x = synth.bf16_bits_to_f32(oracle.rms_norm_bf16(h)).astype(np.float64)
    assert abs(np.sqrt(np.mean(x ** 2)) - 1.0) < 4e-3   # unit RMS up to bf16 rounding


def test_spax_encode_3bit_ramp_layout():
    # a group whose values are exactly mn + q*scale for q = 0..7 (scale = 1/8):
    # the codes are the ramp itself, and the stream packs element i at bits
    # 3i..3i+2, so 8 codes fill 3 bytes and codes straddle byte boundaries
    d, N, group = 16, 1, 8
    vals = np.array([0.0, 0.125, 0.25, 0.375, 0.5, 0.625, 0.75, 0.875] * 2)
    Wd = bf16(vals.reshape(d, N))
    codes, params = oracle.spax_encode(Wd, 3, group)
    assert codes.shape == (1, 6)
    ramp = sum(q << (3 * q) for q in range(8))        # 0b111110101100011010001000
    want = list(ramp.to_bytes(3, "little")) * 2
    assert [int(b) for b in codes[0]] == want
    assert np.allclose(params[0, :, 0], 0.125) and np.allclose(params[0, :, 1], 0.0)
    # the decoder reads the same stream back: mid tier only, a = 1 -> y = w exactly
    y = oracle.spax_down(np.ones(N, np.float32), Wd, codes, params, np.zeros(0, np.int32),
                         np.zeros(1, np.int32), bits=3, group=group)
    assert np.array_equal(y, vals)
