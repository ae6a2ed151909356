"""GPU parity of the tcgen05 activation GEMM: the profiler score (Eq. 1) and
the prefill activation matrix |A| of si_select_dynamic, plus the selection it
drives. Full-size shapes are checked on sampled neurons / token rows that the
oracle computes one by one."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import Guarded, dev, dev_bf16, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def si():
    import activation_sparse_gb300 as si
    return si


PROFILE_CASES = [
    # d, N, T (calibration tokens), neurons sampled for the oracle (None = all)
    (256, 1024, 128, None),       # single-layer workload
    (256, 1000, 100, None),       # ragged N and T
    (128, 130, 1, None),          # one token, ragged tile
    (256, 1000, 600, None),       # 5 token tiles: clusters of 4 with padding tiles
    (256, 300, 300, None),        # 3 token tiles: clusters of 2 with a padding tile
    (2048, 8192, 4096, 96),       # Llama3.2-1B layer, 4096 calibration tokens
    (3072, 8192, 512, 64),        # Llama3.2-3B width
]


@pytest.mark.parametrize("d,N,T,sample", PROFILE_CASES)
def test_profile_scores(si, d, N, T, sample):
    Wg, Wu, _ = synth.layer_weights(60, 0, d, N)
    X = synth.tokens(60, 0, synth.T_CALIB, T, d)
    scores = Guarded((N,), torch().float32, fill=0.0)
    si.si_profile_scores(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(X), scores.t)
    got = scores.numpy().astype(np.float64)
    idx = np.arange(N) if sample is None else np.sort(np.random.default_rng(0).choice(N, sample, replace=False))
    ref = oracle.profile_scores(Wg[idx], Wu[idx], X)
    rel = np.abs(got[idx] - ref) / np.maximum(ref, 1e-30)
    assert rel.max() < 1e-3, rel.max()
    # scores accumulate over calls
    si.si_profile_scores(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(X), scores.t)
    got2 = scores.numpy().astype(np.float64)
    assert np.allclose(got2, 2 * got, rtol=1e-5)


SELECT_CASES = [
    # d, N, gamma, delta, phi, alpha, T, B, sampled rows (None = all)
    (256, 1024, 0.7, 0.2, 0.4, 64, 32, 1, None),          # single-layer workload
    (2048, 8192, 0.7, 0.2, 0.4, 1024, 512, 1, 12),        # Llama3.2-1B prompt
    (3072, 8192, 0.7, 0.25, 0.5, 1024, 1024, 1, 8),       # Llama3.2-3B prompt
    (2048, 11008, 0.8, 0.25, 0.5, 1024, 256, 8, 8),       # Qwen2.5-3B, 8 prompts
    (512, 700, 0.9, 0.3, 0.5, 40, 77, 2, None),           # ragged M and neurons
    (256, 1024, 0.7, 0.2, 0.4, 64, 150, 2, None),         # 3 token tiles: a padding tile in the cluster
]


@pytest.mark.parametrize("d,N,gamma,delta,phi,alpha,T,B,sample", SELECT_CASES)
def test_select_dynamic(si, d, N, gamma, delta, phi, alpha, T, B, sample):
    Wg, Wu, Wd = synth.layer_weights(61, 0, d, N, 1.5 if B > 1 else 1.0)
    s = synth.lognormal_absact(61, 1, N)[0]
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), gamma, delta)
    loaded, st = oracle.rank_loaded(s, s, gamma, delta)
    X = synth.tokens(62, 0, synth.T_PROMPT, B * T, d)
    n_sel = si.si_count(phi, N)
    S = Guarded((B, n_sel), torch().int32, fill=-1)
    A = Guarded((B * T, layer.n_pad), torch().float32, fill=float("nan"))
    si.si_select_dynamic(layer, dev_bf16(X), T, B, alpha, phi, S.t, A.t)
    got_A = A.numpy()
    assert not got_A[:, layer.n_loaded:].any()                 # pad neurons give zero
    rows = np.arange(B * T) if sample is None else np.sort(np.random.default_rng(1).choice(B * T, sample, False))
    ref_A = oracle.absact(Wg, Wu, loaded, X[rows])
    err = np.abs(got_A[rows, :layer.n_loaded] - ref_A)
    assert err.max() <= 1e-3 * ref_A.max() + 1e-6, err.max() / ref_A.max()
    got_S = S.numpy()
    # the selection is the exact selection of the |A| the GPU computed
    S2 = Guarded((B, n_sel), torch().int32, fill=-1)
    si.si_select_from_absact(layer, A.t, T, B, alpha, phi, S2.t)
    assert np.array_equal(got_S, S2.numpy())
    # and agrees with the oracle's selection on its own |A| up to near-ties
    if sample is None:
        ref_S = oracle.select(oracle.absact(Wg, Wu, loaded, X).astype(np.float32), T, B, len(loaded), st, alpha, n_sel)
        for b in range(B):
            overlap = len(np.intersect1d(got_S[b], ref_S[b])) / n_sel
            assert overlap >= 0.98, overlap
    assert np.all(np.diff(got_S, axis=1) > 0)                  # ascending, distinct
    assert np.all(st[got_S].sum(axis=1) == int(st.sum()))      # every static neuron kept
    layer.close()


def test_prefill_absact_matches_select_dynamic(si):
    d, N, T, B = 2048, 8192, 512, 1
    Wg, Wu, Wd = synth.layer_weights(63, 0, d, N)
    s = synth.lognormal_absact(63, 1, N)[0]
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), 0.7, 0.2)
    X = dev_bf16(synth.tokens(64, 0, synth.T_PROMPT, T, d))
    A1 = Guarded((T, layer.n_pad), torch().float32, fill=float("nan"))
    A2 = Guarded((T, layer.n_pad), torch().float32, fill=float("nan"))
    n_sel = si.si_count(0.4, N)
    S1 = Guarded((1, n_sel), torch().int32)
    S2 = Guarded((1, n_sel), torch().int32)
    si.si_prefill_absact(layer, X, T, B, A1.t)
    si.si_select_from_absact(layer, A1.t, T, B, 1024, 0.4, S1.t)
    si.si_select_dynamic(layer, X, T, B, 1024, 0.4, S2.t, A2.t)
    assert np.array_equal(A1.numpy().view(np.uint32), A2.numpy().view(np.uint32))
    assert np.array_equal(S1.numpy(), S2.numpy())
    layer.close()


GEMM_TILES = [64, 80, 96, 112, 128]


@pytest.fixture
def forced_tile(si):
    yield si.si_set_gemm_tile
    si.si_set_gemm_tile(0)


@pytest.mark.parametrize("bnn", GEMM_TILES)
def test_absact_every_tile_width(si, forced_tile, bnn):
    """Each neuron-tile width gives bit-identical |A| (the K order of every
    element is the same) and matches the oracle; ragged tokens and neurons,
    two token tiles, several neuron tiles and a partial last one."""
    d, N, T = 512, 1500, 300
    Wg, Wu, Wd = synth.layer_weights(65, 0, d, N)
    s = synth.lognormal_absact(65, 1, N)[0]
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), 0.7, 0.2)
    loaded, _ = oracle.rank_loaded(s, s, 0.7, 0.2)
    X = synth.tokens(66, 0, synth.T_PROMPT, T, d)
    Xd = dev_bf16(X)
    forced_tile(0)
    A0 = Guarded((T, layer.n_pad), torch().float32, fill=float("nan"))
    si.si_prefill_absact(layer, Xd, T, 1, A0.t)
    forced_tile(bnn)
    A1 = Guarded((T, layer.n_pad), torch().float32, fill=float("nan"))
    si.si_prefill_absact(layer, Xd, T, 1, A1.t)
    got = A1.numpy()
    assert np.array_equal(got.view(np.uint32), A0.numpy().view(np.uint32))
    ref = oracle.absact(Wg, Wu, loaded, X)
    err = np.abs(got[:, :layer.n_loaded] - ref)
    assert err.max() <= 1e-3 * ref.max() + 1e-6, err.max() / ref.max()
    assert not got[:, layer.n_loaded:].any()
    layer.close()


@pytest.mark.parametrize("bnn", GEMM_TILES)
def test_profile_scores_every_tile_width(si, forced_tile, bnn):
    d, N, T = 256, 1000, 600
    Wg, Wu, _ = synth.layer_weights(67, 0, d, N)
    X = synth.tokens(67, 0, synth.T_CALIB, T, d)
    forced_tile(bnn)
    scores = Guarded((N,), torch().float32, fill=0.0)
    si.si_profile_scores(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(X), scores.t)
    ref = oracle.profile_scores(Wg, Wu, X)
    rel = np.abs(scores.numpy().astype(np.float64) - ref) / np.maximum(ref, 1e-30)
    assert rel.max() < 1e-3, rel.max()


def test_tile_choice_fills_the_sms(si):
    """The per-launch width minimises waves * (width + 24), wider on ties."""
    sms = torch().cuda.get_device_properties(0).multi_processor_count

    def cost(M, N, b):
        ctas = -(-N // b) * -(-M // 256)
        return -(-ctas // sms) * (b + 24)

    for M, N in [(512, 5734), (4096, 8192), (1024, 5734), (256, 1000), (8 * 256, 8812), (512, 9728)]:
        b = si.si_gemm_tile_for(M, N)
        assert b in GEMM_TILES
        best = min(cost(M, N, c) for c in GEMM_TILES)
        assert cost(M, N, b) == best
        assert all(cost(M, N, c) > best for c in GEMM_TILES if c > b)
    if sms >= 144:
        assert si.si_gemm_tile_for(512, 5734) == 80   # 144 CTAs instead of 90


def test_weight_aware_salience(si):
    """WiSparse-style ranking key |a_n| * ||Wd[:, n]||_2: the handle's norms,
    the prefill matrix and the selection it drives, against the oracle; the
    default key comes back when the switch is off."""
    from gpu_util import device_view
    d, N, T = 512, 1500, 96
    Wg, Wu, Wd = synth.layer_weights(68, 0, d, N)
    s = synth.lognormal_absact(68, 1, N)[0]
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), 0.7, 0.2)
    loaded, st = oracle.rank_loaded(s, s, 0.7, 0.2)
    nl, n_pad = layer.n_loaded, layer.n_pad
    norms = device_view(si.si_layer_norms(layer), (n_pad,), "<f4").cpu().numpy()
    ref_norms = oracle.down_norms(Wd, loaded)
    assert np.allclose(norms[:nl], ref_norms, rtol=5e-6, atol=0)   # float32 sums of 16 + 5 terms per lane path
    assert not norms[nl:].any()
    X = synth.tokens(69, 0, synth.T_PROMPT, T, d)
    Xd = dev_bf16(X)
    A0 = Guarded((T, n_pad), torch().float32, fill=float("nan"))
    si.si_prefill_absact(layer, Xd, T, 1, A0.t)
    si.si_layer_set_salience(layer, True)
    A1 = Guarded((T, n_pad), torch().float32, fill=float("nan"))
    si.si_prefill_absact(layer, Xd, T, 1, A1.t)
    ref = oracle.absact(Wg, Wu, loaded, X) * ref_norms[None, :]
    got = A1.numpy()
    assert np.abs(got[:, :nl] - ref).max() <= 1e-3 * ref.max()
    assert not got[:, nl:].any()
    # the selection on salience is the exact selection of the matrix the GPU computed
    alpha, phi = 64, 0.4
    n_sel = si.si_count(phi, N)
    S1 = Guarded((1, n_sel), torch().int32, fill=-1)
    S2 = Guarded((1, n_sel), torch().int32, fill=-1)
    si.si_select_dynamic(layer, Xd, T, 1, alpha, phi, S1.t)
    si.si_select_from_absact(layer, A1.t, T, 1, alpha, phi, S2.t)
    assert np.array_equal(S1.numpy(), S2.numpy())
    ref_S = oracle.select(ref.astype(np.float32), T, 1, nl, st, alpha, n_sel)
    overlap = len(np.intersect1d(S1.numpy()[0], ref_S[0])) / n_sel
    assert overlap >= 0.98, overlap
    # and it differs from the |a| ranking somewhere (the norms matter)
    S0 = Guarded((1, n_sel), torch().int32, fill=-1)
    si.si_select_from_absact(layer, A0.t, T, 1, alpha, phi, S0.t)
    assert not np.array_equal(S0.numpy(), S1.numpy())
    # switching back restores |a| bit for bit
    si.si_layer_set_salience(layer, False)
    A2 = Guarded((T, n_pad), torch().float32, fill=float("nan"))
    si.si_prefill_absact(layer, Xd, T, 1, A2.t)
    assert np.array_equal(A2.numpy().view(np.uint32), A0.numpy().view(np.uint32))
    layer.close()
