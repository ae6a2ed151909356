"""GPU parity: selective loading (ranking + packing), score-file merge, and the
prefill selection steps a4..a6 on a given |A| matrix. Integer results must be
bit-exact against the oracle; both sides read the same seeded inputs."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import Guarded, dev, dev_bf16, device_view, torch, u16_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def si():
    import activation_sparse_gb300 as si
    return si


def scores_of(kind, seed, N):
    if kind == "lognormal":
        return synth.lognormal_absact(seed, 1, N)[0]
    if kind == "ties":
        return synth.tie_heavy_absact(seed, 1, N, levels=5)[0]
    if kind == "signed":
        return (synth.normal(seed, 0, synth.T_SCORES_A, N) * 3).astype(np.float32)
    raise ValueError(kind)


def layer_buffers(layer):
    p_loaded, p_static, p_packed = layer.buffers()
    loaded = device_view(p_loaded, (layer.n_loaded,), "<i4").cpu().numpy()
    st = device_view(p_static, (layer.n_loaded,), "|u1").cpu().numpy()
    packed = device_view(p_packed, (layer.n_pad, 3, layer.d), "<i2")
    return loaded, st, packed


# --------------------------------------------------------------- loading

PACK_CASES = [
    # d, N, gamma, delta, score kind
    (256, 1024, 0.7, 0.2, "lognormal"),       # single-layer d=256 workload
    (2048, 8192, 0.7, 0.2, "lognormal"),      # Llama3.2-1B FFN shape
    (3072, 8192, 0.7, 0.25, "ties"),          # Llama3.2-3B FFN shape, tied scores
    (2048, 11008, 0.8, 0.25, "lognormal"),    # Qwen2.5-3B FFN shape
    (64, 100, 1.0, 0.0, "ties"),              # everything loaded, nothing static
    (64, 37, 0.5, 0.5, "signed"),             # all loaded neurons static, negative scores
    (128, 1, 1.0, 1.0, "lognormal"),          # a single neuron
]


@pytest.mark.parametrize("d,N,gamma,delta,kind", PACK_CASES)
def test_pack_loaded_parity(si, d, N, gamma, delta, kind):
    Wg, Wu, Wd = synth.layer_weights(21, 0, d, N)
    task = scores_of(kind, 1, N)
    model = scores_of(kind, 2, N)
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(task), dev(model), gamma, delta)
    torch().cuda.synchronize()
    ref_loaded, ref_static = oracle.rank_loaded(task, model, gamma, delta)
    assert layer.n_loaded == len(ref_loaded) and layer.n_static == int(ref_static.sum())
    loaded, st, packed = layer_buffers(layer)
    assert np.array_equal(loaded, ref_loaded)
    assert np.array_equal(st, ref_static)
    pk = packed.cpu().numpy().view(np.uint16)
    n = layer.n_loaded
    assert np.array_equal(pk[:n, 0, :], Wg[ref_loaded])
    assert np.array_equal(pk[:n, 1, :], Wu[ref_loaded])
    assert np.array_equal(pk[:n, 2, :], Wd[:, ref_loaded].T)
    assert not pk[n:].any()                         # tile padding is zero
    assert layer.n_pad % 128 == 0 and layer.n_pad >= n
    layer.close()


def test_pack_single_score_file_is_top_gamma(si):
    d, N = 64, 512
    Wg, Wu, Wd = synth.layer_weights(22, 0, d, N)
    s = scores_of("lognormal", 5, N)
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), 0.7, 0.2)
    loaded, st, _ = layer_buffers(layer)
    order = np.argsort(-s, kind="stable")
    assert set(loaded) == set(order[:si.si_count(0.7, N)])
    assert set(loaded[st == 1]) == set(order[:si.si_count(0.2, N)])
    layer.close()


def test_merge_scores_bit_exact(si):
    N = 11008
    files = [synth.lognormal_absact(s, 1, N)[0] * 1000 for s in range(4)]
    toks = [4096, 128, 77, 100000]
    out = Guarded((N,), torch().float32)
    si.si_merge_scores([dev(f) for f in files], toks, out.t)
    ref = oracle.merge_scores(files, toks)
    assert np.array_equal(out.numpy().view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------- selection

SEL_CASES = [
    # N, gamma, delta, phi, alpha, T, B, |A| kind
    (1024, 0.7, 0.2, 0.4, 64, 32, 1, "lognormal"),        # single-layer workload
    (8192, 0.7, 0.2, 0.4, 1024, 512, 1, "lognormal"),     # Llama3.2-1B prompt
    (8192, 0.7, 0.25, 0.5, 1024, 1024, 1, "lognormal"),   # Llama3.2-3B prompt
    (11008, 0.8, 0.25, 0.5, 1024, 256, 8, "lognormal"),   # Qwen2.5-3B, 8 prompts
    (1024, 0.7, 0.2, 0.4, 64, 32, 1, "ties"),
    (2000, 0.7, 0.3, 0.4, 100, 40, 3, "ties"),
    (1024, 0.7, 0.2, 0.4, 1, 5, 1, "lognormal"),          # alpha = 1
    (1024, 0.7, 0.2, 0.4, 717, 3, 1, "lognormal"),        # alpha = n_loaded
    (1024, 0.7, 0.2, 0.4, 64, 1, 1, "ties"),              # one token
    (1024, 0.7, 0.2, 0.2, 64, 16, 2, "lognormal"),        # beta = 0
    (1024, 0.7, 0.2, 0.7, 64, 16, 1, "lognormal"),        # phi = gamma: every loaded neuron
    (1024, 0.7, 0.0, 0.4, 64, 16, 1, "ties"),             # no static neurons
    (1000, 1.0, 0.3, 0.4, 50, 8, 1, "zeros"),             # all |A| equal (zero)
    (33, 1.0, 0.1, 0.5, 7, 9, 2, "ties"),                 # tiny, ragged word
    (256, 1.0, 0.1, 0.5, 200, 2100, 1, "lognormal"),      # counts above 2047: top-beta's general path
    (600, 0.7, 0.2, 0.4, 64, 32, 1, "narrow"),            # every key in one top-digit bin: ranked directly
    (1024, 0.7, 0.2, 0.4, 64, 32, 1, "narrow"),           # same, 717 keys: top-alpha's radix passes
]


def absact_of(kind, seed, rows, n, ld):
    if kind == "lognormal":
        A = synth.lognormal_absact(seed, rows, n)
    elif kind == "ties":
        A = synth.tie_heavy_absact(seed, rows, n, levels=6)
    elif kind == "narrow":
        # distinct values in [1, 1.12): one bin of the 11-bit top digit
        A = (1.0 + 0.12 * np.random.default_rng(seed).random((rows, n))).astype(np.float32)
    else:
        A = np.zeros((rows, n), np.float32)
    out = np.full((rows, ld), 1e30, np.float32)   # columns past n_loaded must be ignored
    out[:, :n] = A
    return out


@pytest.mark.parametrize("N,gamma,delta,phi,alpha,T,B,kind", SEL_CASES)
def test_select_from_absact_bit_exact(si, N, gamma, delta, phi, alpha, T, B, kind):
    d = 64
    Wg, Wu, Wd = synth.layer_weights(23, 0, d, N)
    s = scores_of("lognormal", 7, N)
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), gamma, delta)
    _, st, _ = layer_buffers(layer)
    nl = layer.n_loaded
    n_sel = si.si_count(phi, N)
    ld = layer.n_pad + 4
    A = absact_of(kind, 31, B * T, nl, ld)
    words = (nl + 31) // 32
    S = Guarded((B, n_sel), torch().int32, fill=-1)
    tm = Guarded((B * T, words), torch().int32, fill=-1)
    cnt = Guarded((B, nl), torch().int32, fill=-1)
    si.si_select_from_absact(layer, dev(A), T, B, alpha, phi, S.t, tm.t, cnt.t)
    ref_S, ref_cnt, ref_sel = oracle.select(A, T, B, nl, st, alpha, n_sel, want_counts=True, want_sel=True)
    got_S = S.numpy()
    got_cnt = cnt.numpy().view(np.uint32)
    got_tm = tm.numpy().view(np.uint32)
    bits = np.zeros((B * T, words * 32), np.uint64)
    bits[:, :nl] = ref_sel
    ref_tm = (bits.reshape(B * T, words, 32) << np.arange(32, dtype=np.uint64)).sum(axis=2).astype(np.uint32)
    assert np.array_equal(got_tm, ref_tm)
    assert np.array_equal(got_cnt, ref_cnt)
    assert np.array_equal(got_S, ref_S)
    # without optional outputs the same S comes back
    S2 = Guarded((B, n_sel), torch().int32, fill=-1)
    si.si_select_from_absact(layer, dev(A), T, B, alpha, phi, S2.t)
    assert np.array_equal(S2.numpy(), ref_S)
    layer.close()


def test_select_rejects_bad_arguments(si):
    N, d = 256, 64
    Wg, Wu, Wd = synth.layer_weights(24, 0, d, N)
    s = scores_of("lognormal", 8, N)
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), 0.5, 0.2)
    A = dev(np.ones((4, layer.n_pad), np.float32))
    S = dev(np.zeros((1, 200), np.int32))
    for alpha, phi in [(0, 0.3), (layer.n_loaded + 1, 0.3), (4, 0.1), (4, 0.6)]:
        with pytest.raises(si.SIError) as e:
            si.si_select_from_absact(layer, A, 4, 1, alpha, phi, S)
        assert e.value.code == si.SI_ERR_INVALID_ARG
    layer.close()
