"""GPU parity: the sparse SwiGLU decode FFN on the computed set (one token per
sequence) against the oracle, within the FFN tolerance."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL, Guarded, dev, dev_bf16, rel_err, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def si():
    import activation_sparse_gb300 as si
    return si


class Case:
    def __init__(self, si, d, N, gamma, delta, phi, alpha, T, B, sigma=1.0, seed=40):
        self.Wg, self.Wu, self.Wd = synth.layer_weights(seed, 0, d, N, sigma)
        s = synth.lognormal_absact(seed, 1, N)[0]
        self.layer = si.si_pack_loaded(dev_bf16(self.Wg), dev_bf16(self.Wu), dev_bf16(self.Wd), dev(s), dev(s),
                                       gamma, delta)
        self.loaded, self.st = oracle.rank_loaded(s, s, gamma, delta)
        self.n_sel = si.si_count(phi, N)
        nl = len(self.loaded)
        A = synth.lognormal_absact(seed + 1, B * T, nl)
        self.S = oracle.select(A, T, B, nl, self.st, min(alpha, nl), self.n_sel)
        self.d, self.N, self.B = d, N, B


DECODE_CASES = [
    # d, N, gamma, delta, phi, alpha, T, B, sigma
    (256, 1024, 0.7, 0.2, 0.4, 64, 32, 1, 1.0),          # single-layer workload
    (2048, 8192, 0.7, 0.2, 0.4, 1024, 64, 1, 1.0),       # Llama3.2-1B layer
    (3072, 8192, 0.7, 0.25, 0.5, 1024, 64, 1, 1.0),      # Llama3.2-3B layer
    (2048, 11008, 0.8, 0.25, 0.5, 1024, 16, 8, 1.5),     # Qwen2.5-3B layer, 8 sequences
    (2048, 11008, 0.8, 0.25, 0.5, 1024, 16, 3, 1.5),     # 3 sequences
    (4096, 2048, 0.5, 0.2, 0.3, 64, 8, 1, 1.0),          # widest supported d
    (64, 100, 1.0, 0.0, 1.0, 8, 4, 1, 1.0),              # phi = gamma = 1: dense FFN
    (2048, 8192, 1.0, 0.0, 1.0, 1024, 8, 1, 1.0),        # a dense Llama3.2-1B layer (outside the layer range)
    (1088, 300, 0.9, 0.1, 0.2, 8, 4, 2, 1.0),            # d not a multiple of 256
]


@pytest.mark.parametrize("d,N,gamma,delta,phi,alpha,T,B,sigma", DECODE_CASES)
def test_sparse_decode_parity(si, d, N, gamma, delta, phi, alpha, T, B, sigma):
    c = Case(si, d, N, gamma, delta, phi, alpha, T, B, sigma)
    S_dev = dev(c.S)
    if B > 1:
        si.si_decode_plan(c.layer, S_dev, c.n_sel, B)
    # batch 1: two calls without a plan, then three with one (the first of
    # them reads the plan after its dependency wait, the later ones stream
    # the planned records before it)
    for tok in range(2 if B > 1 else 5):
        if B == 1 and tok == 2:
            si.si_decode_plan(c.layer, S_dev, c.n_sel, 1)
        x = synth.tokens(41, tok, synth.T_DECODE, B, d)
        y = Guarded((B, d), torch().float32, fill=float("nan"))
        si.si_sparse_ffn_decode(c.layer, S_dev, c.n_sel, B, dev_bf16(x), y.t)
        got = y.numpy()
        for b in range(B):
            ref = oracle.sparse_ffn(c.Wg, c.Wu, c.Wd, c.loaded, c.S[b], x[b])
            err = rel_err(got[b], ref)
            assert err <= TOL, (tok, b, err)
            assert err <= 2e-5      # fp32 accumulation of bf16 products stays far inside the bar
    c.layer.close()


MMA_CASES = [
    # d, N, gamma, delta, phi, alpha, T, B, sigma: batches at d = 1024 and 2048 take the tensor-core kernel
    (1024, 4096, 0.7, 0.2, 0.4, 256, 8, 8, 1.0),
    (1024, 600, 0.9, 0.1, 0.3, 32, 4, 2, 1.0),           # a few records per CTA: short last batches
    (2048, 11008, 0.8, 0.25, 0.5, 1024, 16, 5, 1.5),
    (2048, 3000, 1.0, 0.0, 1.0, 64, 4, 8, 1.0),          # phi = 1: every sequence computes every neuron
]


@pytest.mark.parametrize("d,N,gamma,delta,phi,alpha,T,B,sigma", MMA_CASES)
def test_batch_decode_tensor_core_path(si, d, N, gamma, delta, phi, alpha, T, B, sigma):
    c = Case(si, d, N, gamma, delta, phi, alpha, T, B, sigma, seed=48)
    S_dev = dev(c.S)
    si.si_decode_plan(c.layer, S_dev, c.n_sel, B)
    x = synth.tokens(49, 0, synth.T_DECODE, B, d)
    ys = []
    for _ in range(2):
        y = Guarded((B, d), torch().float32, fill=float("nan"))
        si.si_sparse_ffn_decode(c.layer, S_dev, c.n_sel, B, dev_bf16(x), y.t)
        y.check()
        ys.append(y.numpy())
    assert np.array_equal(ys[0].view(np.uint32), ys[1].view(np.uint32))   # deterministic
    for b in range(B):
        ref = oracle.sparse_ffn(c.Wg, c.Wu, c.Wd, c.loaded, c.S[b], x[b])
        assert rel_err(ys[0][b], ref) <= 2e-5, b
    c.layer.close()


def test_batch_decode_disjoint_sets(si):
    # four sequences with disjoint computed sets: the union is four times a
    # set and every record serves exactly one sequence
    d, N, B = 2048, 4096, 4
    c = Case(si, d, N, 0.9, 0.0, 0.2, 64, 4, 1, seed=50)
    nl = len(c.loaded)
    n = nl // (2 * B)
    S = np.stack([np.arange(b, nl, B, dtype=np.int32)[:n] for b in range(B)])
    S_dev = dev(S)
    si.si_decode_plan(c.layer, S_dev, n, B)
    x = synth.tokens(51, 0, synth.T_DECODE, B, d)
    y = Guarded((B, d), torch().float32, fill=float("nan"))
    si.si_sparse_ffn_decode(c.layer, S_dev, n, B, dev_bf16(x), y.t)
    got = y.numpy()
    for b in range(B):
        ref = oracle.sparse_ffn(c.Wg, c.Wu, c.Wd, c.loaded, S[b], x[b])
        assert rel_err(got[b], ref) <= 2e-5, b
    c.layer.close()


def test_sparse_decode_dense_limit_matches_library_dense_ffn(si):
    # every neuron loaded and computed: the output is the dense SwiGLU FFN (numpy)
    from scipy.special import expit
    d, N = 512, 768
    c = Case(si, d, N, 1.0, 0.0, 1.0, 16, 4, 1)
    assert np.array_equal(c.S[0], np.arange(N))
    x = synth.tokens(42, 0, synth.T_DECODE, 1, d)
    y = Guarded((1, d), torch().float32)
    si.si_sparse_ffn_decode(c.layer, dev(c.S), N, 1, dev_bf16(x), y.t)
    xf = synth.bf16_bits_to_f32(x[0]).astype(np.float64)
    g = synth.bf16_bits_to_f32(c.Wg).astype(np.float64) @ xf
    u = synth.bf16_bits_to_f32(c.Wu).astype(np.float64) @ xf
    ref = synth.bf16_bits_to_f32(c.Wd).astype(np.float64) @ (g * expit(g) * u)
    assert rel_err(y.numpy()[0], ref) <= 2e-5
    c.layer.close()


def test_sparse_decode_edge_sets(si):
    d, N = 256, 1024
    c = Case(si, d, N, 0.7, 0.0, 0.4, 64, 8, 1)
    x = synth.tokens(43, 0, synth.T_DECODE, 1, d)
    for S in (np.zeros((1, 0), np.int32), np.array([[5]], np.int32), np.array([[c.layer.n_loaded - 1]], np.int32),
              np.arange(c.layer.n_loaded, dtype=np.int32)[None, :]):
        y = Guarded((1, d), torch().float32, fill=float("nan"))
        si.si_sparse_ffn_decode(c.layer, dev(S), S.shape[1], 1, dev_bf16(x), y.t)
        ref = oracle.sparse_ffn(c.Wg, c.Wu, c.Wd, c.loaded, S[0], x[0])
        got = y.numpy()[0]
        if S.shape[1] == 0:
            assert np.all(got == 0)
        else:
            assert rel_err(got, ref) <= 2e-5
    c.layer.close()


@pytest.mark.parametrize("planned", [False, True])
def test_sparse_decode_deterministic_and_repeatable(si, planned):
    d, N = 2048, 8192
    c = Case(si, d, N, 0.7, 0.2, 0.4, 1024, 16, 1)
    x = dev_bf16(synth.tokens(44, 0, synth.T_DECODE, 1, d))
    S = dev(c.S)
    if planned:
        si.si_decode_plan(c.layer, S, c.n_sel, 1)
    ys = []
    for _ in range(5):
        y = Guarded((1, d), torch().float32)
        si.si_sparse_ffn_decode(c.layer, S, c.n_sel, 1, x, y.t)
        ys.append(y.numpy())
    for y in ys[1:]:
        assert np.array_equal(y.view(np.uint32), ys[0].view(np.uint32))
    ref = oracle.sparse_ffn(c.Wg, c.Wu, c.Wd, c.loaded, c.S[0], synth.tokens(44, 0, synth.T_DECODE, 1, d)[0])
    assert rel_err(ys[0][0], ref) <= 2e-5
    c.layer.close()


def test_decode_plan_required_for_batches(si):
    c = Case(si, 256, 1024, 0.7, 0.2, 0.4, 64, 8, 2)
    x = dev_bf16(synth.tokens(45, 0, synth.T_DECODE, 2, 256))
    y = dev(np.zeros((2, 256), np.float32))
    with pytest.raises(si.SIError) as e:
        si.si_sparse_ffn_decode(c.layer, dev(c.S), c.n_sel, 2, x, y)
    assert e.value.code == si.SI_ERR_INVALID_ARG
    c.layer.close()


def test_planned_b1_decode_pipelined_back_to_back(si):
    """Batch-1 decode with a plan: from the second call on, a launch streams its
    records while the previous launch is still finishing (programmatic
    dependent launch). Alternate two layers without host syncs and check every
    output against the oracle."""
    d, N = 2048, 8192
    cases = [Case(si, d, N, 0.7, 0.2, 0.4, 1024, 16, 1, seed=s) for s in (70, 71)]
    S_dev = [dev(c.S) for c in cases]
    for c, S in zip(cases, S_dev):
        si.si_decode_plan(c.layer, S, c.n_sel, 1)
    toks = 6
    xs = [synth.tokens(72, t, synth.T_DECODE, 1, d) for t in range(toks)]
    xd = [dev_bf16(x) for x in xs]
    ys = [[Guarded((1, d), torch().float32, fill=float("nan")) for _ in range(toks)] for _ in cases]
    for t in range(toks):
        for k, c in enumerate(cases):
            si.si_sparse_ffn_decode(c.layer, S_dev[k], c.n_sel, 1, xd[t], ys[k][t].t)
    torch().cuda.synchronize()
    for k, c in enumerate(cases):
        for t in range(toks):
            ref = oracle.sparse_ffn(c.Wg, c.Wu, c.Wd, c.loaded, c.S[0], xs[t][0])
            assert rel_err(ys[k][t].numpy()[0], ref) <= 2e-5, (k, t)
    # the unplanned path agrees within fp32 summation-order noise
    y_plain = Guarded((1, d), torch().float32)
    c2 = Case(si, d, N, 0.7, 0.2, 0.4, 1024, 16, 1, seed=70)
    si.si_sparse_ffn_decode(c2.layer, dev(c2.S), c2.n_sel, 1, xd[toks - 1], y_plain.t)
    assert rel_err(y_plain.numpy()[0], ys[0][toks - 1].numpy()[0]) <= 1e-5
    for c in cases + [c2]:
        c.layer.close()


@pytest.mark.parametrize("planned", [False, True])
def test_residual_decode_accumulates(si, planned):
    """y += FFN(x): the residual form adds the sparse FFN output to y."""
    d, N = 2048, 8192
    c = Case(si, d, N, 0.7, 0.2, 0.4, 1024, 16, 1, seed=75)
    S = dev(c.S)
    if planned:
        si.si_decode_plan(c.layer, S, c.n_sel, 1)
    base = synth.normal(76, 0, synth.T_MISC, d).astype(np.float32)
    y = Guarded((1, d), torch().float32)
    y.t.copy_(torch().from_numpy(base[None, :]))
    xs = [synth.tokens(77, t, synth.T_DECODE, 1, d) for t in range(3)]
    ref = base.astype(np.float64)
    for x in xs:
        si.si_sparse_ffn_decode_residual(c.layer, S, c.n_sel, 1, dev_bf16(x), y.t)
        ref = ref + oracle.sparse_ffn(c.Wg, c.Wu, c.Wd, c.loaded, c.S[0], x[0])
    assert rel_err(y.numpy()[0], ref) <= 2e-5
    with pytest.raises(si.SIError):
        si.si_sparse_ffn_decode_residual(c.layer, S, c.n_sel, 2, dev_bf16(xs[0]), y.t)
    c.layer.close()


def test_layer_range_stack(si):
    """Table 1's layer range on an 8-layer stack: layers 5 .. 5 run selection
    (gamma 0.7, phi 0.4), the first five and the last two keep the dense FFN
    (gamma = phi = 1, S = every position). Every layer matches the oracle."""
    L, d, N = 8, 256, 1024
    mask = si.si_sparse_layers(L, 5, -2)
    assert np.array_equal(mask, oracle.sparse_layers(L, 5, -2))
    for l in range(L):
        if mask[l]:
            c = Case(si, d, N, 0.7, 0.2, 0.4, 64, 16, 1, seed=60 + l)
        else:
            c = Case(si, d, N, 1.0, 0.0, 1.0, 64, 16, 1, seed=60 + l)
            assert c.n_sel == N and np.array_equal(c.S[0], np.arange(N))
        x = synth.tokens(61, l, synth.T_DECODE, 1, d)
        y = Guarded((1, d), torch().float32, fill=float("nan"))
        si.si_sparse_ffn_decode(c.layer, dev(c.S), c.n_sel, 1, dev_bf16(x), y.t)
        ref = oracle.sparse_ffn(c.Wg, c.Wu, c.Wd, c.loaded, c.S[0], x[0])
        assert rel_err(y.numpy()[0], ref) <= TOL
        c.layer.close()


@pytest.mark.parametrize("cluster", [1, 32, 64, 128])
def test_expand_clusters_then_decode(si, cluster):
    """Cluster-granular selection on a Llama3.2-1B layer's computed set:
    bit-exact with the oracle's expansion, and the decode on the expanded set
    matches the oracle's FFN on it."""
    c = Case(si, 2048, 8192, 0.7, 0.2, 0.4, 1024, 16, 1)
    out = Guarded((c.layer.n_loaded,), torch().int32, fill=-1)
    n = si.si_expand_clusters(c.layer, dev(c.S[0]), c.n_sel, cluster, out.t)
    ref = oracle.expand_clusters(c.loaded, c.S[0], c.N, cluster)
    assert n == len(ref)
    assert np.array_equal(out.numpy()[:n], ref)
    assert (n == c.n_sel) == (cluster == 1)
    x = synth.tokens(42, 0, synth.T_DECODE, 1, c.d)
    y = Guarded((1, c.d), torch().float32, fill=float("nan"))
    si.si_sparse_ffn_decode(c.layer, dev(ref).view(1, -1), n, 1, dev_bf16(x), y.t)
    y_ref = oracle.sparse_ffn(c.Wg, c.Wu, c.Wd, c.loaded, ref, x[0])
    assert rel_err(y.numpy()[0], y_ref) <= TOL
    c.layer.close()
