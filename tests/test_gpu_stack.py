"""GPU parity: the decode stack (one launch per token over L sparse FFN layers
on one residual stream) against the oracle's stack, through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL, Guarded, dev, dev_bf16, rel_err, torch, u16_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def si():
    import activation_sparse_gb300 as si
    return si


class StackCase:
    """L packed layers (each with its own seeded weights and computed set)."""

    def __init__(self, si, d, N, L, gamma=0.7, delta=0.2, phi=0.4, alpha=64, T=16, seed=300, dense=()):
        self.layers, self.ref, self.S_dev, self.n_sel = [], [], [], []
        for l in range(L):
            g, dl, ph = (1.0, 0.0, 1.0) if l in dense else (gamma, delta, phi)
            Wg, Wu, Wd = synth.layer_weights(seed, l, d, N)
            s = synth.lognormal_absact(seed + 1, l + 1, N)[l]
            layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), g, dl)
            loaded, st = oracle.rank_loaded(s, s, g, dl)
            n_sel = si.si_count(ph, N)
            nl = len(loaded)
            if l in dense:
                S = np.arange(N, dtype=np.int32)
            else:
                S = oracle.select(synth.lognormal_absact(seed + 2 + l, T, nl), T, 1, nl, st, min(alpha, nl),
                                  n_sel)[0]
            self.layers.append(layer)
            self.ref.append((Wg, Wu, Wd, loaded, S))
            self.S_dev.append(dev(S))
            self.n_sel.append(len(S))
        self.d, self.L = d, L

    def close(self):
        for layer in self.layers:
            layer.close()


def _run(si, stack, h0, L, d):
    h = Guarded((d,), torch().float32)
    h.t.copy_(torch().from_numpy(h0.astype(np.float32)))
    xo = Guarded((L, d), torch().bfloat16, fill=None)
    si.si_sparse_ffn_decode_stack(stack, h.t, xo.t)
    torch().cuda.synchronize()
    return h.numpy().astype(np.float64), u16_of(xo.t), xo


def _signs(seed, d):
    # h = +-1: its RMS norm is +-1/sqrt(1 + 1e-5), which rounds to +-1 in bf16 on
    # either side whatever the order of the sum of squares, so both sides read
    # the same input bit for bit
    return np.where(synth.uniform(seed, 0, 0, d) < 0.5, -1.0, 1.0)


@pytest.mark.parametrize("d,N", [(256, 1024), (1024, 2048), (2048, 8192), (3072, 8192)])
def test_stack_one_layer_matches_oracle(si, d, N):
    c = StackCase(si, d, N, 1, seed=310 + d)
    stack = si.si_stack_create(c.layers)
    si.si_stack_plan(stack, c.S_dev, c.n_sel)
    h0 = _signs(311, d)
    h, xs, xo = _run(si, stack, h0, 1, d)
    xo.check()
    x0 = oracle.rms_norm_bf16(h0)
    assert np.array_equal(x0, synth.to_bf16_bits(h0))
    assert np.array_equal(xs[0], x0)   # the layer's input, bit for bit
    Wg, Wu, Wd, loaded, S = c.ref[0]
    y = oracle.sparse_ffn(Wg, Wu, Wd, loaded, S, x0)
    ref = h0 + y
    # fp32 accumulation of bf16 products (2e-5 of max|y|) plus the rounding of h to fp32
    atol = 2e-5 * np.max(np.abs(y)) + 4 * np.finfo(np.float32).eps * np.max(np.abs(ref))
    assert np.max(np.abs(h - ref)) <= atol
    assert rel_err(h - h0, y) <= TOL
    stack.close()
    c.close()


@pytest.mark.parametrize("d,N,L,dense", [(2048, 4096, 6, (2,)), (3072, 8192, 2, ())])
def test_stack_chain_matches_oracle(si, d, N, L, dense):
    # Past the first layer the two sides' inputs can part by a bf16 step where
    # the normalised stream sits near a rounding midpoint, and such a step moves
    # the next layer's output slightly, so later inputs part more often: the
    # chain is compared at the FFN tolerance, the first input bit for bit.
    c = StackCase(si, d, N, L, seed=330 + d, dense=dense)
    stack = si.si_stack_create(c.layers)
    si.si_stack_plan(stack, c.S_dev, c.n_sel)
    h0 = _signs(331, d)
    h, xs, _ = _run(si, stack, h0, L, d)
    h_ref, xs_ref = oracle.sparse_ffn_stack(h0, c.ref)
    assert np.array_equal(xs[0], xs_ref[0])
    xg = synth.bf16_bits_to_f32(xs).astype(np.float64)
    xr = synth.bf16_bits_to_f32(xs_ref).astype(np.float64)
    assert np.max(np.abs(xg - xr)) <= TOL * np.max(np.abs(xr))
    err = rel_err(h - h0, h_ref - h0)
    assert err <= TOL
    stack.close()
    c.close()


def test_stack_repeated_calls_and_replans(si):
    # scratch (counters, layer sums, error word) is re-zeroed by each launch:
    # calls back to back give the same result; a new plan with other set
    # sizes is picked up
    d, N, L = 1024, 2048, 5
    c = StackCase(si, d, N, L, seed=350)
    stack = si.si_stack_create(c.layers)
    si.si_stack_plan(stack, c.S_dev, c.n_sel)
    h0 = _signs(351, d)
    hs = []
    hbuf = [torch().from_numpy(h0.astype(np.float32)).cuda() for _ in range(3)]
    for hb in hbuf:   # three launches with no host sync between them
        si.si_sparse_ffn_decode_stack(stack, hb)
    torch().cuda.synchronize()
    for hb in hbuf:
        hs.append(hb.cpu().numpy().astype(np.float64))
    h_ref, _ = oracle.sparse_ffn_stack(h0, c.ref)
    for h in hs:
        assert rel_err(h - h0, h_ref - h0) <= TOL
        assert rel_err(h - h0, hs[0] - h0) <= TOL
    # re-plan with smaller sets: the first half of every layer's set
    half = [S[: len(S) // 2].copy() for (_, _, _, _, S) in c.ref]
    si.si_stack_plan(stack, [dev(S) for S in half], [len(S) for S in half])
    h, _, _ = _run(si, stack, h0, L, d)
    ref2 = [(Wg, Wu, Wd, loaded, S2) for (Wg, Wu, Wd, loaded, _), S2 in zip(c.ref, half)]
    h_ref2, _ = oracle.sparse_ffn_stack(h0, ref2)
    assert rel_err(h - h0, h_ref2 - h0) <= TOL
    stack.close()
    c.close()


def test_stack_empty_sets_leave_h(si):
    d, N, L = 512, 1024, 3
    c = StackCase(si, d, N, L, seed=360)
    stack = si.si_stack_create(c.layers)
    si.si_stack_plan(stack, [None] * L, [0] * L)
    h0 = _signs(361, d)
    h, xs, _ = _run(si, stack, h0, L, d)
    assert np.array_equal(h, h0)
    x0 = oracle.rms_norm_bf16(h0)
    assert all(np.array_equal(x, x0) for x in xs)
    stack.close()
    c.close()


def test_stack_rejects_bad_arguments(si):
    Wg, Wu, Wd = synth.layer_weights(370, 0, 4096, 256)
    s = synth.lognormal_absact(370, 1, 256)[0]
    wide = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), 0.5, 0.1)
    with pytest.raises(si.SIError) as e:
        si.si_stack_create([wide])
    assert e.value.code == si.SI_ERR_UNSUPPORTED
    c = StackCase(si, 512, 1024, 1, seed=371)
    Wg2, Wu2, Wd2 = synth.layer_weights(372, 0, 256, 512)
    s2 = synth.lognormal_absact(372, 1, 512)[0]
    other = si.si_pack_loaded(dev_bf16(Wg2), dev_bf16(Wu2), dev_bf16(Wd2), dev(s2), dev(s2), 0.5, 0.1)
    with pytest.raises(si.SIError) as e:
        si.si_stack_create([c.layers[0], other])
    assert e.value.code == si.SI_ERR_INVALID_ARG
    stack = si.si_stack_create(c.layers)
    h = torch().zeros(512, dtype=torch().float32, device="cuda")
    with pytest.raises(si.SIError) as e:   # no plan yet
        si.si_sparse_ffn_decode_stack(stack, h)
    assert e.value.code == si.SI_ERR_INVALID_ARG
    with pytest.raises(si.SIError):        # a set larger than the loaded neurons
        si.si_stack_plan(stack, [c.S_dev[0]], [c.layers[0].n_loaded + 1])
    stack.close()
    c.close()
    wide.close()
    other.close()
