"""The no-allocation batch-1 decode entry point.

Some callers cannot allocate device memory while they run: a server that has
handed all device memory to its own pool, code that runs inside a stream
capture, or a process under a hard memory cap. si_sparse_ffn_decode_noalloc
serves them: its scratch sits in a fixed device array instead of memory the
library allocates. These tests call it through the C ABI twice in a row and
compare with si_sparse_ffn_decode on the same inputs.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes as C

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


def _noalloc_call(si, packed, n_records, d, S_dev, n_sel, x_dev, y_dev):
    lib = si.load()
    stream = C.c_void_p(torch().cuda.current_stream().cuda_stream)
    rc = lib.si_sparse_ffn_decode_noalloc(C.c_void_p(packed), n_records, d,
                                          C.c_void_p(S_dev.data_ptr() if S_dev is not None else 0), n_sel,
                                          C.c_void_p(x_dev.data_ptr()), C.c_void_p(y_dev.data_ptr()), stream)
    assert rc == si.SI_OK, lib.si_last_error_string()


# d = 2048 runs the one-chunk-per-lane kernel; d = 4096 (the largest d the
# fixed scratch holds) the two-chunk kernel, whose last accumulator words sit
# next to the ticket and the error words.
@pytest.mark.parametrize("d,N,gamma,delta,phi", [(2048, 8192, 0.7, 0.2, 0.4), (4096, 2048, 0.7, 0.2, 0.4)])
def test_noalloc_decode_matches_decode_two_calls_in_a_row(si, d, N, gamma, delta, phi):
    Wg, Wu, Wd = synth.layer_weights(90, 0, d, N)
    s = synth.lognormal_absact(90, 1, N)[0]
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), gamma, delta)
    loaded, st = oracle.rank_loaded(s, s, gamma, delta)
    n_sel = si.si_count(phi, N)
    S = oracle.select(synth.lognormal_absact(91, 32, len(loaded)), 32, 1, len(loaded), st, 256, n_sel)
    S_dev = dev(S)
    _, _, packed = layer.buffers()
    xs = [synth.tokens(92, t, synth.T_DECODE, 1, d) for t in range(2)]
    outs = [Guarded((1, d), torch().float32, fill=float("nan")) for _ in xs]
    for x, y in zip(xs, outs):   # two calls back to back, no host sync between them
        _noalloc_call(si, packed, layer.n_pad, d, S_dev, n_sel, dev_bf16(x), y.t)
    torch().cuda.synchronize()
    # failures of these calls would show in the reported word, read and cleared here
    assert si.si_device_error(clear=True) == 0
    for x, y in zip(xs, outs):
        ref = Guarded((1, d), torch().float32)
        si.si_sparse_ffn_decode(layer, S_dev, n_sel, 1, dev_bf16(x), ref.t)
        got, want = y.numpy()[0], ref.numpy()[0]
        assert rel_err(got, want) <= TOL
        assert rel_err(got, want) <= 2e-5
        assert rel_err(got, oracle.sparse_ffn(Wg, Wu, Wd, loaded, S[0], x[0])) <= 2e-5
    layer.close()


def test_noalloc_decode_empty_set_then_full_set(si):
    # n_sel = 0 still runs the ticketed final pass: y = 0 exactly, and the
    # accumulator and ticket come back zeroed for the next call
    d, N, gamma, delta, phi = 2048, 4096, 0.7, 0.2, 0.4
    Wg, Wu, Wd = synth.layer_weights(93, 0, d, N)
    s = synth.lognormal_absact(93, 1, N)[0]
    layer = si.si_pack_loaded(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(Wd), dev(s), dev(s), gamma, delta)
    loaded, st = oracle.rank_loaded(s, s, gamma, delta)
    n_sel = si.si_count(phi, N)
    S = oracle.select(synth.lognormal_absact(94, 16, len(loaded)), 16, 1, len(loaded), st, 128, n_sel)
    _, _, packed = layer.buffers()
    x = synth.tokens(95, 0, synth.T_DECODE, 1, d)
    y0 = Guarded((1, d), torch().float32, fill=float("nan"))
    _noalloc_call(si, packed, layer.n_pad, d, None, 0, dev_bf16(x), y0.t)
    y1 = Guarded((1, d), torch().float32, fill=float("nan"))
    _noalloc_call(si, packed, layer.n_pad, d, dev(S), n_sel, dev_bf16(x), y1.t)
    torch().cuda.synchronize()
    assert si.si_device_error(clear=True) == 0
    assert np.array_equal(y0.numpy(), np.zeros((1, d), np.float32))
    assert rel_err(y1.numpy()[0], oracle.sparse_ffn(Wg, Wu, Wd, loaded, S[0], x[0])) <= 2e-5
    layer.close()


def test_noalloc_decode_rejects_sizes_beyond_its_scratch(si):
    lib = si.load()
    p = C.c_void_p(256)
    assert lib.si_sparse_ffn_decode_noalloc(p, 10, 8192, p, 1, p, p, None) == si.SI_ERR_INVALID_ARG
    assert b"4096" in lib.si_last_error_string()
    assert lib.si_sparse_ffn_decode_noalloc(p, 10, 100, p, 1, p, p, None) == si.SI_ERR_INVALID_ARG
