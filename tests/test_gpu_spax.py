"""GPU parity: SpAx encoding (bit-exact codes), tier choice (bit-exact lists),
dense gate/up activations and the three-tier down-projection (within the FFN
tolerance)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL, Guarded, dev, dev_bf16, device_view, rel_err, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def si():
    import activation_sparse_gb300 as si
    return si


def encoded_buffers(layer):
    """The column-major copy, and the per-column records split into codes
    [N][d*bits/8] and (scale, min) pairs [N][ng_pad][2]."""
    p_wdt, p_codes, p_params = layer.buffers()
    cb = layer.d * layer.bits // 8
    rec = cb + 8 * layer.ngp
    assert p_params == p_codes + cb
    WdT = device_view(p_wdt, (layer.N, layer.d), "<i2").cpu().numpy().view(np.uint16)
    recs = device_view(p_codes, (layer.N, rec), "|u1").cpu().numpy()
    codes = np.ascontiguousarray(recs[:, :cb])
    params = np.ascontiguousarray(recs[:, cb:]).view(np.float32).reshape(layer.N, layer.ngp, 2)
    return WdT, codes, params


@pytest.fixture(scope="module")
def llama8b_layer():
    """One Llama-3.1-8B FFN layer (d=4096, d_ff=14336)."""
    return synth.layer_weights(50, 0, 4096, 14336)


@pytest.mark.parametrize("d,N,group,bits", [(256, 64, 128, 4), (4096, 14336, 128, 4), (512, 300, 64, 4),
                                            (128, 5, 8, 4), (256, 64, 128, 8), (512, 300, 64, 2),
                                            (128, 5, 8, 2), (4096, 14336, 128, 8), (1024, 700, 32, 2),
                                            (4096, 14336, 128, 3), (256, 64, 128, 3), (128, 5, 8, 3)])
def test_spax_encode_bit_exact(si, d, N, group, bits, llama8b_layer):
    if (d, N) == (4096, 14336):
        _, _, Wd = llama8b_layer
    else:
        _, _, Wd = synth.layer_weights(51, 0, d, N)
    layer = si.spax_encode(dev_bf16(Wd), bits, group)
    assert layer.bits == bits
    WdT, codes, params = encoded_buffers(layer)
    rc, rp = oracle.spax_encode(Wd, bits, group)
    assert np.array_equal(WdT, Wd.T)
    assert np.array_equal(codes, rc)
    ng = d // group
    assert np.array_equal(params[:, :ng, :].view(np.uint32), rp.view(np.uint32))
    assert not params[:, ng:, :].any()
    layer.close()


def signed_acts(seed, N, ties=False):
    a = synth.normal(seed, 0, synth.T_SPAX_A, N).astype(np.float32)
    if ties:
        a = (np.round(a * 2) / 2).astype(np.float32)
    return a


@pytest.mark.parametrize("N,top,mid,ties,bits", [(14336, 0.3, 0.3, False, 4), (14336, 0.3, 0.3, True, 4),
                                                 (1000, 0.0, 0.5, True, 4), (1000, 0.5, 0.0, False, 4),
                                                 (1000, 1.0, 0.0, False, 4), (1000, 0.0, 1.0, True, 4),
                                                 (1000, 0.0, 0.0, False, 4), (77, 0.4, 0.6, True, 4),
                                                 (14336, 0.3, 0.3, False, 8), (14336, 0.3, 0.3, True, 2),
                                                 (1000, 0.0, 1.0, True, 8), (1000, 0.2, 0.8, False, 2),
                                                 (14336, 0.3, 0.3, False, 3), (1000, 0.0, 1.0, True, 3)])
def test_spax_tiers_and_down(si, N, top, mid, ties, bits):
    d = 256 if N != 14336 else 4096
    _, _, Wd = synth.layer_weights(52, 0, d, N)
    layer = si.spax_encode(dev_bf16(Wd), bits, 128)
    a = signed_acts(53, N, ties)
    k_top, k_mid = si.si_count(top, N), si.si_count(mid, N)
    ti = Guarded((max(k_top, 1),), torch().int32, fill=-1)
    mi = Guarded((max(k_mid, 1),), torch().int32, fill=-1)
    y = Guarded((d,), torch().float32, fill=float("nan"))
    si.spax_tiered_down(layer, dev(a), top, mid, y.t, ti.t if k_top else None, mi.t if k_mid else None)
    rt, rm = oracle.spax_tiers(a, k_top, k_mid)
    if k_top:
        assert np.array_equal(ti.numpy()[:k_top], rt)
    if k_mid:
        assert np.array_equal(mi.numpy()[:k_mid], rm)
    codes, params = oracle.spax_encode(Wd, bits, 128)
    ref = oracle.spax_down(a, Wd, codes, params, rt, rm, bits=bits)
    got = y.numpy()
    # without the lists each CTA takes the tier members of its own index range
    y2 = Guarded((d,), torch().float32, fill=float("nan"))
    si.spax_tiered_down(layer, dev(a), top, mid, y2.t)
    got2 = y2.numpy()
    if k_top + k_mid == 0:
        assert np.all(got == 0) and np.all(got2 == 0)
    else:
        assert rel_err(got, ref) <= 2e-5
        assert rel_err(got2, ref) <= 2e-5
    layer.close()


@pytest.mark.parametrize("d,N,equal", [(256, 8192, False), (2048, 32768, True)])
def test_spax_tiered_down_fallbacks(si, d, N, equal):
    """a too long to stage beside a small ring (d = 256), and more keys in the
    boundary bins than the candidate space (all |a| equal): the per-CTA rank
    windows give the same tiers."""
    _, _, Wd = synth.layer_weights(56, 0, d, N)
    layer = si.spax_encode(dev_bf16(Wd), 4, 128)
    a = signed_acts(57, N, True)
    if equal:
        a = np.where(a < 0, -1.0, 1.0).astype(np.float32)
    k_top, k_mid = si.si_count(0.3, N), si.si_count(0.3, N)
    rt, rm = oracle.spax_tiers(a, k_top, k_mid)
    codes, params = oracle.spax_encode(Wd, 4, 128)
    ref = oracle.spax_down(a, Wd, codes, params, rt, rm)
    y = Guarded((d,), torch().float32, fill=float("nan"))
    si.spax_tiered_down(layer, dev(a), 0.3, 0.3, y.t)
    assert rel_err(y.numpy(), ref) <= 2e-5
    layer.close()


@pytest.mark.parametrize("d,N", [(4096, 14336), (256, 1000), (1088, 37)])
def test_spax_dense_act(si, d, N, llama8b_layer):
    if (d, N) == (4096, 14336):
        Wg, Wu, _ = llama8b_layer
    else:
        Wg, Wu, _ = synth.layer_weights(54, 0, d, N)
    x = synth.tokens(55, 0, synth.T_DECODE, 1, d)[0]
    a = Guarded((N,), torch().float32, fill=float("nan"))
    si.spax_dense_act(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(x), a.t)
    ref = oracle.dense_act(Wg, Wu, x)
    assert rel_err(a.numpy(), ref) <= 1e-5


@pytest.mark.parametrize("bits", [4, 8, 2, 3])
def test_spax_ffn_decode_full_token(si, llama8b_layer, bits):
    """One Llama-3.1-8B layer token: dense gate/up, 30% bf16 / 30% b-bit / 40% skipped."""
    Wg, Wu, Wd = llama8b_layer
    layer = si.spax_encode(dev_bf16(Wd), bits, 128)
    codes, params = oracle.spax_encode(Wd, bits, 128)
    N = 14336
    k_top, k_mid = si.si_count(0.3, N), si.si_count(0.3, N)
    Wg_d, Wu_d = dev_bf16(Wg), dev_bf16(Wu)
    for tok in range(2):
        x = synth.tokens(56, tok, synth.T_DECODE, 1, 4096)[0]
        y = Guarded((4096,), torch().float32, fill=float("nan"))
        a_out = Guarded((N,), torch().float32)
        si.spax_ffn_decode(layer, Wg_d, Wu_d, dev_bf16(x), 0.3, 0.3, y.t, a_out.t)
        a_ref = oracle.dense_act(Wg, Wu, x).astype(np.float32)
        rt, rm = oracle.spax_tiers(a_ref, k_top, k_mid)
        ref = oracle.spax_down(a_ref, Wd, codes, params, rt, rm, bits=bits)
        assert rel_err(y.numpy(), ref) <= TOL
        assert rel_err(a_out.numpy(), a_ref) <= 1e-5
    layer.close()


def test_spax_dense_act_repeated_calls(si, llama8b_layer):
    """Many back-to-back dense passes at full size: every stage of the ring
    belongs to one consumer warp, so no wait can alias a stale phase (the
    autouse check then finds the device error word clean)."""
    Wg, Wu, _ = llama8b_layer
    gWg, gWu = dev_bf16(Wg), dev_bf16(Wu)
    x = synth.tokens(57, 0, synth.T_DECODE, 1, 4096)[0]
    ref = oracle.dense_act(Wg, Wu, x)
    a = Guarded((14336,), torch().float32)
    xd = dev_bf16(x)
    for _ in range(40):
        si.spax_dense_act(gWg, gWu, xd, a.t)
    assert rel_err(a.numpy(), ref) <= 1e-5
    assert si.si_device_error() == 0


@pytest.mark.parametrize("d,N,frac,top,mid,bits", [(4096, 14336, 0.4, 0.3, 0.3, 4), (256, 1000, 0.5, 0.5, 0.5, 2),
                                                  (256, 1000, 0.05, 0.2, 0.3, 8), (256, 1000, 0.0, 0.3, 0.3, 4),
                                                  (256, 1000, 0.5, 0.3, 0.4, 3)])
def test_spax_select_decode(si, d, N, frac, top, mid, bits, llama8b_layer):
    """SelectInfer x SpAx: gate/up only on a selected set, tiers inside it
    (fractions of the set), the down-projection over its top and middle
    columns; against the oracle's dense activations zeroed outside the set."""
    if (d, N) == (4096, 14336):
        Wg, Wu, Wd = llama8b_layer
    else:
        Wg, Wu, Wd = synth.layer_weights(58, 0, d, N)
    layer = si.spax_encode(dev_bf16(Wd), bits, 128)
    codes, params = oracle.spax_encode(Wd, bits, 128)
    n_rows = si.si_count(frac, N)
    rows = np.sort(np.random.default_rng(59).choice(N, n_rows, replace=False)).astype(np.int32)
    x = synth.tokens(58, 0, synth.T_DECODE, 1, d)[0]
    y = Guarded((d,), torch().float32, fill=float("nan"))
    a_out = Guarded((N,), torch().float32, fill=float("nan"))
    rows_d = dev(rows) if n_rows else torch().empty((0,), dtype=torch().int32, device="cuda")
    si.spax_select_decode(layer, dev_bf16(Wg), dev_bf16(Wu), rows_d, dev_bf16(x), top, mid, y.t, a_out.t)
    if n_rows == 0:
        assert not y.numpy().any() and not a_out.numpy().any()
        layer.close()
        return
    a_ref = np.zeros(N, np.float32)
    a_ref[rows] = oracle.dense_act(Wg[rows], Wu[rows], x).astype(np.float32)
    got_a = a_out.numpy()
    assert not np.delete(got_a, rows).any()
    assert rel_err(got_a[rows], a_ref[rows]) <= 1e-5
    k_top, k_mid = si.si_count(top, n_rows), si.si_count(mid, n_rows)
    rt, rm = oracle.spax_tiers(got_a, k_top, k_mid)        # the tiers of the a the GPU computed
    assert np.isin(rt, rows).all() and np.isin(rm, rows).all()
    ref = oracle.spax_down(got_a, Wd, codes, params, rt, rm, bits=bits)
    assert rel_err(y.numpy(), ref) <= 2e-5
    # and within the FFN bar of the oracle's own activations
    rt2, rm2 = oracle.spax_tiers(a_ref, k_top, k_mid)
    ref2 = oracle.spax_down(a_ref, Wd, codes, params, rt2, rm2, bits=bits)
    assert rel_err(y.numpy(), ref2) <= TOL
    layer.close()


# ------------------------------------------- tiers on gate/up by |x| ("ALL")


def _tie_heavy_x(seed, d, levels=12):
    # bf16 inputs whose magnitudes take few values: many ties at the tier boundaries
    u = synth.uniform(seed, 0, 0, d)
    v = (np.floor(u * levels) - levels / 2 + 0.5) / 4.0
    return synth.to_bf16_bits(v)


@pytest.mark.parametrize("d,N,top,mid,bits,ties", [(4096, 14336, 0.3, 0.3, 4, False), (4096, 14336, 0.2, 0.5, 2, True),
                                                   (256, 512, 0.3, 0.3, 8, False), (256, 512, 0.25, 0.5, 3, True),
                                                   (256, 512, 1.0, 0.0, 4, False), (256, 512, 0.0, 1.0, 4, True),
                                                   (256, 512, 0.0, 0.0, 4, False), (512, 1024, 0.1, 0.0, 4, True)])
def test_spax_gate_up_tiers(si, d, N, top, mid, bits, ties, llama8b_layer):
    """Channel tiers by |x| bit-exact against the oracle (ties to the lower
    index); a = silu(g) * u within 1e-5 of max|a| (fp32 sums of bf16 products
    and of rebuilt weights)."""
    if (d, N) == (4096, 14336):
        Wg, Wu, _ = llama8b_layer
    else:
        Wg, Wu, _ = synth.layer_weights(60, 0, d, N)
    x = _tie_heavy_x(61, d) if ties else synth.tokens(62, 0, synth.T_DECODE, 1, d)[0]
    gate = si.spax_encode_rows(dev_bf16(Wg), bits, 128)
    upe = si.spax_encode_rows(dev_bf16(Wu), bits, 128)
    k_top, k_mid = si.si_count(top, d), si.si_count(mid, d)
    a = Guarded((N,), torch().float32, fill=float("nan"))
    t_out = Guarded((max(k_top, 1),), torch().int32, fill=-1)
    m_out = Guarded((max(k_mid, 1),), torch().int32, fill=-1)
    si.spax_gate_up(gate, upe, dev_bf16(x), top, mid, a.t, t_out.t if k_top else None, m_out.t if k_mid else None)
    got = a.numpy()
    ref, rt, rm = oracle.spax_gate_up(x, Wg, Wu, top, mid, bits=bits, group=128)
    assert np.array_equal(t_out.numpy()[:k_top], rt)
    assert np.array_equal(m_out.numpy()[:k_mid], rm)
    scale = max(np.max(np.abs(ref)), 1e-30)
    assert np.max(np.abs(got - ref)) <= 1e-5 * scale
    gate.close()
    upe.close()


def test_spax_all_decode_llama8b(si, llama8b_layer):
    """One SpAx-ALL token (Llama-3.1-8B layer): channel tiers 30 % / 30 % by |x|
    on gate/up, then neuron tiers 30 % / 30 % by |a| on the down projection;
    y within the FFN tolerance of the oracle's token."""
    Wg, Wu, Wd = llama8b_layer
    d, N = 4096, 14336
    gate = si.spax_encode_rows(dev_bf16(Wg), 4, 128)
    upe = si.spax_encode_rows(dev_bf16(Wu), 4, 128)
    down = si.spax_encode(dev_bf16(Wd), 4, 128)
    codes, params = oracle.spax_encode(Wd, 4, 128)
    for tok in range(2):   # twice: the down tiers' histogram is left clean for the next token
        x = synth.tokens(63, tok, synth.T_DECODE, 1, d)[0]
        y = Guarded((d,), torch().float32, fill=float("nan"))
        a = Guarded((N,), torch().float32, fill=float("nan"))
        si.spax_all_decode(down, gate, upe, dev_bf16(x), 0.3, 0.3, 0.3, 0.3, y.t, a.t)
        a_ref, _, _ = oracle.spax_gate_up(x, Wg, Wu, 0.3, 0.3)
        assert np.max(np.abs(a.numpy() - a_ref)) <= 1e-5 * np.max(np.abs(a_ref))
        a32 = a_ref.astype(np.float32)
        rt, rm = oracle.spax_tiers(a32, si.si_count(0.3, N), si.si_count(0.3, N))
        y_ref = oracle.spax_down(a32, Wd, codes, params, rt, rm)
        assert rel_err(y.numpy(), y_ref) <= TOL
    down.close()
    gate.close()
    upe.close()
