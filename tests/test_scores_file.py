"""Score files ([SI] section 3: the per-neuron scores of one calibration set,
stored with their token count for a later merge): the host-only save / load
pair of the C ABI, its checksum and its rejections. No GPU needed."""
import os

import numpy as np
import pytest


@pytest.fixture(scope="module")
def si():
    import activation_sparse_gb300 as si
    return si


def test_round_trip(si, tmp_path):
    rng = np.random.default_rng(7)
    s = rng.lognormal(0.0, 1.5, 11008).astype(np.float32)
    p = tmp_path / "layer0.scores"
    si.si_scores_save(str(p), s, 4096)
    got, toks = si.si_scores_load(str(p))
    assert toks == 4096
    assert got.dtype == np.float32 and np.array_equal(got.view(np.uint32), s.view(np.uint32))
    # 24-byte header, the scores, a 4-byte checksum
    assert os.path.getsize(p) == 24 + 4 * s.size + 4
    assert open(p, "rb").read(8) == b"SISCORE1"
    assert not os.path.exists(str(p) + ".tmp")


def test_fnv1a_checksum_matches_its_definition(si, tmp_path):
    # FNV-1a, 32 bits: h = 2166136261; for each byte: h ^= byte; h *= 16777619 (mod 2^32)
    s = np.arange(5, dtype=np.float32) * 0.5
    p = tmp_path / "small.scores"
    si.si_scores_save(str(p), s, 3)
    raw = open(p, "rb").read()
    h = 2166136261
    for b in raw[:-4]:
        h = ((h ^ b) * 16777619) & 0xFFFFFFFF
    assert int.from_bytes(raw[-4:], "little") == h


def test_sizing_call_and_small_capacity(si, tmp_path):
    import ctypes as C
    s = np.ones(300, dtype=np.float32)
    p = tmp_path / "s.scores"
    si.si_scores_save(str(p), s, 9)
    lib = si.load()
    n, t = C.c_int(), C.c_longlong()
    buf = np.full(10, -1.0, dtype=np.float32)
    assert lib.si_scores_load(os.fsencode(str(p)), buf.ctypes.data, 10, C.byref(n), C.byref(t)) == si.SI_OK
    assert (n.value, t.value) == (300, 9)
    assert np.all(buf == -1.0)   # too small: nothing copied


@pytest.mark.parametrize("damage", ["flip_score", "flip_checksum", "magic", "truncate", "trailing", "zero_tokens"])
def test_damaged_files_are_rejected(si, tmp_path, damage):
    s = np.linspace(0, 1, 64, dtype=np.float32)
    p = tmp_path / "d.scores"
    si.si_scores_save(str(p), s, 100)
    raw = bytearray(open(p, "rb").read())
    if damage == "flip_score":
        raw[24 + 17] ^= 0x01
    elif damage == "flip_checksum":
        raw[-1] ^= 0x80
    elif damage == "magic":
        raw[0:8] = b"SISCORE2"
    elif damage == "truncate":
        raw = raw[:-9]
    elif damage == "trailing":
        raw += b"\x00"
    elif damage == "zero_tokens":
        raw[16:24] = (0).to_bytes(8, "little")
    open(p, "wb").write(bytes(raw))
    with pytest.raises(si.SIError) as e:
        si.si_scores_load(str(p))
    assert e.value.code == si.SI_ERR_INVALID_ARG


def test_invalid_arguments(si, tmp_path):
    with pytest.raises(si.SIError):
        si.si_scores_save(str(tmp_path / "x"), np.ones(4, np.float32), 0)
    with pytest.raises(si.SIError):
        si.si_scores_save(str(tmp_path / "x"), np.ones(0, np.float32), 5)
    with pytest.raises(si.SIError):
        si.si_scores_load(str(tmp_path / "missing.scores"))
    with pytest.raises(si.SIError):
        si.si_scores_save(str(tmp_path / "no_such_dir" / "x"), np.ones(4, np.float32), 5)


@pytest.mark.gpu
def test_score_files_through_the_profiler_and_the_merge(si, tmp_path):
    # [SI] section 3: profile two calibration sets, store each in a score file
    # with its token count, read both back and merge them on the device; the
    # merge of what was stored equals the oracle's merge of the oracle scores
    import oracle
    import synth
    from gpu_util import dev, dev_bf16, torch
    d, N = 256, 1000
    Wg, Wu, _ = synth.layer_weights(80, 0, d, N)
    files, ref_scores, counts = [], [], []
    for k, T in enumerate((96, 200)):
        X = synth.tokens(81 + k, 0, synth.T_CALIB, T, d)
        s = torch().zeros(N, dtype=torch().float32, device="cuda")
        si.si_profile_scores(dev_bf16(Wg), dev_bf16(Wu), dev_bf16(X), s)
        p = tmp_path / ("set%d.scores" % k)
        si.si_scores_save(str(p), s, T)
        files.append(p)
        ref_scores.append(oracle.profile_scores(Wg, Wu, X).astype(np.float32))
        counts.append(T)
    loaded = [si.si_scores_load(str(p)) for p in files]
    assert [t for _, t in loaded] == counts
    for (got, _), ref in zip(loaded, ref_scores):
        assert np.max(np.abs(got - ref) / np.maximum(ref, 1e-30)) < 1e-3
    out = torch().empty(N, dtype=torch().float32, device="cuda")
    si.si_merge_scores([dev(g) for g, _ in loaded], counts, out)
    merged = out.cpu().numpy()
    # the device merge of the stored scores, bit for bit as the oracle merges them
    assert np.array_equal(merged.view(np.uint32), oracle.merge_scores([g for g, _ in loaded], counts).view(np.uint32))
