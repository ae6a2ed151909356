"""CPU oracle for activation-sparse FFN inference -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package. The product library never does.

``oracle.c`` is plain C compiled with gcc (``-O2 -fopenmp -ffp-contract=off``);
this module builds it on demand and marshals numpy arrays to it. Every
function here is a thin wrapper: the arithmetic lives in ``oracle.c``, which
cites the passages it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to the source (skipped when up to date)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")


def _declare(L):
    i, d, ll = C.c_int, C.c_double, C.c_longlong
    L.oracle_cnt.argtypes, L.oracle_cnt.restype = [d, ll], ll
    L.oracle_num_threads.restype = i
    L.oracle_set_threads.argtypes = [i]
    L.oracle_profile_scores.argtypes = [_u16p, _u16p, i, i, _u16p, i, _f64p]
    L.oracle_merge_scores.argtypes = [C.POINTER(C.c_void_p), C.POINTER(ll), i, i, _f32p]
    L.oracle_sparse_layers.argtypes, L.oracle_sparse_layers.restype = [i, i, i, _u8p], i
    L.oracle_down_norms.argtypes = [_u16p, i, i, _i32p, i, _f64p]
    L.oracle_expand_clusters.argtypes, L.oracle_expand_clusters.restype = [_i32p, i, _i32p, i, i, i, _i32p], i
    L.oracle_rank_loaded.argtypes = [_f32p, _f32p, i, d, d, _i32p, _u8p, C.POINTER(i), C.POINTER(i)]
    L.oracle_rank_loaded.restype = i
    L.oracle_loaded_bytes.argtypes, L.oracle_loaded_bytes.restype = [i, i, i], ll
    L.oracle_absact.argtypes = [_u16p, _u16p, i, _i32p, i, _u16p, i, _f64p]
    L.oracle_topk_rows.argtypes = [_f32p, i, i, i, i, _u8p]
    L.oracle_select.argtypes = [_f32p, i, i, i, i, _u8p, i, i, _i32p, C.c_void_p, C.c_void_p]
    L.oracle_select.restype = i
    L.oracle_sparse_ffn.argtypes = [_u16p, _u16p, _u16p, i, i, _i32p, _i32p, i, _u16p, _f64p]
    L.oracle_dense_act.argtypes = [_u16p, _u16p, i, i, _u16p, _f64p]
    L.oracle_swiglu.argtypes = [_f64p, _f64p, i, _f64p]
    L.oracle_spax_encode.argtypes = [_u16p, i, i, i, i, _u8p, _f32p]
    L.oracle_spax_encode.restype = i
    L.oracle_spax_tiers.argtypes = [_f32p, i, i, i, _i32p, _i32p]
    L.oracle_spax_tiers.restype = i
    L.oracle_spax_down.argtypes = [_f32p, i, i, _u16p, _u8p, _f32p, i, i, _i32p, i, _i32p, i, _f64p]
    L.oracle_bf16_round_array.argtypes = [_f32p, i, _u16p]


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def cnt(r: float, n: int) -> int:
    return int(lib().oracle_cnt(float(r), int(n)))


def profile_scores(Wg, Wu, X, scores=None):
    Wg, Wu, X = _c(Wg, np.uint16), _c(Wu, np.uint16), _c(X, np.uint16)
    N, d = Wg.shape
    s = np.zeros(N, np.float64) if scores is None else _c(scores, np.float64)
    lib().oracle_profile_scores(Wg, Wu, d, N, X, X.shape[0], s)
    return s


def merge_scores(score_list, token_counts):
    arrs = [_c(s, np.float32) for s in score_list]
    N = arrs[0].shape[0]
    ptrs = (C.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    toks = (C.c_longlong * len(arrs))(*[int(t) for t in token_counts])
    out = np.zeros(N, np.float32)
    lib().oracle_merge_scores(ptrs, toks, len(arrs), N, out)
    return out


def sparse_layers(L, first=5, last=-2):
    """Per-layer mask of the layers that run selection (Table 1's range); the
    others keep their dense FFN."""
    out = np.zeros(max(L, 1), np.uint8)
    n = lib().oracle_sparse_layers(int(L), int(first), int(last), out)
    if n < 0:
        raise ValueError("need L >= 0, first >= 0")
    return out[:L].astype(bool)


def down_norms(Wd, loaded):
    """||Wd[:, n]||_2 of each loaded neuron n (float64), the weight half of the
    weight-aware salience |a_n| * ||Wd[:, n]||_2."""
    Wd, loaded = _c(Wd, np.uint16), _c(loaded, np.int32)
    d, N = Wd.shape
    out = np.zeros(loaded.shape[0], np.float64)
    lib().oracle_down_norms(Wd, d, N, loaded, loaded.shape[0], out)
    return out


def expand_clusters(loaded, S, N, cluster):
    """Positions of every loaded neuron in a cluster (contiguous block of
    `cluster` neuron indices) that holds a neuron of the selected positions S."""
    loaded, S = _c(loaded, np.int32), _c(S, np.int32)
    out = np.zeros(max(loaded.shape[0], 1), np.int32)
    n = lib().oracle_expand_clusters(loaded, loaded.shape[0], S, S.shape[0], int(N), int(cluster), out)
    if n < 0:
        raise ValueError("cluster size must be >= 1")
    return out[:n].copy()


def rank_loaded(task, model, gamma, delta):
    task, model = _c(task, np.float32), _c(model, np.float32)
    N = task.shape[0]
    loaded = np.zeros(N, np.int32)
    st = np.zeros(N, np.uint8)
    nl, ns = C.c_int(0), C.c_int(0)
    rc = lib().oracle_rank_loaded(task, model, N, float(gamma), float(delta), loaded, st,
                                  C.byref(nl), C.byref(ns))
    if rc != 0:
        raise ValueError("invalid ratios")
    return loaded[: nl.value].copy(), st[: nl.value].copy()


def loaded_bytes(d, n_loaded, s=2):
    return int(lib().oracle_loaded_bytes(int(d), int(n_loaded), int(s)))


def absact(Wg, Wu, loaded, X):
    Wg, Wu, X, loaded = _c(Wg, np.uint16), _c(Wu, np.uint16), _c(X, np.uint16), _c(loaded, np.int32)
    out = np.zeros((X.shape[0], loaded.shape[0]), np.float64)
    lib().oracle_absact(Wg, Wu, Wg.shape[1], loaded, loaded.shape[0], X, X.shape[0], out)
    return out


def topk_rows(A, k, n=None):
    A = _c(A, np.float32)
    rows, ld = A.shape
    n = ld if n is None else n
    sel = np.zeros((rows, n), np.uint8)
    lib().oracle_topk_rows(A, rows, n, ld, int(k), sel)
    return sel


def select(absA, T, B, n_loaded, is_static, alpha, n_sel, want_counts=False, want_sel=False):
    absA = _c(absA, np.float32)
    ld = absA.shape[1]
    st = _c(is_static, np.uint8)
    S = np.zeros((B, n_sel), np.int32)
    counts = np.zeros((B, n_loaded), np.uint32) if want_counts else None
    sel = np.zeros((B * T, n_loaded), np.uint8) if want_sel else None
    rc = lib().oracle_select(absA, T, B, n_loaded, ld, st, int(alpha), int(n_sel), S,
                             None if counts is None else counts.ctypes.data,
                             None if sel is None else sel.ctypes.data)
    if rc != 0:
        raise ValueError("beta does not fit")
    out = [S]
    if want_counts:
        out.append(counts)
    if want_sel:
        out.append(sel)
    return out[0] if len(out) == 1 else tuple(out)


def sparse_ffn(Wg, Wu, Wd, loaded, S, x):
    Wg, Wu, Wd = _c(Wg, np.uint16), _c(Wu, np.uint16), _c(Wd, np.uint16)
    loaded, S, x = _c(loaded, np.int32), _c(S, np.int32), _c(x, np.uint16)
    N, d = Wg.shape
    y = np.zeros(d, np.float64)
    lib().oracle_sparse_ffn(Wg, Wu, Wd, d, N, loaded, S, S.shape[0], x, y)
    return y


def bf16_round(f):
    """bf16 bit patterns (uint16) of float32 values, round to nearest even."""
    f = _c(np.asarray(f, dtype=np.float32).ravel(), np.float32)
    out = np.zeros(f.shape[0], np.uint16)
    lib().oracle_bf16_round_array(f, f.shape[0], out)
    return out


NORM_EPS = 1e-5  # RMS norm epsilon of a stack layer's input (Llama 3.2's value)


def rms_norm_bf16(h):
    """bf16 bits of h / sqrt(mean(h^2) + eps): computed in float64, rounded to
    float32, then to bf16 (round to nearest even)."""
    hh = np.asarray(h, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(hh * hh) + NORM_EPS)
    return bf16_round((hh * r).astype(np.float32))


def sparse_ffn_stack(h, layers):
    """One decode token through a stack of sparse FFN layers on one residual
    stream. SelectInfer section 5 computes each layer's FFN on its selected
    neurons, the layers in order; in the pages' models (Llama, Qwen) each FFN
    reads the RMS-normalised residual stream and adds its output back to it
    (unit norm gain here):
        for each layer l:  x_l = bf16(h / sqrt(mean(h^2) + eps));  h = h + FFN_l(x_l)
    h: float [d] (kept in float64 here); layers: list of (Wg, Wu, Wd, loaded,
    S) with S the layer's selected packed positions. Returns (h after the
    last layer, float64 [d]; the inputs x_l, uint16 [L][d] bf16 bits)."""
    hh = np.array(h, dtype=np.float64)
    xs = []
    for Wg, Wu, Wd, loaded, S in layers:
        x = rms_norm_bf16(hh)
        xs.append(x)
        hh = hh + sparse_ffn(Wg, Wu, Wd, loaded, S, x)
    return hh, np.stack(xs) if xs else np.zeros((0, hh.shape[0]), np.uint16)


def dense_act(Wg, Wu, x):
    Wg, Wu, x = _c(Wg, np.uint16), _c(Wu, np.uint16), _c(x, np.uint16)
    N, d = Wg.shape
    a = np.zeros(N, np.float64)
    lib().oracle_dense_act(Wg, Wu, d, N, x, a)
    return a


def swiglu(g, u):
    """silu(g) * u elementwise (float64)."""
    g, u = _c(g, np.float64), _c(u, np.float64)
    out = np.zeros(g.shape[0], np.float64)
    lib().oracle_swiglu(g, u, g.shape[0], out)
    return out


def spax_gate_up(x, Wg, Wu, top_frac, mid_frac, bits=4, group=128):
    """SpAx tiers on the gate/up projections by |x| (the pages' "ALL"
    configuration, FFN part): the input channels j ranked by |x_j| (ties to
    the lower index); the top k_top columns of Wg / Wu read in bf16, the next
    k_mid rebuilt from b-bit codes of each column (groups along the neuron
    axis), the rest skipped; then a = silu(g) * u. Wg, Wu: bf16 bits [N x d]
    (output x input, like Wd), x: bf16 bits [d]. Returns (a, top, mid)."""
    Wg, Wu, x = _c(Wg, np.uint16), _c(Wu, np.uint16), _c(x, np.uint16)
    d = x.shape[0]
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    k_top, k_mid = cnt(top_frac, d), cnt(mid_frac, d)
    top, mid = spax_tiers(xf, k_top, k_mid)
    cg, pg = spax_encode(Wg, bits, group)
    cu, pu = spax_encode(Wu, bits, group)
    g = spax_down(xf, Wg, cg, pg, top, mid, bits, group)
    u = spax_down(xf, Wu, cu, pu, top, mid, bits, group)
    return swiglu(g, u), top, mid


def spax_encode(Wd, bits=4, group=128):
    Wd = _c(Wd, np.uint16)
    d, N = Wd.shape
    codes = np.zeros((N, d * bits // 8), np.uint8)
    params = np.zeros((N, d // group, 2), np.float32)
    if lib().oracle_spax_encode(Wd, d, N, int(bits), int(group), codes, params) != 0:
        raise ValueError("unsupported bits/group")
    return codes, params


def spax_tiers(a, k_top, k_mid):
    a = _c(a, np.float32)
    top = np.zeros(max(k_top, 0), np.int32)
    mid = np.zeros(max(k_mid, 0), np.int32)
    if lib().oracle_spax_tiers(a, a.shape[0], int(k_top), int(k_mid), top, mid) != 0:
        raise ValueError("tier sizes do not fit")
    return top, mid


def spax_down(a, Wd, codes, params, top, mid, bits=4, group=128):
    a, Wd = _c(a, np.float32), _c(Wd, np.uint16)
    codes, params = _c(codes, np.uint8), _c(params, np.float32)
    top, mid = _c(top, np.int32), _c(mid, np.int32)
    d, N = Wd.shape
    y = np.zeros(d, np.float64)
    lib().oracle_spax_down(a, N, d, Wd, codes, params, int(bits), int(group), top, top.shape[0],
                           mid, mid.shape[0], y)
    return y
