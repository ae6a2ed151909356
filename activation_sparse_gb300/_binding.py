"""ctypes binding of ``libsi.so`` (declared in ``include/si.h``).

Argument marshalling only: torch tensors supply device pointers, the current
CUDA stream is passed through, status codes become exceptions. Every step of
the method runs in the library's CUDA kernels; there is no fallback. When the
library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes as C
import os

from . import _build

SI_OK, SI_ERR_INVALID_ARG, SI_ERR_CUDA, SI_ERR_OOM, SI_ERR_UNSUPPORTED, SI_ERR_DEVICE = range(6)
SI_DEVERR_WAIT_TIMEOUT, SI_DEVERR_COUNT, SI_DEVERR_RANGE = 1, 2, 4

# every symbol include/si.h declares, with (restype, argtypes)
_vp, _i, _d, _ll, _u32p = C.c_void_p, C.c_int, C.c_double, C.c_longlong, C.POINTER(C.c_uint32)
_ip = C.POINTER(C.c_int)
SIGNATURES = {
    "si_last_error_string": (C.c_char_p, []),
    "si_abi_version": (_i, []),
    "si_count": (_ll, [_d, _ll]),
    "si_counts": (_i, [_i, _d, _d, _d, _ip, _ip, _ip, _ip]),
    "si_packed_bytes": (_ll, [_i, _i]),
    "si_sparse_layers": (_i, [_i, _i, _i, _vp, _ip]),
    "si_device_error": (_i, [_u32p, _i]),
    "si_profile_scores": (_i, [_vp, _vp, _i, _i, _vp, _i, _vp, _vp]),
    "si_merge_scores": (_i, [C.POINTER(_vp), C.POINTER(_ll), _i, _i, _vp, _vp]),
    "si_scores_save": (_i, [C.c_char_p, _vp, _i, _ll]),
    "si_scores_load": (_i, [C.c_char_p, _vp, _i, _ip, C.POINTER(_ll)]),
    "si_pack_loaded": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp, _d, _d, C.POINTER(_vp), _vp]),
    "si_layer_info": (_i, [_vp, _ip, _ip, _ip, _ip, _ip]),
    "si_layer_buffers": (_i, [_vp, C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp)]),
    "si_layer_destroy": (_i, [_vp]),
    "si_select_dynamic": (_i, [_vp, _vp, _i, _i, _i, _d, _vp, _vp, _vp]),
    "si_prefill_absact": (_i, [_vp, _vp, _i, _i, _vp, _vp]),
    "si_set_gemm_tile": (_i, [_i]),
    "si_layer_set_salience": (_i, [_vp, _i]),
    "si_layer_norms": (_i, [_vp, C.POINTER(_vp)]),
    "si_gemm_tile_for": (_i, [_i, _i, _ip]),
    "si_select_from_absact": (_i, [_vp, _vp, _i, _i, _i, _i, _d, _vp, _vp, _vp, _vp]),
    "si_decode_plan": (_i, [_vp, _vp, _i, _i, _vp]),
    "si_expand_clusters": (_i, [_vp, _vp, _i, _i, _vp, _ip, _vp]),
    "si_sparse_ffn_decode": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp]),
    "si_sparse_ffn_decode_residual": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp]),
    "si_sparse_ffn_decode_noalloc": (_i, [_vp, _i, _i, _vp, _i, _vp, _vp, _vp]),
    "si_stack_create": (_i, [C.POINTER(_vp), _i, C.POINTER(_vp)]),
    "si_stack_plan": (_i, [_vp, C.POINTER(_vp), _ip, _vp]),
    "si_sparse_ffn_decode_stack": (_i, [_vp, _vp, _vp, _vp]),
    "si_stack_destroy": (_i, [_vp]),
    "spax_encode": (_i, [_vp, _i, _i, _i, _i, C.POINTER(_vp), _vp]),
    "spax_layer_info": (_i, [_vp, _ip, _ip, _ip, _ip, _ip]),
    "spax_layer_buffers": (_i, [_vp, C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp)]),
    "spax_layer_destroy": (_i, [_vp]),
    "spax_dense_act": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp]),
    "spax_tiered_down": (_i, [_vp, _vp, _d, _d, _vp, _vp, _vp, _vp]),
    "spax_ffn_decode": (_i, [_vp, _vp, _vp, _vp, _d, _d, _vp, _vp, _vp]),
    "spax_select_decode": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _d, _d, _vp, _vp, _vp]),
    "spax_gate_up": (_i, [_vp, _vp, _vp, _d, _d, _vp, _vp, _vp, _vp]),
    "spax_all_decode": (_i, [_vp, _vp, _vp, _vp, _d, _d, _d, _d, _vp, _vp, _vp]),
}

_lib = None


class SIError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("si error %d: %s" % (code, msg))
        self.code = code


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Loads libsi.so (building it first when absent or stale and nvcc exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise ImportError("libsi.so is not built; run __graft_entry__.build() first")
    L = C.CDLL(_build.LIB)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    _lib = L
    return L


def _check(rc):
    if rc != SI_OK:
        raise SIError(rc, _lib.si_last_error_string().decode())


# ------------------------------------------------------------------ helpers

def _torch():
    import torch
    return torch


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    torch = _torch()
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must have dtype %s, got %s" % (name, dtype, t.dtype))
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _bf16(t, name):
    """bf16 tensors travel as their bit patterns: accept torch.bfloat16 or int16/uint16 views."""
    torch = _torch()
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise ValueError("%s must be bf16 (or its 16-bit pattern)" % name)
    return _ptr(t, None, name)


# ------------------------------------------------------------------ API


def si_count(ratio: float, n: int) -> int:
    return int(load().si_count(float(ratio), int(n)))


def si_counts(N, gamma, delta, phi):
    L = load()
    a, b, c, d = C.c_int(), C.c_int(), C.c_int(), C.c_int()
    _check(L.si_counts(int(N), float(gamma), float(delta), float(phi), C.byref(a), C.byref(b), C.byref(c),
                       C.byref(d)))
    return a.value, b.value, c.value, d.value


def si_packed_bytes(d, n_loaded) -> int:
    return int(load().si_packed_bytes(int(d), int(n_loaded)))


def si_device_error(clear: bool = True) -> int:
    L = load()
    v = C.c_uint32()
    _check(L.si_device_error(C.byref(v), 1 if clear else 0))
    return v.value


def si_sparse_layers(L: int, first: int = 5, last: int = -2):
    """Per-layer mask (numpy bool [L]) of the layers that run selection; the others stay dense."""
    import numpy as np
    out = np.zeros(max(int(L), 1), np.uint8)
    n = C.c_int(0)
    _check(load().si_sparse_layers(int(L), int(first), int(last), out.ctypes.data_as(C.c_void_p), C.byref(n)))
    return out[:int(L)].astype(bool)


def si_profile_scores(Wg, Wu, X, scores, stream=None):
    N, d = Wg.shape
    _check(load().si_profile_scores(_bf16(Wg, "Wg"), _bf16(Wu, "Wu"), d, N, _bf16(X, "X"), X.shape[0],
                                    _ptr(scores, _torch().float32, "scores"), _stream(stream)))
    return scores


def si_merge_scores(score_list, token_counts, out, stream=None):
    torch = _torch()
    ptrs = (C.c_void_p * len(score_list))(*[s.data_ptr() for s in score_list])
    for s in score_list:
        _ptr(s, torch.float32, "scores")
    toks = (C.c_longlong * len(score_list))(*[int(t) for t in token_counts])
    _check(load().si_merge_scores(ptrs, toks, len(score_list), out.shape[0], _ptr(out, torch.float32, "out"),
                                  _stream(stream)))
    return out


def si_scores_save(path, scores, token_count):
    """Writes a score file: `scores` (fp32 [N], on any device) and the token
    count they were summed over."""
    import numpy as np
    if hasattr(scores, "detach"):
        scores = scores.detach().to("cpu")
        scores = scores.numpy()
    h = np.ascontiguousarray(scores, dtype=np.float32).reshape(-1)
    _check(load().si_scores_save(os.fsencode(path), h.ctypes.data, int(h.size), int(token_count)))


def si_scores_load(path):
    """Reads a score file: (scores as a float32 numpy array [N], token count)."""
    import numpy as np
    n, t = C.c_int(), C.c_longlong()
    L = load()
    _check(L.si_scores_load(os.fsencode(path), None, 0, C.byref(n), C.byref(t)))
    out = np.empty(n.value, dtype=np.float32)
    _check(L.si_scores_load(os.fsencode(path), out.ctypes.data, int(out.size), C.byref(n), C.byref(t)))
    return out, t.value


class Layer:
    """A packed SelectInfer layer (owns the library handle)."""

    def __init__(self, handle):
        self._h = handle
        L = load()
        v = [C.c_int() for _ in range(5)]
        _check(L.si_layer_info(self._h, *[C.byref(x) for x in v]))
        self.d, self.N, self.n_loaded, self.n_static, self.n_pad = [x.value for x in v]

    @property
    def handle(self):
        return self._h

    def buffers(self):
        """(loaded_idx, is_static, packed) device pointers as ints."""
        a, b, c = C.c_void_p(), C.c_void_p(), C.c_void_p()
        _check(load().si_layer_buffers(self._h, C.byref(a), C.byref(b), C.byref(c)))
        return a.value, b.value, c.value

    def close(self):
        if self._h:
            load().si_layer_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def si_pack_loaded(Wg, Wu, Wd, task_scores, model_scores, gamma, delta, stream=None) -> Layer:
    torch = _torch()
    N, d = Wg.shape
    h = C.c_void_p()
    _check(load().si_pack_loaded(_bf16(Wg, "Wg"), _bf16(Wu, "Wu"), _bf16(Wd, "Wd"), d, N,
                                 _ptr(task_scores, torch.float32, "task_scores"),
                                 _ptr(model_scores, torch.float32, "model_scores"), float(gamma), float(delta),
                                 C.byref(h), _stream(stream)))
    return Layer(h)


def si_select_dynamic(layer: Layer, X, T, B, alpha, phi, S, absact_out=None, stream=None):
    torch = _torch()
    _check(load().si_select_dynamic(layer.handle, _bf16(X, "X"), int(T), int(B), int(alpha), float(phi),
                                    _ptr(S, torch.int32, "S"), _ptr(absact_out, torch.float32, "absact_out"),
                                    _stream(stream)))
    return S


def si_layer_set_salience(layer: Layer, weight_aware: bool):
    """Prefill ranking key of this layer: |a| (False, default) or |a| * ||Wd[:, n]||_2 (True)."""
    _check(load().si_layer_set_salience(layer.handle, 1 if weight_aware else 0))


def si_layer_norms(layer: Layer) -> int:
    """Device pointer of the layer's fp32 [n_pad] down-column norms."""
    p = C.c_void_p()
    _check(load().si_layer_norms(layer.handle, C.byref(p)))
    return p.value


def si_set_gemm_tile(bnn: int):
    """Forces the activation GEMM's neuron-tile width (64, 80, 96, 112, 128) or, with 0, restores the per-launch choice."""
    _check(load().si_set_gemm_tile(int(bnn)))


def si_gemm_tile_for(M: int, N: int) -> int:
    """The neuron-tile width a GEMM launch over M token rows and N neurons would use now."""
    b = C.c_int(0)
    _check(load().si_gemm_tile_for(int(M), int(N), C.byref(b)))
    return b.value


def si_prefill_absact(layer: Layer, X, T, B, absact_out, stream=None):
    _check(load().si_prefill_absact(layer.handle, _bf16(X, "X"), int(T), int(B),
                                    _ptr(absact_out, _torch().float32, "absact_out"), _stream(stream)))
    return absact_out


def si_select_from_absact(layer: Layer, absA, T, B, alpha, phi, S, topmask=None, counts=None, stream=None):
    torch = _torch()
    u32 = torch.int32  # uint32 words travel in int32 tensors
    _check(load().si_select_from_absact(layer.handle, _ptr(absA, torch.float32, "absA"), absA.shape[1], int(T),
                                        int(B), int(alpha), float(phi), _ptr(S, torch.int32, "S"),
                                        _ptr(topmask, u32, "topmask"), _ptr(counts, u32, "counts"),
                                        _stream(stream)))
    return S


def si_expand_clusters(layer: Layer, S, n_sel, cluster, S_out, stream=None) -> int:
    """Whole clusters of `cluster` contiguous neurons around the selected positions S; returns len."""
    n = C.c_int(0)
    _check(load().si_expand_clusters(layer.handle, _ptr(S, _torch().int32, "S") if n_sel else None, int(n_sel),
                                     int(cluster), _ptr(S_out, _torch().int32, "S_out"), C.byref(n),
                                     _stream(stream)))
    return n.value


def si_decode_plan(layer: Layer, S, n_sel, B, stream=None):
    _check(load().si_decode_plan(layer.handle, _ptr(S, _torch().int32, "S"), int(n_sel), int(B), _stream(stream)))


def si_sparse_ffn_decode(layer: Layer, S, n_sel, B, x, y, stream=None):
    torch = _torch()
    _check(load().si_sparse_ffn_decode(layer.handle, _ptr(S, torch.int32, "S"), int(n_sel), int(B), _bf16(x, "x"),
                                       _ptr(y, torch.float32, "y"), _stream(stream)))
    return y


def si_sparse_ffn_decode_residual(layer: Layer, S, n_sel, B, x, y, stream=None):
    torch = _torch()
    _check(load().si_sparse_ffn_decode_residual(layer.handle, _ptr(S, torch.int32, "S"), int(n_sel), int(B),
                                                _bf16(x, "x"), _ptr(y, torch.float32, "y"), _stream(stream)))
    return y


def si_sparse_ffn_decode_noalloc(packed_ptr: int, n_records: int, d: int, S, n_sel, x, y, stream=None):
    """The no-allocation batch-1 decode; packed_ptr is a device address (int)."""
    torch = _torch()
    _check(load().si_sparse_ffn_decode_noalloc(C.c_void_p(packed_ptr), int(n_records), int(d),
                                               _ptr(S, torch.int32, "S"), int(n_sel), _bf16(x, "x"),
                                               _ptr(y, torch.float32, "y"), _stream(stream)))
    return y


class Stack:
    """A decode stack over packed layers (owns the library handle; the layers
    must outlive it, and it keeps references to them)."""

    def __init__(self, handle, layers):
        self._h = handle
        self.layers = list(layers)
        self.L = len(self.layers)
        self.d = self.layers[0].d

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            load().si_stack_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def si_stack_create(layers) -> Stack:
    hs = (C.c_void_p * len(layers))(*[l.handle for l in layers])
    h = C.c_void_p()
    _check(load().si_stack_create(hs, len(layers), C.byref(h)))
    return Stack(h, layers)


def si_stack_plan(stack: Stack, S_list, n_sel_list, stream=None):
    """Copies each layer's computed set (device int32, ascending positions) into the stack."""
    torch = _torch()
    ptrs = []
    for S, n in zip(S_list, n_sel_list):
        ptrs.append(_ptr(S, torch.int32, "S").value if int(n) > 0 else None)
    arr = (C.c_void_p * stack.L)(*ptrs)
    ns = (C.c_int * stack.L)(*[int(n) for n in n_sel_list])
    _check(load().si_stack_plan(stack.handle, arr, ns, _stream(stream)))


def si_sparse_ffn_decode_stack(stack: Stack, h, x_out=None, stream=None):
    """One decode token through every layer of the stack: h (fp32 [d], read
    and written) is the residual stream; x_out (optional bf16 [L][d]) gets each
    layer's input."""
    torch = _torch()
    _check(load().si_sparse_ffn_decode_stack(stack.handle, _ptr(h, torch.float32, "h"),
                                             _bf16(x_out, "x_out") if x_out is not None else None,
                                             _stream(stream)))
    return h


class SpaxLayer:
    """An encoded SpAx down-projection (owns the library handle)."""

    def __init__(self, handle):
        self._h = handle
        v = [C.c_int() for _ in range(5)]
        _check(load().spax_layer_info(self._h, *[C.byref(x) for x in v]))
        self.d, self.N, self.bits, self.group, self.ngp = [x.value for x in v]

    @property
    def handle(self):
        return self._h

    def buffers(self):
        """(WdT, codes, params) device pointers as ints."""
        a, b, c = C.c_void_p(), C.c_void_p(), C.c_void_p()
        _check(load().spax_layer_buffers(self._h, C.byref(a), C.byref(b), C.byref(c)))
        return a.value, b.value, c.value

    def close(self):
        if self._h:
            load().spax_layer_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spax_encode(Wd, bits=4, group=128, stream=None) -> SpaxLayer:
    d, N = Wd.shape
    h = C.c_void_p()
    _check(load().spax_encode(_bf16(Wd, "Wd"), d, N, int(bits), int(group), C.byref(h), _stream(stream)))
    return SpaxLayer(h)


def spax_dense_act(Wg, Wu, x, a, stream=None):
    N, d = Wg.shape
    _check(load().spax_dense_act(_bf16(Wg, "Wg"), _bf16(Wu, "Wu"), d, N, _bf16(x, "x"),
                                 _ptr(a, _torch().float32, "a"), _stream(stream)))
    return a


def spax_tiered_down(layer: SpaxLayer, a, top_frac, mid_frac, y, top_idx=None, mid_idx=None, stream=None):
    torch = _torch()
    _check(load().spax_tiered_down(layer.handle, _ptr(a, torch.float32, "a"), float(top_frac), float(mid_frac),
                                   _ptr(y, torch.float32, "y"), _ptr(top_idx, torch.int32, "top_idx"),
                                   _ptr(mid_idx, torch.int32, "mid_idx"), _stream(stream)))
    return y


def spax_select_decode(layer: SpaxLayer, Wg, Wu, rows, x, top_frac, mid_frac, y, a_out=None, stream=None):
    """SpAx tiers inside a selected set: rows (device int32) are the neurons computed."""
    torch = _torch()
    n_rows = int(rows.numel()) if rows is not None else 0
    _check(load().spax_select_decode(layer.handle, _bf16(Wg, "Wg"), _bf16(Wu, "Wu"),
                                     _ptr(rows, torch.int32, "rows") if n_rows else None, n_rows, _bf16(x, "x"),
                                     float(top_frac), float(mid_frac), _ptr(y, torch.float32, "y"),
                                     _ptr(a_out, torch.float32, "a_out"), _stream(stream)))
    return y


def spax_ffn_decode(layer: SpaxLayer, Wg, Wu, x, top_frac, mid_frac, y, a_out=None, stream=None):
    torch = _torch()
    _check(load().spax_ffn_decode(layer.handle, _bf16(Wg, "Wg"), _bf16(Wu, "Wu"), _bf16(x, "x"), float(top_frac),
                                  float(mid_frac), _ptr(y, torch.float32, "y"),
                                  _ptr(a_out, torch.float32, "a_out"), _stream(stream)))
    return y


def spax_encode_rows(W, bits=4, group=128, stream=None) -> SpaxLayer:
    """Encodes a gate or up matrix W [N x d] for spax_gate_up: its columns
    (input channels) get the records, with groups along the N neurons."""
    N, d = W.shape
    h = C.c_void_p()
    _check(load().spax_encode(_bf16(W, "W"), N, d, int(bits), int(group), C.byref(h), _stream(stream)))
    return SpaxLayer(h)


def spax_gate_up(gate: SpaxLayer, up: SpaxLayer, x, top_frac, mid_frac, a, top_idx=None, mid_idx=None, stream=None):
    """a = silu(g) * u with g, u tiered over the input channels by |x|."""
    torch = _torch()
    _check(load().spax_gate_up(gate.handle, up.handle, _bf16(x, "x"), float(top_frac), float(mid_frac),
                               _ptr(a, torch.float32, "a"), _ptr(top_idx, torch.int32, "top_idx"),
                               _ptr(mid_idx, torch.int32, "mid_idx"), _stream(stream)))
    return a


def spax_all_decode(down: SpaxLayer, gate: SpaxLayer, up: SpaxLayer, x, in_top, in_mid, top_frac, mid_frac, y,
                    a_out=None, stream=None):
    """One SpAx-ALL FFN token: gate/up tiers by |x|, then the down tiers by |a|."""
    torch = _torch()
    _check(load().spax_all_decode(down.handle, gate.handle, up.handle, _bf16(x, "x"), float(in_top), float(in_mid),
                                  float(top_frac), float(mid_frac), _ptr(y, torch.float32, "y"),
                                  _ptr(a_out, torch.float32, "a_out"), _stream(stream)))
    return y
