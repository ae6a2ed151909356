"""activation_sparse_gb300 -- neuron-level activation-sparse FFN inference on
GB300 (sm_103a): SelectInfer profiling / selective loading / prefill selection /
sparse decode, and the SpAx three-tier down-projection.

The compute lives in ``libsi.so`` (CUDA kernels behind the C ABI of
``include/si.h``); this package is its thin binding. Importing it loads the
library and raises when it cannot be found or built.
"""
from ._binding import (  # noqa: F401
    SIGNATURES, SIError, Layer, SpaxLayer, load, lib_path,
    si_count, si_counts, si_packed_bytes, si_sparse_layers, si_device_error,
    si_profile_scores, si_merge_scores, si_scores_save, si_scores_load, si_pack_loaded,
    si_select_dynamic, si_prefill_absact, si_select_from_absact,
    si_set_gemm_tile, si_gemm_tile_for, si_layer_set_salience, si_layer_norms,
    si_decode_plan, si_expand_clusters, si_sparse_ffn_decode, si_sparse_ffn_decode_residual, si_sparse_ffn_decode_noalloc,
    Stack, si_stack_create, si_stack_plan, si_sparse_ffn_decode_stack,
    spax_encode, spax_dense_act, spax_tiered_down, spax_ffn_decode, spax_select_decode,
    spax_encode_rows, spax_gate_up, spax_all_decode,
    SI_OK, SI_ERR_INVALID_ARG, SI_ERR_CUDA, SI_ERR_OOM, SI_ERR_UNSUPPORTED, SI_ERR_DEVICE,
)

load()
