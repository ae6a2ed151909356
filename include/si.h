/*
 * si.h -- C ABI of the GB300 (sm_103a) activation-sparse FFN library.
 *
 * Method sources (cited per entry point below):
 *   [SI]   "SelectInfer: Selective Neuron Loading and Computation for
 *          On-Device LLMs" (arXiv 2607.18081v1): section 3 LLM Profiler,
 *          Eq. (1); section 4 Selective Loading, Fig. 6; section 5 Selective
 *          Computation, Fig. 7; section 6.6 Eq. (2); Table 1.
 *   [SPAX] "Activation Sparsity with Weight Approximation for Faster LLM
 *          Decoding on Offloaded Weights": abstract; Fig. 2 (offline
 *          encoding, per-token tier choice); Fig. 3 (middle-tier column
 *          rebuilt from its own b-bit codes).
 *   [WI]   WiSparse ("Weight-aware Mixed-Granularity Training-free
 *          Activation Sparsity"), abstract: activation magnitudes combined
 *          with precomputed weight norms (si_layer_set_salience).
 *   [LS]   "LeanStream: A Speculate-and-Refine Streaming Framework for
 *          Efficient on-Device LLM Inference", permutation-invariant
 *          execution: a SwiGLU FFN output is a sum over hidden neurons, so
 *          neuron order in memory is free.
 *
 * Conventions (all entry points):
 *   - Every function returns an int status: SI_OK, or an SI_ERR_* code;
 *     si_last_error_string() then describes the failure (thread-local).
 *     Nothing throws or aborts across this boundary.
 *   - Pointers are DEVICE pointers unless the argument is marked (host).
 *     The caller owns inputs and outputs; the library owns the si_layer /
 *     spax_layer handles and everything inside them.
 *   - Every entry point that launches work or waits on the device opens an
 *     NVTX range named after itself for the length of the call (visible to
 *     Nsight tools; a pointer check when none is attached).
 *   - bf16 tensors are passed as uint16_t bit patterns. HF layouts:
 *     Wg, Wu are [N x d] row-major (neuron n = row n), Wd is [d x N]
 *     row-major (neuron n = column n). Activations X are [rows x d].
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued asynchronously on it; calls that allocate
 *     (layer creation, first use of a larger scratch size) do so before
 *     enqueueing and must not run during stream capture.
 *   - Ratios follow the pages' parameters (gamma loaded, delta static, phi
 *     computed = delta + epsilon, tier fractions); a count is
 *     si_count(ratio, N) = floor(ratio*N + 0.5) in double.
 *   - Calls that use the same handle must not overlap on the GPU (they
 *     share the handle's scratch); order them on one stream.
 *   - Kernels never spin without a bound. A bounded wait that runs out sets
 *     a device error word, read with si_device_error().
 */
#ifndef SI_H
#define SI_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SI_OK 0
#define SI_ERR_INVALID_ARG 1
#define SI_ERR_CUDA 2
#define SI_ERR_OOM 3
#define SI_ERR_UNSUPPORTED 4
#define SI_ERR_DEVICE 5

typedef struct si_layer si_layer;
typedef struct spax_layer spax_layer;

/* ------------------------------------------------------------ utilities */

/* Message of the last failing call on this thread ("" if none). The string
 * is owned by the library and valid until the next call on this thread. */
const char *si_last_error_string(void);

/* ABI version of this header (increments on incompatible change). */
int si_abi_version(void);

/* Count of neurons for a ratio: floor(ratio * n + 0.5) computed in double.
 * [SI] section 4/5 and Table 1 give ratios; counts round to nearest. */
long long si_count(double ratio, long long n);

/* Counts used by selective loading/computation for a layer of N neurons:
 * n_loaded = si_count(gamma, N), n_static = si_count(delta, N),
 * n_sel = si_count(phi, N), beta = n_sel - n_static ([SI] section 5:
 * static + dynamic until phi = delta + epsilon). Any output pointer (host)
 * may be NULL. Fails with SI_ERR_INVALID_ARG unless
 * 0 <= delta <= phi <= gamma <= 1 and N >= 1. */
int si_counts(int N, double gamma, double delta, double phi,
              int *n_loaded, int *n_static, int *n_sel, int *beta);

/* Bytes one packed layer keeps for n_loaded neurons of width d: gate row, up
 * row and down column per neuron at 2 bytes per parameter (the complement of
 * [SI] Eq. (2)'s saving, before tile padding). */
long long si_packed_bytes(int d, int n_loaded);

/* Layer range of selection, [SI] section 6.4 Table 1 (first layer 5, last
 * layer -2: "skip last 2"): sparse[l] (host, L bytes) = 1 for the layers
 * first <= l < end that run selective loading and computation, 0 for the
 * layers that keep their dense FFN. `last` is a slice end: end = L + last
 * when last <= 0, else end = last, clipped to L. A dense layer runs through
 * the same decode with a layer packed at gamma = 1 and S = every position
 * (phi = 1). Returns SI_OK and the number of sparse layers in *n_sparse
 * (may be NULL); SI_ERR_INVALID_ARG for L < 0, first < 0 or sparse NULL
 * with L > 0. */
int si_sparse_layers(int L, int first, int last, uint8_t *sparse, int *n_sparse);

/* Reads (and with clear != 0 resets) the device error words of the current
 * device: the one every entry point's kernels write, and the one of
 * si_sparse_ffn_decode_noalloc (inside its static array). *code (host)
 * receives 0 when no kernel reported a failure, else the bit set (OR of both
 * words) of SI_DEVERR_* values. Synchronises the device; allocates nothing. */
#define SI_DEVERR_WAIT_TIMEOUT 1u   /* a bounded mbarrier wait ran out */
#define SI_DEVERR_COUNT 2u          /* an index or count check failed (bad S / tier list, count mismatch) */
#define SI_DEVERR_RANGE 4u          /* a decode partial exceeded a fixed-point accumulator's range (|y| >= 2^23) */
/* With SI_DEVERR_WAIT_TIMEOUT, bits 8-15 name the kernel whose wait ran out
 * (1 sparse decode, 2 dense activation pass, 3 tiered down-projection,
 * 4 activation GEMM, 5 decode stack) and bits 16-19 the barrier (1 stage
 * full, 2 stage empty, 3 stage full in the down-projection phase,
 * 4 accumulator ready, 5 grid barrier between layers). */
int si_device_error(uint32_t *code, int clear);

/* --------------------------------------------------- a1: profiler score */

/* Profiler score, [SI] section 3 Eq. (1): scores[n] += sum_t |a_n(x_t)| with
 * a_n(x) = silu(Wg[n].x) * (Wu[n].x), the down_proj input. Runs on the
 * tcgen05 tensor cores (bf16 inputs, fp32 accumulation).
 *   Wg, Wu  bf16 [N x d]; X bf16 [T x d]; scores fp32 [N], accumulated (the
 *   caller zeroes it and keeps the token count for merging).
 * Requires d % 64 == 0, N >= 1, T >= 1. */
int si_profile_scores(const uint16_t *Wg, const uint16_t *Wu, int d, int N,
                      const uint16_t *X, int T, float *scores, void *stream);

/* Merge of score files, [SI] section 3: out[n] = sum over files f (in the
 * given order) of scores[f][n] / (float)token_counts[f], in float32.
 *   scores (host array of nfiles DEVICE pointers, each fp32 [N]);
 *   token_counts (host) int64 [nfiles], each >= 1; out fp32 [N] (device).
 * 1 <= nfiles <= 16. */
int si_merge_scores(const float *const *scores, const long long *token_counts, int nfiles,
                    int N, float *out, void *stream);

/* Score files, [SI] section 3: the profiler's per-neuron scores of one
 * calibration set are stored in a score file with the number of tokens they
 * were summed over, so that files from several sets can be merged later
 * (si_merge_scores) and the merged scores ranked (si_pack_loaded).
 * File layout (little-endian): the 8 bytes "SISCORE1", int32 N, int32 0,
 * int64 token_count, N float32 scores, then a uint32 FNV-1a checksum of
 * every preceding byte.
 *   si_scores_save: scores (host) fp32 [N], N >= 1, token_count >= 1;
 *     writes `path` (replacing it) through a temporary file and a rename.
 *   si_scores_load: reads `path`; *N_out and *token_count_out (host)
 *     receive the stored N and count; scores (host) fp32 [capacity]
 *     receives the scores when capacity >= N (when it is smaller, or scores
 *     is NULL, only *N_out and *token_count_out are set and the call returns
 *     SI_OK, so a caller can size its buffer first).
 * SI_ERR_INVALID_ARG for NULL path / counts, N < 1, token_count < 1, a
 * missing or short file, another magic, or a checksum that does not match;
 * SI_ERR_CUDA never (host only: no CUDA call). */
int si_scores_save(const char *path, const float *scores, int N, long long token_count);
int si_scores_load(const char *path, float *scores, int capacity, int *N_out, long long *token_count_out);

/* ------------------------------------------------- a2: selective loading */

/* Selective loading, [SI] section 4 / Fig. 6: base (static) neurons are the
 * top si_count(delta, N) by task_scores; secondary neurons are the top by
 * model_scores among the rest until si_count(gamma, N) neurons are loaded.
 * Ties go to the lower neuron index. Pass the same pointer twice for a single
 * score file. The loaded neurons are kept in ascending index order in a
 * neuron-major packed buffer [n_pad][3][d] bf16 (gate row, up row, down
 * column contiguous per neuron; [LS] permutation invariance makes the order
 * free), n_pad = n_loaded rounded up to 128, pad rows zero.
 *   Wg, Wu bf16 [N x d], Wd bf16 [d x N]; task_scores, model_scores fp32 [N]
 *   (finite). *out (host) receives a new handle. Synchronous: allocates, then
 *   enqueues the ranking and packing kernels on `stream` and waits for them.
 * Requires d % 64 == 0, N <= 32768, 0 <= delta <= gamma <= 1, n_loaded >= 1. */
int si_pack_loaded(const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd, int d, int N,
                   const float *task_scores, const float *model_scores, double gamma,
                   double delta, si_layer **out, void *stream);

/* Shape of a packed layer; any output (host) may be NULL. */
int si_layer_info(const si_layer *layer, int *d, int *N, int *n_loaded, int *n_static,
                  int *n_pad);

/* Device buffers owned by the layer (read-only for the caller):
 * loaded_idx int32 [n_loaded] (original neuron index of packed position p,
 * ascending), is_static uint8 [n_loaded], packed bf16 [n_pad][3][d].
 * Outputs (host) may be NULL. */
int si_layer_buffers(const si_layer *layer, const int32_t **loaded_idx,
                     const uint8_t **is_static, const uint16_t **packed);

/* Frees the handle and its device memory (synchronises the device first). */
int si_layer_destroy(si_layer *layer);

/* ------------------------------------------ a3..a6: prefill selection */

/* Dynamic neuron selection during prefill, [SI] section 5 / Fig. 7, for B
 * prompts of T tokens each (X rows are sequence-major: row b*T + t):
 *   a3  |A|[r, p] = |a_{loaded[p]}(x_r)| for every loaded neuron, on the
 *       tcgen05 tensor cores (bf16 x bf16 -> fp32, SiLU*up epilogue);
 *   a4  per token, the top-alpha loaded positions by |A| (ties to the lower
 *       position, which is the lower neuron index);
 *   a5  per prompt, how often each position occurs in those lists;
 *   a6  the top-beta positions by count among non-static positions (ties to
 *       the lower position), beta = si_count(phi,N) - n_static, combined with
 *       the static positions.
 *   X bf16 [B*T x d]; S int32 [B x n_sel] receives ascending packed
 *   positions, n_sel = si_count(phi, N); absact_out (optional, may be NULL)
 *   fp32 [B*T x n_pad], 16-byte aligned (the kernel stores it with TMA;
 *   SI_ERR_INVALID_ARG otherwise), receives |A| (pad columns zero).
 * Requires 1 <= alpha <= n_loaded, n_static <= n_sel <= n_loaded, T, B >= 1. */
int si_select_dynamic(si_layer *layer, const uint16_t *X, int T, int B, int alpha, double phi,
                      int32_t *S, float *absact_out, void *stream);

/* Step a3 of si_select_dynamic alone: absact_out fp32 [B*T x n_pad], 16-byte
 * aligned, receives |A| for every token row and packed position (pad columns
 * zero), computed on the tcgen05 tensor cores exactly as si_select_dynamic
 * does. Together with si_select_from_absact(layer, absact_out, n_pad, ...) it
 * gives the same S. */
int si_prefill_absact(si_layer *layer, const uint16_t *X, int T, int B, float *absact_out,
                      void *stream);

/* Neuron-tile width of the activation GEMM behind si_profile_scores,
 * si_select_dynamic and si_prefill_absact. Each launch covers 256 token rows
 * by `bnn` neurons per CTA; bnn = 0 (the default) lets every launch pick,
 * among 64, 80, 96, 112 and 128, the width that fills the GPU's SMs best;
 * 64, 80, 96, 112 or 128 forces that width for every later launch in this
 * process (any other value fails with SI_ERR_INVALID_ARG). A tuning and test
 * knob: the width changes no result, since every output element sums its K
 * products in the same order whatever the tile. */
int si_set_gemm_tile(int bnn);

/* The width (see si_set_gemm_tile) that a launch over M token rows and N
 * neurons would use on the current device right now, in *bnn. */
int si_gemm_tile_for(int M, int N, int *bnn);

/* Ranking key of the prefill selection of this handle (si_select_dynamic and
 * si_prefill_absact): weight_aware = 0 (the default) ranks by |a_n| as
 * SelectInfer does; 1 ranks by the weight-aware salience |a_n| *
 * ||Wd[:, n]||_2 (WiSparse abstract: activation magnitudes combined with
 * precomputed weight norms, read as the size of neuron n's contribution to
 * the FFN output), which is then what absact_out receives. The profiler
 * score (si_profile_scores, Eq. (1)) is unaffected. SI_ERR_INVALID_ARG for
 * other values. */
int si_layer_set_salience(si_layer *layer, int weight_aware);

/* Device pointer (read-only) to the handle's down-column norms: fp32
 * [n_pad], norms[p] = ||Wd[:, loaded[p]]||_2 (float32 sum of squares of the
 * bf16 column, then sqrt), 0 for pad positions; computed by si_pack_loaded. */
int si_layer_norms(const si_layer *layer, const float **norms);

/* Steps a4..a6 of si_select_dynamic on a given |A| matrix (fp32 [B*T x ld],
 * ld >= n_loaded, finite; only the first n_loaded columns are read, and they
 * are ranked by magnitude). Optional outputs (may be NULL): topmask
 * uint32 [B*T x ceil(n_loaded/32)] (bit p%32 of word p/32 set when p is in
 * the row's top-alpha) and counts uint32 [B x n_loaded] (step a5). */
int si_select_from_absact(si_layer *layer, const float *absA, int ld, int T, int B, int alpha,
                          double phi, int32_t *S, uint32_t *topmask, uint32_t *counts,
                          void *stream);

/* --------------------------------------------------- a7: sparse decode */

/* Cluster-granular selection (the PowerInfer-2 neuron clusters the pages
 * quote: contiguous blocks of `cluster` neuron indices, k*cluster ..
 * (k+1)*cluster - 1; when one neuron of a cluster is predicted active the
 * whole cluster is brought in), applied to one computed set: S_out (device
 * int32, capacity n_loaded) receives, ascending, every packed position whose
 * loaded neuron lies in a cluster that holds the neuron of some position of
 * S (device int32 [n_sel], packed positions); *n_out (host) its length. The
 * result is a computed set for si_decode_plan / the decode calls. For B
 * sequences call it once per sequence. Synchronous (reads the count back;
 * not during stream capture). A position of S outside [0, n_loaded) sets
 * SI_DEVERR_COUNT and is ignored. Requires cluster >= 1, 0 <= n_sel <=
 * n_loaded. */
int si_expand_clusters(si_layer *layer, const int32_t *S, int n_sel, int cluster, int32_t *S_out,
                       int *n_out, void *stream);

/* Builds, inside the handle, the decode plan for the computed sets S[b]
 * (b < B): the union of the B ascending lists S[b][0..n_sel) with, per union
 * entry, a bit mask of the sequences that selected it, so decode reads each
 * selected neuron once. Required before decoding with B > 1; optional for
 * B == 1, where it lets decode start streaming the selected weights while the
 * previous kernel on the stream is still finishing (from the second decode
 * call after the plan on; the first one follows the plan kernel and waits for
 * it). S must stay unchanged while the plan is used; calling si_decode_plan
 * again replaces it. Plan and decode calls of a handle go on one stream.
 * Requires 1 <= B <= 8. */
int si_decode_plan(si_layer *layer, const int32_t *S, int n_sel, int B, void *stream);

/* Sparse decode FFN on the computed set, [SI] section 5 (only the selected
 * neurons are computed at decode):
 *   y[b, :] = sum over p in S[b] of a_{loaded[p]}(x_b) * Wd[:, loaded[p]].
 * Reads only the selected packed records (gate row, up row, down column) with
 * bulk copies and reduces over neurons inside the kernel, split over neurons
 * across the SMs. For B == 1 the CTA partials are summed through cluster
 * shared memory and then in a fixed cross-cluster order. For 2 <= B <= 8 at
 * d = 1024 or 2048 the gate/up and down products run on the tensor cores
 * (bf16 operands, fp32 accumulation; a enters as two bf16 terms, so it is
 * applied to within 2^-18 |a|) and the CTA partials meet in a grid-wide
 * reduction in a fixed CTA order (a cooperative launch, one CTA per SM);
 * other B > 1 go through cluster shared memory and a fixed cross-cluster
 * order. Either way results are deterministic.
 *   S int32 [B x n_sel] ascending positions (as written by the selection
 *   calls); x bf16 [B x d]; y fp32 [B x d] (overwritten).
 * For B > 1, si_decode_plan(layer, S, n_sel, B) must have been called with
 * the same S pointer, n_sel and B. No allocation: safe to capture. */
int si_sparse_ffn_decode(si_layer *layer, const int32_t *S, int n_sel, int B,
                         const uint16_t *x, float *y, void *stream);

/* Residual form of si_sparse_ffn_decode for one sequence (B == 1):
 * y += sum over p in S of a_{loaded[p]}(x) * Wd[:, loaded[p]], the way a
 * transformer adds the FFN output to its residual stream. The CTAs add their
 * partial sums into y with float atomics as they finish, so there is no
 * cross-CTA pass at the end of the kernel; the order of those additions is
 * not fixed, so repeated calls can differ in the last bits (within fp32
 * rounding of the si_sparse_ffn_decode result). A plan built with
 * si_decode_plan lets a call stream its weights while the previous kernel on
 * the stream finishes. y fp32 [d] (read and written). */
int si_sparse_ffn_decode_residual(si_layer *layer, const int32_t *S, int n_sel, int B,
                                  const uint16_t *x, float *y, void *stream);

/* Batch-1 sparse decode that allocates no memory: the same computation as
 * si_sparse_ffn_decode with B == 1 (y = sum over p in S of a_p(x) * down_p,
 * overwritten, deterministic), for callers that must not call cudaMalloc
 * while they run -- a server that owns all device memory through its own
 * pool, code inside a stream capture, or a process under a hard memory cap.
 * The methods this library implements have no counterpart of it.
 *   packed bf16 [n_records][3][d] neuron records (gate row, up row, down
 *   column), e.g. the buffer si_layer_buffers() returns with n_records =
 *   n_pad; S int32 [n_sel] positions in [0, n_records); x bf16 [d]; y fp32 [d].
 * Its scratch (a 64-bit fixed-point accumulator of d words, a ticket and an
 * error word) lives in one fixed device array of 4096 + 2 words that every
 * GPU loading the library keeps until the process exits, so d is limited to
 * 4096 (larger d fails with SI_ERR_INVALID_ARG); also 256 <= d, d % 64 == 0.
 * The first call on a device looks up that array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * All calls share the array: calls that overlap on the GPU (other streams,
 * other threads) race and give wrong results; order them on one stream.
 * Each call leaves the accumulator and ticket at zero for the next one.
 * Device-side failures (a position outside [0, n_records), a bounded wait that
 * ran out, a partial beyond the accumulator's range) are recorded per launch
 * and moved by the launch's last CTA into a reported word in the same array:
 * read and clear it with si_device_error(). A failed launch's y is not valid;
 * later calls are unaffected (their waits watch only their own launch). */
int si_sparse_ffn_decode_noalloc(const uint16_t *packed, int n_records, int d, const int32_t *S,
                                 int n_sel, const uint16_t *x, float *y, void *stream);

/* Decode stack: one launch per decode token over L sparse FFN layers.
 * [SI] section 5 computes, at every decode step, each layer's FFN on that
 * layer's selected neurons only, the layers one after another. In the pages'
 * models (Llama, Qwen) a layer's FFN reads the RMS-normalised residual stream
 * and adds its output back to it; for a stack of FFN layers (unit norm gain):
 *     for l = 0 .. L-1:  x_l = bf16(h / sqrt(mean(h^2) + 1e-5));
 *                        h += sum over p in S_l of a_p(x_l) * down_p
 * (h in fp32, the mean over the d elements, round to nearest even; a_p and
 * down_p as in si_sparse_ffn_decode). The
 * whole token is one cooperative grid, one CTA per SM: the selected records
 * of layer l+1 stream into the ring while layer l's partial sums are added
 * up across the grid, so the weight stream does not stop at layer
 * boundaries. The sum over a layer's CTAs uses float atomics: repeated calls
 * can differ in the last bits (as si_sparse_ffn_decode_residual).
 *
 * si_stack_create: layers (host array of L handles, 1 <= L <= 64, all of the
 *   same d, d in {256, 512, 1024, 2048, 3072}, else SI_ERR_UNSUPPORTED) are borrowed, not owned: they must
 *   outlive the stack. Allocates (synchronous; not during capture).
 * si_stack_plan: the computed sets, S (host array of L device pointers, each
 *   int32 [n_sel[l]] ascending packed positions of layer l, as the selection
 *   calls write them) and n_sel (host, L counts, 0 <= n_sel[l] <= n_loaded),
 *   are copied into the stack by stream-ordered device copies; the caller may
 *   reuse S afterwards. When the counts differ from the previous plan's, the
 *   call first synchronises the stream and uploads the stack's layer table
 *   (then it must not run during capture); with the same counts it only
 *   enqueues the copies and may be captured.
 * si_sparse_ffn_decode_stack: h fp32 [d] (16-byte aligned) holds the residual
 *   stream; it is read at the start and receives h after layer L-1. x_out
 *   (optional, may be NULL; 16-byte aligned) bf16 [L][d] receives each layer's
 *   input x_l. Needs a plan; calls of one stack go on one stream (they share
 *   its scratch). An index outside a layer's records sets SI_DEVERR_COUNT and
 *   reads record 0; a grid barrier that runs out sets SI_DEVERR_WAIT_TIMEOUT
 *   with kernel id 5 and barrier kind 5 (see si_device_error).
 * si_stack_destroy frees the stack (synchronises the device first). */
typedef struct si_stack si_stack;
int si_stack_create(si_layer *const *layers, int L, si_stack **out);
int si_stack_plan(si_stack *stack, const int32_t *const *S, const int *n_sel, void *stream);
int si_sparse_ffn_decode_stack(si_stack *stack, float *h, uint16_t *x_out, void *stream);
int si_stack_destroy(si_stack *stack);

/* ------------------------------------------------------------- SpAx */

/* SpAx offline encoding, [SPAX] Fig. 2 / Fig. 3: for each column n of Wd and
 * each group of `group` consecutive rows: scale = (max - min) / (2^bits - 1),
 * q = clamp(floor((w - min) / scale + 0.5), 0, 2^bits - 1) (q = 0 when
 * scale == 0), all in float32; a middle-tier weight is rebuilt as
 * min + q * scale. The handle keeps a column-major bf16 copy of Wd (top tier,
 * one contiguous column per neuron) and, per column, one record of
 * rec = d*bits/8 + 8*ng_pad bytes (ng_pad = d/group rounded up to even): the
 * codes (one bit stream per column: element i in bits i*bits .. i*bits +
 * bits - 1, bit k being bit k % 8 of byte k / 8; element 2i in the low
 * nibble of byte i for bits = 4, and 3-bit codes straddle bytes), then
 * ng_pad fp32 (scale, min) pairs, so a middle-tier column is one contiguous
 * read.
 *   Wd bf16 [d x N]. Synchronous (allocates, enqueues, waits).
 * Requires bits 2, 3, 4 or 8 (SI_ERR_UNSUPPORTED otherwise), group a power
 * of two >= 8 dividing d, d % 64 == 0 (d % 128 == 0 for bits = 3),
 * d <= 32768; the tiered down-projection calls need d <= 4096 (an encoding
 * of Wg / Wu for spax_gate_up has d = N neurons). */
int spax_encode(const uint16_t *Wd, int d, int N, int bits, int group, spax_layer **out,
                void *stream);

/* Shape of an encoded layer; outputs (host) may be NULL. */
int spax_layer_info(const spax_layer *layer, int *d, int *N, int *bits, int *group, int *ng_pad);

/* Device buffers of an encoded layer (read-only): WdT bf16 [N][d]; codes
 * points at column 0's record and params at its (scale, min) pairs
 * (codes + d*bits/8); column n's codes and params are at the same offsets
 * n * rec bytes further, rec = d*bits/8 + 8*ng_pad. */
int spax_layer_buffers(const spax_layer *layer, const uint16_t **WdT, const uint8_t **codes,
                       const float **params);

/* Frees the handle (synchronises the device first). */
int spax_layer_destroy(spax_layer *layer);

/* Dense gate/up pass of a SpAx decode token: a[n] = silu(Wg[n].x) *
 * (Wu[n].x) for every neuron (the activation magnitudes that choose the
 * tiers, [SPAX] Fig. 2). Wg, Wu bf16 [N x d]; x bf16 [d]; a fp32 [N]. */
int spax_dense_act(const uint16_t *Wg, const uint16_t *Wu, int d, int N, const uint16_t *x,
                   float *a, void *stream);

/* Three-tier down-projection for one token, [SPAX] abstract / Fig. 2:
 * k_top = si_count(top_frac, N) columns with the largest |a| are read in
 * bf16, the next k_mid = si_count(mid_frac, N) are rebuilt from their codes,
 * the rest skipped (ranking by |a| descending, ties to the lower index):
 *   y = sum_{n in top} a[n] Wd[:, n] + sum_{n in mid} a[n] w^_n.
 *   a fp32 [N] (finite); y fp32 [d] (overwritten, deterministic); top_idx /
 *   mid_idx (optional, may be NULL) int32 [k_top] / [k_mid] receive the tier
 *   lists in ascending column order. Requires top_frac + mid_frac <= 1.
 * The tiers are chosen inside the down-projection kernel from a histogram of
 * |a| that this call builds first; spax_ffn_decode gets that histogram from
 * its dense pass instead. Calls on one handle go on one stream. */
int spax_tiered_down(spax_layer *layer, const float *a, double top_frac, double mid_frac,
                     float *y, int32_t *top_idx, int32_t *mid_idx, void *stream);

/* One SpAx decode token: spax_dense_act, then spax_tiered_down on its a
 * (two kernels: the dense pass also counts the tier histogram).
 * a_out (optional) fp32 [N] receives the activations. */
int spax_ffn_decode(spax_layer *layer, const uint16_t *Wg, const uint16_t *Wu,
                    const uint16_t *x, double top_frac, double mid_frac, float *y,
                    float *a_out, void *stream);

/* SelectInfer x SpAx: the SpAx token restricted to a selected set. Only the
 * n_rows neurons listed in rows (device int32, distinct, in [0, N); e.g. the
 * loaded indices of si_select_dynamic's S) get their gate/up dot products
 * (a[n] = silu(Wg[n].x) * (Wu[n].x)); every other neuron has a = 0. The
 * tiers are then taken inside the selected set: k_top = si_count(top_frac,
 * n_rows) columns by |a| in bf16, the next k_mid = si_count(mid_frac, n_rows)
 * from their codes, the rest (and every unselected column) skipped, so the
 * call reads only the selected rows of Wg/Wu and the top/middle columns of
 * the selected set. y fp32 [d]; a_out (optional) fp32 [N] receives a (zeros
 * outside the set). n_rows = 0 gives y = 0. An index outside [0, N) sets
 * SI_DEVERR_COUNT and reads neuron 0 instead. Requires top_frac, mid_frac
 * >= 0, top_frac + mid_frac <= 1. */
int spax_select_decode(spax_layer *layer, const uint16_t *Wg, const uint16_t *Wu, const int32_t *rows,
                       int n_rows, const uint16_t *x, double top_frac, double mid_frac, float *y,
                       float *a_out, void *stream);

/* SpAx tiers on the gate/up projections by |x| ([SPAX] Table 1 "ALL":
 * every offloaded projection tiered; the FFN part adds gate and up to the
 * down projection; Table 2 "SpAx-ALL"). Input channel j (column j of Wg and
 * of Wu) is ranked by |x_j| (ties to the lower index): the k_top =
 * si_count(top_frac, d) largest are read in bf16, the next k_mid =
 * si_count(mid_frac, d) are rebuilt from their own b-bit codes (Fig. 3), the
 * rest are skipped:
 *   g = sum_{j in top} x_j Wg[:, j] + sum_{j in mid} x_j w^_j,  u likewise,
 *   a[n] = silu(g[n]) * u[n].
 * gate / up: made by spax_encode on Wg / Wu read as [N x d] matrices
 * (spax_encode(Wg, N, d, bits, group, ...): rows = neurons, columns = input
 * channels), same shape, bits and group; N % 4 == 0, d <= 8192.
 *   x bf16 [d]; a fp32 [N] (written); top_idx / mid_idx (optional, may be
 *   NULL) int32 [k_top] / [k_mid] receive the channel tiers, ascending.
 * Requires top_frac, mid_frac >= 0, top_frac + mid_frac <= 1. */
int spax_gate_up(const spax_layer *gate, const spax_layer *up, const uint16_t *x, double top_frac,
                 double mid_frac, float *a, int32_t *top_idx, int32_t *mid_idx, void *stream);

/* One SpAx-ALL decode token for the FFN ([SPAX] Table 1 "ALL"): spax_gate_up
 * with the input-channel fractions in_top_frac / in_mid_frac, then
 * spax_tiered_down on its a with top_frac / mid_frac over the N neurons (two
 * kernels; the gate/up pass also counts the down tiers' histogram).
 *   down: spax_encode of Wd [d x N] (d <= 4096); gate / up as for
 *   spax_gate_up, with rows = the down encoding's columns (N) and columns =
 *   its rows (d). y fp32 [d] (overwritten, deterministic); a_out (optional)
 *   fp32 [N] receives a. Calls on one down handle go on one stream. */
int spax_all_decode(spax_layer *down, const spax_layer *gate, const spax_layer *up, const uint16_t *x,
                    double in_top_frac, double in_mid_frac, double top_frac, double mid_frac, float *y,
                    float *a_out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* SI_H */
