// internal.h -- launcher interface between the C-ABI layer (api.cu) and the
// kernels. Not installed; not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace si {

struct SparseDecodeParams {
    const uint16_t* packed;   // [n_pad][3][d] bf16
    int d;
    const int32_t* pos;       // plan positions
    int n_records;            // records in `packed` (positions must be below it)
    const uint32_t* pmask;    // per-entry sequence mask, or nullptr (all sequences)
    const int* n_dev;         // device-resident entry count, or nullptr
    int n_host;               // entry count when n_dev == nullptr
    const uint16_t* x;        // [B][d] bf16
    float* y;                 // [B][d] fp32
    float* part;              // [clusters][B*d] scratch
    long long part_floats;    // capacity of part
    unsigned* tickets;        // [16], zero between launches
    unsigned* err;            // device error word
    int R;                    // ring stages
    int stable_plan;          // pos / n_dev come from a completed decode plan: records may be
                              // streamed before this grid's dependency wait
    unsigned long long* acc;  // [B*d] fixed-point accumulator, zero between launches
    unsigned* acc_ticket;     // zero between launches
    int accumulate;           // 1: y += result with float atomics (no cross-CTA ordering)
    unsigned* err_report;     // optional (overwrite form only): the last CTA moves the bits of *err, which
                              // then covers this launch alone, into *err_report and clears *err
};


// Tier histogram: bin b counts the neurons whose |a| key (the float's bits
// with the sign cleared) has bits 30..20 equal to b; word kTierBins is the
// ticket of the CTAs that have read it (the last one re-zeroes everything).
constexpr int kTierBins = 2048;
constexpr int kTierShift = 20;
// Per-bin member lists of the tier histogram ("slabs"): bin b's first
// kSlabCap members (neuron indices, any order) at slab + b * kSlabCap. A bin
// whose count exceeds kSlabCap has an incomplete list and is not read.
constexpr int kSlabCap = 512;

struct DenseActParams {
    const uint16_t* Wg;
    const uint16_t* Wu;
    int d, N;
    const uint16_t* x;
    float* a;
    unsigned* hist;           // optional tier histogram of a (kTierBins + 1 words, zero on entry)
    int32_t* slab;            // optional per-bin member lists of hist ([kTierBins][kSlabCap]); needs hist
    const int32_t* rows;      // optional: compute only these n_rows neurons (others untouched, counted as a = 0)
    int n_rows;
    unsigned* err;
    int R;
};

struct TieredDownParams {
    const uint16_t* WdT;      // [N][d] bf16
    const uint8_t* codes;     // [N] records of rec_bytes: d*bits/8 code bytes, then ngp (scale, min) pairs
    int rec_bytes;
    int bits;                 // code width: 2, 3, 4 or 8
    const float* a;           // [N]
    unsigned* hist;           // tier histogram of a (kTierBins + 1 words), re-zeroed by the kernel
    const int32_t* slab;      // optional per-bin member lists of hist (see kSlabCap)
    int32_t* top_out;         // optional [k_top]: the top tier, ascending
    int32_t* mid_out;         // optional [k_mid]: the middle tier, ascending
    int d, group, ngp, k_top, k_mid;
    int N;                    // columns
    float* y;                 // [d]
    float* part;
    long long part_floats;
    unsigned* tickets;
    unsigned* err;
    int ring_bytes;           // shared-memory ring (split into one byte ring per warp)
    int aux_floats;           // per-CTA buffer: activations in the first half, columns in the second
};

// SpAx tiers on the gate/up projections by |x| (spax_in.cu). Channel j of the
// gate (up) weights is column j of Wg (Wu): WgT [d][N] bf16 holds the columns
// contiguously, gcodes [d] the per-channel records (N*bits/8 code bytes, then
// ngp (scale, min) pairs for groups of `group` consecutive neurons).
struct GateUpTierParams {
    const uint16_t* WgT;
    const uint16_t* WuT;
    const uint8_t* gcodes;
    const uint8_t* ucodes;
    int rec_bytes, bits, group;
    int d, N;                 // input channels, neurons
    const uint16_t* x;        // [d] bf16
    int k_top, k_mid;         // channel tiers
    float* a;                 // [N] out
    unsigned* hist;           // optional tier histogram of a (kTierBins + 1 words, zero on entry)
    int32_t* slab;            // optional member lists of hist
    int32_t* top_out;         // optional [k_top] channel lists, ascending
    int32_t* mid_out;         // optional [k_mid]
    int S;                    // neurons per CTA (multiple of 4, <= 128)
    unsigned* err;
};
int spax_gate_up_slice(int N);
size_t spax_gate_up_smem(int d, int S);
cudaError_t launch_spax_gate_up(const GateUpTierParams& P, cudaStream_t st);

// select.cu
cudaError_t launch_topk_alpha(const float* absA, int ld, int n, int T, int B, int alpha, uint32_t* counts,
                              uint32_t* topmask, cudaStream_t st);
cudaError_t launch_topk_beta(const uint32_t* counts, const uint8_t* is_static, int n, int B, int beta, int n_sel,
                             int32_t* S, unsigned* err, cudaStream_t st);
cudaError_t launch_rank_loaded(const float* task, const float* model, int N, int n_base, int n_load,
                               int32_t* loaded, uint8_t* is_static, unsigned* err, cudaStream_t st);
cudaError_t launch_decode_plan(const int32_t* S, int n_sel, int B, int n, int32_t* pos, uint32_t* pmask,
                               int* count, unsigned* err, cudaStream_t st);
cudaError_t launch_expand_clusters(const int32_t* loaded, int n_loaded, const int32_t* S, int n_sel, int N,
                                  int csize, int32_t* out, int* count, unsigned* err, cudaStream_t st);
cudaError_t launch_merge_scores(const float* const* s, const float* tok, int nfiles, int N, float* out,
                                cudaStream_t st);

// pack.cu
cudaError_t launch_pack_loaded(const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, int d, int N,
                               const int32_t* loaded, int n_loaded, int n_pad, uint16_t* packed, cudaStream_t st);
cudaError_t launch_down_norms(const uint16_t* packed, int d, int n_loaded, int n_pad, float* norms, cudaStream_t st);
cudaError_t launch_spax_encode(const uint16_t* Wd, int d, int N, int bits, int group, int ngp, uint16_t* WdT,
                               uint8_t* recs, int rec_bytes, cudaStream_t st);

// api.cu: sets the message si_last_error_string() returns on this thread
void set_error_message(const char* msg);

// One layer of a decode stack: the packed records of a handle and the copy of
// its computed set that si_stack_plan made.
struct StackLayerDesc {
    const uint16_t* packed;   // [n_records][3][d] bf16
    const int32_t* pos;       // n ascending packed positions
    int n;
    int n_records;
};

constexpr int kStackMaxLayers = 64;
// Layer sums: kDeltaCopies copies of [d] per layer (CTA b adds into copy
// b % kDeltaCopies). Grid barrier of layer l: kBarLines counters, each in its
// own 128-byte line (kLineWords words); then the exit ticket and the launch's
// error word, each in its own line.
constexpr int kDeltaCopies = 4;
constexpr int kBarLines = 16;
constexpr int kLineWords = 32;
__host__ __device__ inline int stack_bar_word(int l, int k) { return (l * kBarLines + k) * kLineWords; }
__host__ __device__ inline int stack_ticket_word(int L) { return L * kBarLines * kLineWords; }
__host__ __device__ inline int stack_lerr_word(int L) { return (L * kBarLines + 1) * kLineWords; }
__host__ __device__ inline int stack_sync_words(int L) { return (L * kBarLines + 2) * kLineWords; }

struct StackParams {
    const StackLayerDesc* layers;  // [L], device
    int L, d, R;
    float* h;                 // [d] residual stream: read at entry, written at exit
    uint16_t* x_out;          // optional [L][d]: the bf16 input each layer used
    float* delta;             // [L][kDeltaCopies][d] per-layer output sums, zero on entry (the kernel
                              // re-zeroes them)
    unsigned* sync;           // [stack_sync_words(L)] barrier counters, exit ticket, the launch's error
                              // word; zero on entry (the kernel re-zeroes them)
    unsigned* err;            // device error word (the launch's failures are moved here at exit)
};

// stack.cu
int sparse_decode_stack_stages(int d);
cudaError_t launch_sparse_decode_stack(const StackParams& P, cudaStream_t st);

// noalloc.cu: device address of the no-allocation entry point's reported
// error word on the current device (looked up once per device; allocates nothing)
int noalloc_error_word(unsigned** out);

// decode.cu
int sparse_decode_b1_stages(int d, int extra_static = 0);  // extra: static shared memory beyond the usual 2 KB
int sparse_decode_stages(int d, int B);
int decode_max_partial_floats(int d, int B);
cudaError_t launch_sparse_decode(SparseDecodeParams P, int B, cudaStream_t st);
int dense_act_stages(int d);
cudaError_t launch_dense_act(DenseActParams P, cudaStream_t st);
cudaError_t launch_abs_hist(const float* a, int N, unsigned* hist, int32_t* slab, cudaStream_t st);
int tiered_down_ring(int d, int aux_floats, int rec_bytes);
int tiered_max_partial_floats(int d);  // partial floats for the tiered kernel (at most one per CTA, one CTA per SM)
cudaError_t launch_tiered_down(TieredDownParams P, cudaStream_t st);
int streaming_grid_upper_bound();

// gemm.cu -- tcgen05 activation GEMM: rows of X against gate/up row pairs.
//   mode 0: out[r * ldo + p] = |silu(g) * u| for r < M, p < Npad (fp32)
//   mode 1: colsum[p] += sum_r |silu(g) * u| over r < M, p < Nvalid
struct ActGemmParams {
    const uint16_t* X;        // [M][K] bf16
    int M, K;
    const uint16_t* Wgate;    // row p at Wgate + p * w_stride (elements)
    const uint16_t* Wup;      // row p at Wup + p * w_stride
    long long w_stride;       // elements between consecutive neuron rows
    int Nrows;                // rows addressable in the weight tensors
    int Nvalid;               // columns written / summed
    int mode;
    float* out;
    long long ldo;
    const float* wnorm;       // optional [Nvalid]: mode 0 writes |a| * wnorm[col] (weight-aware salience)
    float* colsum;
    unsigned* err;
};
cudaError_t launch_act_gemm(const ActGemmParams& P, cudaStream_t st);
// Neuron-tile width override for the activation GEMM (0 = per-launch choice).
cudaError_t set_gemm_tile(int bnn);
// The width a launch over M token rows and Nvalid neurons would use now.
int gemm_tile_for(int M, int Nvalid);

}  // namespace si
