// api.cu -- the C ABI declared in include/si.h: argument validation, handle
// lifetime, scratch management and kernel launches. No arithmetic of the
// method happens here; every step runs in the kernels.
#include <vector>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/si.h"
#include "internal.h"
#include <nvtx3/nvToolsExt.h>

namespace {
// An NVTX range named after the entry point, open for the call (a pointer
// check when no profiler is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace
#define SI_TRACE(name) NvtxRange si_trace_range_(name)

namespace {

thread_local std::string g_msg;

int fail(int code, const std::string& msg) {
    g_msg = msg;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    g_msg = std::string(what) + ": " + cudaGetErrorString(e);
    return e == cudaErrorMemoryAllocation ? SI_ERR_OOM : SI_ERR_CUDA;
}

#define SI_CK(call)                                        \
    do {                                                   \
        cudaError_t e_ = (call);                           \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

long long count_of(double r, long long n) { return (long long)std::floor(r * (double)n + 0.5); }

int round_up(int x, int m) { return (x + m - 1) / m * m; }

bool capturing(cudaStream_t st) {
    cudaStreamCaptureStatus s = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &s) != cudaSuccess) return false;
    return s != cudaStreamCaptureStatusNone;
}

// Device error word, one per device, allocated on first use.
std::mutex g_err_mu;
unsigned* g_err_word[128] = {};

int err_word(unsigned** out) {
    int dev = 0;
    SI_CK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 128) return fail(SI_ERR_UNSUPPORTED, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_word[dev]) {
        unsigned* p = nullptr;
        SI_CK(cudaMalloc(&p, sizeof(unsigned)));
        SI_CK(cudaMemset(p, 0, sizeof(unsigned)));
        g_err_word[dev] = p;
    }
    *out = g_err_word[dev];
    return SI_OK;
}

template <class T>
int dalloc(T** p, size_t count, const char* what) {
    *p = nullptr;
    if (count == 0) count = 1;
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(SI_ERR_OOM, std::string("cudaMalloc failed for ") + what);
    }
    return SI_OK;
}

template <class T>
void dfree(T*& p) {
    if (p) cudaFree(p);
    p = nullptr;
}

bool ratios_ok(double delta, double phi, double gamma) {
    return std::isfinite(delta) && std::isfinite(phi) && std::isfinite(gamma) && delta >= 0.0 && delta <= phi &&
           phi <= gamma && gamma <= 1.0;
}

}  // namespace

namespace si {
void set_error_message(const char* msg) { g_msg = msg; }
}  // namespace si

struct si_layer {
    int device = 0;
    int d = 0, N = 0, n_loaded = 0, n_static = 0, n_pad = 0;
    int32_t* loaded = nullptr;
    uint8_t* is_static = nullptr;
    uint16_t* packed = nullptr;
    float* wnorm = nullptr;     // ||Wd[:, n]||_2 per packed position (pads 0)
    int salience = 0;           // 1: prefill ranks by |a| * wnorm (weight-aware)
    uint32_t* counts = nullptr;
    int counts_B = 0;
    float* absA = nullptr;
    size_t absA_floats = 0;
    float* part = nullptr;
    long long part_floats = 0;
    unsigned* tickets = nullptr;
    unsigned long long* acc = nullptr;  // batch-1 decode accumulator [d] (+ its ticket in tickets[15])
    int32_t* plan_pos = nullptr;
    uint32_t* plan_mask = nullptr;
    int* plan_n = nullptr;
    int* cluster_n = nullptr;   // count of si_expand_clusters (allocated on first use)
    const int32_t* plan_S = nullptr;
    int plan_nsel = -1, plan_B = 0;
    // True from si_decode_plan until the next decode launch on this handle: that
    // launch may directly follow the plan kernel, so it reads the plan only after
    // its dependency wait; later launches are ordered after it and may stream early.
    bool plan_fresh = false;
};

struct spax_layer {
    int device = 0;
    int d = 0, N = 0, bits = 0, group = 0, ngp = 0;
    uint16_t* WdT = nullptr;
    uint8_t* codes = nullptr;
    float* params = nullptr;    // inside the records: codes + d / 2 (not a separate allocation)
    int rec_bytes = 0;          // per-column record: d * bits / 8 code bytes, then ngp (scale, min) pairs
    unsigned* hist = nullptr;  // tier histogram of the current a (zero between calls) + its ticket
    int32_t* slab = nullptr;   // the histogram's per-bin member lists [kTierBins][kSlabCap]
    float* a = nullptr;
    float* part = nullptr;
    long long part_floats = 0;
    unsigned* tickets = nullptr;
};

// A decode stack: L packed layers (not owned) decoded one token at a time by
// one launch (si_sparse_ffn_decode_stack).
struct si_stack {
    int device = 0;
    int L = 0, d = 0;
    si_layer* layers[si::kStackMaxLayers] = {};
    long long pos_off[si::kStackMaxLayers + 1] = {};  // offsets of the plan copies in pos
    int32_t* pos = nullptr;                  // plan copies of the computed sets (capacity sum of n_loaded)
    si::StackLayerDesc* desc = nullptr;      // [L] device
    si::StackLayerDesc* desc_host = nullptr; // [L] pinned host staging of desc
    float* delta = nullptr;                  // [L][kDeltaCopies][d], zero between launches
    unsigned* sync = nullptr;                // barrier counters, ticket, error word; zero between launches
    bool planned = false;
};

namespace {

int grow_part(float** part, long long* cap, int d, int B) {
    const long long need = si::decode_max_partial_floats(d, B);
    if (need <= 0) return fail(SI_ERR_CUDA, "cannot query the device for the decode grid");
    if (*cap >= need) return SI_OK;
    dfree(*part);
    *cap = 0;
    int rc = dalloc(part, (size_t)need, "decode partials");
    if (rc) return rc;
    *cap = need;
    return SI_OK;
}

void destroy_layer(si_layer* L) {
    if (!L) return;
    dfree(L->loaded);
    dfree(L->is_static);
    dfree(L->packed);
    dfree(L->wnorm);
    dfree(L->counts);
    dfree(L->absA);
    dfree(L->part);
    dfree(L->tickets);
    dfree(L->acc);
    dfree(L->plan_pos);
    dfree(L->plan_mask);
    dfree(L->plan_n);
    dfree(L->cluster_n);
    delete L;
}

void destroy_spax(spax_layer* L) {
    if (!L) return;
    dfree(L->WdT);
    dfree(L->codes);
    dfree(L->hist);
    dfree(L->slab);
    dfree(L->a);
    dfree(L->part);
    dfree(L->tickets);
    delete L;
}

int select_core(si_layer* L, const float* absA, int ld, int T, int B, int alpha, double phi, int32_t* S,
                uint32_t* topmask, uint32_t* counts, cudaStream_t st) {
    const long long n_sel = count_of(phi, L->N);
    if (n_sel < L->n_static || n_sel > L->n_loaded)
        return fail(SI_ERR_INVALID_ARG, "phi must give n_static <= n_sel <= n_loaded");
    const int beta = (int)n_sel - L->n_static;
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    uint32_t* cnt = counts;
    if (!cnt) {
        if (L->counts_B < B) {
            if (capturing(st)) return fail(SI_ERR_INVALID_ARG, "count scratch must grow; call once before capture");
            dfree(L->counts);
            L->counts_B = 0;
            rc = dalloc(&L->counts, (size_t)B * L->n_loaded, "selection counts");
            if (rc) return rc;
            L->counts_B = B;
        }
        cnt = L->counts;
    }
    SI_CK(cudaMemsetAsync(cnt, 0, (size_t)B * L->n_loaded * sizeof(uint32_t), st));
    SI_CK(si::launch_topk_alpha(absA, ld, L->n_loaded, T, B, alpha, cnt, topmask, st));
    SI_CK(si::launch_topk_beta(cnt, L->is_static, L->n_loaded, B, beta, (int)n_sel, S, err, st));
    return SI_OK;
}

}  // namespace

extern "C" {

const char* si_last_error_string(void) { return g_msg.c_str(); }

int si_abi_version(void) { return 1; }

long long si_count(double ratio, long long n) { return count_of(ratio, n); }

int si_sparse_layers(int L, int first, int last, uint8_t* sparse, int* n_sparse) {
    if (L < 0 || first < 0) return fail(SI_ERR_INVALID_ARG, "need L >= 0, first >= 0");
    if (L > 0 && !sparse) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    const long long end_raw = last <= 0 ? (long long)L + last : (long long)last;
    const long long end = end_raw > L ? L : end_raw;
    int n = 0;
    for (int l = 0; l < L; ++l) {
        const bool in = l >= first && l < end;
        sparse[l] = in ? 1 : 0;
        n += in ? 1 : 0;
    }
    if (n_sparse) *n_sparse = n;
    return SI_OK;
}

int si_counts(int N, double gamma, double delta, double phi, int* n_loaded, int* n_static, int* n_sel, int* beta) {
    if (N < 1 || !ratios_ok(delta, phi, gamma))
        return fail(SI_ERR_INVALID_ARG, "need N >= 1 and 0 <= delta <= phi <= gamma <= 1");
    const long long nl = count_of(gamma, N), ns = count_of(delta, N), nq = count_of(phi, N);
    if (n_loaded) *n_loaded = (int)nl;
    if (n_static) *n_static = (int)ns;
    if (n_sel) *n_sel = (int)nq;
    if (beta) *beta = (int)(nq - ns);
    return SI_OK;
}

long long si_packed_bytes(int d, int n_loaded) { return 3LL * d * n_loaded * 2; }

int si_device_error(uint32_t* code, int clear) {
    SI_TRACE("si_device_error");
    if (!code) return fail(SI_ERR_INVALID_ARG, "code is NULL");
    int dev = 0;
    SI_CK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 128) return fail(SI_ERR_UNSUPPORTED, "device ordinal out of range");
    unsigned* w = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_err_mu);
        w = g_err_word[dev];  // not allocated yet: no kernel has used it, so it reads as 0
    }
    unsigned* wn = nullptr;   // the no-allocation decode's reported word (a static device array)
    int rc = si::noalloc_error_word(&wn);
    if (rc) return rc;
    SI_CK(cudaDeviceSynchronize());
    unsigned v = 0, vn = 0;
    if (w) SI_CK(cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost));
    SI_CK(cudaMemcpy(&vn, wn, sizeof vn, cudaMemcpyDeviceToHost));
    if (clear) {
        if (w) SI_CK(cudaMemset(w, 0, sizeof(unsigned)));
        SI_CK(cudaMemset(wn, 0, sizeof(unsigned)));
    }
    *code = v | vn;
    return SI_OK;
}

// ------------------------------------------------------------------ a1

int si_profile_scores(const uint16_t* Wg, const uint16_t* Wu, int d, int N, const uint16_t* X, int T, float* scores,
                      void* stream) {
    SI_TRACE("si_profile_scores");
    if (!Wg || !Wu || !X || !scores) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (d < 64 || d % 64 || N < 1 || T < 1) return fail(SI_ERR_INVALID_ARG, "need d % 64 == 0, N >= 1, T >= 1");
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    si::ActGemmParams P = {};
    P.X = X;
    P.M = T;
    P.K = d;
    P.Wgate = Wg;
    P.Wup = Wu;
    P.w_stride = d;
    P.Nrows = N;
    P.Nvalid = N;
    P.mode = 1;
    P.colsum = scores;
    P.err = err;
    SI_CK(si::launch_act_gemm(P, (cudaStream_t)stream));
    return SI_OK;
}

int si_merge_scores(const float* const* scores, const long long* token_counts, int nfiles, int N, float* out,
                    void* stream) {
    SI_TRACE("si_merge_scores");
    if (!scores || !token_counts || !out) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (nfiles < 1 || nfiles > 16 || N < 1) return fail(SI_ERR_INVALID_ARG, "need 1 <= nfiles <= 16, N >= 1");
    float tok[16];
    for (int f = 0; f < nfiles; ++f) {
        if (!scores[f]) return fail(SI_ERR_INVALID_ARG, "NULL score file");
        if (token_counts[f] < 1) return fail(SI_ERR_INVALID_ARG, "token counts must be >= 1");
        tok[f] = (float)token_counts[f];
    }
    SI_CK(si::launch_merge_scores(scores, tok, nfiles, N, out, (cudaStream_t)stream));
    return SI_OK;
}

// ----------------------------------------------------------- score files

namespace {

constexpr char kScoreMagic[8] = {'S', 'I', 'S', 'C', 'O', 'R', 'E', '1'};

// 32-bit FNV-1a (offset basis 2166136261, prime 16777619) over a byte range,
// continuing from h
uint32_t fnv1a(const void* data, size_t n, uint32_t h) {
    const unsigned char* p = static_cast<const unsigned char*>(data);
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= 16777619u;
    }
    return h;
}

struct ScoreHeader {
    char magic[8];
    int32_t n;
    int32_t zero;
    int64_t tokens;
};
static_assert(sizeof(ScoreHeader) == 24, "score file header is 24 bytes");

}  // namespace

int si_scores_save(const char* path, const float* scores, int N, long long token_count) {
    SI_TRACE("si_scores_save");
    if (!path || !scores) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (N < 1 || token_count < 1) return fail(SI_ERR_INVALID_ARG, "need N >= 1 and token_count >= 1");
    ScoreHeader h = {};
    std::memcpy(h.magic, kScoreMagic, 8);
    h.n = N;
    h.zero = 0;
    h.tokens = token_count;
    uint32_t sum = fnv1a(&h, sizeof(h), 2166136261u);
    sum = fnv1a(scores, (size_t)N * sizeof(float), sum);
    const std::string tmp = std::string(path) + ".tmp";
    FILE* f = std::fopen(tmp.c_str(), "wb");
    if (!f) return fail(SI_ERR_INVALID_ARG, "cannot open the score file for writing");
    const bool ok = std::fwrite(&h, sizeof(h), 1, f) == 1 &&
                    std::fwrite(scores, sizeof(float), (size_t)N, f) == (size_t)N &&
                    std::fwrite(&sum, sizeof(sum), 1, f) == 1;
    const bool closed = std::fclose(f) == 0;
    if (!ok || !closed || std::rename(tmp.c_str(), path) != 0) {
        std::remove(tmp.c_str());
        return fail(SI_ERR_INVALID_ARG, "cannot write the score file");
    }
    return SI_OK;
}

int si_scores_load(const char* path, float* scores, int capacity, int* N_out, long long* token_count_out) {
    SI_TRACE("si_scores_load");
    if (!path || !N_out || !token_count_out) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    FILE* f = std::fopen(path, "rb");
    if (!f) return fail(SI_ERR_INVALID_ARG, "cannot open the score file");
    ScoreHeader h = {};
    const bool head = std::fread(&h, sizeof(h), 1, f) == 1;
    if (!head || std::memcmp(h.magic, kScoreMagic, 8) != 0 || h.n < 1 || h.zero != 0 || h.tokens < 1) {
        std::fclose(f);
        return fail(SI_ERR_INVALID_ARG, "not a score file (magic, N or token count)");
    }
    std::vector<float> v((size_t)h.n);
    uint32_t stored = 0;
    unsigned char extra;
    const bool body = std::fread(v.data(), sizeof(float), v.size(), f) == v.size() &&
                      std::fread(&stored, sizeof(stored), 1, f) == 1 && std::fread(&extra, 1, 1, f) == 0;
    std::fclose(f);
    if (!body) return fail(SI_ERR_INVALID_ARG, "score file is short or has trailing bytes");
    uint32_t sum = fnv1a(&h, sizeof(h), 2166136261u);
    sum = fnv1a(v.data(), v.size() * sizeof(float), sum);
    if (sum != stored) return fail(SI_ERR_INVALID_ARG, "score file checksum does not match");
    *N_out = h.n;
    *token_count_out = h.tokens;
    if (scores && capacity >= h.n) std::memcpy(scores, v.data(), v.size() * sizeof(float));
    return SI_OK;
}

// ------------------------------------------------------------------ a2

int si_pack_loaded(const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, int d, int N, const float* task_scores,
                   const float* model_scores, double gamma, double delta, si_layer** out, void* stream) {
    SI_TRACE("si_pack_loaded");
    if (!out) return fail(SI_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!Wg || !Wu || !Wd || !task_scores || !model_scores) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (d < 64 || d % 64) return fail(SI_ERR_INVALID_ARG, "need d % 64 == 0");
    if (N < 1 || N > 32768) return fail(SI_ERR_INVALID_ARG, "need 1 <= N <= 32768");
    if (!ratios_ok(delta, delta, gamma)) return fail(SI_ERR_INVALID_ARG, "need 0 <= delta <= gamma <= 1");
    const int n_loaded = (int)count_of(gamma, N), n_static = (int)count_of(delta, N);
    if (n_loaded < 1) return fail(SI_ERR_INVALID_ARG, "gamma loads no neuron");
    cudaStream_t st = (cudaStream_t)stream;
    if (capturing(st)) return fail(SI_ERR_INVALID_ARG, "si_pack_loaded allocates; not allowed during capture");
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    si_layer* L = new si_layer();
    SI_CK(cudaGetDevice(&L->device));
    L->d = d;
    L->N = N;
    L->n_loaded = n_loaded;
    L->n_static = n_static;
    L->n_pad = round_up(n_loaded, 128);
    if ((rc = dalloc(&L->loaded, n_loaded, "loaded index")) || (rc = dalloc(&L->is_static, n_loaded, "static flags")) ||
        (rc = dalloc(&L->packed, (size_t)L->n_pad * 3 * d, "packed weights")) ||
        (rc = dalloc(&L->wnorm, L->n_pad, "down-column norms")) ||
        (rc = dalloc(&L->tickets, 16, "tickets")) || (rc = dalloc(&L->acc, d, "decode accumulator")) ||
        (rc = grow_part(&L->part, &L->part_floats, d, 1))) {
        destroy_layer(L);
        return rc;
    }
    cudaError_t e = cudaMemsetAsync(L->tickets, 0, 16 * sizeof(unsigned), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L->acc, 0, (size_t)d * sizeof(unsigned long long), st);
    if (e == cudaSuccess) e = si::launch_rank_loaded(task_scores, model_scores, N, n_static, n_loaded, L->loaded,
                                                     L->is_static, err, st);
    if (e == cudaSuccess) e = si::launch_pack_loaded(Wg, Wu, Wd, d, N, L->loaded, n_loaded, L->n_pad, L->packed, st);
    if (e == cudaSuccess) e = si::launch_down_norms(L->packed, d, n_loaded, L->n_pad, L->wnorm, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        destroy_layer(L);
        return cuda_fail(e, "si_pack_loaded");
    }
    *out = L;
    return SI_OK;
}

int si_layer_info(const si_layer* L, int* d, int* N, int* n_loaded, int* n_static, int* n_pad) {
    SI_TRACE("si_layer_info");
    if (!L) return fail(SI_ERR_INVALID_ARG, "layer is NULL");
    if (d) *d = L->d;
    if (N) *N = L->N;
    if (n_loaded) *n_loaded = L->n_loaded;
    if (n_static) *n_static = L->n_static;
    if (n_pad) *n_pad = L->n_pad;
    return SI_OK;
}

int si_layer_buffers(const si_layer* L, const int32_t** loaded_idx, const uint8_t** is_static,
                     const uint16_t** packed) {
    SI_TRACE("si_layer_buffers");
    if (!L) return fail(SI_ERR_INVALID_ARG, "layer is NULL");
    if (loaded_idx) *loaded_idx = L->loaded;
    if (is_static) *is_static = L->is_static;
    if (packed) *packed = L->packed;
    return SI_OK;
}

int si_layer_norms(const si_layer* L, const float** norms) {
    SI_TRACE("si_layer_norms");
    if (!L || !norms) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    *norms = L->wnorm;
    return SI_OK;
}

int si_layer_set_salience(si_layer* L, int weight_aware) {
    SI_TRACE("si_layer_set_salience");
    if (!L) return fail(SI_ERR_INVALID_ARG, "layer is NULL");
    if (weight_aware != 0 && weight_aware != 1) return fail(SI_ERR_INVALID_ARG, "weight_aware must be 0 or 1");
    L->salience = weight_aware;
    return SI_OK;
}

int si_layer_destroy(si_layer* L) {
    SI_TRACE("si_layer_destroy");
    if (!L) return SI_OK;
    cudaDeviceSynchronize();
    destroy_layer(L);
    return SI_OK;
}

// ------------------------------------------------------------ a3 .. a6

int si_select_from_absact(si_layer* L, const float* absA, int ld, int T, int B, int alpha, double phi, int32_t* S,
                          uint32_t* topmask, uint32_t* counts, void* stream) {
    SI_TRACE("si_select_from_absact");
    if (!L || !absA || !S) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (T < 1 || B < 1 || ld < L->n_loaded) return fail(SI_ERR_INVALID_ARG, "need T, B >= 1 and ld >= n_loaded");
    if (alpha < 1 || alpha > L->n_loaded) return fail(SI_ERR_INVALID_ARG, "need 1 <= alpha <= n_loaded");
    if (!std::isfinite(phi)) return fail(SI_ERR_INVALID_ARG, "phi is not finite");
    return select_core(L, absA, ld, T, B, alpha, phi, S, topmask, counts, (cudaStream_t)stream);
}

namespace {

int absact_core(si_layer* L, const uint16_t* X, int M, float* A, cudaStream_t st) {
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    si::ActGemmParams P = {};
    P.X = X;
    P.M = M;
    P.K = L->d;
    P.Wgate = L->packed;
    P.Wup = L->packed + L->d;
    P.w_stride = 3LL * L->d;
    P.Nrows = L->n_pad;
    P.Nvalid = L->n_pad;
    P.mode = 0;
    P.out = A;
    P.ldo = L->n_pad;
    P.wnorm = L->salience ? L->wnorm : nullptr;
    P.err = err;
    SI_CK(si::launch_act_gemm(P, st));
    return SI_OK;
}

}  // namespace

int si_prefill_absact(si_layer* L, const uint16_t* X, int T, int B, float* absact_out, void* stream) {
    SI_TRACE("si_prefill_absact");
    if (!L || !X || !absact_out) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (reinterpret_cast<uintptr_t>(absact_out) & 15u) return fail(SI_ERR_INVALID_ARG, "absact_out must be 16-byte aligned");
    if (T < 1 || B < 1) return fail(SI_ERR_INVALID_ARG, "need T, B >= 1");
    if ((long long)T * B > (1LL << 30) / L->n_pad) return fail(SI_ERR_INVALID_ARG, "T * B too large");
    return absact_core(L, X, T * B, absact_out, (cudaStream_t)stream);
}

int si_set_gemm_tile(int bnn) {
    SI_TRACE("si_set_gemm_tile");
    if (si::set_gemm_tile(bnn) != cudaSuccess) return fail(SI_ERR_INVALID_ARG, "bnn must be 0, 64, 80, 96, 112 or 128");
    return SI_OK;
}

int si_gemm_tile_for(int M, int N, int* bnn) {
    SI_TRACE("si_gemm_tile_for");
    if (!bnn) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (M < 1 || N < 1) return fail(SI_ERR_INVALID_ARG, "need M, N >= 1");
    const int b = si::gemm_tile_for(M, N);
    if (!b) return fail(SI_ERR_CUDA, "no current CUDA device");
    *bnn = b;
    return SI_OK;
}

int si_select_dynamic(si_layer* L, const uint16_t* X, int T, int B, int alpha, double phi, int32_t* S,
                      float* absact_out, void* stream) {
    SI_TRACE("si_select_dynamic");
    if (!L || !X || !S) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (reinterpret_cast<uintptr_t>(absact_out) & 15u) return fail(SI_ERR_INVALID_ARG, "absact_out must be 16-byte aligned");
    if (T < 1 || B < 1) return fail(SI_ERR_INVALID_ARG, "need T, B >= 1");
    if ((long long)T * B > (1LL << 30) / L->n_pad) return fail(SI_ERR_INVALID_ARG, "T * B too large");
    if (alpha < 1 || alpha > L->n_loaded) return fail(SI_ERR_INVALID_ARG, "need 1 <= alpha <= n_loaded");
    if (!std::isfinite(phi)) return fail(SI_ERR_INVALID_ARG, "phi is not finite");
    const long long n_sel = count_of(phi, L->N);
    if (n_sel < L->n_static || n_sel > L->n_loaded)
        return fail(SI_ERR_INVALID_ARG, "phi must give n_static <= n_sel <= n_loaded");
    cudaStream_t st = (cudaStream_t)stream;
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    const int M = T * B;
    float* A = absact_out;
    if (!A) {
        const size_t need = (size_t)M * L->n_pad;
        if (L->absA_floats < need) {
            if (capturing(st)) return fail(SI_ERR_INVALID_ARG, "|A| scratch must grow; call once before capture");
            dfree(L->absA);
            L->absA_floats = 0;
            rc = dalloc(&L->absA, need, "|A| scratch");
            if (rc) return rc;
            L->absA_floats = need;
        }
        A = L->absA;
    }
    rc = absact_core(L, X, M, A, st);
    if (rc) return rc;
    return select_core(L, A, L->n_pad, T, B, alpha, phi, S, nullptr, nullptr, st);
}

// ------------------------------------------------------------------ a7

int si_expand_clusters(si_layer* L, const int32_t* S, int n_sel, int cluster, int32_t* S_out, int* n_out,
                       void* stream) {
    SI_TRACE("si_expand_clusters");
    if (!L || !S_out || !n_out || (n_sel > 0 && !S)) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (cluster < 1) return fail(SI_ERR_INVALID_ARG, "cluster size must be >= 1");
    if (n_sel < 0 || n_sel > L->n_loaded) return fail(SI_ERR_INVALID_ARG, "need 0 <= n_sel <= n_loaded");
    cudaStream_t st = (cudaStream_t)stream;
    if (capturing(st)) return fail(SI_ERR_INVALID_ARG, "si_expand_clusters reads its count back; not during capture");
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    if (!L->cluster_n && (rc = dalloc(&L->cluster_n, 1, "cluster count"))) return rc;
    SI_CK(si::launch_expand_clusters(L->loaded, L->n_loaded, S, n_sel, L->N, cluster, S_out, L->cluster_n, err, st));
    int n = 0;
    SI_CK(cudaMemcpyAsync(&n, L->cluster_n, sizeof(int), cudaMemcpyDeviceToHost, st));
    SI_CK(cudaStreamSynchronize(st));
    *n_out = n;
    return SI_OK;
}

int si_decode_plan(si_layer* L, const int32_t* S, int n_sel, int B, void* stream) {
    SI_TRACE("si_decode_plan");
    if (!L || (!S && n_sel > 0)) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (B < 1 || B > 8) return fail(SI_ERR_INVALID_ARG, "need 1 <= B <= 8");
    if (n_sel < 0 || n_sel > L->n_loaded) return fail(SI_ERR_INVALID_ARG, "need 0 <= n_sel <= n_loaded");
    cudaStream_t st = (cudaStream_t)stream;
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    if (!L->plan_pos) {
        if (capturing(st)) return fail(SI_ERR_INVALID_ARG, "plan buffers must be allocated before capture");
        if ((rc = dalloc(&L->plan_pos, L->n_loaded, "plan positions")) ||
            (rc = dalloc(&L->plan_mask, L->n_loaded, "plan masks")) || (rc = dalloc(&L->plan_n, 1, "plan count")))
            return rc;
    }
    if (L->part_floats < si::decode_max_partial_floats(L->d, B)) {
        if (capturing(st)) return fail(SI_ERR_INVALID_ARG, "partials must grow; call once before capture");
        rc = grow_part(&L->part, &L->part_floats, L->d, B);
        if (rc) return rc;
    }
    if (B == 1) {
        // batch 1: the plan is a copy of S that later calls may read before
        // their dependency wait (nothing but si_decode_plan writes it)
        if (n_sel > 0) SI_CK(cudaMemcpyAsync(L->plan_pos, S, (size_t)n_sel * 4, cudaMemcpyDeviceToDevice, st));
    } else {
        SI_CK(si::launch_decode_plan(S, n_sel, B, L->n_loaded, L->plan_pos, L->plan_mask, L->plan_n, err, st));
    }
    L->plan_fresh = true;
    L->plan_S = S;
    L->plan_nsel = n_sel;
    L->plan_B = B;
    return SI_OK;
}

namespace {
int sparse_decode_impl(si_layer* L, const int32_t* S, int n_sel, int B, const uint16_t* x, float* y,
                       void* stream, bool accumulate);
}

int si_sparse_ffn_decode(si_layer* L, const int32_t* S, int n_sel, int B, const uint16_t* x, float* y,
                         void* stream) {
    SI_TRACE("si_sparse_ffn_decode");
    return sparse_decode_impl(L, S, n_sel, B, x, y, stream, false);
}

int si_sparse_ffn_decode_residual(si_layer* L, const int32_t* S, int n_sel, int B, const uint16_t* x, float* y,
                                  void* stream) {
    SI_TRACE("si_sparse_ffn_decode_residual");
    if (B != 1) return fail(SI_ERR_UNSUPPORTED, "the residual form is implemented for B == 1");
    return sparse_decode_impl(L, S, n_sel, B, x, y, stream, true);
}

}  // extern "C"

namespace {
int sparse_decode_impl(si_layer* L, const int32_t* S, int n_sel, int B, const uint16_t* x, float* y,
                       void* stream, bool accumulate) {
    if (!L || (!S && n_sel > 0) || !x || !y) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (B < 1 || B > 8) return fail(SI_ERR_INVALID_ARG, "need 1 <= B <= 8");
    if (n_sel < 0 || n_sel > L->n_loaded) return fail(SI_ERR_INVALID_ARG, "need 0 <= n_sel <= n_loaded");
    if (L->d > 4096) return fail(SI_ERR_UNSUPPORTED, "decode supports d <= 4096");
    if (B > 1 && (L->plan_S != S || L->plan_nsel != n_sel || L->plan_B != B))
        return fail(SI_ERR_INVALID_ARG, "B > 1 needs si_decode_plan with the same S, n_sel and B first");
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    si::SparseDecodeParams P = {};
    P.packed = L->packed;
    P.n_records = L->n_pad;
    P.d = L->d;
    P.x = x;
    P.y = y;
    P.part = L->part;
    P.part_floats = L->part_floats;
    P.tickets = L->tickets;
    P.acc = L->acc;
    P.acc_ticket = L->tickets + 15;
    P.accumulate = accumulate ? 1 : 0;
    P.err = err;
    P.R = si::sparse_decode_stages(L->d, B);
    if (P.R < 8) return fail(SI_ERR_UNSUPPORTED, "d too large for the decode ring");
    const bool have_plan = L->plan_S == S && L->plan_nsel == n_sel && L->plan_B == B;
    const bool stable = have_plan && !L->plan_fresh;
    P.stable_plan = stable ? 1 : 0;
    if (B == 1) {
        // a batch-1 plan is a copy of S (n_sel entries); the count is the host's
        P.pos = stable ? L->plan_pos : S;
        P.pmask = nullptr;
        P.n_dev = nullptr;
        P.n_host = n_sel;
    } else {
        P.pos = L->plan_pos;
        P.pmask = B > 1 ? L->plan_mask : nullptr;
        P.n_dev = L->plan_n;
        P.n_host = n_sel;
    }
    SI_CK(si::launch_sparse_decode(P, B, (cudaStream_t)stream));
    if (have_plan) L->plan_fresh = false;
    return SI_OK;
}

}  // namespace

extern "C" {

// ------------------------------------------------------------------ SpAx

int spax_encode(const uint16_t* Wd, int d, int N, int bits, int group, spax_layer** out, void* stream) {
    SI_TRACE("spax_encode");
    if (!out) return fail(SI_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!Wd) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (bits != 2 && bits != 3 && bits != 4 && bits != 8)
        return fail(SI_ERR_UNSUPPORTED, "codes are 2, 3, 4 or 8 bits wide");
    if (group < 8 || (group & (group - 1)) || d < 64 || d % 64 || d % group)
        return fail(SI_ERR_INVALID_ARG, "need group a power of two >= 8, d % 64 == 0, d % group == 0");
    if (bits == 3 && d % 128)
        return fail(SI_ERR_INVALID_ARG, "3-bit codes need d % 128 == 0 (records of whole 16-byte units)");
    if (d > 32768) return fail(SI_ERR_UNSUPPORTED, "need d <= 32768");
    if (N < 1 || N > 32768) return fail(SI_ERR_INVALID_ARG, "need 1 <= N <= 32768");
    cudaStream_t st = (cudaStream_t)stream;
    if (capturing(st)) return fail(SI_ERR_INVALID_ARG, "spax_encode allocates; not allowed during capture");
    spax_layer* L = new spax_layer();
    SI_CK(cudaGetDevice(&L->device));
    L->d = d;
    L->N = N;
    L->bits = bits;
    L->group = group;
    L->ngp = round_up(d / group, 2);
    L->rec_bytes = d * bits / 8 + 8 * L->ngp;
    int rc;
    if ((rc = dalloc(&L->WdT, (size_t)N * d, "column-major Wd")) ||
        (rc = dalloc(&L->codes, (size_t)N * L->rec_bytes, "code records")) ||
        (rc = dalloc(&L->hist, si::kTierBins + 1, "tier histogram")) ||
        (rc = dalloc(&L->slab, (size_t)si::kTierBins * si::kSlabCap, "tier member lists")) ||
        (rc = dalloc(&L->a, N, "activations")) ||
        (rc = dalloc(&L->tickets, 16, "tickets"))) {
        destroy_spax(L);
        return rc;
    }
    L->part_floats = si::tiered_max_partial_floats(d);
    if (L->part_floats <= 0) {
        destroy_spax(L);
        return fail(SI_ERR_CUDA, "cannot query the device for the tiered grid");
    }
    if ((rc = dalloc(&L->part, (size_t)L->part_floats, "tiered partials"))) {
        destroy_spax(L);
        return rc;
    }
    L->params = reinterpret_cast<float*>(L->codes + d * bits / 8);
    cudaError_t e = cudaMemsetAsync(L->tickets, 0, 16 * sizeof(unsigned), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L->hist, 0, (si::kTierBins + 1) * sizeof(unsigned), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L->codes, 0, (size_t)N * L->rec_bytes, st);
    if (e == cudaSuccess)
        e = si::launch_spax_encode(Wd, d, N, bits, group, L->ngp, L->WdT, L->codes, L->rec_bytes, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        destroy_spax(L);
        return cuda_fail(e, "spax_encode");
    }
    *out = L;
    return SI_OK;
}

int spax_layer_info(const spax_layer* L, int* d, int* N, int* bits, int* group, int* ngp) {
    SI_TRACE("spax_layer_info");
    if (!L) return fail(SI_ERR_INVALID_ARG, "layer is NULL");
    if (d) *d = L->d;
    if (N) *N = L->N;
    if (bits) *bits = L->bits;
    if (group) *group = L->group;
    if (ngp) *ngp = L->ngp;
    return SI_OK;
}

int spax_layer_buffers(const spax_layer* L, const uint16_t** WdT, const uint8_t** codes, const float** params) {
    SI_TRACE("spax_layer_buffers");
    if (!L) return fail(SI_ERR_INVALID_ARG, "layer is NULL");
    if (WdT) *WdT = L->WdT;
    if (codes) *codes = L->codes;
    if (params) *params = L->params;
    return SI_OK;
}

int spax_layer_destroy(spax_layer* L) {
    SI_TRACE("spax_layer_destroy");
    if (!L) return SI_OK;
    cudaDeviceSynchronize();
    destroy_spax(L);
    return SI_OK;
}

}  // extern "C"

namespace {

int dense_act_core(const uint16_t* Wg, const uint16_t* Wu, int d, int N, const uint16_t* x, float* a, unsigned* hist,
                   int32_t* slab, cudaStream_t stream, const int32_t* rows = nullptr, int n_rows = 0) {
    if (!Wg || !Wu || !x || !a) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (d < 8 || d % 8 || N < 1) return fail(SI_ERR_INVALID_ARG, "need d % 8 == 0, N >= 1");
    if (d > 4096) return fail(SI_ERR_UNSUPPORTED, "dense activation pass supports d <= 4096");
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    si::DenseActParams P = {};
    P.Wg = Wg;
    P.Wu = Wu;
    P.d = d;
    P.N = N;
    P.x = x;
    P.a = a;
    P.hist = hist;
    P.slab = hist ? slab : nullptr;
    P.rows = rows;
    P.n_rows = n_rows;
    P.err = err;
    P.R = si::dense_act_stages(d);
    if (P.R < 8) return fail(SI_ERR_UNSUPPORTED, "d too large for the activation ring");
    SI_CK(si::launch_dense_act(P, stream));
    return SI_OK;
}

int tier_counts(const spax_layer* L, double top_frac, double mid_frac, long long* k_top, long long* k_mid) {
    if (!(top_frac >= 0.0 && mid_frac >= 0.0 && top_frac <= 1.0 && mid_frac <= 1.0))
        return fail(SI_ERR_INVALID_ARG, "tier fractions must be in [0, 1]");
    *k_top = count_of(top_frac, L->N);
    *k_mid = count_of(mid_frac, L->N);
    if (*k_top + *k_mid > L->N) return fail(SI_ERR_INVALID_ARG, "top + mid tiers exceed N");
    return SI_OK;
}

// The tiered down-projection with the tier choice inside the kernel; L->hist
// must hold the tier histogram of a (the kernel re-zeroes it).
int tiered_core(spax_layer* L, const float* a, long long k_top, long long k_mid, float* y, int32_t* top_out,
                int32_t* mid_out, cudaStream_t st) {
    if (L->d > 4096) return fail(SI_ERR_UNSUPPORTED, "the tiered down-projection supports d <= 4096");
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    si::TieredDownParams P = {};
    P.WdT = L->WdT;
    P.codes = L->codes;
    P.rec_bytes = L->rec_bytes;
    P.bits = L->bits;
    P.a = a;
    P.hist = L->hist;
    P.slab = L->slab;
    P.top_out = top_out;
    P.mid_out = mid_out;
    P.d = L->d;
    P.group = L->group;
    P.ngp = L->ngp;
    P.k_top = (int)k_top;
    P.k_mid = (int)k_mid;
    P.N = L->N;
    P.y = y;
    P.part = L->part;
    P.part_floats = L->part_floats;
    P.tickets = L->tickets;
    P.err = err;
    const int gmin = si::streaming_grid_upper_bound() / 4;  // grids are at least a quarter of the SMs
    P.aux_floats = round_up((int)(L->N / (gmin > 0 ? gmin : 1)) * 2 + 8, 32);
    P.ring_bytes = si::tiered_down_ring(L->d, P.aux_floats, L->rec_bytes);
    if (P.ring_bytes <= 0) return fail(SI_ERR_UNSUPPORTED, "d too large for the tier ring");
    SI_CK(si::launch_tiered_down(P, st));
    return SI_OK;
}

}  // namespace

extern "C" {

int spax_dense_act(const uint16_t* Wg, const uint16_t* Wu, int d, int N, const uint16_t* x, float* a, void* stream) {
    SI_TRACE("spax_dense_act");
    return dense_act_core(Wg, Wu, d, N, x, a, nullptr, nullptr, (cudaStream_t)stream);
}

int spax_tiered_down(spax_layer* L, const float* a, double top_frac, double mid_frac, float* y, int32_t* top_idx,
                     int32_t* mid_idx, void* stream) {
    SI_TRACE("spax_tiered_down");
    if (!L || !a || !y) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    long long k_top = 0, k_mid = 0;
    int rc = tier_counts(L, top_frac, mid_frac, &k_top, &k_mid);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    SI_CK(si::launch_abs_hist(a, L->N, L->hist, L->slab, st));
    return tiered_core(L, a, k_top, k_mid, y, top_idx, mid_idx, st);
}

int spax_select_decode(spax_layer* L, const uint16_t* Wg, const uint16_t* Wu, const int32_t* rows, int n_rows,
                       const uint16_t* x, double top_frac, double mid_frac, float* y, float* a_out, void* stream) {
    SI_TRACE("spax_select_decode");
    if (!L || !Wg || !Wu || !x || !y || (n_rows > 0 && !rows)) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (n_rows < 0 || n_rows > L->N) return fail(SI_ERR_INVALID_ARG, "need 0 <= n_rows <= N");
    if (!(top_frac >= 0.0 && mid_frac >= 0.0 && top_frac + mid_frac <= 1.0))
        return fail(SI_ERR_INVALID_ARG, "tier fractions must be >= 0 with top + mid <= 1");
    const long long k_top = count_of(top_frac, n_rows), k_mid = count_of(mid_frac, n_rows);
    if (k_top + k_mid > n_rows) return fail(SI_ERR_INVALID_ARG, "top + mid tiers exceed the selected rows");
    cudaStream_t st = (cudaStream_t)stream;
    float* a = a_out ? a_out : L->a;
    // unlisted neurons have a = 0; the dense pass over the listed rows fills
    // the rest and counts the zeros in the tier histogram
    SI_CK(cudaMemsetAsync(a, 0, (size_t)L->N * sizeof(float), st));
    if (n_rows == 0) {
        SI_CK(cudaMemsetAsync(y, 0, (size_t)L->d * sizeof(float), st));
        return SI_OK;
    }
    int rc = dense_act_core(Wg, Wu, L->d, L->N, x, a, L->hist, L->slab, st, rows, n_rows);
    if (rc) return rc;
    if ((rc = tiered_core(L, a, k_top, k_mid, y, nullptr, nullptr, st))) {
        cudaMemsetAsync(L->hist, 0, (si::kTierBins + 1) * sizeof(unsigned), st);  // leave it clean
        return rc;
    }
    return SI_OK;
}

int spax_ffn_decode(spax_layer* L, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* x, double top_frac,
                    double mid_frac, float* y, float* a_out, void* stream) {
    SI_TRACE("spax_ffn_decode");
    if (!L || !y) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    long long k_top = 0, k_mid = 0;
    int rc = tier_counts(L, top_frac, mid_frac, &k_top, &k_mid);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    float* a = a_out ? a_out : L->a;
    // the dense pass builds the tier histogram of a as it writes it
    if ((rc = dense_act_core(Wg, Wu, L->d, L->N, x, a, L->hist, L->slab, st))) return rc;
    if ((rc = tiered_core(L, a, k_top, k_mid, y, nullptr, nullptr, st))) {
        cudaMemsetAsync(L->hist, 0, (si::kTierBins + 1) * sizeof(unsigned), st);  // leave it clean
        return rc;
    }
    return SI_OK;
}

}  // extern "C"

namespace {

void destroy_stack(si_stack* K) {
    if (!K) return;
    dfree(K->pos);
    dfree(K->desc);
    dfree(K->delta);
    dfree(K->sync);
    if (K->desc_host) cudaFreeHost(K->desc_host);
    delete K;
}

}  // namespace

extern "C" {

// ------------------------------------------------------- a7: decode stack

int si_stack_create(si_layer* const* layers, int L, si_stack** out) {
    SI_TRACE("si_stack_create");
    if (!out) return fail(SI_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!layers) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (L < 1 || L > si::kStackMaxLayers) return fail(SI_ERR_INVALID_ARG, "need 1 <= L <= 64");
    for (int l = 0; l < L; ++l)
        if (!layers[l]) return fail(SI_ERR_INVALID_ARG, "NULL layer handle");
    const int d = layers[0]->d;
    for (int l = 1; l < L; ++l)
        if (layers[l]->d != d) return fail(SI_ERR_INVALID_ARG, "every layer of a stack must have the same d");
    if (si::sparse_decode_stack_stages(d) < 8)
        return fail(SI_ERR_UNSUPPORTED, "the decode stack supports d = 256, 512, 1024, 2048 or 3072");
    si_stack* K = new si_stack();
    SI_CK(cudaGetDevice(&K->device));
    K->L = L;
    K->d = d;
    for (int l = 0; l < L; ++l) {
        K->layers[l] = layers[l];
        K->pos_off[l + 1] = K->pos_off[l] + layers[l]->n_loaded;
    }
    int rc;
    if ((rc = dalloc(&K->pos, (size_t)K->pos_off[L], "stack plan copies")) ||
        (rc = dalloc(&K->desc, (size_t)L, "stack layer table")) ||
        (rc = dalloc(&K->delta, (size_t)L * si::kDeltaCopies * d, "stack layer sums")) ||
        (rc = dalloc(&K->sync, (size_t)si::stack_sync_words(L), "stack barrier counters"))) {
        destroy_stack(K);
        return rc;
    }
    if (cudaMallocHost(reinterpret_cast<void**>(&K->desc_host), sizeof(si::StackLayerDesc) * L) != cudaSuccess) {
        (void)cudaGetLastError();
        K->desc_host = nullptr;
        destroy_stack(K);
        return fail(SI_ERR_OOM, "cudaMallocHost failed for the stack layer table");
    }
    cudaError_t e = cudaMemset(K->delta, 0, sizeof(float) * (size_t)L * si::kDeltaCopies * d);
    if (e == cudaSuccess) e = cudaMemset(K->sync, 0, sizeof(unsigned) * (size_t)si::stack_sync_words(L));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        destroy_stack(K);
        return cuda_fail(e, "si_stack_create");
    }
    *out = K;
    return SI_OK;
}

int si_stack_plan(si_stack* K, const int32_t* const* S, const int* n_sel, void* stream) {
    SI_TRACE("si_stack_plan");
    if (!K || !S || !n_sel) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    bool same = K->planned;
    for (int l = 0; l < K->L; ++l) {
        if (n_sel[l] < 0 || n_sel[l] > K->layers[l]->n_loaded)
            return fail(SI_ERR_INVALID_ARG, "need 0 <= n_sel[l] <= n_loaded of layer l");
        if (n_sel[l] > 0 && !S[l]) return fail(SI_ERR_INVALID_ARG, "NULL computed set");
        same = same && K->desc_host[l].n == n_sel[l];
    }
    cudaStream_t st = (cudaStream_t)stream;
    if (!same) {
        // the layer table changes: it goes to the device by a stream-ordered copy
        // from the pinned staging table, which an earlier copy may still read
        if (capturing(st)) return fail(SI_ERR_INVALID_ARG, "the set sizes changed; plan once before capture");
        SI_CK(cudaStreamSynchronize(st));
        for (int l = 0; l < K->L; ++l) {
            si::StackLayerDesc D;
            D.packed = K->layers[l]->packed;
            D.pos = K->pos + K->pos_off[l];
            D.n = n_sel[l];
            D.n_records = K->layers[l]->n_pad;
            K->desc_host[l] = D;
        }
        SI_CK(cudaMemcpyAsync(K->desc, K->desc_host, sizeof(si::StackLayerDesc) * K->L, cudaMemcpyHostToDevice,
                              st));
    }
    // the sets themselves: stream-ordered device copies (capturable)
    for (int l = 0; l < K->L; ++l)
        if (n_sel[l] > 0)
            SI_CK(cudaMemcpyAsync(K->pos + K->pos_off[l], S[l], sizeof(int32_t) * (size_t)n_sel[l],
                                  cudaMemcpyDeviceToDevice, st));
    K->planned = true;
    return SI_OK;
}

int si_sparse_ffn_decode_stack(si_stack* K, float* h, uint16_t* x_out, void* stream) {
    SI_TRACE("si_sparse_ffn_decode_stack");
    if (!K || !h) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (!K->planned) return fail(SI_ERR_INVALID_ARG, "call si_stack_plan before decoding");
    if ((reinterpret_cast<uintptr_t>(h) & 15u) || (reinterpret_cast<uintptr_t>(x_out) & 15u))
        return fail(SI_ERR_INVALID_ARG, "h and x_out must be 16-byte aligned");
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    si::StackParams P = {};
    P.layers = K->desc;
    P.L = K->L;
    P.d = K->d;
    P.R = si::sparse_decode_stack_stages(K->d);
    P.h = h;
    P.x_out = x_out;
    P.delta = K->delta;
    P.sync = K->sync;
    P.err = err;
    SI_CK(si::launch_sparse_decode_stack(P, (cudaStream_t)stream));
    return SI_OK;
}

int si_stack_destroy(si_stack* K) {
    SI_TRACE("si_stack_destroy");
    if (!K) return SI_OK;
    cudaDeviceSynchronize();
    destroy_stack(K);
    return SI_OK;
}

}  // extern "C"

namespace {

// The gate/up tiers by |x| into a (and, when hist is given, the down
// projection's tier histogram of a).
int gate_up_core(const spax_layer* G, const spax_layer* U, const uint16_t* x, double top_frac, double mid_frac,
                 float* a, int32_t* top_idx, int32_t* mid_idx, unsigned* hist, int32_t* slab, cudaStream_t st) {
    if (!G || !U || !x || !a) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    // an encoded gate/up matrix: rows = neurons (handle d), columns = input channels (handle N)
    if (G->d != U->d || G->N != U->N || G->bits != U->bits || G->group != U->group)
        return fail(SI_ERR_INVALID_ARG, "gate and up encodings must have the same shape, bits and group");
    const int N = G->d, d = G->N;
    if (N % 4 || G->group % 4) return fail(SI_ERR_INVALID_ARG, "need N % 4 == 0");
    if (d > 8192) return fail(SI_ERR_UNSUPPORTED, "gate/up tiers support d <= 8192 input channels");
    if (!(top_frac >= 0.0 && mid_frac >= 0.0 && top_frac + mid_frac <= 1.0))
        return fail(SI_ERR_INVALID_ARG, "tier fractions must be >= 0 with top + mid <= 1");
    const long long k_top = count_of(top_frac, d), k_mid = count_of(mid_frac, d);
    if (k_top + k_mid > d) return fail(SI_ERR_INVALID_ARG, "top + mid tiers exceed the channels");
    unsigned* err = nullptr;
    int rc = err_word(&err);
    if (rc) return rc;
    si::GateUpTierParams P = {};
    P.WgT = G->WdT;
    P.WuT = U->WdT;
    P.gcodes = G->codes;
    P.ucodes = U->codes;
    P.rec_bytes = G->rec_bytes;
    P.bits = G->bits;
    P.group = G->group;
    P.d = d;
    P.N = N;
    P.x = x;
    P.k_top = (int)k_top;
    P.k_mid = (int)k_mid;
    P.a = a;
    P.hist = hist;
    P.slab = hist ? slab : nullptr;
    P.top_out = top_idx;
    P.mid_out = mid_idx;
    P.S = si::spax_gate_up_slice(N);
    P.err = err;
    if (P.S < 4) return fail(SI_ERR_CUDA, "cannot query the device");
    SI_CK(si::launch_spax_gate_up(P, st));
    return SI_OK;
}

}  // namespace

extern "C" {

int spax_gate_up(const spax_layer* gate, const spax_layer* up, const uint16_t* x, double top_frac, double mid_frac,
                 float* a, int32_t* top_idx, int32_t* mid_idx, void* stream) {
    SI_TRACE("spax_gate_up");
    return gate_up_core(gate, up, x, top_frac, mid_frac, a, top_idx, mid_idx, nullptr, nullptr, (cudaStream_t)stream);
}

int spax_all_decode(spax_layer* down, const spax_layer* gate, const spax_layer* up, const uint16_t* x,
                    double in_top_frac, double in_mid_frac, double top_frac, double mid_frac, float* y,
                    float* a_out, void* stream) {
    SI_TRACE("spax_all_decode");
    if (!down || !gate || !up || !y) return fail(SI_ERR_INVALID_ARG, "NULL pointer");
    if (down->N != gate->d || down->d != gate->N)
        return fail(SI_ERR_INVALID_ARG, "the down encoding's columns must be the gate/up encodings' rows");
    long long k_top = 0, k_mid = 0;
    int rc = tier_counts(down, top_frac, mid_frac, &k_top, &k_mid);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    float* a = a_out ? a_out : down->a;
    // the gate/up pass builds the down tiers' histogram of a as it writes it
    if ((rc = gate_up_core(gate, up, x, in_top_frac, in_mid_frac, a, nullptr, nullptr, down->hist, down->slab, st)))
        return rc;
    if ((rc = tiered_core(down, a, k_top, k_mid, y, nullptr, nullptr, st))) {
        cudaMemsetAsync(down->hist, 0, (si::kTierBins + 1) * sizeof(unsigned), st);  // leave it clean
        return rc;
    }
    return SI_OK;
}

}  // extern "C"
