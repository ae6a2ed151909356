// select.cu -- exact top-k selection kernels.
//
// Every ranking of the method is "the k largest by a key, ties to the lower
// index": per-token top-alpha of |a| and top-beta of counts (SelectInfer
// section 5, Fig. 7) and base/secondary neurons by profiler score (section 4,
// Fig. 6). All of them use one block-wide primitive (the SpAx tiers are
// selected inside the tiered down-projection kernel, decode.cu):
//   block_topk_cut   4 passes of an 8-bit radix histogram over 32-bit
//                    order-preserving keys find the k-th largest key `thr`
//                    and how many elements equal to it are still needed;
//   block_topk_emit  walks the elements in index order with warp ballots,
//                    takes every key > thr and the first `take_eq` keys == thr,
//                    and reports each selected element with its rank.
// Only integer compares decide, so results are bit-exact and independent of
// thread scheduling.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace si {

struct TopkCut {
    uint32_t thr;
    int take_eq;
};

// Scratch: hist[257], state[2] in shared memory.
template <int NT, class KeyF, class EligF>
__device__ TopkCut block_topk_cut(int n, int k, KeyF key, EligF elig, uint32_t* hist, uint32_t* state) {
    TopkCut cut;
    if (k <= 0) {
        cut.thr = 0xFFFFFFFFu;
        cut.take_eq = 0;
        return cut;
    }
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0, pmask = 0;
    int kk = k;
    const int rounds = (n + NT - 1) / NT;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 257; i += NT) hist[i] = 0;
        __syncthreads();
        for (int r = 0; r < rounds; ++r) {
            const int i = r * NT + threadIdx.x;
            uint32_t bin = 256;
            if (i < n && elig(i)) {
                const uint32_t kv = key(i);
                if ((kv & pmask) == prefix) bin = (kv >> shift) & 255u;
            }
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bin);
            if (bin != 256u && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l owns bins 255-8l .. 248-8l, visited from the top down
            uint32_t c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[255 - 8 * lane - j];
                sum += c[j];
            }
            uint32_t inc = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += v;
            }
            const uint32_t exc = inc - sum;
            const bool hit = exc < (uint32_t)kk && (uint32_t)kk <= inc;
            if (hit) {
                uint32_t run = exc;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (run + c[j] >= (uint32_t)kk) {
                        state[0] = (uint32_t)(255 - 8 * lane - j);
                        state[1] = (uint32_t)kk - run;
                        break;
                    }
                    run += c[j];
                }
            }
            if (__ballot_sync(0xFFFFFFFFu, hit) == 0u && lane == 0) state[0] = 0xFFFFFFFFu;
        }
        __syncthreads();
        const uint32_t digit = state[0];
        const int nkk = (int)state[1];
        __syncthreads();
        if (digit == 0xFFFFFFFFu) {  // fewer eligible elements than k: take them all
            cut.thr = 0u;
            cut.take_eq = INT_MAX;
            return cut;
        }
        prefix |= digit << shift;
        pmask |= 0xFFu << shift;
        kk = nkk;
    }
    cut.thr = prefix;
    cut.take_eq = kk;
    return cut;
}

// Scratch: scnt[2 * NT / 32]. Calls out(i, rank) for each selected element
// (rank = position among selected ones in index order) and, when WORDS,
// word(i / 32, ballot) once per 32 elements. Returns the number selected.
template <int NT, bool WORDS, class KeyF, class EligF, class OutF, class WordF>
__device__ int block_topk_emit(int n, TopkCut cut, KeyF key, EligF elig, OutF out, WordF word,
                               uint32_t* scnt) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int eq_base = 0, sel_base = 0;
    const int rounds = (n + NT - 1) / NT;
    for (int r = 0; r < rounds; ++r) {
        const int i = r * NT + threadIdx.x;
        bool gt = false, eq = false;
        if (i < n && elig(i)) {
            const uint32_t kv = key(i);
            gt = kv > cut.thr;
            eq = kv == cut.thr;
        }
        const uint32_t meq = __ballot_sync(0xFFFFFFFFu, eq);
        if (lane == 0) scnt[warp] = (uint32_t)__popc(meq);
        __syncthreads();
        int eq_off = 0, eq_tot = 0;
        for (int w = 0; w < NW; ++w) {
            const int c = (int)scnt[w];
            eq_off += (w < warp) ? c : 0;
            eq_tot += c;
        }
        const int eq_rank = eq_base + eq_off + __popc(meq & lanemask_lt());
        const bool s = gt || (eq && eq_rank < cut.take_eq);
        const uint32_t ms = __ballot_sync(0xFFFFFFFFu, s);
        if (lane == 0) {
            scnt[NW + warp] = (uint32_t)__popc(ms);
            if (WORDS && r * NT + warp * 32 < n) word((r * NT + warp * 32) >> 5, ms);
        }
        __syncthreads();
        int s_off = 0, s_tot = 0;
        for (int w = 0; w < NW; ++w) {
            const int c = (int)scnt[NW + w];
            s_off += (w < warp) ? c : 0;
            s_tot += c;
        }
        if (s) out(i, sel_base + s_off + __popc(ms & lanemask_lt()));
        eq_base += eq_tot;
        sel_base += s_tot;
        __syncthreads();
    }
    return sel_base;
}

struct NoWord {
    __device__ void operator()(int, uint32_t) const {}
};

// Ordered compaction: out(i, rank) for every i with pred(i), in index order.
template <int NT, class PredF, class OutF>
__device__ int block_compact(int n, PredF pred, OutF out, uint32_t* scnt) {
    TopkCut all;
    all.thr = 0u;
    all.take_eq = 0;
    auto key = [&](int i) -> uint32_t { return pred(i) ? 1u : 0u; };
    auto elig = [](int) { return true; };
    return block_topk_emit<NT, false>(n, all, key, elig, out, NoWord(), scnt);
}

// ------------------------------------------------------------------- kernels

// Exclusive scan of one value per thread over an NT-thread CTA (NT a
// multiple of 32, at most 1024); *total gets the sum. s_w: 33 words of shared
// scratch. Every thread of the CTA calls it.
template <int NT>
__device__ __forceinline__ uint32_t cta_excl_scan(uint32_t v, uint32_t* s_w, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = lane < NT / 32 ? s_w[lane] : 0u;
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += t;
        }
        s_w[lane] = wi - w;  // exclusive prefix of the warp totals
        if (lane == 31) s_w[32] = wi;
    }
    __syncthreads();
    const uint32_t r = s_w[warp] + incl - v;
    *total = s_w[32];
    __syncthreads();  // s_w may be reused
    return r;
}

constexpr int kSelNT = 512;

// a4 + a5: one CTA per token row. Per-token top-alpha over the loaded
// positions by |A| (SelectInfer section 5); every selected position adds 1 to
// its sequence's count. Optional bit mask of the selection per row.
// The threshold comes from three radix passes over the 31-bit |A| key
// (digits of 11, 11 and 9 bits, shared-memory histograms); the emit walks
// word-aligned runs of 32 positions per warp, so a selection ballot is the
// row's mask word. Ranks among equal keys are counted only when the
// threshold splits a run of them.
constexpr int kAlphaBins = 2048;

__global__ void __launch_bounds__(kSelNT) k_topk_alpha(const float* __restrict__ absA, int ld, int n, int T,
                                                      int alpha, uint32_t* __restrict__ counts,
                                                      uint32_t* __restrict__ topmask, int words) {
    extern __shared__ __align__(16) uint32_t s_keys[];
    __shared__ uint32_t hist[kAlphaBins];
    __shared__ uint32_t s_w[33];
    __shared__ uint32_t s_state[3];  // bin, rank left inside it, its count
    const int row = blockIdx.x, b = row / T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* src = absA + (size_t)row * ld;
    grid_launch_dependents();
    grid_dependency_wait();  // |A| and the zeroed counts come from earlier work in the stream
    for (int i = tid; i < n; i += kSelNT) s_keys[i] = abs_key(__ldg(src + i));
    const bool act = alpha > 0 && alpha < n;
    uint32_t prefix = 0u, pmask = 0u, kk = (uint32_t)alpha, eqn = 0u;
    if (act) {
        constexpr int kShift[3] = {20, 9, 0}, kBits[3] = {11, 11, 9};
#pragma unroll
        for (int p = 0; p < 3; ++p) {
            const int shift = kShift[p], nb = 1 << kBits[p], per = nb / kSelNT;
            for (int i = tid; i < kAlphaBins; i += kSelNT) hist[i] = 0u;
            __syncthreads();
            for (int i = tid; i < n; i += kSelNT) {
                const uint32_t k = s_keys[i];
                if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & (uint32_t)(nb - 1)], 1u);
            }
            __syncthreads();
            // thread t owns bins nb-1-per*t ... nb-per*(t+1), highest first
            uint32_t c = 0u;
            for (int j = 0; j < per; ++j) c += hist[nb - 1 - per * tid - j];
            uint32_t tot;
            const uint32_t e = cta_excl_scan<kSelNT>(c, s_w, &tot);  // keys in higher bins
            if (e < kk && kk <= e + c) {
                uint32_t run = e;
                for (int j = 0; j < per; ++j) {
                    const int bin = nb - 1 - per * tid - j;
                    if (run + hist[bin] >= kk) {
                        s_state[0] = (uint32_t)bin;
                        s_state[1] = kk - run;
                        s_state[2] = hist[bin];
                        break;
                    }
                    run += hist[bin];
                }
            }
            __syncthreads();
            prefix |= s_state[0] << shift;
            pmask |= (uint32_t)(nb - 1) << shift;
            kk = s_state[1];
            eqn = s_state[2];
        }
    } else {
        __syncthreads();  // the keys are in place
    }
    // every key > thr and the first `take` keys == thr, in index order
    const uint32_t thr = act ? prefix : (alpha <= 0 ? 0xFFFFFFFFu : 0u);
    const uint32_t take = act ? kk : (alpha <= 0 ? 0u : 0xFFFFFFFFu);
    const bool split = act && kk < eqn;
    // warp w owns positions [w * SEG, (w + 1) * SEG), SEG a multiple of 32
    const int SEG = ((n + kSelNT - 1) / kSelNT) * 32;
    const int lo = warp * SEG, hi = min(n, lo + SEG);
    const uint32_t lt = lanemask_lt();
    uint32_t r = 0u;  // keys equal to thr before the current position
    if (split) {
        uint32_t q = 0u;
        for (int i0 = lo; i0 < hi; i0 += 32) {
            const int i = i0 + lane;
            q += __popc(__ballot_sync(0xFFFFFFFFu, i < hi && s_keys[i] == thr));
        }
        uint32_t tot;
        const uint32_t ex = cta_excl_scan<kSelNT>(lane == 0 ? q : 0u, s_w, &tot);
        r = __shfl_sync(0xFFFFFFFFu, ex, 0);
    }
    uint32_t* cnt = counts + (size_t)b * n;
    uint32_t* tm = topmask ? topmask + (size_t)row * words : nullptr;
    for (int i0 = lo; i0 < hi; i0 += 32) {
        const int i = i0 + lane;
        const bool in = i < hi;
        const uint32_t k = in ? s_keys[i] : 0u;
        const uint32_t me = __ballot_sync(0xFFFFFFFFu, in && k == thr);
        const bool sel = in && (k > thr || (k == thr && r + __popc(me & lt) < take));
        r += __popc(me);
        const uint32_t ms = __ballot_sync(0xFFFFFFFFu, sel);
        if (sel) atomicAdd(cnt + i, 1u);
        if (tm && lane == 0) tm[i0 >> 5] = ms;
    }
}

// a6: one CTA per sequence. Top-beta of the counts among non-static positions
// (ties to the lower position), united with the static positions, written as
// an ascending list of n_sel positions.
// Counts are small integers (at most the prompt length), so one 2048-bin
// histogram of min(count, 2047) finds the threshold count and how many
// neurons equal to it are taken (in index order). One blocked pass with two
// CTA scans (ranks among equal counts, then output slots) writes S. Only a
// threshold in the saturated top bin (counts >= 2047) falls back to the
// general radix selection.
constexpr int kBetaBins = 2048;
// threads of the one CTA per sequence: the per-thread runs and scans are
// latency-bound, so more threads win (top-alpha + top-beta per Llama3.2-1B
// layer: 24.3 us with 256, 22.3 with 512, 20.4 with 1024)
constexpr int kBetaNT = 1024;
static_assert(kBetaBins % kBetaNT == 0, "whole bins per thread");

__global__ void __launch_bounds__(kBetaNT) k_topk_beta(const uint32_t* __restrict__ counts,
                                                      const uint8_t* __restrict__ is_static, int n, int beta,
                                                      int n_sel, int32_t* __restrict__ S, unsigned* err) {
    extern __shared__ __align__(16) uint32_t s_keys[];  // n keys, then n flag bytes
    uint8_t* s_take = reinterpret_cast<uint8_t*>(s_keys + n);
    __shared__ uint32_t hist[kBetaBins];
    __shared__ uint32_t s_w[33];
    __shared__ uint32_t s_cut[2];  // threshold count, equal counts taken
    constexpr int NT = kBetaNT, PER = kBetaBins / kBetaNT;
    const int b = blockIdx.x, tid = threadIdx.x;
    grid_launch_dependents();
    grid_dependency_wait();  // the counts are the previous grid's output
    for (int i = tid; i < n; i += NT) {
        s_keys[i] = counts[(size_t)b * n + i];
        s_take[i] = is_static[i] ? 1 : 0;
    }
    for (int i = tid; i < kBetaBins; i += NT) hist[i] = 0u;
    if (tid == 0) {
        s_cut[0] = 0xFFFFFFFFu;  // beta == 0: no count is above or at it
        s_cut[1] = 0u;
    }
    __syncthreads();
    for (int i = tid; i < n; i += NT)
        if (!s_take[i]) atomicAdd(&hist[min(s_keys[i], (uint32_t)(kBetaBins - 1))], 1u);
    __syncthreads();
    // thread t owns bins 2047 - PER t ... 2048 - PER (t + 1) (counting from the top)
    uint32_t hsum = 0u;
#pragma unroll
    for (int j = 0; j < PER; ++j) hsum += hist[kBetaBins - 1 - PER * tid - j];
    uint32_t eligible;
    const uint32_t above = cta_excl_scan<NT>(hsum, s_w, &eligible);
    if (beta > 0 && above < (uint32_t)beta && (uint32_t)beta <= above + hsum) {
        uint32_t run = above;
        for (int j = 0; j < PER; ++j) {
            const int bin = kBetaBins - 1 - PER * tid - j;
            const uint32_t h = hist[bin];
            if ((uint32_t)beta <= run + h) {
                s_cut[0] = (uint32_t)bin;
                s_cut[1] = (uint32_t)beta - run;
                break;
            }
            run += h;
        }
    }
    __syncthreads();
    const uint32_t thr = s_cut[0], take = s_cut[1];
    int32_t* dst = S + (size_t)b * n_sel;
    if (beta > 0 && (eligible < (uint32_t)beta || thr == (uint32_t)(kBetaBins - 1))) {
        // fewer eligible neurons than beta, or a threshold among saturated
        // counts: the general radix selection decides
        __syncthreads();
        __shared__ uint32_t rhist[257], rstate[2], scnt[2 * NT / 32];
        auto key = [&](int i) -> uint32_t { return s_keys[i]; };
        auto elig = [&](int i) { return is_static[i] == 0; };
        const TopkCut cut = block_topk_cut<NT>(n, beta, key, elig, rhist, rstate);
        auto mark = [&](int i, int) { s_take[i] = 1; };
        block_topk_emit<NT, false>(n, cut, key, elig, mark, NoWord(), scnt);
        __syncthreads();
        auto pred = [&](int i) { return s_take[i] != 0; };
        auto put = [&](int i, int r) {
            if (r < n_sel) dst[r] = i;
        };
        const int total = block_compact<NT>(n, pred, put, scnt);
        if (tid == 0 && total != n_sel) atomicOr(err, SI_DEVERR_COUNT);
        return;
    }
    // each thread takes a contiguous run of positions, in index order
    const int CH = (n + NT - 1) / NT;
    const int lo = tid * CH, hi = min(n, lo + CH);
    uint32_t q = 0u;
    for (int i = lo; i < hi; ++i) q += (!s_take[i] && s_keys[i] == thr) ? 1u : 0u;
    uint32_t unused;
    const uint32_t r0 = cta_excl_scan<NT>(q, s_w, &unused);  // equal counts before this run
    uint32_t r = r0, c = 0u;
    for (int i = lo; i < hi; ++i) {
        const uint32_t k = s_keys[i];
        bool sel = s_take[i] != 0;
        if (!sel) {
            sel = k > thr || (k == thr && r < take);
            r += (k == thr) ? 1u : 0u;
        }
        c += sel ? 1u : 0u;
    }
    uint32_t total;
    uint32_t pos = cta_excl_scan<NT>(c, s_w, &total);
    r = r0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t k = s_keys[i];
        bool sel = s_take[i] != 0;
        if (!sel) {
            sel = k > thr || (k == thr && r < take);
            r += (k == thr) ? 1u : 0u;
        }
        if (sel) {
            if (pos < (uint32_t)n_sel) dst[pos] = i;
            ++pos;
        }
    }
    if (tid == 0 && total != (uint32_t)n_sel) atomicOr(err, SI_DEVERR_COUNT);
}

// a2: selective loading ranking (SelectInfer section 4, Fig. 6), one CTA.
// base = top n_base by task score; secondary = top (n_load - n_base) by model
// score among the rest; loaded positions ascending by neuron index.
__global__ void __launch_bounds__(1024) k_rank_loaded(const float* __restrict__ task,
                                                     const float* __restrict__ model, int N, int n_base,
                                                     int n_load, int32_t* __restrict__ loaded,
                                                     uint8_t* __restrict__ is_static, unsigned* err) {
    extern __shared__ __align__(16) uint8_t s_flags[];  // N base flags, N take flags
    uint8_t* s_base = s_flags;
    uint8_t* s_take = s_flags + N;
    __shared__ uint32_t hist[257], state[2], scnt[2 * 1024 / 32];
    for (int i = threadIdx.x; i < N; i += 1024) {
        s_base[i] = 0;
        s_take[i] = 0;
    }
    __syncthreads();
    auto key1 = [&](int i) -> uint32_t { return value_key(task[i]); };
    auto all = [](int) { return true; };
    const TopkCut c1 = block_topk_cut<1024>(N, n_base, key1, all, hist, state);
    auto mark1 = [&](int i, int) {
        s_base[i] = 1;
        s_take[i] = 1;
    };
    block_topk_emit<1024, false>(N, c1, key1, all, mark1, NoWord(), scnt);
    __syncthreads();
    auto key2 = [&](int i) -> uint32_t { return value_key(model[i]); };
    auto notbase = [&](int i) { return s_base[i] == 0; };
    const TopkCut c2 = block_topk_cut<1024>(N, n_load - n_base, key2, notbase, hist, state);
    auto mark2 = [&](int i, int) { s_take[i] = 1; };
    block_topk_emit<1024, false>(N, c2, key2, notbase, mark2, NoWord(), scnt);
    __syncthreads();
    auto pred = [&](int i) { return s_take[i] != 0; };
    auto put = [&](int i, int r) {
        if (r < n_load) {
            loaded[r] = i;
            is_static[r] = s_base[i];
        }
    };
    const int total = block_compact<1024>(N, pred, put, scnt);
    if (threadIdx.x == 0 && total != n_load) atomicOr(err, SI_DEVERR_COUNT);
}

// Decode plan for B sequences: union of the B position lists with a per-entry
// mask of the sequences that selected it (one CTA).
__global__ void __launch_bounds__(1024) k_decode_plan(const int32_t* __restrict__ S, int n_sel, int B, int n,
                                                     int32_t* __restrict__ pos, uint32_t* __restrict__ pmask,
                                                     int* __restrict__ count, unsigned* err) {
    extern __shared__ __align__(16) uint32_t s_mask[];
    __shared__ uint32_t scnt[2 * 1024 / 32];
    for (int i = threadIdx.x; i < n; i += 1024) s_mask[i] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < B * n_sel; j += 1024) {
        const int p = S[j];
        if (p >= 0 && p < n)
            atomicOr(&s_mask[p], 1u << (j / n_sel));
        else
            atomicOr(err, SI_DEVERR_COUNT);
    }
    __syncthreads();
    auto pred = [&](int i) { return s_mask[i] != 0u; };
    auto put = [&](int i, int r) {
        pos[r] = i;
        pmask[r] = s_mask[i];
    };
    const int total = block_compact<1024>(n, pred, put, scnt);
    if (threadIdx.x == 0) *count = total;
}

// Score-file merge (SelectInfer section 3): out[n] = sum_f s_f[n] / T_f in
// float32, files in order, each step rounded (no contraction).
struct MergeArgs {
    const float* s[16];
    float tok[16];
    int nfiles;
};

__global__ void k_merge_scores(MergeArgs args, int N, float* __restrict__ out) {
    for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += gridDim.x * blockDim.x) {
        float acc = 0.0f;
        for (int f = 0; f < args.nfiles; ++f) acc = __fadd_rn(acc, __fdiv_rn(args.s[f][n], args.tok[f]));
        out[n] = acc;
    }
}

// Cluster-granular selection (PowerInfer-2 neuron clusters: contiguous blocks
// of csize neuron indices; when one neuron of a cluster is predicted active
// the whole cluster is brought in), applied to a computed set S. One CTA:
// the clusters of the selected positions' neurons are marked in a shared
// bitmap, then every packed position whose neuron's cluster is marked is
// written in ascending order (ballot compaction), with the count.
__global__ void __launch_bounds__(1024) k_expand_clusters(const int32_t* __restrict__ loaded, int n_loaded,
                                                         const int32_t* __restrict__ S, int n_sel, int N, int csize,
                                                         int32_t* __restrict__ out, int* __restrict__ count,
                                                         unsigned* err) {
    extern __shared__ uint32_t s_hit[];  // one bit per cluster
    __shared__ uint32_t scnt[2 * 1024 / 32];
    const int nc = (N + csize - 1) / csize, nw = (nc + 31) / 32;
    for (int i = threadIdx.x; i < nw; i += 1024) s_hit[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n_sel; i += 1024) {
        const int p = S[i];
        if (p < 0 || p >= n_loaded) {
            atomicOr(err, SI_DEVERR_COUNT);
            continue;
        }
        const int c = loaded[p] / csize;
        atomicOr(&s_hit[c >> 5], 1u << (c & 31));
    }
    __syncthreads();
    auto pred = [&](int p) -> bool {
        const int c = loaded[p] / csize;
        return (s_hit[c >> 5] >> (c & 31)) & 1u;
    };
    auto put = [&](int p, int r) { out[r] = p; };
    const int total = block_compact<1024>(n_loaded, pred, put, scnt);
    if (threadIdx.x == 0) *count = total;
}

// ------------------------------------------------------------------ launchers

namespace {
// Launch with programmatic dependent launch: the kernel's launch and
// set-up overlap the previous grid in the stream; it waits for that grid
// before reading anything.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
}  // namespace

cudaError_t launch_topk_alpha(const float* absA, int ld, int n, int T, int B, int alpha, uint32_t* counts,
                              uint32_t* topmask, cudaStream_t st) {
    const size_t smem = (size_t)n * 4;
    cudaError_t e = allow_max_smem(k_topk_alpha);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_topk_alpha, (unsigned)(B * T), kSelNT, smem, st, absA, ld, n, T, alpha, counts, topmask,
                      (n + 31) / 32);
}

cudaError_t launch_topk_beta(const uint32_t* counts, const uint8_t* is_static, int n, int B, int beta, int n_sel,
                             int32_t* S, unsigned* err, cudaStream_t st) {
    const size_t smem = (size_t)n * 5 + 16;
    cudaError_t e = allow_max_smem(k_topk_beta);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_topk_beta, (unsigned)B, kBetaNT, smem, st, counts, is_static, n, beta, n_sel, S, err);
}

cudaError_t launch_rank_loaded(const float* task, const float* model, int N, int n_base, int n_load,
                               int32_t* loaded, uint8_t* is_static, unsigned* err, cudaStream_t st) {
    const size_t smem = (size_t)N * 2 + 16;
    cudaError_t e = allow_max_smem(k_rank_loaded);
    if (e != cudaSuccess) return e;
    k_rank_loaded<<<1, 1024, smem, st>>>(task, model, N, n_base, n_load, loaded, is_static, err);
    return cudaGetLastError();
}

cudaError_t launch_decode_plan(const int32_t* S, int n_sel, int B, int n, int32_t* pos, uint32_t* pmask,
                               int* count, unsigned* err, cudaStream_t st) {
    const size_t smem = (size_t)n * 4;
    cudaError_t e = allow_max_smem(k_decode_plan);
    if (e != cudaSuccess) return e;
    k_decode_plan<<<1, 1024, smem, st>>>(S, n_sel, B, n, pos, pmask, count, err);
    return cudaGetLastError();
}

cudaError_t launch_merge_scores(const float* const* s, const float* tok, int nfiles, int N, float* out,
                                cudaStream_t st) {
    MergeArgs a;
    for (int f = 0; f < 16; ++f) {
        a.s[f] = f < nfiles ? s[f] : nullptr;
        a.tok[f] = f < nfiles ? tok[f] : 1.0f;
    }
    a.nfiles = nfiles;
    const int blocks = (N + 255) / 256 < 1024 ? (N + 255) / 256 : 1024;
    k_merge_scores<<<blocks, 256, 0, st>>>(a, N, out);
    return cudaGetLastError();
}

cudaError_t launch_expand_clusters(const int32_t* loaded, int n_loaded, const int32_t* S, int n_sel, int N,
                                  int csize, int32_t* out, int* count, unsigned* err, cudaStream_t st) {
    const int nc = (N + csize - 1) / csize;
    const size_t smem = (size_t)((nc + 31) / 32) * 4;
    k_expand_clusters<<<1, 1024, smem, st>>>(loaded, n_loaded, S, n_sel, N, csize, out, count, err);
    return cudaGetLastError();
}

}  // namespace si
