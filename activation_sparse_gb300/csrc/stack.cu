// stack.cu -- one launch per decode token over a stack of sparse FFN layers.
//
// SelectInfer (section 5) computes, at every decode step, each layer's FFN on
// that layer's selected neurons only; the layers run one after another, the
// output of one feeding the input of the next. In the pages' models (Llama,
// Qwen) a layer's FFN reads the RMS-normalised residual stream and adds its
// output back to it; for a stack of FFN layers (unit norm gain) that is
//
//     for l = 0 .. L-1:   x_l = bf16(h / sqrt(mean(h^2) + eps));   h += sum over p in S_l of a_p(x_l) * down_p
//
// with h kept in fp32 and eps = 1e-5. k_sparse_decode_stack runs the whole token as one
// cooperative grid, one CTA per SM, so that the weight stream never stops at
// a layer boundary:
//   * the producer warp streams the records of layer 0, then layer 1, ... into
//     one ring, numbering them consecutively; it never waits for a layer's
//     result, because which records a layer reads does not depend on x;
//   * the eight consumer warps compute layer l's records (as the batch-1
//     decode does: a = silu(g.x) * (u.x) per record, a * down into a per-warp
//     register partial of y), reduce the eight partials through shared memory
//     in a fixed order, add the CTA's sum into one of kDeltaCopies copies of
//     delta_l (copy b % kDeltaCopies) with float4 reductions and arrive on
//     layer l's grid barrier. Atomics on one address are serialised where the
//     address lives, so spreading the 152 CTAs' sums over four copies, and
//     the barrier's arrivals over kBarLines counters in separate cache lines,
//     keeps those queues short;
//   * once every CTA has arrived, each CTA adds the copies of delta_l, in copy
//     order, to its own copy of h and forms x_{l+1} from it in shared memory (every CTA performs the same
//     fp32 operations in the same order, so the copies agree), then goes on
//     with layer l+1, whose first records are already in the ring.
// So DRAM idles only when a layer boundary takes longer than the ring's
// look-ahead (R stages of 6d bytes per SM). The counters, the delta buffers
// and the launch's error word are zero on entry and zeroed again before the
// grid ends (each CTA zeroes a slice of delta_{l-1} once it has passed barrier
// l; the last CTA to leave zeroes delta_{L-1} and the counters).
#include "common.cuh"
#include "internal.h"
#include "ring.cuh"

namespace si {

namespace {

constexpr float kNormEps = 1e-5f;  // RMS norm epsilon of the layer input
constexpr int kStackMaxStages = 32;
constexpr unsigned kSiteStack = 5u << 8;
constexpr unsigned kSiteGrid = 5u << 16;

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier of layer l, run by one whole warp: lane 0 arrives on counter
// b % kBarLines (each counter in its own 128-byte line) with a release
// pattern, then lanes 0 .. kBarLines-1 each wait (bounded, acquire loads)
// until their counter holds all of its CTAs. The caller orders the CTA's
// writes before the arrival and its later reads after the wait with CTA
// barriers.
__device__ bool grid_arrive_wait(unsigned* ctrs, int G, unsigned* err) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        // release: the CTA's sums (ordered before this thread by the CTA
        // barrier) become visible before the arrival
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(ctrs + (blockIdx.x % kBarLines) * kLineWords)
                     : "memory");
    }
    __syncwarp();
    const unsigned want = lane < kBarLines ? (unsigned)((G - lane + kBarLines - 1) / kBarLines) : 0u;
    const unsigned* mine = ctrs + (lane < kBarLines ? lane : 0) * kLineWords;
    bool ok = true;
    const long long t0 = cycles();
    for (uint32_t it = 1;; ++it) {
        const bool here = lane >= kBarLines || ld_acquire_gpu(mine) >= want;
        if (__all_sync(0xFFFFFFFFu, here)) break;
        if ((it & 255u) == 0) {
            bool stop = (*reinterpret_cast<volatile unsigned*>(err) & SI_DEVERR_WAIT_TIMEOUT) != 0;
            if (!stop && cycles() - t0 > kWaitLimitCycles) {
                if (lane == 0) atomicOr(err, SI_DEVERR_WAIT_TIMEOUT | kSiteStack | kSiteGrid);
                stop = true;
            }
            if (__any_sync(0xFFFFFFFFu, stop)) {
                ok = false;
                break;
            }
        }
    }
    return ok;  // the acquire loads order the CTA's later reads (after a CTA barrier)
}

// y += v on four consecutive floats in global memory, without a return value
__device__ __forceinline__ void red_add4(float* p, const float4 v) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// bf16 of four fp32 values (round to nearest even), packed in element order
__device__ __forceinline__ uint2 bf16x4(const float4 v) {
    const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(v.x));
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v.y));
    const uint32_t c = __bfloat16_as_ushort(__float2bfloat16_rn(v.z));
    const uint32_t e = __bfloat16_as_ushort(__float2bfloat16_rn(v.w));
    return make_uint2(a | (b << 16), c | (e << 16));
}

// Shared memory besides the ring: the stages' record numbers (R ints) and x
// (bf16 [d]).
__host__ __device__ inline RingLayout stack_layout(int R, int d) {
    return ring_layout(R, 6 * d, 4 * kStackMaxStages, 2 * d);
}

}  // namespace

bool sparse_decode_stack_width_ok(int d);

// XJ = d / 256: 16-byte chunks of a row per lane (chunk c = lane + 32 j).
//
// Ring discipline. Records are numbered consecutively over the layers; record
// i goes to stage i % R and to consumer warp i % 8. R need not be a multiple
// of 8, so a stage's consecutive fills belong to different warps, and a parity
// wait alone could be answered by a fill two phases old. The producer
// therefore writes the record number into the stage's slot before issuing the
// copy (it can only do so once the stage's previous fill was consumed and
// released), and a consumer first waits for its record number to appear, then
// for the stage's full barrier.
//
// Layer end. A warp keeps the stage of its last record of the layer instead of
// releasing it, and writes its register partial of y there (4d bytes fit the
// 6d-byte stage); after one CTA barrier every thread sums its columns over the
// eight warps' stages in warp order and adds the sum into the CTA's copy of
// delta_l; after a second barrier the warps release those stages.
template <int XJ>
__global__ void __launch_bounds__(kDecThreads, 1) k_sparse_decode_stack(StackParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ StackLayerDesc s_desc[kStackMaxLayers];
    __shared__ unsigned s_flag;
    __shared__ float s_ss[kConsWarps];
    const int d = P.d, L = P.L;
    const int G = (int)gridDim.x;
    const RingLayout RL = stack_layout(P.R, d);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RL.off_full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + RL.off_empty);
    int* seq = reinterpret_cast<int*>(smem + RL.off_aux);  // record number of each stage's latest fill
    uint4* s_x = reinterpret_cast<uint4*>(smem + RL.off_x);
    uint8_t* ring = smem + RL.off_ring;
    const int R = RL.R;
    unsigned* lerr = P.sync + stack_lerr_word(L);  // this launch's failures; bounded waits watch it
    // the host never launches an invalid ring or stack; refuse one rather than misbehave
    if (R < kConsWarps || R > kStackMaxStages || L < 1 || L > kStackMaxLayers || d != 256 * XJ ||
        RL.stage < 4 * d) {
        if (threadIdx.x == 0) atomicOr(P.err, SI_DEVERR_COUNT);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = d / 8;
    constexpr int KV = (XJ + 3) / 4;  // float4 columns of h per consumer thread (d / 4 over 256 threads)

    for (int l = threadIdx.x; l < L; l += blockDim.x) s_desc[l] = P.layers[l];
    for (int s = threadIdx.x; s < R; s += blockDim.x) seq[s] = -1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // CTA b's share of layer l: an even slice of the layer's list, with the
    // slice index rotated by l so that no CTA takes the larger share of every
    // layer
    auto share = [&](int l, int& lo, int& cnt) {
        const int n = s_desc[l].n;
        const int b = (int)((blockIdx.x + (unsigned)l) % (unsigned)G);
        lo = (int)((long long)n * b / G);
        cnt = (int)((long long)n * (b + 1) / G) - lo;
    };

    if (warp == kConsWarps) {
        const uint64_t pol = policy_evict_first();
        const uint32_t rec_bytes = (uint32_t)(6 * d);
        int ibase = 0;
        for (int l = 0; l < L; ++l) {
            int lo, cnt;
            share(l, lo, cnt);
            const uint16_t* packed = s_desc[l].packed;
            produce_by_index(
                s_desc[l].pos + lo, cnt, s_desc[l].n_records, R, empty, lerr, kSiteStack | kSiteEmpty,
                [&](int i, int s, int p) {
                    *reinterpret_cast<volatile int*>(seq + s) = i;
                    mbar_arrive_expect_tx(&full[s], rec_bytes);
                    bulk_g2s_hint(ring + (size_t)s * RL.stage, packed + (size_t)p * 3 * d, rec_bytes, &full[s], pol);
                },
                ibase);
            ibase += cnt;
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int tid = threadIdx.x;  // 0 .. 255
    const int q4 = d / 4;         // float4 columns of h
    // the CTA's slice of float4 columns (writing of h) and of a layer's
    // delta copies (zeroing)
    const int z0 = (int)((long long)q4 * blockIdx.x / G), z1 = (int)((long long)q4 * (blockIdx.x + 1) / G);
    const int zc0 = (int)((long long)q4 * kDeltaCopies * blockIdx.x / G);
    const int zc1 = (int)((long long)q4 * kDeltaCopies * (blockIdx.x + 1) / G);
    float4 h[KV];
    // x_l = bf16(h * r), r = 1 / sqrt(mean(h^2) + eps), into shared memory (and
    // x_out[l] from CTA 0). The sum of squares runs in the same order in every
    // CTA (thread columns, warp butterfly, warps 0..7), so every CTA gets the same r.
    auto form_x = [&](int l) {
        float ss = 0.0f;
#pragma unroll
        for (int t = 0; t < KV; ++t) {
            const int k = tid + kConsThreads * t;
            if (k < q4) ss += (h[t].x * h[t].x + h[t].y * h[t].y) + (h[t].z * h[t].z + h[t].w * h[t].w);
        }
        ss = warp_sum(ss);
        if (lane == 0) s_ss[warp] = ss;
        named_bar_sync(1, kConsThreads);
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsWarps; ++w) tot += s_ss[w];
        const float r = 1.0f / sqrtf(tot / (float)d + kNormEps);
#pragma unroll
        for (int t = 0; t < KV; ++t) {
            const int k = tid + kConsThreads * t;
            if (k < q4) {
                const uint2 v = bf16x4(make_float4(h[t].x * r, h[t].y * r, h[t].z * r, h[t].w * r));
                reinterpret_cast<uint2*>(s_x)[k] = v;
                if (P.x_out && blockIdx.x == 0) reinterpret_cast<uint2*>(P.x_out + (size_t)l * d)[k] = v;
            }
        }
    };
#pragma unroll
    for (int t = 0; t < KV; ++t) {
        const int k = tid + kConsThreads * t;
        h[t] = k < q4 ? __ldcg(reinterpret_cast<const float4*>(P.h) + k) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    form_x(0);
    named_bar_sync(1, kConsThreads);

    float acc[XJ][8];
    int ibase = 0;
    for (int l = 0; l < L; ++l) {
        int lo, cnt;
        share(l, lo, cnt);
        (void)lo;
#pragma unroll
        for (int j = 0; j < XJ; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;
        const int iend = ibase + cnt;
        // this warp's records of the layer: ring indices i == warp (mod 8)
        const int ifirst = ibase + ((warp - ibase % kConsWarps) + kConsWarps) % kConsWarps;
        for (int i = ifirst; i < iend; i += kConsWarps) {
            const int s = i % R;
            if (*reinterpret_cast<volatile int*>(seq + s) != i) {
                const long long t0 = cycles();
                while (*reinterpret_cast<volatile int*>(seq + s) != i) {
                    if (cycles() - t0 > kWaitLimitCycles) {
                        if (lane == 0) atomicOr(lerr, SI_DEVERR_WAIT_TIMEOUT | kSiteStack | kSiteFull);
                        break;
                    }
                }
            }
            mbar_wait(&full[s], (uint32_t)((i / R) & 1), lerr, kSiteStack | kSiteFull);
            const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)s * RL.stage);
            float ga[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                const int c = lane + 32 * j;
                const uint4 xv = s_x[c];
                ga[j & 3] = dot8(st[c], xv, ga[j & 3]);
                ua[j & 3] = dot8(st[nch + c], xv, ua[j & 3]);
            }
            const float g = warp_sum((ga[0] + ga[1]) + (ga[2] + ga[3]));
            const float u = warp_sum((ua[0] + ua[1]) + (ua[2] + ua[3]));
            const float a = swiglu(g, u);
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                float f[8];
                unpack8(st[2 * nch + lane + 32 * j], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(a, f[e], acc[j][e]);
            }
            __syncwarp();
            // the stage of the warp's last record of the layer is kept for its partial
            if (lane == 0 && i + kConsWarps < iend) mbar_arrive(&empty[s]);
        }
        // The last record of warp w in [ibase, iend) and its stage (none when
        // the warp had no record of this layer).
        auto last_of = [&](int w) -> int {
            const int ilast = iend - 1 - ((iend - 1 - w) % kConsWarps + kConsWarps) % kConsWarps;
            return ilast >= ibase ? ilast : -1;
        };
        const int my_last = last_of(warp);
        if (my_last >= 0) {
            // layout per warp stage: for chunk j, the lanes' first halves (4
            // floats each), then their second halves (bank-conflict free)
            float4* wst = reinterpret_cast<float4*>(ring + (size_t)(my_last % R) * RL.stage);
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                wst[j * 64 + lane] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
                wst[j * 64 + 32 + lane] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
            }
        }
        named_bar_sync(1, kConsThreads);  // every warp's partial is in its stage
        float* dl = P.delta + (size_t)l * kDeltaCopies * d;   // delta_l: kDeltaCopies copies of [d]
        float* mine = dl + (size_t)(blockIdx.x % kDeltaCopies) * d;
        {
            int wstage[kConsWarps];
#pragma unroll
            for (int w = 0; w < kConsWarps; ++w) {
                const int il = last_of(w);
                wstage[w] = il >= 0 ? il % R : -1;
            }
#pragma unroll
            for (int t = 0; t < KV; ++t) {
                const int k = tid + kConsThreads * t;
                if (k < q4) {
                    const int c = k >> 1, off = (c >> 5) * 64 + (k & 1) * 32 + (c & 31);
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int w = 0; w < kConsWarps; ++w)
                        if (wstage[w] >= 0) {
                            const float4 q = reinterpret_cast<const float4*>(ring + (size_t)wstage[w] * RL.stage)[off];
                            v.x += q.x; v.y += q.y; v.z += q.z; v.w += q.w;
                        }
                    red_add4(mine + 4 * k, v);
                }
            }
        }
        named_bar_sync(1, kConsThreads);  // the stages have been read; the CTA's sum is on its way
        if (lane == 0 && my_last >= 0) mbar_arrive(&empty[my_last % R]);
        if (warp == 0) grid_arrive_wait(P.sync + stack_bar_word(l, 0), G, lerr);
        named_bar_sync(1, kConsThreads);  // every CTA's sum is in delta_l
        // every CTA has read delta_{l-1} (before arriving at barrier l): zero this CTA's slice of it
        if (l >= 1) {
            float4* dp = reinterpret_cast<float4*>(P.delta + (size_t)(l - 1) * kDeltaCopies * d);
            for (int k = zc0 + tid; k < zc1; k += kConsThreads) dp[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // h += sum of the copies in copy order (the same in every CTA)
#pragma unroll
        for (int t = 0; t < KV; ++t) {
            const int k = tid + kConsThreads * t;
            if (k < q4) {
                float4 v[kDeltaCopies];
#pragma unroll
                for (int c = 0; c < kDeltaCopies; ++c) v[c] = __ldcg(reinterpret_cast<const float4*>(dl + (size_t)c * d) + k);
                float4 sum = v[0];
#pragma unroll
                for (int c = 1; c < kDeltaCopies; ++c) {
                    sum.x += v[c].x; sum.y += v[c].y; sum.z += v[c].z; sum.w += v[c].w;
                }
                h[t].x += sum.x; h[t].y += sum.y; h[t].z += sum.z; h[t].w += sum.w;
            }
        }
        if (l + 1 < L) form_x(l + 1);
        named_bar_sync(1, kConsThreads);  // x_{l+1} is in place
        ibase = iend;
    }

    // h after the last layer: each CTA writes its slice (every CTA read the
    // input h before arriving at barrier 0)
#pragma unroll
    for (int t = 0; t < KV; ++t) {
        const int k = tid + kConsThreads * t;
        if (k >= z0 && k < z1) reinterpret_cast<float4*>(P.h)[k] = h[t];
    }
    named_bar_sync(1, kConsThreads);
    if (tid == 0) {
        __threadfence();
        s_flag = (atomicAdd(P.sync + stack_ticket_word(L), 1u) == (unsigned)G - 1) ? 1u : 0u;
    }
    named_bar_sync(1, kConsThreads);
    if (s_flag) {
        // the last CTA out: every CTA has passed every barrier and read delta_{L-1}
        __threadfence();
        float4* dp = reinterpret_cast<float4*>(P.delta + (size_t)(L - 1) * kDeltaCopies * d);
        for (int k = tid; k < q4 * kDeltaCopies; k += kConsThreads) dp[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = tid; i < L * kBarLines; i += kConsThreads) P.sync[stack_bar_word(i / kBarLines, i % kBarLines)] = 0u;
        if (tid == 0) P.sync[stack_ticket_word(L)] = 0u;
        if (tid == 0) {
            const unsigned v = atomicExch(lerr, 0u);
            if (v) atomicOr(P.err, v);
        }
    }
}

int sparse_decode_stack_stages(int d) {
    if (!sparse_decode_stack_width_ok(d)) return 0;
    constexpr int kBudget = 227 * 1024 - 4096;  // leaves room for the static shared memory
    const int fixed = stack_layout(0, d).total;
    int R = (kBudget - fixed - 16 * kStackMaxStages) / round_up(6 * d, 128);
    if (R > kStackMaxStages) R = kStackMaxStages;
    return R >= kConsWarps ? R : 0;
}

namespace {
template <int XJ>
cudaError_t launch_stack(const StackParams& P, int sms, cudaStream_t st) {
    auto kern = k_sparse_decode_stack<XJ>;
    cudaError_t e = allow_max_smem(kern);
    if (e != cudaSuccess) return e;
    StackParams Pc = P;
    void* args[] = {&Pc};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms, 1, 1);  // one CTA per SM; the cooperative launch guarantees co-residency
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)stack_layout(P.R, P.d).total;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kern), args);
}
}  // namespace

bool sparse_decode_stack_width_ok(int d) {
    return d == 256 || d == 512 || d == 1024 || d == 2048 || d == 3072;
}

cudaError_t launch_sparse_decode_stack(const StackParams& P, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    switch (P.d) {
        case 256: return launch_stack<1>(P, sms, st);
        case 512: return launch_stack<2>(P, sms, st);
        case 1024: return launch_stack<4>(P, sms, st);
        case 2048: return launch_stack<8>(P, sms, st);
        case 3072: return launch_stack<12>(P, sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace si
