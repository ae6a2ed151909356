// spax_in.cu -- SpAx tiers on the gate/up projections, chosen by |x|.
//
// The SpAx page's "ALL" configuration applies the three-tier approximation to
// every projection whose weights are offloaded; for the FFN that adds the
// gate and up projections to the down projection. For gate/up the tiers are
// over input channels j (the columns of Wg and Wu), ranked by |x_j| (ties to
// the lower index): the top k_top channels are read in bf16, the next k_mid
// are rebuilt from their own b-bit codes (groups of consecutive neurons along
// the column), the rest are skipped:
//     g = sum_{j in top} x_j Wg[:, j] + sum_{j in mid} x_j w^_j      (u likewise)
//     a = silu(g) * u
// The encoded gate (up) weights are a spax_layer made from Wg (Wu) read as a
// [N x d] matrix whose columns are the input channels: its column-major copy
// is Wg^T (channel j's N gate weights contiguous) and its records hold each
// channel's codes over the N neurons, then the (scale, min) pairs.
//
// k_spax_gate_up: one CTA per slice of S <= 128 consecutive neurons, 16
// warps. Every CTA takes the channel tiers itself from x (4096 keys fit a
// CTA: a two-digit radix selection on the 15-bit bf16 magnitude, then the
// members in index order), then streams its slice of every top and middle
// channel -- 2S bytes of a bf16 column, or S*b/8 code bytes and one (scale,
// min) pair -- with vector loads: the pieces are far too small for bulk copies.
// Warps take list entries round robin, lanes take four neurons each; the 16
// warp partials of g and u are summed in warp order (deterministic), and the
// CTA writes a for its slice together with the down projection's tier
// histogram and member lists, so the tiered down-projection can follow.
#include "common.cuh"
#include "internal.h"

namespace si {

namespace {

constexpr int kGuWarps = 16;
constexpr int kGuThreads = kGuWarps * 32;
constexpr int kGuUnroll = 8;  // list entries in flight per warp and pass

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// The b-bit codes of four consecutive neurons starting at neuron n (n % 4 ==
// 0), element i at bit i*b of the channel's stream.
template <int BITS>
__device__ __forceinline__ uint32_t codes4(const uint8_t* __restrict__ rec, int n) {
    if constexpr (BITS == 8) {
        return __ldcs(reinterpret_cast<const unsigned*>(rec + n));
    } else if constexpr (BITS == 4) {
        return __ldcs(reinterpret_cast<const unsigned short*>(rec + n / 2));
    } else if constexpr (BITS == 2) {
        return __ldcs(rec + n / 4);
    } else {  // BITS == 3: 12 bits from bit 3n, which starts a byte or the middle of one
        const int bit = 3 * n;
        const uint8_t* p = rec + bit / 8;
        const uint32_t w = (uint32_t)__ldcs(p) | ((uint32_t)__ldcs(p + 1) << 8);
        return (w >> (bit % 8)) & 0xFFFu;
    }
}

}  // namespace

template <int BITS>
__global__ void __launch_bounds__(kGuThreads, 1) k_spax_gate_up(GateUpTierParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int d = P.d, N = P.N, S = P.S;
    float* s_xf = reinterpret_cast<float*>(smem);                       // [d] x as float
    uint16_t* s_key = reinterpret_cast<uint16_t*>(s_xf + d);            // [d] |x| keys
    int32_t* s_list = reinterpret_cast<int32_t*>(s_key + ((d + 7) & ~7));  // top then middle channels
    float* s_part = reinterpret_cast<float*>(s_list + d);               // [kGuWarps][2S] partials
    __shared__ unsigned s_h[2][256];
    __shared__ unsigned s_w[kGuWarps][4];
    __shared__ unsigned s_state[8];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * S;
    const int n1 = min(N, n0 + S);

    grid_launch_dependents();
    grid_dependency_wait();  // x may be the previous grid's output

    // ---- x and the |x| keys (bf16 magnitude: the sign bit cleared)
    for (int j = tid; j < d; j += kGuThreads) {
        const uint16_t xb = P.x[j];
        s_xf[j] = bf2f(xb);
        s_key[j] = (uint16_t)(xb & 0x7FFFu);
    }
    for (int i = tid; i < 512; i += kGuThreads) (&s_h[0][0])[i] = 0u;
    __syncthreads();

    // ---- the two rank boundaries K0 = k_top, K1 = k_top + k_mid (largest first)
    const int K[2] = {P.k_top, P.k_top + P.k_mid};
    const bool act[2] = {K[0] > 0 && K[0] < d, K[1] > 0 && K[1] < d};
    for (int j = tid; j < d; j += kGuThreads) atomicAdd(&s_h[0][s_key[j] >> 7], 1u);
    __syncthreads();
    // warp 0: the digit-1 bin holding each boundary's K-th largest key. Lane l
    // owns bins 255 - 8l - i (i < 8): lanes in descending bin order.
    if (warp == 0) {
        uint32_t c[8], tot = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = s_h[0][255 - 8 * lane - i];
            tot += c[i];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        const uint32_t excl = incl - tot;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t k = (uint32_t)K[t];
            if (act[t] && excl < k && k <= incl) {
                uint32_t run = excl;
                for (int i = 0; i < 8; ++i) {
                    if (run + c[i] >= k) {
                        s_state[2 * t] = (uint32_t)(255 - 8 * lane - i);
                        s_state[2 * t + 1] = k - run;  // rank left inside the bin
                        break;
                    }
                    run += c[i];
                }
            }
        }
    }
    __syncthreads();
    const uint32_t b0 = act[0] ? s_state[0] : 0xFFFFu, b1 = act[1] ? s_state[2] : 0xFFFFu;
    const uint32_t r0 = act[0] ? s_state[1] : 0u, r1 = act[1] ? s_state[3] : 0u;
    for (int i = tid; i < 512; i += kGuThreads) (&s_h[0][0])[i] = 0u;
    __syncthreads();
    for (int j = tid; j < d; j += kGuThreads) {
        const uint32_t k = s_key[j];
        if ((k >> 7) == b0) atomicAdd(&s_h[0][k & 127u], 1u);
        if ((k >> 7) == b1) atomicAdd(&s_h[1][k & 127u], 1u);
    }
    __syncthreads();
    // warp 0: the exact key of each boundary and how many keys equal to it it takes
    if (warp == 0) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (!act[t]) continue;
            const uint32_t k = t ? r1 : r0;
            uint32_t c[4], tot = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                c[i] = s_h[t][127 - 4 * lane - i];
                tot += c[i];
            }
            uint32_t incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            const uint32_t excl = incl - tot;
            if (excl < k && k <= incl) {
                uint32_t run = excl;
                for (int i = 0; i < 4; ++i) {
                    if (run + c[i] >= k) {
                        s_state[4 + 2 * t] = ((t ? b1 : b0) << 7) | (uint32_t)(127 - 4 * lane - i);
                        s_state[5 + 2 * t] = k - run;
                        break;
                    }
                    run += c[i];
                }
            }
        }
    }
    __syncthreads();
    // Boundary t takes every key > thr[t] and the first take[t] keys == thr[t]
    // in index order; K == 0 takes nothing, K == d everything.
    uint32_t thr[2], take[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (act[t]) {
            thr[t] = s_state[4 + 2 * t];
            take[t] = s_state[5 + 2 * t];
        } else if (K[t] <= 0) {
            thr[t] = 0xFFFFu;  // above every key
            take[t] = 0u;
        } else {
            thr[t] = 0u;
            take[t] = 0xFFFFFFFFu;
        }
    }

    // ---- members in index order: warp w owns indices [w * SEG, (w + 1) * SEG)
    const int SEG = ((d + kGuWarps * 32 - 1) / (kGuWarps * 32)) * 32;
    const int lo = warp * SEG, hi = min(d, lo + SEG);
    const uint32_t lt = lanemask_lt();
    // pass 1: keys equal to each threshold, per warp
    uint32_t q0 = 0u, q1 = 0u;
    for (int i0 = lo; i0 < hi; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t k = i < hi ? s_key[i] : 0x10000u;
        q0 += __popc(__ballot_sync(0xFFFFFFFFu, k == thr[0]));
        q1 += __popc(__ballot_sync(0xFFFFFFFFu, k == thr[1]));
    }
    if (lane == 0) {
        s_w[warp][0] = q0;
        s_w[warp][1] = q1;
    }
    __syncthreads();
    uint32_t e0 = 0u, e1 = 0u;
    for (int w = 0; w < warp; ++w) {
        e0 += s_w[w][0];
        e1 += s_w[w][1];
    }
    __syncthreads();
    // pass 2 counts the warp's members, pass 3 writes them at their list slots
    uint32_t base_t = 0u, base_m = 0u;
    for (int pass = 0; pass < 2; ++pass) {
        uint32_t ra = e0, rb = e1, ct = 0u, cm = 0u;
        for (int i0 = lo; i0 < hi; i0 += 32) {
            const int i = i0 + lane;
            const bool in = i < hi;
            const uint32_t k = in ? s_key[i] : 0x10000u;
            const uint32_t ea = __ballot_sync(0xFFFFFFFFu, in && k == thr[0]);
            const uint32_t eb = __ballot_sync(0xFFFFFFFFu, in && k == thr[1]);
            const bool sel0 = in && (k > thr[0] || (k == thr[0] && ra + __popc(ea & lt) < take[0]));
            const bool sel1 = in && (k > thr[1] || (k == thr[1] && rb + __popc(eb & lt) < take[1]));
            ra += __popc(ea);
            rb += __popc(eb);
            const bool mid = sel1 && !sel0;
            const uint32_t bt = __ballot_sync(0xFFFFFFFFu, sel0), bm = __ballot_sync(0xFFFFFFFFu, mid);
            if (pass == 1) {
                if (sel0) s_list[base_t + ct + __popc(bt & lt)] = i;
                if (mid) s_list[P.k_top + base_m + cm + __popc(bm & lt)] = i;
            }
            ct += __popc(bt);
            cm += __popc(bm);
        }
        if (pass == 0) {
            if (lane == 0) {
                s_w[warp][2] = ct;
                s_w[warp][3] = cm;
            }
            __syncthreads();
            uint32_t nt = 0u, nm = 0u;
            for (int w = 0; w < kGuWarps; ++w) {
                if (w < warp) {
                    base_t += s_w[w][2];
                    base_m += s_w[w][3];
                }
                nt += s_w[w][2];
                nm += s_w[w][3];
            }
            if (tid == 0 && (nt != (uint32_t)P.k_top || nm != (uint32_t)P.k_mid)) atomicOr(P.err, SI_DEVERR_COUNT);
            if (nt != (uint32_t)P.k_top || nm != (uint32_t)P.k_mid) {
                // never write outside the list: leave it empty
                base_t = base_m = 0xFFFFFFFFu;
                break;
            }
        }
    }
    __syncthreads();
    const bool lists_ok = base_t != 0xFFFFFFFFu;
    if (blockIdx.x == 0 && lists_ok) {
        if (P.top_out)
            for (int e = tid; e < P.k_top; e += kGuThreads) P.top_out[e] = s_list[e];
        if (P.mid_out)
            for (int e = tid; e < P.k_mid; e += kGuThreads) P.mid_out[e] = s_list[P.k_top + e];
    }
    const int n_top = lists_ok ? P.k_top : 0, n_mid = lists_ok ? P.k_mid : 0;

    // ---- streaming: lane l takes neurons n0 + 4l .. n0 + 4l + 3
    const int nb = n0 + 4 * lane;
    const bool live = 4 * lane < S && nb < n1;  // slices are whole multiples of 4 neurons
    float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
    for (int e0 = warp; e0 < n_top; e0 += kGuWarps * kGuUnroll) {
        uint2 gv[kGuUnroll], uv[kGuUnroll];
        float xv[kGuUnroll];
#pragma unroll
        for (int k = 0; k < kGuUnroll; ++k) {
            const int e = e0 + kGuWarps * k;
            xv[k] = 0.0f;
            gv[k] = uv[k] = make_uint2(0u, 0u);
            if (e < n_top && live) {
                const int j = s_list[e];
                xv[k] = s_xf[j];
                gv[k] = __ldcs(reinterpret_cast<const uint2*>(P.WgT + (size_t)j * N + nb));
                uv[k] = __ldcs(reinterpret_cast<const uint2*>(P.WuT + (size_t)j * N + nb));
            }
        }
#pragma unroll
        for (int k = 0; k < kGuUnroll; ++k) {
            g[0] = fmaf(xv[k], bf_lo(gv[k].x), g[0]);
            g[1] = fmaf(xv[k], bf_hi(gv[k].x), g[1]);
            g[2] = fmaf(xv[k], bf_lo(gv[k].y), g[2]);
            g[3] = fmaf(xv[k], bf_hi(gv[k].y), g[3]);
            u[0] = fmaf(xv[k], bf_lo(uv[k].x), u[0]);
            u[1] = fmaf(xv[k], bf_hi(uv[k].x), u[1]);
            u[2] = fmaf(xv[k], bf_lo(uv[k].y), u[2]);
            u[3] = fmaf(xv[k], bf_hi(uv[k].y), u[3]);
        }
    }
    const int code_bytes = N * BITS / 8;
    const int gi = live ? nb / P.group : 0;  // the four neurons share one group (group % 4 == 0)
    constexpr uint32_t kMask = (1u << BITS) - 1u;
    for (int e0 = warp; e0 < n_mid; e0 += kGuWarps * kGuUnroll) {
        uint32_t gq[kGuUnroll], uq[kGuUnroll];
        float2 gp[kGuUnroll], up[kGuUnroll];
        float xv[kGuUnroll];
#pragma unroll
        for (int k = 0; k < kGuUnroll; ++k) {
            const int e = e0 + kGuWarps * k;
            xv[k] = 0.0f;
            gq[k] = uq[k] = 0u;
            gp[k] = up[k] = make_float2(0.f, 0.f);
            if (e < n_mid && live) {
                const int j = s_list[P.k_top + e];
                xv[k] = s_xf[j];
                const uint8_t* rg = P.gcodes + (size_t)j * P.rec_bytes;
                const uint8_t* ru = P.ucodes + (size_t)j * P.rec_bytes;
                gq[k] = codes4<BITS>(rg, nb);
                uq[k] = codes4<BITS>(ru, nb);
                gp[k] = __ldcs(reinterpret_cast<const float2*>(rg + code_bytes) + gi);
                up[k] = __ldcs(reinterpret_cast<const float2*>(ru + code_bytes) + gi);
            }
        }
#pragma unroll
        for (int k = 0; k < kGuUnroll; ++k) {
            // x_j * (min + q * scale) = x_j * min + (x_j * scale) * q
            const float gs = xv[k] * gp[k].x, gm = xv[k] * gp[k].y;
            const float us = xv[k] * up[k].x, um = xv[k] * up[k].y;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                g[i] = fmaf(gs, (float)((gq[k] >> (BITS * i)) & kMask), g[i] + gm);
                u[i] = fmaf(us, (float)((uq[k] >> (BITS * i)) & kMask), u[i] + um);
            }
        }
    }

    // ---- warp partials -> the slice's a, in warp order
    if (live) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s_part[warp * 2 * S + 4 * lane + i] = g[i];
            s_part[warp * 2 * S + S + 4 * lane + i] = u[i];
        }
    }
    __syncthreads();
    for (int t = tid; t < n1 - n0; t += kGuThreads) {
        float gs = 0.0f, us = 0.0f;
        for (int w = 0; w < kGuWarps; ++w) {
            gs += s_part[w * 2 * S + t];
            us += s_part[w * 2 * S + S + t];
        }
        const float av = swiglu(gs, us);
        const int n = n0 + t;
        P.a[n] = av;
        if (P.hist) {
            const uint32_t bin = abs_key(av) >> kTierShift;
            const uint32_t slot = atomicAdd(P.hist + bin, 1u);
            if (P.slab && slot < (uint32_t)kSlabCap) P.slab[(size_t)bin * kSlabCap + slot] = n;
        }
    }
}

int spax_gate_up_slice(int N) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) return 0;
    int S = (N + sms - 1) / sms;
    S = (S + 3) / 4 * 4;
    return S < 128 ? (S < 4 ? 4 : S) : 128;
}

size_t spax_gate_up_smem(int d, int S) {
    return (size_t)d * 4 + (size_t)((d + 7) & ~7) * 2 + (size_t)d * 4 + (size_t)kGuWarps * 2 * S * 4;
}

cudaError_t launch_spax_gate_up(const GateUpTierParams& P, cudaStream_t st) {
    if (P.S < 4 || P.S % 4 || P.S > 128 || P.group % 4) return cudaErrorInvalidValue;
    const size_t smem = spax_gate_up_smem(P.d, P.S);
    const int grid = (P.N + P.S - 1) / P.S;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kGuThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    switch (P.bits) {
#define SI_GU(b)                                                              \
    case b:                                                                   \
        if ((e = allow_max_smem(k_spax_gate_up<b>)) != cudaSuccess) return e; \
        return cudaLaunchKernelEx(&cfg, k_spax_gate_up<b>, P);
        SI_GU(2)
        SI_GU(3)
        SI_GU(4)
        SI_GU(8)
#undef SI_GU
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace si
