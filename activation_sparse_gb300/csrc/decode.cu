// decode.cu -- HBM-streaming decode kernels (one token per sequence).
//
//  k_sparse_decode  SelectInfer sparse decode FFN (section 5: only the
//                   selected neurons are computed): for each selected packed
//                   record [gate row | up row | down column] it forms
//                   a = silu(g.x) * (u.x) and accumulates a * down into a
//                   per-CTA partial of y.
//  k_dense_act      SpAx dense gate/up pass: a[n] for every neuron.
//  k_tiered_down    SpAx three-tier down-projection (abstract, Fig. 2/3):
//                   top columns in bf16, middle columns rebuilt from 4-bit
//                   codes (min + q * scale), the rest never read.
//
// Common structure (warp-specialised, one CTA per SM):
//   * warp 8, lane 0 streams whole records into a ring of shared-memory
//     stages with 1-D bulk copies (cp.async.bulk, completion counted in bytes
//     on a per-stage "full" mbarrier); consumer warps release a stage through
//     its "empty" mbarrier. Every wait is bounded.
//   * records are split evenly over the CTAs of the grid (split-K over
//     neurons / columns), each CTA keeps its partial y in registers;
//   * reduction: the CTAs of a thread-block cluster sum their partials
//     through distributed shared memory (each CTA owns a slice of y), write
//     one partial per cluster, and the last cluster to finish a slice (an
//     atomic ticket, no waiting) sums the cluster partials in fixed order.
//     The result is deterministic run to run.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace si {

constexpr int kConsWarps = 8;
constexpr int kConsThreads = kConsWarps * 32;
constexpr int kDecThreads = kConsThreads + 32;

__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Shared-memory layout of the streaming kernels (host and device agree).
struct RingLayout {
    int off_full, off_empty, off_aux, off_x, off_ring, stage, R, total;
};

__host__ __device__ inline RingLayout ring_layout(int R, int stage_bytes, int aux_bytes, int x_bytes) {
    RingLayout L;
    L.R = R;
    L.stage = round_up(stage_bytes, 128);
    L.off_full = 0;
    L.off_empty = 8 * R;
    L.off_aux = round_up(16 * R, 128);
    L.off_x = L.off_aux + round_up(aux_bytes, 128);
    L.off_ring = L.off_x + round_up(x_bytes, 128);
    L.total = L.off_ring + R * L.stage;
    return L;
}

// Cluster-level then grid-level reduction of the per-CTA partials ypart[BD]
// (shared memory) into y[BD]. Must be called by every thread of every CTA.
__device__ void cluster_ticket_reduce(float* ypart, int BD, float* __restrict__ part, unsigned* tickets,
                                      float* __restrict__ y) {
    __shared__ unsigned s_last;
    cg::cluster_group cl = cg::this_cluster();
    const unsigned C = cl.num_blocks();
    const unsigned r = cl.block_rank();
    const unsigned ncl = gridDim.x / C;
    const unsigned cid = blockIdx.x / C;
    cl.sync();
    const int per = (BD + (int)C - 1) / (int)C;
    const int s0 = (int)r * per;
    const int s1 = min(BD, s0 + per);
    for (int idx = s0 + (int)threadIdx.x; idx < s1; idx += blockDim.x) {
        float v = 0.0f;
        for (unsigned c = 0; c < C; ++c) v += cl.map_shared_rank(ypart, c)[idx];
        __stcg(part + (size_t)cid * BD + idx, v);
    }
    __threadfence();
    cl.sync();  // no CTA leaves while a peer still reads its shared memory
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned t = atomicAdd(tickets + r, 1u);
        s_last = (t == ncl - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int idx = s0 + (int)threadIdx.x; idx < s1; idx += blockDim.x) {
            float v = 0.0f;
            for (unsigned k = 0; k < ncl; ++k) v += __ldcg(part + (size_t)k * BD + idx);
            y[idx] = v;
        }
        if (threadIdx.x == 0) tickets[r] = 0u;
    }
}

// ----------------------------------------------------------- sparse decode

// B sequences (B <= 8); MAXC = ceil(d / 2048) column chunks of 8 per thread.
template <int B, int MAXC>
__global__ void __launch_bounds__(kDecThreads, 1) k_sparse_decode(SparseDecodeParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int d = P.d;
    const RingLayout L = ring_layout(P.R, 6 * d, 2 * kConsWarps * B * 4, B * d * 2);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    float* s_a = reinterpret_cast<float*>(smem + L.off_aux);
    uint16_t* s_x = reinterpret_cast<uint16_t*>(smem + L.off_x);
    uint8_t* ring = smem + L.off_ring;
    const int R = L.R;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = P.n_dev ? *P.n_dev : P.n_host;
    const int lo = (int)((long long)n * blockIdx.x / gridDim.x);
    const int hi = (int)((long long)n * (blockIdx.x + 1) / gridDim.x);
    const int cnt = hi - lo;
    const uint32_t rec_bytes = (uint32_t)(6 * d);

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsWarps);
        }
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < B * d / 8; i += blockDim.x)
        reinterpret_cast<uint4*>(s_x)[i] = reinterpret_cast<const uint4*>(P.x)[i];
    __syncthreads();

    if (warp == kConsWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < cnt; ++i) {
                const int s = i % R;
                if (i >= R) mbar_wait(&empty[s], (uint32_t)((i / R - 1) & 1), P.err, kSiteDecode | kSiteEmpty);
                int p = P.pos[lo + i];
                if (p < 0 || p >= P.n_records) {  // never read outside the packed buffer
                    atomicOr(P.err, SI_DEVERR_COUNT);
                    p = 0;
                }
                mbar_arrive_expect_tx(&full[s], rec_bytes);
                bulk_g2s_hint(ring + (size_t)s * L.stage, P.packed + (size_t)p * 3 * d, rec_bytes, &full[s], pol);
            }
        }
        __syncwarp();
    } else {
        float acc[MAXC][8][B];
#pragma unroll
        for (int j = 0; j < MAXC; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int b = 0; b < B; ++b) acc[j][e][b] = 0.0f;
        constexpr int XJ = 8 * MAXC;  // lane chunks of x kept in registers (B == 1)
        uint4 xr[B == 1 ? XJ : 1];
        if constexpr (B == 1) {
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                const int c = lane + 32 * j;
                xr[j] = (c < d / 8) ? reinterpret_cast<const uint4*>(s_x)[c] : make_uint4(0u, 0u, 0u, 0u);
            }
        }
        const int tid = threadIdx.x;  // 0 .. 255
        const int iters = (cnt + kConsWarps - 1) / kConsWarps;
        for (int it = 0; it < iters; ++it) {
            float* a_buf = s_a + (it & 1) * kConsWarps * B;
            const int i = it * kConsWarps + warp;
            if (i < cnt) {
                const int s = i % R;
                mbar_wait(&full[s], (uint32_t)((i / R) & 1), P.err, kSiteDecode | kSiteFull);
                const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)s * L.stage);
                float g[B], u[B];
#pragma unroll
                for (int b = 0; b < B; ++b) g[b] = u[b] = 0.0f;
                if constexpr (B == 1) {
#pragma unroll
                    for (int j = 0; j < XJ; ++j) {
                        const int c = lane + 32 * j;
                        if (c < d / 8) {
                            g[0] = dot8(st[c], xr[j], g[0]);
                            u[0] = dot8(st[d / 8 + c], xr[j], u[0]);
                        }
                    }
                } else {
                    for (int c = lane; c < d / 8; c += 32) {
                        const uint4 gv = st[c], uv = st[d / 8 + c];
#pragma unroll
                        for (int b = 0; b < B; ++b) {
                            const uint4 xv = reinterpret_cast<const uint4*>(s_x + b * d)[c];
                            g[b] = dot8(gv, xv, g[b]);
                            u[b] = dot8(uv, xv, u[b]);
                        }
                    }
                }
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    g[b] = warp_sum(g[b]);
                    u[b] = warp_sum(u[b]);
                }
                const uint32_t m = P.pmask ? P.pmask[lo + i] : 0xFFFFFFFFu;
                if (lane == 0) {
#pragma unroll
                    for (int b = 0; b < B; ++b) a_buf[warp * B + b] = ((m >> b) & 1u) ? swiglu(g[b], u[b]) : 0.0f;
                }
            }
            named_bar_sync(1, kConsThreads);
            const int nb = min(kConsWarps, cnt - it * kConsWarps);
            for (int w2 = 0; w2 < nb; ++w2) {
                const int i2 = it * kConsWarps + w2;
                const int s2 = i2 % R;
                mbar_wait(&full[s2], (uint32_t)((i2 / R) & 1), P.err, kSiteDecode | kSiteFullB);
                const uint4* dn = reinterpret_cast<const uint4*>(ring + (size_t)s2 * L.stage) + 2 * (d / 8);
                float av[B];
#pragma unroll
                for (int b = 0; b < B; ++b) av[b] = a_buf[w2 * B + b];
#pragma unroll
                for (int j = 0; j < MAXC; ++j) {
                    const int c = tid + kConsThreads * j;
                    if (c < d / 8) {
                        float f[8];
                        unpack8(dn[c], f);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
#pragma unroll
                            for (int b = 0; b < B; ++b) acc[j][e][b] = fmaf(av[b], f[e], acc[j][e][b]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                for (int w2 = 0; w2 < nb; ++w2) mbar_arrive(&empty[(it * kConsWarps + w2) % R]);
        }
        named_bar_sync(1, kConsThreads);  // every consumer is done with the ring
        float* ypart = reinterpret_cast<float*>(ring);
#pragma unroll
        for (int j = 0; j < MAXC; ++j) {
            const int c = tid + kConsThreads * j;
            if (c < d / 8) {
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    float4* dst = reinterpret_cast<float4*>(ypart + (size_t)b * d + c * 8);
                    dst[0] = make_float4(acc[j][0][b], acc[j][1][b], acc[j][2][b], acc[j][3][b]);
                    dst[1] = make_float4(acc[j][4][b], acc[j][5][b], acc[j][6][b], acc[j][7][b]);
                }
            }
        }
    }
    __syncthreads();
    cluster_ticket_reduce(reinterpret_cast<float*>(ring), B * d, P.part, P.tickets, P.y);
}

// --------------------------------------------------------------- dense act

template <int MAXC>
__global__ void __launch_bounds__(kDecThreads, 1) k_dense_act(DenseActParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int d = P.d;
    const RingLayout L = ring_layout(P.R, 4 * d, 0, d * 2);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    uint16_t* s_x = reinterpret_cast<uint16_t*>(smem + L.off_x);
    uint8_t* ring = smem + L.off_ring;
    const int R = L.R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lo = (int)((long long)P.N * blockIdx.x / gridDim.x);
    const int hi = (int)((long long)P.N * (blockIdx.x + 1) / gridDim.x);
    const int cnt = hi - lo;
    const uint32_t row_bytes = (uint32_t)(2 * d);

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x)
        reinterpret_cast<uint4*>(s_x)[i] = reinterpret_cast<const uint4*>(P.x)[i];
    __syncthreads();

    if (warp == kConsWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < cnt; ++i) {
                const int s = i % R;
                if (i >= R) mbar_wait(&empty[s], (uint32_t)((i / R - 1) & 1), P.err, kSiteDenseAct | kSiteEmpty);
                const size_t n = (size_t)(lo + i);
                uint8_t* dst = ring + (size_t)s * L.stage;
                mbar_arrive_expect_tx(&full[s], 2 * row_bytes);
                bulk_g2s_hint(dst, P.Wg + n * d, row_bytes, &full[s], pol);
                bulk_g2s_hint(dst + row_bytes, P.Wu + n * d, row_bytes, &full[s], pol);
            }
        }
        __syncwarp();
    } else {
        constexpr int XJ = 8 * MAXC;
        uint4 xr[XJ];
#pragma unroll
        for (int j = 0; j < XJ; ++j) {
            const int c = lane + 32 * j;
            xr[j] = (c < d / 8) ? reinterpret_cast<const uint4*>(s_x)[c] : make_uint4(0u, 0u, 0u, 0u);
        }
        for (int i = warp; i < cnt; i += kConsWarps) {
            const int s = i % R;
            mbar_wait(&full[s], (uint32_t)((i / R) & 1), P.err, kSiteDenseAct | kSiteFull);
            const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)s * L.stage);
            float g = 0.0f, u = 0.0f;
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                const int c = lane + 32 * j;
                if (c < d / 8) {
                    g = dot8(st[c], xr[j], g);
                    u = dot8(st[d / 8 + c], xr[j], u);
                }
            }
            g = warp_sum(g);
            u = warp_sum(u);
            __syncwarp();
            if (lane == 0) {
                P.a[lo + i] = swiglu(g, u);
                mbar_arrive(&empty[s]);
            }
        }
    }
}

// ---------------------------------------------------------- tiered down

template <int MAXC>
__global__ void __launch_bounds__(kDecThreads, 1) k_tiered_down(TieredDownParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int d = P.d;
    const int mid_bytes = d / 2 + P.ngp * 8;
    const RingLayout L = ring_layout(P.R, 2 * d, P.aux_floats * 4, 0);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    float* s_av = reinterpret_cast<float*>(smem + L.off_aux);
    uint8_t* ring = smem + L.off_ring;
    const int R = L.R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = (int)((long long)P.k_top * blockIdx.x / gridDim.x);
    const int t1 = (int)((long long)P.k_top * (blockIdx.x + 1) / gridDim.x);
    const int m0 = (int)((long long)P.k_mid * blockIdx.x / gridDim.x);
    const int m1 = (int)((long long)P.k_mid * (blockIdx.x + 1) / gridDim.x);
    const int ntop = t1 - t0, nrec = ntop + (m1 - m0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsWarps);
        }
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < nrec; i += blockDim.x) {
        const int col = i < ntop ? P.top[t0 + i] : P.mid[m0 + i - ntop];
        s_av[i] = (col >= 0 && col < P.N) ? P.a[col] : 0.0f;
    }
    __syncthreads();

    if (warp == kConsWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < nrec; ++i) {
                const int s = i % R;
                if (i >= R) mbar_wait(&empty[s], (uint32_t)((i / R - 1) & 1), P.err, kSiteTiered | kSiteEmpty);
                uint8_t* dst = ring + (size_t)s * L.stage;
                int ci = i < ntop ? P.top[t0 + i] : P.mid[m0 + i - ntop];
                if (ci < 0 || ci >= P.N) {  // never read outside the encoded buffers
                    atomicOr(P.err, SI_DEVERR_COUNT);
                    ci = 0;
                }
                const size_t col = (size_t)ci;
                if (i < ntop) {
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * d));
                    bulk_g2s_hint(dst, P.WdT + col * d, (uint32_t)(2 * d), &full[s], pol);
                } else {
                    mbar_arrive_expect_tx(&full[s], (uint32_t)mid_bytes);
                    bulk_g2s_hint(dst, P.codes + col * (d / 2), (uint32_t)(d / 2), &full[s], pol);
                    bulk_g2s_hint(dst + d / 2, P.params + col * P.ngp * 2, (uint32_t)(P.ngp * 8), &full[s], pol);
                }
            }
        }
        __syncwarp();
    } else {
        float acc[MAXC][8];
#pragma unroll
        for (int j = 0; j < MAXC; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;
        const int tid = threadIdx.x;
        for (int i = 0; i < nrec; ++i) {
            const int s = i % R;
            mbar_wait(&full[s], (uint32_t)((i / R) & 1), P.err, kSiteTiered | kSiteFull);
            const uint8_t* st = ring + (size_t)s * L.stage;
            const float av = s_av[i];
            if (i < ntop) {
#pragma unroll
                for (int j = 0; j < MAXC; ++j) {
                    const int c = tid + kConsThreads * j;
                    if (c < d / 8) {
                        float f[8];
                        unpack8(reinterpret_cast<const uint4*>(st)[c], f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(av, f[e], acc[j][e]);
                    }
                }
            } else {
                const float2* prm = reinterpret_cast<const float2*>(st + d / 2);
#pragma unroll
                for (int j = 0; j < MAXC; ++j) {
                    const int c = tid + kConsThreads * j;
                    if (c < d / 8) {
                        const uint32_t q = reinterpret_cast<const uint32_t*>(st)[c];
                        const float2 sm = prm[(8 * c) / P.group];  // (scale, min)
                        const float c1 = av * sm.x, c0 = av * sm.y;
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            acc[j][e] += fmaf(c1, (float)((q >> (4 * e)) & 15u), c0);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        named_bar_sync(1, kConsThreads);
        float* ypart = reinterpret_cast<float*>(ring);
#pragma unroll
        for (int j = 0; j < MAXC; ++j) {
            const int c = tid + kConsThreads * j;
            if (c < d / 8) {
                float4* dst = reinterpret_cast<float4*>(ypart + c * 8);
                dst[0] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
                dst[1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
            }
        }
    }
    __syncthreads();
    cluster_ticket_reduce(reinterpret_cast<float*>(ring), d, P.part, P.tickets, P.y);
}

// ------------------------------------------------------------------ launch

namespace {

constexpr int kSmemBudget = 227 * 1024 - 2048;  // dynamic budget, leaves room for static smem

template <class K>
cudaError_t launch_clustered(K kernel, int grid, int cluster, size_t smem, cudaStream_t st, void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kernel), args);
}

// Largest co-resident grid for a clustered streaming kernel: tries cluster
// sizes 8, 4, 2 and keeps the one that puts the most CTAs on the GPU at once.
template <class K>
cudaError_t pick_grid(K kernel, size_t smem, int* grid, int* cluster) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = allow_max_smem(kernel);
    if (e != cudaSuccess) return e;
    int best = 0, bestC = 2;
    for (int C = 8; C >= 2; C /= 2) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((sms / C) * C, 1, 1);
        cfg.blockDim = dim3(kDecThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int ncl = 0;
        e = cudaOccupancyMaxActiveClusters(&ncl, reinterpret_cast<const void*>(kernel), &cfg);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            continue;
        }
        // one CTA per SM at most: the partial buffers are sized for that
        const int ctas = ncl * C < (sms / C) * C ? ncl * C : (sms / C) * C;
        if (ctas > best) {
            best = ctas;
            bestC = C;
        }
    }
    if (best <= 0) return cudaErrorInvalidConfiguration;
    *grid = best;
    *cluster = bestC;
    return cudaSuccess;
}

struct GridCache {
    const void* fn = nullptr;
    size_t smem = 0;
    int dev = -1, grid = 0, cluster = 0;
};

template <class K>
cudaError_t cached_grid(K kernel, size_t smem, int* grid, int* cluster) {
    static thread_local GridCache cache[32];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void* fn = reinterpret_cast<const void*>(kernel);
    for (auto& c : cache)
        if (c.fn == fn && c.smem == smem && c.dev == dev) {
            *grid = c.grid;
            *cluster = c.cluster;
            return cudaSuccess;
        }
    e = pick_grid(kernel, smem, grid, cluster);
    if (e != cudaSuccess) return e;
    for (auto& c : cache)
        if (c.fn == nullptr) {
            c.fn = fn;
            c.smem = smem;
            c.dev = dev;
            c.grid = *grid;
            c.cluster = *cluster;
            break;
        }
    return cudaSuccess;
}

template <int B, int MAXC>
cudaError_t launch_sd(SparseDecodeParams& P, cudaStream_t st, int* grid_out) {
    auto kern = k_sparse_decode<B, MAXC>;
    int grid = 0, cluster = 0;
    const size_t smem = (size_t)ring_layout(P.R, 6 * P.d, 2 * kConsWarps * B * 4, B * P.d * 2).total;
    cudaError_t e = cached_grid(kern, smem, &grid, &cluster);
    if (e != cudaSuccess) return e;
    if (grid_out) *grid_out = grid;
    if (P.part_floats < (long long)(grid / cluster) * B * P.d) return cudaErrorInvalidValue;
    void* args[] = {&P};
    return launch_clustered(kern, grid, cluster, smem, st, args);
}

}  // namespace

int sparse_decode_stages(int d, int B) {
    const int fixed = ring_layout(0, 6 * d, 2 * kConsWarps * B * 4, B * d * 2).total;
    const int stage = round_up(6 * d, 128);
    int R = (kSmemBudget - fixed - 256) / stage;
    if (R > 32) R = 32;
    return R;
}

int decode_max_partial_floats(int d, int B) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return (sms / 2 + 1) * B * d;  // clusters have at least 2 CTAs
}

cudaError_t launch_sparse_decode(SparseDecodeParams P, int B, cudaStream_t st) {
    const bool wide = P.d > 2048;
    switch (B) {
#define SI_CASE(b)                                                         \
    case b:                                                                \
        return wide ? launch_sd<b, 2>(P, st, nullptr) : launch_sd<b, 1>(P, st, nullptr);
        SI_CASE(1)
        SI_CASE(2)
        SI_CASE(3)
        SI_CASE(4)
        SI_CASE(5)
        SI_CASE(6)
        SI_CASE(7)
        SI_CASE(8)
#undef SI_CASE
        default:
            return cudaErrorInvalidValue;
    }
}

// The dense pass hands neuron i to warp i % 8 and stage i % R. R is kept a
// multiple of the consumer-warp count so that every stage belongs to one warp:
// a warp then always consumed the previous fill of a stage before it waits on
// the next one, and a parity wait can never be two phases behind (which would
// read as complete).
int dense_act_stages(int d) {
    const int fixed = ring_layout(0, 4 * d, 0, d * 2).total;
    int R = (kSmemBudget - fixed - 256) / round_up(4 * d, 128);
    if (R > 32) R = 32;
    return (R / kConsWarps) * kConsWarps;
}

cudaError_t launch_dense_act(DenseActParams P, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t smem = (size_t)ring_layout(P.R, 4 * P.d, 0, P.d * 2).total;
    const int grid = P.N < sms ? P.N : sms;
    if (P.d > 2048) {
        if ((e = allow_max_smem(k_dense_act<2>)) != cudaSuccess) return e;
        k_dense_act<2><<<grid, kDecThreads, smem, st>>>(P);
    } else {
        if ((e = allow_max_smem(k_dense_act<1>)) != cudaSuccess) return e;
        k_dense_act<1><<<grid, kDecThreads, smem, st>>>(P);
    }
    return cudaGetLastError();
}

int tiered_down_stages(int d, int aux_floats) {
    const int fixed = ring_layout(0, 2 * d, aux_floats * 4, 0).total;
    int R = (kSmemBudget - fixed - 256) / round_up(2 * d, 128);
    return R > 32 ? 32 : R;
}

cudaError_t launch_tiered_down(TieredDownParams P, cudaStream_t st) {
    const size_t smem = (size_t)ring_layout(P.R, 2 * P.d, P.aux_floats * 4, 0).total;
    int grid = 0, cluster = 0;
    cudaError_t e;
    if (P.d > 2048) {
        e = cached_grid(k_tiered_down<2>, smem, &grid, &cluster);
    } else {
        e = cached_grid(k_tiered_down<1>, smem, &grid, &cluster);
    }
    if (e != cudaSuccess) return e;
    if (P.part_floats < (long long)(grid / cluster) * P.d) return cudaErrorInvalidValue;
    // per-CTA record counts must fit the activation buffer
    const long long per = (long long)(P.k_top + grid - 1) / grid + (P.k_mid + grid - 1) / grid;
    if (per > P.aux_floats) return cudaErrorInvalidValue;
    void* args[] = {&P};
    if (P.d > 2048) return launch_clustered(k_tiered_down<2>, grid, cluster, smem, st, args);
    return launch_clustered(k_tiered_down<1>, grid, cluster, smem, st, args);
}

int streaming_grid_upper_bound() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace si
