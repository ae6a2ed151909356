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
// Producer loop of the ring kernels whose records are picked by an index
// list (idx[0, cnt), each in [0, limit)): the warp loads the indices 32 at a
// time, with the next block's load in flight while this block is issued, and
// lane 0 issues record i into stage i % R once that stage's previous fill has
// been released. An index out of range is flagged and replaced by 0. Called
// by the whole producer warp.
template <class IssueF>
__device__ __forceinline__ void produce_by_index(const int32_t* __restrict__ idx, int cnt, int limit, int R,
                                                 uint64_t* empty, unsigned* err, unsigned site, IssueF issue) {
    const int lane = threadIdx.x & 31;
    int pn = lane < cnt ? __ldcg(idx + lane) : 0;
    for (int base = 0; base < cnt; base += 32) {
        int p = pn;
        pn = base + 32 + lane < cnt ? __ldcg(idx + base + 32 + lane) : 0;
        const bool bad = base + lane < cnt && (p < 0 || p >= limit);
        if (bad) p = 0;
        if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(err, SI_DEVERR_COUNT);
        const int m = cnt - base < 32 ? cnt - base : 32;
        for (int k = 0; k < m; ++k) {
            const int pk = __shfl_sync(0xFFFFFFFFu, p, k);
            if (lane == 0) {
                const int i = base + k, s = i % R;
                if (i >= R) mbar_wait(&empty[s], (uint32_t)((i / R - 1) & 1), err, site);
                issue(i, s, pk);
            }
        }
    }
    __syncwarp();
}

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
            // eight loads in flight, summed in cluster order (deterministic)
            float v = 0.0f;
            unsigned k = 0;
            for (; k + 8 <= ncl; k += 8) {
                float t[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) t[q] = __ldcg(part + (size_t)(k + q) * BD + idx);
#pragma unroll
                for (int q = 0; q < 8; ++q) v += t[q];
            }
            for (; k < ncl; ++k) v += __ldcg(part + (size_t)k * BD + idx);
            y[idx] = v;
        }
        if (threadIdx.x == 0) tickets[r] = 0u;
    }
}

// Cluster arrive / wait halves (all threads of every CTA in the cluster).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Same reduction as cluster_ticket_reduce, in float4 units (BD % (4 * C) == 0):
// cluster peers' partials are summed through distributed shared memory in
// rank order, the cluster partial goes to global memory, and the last cluster
// to finish a slice sums the cluster partials in cluster order. The second
// cluster barrier is split so that the ticket and the final sum overlap the
// peers' reads of this CTA's shared memory; only thread 0 fences.
__device__ void cluster_ticket_reduce4(const float* ypart, int BD, float* __restrict__ part, unsigned* tickets,
                                       float* __restrict__ y) {
    __shared__ unsigned s_last;
    __shared__ float4 s_grp[kDecThreads];
    cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks();
    const int r = (int)cl.block_rank();
    const int ncl = (int)(gridDim.x / C);
    const int cid = (int)(blockIdx.x / C);
    const int Q = BD / (4 * C);  // float4 columns of this CTA's slice
    const int q0 = r * Q;
    float4* part4 = reinterpret_cast<float4*>(part);
    float4* y4 = reinterpret_cast<float4*>(y);
    const int BD4 = BD / 4;
    cluster_arrive();
    cluster_wait();
    for (int q = threadIdx.x; q < Q; q += blockDim.x) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < C; ++c) {
            const float4 t = reinterpret_cast<const float4*>(cl.map_shared_rank(ypart, c))[q0 + q];
            v.x += t.x; v.y += t.y; v.z += t.z; v.w += t.w;
        }
        __stcg(part4 + (size_t)cid * BD4 + q0 + q, v);
    }
    cluster_arrive();  // done reading the peers' shared memory
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned t = atomicAdd(tickets + r, 1u);
        s_last = (t == (unsigned)ncl - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        // Sum of clusters k = g, g + G, g + 2G, ... of column q, eight loads in flight.
        auto sum_clusters = [&](int q, int g, int G) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            int k = g;
            for (; k + 7 * G < ncl; k += 8 * G) {
                float4 t[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) t[u] = __ldcg(part4 + (size_t)(k + u * G) * BD4 + q0 + q);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    v.x += t[u].x; v.y += t[u].y; v.z += t[u].z; v.w += t[u].w;
                }
            }
            for (; k < ncl; k += G) {
                const float4 t = __ldcg(part4 + (size_t)k * BD4 + q0 + q);
                v.x += t.x; v.y += t.y; v.z += t.z; v.w += t.w;
            }
            return v;
        };
        if (Q >= (int)blockDim.x) {
            // at least one column per thread: each thread sums its columns alone
            for (int q = threadIdx.x; q < Q; q += blockDim.x) y4[q0 + q] = sum_clusters(q, 0, 1);
        } else {
            // G groups of Q threads; group sums are added in group order
            const int G = (int)blockDim.x / Q;
            const int q = (int)threadIdx.x % Q, g = (int)threadIdx.x / Q;
            if (g < G) s_grp[g * Q + q] = sum_clusters(q, g, G);
            __syncthreads();
            for (int qq = threadIdx.x; qq < Q; qq += blockDim.x) {
                float4 acc = s_grp[qq];
                for (int gg = 1; gg < G; ++gg) {
                    const float4 t = s_grp[gg * Q + qq];
                    acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
                }
                y4[q0 + qq] = acc;
            }
        }
        if (threadIdx.x == 0) tickets[r] = 0u;
    }
    cluster_wait();  // peers have finished reading this CTA's partial
}

// Grid-wide sum of per-CTA partials without any barrier between CTAs: each
// CTA adds its partial (shared memory, BD floats) into a 64-bit fixed-point
// accumulator (value * 2^32, rounded to nearest) with integer atomics. Integer
// addition is exact and order-independent, so the sum is deterministic; the
// last CTA to take a ticket converts it to float, writes y and re-zeroes the
// accumulator and the ticket for the next launch. A partial of magnitude
// >= 2^23 sets SI_DEVERR_RANGE (the sum of up to 152 such partials would no
// longer be guaranteed to fit).
constexpr double kFixScale = 4294967296.0;          // 2^32
constexpr double kFixInv = 1.0 / 4294967296.0;
constexpr float kFixLimit = 8388608.0f;               // 2^23

__device__ void fixed_point_reduce(const float* ypart, int BD, unsigned long long* __restrict__ acc,
                                   unsigned* ticket, float* __restrict__ y, unsigned* err) {
    __shared__ unsigned s_last;
    bool range_ok = true;
    for (int k = threadIdx.x; k < BD; k += blockDim.x) {
        const float v = ypart[k];
        if (!(fabsf(v) < kFixLimit)) range_ok = false;
        const long long q = __double2ll_rn((double)v * kFixScale);
        atomicAdd(acc + k, (unsigned long long)q);
    }
    if (!range_ok) atomicOr(err, SI_DEVERR_RANGE);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int k = threadIdx.x; k < BD; k += blockDim.x) {
            const long long q = (long long)__ldcg(acc + k);
            y[k] = (float)((double)q * kFixInv);
            __stcg(acc + k, 0ull);
        }
        if (threadIdx.x == 0) *ticket = 0u;
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
    if (R < 1) {  // the host never launches without stages; refuse rather than divide by zero
        if (threadIdx.x == 0) atomicOr(P.err, SI_DEVERR_COUNT);
        return;
    }

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
        const uint64_t pol = policy_evict_first();
        produce_by_index(P.pos + lo, cnt, P.n_records, R, empty, P.err, kSiteDecode | kSiteEmpty,
                         [&](int, int s, int p) {
                             mbar_arrive_expect_tx(&full[s], rec_bytes);
                             bulk_g2s_hint(ring + (size_t)s * L.stage, P.packed + (size_t)p * 3 * d, rec_bytes,
                                           &full[s], pol);
                         });
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
                    // four independent accumulator chains per projection keep the
                    // FMA pipe busy instead of one long dependent chain
                    float ga[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < XJ; ++j) {
                        const int c = lane + 32 * j;
                        if (c < d / 8) {
                            ga[j & 3] = dot8(st[c], xr[j], ga[j & 3]);
                            ua[j & 3] = dot8(st[d / 8 + c], xr[j], ua[j & 3]);
                        }
                    }
                    g[0] = (ga[0] + ga[1]) + (ga[2] + ga[3]);
                    u[0] = (ua[0] + ua[1]) + (ua[2] + ua[3]);
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

// Batch-1 decode with decoupled warps: neuron i belongs to warp i % 8 and ring
// stage i % R (R a multiple of 8, so a warp always consumed the previous fill
// of its own stages). Each warp computes a = silu(g.x) * (u.x) for its neuron
// and accumulates a * down into its own register partial of y; there is no
// CTA-wide barrier in the main loop, so a slow record stalls one warp only.
// x is read straight into registers; the producer starts streaming as soon as
// the barriers exist.
template <int MAXC>
__global__ void __launch_bounds__(kDecThreads, 1) k_sparse_decode_b1(SparseDecodeParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int d = P.d;
    // x stays in registers when it fits (d <= 2048); wider rows read it from shared memory
    constexpr bool kXReg = (MAXC == 1);
    const RingLayout L = ring_layout(P.R, 6 * d, 0, kXReg ? 0 : 2 * d);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    const uint4* s_x = reinterpret_cast<const uint4*>(smem + L.off_x);
    uint8_t* ring = smem + L.off_ring;
    const int R = L.R;
    if (R < 1) {  // the host never launches without stages; refuse rather than divide by zero
        if (threadIdx.x == 0) atomicOr(P.err, SI_DEVERR_COUNT);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a stable plan's count is read before the dependency wait (nothing before
    // this grid writes it); otherwise the count is the host's
    const int n = (P.stable_plan && P.n_dev) ? *P.n_dev : P.n_host;
    const int lo = (int)((long long)n * blockIdx.x / gridDim.x);
    const int hi = (int)((long long)n * (blockIdx.x + 1) / gridDim.x);
    const int cnt = hi - lo;
    const uint32_t rec_bytes = (uint32_t)(6 * d);
    constexpr int XJ = 8 * MAXC;  // 16-byte chunks of a row per lane (c = lane + 32 j)
    const int nch = d / 8;

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // Let the next launch in the stream begin scheduling now: its CTAs take
    // SMs as ours leave, and everything they do before their own dependency
    // wait is an L2 prefetch hint.
    grid_launch_dependents();

    if (warp == kConsWarps) {
        // With a stable plan the records (weights and positions) cannot be
        // written by the grid before this one, so the ring fills while that
        // grid finishes. Otherwise the index list may be that grid's output:
        // only an L2 prefetch hint is issued before the dependency wait.
        if (!P.stable_plan) {
            for (int i = lane; i < cnt && i < R; i += 32) {
                const int p = P.pos[lo + i];
                if (p >= 0 && p < P.n_records) prefetch_l2(P.packed + (size_t)p * 3 * d, rec_bytes);
            }
            grid_dependency_wait();
        }
        const uint64_t pol = policy_evict_first();
        produce_by_index(P.pos + lo, cnt, P.n_records, R, empty, P.err, kSiteDecode | kSiteEmpty,
                         [&](int, int s, int p) {
                             mbar_arrive_expect_tx(&full[s], rec_bytes);
                             bulk_g2s_hint(ring + (size_t)s * L.stage, P.packed + (size_t)p * 3 * d, rec_bytes,
                                           &full[s], pol);
                         });
        if (P.stable_plan) grid_dependency_wait();  // before the tail touches y and the partials
    } else {
        grid_dependency_wait();  // x may be the previous grid's output
        uint4 xr[kXReg ? XJ : 1];
        float acc[XJ][8];
        if constexpr (!kXReg) {
            for (int c = threadIdx.x; c < nch; c += kConsThreads)
                const_cast<uint4*>(s_x)[c] = __ldg(reinterpret_cast<const uint4*>(P.x) + c);
            named_bar_sync(1, kConsThreads);
        }
#pragma unroll
        for (int j = 0; j < XJ; ++j) {
            const int c = lane + 32 * j;
            if constexpr (kXReg)
                xr[j] = (c < nch) ? __ldg(reinterpret_cast<const uint4*>(P.x) + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;
        }
        for (int i = warp; i < cnt; i += kConsWarps) {
            const int s = i % R;
            mbar_wait(&full[s], (uint32_t)((i / R) & 1), P.err, kSiteDecode | kSiteFull);
            const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)s * L.stage);
            float ga[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                const int c = lane + 32 * j;
                if (c < nch) {
                    uint4 xv;
                    if constexpr (kXReg) xv = xr[j];
                    else xv = s_x[c];
                    ga[j & 3] = dot8(st[c], xv, ga[j & 3]);
                    ua[j & 3] = dot8(st[nch + c], xv, ua[j & 3]);
                }
            }
            const float g = warp_sum((ga[0] + ga[1]) + (ga[2] + ga[3]));
            const float u = warp_sum((ua[0] + ua[1]) + (ua[2] + ua[3]));
            const float a = swiglu(g, u);
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                const int c = lane + 32 * j;
                if (c < nch) {
                    float f[8];
                    unpack8(st[2 * nch + c], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(a, f[e], acc[j][e]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // Warp partial -> the warp's own first ring stage (free: the warp has
        // consumed every record of its stages), no barrier needed before it.
        // Layout per warp: for chunk j, the lanes' first halves (4 floats each)
        // then their second halves, so the stores are bank-conflict free.
        float4* wst = reinterpret_cast<float4*>(ring + (size_t)warp * L.stage);
#pragma unroll
        for (int j = 0; j < XJ; ++j) {
            if (32 * j < nch) {  // blocks of 32 chunks that exist (ceil(d / 256) KB per warp)
                wst[j * 64 + lane] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
                wst[j * 64 + 32 + lane] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
            }
        }
        named_bar_sync(1, kConsThreads);
        // float4 k of y = chunk c = k / 2, half k % 2 -> (j, lane) = (c / 32, c % 32)
        constexpr int KV = 2 * MAXC;  // float4 columns per consumer thread
        float4 v[KV];
#pragma unroll
        for (int t = 0; t < KV; ++t) {
            const int k = threadIdx.x + t * kConsThreads;
            v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < d / 4) {
                const int c = k >> 1, off = (c >> 5) * 64 + (k & 1) * 32 + (c & 31);
#pragma unroll
                for (int w = 0; w < kConsWarps; ++w) {
                    const float4 q = reinterpret_cast<const float4*>(ring + (size_t)w * L.stage)[off];
                    v[t].x += q.x; v[t].y += q.y; v[t].z += q.z; v[t].w += q.w;
                }
                // residual form y += FFN(x): vector float atomics, then this thread is done
                if (P.accumulate) atomicAdd(reinterpret_cast<float4*>(P.y) + k, v[t]);
            }
        }
        if (!P.accumulate) {
            named_bar_sync(1, kConsThreads);  // every warp stage has been read
#pragma unroll
            for (int t = 0; t < KV; ++t) {
                const int k = threadIdx.x + t * kConsThreads;
                if (k < d / 4) reinterpret_cast<float4*>(ring)[k] = v[t];
            }
        }
    }
    if (!P.accumulate) {
        __syncthreads();
        fixed_point_reduce(reinterpret_cast<float*>(ring), d, P.acc, P.acc_ticket, P.y, P.err);
    }
}

// ------------------------------------------------------ planned batch-1 decode

// Plan repack: Wp[j][i] = down column of record pos[i], element j, so that a
// CTA that owns output rows reads them contiguously. Pad columns i >= n are
// zero. 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) k_repack_down(const uint16_t* __restrict__ packed, int d,
                                                    const int32_t* __restrict__ pos, int n, int np,
                                                    uint16_t* __restrict__ Wp) {
    __shared__ uint16_t tile[32][34];
    __shared__ int s_p[32];
    const int i0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    if (threadIdx.x < 32) s_p[threadIdx.x] = (i0 + threadIdx.x < n) ? pos[i0 + threadIdx.x] : -1;
    __syncthreads();
    for (int ii = ty; ii < 32; ii += 8) {
        const int p = s_p[ii];
        tile[ii][tx] = (p >= 0 && j0 + tx < d) ? packed[((size_t)p * 3 + 2) * d + j0 + tx] : (uint16_t)0;
    }
    __syncthreads();
    for (int jj = ty; jj < 32; jj += 8)
        if (j0 + jj < d && i0 + tx < np) Wp[(size_t)(j0 + jj) * np + i0 + tx] = tile[tx][jj];
}

// K5a: a[i] = silu(gate[pos[i]] . x) * (up[pos[i]] . x). Warp w owns records
// i = w, w + 8, ... of its CTA's range and ring stages i % R (R a multiple of
// 8); only the gate and up rows (the first 4d bytes of a record) are read.
// With a stable plan the ring fills before the dependency wait; x is read
// after it.
template <int MAXC>
__global__ void __launch_bounds__(kDecThreads, 1) k_plan_act(PlanActParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int d = P.d;
    const RingLayout L = ring_layout(P.R, 4 * d, 0, 0);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    uint8_t* ring = smem + L.off_ring;
    const int R = L.R;
    if (R < 1) {  // the host never launches without stages; refuse rather than divide by zero
        if (threadIdx.x == 0) atomicOr(P.err, SI_DEVERR_COUNT);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lo = (int)((long long)P.n * blockIdx.x / gridDim.x);
    const int hi = (int)((long long)P.n * (blockIdx.x + 1) / gridDim.x);
    const int cnt = hi - lo;
    const uint32_t row2 = (uint32_t)(4 * d);
    constexpr int XJ = 8 * MAXC;
    const int nch = d / 8;

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    grid_launch_dependents();

    if (warp == kConsWarps) {
        if (!P.stable_plan) grid_dependency_wait();
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < cnt; ++i) {
                const int s = i % R;
                if (i >= R) mbar_wait(&empty[s], (uint32_t)((i / R - 1) & 1), P.err, kSiteDecode | kSiteEmpty);
                int p = P.pos[lo + i];
                if (p < 0 || p >= P.n_records) {
                    atomicOr(P.err, SI_DEVERR_COUNT);
                    p = 0;
                }
                mbar_arrive_expect_tx(&full[s], row2);
                bulk_g2s_hint(ring + (size_t)s * L.stage, P.packed + (size_t)p * 3 * d, row2, &full[s], pol);
            }
        }
        __syncwarp();
    } else {
        grid_dependency_wait();  // x may be the previous grid's output; a may still be read by it
        uint4 xr[XJ];
#pragma unroll
        for (int j = 0; j < XJ; ++j) {
            const int c = lane + 32 * j;
            xr[j] = (c < nch) ? __ldg(reinterpret_cast<const uint4*>(P.x) + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        for (int i = warp; i < cnt; i += kConsWarps) {
            const int s = i % R;
            mbar_wait(&full[s], (uint32_t)((i / R) & 1), P.err, kSiteDecode | kSiteFull);
            const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)s * L.stage);
            float ga[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                const int c = lane + 32 * j;
                if (c < nch) {
                    ga[j & 3] = dot8(st[c], xr[j], ga[j & 3]);
                    ua[j & 3] = dot8(st[nch + c], xr[j], ua[j & 3]);
                }
            }
            const float g = warp_sum((ga[0] + ga[1]) + (ga[2] + ga[3]));
            const float u = warp_sum((ua[0] + ua[1]) + (ua[2] + ua[3]));
            __syncwarp();
            if (lane == 0) {
                P.a[lo + i] = swiglu(g, u);
                mbar_arrive(&empty[s]);
            }
        }
    }
}

// K5b: y[j] = sum_i a[i] * Wp[j][i] for the CTA's rows. The rows (plan data)
// stream into shared memory before the dependency wait when the plan is
// stable; a is read after it. Warp w handles rows w, w + 8, ...; lanes stride
// over 8-column chunks with four accumulators, summed in a fixed order.
__global__ void __launch_bounds__(256, 2) k_plan_down(PlanDownParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    float* s_a = reinterpret_cast<float*>(smem + 128);
    uint16_t* s_w = reinterpret_cast<uint16_t*>(smem + 128 + round_up(P.np * 4, 128));
    const int r0 = blockIdx.x * P.rows;
    const int nr = min(P.rows, P.d - r0);
    const uint32_t row_bytes = (uint32_t)(P.np * 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    grid_launch_dependents();
    if (!P.stable_plan) grid_dependency_wait();
    if (threadIdx.x == 0 && nr > 0) {
        mbar_arrive_expect_tx(bar, row_bytes * (uint32_t)nr);
        const uint64_t pol = policy_evict_first();
        for (int r = 0; r < nr; ++r)
            bulk_g2s_hint(s_w + (size_t)r * P.np, P.Wp + (size_t)(r0 + r) * P.np, row_bytes, bar, pol);
    }
    grid_dependency_wait();  // a is the previous grid's output
    for (int k = threadIdx.x; k < P.np / 4; k += blockDim.x)
        reinterpret_cast<float4*>(s_a)[k] = __ldcg(reinterpret_cast<const float4*>(P.a) + k);
    __syncthreads();
    if (nr > 0) mbar_wait(bar, 0u, P.err, kSiteDecode | kSiteFullB);
    const int nch = P.np / 8;
    for (int r = warp; r < nr; r += 8) {
        const uint4* w = reinterpret_cast<const uint4*>(s_w + (size_t)r * P.np);
        const float4* av = reinterpret_cast<const float4*>(s_a);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        int q = 0;
        for (int c = lane; c < nch; c += 32, ++q) {
            float f[8];
            unpack8(w[c], f);
            const float4 a0 = av[2 * c], a1 = av[2 * c + 1];
            float t = acc[q & 3];
            t = fmaf(f[0], a0.x, t);
            t = fmaf(f[1], a0.y, t);
            t = fmaf(f[2], a0.z, t);
            t = fmaf(f[3], a0.w, t);
            t = fmaf(f[4], a1.x, t);
            t = fmaf(f[5], a1.y, t);
            t = fmaf(f[6], a1.z, t);
            t = fmaf(f[7], a1.w, t);
            acc[q & 3] = t;
        }
        const float v = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
        if (lane == 0) P.y[r0 + r] = P.accumulate ? P.y[r0 + r] + v : v;
    }
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
    if (R < 1) {  // the host never launches without stages; refuse rather than divide by zero
        if (threadIdx.x == 0) atomicOr(P.err, SI_DEVERR_COUNT);
        return;
    }
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
    grid_launch_dependents();
    // The weights belong to the caller and may be the previous grid's output,
    // so before the dependency wait they are only prefetched into L2; x and a
    // are touched after it.
    if (warp == kConsWarps)
        for (int i = lane; i < cnt && i < R; i += 32) {
            prefetch_l2(P.Wg + (size_t)(lo + i) * d, row_bytes);
            prefetch_l2(P.Wu + (size_t)(lo + i) * d, row_bytes);
        }
    grid_dependency_wait();
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
            float ga[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                const int c = lane + 32 * j;
                if (c < d / 8) {
                    ga[j & 3] = dot8(st[c], xr[j], ga[j & 3]);
                    ua[j & 3] = dot8(st[d / 8 + c], xr[j], ua[j & 3]);
                }
            }
            const float g = warp_sum((ga[0] + ga[1]) + (ga[2] + ga[3]));
            const float u = warp_sum((ua[0] + ua[1]) + (ua[2] + ua[3]));
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
    if (R < 1) {  // the host never launches without stages; refuse rather than divide by zero
        if (threadIdx.x == 0) atomicOr(P.err, SI_DEVERR_COUNT);
        return;
    }
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
    // the tier lists and a are the previous grids' output
    grid_launch_dependents();
    grid_dependency_wait();
    int* s_col = reinterpret_cast<int*>(s_av + P.aux_floats / 2);
    for (int i = threadIdx.x; i < nrec; i += blockDim.x) {
        const int col = i < ntop ? P.top[t0 + i] : P.mid[m0 + i - ntop];
        const bool ok = col >= 0 && col < P.N;
        s_col[i] = ok ? col : -1;
        s_av[i] = ok ? P.a[col] : 0.0f;
    }
    __syncthreads();

    if (warp == kConsWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < nrec; ++i) {
                const int s = i % R;
                if (i >= R) mbar_wait(&empty[s], (uint32_t)((i / R - 1) & 1), P.err, kSiteTiered | kSiteEmpty);
                uint8_t* dst = ring + (size_t)s * L.stage;
                int ci = s_col[i];
                if (ci < 0) {  // never read outside the encoded buffers
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
    cluster_ticket_reduce4(reinterpret_cast<float*>(ring), d, P.part, P.tickets, P.y);
}

// ------------------------------------------------------------------ launch

namespace {

constexpr int kSmemBudget = 227 * 1024 - 2048;  // dynamic budget, leaves room for static smem

// Clustered launch; with `pdl` the launch may overlap the previous grid in
// the stream (programmatic stream serialization: the kernel itself waits with
// griddepcontrol.wait before it reads anything that grid may write).
template <class K>
cudaError_t launch_clustered(K kernel, int grid, int cluster, size_t smem, cudaStream_t st, void** args,
                             bool pdl = false) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
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
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) (void)cudaGetLastError();
    int ctas_of[17] = {0};
    for (int C = 16; C >= 2; C /= 2) {
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
        ctas_of[C] = ncl * C < (sms / C) * C ? ncl * C : (sms / C) * C;
    }
    // Larger clusters leave fewer partials for the cross-cluster sum (its
    // cost grows with the partial count), so take the largest cluster that
    // still keeps most SMs streaming; otherwise the one with the most CTAs.
    int bestC = 0;
    for (int C = 16; C >= 2 && !bestC; C /= 2)
        if (ctas_of[C] * 100 >= sms * 84) bestC = C;
    if (!bestC)
        for (int C = 2; C <= 16; C *= 2)
            if (!bestC || ctas_of[C] > ctas_of[bestC]) bestC = C;
    if (ctas_of[bestC] <= 0) return cudaErrorInvalidConfiguration;
    *grid = ctas_of[bestC];
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

// One CTA per SM minus a few: with programmatic dependent launch the next
// launch's CTAs take SMs as this launch's CTAs leave, and the spare SMs keep
// the last CTA's tail from delaying the next launch's start.
constexpr int kSpareSms = 4;

template <int MAXC>
cudaError_t launch_sd1(SparseDecodeParams& P, cudaStream_t st) {
    auto kern = k_sparse_decode_b1<MAXC>;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = allow_max_smem(kern)) != cudaSuccess) return e;
    const size_t smem = (size_t)ring_layout(P.R, 6 * P.d, 0, MAXC == 1 ? 0 : 2 * P.d).total;
    void* args[] = {&P};
    return launch_clustered(kern, sms > 2 * kSpareSms ? sms - kSpareSms : sms, 1, smem, st, args, /*pdl=*/true);
}

}  // namespace

cudaError_t launch_repack_down(const uint16_t* packed, int d, const int32_t* pos, int n, int np, uint16_t* Wp,
                               cudaStream_t st) {
    dim3 grid((np + 31) / 32, (d + 31) / 32);
    k_repack_down<<<grid, 256, 0, st>>>(packed, d, pos, n, np, Wp);
    return cudaGetLastError();
}

// Small rings so that the down kernel's CTAs fit beside this kernel's on an SM.
int plan_act_stages(int d) {
    const int stage = round_up(4 * d, 128);
    int R = (80 * 1024) / stage;
    R = (R / kConsWarps) * kConsWarps;
    return R < kConsWarps ? kConsWarps : R;
}

cudaError_t launch_plan_act(PlanActParams P, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const size_t smem = (size_t)ring_layout(P.R, 4 * P.d, 0, 0).total;
    const int grid = P.n < sms ? (P.n > 0 ? P.n : 1) : sms;
    void* args[] = {&P};
    if (P.d > 2048) {
        if ((e = allow_max_smem(k_plan_act<2>)) != cudaSuccess) return e;
        return launch_clustered(k_plan_act<2>, grid, 1, smem, st, args, true);
    }
    if ((e = allow_max_smem(k_plan_act<1>)) != cudaSuccess) return e;
    return launch_clustered(k_plan_act<1>, grid, 1, smem, st, args, true);
}

int plan_down_rows(int d, int np) {
    // rows per CTA: enough CTAs to cover the SMs about twice, rows buffer <= 96 KB
    int rows = 8;
    while (rows > 1 && (size_t)rows * np * 2 > 96 * 1024) rows /= 2;
    (void)d;
    return rows;
}

cudaError_t launch_plan_down(PlanDownParams P, cudaStream_t st) {
    cudaError_t e = allow_max_smem(k_plan_down);
    if (e != cudaSuccess) return e;
    const size_t smem = 128 + (size_t)round_up(P.np * 4, 128) + (size_t)P.rows * P.np * 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((P.d + P.rows - 1) / P.rows, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&P};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(k_plan_down), args);
}

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

int sparse_decode_b1_stages(int d) {
    const int stage = round_up(6 * d, 128);
    int R = (kSmemBudget - 512 - (d > 2048 ? round_up(2 * d, 128) : 0)) / stage;
    if (R > 32) R = 32;
    R = (R / kConsWarps) * kConsWarps;
    // warp w's partial (blocks of 32 chunks: round_up(d, 256) floats) reuses
    // its stage w, then the CTA partial stage 0
    return (R >= kConsWarps && stage >= round_up(d, 256) * 4) ? R : 0;
}

cudaError_t launch_sparse_decode(SparseDecodeParams P, int B, cudaStream_t st) {
    const bool wide = P.d > 2048;
    if (B == 1 && P.pmask == nullptr && (P.n_dev == nullptr || P.stable_plan)) {
        const int R1 = sparse_decode_b1_stages(P.d);
        if (R1 >= kConsWarps) {
            SparseDecodeParams P1 = P;
            P1.R = R1;
            return wide ? launch_sd1<2>(P1, st) : launch_sd1<1>(P1, st);
        }
    }
    if (P.R < 1) return cudaErrorInvalidValue;
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
    void* args[] = {&P};
    if (P.d > 2048) {
        if ((e = allow_max_smem(k_dense_act<2>)) != cudaSuccess) return e;
        return launch_clustered(k_dense_act<2>, grid, 1, smem, st, args, /*pdl=*/true);
    }
    if ((e = allow_max_smem(k_dense_act<1>)) != cudaSuccess) return e;
    return launch_clustered(k_dense_act<1>, grid, 1, smem, st, args, /*pdl=*/true);
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
    // (activations in the first half of the buffer, columns in the second)
    const long long per = (long long)(P.k_top + grid - 1) / grid + (P.k_mid + grid - 1) / grid;
    if (2 * per > P.aux_floats) return cudaErrorInvalidValue;
    void* args[] = {&P};
    if (P.d > 2048) return launch_clustered(k_tiered_down<2>, grid, cluster, smem, st, args, /*pdl=*/true);
    return launch_clustered(k_tiered_down<1>, grid, cluster, smem, st, args, /*pdl=*/true);
}

int streaming_grid_upper_bound() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace si
