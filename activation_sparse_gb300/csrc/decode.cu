// decode.cu -- HBM-streaming decode kernels (one token per sequence).
//
//  k_sparse_decode_b1  SelectInfer sparse decode FFN for one sequence
//                      (section 5: only the selected neurons are computed):
//                      for each selected packed record [gate row | up row |
//                      down column] it forms a = silu(g.x) * (u.x) and adds
//                      a * down into a per-warp partial of y.
//  k_sparse_decode     the same for B <= 8 sequences over the union of their
//                      selections (each record carries a mask of the
//                      sequences that selected it).
//  k_dense_act         SpAx dense gate/up pass: a[n] for every neuron.
//  k_tiered_down       SpAx three-tier down-projection (abstract, Fig. 2/3):
//                      top columns in bf16, middle columns rebuilt from 2-, 3-,
//                      4- or 8-bit codes (min + q * scale), the rest never read.
//
// Common structure (warp-specialised, one CTA per SM):
//   * the producer warp streams whole records into a ring of shared-memory
//     stages with 1-D bulk copies (cp.async.bulk, completion counted in bytes
//     on a per-stage "full" mbarrier); consumers release a stage through its
//     "empty" mbarrier. Every wait is bounded.
//   * records are split evenly over the CTAs of the grid (split-K over
//     neurons / columns); partial sums of y stay in registers.
//   * cross-CTA sum of y: 64-bit fixed-point atomics with a ticketed final
//     conversion (batch-1 overwrite; deterministic), float atomics into y
//     (batch-1 residual form), or cluster reduction through distributed
//     shared memory plus a ticketed fixed-order final pass over float4
//     columns (batch B and tiered down; deterministic).
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "ring.cuh"

namespace cg = cooperative_groups;

namespace si {

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
        // the peers' values in rank order, up to eight loads in flight before
        // the adds (the rank order of the sum is kept)
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < C; c += 8) {
            float4 t[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + u < C) t[u] = reinterpret_cast<const float4*>(cl.map_shared_rank(ypart, c + u))[q0 + q];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + u < C) {
                    v.x += t[u].x; v.y += t[u].y; v.z += t[u].z; v.w += t[u].w;
                }
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
        // Sum of clusters k = g, g + G, g + 2G, ... of column q, sixteen (then
        // eight) loads in flight.
        auto sum_clusters = [&](int q, int g, int G) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            int k = g;
            for (; k + 15 * G < ncl; k += 16 * G) {
                float4 t[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) t[u] = __ldcg(part4 + (size_t)(k + u * G) * BD4 + q0 + q);
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    v.x += t[u].x; v.y += t[u].y; v.z += t[u].z; v.w += t[u].w;
                }
            }
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

// With err_report set, *err is a word that only this launch writes into (its
// bounded waits stop early once it holds a timeout): the last CTA, which runs
// after every other CTA has recorded its failures, moves its bits into
// *err_report and clears it, so a failure never cuts short a later launch's waits.
__device__ void fixed_point_reduce(const float* ypart, int BD, unsigned long long* __restrict__ acc,
                                   unsigned* ticket, float* __restrict__ y, unsigned* err,
                                   unsigned* err_report = nullptr) {
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
        if (threadIdx.x == 0) {
            *ticket = 0u;
            if (err_report) {
                const unsigned v = atomicExch(err, 0u);
                if (v) atomicOr(err_report, v);
            }
        }
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
    // float4 columns, each summed over the clusters by one thread of the last
    // cluster (fixed cluster order: deterministic)
    cluster_ticket_reduce4(reinterpret_cast<float*>(ring), B * d, P.part, P.tickets, P.y);
}

// ------------------------------------------------ batch decode on tensor cores

// Warp-level bf16 tensor-core pieces: ldmatrix of 8x8 b16 tiles from any
// 16-byte-aligned row addresses (one per lane 0-15), and the m16n8k16 MMA
// with fp32 accumulation.
__device__ __forceinline__ void ldsm_x2(const void* row, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(smem_u32(row)));
}
__device__ __forceinline__ void ldsm_x4(const void* row, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(row)));
}
__device__ __forceinline__ void ldsm_x2_trans(const void* row, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(smem_u32(row)));
}
// d += A (16 x 16, rows a0..a3 as the fragment) * B (16 x 8), A's rows 8-15
// and k 8-15 given as registers (zero where absent)
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    // a register-only operation: not volatile, so independent MMAs can be
    // interleaved by the compiler
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Shared-memory layout of the tensor-core batch decode: full / empty
// barriers, the cross-warp sums of the gate and up products, a, then the
// stages. A stage is one packed record (gate row, up row, down column) plus
// 16 bytes, so that the same 16-byte row of eight consecutive records falls
// in eight different bank groups (conflict-free ldmatrix).
constexpr int kMmaBatch = 8;  // records per batch: a batch's stages are held until its down products are done
struct MmaLayout {
    int off_full, off_empty, off_red, off_a, off_ring, stage, R, total;
};
__host__ __device__ inline MmaLayout mma_layout(int R, int d) {
    MmaLayout L;
    L.R = R;
    L.stage = round_up(6 * d, 128) + 16;
    L.off_full = 0;
    L.off_empty = 8 * R;
    L.off_red = round_up(16 * R, 128);
    L.off_a = L.off_red + kConsWarps * 128 * 4;
    L.off_ring = L.off_a + round_up(8 * 8 * 4, 128);
    L.total = L.off_ring + R * L.stage;
    return L;
}

// Grid-wide sum of the CTAs' partials for a cooperative launch (every CTA
// resident): each CTA stores its partial (BD floats in shared memory) to
// part[blockIdx], arrives on ctr[0] and waits (bounded) until all G CTAs
// have arrived; then it sums its slice of the BD floats over the G partials
// in a fixed order (groups of threads take every ng-th partial, the group
// sums are added in group order) and writes y. The last CTA to leave resets
// ctr[0] and ctr[1] for the next launch. BD % 4 == 0. With `trigger` the
// grid lets its dependents launch once all its CTAs have arrived.
__device__ void grid_slice_reduce4(const float* ypart, int BD, float* __restrict__ part, unsigned* ctr,
                                   float* __restrict__ y, unsigned* err, unsigned site, bool trigger = false) {
    __shared__ float4 s_grp[kDecThreads];
    __shared__ unsigned s_last;
    const int G = (int)gridDim.x, BD4 = BD / 4;
    float4* part4 = reinterpret_cast<float4*>(part);
    const float4* yp4 = reinterpret_cast<const float4*>(ypart);
    for (int k = threadIdx.x; k < BD4; k += blockDim.x) __stcg(part4 + (size_t)blockIdx.x * BD4 + k, yp4[k]);
    __syncthreads();
    if (threadIdx.x == 0) {
        // release: the partial (ordered before this thread by the CTA barrier)
        // is visible before the arrival; acquire: the others' partials after it
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
        const long long t0 = cycles();
        for (uint32_t it = 1;; ++it) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
            if (v >= (unsigned)G) break;
            if ((it & 255u) == 0) {
                if (*reinterpret_cast<volatile unsigned*>(err) & SI_DEVERR_WAIT_TIMEOUT) break;
                if (cycles() - t0 > kWaitLimitCycles) {
                    atomicOr(err, SI_DEVERR_WAIT_TIMEOUT | site);
                    break;
                }
            }
        }
    }
    __syncthreads();
    // every CTA of the grid is resident now: the next grid in the stream may
    // begin (it cannot take an SM this grid still needs)
    if (trigger) grid_launch_dependents();
    const int q0 = (int)((long long)BD4 * blockIdx.x / G), q1 = (int)((long long)BD4 * (blockIdx.x + 1) / G);
    const int nq = q1 - q0;
    auto sum_parts = [&](int q, int first, int step) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        int k = first;
        for (; k + 7 * step < G; k += 8 * step) {
            float4 t[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) t[u] = __ldcg(part4 + (size_t)(k + u * step) * BD4 + q);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                v.x += t[u].x; v.y += t[u].y; v.z += t[u].z; v.w += t[u].w;
            }
        }
        for (; k < G; k += step) {
            const float4 t = __ldcg(part4 + (size_t)k * BD4 + q);
            v.x += t.x; v.y += t.y; v.z += t.z; v.w += t.w;
        }
        return v;
    };
    float4* y4 = reinterpret_cast<float4*>(y);
    if (nq > 0 && nq <= (int)blockDim.x) {
        const int ng = (int)blockDim.x / nq;
        const int q = (int)threadIdx.x % nq, grp = (int)threadIdx.x / nq;
        if (grp < ng) s_grp[grp * nq + q] = sum_parts(q0 + q, grp, ng);
        __syncthreads();
        if ((int)threadIdx.x < nq) {
            float4 acc = s_grp[threadIdx.x];
            for (int gg = 1; gg < ng; ++gg) {
                const float4 t = s_grp[gg * nq + threadIdx.x];
                acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
            }
            y4[q0 + threadIdx.x] = acc;
        }
    } else {
        for (int q = q0 + (int)threadIdx.x; q < q1; q += blockDim.x) y4[q] = sum_parts(q, 0, 1);
    }
    __syncthreads();  // every read of the partials is done before leaving
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(ctr + 1, 1u) == (unsigned)G - 1) ? 1u : 0u;
        if (s_last) {
            ctr[0] = 0u;
            ctr[1] = 0u;
        }
    }
}

// Batch-B decode (B <= 8 sequences over the union plan) on the tensor cores.
// The CTA takes its records in batches of eight. Gate and up products in one
// MMA per k-step: A's rows 0-7 are the batch's gate rows and rows 8-15 their
// up rows, times x^T (N = the 8 sequences); K is split over the eight
// consumer warps (warp w takes k in [w d / 8, (w + 1) d / 8), its x
// fragments held in registers for the whole launch), and the warps' partial
// sums meet in shared memory, added in warp order. a = silu(g) u where the
// sequence selected the record, else 0. Down: warp w takes rows
// [w d / 8, (w + 1) d / 8); the batch's down columns (ldmatrix.trans) enter
// K twice, against a's leading bf16 term in k 0-7 and its remainder in
// k 8-15, so one MMA per tile applies a to within 2^-18 |a| (fp32-level
// products). The launch is cooperative (one CTA per SM,
// all resident) and the CTA sums meet in a grid-wide slice reduction in a
// fixed order (deterministic).
// DT = d / 128: k-steps of 16 per warp slice and m-tiles of 16 rows per warp.
template <int DT>
__global__ void __launch_bounds__(kDecThreads, 1) k_sparse_decode_mma(SparseDecodeParams P, int B) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int d = 128 * DT;
    const MmaLayout L = mma_layout(P.R, d);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    float* s_red = reinterpret_cast<float*>(smem + L.off_red);  // [warp][gate 64 | up 64]
    float* s_av = reinterpret_cast<float*>(smem + L.off_a);     // [record][sequence]
    uint8_t* ring = smem + L.off_ring;
    const int R = L.R;
    // the host never launches fewer stages than a batch, another d or B > 8
    if (R < kMmaBatch || P.d != d || B < 1 || B > 8) {
        if (threadIdx.x == 0) atomicOr(P.err, SI_DEVERR_COUNT);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // A stable plan (its records, masks and count) cannot be written by the
    // grid before this one, so the ring fills while that grid finishes; x,
    // y, the partials and the counters are touched only after the
    // dependency wait. A fresh plan may be that grid's output: wait first.
    if (!P.stable_plan) grid_dependency_wait();
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
        if (P.stable_plan) grid_dependency_wait();  // x may be the previous grid's output
        const int g = lane >> 2, t = lane & 3;  // fragment row / column group
        // x^T fragments of this warp's k-slice: b0b1 = x[g][k0 + 2t ..], b2b3 = x[g][k0 + 8 + 2t ..]
        uint32_t xb[DT][2];
        {
            const uint32_t* xg = reinterpret_cast<const uint32_t*>(P.x + (size_t)(g < B ? g : 0) * d);
#pragma unroll
            for (int ks = 0; ks < DT; ++ks) {
                const int k0 = warp * (d / 8) + 16 * ks;
                xb[ks][0] = g < B ? __ldg(xg + (k0 + 2 * t) / 2) : 0u;
                xb[ks][1] = g < B ? __ldg(xg + (k0 + 8 + 2 * t) / 2) : 0u;
            }
        }
        float acc[DT][4];
#pragma unroll
        for (int mt = 0; mt < DT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
        const int nbat = (cnt + kMmaBatch - 1) / kMmaBatch;
        for (int bt = 0; bt < nbat; ++bt) {
            const int i0 = bt * kMmaBatch;
            const int nb = min(kMmaBatch, cnt - i0);
            // the sequence mask of this thread's record, read ahead of the products
            const int rm = threadIdx.x >> 3;
            const uint32_t pm = (threadIdx.x < 64 && rm < nb && P.pmask) ? __ldg(P.pmask + lo + i0 + rm) : 0xFFFFFFFFu;
            for (int r = 0; r < nb; ++r) {
                const int i = i0 + r;
                mbar_wait(&full[i % R], (uint32_t)((i / R) & 1), P.err, kSiteDecode | kSiteFull);
            }
            // lanes 0-15 address record (lane & 7) (record 0 where the batch is short)
            const int rr = (lane & 7) < nb ? (lane & 7) : 0;
            const uint8_t* rec = ring + (size_t)((i0 + rr) % R) * L.stage;
            const int half8 = (lane >> 3) & 1;  // second 8x8 tile of the pair
            // gate (rows g) and up (rows g + 8): D[record][sequence] over this
            // warp's k-slice. ldmatrix.x4 tiles: lanes 0-7 gate rows at k0,
            // 8-15 up rows at k0, 16-23 gate rows at k0 + 8, 24-31 up rows at
            // k0 + 8. Two accumulator chains (even and odd k-steps), so that
            // consecutive MMAs do not wait on each other.
            const uint8_t* gu = ring + (size_t)((i0 + ((lane & 7) < nb ? (lane & 7) : 0)) % R) * L.stage +
                                (size_t)(((lane >> 3) & 1) * 2 * d) + (size_t)(((lane >> 4) & 1) * 8) * 2;
            float cgu[2][4] = {};
#pragma unroll
            for (int ks = 0; ks < DT; ++ks) {
                const int k0 = warp * (d / 8) + 16 * ks;
                uint32_t a0, a1, a2, a3;
                ldsm_x4(gu + (size_t)k0 * 2, a0, a1, a2, a3);
                mma_bf16(cgu[ks & 1], a0, a1, a2, a3, xb[ks][0], xb[ks][1]);
            }
            float cg[1][2] = {{cgu[0][0] + cgu[1][0], cgu[0][1] + cgu[1][1]}};
            float cu[1][2] = {{cgu[0][2] + cgu[1][2], cgu[0][3] + cgu[1][3]}};
            // rows g (the records) of the fragments: sequences 2t, 2t + 1
            *reinterpret_cast<float2*>(s_red + warp * 128 + g * 8 + 2 * t) = make_float2(cg[0][0], cg[0][1]);
            *reinterpret_cast<float2*>(s_red + warp * 128 + 64 + g * 8 + 2 * t) = make_float2(cu[0][0], cu[0][1]);
            named_bar_sync(1, kConsThreads);
            if (threadIdx.x < 64) {
                const int r = threadIdx.x >> 3, b = threadIdx.x & 7;
                float gs = 0.0f, us = 0.0f;
#pragma unroll
                for (int w = 0; w < kConsWarps; ++w) {
                    gs += s_red[w * 128 + threadIdx.x];
                    us += s_red[w * 128 + 64 + threadIdx.x];
                }
                s_av[r * 8 + b] = (r < nb && b < B && ((pm >> b) & 1u)) ? swiglu(gs, us) : 0.0f;
            }
            named_bar_sync(1, kConsThreads);
            // a as B fragments: k = 2t, 2t + 1 (records) -> (a[2t][g], a[2t + 1][g]),
            // its leading bf16 term for k < 8 and the bf16 of the remainder for k >= 8
            uint32_t bh, bl;
            {
                const float a0 = s_av[(2 * t) * 8 + g], a1 = s_av[(2 * t + 1) * 8 + g];
                const float h0 = __bfloat162float(__float2bfloat16_rn(a0)), h1 = __bfloat162float(__float2bfloat16_rn(a1));
                bh = pack_bf16(h0, h1);
                bl = pack_bf16(a0 - h0, a1 - h1);
            }
            // down: Y[row][sequence] += Dn[row][record] a[record][sequence] over this warp's rows
            const uint8_t* dn = rec + (size_t)4 * d + (size_t)(8 * half8) * 2;
            // (the records' columns enter K twice: k 0-7 and k 8-15 both hold
            // records 0-7, against a's two terms)
#pragma unroll
            for (int mt = 0; mt < DT; ++mt) {
                uint32_t a0, a1;
                ldsm_x2_trans(dn + (size_t)(warp * (d / 8) + 16 * mt) * 2, a0, a1);
                mma_bf16(acc[mt], a0, a1, a0, a1, bh, bl);
            }
            __syncwarp();
            if (lane == 0)
                for (int r = 0; r < nb; ++r) mbar_arrive(&empty[(i0 + r) % R]);
        }
        named_bar_sync(1, kConsThreads);  // every consumer is done with the ring
        float* ypart = reinterpret_cast<float*>(ring);
#pragma unroll
        for (int mt = 0; mt < DT; ++mt) {
            const int m0 = warp * (d / 8) + 16 * mt;
            if (2 * t < B) {
                ypart[(size_t)(2 * t) * d + m0 + g] = acc[mt][0];
                ypart[(size_t)(2 * t) * d + m0 + 8 + g] = acc[mt][2];
            }
            if (2 * t + 1 < B) {
                ypart[(size_t)(2 * t + 1) * d + m0 + g] = acc[mt][1];
                ypart[(size_t)(2 * t + 1) * d + m0 + 8 + g] = acc[mt][3];
            }
        }
    }
    __syncthreads();  // (the consumers' dependency wait orders every write below after the previous grid)
    grid_slice_reduce4(reinterpret_cast<float*>(ring), B * d, P.part, P.tickets, P.y, P.err, kSiteDecode | kSiteAccum,
                       /*trigger=*/true);
}

// The overwrite form (y = FFN(x)) sums the CTAs' partials either through
// the cluster and a fixed-order final pass (CR: clustered launches with a
// partial buffer) or with the 64-bit fixed-point accumulator (no partial
// buffer: the allocation-free entry point); both are deterministic. The
// residual form (y += FFN(x)) adds each CTA's sum with vector atomics.
// Batch-1 decode with decoupled warps: neuron i belongs to warp i % 8 and ring
// stage i % R. Each warp computes a = silu(g.x) * (u.x) for its neuron and
// accumulates a * down into its own register partial of y; there is no
// CTA-wide barrier in the main loop, so a slow record stalls one warp only.
// x is staged once per CTA in shared memory after the dependency wait; the
// producer starts streaming as soon as the barriers exist.
// R need not be a multiple of 8, so consecutive fills of a stage belong to
// different warps and a parity wait alone could be answered by a fill two
// phases old: the producer writes the record number into the stage's slot
// before issuing its copy (only possible once the previous fill was released)
// and a consumer waits for its number to appear before the parity wait.
constexpr int kB1MaxStages = 32;  // stages of the batch-1 ring (their record numbers sit in the aux area)

template <int MAXC, bool CR>
__global__ void __launch_bounds__(kDecThreads, 1) k_sparse_decode_b1(SparseDecodeParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int d = P.d;
    // x is staged once per CTA in shared memory (one L2 read of x per CTA
    // rather than one per warp)
    const RingLayout L = ring_layout(P.R, 6 * d, 4 * kB1MaxStages, 2 * d);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    int* seq = reinterpret_cast<int*>(smem + L.off_aux);  // record number of each stage's latest fill
    const uint4* s_x = reinterpret_cast<const uint4*>(smem + L.off_x);
    uint8_t* ring = smem + L.off_ring;
    const int R = L.R;
    // the host never launches a ring shorter than the eight warp partials need
    if (R < kConsWarps || R > kB1MaxStages) {
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

    for (int s = threadIdx.x; s < R; s += blockDim.x) seq[s] = -1;
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
                         [&](int i, int s, int p) {
                             *reinterpret_cast<volatile int*>(seq + s) = i;
                             mbar_arrive_expect_tx(&full[s], rec_bytes);
                             bulk_g2s_hint(ring + (size_t)s * L.stage, P.packed + (size_t)p * 3 * d, rec_bytes,
                                           &full[s], pol);
                         });
        if (P.stable_plan) grid_dependency_wait();  // before the tail touches y and the partials
    } else {
        grid_dependency_wait();  // x may be the previous grid's output
        float acc[XJ][8];
        for (int c = threadIdx.x; c < nch; c += kConsThreads)
            const_cast<uint4*>(s_x)[c] = __ldg(reinterpret_cast<const uint4*>(P.x) + c);
        named_bar_sync(1, kConsThreads);
#pragma unroll
        for (int j = 0; j < XJ; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;
        for (int i = warp; i < cnt; i += kConsWarps) {
            const int s = i % R;
            if (*reinterpret_cast<volatile int*>(seq + s) != i) {
                const long long t0 = cycles();
                while (*reinterpret_cast<volatile int*>(seq + s) != i) {
                    if (cycles() - t0 > kWaitLimitCycles) {
                        if (lane == 0) atomicOr(P.err, SI_DEVERR_WAIT_TIMEOUT | kSiteDecode | kSiteFull);
                        break;
                    }
                }
            }
            mbar_wait(&full[s], (uint32_t)((i / R) & 1), P.err, kSiteDecode | kSiteFull);
            const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)s * L.stage);
            float ga[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < XJ; ++j) {
                const int c = lane + 32 * j;
                if (c < nch) {
                    const uint4 xv = s_x[c];
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
        // Warp partial -> ring stage `warp`, once every warp has consumed all
        // of its records (the producer has issued its last record by then, so
        // no stage is refilled). Layout per warp: for chunk j, the lanes'
        // first halves (4 floats each) then their second halves, so the
        // stores are bank-conflict free.
        named_bar_sync(1, kConsThreads);
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
        if constexpr (CR)
            cluster_ticket_reduce4(reinterpret_cast<float*>(ring), d, P.part, P.tickets, P.y);
        else
            fixed_point_reduce(reinterpret_cast<float*>(ring), d, P.acc, P.acc_ticket, P.y, P.err, P.err_report);
    }
}

// ------------------------------------------------------ planned batch-1 decode


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
    // the rows this CTA computes: an even share of all N neurons, or of the
    // n_rows listed ones (their indices in P.rows)
    const int total = P.rows ? P.n_rows : P.N;
    const int lo = (int)((long long)total * blockIdx.x / gridDim.x);
    const int hi = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
    const int cnt = hi - lo;
    const uint32_t row_bytes = (uint32_t)(2 * d);
    // neuron of the CTA's i-th row; a listed index outside [0, N) is flagged
    // and read as neuron 0 (never outside the weights)
    auto row = [&](int i) -> int {
        if (!P.rows) return lo + i;
        const int n = P.rows[lo + i];
        return (n >= 0 && n < P.N) ? n : 0;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    grid_launch_dependents();
    // The weights belong to the caller and may be the previous grid's output,
    // so before the dependency wait they are only prefetched into L2; x, a and
    // a row list (which may be that grid's output too) are touched after it.
    if (warp == kConsWarps && !P.rows)
        for (int i = lane; i < cnt && i < R; i += 32) {
            prefetch_l2(P.Wg + (size_t)row(i) * d, row_bytes);
            prefetch_l2(P.Wu + (size_t)row(i) * d, row_bytes);
        }
    grid_dependency_wait();
    // with a row list, every unlisted neuron has a = 0 (the caller zeroes a):
    // its key falls in bin 0 of the tier histogram
    if (P.rows && P.hist && blockIdx.x == 0 && threadIdx.x == 0 && P.N > P.n_rows)
        atomicAdd(P.hist, (unsigned)(P.N - P.n_rows));
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x)
        reinterpret_cast<uint4*>(s_x)[i] = reinterpret_cast<const uint4*>(P.x)[i];
    __syncthreads();

    if (warp == kConsWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < cnt; ++i) {
                const int s = i % R;
                if (i >= R) mbar_wait(&empty[s], (uint32_t)((i / R - 1) & 1), P.err, kSiteDenseAct | kSiteEmpty);
                if (P.rows && (P.rows[lo + i] < 0 || P.rows[lo + i] >= P.N)) atomicOr(P.err, SI_DEVERR_COUNT);
                const size_t n = (size_t)row(i);
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
        // the histogram slot of this warp's previous record: its slab entry
        // is written one record later, so the atomic's round trip overlaps
        // the next record's dot products
        uint32_t pend_pos = 0xFFFFFFFFu, pend_bin = 0u;
        int pend_n = -1;
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
                const float av = swiglu(g, u);
                P.a[row(i)] = av;
                mbar_arrive(&empty[s]);
                if (P.hist) {
                    if (P.slab) {
                        if (pend_pos < (uint32_t)kSlabCap) P.slab[(size_t)pend_bin * kSlabCap + pend_pos] = pend_n;
                        pend_bin = abs_key(av) >> kTierShift;
                        pend_pos = atomicAdd(P.hist + pend_bin, 1u);
                        pend_n = row(i);
                    } else {
                        atomicAdd(P.hist + (abs_key(av) >> kTierShift), 1u);
                    }
                }
            }
        }
        if (lane == 0 && pend_pos < (uint32_t)kSlabCap) P.slab[(size_t)pend_bin * kSlabCap + pend_pos] = pend_n;
    }
}

// Tier histogram of a given activation vector, for a tiered call whose a
// did not come from the dense pass (which builds the same histogram), and
// its per-bin member lists: each CTA reserves one run of slots per bin with
// a single global atomic, then places its members by shared-memory rank.
__global__ void __launch_bounds__(256) k_abs_hist(const float* __restrict__ a, int N, unsigned* __restrict__ hist,
                                                 int32_t* __restrict__ slab) {
    __shared__ unsigned h[kTierBins];
    __shared__ unsigned base[kTierBins];
    grid_launch_dependents();
    grid_dependency_wait();  // a may be the previous grid's output
    for (int i = threadIdx.x; i < kTierBins; i += blockDim.x) h[i] = 0u;
    __syncthreads();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x)
        atomicAdd(&h[abs_key(__ldcg(a + i)) >> kTierShift], 1u);
    __syncthreads();
    for (int i = threadIdx.x; i < kTierBins; i += blockDim.x) {
        base[i] = h[i] ? atomicAdd(hist + i, h[i]) : 0u;
        h[i] = 0u;
    }
    if (!slab) return;
    __syncthreads();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x) {
        const uint32_t bin = abs_key(__ldcg(a + i)) >> kTierShift;
        const uint32_t pos = base[bin] + atomicAdd(&h[bin], 1u);
        if (pos < (uint32_t)kSlabCap) slab[(size_t)bin * kSlabCap + pos] = i;
    }
}

// ---------------------------------------------------------- tiered down

// Tier choice inside the tiered kernel (abstract, Fig. 2: Top = the k_top
// largest |a|, Mid = the next k_mid, ties to the lower index). Every CTA
// derives the same two rank boundaries, K0 = k_top and K1 = k_top + k_mid:
// the tier histogram (bits 30..20 of the |a| key) gives each boundary's
// top digit, two passes over the keys of that bin (bits 19..9, then 8..0)
// give the exact key `thr` and how many keys equal to it are taken. The
// CTA then counts the members of each tier in index order and takes its
// window of ranks of both tiers (balanced over the CTAs).
constexpr int kTdThreads = 256;          // threads of the tiered kernel: eight warps
constexpr int kTDW = kTdThreads / 32;    // warps of the tiered kernel
constexpr int kTdSplit = 1;              // warps that share a record, each a slice of its rows
constexpr int kTdPairs = kTDW / kTdSplit;  // record streams (one per group of kTdSplit warps)
constexpr int kTdSlots = 16;             // records in flight per stream at most (one barrier pair each)

// Exclusive scan over the CTA's warps of two per-warp counts (the same value
// in every lane of a warp); gives the warp's offsets and the CTA totals.
__device__ __forceinline__ void cta_scan2(uint32_t c0, uint32_t c1, uint2* s_w, uint32_t& o0, uint32_t& o1,
                                          uint32_t& n0, uint32_t& n1) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) s_w[warp] = make_uint2(c0, c1);
    __syncthreads();
    uint32_t a0 = 0u, a1 = 0u, t0 = 0u, t1 = 0u;
#pragma unroll
    for (int w = 0; w < kTDW; ++w) {
        const uint2 v = s_w[w];
        if (w < warp) {
            a0 += v.x;
            a1 += v.y;
        }
        t0 += v.x;
        t1 += v.y;
    }
    o0 = a0;
    o1 = a1;
    n0 = t0;
    n1 = t1;
    __syncthreads();  // s_w may be reused
}

// For each active boundary t: the bin of h[t] (nb bins, a power of two >= 256,
// counted from the highest bin down) holding its kk[t]-th largest key.
// Updates kk[t] to the rank left inside that bin and returns the bin and its
// count; `total` is the sum of h[0]. Threads 0..255 own nb/256 bins each.
__device__ void find_bins2(const unsigned* h0, const unsigned* h1, int nb, const bool* act, uint32_t* kk,
                           uint32_t* bin, uint32_t* cnt, uint32_t* total, uint2* s_w, uint32_t* s_state) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int per = nb / 256;
    const bool own = tid < 256;
    uint32_t c[2] = {0u, 0u};
    if (own)
        for (int j = 0; j < per; ++j) {
            c[0] += h0[nb - 1 - per * tid - j];
            c[1] += h1[nb - 1 - per * tid - j];
        }
    uint32_t w0 = c[0], w1 = c[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t a0 = __shfl_up_sync(0xFFFFFFFFu, w0, o), a1 = __shfl_up_sync(0xFFFFFFFFu, w1, o);
        if (lane >= o) {
            w0 += a0;
            w1 += a1;
        }
    }
    uint32_t o0, o1, n0, n1;
    cta_scan2(__shfl_sync(0xFFFFFFFFu, w0, 31), __shfl_sync(0xFFFFFFFFu, w1, 31), s_w, o0, o1, n0, n1);
    const uint32_t e[2] = {o0 + w0 - c[0], o1 + w1 - c[1]};  // keys in higher bins
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (own && act[t] && e[t] < kk[t] && kk[t] <= e[t] + c[t]) {
            const unsigned* h = t ? h1 : h0;
            uint32_t run = e[t];
            for (int j = 0; j < per; ++j) {
                const int b = nb - 1 - per * tid - j;
                if (run + h[b] >= kk[t]) {
                    s_state[3 * t] = (uint32_t)b;
                    s_state[3 * t + 1] = kk[t] - run;
                    s_state[3 * t + 2] = h[b];
                    break;
                }
                run += h[b];
            }
        }
    }
    *total = n0;
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (act[t]) {
            bin[t] = s_state[3 * t];
            kk[t] = s_state[3 * t + 1];
            cnt[t] = s_state[3 * t + 2];
        }
    }
    __syncthreads();
}


// Tier choice of one CTA (the scheme above): both boundaries from the tier
// histogram (already in s_hist[0]) and two passes over the keys, then this
// CTA's windows [t0, t1) of the top ranks and [m0, m1) of the middle ranks
// into s_col / s_av (top first), and the optional global lists for exactly
// those windows. aval(i) reads a[i]. Called by every thread of the CTA.
template <class ValF>
__device__ __forceinline__ void tier_windows(const TieredDownParams& P, ValF aval, int t0, int t1, int m0, int m1,
                                               int* s_col, float* s_av, unsigned (*s_hist)[kTierBins], uint2* s_w,
                                               uint32_t* s_state) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = P.N, ntop = t1 - t0;
    auto key = [&](int i) -> uint32_t { return abs_key(aval(i)); };
    // --- the two boundaries: digits 30..20 (histogram), 19..9, 8..0
    const int K[2] = {P.k_top, P.k_top + P.k_mid};
    bool act[2] = {K[0] > 0 && K[0] < N, K[1] > 0 && K[1] < N};
    uint32_t kk[2] = {(uint32_t)K[0], (uint32_t)K[1]}, d0[2] = {0u, 0u}, d1[2] = {0u, 0u}, d2[2] = {0u, 0u};
    uint32_t eqn[2] = {0u, 0u}, total = 0u, unused = 0u;
    find_bins2(s_hist[0], s_hist[0], kTierBins, act, kk, d0, eqn, &total, s_w, s_state);
    const bool bad = total != (uint32_t)N;  // a histogram that does not describe a
    if (bad) act[0] = act[1] = false;
    const bool same1 = act[0] && act[1] && d0[0] == d0[1];
    for (int i = tid; i < 2 * kTierBins; i += blockDim.x) (&s_hist[0][0])[i] = 0u;
    __syncthreads();
    // keys are read eight at a time ahead of the atomics (which the compiler
    // cannot move loads across); 0xFFFFFFFF pads past the end and matches no bin
    if (act[0] || act[1])
        for (int i0 = tid; i0 < N; i0 += 8 * kTdThreads) {
            uint32_t kv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) kv[u] = i0 + u * kTdThreads < N ? key(i0 + u * kTdThreads) : 0xFFFFFFFFu;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t top = kv[u] >> kTierShift, b = (kv[u] >> 9) & 2047u;
                if (act[0] && top == d0[0]) atomicAdd(&s_hist[0][b], 1u);
                if (act[1] && !same1 && top == d0[1]) atomicAdd(&s_hist[1][b], 1u);
            }
        }
    __syncthreads();
    find_bins2(s_hist[0], same1 ? s_hist[0] : s_hist[1], 2048, act, kk, d1, eqn, &unused, s_w, s_state);
    const uint32_t pre[2] = {(d0[0] << 11) | d1[0], (d0[1] << 11) | d1[1]};
    const bool same2 = same1 && pre[0] == pre[1];
    for (int i = tid; i < 2 * kTierBins; i += blockDim.x) (&s_hist[0][0])[i] = 0u;
    __syncthreads();
    if (act[0] || act[1])
        for (int i0 = tid; i0 < N; i0 += 8 * kTdThreads) {
            uint32_t kv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) kv[u] = i0 + u * kTdThreads < N ? key(i0 + u * kTdThreads) : 0xFFFFFFFFu;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t b = kv[u] & 511u;
                if (act[0] && (kv[u] >> 9) == pre[0]) atomicAdd(&s_hist[0][b], 1u);
                if (act[1] && !same2 && (kv[u] >> 9) == pre[1]) atomicAdd(&s_hist[1][b], 1u);
            }
        }
    __syncthreads();
    find_bins2(s_hist[0], same2 ? s_hist[0] : s_hist[1], 512, act, kk, d2, eqn, &unused, s_w, s_state);
    // Boundary t takes every key > thr[t] and the first take[t] keys == thr[t]
    // in index order; K == 0 (or a bad histogram) takes nothing, K == N all.
    uint32_t thr[2], take[2];
    bool split = false;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (act[t]) {
            thr[t] = (d0[t] << kTierShift) | (d1[t] << 9) | d2[t];
            take[t] = kk[t];
            split |= kk[t] < eqn[t];
        } else if (K[t] <= 0 || bad) {
            thr[t] = 0xFFFFFFFFu;  // keys are below 2^31: nothing is greater or equal
            take[t] = 0u;
        } else {
            thr[t] = 0u;
            take[t] = 0xFFFFFFFFu;
        }
    }

    // --- members in index order; this CTA takes ranks [t0, t1) and [m0, m1).
    // Warp w covers indices [w * SEG, (w + 1) * SEG), 32 at a time.
    const int SEG = ((N + kTDW * 32 - 1) / (kTDW * 32)) * 32;
    const int lo = warp * SEG, hi = min(N, lo + SEG);
    const uint32_t lt = lanemask_lt();
    uint32_t eqb0 = 0u, eqb1 = 0u;
    if (split) {  // ranks among equal keys need the equal keys before each warp
        uint32_t q0 = 0u, q1 = 0u, u0, u1;
        for (int i0 = lo; i0 < hi; i0 += 128) {
            uint32_t kv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) kv[u] = i0 + 32 * u + lane < hi ? key(i0 + 32 * u + lane) : 0xFFFFFFFFu;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool in = i0 + 32 * u + lane < hi;
                q0 += __popc(__ballot_sync(0xFFFFFFFFu, in && kv[u] == thr[0]));
                q1 += __popc(__ballot_sync(0xFFFFFFFFu, in && kv[u] == thr[1]));
            }
        }
        cta_scan2(q0, q1, s_w, eqb0, eqb1, u0, u1);
    }
    uint32_t base0 = 0u, base1 = 0u, n0 = 0u, n1 = 0u, w0 = 0u, w1 = 0u;
    for (int pass = 0; pass < 2; ++pass) {
        // pass 0 counts the warp's members, pass 1 places those in this CTA's windows
        if (pass == 1 && !(base0 < (uint32_t)t1 && base0 + w0 > (uint32_t)t0) &&
            !(base1 < (uint32_t)m1 && base1 + w1 > (uint32_t)m0) && !(P.top_out || P.mid_out))
            break;
        uint32_t r0 = eqb0, r1 = eqb1, c0 = 0u, c1 = 0u;
        for (int i4 = lo; i4 < hi; i4 += 128) {
            uint32_t kv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) kv[u] = i4 + 32 * u + lane < hi ? key(i4 + 32 * u + lane) : 0u;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i4 + 32 * u + lane;
                const bool in = i < hi;
                const uint32_t k = kv[u];
                const uint32_t e0 = __ballot_sync(0xFFFFFFFFu, in && k == thr[0]);
                const uint32_t e1 = __ballot_sync(0xFFFFFFFFu, in && k == thr[1]);
                const bool sel0 = in && (k > thr[0] || (k == thr[0] && r0 + __popc(e0 & lt) < take[0]));
                const bool sel1 = in && (k > thr[1] || (k == thr[1] && r1 + __popc(e1 & lt) < take[1]));
                r0 += __popc(e0);
                r1 += __popc(e1);
                const bool is_mid = sel1 && !sel0;
                const uint32_t bt = __ballot_sync(0xFFFFFFFFu, sel0), bm = __ballot_sync(0xFFFFFFFFu, is_mid);
                if (pass == 1) {
                    if (sel0) {
                        const uint32_t r = base0 + c0 + __popc(bt & lt);
                        if (r >= (uint32_t)t0 && r < (uint32_t)t1) {
                            s_col[r - t0] = i;
                            s_av[r - t0] = aval(i);
                            if (P.top_out) P.top_out[r] = i;
                        }
                    }
                    if (is_mid) {
                        const uint32_t r = base1 + c1 + __popc(bm & lt);
                        if (r >= (uint32_t)m0 && r < (uint32_t)m1) {
                            s_col[ntop + r - m0] = i;
                            s_av[ntop + r - m0] = aval(i);
                            if (P.mid_out) P.mid_out[r] = i;
                        }
                    }
                }
                c0 += __popc(bt);
                c1 += __popc(bm);
            }
        }
        if (pass == 0) {
            w0 = c0;
            w1 = c1;
            cta_scan2(c0, c1, s_w, base0, base1, n0, n1);
        }
    }
    if (tid == 0 && !bad && (n0 != (uint32_t)P.k_top || n1 != (uint32_t)P.k_mid)) atomicOr(P.err, SI_DEVERR_COUNT);
    if (tid == 0 && bad) atomicOr(P.err, SI_DEVERR_COUNT);
}

// Thresholds of both boundaries from the candidates: pass `p` (1: bits
// 19..9, 2: bits 8..0) over the keys in cand[0, C) that share the prefix
// found so far. Every thread of the CTA calls it.
template <class KeyF>
__device__ __forceinline__ void tier_refine(KeyF key, const int* cand, int C, int p, const bool* act,
                                            const uint32_t* pre, unsigned (*s_hist)[kTierBins], uint32_t* kk,
                                            uint32_t* dig, uint32_t* eqn, uint2* s_w, uint32_t* s_state) {
    const int shift = p == 1 ? kTierShift : 9;   // bits above the digit: the prefix
    const int dshift = p == 1 ? 9 : 0;
    const uint32_t dmask = p == 1 ? 2047u : 511u;
    const bool same = act[0] && act[1] && pre[0] == pre[1];
    for (int i = threadIdx.x; i < 2 * kTierBins; i += blockDim.x) (&s_hist[0][0])[i] = 0u;
    __syncthreads();
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        const uint32_t k = key(cand[c]), hi = k >> shift, b = (k >> dshift) & dmask;
        if (act[0] && hi == pre[0]) atomicAdd(&s_hist[0][b], 1u);
        if (act[1] && !same && hi == pre[1]) atomicAdd(&s_hist[1][b], 1u);
    }
    __syncthreads();
    uint32_t unused;
    find_bins2(s_hist[0], same ? s_hist[0] : s_hist[1], (int)dmask + 1, act, kk, dig, eqn, &unused, s_w, s_state);
}

// Tier choice of one CTA when a is staged in shared memory (s_a) and no
// global lists are wanted: the CTA owns the contiguous index range
// [n0, n1) and takes the tier members in it, top ones first, then middle
// ones, each in index order, into s_col / s_av, with their counts in s_n.
// Only the keys in the two boundary bins of the histogram (the candidates,
// gathered once into cand) are needed to finish both thresholds and to
// count the keys equal to a threshold before n0. Returns false (before
// touching the histogram in s_hist[0]) when the candidates exceed cap; the
// caller then takes the rank windows instead. Every thread calls it.
__device__ bool tier_own_range(const TieredDownParams& P, const float* s_a, int* cand, int cap, int n0, int n1,
                               int* s_col, float* s_av, unsigned (*s_hist)[kTierBins], uint2* s_w,
                               uint32_t* s_state, int* s_n) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = P.N;
    auto key = [&](int i) -> uint32_t { return abs_key(s_a[i]); };
    const int K[2] = {P.k_top, P.k_top + P.k_mid};
    bool act[2] = {K[0] > 0 && K[0] < N, K[1] > 0 && K[1] < N};
    uint32_t kk[2] = {(uint32_t)K[0], (uint32_t)K[1]}, d0[2] = {0u, 0u}, d1[2] = {0u, 0u}, d2[2] = {0u, 0u};
    uint32_t eqn[2] = {0u, 0u}, total = 0u;
    // the top digit of each boundary from the histogram (read only)
    find_bins2(s_hist[0], s_hist[0], kTierBins, act, kk, d0, eqn, &total, s_w, s_state);
    const bool bad = total != (uint32_t)N;  // a histogram that does not describe a
    if (bad) act[0] = act[1] = false;

    // candidates: indices of the keys in either boundary bin, in index order.
    // Each lane owns a contiguous run of LQ quads (four consecutive keys, one
    // 16-byte read each); the lanes' runs tile the warps' runs in order. Pass
    // 0 counts per lane (no cross-lane work in the loop), one scan gives each
    // lane its first slot, pass 1 writes.
    const uint32_t lt = lanemask_lt();
    const int NQ = (N + 3) / 4;
    const int LQ = ((NQ + kTDW * 32 - 1) / (kTDW * 32)) | 1;  // odd: spreads the lanes over the banks
    const int q_lo = (warp * 32 + lane) * LQ, q_hi = min(NQ, q_lo + LQ);
    const float4* s_a4 = reinterpret_cast<const float4*>(s_a);
    auto quad_matches = [&](int q) -> uint32_t {  // bit u: key 4q + u is a candidate
        const float4 v = s_a4[q];
        const float f[4] = {v.x, v.y, v.z, v.w};
        uint32_t m = 0u;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t t = abs_key(f[u]) >> kTierShift;
            if (4 * q + u < N && ((act[0] && t == d0[0]) || (act[1] && t == d0[1]))) m |= 1u << u;
        }
        return m;
    };
    // When both boundary bins fit their member lists (filled by the pass that
    // built the histogram), the candidates are read from those lists rather
    // than found by a scan of every key; their order does not matter below.
    const bool two = act[1] && !(act[0] && d0[1] == d0[0]);
    const uint32_t h0 = act[0] ? s_hist[0][d0[0]] : 0u, h1 = two ? s_hist[0][d0[1]] : 0u;
    uint32_t C;
    // (bin 0 holds a = 0; a dense pass over a row list counts the unlisted
    // zeros there without listing them, so bin 0 is always scanned)
    const bool zero_bin = (act[0] && d0[0] == 0u) || (two && d0[1] == 0u);
    if (P.slab && !zero_bin && h0 <= (uint32_t)kSlabCap && h1 <= (uint32_t)kSlabCap && h0 + h1 <= (uint32_t)cap) {
        C = h0 + h1;
        const uint32_t b0 = act[0] ? d0[0] : d0[1];  // the first list's bin
        auto slot = [&](uint32_t c) -> size_t {
            return c < h0 ? (size_t)b0 * kSlabCap + c : (size_t)d0[1] * kSlabCap + (c - h0);
        };
        // eight loads in flight per thread before any store (C <= 2 * kSlabCap:
        // one round trip for up to 8 * 288 candidates)
        for (uint32_t c0 = (uint32_t)tid; c0 < C; c0 += 8u * blockDim.x) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t c = c0 + (uint32_t)u * blockDim.x;
                v[u] = c < C ? __ldcg(P.slab + slot(c)) : 0;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t c = c0 + (uint32_t)u * blockDim.x;
                if (c < C) cand[c] = v[u];
            }
        }
        __syncthreads();
    } else {
        uint32_t n = 0u;
        if (act[0] || act[1])
            for (int q = q_lo; q < q_hi; ++q) n += __popc(quad_matches(q));
        uint32_t incl = n;  // lanes' counts, inclusive scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        uint32_t wbase, unused0, unused1;
        cta_scan2(__shfl_sync(0xFFFFFFFFu, incl, 31), 0u, s_w, wbase, unused0, C, unused1);
        if (C > (uint32_t)cap) return false;  // the same decision in every thread
        if (n) {
            uint32_t pos = wbase + incl - n;
            for (int q = q_lo; q < q_hi; ++q) {
                const uint32_t m = quad_matches(q);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (m & (1u << u)) cand[pos++] = 4 * q + u;
            }
        }
        __syncthreads();
    }

    // both thresholds: bits 19..9, then 8..0, over the candidates
    const uint32_t pre1[2] = {d0[0], d0[1]};
    tier_refine(key, cand, (int)C, 1, act, pre1, s_hist, kk, d1, eqn, s_w, s_state);
    const uint32_t pre2[2] = {(d0[0] << 11) | d1[0], (d0[1] << 11) | d1[1]};
    tier_refine(key, cand, (int)C, 2, act, pre2, s_hist, kk, d2, eqn, s_w, s_state);
    uint32_t thr[2], take[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (act[t]) {
            thr[t] = (d0[t] << kTierShift) | (d1[t] << 9) | d2[t];
            take[t] = kk[t];
        } else if (K[t] <= 0 || bad) {
            thr[t] = 0xFFFFFFFFu;  // keys are below 2^31: nothing is greater or equal
            take[t] = 0u;
        } else {
            thr[t] = 0u;
            take[t] = 0xFFFFFFFFu;
        }
    }

    // keys equal to a threshold before n0: all of them are candidates
    uint32_t e0 = 0u, e1 = 0u;
    for (int c = tid; c < (int)C; c += blockDim.x) {
        const int i = cand[c];
        if (i < n0) {
            const uint32_t k = key(i);
            e0 += k == thr[0];
            e1 += k == thr[1];
        }
    }
    uint32_t o0, o1, E0, E1;
    cta_scan2(__reduce_add_sync(0xFFFFFFFFu, e0), __reduce_add_sync(0xFFFFFFFFu, e1), s_w, o0, o1, E0, E1);

    // the CTA's own range, in index order: top members, then middle members
    if (warp == 0) {
        int ntop = 0;
        for (int part = 0; part < 2; ++part) {
            uint32_t r0 = E0, r1 = E1;
            int c = 0;
            for (int i0 = n0; i0 < n1; i0 += 32) {
                const int i = i0 + lane;
                const bool in = i < n1;
                const uint32_t k = in ? key(i) : 0u;
                const uint32_t q0 = __ballot_sync(0xFFFFFFFFu, in && k == thr[0]);
                const uint32_t q1 = __ballot_sync(0xFFFFFFFFu, in && k == thr[1]);
                const bool sel0 = in && (k > thr[0] || (k == thr[0] && r0 + __popc(q0 & lt) < take[0]));
                const bool sel1 = in && (k > thr[1] || (k == thr[1] && r1 + __popc(q1 & lt) < take[1]));
                r0 += __popc(q0);
                r1 += __popc(q1);
                const bool want = part == 0 ? sel0 : (sel1 && !sel0);
                const uint32_t bw = __ballot_sync(0xFFFFFFFFu, want);
                if (want) {
                    const int pos = (part == 0 ? 0 : ntop) + c + __popc(bw & lt);
                    s_col[pos] = i;
                    s_av[pos] = s_a[i];
                }
                c += __popc(bw);
            }
            if (part == 0) ntop = c;
            else if (lane == 0) {
                s_n[0] = ntop;
                s_n[1] = c;
            }
        }
    }
    if (tid == 0 && bad) atomicOr(P.err, SI_DEVERR_COUNT);
    return true;
}

// Shared-memory layout of the tiered kernel: per record stream kTdSlots
// "full" and "empty" barriers, the activation / column buffer, then the ring
// (ring_bytes, the CTA's sum of y in its last 4d bytes).
__host__ __device__ inline int td_off_aux() { return round_up(16 * kTdPairs * kTdSlots, 128); }
__host__ __device__ inline int td_off_ring(int aux_floats) { return td_off_aux() + round_up(aux_floats * 4, 128); }

// The eight 4-bit codes of a 32-bit word (element i at bits 4i) as the floats
// 1 + q / 16 (exact: q sits in the top mantissa bits of 1.0f), in element
// pairs: element 2m is the low nibble of byte m, 2m + 1 the high one.
__device__ __forceinline__ void codes4_unit(uint32_t q, float2 (&w)[4]) {
    const uint32_t lo = ((q << 3) & 0x78787878u) | 0x80808080u;  // byte m: 0x80 | low nibble << 3
    const uint32_t hi = ((q >> 1) & 0x78787878u) | 0x80808080u;  // byte m: 0x80 | high nibble << 3
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t sel = 0x7044u | ((uint32_t)m << 8);  // bytes: 0, 0, lo/hi byte m, 0x3F
        w[m] = make_float2(__uint_as_float(__byte_perm(lo, 0x3F000000u, sel)),
                           __uint_as_float(__byte_perm(hi, 0x3F000000u, sel)));
    }
}

// SpAx tiered down-projection (abstract, Fig. 2; middle columns rebuilt from
// their codes as in Fig. 3): y = sum over Top of a_n Wd[:, n] + sum over Mid
// of a_n (min_g + q * scale_g). Each CTA takes its own index range (or an
// even share of both tier lists), its top columns first, then its middle
// ones. Record i goes to stream i % S (S = 8 / kTdSplit streams of kTdSplit
// warps): each warp of the stream reads it, a slice of the d rows each (lane
// l: chunks l + 32 j of 8 rows of the slice). The stream's first warp issues
// the stream's copies into the stream's own byte ring, records back to back
// at their own size (a bf16 column 2d bytes, a code record rec_bytes), and
// reuses bytes once every warp of the stream has released them. The
// streams' partials meet in shared memory at the end (summed in stream
// order) and the CTAs' sums are reduced through the cluster and a
// fixed-order final pass (deterministic). FULL: d == 2048 * MAXC, every
// lane's chunks exist (no bounds checks in the per-record code).
template <int MAXC, int BITS, bool FULL>
__global__ void __launch_bounds__(kTdThreads, 1) k_tiered_down(TieredDownParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int d = P.d;
    const int mid_bytes = P.rec_bytes;  // d * BITS / 8 code bytes, then ngp (scale, min) pairs
    uint64_t* full_all = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty_all = full_all + kTdPairs * kTdSlots;
    float* s_av = reinterpret_cast<float*>(smem + td_off_aux());
    uint8_t* ring = smem + td_off_ring(P.aux_floats);
    const int ring_bytes = P.ring_bytes;
    // each stream's ring (records only; the CTA sum of y follows them)
    const int RP = ((ring_bytes - 4 * d) / kTdPairs) / 128 * 128;
    float* ycta = reinterpret_cast<float*>(ring + ring_bytes) - d;
    // a stream's ring holds one record of either kind, the streams' partials
    // and the CTA sum fit the ring, a slice's chunks fit 8 * MAXC / kTdSplit
    // per lane; refuse a launch where they do not (the host never makes one)
    if (RP < 2 * d || RP < mid_bytes || (mid_bytes & 15) || (d % (8 * kTdSplit)) || d > 2048 * MAXC ||
        (FULL && d != 2048 * MAXC) || (long long)ring_bytes < (4LL * kTdPairs + 4) * d) {
        if (threadIdx.x == 0) atomicOr(P.err, SI_DEVERR_COUNT);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // rank windows of the two tiers (fallback) and own index range (fast path)
    const int t0 = (int)((long long)P.k_top * blockIdx.x / gridDim.x);
    const int t1 = (int)((long long)P.k_top * (blockIdx.x + 1) / gridDim.x);
    const int m0 = (int)((long long)P.k_mid * blockIdx.x / gridDim.x);
    const int m1 = (int)((long long)P.k_mid * (blockIdx.x + 1) / gridDim.x);
    const int n0 = (int)((long long)P.N * blockIdx.x / gridDim.x);
    const int n1 = (int)((long long)P.N * (blockIdx.x + 1) / gridDim.x);

    if (threadIdx.x == 0) {
        for (int b = 0; b < kTdPairs * kTdSlots; ++b) {
            mbar_init(&full_all[b], 1);
            mbar_init(&empty_all[b], kTdSplit);
        }
        fence_mbar_init();
    }
    __shared__ unsigned s_hist[2][kTierBins];
    __shared__ uint2 s_w[kTDW];
    __shared__ uint32_t s_state[6];
    __shared__ unsigned s_last;
    __shared__ __align__(8) uint64_t s_stage_bar;
    __shared__ int s_n[2];
    grid_launch_dependents();
    grid_dependency_wait();  // a and its tier histogram are the previous grids' output
    const int tid = threadIdx.x;
    const int N = P.N;
    int* s_col = reinterpret_cast<int*>(s_av + P.aux_floats / 2);
    // a is staged in the ring when it fits (the ring is idle until streaming):
    // one bulk copy when a is 16-byte aligned and sized, else vector loads
    const int RB = kTdPairs * RP;
    float* s_a = reinterpret_cast<float*>(ring);
    const bool staged = (long long)N * 4 <= (long long)RB;
    const bool bulk = staged && (N % 4) == 0 && (reinterpret_cast<uintptr_t>(P.a) & 15) == 0;
    if (bulk && tid == 0) {
        mbar_init(&s_stage_bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&s_stage_bar, (uint32_t)(N * 4));
        bulk_g2s(s_a, P.a, (uint32_t)(N * 4), &s_stage_bar);
    } else if (staged && !bulk) {
        for (int i = tid; i < N; i += blockDim.x) s_a[i] = __ldcg(P.a + i);
    }
    for (int i = tid; i < kTierBins; i += blockDim.x) s_hist[0][i] = __ldcg(P.hist + i);
    __syncthreads();
    if (bulk) mbar_wait(&s_stage_bar, 0u, P.err, kSiteTiered | kSiteFullB);

    // Fast path: own index range, candidates in the ring after the staged a.
    int ntop = 0, nrec = 0;
    bool own = false;
    if (staged && !P.top_out && !P.mid_out) {
        const long long off = ((long long)N * 4 + 15) / 16 * 16;
        const long long cap = ((long long)RB - off) / 4;
        own = tier_own_range(P, s_a, reinterpret_cast<int*>(ring + off), (int)(cap < N ? cap : N), n0, n1, s_col,
                             s_av, s_hist, s_w, s_state, s_n);
        __syncthreads();
        if (own) {
            ntop = s_n[0];
            nrec = s_n[0] + s_n[1];
        }
    }
    if (!own) {
        // Rank windows: balanced, and exact global lists; every CTA counts
        // the members over all N. The selection reads a through one path
        // only (a generic "shared or global" load would make the compiler
        // issue the global load every time).
        ntop = t1 - t0;
        nrec = ntop + (m1 - m0);
        for (int i = tid; i < nrec; i += blockDim.x) s_col[i] = -1;
        if (staged)
            tier_windows(P, [&](int i) -> float { return s_a[i]; }, t0, t1, m0, m1, s_col, s_av, s_hist, s_w,
                         s_state);
        else
            tier_windows(P, [&](int i) -> float { return __ldcg(P.a + i); }, t0, t1, m0, m1, s_col, s_av, s_hist,
                         s_w, s_state);
    }
    __syncthreads();  // the records are in place and the staged keys are no longer read

    constexpr int JH = 8 * MAXC / kTdSplit;  // chunks per lane in a slice
    const int pair = warp / kTdSplit, half = warp % kTdSplit;  // stream, slice
    const int nch = d / 8, hch = nch / kTdSplit;  // chunks of a column, of a slice
    const int cbase = half * hch;                 // this warp's first chunk
    float2 acc[JH][4];
    float amin[JH];
#pragma unroll
    for (int j = 0; j < JH; ++j) {
        amin[j] = 0.0f;
#pragma unroll
        for (int m = 0; m < 4; ++m) acc[j][m] = make_float2(0.0f, 0.0f);
    }
    {
        uint8_t* reg = ring + (size_t)pair * RP;
        uint64_t* full = full_all + pair * kTdSlots;
        uint64_t* empty = empty_all + pair * kTdSlots;
        const int nw = nrec > pair ? (nrec - pair + kTdPairs - 1) / kTdPairs : 0;  // the stream's records
        const int gshift = 31 - __clz(P.group);  // group is a power of two (checked by the host)
        auto rec_size = [&](int k) -> uint32_t {
            return pair + kTdPairs * k < ntop ? (uint32_t)(2 * d) : (uint32_t)mid_bytes;
        };
        // Placement in the stream's ring: a running position and offset; a
        // record that would run past the ring's end starts at its beginning.
        // Issuer and consumers replay the same sequence.
        struct Cursor {
            uint32_t mono, off;  // monotonic byte position, its offset in the ring
        };
        auto place = [&](Cursor& c, uint32_t sz) -> uint32_t {
            if (c.off + sz > (uint32_t)RP) {
                c.mono += (uint32_t)RP - c.off;
                c.off = 0u;
            }
            const uint32_t at = c.off;
            c.mono += sz;
            c.off += sz;
            return at;
        };
        const bool issuer = half == 0 && lane == 0;
        const uint64_t pol = policy_evict_first();
        Cursor head = {0u, 0u}, rel = {0u, 0u}, cons = {0u, 0u};
        int ki = 0, jr = 0;  // records issued, records known released (issuer only)
        for (int k = 0; k < nw; ++k) {
            if (issuer) {
                while (ki < nw) {
                    const uint32_t sz = rec_size(ki);
                    Cursor h2 = head;
                    const uint32_t at = place(h2, sz);
                    const bool fits = ki - jr < kTdSlots && (jr == ki || h2.mono - rel.mono <= (uint32_t)RP);
                    if (fits) {
                        const int i = pair + kTdPairs * ki;
                        int ci = s_col[i];
                        if (ci < 0 || ci >= N) {  // never read outside the encoded buffers
                            atomicOr(P.err, SI_DEVERR_COUNT);
                            ci = 0;
                        }
                        const size_t col = (size_t)ci;
                        const void* src = i < ntop ? static_cast<const void*>(P.WdT + col * d)
                                                   : static_cast<const void*>(P.codes + col * (size_t)P.rec_bytes);
                        mbar_arrive_expect_tx(&full[ki % kTdSlots], sz);
                        bulk_g2s_hint(reg + at, src, sz, &full[ki % kTdSlots], pol);
                        head = h2;
                        ++ki;
                        continue;
                    }
                    if (jr >= k) break;  // nothing this warp has consumed is still unreleased
                    // record jr: this warp is done with it; take its release when
                    // the stream's other warps have released it too (wait only if
                    // record k itself still needs the room)
                    const uint32_t par = (uint32_t)((jr / kTdSlots) & 1);
                    if (ki > k) {
                        if (!mbar_test_wait(&empty[jr % kTdSlots], par)) break;
                    } else if (!mbar_wait(&empty[jr % kTdSlots], par, P.err, kSiteTiered | kSiteEmpty)) {
                        break;
                    }
                    place(rel, rec_size(jr));
                    ++jr;
                }
            }
            const int i = pair + kTdPairs * k;
            const uint32_t at = place(cons, rec_size(k));
            mbar_wait(&full[k % kTdSlots], (uint32_t)((k / kTdSlots) & 1), P.err, kSiteTiered | kSiteFull);
            const uint8_t* st = reg + at;
            const float av = s_av[i];
            if (i < ntop) {
                const float2 a2 = make_float2(av, av);
#pragma unroll
                for (int j = 0; j < JH; ++j) {
                    const int c = lane + 32 * j;
                    if (FULL || c < hch) {
                        float f[8];
                        unpack8(reinterpret_cast<const uint4*>(st)[cbase + c], f);
#pragma unroll
                        for (int m = 0; m < 4; ++m) acc[j][m] = __ffma2_rn(a2, make_float2(f[2 * m], f[2 * m + 1]), acc[j][m]);
                    }
                }
            } else {
                const float2* prm = reinterpret_cast<const float2*>(st + (d * BITS) / 8);
#pragma unroll
                for (int j = 0; j < JH; ++j) {
                    const int c = lane + 32 * j;
                    if (FULL || c < hch) {
                        const int cc = cbase + c;
                        const float2 sm = prm[(8 * cc) >> gshift];  // (scale, min)
                        if constexpr (BITS == 4) {
                            // codes as 1 + q / 16: a (min + q scale) = 16 a scale (1 + q / 16) + a (min - 16 scale)
                            const float c1 = (16.0f * av) * sm.x;
                            amin[j] += fmaf(av, sm.y, -c1);
                            const float2 c2 = make_float2(c1, c1);
                            float2 w[4];
                            codes4_unit(reinterpret_cast<const uint32_t*>(st)[cc], w);
#pragma unroll
                            for (int m = 0; m < 4; ++m) acc[j][m] = __ffma2_rn(c2, w[m], acc[j][m]);
                        } else {
                            const float c1 = av * sm.x;
                            amin[j] = fmaf(av, sm.y, amin[j]);
                            // a code arrives as the float bits of 2^23 + code,
                            // exact for codes below 2^23, and 2^23 is subtracted
                            uint32_t wd[8];
                            if constexpr (BITS == 8) {
                                // one byte per element
                                const uint2 q = reinterpret_cast<const uint2*>(st)[cc];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    wd[e] = __byte_perm(q.x, 0x4B000000u, 0x7440u | (uint32_t)e);
                                    wd[4 + e] = __byte_perm(q.y, 0x4B000000u, 0x7440u | (uint32_t)e);
                                }
                            } else if constexpr (BITS == 3) {
                                // 24 bits per chunk, in bytes 3c .. 3c + 2; element e at bits 3e .. 3e + 2
                                const uint8_t* b3 = st + 3 * cc;
                                const uint32_t q = (uint32_t)b3[0] | ((uint32_t)b3[1] << 8) | ((uint32_t)b3[2] << 16);
#pragma unroll
                                for (int e = 0; e < 8; ++e) wd[e] = 0x4B000000u | ((q >> (3 * e)) & 7u);
                            } else {
                                // BITS == 2: sixteen bits per chunk, element e at bits 2e, 2e + 1
                                const uint32_t q = reinterpret_cast<const uint16_t*>(st)[cc];
#pragma unroll
                                for (int e = 0; e < 8; ++e) wd[e] = 0x4B000000u | ((q >> (2 * e)) & 3u);
                            }
                            const float2 c2 = make_float2(c1, c1);
#pragma unroll
                            for (int m = 0; m < 4; ++m)
                                acc[j][m] = __ffma2_rn(c2, make_float2(__uint_as_float(wd[2 * m]) - 8388608.0f,
                                                                       __uint_as_float(wd[2 * m + 1]) - 8388608.0f),
                                                       acc[j][m]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[k % kTdSlots]);
        }
    }
    // All records consumed and every copy landed: the stream's partial goes
    // to ring region `pair` (d floats; this warp writes its slice), then each
    // thread sums its float4 columns over the streams in stream order.
    __syncthreads();
    {
        float* part = reinterpret_cast<float*>(ring) + (size_t)pair * d;
#pragma unroll
        for (int j = 0; j < JH; ++j) {
            const int c = lane + 32 * j;
            if (FULL || c < hch) {
                float4* pc = reinterpret_cast<float4*>(part + 8 * (cbase + c));
                pc[0] = make_float4(acc[j][0].x + amin[j], acc[j][0].y + amin[j], acc[j][1].x + amin[j],
                                    acc[j][1].y + amin[j]);
                pc[1] = make_float4(acc[j][2].x + amin[j], acc[j][2].y + amin[j], acc[j][3].x + amin[j],
                                    acc[j][3].y + amin[j]);
            }
        }
    }
    __syncthreads();
    {
        const float4* part4 = reinterpret_cast<const float4*>(ring);
        for (int k = tid; k < d / 4; k += blockDim.x) {
            float4 v = part4[k];
#pragma unroll
            for (int p = 1; p < kTdPairs; ++p) {
                const float4 u = part4[(size_t)p * (d / 4) + k];
                v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
            }
            reinterpret_cast<float4*>(ycta)[k] = v;
        }
    }
    __syncthreads();
    cluster_ticket_reduce4(ycta, d, P.part, P.tickets, P.y);
    // every CTA read the histogram at its start; the last one to finish
    // re-zeroes it for the next token
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(P.hist + kTierBins, 1u) == gridDim.x - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (s_last) {
        for (int i = threadIdx.x; i < kTierBins; i += blockDim.x) P.hist[i] = 0u;
        if (threadIdx.x == 0) P.hist[kTierBins] = 0u;
    }
}

// ------------------------------------------------------------------ launch

namespace {

constexpr int kSmemBudget = 227 * 1024 - 2048;  // dynamic budget, leaves room for static smem

// Clustered launch; with `pdl` the launch may overlap the previous grid in
// the stream (programmatic stream serialization: the kernel itself waits with
// griddepcontrol.wait before it reads anything that grid may write).
template <class K>
cudaError_t launch_clustered(K kernel, int grid, int cluster, size_t smem, cudaStream_t st, void** args,
                             bool pdl = false, int threads = kDecThreads) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
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
cudaError_t pick_grid(K kernel, size_t smem, int* grid, int* cluster, int threads) {
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
        cfg.blockDim = dim3(threads, 1, 1);
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
cudaError_t cached_grid(K kernel, size_t smem, int* grid, int* cluster, int threads = kDecThreads) {
    static thread_local GridCache cache[64];
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
    e = pick_grid(kernel, smem, grid, cluster, threads);
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
    if ((B * P.d) % (4 * cluster)) return cudaErrorInvalidValue;  // float4 slices per cluster rank
    void* args[] = {&P};
    return launch_clustered(kern, grid, cluster, smem, st, args);
}

// One CTA per SM minus a few: with programmatic dependent launch the next
// launch's CTAs take SMs as this launch's CTAs leave, and the spare SMs keep
// the last CTA's tail from delaying the next launch's start.
constexpr int kSpareSms = 4;

template <int MAXC>
cudaError_t launch_sd1(SparseDecodeParams& P, cudaStream_t st) {
    auto kern = k_sparse_decode_b1<MAXC, false>;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = allow_max_smem(kern)) != cudaSuccess) return e;
    const size_t smem = (size_t)ring_layout(P.R, 6 * P.d, 4 * kB1MaxStages, 2 * P.d).total;
    void* args[] = {&P};
    return launch_clustered(kern, sms > 2 * kSpareSms ? sms - kSpareSms : sms, 1, smem, st, args, /*pdl=*/true);
}

// The overwrite form with the cluster reduction: clusters from the occupancy
// of this kernel (as the other clustered decode kernels).
template <int MAXC>
cudaError_t launch_sd1_cr(SparseDecodeParams& P, cudaStream_t st) {
    auto kern = k_sparse_decode_b1<MAXC, true>;
    const size_t smem = (size_t)ring_layout(P.R, 6 * P.d, 4 * kB1MaxStages, 2 * P.d).total;
    int grid = 0, cluster = 0;
    cudaError_t e = cached_grid(kern, smem, &grid, &cluster);
    if (e != cudaSuccess) return e;
    if (P.part_floats < (long long)(grid / cluster) * P.d) return cudaErrorInvalidValue;
    if (P.d % (4 * cluster)) return cudaErrorInvalidValue;  // float4 slices per cluster rank
    void* args[] = {&P};
    return launch_clustered(kern, grid, cluster, smem, st, args, /*pdl=*/true);
}

}  // namespace


int sparse_decode_stages(int d, int B) {
    const int fixed = ring_layout(0, 6 * d, 2 * kConsWarps * B * 4, B * d * 2).total;
    const int stage = round_up(6 * d, 128);
    // the cluster reduction's static shared memory (a float4 per thread) comes
    // out of the same 227 KB
    int R = (kSmemBudget - (int)sizeof(float4) * kDecThreads - fixed - 256) / stage;
    if (R > 32) R = 32;
    return R;
}

int tiered_max_partial_floats(int d) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms * d;  // one partial per CTA, one CTA per SM
}

int decode_max_partial_floats(int d, int B) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    // one partial per CTA for the tensor-core batch kernel (one CTA per SM),
    // one per cluster (at least 2 CTAs) otherwise
    return (B > 1 ? sms : sms / 2 + 1) * B * d;
}

int sparse_decode_b1_stages(int d, int extra_static) {
    const int stage = round_up(6 * d, 128);
    int R = (kSmemBudget - extra_static - ring_layout(kB1MaxStages, 0, 4 * kB1MaxStages, 2 * d).total) / stage;
    if (R > kB1MaxStages) R = kB1MaxStages;
    // warp w's partial (blocks of 32 chunks: round_up(d, 256) floats) reuses
    // its stage w, then the CTA partial stage 0
    return (R >= kConsWarps && stage >= round_up(d, 256) * 4) ? R : 0;
}

// Cooperative launch (one CTA per SM, all resident: a grid-wide slice
// reduction waits on every CTA), with programmatic stream serialization when
// the runtime accepts the two together (probed once, outside stream capture;
// during a capture before the probe, cooperative alone).
cudaError_t launch_coop(const void* kern, cudaLaunchConfig_t cfg, void** args) {
    static int state = 0;  // 0 unknown, 1 cooperative + PDL accepted, 2 cooperative only
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    if (state == 0) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(cfg.stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
            cfg.numAttrs = 1;
            return cudaLaunchKernelExC(&cfg, kern, args);
        }
        cfg.numAttrs = 2;
        const cudaError_t e = cudaLaunchKernelExC(&cfg, kern, args);
        if (e == cudaSuccess) {
            state = 1;
            return e;
        }
        (void)cudaGetLastError();
        state = 2;
    }
    cfg.numAttrs = state == 1 ? 2 : 1;
    return cudaLaunchKernelExC(&cfg, kern, args);
}

// Stages of the tensor-core batch decode for width d (at most 32; 0 when
// fewer than one batch of records fits).
int sparse_decode_mma_stages(int d) {
    const MmaLayout L = mma_layout(0, d);
    int R = (kSmemBudget - (int)sizeof(float4) * kDecThreads - L.off_ring - 256) / L.stage;
    if (R > 32) R = 32;
    return R >= kMmaBatch ? R : 0;
}

template <int DT>
cudaError_t launch_sd_mma(SparseDecodeParams& P, int B, cudaStream_t st) {
    auto kern = k_sparse_decode_mma<DT>;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = allow_max_smem(kern)) != cudaSuccess) return e;
    if (P.part_floats < (long long)sms * B * P.d) return cudaErrorInvalidValue;
    void* args[] = {&P, &B};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms, 1, 1);  // one CTA per SM; the cooperative launch guarantees co-residency
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)mma_layout(P.R, P.d).total;
    cfg.stream = st;
    return launch_coop(reinterpret_cast<const void*>(kern), cfg, args);
}

cudaError_t launch_sparse_decode(SparseDecodeParams P, int B, cudaStream_t st) {
    const bool wide = P.d > 2048;
    // B > 1 at d = 1024 or 2048: the tensor-core kernel (wider d would not
    // keep its x fragments and partial sums in the registers of a 9-warp CTA)
    if (B >= 2 && B <= 8 && (P.d == 1024 || P.d == 2048)) {
        SparseDecodeParams P2 = P;
        P2.R = sparse_decode_mma_stages(P.d);
        if (P2.R >= kMmaBatch) return P.d == 1024 ? launch_sd_mma<8>(P2, B, st) : launch_sd_mma<16>(P2, B, st);
    }
    if (B == 1 && P.pmask == nullptr && (P.n_dev == nullptr || P.stable_plan)) {
        // the overwrite form with a partial buffer: the cluster reduction
        // (its static shared memory, a float4 per thread, comes out of the ring)
        if (!P.accumulate && P.part && P.tickets) {
            const int Rc = sparse_decode_b1_stages(P.d, (int)sizeof(float4) * kDecThreads + 64);
            if (Rc >= kConsWarps) {
                SparseDecodeParams P1 = P;
                P1.R = Rc;
                return wide ? launch_sd1_cr<2>(P1, st) : launch_sd1_cr<1>(P1, st);
            }
        }
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
    const int rows = P.rows ? P.n_rows : P.N;
    if (rows < 1) return cudaErrorInvalidValue;
    const int grid = rows < sms ? rows : sms;
    void* args[] = {&P};
    if (P.d > 2048) {
        if ((e = allow_max_smem(k_dense_act<2>)) != cudaSuccess) return e;
        return launch_clustered(k_dense_act<2>, grid, 1, smem, st, args, /*pdl=*/true);
    }
    if ((e = allow_max_smem(k_dense_act<1>)) != cudaSuccess) return e;
    return launch_clustered(k_dense_act<1>, grid, 1, smem, st, args, /*pdl=*/true);
}

// Bytes of the tiered kernel's ring: what is left of the shared memory after
// the barriers and the activation buffer, the CTA sum of y (4d bytes) at its
// end. 0 when a stream's share cannot hold one record of either kind, or the
// ring the streams' partials and the CTA sum.
int tiered_down_ring(int d, int aux_floats, int rec_bytes) {
    // the kernel's static shared memory (tier histograms, reduction scratch)
    // takes about 21 KB of the 227 KB
    constexpr int kTieredBudget = 227 * 1024 - 24 * 1024;
    const int bytes = (kTieredBudget - td_off_ring(aux_floats)) / 1024 * 1024;
    const int RP = ((bytes - 4 * d) / kTdPairs) / 128 * 128;
    return (RP >= 2 * d && RP >= rec_bytes && bytes >= (4 * kTdPairs + 4) * d) ? bytes : 0;
}

template <int MAXC, int BITS, bool FULL>
cudaError_t launch_tiered(TieredDownParams& P, size_t smem, cudaStream_t st) {
    auto kern = k_tiered_down<MAXC, BITS, FULL>;
    int grid = 0, cluster = 0;
    cudaError_t e = cached_grid(kern, smem, &grid, &cluster, kTdThreads);
    if (e != cudaSuccess) return e;
    if (P.part_floats < (long long)(grid / cluster) * P.d) return cudaErrorInvalidValue;
    // per-CTA record counts (rank windows, or an own range of N / grid
    // columns) must fit the activation buffer (activations in the first half
    // of the buffer, columns in the second)
    long long per = (long long)(P.k_top + grid - 1) / grid + (P.k_mid + grid - 1) / grid;
    const long long own = ((long long)P.N + grid - 1) / grid;
    if (own > per) per = own;
    if (2 * per > P.aux_floats) return cudaErrorInvalidValue;
    void* args[] = {&P};
    return launch_clustered(kern, grid, cluster, smem, st, args, /*pdl=*/true, kTdThreads);
}

cudaError_t launch_tiered_down(TieredDownParams P, cudaStream_t st) {
    const size_t smem = (size_t)td_off_ring(P.aux_floats) + (size_t)P.ring_bytes;
    // d = 2048 or 4096: every lane's chunks exist, no bounds checks
    const bool wide = P.d > 2048, full = P.d == 2048 || P.d == 4096;
#define SI_TIERED_CASE(B)                                                                  \
    case B:                                                                                \
        if (full) return wide ? launch_tiered<2, B, true>(P, smem, st) : launch_tiered<1, B, true>(P, smem, st); \
        return wide ? launch_tiered<2, B, false>(P, smem, st) : launch_tiered<1, B, false>(P, smem, st);
    switch (P.bits) {
        SI_TIERED_CASE(2)
        SI_TIERED_CASE(3)
        SI_TIERED_CASE(4)
        SI_TIERED_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef SI_TIERED_CASE
}

cudaError_t launch_abs_hist(const float* a, int N, unsigned* hist, int32_t* slab, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int grid = (N + 2047) / 2048;
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_abs_hist, a, N, hist, slab);
}

int streaming_grid_upper_bound() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace si
