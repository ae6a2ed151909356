// gemm.cu -- activation GEMM on the 5th-generation tensor cores (tcgen05).
//
// Computes, for a block of token rows X[m, :] and a block of neurons p,
//     g = X[m] . Wgate[p],  u = X[m] . Wup[p],  a = silu(g) * u,
// the down_proj input of every (token, neuron) pair. It serves two steps:
//   mode 0  prefill activation pass of SelectInfer (section 5, Fig. 7):
//           writes |a| for every token and every loaded neuron;
//   mode 1  offline profiler score (section 3, Eq. (1)): adds
//           sum over tokens of |a| into a per-neuron score.
//
// Tile: 256 tokens x BNN neurons, K in blocks of 64 (one 128-byte swizzle
// row). BNN (64 .. 128, a multiple of 16) is picked per launch so that the
// grid fills the SMs: a 512-token prompt over 5734 loaded neurons gives 90
// tiles of 128 neurons (0.6 of the SMs busy) but 144 tiles of 80. The gate
// rows and the up rows of the same BNN neurons are loaded side by side into
// one 2*BNN-row B tile, so one tcgen05.mma (M=128, N=2*BNN, K=16, bf16 in,
// fp32 accumulate) produces both projections for 128 tokens; the two token
// halves share each B tile. Half t accumulates at TMEM columns 256*t (gate
// in the first BNN columns, up in the next BNN) and the epilogue reads
// matching gate/up columns of the same row with tcgen05.ld. One wide MMA
// rather than a gate MMA and an up MMA matters: each MMA reads its A tile
// from shared memory again, and at N = BNN that re-read would outrun the
// shared-memory bandwidth.
//
// Warp roles (320 threads): warp 0 lane 0 issues TMA loads into a 3- or
// 4-stage shared-memory ring; warp 1 owns TMEM and lane 0 issues the MMAs
// (tcgen05.commit releases a stage once its MMAs are done); warps 2..9 run
// the epilogue, warp w reading TMEM lanes 32*(w%4) .. +31 of token half
// (w-2)/4. All waits are bounded; TMEM is always released. Launched with
// programmatic dependent launch: barrier set-up, TMEM allocation and the
// tensor-map prefetch overlap the previous launch in the stream.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace si {

namespace {

constexpr int BM = 128;                       // token rows per MMA (MMA M)
constexpr int MT = 2;                         // MMA row blocks per tile: 256 token rows
constexpr int BK = 64;                        // K per stage (128 bytes of bf16)
constexpr int A_BYTES = BM * BK * 2;          // 16 KB per row block
constexpr int STAGE_A = MT * A_BYTES;         // 32 KB
constexpr int ACC_STRIDE = 256;               // TMEM columns per token half: gate at +0, up at +BNN
constexpr int TMEM_COLS = MT * ACC_STRIDE;    // 512: all of TMEM
constexpr int kEpiWarps = 8;                  // two per TMEM lane quarter: one per token half
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int COLSUM_FLOATS = kEpiWarps * 32 * 65;
constexpr int kStageOutBytes = 32 * 128 * 4;  // one warp's [32][BNN <= 128] fp32 output tile
static_assert(kEpiWarps == 4 * MT, "one epilogue warp per TMEM lane quarter and token half");
constexpr int kSmemLimit = 227 * 1024;

// Per neuron-tile width: shared-memory layout (offsets from a 1024-aligned
// base) and the instruction descriptor.
template <int BNN>
struct GemmCfg {
    static_assert(BNN % 16 == 0 && BNN >= 64 && BNN <= 128, "neuron tile: M = 128 MMAs need N % 16 == 0");
    static constexpr int B_BYTES = 2 * BNN * BK * 2;  // gate tile then up tile, each BNN 128-byte rows
    static constexpr int STAGE_BYTES = STAGE_A + B_BYTES;
    static constexpr int FIXED = (2 * 4 + 1) * 8 + 16 + 1024;  // barriers, TMEM slot, alignment slack
    static constexpr int STAGES = (kSmemLimit - FIXED) / STAGE_BYTES >= 4 ? 4 : 3;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = STAGES * STAGE_A;
    static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + (2 * STAGES + 1) * 8;
    static constexpr int SMEM_BYTES = OFF_TMEM_SLOT + 16 + 1024;
    static_assert(SMEM_BYTES <= kSmemLimit, "shared memory");
    static_assert(B_BYTES % 1024 == 0 && (BNN * 128) % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
    static_assert(COLSUM_FLOATS * 4 <= OFF_BAR && kEpiWarps * kStageOutBytes <= OFF_BAR,
                  "the output tiles and the column-sum scratch reuse the drained ring");
    // kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9 = 1), B bf16 (bits
    // 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
    // M >> 4 at bits 24-28. N = 2 * BNN: gate and up rows in one MMA.
    static constexpr uint32_t IDESC =
        (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(2 * BNN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
};

// Shared-memory matrix descriptor for a K-major tile written by TMA with
// 128-byte swizzle: start address >> 4 (bits 0-13), leading byte offset 16 B
// (unused for this layout, bits 16-29), stride byte offset 1024 B between
// 8-row groups (bits 32-45), descriptor version 1 (bits 46-47), swizzle mode
// 128B = 2 (bits 61-63). The tile base is 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Bounded wait used only to drain in-flight copies before exit; ignores the
// short-circuit so that a CTA never leaves with a TMA write pending.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const long long t0 = cycles();
    while (!mbar_try_wait(bar, parity)) {
        if (cycles() - t0 > kDrainLimitCycles) return;
    }
}

// 16 consecutive fp32 columns of this thread's TMEM lane into r[0..15].
__device__ __forceinline__ void tmem_ld16p(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// |silu(g) * u| for the prefill activations. The sigmoid's division uses the
// fast reciprocal (__fdividef, a few ulp): the epilogue is ALU-bound at
// BNN values per thread, and |A| only ranks neurons (tolerance 1e-3 of the
// largest value against the float64 definition). A denominator past 2^126
// (g < -87) gives 0, which is silu's limit there.
__device__ __forceinline__ float abs_act(float g, float u) {
    return fabsf(__fdividef(g * u, 1.0f + __expf(-g)));
}

// One epilogue group: NC (a multiple of 16, at most 64) columns of gate (at
// TMEM column tg + j0) and up (tg + BNN + j0) for this thread's token row,
// loaded with one wait, turned into |silu(g) * u| and either staged in shared
// memory (mode 0: row `lane` of the warp's [32][BNN] fp32 tile, stored by one
// TMA copy afterwards) or summed over the warp's 32 rows into per-neuron
// scores (mode 1, through the [32][NC+1] scratch cs).
template <int NC, int BNN>
__device__ __forceinline__ void epi_group(const ActGemmParams& P, uint32_t tg, int j0, int col0, float* stage,
                                          float* cs, int lane) {
    static_assert(NC % 16 == 0 && NC <= 64, "group width");
    uint32_t g[NC], u[NC];
#pragma unroll
    for (int c = 0; c < NC; c += 16) {
        tmem_ld16p(tg + (uint32_t)(j0 + c), g + c);
        tmem_ld16p(tg + (uint32_t)(BNN + j0 + c), u + c);
    }
    tmem_ld_wait();
    float v[NC];
#pragma unroll
    for (int e = 0; e < NC; ++e) v[e] = abs_act(__uint_as_float(g[e]), __uint_as_float(u[e]));
    if (P.wnorm) {
        // weight-aware salience |a| * ||Wd[:, n]||_2 (columns past Nvalid are clipped by the store)
#pragma unroll
        for (int e = 0; e < NC; ++e) v[e] *= (col0 + e < P.Nvalid) ? __ldg(P.wnorm + col0 + e) : 0.0f;
    }
    if (P.mode == 0) {
        float* dst = stage + lane * BNN + j0;
#pragma unroll
        for (int e = 0; e < NC; e += 4)
            *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    } else {
        // column sums over this warp's 32 rows (rows past M are zero: TMA fills them)
#pragma unroll
        for (int e = 0; e < NC; ++e) cs[lane * (NC + 1) + e] = v[e];
        __syncwarp();
#pragma unroll
        for (int c = lane; c < NC; c += 32) {
            float sum = 0.0f;
#pragma unroll 8
            for (int r2 = 0; r2 < 32; ++r2) sum += cs[r2 * (NC + 1) + c];
            if (col0 + c < P.Nvalid) atomicAdd(P.colsum + col0 + c, sum);
        }
        __syncwarp();
    }
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}

}  // namespace

template <int BNN>
__global__ void __launch_bounds__(kThreads, 1)
    k_act_gemm(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_g,
               const __grid_constant__ CUtensorMap map_u, const __grid_constant__ CUtensorMap map_o,
               ActGemmParams P) {
    using C = GemmCfg<BNN>;
    constexpr int STAGES = C::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + STAGES;
    uint64_t* accum = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BNN;
    const int m0 = blockIdx.y * (MT * BM);
    const int KB = P.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
        fence_mbar_init();
    } else if (threadIdx.x == 32) {
        // fetch the descriptors the first copies need while the barriers are set up
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_x)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_g)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_u)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The set-up above overlaps the previous launch's tail; X, the weights
    // and the outputs may belong to that launch, so every thread waits for
    // it before touching global memory, and lets the next launch begin
    // scheduling.
    grid_launch_dependents();
    grid_dependency_wait();

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % STAGES;
                if (kb >= STAGES) mbar_wait(&empty[s], (uint32_t)((kb / STAGES - 1) & 1), P.err, kSiteGemm | kSiteEmpty);
                mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                uint8_t* a_dst = smem + C::OFF_A + s * STAGE_A;
                uint8_t* b_dst = smem + C::OFF_B + s * C::B_BYTES;
#pragma unroll
                for (int t = 0; t < MT; ++t) tma_load_2d(a_dst + t * A_BYTES, &map_x, kb * BK, m0 + t * BM, &full[s]);
                tma_load_2d(b_dst, &map_g, kb * BK, n0, &full[s]);
                tma_load_2d(b_dst + C::B_BYTES / 2, &map_u, kb * BK, n0, &full[s]);
            }
            // every issued copy has landed before this CTA may exit
            for (int s = 0; s < STAGES && s < KB; ++s) {
                const int fills = (KB - s + STAGES - 1) / STAGES;
                mbar_drain(&full[s], (uint32_t)((fills - 1) & 1));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % STAGES;
                mbar_wait(&full[s], (uint32_t)((kb / STAGES) & 1), P.err, kSiteGemm | kSiteFull);
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + C::OFF_A + s * STAGE_A);
                const uint32_t b_addr = smem_u32(smem + C::OFF_B + s * C::B_BYTES);
                const uint64_t bdesc = sw128_desc(b_addr);
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const uint64_t adesc = sw128_desc(a_addr + (uint32_t)(t * A_BYTES));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // +32 bytes per K step of 16 bf16 inside the swizzled 128-byte row
                        tc_mma(tmem + (uint32_t)(t * ACC_STRIDE), adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k),
                               C::IDESC, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                }
                tc_commit(&empty[s]);
            }
            tc_commit(accum);
        }
        __syncwarp();
    } else {
        // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 of token half
        // (w-2)/4, one token row per thread
        const int q = warp & 3;
        const int t = (warp - 2) >> 2;
        mbar_wait(accum, 0u, P.err, kSiteGemm | kSiteAccum);
        tc_fence_after();
        // every MMA has completed, so every copy into the ring has landed
        // and the ring is free for the output tiles and column-sum scratch
        float* stage = reinterpret_cast<float*>(smem + C::OFF_A + (warp - 2) * kStageOutBytes);
        float* cs = reinterpret_cast<float*>(smem + C::OFF_A) + (warp - 2) * 32 * 65;
        const int row0 = m0 + t * BM + q * 32;
        const uint32_t tg = tmem + (uint32_t)(t * ACC_STRIDE) + ((uint32_t)(q * 32) << 16);
        // groups of 64 columns, then the remainder (16, 32 or 48)
        epi_group<64, BNN>(P, tg, 0, n0, stage, cs, lane);
        if constexpr (BNN >= 128) epi_group<64, BNN>(P, tg, 64, n0 + 64, stage, cs, lane);
        if constexpr (BNN > 64 && BNN < 128) epi_group<BNN - 64, BNN>(P, tg, 64, n0 + 64, stage, cs, lane);
        tc_fence_before();
        if (P.mode == 0 && row0 < P.M) {
            // the tile's 32 rows x BNN columns in one TMA store; the tensor
            // map clips rows past M and columns past Nvalid
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&map_o, stage, n0, row0);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                // the CTA may leave once the tile has been read out of shared
                // memory; the global writes complete with the grid
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            }
            __syncwarp();
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ------------------------------------------------------------------ host

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

cudaError_t get_encoder() {
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (g_encode) return cudaSuccess;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// 2-D bf16 map over rows of `cols` elements, row stride `stride_elems`,
// box 64 x box_rows, 128-byte swizzle, zero fill outside.
cudaError_t make_map(CUtensorMap* map, const void* base, long long cols, long long rows, long long stride_elems,
                     int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(stride_elems * 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D fp32 map for the |A| output: `cols` x `rows`, row stride `ld`
// elements, box BNN x 32 (one epilogue warp's tile), no swizzle.
cudaError_t make_out_map(CUtensorMap* map, float* base, long long cols, long long rows, long long ld, int box_cols) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 4)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, 32u};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

std::atomic<int> g_forced_bnn{0};

// Neuron-tile width for a launch: the fewest waves of the widest useful
// tile. A CTA's time grows with its width plus a fixed share for the token
// rows it loads (about 24 neurons' worth), so among 128, 112, 96, 80 and 64
// the width with the smallest waves * (width + 24) wins, the wider on ties.
int pick_bnn(int nvalid, int mtiles, int sms) {
    const int forced = g_forced_bnn.load(std::memory_order_relaxed);
    if (forced) return forced;
    static const int cand[] = {128, 112, 96, 80, 64};
    int best = 128;
    long long best_cost = -1;
    for (int c : cand) {
        const long long ctas = (long long)((nvalid + c - 1) / c) * mtiles;
        const long long waves = (ctas + sms - 1) / sms;
        const long long cost = waves * (c + 24);
        if (best_cost < 0 || cost < best_cost) {
            best = c;
            best_cost = cost;
        }
    }
    return best;
}

template <int BNN>
cudaError_t launch_tile(const CUtensorMap& mx, const ActGemmParams& P, int mtiles, cudaStream_t st) {
    CUtensorMap mg, mu, mo;
    cudaError_t e;
    if ((e = make_map(&mg, P.Wgate, P.K, P.Nrows, P.w_stride, BNN)) != cudaSuccess) return e;
    if ((e = make_map(&mu, P.Wup, P.K, P.Nrows, P.w_stride, BNN)) != cudaSuccess) return e;
    memset(&mo, 0, sizeof(mo));  // mode 1 writes no |A|
    if (P.mode == 0 && (e = make_out_map(&mo, P.out, P.Nvalid, P.M, P.ldo, BNN)) != cudaSuccess) return e;
    if ((e = allow_max_smem(k_act_gemm<BNN>)) != cudaSuccess) return e;
    // programmatic dependent launch: this grid's set-up overlaps the tail of
    // the previous launch in the stream (the kernel waits before any access)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((P.Nvalid + BNN - 1) / BNN, mtiles, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = GemmCfg<BNN>::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_act_gemm<BNN>, mx, mg, mu, mo, P);
}

}  // namespace

cudaError_t set_gemm_tile(int bnn) {
    if (bnn != 0 && bnn != 64 && bnn != 80 && bnn != 96 && bnn != 112 && bnn != 128) return cudaErrorInvalidValue;
    g_forced_bnn.store(bnn, std::memory_order_relaxed);
    return cudaSuccess;
}

int gemm_tile_for(int M, int Nvalid) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) return 0;
    return pick_bnn(Nvalid, (M + MT * BM - 1) / (MT * BM), sms);
}

cudaError_t launch_act_gemm(const ActGemmParams& P, cudaStream_t st) {
    if (P.K % BK || P.M < 1 || P.Nvalid < 1 || P.Nrows < 1) return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(P.X) | reinterpret_cast<uintptr_t>(P.Wgate) |
         reinterpret_cast<uintptr_t>(P.Wup)) & 15u)
        return cudaErrorMisalignedAddress;
    if ((P.w_stride * 2) % 16 || P.mode < 0 || P.mode > 1) return cudaErrorInvalidValue;
    // the |A| tile goes out by TMA: 16-byte aligned base and row stride
    if (P.mode == 0 && ((reinterpret_cast<uintptr_t>(P.out) & 15u) || P.ldo % 4 || P.ldo < P.Nvalid))
        return cudaErrorMisalignedAddress;
    const long long mtiles = (P.M + MT * BM - 1) / (MT * BM);
    if (mtiles > 65535) return cudaErrorInvalidValue;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    CUtensorMap mx;
    if ((e = make_map(&mx, P.X, P.K, P.M, P.K, BM)) != cudaSuccess) return e;
    switch (pick_bnn(P.Nvalid, (int)mtiles, sms)) {
        case 64: return launch_tile<64>(mx, P, (int)mtiles, st);
        case 80: return launch_tile<80>(mx, P, (int)mtiles, st);
        case 96: return launch_tile<96>(mx, P, (int)mtiles, st);
        case 112: return launch_tile<112>(mx, P, (int)mtiles, st);
        default: return launch_tile<128>(mx, P, (int)mtiles, st);
    }
}

}  // namespace si
