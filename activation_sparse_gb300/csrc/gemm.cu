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
// Tile: 256 tokens x 128 neurons, K in blocks of 64 (one 128-byte swizzle
// row). The gate rows and the up rows of the same 128 neurons are loaded side
// by side into one 256-row B tile, so one tcgen05.mma (M=128, N=256, K=16,
// bf16 in, fp32 accumulate) produces both projections for 128 tokens; two
// such MMAs (token rows 0..127 and 128..255) share each B tile, which halves
// the B traffic per flop. The two accumulators fill the 512 TMEM columns
// (per 128-token half: gate in 0..127, up in 128..255) and the epilogue reads
// matching gate/up columns of the same row with tcgen05.ld.
//
// Warp roles (192 threads): warp 0 lane 0 issues TMA loads into a 4-stage
// shared-memory ring; warp 1 owns TMEM and lane 0 issues the MMAs
// (tcgen05.commit releases a stage once its MMAs are done); warps 2..5 run
// the epilogue, warp w reading TMEM lanes 32*(w%4) .. +31. All waits are
// bounded; TMEM is always released.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace si {

namespace {

constexpr int BM = 128;       // token rows per MMA (MMA M)
constexpr int MT = 2;         // MMA row blocks per tile: 256 token rows
constexpr int BNN = 128;      // neurons per tile (gate + up -> MMA N = 256)
constexpr int BK = 64;        // K per stage (128 bytes of bf16)
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB per row block
constexpr int STAGE_A = MT * A_BYTES;         // 32 KB
constexpr int B_BYTES = 2 * BNN * BK * 2;     // 32 KB (gate tile then up tile)
constexpr int STAGE_BYTES = STAGE_A + B_BYTES;
constexpr int ACC_COLS = 2 * BNN;             // TMEM columns of one accumulator
constexpr int TMEM_COLS = MT * ACC_COLS;      // 512: all of TMEM
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int COLSUM_FLOATS = kEpiWarps * 32 * 33;

// shared-memory layout (offsets from a 1024-aligned base)
constexpr int OFF_A = 0;
constexpr int OFF_B = STAGES * STAGE_A;
constexpr int OFF_COLSUM = OFF_B + STAGES * B_BYTES;
constexpr int OFF_BAR = OFF_COLSUM + COLSUM_FLOATS * 4;
constexpr int OFF_TMEM_SLOT = OFF_BAR + (2 * STAGES + 1) * 8;
constexpr int SMEM_BYTES = OFF_TMEM_SLOT + 16 + 1024;  // + alignment slack

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9
// = 1), B bf16 (bits 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(2 * BNN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

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

#define SI_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                 "=r"(r[i + 6]), "=r"(r[i + 7])

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : SI_R8(0), SI_R8(8), SI_R8(16), SI_R8(24)
        : "r"(taddr));
}
#undef SI_R8

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Bounded wait used only to drain in-flight copies before exit; ignores the
// short-circuit so that a CTA never leaves with a TMA write pending.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const long long t0 = cycles();
    while (!mbar_try_wait(bar, parity)) {
        if (cycles() - t0 > kDrainLimitCycles) return;
    }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_act_gemm(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_g,
               const __grid_constant__ CUtensorMap map_u, ActGemmParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* empty = full + STAGES;
    uint64_t* accum = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM_SLOT);

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

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % STAGES;
                if (kb >= STAGES) mbar_wait(&empty[s], (uint32_t)((kb / STAGES - 1) & 1), P.err, kSiteGemm | kSiteEmpty);
                mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                uint8_t* a_dst = smem + OFF_A + s * STAGE_A;
                uint8_t* b_dst = smem + OFF_B + s * B_BYTES;
#pragma unroll
                for (int t = 0; t < MT; ++t) tma_load_2d(a_dst + t * A_BYTES, &map_x, kb * BK, m0 + t * BM, &full[s]);
                tma_load_2d(b_dst, &map_g, kb * BK, n0, &full[s]);
                tma_load_2d(b_dst + B_BYTES / 2, &map_u, kb * BK, n0, &full[s]);
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
                const uint32_t a_addr = smem_u32(smem + OFF_A + s * STAGE_A);
                const uint32_t b_addr = smem_u32(smem + OFF_B + s * B_BYTES);
                const uint64_t bdesc = sw128_desc(b_addr);
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const uint64_t adesc = sw128_desc(a_addr + (uint32_t)(t * A_BYTES));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // +32 bytes per K step of 16 bf16 inside the swizzled 128-byte row
                        tc_mma(tmem + (uint32_t)(t * ACC_COLS), adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k),
                               kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                }
                tc_commit(&empty[s]);
            }
            tc_commit(accum);
        }
        __syncwarp();
    } else {
        // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, one token row per
        // thread in each of the two 128-token halves
        const int q = warp & 3;
        mbar_wait(accum, 0u, P.err, kSiteGemm | kSiteAccum);
        tc_fence_after();
        float* cs = reinterpret_cast<float*>(smem + OFF_COLSUM) + (warp - 2) * 32 * 33;
        for (int t = 0; t < MT; ++t)
        for (int j0 = 0; j0 < BNN; j0 += 32) {
            const int row = m0 + t * BM + q * 32 + lane;
            const uint32_t tbase = tmem + (uint32_t)(t * ACC_COLS) + ((uint32_t)(q * 32) << 16);
            uint32_t g[32], u[32];
            tmem_ld32(tbase + (uint32_t)j0, g);
            tmem_ld32(tbase + (uint32_t)(BNN + j0), u);
            tmem_ld_wait();
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = fabsf(swiglu(__uint_as_float(g[e]), __uint_as_float(u[e])));
            if (P.mode == 0) {
                if (row < P.M) {
                    float* dst = P.out + (size_t)row * P.ldo + n0 + j0;
                    if (n0 + j0 + 32 <= P.Nvalid) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                    } else {
                        for (int e = 0; e < 32; ++e)
                            if (n0 + j0 + e < P.Nvalid) dst[e] = v[e];
                    }
                }
            } else {
                // column sums over this warp's 32 rows (rows past M are zero: TMA fills them)
#pragma unroll
                for (int e = 0; e < 32; ++e) cs[lane * 33 + e] = v[e];
                __syncwarp();
                float sum = 0.0f;
#pragma unroll 8
                for (int r2 = 0; r2 < 32; ++r2) sum += cs[r2 * 33 + lane];
                __syncwarp();
                const int col = n0 + j0 + lane;
                if (col < P.Nvalid) atomicAdd(P.colsum + col, sum);
            }
        }
        tc_fence_before();
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
// box 64 x 128, 128-byte swizzle, zero fill outside.
cudaError_t make_map(CUtensorMap* map, const void* base, long long cols, long long rows, long long stride_elems) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(stride_elems * 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_act_gemm(const ActGemmParams& P, cudaStream_t st) {
    if (P.K % BK || P.M < 1 || P.Nvalid < 1 || P.Nrows < 1) return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(P.X) | reinterpret_cast<uintptr_t>(P.Wgate) |
         reinterpret_cast<uintptr_t>(P.Wup)) & 15u)
        return cudaErrorMisalignedAddress;
    if ((P.w_stride * 2) % 16 || P.mode < 0 || P.mode > 1) return cudaErrorInvalidValue;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    CUtensorMap mx, mg, mu;
    if ((e = make_map(&mx, P.X, P.K, P.M, P.K)) != cudaSuccess) return e;
    if ((e = make_map(&mg, P.Wgate, P.K, P.Nrows, P.w_stride)) != cudaSuccess) return e;
    if ((e = make_map(&mu, P.Wup, P.K, P.Nrows, P.w_stride)) != cudaSuccess) return e;
    if ((e = allow_max_smem(k_act_gemm)) != cudaSuccess) return e;
    dim3 grid((P.Nvalid + BNN - 1) / BNN, (P.M + MT * BM - 1) / (MT * BM));
    if (grid.y > 65535) return cudaErrorInvalidValue;
    k_act_gemm<<<grid, kThreads, SMEM_BYTES, st>>>(mx, mg, mu, P);
    return cudaGetLastError();
}

}  // namespace si
