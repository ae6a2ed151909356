// pack.cu -- offline layout kernels.
//
//  k_pack_loaded   selective loading (SelectInfer section 4, Fig. 6): copy the
//                  gate row, up row and down column of every loaded neuron into
//                  one contiguous neuron-major record [3][d] (LeanStream's
//                  permutation-invariance argument: a SwiGLU FFN output is a
//                  sum over neurons, so the records can sit in any order; this
//                  library keeps ascending neuron index).
//  k_down_norms    ||Wd[:, n]||_2 per packed neuron, for the weight-aware
//                  salience |a_n| * ||Wd[:, n]||_2 (WiSparse abstract).
//  k_spax_encode   SpAx offline encoding (Fig. 2, Fig. 3): per column and
//                  per row group, float32 min / max / scale and 2-, 3-, 4-
//                  or 8-bit codes, plus a column-major bf16 copy of Wd so that a top-tier
//                  column is one contiguous read. A column's codes and its
//                  (scale, min) pairs form one record, so a middle-tier
//                  column is one contiguous read too.
#include "common.cuh"
#include "internal.h"

namespace si {

// One CTA per 32 packed positions; pad positions (>= n_loaded) become zeros.
__global__ void __launch_bounds__(256) k_pack_loaded(const uint16_t* __restrict__ Wg, const uint16_t* __restrict__ Wu,
                                                    const uint16_t* __restrict__ Wd, int d, int N,
                                                    const int32_t* __restrict__ loaded, int n_loaded,
                                                    uint16_t* __restrict__ packed) {
    __shared__ uint16_t tile[32][34];
    __shared__ int s_n[32];
    const int p0 = blockIdx.x * 32;
    if (threadIdx.x < 32) {
        const int p = p0 + threadIdx.x;
        s_n[threadIdx.x] = p < n_loaded ? loaded[p] : -1;
    }
    __syncthreads();
    const int chunks = d / 8;
    for (int idx = threadIdx.x; idx < 32 * 2 * chunks; idx += 256) {
        const int r = idx / (2 * chunks);
        const int rem = idx - r * 2 * chunks;
        const int which = rem / chunks;
        const int c = rem - which * chunks;
        const int n = s_n[r];
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n >= 0) v = reinterpret_cast<const uint4*>((which ? Wu : Wg) + (size_t)n * d)[c];
        reinterpret_cast<uint4*>(packed + ((size_t)(p0 + r) * 3 + which) * d)[c] = v;
    }
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int j0 = 0; j0 < d; j0 += 32) {
        const int n = s_n[tx];
        for (int jj = ty; jj < 32; jj += 8) tile[tx][jj] = (n >= 0) ? Wd[(size_t)(j0 + jj) * N + n] : (uint16_t)0;
        __syncthreads();
        for (int rr = ty; rr < 32; rr += 8) packed[((size_t)(p0 + rr) * 3 + 2) * d + j0 + tx] = tile[rr][tx];
        __syncthreads();
    }
}

// grid (ceil(N/32), d/group); block 256 = 8 warps, each warp owns 4 columns.
// Column n's record at recs + n * rec_bytes: d * BITS / 8 code bytes (element
// i at bit i * BITS, little-endian), then ngp (scale, min) float pairs.
// All quantisation arithmetic is float32 with explicit round-to-nearest
// intrinsics (no contraction), so codes are reproducible bit for bit.
template <int BITS>
__global__ void __launch_bounds__(256) k_spax_encode(const uint16_t* __restrict__ Wd, int d, int N, int group,
                                                    int ngp, uint16_t* __restrict__ WdT,
                                                    uint8_t* __restrict__ recs, int rec_bytes) {
    // codes per store unit: one byte (2-, 4-, 8-bit codes) or, for 3-bit
    // codes, eight codes in three bytes (a code may straddle two bytes)
    constexpr int EPU = BITS == 3 ? 8 : 8 / BITS;
    constexpr int QMAX = (1 << BITS) - 1;
    extern __shared__ __align__(16) uint16_t s_tile[];  // [group][33]
    const int n0 = blockIdx.x * 32;
    const int g = blockIdx.y;
    const int r0 = g * group;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int r = ty; r < group; r += 8) {
        const int n = n0 + tx;
        s_tile[r * 33 + tx] = (n < N) ? Wd[(size_t)(r0 + r) * N + n] : (uint16_t)0;
    }
    __syncthreads();
    for (int cc = ty; cc < 32; cc += 8) {
        const int n = n0 + cc;
        if (n >= N) break;  // warp-uniform
        float mn = INFINITY, mx = -INFINITY;
        for (int r = tx; r < group; r += 32) {
            const float w = __uint_as_float((uint32_t)s_tile[r * 33 + cc] << 16);
            mn = fminf(mn, w);
            mx = fmaxf(mx, w);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        }
        const float scale = __fdiv_rn(__fsub_rn(mx, mn), (float)QMAX);
        for (int r = EPU * tx; r < group; r += 32 * EPU) {
            uint32_t word = 0u;
#pragma unroll
            for (int h = 0; h < EPU; ++h) {
                const uint16_t hb = s_tile[(r + h) * 33 + cc];
                WdT[(size_t)n * d + r0 + r + h] = hb;
                const float w = __uint_as_float((uint32_t)hb << 16);
                int v = 0;
                if (scale != 0.0f) {
                    float t = __fdiv_rn(__fsub_rn(w, mn), scale);
                    t = __fadd_rn(t, 0.5f);
                    v = (int)floorf(t);
                    v = v < 0 ? 0 : (v > QMAX ? QMAX : v);
                }
                word |= (uint32_t)v << (h * BITS);
            }
            // element i at bit i * BITS of the column's little-endian stream
            uint8_t* dst = recs + (size_t)n * rec_bytes + (size_t)(r0 + r) * BITS / 8;
            dst[0] = (uint8_t)word;
            if constexpr (BITS == 3) {
                dst[1] = (uint8_t)(word >> 8);
                dst[2] = (uint8_t)(word >> 16);
            }
        }
        if (tx == 0) {
            float* prm = reinterpret_cast<float*>(recs + (size_t)n * rec_bytes + (size_t)d * BITS / 8);
            prm[g * 2 + 0] = scale;
            prm[g * 2 + 1] = mn;
        }
    }
}

// ||Wd[:, n]||_2 of each packed neuron, from its record's down column: one
// warp per position, lane-strided float32 squares summed in a fixed order
// (deterministic), then a butterfly; pad positions get 0.
__global__ void __launch_bounds__(256) k_down_norms(const uint16_t* __restrict__ packed, int d, int n_loaded,
                                                   int n_pad, float* __restrict__ norms) {
    const int p = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (p >= n_pad) return;
    float acc = 0.0f;
    if (p < n_loaded) {
        const uint16_t* col = packed + ((size_t)p * 3 + 2) * d;
        for (int j = lane; j < d; j += 32) {
            const float w = __uint_as_float((uint32_t)col[j] << 16);
            acc = fmaf(w, w, acc);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) norms[p] = sqrtf(acc);
}

cudaError_t launch_down_norms(const uint16_t* packed, int d, int n_loaded, int n_pad, float* norms, cudaStream_t st) {
    k_down_norms<<<(n_pad + 7) / 8, 256, 0, st>>>(packed, d, n_loaded, n_pad, norms);
    return cudaGetLastError();
}

cudaError_t launch_pack_loaded(const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, int d, int N,
                               const int32_t* loaded, int n_loaded, int n_pad, uint16_t* packed, cudaStream_t st) {
    k_pack_loaded<<<n_pad / 32, 256, 0, st>>>(Wg, Wu, Wd, d, N, loaded, n_loaded, packed);
    return cudaGetLastError();
}

cudaError_t launch_spax_encode(const uint16_t* Wd, int d, int N, int bits, int group, int ngp, uint16_t* WdT,
                               uint8_t* recs, int rec_bytes, cudaStream_t st) {
    const size_t smem = (size_t)group * 33 * 2;
    dim3 grid((N + 31) / 32, d / group);
    cudaError_t e;
    switch (bits) {
        case 2:
            if ((e = allow_max_smem(k_spax_encode<2>)) != cudaSuccess) return e;
            k_spax_encode<2><<<grid, 256, smem, st>>>(Wd, d, N, group, ngp, WdT, recs, rec_bytes);
            break;
        case 3:
            if ((e = allow_max_smem(k_spax_encode<3>)) != cudaSuccess) return e;
            k_spax_encode<3><<<grid, 256, smem, st>>>(Wd, d, N, group, ngp, WdT, recs, rec_bytes);
            break;
        case 4:
            if ((e = allow_max_smem(k_spax_encode<4>)) != cudaSuccess) return e;
            k_spax_encode<4><<<grid, 256, smem, st>>>(Wd, d, N, group, ngp, WdT, recs, rec_bytes);
            break;
        case 8:
            if ((e = allow_max_smem(k_spax_encode<8>)) != cudaSuccess) return e;
            k_spax_encode<8><<<grid, 256, smem, st>>>(Wd, d, N, group, ngp, WdT, recs, rec_bytes);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace si
