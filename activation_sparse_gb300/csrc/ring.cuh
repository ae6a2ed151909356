// ring.cuh -- the shared-memory ring of the streaming decode kernels: the
// warp roles, the layout of barriers / auxiliary space / x / stages, and the
// producer loop that streams records picked by an index list.
#pragma once

#include "common.cuh"

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

// Producer loop of the ring kernels whose records are picked by an index
// list (idx[0, cnt), each in [0, limit)): the warp loads the indices 32 at a
// time, with the next block's load in flight while this block is issued, and
// lane 0 issues record i into stage i % R once that stage's previous fill has
// been released. An index out of range is flagged and replaced by 0. Called
// by the whole producer warp.
// `ibase` is the ring index of the list's first record (a kernel that streams
// several lists through one ring numbers their records consecutively).
template <class IssueF>
__device__ __forceinline__ void produce_by_index(const int32_t* __restrict__ idx, int cnt, int limit, int R,
                                                 uint64_t* empty, unsigned* err, unsigned site, IssueF issue,
                                                 int ibase = 0) {
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
                const int i = ibase + base + k, s = i % R;
                if (i >= R) mbar_wait(&empty[s], (uint32_t)((i / R - 1) & 1), err, site);
                issue(i, s, pk);
            }
        }
    }
    __syncwarp();
}

}  // namespace si
