// Warp-level exact top-k of up to a few hundred 32-bit order keys: the k-th
// largest key by four 8-bit radix passes over a per-warp shared-memory
// histogram, then the selection written in ascending position order (every
// key above the k-th, and of the keys equal to it the lowest positions until
// k are taken). Used by the dense-row select.
#pragma once

#include "mita_internal.cuh"

namespace mita {

// 32-bit order key of a raw landmark logit: larger tau * raw first (the
// score bits of topk_key; ties are broken by position in warp_take).
__device__ __forceinline__ uint32_t score_key32(float raw) {
    return static_cast<uint32_t>(topk_key(raw * 0.125f, 0u) >> 32);
}

// k-th largest of `cnt` keys get(e) (e < cnt) by four 8-bit radix passes;
// returns it and sets *remaining to how many keys equal to it belong to the
// k largest (warp-uniform results).
template <class Get>
__device__ __forceinline__ uint32_t warp_radix_kth(int cnt, unsigned k, unsigned* hist, Get get,
                                                   unsigned* remaining_out) {
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0, mask = 0;
    unsigned remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = lane; b < 256; b += 32) hist[b] = 0;
        __syncwarp();
        for (int e = lane; e < cnt; e += 32) {
            const uint32_t x = get(e);
            if ((x & mask) == prefix) atomicAdd(&hist[(x >> shift) & 255u], 1u);
        }
        __syncwarp();
        // lane l holds bins 255-8l .. 248-8l (descending digits)
        unsigned c[8], tot = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            c[t] = hist[255 - 8 * lane - t];
            tot += c[t];
        }
        unsigned incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned excl = incl - tot;
        const bool mine = excl < remaining && remaining <= incl;
        int digit = 0;
        unsigned above = 0;
        if (mine) {
            unsigned run = excl;
            for (int t = 0; t < 8; ++t) {
                if (run + c[t] >= remaining) {
                    digit = 255 - 8 * lane - t;
                    above = run;
                    break;
                }
                run += c[t];
            }
        }
        const int src_lane = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
        digit = __shfl_sync(0xffffffffu, digit, src_lane);
        above = __shfl_sync(0xffffffffu, above, src_lane);
        remaining -= above;
        prefix |= static_cast<uint32_t>(digit) << shift;
        mask |= 0xFFu << shift;
        __syncwarp();
    }
    *remaining_out = remaining;
    return prefix;
}

// Calls put(r, idx(e)) for the r-th (r = 0, 1, ...) in ascending order of
// position e < cnt of every key above kth and of the first `remaining` keys
// equal to it.
template <class Get, class Idx, class Put>
__device__ __forceinline__ void warp_take(int cnt, uint32_t kth, unsigned remaining, Get get, Idx idx, Put put) {
    const int lane = threadIdx.x & 31;
    const unsigned below = (1u << lane) - 1u;
    unsigned taken = 0, eq_seen = 0;
    for (int e0 = 0; e0 < cnt; e0 += 32) {
        const int e = e0 + lane;
        const uint32_t x = e < cnt ? get(e) : 0u;
        const bool gt = e < cnt && x > kth, eq = e < cnt && x == kth;
        const unsigned eqb = __ballot_sync(0xffffffffu, eq);
        const bool sel = gt || (eq && eq_seen + __popc(eqb & below) < remaining);
        const unsigned sb = __ballot_sync(0xffffffffu, sel);
        if (sel) put(static_cast<int>(taken + __popc(sb & below)), idx(e));
        taken += __popc(sb);
        eq_seen += __popc(eqb);
    }
}

}  // namespace mita
