// Streaming top-k support for the landmark scan: candidate buffers with a
// running threshold, compacted by a warp-cooperative radix select.
//
// Each (head, key chunk, landmark) owns a buffer of `cap` 64-bit keys built by
// topk_key(): larger score first, then lower key index, so every key in a
// buffer is distinct and "the k largest keys" is exactly the routed expert's
// selection rule with ties going to the lower index. A score is appended only
// when its key beats the buffer's threshold (initially 0, below every real
// key). When a buffer would overflow, the owning warp selects its k largest
// keys in place and raises the threshold to the k-th largest: a later key
// below it can never enter this chunk's top k, because k kept keys beat it.
#pragma once

#include "mita_internal.cuh"

namespace mita {

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned r;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
    return r;
}

// k-th largest of the (distinct) keys buf[0..cnt) that match `prefix` under
// `mask` on the digits already fixed. Radix select, 8 bits per pass from the
// top, 256-bin histogram in `hist` (shared memory, one per warp). All 32
// lanes call it; every lane gets the result.
__device__ __forceinline__ uint64_t warp_kth_largest(const uint64_t* buf, int cnt, int kth, unsigned* hist) {
    const int lane = threadIdx.x & 31;
    uint64_t prefix = 0, mask = 0;
    unsigned remaining = static_cast<unsigned>(kth);
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int b = lane; b < 256; b += 32) hist[b] = 0;
        __syncwarp();
        for (int e = lane; e < cnt; e += 32) {
            const uint64_t x = buf[e];
            if ((x & mask) == prefix) atomicAdd(&hist[(x >> shift) & 255u], 1u);
        }
        __syncwarp();
        // lane L holds bins 255-8L .. 248-8L, i.e. descending digit order
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
        const unsigned who = __ballot_sync(0xffffffffu, mine);
        int digit = 0;
        unsigned above = 0;
        if (mine) {
            unsigned run = excl;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (run + c[t] >= remaining) {
                    digit = 255 - 8 * lane - t;
                    above = run;
                    break;
                }
                run += c[t];
            }
        }
        const int src = __ffs(who) - 1;
        digit = __shfl_sync(0xffffffffu, digit, src);
        above = __shfl_sync(0xffffffffu, above, src);
        remaining -= above;
        prefix |= static_cast<uint64_t>(digit) << shift;
        mask |= 0xFFull << shift;
        __syncwarp();
    }
    return prefix;
}

// Keeps the k largest keys of buf[0..cnt) (cnt >= k) in buf[0..k), in place.
// Returns the k-th largest key, the buffer's new threshold. Not inlined: it runs
// rarely, and inlined it would add its registers to its callers' hot loops.
static __device__ __noinline__ uint64_t warp_compact_topk(uint64_t* buf, int cnt, int k, unsigned* hist) {
    const int lane = threadIdx.x & 31;
    const uint64_t kth = warp_kth_largest(buf, cnt, k, hist);
    int out = 0;
    for (int base = 0; base < cnt; base += 32) {
        const int e = base + lane;
        const uint64_t x = e < cnt ? buf[e] : 0;
        const bool keep = e < cnt && x >= kth;
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        __syncwarp();  // this chunk is read before any lane overwrites it
        if (keep) buf[out + __popc(bal & lanemask_lt())] = x;
        out += __popc(bal);
        __syncwarp();
    }
    return kth;
}

// One 32-key step of a warp's candidate buffer: lane j offers `key` when
// `valid`. Appends the keys above the threshold, compacting first when the
// buffer would overflow (cap >= k + 32 guarantees room afterwards).
__device__ __forceinline__ void warp_offer(uint64_t* buf, int& cnt, uint64_t& theta, int cap, int k, bool valid,
                                           uint64_t key, unsigned* hist) {
    bool acc = valid && key > theta;
    unsigned bal = __ballot_sync(0xffffffffu, acc);
    if (bal == 0) return;
    if (cnt + __popc(bal) > cap) {
        __syncwarp();
        theta = warp_compact_topk(buf, cnt, k, hist);
        cnt = k;
        acc = valid && key > theta;
        bal = __ballot_sync(0xffffffffu, acc);
    }
    if (acc) buf[cnt + __popc(bal & lanemask_lt())] = key;
    cnt += __popc(bal);
    __syncwarp();
}

}  // namespace mita
