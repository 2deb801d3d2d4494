// Which keys two routed experts share (s routed experts per query, tensor-core
// attention passes).
//
// With s > 1 a query attends to the union of its s experts' keys, each key
// once (the one softmax of "NeurIPS 2026 | Mixture-of-Top-k 注意力"
// (shuwu5.cn), section "MiTA：用少量地标查询，同时完成压缩与专家构造", taken over a
// set of keys). The pass of rank j skips the keys of its expert e that an
// earlier-ranked expert of the query already held; this table gives them as
// bit masks: ovl[bh][a][b][w] bit c is set iff key E_b[64 w + c] is also in
// E_a (the entry (a, a) is all ones; a query's experts are distinct, so it
// is never read).
//
// Membership in E_a is a lookup in a hash table of its keys in shared memory
// (open addressing, linear probing, at most half full: about 1.5 probes per
// lookup). One CTA per (head, expert a); its warps take the experts b in
// turn, the lanes 32 positions of E_b at a time (one ballot per 32).
#include "mita_internal.cuh"

namespace mita {

namespace {

constexpr int OT = 256;
constexpr int HT = 2 * MITA_MAX_K;  // hash slots (a power of two)
static_assert((HT & (HT - 1)) == 0, "HT must be a power of two");

__device__ __forceinline__ int slot_of(int key) {  // Fibonacci hashing
    return static_cast<int>((static_cast<uint32_t>(key) * 2654435769u) >> (32 - 11)) & (HT - 1);
}

__global__ void __launch_bounds__(OT) overlap_kernel(const int32_t* __restrict__ expert_idx, int m, int k, int nbw,
                                                     uint64_t* __restrict__ ovl) {
    __shared__ int tab[HT];  // keys of E_a (distinct, >= 0); -1: empty
    const int64_t bh = blockIdx.x / m;
    const int a = static_cast<int>(blockIdx.x % m);
    const int32_t* A = expert_idx + (bh * m + a) * static_cast<int64_t>(k);
    for (int x = threadIdx.x; x < HT; x += OT) tab[x] = -1;
    __syncthreads();
    for (int p = threadIdx.x; p < k; p += OT) {
        const int key = A[p];
        int x = slot_of(key);
        for (int it = 0; it < HT; ++it, x = (x + 1) & (HT - 1))  // k <= HT / 2: a free slot exists
            if (atomicCAS(&tab[x], -1, key) == -1) break;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* dst = ovl + (bh * m + a) * static_cast<int64_t>(m) * nbw;
    for (int b = warp; b < m; b += OT / 32) {
        const int32_t* Bl = expert_idx + (bh * m + b) * static_cast<int64_t>(k);
        for (int p0 = 0; p0 < k; p0 += 256) {  // 256 positions of E_b: 8 per lane, loaded together
            int key[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int p = p0 + 32 * u + lane;
                key[u] = p < k ? Bl[p] : 0;
            }
            uint32_t bits[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                bool in = false;
                if (p0 + 32 * u + lane < k) {
                    int x = slot_of(key[u]);
                    for (int it = 0; it < HT; ++it, x = (x + 1) & (HT - 1)) {
                        const int t = tab[x];
                        if (t == key[u]) in = true;
                        if (t == key[u] || t == -1) break;
                    }
                }
                bits[u] = __ballot_sync(0xffffffffu, in);
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) {  // lane x writes the 64-bit word of positions p0 + 64 x ..
                const int w = p0 / 64 + x;
                if (lane == x && w < nbw)
                    dst[b * nbw + w] = (static_cast<uint64_t>(bits[2 * x + 1]) << 32) | bits[2 * x];
            }
        }
    }
}

// The masks of one rank j >= 1, in grouping-slot order (the order the
// attention pass reads its queries): for slot x of head bh, with n the query
// there and e its j-th expert, word w is the OR over the query's earlier
// experts r_0 .. r_{j-1} of ovl[bh][r_i][e][w].
__global__ void __launch_bounds__(256) pass_mask_kernel(const int* __restrict__ perm, const int32_t* __restrict__ route,
                                                        const uint64_t* __restrict__ ovl, int64_t BH, int64_t N,
                                                        int m, int s, int j, int nbw, uint64_t* __restrict__ mask) {
    const int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (x >= BH * N) return;
    const int64_t bh = x / N;
    const int n = perm[x];
    const int32_t* r = route + (bh * N + n) * s;
    const int e = r[j];
    uint64_t* dst = mask + x * nbw;
    for (int w = 0; w < nbw; ++w) {
        uint64_t v = 0;
        for (int i = 0; i < j; ++i) v |= ovl[((bh * m + r[i]) * m + e) * static_cast<int64_t>(nbw) + w];
        dst[w] = v;
    }
}

}  // namespace

size_t pass_mask_bytes(const Shape& s) {
    const size_t nbw = static_cast<size_t>((s.k + 63) / 64);
    return static_cast<size_t>(s.s_route > 1 ? s.s_route - 1 : 0) * s.BH * s.N * nbw * sizeof(uint64_t);
}

size_t overlap_bytes(const Shape& s) {
    const size_t nbw = static_cast<size_t>((s.k + 63) / 64);
    return static_cast<size_t>(s.BH) * s.m * s.m * nbw * sizeof(uint64_t);
}

// The overlap table, then the masks of ranks 1 .. s-1 (after the grouping).
cudaError_t launch_overlap(const Plan& p, const Work& w, const int32_t* expert_idx, const int32_t* route,
                           cudaStream_t st) {
    const int nbw = (p.s.k + 63) / 64;
    overlap_kernel<<<static_cast<unsigned>(p.s.BH * p.s.m), OT, 0, st>>>(expert_idx, p.s.m, p.s.k, nbw, w.ovl);
    const int64_t slots = p.s.BH * p.s.N;
    for (int j = 1; j < p.s.s_route; ++j)
        pass_mask_kernel<<<static_cast<unsigned>((slots + 255) / 256), 256, 0, st>>>(
            w.perm + static_cast<size_t>(j) * slots, route, w.ovl, p.s.BH, p.s.N, p.s.m, p.s.s_route, j, nbw,
            w.mask + static_cast<size_t>(j - 1) * slots * nbw);
    return cudaGetLastError();
}

}  // namespace mita
