// Stage 4: query-expert attention on the tensor cores (tcgen05, TMEM).
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造", and Figure 3 / Algorithm 1 of
// "And attention is also FFN? …" (en.roboind.com): a query routed to expert e
// attends to the m shared pairs (keys Lq_i, values LV_i) and the k routed pairs
// (K_j, V_j, j in E_e) under one softmax over all m+k logits; the page's
// implementation groups queries by expert and combines by online softmax.
//
// Persistent CTAs walk a contiguous range of the flat, expert-ordered item
// list (<= 128 queries of one expert per item), in rounds of up to two items
// of the same expert, one per row warpgroup. The expert's key list
// [Lq_0..Lq_{m-1}, K_e] and value list [LV_0..LV_{m-1}, V_e] (bf16, 128-byte
// swizzled rows, zero padded to whole 64-row blocks) stay in shared memory
// while consecutive rounds share the expert.
//   warp 0:         producer: gathers the key/value lists when the expert
//                   changes (the shared rows only when the head changes) and
//                   each item's query rows (through the grouping permutation),
//                   all with cp.async;
//   warps 1, 2 (lane 0): one MMA issuer per warpgroup: per 64-key block j of its
//                   item, S = Q keys_j^T into one of two TMEM buffers, and one
//                   block later O += P_j values_j into the warpgroup's TMEM
//                   accumulator;
//   warps 3-6, 7-10: one warpgroup per item (4 consecutive warps cover the 4
//                   TMEM lane quarters), one thread per query row: load the
//                   64 logits, update the running max (kept while it grows by
//                   < 2^8, so O rarely needs rescaling), p = 2^(s tau log2e -
//                   max) in registers, P (bf16) into shared memory once the
//                   previous block's P.V is done; at the end O / rowsum ->
//                   bf16 -> the query's row. Query rows are double-buffered, so
//                   the producer gathers the next item while this one runs.
// Handshakes are mbarriers, each completed exactly once per event its waiter
// consumes; row threads arrive individually (128-arrival barriers) and make
// their waits warp-uniform, so no named barrier can block forever. Every
// wait is bounded (umma.cuh).
#include "umma.cuh"

namespace mita {

namespace {

using namespace umma;

constexpr float kC = 0.125f * kLog2e;  // tau * log2(e), tau = 1/sqrt(64)
constexpr float kLazy = 8.0f;          // keep the running max while the new one is within 2^8
constexpr int KB = 64;                 // keys per block
constexpr int NWG = 3;                 // row warpgroups
constexpr int QB = 1;                  // query-row buffers per warpgroup
constexpr int SB = 1;                  // TMEM score buffers per warpgroup
constexpr int NT = 32 * (1 + NWG) + NWG * 128;  // producer, one issuer warp per group, rows
constexpr uint32_t kTStride = (SB + 1) * 64;    // TMEM columns per warpgroup: SB x S, then O
static_assert(NWG * kTStride <= 512, "TMEM holds 512 columns");
constexpr uint32_t kIdescS = idesc_bf16(128, KB, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 64, true);

struct Args {
    const __nv_bfloat16* Q;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    const __nv_bfloat16* lqhi;
    const __nv_bfloat16* lvbf;
    const int4* items;
    const int* nitems;
    const int* perm;
    const int32_t* expert_idx;
    __nv_bfloat16* out;
    int* status;
    int64_t N;
    int m, k, nblk;
};

struct Layout {
    uint8_t* keys;  // nblk * 8 KB
    uint8_t* vals;  // nblk * 8 KB
    uint8_t* q;     // [NWG][QB] * 16 KB: query rows
    uint8_t* p;     // [NWG] * 16 KB: P of the current block
};

__device__ __forceinline__ Layout layout(uint8_t* base, int nblk) {
    Layout L;
    L.keys = base;
    L.vals = L.keys + nblk * 8192;
    L.q = L.vals + nblk * 8192;
    L.p = L.q + NWG * QB * 16384;
    return L;
}

// The round starting at item r of [r, i1): up to NWG consecutive items of
// the same expert, one per warpgroup.
__device__ __forceinline__ int round_size(const Args& a, int r, int i1, int4* it) {
    it[0] = a.items[r];
    int n = 1;
    while (n < NWG && r + n < i1) {
        const int4 x = a.items[r + n];
        if (x.x != it[0].x || x.w != it[0].w) break;
        it[n++] = x;
    }
    return n;
}

__device__ __forceinline__ void zero16(uint8_t* p) { *reinterpret_cast<uint4*>(p) = make_uint4(0, 0, 0, 0); }

__global__ void __launch_bounds__(NT, 1) expert_tc_kernel(Args a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t kvfull, kvfree, qfull[NWG * QB], qfree[NWG * QB], ofree[NWG];
    __shared__ uint64_t sfull[NWG * SB], sfree[NWG * SB], pfull[NWG], pvdone[NWG];
    __shared__ uint32_t tmem_base;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Layout S = layout(base, a.nblk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nkeys = a.m + a.k;

    if (tid == 0) {
        mbar_init(&kvfull, 1);
        mbar_init(&kvfree, NWG);  // one commit per MMA issuer
        for (int w = 0; w < NWG; ++w) {
            mbar_init(&ofree[w], 128);
            mbar_init(&pfull[w], 128);
            mbar_init(&pvdone[w], 1);
        }
        for (int b = 0; b < NWG * QB; ++b) {
            mbar_init(&qfull[b], 1);
            mbar_init(&qfree[b], 1);
        }
        for (int b = 0; b < NWG * SB; ++b) {
            mbar_init(&sfull[b], 1);
            mbar_init(&sfree[b], 128);
        }
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;

    const int total = *a.nitems;
    const int i0 = static_cast<int>(static_cast<int64_t>(total) * blockIdx.x / gridDim.x);
    const int i1 = static_cast<int>(static_cast<int64_t>(total) * (blockIdx.x + 1) / gridDim.x);

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        int64_t cur_bh = -1;
        int cur_e = -1, changes = 0;
        uint32_t nq[NWG] = {};
        bool ok = true;
        for (int r = i0; r < i1 && ok;) {
            int4 it[NWG];
            const int cnt = round_size(a, r, i1, it);
            if (it[0].w != cur_bh || it[0].x != cur_e) {
                // wait until the MMAs reading the previous lists are done
                if (changes > 0) ok = __all_sync(0xffffffffu, mbar_wait(&kvfree, (changes - 1) & 1, a.status));
                if (!ok) break;
                const int64_t bh = it[0].w;
                const int32_t* sel = a.expert_idx + (bh * a.m + it[0].x) * static_cast<int64_t>(a.k);
                const int r0 = (it[0].w != cur_bh) ? 0 : a.m;  // shared rows only on a new head
                const uint32_t kb = smem_u32(S.keys), vb = smem_u32(S.vals);
                // lane l stages rows r0 + l, r0 + l + 32, ...: the row indices of a
                // batch of 8 rows are loaded first, then all of their copies issued
                const int rows = a.nblk * KB;
                for (int rb = r0; rb < rows; rb += 32 * 8) {
                    int64_t src[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int row = rb + u * 32 + lane;
                        src[u] = -1;
                        if (row < a.m) src[u] = (bh * a.m + row) * D;
                        else if (row < nkeys) src[u] = (bh * a.N + sel[row - a.m]) * D;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int row = rb + u * 32 + lane;
                        if (row >= rows) continue;
                        const __nv_bfloat16* ks = row < a.m ? a.lqhi : a.K;
                        const __nv_bfloat16* vs = row < a.m ? a.lvbf : a.V;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint32_t off = swz128(row, c);
                            if (src[u] >= 0) {
                                cp_async16(kb + off, ks + src[u] + c * 8);
                                cp_async16(vb + off, vs + src[u] + c * 8);
                            } else {
                                zero16(S.keys + off);
                                zero16(S.vals + off);
                            }
                        }
                    }
                }
                cp_async_wait_all();
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&kvfull);
                cur_bh = it[0].w;
                cur_e = it[0].x;
                ++changes;
            }
            for (int w = 0; w < cnt && ok; ++w) {
                // this Q buffer of the warpgroup was last used QB items back
                const uint32_t qb = w * QB + (nq[w] % QB);
                if (nq[w] >= QB)
                    ok = __all_sync(0xffffffffu, mbar_wait(&qfree[qb], ((nq[w] / QB) - 1) & 1, a.status));
                if (!ok) break;
                const int64_t bh = it[w].w;
                const uint32_t qa = smem_u32(S.q + qb * 16384);
                // lane l gathers rows l, l+32, l+64, l+96: indices first, then copies
                int n[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int row = u * 32 + lane;
                    n[u] = row < it[w].z ? a.perm[bh * a.N + it[w].y + row] : -1;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int row = u * 32 + lane;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        if (n[u] >= 0)
                            cp_async16(qa + swz128(row, c), a.Q + (bh * a.N + n[u]) * D + c * 8);
                        else
                            zero16(S.q + qb * 16384 + swz128(row, c));
                    }
                }
                cp_async_wait_all();
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&qfull[qb]);
                ++nq[w];
            }
            r += cnt;
        }
    } else if (warp <= NWG) {
        // ---------------- MMA issuers: lane 0 of warp 1 + w serves warpgroup w ----------------
        // (each issuer has a warp of its own: tcgen05.mma is a single-thread instruction)
        if (lane == 0) {
            const int w = warp - 1;
            int64_t cur_bh = -1;
            int cur_e = -1, changes = 0;
            uint32_t nq = 0, gb = 0;
            const uint32_t ka = smem_u32(S.keys), va = smem_u32(S.vals);
            const uint32_t pa = smem_u32(S.p + w * 16384);
            const uint32_t tO = tb + w * kTStride + SB * 64;
            bool ok = true;
            for (int r = i0; r < i1 && ok;) {
                int4 it[NWG];
                const int cnt = round_size(a, r, i1, it);
                if (it[0].w != cur_bh || it[0].x != cur_e) {
                    if (!mbar_wait(&kvfull, changes & 1, a.status)) break;
                    cur_bh = it[0].w;
                    cur_e = it[0].x;
                    ++changes;
                }
                r += cnt;
                if (w < cnt) {
                    const uint32_t qb = w * QB + (nq % QB);
                    if (!mbar_wait(&qfull[qb], (nq / QB) & 1, a.status)) break;
                    tc_fence_after();
                    const uint32_t qa = smem_u32(S.q + qb * 16384);
                    // S for block j, then P.V for block j-1
                    for (int j = 0; j <= a.nblk && ok; ++j) {
                        if (j < a.nblk) {
                            const uint32_t g = gb + j, sb = g % SB;
                            if (g >= SB) {  // the rows have read this S buffer (block g - SB)
                                ok = mbar_wait(&sfree[w * SB + sb], ((g / SB) - 1) & 1, a.status);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            const uint32_t tS = tb + w * kTStride + sb * KB;
#pragma unroll
                            for (int s = 0; s < 4; ++s)
                                mma_ss(tS, sdesc_sw128(qa + s * 32), sdesc_sw128(ka + j * 8192 + s * 32), kIdescS,
                                       s > 0);
                            mma_commit(&sfull[w * SB + sb]);
                            if (j == a.nblk - 1) mma_commit(&qfree[qb]);
                        }
                        if (j > 0) {
                            const uint32_t g = gb + j - 1;
                            // the first P.V of an item overwrites O: the previous
                            // item's epilogue must have read it
                            if (j == 1 && nq > 0) ok = mbar_wait(&ofree[w], (nq - 1) & 1, a.status);
                            if (ok) ok = mbar_wait(&pfull[w], g & 1, a.status);
                            if (!ok) break;
                            tc_fence_after();
#pragma unroll
                            for (int s = 0; s < 4; ++s)
                                mma_ss(tO, sdesc_sw128(pa + s * 32), sdesc_sw128(va + (j - 1) * 8192 + s * 2048),
                                       kIdescPV, (j > 1 || s > 0) ? 1u : 0u);
                            mma_commit(&pvdone[w]);
                        }
                    }
                    gb += a.nblk;
                    ++nq;
                }
                // the next round needs other lists: let the producer overwrite them
                if (r >= i1 || a.items[r].w != cur_bh || a.items[r].x != cur_e) mma_commit(&kvfree);
            }
        }
    } else {
        // ------------------------------ row warpgroups ------------------------------
        const int w = (warp - 1 - NWG) >> 2;  // 4 consecutive warps cover the 4 TMEM lane quarters
        const int t = (warp & 3) * 32 + lane;  // TMEM lane = query row of the item
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tO = tb + w * kTStride + SB * 64;
        uint32_t gb = 0, nitem = 0;
        bool ok = true;
        for (int r = i0; r < i1 && ok;) {
            int4 it[NWG];
            const int cnt = round_size(a, r, i1, it);
            r += cnt;
            if (w >= cnt) continue;
            const int4 item = it[w];
            const int64_t bh = item.w;
            const int n = t < item.z ? a.perm[bh * a.N + item.y + t] : 0;
            float mrun = -INFINITY, lrun = 0.f;
            for (int j = 0; j < a.nblk; ++j, ++gb) {
                const uint32_t sb = gb % SB;
                ok = __all_sync(0xffffffffu, mbar_wait(&sfull[w * SB + sb], (gb / SB) & 1, a.status));
                if (!ok) break;
                tc_fence_after();
                float s[KB];
                tmem_ld32(tb + w * kTStride + sb * KB + lane_off, s);
                tmem_ld32(tb + w * kTStride + sb * KB + lane_off + 32, s + 32);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&sfree[w * SB + sb]);
                const int valid = min(KB, nkeys - j * KB);
                if (valid < KB) {  // last, partial block (warp-uniform)
#pragma unroll
                    for (int c = 0; c < KB; ++c) s[c] = c < valid ? s[c] : -INFINITY;
                }
                // 8 independent partial maxima / sums: short dependency chains
                float pm[8];
                static_assert(KB == 64, "the partial maxima below cover exactly 64 columns");
#pragma unroll
                for (int u = 0; u < 8; ++u) {  // columns u, u+8, ..., u+56
                    pm[u] = fmax3(s[u], s[u + 8], s[u + 16]);
                    pm[u] = fmax3(pm[u], s[u + 24], s[u + 32]);
                    pm[u] = fmax3(pm[u], s[u + 40], s[u + 48]);
                    pm[u] = fmaxf(pm[u], s[u + 56]);
                }
                const float bmax = fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(fmax3(pm[3], pm[4], pm[5]), pm[6], pm[7])) * kC;
                const float mnew = (bmax > mrun + kLazy) ? bmax : mrun;
                const float alpha = exp2f(mrun - mnew);  // 0 on the first block, 1 when the max is kept
                // packed pairs: one f32x2 FMA forms two exponents, one f32x2 add
                // accumulates two weights
                const float2 c2 = make_float2(kC, kC), m2 = make_float2(-mnew, -mnew);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < KB; c += 2) {
                    const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), c2, m2);
                    s[c] = exp2f(x.x);
                    s[c + 1] = exp2f(x.y);
                    acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], make_float2(s[c], s[c + 1]));
                }
                const float sum = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
                lrun = lrun * alpha + sum;
                // P.V of the previous block must be done before P is overwritten
                // (and before O is rescaled, when a running max grew by > 2^8)
                const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
                if (gb >= 1) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&pvdone[w], (gb - 1) & 1, a.status));
                    if (!ok) break;
                }
                tc_fence_after();
                if (rescale) {
                    float o[16];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        tmem_ld16(tO + lane_off + h * 16, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 16; ++c) o[c] *= alpha;
                        tmem_st16(tO + lane_off + h * 16, o);
                    }
                    tmem_st_wait();
                }
                uint8_t* pdst = S.p + w * 16384;
#pragma unroll
                for (int g = 0; g < KB / 8; ++g) {
                    uint4 pk;
                    __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
                    for (int u = 0; u < 4; ++u) h2[u] = __floats2bfloat162_rn(s[8 * g + 2 * u], s[8 * g + 2 * u + 1]);
                    *reinterpret_cast<uint4*>(pdst + swz128(t, g)) = pk;
                }
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(&pfull[w]);
                mrun = mnew;
            }
            if (!ok) break;
            // epilogue: the last P.V of the item (and with it every earlier one) is done
            ok = __all_sync(0xffffffffu, mbar_wait(&pvdone[w], (gb - 1) & 1, a.status));
            if (!ok) break;
            tc_fence_after();
            const float inv = 1.f / lrun;
            uint4* dst = reinterpret_cast<uint4*>(a.out + (bh * a.N + n) * D);
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // two 32-column halves of the output row
                float o[32];
                tmem_ld32(tO + lane_off + h * 32, o);
                tmem_ld_wait();
                if (h == 1) {
                    tc_fence_before();
                    mbar_arrive(&ofree[w]);
                }
                if (t < item.z) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 pk;
                        __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            h2[u] = __floats2bfloat162_rn(o[8 * c + 2 * u] * inv, o[8 * c + 2 * u + 1] * inv);
                        dst[h * 4 + c] = pk;
                    }
                }
            }
            ++nitem;
        }
        (void)nitem;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tb, 512);
}

size_t smem_bytes(int nblk) { return 1024 + static_cast<size_t>(nblk) * 16384 + NWG * (QB * 16384 + 16384); }

}  // namespace

bool expert_tc_supported(const Plan& p) {
    const int nkeys = p.s.m + p.s.k;
    return nkeys <= 512 && smem_bytes((nkeys + KB - 1) / KB) <= 232448;
}

cudaError_t launch_expert_tc(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                             const __nv_bfloat16* V, const int32_t* expert_idx, __nv_bfloat16* out,
                             cudaStream_t st) {
    Args a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.lqhi = w.lqhi;
    a.lvbf = w.lvbf;
    a.items = w.items;
    a.nitems = w.nitems;
    a.perm = w.perm;
    a.expert_idx = expert_idx;
    a.out = out;
    a.status = w.status;
    a.N = p.s.N;
    a.m = p.s.m;
    a.k = p.s.k;
    a.nblk = (p.s.m + p.s.k + KB - 1) / KB;
    const size_t sm = smem_bytes(a.nblk);
    cudaError_t e = cudaFuncSetAttribute(expert_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sm));
    if (e != cudaSuccess) return e;
    expert_tc_kernel<<<device_sms(), NT, sm, st>>>(a);
    return cudaGetLastError();
}

}  // namespace mita
