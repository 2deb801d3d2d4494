// Stage 3 on the tensor cores: routing.
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造": each query picks the expert of
// the landmark query it matches best (s = 1), reusing the query-to-landmark
// logits: e(n) = argmax_i <q_n, Lq_i> (tau > 0 does not change the argmax),
// ties to the lowest i.
//
// Persistent CTAs, each over a contiguous range of 128-query tiles (so the
// head, and with it the landmark operand, changes rarely).
//   warp 4 lane 0: TMA loads of Q tiles (4-stage ring) and of the head's
//                  landmark queries (bf16 hi/lo pair, m_pad <= 256 rows);
//   warps 9, 10 (lane 0): MMA issuers, one per TMEM buffer b (tiles t = b mod
//                  2): D = Q Lq_hi^T + Q Lq_lo^T (M = 128, N = m_pad, exact to
//                  ~2^-16 of the fp32 landmarks); a tcgen05.mma holds its
//                  issuing thread about as long as it runs, so the two
//                  buffers' MMAs come from separate threads;
//   warps 0-3, 5-8: two argmax warpgroups, one per TMEM buffer: one query row
//                  per thread, argmax over the m logits, the route, and a
//                  shared-memory histogram (one per warpgroup) of the head's
//                  routes that is added to the per-head expert counts.
// With s routed experts per query (MULTI; the pages' setting is s = 1, the
// general form takes the s highest logits, highest first, ties to the lower
// landmark) each row keeps its s best (logit, landmark) pairs as a sorted
// list instead of the argmax, and the histograms count per rank of the list.
// Every wait is bounded (umma.cuh).
#include <algorithm>

#include "tensormap.cuh"
#include "umma.cuh"

namespace mita {

namespace {

using namespace umma;

constexpr int QST = 4;  // Q tile stages
constexpr size_t OFF_LO = 32768;
constexpr size_t OFF_Q = 65536;
constexpr size_t SMEM = OFF_Q + QST * 16384 + 1024;

struct RouteArgs {
    int32_t* route;  // [BH][N][s]
    int* counts;     // [s][BH][m]
    int* status;
    int64_t N, BH, tiles_per_head, total_tiles;
    int m, m_pad, s;
};

constexpr int RT_THREADS = 352;  // warps 0-3 and 5-8: argmax groups; 4: loads; 9, 10: MMA issuers

template <bool MULTI>
__global__ void __launch_bounds__(RT_THREADS, 1) route_tc_kernel(const __grid_constant__ CUtensorMap tq,
                                                          const __grid_constant__ CUtensorMap thi,
                                                          const __grid_constant__ CUtensorMap tlo, RouteArgs a) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t qfull[QST], qempty[QST], dfull[2], dfree[2], lqfull, lqfree, drain;
    __shared__ uint32_t tmem_base;
    constexpr int HS = MULTI ? MITA_MAX_S : 1;  // histogram planes (ranks)
    __shared__ int hist[2][HS][256];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t t0 = a.total_tiles * blockIdx.x / gridDim.x;
    const int64_t t1 = a.total_tiles * (blockIdx.x + 1) / gridDim.x;
    const int nt = static_cast<int>(t1 - t0);

    if (tid == 0) {
        for (int i = 0; i < QST; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&dfull[i], 1);
            mbar_init(&dfree[i], 4);  // every warp of the buffer's group arrives
        }
        mbar_init(&lqfull, 1);
        mbar_init(&lqfree, 2);  // one commit per MMA issuer
        mbar_init(&drain, 2);   // exit path: one commit per MMA issuer
        fence_barrier_init();
    }
    for (int e = tid; e < 2 * HS * 256; e += blockDim.x) (&hist[0][0][0])[e] = 0;
    if (warp == 0) tmem_alloc(&tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;

    if (warp == 4) {
        // ---------------- loads (lane 0) ----------------
        if (lane == 0) {
            auto load_q = [&](int t) {
                const int st = t % QST;
                const int64_t g = t0 + t;
                const int64_t bh = g / a.tiles_per_head, tile = g % a.tiles_per_head;
                mbar_arrive_expect_tx(&qfull[st], 16384);
                tma_load_2d(base + OFF_Q + st * 16384, &tq, 0, static_cast<int>(bh * a.N + tile * 128), &qfull[st]);
            };
            int loaded = 0;
            for (int t = 0; t < nt && t < QST; ++t, ++loaded) load_q(t);
            int64_t cur = -1;
            int changes = 0;
            for (int t = 0; t < nt; ++t) {
                const int64_t bh = (t0 + t) / a.tiles_per_head;
                if (bh != cur) {  // restage the landmarks once the MMAs reading them are done
                    if (changes > 0 && !mbar_wait(&lqfree, (changes - 1) & 1, a.status)) break;
                    mbar_arrive_expect_tx(&lqfull, 2u * a.m_pad * 128u);
                    tma_load_2d(base, &thi, 0, static_cast<int>(bh * a.m), &lqfull);
                    tma_load_2d(base + OFF_LO, &tlo, 0, static_cast<int>(bh * a.m), &lqfull);
                    ++changes;
                    cur = bh;
                }
                // refill the stage of tile t once its MMAs are done
                if (t + QST < nt) {
                    if (!mbar_wait(&qempty[t % QST], (t / QST) & 1, a.status)) break;
                    load_q(t + QST);
                    ++loaded;
                }
            }
            // exit: the last load of every barrier armed here has landed
            if (changes > 0) mbar_drain(&lqfull, (changes - 1) & 1);
            for (int st = 0; st < QST; ++st) {
                const int arms = loaded > st ? (loaded - st + QST - 1) / QST : 0;
                if (arms > 0) mbar_drain(&qfull[st], (arms - 1) & 1);
            }
        }
    } else if (warp >= 9) {
        // ---------------- MMA issuer of TMEM buffer b (lane 0) ----------------
        // Walks every tile to follow the landmark restages (each head change
        // is released, then waited for), and issues the tiles t = b mod 2.
        if (lane == 0) {
            const int b = warp - 9;
            const uint32_t idesc = idesc_bf16(128, a.m_pad, false);
            const uint32_t hi = smem_u32(base), lo = smem_u32(base + OFF_LO);
            const uint32_t d = tb + b * 256;
            int64_t cur = -1;
            int changes = 0;
            for (int t = 0; t < nt; ++t) {
                const int64_t bh = (t0 + t) / a.tiles_per_head;
                if (bh != cur) {
                    if (changes > 0) mma_commit(&lqfree);  // once this thread's MMAs on the old landmarks are done
                    if (!mbar_wait(&lqfull, changes & 1, a.status)) break;
                    ++changes;
                    cur = bh;
                }
                if ((t & 1) != b) continue;
                const int st = t % QST;
                if (!mbar_wait(&qfull[st], (t / QST) & 1, a.status)) break;
                // the argmax group has read this buffer's previous tile (t - 2)
                if (t >= 2 && !mbar_wait(&dfree[b], ((t >> 1) - 1) & 1, a.status)) break;
                tc_fence_after();
                const uint32_t qa = smem_u32(base + OFF_Q + st * 16384);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ss(d, sdesc_sw128(qa + s * 32), sdesc_sw128(hi + s * 32), idesc, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_ss(d, sdesc_sw128(qa + s * 32), sdesc_sw128(lo + s * 32), idesc, 1u);
                mma_commit(&dfull[b]);
                mma_commit(&qempty[st]);
            }
            mma_drain(&drain);  // exit: this issuer's MMAs are done
        }
    } else {
        // ---------------- argmax warpgroups: group b takes the tiles t = b (mod 2) ----------------
        const int b = warp < 4 ? 0 : 1;
        const int row = (warp & 3) * 32 + lane;  // TMEM lane quarter = warp % 4
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int(*h)[256] = hist[b];
        const int ns = MULTI ? a.s : 1;
        int64_t cur = -1;
        for (int t = b; t < nt; t += 2) {
            const int64_t g = t0 + t;
            const int64_t bh = g / a.tiles_per_head, tile = g % a.tiles_per_head;
            if (bh != cur) {
                named_bar(1 + b, 128);
                if (cur >= 0)
                    for (int j = 0; j < ns; ++j)
                        for (int e = row; e < a.m; e += 128)
                            if (h[j][e]) atomicAdd(&a.counts[(j * a.BH + cur) * a.m + e], h[j][e]);
                named_bar(1 + b, 128);
                for (int j = 0; j < ns; ++j)
                    for (int e = row; e < a.m; e += 128) h[j][e] = 0;
                named_bar(1 + b, 128);
                cur = bh;
            }
            if (!named_bar_and(1 + b, 128, mbar_wait(&dfull[b], (t >> 1) & 1, a.status))) break;
            tc_fence_after();
            const uint32_t d = tb + b * 256 + lane_off;
            const int64_t n = tile * 128 + row;
            if constexpr (!MULTI) {
                // 4 interleaved (value, index) chains; on equal values the lower
                // index wins, as in a left-to-right scan with a strict comparison
                float bv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                int bi[4] = {0, 1, 2, 3};
                for (int c0 = 0; c0 < a.m_pad; c0 += 32) {
                    float v[32];
                    tmem_ld32(d + c0, v);
                    tmem_ld_wait();
                    if (c0 + 32 > a.m) {  // (uniform) the last chunk: columns past m are another head's
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = c0 + j < a.m ? v[j] : -INFINITY;
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int u = j & 3;
                        if (v[j] > bv[u]) {
                            bv[u] = v[j];
                            bi[u] = c0 + j;
                        }
                    }
                }
                tc_fence_before();
                warp_arrive(&dfree[b]);
                float best = bv[0];
                int arg = bi[0];
#pragma unroll
                for (int u = 1; u < 4; ++u)
                    if (bv[u] > best || (bv[u] == best && bi[u] < arg)) {
                        best = bv[u];
                        arg = bi[u];
                    }
                arg = min(arg, a.m - 1);  // in range whatever the logits (non-finite ones are out of contract)
                if (n < a.N) {
                    a.route[bh * a.N + n] = arg;
                    atomicAdd(&h[0][arg], 1);
                }
            } else {
                // s rounds of the argmax above, each over the columns not
                // taken by an earlier round (those read as -inf): round u
                // gives the u-th entry in the order (logit descending,
                // landmark ascending). The winners so far are kept as bytes
                // (m <= 256 here) in two words; the rounds stay a loop.
                uint32_t won0 = 0u, won1 = 0u;  // winners 0-3 and 4-7, one byte each
#pragma unroll 1
                for (int u = 0; u < ns; ++u) {
                    float bv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                    int bi[4] = {a.m, a.m, a.m, a.m};
                    for (int c0 = 0; c0 < a.m_pad; c0 += 32) {
                        float v[32];
                        tmem_ld32(d + c0, v);
                        tmem_ld_wait();
                        if (c0 + 32 > a.m) {
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj) v[jj] = c0 + jj < a.m ? v[jj] : -INFINITY;
                        }
                        uint32_t ex = 0;  // columns of this chunk taken before
                        for (int x = 0; x < u; ++x) {
                            const int wc = static_cast<int>(((x < 4 ? won0 : won1) >> (8 * (x & 3))) & 255u);
                            if ((wc >> 5) == (c0 >> 5)) ex |= 1u << (wc & 31);
                        }
                        if (ex) {
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj) v[jj] = ((ex >> jj) & 1u) ? -INFINITY : v[jj];
                        }
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const int ch = jj & 3;
                            if (v[jj] > bv[ch]) {
                                bv[ch] = v[jj];
                                bi[ch] = c0 + jj;
                            }
                        }
                    }
                    float best = bv[0];
                    int arg = bi[0];
#pragma unroll
                    for (int c = 1; c < 4; ++c)
                        if (bv[c] > best || (bv[c] == best && bi[c] < arg)) {
                            best = bv[c];
                            arg = bi[c];
                        }
                    // in range whatever the logits (non-finite ones are out of contract)
                    const int r = min(max(arg, 0), a.m - 1);
                    if (u < 4)
                        won0 |= static_cast<uint32_t>(r) << (8 * u);
                    else
                        won1 |= static_cast<uint32_t>(r) << (8 * (u - 4));
                    if (n < a.N) {
                        a.route[(bh * a.N + n) * ns + u] = r;
                        atomicAdd(&h[u][r], 1);
                    }
                }
                tc_fence_before();
                warp_arrive(&dfree[b]);
            }
        }
        named_bar(1 + b, 128);
        if (cur >= 0)
            for (int j = 0; j < ns; ++j)
                for (int e = row; e < a.m; e += 128)
                    if (h[j][e]) atomicAdd(&a.counts[(j * a.BH + cur) * a.m + e], h[j][e]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tb, 512);
}

}  // namespace

bool route_tc_supported(const Plan& p) { return p.s.m <= 256 && p.s.BH * p.s.N < (int64_t(1) << 31); }

// The route of each query (s = 1: [BH][N]) or its s best landmarks ([BH][N][s]).

cudaError_t launch_route_tc(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route, cudaStream_t st) {
    RouteArgs a;
    a.route = route;
    a.counts = w.counts;
    a.status = w.status;
    a.N = p.s.N;
    a.BH = p.s.BH;
    a.s = p.s.s_route;
    a.tiles_per_head = (p.s.N + 127) / 128;
    a.total_tiles = a.tiles_per_head * p.s.BH;
    a.m = p.s.m;
    a.m_pad = (p.s.m + 15) / 16 * 16;
    CUtensorMap tq, thi, tlo;
    const uint64_t mrows = static_cast<uint64_t>(p.s.BH) * p.s.m;
    if (!make_row_tmap(&tq, Q, static_cast<uint64_t>(p.s.BH * p.s.N), 128) ||
        !make_row_tmap(&thi, w.lqhi, mrows, a.m_pad) || !make_row_tmap(&tlo, w.lqlo, mrows, a.m_pad))
        return cudaErrorInvalidValue;
    auto kern = a.s > 1 ? route_tc_kernel<true> : route_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM));
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(device_sms(), a.total_tiles);
    return launch_dep(kern, dim3(static_cast<unsigned>(grid)), dim3(RT_THREADS), SMEM, st, tq, thi, tlo, a);
}

}  // namespace mita
