// Backward pass on the tensor cores (tcgen05, TMEM): the four dense products
// of the two attentions of MiTA, for the gradients declared in backward.cu.
//
// The forward pass is written in "NeurIPS 2026 | Mixture-of-Top-k 注意力"
// (shuwu5.cn), section "MiTA：用少量地标查询，同时完成压缩与专家构造"; the pages
// train MiTA models (results section) but do not describe their backward
// pass. With tau = 1/sqrt(64), z = tau <row, key> log2(e), and per row its
// log-sum-exp L (log2 units) and Delta = dR . out:
//   p = 2^(z - L),   ds = p (<dR, value> - Delta),
//   row gradient     G_row = tau sum_key ds key           (rows kernel)
//   key gradients    dK_key = tau sum_row ds row,  dV_key = sum_row p dR
//                                                          (keys kernel)
// Two attentions have this form:
//   expert attention (EXP): rows = the queries routed to an expert (dR = dO),
//     keys = its list [Lq_0..Lq_{m-1} (bf16, as the forward pass reads them),
//     K_j (j in E_e)], values [LV_0..LV_{m-1} (bf16), V_j]: G -> dQ, dK/dV of
//     the shared keys -> dLq, dLV, of the routed keys -> dK, dV;
//   landmark attention (LMK): rows = the landmarks (Lq as a bf16 hi/lo pair,
//     as the forward scan reads them; dR = dLV), keys = all of the head's K,
//     values V: G -> dLq, dK/dV -> dK, dV.
//
// Rows kernel (rows on the MMA's M dimension, one thread per row): per block
// of 64 keys S = R K^T and dP = dR V^T into TMEM, the rows form ds (bf16) in
// TMEM, and G += ds K (A in TMEM, the same key rows as the MN-major B). One
// work unit = 128 rows: an item (<= 128 queries of one expert) or a landmark
// tile with one chunk of keys.
// Keys kernel (keys on M, one thread per key): per tile of 128 rows
// S^T = K R^T and dP^T = V dR^T, the key threads form p^T and ds^T (bf16) in
// TMEM with each row's L and Delta read from shared memory, then
// dV += p^T dR and dK += ds^T R (A in TMEM, the row tiles as MN-major B),
// accumulated over all the rows of the unit. One work unit = 128 keys: a
// block of an expert's list (rows: that expert's queries) or a tile of the
// head's keys (rows: its landmarks).
// Warps: 0-15 the row (or key) threads, four per TMEM lane quarter, each
// taking a quarter of a block's columns (p and ds are elementwise once the
// row statistics are known, so nothing is reduced across them); 16 the
// producer (TMA), 17 and 18 the MMA issuers: one for the products that
// read the rows and keys (S, dP), one for the gradient products (G; dV and
// dK), so the next block's S and dP run while the threads and G work on
// this one. Every wait is bounded (umma.cuh).
#include <algorithm>

#include "pool_grad.cuh"
#include "tensormap.cuh"
#include "umma.cuh"

namespace mita {

namespace {

using namespace umma;

constexpr float kTau = 0.125f;
constexpr float kC = 0.125f * kLog2e;  // tau * log2(e)
constexpr int kExp = 0, kLmk = 1;       // expert attention / landmark attention
constexpr int RW = 4;                  // row (key) warps per TMEM lane quarter
constexpr int NRW = 4 * RW;            // row (key) warps: 0 .. NRW - 1
constexpr int PW = NRW;                // producer warp; the MMA issuers are PW + 1 (S, dP), PW + 2 (G)
constexpr int NTB = (NRW + 3) * 32;
constexpr int TILE = 16384;            // 128 rows of 64 bf16

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Problem description shared by both kernels (pointers a mode does not use are null).
struct BArgs {
    const int4* items;          // EXP rows kernel: the flat item list and its length
    const int* nitems;
    const int* expoff;          // EXP keys kernel: [BH][m+1] each expert's first grouped query
    const int* perm;            // [BH][N] queries grouped by expert
    const int32_t* expert_idx;  // [BH][m][k]
    const float* lse;           // EXP: [BH][N] per query in grouped order; LMK: [BH][m] per landmark (log2 units)
    const float* delta;         // same layout: Delta of each row
    float* gk;                  // keys kernel: dK target ([BH][N][64], += ), rows kernel: G target (EXP: dQ, =)
    float* gv;                  // keys kernel: dV target ([BH][N][64], +=); LMK rows kernel: dLq (atomic)
    float* slq;                 // EXP keys kernel: dLq of the shared keys ([BH][m][64], atomic)
    float* slv;                 // EXP keys kernel: dLV of the shared keys ([BH][m][64], atomic)
    int* status;
    int64_t N, units, chunk_len;
    int m, k, m4, nblk, chunks;
    int gh, gw, p;              // EXP rows kernel: the landmark windows (dQ gets the pooling's share of dLq)
};


// Rows of expert list position x (EXP): the shared rows [0, m) are landmark
// rows (clamped), positions [m, m4) are unused, [m4, m4 + k) routed keys
// (clamped to the last). Four consecutive positions never straddle m4.
__device__ __forceinline__ void list_rows4(const BArgs& a, int64_t bh, const int32_t* sel, int x, int* y, bool* shared) {
    *shared = x < a.m4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int xx = x + u;
        y[u] = *shared ? static_cast<int>(bh * a.m + min(xx, a.m - 1))
                       : static_cast<int>(bh * a.N + sel[min(xx - a.m4, a.k - 1)]);
    }
}

// ============================================================================
// Keys kernel
// ============================================================================
// shared memory: key blocks c = 0, 1 (KB, VB) at 32 KB c; then the row tile
// buffers: EXP four of R, dR, L[128], Delta[128] (33 KB each), LMK two of
// R, R_lo, dR, L, Delta (49 KB each)
constexpr size_t KOFF_BUF = 65536;
template <int MODE>
struct KRow {
    static constexpr int n = MODE == kExp ? 4 : 2;                         // buffers
    static constexpr size_t dr = MODE == kExp ? TILE : 2 * TILE;           // dR
    static constexpr size_t st = MODE == kExp ? 2 * TILE : 3 * TILE;       // L, Delta
    static constexpr size_t size = st + 1024;
};
constexpr size_t KSMEM = KOFF_BUF + 4 * (2 * TILE + 1024) + 1024;
static_assert(4 * (2 * TILE + 1024) >= 2 * (3 * TILE + 1024), "row buffers of both modes fit");
// TMEM columns
constexpr uint32_t cS = 0, cDP = 128, cP = 256, cDS = 320, cV = 384, cK = 448;

template <int MODE>
__device__ __forceinline__ void keys_unit(const BArgs& a, int64_t u, int64_t& bh, int& e, int& b, int& ntiles,
                                          int& qoff, int& qcnt) {
    if (MODE == kExp) {
        bh = u / (static_cast<int64_t>(a.m) * a.nblk);
        e = static_cast<int>((u / a.nblk) % a.m);
        b = static_cast<int>(u % a.nblk);
        const int* eo = a.expoff + bh * (a.m + 1);
        qoff = eo[e];
        qcnt = eo[e + 1] - qoff;
        ntiles = (qcnt + 127) / 128;
    } else {
        const int64_t nkt = (a.N + 127) / 128;
        bh = u / nkt;
        b = static_cast<int>(u % nkt);
        e = 0;
        qoff = 0;
        qcnt = a.m;
        ntiles = (a.m + 127) / 128;
    }
}

template <int MODE>
__global__ void __launch_bounds__(NTB, 1)
    bwd_keys_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tsk, const __grid_constant__ CUtensorMap tsv,
                    const __grid_constant__ CUtensorMap tr, const __grid_constant__ CUtensorMap tdr, BArgs a) {
    // EXP: tk, tv, tsk, tsv: K, V, Lq (bf16), LV (bf16) rows, one row high
    //      (gathers); tr, tdr: Q, dO rows, one row high.
    // LMK: tk, tv: K, V, 128 rows high; tr, tsk: Lq hi, lo; tdr: dLV (bf16),
    //      128 rows high.
    extern __shared__ uint8_t smem_raw[];
    using RB = KRow<MODE>;
    __shared__ uint64_t kvfull[2], kvfree[2], rfull[4], rfree[4], sfull, sfree, pfull, pvdone, afree, drain[2];
    __shared__ uint32_t tmem_base;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t u0 = a.units * blockIdx.x / gridDim.x, u1 = a.units * (blockIdx.x + 1) / gridDim.x;
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&kvfull[b], 1);
            mbar_init(&kvfree[b], 1);
        }
        for (int b = 0; b < RB::n; ++b) {
            mbar_init(&rfull[b], 2);  // the loads' transaction count, and the statistics
            mbar_init(&rfree[b], 1);
        }
        mbar_init(&sfull, 1);
        mbar_init(&sfree, NRW);
        mbar_init(&pfull, NRW);
        mbar_init(&pvdone, 1);
        mbar_init(&afree, NRW);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    auto kbuf = [&](int c) { return base + c * 2 * TILE; };  // keys, then values at + TILE
    auto rbuf = [&](int b) { return base + KOFF_BUF + b * RB::size; };

    if (warp == PW) {
        // ---------------------------------- producer ----------------------------------
        // Tiles in order (units with no tiles skipped). The global values a
        // tile needs (EXP: its queries, the key list rows of a unit's first
        // tile; both: the rows' statistics) are loaded into registers one tile
        // ahead, so their latency overlaps the wait for a free buffer.
        struct Cur {
            int64_t u, bh;
            int e, b, ntiles, qoff, qcnt, t;
        };
        auto first_of = [&](int64_t u, Cur& c) -> bool {  // the first tile at or after unit u
            for (; u < u1; ++u) {
                keys_unit<MODE>(a, u, c.bh, c.e, c.b, c.ntiles, c.qoff, c.qcnt);
                if (c.ntiles > 0) {
                    c.u = u;
                    c.t = 0;
                    return true;
                }
            }
            return false;
        };
        const int r0 = 4 * lane;
        int y[4];
        bool sh = false;
        float L4[4], D4[4];
        auto fetch = [&](const Cur& c) {
            if (MODE == kExp) {
                const int cnt = min(128, c.qcnt - 128 * c.t);
                const int64_t gp = c.bh * a.N + c.qoff + 128 * c.t + r0;  // statistics in grouped order
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const bool v = r0 + x < cnt;
                    L4[x] = v ? a.lse[gp + x] : INFINITY;
                    D4[x] = v ? a.delta[gp + x] : 0.f;
                }
                if (c.t == 0) {
                    const int32_t* sel = a.expert_idx + (c.bh * a.m + c.e) * static_cast<int64_t>(a.k);
                    list_rows4(a, c.bh, sel, 128 * c.b + r0, y, &sh);
                }
            } else {
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int li = 128 * c.t + r0 + x;
                    const bool v = li < a.m;
                    L4[x] = v ? a.lse[c.bh * a.m + li] : INFINITY;
                    D4[x] = v ? a.delta[c.bh * a.m + li] : 0.f;
                }
            }
        };
        int ucount = 0, tseq = 0;
        bool ok = true;
        Cur c;
        bool have = first_of(u0, c);
        if (have) fetch(c);
        while (have && ok) {
            if (c.t == 0) {
                const int kb = ucount & 1;  // this unit's key block buffer, last used two units back
                if (ucount >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&kvfree[kb], ((ucount >> 1) - 1) & 1, a.status));
                if (!ok) break;
                uint8_t* KBs = kbuf(kb);
                uint8_t* VBs = KBs + TILE;
                if (lane == 0) mbar_arrive_expect_tx(&kvfull[kb], 2 * TILE);
                __syncwarp();
                if (MODE == kExp) {  // list positions 128 b + 4 lane .. + 3
                    tma_gather4(KBs + r0 * 128, sh ? &tsk : &tk, 0, y[0], y[1], y[2], y[3], &kvfull[kb]);
                    tma_gather4(VBs + r0 * 128, sh ? &tsv : &tv, 0, y[0], y[1], y[2], y[3], &kvfull[kb]);
                } else if (lane == 0) {
                    tma_load_2d(KBs, &tk, 0, static_cast<int>(c.bh * a.N + 128 * c.b), &kvfull[kb]);
                    tma_load_2d(VBs, &tv, 0, static_cast<int>(c.bh * a.N + 128 * c.b), &kvfull[kb]);
                }
                ++ucount;
            }
            const int buf = tseq % RB::n;
            if (tseq >= RB::n) ok = __all_sync(0xffffffffu, mbar_wait(&rfree[buf], ((tseq / RB::n) - 1) & 1, a.status));
            if (!ok) break;
            uint8_t* rb = rbuf(buf);
            float* sl = reinterpret_cast<float*>(rb + RB::st);
            if (lane == 0) mbar_arrive_expect_tx(&rfull[buf], (MODE == kExp ? 2 : 3) * TILE);
            __syncwarp();
            if (MODE == kExp) {
                // the tile's queries and their dO, in grouped order (rows past
                // the expert's queries belong to the next expert or lie past
                // the end, zero-filled: their statistics mask them)
                if (lane == 0) {
                    const int yg = static_cast<int>(c.bh * a.N + c.qoff + 128 * c.t);
                    tma_load_2d(rb, &tr, 0, yg, &rfull[buf]);
                    tma_load_2d(rb + RB::dr, &tdr, 0, yg, &rfull[buf]);
                }
            } else if (lane == 0) {
                const int yl = static_cast<int>(c.bh * a.m + 128 * c.t);
                tma_load_2d(rb, &tr, 0, yl, &rfull[buf]);
                tma_load_2d(rb + TILE, &tsk, 0, yl, &rfull[buf]);
                tma_load_2d(rb + RB::dr, &tdr, 0, yl, &rfull[buf]);
            }
            *reinterpret_cast<float4*>(sl + r0) = make_float4(L4[0], L4[1], L4[2], L4[3]);
            *reinterpret_cast<float4*>(sl + 128 + r0) = make_float4(D4[0], D4[1], D4[2], D4[3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&rfull[buf]);  // the statistics are in place
            ++tseq;
            // the next tile, and its values
            if (++c.t == c.ntiles) have = first_of(c.u + 1, c);
            if (have) fetch(c);
        }
        if (lane == 0) {  // exit: the last phase of every barrier armed here has landed
            for (int b = 0; b < 2; ++b) {
                const int karms = ucount > b ? (ucount - b + 1) / 2 : 0;
                if (karms > 0) mbar_drain(&kvfull[b], (karms - 1) & 1);
            }
            for (int b = 0; b < RB::n; ++b) {
                const int arms = tseq > b ? (tseq - b + RB::n - 1) / RB::n : 0;
                if (arms > 0) mbar_drain(&rfull[b], (arms - 1) & 1);
            }
        }
    } else if (warp == PW + 1) {
        // ------------------------------ S, dP issuer ------------------------------
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(128, 128, false);
            int ucount = 0, tseq = 0;
            bool ok = true;
            for (int64_t u = u0; u < u1 && ok; ++u) {
                int64_t bh;
                int e, b, ntiles, qoff, qcnt;
                keys_unit<MODE>(a, u, bh, e, b, ntiles, qoff, qcnt);
                if (ntiles == 0) continue;
                const int kb = ucount & 1;
                if (!(ok = mbar_wait(&kvfull[kb], (ucount >> 1) & 1, a.status))) break;
                const uint64_t kd = sdesc_sw128(smem_u32(kbuf(kb))), vd = sdesc_sw128(smem_u32(kbuf(kb) + TILE));
                for (int t = 0; t < ntiles; ++t) {
                    const int buf = tseq % RB::n;
                    if (!(ok = mbar_wait(&rfull[buf], (tseq / RB::n) & 1, a.status))) break;
                    // the key threads have read the previous tile's S and dP
                    if (tseq >= 1 && !(ok = mbar_wait(&sfree, (tseq - 1) & 1, a.status))) break;
                    tc_fence_after();
                    const uint32_t rs = smem_u32(rbuf(buf));
                    mma_ss_k64(tb + cS, kd, sdesc_sw128(rs), idS, 0u);
                    if (MODE == kLmk) mma_ss_k64(tb + cS, kd, sdesc_sw128(rs + TILE), idS, 1u);
                    mma_ss_k64(tb + cDP, vd, sdesc_sw128(rs + RB::dr), idS, 0u);
                    mma_commit(&sfull);
                    ++tseq;
                }
                if (!ok) break;
                mma_commit(&kvfree[kb]);  // the key block is read by S and dP only
                ++ucount;
            }
            mma_drain(&drain[0]);
        }
    } else if (warp == PW + 2) {
        // -------------------------------- G issuer --------------------------------
        if (lane == 0) {
            const uint32_t idG = idesc_bf16(128, 64, true);
            int ucount = 0, tseq = 0;
            bool ok = true;
            for (int64_t u = u0; u < u1 && ok; ++u) {
                int64_t bh;
                int e, b, ntiles, qoff, qcnt;
                keys_unit<MODE>(a, u, bh, e, b, ntiles, qoff, qcnt);
                if (ntiles == 0) continue;
                for (int t = 0; t < ntiles; ++t) {
                    const int buf = tseq % RB::n;
                    // the row tile (for its layout in shared memory) and the
                    // threads' p^T and ds^T of it
                    if (!(ok = mbar_wait(&rfull[buf], (tseq / RB::n) & 1, a.status))) break;
                    if (!(ok = mbar_wait(&pfull, tseq & 1, a.status))) break;
                    // the first products of a unit overwrite the accumulators: the
                    // key threads have read the previous unit's
                    if (t == 0 && ucount >= 1 && !(ok = mbar_wait(&afree, (ucount - 1) & 1, a.status))) break;
                    tc_fence_after();
                    const uint32_t rs = smem_u32(rbuf(buf));
                    const uint64_t dr = sdesc_sw128(rs + RB::dr), rr = sdesc_sw128(rs);
#pragma unroll 1
                    for (int s = 0; s < 8; ++s) {  // K = the tile's 128 rows, 16 per step
                        const uint32_t acc = (t > 0 || s > 0) ? 1u : 0u;
                        mma_ts(tb + cV, tb + cP + 8 * s, dr + static_cast<uint64_t>(s) * 128, idG, acc);
                        mma_ts(tb + cK, tb + cDS + 8 * s, rr + static_cast<uint64_t>(s) * 128, idG, acc);
                    }
                    mma_commit(&pvdone);
                    mma_commit(&rfree[buf]);  // S and dP of the tile completed before pfull
                    ++tseq;
                }
                if (!ok) break;
                ++ucount;
            }
            mma_drain(&drain[1]);
        }
    } else {
        // ------------------------------- key threads -------------------------------
        // warp w: TMEM lanes 32 (w % 4) .. + 31 (the unit's keys), rows
        // 32 (w / 4) .. + 31 of each row tile, and accumulator columns
        // 16 (w / 4) .. + 15
        static_assert(RW == 4, "one 32-row chunk of the tile per key warp");
        const int t_ = (warp & 3) * 32 + lane;  // TMEM lane = key row of the unit
        const int cg = warp >> 2;
        const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int ucount = 0, tseq = 0;
        bool ok = true;
        for (int64_t u = u0; u < u1 && ok; ++u) {
            int64_t bh;
            int e, b, ntiles, qoff, qcnt;
            keys_unit<MODE>(a, u, bh, e, b, ntiles, qoff, qcnt);
            if (ntiles == 0) continue;
            for (int t = 0; t < ntiles && ok; ++t) {
                const int buf = tseq % RB::n;
                ok = __all_sync(0xffffffffu, mbar_wait(&sfull, tseq & 1, a.status));
                if (!ok) break;
                tc_fence_after();
                const float* sl = reinterpret_cast<const float*>(rbuf(buf) + RB::st) + 32 * cg;
#pragma unroll
                for (int h = 0; h < 2 && ok; ++h) {  // 16 rows at a time
                    float sv[16], dv[16];
                    tmem_ld16(tb + cS + 32 * cg + 16 * h + lo, sv);
                    tmem_ld16(tb + cDP + 32 * cg + 16 * h + lo, dv);
                    tmem_ld_wait();
                    if (h == 1) {
                        tc_fence_before();
                        warp_arrive(&sfree);
                    }
                    uint32_t pk[8], dk[8];
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float4 L = *reinterpret_cast<const float4*>(sl + 16 * h + j);
                        const float4 Dl = *reinterpret_cast<const float4*>(sl + 128 + 16 * h + j);
                        const float p0 = exp2f(fmaf(sv[j], kC, -L.x)), p1 = exp2f(fmaf(sv[j + 1], kC, -L.y));
                        const float p2 = exp2f(fmaf(sv[j + 2], kC, -L.z)), p3 = exp2f(fmaf(sv[j + 3], kC, -L.w));
                        pk[j >> 1] = pack_bf16(p0, p1);
                        pk[(j >> 1) + 1] = pack_bf16(p2, p3);
                        dk[j >> 1] = pack_bf16(p0 * (dv[j] - Dl.x), p1 * (dv[j + 1] - Dl.y));
                        dk[(j >> 1) + 1] = pack_bf16(p2 * (dv[j + 2] - Dl.z), p3 * (dv[j + 3] - Dl.w));
                    }
                    // p^T and ds^T go where the previous tile's products read them
                    if (h == 0 && tseq >= 1) {
                        ok = __all_sync(0xffffffffu, mbar_wait(&pvdone, (tseq - 1) & 1, a.status));
                        if (!ok) break;
                        tc_fence_after();
                    }
                    tmem_st8u(tb + cP + 16 * cg + 8 * h + lo, pk);
                    tmem_st8u(tb + cDS + 16 * cg + 8 * h + lo, dk);
                }
                if (!ok) break;
                tmem_st_wait();
                tc_fence_before();
                warp_arrive(&pfull);
                ++tseq;
            }
            if (!ok) break;
            // the unit's gradients of its 128 keys, columns 16 cg .. + 15
            ok = __all_sync(0xffffffffu, mbar_wait(&pvdone, (tseq - 1) & 1, a.status));
            if (!ok) break;
            tc_fence_after();
            float gvv[16], gkk[16];
            tmem_ld16(tb + cV + 16 * cg + lo, gvv);
            tmem_ld16(tb + cK + 16 * cg + lo, gkk);
            tmem_ld_wait();
            tc_fence_before();
            warp_arrive(&afree);
            float* dkp = nullptr;
            float* dvp = nullptr;
            if (MODE == kExp) {
                const int x = 128 * b + t_;
                if (x < a.m) {
                    dkp = a.slq + (bh * a.m + x) * D;
                    dvp = a.slv + (bh * a.m + x) * D;
                } else if (x >= a.m4 && x < a.m4 + a.k) {
                    const int j = a.expert_idx[(bh * a.m + e) * static_cast<int64_t>(a.k) + (x - a.m4)];
                    dkp = a.gk + (bh * a.N + j) * D;
                    dvp = a.gv + (bh * a.N + j) * D;
                }
            } else {
                const int64_t j = 128LL * b + t_;
                if (j < a.N) {
                    dkp = a.gk + (bh * a.N + j) * D;
                    dvp = a.gv + (bh * a.N + j) * D;
                }
            }
            if (dkp) {
#pragma unroll
                for (int c = 0; c < 16; c += 4) {
                    const float4 kk = make_float4(gkk[c] * kTau, gkk[c + 1] * kTau, gkk[c + 2] * kTau, gkk[c + 3] * kTau);
                    const float4 vv = make_float4(gvv[c], gvv[c + 1], gvv[c + 2], gvv[c + 3]);
                    // reductions (no value returned): nothing waits for them
                    atomicAdd(reinterpret_cast<float4*>(dkp + 16 * cg + c), kk);
                    atomicAdd(reinterpret_cast<float4*>(dvp + 16 * cg + c), vv);
                }
            }
            ++ucount;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tb, 512);
}

// ============================================================================
// Rows kernel
// ============================================================================
// shared memory: row buffers b = 0, 1 at 49 KB b: R, R_lo (LMK), dR; then
// LMK: a ring of RST key stages of K (8 KB) and V (8 KB) rows, 64 keys each;
// EXP: the expert's whole key list (nblk blocks of 64 rows) and then its
// value list, kept while consecutive items share the expert
constexpr int RST = 4;
constexpr size_t RBUF = 3 * TILE + 1024, ROFF_K = 2 * RBUF;
constexpr size_t RSMEM = ROFF_K + RST * 16384 + 1024;
constexpr int RMAXBLK = 8;  // EXP: list blocks of 64 (m4 + k <= 512)
// EXP row buffers hold R and dR only (2 x 32 KB)
constexpr size_t RSMEM_EXP = 2 * 2 * TILE + RMAXBLK * 16384 + 1024;
// TMEM: S buffers at 0, 64; dP at 128, 192; ds (bf16 pairs) at 256, 288; G at 384
constexpr uint32_t rS = 0, rDP = 128, rDS = 256, rG = 384;

template <int MODE>
__device__ __forceinline__ void rows_unit(const BArgs& a, int64_t u, int64_t& bh, int4& item, int& lt, int& nb,
                                          int64_t& c0, int64_t& c1) {
    if (MODE == kExp) {
        item = a.items[u];
        bh = item.w;
        lt = 0;
        nb = a.nblk;
        c0 = c1 = 0;
    } else {
        const int lts = (a.m + 127) / 128;
        bh = u / (static_cast<int64_t>(lts) * a.chunks);
        lt = static_cast<int>((u / a.chunks) % lts);
        const int c = static_cast<int>(u % a.chunks);
        c0 = static_cast<int64_t>(c) * a.chunk_len;
        c1 = min(a.N, c0 + a.chunk_len);
        nb = static_cast<int>((c1 - c0 + 63) / 64);
        item = make_int4(0, 0, 0, 0);
    }
}

template <int MODE>
__global__ void __launch_bounds__(NTB, 1)
    bwd_rows_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tsk, const __grid_constant__ CUtensorMap tsv,
                    const __grid_constant__ CUtensorMap tr, const __grid_constant__ CUtensorMap tdr, BArgs a) {
    // EXP: tk, tv, tsk, tsv: K, V, Lq (bf16), LV (bf16) rows one row high
    //      (the key list gathers); tr, tdr: Q, dO rows one row high.
    // LMK: tk, tv: K, V, 64 rows high; tr, tsk: Lq hi, lo; tdr: dLV (bf16),
    //      128 rows high.
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t rfull[2], rfree[2], kfull[RST], kempty[RST], sfull[2], sfree[2], pfull[2], dsfree[2];
    __shared__ uint64_t gdone, gfree, drain[2], kvfull, kvfree;
    __shared__ uint32_t tmem_base;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t total = MODE == kExp ? *a.nitems : a.units;
    const int64_t u0 = total * blockIdx.x / gridDim.x, u1 = total * (blockIdx.x + 1) / gridDim.x;
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&rfull[b], 1);
            mbar_init(&rfree[b], 1);
            mbar_init(&sfull[b], 1);
            mbar_init(&sfree[b], NRW);
            mbar_init(&pfull[b], NRW);
            mbar_init(&dsfree[b], 1);
        }
        for (int s = 0; s < RST; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&kempty[s], 1);
        }
        mbar_init(&gdone, 1);
        mbar_init(&gfree, NRW);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        mbar_init(&kvfull, 1);
        mbar_init(&kvfree, 2);  // both issuers read the expert's list
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    constexpr size_t RB = MODE == kExp ? 2 * TILE : RBUF;    // row buffer stride
    constexpr size_t DROFF = MODE == kExp ? TILE : 2 * TILE;  // dR within a row buffer
    auto rbuf = [&](int b) { return base + b * RB; };
    auto kst = [&](int s) { return base + ROFF_K + s * 16384; };  // K rows, then V rows at +8 KB
    uint8_t* listk = base + 2 * RB;                                  // EXP: list block j at + 8 KB j
    uint8_t* listv = listk + a.nblk * 8192;

    if (warp == PW) {
        // ---------------------------------- producer ----------------------------------
        int useq = 0, g = 0, changes = 0, cur_e = -1;
        int64_t cur_bh = -1;
        bool ok = true;
        for (int64_t u = u0; u < u1 && ok; ++u) {
            int64_t bh, c0, c1;
            int4 item;
            int lt, nb;
            rows_unit<MODE>(a, u, bh, item, lt, nb, c0, c1);
            if (MODE == kExp && (bh != cur_bh || item.x != cur_e)) {
                // the expert's list, once the MMAs reading the previous one are done
                if (changes > 0) ok = __all_sync(0xffffffffu, mbar_wait(&kvfree, (changes - 1) & 1, a.status));
                if (!ok) break;
                if (lane == 0) mbar_arrive_expect_tx(&kvfull, static_cast<uint32_t>(a.nblk) * 16384u);
                __syncwarp();
                const int32_t* sel = a.expert_idx + (bh * a.m + item.x) * static_cast<int64_t>(a.k);
                for (int gi = lane; gi < a.nblk * 16; gi += 32) {  // list positions 4 gi .. + 3
                    int y[4];
                    bool sh;
                    list_rows4(a, bh, sel, 4 * gi, y, &sh);
                    tma_gather4(listk + 4 * gi * 128, sh ? &tsk : &tk, 0, y[0], y[1], y[2], y[3], &kvfull);
                    tma_gather4(listv + 4 * gi * 128, sh ? &tsv : &tv, 0, y[0], y[1], y[2], y[3], &kvfull);
                }
                cur_bh = bh;
                cur_e = item.x;
                ++changes;
            }
            const int buf = useq & 1;
            if (useq >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&rfree[buf], ((useq >> 1) - 1) & 1, a.status));
            if (!ok) break;
            uint8_t* rb = rbuf(buf);
            if (lane == 0) mbar_arrive_expect_tx(&rfull[buf], (MODE == kExp ? 2 : 3) * TILE);
            __syncwarp();
            if (MODE == kExp) {
                // the item's queries and their dO, in grouped order (rows past
                // the item are masked: those threads' rows are not the item's)
                if (lane == 0) {
                    const int y = static_cast<int>(bh * a.N + item.y);
                    tma_load_2d(rb, &tr, 0, y, &rfull[buf]);
                    tma_load_2d(rb + DROFF, &tdr, 0, y, &rfull[buf]);
                }
            } else if (lane == 0) {
                const int y = static_cast<int>(bh * a.m + 128 * lt);
                tma_load_2d(rb, &tr, 0, y, &rfull[buf]);
                tma_load_2d(rb + TILE, &tsk, 0, y, &rfull[buf]);
                tma_load_2d(rb + 2 * TILE, &tdr, 0, y, &rfull[buf]);
            }
            for (int j = 0; j < nb && ok && MODE == kLmk; ++j, ++g) {
                const int s = g % RST;
                if (g >= RST) ok = __all_sync(0xffffffffu, mbar_wait(&kempty[s], ((g / RST) - 1) & 1, a.status));
                if (!ok) break;
                if (lane == 0) mbar_arrive_expect_tx(&kfull[s], 16384);
                __syncwarp();
                uint8_t* ks = kst(s);
                if (lane == 0) {
                    const int y = static_cast<int>(bh * a.N + c0 + 64 * j);
                    tma_load_2d(ks, &tk, 0, y, &kfull[s]);
                    tma_load_2d(ks + 8192, &tv, 0, y, &kfull[s]);
                }
            }
            ++useq;
        }
        if (lane == 0) {
            if (changes > 0) mbar_drain(&kvfull, (changes - 1) & 1);
            for (int b = 0; b < 2; ++b) {
                const int arms = useq > b ? (useq - b + 1) / 2 : 0;
                if (arms > 0) mbar_drain(&rfull[b], (arms - 1) & 1);
            }
            for (int s = 0; s < RST; ++s) {
                const int arms = g > s ? (g - s + RST - 1) / RST : 0;
                if (arms > 0) mbar_drain(&kfull[s], (arms - 1) & 1);
            }
        }
    } else if (warp == PW + 1 || warp == PW + 2) {
        // ------------------- MMA issuers: S and dP (PW + 1), G (PW + 2) -------------------
        if (lane == 0) {
            const bool gi = warp == PW + 2;
            const uint32_t idS = idesc_bf16(128, 64, false), idG = idesc_bf16(128, 64, true);
            int useq = 0, g = 0, changes = 0, cur_e = -1;
            int64_t cur_bh = -1;
            bool ok = true;
            for (int64_t u = u0; u < u1 && ok; ++u) {
                int64_t bh, c0, c1;
                int4 item;
                int lt, nb;
                rows_unit<MODE>(a, u, bh, item, lt, nb, c0, c1);
                const int buf = useq & 1;
                if (MODE == kExp && (bh != cur_bh || item.x != cur_e)) {
                    // release the previous list (once this thread's MMAs on it are
                    // done), then wait for this expert's; before the unit's rows,
                    // which the producer loads only after the list
                    if (changes > 0) mma_commit(&kvfree);
                    if (!(ok = mbar_wait(&kvfull, changes & 1, a.status))) break;
                    cur_bh = bh;
                    cur_e = item.x;
                    ++changes;
                }
                if (!(ok = mbar_wait(&rfull[buf], (useq >> 1) & 1, a.status))) break;
                const uint32_t rs = smem_u32(rbuf(buf));
                if (!gi) {
                    for (int j = 0; j < nb && ok; ++j, ++g) {
                        const int s = g % RST, sb = g & 1;
                        if (MODE == kLmk && !(ok = mbar_wait(&kfull[s], (g / RST) & 1, a.status))) break;
                        // the rows have read block g - 2's S and dP
                        if (g >= 2 && !(ok = mbar_wait(&sfree[sb], ((g >> 1) - 1) & 1, a.status))) break;
                        tc_fence_after();
                        const uint32_t ks = MODE == kExp ? smem_u32(listk + j * 8192) : smem_u32(kst(s));
                        const uint32_t vs = MODE == kExp ? smem_u32(listv + j * 8192) : ks + 8192;
                        mma_ss_k64(tb + rS + 64 * sb, sdesc_sw128(rs), sdesc_sw128(ks), idS, 0u);
                        if (MODE == kLmk)
                            mma_ss_k64(tb + rS + 64 * sb, sdesc_sw128(rs + TILE), sdesc_sw128(ks), idS, 1u);
                        mma_ss_k64(tb + rDP + 64 * sb, sdesc_sw128(rs + DROFF), sdesc_sw128(vs), idS, 0u);
                        mma_commit(&sfull[sb]);
                    }
                } else {
                    // G += ds(j) K(j) (the first block of the unit overwrites G)
                    for (int j = 0; j < nb && ok; ++j, ++g) {
                        const int s = g % RST, sb = g & 1;
                        if (!(ok = mbar_wait(&pfull[sb], (g >> 1) & 1, a.status))) break;
                        if (j == 0 && useq >= 1 && !(ok = mbar_wait(&gfree, (useq - 1) & 1, a.status))) break;
                        tc_fence_after();
                        const uint64_t kmn = sdesc_sw128(smem_u32(MODE == kExp ? listk + j * 8192 : kst(s)));
                        mma_ts_k64(tb + rG, tb + rDS + 32 * sb, kmn, idG, j == 0 ? 0u : 1u);
                        mma_commit(&dsfree[sb]);
                        if (MODE == kLmk) mma_commit(&kempty[s]);  // (S and dP of the block completed before pfull)
                    }
                    if (!ok) break;
                    mma_commit(&gdone);
                    mma_commit(&rfree[buf]);
                }
                if (!ok) break;
                ++useq;
            }
            mma_drain(&drain[gi ? 1 : 0]);
        }
    } else {
        // ------------------------------- row threads -------------------------------
        // warp w: TMEM lanes 32 (w % 4) .. + 31 (the unit's rows), key
        // columns 16 (w / 4) .. + 15 of each 64-key block, and columns
        // 16 (w / 4) .. + 15 of G
        static_assert(RW == 4, "16 of each block's 64 columns per row warp");
        const int t = (warp & 3) * 32 + lane;  // TMEM lane = row of the unit
        const int cg = warp >> 2;
        const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int useq = 0, g = 0;
        bool ok = true;
        for (int64_t u = u0; u < u1 && ok; ++u) {
            int64_t bh, c0, c1;
            int4 item;
            int lt, nb;
            rows_unit<MODE>(a, u, bh, item, lt, nb, c0, c1);
            // this row's statistics and where its gradient goes
            bool row_ok;
            int64_t orow;
            int64_t srow;  // where its statistics are (EXP: grouped order)
            if (MODE == kExp) {
                row_ok = t < item.z;
                const int n = row_ok ? a.perm[bh * a.N + item.y + t] : 0;
                orow = bh * a.N + n;
                srow = bh * a.N + item.y + (row_ok ? t : 0);
            } else {
                const int li = 128 * lt + t;
                row_ok = li < a.m;
                orow = bh * a.m + (row_ok ? li : 0);
                srow = orow;
            }
            const float L = row_ok ? a.lse[srow] : INFINITY;
            const float Dl = row_ok ? a.delta[srow] : 0.f;
            const int nkeys = MODE == kExp ? a.m4 + a.k : static_cast<int>(c1 - c0);  // valid list positions / keys
            for (int j = 0; j < nb && ok; ++j, ++g) {
                const int sb = g & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&sfull[sb], (g >> 1) & 1, a.status));
                if (!ok) break;
                tc_fence_after();
                float sv[16], dv[16];
                tmem_ld16(tb + rS + 64 * sb + 16 * cg + lo, sv);
                tmem_ld16(tb + rDP + 64 * sb + 16 * cg + lo, dv);
                tmem_ld_wait();
                tc_fence_before();
                warp_arrive(&sfree[sb]);
                const int x0 = 64 * j + 16 * cg;
                uint32_t pk[8];
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    const int x = x0 + c;
                    // EXP: the unused positions [m, m4) and those past the list; LMK: past the chunk
                    const bool v0 = x < nkeys && (MODE == kLmk || x < a.m || x >= a.m4);
                    const bool v1 = x + 1 < nkeys && (MODE == kLmk || x + 1 < a.m || x + 1 >= a.m4);
                    const float p0 = v0 ? exp2f(fmaf(sv[c], kC, -L)) : 0.f;
                    const float p1 = v1 ? exp2f(fmaf(sv[c + 1], kC, -L)) : 0.f;
                    pk[c >> 1] = pack_bf16(p0 * (dv[c] - Dl), p1 * (dv[c + 1] - Dl));
                }
                if (g >= 2) {  // ds buffer sb was last read by G of block g - 2
                    ok = __all_sync(0xffffffffu, mbar_wait(&dsfree[sb], ((g >> 1) - 1) & 1, a.status));
                    if (!ok) break;
                }
                tc_fence_after();
                tmem_st8u(tb + rDS + 32 * sb + 8 * cg + lo, pk);
                tmem_st_wait();
                tc_fence_before();
                warp_arrive(&pfull[sb]);
            }
            if (!ok) break;
            ok = __all_sync(0xffffffffu, mbar_wait(&gdone, useq & 1, a.status));
            if (!ok) break;
            tc_fence_after();
            float gg[16];
            tmem_ld16(tb + rG + 16 * cg + lo, gg);
            tmem_ld_wait();
            tc_fence_before();
            warp_arrive(&gfree);
            if (row_ok) {
                if (MODE == kExp) {
                    // dQ of the query: its expert attention's share and the
                    // pooling's share of the (complete) dLq of its windows
#pragma unroll
                    for (int c = 0; c < 16; ++c) gg[c] *= kTau;
                    pool_windows_of(a.N, a.gh, a.gw, a.p, a.m, orow - bh * a.N, [&](int i, float wgt) {
                        const float4* s4 = reinterpret_cast<const float4*>(a.slq + (bh * a.m + i) * D + 16 * cg);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float4 v = s4[c];
                            gg[4 * c] = fmaf(v.x, wgt, gg[4 * c]);
                            gg[4 * c + 1] = fmaf(v.y, wgt, gg[4 * c + 1]);
                            gg[4 * c + 2] = fmaf(v.z, wgt, gg[4 * c + 2]);
                            gg[4 * c + 3] = fmaf(v.w, wgt, gg[4 * c + 3]);
                        }
                    });
                    float4* dst = reinterpret_cast<float4*>(a.gk + orow * D + 16 * cg);
#pragma unroll
                    for (int c = 0; c < 16; c += 4) dst[c / 4] = make_float4(gg[c], gg[c + 1], gg[c + 2], gg[c + 3]);
                } else {  // dLq of the landmark, summed over the key chunks
                    float4* dst = reinterpret_cast<float4*>(a.gv + orow * D + 16 * cg);
#pragma unroll
                    for (int c = 0; c < 16; c += 4)
                        atomicAdd(dst + c / 4,
                                  make_float4(gg[c] * kTau, gg[c + 1] * kTau, gg[c + 2] * kTau, gg[c + 3] * kTau));
                }
            }
            ++useq;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tb, 512);
}

template <class Kern>
cudaError_t launch6(Kern kern, size_t smem, int64_t grid, const CUtensorMap* m, const BArgs& a, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (grid <= 0) return cudaSuccess;
    kern<<<static_cast<unsigned>(grid), NTB, smem, st>>>(m[0], m[1], m[2], m[3], m[4], m[5], a);
    return cudaGetLastError();
}

}  // namespace

bool backward_tc_supported(const Plan& p) {
    // the key list of an expert fits the key kernel's 128-key blocks and the
    // rows kernel's staged 64-key blocks; the landmarks fit two 128-row tiles
    return p.s.m <= 256 && p.s.s_route == 1 && p.s.BH * p.s.N < (int64_t(1) << 31) &&
           p.s.BH * (p.s.m + 1) < (int64_t(1) << 31);
}

// EXP maps and arguments shared by the two expert-side launches
static int exp_setup(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                     const __nv_bfloat16* V, const __nv_bfloat16* dO, const int32_t* expert_idx, const float* st_lse,
                     const float* st_delta, CUtensorMap* maps, BArgs& a) {
    a = BArgs{};
    a.items = w.items;
    a.nitems = w.nitems;
    a.expoff = w.expoff;
    a.perm = w.perm;
    a.expert_idx = expert_idx;
    a.lse = st_lse;
    a.delta = st_delta;
    a.status = w.status;
    a.N = p.s.N;
    a.m = p.s.m;
    a.k = p.s.k;
    a.m4 = (p.s.m + 3) & ~3;
    a.gh = p.s.gh;
    a.gw = p.s.gw;
    a.p = p.s.p;
    const uint64_t rows = static_cast<uint64_t>(p.s.BH) * p.s.N, lrows = static_cast<uint64_t>(p.s.BH) * p.s.m;
    return make_row_tmap(&maps[0], K, rows, 1) && make_row_tmap(&maps[1], V, rows, 1) &&
           make_row_tmap(&maps[2], w.lqhi, lrows, 1) && make_row_tmap(&maps[3], w.lvbf, lrows, 1) &&
           make_row_tmap(&maps[4], Q, rows, 1) && make_row_tmap(&maps[5], dO, rows, 1);
}

cudaError_t launch_backward_tc_expert_keys(const Plan& p, const Work& w, const __nv_bfloat16* Qg,
                                           const __nv_bfloat16* K, const __nv_bfloat16* V, const __nv_bfloat16* dOg,
                                           const int32_t* expert_idx, const float* st_lse, const float* st_delta,
                                           float* dK, float* dV, float* dlq, float* dlv, cudaStream_t st) {
    BArgs a;
    CUtensorMap maps[6];
    if (!exp_setup(p, w, Qg, K, V, dOg, expert_idx, st_lse, st_delta, maps, a)) return cudaErrorInvalidValue;
    // the row tiles: 128 consecutive rows of the grouped copies
    const uint64_t rows = static_cast<uint64_t>(p.s.BH) * p.s.N;
    if (!make_row_tmap(&maps[4], Qg, rows, 128) || !make_row_tmap(&maps[5], dOg, rows, 128)) return cudaErrorInvalidValue;
    // one unit per (head, expert, 128-key block of its list)
    a.nblk = (a.m4 + a.k + 127) / 128;
    a.units = p.s.BH * static_cast<int64_t>(p.s.m) * a.nblk;
    a.gk = dK;
    a.gv = dV;
    a.slq = dlq;
    a.slv = dlv;
    return launch6(bwd_keys_kernel<kExp>, KSMEM, std::min<int64_t>(device_sms(), a.units), maps, a, st);
}

cudaError_t launch_backward_tc_expert_rows(const Plan& p, const Work& w, const __nv_bfloat16* Qg,
                                           const __nv_bfloat16* K, const __nv_bfloat16* V, const __nv_bfloat16* dOg,
                                           const int32_t* expert_idx, const float* st_lse, const float* st_delta,
                                           const float* dlq, float* dQ, cudaStream_t st) {
    BArgs a;
    CUtensorMap maps[6];
    if (!exp_setup(p, w, Qg, K, V, dOg, expert_idx, st_lse, st_delta, maps, a)) return cudaErrorInvalidValue;
    // an item's rows: 128 consecutive rows of the grouped copies
    const uint64_t rows = static_cast<uint64_t>(p.s.BH) * p.s.N;
    if (!make_row_tmap(&maps[4], Qg, rows, 128) || !make_row_tmap(&maps[5], dOg, rows, 128)) return cudaErrorInvalidValue;
    // one unit per item, over the expert's list in 64-key blocks
    a.nblk = (a.m4 + a.k + 63) / 64;
    a.gk = dQ;
    a.slq = const_cast<float*>(dlq);  // (read: the pooling's share)
    return launch6(bwd_rows_kernel<kExp>, RSMEM_EXP, device_sms(), maps, a, st);
}

cudaError_t launch_backward_tc_landmark(const Plan& p, const Work& w, const __nv_bfloat16* K, const __nv_bfloat16* V,
                                        const __nv_bfloat16* dlv_bf16, const float* lse2, const float* delta,
                                        float* dK, float* dV, float* dlq, cudaStream_t st) {
    BArgs a{};
    a.lse = lse2;
    a.delta = delta;
    a.status = w.status;
    a.N = p.s.N;
    a.m = p.s.m;
    a.k = p.s.k;
    a.m4 = (p.s.m + 3) & ~3;
    const uint64_t rows = static_cast<uint64_t>(p.s.BH) * p.s.N, lrows = static_cast<uint64_t>(p.s.BH) * p.s.m;
    const int sms = device_sms();
    // dK, dV: one unit per (head, 128 keys), rows = the head's landmarks
    {
        CUtensorMap mk, mv, mlo, mhi, mdl;
        if (!make_row_tmap(&mk, K, rows, 128) || !make_row_tmap(&mv, V, rows, 128) ||
            !make_row_tmap(&mhi, w.lqhi, lrows, 128) || !make_row_tmap(&mlo, w.lqlo, lrows, 128) ||
            !make_row_tmap(&mdl, dlv_bf16, lrows, 128))
            return cudaErrorInvalidValue;
        const CUtensorMap maps[6] = {mk, mv, mlo, mlo, mhi, mdl};
        a.units = p.s.BH * ((p.s.N + 127) / 128);
        a.gk = dK;
        a.gv = dV;
        cudaError_t e = launch6(bwd_keys_kernel<kLmk>, KSMEM, std::min<int64_t>(sms, a.units), maps, a, st);
        if (e != cudaSuccess) return e;
    }
    // dLq: one unit per (head, 128 landmarks, chunk of keys), about 4 units per SM
    {
        CUtensorMap mk, mv, mlo, mhi, mdl;
        if (!make_row_tmap(&mk, K, rows, 64) || !make_row_tmap(&mv, V, rows, 64) ||
            !make_row_tmap(&mhi, w.lqhi, lrows, 128) || !make_row_tmap(&mlo, w.lqlo, lrows, 128) ||
            !make_row_tmap(&mdl, dlv_bf16, lrows, 128))
            return cudaErrorInvalidValue;
        const CUtensorMap maps[6] = {mk, mv, mlo, mlo, mhi, mdl};
        const int lts = (p.s.m + 127) / 128;
        int64_t chunks = std::max<int64_t>(1, (4LL * sms + p.s.BH * lts - 1) / (p.s.BH * lts));
        chunks = std::min<int64_t>(chunks, (p.s.N + 63) / 64);
        a.chunk_len = ((p.s.N + chunks - 1) / chunks + 63) / 64 * 64;
        a.chunks = static_cast<int>((p.s.N + a.chunk_len - 1) / a.chunk_len);
        a.units = p.s.BH * lts * static_cast<int64_t>(a.chunks);
        a.gv = dlq;
        return launch6(bwd_rows_kernel<kLmk>, RSMEM, std::min<int64_t>(sms, a.units), maps, a, st);
    }
}

}  // namespace mita
