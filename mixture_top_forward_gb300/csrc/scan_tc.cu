// Stage 2 on the tensor cores: the landmark scan, and the sample pilots that
// give it its top-k thresholds.
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造": each landmark query is matched
// against every key; its k best keys form its routed expert, and the same
// landmark's cross-attention over the whole sequence gives the shared-expert
// value LV_i. One pass over K and V does both.
//
// One CTA per (head, chunk of keys); it holds all m <= 256 landmark queries
// (NL = 1 or 2 tiles of 128 rows) in shared memory as a bf16 hi/lo pair,
// hi = bf16(Lq), lo = bf16(Lq - hi), so that S = Lq_hi K^T + Lq_lo K^T (two
// accumulating MMAs) matches the fp32 landmark to ~2^-16 relative: exact
// enough for the top-k comparisons.
//   warp 0:        TMEM allocation; lane 0: TMA producer of 128-key tiles of
//                  K (3-4 stage ring); lane 1: TMA producer of V tiles (2-3
//                  stages; full scans only);
//   warps 1..NL (lane 0): one MMA issuer per landmark tile L: S_L = Lq_L K^T
//                  into TMEM (two buffers);
//   warp NL+1 (lane 0, full scans only): MMA issuer of O_L += P_L V, one tile
//                  behind (a tcgen05.mma holds its issuing thread for about a
//                  hundred cycles, so independent chains from separate warps
//                  keep the tensor pipe busy);
//   warps NL+2..:  one warpgroup (4 consecutive warps: warp w reads TMEM lane
//                  quarter w % 4) per landmark tile, one thread per landmark.
//                  Per 64-key tile a thread loads its 64 scores and offers
//                  them to its landmark's candidate buffers: an 8-column
//                  group whose maximum reaches the threshold goes out whole
//                  as a record in pilot scans (the select expands it), and
//                  key by key otherwise, or once the records are full
//                  (topk.cuh: append when the 64-bit order key reaches the
//                  threshold, warp-cooperative compaction on overflow); in
//                  full scans it also runs the online softmax (lazy running
//                  max), writes P (bf16) into TMEM and leaves a (max, sum,
//                  o[64]) partial at the end of the chunk. Dense levels
//                  write every raw logit instead of candidates.
// Keys are read through a 3-D tensor map (row, head) whose row stride may be
// > 1: a pilot scan reads every stride-th key of each head. A pilot does only
// the top-k part; its k-th best order key (select.cu) is a lower bound of the
// true k-th best of the whole head, because the sample keys are keys of the
// head, so the next scan may start from it and still keep every key of the
// true top k. Every wait is bounded (umma.cuh).
#include "tensormap.cuh"
#include "topk.cuh"
#include "umma.cuh"

namespace mita {

namespace {

using namespace umma;

constexpr float kC = 0.125f * kLog2e;  // tau * log2(e)
constexpr float kLazy = 8.0f;
constexpr uint32_t kIdescS = idesc_bf16(128, 64, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 64, true);

struct ScanArgs {
    const __nv_bfloat16* lqhi;
    const __nv_bfloat16* lqlo;
    const uint64_t* theta;  // [BH][m] starting thresholds, or null (0: accept everything)
    float* part;            // [BH][chunks][m][68], full scans only
    uint64_t* cand;         // [BH][chunks][m][cap]
    int* ccount;            // [BH][chunks][m]
    uint32_t* ridx;         // [BH][chunks][m][rcap] group records: sample index of column 0 of the group
    float* rval;            // [BH][chunks][m][rcap][8] group records: the group's raw logits
    int* rcount;            // [BH][chunks][m]
    float* dense;           // dense top-k: [BH][m][ld] raw logits, else null
    int64_t ld;             // row stride of dense
    int* status;
    const int* skip;    // [BH] or null: a head whose entry is 0 is not scanned (its CTAs return at once)
    int64_t S;          // keys (samples) per head in this scan
    int64_t stride;     // key index of sample s is s * stride
    int64_t chunk_len;  // multiple of 128
    int chunks, cap, rcap, m, k;
};

template <bool FULL, int NL>
struct Cfg {
    static constexpr int KT = 64;                     // keys per tile
    static constexpr int TB = KT * 128;               // bytes of one K or V tile
    static constexpr int KST = NL == 1 ? 4 : 6;       // K ring stages
    static constexpr int VST = FULL ? (NL == 1 ? 3 : 4) : 0;  // V ring stages
    static constexpr int MINB = NL == 1 ? 2 : 1;      // CTAs per SM
    static constexpr int NT = 32 * (NL + 2) + NL * 128;  // producer, NL S issuers, P.V issuer, rows
    static constexpr int ROW0 = NL + 2;                  // first row warp
    static constexpr size_t OFF_LQLO = NL * 16384;
    static constexpr size_t OFF_K = 2 * NL * 16384;
    static constexpr size_t OFF_V = OFF_K + KST * TB;
    static constexpr size_t OFF_HIST = OFF_V + VST * TB;
    static constexpr size_t SMEM = OFF_HIST + NL * 4 * 1024 + 1024;
    // TMEM per landmark tile L (256 columns apart): S buffers at +0 and +64, O at +128,
    // P (bf16 pairs) buffers at +192 and +224
    static constexpr uint32_t TCOLS = NL * 256;
};

// Score of an order key (the inverse of topk_key's float mapping); -inf for 0.
__device__ __forceinline__ float key_score(uint64_t key) {
    if (key == 0) return -INFINITY;
    uint32_t u = static_cast<uint32_t>(key >> 32);
    u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
    return __uint_as_float(u);
}

struct Bars {
    uint64_t* vfull;
    uint64_t* vempty;
    uint64_t* pfull;   // [NL][2]
    uint64_t* pvdone;  // [NL][2]
};

// Issues O_L += P_L(i) V(i) for every landmark tile L of key tile i (P.V issuer).
template <class C, int NL>
__device__ __forceinline__ bool issue_pv(const ScanArgs& a, uint8_t* base, uint32_t tb, int i, const Bars& b) {
    const int vs = i % C::VST, pbuf = i & 1;
    if (!mbar_wait(&b.vfull[vs], (i / C::VST) & 1, a.status)) return false;
    const uint64_t vd = sdesc_sw128(smem_u32(base + C::OFF_V + vs * C::TB));
    for (int l = 0; l < NL; ++l) {
        if (!mbar_wait(&b.pfull[l * 2 + pbuf], (i >> 1) & 1, a.status)) return false;
        tc_fence_after();
        mma_ts_k64(tb + l * 256 + 128, tb + l * 256 + 192 + pbuf * 32, vd, kIdescPV, i > 0 ? 1u : 0u);
        mma_commit(&b.pvdone[l * 2 + pbuf]);
    }
    mma_commit(&b.vempty[vs]);
    return true;
}

template <bool FULL, int NL>
__global__ void __launch_bounds__(Cfg<FULL, NL>::NT, Cfg<FULL, NL>::MINB)
    scan_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, ScanArgs a) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    using C = Cfg<FULL, NL>;
    constexpr int KT = C::KT;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t kfull[C::KST], kempty[C::KST];
    __shared__ uint64_t vfull[C::VST > 0 ? C::VST : 1], vempty[C::VST > 0 ? C::VST : 1];
    __shared__ uint64_t sfull[NL * 2], sfree[NL * 2], pfull[NL * 2], pvdone[NL * 2], drain;
    __shared__ uint32_t tmem_base;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.chunks));
    const int64_t bh = blockIdx.x / static_cast<unsigned>(a.chunks);
    if (a.skip && a.skip[bh] == 0) return;  // (uniform: before any barrier or TMEM allocation)
    const int64_t s0 = static_cast<int64_t>(c) * a.chunk_len;
    const int64_t s1 = min(a.S, s0 + a.chunk_len);
    const int T = static_cast<int>((s1 - s0 + KT - 1) / KT);

    if (tid == 0) {
        for (int i = 0; i < C::KST; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], NL);  // one commit per S issuer
        }
        for (int i = 0; i < C::VST; ++i) {
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], 1);
        }
        for (int l = 0; l < NL * 2; ++l) {
            mbar_init(&sfull[l], 1);
            mbar_init(&sfree[l], 4);  // every row warp arrives after reading S
            mbar_init(&pfull[l], 4);  // every row warp arrives after writing its P rows
            mbar_init(&pvdone[l], 1);
        }
        mbar_init(&drain, FULL ? NL + 1 : NL);  // exit path: one commit per MMA issuer
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base, C::TCOLS);
    {   // landmark queries of this head, hi and lo, rows >= m zero
        const uint32_t hb = smem_u32(base), lb = smem_u32(base + C::OFF_LQLO);
        for (int x = tid; x < NL * 128 * 8; x += C::NT) {
            const int row = x >> 3, ch = x & 7;
            const uint32_t off = swz128(row, ch);
            if (row < a.m) {
                const int64_t src = (bh * a.m + row) * D + ch * 8;
                cp_async16(hb + off, a.lqhi + src);
                cp_async16(lb + off, a.lqlo + src);
            } else {
                *reinterpret_cast<uint4*>(base + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(base + C::OFF_LQLO + off) = make_uint4(0, 0, 0, 0);
            }
        }
        cp_async_wait_all();
        fence_proxy_async();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const Bars bars{vfull, vempty, pfull, pvdone};

    if (warp == 0) {
        // ---------------- K producer (lane 0) ----------------
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < T; ++i) {
                const int st = i % C::KST;
                if (i >= C::KST && !mbar_wait(&kempty[st], ((i / C::KST) & 1) ^ 1, a.status)) break;
                mbar_arrive_expect_tx(&kfull[st], C::TB);
                tma_load_3d(base + C::OFF_K + st * C::TB, &tk, 0, static_cast<int>(s0 + i * KT),
                            static_cast<int>(bh), &kfull[st]);
                ++issued;
            }
            for (int st = 0; st < C::KST; ++st) {  // exit: the last load of every stage has landed
                const int arms = issued > st ? (issued - st + C::KST - 1) / C::KST : 0;
                if (arms > 0) mbar_drain(&kfull[st], (arms - 1) & 1);
            }
        }
        if constexpr (FULL) {
            // ---------------- V producer (lane 1) ----------------
            if (lane == 1) {
                int issued = 0;
                for (int i = 0; i < T; ++i) {
                    const int st = i % C::VST;
                    if (i >= C::VST && !mbar_wait(&vempty[st], ((i / C::VST) & 1) ^ 1, a.status)) break;
                    mbar_arrive_expect_tx(&vfull[st], C::TB);
                    tma_load_3d(base + C::OFF_V + st * C::TB, &tv, 0, static_cast<int>(s0 + i * KT),
                                static_cast<int>(bh), &vfull[st]);
                    ++issued;
                }
                for (int st = 0; st < C::VST; ++st) {
                    const int arms = issued > st ? (issued - st + C::VST - 1) / C::VST : 0;
                    if (arms > 0) mbar_drain(&vfull[st], (arms - 1) & 1);
                }
            }
        }
    } else if (warp <= NL) {
        // ---------------- S issuer of landmark tile L = warp - 1 ----------------
        if (lane == 0) {
            const int l = warp - 1;
            const uint64_t hd = sdesc_sw128(smem_u32(base + l * 16384));
            const uint64_t ld = sdesc_sw128(smem_u32(base + C::OFF_LQLO + l * 16384));
            for (int i = 0; i < T; ++i) {
                const int st = i % C::KST, sb = i & 1;
                if (!mbar_wait(&kfull[st], (i / C::KST) & 1, a.status)) break;
                // the rows have read S buffer sb of tile i-2
                if (i >= 2 && !mbar_wait(&sfree[l * 2 + sb], ((i >> 1) - 1) & 1, a.status)) break;
                tc_fence_after();
                const uint64_t kd = sdesc_sw128(smem_u32(base + C::OFF_K + st * C::TB));
                const uint32_t tS = tb + l * 256 + sb * KT;
                mma_ss_k64(tS, hd, kd, kIdescS, 0u);
                mma_ss_k64(tS, ld, kd, kIdescS, 1u);
                mma_commit(&sfull[l * 2 + sb]);
                mma_commit(&kempty[st]);
            }
            mma_drain(&drain);  // exit: this issuer's MMAs are done
        }
    } else if (warp == NL + 1) {
        // ---------------- P.V issuer ----------------
        if constexpr (FULL) {
            if (lane == 0) {
                for (int i = 0; i < T; ++i)
                    if (!issue_pv<C, NL>(a, base, tb, i, bars)) break;
                mma_drain(&drain);
            }
        }
    } else {
        // ---------------- landmark rows: top-k filter and softmax ----------------
        const int L = (warp - C::ROW0) >> 2;
        const int t = (warp & 3) * 32 + lane;  // TMEM lane = landmark row in the tile
        const int li = L * 128 + t;
        const bool row_ok = li < a.m;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tO = tb + L * 256 + 128;
        const int64_t slot = (bh * a.chunks + c) * a.m + (row_ok ? li : 0);
        uint64_t* buf = a.cand + slot * static_cast<int64_t>(a.cap);
        uint32_t* rix = a.ridx + slot * static_cast<int64_t>(a.rcap);
        float4* rvl = reinterpret_cast<float4*>(a.rval) + slot * static_cast<int64_t>(a.rcap) * 2;
        int rc = 0;  // records so far
        uint64_t theta = (a.theta && row_ok) ? a.theta[bh * a.m + li] : 0;
        float theta_s = key_score(theta);
        int cnt = 0;
        unsigned* hist = reinterpret_cast<unsigned*>(base + C::OFF_HIST + (warp - C::ROW0) * 1024);
        float mrun = -INFINITY, lrun = 0.f;
        bool ok = true;
        for (int i = 0; i < T; ++i) {
            const int sb = i & 1;
            // waits are made warp-uniform (TMEM loads and stores are warp-wide);
            // the warps of the group run on their own, so nothing blocks unboundedly
            ok = __all_sync(0xffffffffu, mbar_wait(&sfull[L * 2 + sb], (i >> 1) & 1, a.status));
            if (!ok) break;
            tc_fence_after();
            float s[KT];
            tmem_ld32(tb + L * 256 + sb * KT + lane_off, s);
            tmem_ld32(tb + L * 256 + sb * KT + lane_off + 32, s + 32);
            tmem_ld_wait();
            tc_fence_before();
            warp_arrive(&sfree[L * 2 + sb]);
            const int64_t col0 = s0 + static_cast<int64_t>(i) * KT;
            const int nvalid = static_cast<int>(s1 - col0 < KT ? s1 - col0 : KT);
            if (nvalid < KT) {  // last, partial tile of the chunk (warp-uniform)
#pragma unroll
                for (int col = 0; col < KT; ++col) s[col] = col < nvalid ? s[col] : -INFINITY;
            }
            // raw maxima per 8-column group; a group can only hold a candidate
            // if its maximum reaches the threshold (s_raw >= 8 theta_s is exact:
            // tau = 1/8 is a power of two)
            static_assert(KT == 64, "eight groups of eight columns");
            float gm[KT / 8];
#pragma unroll
            for (int g = 0; g < KT / 8; ++g) {
                const float* v = s + 8 * g;
                gm[g] = fmax3(fmax3(v[0], v[1], v[2]), fmax3(v[3], v[4], v[5]), fmaxf(v[6], v[7]));
            }
            const float bmax = fmax3(fmax3(gm[0], gm[1], gm[2]), fmax3(gm[3], gm[4], gm[5]), fmaxf(gm[6], gm[7]));

            if (a.dense) {  // (uniform) dense top-k: every logit of the row goes out
                if (row_ok) {
                    float* dst = a.dense + (bh * a.m + li) * a.ld + col0;
                    if (nvalid == KT) {
#pragma unroll
                        for (int q = 0; q < KT; q += 4)
                            *reinterpret_cast<float4*>(dst + q) = make_float4(s[q], s[q + 1], s[q + 2], s[q + 3]);
                    } else {
#pragma unroll
                        for (int q = 0; q < KT; ++q)
                            if (q < nvalid) dst[q] = s[q];
                    }
                }
            } else {
            // top-k candidates (compaction first if this tile could overflow a buffer)
            unsigned need = __ballot_sync(0xffffffffu, row_ok && cnt + nvalid > a.cap);
            while (need) {
                const int src = __ffs(need) - 1;
                need &= need - 1;
                uint64_t* b = reinterpret_cast<uint64_t*>(
                    __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(buf), src));
                const int bc = __shfl_sync(0xffffffffu, cnt, src);
                const uint64_t kth = warp_compact_topk(b, bc, a.k, hist);
                if (lane == src) {
                    cnt = a.k;
                    theta = kth + 1;
                    theta_s = key_score(kth);
                }
            }
            // masked columns hold -inf: never let them through, even while the
            // threshold is still -inf (every finite score passes -FLT_MAX)
            const float thr = fmaxf(theta_s * 8.0f, -3.402823466e38f);
            if (row_ok && bmax >= thr) {
                // A group whose maximum reaches the threshold goes out whole as
                // a record (its first sample index and its 8 raw logits; the
                // select keeps the ones at or above the threshold). Once the
                // landmark's records are full, its keys go one by one: a lane
                // entering a group stashes the group's 8 scores in its own
                // 32-byte slot of the warp's scratch (the compaction histogram,
                // idle here), so each hit is one shared-memory load.
                float* slot = reinterpret_cast<float*>(hist) + lane * 8;
#pragma unroll
                for (int g = 0; g < KT / 8; ++g) {
                    if (!FULL && gm[g] >= thr && rc < a.rcap) {  // (pilot scans only)
                        rix[rc] = static_cast<uint32_t>(col0 + 8 * g);
                        rvl[2 * rc] = make_float4(s[8 * g], s[8 * g + 1], s[8 * g + 2], s[8 * g + 3]);
                        rvl[2 * rc + 1] = make_float4(s[8 * g + 4], s[8 * g + 5], s[8 * g + 6], s[8 * g + 7]);
                        ++rc;
                    } else if (gm[g] >= thr) {
                        reinterpret_cast<float4*>(slot)[0] =
                            make_float4(s[8 * g], s[8 * g + 1], s[8 * g + 2], s[8 * g + 3]);
                        reinterpret_cast<float4*>(slot)[1] =
                            make_float4(s[8 * g + 4], s[8 * g + 5], s[8 * g + 6], s[8 * g + 7]);
                        unsigned msk = 0;
#pragma unroll
                        for (int j = 0; j < 8; ++j) msk |= (s[8 * g + j] >= thr ? 1u : 0u) << j;
                        while (msk) {
                            const int j = __ffs(msk) - 1;
                            msk &= msk - 1;
                            const uint64_t key =
                                topk_key(slot[j] * 0.125f, static_cast<uint32_t>((col0 + 8 * g + j) * a.stride));
                            if (key >= theta) buf[cnt++] = key;
                        }
                    }
                }
            }
            }
            if constexpr (FULL) {
                const float bm2 = bmax * kC;
                const float mnew = (bm2 > mrun + kLazy) ? bm2 : mrun;
                const float alpha = exp2f(mrun - mnew);
                // packed pairs: one f32x2 FMA forms two exponents, one f32x2 add
                // accumulates two weights
                const float2 c2 = make_float2(kC, kC), m2 = make_float2(-mnew, -mnew);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
#pragma unroll
                for (int col = 0; col < KT; col += 2) {
                    const float2 x = __ffma2_rn(make_float2(s[col], s[col + 1]), c2, m2);
                    s[col] = exp2f(x.x);
                    s[col + 1] = exp2f(x.y);
                    acc[(col >> 1) & 3] = __fadd2_rn(acc[(col >> 1) & 3], make_float2(s[col], s[col + 1]));
                }
                const float sum = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
                lrun = lrun * alpha + sum;
                const int pb = L * 2 + sb;
                // this warp's rows of O need rescaling only when a running max
                // grew by more than 2^8 (rare); that needs PV(i-1) done
                const bool rescale = i > 0 && __any_sync(0xffffffffu, alpha != 1.f);
                if (rescale) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&pvdone[L * 2 + (sb ^ 1)], ((i - 1) >> 1) & 1, a.status));
                    if (!ok) break;
                }
                if (i >= 2) {  // the P buffer of this tile was last read by PV(i-2)
                    ok = __all_sync(0xffffffffu, mbar_wait(&pvdone[pb], ((i >> 1) - 1) & 1, a.status));
                    if (!ok) break;
                }
                tc_fence_after();
                if (rescale) tmem_scale64(tO + lane_off, alpha);
                uint32_t pk[KT / 2];
#pragma unroll
                for (int q = 0; q < KT / 2; ++q) {
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(s[2 * q], s[2 * q + 1]);
                    pk[q] = *reinterpret_cast<uint32_t*>(&h2);
                }
                tmem_st32u(tb + L * 256 + 192 + sb * 32 + lane_off, pk);
                tmem_st_wait();
                tc_fence_before();
                warp_arrive(&pfull[pb]);
                mrun = mnew;
            }
        }
        if constexpr (FULL) {
            if (ok && T > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(&pvdone[L * 2 + ((T - 1) & 1)], ((T - 1) >> 1) & 1, a.status));
                if (ok) {
                    tc_fence_after();
                    float o[64];
                    tmem_ld32(tO + lane_off, o);
                    tmem_ld32(tO + lane_off + 32, o + 32);
                    tmem_ld_wait();
                    if (row_ok) {
                        float* pp = a.part + slot * 68;
                        pp[0] = mrun / kLog2e;  // running max in natural-log units of tau <Lq, K>
                        pp[1] = lrun;
#pragma unroll
                        for (int q = 0; q < 64; q += 4)
                            *reinterpret_cast<float4*>(pp + 4 + q) =
                                make_float4(o[q], o[q + 1], o[q + 2], o[q + 3]);
                    }
                }
            }
        }
        if (row_ok && !a.dense) a.ccount[slot] = cnt;
        if (!FULL && row_ok && a.rcap > 0) a.rcount[slot] = rc;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tb, C::TCOLS);
}

template <bool FULL, int NL>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const ScanArgs& a, int64_t BH,
                       cudaStream_t st) {
    using C = Cfg<FULL, NL>;
    cudaError_t e = cudaFuncSetAttribute(scan_tc_kernel<FULL, NL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(BH * a.chunks);
    return launch_dep(scan_tc_kernel<FULL, NL>, dim3(grid), dim3(C::NT), C::SMEM, st, tk, tv, a);
}

// One thread per landmark: the candidates its chunks kept; a head with a
// landmark below k is flagged (every head's flag is written).
__global__ void __launch_bounds__(256) scan_check_kernel(const int* __restrict__ ccount, int chunks, int m, int k,
                                                         int* __restrict__ hflag) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    const int64_t bh = blockIdx.x;
    bool bad = false;
    for (int i = threadIdx.x; i < m; i += 256) {
        int n = 0;
        for (int c = 0; c < chunks; ++c) n += ccount[(bh * chunks + c) * m + i];
        bad = bad || n < k;
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) hflag[bh] = bad ? 1 : 0;
}

ScanArgs scan_args(const Plan& p, const Work& w, const ScanLevel& L) {
    ScanArgs a;
    a.lqhi = w.lqhi;
    a.lqlo = w.lqlo;
    a.theta = w.theta;
    a.part = w.part;
    a.cand = w.cand;
    a.ccount = w.ccount;
    a.dense = L.dense ? w.dense : nullptr;
    a.ld = L.ld;
    a.status = w.status;
    a.skip = nullptr;
    a.S = L.S;
    a.stride = L.stride;
    a.chunk_len = L.chunk_len;
    a.chunks = L.chunks;
    a.cap = L.cap;
    a.rcap = L.rcap;
    a.ridx = w.ridx;
    a.rval = w.rval;
    a.rcount = w.rcount;
    a.m = p.s.m;
    a.k = p.s.k;
    return a;
}

}  // namespace

cudaError_t launch_scan_tc(const Plan& p, const Work& w, const __nv_bfloat16* K, const __nv_bfloat16* V, int level,
                           cudaStream_t st) {
    const ScanLevel& L = p.lev[level];
    const bool full = level == p.nlev - 1 && p.shared;  // (no LV without the shared branch)
    CUtensorMap tk, tv;
    if (!make_head_tmap(&tk, K, static_cast<uint64_t>(L.S), static_cast<uint64_t>(p.s.BH),
                        static_cast<uint64_t>(L.stride), static_cast<uint64_t>(p.s.N), 64))
        return cudaErrorInvalidValue;
    if (full) {
        if (!make_head_tmap(&tv, V, static_cast<uint64_t>(p.s.N), static_cast<uint64_t>(p.s.BH), 1,
                            static_cast<uint64_t>(p.s.N), 64))
            return cudaErrorInvalidValue;
    } else {
        tv = tk;
    }
    ScanArgs a = scan_args(p, w, L);
    a.theta = level > 0 ? w.theta : nullptr;
    const bool two = p.s.m > 128;
    if (full) return two ? launch_one<true, 2>(tk, tv, a, p.s.BH, st) : launch_one<true, 1>(tk, tv, a, p.s.BH, st);
    return two ? launch_one<false, 2>(tk, tv, a, p.s.BH, st) : launch_one<false, 1>(tk, tv, a, p.s.BH, st);
}

cudaError_t launch_scan_verify(const Plan& p, const Work& w, const __nv_bfloat16* K, cudaStream_t st) {
    const ScanLevel& L = p.lev[p.nlev - 1];
    cudaError_t e = launch_dep(scan_check_kernel, dim3(static_cast<unsigned>(p.s.BH)), dim3(256), 0, st, w.ccount,
                               L.chunks, p.s.m, p.s.k, w.hflag);
    if (e != cudaSuccess) return e;
    CUtensorMap tk;
    if (!make_head_tmap(&tk, K, static_cast<uint64_t>(L.S), static_cast<uint64_t>(p.s.BH),
                        static_cast<uint64_t>(L.stride), static_cast<uint64_t>(p.s.N), 64))
        return cudaErrorInvalidValue;
    // the flagged heads' candidates again (the same chunks and buffers; LV is
    // already merged from the main scan's partials), from the k-th best keys
    ScanArgs a = scan_args(p, w, L);
    a.theta = w.theta_safe;
    a.skip = w.hflag;
    return p.s.m > 128 ? launch_one<false, 2>(tk, tk, a, p.s.BH, st) : launch_one<false, 1>(tk, tk, a, p.s.BH, st);
}

}  // namespace mita
