// Stage 3 with the shared branch of stage 4, on the tensor cores.
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造": each query picks the expert of
// the landmark query it matches best, reusing the query-to-landmark logits,
// and attends to the m shared pairs (Lq_i, LV_i) and its expert's k routed
// pairs under one softmax. The Algorithm 1 caption of "And attention is also
// FFN? …" (en.roboind.com) combines the two branches by online softmax. This
// kernel computes, per query n, the logits t_i = tau <q_n, Lq_i> once and uses
// them twice:
//   route(n) = argmax_i t_i (ties to the lowest i), and
//   the shared branch's softmax partial over those m logits:
//     lse_n = max_i t_i log2(e) + log2(sum_i 2^(t_i log2(e) - max)), and
//     o_n   = sum_i p_i LV_i / sum_i p_i  (bf16),
// from which the expert kernel continues the same softmax over the routed
// keys: (lse_n, o_n) is exactly one pre-merged pair of logit lse_n (log2
// units) and value o_n.
//
// Persistent CTAs over 128-query tiles (a contiguous range each, so the head
// and with it the landmark operands change rarely). TMEM: two buffers of 256
// columns (tiles t = b mod 2). In buffer b the logits D = Q Lq^T (hi + lo,
// exact to ~2^-16 of the fp32 landmarks) fill columns [0, m_pad); once the
// rows have read them, P (bf16 pairs) takes columns [0, m_pad / 2) and the
// two halves of the P.LV product accumulate in columns [128, 192) (landmarks
// below 128) and [192, 256) (the rest).
//   warp 8 lane 0:   TMA loads of Q tiles (4-stage ring) and of the head's
//                    Lq hi / lo and LV rows (m_pad <= 256 each);
//   warp 9 lane 0:   logits issuer, both buffers: D = Q Lq_hi^T + Q Lq_lo^T;
//   warps 10, 11 lane 0: P.LV issuer of landmark half g (g = 0: landmarks
//                    [0, 128), g = 1: [128, m_pad)) for both buffers;
//   warps 0-3, 4-7:  row warpgroup b for buffer b, one query per thread:
//                    argmax and maximum over the logits, the weights
//                    p_i = 2^(t_i log2 e - max) into TMEM as bf16 (row sum
//                    from the same rounded weights the product sees), then
//                    o = (O_0 + O_1) / sum, lse, the route and a histogram of
//                    the head's routes for the grouping.
// Every wait is bounded (umma.cuh).
#include <algorithm>

#include "tensormap.cuh"
#include "umma.cuh"

namespace mita {

namespace {

using namespace umma;

constexpr float kC = 0.125f * kLog2e;  // tau * log2(e), tau = 1/sqrt(64)
constexpr int QST = 4;                 // Q tile stages
constexpr size_t OFF_LO = 32768;
constexpr size_t OFF_LV = 65536;
constexpr size_t OFF_Q = 98304;
constexpr size_t SMEM = OFF_Q + QST * 16384 + 1024;
constexpr int NTH = 384;  // warps 0-7 rows, 8 loads, 9 logits issuer, 10-11 P.LV issuers
constexpr uint32_t kIdescPV = idesc_bf16(128, 64, true);
constexpr uint32_t kColO = 128;  // O half g at kColO + 64 g within the buffer

struct Args {
    int32_t* route;        // [BH][N]
    int* counts;           // [BH][m]
    __nv_bfloat16* osh;    // [BH][N][64] shared-branch output, normalised
    float* lse;            // [BH][N] its log-sum-exp (log2 units of the tau-scaled logits)
    int* status;
    int64_t N, tiles_per_head, total_tiles;
    int m, m_pad;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(NTH, 1)
    route_shared_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap thi,
                        const __grid_constant__ CUtensorMap tlo, const __grid_constant__ CUtensorMap tlv, Args a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t qfull[QST], qempty[QST], dfull[2], pfull[2], odone[2], dfree[2], lqfull, lqfree, drain;
    __shared__ uint32_t tmem_base;
    __shared__ int hist[2][256];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t t0 = a.total_tiles * blockIdx.x / gridDim.x;
    const int64_t t1 = a.total_tiles * (blockIdx.x + 1) / gridDim.x;
    const int nt = static_cast<int>(t1 - t0);
    const int npv = a.m_pad > 128 ? 2 : 1;  // P.LV halves in use

    if (tid == 0) {
        for (int i = 0; i < QST; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&dfull[b], 1);
            mbar_init(&pfull[b], 4);    // the buffer's row warps, after writing P
            mbar_init(&odone[b], npv);  // one commit per P.LV half in use
            mbar_init(&dfree[b], 4);    // the buffer's row warps, after reading O
        }
        mbar_init(&lqfull, 1);
        mbar_init(&lqfree, 1 + npv);  // every issuer that reads the landmark operands
        mbar_init(&drain, 3);         // exit path: one commit per issuer warp
        fence_barrier_init();
    }
    for (int e = tid; e < 2 * 256; e += NTH) (&hist[0][0])[e] = 0;
    if (warp == 0) tmem_alloc(&tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;

    if (warp == 8) {
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
                if (bh != cur) {  // restage the landmarks once every MMA reading them is done
                    if (changes > 0 && !mbar_wait(&lqfree, (changes - 1) & 1, a.status)) break;
                    mbar_arrive_expect_tx(&lqfull, 3u * a.m_pad * 128u);
                    tma_load_2d(base, &thi, 0, static_cast<int>(bh * a.m), &lqfull);
                    tma_load_2d(base + OFF_LO, &tlo, 0, static_cast<int>(bh * a.m), &lqfull);
                    tma_load_2d(base + OFF_LV, &tlv, 0, static_cast<int>(bh * a.m), &lqfull);
                    ++changes;
                    cur = bh;
                }
                if (t + QST < nt) {  // refill the stage of tile t once its logits are done
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
    } else if (warp == 9) {
        // ---------------- logits issuer (lane 0), both buffers ----------------
        // Walks every tile to follow the landmark restages (each head change is
        // released, then waited for).
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, a.m_pad, false);
            const uint32_t hi = smem_u32(base), lo = smem_u32(base + OFF_LO);
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
                const int b = t & 1, st = t % QST;
                if (!mbar_wait(&qfull[st], (t / QST) & 1, a.status)) break;
                // the rows have read this buffer's O of tile t - 2
                if (t >= 2 && !mbar_wait(&dfree[b], ((t >> 1) - 1) & 1, a.status)) break;
                tc_fence_after();
                const uint32_t qa = smem_u32(base + OFF_Q + st * 16384);
                const uint32_t d = tb + b * 256;
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
    } else if (warp >= 10) {
        // ---------------- P.LV issuer of landmark half g (lane 0) ----------------
        if (lane == 0) {
            const int g = warp - 10;
            const int k0 = 128 * g;                                  // first landmark of the half
            const int ksteps = g < npv ? (min(a.m_pad, k0 + 128) - k0) / 16 : 0;
            const uint64_t lvd = sdesc_sw128(smem_u32(base + OFF_LV + k0 * 128));
            int64_t cur = -1;
            int changes = 0;
            for (int t = 0; t < nt && ksteps > 0; ++t) {
                const int64_t bh = (t0 + t) / a.tiles_per_head;
                if (bh != cur) {
                    if (changes > 0) mma_commit(&lqfree);
                    if (!mbar_wait(&lqfull, changes & 1, a.status)) break;
                    ++changes;
                    cur = bh;
                }
                const int b = t & 1;
                if (!mbar_wait(&pfull[b], (t >> 1) & 1, a.status)) break;
                tc_fence_after();
                const uint32_t d = tb + b * 256;
                // P of landmarks k0.. sits in columns k0 / 2.. (bf16 pairs); LV rows
                // are MN-major, 16 rows (2048 bytes) per K step
                for (int s = 0; s < ksteps; ++s)
                    mma_ts(d + kColO + 64 * g, d + k0 / 2 + 8 * s, lvd + static_cast<uint64_t>(s) * 128, kIdescPV,
                           s > 0 ? 1u : 0u);
                mma_commit(&odone[b]);
            }
            mma_drain(&drain);
        }
    } else {
        // ---------------- row warpgroup b: tiles t = b (mod 2) ----------------
        const int b = warp >> 2;
        const int row = (warp & 3) * 32 + lane;  // TMEM lane quarter = warp % 4
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t d = tb + b * 256 + lane_off;
        int* h = hist[b];
        int64_t cur = -1;
        for (int t = b; t < nt; t += 2) {
            const int64_t g = t0 + t;
            const int64_t bh = g / a.tiles_per_head, tile = g % a.tiles_per_head;
            if (bh != cur) {  // flush the previous head's route counts
                named_bar(1 + b, 128);
                if (cur >= 0)
                    for (int e = row; e < a.m; e += 128)
                        if (h[e]) atomicAdd(&a.counts[cur * a.m + e], h[e]);
                named_bar(1 + b, 128);
                for (int e = row; e < a.m; e += 128) h[e] = 0;
                named_bar(1 + b, 128);
                cur = bh;
            }
            if (!named_bar_and(1 + b, 128, mbar_wait(&dfull[b], (t >> 1) & 1, a.status))) break;
            tc_fence_after();
            // pass 1: argmax (ties to the lower index) and maximum; 4 interleaved chains
            float bv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            int bi[4] = {0, 1, 2, 3};
            for (int c0 = 0; c0 < a.m_pad; c0 += 32) {
                float v[32];
                tmem_ld32(d + c0, v);
                tmem_ld_wait();
                if (c0 + 32 > a.m) {  // (uniform) columns past m are another head's landmarks
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
            float best = bv[0];
            int arg = bi[0];
#pragma unroll
            for (int u = 1; u < 4; ++u)
                if (bv[u] > best || (bv[u] == best && bi[u] < arg)) {
                    best = bv[u];
                    arg = bi[u];
                }
            arg = min(arg, a.m - 1);  // in range whatever the logits (non-finite ones are out of contract)
            // pass 2: weights, as bf16 pairs over the logits already read. The
            // largest weight is 2^0, exact in bf16; the row sum adds the fp32
            // weights (their bf16 roundings are independent, relative 2^-9)
            const float mx = best * kC;
            const float2 c2 = make_float2(kC, kC), m2 = make_float2(-mx, -mx);
            float2 acc = make_float2(0.f, 0.f);
            for (int c0 = 0; c0 < a.m_pad; c0 += 32) {
                float v[32];
                tmem_ld32(d + c0, v);
                tmem_ld_wait();
                if (c0 + 32 > a.m) {  // (uniform) columns past m get weight 0
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = c0 + j < a.m ? v[j] : -INFINITY;
                }
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float2 x = __ffma2_rn(make_float2(v[j], v[j + 1]), c2, m2);
                    const float2 e = make_float2(exp2f(x.x), exp2f(x.y));
                    acc = __fadd2_rn(acc, e);
                    pk[j >> 1] = pack_bf16(e.x, e.y);
                }
                // P columns c0/2 .. c0/2+15 hold logits already read (c0/2 + 15 < c0 + 32)
                tmem_st16u(d + c0 / 2, pk);
            }
            const float lsum = acc.x + acc.y;
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&pfull[b]);
            const int64_t n = tile * 128 + row;
            if (n < a.N) {
                a.route[bh * a.N + n] = arg;
                atomicAdd(&h[arg], 1);
            }
            // o = (O_0 + O_1) / sum and lse, once the product is done
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&odone[b], (t >> 1) & 1, a.status));
            if (!ok) break;
            tc_fence_after();
            const float inv = 1.f / lsum;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float o[32], o2[32];
                tmem_ld32(d + kColO + 32 * hh, o);
                if (npv > 1) tmem_ld32(d + kColO + 64 + 32 * hh, o2);
                tmem_ld_wait();
                if (npv > 1) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] += o2[j];
                }
                if (n < a.N) {
                    uint4* dst = reinterpret_cast<uint4*>(a.osh + (bh * a.N + n) * D + 32 * hh);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        dst[c] = make_uint4(pack_bf16(o[8 * c] * inv, o[8 * c + 1] * inv),
                                            pack_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                            pack_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                            pack_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
                }
            }
            tc_fence_before();
            warp_arrive(&dfree[b]);
            if (n < a.N) a.lse[bh * a.N + n] = mx + __log2f(lsum);
        }
        named_bar(1 + b, 128);
        if (cur >= 0)
            for (int e = row; e < a.m; e += 128)
                if (h[e]) atomicAdd(&a.counts[cur * a.m + e], h[e]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tb, 512);
}

}  // namespace

bool route_shared_supported(const Plan& p) {
    return p.s.m <= 256 && p.s.s_route == 1 && p.shared && p.s.BH * p.s.N < (int64_t(1) << 31);
}

cudaError_t launch_route_shared(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route,
                                cudaStream_t st) {
    Args a;
    a.route = route;
    a.counts = w.counts;
    a.osh = w.osh;
    a.lse = w.lse;
    a.status = w.status;
    a.N = p.s.N;
    a.tiles_per_head = (p.s.N + 127) / 128;
    a.total_tiles = a.tiles_per_head * p.s.BH;
    a.m = p.s.m;
    a.m_pad = (p.s.m + 15) / 16 * 16;
    CUtensorMap tq, thi, tlo, tlv;
    const uint64_t mrows = static_cast<uint64_t>(p.s.BH) * p.s.m;
    if (!make_row_tmap(&tq, Q, static_cast<uint64_t>(p.s.BH * p.s.N), 128) ||
        !make_row_tmap(&thi, w.lqhi, mrows, a.m_pad) || !make_row_tmap(&tlo, w.lqlo, mrows, a.m_pad) ||
        !make_row_tmap(&tlv, w.lvbf, mrows, a.m_pad))
        return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(route_shared_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM));
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(device_sms(), a.total_tiles);
    route_shared_kernel<<<static_cast<unsigned>(grid), NTH, SMEM, st>>>(tq, thi, tlo, tlv, a);
    return cudaGetLastError();
}

}  // namespace mita
