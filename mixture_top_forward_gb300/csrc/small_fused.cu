// The whole MiTA forward pass of a short head in one kernel (one CTA per
// head), for heads whose queries, keys and values fit in shared memory
// (N <= 256 tokens, m <= 32 landmarks): the ViT shapes of the pages' image
// experiments ("NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), results
// section: DeiT-S on 14 x 14 patch grids).
//
// The stages are those of section "MiTA：用少量地标查询，同时完成压缩与专家构造"
// of the same page, in its order:
//   1. landmarks Lq_i = mean of Q over window i (1-D windows or 2-D adaptive
//      pooling of the token grid, as pool.cu), fp32;
//   2. landmark scan (tensor cores): raw_ij = <Lq_i, K_j> as two bf16
//      products (Lq = hi + lo, exact to ~2^-16), into TMEM; the shared-expert
//      value LV_i = softmax_j(tau raw_ij) V by a second product (P in bf16);
//      the routed expert E_i = the k keys with the largest tau raw_ij, ties
//      to the lower index, in ascending index order (one warp per landmark,
//      the k-th largest order key found bit by bit);
//   3. routing (tensor cores): e(n) = argmax_i <q_n, Lq_hi_i + Lq_lo_i> (two
//      bf16 products, fp32 accumulation), ties to the lowest i;
//   4. expert attention (tensor cores): each 128-query tile against the
//      whole list [Lq; K] in 64-key blocks (S = Q list^T, then O += P [LV; V]
//      with P in TMEM), each query's logits masked to its expert: the m
//      shared keys and the k routed ones (a bit set per expert); one online
//      softmax over the blocks. A short head's whole key list is about as
//      long as one expert's, so the dense product wastes little.
// At these sizes the general path spends its time on launches, short rows
// and work items of a few queries each; here every operand is read from HBM
// once and the head's rows stay in shared memory throughout.
//
// Shared memory: Q (256 rows, zero past N), the key list [Lq in bf16 (rows
// < m), zero rows to 32, K, zero rows to a multiple of 64] and the value
// list [LV in bf16, zeros, V, zeros], all bf16 rows of 128 bytes in the
// 128-byte swizzle the MMAs read (16-byte chunk c of row r at chunk position
// c ^ (r & 7)); the landmark tile (Lq hi and lo, 128 rows each, zero past
// m); the landmarks' raw logits, fp32; Lq and LV in fp32; the experts E, one
// byte an index; each expert's keys as 256 bits. TMEM per query tile: S (64 columns), P (32), O
// (64), routing logits (32). Warps: all 16 for pooling and the top-k;
// warps 0 and 4 (both reach TMEM lanes 0-31) hold the landmark rows of stage
// 2, each for half of the key blocks; warps 0-7 the query rows of stages
// 3-4; warp 8 issues the MMAs. Every wait is bounded.
#include "mita_internal.cuh"
#include "umma.cuh"

namespace mita {

namespace {

constexpr int SF_THREADS = 512;  // 16 warps; two threads per query in routing (N <= 256)
constexpr int SF_WARPS = SF_THREADS / 32;
static_assert(SF_THREADS == 2 * 256, "two threads per query of up to 256");
constexpr int SF_MAX_N = 256;
constexpr int SF_MAX_M = 32;
constexpr float kTauSF = 0.125f;  // 1 / sqrt(64)

struct SFArgs {
    const __nv_bfloat16* Q;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    __nv_bfloat16* out;
    int32_t* expert_idx;  // [BH][m][k]
    int32_t* route;       // [BH][N]
    float* lq_out;        // [BH][m][64] or null
    float* lv_out;        // [BH][m][64] or null
    int* status;          // the workspace's status word (bounded waits)
    int N, m, k, gh, gw, p;
};


// byte offset of 16-byte chunk c of bf16 row r (128 bytes a row)
__device__ __forceinline__ uint32_t sf_chunk(int r, int c) {
    return static_cast<uint32_t>(r) * 128u + (static_cast<uint32_t>(c ^ (r & 7)) << 4);
}
// order key of a logit: larger tau * raw first (the score bits of topk_key)
__device__ __forceinline__ uint32_t sf_key(float raw) {
    return static_cast<uint32_t>(topk_key(raw * kTauSF, 0u) >> 32);
}

struct SFLayout {
    size_t kl, vl, lqh, lql, raw, lq, lv, e, bits, total;
    int nkl;  // rows of the key and value lists: 32 landmark rows, then the N key rows, to a multiple of 64
};

__host__ __device__ inline SFLayout sf_layout(int N, int m, int k) {
    SFLayout L;
    L.nkl = (32 + N + 63) / 64 * 64;
    // Q: 256 rows at offset 0 (two 128-row MMA tiles); every list 1024-byte aligned
    L.kl = 256 * 128;
    L.vl = L.kl + static_cast<size_t>(L.nkl) * 128;
    L.lqh = L.vl + static_cast<size_t>(L.nkl) * 128;  // the landmark tile: Lq in bf16 (hi), 128 rows
    L.lql = L.lqh + 128 * 128;                           // and the remainder Lq - hi in bf16 (lo)
    L.raw = L.lql + 128 * 128;                           // the landmarks' raw logits, fp32 [m][256]
    L.lq = L.raw + static_cast<size_t>(m) * 256 * 4;
    L.lv = L.lq + static_cast<size_t>(m) * 64 * 4;
    L.e = L.lv + static_cast<size_t>(m) * 64 * 4;
    L.bits = (L.e + static_cast<size_t>(m) * k + 15) & ~static_cast<size_t>(15);
    L.total = L.bits + 32 * 8 * 4 + 1024;  // (+ alignment of the dynamic base)
    return L;
}

constexpr uint32_t kSfIdescS = umma::idesc_bf16(128, 64, false);   // S = Q keys^T, both K-major
constexpr uint32_t kSfIdescPV = umma::idesc_bf16(128, 64, true);   // O += P values, values MN-major
constexpr uint32_t kSfIdescR = umma::idesc_bf16(128, 32, false);   // routing: Q landmarks^T

__global__ void __launch_bounds__(SF_THREADS, 1) small_fused_kernel(SFArgs a) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    extern __shared__ uint8_t sm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t sfull[2], sfree[2], pfull[2], pvdone[2], rfull[2], drain, cfull, cpfull, cvdone;
    __shared__ uint32_t tmem_base;
    __shared__ float red[2][2][32];  // the landmark-row warps' partial maxima and sums
    const SFLayout Ly = sf_layout(a.N, a.m, a.k);
    uint8_t* Qs = sm;
    uint8_t* KL = sm + Ly.kl;  // [Lq (bf16, rows < m), zeros to row 32, K rows, zeros]
    uint8_t* VL = sm + Ly.vl;  // [LV (bf16), zeros, V rows, zeros]
    uint8_t* Ks = KL + 32 * 128;
    uint8_t* Vs = VL + 32 * 128;
    float* Lq = reinterpret_cast<float*>(sm + Ly.lq);
    float* LV = reinterpret_cast<float*>(sm + Ly.lv);
    uint8_t* E = sm + Ly.e;
    uint32_t* bits = reinterpret_cast<uint32_t*>(sm + Ly.bits);  // [expert][8]: its keys as a bit set
    uint8_t* LqH = sm + Ly.lqh;
    uint8_t* LqL = sm + Ly.lql;
    float* raw_s = reinterpret_cast<float*>(sm + Ly.raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = a.N, m = a.m, k = a.k;
    const int nkl = Ly.nkl;
    const int64_t bh = blockIdx.x;
    const int64_t row0 = bh * N;

    if (tid == 0) {
        for (int t = 0; t < 2; ++t) {
            umma::mbar_init(&sfull[t], 1);
            umma::mbar_init(&sfree[t], 4);
            umma::mbar_init(&pfull[t], 4);
            umma::mbar_init(&pvdone[t], 1);
            umma::mbar_init(&rfull[t], 1);
        }
        umma::mbar_init(&drain, 1);
        umma::mbar_init(&cfull, 1);
        umma::mbar_init(&cpfull, 2);  // the two landmark-row warps
        umma::mbar_init(&cvdone, 1);
        umma::fence_barrier_init();
    }
    if (warp == 0) umma::tmem_alloc(&tmem_base, 512);

    // ---- the head's rows into shared memory (16-byte copies); zero rows
    //      past them (finite operands for the masked MMA rows) ----
    {
        const __nv_bfloat16* src[3] = {a.Q + row0 * 64, a.K + row0 * 64, a.V + row0 * 64};
        uint8_t* dst[3] = {Qs, Ks, Vs};
#pragma unroll
        for (int t = 0; t < 3; ++t)
            for (int x = tid; x < N * 8; x += SF_THREADS) {
                const int r = x >> 3, c = x & 7;
                umma::cp_async16(umma::smem_u32(dst[t] + sf_chunk(r, c)), src[t] + static_cast<int64_t>(r) * 64 + c * 8);
            }
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int x = N * 8 + tid; x < 256 * 8; x += SF_THREADS) *reinterpret_cast<uint4*>(Qs + 16 * x) = z;
        for (int x = tid; x < 32 * 8; x += SF_THREADS) {  // landmark rows (written below for r < m)
            *reinterpret_cast<uint4*>(KL + 16 * x) = z;
            *reinterpret_cast<uint4*>(VL + 16 * x) = z;
        }
        for (int x = (32 + N) * 8 + tid; x < nkl * 8; x += SF_THREADS) {
            *reinterpret_cast<uint4*>(KL + 16 * x) = z;
            *reinterpret_cast<uint4*>(VL + 16 * x) = z;
        }
        for (int x = tid; x < 32 * 8; x += SF_THREADS) bits[x] = 0u;
        for (int x = tid; x < 128 * 8; x += SF_THREADS) {  // rows >= m stay zero
            *reinterpret_cast<uint4*>(LqH + 16 * x) = z;
            *reinterpret_cast<uint4*>(LqL + 16 * x) = z;
        }
        umma::cp_async_wait_all();
    }
    umma::tc_fence_before();
    __syncthreads();
    umma::tc_fence_after();
    const uint32_t tb = tmem_base;

    // ---- 1. landmarks: window means of Q (fp32, and bf16 into the key list) ----
    // (windows as pool.cu: [floor(i L / w), ceil((i + 1) L / w)); all
    // products here stay below 2^16)
    // (one warp per landmark; lane l sums columns 2l, 2l + 1 over the window)
    for (int i = warp; i < m; i += SF_WARPS) {
        int y0, y1, x0, x1, gw;
        if (a.p == 0) {
            y0 = 0;
            y1 = 1;
            x0 = (i * N) / m;
            x1 = ((i + 1) * N + m - 1) / m;
            gw = 0;
        } else {
            const int r = i / a.p, cc = i % a.p;
            y0 = (r * a.gh) / a.p;
            y1 = ((r + 1) * a.gh + a.p - 1) / a.p;
            x0 = (cc * a.gw) / a.p;
            x1 = ((cc + 1) * a.gw + a.p - 1) / a.p;
            gw = a.gw;
        }
        const uint32_t woff = static_cast<uint32_t>(lane & 3) * 4;
        float s0 = 0.f, s1 = 0.f;
        for (int y = y0; y < y1; ++y)
            for (int x = x0; x < x1; ++x) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(Qs + sf_chunk(y * gw + x, lane >> 2) + woff);
                s0 += __uint_as_float(w << 16);
                s1 += __uint_as_float(w & 0xFFFF0000u);
            }
        const float cnt = static_cast<float>((y1 - y0) * (x1 - x0));
        const float v0 = s0 / cnt, v1 = s1 / cnt;
        reinterpret_cast<float2*>(Lq + i * 64)[lane] = make_float2(v0, v1);
        if (a.lq_out) reinterpret_cast<float2*>(a.lq_out + (bh * m + i) * 64)[lane] = make_float2(v0, v1);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(v0, v1);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v0 - __low2float(hi), v1 - __high2float(hi));
        const uint32_t at = sf_chunk(i, lane >> 2) + woff;
        *reinterpret_cast<__nv_bfloat162*>(KL + at) = hi;
        *reinterpret_cast<__nv_bfloat162*>(LqH + at) = hi;
        *reinterpret_cast<__nv_bfloat162*>(LqL + at) = lo;
    }
    umma::fence_proxy_async();  // the bf16 rows written here feed the tensor cores
    __syncthreads();

    // ---- 2. landmark scan on the tensor cores: S = (Lq_hi + Lq_lo) K^T (two
    //      bf16 products, exact to ~2^-16 of the fp32 landmarks) for all key
    //      blocks into TMEM; warp 0 (lane i = landmark i) writes the raw
    //      logits to shared memory and forms P = exp(tau (S - max)) in bf16;
    //      LV = P V / sum by a second product ----
    const int nkb = (N + 63) / 64;
    const uint32_t cS = tb, cP = tb + 256, cO = tb + 384;  // (stage 4 reuses the columns afterwards)
    constexpr float kC2 = kTauSF * 1.4426950408889634f;    // tau log2(e)
    if (warp == 8) {
        if (lane == 0) {
            const uint64_t hd = umma::sdesc_sw128(umma::smem_u32(LqH)), ld = umma::sdesc_sw128(umma::smem_u32(LqL));
            const uint64_t kd = umma::sdesc_sw128(umma::smem_u32(Ks)), vd = umma::sdesc_sw128(umma::smem_u32(Vs));
            umma::tc_fence_after();
            for (int b = 0; b < nkb; ++b) {
                umma::mma_ss_k64(cS + 64 * b, hd, kd + static_cast<uint64_t>(b) * 512, kSfIdescS, 0u);
                umma::mma_ss_k64(cS + 64 * b, ld, kd + static_cast<uint64_t>(b) * 512, kSfIdescS, 1u);
            }
            umma::mma_commit(&cfull);
            if (umma::mbar_wait(&cpfull, 0, a.status)) {
                umma::tc_fence_after();
                for (int b = 0; b < nkb; ++b)
                    umma::mma_ts_k64(cO, cP + 32 * b, vd + static_cast<uint64_t>(b) * 512, kSfIdescPV, b > 0 ? 1u : 0u);
            }
            umma::mma_commit(&cvdone);
        }
    } else if (warp == 0 || warp == 4) {
        // warps 0 and 4 both reach TMEM lanes 0-31 (the landmarks, m <= 32);
        // warp 4 h takes the key blocks b = h, h + 2, ...
        const int hw = warp >> 2, i = lane;
        float* ri = raw_s + (i < m ? i : 0) * 256;
        bool ok = __all_sync(0xffffffffu, umma::mbar_wait(&cfull, 0, a.status));
        if (ok) umma::tc_fence_after();
        float mx = -INFINITY;
        for (int b = hw; b < nkb && ok; b += 2) {
            float sv[64];
            umma::tmem_ld32(cS + 64 * b, sv);
            umma::tmem_ld32(cS + 64 * b + 32, sv + 32);
            umma::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const int j = 64 * b + c;
                if (j < N) {
                    if (i < m) ri[j] = sv[c];
                    mx = fmaxf(mx, sv[c]);
                }
            }
        }
        red[0][hw][lane] = mx;
        umma::named_bar(1, 64);
        mx = fmaxf(red[0][0][lane], red[0][1][lane]);
        float sum = 0.f;
        for (int b = hw; b < nkb && ok; b += 2) {
            float sv[64];
            umma::tmem_ld32(cS + 64 * b, sv);
            umma::tmem_ld32(cS + 64 * b + 32, sv + 32);
            umma::tmem_ld_wait();
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const int j = 64 * b + c;
                const float p0 = j < N ? exp2f((sv[c] - mx) * kC2) : 0.f;
                const float p1 = j + 1 < N ? exp2f((sv[c + 1] - mx) * kC2) : 0.f;
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
                pk[c >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
                sum += __low2float(b2) + __high2float(b2);  // the weights the product sees
            }
            umma::tmem_st32u(cP + 32 * b, pk);
        }
        red[1][hw][lane] = sum;
        umma::tmem_st_wait();
        umma::tc_fence_before();
        umma::warp_arrive(&cpfull);
        umma::named_bar(1, 64);
        if (hw == 0) {
            ok = ok && __all_sync(0xffffffffu, umma::mbar_wait(&cvdone, 0, a.status));
            if (ok) {
                umma::tc_fence_after();
                const float inv = 1.f / (red[1][0][lane] + red[1][1][lane]);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float o[32];
                    umma::tmem_ld32(cO + 32 * hh, o);
                    umma::tmem_ld_wait();
                    if (i < m) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] *= inv;
                        float* lvr = LV + i * 64 + 32 * hh;
#pragma unroll
                        for (int c = 0; c < 32; c += 4)
                            *reinterpret_cast<float4*>(lvr + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
                        if (a.lv_out) {
                            float* g = a.lv_out + (bh * m + i) * 64 + 32 * hh;
#pragma unroll
                            for (int c = 0; c < 32; c += 4)
                                *reinterpret_cast<float4*>(g + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
                        }
#pragma unroll
                        for (int c = 0; c < 4; ++c) {  // bf16 row i of the value list, chunks 4 hh + c
                            uint32_t w[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[8 * c + 2 * u], o[8 * c + 2 * u + 1]);
                                w[u] = *reinterpret_cast<const uint32_t*>(&b2);
                            }
                            *reinterpret_cast<uint4*>(VL + sf_chunk(i, 4 * hh + c)) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
        }
        umma::tc_fence_before();
    }
    umma::fence_proxy_async();
    __syncthreads();

    // ---- E_i: the k largest raw logits of landmark i, ties to the lower
    //      index, in ascending index order (one warp per landmark). Their
    //      threshold (the k-th largest key) bit by bit from the top: the
    //      largest value with at least k keys at or above it; then every key
    //      above it and, of the keys equal to it, the lowest indices ----
    constexpr int T = SF_MAX_N / 32;
    for (int i = warp; i < m; i += SF_WARPS) {
        const float* ri = raw_s + i * 256;
        uint32_t kk[T];
#pragma unroll
        for (int t = 0; t < T; ++t) kk[t] = 32 * t + lane < N ? sf_key(ri[32 * t + lane]) : 0u;  // real keys are > 0
        uint32_t thr = 0;
        for (int bt = 31; bt >= 0; --bt) {
            const uint32_t cand = thr | (1u << bt);
            unsigned c = 0;
#pragma unroll
            for (int t = 0; t < T; ++t) c += kk[t] >= cand ? 1u : 0u;
            if (__reduce_add_sync(0xffffffffu, c) >= static_cast<unsigned>(k)) thr = cand;
        }
        unsigned above = 0;
#pragma unroll
        for (int t = 0; t < T; ++t) above += kk[t] > thr ? 1u : 0u;
        const unsigned remaining = static_cast<unsigned>(k) - __reduce_add_sync(0xffffffffu, above);
        int32_t* dst = a.expert_idx + (bh * m + i) * static_cast<int64_t>(k);
        uint8_t* ei = E + i * k;
        const unsigned below = (1u << lane) - 1u;
        unsigned taken = 0, eq_seen = 0;
#pragma unroll
        for (int t = 0; t < T; ++t) {
            if (32 * t >= N) break;  // (warp-uniform)
            const bool eq = kk[t] == thr && kk[t] != 0u;
            const unsigned eqb = __ballot_sync(0xffffffffu, eq);
            const bool sel = kk[t] > thr || (eq && eq_seen + __popc(eqb & below) < remaining);
            const unsigned sb = __ballot_sync(0xffffffffu, sel);
            if (sel) {
                const int r = static_cast<int>(taken + __popc(sb & below));
                dst[r] = 32 * t + lane;
                ei[r] = static_cast<uint8_t>(32 * t + lane);
            }
            if (lane == 0) bits[i * 8 + t] = sb;  // the expert's key set as bits
            taken += __popc(sb);
            eq_seen += __popc(eqb);
        }
    }
    __syncthreads();

    // ---- 4. expert attention on the tensor cores: each 128-query tile t
    //      against the whole list [Lq; K] in 64-key blocks, masked per query
    //      to its expert (the m shared keys and the expert's k routed keys);
    //      one online softmax over the blocks, as in the expert kernel ----
    const int ntile = (N + 127) / 128, nblk = nkl / 64;
    // TMEM per tile: S (64 columns), P (bf16 pairs, 32), O (64)
    auto tS = [&](int t) { return tb + t * 160; };
    auto tP = [&](int t) { return tb + t * 160 + 64; };
    auto tO = [&](int t) { return tb + t * 160 + 96; };
    auto tR = [&](int t) { return tb + 320 + t * 32; };  // routing logits: 32 columns per tile
    if (warp == 8) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            const uint64_t qd = umma::sdesc_sw128(umma::smem_u32(Qs));
            const uint64_t kd = umma::sdesc_sw128(umma::smem_u32(KL));
            const uint64_t vd = umma::sdesc_sw128(umma::smem_u32(VL));
            // routing logits <q, Lq_hi + Lq_lo> of each tile (landmarks 0-31)
            const uint64_t hd = umma::sdesc_sw128(umma::smem_u32(LqH)), ld = umma::sdesc_sw128(umma::smem_u32(LqL));
            umma::tc_fence_after();
            for (int t = 0; t < ntile; ++t) {
                umma::mma_ss_k64(tR(t), qd + static_cast<uint64_t>(t) * 1024, hd, kSfIdescR, 0u);
                umma::mma_ss_k64(tR(t), qd + static_cast<uint64_t>(t) * 1024, ld, kSfIdescR, 1u);
                umma::mma_commit(&rfull[t]);
            }
            bool ok = true;
            for (int j = 0; j < nblk && ok; ++j) {
                for (int t = 0; t < ntile && ok; ++t) {
                    // the rows have read S of the previous block
                    if (j > 0 && !(ok = umma::mbar_wait(&sfree[t], (j - 1) & 1, a.status))) break;
                    umma::tc_fence_after();
                    umma::mma_ss_k64(tS(t), qd + static_cast<uint64_t>(t) * 1024, kd + static_cast<uint64_t>(j) * 512,
                                     kSfIdescS, 0u);
                    umma::mma_commit(&sfull[t]);
                }
                for (int t = 0; t < ntile && ok; ++t) {
                    if (!(ok = umma::mbar_wait(&pfull[t], j & 1, a.status))) break;
                    umma::tc_fence_after();
                    umma::mma_ts_k64(tO(t), tP(t), vd + static_cast<uint64_t>(j) * 512, kSfIdescPV, j > 0 ? 1u : 0u);
                    umma::mma_commit(&pvdone[t]);
                }
            }
            umma::mma_drain(&drain);
        }
    } else if (warp < 4 * ntile) {
        // ------------------------- query rows of tile t -------------------------
        const int t = warp >> 2;
        const int n = 128 * t + (warp & 3) * 32 + lane;  // TMEM lane = row of the tile
        const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const bool valid = n < N;
        // routing: e(n) = argmax_i <q_n, Lq_i> (hi + lo, fp32 accumulation);
        // a strict comparison in ascending i keeps the lowest i on ties
        int e = 0;
        {
            if (!__all_sync(0xffffffffu, umma::mbar_wait(&rfull[t], 0, a.status))) e = 0;
            umma::tc_fence_after();
            float r[32];
            umma::tmem_ld32(tR(t) + lo, r);
            umma::tmem_ld_wait();
            float best = r[0];
#pragma unroll
            for (int i = 1; i < 32; ++i)
                if (i < m && r[i] > best) {
                    best = r[i];
                    e = i;
                }
            if (valid) a.route[row0 + n] = e;
        }
        const uint32_t lmask = m >= 32 ? 0xFFFFFFFFu : ((1u << m) - 1u);  // the shared keys of block 0
        constexpr float kC = kTauSF * 1.4426950408889634f;  // tau log2(e)
        float M = -INFINITY, L = 0.f;
        bool ok = true;
        for (int j = 0; j < nblk && ok; ++j) {
            ok = __all_sync(0xffffffffu, umma::mbar_wait(&sfull[t], j & 1, a.status));
            if (!ok) break;
            umma::tc_fence_after();
            float s[64];
            umma::tmem_ld32(tS(t) + lo, s);
            umma::tmem_ld32(tS(t) + 32 + lo, s + 32);
            umma::tmem_ld_wait();
            umma::tc_fence_before();
            umma::warp_arrive(&sfree[t]);
            // list row 64 j + c: rows 0-31 landmarks, key 64 j + c - 32 after
            const uint32_t w0 = j == 0 ? lmask : bits[e * 8 + 2 * j - 1];
            const uint32_t w1 = 2 * j < 8 ? bits[e * 8 + 2 * j] : 0u;
            float bm = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const bool in = ((c < 32 ? w0 : w1) >> (c & 31)) & 1u;
                s[c] = in ? s[c] * kC : -INFINITY;
                bm = fmaxf(bm, s[c]);
            }
            const float mnew = fmaxf(M, bm);
            const float alpha = exp2f(M - mnew);  // 0 on the first block with a key
            uint32_t pk[32];
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const float p0 = exp2f(s[c] - mnew), p1 = exp2f(s[c + 1] - mnew);
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
                pk[c >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
                sum += __low2float(b2) + __high2float(b2);  // the weights the P.V product sees
            }
            L = L * alpha + sum;
            M = mnew;
            // the previous block's P.V must be done before P is overwritten or O rescaled
            if (j > 0) {
                ok = __all_sync(0xffffffffu, umma::mbar_wait(&pvdone[t], (j - 1) & 1, a.status));
                if (!ok) break;
                umma::tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) umma::tmem_scale64(tO(t) + lo, alpha);
            }
            umma::tmem_st32u(tP(t) + lo, pk);
            umma::tmem_st_wait();
            umma::tc_fence_before();
            umma::warp_arrive(&pfull[t]);
        }
        if (ok && __all_sync(0xffffffffu, umma::mbar_wait(&pvdone[t], (nblk - 1) & 1, a.status))) {
            umma::tc_fence_after();
            const float inv = 1.f / L;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float o[32];
                umma::tmem_ld32(tO(t) + 32 * hh + lo, o);
                umma::tmem_ld_wait();
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(a.out + (row0 + n) * 64 + 32 * hh);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t w[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const __nv_bfloat162 b2 =
                                __floats2bfloat162_rn(o[8 * c + 2 * u] * inv, o[8 * c + 2 * u + 1] * inv);
                            w[u] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }
    umma::tc_fence_before();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tb, 512);
}

}  // namespace

bool small_fused_applies(const Plan& p) {
    return p.shared && !p.split && p.s.s_route == 1 && p.s.N <= SF_MAX_N && p.s.m <= SF_MAX_M && p.s.k <= p.s.N &&
           p.s.BH < (int64_t(1) << 31) && sf_layout(static_cast<int>(p.s.N), p.s.m, p.s.k).total <= 232448;
}

cudaError_t launch_small_fused(const Plan& p, const __nv_bfloat16* Q, const __nv_bfloat16* K, const __nv_bfloat16* V,
                               __nv_bfloat16* out, int32_t* expert_idx, int32_t* route, float* lq_out, float* lv_out,
                               int* status, cudaStream_t st) {
    SFArgs a;
    a.status = status;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.out = out;
    a.expert_idx = expert_idx;
    a.route = route;
    a.lq_out = lq_out;
    a.lv_out = lv_out;
    a.N = static_cast<int>(p.s.N);
    a.m = p.s.m;
    a.k = p.s.k;
    a.gh = p.s.gh;
    a.gw = p.s.gw;
    a.p = p.s.p;
    const size_t smem = sf_layout(a.N, a.m, a.k).total;
    cudaError_t e =
        cudaFuncSetAttribute(small_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_dep(small_fused_kernel, dim3(static_cast<unsigned>(p.s.BH)), dim3(SF_THREADS), smem, st, a);
}

}  // namespace mita
