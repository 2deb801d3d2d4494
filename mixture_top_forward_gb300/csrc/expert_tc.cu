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
// list (<= 128 queries of one expert per item), in rounds of up to three items
// of the same expert, one per row warpgroup. The expert's key list
// [Lq_0..Lq_{m-1}, K_e] and value list [LV_0..LV_{m-1}, V_e] (bf16, 128-byte
// swizzled rows, zero padded to whole 64-row blocks) stay in shared memory
// while consecutive rounds share the expert.
//   warp 0:         producer: gathers the key/value lists when the expert
//                   changes (the shared rows only when the head changes) and
//                   each item's query rows (through the grouping permutation)
//                   into the warpgroup's next query buffer, all with TMA 4-row
//                   gathers that complete on the consumer's mbarrier. A gather
//                   costs its issuing warp about a hundred cycles, so where
//                   lists change often the row warps, idle at a list change,
//                   load the lists instead (RL: all 12; IND: each warpgroup its
//                   own list and query rows), and the producer keeps the rest;
//   warps 1-3 (lane 0): one MMA issuer per warpgroup: per 64-key block j of
//                   its item, S = Q keys_j^T (A and B in shared memory) into
//                   the warpgroup's TMEM score columns, and one block later
//                   O += P_j values_j with P read from TMEM (A in tensor
//                   memory, B in shared memory) into its TMEM accumulator;
//   warps 4-7, 8-11, 12-15: one warpgroup per item (4 consecutive warps cover
//                   the 4 TMEM lane quarters), one thread per query row: load
//                   the 64 logits, update the running max, p = 2^(s tau log2e
//                   - max) in registers, P as bf16 pairs into TMEM once the
//                   previous block's P.V is done; at the end O / rowsum ->
//                   bf16 -> the query's row. The row sum takes each block's
//                   largest weight as rounded to bf16 for the P.V product, so
//                   a dominant key's rounding cancels in O / rowsum.
// The running max is kept while a new block maximum stays within 2^32 of it,
// so O is rescaled (after the block's P.V wait) only for extreme logit
// ranges. Weights up to 2^32 stay far inside the bf16/fp32 range; O overflows
// only for values beyond ~2^86 in magnitude.
// TMEM per warpgroup: 64 columns of S, 32 of P (bf16 pairs), 64 of O, so three
// warpgroups (three row warps per SM sub-partition) fit in the 512 columns.
// Handshakes are mbarriers, each completed exactly once per event its waiter
// consumes; row warps arrive once each (4-arrival barriers) and make
// their waits warp-uniform, so no named barrier can block forever. Every
// wait is bounded (umma.cuh).
//
// With the shared branch split off (SPLIT, s = 1: route_shared.cu has already
// formed each query's softmax partial over the m landmark logits, as the
// Algorithm 1 caption's online-softmax combine allows), the key list holds
// the k routed keys alone and each row starts its online softmax from that
// partial: running max lse_n (log2 units), row sum 1 and O = o_n (the shared
// output, gathered like the query rows), i.e. one pre-merged pair of logit
// lse_n and value o_n. Each row thread copies its o_n row into its warpgroup's
// staging rows with cp.async when its item starts, and writes it, scaled to
// its first block's running max, into its O accumulator before that block's
// P.V accumulates (the producer is not involved, so it keeps running ahead).
//
// s routed experts per query (MULTI; the pages' setting is s = 1): one launch
// per rank j of the routes, over the queries grouped by their j-th expert.
// Pass 0 takes the shared pairs and the expert's keys, later passes the
// expert's keys alone, with the keys an earlier-ranked expert of the query
// already held masked out (their logits set to -inf, from the expert overlap
// table), so the union of the s experts enters the softmax once. Each pass
// runs its own online softmax; the epilogue merges it with the query's fp32
// state row of the earlier passes (log-sum-exp merge of (max, sum, O)) and
// either stores the merged state or, in the last pass, the normalised output.
#include "tensormap.cuh"
#include "umma.cuh"

namespace mita {

namespace {

using namespace umma;

constexpr float kC = 0.125f * kLog2e;  // tau * log2(e), tau = 1/sqrt(64)
constexpr float kLazy = 32.0f;         // keep the running max while the new one is within 2^32
constexpr int KB = 64;                 // keys per block
constexpr int NWG = 3;                 // row warpgroups
constexpr int QB = 2;                  // query-row buffers per warpgroup
constexpr int NT = 32 * (1 + NWG) + NWG * 128;  // producer, one issuer warp per group, rows
// TMEM columns of warpgroup w: S (64) at 64 w, O (64) at 192 + 64 w, P (32,
// bf16 pairs) at 384 + 32 w; every S and O starts on a multiple of 64
__host__ __device__ constexpr uint32_t tcol_s(int w) { return 64u * w; }
__host__ __device__ constexpr uint32_t tcol_o(int w) { return 192u + 64u * w; }
__host__ __device__ constexpr uint32_t tcol_p(int w) { return 384u + 32u * w; }
static_assert(tcol_p(NWG - 1) + 32 <= 512 && tcol_s(NWG - 1) + 64 <= tcol_o(0) && tcol_o(NWG - 1) + 64 <= tcol_p(0),
              "TMEM holds 512 columns");
constexpr uint32_t kIdescS = idesc_bf16(128, KB, false);
// kernel modes; kStats (the backward pass's statistics) runs the plain pass
// but writes each query's log-sum-exp and Delta = dO . out instead of out
constexpr int kPlain = 0, kMulti = 1, kSplit = 2, kStats = 3;
constexpr uint32_t kIdescPV = idesc_bf16(128, 64, true);

struct Args {
    const int4* items;
    const int* nitems;
    const int* perm;
    const int32_t* expert_idx;
    __nv_bfloat16* out;
    int* status;
    int64_t N;
    int m, msh, k, nblk;  // msh: shared pairs taken (m, or 0 for the routing-only ablation / passes j > 0)
    int s, j, nbw;        // MULTI: this launch is the pass of rank j of s; nbw mask words per row
    // the pointers only one mode reads share their storage (kept within 128
    // bytes: a larger argument block made the plain kernel spill registers)
    union {
        struct {                   // MULTI (s > 1 routing)
            const uint64_t* mask;  // j > 0: [BH][N][nbw] per grouping slot, bit c of word b: key c of block b counted before
            float* state;          // [BH][N][68]: O[64] (unnormalised), max (log2 units), sum
        };
        struct {                        // SPLIT
            const float* lse;           // [BH][N] the shared branch's log-sum-exp (log2 units)
            const __nv_bfloat16* osh;   // [BH][N][64] its output rows
        };
        struct {                        // plain: the key and value rows (L2 prefetches of the next list)
            const __nv_bfloat16* kp;    // [BH][N][64]
            const __nv_bfloat16* vp;    // [BH][N][64]
        };
        struct {                        // STATS
            const __nv_bfloat16* dO;    // [BH][N][64] output gradients
            float* st_lse;              // [BH][N] log-sum-exp of the m + k logits (log2 units of tau <q, key>)
            float* st_delta;            // [BH][N] dO . out (out unrounded); both in grouped order
        };
    };
};
static_assert(sizeof(Args) <= 128, "the kernel argument block stays within 128 bytes");

struct Layout {
    uint8_t* keys;    // nblk * 8 KB (IND: warpgroup w's at + w * kvstride)
    uint8_t* vals;    // nblk * 8 KB (likewise)
    uint32_t kvstride;  // bytes between the warpgroups' lists (0: one shared list)
    uint8_t* q;       // [NWG][QB] * 16 KB: query rows
    uint8_t* ps;      // SPLIT: [NWG] * 16 KB: the rows' shared-branch outputs (each thread its own row)
};

__device__ __forceinline__ Layout layout(uint8_t* base, int nblk, bool ind) {
    Layout L;
    L.keys = base;
    L.vals = L.keys + nblk * 8192;
    L.kvstride = ind ? static_cast<uint32_t>(nblk) * 16384u : 0u;
    L.q = base + (ind ? NWG : 1) * nblk * 16384;
    L.ps = L.q + NWG * QB * 16384;
    return L;
}

// The round starting at item r of [r, i1): the item there and, if the next
// item has the same expert (and head), that one too; one per warpgroup. With
// independent warpgroups (one = true) every round is one item of the
// warpgroup's own range.
__device__ __forceinline__ int round_items(const Args& a, int r, int i1, int4& x0, int4& x1, int4& x2,
                                           bool one = false) {
    x0 = a.items[r];
    if (one || r + 1 >= i1) return 1;
    x1 = a.items[r + 1];
    if (x1.x != x0.x || x1.w != x0.w) return 1;
    if (r + 2 >= i1) return 2;
    x2 = a.items[r + 2];
    return (x2.x == x0.x && x2.w == x0.w) ? 3 : 2;
}
__device__ __forceinline__ int4 pick(int w, const int4& x0, const int4& x1, const int4& x2) {
    return w == 0 ? x0 : (w == 1 ? x1 : x2);
}

// Walks the rounds from r to the next item of warpgroup w (returned in out).
// Each list change on the way is first released (kvfree: once this thread's
// MMAs so far are done) and then waited for (kvfull), strictly in turn, so
// every issuer sees every phase of both barriers. Returns 1 (item), 0 (none
// left) or -1 (a wait timed out).
__device__ __forceinline__ int next_item(const Args& a, int w, int& r, int i1, int& cur_bh, int& cur_e, int& changes,
                                         uint64_t* kvfull, uint64_t* kvfree, int4& out, bool one) {
    while (r < i1) {
        int4 x0, x1, x2;
        const int cnt = round_items(a, r, i1, x0, x1, x2, one);
        if (x0.w != cur_bh || x0.x != cur_e) {
            // (IND: the row warps load the next list once they see the last
            // P.V of the current one done; nothing waits for a release)
            if (changes > 0 && !one) umma::mma_commit(kvfree);
            if (!umma::mbar_wait(kvfull, changes & 1, a.status)) return -1;
            umma::tc_fence_after();
            cur_bh = x0.w;
            cur_e = x0.x;
            ++changes;
        }
        r += cnt;
        if (w < cnt) {
            out = pick(w, x0, x1, x2);
            return 1;
        }
    }
    return 0;
}

// Whether warpgroup w has another item before the next list change.
__device__ __forceinline__ bool next_same(const Args& a, int w, int r, int i1, int cur_bh, int cur_e, bool one) {
    while (r < i1) {
        int4 x0, x1, x2;
        const int cnt = round_items(a, r, i1, x0, x1, x2, one);
        if (x0.w != cur_bh || x0.x != cur_e) return false;
        if (w < cnt) return true;
        r += cnt;
    }
    return false;
}

__device__ __forceinline__ void zero16(uint8_t* p) { *reinterpret_cast<uint4*>(p) = make_uint4(0, 0, 0, 0); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// SPLIT: writes row t's shared-branch output (bf16, a 128-byte swizzled row
// of `rows`), times alpha, into this warp's 64 O columns at tO, and orders
// the stores before the caller's barrier arrival. Once per item: kept out of
// line so that its registers do not count in the block loop.
static __device__ __noinline__ void preload_shared(uint32_t tO, const uint8_t* rows, int t, float alpha) {
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        float o[32];
#pragma unroll
        for (int c = 0; c < 4; ++c)
            unpack_bf16x8(*reinterpret_cast<const uint4*>(rows + swz128(t, 4 * hh + c)), o + 8 * c);
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] *= alpha;
        tmem_st32(tO + 32 * hh, o);
    }
    tmem_st_wait();
    tc_fence_before();
}

// STATS: dO_row . (O * inv) over this warp's 64 O columns at tO (row = false:
// the O columns are still read, the dot is 0). Out of line, like the
// preload above.
static __device__ __noinline__ float stats_delta(uint32_t tO, const __nv_bfloat16* g, float inv, bool row) {
    float dl = 0.f;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
        float o[32];
        tmem_ld32(tO + h * 32, o);
        tmem_ld_wait();
        if (row) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float gv[8];
                unpack_bf16x8(ldg_nc_v4(g + 32 * h + 8 * c), gv);
#pragma unroll
                for (int u = 0; u < 8; ++u) dl = fmaf(o[8 * c + u] * inv, gv[u], dl);
            }
        }
    }
    return dl;
}

// IND (independent warpgroups, short lists only): each warpgroup takes a
// contiguous third of the CTA's items with a key/value list of its own, so
// experts of one item each (short sequences, ViT shapes) run three at a time
// instead of one per round.
// RL (long lists, few items per expert): the row warps load the CTA's key
// lists instead of the producer, spread over all of them.
template <int MODE, bool IND, bool RL = false>
__global__ void __launch_bounds__(NT, 1)
    expert_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tlq,
                     const __grid_constant__ CUtensorMap tlv, Args a) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    constexpr bool MULTI = MODE == kMulti, SPLIT = MODE == kSplit, STATS = MODE == kStats;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t kvfull[NWG], kvfree[NWG], qfull[NWG * QB], qfree[NWG * QB], ofree[NWG];
    __shared__ uint64_t sfull[NWG], sfree[NWG], pfull[NWG], pvdone[NWG], drain;
    __shared__ uint32_t tmem_base;
    // per row warp: the head and expert of the key list held, lists armed
    // (read only between items: kept out of the registers of the block loop)
    __shared__ int s_list[4 * NWG][3];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Layout S = layout(base, a.nblk, IND);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // key rows: [0, msh) shared, [msh, m4) unused, [m4, m4 + k) routed (m4 =
    // msh rounded up to 4, so every 4-row gather starts 512-byte aligned);
    // msh = m, or 0 in the routing-only ablation (no shared pairs)
    const int msh = a.msh;
    const int m4 = (msh + 3) & ~3;
    const int nkeys = m4 + a.k;

    if (tid == 0) {
        for (int w = 0; w < NWG; ++w) {
            // the producer loads the lists (one arrival), or the row warps do
            // (IND: the warpgroup's 4, RL: all of them)
            mbar_init(&kvfull[w], IND ? 4 : (RL ? 4 * NWG : 1));
            mbar_init(&kvfree[w], IND ? 1 : NWG);  // shared lists: one commit per MMA issuer
        }
        for (int w = 0; w < NWG; ++w) {
            mbar_init(&ofree[w], 4);  // one arrival per row warp
            mbar_init(&pfull[w], 4);
            mbar_init(&pvdone[w], 1);
            mbar_init(&sfull[w], 1);
            mbar_init(&sfree[w], 4);
        }
        for (int b = 0; b < NWG * QB; ++b) {
            mbar_init(&qfull[b], IND ? 4 : 1);  // IND: the warpgroup's 4 row warps load the rows
            mbar_init(&qfree[b], 1);
        }
        mbar_init(&drain, NWG);  // exit path: one commit per MMA issuer
        fence_barrier_init();
    }
    // query buffers zeroed before anything copies into them: an item's rows
    // past its last query keep an earlier item's queries or these zeros
    for (int x = tid; x < NWG * QB * 1024; x += NT) zero16(S.q + 16 * x);
    // likewise the list rows past the last gather: zero (their logits are
    // masked; their values must be finite)
    for (int w = 0; w < (IND ? NWG : 1); ++w)
        for (int x = ((nkeys + 3) & ~3) * 8 + tid; x < a.nblk * KB * 8; x += NT) {
            zero16(S.keys + w * S.kvstride + swz128(x >> 3, x & 7));
            zero16(S.vals + w * S.kvstride + swz128(x >> 3, x & 7));
        }
    fence_proxy_async();
    if (warp == 0) tmem_alloc(&tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;

    const int total = *a.nitems;
    const int i0 = static_cast<int>(static_cast<int64_t>(total) * blockIdx.x / gridDim.x);
    const int i1 = static_cast<int>(static_cast<int64_t>(total) * (blockIdx.x + 1) / gridDim.x);
    // IND: warpgroup w's items [j0(w), j0(w + 1))
    auto j0 = [&](int w) { return i0 + static_cast<int>(static_cast<int64_t>(i1 - i0) * w / NWG); };

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        // Every row arrives by TMA 4-row gathers that complete on the consumer's
        // mbarrier: the producer never waits for its own copies. Rows past the
        // last gather stay zero (their logits are masked; their values must be
        // finite).
        // the key/value list of item `it` into list copy w (the shared rows
        // only when the copy held another head's list)
        auto gather_list = [&](const int4& it, int w, bool new_head) {
            uint8_t* keys = S.keys + w * S.kvstride;
            uint8_t* vals = S.vals + w * S.kvstride;
            uint64_t* bar = &kvfull[w];
            const int bh = it.w;
            const int32_t* sel = a.expert_idx + (static_cast<int64_t>(bh) * a.m + it.x) * a.k;
            const int ns = new_head ? m4 / 4 : 0;
            const int nr = (a.k + 3) / 4;
            if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(ns + nr) * 1024u);
            __syncwarp();
            for (int g = lane; g < ns; g += 32) {  // shared rows 4g..4g+3 (the last ones repeat row m-1)
                const int y = bh * a.m;
                const int r0 = 4 * g;
                const int y0 = y + min(r0, a.m - 1), y1 = y + min(r0 + 1, a.m - 1);
                const int y2 = y + min(r0 + 2, a.m - 1), y3 = y + min(r0 + 3, a.m - 1);
                tma_gather4(keys + r0 * 128, &tlq, 0, y0, y1, y2, y3, bar);
                tma_gather4(vals + r0 * 128, &tlv, 0, y0, y1, y2, y3, bar);
            }
            for (int g = lane; g < nr; g += 32) {  // routed rows m4 + 4g.. (the last ones repeat key k-1)
                const int r0 = 4 * g;
                const int y = bh * static_cast<int>(a.N);
                const int y0 = y + sel[min(r0, a.k - 1)], y1 = y + sel[min(r0 + 1, a.k - 1)];
                const int y2 = y + sel[min(r0 + 2, a.k - 1)], y3 = y + sel[min(r0 + 3, a.k - 1)];
                tma_gather4(keys + (m4 + r0) * 128, &tk, 0, y0, y1, y2, y3, bar);
                tma_gather4(vals + (m4 + r0) * 128, &tv, 0, y0, y1, y2, y3, bar);
            }
        };
        uint32_t nq[NWG] = {};
        // the query rows of item `it` into warpgroup w's next query buffer
        auto gather_q = [&](const int4& it, int w) -> bool {
            // this Q buffer of the warpgroup was last used QB items back
            const uint32_t qb = w * QB + (nq[w] % QB);
            if (nq[w] >= QB && !__all_sync(0xffffffffu, mbar_wait(&qfree[qb], ((nq[w] / QB) - 1) & 1, a.status)))
                return false;
            // lane l gathers query rows 4l..4l+3 while 4l < z (the last group
            // repeats the item's last query); the groups after are not copied
            // (a gather costs the issuing warp about a hundred cycles), so
            // those rows keep an earlier item's queries or the initial zeros
            const int ng = (it.z + 3) >> 2;
            if (lane == 0) mbar_arrive_expect_tx(&qfull[qb], static_cast<uint32_t>(ng) * 512u);
            __syncwarp();
            const int bh = it.w;
            const int* pp = a.perm + static_cast<int64_t>(bh) * a.N + it.y;
            const int last = it.z - 1, r0 = 4 * lane;
            const int y = bh * static_cast<int>(a.N);
            if (lane < ng)
                tma_gather4(S.q + qb * 16384 + r0 * 128, &tq, 0, y + pp[min(r0, last)], y + pp[min(r0 + 1, last)],
                            y + pp[min(r0 + 2, last)], y + pp[min(r0 + 3, last)], &qfull[qb]);
            ++nq[w];
            return true;
        };
        bool ok = true;
        // (IND: the row warps load the key lists and their query rows; RL: the
        // key lists)
        int64_t cur_bh = -1;
        int cur_e = -1, changes = 0;
        if constexpr (!IND) {
            for (int r = i0; r < i1 && ok;) {
                int4 it[NWG];
                const int cnt = round_items(a, r, i1, it[0], it[1], it[2]);
                if (!RL && (it[0].w != cur_bh || it[0].x != cur_e)) {
                    // wait until the MMAs reading the previous lists are done
                    if (changes > 0)
                        ok = __all_sync(0xffffffffu, mbar_wait(&kvfree[0], (changes - 1) & 1, a.status));
                    if (!ok) break;
                    gather_list(it[0], 0, it[0].w != cur_bh);
                    cur_bh = it[0].w;
                    cur_e = it[0].x;
                    ++changes;
                }
#pragma unroll
                for (int w = 0; w < NWG; ++w) {
                    if (w >= cnt || !ok) break;
                    ok = gather_q(it[w], w);
                }
                r += cnt;
                if constexpr (MODE == kPlain) {
                    // the next round's expert, if it is another one: its routed
                    // key and value rows into L2 now (a round or two before
                    // its list is gathered), so that the gathers at the list
                    // change find them there instead of in DRAM
                    if (r < i1) {
                        const int4 nx = a.items[r];
                        if (nx.w != it[0].w || nx.x != it[0].x) {
                            const int32_t* sel = a.expert_idx + (static_cast<int64_t>(nx.w) * a.m + nx.x) * a.k;
                            const int64_t hb = static_cast<int64_t>(nx.w) * a.N;
                            for (int i = lane; i < a.k; i += 32) {
                                const int64_t row = hb + sel[i];
                                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.kp + row * D));
                                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.vp + row * D));
                            }
                        }
                    }
                }
            }
        }
        // exit: the last phase of every barrier this warp armed has landed
        if (lane == 0) {
            if (changes > 0) mbar_drain(&kvfull[0], (changes - 1) & 1);
            for (int w = 0; w < NWG; ++w) {
                for (uint32_t b = 0; b < QB; ++b) {
                    const uint32_t arms = nq[w] > b ? (nq[w] - b + QB - 1) / QB : 0;
                    if (arms > 0) mbar_drain(&qfull[w * QB + b], (arms - 1) & 1);
                }
            }
        }
    } else if (warp <= NWG) {
        // ---------------- MMA issuers: lane 0 of warp 1 + w serves warpgroup w ----------------
        // (each issuer has a warp of its own: tcgen05.mma is a single-thread instruction)
        // Per item: S(0), then S(j) and P.V(j - 1) in turn. The next item's
        // S(0) goes out before this item's last P.V when it keeps the
        // key/value lists, so the rows find it ready when they start it. Every
        // MMA covers a whole block: past the key list the logits are masked and
        // the staged rows are finite (zero or repeated), so P = 0 there.
        if (lane == 0) {
            const int w = warp - 1;
            const uint32_t tS = tb + tcol_s(w), tP = tb + tcol_p(w), tO = tb + tcol_o(w);
            // IND: this warpgroup's own list, items and list barriers; the rounds
            // below then hold one item each, all of them this warpgroup's
            const uint64_t kd = sdesc_sw128(smem_u32(S.keys + w * S.kvstride));
            const uint64_t vd = sdesc_sw128(smem_u32(S.vals + w * S.kvstride));
            const uint64_t qd = sdesc_sw128(smem_u32(S.q + w * QB * 16384));  // + 1024 per buffer
            const int we = IND ? 0 : w, ie = IND ? j0(w + 1) : i1;
            uint64_t* kvf = &kvfull[IND ? w : 0];
            uint64_t* kve = &kvfree[IND ? w : 0];
            int r = IND ? j0(w) : i0, cur_bh = -1, cur_e = -1, changes = 0;
            uint32_t gs = 0, gp = 0;  // S and P.V blocks issued
            uint32_t nq = 0;          // items whose S has started (query buffer sequence)
            uint32_t npv = 0;         // items whose P.V is complete
            // S of block j of the item in query buffer sequence q
            auto issue_s = [&](uint32_t q, int j) -> bool {
                const uint32_t qb = w * QB + q % QB;
                if (j == 0) {
                    if (!mbar_wait(&qfull[qb], (q / QB) & 1, a.status)) return false;
                }
                if (gs >= 1 && !mbar_wait(&sfree[w], (gs - 1) & 1, a.status)) return false;  // rows read S(gs - 1)
                tc_fence_after();
                mma_ss_k64(tS, qd + (q % QB) * 1024, kd + j * 512, kIdescS, 0u);
                mma_commit(&sfull[w]);
                if (j == a.nblk - 1) mma_commit(&qfree[qb]);
                ++gs;
                return true;
            };
            // P.V of block j of the current item
            auto issue_pv = [&](int j) -> bool {
                // the first P.V of an item overwrites O (SPLIT: adds to the
                // preloaded shared output): the previous item's epilogue must
                // have read it (SPLIT: the rows have preloaded this item's)
                if (j == 0) {
                    if (SPLIT && !mbar_wait(&ofree[w], npv & 1, a.status)) return false;
                    if (!SPLIT && npv > 0 && !mbar_wait(&ofree[w], (npv - 1) & 1, a.status)) return false;
                }
                if (!mbar_wait(&pfull[w], gp & 1, a.status)) return false;
                tc_fence_after();
                mma_ts_k64(tO, tP, vd + j * 512, kIdescPV, (j > 0 || SPLIT) ? 1u : 0u);
                mma_commit(&pvdone[w]);
                ++gp;
                return true;
            };
            int4 cur;
            int st = next_item(a, we, r, ie, cur_bh, cur_e, changes, kvf, kve, cur, IND);
            bool ok = st >= 0, s0 = false;
            while (ok && st > 0) {
                const uint32_t q = nq++;
                if (!s0) ok = issue_s(q, 0);
                for (int j = 1; j < a.nblk && ok; ++j) ok = issue_s(q, j) && issue_pv(j - 1);
                if (!ok) break;
                s0 = next_same(a, we, r, ie, cur_bh, cur_e, IND);
                if (s0 && !(ok = issue_s(nq, 0))) break;
                if (!(ok = issue_pv(a.nblk - 1))) break;
                ++npv;
                st = next_item(a, we, r, ie, cur_bh, cur_e, changes, kvf, kve, cur, IND);
                ok = st >= 0;
            }
            mma_drain(&drain);  // exit: this issuer's MMAs are done
        }
    } else {
        // ------------------------------ row warpgroups ------------------------------
        // An item's epilogue (O / rowsum -> its output rows) waits until the
        // rows have written the next item's first P: by then its last P.V is
        // done, and the wait for it has overlapped that block's softmax.
        const int w = (warp - 1 - NWG) >> 2;  // 4 consecutive warps cover the 4 TMEM lane quarters
        const int t = (warp & 3) * 32 + lane;  // TMEM lane = query row of the item
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tb + tcol_s(w) + lane_off, tP = tb + tcol_p(w) + lane_off, tO = tb + tcol_o(w) + lane_off;
        uint32_t gb = 0;
        bool ok = true;
        bool pend = false, pend_row = false;  // an item whose epilogue is pending
        float pend_inv = 0.f;
        uint4* pend_dst = nullptr;
        float pend_m = 0.f, pend_l = 0.f;  // MULTI, STATS: the running max and sum
        int64_t pend_pos = 0;              // STATS: head * N + the row's position in the grouping
        float* pend_state = nullptr;       // MULTI: the query's state row
        auto epilogue = [&]() {
            if constexpr (STATS) {
                // Delta = dO . (O / rowsum) in fp32, and the log-sum-exp
                const float dl = stats_delta(tO, reinterpret_cast<const __nv_bfloat16*>(pend_dst), pend_inv,
                                             pend_row);
                tc_fence_before();
                warp_arrive(&ofree[w]);
                if (pend_row) {  // (in grouped order: the row's position in the grouping)
                    a.st_delta[pend_pos] = dl;
                    a.st_lse[pend_pos] = pend_m + __log2f(pend_l);
                }
            } else if constexpr (!MULTI) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // two 32-column halves of the output row
                    float o[32];
                    tmem_ld32(tO + h * 32, o);
                    tmem_ld_wait();
                    if (h == 1 && !SPLIT) {  // (SPLIT: the next item's preload releases O)
                        tc_fence_before();
                        warp_arrive(&ofree[w]);
                    }
                    if (pend_row) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint4 q;
                            q.x = pack_bf16(o[8 * c + 0] * pend_inv, o[8 * c + 1] * pend_inv);
                            q.y = pack_bf16(o[8 * c + 2] * pend_inv, o[8 * c + 3] * pend_inv);
                            q.z = pack_bf16(o[8 * c + 4] * pend_inv, o[8 * c + 5] * pend_inv);
                            q.w = pack_bf16(o[8 * c + 6] * pend_inv, o[8 * c + 7] * pend_inv);
                            pend_dst[h * 4 + c] = q;
                        }
                    }
                }
            } else {
                // merge (pend_m, pend_l, O of this pass) with the state of the
                // earlier passes (none in pass 0); max -inf: nothing there
                float ms = -INFINITY, ls = 0.f;
                if (pend_row && a.j > 0) {
                    const float2 ml = *reinterpret_cast<const float2*>(pend_state + D);
                    ms = ml.x;
                    ls = ml.y;
                }
                const float mt = fmaxf(ms, pend_m);
                const float fs = ms == -INFINITY ? 0.f : exp2f(ms - mt);
                const float fp = pend_m == -INFINITY ? 0.f : exp2f(pend_m - mt);
                const float lt = ls * fs + pend_l * fp;
                const bool last = a.j == a.s - 1;
                const float inv = last ? 1.f / lt : 1.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float o[32];
                    tmem_ld32(tO + h * 32, o);
                    tmem_ld_wait();
                    if (h == 1) {
                        tc_fence_before();
                        warp_arrive(&ofree[w]);
                    }
                    if (pend_row) {
                        float4* sr = reinterpret_cast<float4*>(pend_state + h * 32);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            float4 x = make_float4(o[4 * c] * fp, o[4 * c + 1] * fp, o[4 * c + 2] * fp,
                                                   o[4 * c + 3] * fp);
                            if (a.j > 0) {
                                const float4 y = sr[c];
                                x.x = fmaf(y.x, fs, x.x);
                                x.y = fmaf(y.y, fs, x.y);
                                x.z = fmaf(y.z, fs, x.z);
                                x.w = fmaf(y.w, fs, x.w);
                            }
                            if (last) {
                                uint2 q;
                                q.x = pack_bf16(x.x * inv, x.y * inv);
                                q.y = pack_bf16(x.z * inv, x.w * inv);
                                reinterpret_cast<uint2*>(pend_dst)[h * 8 + c] = q;
                            } else {
                                sr[c] = x;
                            }
                        }
                    }
                }
                if (pend_row && !last) *reinterpret_cast<float2*>(pend_state + D) = make_float2(mt, lt);
            }
            pend = false;
        };
        // IND: this warpgroup's own range, one item per round. Its row warps
        // load the query rows themselves (the producer's TMA gathers are the
        // bottleneck of short lists, and these warps are mostly waiting):
        // each warp its 32 rows of the next item, lanes 0-7 one 4-row gather
        // each, during the current item's first block; the first item's at
        // the start.
        const int re = IND ? j0(w + 1) : i1;
        uint32_t qseq = 0;                    // IND: items of this warpgroup so far
        int qarm_b = -1;                      // IND: the last query buffer this warp armed
        uint32_t qarm_par = 0;
        const int qg = 8 * (warp & 3) + lane;  // IND: this lane's 4-row group of an item (lanes 0-7)
        // IND: the sources of this lane's group of item x (rows past z repeat its last query)
        auto q_src = [&](const int4& x, int* pq) {
            const int* pp = a.perm + static_cast<int64_t>(x.w) * a.N + x.y;
            const int last = x.z - 1, r0 = 4 * qg, y = x.w * static_cast<int>(a.N);
#pragma unroll
            for (int i = 0; i < 4; ++i) pq[i] = (lane < 8 && r0 < x.z) ? y + pp[min(r0 + i, last)] : 0;
        };
        // IND: item number u of this warpgroup (z queries, rows from pq) into its query buffer
        auto q_load = [&](int z, uint32_t u, const int* pq) -> bool {
            const uint32_t qb = w * QB + u % QB;
            // the buffer's previous item (u - QB) must be done with it (its S products)
            if (u >= QB && !__all_sync(0xffffffffu, mbar_wait(&qfree[qb], ((u / QB) - 1) & 1, a.status)))
                return false;
            const int ng = min(8, max(0, (z - 32 * (warp & 3) + 3) >> 2));  // this warp's groups
            if (lane == 0) mbar_arrive_expect_tx(&qfull[qb], static_cast<uint32_t>(ng) * 512u);
            __syncwarp();
            if (lane < ng) tma_gather4(S.q + qb * 16384 + qg * 512, &tq, 0, pq[0], pq[1], pq[2], pq[3], &qfull[qb]);
            qarm_b = static_cast<int>(qb);
            qarm_par = (u / QB) & 1;
            return true;
        };
        // The key/value list of item x (the head's shared rows too when
        // new_head) into the warpgroup's list (IND) or the CTA's: its 4-row
        // gathers, keys and values, spread over the warpgroup's 4 row warps
        // (IND) or all 4 NWG of them (op o: row warp o mod nw, lane o / nw);
        // each warp arrives once on kvfull with its own bytes. A TMA gather
        // costs its issuing warp about a hundred cycles, so one warp alone
        // would take ~10K cycles per list at k = 256.
        constexpr int NWL = IND ? 4 : 4 * NWG;  // warps sharing a list's gathers
        int* ls = s_list[warp - 1 - NWG];        // [0] head, [1] expert of the list held, [2] lists armed
        if (lane == 0) {
            ls[0] = -1;
            ls[1] = -1;
            ls[2] = 0;
        }
        __syncwarp();
        auto l_load = [&](const int4& x, bool new_head) {
            const int wl = IND ? (warp & 3) : (warp - 1 - NWG);
            uint64_t* kvf = &kvfull[IND ? w : 0];
            uint8_t* keys = S.keys + (IND ? w * S.kvstride : 0);
            uint8_t* vals = S.vals + (IND ? w * S.kvstride : 0);
            const int32_t* sel = a.expert_idx + (static_cast<int64_t>(x.w) * a.m + x.x) * a.k;
            const int ns = new_head ? m4 / 4 : 0, nr = (a.k + 3) / 4, nops = 2 * (ns + nr);
            const int mine = nops > wl ? (nops - wl + NWL - 1) / NWL : 0;  // ops o = wl + NWL i
            if (lane == 0) mbar_arrive_expect_tx(kvf, static_cast<uint32_t>(mine) * 512u);
            __syncwarp();
            for (int o = wl + NWL * lane; o < nops; o += 32 * NWL) {
                const int g = o >> 1;
                const bool isv = o & 1;
                if (g < ns) {  // shared rows 4g..4g+3 (the last ones repeat row m-1)
                    const int y = x.w * a.m, r0 = 4 * g;
                    tma_gather4((isv ? vals : keys) + r0 * 128, isv ? &tlv : &tlq, 0, y + min(r0, a.m - 1),
                                y + min(r0 + 1, a.m - 1), y + min(r0 + 2, a.m - 1), y + min(r0 + 3, a.m - 1), kvf);
                } else {  // routed rows m4 + 4(g - ns).. (the last ones repeat key k-1)
                    const int r0 = 4 * (g - ns), y = x.w * static_cast<int>(a.N);
                    tma_gather4((isv ? vals : keys) + (m4 + r0) * 128, isv ? &tv : &tk, 0,
                                y + sel[min(r0, a.k - 1)], y + sel[min(r0 + 1, a.k - 1)],
                                y + sel[min(r0 + 2, a.k - 1)], y + sel[min(r0 + 3, a.k - 1)], kvf);
                }
            }
            __syncwarp();
            if (lane == 0) {
                ls[0] = x.w;
                ls[1] = x.x;
                ++ls[2];
            }
            __syncwarp();
        };
        if constexpr (RL && !IND) {
            if (i0 < i1) l_load(a.items[i0], true);  // the first list (every row warp of the CTA)
        }
        if constexpr (IND) {
            if (j0(w) < re) {
                const int4 x = a.items[j0(w)];
                l_load(x, true);
                int pq[4];
                q_src(x, pq);
                ok = q_load(x.z, 0, pq);
            }
        }
        for (int r = IND ? j0(w) : i0; r < re && ok;) {
            int4 x0, x1, x2;
            const int cnt = round_items(a, r, re, x0, x1, x2, IND);
            r += cnt;
            if constexpr (RL && !IND) {
                // a new list: once every MMA issuer has released the old one
                // (its products are done), every row warp loads its share
                if (x0.w != ls[0] || x0.x != ls[1]) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&kvfree[0], (ls[2] - 1) & 1, a.status));
                    if (!ok) break;
                    l_load(x0, x0.w != ls[0]);
                }
            }
            if (!IND && w >= cnt) continue;
            const int4 item = IND ? x0 : pick(w, x0, x1, x2);
            const int64_t bh = item.w;
            const int n = t < item.z ? a.perm[bh * a.N + item.y + t] : 0;
            // IND: the next item's query rows load after this item's first block
            const bool qnext = IND && r < re;
            // SPLIT: the shared branch as one pre-merged pair (logit lse, weight 1);
            // its output row comes in now, and is read in the first block
            float mrun = -INFINITY, lrun = 0.f;
            if constexpr (SPLIT) {
                mrun = t < item.z ? a.lse[bh * a.N + n] : 0.f;
                lrun = 1.f;
                const __nv_bfloat16* src = a.osh + (bh * a.N + n) * D;  // (padding rows: query 0's, finite)
                const uint32_t dst = smem_u32(S.ps + w * 16384);
#pragma unroll
                for (int c = 0; c < 8; ++c) cp_async16(dst + swz128(t, c), src + 8 * c);
                asm volatile("cp.async.commit_group;" ::: "memory");
            }
            float* srow = nullptr;
            const uint64_t* mrow = nullptr;  // MULTI, passes j > 0: this row's masks, one word per block
            uint64_t dm0 = 0;                // the word of the next block (first: loaded with the item)
            if constexpr (MULTI) {
                if (a.j > 0 && t < item.z) {
                    mrow = a.mask + (bh * a.N + item.y + t) * static_cast<int64_t>(a.nbw);
                    dm0 = mrow[0];
                }
                srow = a.state + (bh * a.N + n) * 68;
                if (a.j > 0 && t < item.z) {  // the epilogue reads it: start bringing it in
                    const char* p0 = reinterpret_cast<const char*>(srow);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(p0 + (x < 3 ? 128 * x : 271)));
                }
            }
            for (int j = 0; j < a.nblk; ++j, ++gb) {
                // MULTI, passes j > 0: the block's keys an earlier-ranked expert
                // of the query holds (bit c: key column c)
                uint64_t dm = 0;
                if constexpr (MULTI) {
                    if (mrow) {  // this block's word; the next one loads during this block
                        dm = dm0;
                        if (j + 1 < a.nblk) dm0 = mrow[j + 1];
                    }
                }
                ok = __all_sync(0xffffffffu, mbar_wait(&sfull[w], gb & 1, a.status));
                if (!ok) break;
                tc_fence_after();
                float s[KB];
#pragma unroll
                for (int c = 0; c < KB; c += 32) tmem_ld32(tS + c, s + c);
                tmem_ld_wait();
                tc_fence_before();
                warp_arrive(&sfree[w]);
                const int k0 = j * KB;  // key row of column 0
                if (k0 + KB > nkeys || (k0 < m4 && k0 + KB > msh && m4 > msh)) {
                    // (warp-uniform) the block holds the unused rows [m, m4) or
                    // ends past the key list, where the logits are not keys'
#pragma unroll
                    for (int c = 0; c < KB; ++c) {
                        const int g = k0 + c;
                        s[c] = (g >= nkeys || (g >= msh && g < m4)) ? -INFINITY : s[c];
                    }
                }
                if constexpr (MULTI) {
                    if (dm) {
#pragma unroll
                        for (int c = 0; c < KB; ++c) s[c] = ((dm >> c) & 1) ? -INFINITY : s[c];
                    }
                }
                // 8 independent partial maxima: short dependency chains
                float pm[8];
                static_assert(KB == 64, "the partial maxima below cover exactly 64 columns");
#pragma unroll
                for (int u = 0; u < 8; ++u)  // columns u, u+8, ..., u+56
                    pm[u] = fmax3(fmax3(s[u], s[u + 8], s[u + 16]), fmax3(s[u + 24], s[u + 32], s[u + 40]),
                                  fmaxf(s[u + 48], s[u + 56]));
                const float smax = fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(fmax3(pm[3], pm[4], pm[5]), pm[6], pm[7]));
                const float bmax = smax * kC;
                const float mnew = (bmax > mrun + kLazy) ? bmax : mrun;
                // 0 on the first block, 1 when the max is kept. MULTI: a row
                // may have no key yet (max -inf): then every weight is 0
                const float alpha = (MULTI && mnew == -INFINITY) ? 1.f : exp2f(mrun - mnew);
                const float mexp = (MULTI && mnew == -INFINITY) ? 0.f : mnew;
                // The P.V product sees the weights rounded to bf16, the row sum
                // below adds them unrounded; the block's largest weight
                // dominates the difference, so the sum takes its rounding
                // (computed exactly as in the loop: same fused multiply-add).
                const float emax = exp2f(fmaf(smax, kC, -mexp));
                const float corr = __bfloat162float(__float2bfloat16_rn(emax)) - emax;
                // packed pairs: one f32x2 FMA forms two exponents, one f32x2 add
                // accumulates two weights; P goes out as bf16 pairs
                const float2 c2 = make_float2(kC, kC), m2 = make_float2(-mexp, -mexp);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                uint32_t pk[KB / 2];
#pragma unroll
                for (int c = 0; c < KB; c += 2) {
                    const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), c2, m2);
                    const float2 e = make_float2(exp2f(x.x), exp2f(x.y));
                    acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], e);
                    pk[c >> 1] = pack_bf16(e.x, e.y);
                }
                const float sum = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
                lrun = lrun * alpha + (sum + corr);
                // P.V of the previous block (for j = 0 the previous item's last)
                // must be done before P is overwritten or O rescaled
                const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
                if (gb >= 1) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&pvdone[w], (gb - 1) & 1, a.status));
                    if (!ok) break;
                }
                tc_fence_after();
                if (rescale) tmem_scale64(tO, alpha);
                tmem_st32u(tP, pk);
                tmem_st_wait();
                tc_fence_before();
                warp_arrive(&pfull[w]);
                if (pend) epilogue();  // the previous item's O is final (its last P.V is done)
                if (qnext && j == 0) {
                    const int4 xn = a.items[r];
                    int pqn[4];
                    q_src(xn, pqn);
                    if (!(ok = q_load(xn.z, qseq + 1, pqn))) break;
                }
                if (SPLIT && j == 0) {
                    // O := alpha o_n (the shared output at this block's running
                    // max), before this item's first P.V adds to it; each thread
                    // reads back only the row it copied itself
                    cp_async_wait_all();
                    preload_shared(tO, S.ps + w * 16384, t, alpha);
                    warp_arrive(&ofree[w]);
                }
                mrun = mnew;
            }
            if (!ok) break;
            if (qnext) {
                // IND: the next item's list, once this item's last P.V (and
                // with it every product reading the list) is done
                const int4 xn = a.items[r];
                if (xn.w != ls[0] || xn.x != ls[1]) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&pvdone[w], (gb - 1) & 1, a.status));
                    if (!ok) break;
                    tc_fence_after();
                    l_load(xn, xn.w != ls[0]);
                }
            }
            ++qseq;
            pend = true;
            pend_row = t < item.z;
            pend_inv = 1.f / lrun;
            // (STATS: the query's dO row instead of its output row)
            pend_dst = reinterpret_cast<uint4*>((STATS ? const_cast<__nv_bfloat16*>(a.dO) : a.out) + (bh * a.N + n) * D);
            if constexpr (STATS) pend_pos = bh * a.N + item.y + t;
            pend_m = mrun;
            pend_l = lrun;
            pend_state = srow;
        }
        if (ok && pend) {  // the last item: wait for its last P.V
            ok = __all_sync(0xffffffffu, mbar_wait(&pvdone[w], (gb - 1) & 1, a.status));
            if (ok) {
                tc_fence_after();
                epilogue();
            }
        }
        // IND exit: this warp's last query copies have landed (on the normal
        // path the issuer has waited for them already)
        if (IND && qarm_b >= 0 && lane == 0) mbar_drain(&qfull[qarm_b], qarm_par);
        if ((IND || RL) && ls[2] > 0 && lane == 0) mbar_drain(&kvfull[IND ? w : 0], (ls[2] - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tb, 512);
}

size_t smem_bytes(int nblk, bool split, bool ind = false) {
    return 1024 + static_cast<size_t>(nblk) * 16384 * (ind ? NWG : 1) + NWG * QB * 16384 + (split ? NWG * 16384 : 0);
}

// the shared pairs enter the key list unless they are absent (routing-only
// ablation) or already folded into each query's shared-branch partial
int key_rows(const Plan& p) { return (p.shared && !p.split ? (p.s.m + 3) & ~3 : 0) + p.s.k; }

}  // namespace

bool expert_tc_supported(const Plan& p) {
    return key_rows(p) <= 512 && p.s.BH * p.s.N < (int64_t(1) << 31) &&
           smem_bytes((key_rows(p) + KB - 1) / KB, p.split) <= 232448;
}

bool expert_split_fits(const Plan& p) {
    const int rows = p.s.k;  // the routed keys alone
    return rows <= 512 && p.s.BH * p.s.N < (int64_t(1) << 31) && smem_bytes((rows + KB - 1) / KB, true) <= 232448;
}

cudaError_t launch_expert_tc(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                             const __nv_bfloat16* V, const int32_t* expert_idx, __nv_bfloat16* out, cudaStream_t st,
                             const int32_t* route, int j) {
    (void)route;  // the passes read the per-slot masks built from it
    const bool multi = p.s.s_route > 1;
    Args a{};
    a.items = w.items + static_cast<size_t>(j) * p.s.BH * p.max_items;  // the plane of rank j
    a.nitems = w.nitems + j;
    a.perm = w.perm + static_cast<size_t>(j) * p.s.BH * p.s.N;
    a.expert_idx = expert_idx;
    a.out = out;
    a.status = w.status;
    a.N = p.s.N;
    a.m = p.s.m;
    a.msh = p.shared && j == 0 && !p.split ? p.s.m : 0;
    a.k = p.s.k;
    a.nblk = ((a.msh + 3) / 4 * 4 + a.k + KB - 1) / KB;
    a.s = p.s.s_route;
    a.j = j;
    a.nbw = (p.s.k + 63) / 64;
    if (multi) {  // (the union holds one mode's pointers)
        a.mask = j > 0 ? w.mask + static_cast<size_t>(j - 1) * p.s.BH * p.s.N * ((p.s.k + 63) / 64) : nullptr;
        a.state = w.state;
    } else if (p.split) {
        a.lse = w.lse;
        a.osh = w.osh;
    } else {
        a.kp = K;
        a.vp = V;
    }
    CUtensorMap tq, tk, tv, tlq, tlv;
    const uint64_t rows = static_cast<uint64_t>(p.s.BH) * p.s.N, lrows = static_cast<uint64_t>(p.s.BH) * p.s.m;
    if (!make_row_tmap(&tq, Q, rows, 1) || !make_row_tmap(&tk, K, rows, 1) || !make_row_tmap(&tv, V, rows, 1) ||
        !make_row_tmap(&tlq, w.lqhi, lrows, 1) || !make_row_tmap(&tlv, w.lvbf, lrows, 1))
        return cudaErrorInvalidValue;
    const size_t sm = smem_bytes(a.nblk, p.split);
    // short lists (the ViT shapes, short sequences): a list per warpgroup
    const bool ind = !multi && !p.split && smem_bytes(a.nblk, false, true) <= 232448;
    const size_t smi = ind ? smem_bytes(a.nblk, false, true) : sm;
    // the row warps load the key lists when an expert owns few items (its
    // list is reloaded every few rounds): N / m queries per expert, <= 16 items
    const bool rl = !multi && !p.split && !ind && p.s.N / p.s.m <= 16 * 128;
    auto kern = multi ? expert_tc_kernel<kMulti, false>
                      : (p.split ? expert_tc_kernel<kSplit, false>
                                 : (ind ? expert_tc_kernel<kPlain, true>
                                        : (rl ? expert_tc_kernel<kPlain, false, true> : expert_tc_kernel<kPlain, false>)));
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smi));
    if (e != cudaSuccess) return e;
    if (multi) {
        // (the s > 1 passes follow each other directly: launched early, the
        // next pass's attention measured 1.1 ms slower at long1m, s = 2)
        kern<<<device_sms(), NT, smi, st>>>(tq, tk, tv, tlq, tlv, a);
        return cudaGetLastError();
    }
    return launch_dep(kern, dim3(device_sms()), dim3(NT), smi, st, tq, tk, tv, tlq, tlv, a);
}

cudaError_t launch_expert_stats(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                                const __nv_bfloat16* V, const int32_t* expert_idx, const __nv_bfloat16* dO,
                                float* st_lse, float* st_delta, cudaStream_t st) {
    Args a{};
    a.items = w.items;
    a.nitems = w.nitems;
    a.perm = w.perm;
    a.expert_idx = expert_idx;
    a.out = nullptr;
    a.status = w.status;
    a.N = p.s.N;
    a.m = p.s.m;
    a.msh = p.s.m;
    a.k = p.s.k;
    a.nblk = ((a.msh + 3) / 4 * 4 + a.k + KB - 1) / KB;
    a.s = 1;
    a.dO = dO;
    a.st_lse = st_lse;
    a.st_delta = st_delta;
    CUtensorMap tq, tk, tv, tlq, tlv;
    const uint64_t rows = static_cast<uint64_t>(p.s.BH) * p.s.N, lrows = static_cast<uint64_t>(p.s.BH) * p.s.m;
    if (!make_row_tmap(&tq, Q, rows, 1) || !make_row_tmap(&tk, K, rows, 1) || !make_row_tmap(&tv, V, rows, 1) ||
        !make_row_tmap(&tlq, w.lqhi, lrows, 1) || !make_row_tmap(&tlv, w.lvbf, lrows, 1))
        return cudaErrorInvalidValue;
    const size_t sm = smem_bytes(a.nblk, false);
    cudaError_t e = cudaFuncSetAttribute(expert_tc_kernel<kStats, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sm));
    if (e != cudaSuccess) return e;
    return launch_dep(expert_tc_kernel<kStats, false>, dim3(device_sms()), dim3(NT), sm, st, tq, tk, tv, tlq, tlv, a);
}

}  // namespace mita
