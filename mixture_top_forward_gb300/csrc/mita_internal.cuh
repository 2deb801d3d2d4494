// Internal declarations shared by the kernels of libmita.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mita.h"

// Largest m and k the kernels' shared-memory tables hold (the public limits
// MITA_MAX_M / MITA_MAX_K in mita.h must not exceed these).
#define MITA_MAX_M_INTERNAL 1024
#define MITA_SORT_MAX 1024

namespace mita {

constexpr int D = 64;  // head dimension the kernels are built for

// ----------------------------------------------------------------------------
// Problem shape and the workspace plan of one call.
// ----------------------------------------------------------------------------
struct Shape {
    int64_t BH;     // B*H heads
    int64_t N;      // tokens per head
    int gh, gw;     // token grid (0,0 = 1-D)
    int p;          // landmark grid side for 2-D (m = p*p), 0 for 1-D
    int m, k;       // landmarks, keys per routed expert
    int s_route;    // routed experts per query (s)
};

// One scan over (a sample of) every head's keys.
struct ScanLevel {
    int64_t S;          // keys scanned per head (samples 0..S-1)
    int64_t stride;     // sample s is key s * stride
    int64_t chunk_len;  // samples per chunk (last one may be shorter)
    int chunks;         // chunks per head (one CTA each)
    int cap;            // candidate slots per (head, chunk, landmark)
    int rcap;           // group records per (head, chunk, landmark) (tensor-core scans; 0: none)
    bool dense;         // write every logit ([BH][m][ld] floats) instead of candidates
    int64_t ld;         // row stride of those logits (S rounded up to 4)
};

struct Plan {
    Shape s;
    // landmark scan: pilot levels on strided samples, then the main scan
    // (lev[nlev-1], stride 1); scan_tc selects the tensor-core kernels
    bool scan_tc;
    // false: the routing-only ablation (no shared pairs in the attention; the
    // main scan then computes no LV)
    bool shared;
    int nlev;
    ScanLevel lev[4];
    // dense top-k: when no sample threshold could keep the main scan's
    // candidates rare, the main scan writes every logit and the select ranks
    // whole rows (no pilots, no candidate buffers)
    bool dense;
    int64_t dense_ld;  // row stride of the dense logits (N rounded up to 4)
    // speculative main-scan threshold (0: off): the last pilot passes the
    // spec_j-th best key of its sample instead of the k-th; a head where a
    // landmark then keeps fewer than k candidates is scanned again from the
    // k-th (safe) thresholds
    int spec_j;
    // routing / grouping
    int rblock;         // queries per routing CTA
    int64_t nrblocks;   // routing CTAs per head
    // expert attention
    int qtile;          // queries per expert work item
    int64_t max_items;  // work items per head, upper bound
    // s > 1 routing: the attention passes run on the tensor cores (with the
    // expert overlap table) or, where that kernel does not apply, on the CUDA cores
    bool multi_tc;
    // s = 1 with the shared branch on the tensor cores: the routing kernel also
    // forms each query's softmax partial over the m landmark logits (o, lse)
    // and the expert kernel attends to the routed keys alone, continuing it
    bool split;
    // workspace layout (byte offsets)
    size_t off_status, off_lq32, off_lqhi, off_lqlo, off_lv32, off_lvbf, off_part, off_cand, off_ccount, off_theta,
        off_counts, off_expoff, off_cursor, off_perm, off_items, off_nitems, off_dense, off_ridx, off_rval, off_rcount,
        off_state, off_ovl, off_mask, off_osh, off_lse, off_theta_safe, off_hflag, total;
};

// Builds the plan; returns false if a size does not fit the int ranges used.
// split: fold the shared branch into the routing kernel where its kernels
// apply (mita_forward_split).
bool make_plan(const Shape& s, Plan* p, bool shared = true, bool split = false);

// Workspace pointers derived from a plan.
struct Work {
    int* status;            // device status word (MITA_ERR_TIMEOUT etc.)
    float* lq32;            // [BH][m][64]
    __nv_bfloat16* lqhi;    // [BH][m][64]  bf16(Lq)
    __nv_bfloat16* lqlo;    // [BH][m][64]  bf16(Lq - bf16(Lq))
    float* lv32;            // [BH][m][64]
    __nv_bfloat16* lvbf;    // [BH][m][64]
    float* part;            // [BH][chunks][m][68]: max, sum, -, -, o[64]
    uint64_t* cand;         // [BH][chunks][m][cap] composite top-k keys
    int* ccount;            // [BH][chunks][m]
    uint32_t* ridx;         // [BH][chunks][m][rcap] group records: sample index of the group's first key
    float* rval;            // [BH][chunks][m][rcap][8] group records: the group's 8 raw logits
    int* rcount;            // [BH][chunks][m]
    uint64_t* theta;        // [BH][m] top-k thresholds from the pilot scans
    uint64_t* theta_safe;   // [BH][m] spec_j: the last pilot's k-th best keys (the fallback thresholds)
    int* hflag;             // [BH] spec_j: heads to scan again from theta_safe
    float* dense;           // [BH][m][dense_ld] raw logits <Lq_i, K_j> (dense top-k only)
    int* counts;            // [s][BH][m] queries routed to each expert (per rank of the routes)
    int* expoff;            // [BH][m+1] exclusive prefix of counts
    int* cursor;            // [BH][m] scatter cursors
    int* perm;              // [s][BH][N] queries grouped by expert (rank j of the routes: plane j)
    int4* items;            // [s][BH*max_items] flat lists: (expert, start, len, head)
    int* nitems;            // [s] number of items in each flat list
    float* state;           // [BH][N][68] running softmax state between the passes of s > 1 routing
    uint64_t* ovl;          // [BH][m][m][ceil(k/64)] expert overlap bit masks (s > 1, tensor cores)
    uint64_t* mask;         // [s-1][BH][N][ceil(k/64)] per grouping slot of ranks 1..s-1: keys already counted
    __nv_bfloat16* osh;     // split: [BH][N][64] each query's shared-branch output (normalised)
    float* lse;             // split: [BH][N] its log-sum-exp (log2 units of the tau-scaled logits)
};

Work carve(const Plan& p, void* base);

// ----------------------------------------------------------------------------
// Device helpers.
// ----------------------------------------------------------------------------
// Top-k order key: larger score first, then lower key index. The float is
// mapped to an order-preserving unsigned integer (-0 folded onto +0), the
// index is stored inverted so that a lower index compares larger.
__device__ __forceinline__ uint64_t topk_key(float s, uint32_t j) {
    uint32_t u = __float_as_uint(s);
    if ((u << 1) == 0) u = 0;  // -0 -> +0
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<uint64_t>(u) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - j);
}
__device__ __forceinline__ uint32_t topk_key_index(uint64_t key) {
    return 0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFu);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& raw, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        float2 x = __bfloat1622float2(h[t]);
        f[2 * t] = x.x;
        f[2 * t + 1] = x.y;
    }
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

constexpr float kLog2e = 1.4426950408889634f;

// ----------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched by launch_dep may be
// scheduled while the kernel before it in the stream is still finishing, so
// the launch latency overlaps that kernel's tail (about 2.5 us per kernel
// boundary, measured on GB300). Such a kernel calls dep_entry() first, before
// it touches memory or allocates tensor memory: the wait returns once the
// kernel before has completed and its writes are visible (at once when there
// is no such dependency), and the trigger lets the next kernel's launch start.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void dep_entry() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... P, typename... A>
cudaError_t launch_dep(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<P>(args)...);
}

// ----------------------------------------------------------------------------
// Launchers (each returns cudaGetLastError() of its launches).
// ----------------------------------------------------------------------------
cudaError_t launch_pool(const Plan& p, const Work& w, const __nv_bfloat16* Q, cudaStream_t st);
cudaError_t launch_scan(const Plan& p, const Work& w, const __nv_bfloat16* K, const __nv_bfloat16* V,
                        cudaStream_t st);
cudaError_t launch_scan_tc(const Plan& p, const Work& w, const __nv_bfloat16* K, const __nv_bfloat16* V, int level,
                           cudaStream_t st);
// After the main scan from a speculative threshold (p.spec_j): flags every
// head with a landmark that kept fewer than k candidates and scans those
// heads' keys again, candidates only, from the safe thresholds.
cudaError_t launch_scan_verify(const Plan& p, const Work& w, const __nv_bfloat16* K, cudaStream_t st);
// lse_out (optional): each landmark's log-sum-exp over all keys of tau <Lq_i, K_j>.
// Dense rows of at most 4096 logits take a warp-per-landmark kernel.
bool dense_row_select_applies(const Plan& p);
cudaError_t launch_select(const Plan& p, const Work& w, int32_t* expert_idx, cudaStream_t st,
                          float* lse_out = nullptr);
cudaError_t launch_pilot_select(const Plan& p, const Work& w, int level, cudaStream_t st);
cudaError_t launch_route(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route, cudaStream_t st);
cudaError_t launch_route_simt(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route,
                              cudaStream_t st);
cudaError_t launch_route_tc(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route, cudaStream_t st);
bool route_tc_supported(const Plan& p);

cudaError_t launch_group(const Plan& p, const Work& w, const int32_t* route, int j, cudaStream_t st);
cudaError_t launch_route_multi(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route,
                               cudaStream_t st);
cudaError_t launch_expert_multi(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                                const __nv_bfloat16* V, const int32_t* expert_idx, const int32_t* route, int j,
                                __nv_bfloat16* out, cudaStream_t st);
size_t expert_multi_state_bytes(const Plan& p);
size_t overlap_bytes(const Shape& s);
size_t pass_mask_bytes(const Shape& s);
cudaError_t launch_overlap(const Plan& p, const Work& w, const int32_t* expert_idx, const int32_t* route,
                           cudaStream_t st);
cudaError_t launch_expert(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                          const __nv_bfloat16* V, const int32_t* expert_idx, __nv_bfloat16* out, cudaStream_t st);
cudaError_t launch_expert_simt(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                               const __nv_bfloat16* V, const int32_t* expert_idx, __nv_bfloat16* out,
                               cudaStream_t st);
// route/j: s > 1 routing, the pass of rank j (route is [BH][N][s]); s = 1: nullptr, 0
cudaError_t launch_expert_tc(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                             const __nv_bfloat16* V, const int32_t* expert_idx, __nv_bfloat16* out, cudaStream_t st,
                             const int32_t* route = nullptr, int j = 0);
bool expert_tc_supported(const Plan& p);
// The backward pass's statistics of the query-expert attention (the plain
// forward pass's sequence with the shared pairs in the key list): per query
// the log-sum-exp of its m + k logits (log2 units of tau <q, key>) and
// Delta = dO . out, into st_lse and st_delta ([BH][N] each, in the grouped
// order: entry head * N + p is the query perm[head][p]).
cudaError_t launch_expert_stats(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                                const __nv_bfloat16* V, const int32_t* expert_idx, const __nv_bfloat16* dO,
                                float* st_lse, float* st_delta, cudaStream_t st);
bool expert_split_fits(const Plan& p);
bool route_shared_supported(const Plan& p);
cudaError_t launch_route_shared(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route,
                                cudaStream_t st);

// Backward pass: its own workspace (byte offsets) next to the forward plan's.
struct BwdLayout {
    int ltiles, chunks;      // landmark tiles of 128; key chunks of the landmark-side kernels
    int64_t chunk_len;
    size_t off_lv, off_lse, off_part, off_dlq, off_dlv, off_dlt, off_route;
    // tensor-core path: per-query statistics, the recomputed expert sets, the
    // landmarks' log-sum-exp (log2 units) and dLV in bf16
    size_t off_qlse, off_qdelta, off_eidx, off_lse2, off_dlvb, off_qg, off_dog, total;
};
BwdLayout backward_layout(const Plan& p);
// Gradients dQ, dK, dV (fp32, [BH][N][64], overwritten) of sum(out * dO) with
// the given experts and routes held fixed; uses the forward plan's workspace
// for pooling and grouping and `bbase` (BwdLayout::total bytes) for the rest.
cudaError_t launch_backward(const Plan& p, const Work& w, const BwdLayout& L, void* bbase, const __nv_bfloat16* Q,
                            const __nv_bfloat16* K, const __nv_bfloat16* V, const __nv_bfloat16* dO,
                            const int32_t* expert_idx, const int32_t* route, float* dQ, float* dK, float* dV,
                            cudaStream_t st);

// One thread waits, with the kernels' bounded wait and the given limit, on an
// mbarrier nothing completes; records MITA_ERR_TIMEOUT in *status.
cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t st);

// Backward pass on the tensor cores (backward_tc.cu). The expert part: dK,
// dV of the routed keys (added atomically) and dLq, dLV of the shared keys
// (added atomically), then dQ, from the statistics of launch_expert_stats. The landmark part: dK, dV (added) and dLq (added
// atomically), from each landmark's log-sum-exp (log2 units) and
// Delta' = dLV . LV, with dLV rounded to bf16.
bool backward_tc_supported(const Plan& p);
// (Qg, dOg: Q and dO rows in grouped order, [BH][N][64] bf16)
cudaError_t launch_backward_tc_expert_keys(const Plan& p, const Work& w, const __nv_bfloat16* Qg,
                                           const __nv_bfloat16* K, const __nv_bfloat16* V, const __nv_bfloat16* dOg,
                                           const int32_t* expert_idx, const float* st_lse, const float* st_delta,
                                           float* dK, float* dV, float* dlq, float* dlv, cudaStream_t st);
// dQ (written): the expert attention's share plus the pooling's share of
// the complete dLq, so it runs after the landmark part
cudaError_t launch_backward_tc_expert_rows(const Plan& p, const Work& w, const __nv_bfloat16* Qg,
                                           const __nv_bfloat16* K, const __nv_bfloat16* V, const __nv_bfloat16* dOg,
                                           const int32_t* expert_idx, const float* st_lse, const float* st_delta,
                                           const float* dlq, float* dQ, cudaStream_t st);
cudaError_t launch_backward_tc_landmark(const Plan& p, const Work& w, const __nv_bfloat16* K, const __nv_bfloat16* V,
                                        const __nv_bfloat16* dlv_bf16, const float* lse2, const float* delta,
                                        float* dK, float* dV, float* dlq, cudaStream_t st);

// The whole forward pass of a short head in one kernel (small_fused.cu):
// N <= 256, m <= 32, s = 1, with the shared branch, not split. Writes out,
// expert_idx, route and (when not null) Lq, LV [BH][m][64] fp32.
bool small_fused_applies(const Plan& p);
cudaError_t launch_small_fused(const Plan& p, const __nv_bfloat16* Q, const __nv_bfloat16* K, const __nv_bfloat16* V,
                               __nv_bfloat16* out, int32_t* expert_idx, int32_t* route, float* lq_out, float* lv_out,
                               int* status, cudaStream_t st);

// Number of SMs of the current device (cached per device).
int device_sms();

}  // namespace mita
