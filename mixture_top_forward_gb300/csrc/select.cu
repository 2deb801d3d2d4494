// Stage 2, merge: per (head, landmark), combine the scan's per-chunk results.
//
//  * shared-expert value: the chunks' softmax partials (max_c, sum_c, o_c)
//    are merged by rescaling to the common maximum (log-sum-exp merge), giving
//    LV_i = softmax(s_i) V over all N keys;
//  * routed expert: the k largest top-k keys over all chunks' candidate
//    buffers, found by radix select on the 64-bit keys (8 bits per pass,
//    256-bin shared-memory histogram), then written as key indices in
//    ascending order (each selected index placed by counting the selected
//    indices below it).
// Each chunk's buffer holds at least min(chunk length, k) of its best keys,
// so the union always contains the global top k.
//
// Dense top-k (shapes whose sample thresholds would pass too many keys): the
// candidates are the landmark's whole row of logits, written by the scan.
//
// The pilot variant (after a scan of a strided key sample) only finds each
// landmark's k-th largest sample key and raises the landmark's threshold to
// it: k keys of the head reach that value, so the true k-th best does too.
#include "topk.cuh"
#include "warp_select.cuh"

namespace mita {

namespace {

constexpr int ST = 256;         // threads per CTA
constexpr int SEL_CAP = 4608;   // candidates staged in shared memory (36 KB)

template <bool PILOT>
__global__ void __launch_bounds__(ST) select_kernel(int m, int k, int chunks, int cap,
                                                    const float* __restrict__ part,
                                                    const uint64_t* __restrict__ cand,
                                                    const int* __restrict__ ccount, float* __restrict__ lv32,
                                                    __nv_bfloat16* __restrict__ lvbf,
                                                    int32_t* __restrict__ expert_idx, uint64_t* __restrict__ theta,
                                                    const float* __restrict__ dense, int64_t N, int64_t ld,
                                                    int64_t stride, const uint32_t* __restrict__ ridx,
                                                    const float* __restrict__ rval, const int* __restrict__ rcount,
                                                    int rcap, const uint64_t* __restrict__ thr_in,
                                                    float* __restrict__ lse_out, int jspec,
                                                    uint64_t* __restrict__ theta_safe) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    __shared__ unsigned hist[256];
    __shared__ unsigned hist2[256];     // (two-target radix select: the second target's histogram)
    __shared__ int s_dg[2];             // (two-target radix select: each target's digit and keys above it)
    __shared__ unsigned s_ab[2];
    __shared__ int offs[ST + 1];        // chunk offsets into staged[] (chunks <= ST)
    __shared__ float red[ST / 32 + 1];  // block reductions
    __shared__ float fac[ST];           // LV merge: per-chunk rescale factors
    __shared__ float osum[4][D];
    __shared__ uint64_t staged[SEL_CAP];
    __shared__ int sel[MITA_SORT_MAX];
    __shared__ int nsel;
    __shared__ int wcnt[ST / 32];  // ordered take: selected keys per warp in the round
    __shared__ int nst;  // keys staged (records expanded); counts past SEL_CAP too
    __shared__ int s_digit;
    __shared__ unsigned s_above;

    const int i = static_cast<int>(blockIdx.x % static_cast<unsigned>(m));
    const int64_t bh = blockIdx.x / static_cast<unsigned>(m);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const bool small = chunks <= ST;  // per-chunk values fit the shared arrays
    auto part_of = [&](int c) { return part + ((bh * chunks + c) * m + i) * 68; };

    // ---- shared-expert value ------------------------------------------------
    if (!PILOT && part) {
        if (small) {
            // M = max of the chunks' maxima; factors exp(max_c - M); L = sum sum_c f_c
            const float mc = tid < chunks ? part_of(tid)[0] : -INFINITY;
            const float lc = tid < chunks ? part_of(tid)[1] : 0.f;
            float x = mc;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
            if (lane == 0) red[wid] = x;
            __syncthreads();
            float M = red[0];
            for (int w = 1; w < ST / 32; ++w) M = fmaxf(M, red[w]);
            const float f = tid < chunks ? exp2f((mc - M) * kLog2e) : 0.f;
            if (tid < chunks) fac[tid] = f;
            float y = lc * f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
            __syncthreads();
            if (lane == 0) red[wid] = y;
            __syncthreads();
            float L = 0.f;
            for (int w = 0; w < ST / 32; ++w) L += red[w];
            // O_d = sum_c o_c[d] f_c: four threads per column d, chunks q, q+4, ...
            const int dd = tid & (D - 1), q = tid >> 6;
            float acc = 0.f;
            for (int c = q; c < chunks; c += ST / D) acc += part_of(c)[4 + dd] * fac[c];
            osum[q][dd] = acc;
            __syncthreads();
            if (tid < D) {
                const float v = (osum[0][tid] + osum[1][tid] + osum[2][tid] + osum[3][tid]) / L;
                lv32[(bh * m + i) * D + tid] = v;
                if (lse_out && tid == 0) lse_out[bh * m + i] = M + logf(L);
                lvbf[(bh * m + i) * D + tid] = __float2bfloat16_rn(v);
            }
        } else if (tid < D) {
            float M = -INFINITY;
            for (int c = 0; c < chunks; ++c) M = fmaxf(M, part_of(c)[0]);
            float L = 0.f, O = 0.f;
            for (int c = 0; c < chunks; ++c) {
                const float* pp = part_of(c);
                const float f = exp2f((pp[0] - M) * kLog2e);
                L += pp[1] * f;
                O += pp[4 + tid] * f;
            }
            const float v = O / L;
            lv32[(bh * m + i) * D + tid] = v;
            if (lse_out && tid == 0) lse_out[bh * m + i] = M + logf(L);
            lvbf[(bh * m + i) * D + tid] = __float2bfloat16_rn(v);
        }
    }

    // ---- routed expert: k largest keys over all chunk buffers ---------------
    auto buf_of = [&](int c) { return cand + ((bh * chunks + c) * m + i) * static_cast<int64_t>(cap); };
    auto count_of = [&](int c) { return ccount[(bh * chunks + c) * m + i]; };
    // dense top-k: the landmark's whole row of logits, as order keys
    const float* drow = dense ? dense + (bh * m + i) * ld : nullptr;
    // group records (tensor-core scans): each record's logits at or above the
    // landmark's threshold key become keys, as the scan's own key appends
    // would have made them (non-finite logits are masked columns: dropped)
    const uint64_t thr_key = thr_in ? thr_in[bh * m + i] : 0;
    auto recs_of = [&](int c) { return rcap > 0 ? rcount[(bh * chunks + c) * m + i] : 0; };
    // f(j, key) for each column j (0..7, unrolled) of record r of chunk c that becomes a key
    auto rec_keys_at = [&](int c, int r, auto&& f) {
        const int64_t at = ((bh * chunks + c) * m + i) * static_cast<int64_t>(rcap) + r;
        const uint32_t b0 = ridx[at];
        const float4 v0 = reinterpret_cast<const float4*>(rval)[2 * at];
        const float4 v1 = reinterpret_cast<const float4*>(rval)[2 * at + 1];
        const float sc[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (sc[j] >= -3.402823466e38f && sc[j] <= 3.402823466e38f) {
                const uint64_t key = topk_key(sc[j] * 0.125f, static_cast<uint32_t>((b0 + j) * stride));
                if (key >= thr_key) f(j, key);
            }
        }
    };
    auto rec_keys = [&](int c, int r, auto&& f) { rec_keys_at(c, r, [&](int, uint64_t key) { f(key); }); };
    int total = 0;
    if (drow) {
        total = static_cast<int>(N);
    } else if (small) {
        // chunk counts, one per thread, and their exclusive prefix sums
        const int n = tid < chunks ? count_of(tid) : 0;
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncthreads();
        if (lane == 31) red[wid] = __int_as_float(incl);
        __syncthreads();
        int base = 0;
        for (int w = 0; w < wid; ++w) base += __float_as_int(red[w]);
        offs[tid] = base + incl - n;
        if (tid == ST - 1) offs[ST] = base + incl;
        if (tid == 0) nst = 0;
        __syncthreads();
        total = offs[ST];
        // the records' keys go after the plain keys (one warp per chunk, a
        // record per lane; one shared-memory atomic per warp and round
        // reserves the round's slots); the count stays exact past SEL_CAP
        if (rcap > 0) {
            if (tid == 0) nst = total;
            __syncthreads();
            for (int c = wid; c < chunks; c += ST / 32) {
                const int nr = recs_of(c);
                for (int r0 = 0; r0 < nr; r0 += 32) {
                    uint64_t key[8];
                    unsigned acc = 0;
                    if (r0 + lane < nr)
                        rec_keys_at(c, r0 + lane, [&](int j, uint64_t x) {
                            key[j] = x;
                            acc |= 1u << j;
                        });
                    const int mine = __popc(acc);
                    int incl = mine;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += y;
                    }
                    int base = 0;
                    if (lane == 31) base = atomicAdd(&nst, incl);
                    int pos = __shfl_sync(0xffffffffu, base, 31) + incl - mine;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if ((acc >> j) & 1u) {
                            if (pos < SEL_CAP) staged[pos] = key[j];
                            ++pos;
                        }
                }
            }
            __syncthreads();
            total = nst;
        }
    } else {
        for (int c = 0; c < chunks; ++c) total += count_of(c);
        if (rcap > 0) {  // count the records' keys
            int mine = 0;
            for (int c = 0; c < chunks; ++c)
                for (int r = tid; r < recs_of(c); r += ST) rec_keys(c, r, [&](uint64_t) { ++mine; });
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
            __syncthreads();
            if (lane == 0) red[wid] = __int_as_float(mine);
            __syncthreads();
            for (int w = 0; w < ST / 32; ++w) total += __float_as_int(red[w]);
            __syncthreads();
        }
    }

    // all of this landmark's candidates in shared memory when they fit. A
    // dense pilot row only needs its k-th largest score: its scores go in as
    // the upper 32 bits of their keys (index bits zero), twice as many fit,
    // and the k-th largest of those keys is still at or below the true k-th
    // largest key of the head.
    uint32_t* staged32 = reinterpret_cast<uint32_t*>(staged);
    const bool in_smem32 = PILOT && drow && total <= 2 * SEL_CAP;
    const bool in_smem = !in_smem32 && (drow || small) && total <= SEL_CAP;
    if (in_smem32) {
        for (int e = tid; e < total; e += ST)
            staged32[e] = static_cast<uint32_t>(topk_key(drow[e] * 0.125f, 0xFFFFFFFFu) >> 32);
        __syncthreads();
    } else if (in_smem && drow) {
        for (int e = tid; e < total; e += ST) staged[e] = topk_key(drow[e] * 0.125f, static_cast<uint32_t>(e * stride));
        __syncthreads();
    } else if (in_smem) {  // one warp per chunk buffer, so the chunks' loads overlap
        // (the records' keys are already in place after the plain keys)
        for (int c = wid; c < chunks; c += ST / 32) {
            const uint64_t* b = buf_of(c);
            const int o = offs[c], n = offs[c + 1] - o;
            for (int e = lane; e < n; e += 32) staged[o + e] = b[e];
        }
        __syncthreads();
    }
    auto for_each = [&](auto&& f) {
        if (in_smem32) {
            for (int e = tid; e < total; e += ST) f(static_cast<uint64_t>(staged32[e]) << 32);
        } else if (in_smem) {
            for (int e = tid; e < total; e += ST) f(staged[e]);
        } else if (drow) {
            for (int e = tid; e < total; e += ST) f(topk_key(drow[e] * 0.125f, static_cast<uint32_t>(e * stride)));
        } else {
            for (int c = 0; c < chunks; ++c) {
                const uint64_t* b = buf_of(c);
                const int n = count_of(c);
                for (int e = tid; e < n; e += ST) f(b[e]);
                const int nr = recs_of(c);
                for (int r = tid; r < nr; r += ST) rec_keys(c, r, f);
            }
        }
    };

    // Radix select, 8 bits per pass from the top. It stops early once the bin
    // holding the k-th largest key holds exactly the keys still needed: then
    // every key whose leading digits reach the prefix is selected, and the
    // prefix (lower bits zero) separates them from the rest.
    // (each: the key set, as for_each; returns a value with exactly `target`
    // of the keys at or above it)
    auto radix_select = [&](unsigned target, auto&& each) -> uint64_t {
        uint64_t prefix = 0, mask = 0;
        unsigned remaining = target;
        for (int shift = 56; shift >= 0; shift -= 8) {
            hist[tid] = 0;
            __syncthreads();
            each([&](uint64_t x) {
                if ((x & mask) == prefix) atomicAdd(&hist[(x >> shift) & 255u], 1u);
            });
            __syncthreads();
            if (tid < 32) {  // warp 0 finds the digit holding the k-th largest
                const int lane = tid;
                unsigned cc[8], tot = 0;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    cc[t] = hist[255 - 8 * lane - t];
                    tot += cc[t];
                }
                unsigned incl = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const unsigned excl = incl - tot;
                if (excl < remaining && remaining <= incl) {
                    unsigned run = excl;
                    for (int t = 0; t < 8; ++t) {
                        if (run + cc[t] >= remaining) {
                            s_digit = 255 - 8 * lane - t;
                            s_above = run;
                            break;
                        }
                        run += cc[t];
                    }
                }
            }
            __syncthreads();
            remaining -= s_above;
            prefix |= static_cast<uint64_t>(s_digit) << shift;
            mask |= 0xFFull << shift;
            const bool whole_bin = hist[s_digit] == remaining;
            __syncthreads();
            if (whole_bin) break;
        }
        return prefix;
    };
    // The k-th and the j-th largest (j < k) in the same passes: one histogram
    // while both are searching with the same prefix, one each once they
    // differ (or one of them is done); warp 0 finds the k-th's digit, warp 1
    // the j-th's.
    auto radix_select2 = [&](unsigned tk, unsigned tj, auto&& each, uint64_t& out_k, uint64_t& out_j) {
        uint64_t pk = 0, pj = 0, mask = 0;
        unsigned rk = tk, rj = tj;
        bool dk = false, dj = false;
        for (int shift = 56; shift >= 0; shift -= 8) {
            const bool same = pk == pj && !dk && !dj;
            hist[tid] = 0;
            hist2[tid] = 0;
            __syncthreads();
            each([&](uint64_t x) {
                const uint64_t xm = x & mask;
                const unsigned dg = (x >> shift) & 255u;
                if (!dk && xm == pk) atomicAdd(&hist[dg], 1u);
                if (!dj && !same && xm == pj) atomicAdd(&hist2[dg], 1u);
            });
            __syncthreads();
            if (tid < 64) {
                const int t2 = tid >> 5, ln = tid & 31;
                if (t2 == 0 ? !dk : !dj) {
                    const unsigned* h = (t2 == 1 && !same) ? hist2 : hist;
                    const unsigned remaining = t2 == 0 ? rk : rj;
                    unsigned cc[8], tot = 0;
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        cc[t] = h[255 - 8 * ln - t];
                        tot += cc[t];
                    }
                    unsigned incl = tot;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (ln >= o) incl += y;
                    }
                    const unsigned excl = incl - tot;
                    if (excl < remaining && remaining <= incl) {
                        unsigned run = excl;
                        for (int t = 0; t < 8; ++t) {
                            if (run + cc[t] >= remaining) {
                                s_dg[t2] = 255 - 8 * ln - t;
                                s_ab[t2] = run;
                                break;
                            }
                            run += cc[t];
                        }
                    }
                }
            }
            __syncthreads();
            bool wk = dk, wj = dj;
            if (!dk) {
                rk -= s_ab[0];
                pk |= static_cast<uint64_t>(s_dg[0]) << shift;
                wk = hist[s_dg[0]] == rk;  // the whole bin is selected: the prefix separates it
            }
            if (!dj) {
                rj -= s_ab[1];
                pj |= static_cast<uint64_t>(s_dg[1]) << shift;
                wj = (same ? hist : hist2)[s_dg[1]] == rj;
            }
            mask |= 0xFFull << shift;
            __syncthreads();
            dk = wk;
            dj = wj;
            if (dk && dj) break;
        }
        out_k = pk;
        out_j = pj;
    };
    uint64_t kth = 0;  // keep every key >= kth
    uint64_t kj = 0;   // the last speculative pilot: its jspec-th largest key
    bool ranked = false;
    if (total > k || (PILOT && total == k)) {
        if (PILOT && theta_safe && jspec > 0 && jspec < k) {
            radix_select2(static_cast<unsigned>(k), static_cast<unsigned>(jspec), for_each, kth, kj);
            ranked = true;
        } else {
            kth = radix_select(static_cast<unsigned>(k), for_each);
        }
    }
    if (PILOT) {
        // The last pilot of a speculative scan (theta_safe set) has also
        // found the jspec-th largest key (jspec < k, in the same passes): it
        // becomes the threshold, the k-th the fallback.
        if (tid == 0) {
            const uint64_t old = theta[bh * m + i];
            const uint64_t safe = (total >= k && kth > old) ? kth : old;
            const uint64_t spec = ranked && kj > safe ? kj : safe;
            theta[bh * m + i] = spec;
            if (theta_safe) theta_safe[bh * m + i] = safe;
        }
        return;
    }

    int32_t* dst = expert_idx + (bh * m + i) * static_cast<int64_t>(k);
    if (in_smem) {
        // ---- the selected indices, ascending, by an ordered take ----------
        // The staged keys are in ascending index order: the chunks cover the
        // keys in order, each appends its candidates in key order and its
        // compaction keeps their order (a dense row is staged in order).
        // Round by round (ST keys), each selected key goes to the number of
        // selected keys before it. Exactly k keys reach kth (every landmark
        // keeps at least k candidates); were it ever fewer, the rest become
        // key 0, so every index written is in range.
        int base = 0;  // selected in earlier rounds (block-uniform)
        for (int e0 = 0; e0 < total; e0 += ST) {
            const int e = e0 + tid;
            const bool f = e < total && staged[e] >= kth;
            const unsigned bal = __ballot_sync(0xffffffffu, f);
            if (lane == 0) wcnt[wid] = __popc(bal);
            __syncthreads();
            int before = 0, all = 0;
#pragma unroll
            for (int w = 0; w < ST / 32; ++w) {
                const int c = wcnt[w];
                before += w < wid ? c : 0;
                all += c;
            }
            const int pos = base + before + __popc(bal & lanemask_lt());
            if (f && pos < k) dst[pos] = static_cast<int>(topk_key_index(staged[e]));
            base += all;
            __syncthreads();  // (wcnt is rewritten next round)
        }
        for (int t = base + tid; t < k; t += ST) dst[t] = 0;
        return;
    }
    // ---- otherwise: gather the selected indices and sort them ascending -----
    if (tid == 0) nsel = 0;
    __syncthreads();
    for_each([&](uint64_t x) {
        if (x >= kth) sel[atomicAdd(&nsel, 1)] = static_cast<int>(topk_key_index(x));
    });
    __syncthreads();
    // Exactly k keys reach kth (every landmark has at least k candidates). If
    // that were ever not so, the missing entries become key 0, so every index
    // written is in range.
    for (int t = nsel + tid; t < k; t += ST) sel[t] = 0;
    __syncthreads();
    // ascending order: each selected index goes to the place given by the
    // number of selected indices below it (equal ones ordered by position)
    for (int t = tid; t < k; t += ST) {
        const int x = sel[t];
        int r = 0;
        for (int u = 0; u < k; ++u) r += (sel[u] < x || (sel[u] == x && u < t)) ? 1 : 0;
        dst[r] = x;
    }
}

// ---------------------------------------------------------------------------
// Dense rows (short sequences: the dense buffer holds every logit of the
// landmark's row), one warp per landmark, k <= 32 C. Scores become 32-bit
// order keys (larger score first). Each lane keeps its C largest keys while
// the row streams in; theta = the smallest of the lanes' C-th largest is a
// lower bound on the row's k-th largest key, since every lane holds C keys
// at or above it (32 C >= k; a lane with fewer than C keys leaves theta = 0,
// below every key). The keys at or above theta are compacted in index order
// into shared memory; a radix select over them (8-bit digits, per-warp
// histogram) finds the k-th largest key, and a walk in index order takes
// every key above it and, of the keys equal to it, the lowest indices until
// k are taken: the set ranked by (score desc, index asc), written in
// ascending index order. More survivors than kSurv (heavy ties) run the same
// select over the whole row. The warp also merges the landmark's LV partials.
// ---------------------------------------------------------------------------
constexpr int DW = 8;        // warps (landmarks) per CTA
constexpr int kSurv = 512;   // survivors staged per warp
constexpr int kDenseMaxC = 4;

template <int C>
__global__ void __launch_bounds__(DW * 32) dense_row_select_kernel(
    int64_t rows, int m, int k, int chunks, const float* __restrict__ part, float* __restrict__ lv32,
    __nv_bfloat16* __restrict__ lvbf, int32_t* __restrict__ expert_idx, const float* __restrict__ dense, int n,
    int64_t ld, float* __restrict__ lse_out) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    __shared__ uint32_t s_key[DW][kSurv];
    __shared__ int32_t s_idx[DW][kSurv];
    __shared__ unsigned s_hist[DW][256];
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * DW + wid;  // (head, landmark)
    if (row >= rows) return;  // (warp-uniform; no block-wide barrier below)

    // ---- shared-expert value: merge of the chunks' partials ----
    if (part) {
        const int64_t bh = row / m, i = row % m;
        auto part_of = [&](int c) { return part + ((bh * chunks + c) * m + i) * 68; };
        float M = -INFINITY;
        for (int c = 0; c < chunks; ++c) M = fmaxf(M, part_of(c)[0]);
        float L = 0.f, o0 = 0.f, o1 = 0.f;
        for (int c = 0; c < chunks; ++c) {
            const float* pp = part_of(c);
            const float f = exp2f((pp[0] - M) * kLog2e);
            L += pp[1] * f;
            o0 += pp[4 + lane] * f;
            o1 += pp[36 + lane] * f;
        }
        o0 /= L;
        o1 /= L;
        lv32[row * D + lane] = o0;
        lv32[row * D + 32 + lane] = o1;
        lvbf[row * D + lane] = __float2bfloat16_rn(o0);
        lvbf[row * D + 32 + lane] = __float2bfloat16_rn(o1);
        if (lse_out && lane == 0) lse_out[row] = M + logf(L);
    }

    // ---- routed expert: the k best of the row ----
    const float* src = dense + row * ld;  // ld is a multiple of 4: float4 rows
    // The per-lane top C runs on the raw logits: tau = 1/8 is exact and the
    // order key is monotone in the float (with -0 = +0, as a float compare
    // has it), so comparing raw values orders them as their keys do, and
    // only the survivors need their keys.
    float t[C];
#pragma unroll
    for (int c = 0; c < C; ++c) t[c] = -INFINITY;
    // eight 16-byte loads of the row in flight per lane
    for (int g0 = 0; g0 < n; g0 += 8 * 128) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e0 = g0 + 128 * u + 4 * lane;
            v[u] = e0 < n ? __ldg(reinterpret_cast<const float4*>(src + e0))
                          : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float x = f[j];  // (past the row: -inf, below every logit)
#pragma unroll
                for (int c = 0; c < C; ++c) {  // insert into t[0] >= t[1] >= ...
                    const float hi = fmaxf(t[c], x);
                    x = fminf(t[c], x);
                    t[c] = hi;
                }
            }
        }
    }
    // theta: the smallest of the lanes' C-th largest keys, and the raw logit
    // it stands for (-inf when a lane holds fewer than C logits)
    const uint32_t theta = __reduce_min_sync(0xffffffffu, t[C - 1] == -INFINITY ? 0u : score_key32(t[C - 1]));
    float thr_raw = -INFINITY;
    if (theta != 0u) {
        const uint32_t u = theta;
        thr_raw = __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u) * 8.0f;
    }
    // survivors (keys >= theta) in index order; the second read of the row
    // also keeps eight 16-byte loads per lane in flight
    const unsigned below = (1u << lane) - 1u;
    unsigned total = 0;
    for (int g0 = 0; g0 < n; g0 += 8 * 128) {
        float4 vv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e0 = g0 + 128 * u + 4 * lane;
            vv[u] = e0 < n ? __ldg(reinterpret_cast<const float4*>(src + e0)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e0 = g0 + 128 * u + 4 * lane;
            const float f[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
            unsigned bl[4], before = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                bl[j] = __ballot_sync(0xffffffffu, e0 + j < n && f[j] >= thr_raw);
                before += __popc(bl[j] & below);
            }
            unsigned pos = total + before;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if ((bl[j] >> lane) & 1u) {
                    if (pos < kSurv) {
                        s_key[wid][pos] = score_key32(f[j]);
                        s_idx[wid][pos] = e0 + j;
                    }
                    ++pos;
                }
            }
            total += __popc(bl[0]) + __popc(bl[1]) + __popc(bl[2]) + __popc(bl[3]);
        }
    }
    __syncwarp();
    int32_t* dst = expert_idx + row * static_cast<int64_t>(k);
    unsigned remaining;
    if (total <= static_cast<unsigned>(kSurv)) {
        const int cnt = static_cast<int>(total);
        auto get = [&](int e) { return s_key[wid][e]; };
        const uint32_t kth = warp_radix_kth(cnt, static_cast<unsigned>(k), s_hist[wid], get, &remaining);
        warp_take(cnt, kth, remaining, get, [&](int e) { return s_idx[wid][e]; }, [&](int r, int32_t x) { dst[r] = x; });
    } else {
        auto get = [&](int e) { return score_key32(src[e]); };
        const uint32_t kth = warp_radix_kth(n, static_cast<unsigned>(k), s_hist[wid], get, &remaining);
        warp_take(n, kth, remaining, get, [](int e) { return e; }, [&](int r, int32_t x) { dst[r] = x; });
    }
}

}  // namespace

bool dense_row_select_applies(const Plan& p) {
    const ScanLevel& L = p.lev[p.nlev - 1];
    return L.dense && p.s.k <= p.s.N && p.s.k <= 32 * kDenseMaxC;
}

cudaError_t launch_select(const Plan& p, const Work& w, int32_t* expert_idx, cudaStream_t st, float* lse_out) {
    const unsigned grid = static_cast<unsigned>(p.s.BH * p.s.m);
    const ScanLevel& L = p.lev[p.nlev - 1];
    if (dense_row_select_applies(p)) {
        const int64_t rows = p.s.BH * p.s.m;
        const unsigned grid = static_cast<unsigned>((rows + DW - 1) / DW);
        auto go = [&](auto kern) {
            return launch_dep(kern, dim3(grid), dim3(DW * 32), 0, st, rows, p.s.m, p.s.k, L.chunks,
                              p.shared ? w.part : nullptr, w.lv32, w.lvbf, expert_idx, w.dense,
                              static_cast<int>(p.s.N), L.ld, lse_out);
        };
        switch ((p.s.k + 31) / 32) {
            case 1: return go(dense_row_select_kernel<1>);
            case 2: return go(dense_row_select_kernel<2>);
            case 3: return go(dense_row_select_kernel<3>);
            default: return go(dense_row_select_kernel<4>);
        }
    }
    return launch_dep(select_kernel<false>, dim3(grid), dim3(ST), 0, st, p.s.m, p.s.k, L.chunks, L.cap,
                      p.shared ? w.part : nullptr, w.cand, w.ccount, w.lv32, w.lvbf, expert_idx, nullptr,
                      L.dense ? w.dense : nullptr, p.s.N, L.ld, int64_t(1), w.ridx, w.rval, w.rcount, L.rcap,
                      p.nlev > 1 ? w.theta : nullptr, lse_out, 0, nullptr);
}

cudaError_t launch_pilot_select(const Plan& p, const Work& w, int level, cudaStream_t st) {
    const unsigned grid = static_cast<unsigned>(p.s.BH * p.s.m);
    const ScanLevel& L = p.lev[level];
    return launch_dep(select_kernel<true>, dim3(grid), dim3(ST), 0, st, p.s.m, p.s.k, L.chunks, L.cap, nullptr,
                      w.cand, w.ccount, nullptr, nullptr, nullptr, w.theta, L.dense ? w.dense : nullptr, L.S, L.ld,
                      L.stride, w.ridx, w.rval, w.rcount, L.rcap, level > 0 ? w.theta : nullptr, nullptr, p.spec_j,
                      p.spec_j && level == p.nlev - 2 ? w.theta_safe : nullptr);
}

}  // namespace mita
