// C ABI of libmita.so: argument checks, workspace, and the launch sequence
// of the forward pass (declared and documented in include/mita.h).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "mita.h"
#include "mita_internal.cuh"

static_assert(MITA_MAX_M <= MITA_MAX_M_INTERNAL, "routing/grouping tables hold MITA_MAX_M experts");
static_assert(MITA_MAX_K <= MITA_SORT_MAX, "the expert sort holds MITA_MAX_K indices");

namespace mita {

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(MITA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The host entry point pipelines up to kHostGroups head groups once Q, K and V
// together reach kHostPipelineBytes.
constexpr int kHostGroups = 8;
constexpr size_t kHostPipelineBytes = size_t(256) << 20;

int isqrt_exact(int m) {
    int p = 0;
    while ((p + 1) * (p + 1) <= m) ++p;
    return p * p == m ? p : -1;
}

// Validates the arguments common to every entry point and fills `s`.
// Returns MITA_OK, or an error code with the message set.
int check_shape(int B, int H, int N, int d, int gh, int gw, int m, int k, Shape* s, bool* empty) {
    *empty = false;
    if (B < 0 || H < 0) return fail(MITA_ERR_INVALID_ARG, "B=%d, H=%d must be >= 0", B, H);
    if (static_cast<int64_t>(B) * H == 0) {
        *empty = true;
        return MITA_OK;
    }
    if (N < 1) return fail(MITA_ERR_INVALID_ARG, "N=%d must be >= 1", N);
    if (d != D) return fail(MITA_ERR_UNSUPPORTED, "d=%d: only d=64 is built", d);
    if (m < 1 || m > N) return fail(MITA_ERR_INVALID_ARG, "m=%d must be in [1, N=%d]", m, N);
    if (k < 1 || k > N) return fail(MITA_ERR_INVALID_ARG, "k=%d must be in [1, N=%d]", k, N);
    if (m > MITA_MAX_M) return fail(MITA_ERR_UNSUPPORTED, "m=%d exceeds MITA_MAX_M=%d", m, MITA_MAX_M);
    if (k > MITA_MAX_K) return fail(MITA_ERR_UNSUPPORTED, "k=%d exceeds MITA_MAX_K=%d", k, MITA_MAX_K);
    int p = 0;
    if (gh != 0 || gw != 0) {
        if (gh < 1 || gw < 1 || static_cast<int64_t>(gh) * gw != N)
            return fail(MITA_ERR_INVALID_ARG, "grid %dx%d does not tile N=%d", gh, gw, N);
        p = isqrt_exact(m);
        if (p < 0) return fail(MITA_ERR_UNSUPPORTED, "2-D pooling needs a square m, got m=%d", m);
        if (p > gh || p > gw) return fail(MITA_ERR_INVALID_ARG, "landmark grid %dx%d exceeds the token grid", p, p);
    }
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (BH * N > (static_cast<int64_t>(1) << 40))
        return fail(MITA_ERR_UNSUPPORTED, "B*H*N=%lld is too large", static_cast<long long>(BH * N));
    *s = Shape{BH, N, gh, gw, p, m, k, 1};
    return MITA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// Workspace cache, one buffer per (device, stream, purpose).
// ---------------------------------------------------------------------------
struct Slot {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mu;
std::map<std::pair<int, std::pair<uintptr_t, int>>, Slot> g_ws;

// Grows in stream order: the old buffer is released with cudaFreeAsync and
// the new one taken with cudaMallocAsync, both on `st`, so the work already
// queued on `st` finishes with the old buffer before the pool hands its
// memory out again, and the host never waits. The status word travels with
// the workspace: a code still pending in the old buffer is carried over.
int workspace(cudaStream_t st, int purpose, size_t bytes, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Slot& s = g_ws[{dev, {reinterpret_cast<uintptr_t>(st), purpose}}];
    if (s.bytes < bytes) {
        const size_t want = bytes + bytes / 8;  // some headroom for growth
        void* p = nullptr;
        e = cudaMallocAsync(&p, want, st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(MITA_ERR_ALLOC, "cudaMallocAsync(%zu) for the workspace: %s", want, cudaGetErrorString(e));
        }
        e = cudaMemsetAsync(p, 0, want, st);
        // the forward workspace's status word sits at offset 0 of every plan
        if (e == cudaSuccess && s.ptr && purpose == 0)
            e = cudaMemcpyAsync(p, s.ptr, sizeof(int), cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && s.ptr) e = cudaFreeAsync(s.ptr, st);
        if (e != cudaSuccess) {
            cudaFreeAsync(p, st);
            return cuda_fail(e, "workspace growth");
        }
        s.ptr = p;
        s.bytes = want;
    }
    *out = s.ptr;
    return MITA_OK;
}

}  // namespace

int device_sms() {
    static std::mutex mu;
    static std::map<int, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
    return n;
}

cudaError_t launch_route(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route, cudaStream_t st) {
    if (route_tc_supported(p)) return launch_route_tc(p, w, Q, route, st);  // any s
    if (p.s.s_route > 1) return launch_route_multi(p, w, Q, route, st);
    return launch_route_simt(p, w, Q, route, st);
}

cudaError_t launch_expert(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                          const __nv_bfloat16* V, const int32_t* expert_idx, __nv_bfloat16* out, cudaStream_t st) {
    // tensor cores wherever the kernel applies, also for experts with few
    // queries (the 128-row tiles run part-empty; still several times faster
    // than the CUDA-core kernel, measured on the ViT shapes)
    if (expert_tc_supported(p)) return launch_expert_tc(p, w, Q, K, V, expert_idx, out, st);
    return launch_expert_simt(p, w, Q, K, V, expert_idx, out, st);
}

namespace {

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// Chunking and candidate capacity of one scan level. prevS = samples of the
// pilot whose threshold this level starts from (0: none, every key is kept).
ScanLevel scan_level(const Shape& s, int64_t S, int64_t stride, int64_t prevS, int64_t min_chunk, int sms) {
    ScanLevel L{};
    L.S = S;
    L.stride = stride;
    int64_t chunks = std::max<int64_t>(1, cdiv(sms, s.BH));  // about one wave of CTAs
    chunks = std::min(chunks, cdiv(S, min_chunk));
    if (prevS == 0) chunks = std::max(chunks, cdiv(S, 2048));  // bound what an unfiltered chunk keeps
    L.chunk_len = round_up(cdiv(S, chunks), 128);
    L.chunks = static_cast<int>(cdiv(S, L.chunk_len));
    // A chunk holds at most min(chunk_len, S) keys: with that capacity it never
    // compacts. A filtered level expects ~k * chunk_len / prevS survivors per
    // landmark; give it 1.5x that (compaction handles the rest, and needs
    // room for k plus one 128-key tile).
    const int64_t room = round_up(std::min(L.chunk_len, S), 32);
    int64_t cap = room;
    // group records (pilot scans) overflow into the key buffer, so they need
    // room for the expected groups only: each holds at least one survivor
    int64_t rcap = cdiv(room, 8);
    if (prevS > 0) {
        const int64_t expect = cdiv(static_cast<int64_t>(s.k) * L.chunk_len, prevS);
        cap = std::max<int64_t>(round_up(expect + expect / 2 + 64, 32), s.k + 128);
        cap = std::min(cap, room);
        rcap = std::min(round_up(expect + expect / 2 + 64, 32), cap);
    }
    L.cap = static_cast<int>(cap);
    L.rcap = static_cast<int>(rcap);  // (kept only for the tensor-core pilot levels: make_plan)
    return L;
}

}  // namespace

bool make_plan(const Shape& s, Plan* p, bool shared, bool split) {
    Plan P{};
    P.s = s;
    P.shared = shared;
    const int sms = device_sms();
    P.scan_tc = s.m <= 256;
    if (P.scan_tc) {
        // Pilots: strided samples, the first of max(2k, min(N/8, 8k)) keys,
        // then up to 16x larger while within N/32; each starts from the
        // previous level's threshold. The main scan starts from the last
        // level's speculative key (below), which keeps about 2k + 8 N / S
        // candidates per landmark and head: 2k + 256 after N/32 samples,
        // against 2k + 64 after N/8, for a quarter of the last level's cost
        // (at 1M: levels of 8192 and 32768 samples instead of three).
        int64_t prevS = 0;
        const int64_t K8 = 8LL * s.k;
        int64_t t = std::max<int64_t>(2LL * s.k, std::min<int64_t>(s.N / 8, K8));
        if (8 * t <= s.N) {
            // The first level has no threshold. When a sample up to 4x larger
            // (within N/16: as the last level it is the speculative threshold's
            // sample, see above) still fits below N/8 and its logits in 1 GB,
            // it writes every logit of that sample and its select ranks whole
            // rows (dense): appending each sampled key as a candidate costs
            // more, and the larger sample makes the next level's threshold
            // tighter.
            const int64_t t0 = std::min<int64_t>(4 * t, s.N / 16);
            const bool dense0 = t0 >= t && t0 <= s.N / 8 && s.BH * s.m * round_up(t0, 4) * 4 <= (1LL << 30);
            while (P.nlev < 3) {
                const int64_t ts = (P.nlev == 0 && dense0) ? t0 : t;
                const int64_t stride = s.N / ts;
                const int64_t S = cdiv(s.N, stride);
                // the unfiltered first level keeps every sampled key: small chunks spread it over the SMs
                ScanLevel L = scan_level(s, S, stride, prevS, prevS == 0 ? 128 : 512, sms);
                if (P.nlev == 0 && dense0) {
                    L.dense = true;
                    L.ld = round_up(S, 4);
                    L.cap = 0;
                }
                P.lev[P.nlev++] = L;
                prevS = S;
                const int64_t next = std::min<int64_t>(16 * t, s.N / 32);
                if (next <= S) break;
                t = next;
            }
        }
        // Dense top-k when the last sample could only pass more than one key in
        // 16 to the main scan (or there is no sample at all) and the logit rows
        // stay small: appending that many candidates one by one costs more than
        // writing every logit and ranking whole rows.
        const int64_t dense_bytes = s.BH * s.m * round_up(s.N, 4) * 4;
        if ((prevS == 0 || 16LL * s.k > prevS) && s.N <= 65536 && dense_bytes <= (1LL << 30)) {
            P.dense = true;
            P.dense_ld = round_up(s.N, 4);
            P.nlev = 0;
            prevS = 1;  // chunking as for a filtered scan; no candidate buffers
        }
        P.lev[P.nlev++] = scan_level(s, s.N, 1, prevS, 512, sms);
        if (P.dense) {
            P.lev[0].cap = 0;
            P.lev[0].dense = true;
            P.lev[0].ld = P.dense_ld;
        }
        // The last pilot's k-th best sample key is a safe main-scan threshold
        // but a loose one: with a sample of S of the N keys, about k S / N
        // sample keys are among the head's k best, so about k N / S keys pass
        // it. Its j-th best with j = 2 k S / N + 8 keeps about 2k + 8 N / S
        // and still lies below the head's k-th best unless the sample holds
        // j of the head's best k (the main scan's candidate counts tell; a
        // head where that happened is scanned again from the k-th).
        if (P.nlev > 1) {
            const int64_t j = cdiv(2 * static_cast<int64_t>(s.k) * P.lev[P.nlev - 2].S, s.N) + 8;
            if (j < s.k) P.spec_j = static_cast<int>(j);
        }
    } else {
        // CUDA-core scan: 32 landmarks per CTA, ~8 CTAs per SM, >= 1024 keys per chunk
        const int64_t ltiles = cdiv(s.m, 32);
        int64_t chunks = cdiv(static_cast<int64_t>(sms) * 8, s.BH * ltiles);
        chunks = std::max<int64_t>(1, std::min<int64_t>(chunks, s.N / 1024));
        ScanLevel L{};
        L.S = s.N;
        L.stride = 1;
        L.chunk_len = cdiv(s.N, chunks);
        L.chunks = static_cast<int>(cdiv(s.N, L.chunk_len));
        const int64_t room = round_up(L.chunk_len, 32) + 32;
        int64_t cap = round_up(2LL * s.k + 64, 32);
        cap = std::min(cap, room);
        cap = std::max<int64_t>(cap, s.k + 32);
        L.cap = static_cast<int>(cap);
        P.nlev = 1;
        P.lev[0] = L;
    }
    // on request, the shared branch goes with the routing when the
    // tensor-core kernels of both sides apply (and the scan is the
    // tensor-core one)
    P.split = split && P.scan_tc && route_shared_supported(P) && expert_split_fits(P);
    P.rblock = 256;
    P.nrblocks = (s.N + P.rblock - 1) / P.rblock;
    P.qtile = 128;
    P.max_items = (s.N + P.qtile - 1) / P.qtile + s.m;

    const size_t BH = static_cast<size_t>(s.BH), m = static_cast<size_t>(s.m);
    size_t cand = 0, cnts = 0, recs = 0;
    for (int l = 0; l < P.nlev; ++l) {
        // the tensor-core pilot scans append 8-column groups as records first
        // (keys only once a landmark's records are full); the main scan and
        // the CUDA-core scan append keys (records in the main scan measured
        // faster there at 256K and 64K, but the select's expansion of them
        // costs more than that: a net loss at 1M, even at 64K)
        if (!(P.scan_tc && !P.lev[l].dense && l + 1 < P.nlev)) P.lev[l].rcap = 0;
        cand = std::max(cand, BH * P.lev[l].chunks * m * static_cast<size_t>(P.lev[l].cap));
        recs = std::max(recs, BH * P.lev[l].chunks * m * static_cast<size_t>(P.lev[l].rcap));
        cnts = std::max(cnts, BH * P.lev[l].chunks * m);
    }
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    P.off_status = take(sizeof(int));
    P.off_lq32 = take(BH * m * D * sizeof(float));
    P.off_lqhi = take(BH * m * D * 2);
    P.off_lqlo = take(BH * m * D * 2);
    P.off_lv32 = take(BH * m * D * sizeof(float));
    P.off_lvbf = take(BH * m * D * 2);
    P.off_part = take(BH * P.lev[P.nlev - 1].chunks * m * 68 * sizeof(float));
    P.off_cand = take(cand * sizeof(uint64_t));
    P.off_ccount = take(cnts * sizeof(int));
    P.off_theta = take(BH * m * sizeof(uint64_t));
    const size_t sr = static_cast<size_t>(s.s_route);  // one grouping plane per rank of the routes
    P.off_counts = take(sr * BH * m * sizeof(int));
    P.off_expoff = take(BH * (m + 1) * sizeof(int));
    P.off_cursor = take(BH * m * sizeof(int));
    P.off_perm = take(sr * BH * static_cast<size_t>(s.N) * sizeof(int));
    P.off_items = take(sr * BH * static_cast<size_t>(P.max_items) * sizeof(int4));
    P.off_nitems = take(sr * sizeof(int));
    size_t dense_floats = 0;  // the largest dense level's logits
    for (int l = 0; l < P.nlev; ++l)
        if (P.lev[l].dense) dense_floats = std::max(dense_floats, BH * m * static_cast<size_t>(P.lev[l].ld));
    P.off_dense = take(dense_floats * sizeof(float));
    P.off_ridx = take(recs * sizeof(uint32_t));
    P.off_rval = take(recs * 8 * sizeof(float));
    P.off_rcount = take(recs ? cnts * sizeof(int) : 0);
    P.off_state = take(expert_multi_state_bytes(P));
    // s > 1: tensor-core passes where the one-expert kernel applies (same
    // conditions as launch_expert) and the overlap table stays below 1 GB
    P.multi_tc = s.s_route > 1 && expert_tc_supported(P) && s.m <= 256 &&
                 overlap_bytes(s) <= (size_t(1) << 30) && pass_mask_bytes(s) <= (size_t(4) << 30);
    P.off_ovl = take(P.multi_tc ? overlap_bytes(s) : 0);
    P.off_mask = take(P.multi_tc ? pass_mask_bytes(s) : 0);
    P.off_osh = take(P.split ? BH * static_cast<size_t>(s.N) * D * 2 : 0);
    P.off_lse = take(P.split ? BH * static_cast<size_t>(s.N) * sizeof(float) : 0);
    P.off_theta_safe = take(P.spec_j ? BH * m * sizeof(uint64_t) : 0);
    P.off_hflag = take(P.spec_j ? BH * sizeof(int) : 0);
    P.total = off;
    if (P.max_items * s.BH > 0x7FFFFFFFLL || s.BH * P.nrblocks > 0x7FFFFFFFLL) return false;
    for (int l = 0; l < P.nlev; ++l)
        if (s.BH * P.lev[l].chunks * 32 > 0x7FFFFFFFLL) return false;
    *p = P;
    return true;
}

Work carve(const Plan& p, void* base) {
    char* b = static_cast<char*>(base);
    Work w;
    w.status = reinterpret_cast<int*>(b + p.off_status);
    w.lq32 = reinterpret_cast<float*>(b + p.off_lq32);
    w.lqhi = reinterpret_cast<__nv_bfloat16*>(b + p.off_lqhi);
    w.lqlo = reinterpret_cast<__nv_bfloat16*>(b + p.off_lqlo);
    w.lv32 = reinterpret_cast<float*>(b + p.off_lv32);
    w.lvbf = reinterpret_cast<__nv_bfloat16*>(b + p.off_lvbf);
    w.part = reinterpret_cast<float*>(b + p.off_part);
    w.cand = reinterpret_cast<uint64_t*>(b + p.off_cand);
    w.ccount = reinterpret_cast<int*>(b + p.off_ccount);
    w.ridx = reinterpret_cast<uint32_t*>(b + p.off_ridx);
    w.rval = reinterpret_cast<float*>(b + p.off_rval);
    w.rcount = reinterpret_cast<int*>(b + p.off_rcount);
    w.theta = reinterpret_cast<uint64_t*>(b + p.off_theta);
    w.theta_safe = reinterpret_cast<uint64_t*>(b + p.off_theta_safe);
    w.hflag = reinterpret_cast<int*>(b + p.off_hflag);
    w.counts = reinterpret_cast<int*>(b + p.off_counts);
    w.expoff = reinterpret_cast<int*>(b + p.off_expoff);
    w.cursor = reinterpret_cast<int*>(b + p.off_cursor);
    w.perm = reinterpret_cast<int*>(b + p.off_perm);
    w.items = reinterpret_cast<int4*>(b + p.off_items);
    w.nitems = reinterpret_cast<int*>(b + p.off_nitems);
    w.state = reinterpret_cast<float*>(b + p.off_state);
    w.ovl = reinterpret_cast<uint64_t*>(b + p.off_ovl);
    w.mask = reinterpret_cast<uint64_t*>(b + p.off_mask);
    w.osh = reinterpret_cast<__nv_bfloat16*>(b + p.off_osh);
    w.lse = reinterpret_cast<float*>(b + p.off_lse);
    bool any_dense = false;
    for (int l = 0; l < p.nlev; ++l) any_dense = any_dense || p.lev[l].dense;
    w.dense = any_dense ? reinterpret_cast<float*>(b + p.off_dense) : nullptr;
    return w;
}

namespace {

// ---------------------------------------------------------------------------
// Stage timing: per host thread, events recorded between stages.
// ---------------------------------------------------------------------------
constexpr int kStages = 7;
const char* const kStageNames[kStages] = {"pool", "pilot", "scan", "select", "route", "group", "expert"};
struct Recorded {
    cudaStream_t stream;
    cudaEvent_t ev[kStages + 1];
    cudaEvent_t side[2];  // the select stage when it ran on the side stream (else unused)
    bool side_on;
    int launches[kStages];
    int first;  // stages before `first` ran no kernel (their events are not recorded)
};
thread_local bool t_profile = false;
thread_local std::vector<Recorded> t_records;
// Events are reused across calls: creating eight per call made the host, not
// the GPU, set the pace of short passes while profiling.
thread_local std::vector<cudaEvent_t> t_free_events;

cudaEvent_t take_event() {
    if (!t_free_events.empty()) {
        cudaEvent_t e = t_free_events.back();
        t_free_events.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    return cudaEventCreate(&e) == cudaSuccess ? e : nullptr;
}

struct StageMarks {
    Recorded rec{};
    bool on = false;
    explicit StageMarks(cudaStream_t st) {
        if (!t_profile) return;
        rec.stream = st;
        rec.side_on = false;
        for (auto& e : rec.ev)
            if (!(e = take_event())) {
                release();
                return;
            }
        for (auto& e : rec.side)
            if (!(e = take_event())) {
                release();
                return;
            }
        on = true;
    }
    void release() {
        for (auto& e : rec.ev)
            if (e) t_free_events.push_back(e);
        for (auto& e : rec.side)
            if (e) t_free_events.push_back(e);
        for (auto& e : rec.ev) e = nullptr;
        for (auto& e : rec.side) e = nullptr;
    }
    void mark(int i) {
        if (on) cudaEventRecord(rec.ev[i], rec.stream);
    }
    // the select stage's own bounds on the side stream
    void side_mark(int i, cudaStream_t ss) {
        if (on) {
            cudaEventRecord(rec.side[i], ss);
            rec.side_on = true;
        }
    }
    void commit(const int* launches, int first = 0) {
        if (on) {
            for (int i = 0; i < kStages; ++i) rec.launches[i] = launches[i];
            rec.first = first;
            t_records.push_back(rec);
        }
        on = false;
    }
    ~StageMarks() {
        if (on) release();
    }
};

// The expert selection needs the scan, routing only Q and the landmarks:
// the selection runs on a side stream (one per device and caller stream,
// forked and joined with events) concurrently with routing and grouping.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::map<std::pair<int, uintptr_t>, SideStream> g_side;

SideStream* side_stream(cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    SideStream& h = g_side[{dev, reinterpret_cast<uintptr_t>(st)}];
    if (!h.s) {
        if (cudaStreamCreateWithFlags(&h.s, cudaStreamNonBlocking) != cudaSuccess) {
            h.s = nullptr;
            return nullptr;
        }
        if (cudaEventCreateWithFlags(&h.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&h.join, cudaEventDisableTiming) != cudaSuccess) {
            if (h.fork) cudaEventDestroy(h.fork);
            if (h.join) cudaEventDestroy(h.join);
            cudaStreamDestroy(h.s);
            h = SideStream{};
            return nullptr;
        }
    }
    return &h;
}

// The four stages on a prepared workspace.
int run_forward(const Plan& P, const Work& W, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                const __nv_bfloat16* V, __nv_bfloat16* out, int32_t* expert_idx, int32_t* route, float* lq_out,
                float* lv_out, cudaStream_t st) {
    cudaError_t e;
    if (small_fused_applies(P)) {  // a short head: every stage in one kernel (timed as the expert stage)
        StageMarks marks(st);
        marks.mark(6);
        if ((e = launch_small_fused(P, Q, K, V, out, expert_idx, route, lq_out, lv_out, W.status, st)) != cudaSuccess)
            return cuda_fail(e, "fused short-head launch");
        marks.mark(7);
        const int launches[kStages] = {0, 0, 0, 0, 0, 0, 1};
        marks.commit(launches, 6);
        return MITA_OK;
    }
    const size_t mrows = static_cast<size_t>(P.s.BH) * P.s.m;
    const int sr = P.s.s_route;
    // (all before the first kernel, so that the kernels that follow each
    // other in the stream can overlap their launches)
    if ((e = cudaMemsetAsync(W.counts, 0, sr * mrows * sizeof(int), st)) != cudaSuccess ||
        (e = cudaMemsetAsync(W.nitems, 0, sr * sizeof(int), st)) != cudaSuccess ||
        (P.scan_tc && P.nlev > 1 && (e = cudaMemsetAsync(W.theta, 0, mrows * sizeof(uint64_t), st)) != cudaSuccess))
        return cuda_fail(e, "cudaMemsetAsync");
    StageMarks marks(st);
    marks.mark(0);
    if ((e = launch_pool(P, W, Q, st)) != cudaSuccess) return cuda_fail(e, "landmark pooling launch");
    marks.mark(1);
    if (P.scan_tc) {
        for (int l = 0; l + 1 < P.nlev; ++l) {
            if ((e = launch_scan_tc(P, W, K, V, l, st)) != cudaSuccess) return cuda_fail(e, "pilot scan launch");
            if ((e = launch_pilot_select(P, W, l, st)) != cudaSuccess) return cuda_fail(e, "pilot select launch");
        }
        marks.mark(2);
        if ((e = launch_scan_tc(P, W, K, V, P.nlev - 1, st)) != cudaSuccess)
            return cuda_fail(e, "landmark scan launch");
        if (P.spec_j && (e = launch_scan_verify(P, W, K, st)) != cudaSuccess)
            return cuda_fail(e, "landmark scan check launch");
    } else {
        marks.mark(2);
        if ((e = launch_scan(P, W, K, V, st)) != cudaSuccess) return cuda_fail(e, "landmark scan launch");
    }
    marks.mark(3);
    // (the split form's routing reads LV from the selection: in order)
    SideStream* ss = P.split ? nullptr : side_stream(st);
    if (ss) {
        if ((e = cudaEventRecord(ss->fork, st)) != cudaSuccess || (e = cudaStreamWaitEvent(ss->s, ss->fork, 0)) != cudaSuccess)
            return cuda_fail(e, "side stream fork");
        marks.side_mark(0, ss->s);
        if ((e = launch_select(P, W, expert_idx, ss->s)) != cudaSuccess)
            return cuda_fail(e, "expert selection launch");
        marks.side_mark(1, ss->s);
        if ((e = cudaEventRecord(ss->join, ss->s)) != cudaSuccess) return cuda_fail(e, "side stream join");
    } else if ((e = launch_select(P, W, expert_idx, st)) != cudaSuccess) {
        return cuda_fail(e, "expert selection launch");
    }
    marks.mark(4);
    e = P.split ? launch_route_shared(P, W, Q, route, st) : launch_route(P, W, Q, route, st);
    if (e != cudaSuccess) return cuda_fail(e, "routing launch");
    marks.mark(5);
    for (int j = 0; j < sr; ++j)
        if ((e = launch_group(P, W, route, j, st)) != cudaSuccess) return cuda_fail(e, "grouping launch");
    // the expert sets are read from here on
    if (ss && (e = cudaStreamWaitEvent(st, ss->join, 0)) != cudaSuccess) return cuda_fail(e, "side stream join");
    if (P.multi_tc && (e = launch_overlap(P, W, expert_idx, route, st)) != cudaSuccess)
        return cuda_fail(e, "expert overlap launch");
    marks.mark(6);
    if (sr == 1) {
        if ((e = launch_expert(P, W, Q, K, V, expert_idx, out, st)) != cudaSuccess)
            return cuda_fail(e, "expert attention launch");
    } else {  // one pass per rank of the routes
        for (int j = 0; j < sr; ++j) {
            e = P.multi_tc ? launch_expert_tc(P, W, Q, K, V, expert_idx, out, st, route, j)
                           : launch_expert_multi(P, W, Q, K, V, expert_idx, route, j, out, st);
            if (e != cudaSuccess) return cuda_fail(e, "expert attention launch");
        }
    }
    marks.mark(7);
    const int launches[kStages] = {1, P.scan_tc ? 2 * (P.nlev - 1) : 0, 1 + (P.spec_j ? 2 : 0), 1, 1,
                                   2 * sr + (P.multi_tc ? sr : 0), sr};
    marks.commit(launches);
    if (lq_out && (e = cudaMemcpyAsync(lq_out, W.lq32, mrows * D * sizeof(float), cudaMemcpyDeviceToDevice, st)) !=
                      cudaSuccess)
        return cuda_fail(e, "copy of Lq");
    if (lv_out && (e = cudaMemcpyAsync(lv_out, W.lv32, mrows * D * sizeof(float), cudaMemcpyDeviceToDevice, st)) !=
                      cudaSuccess)
        return cuda_fail(e, "copy of LV");
    return MITA_OK;
}

}  // namespace
}  // namespace mita

using namespace mita;

namespace {

// The device-buffer entry points: MiTA (shared = true) or its routing-only
// ablation.
int forward_device(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h, int grid_w,
                   int m, int k, void* out, int32_t* expert_idx, int32_t* route, float* lq, float* lv, void* stream,
                   bool shared, int s_route = 1, bool split = false) {
    g_err[0] = 0;
    Shape s;
    bool empty;
    int rc = check_shape(B, H, N, d, grid_h, grid_w, m, k, &s, &empty);
    if (rc != MITA_OK || empty) return rc;
    if (s_route < 1 || s_route > m || s_route > MITA_MAX_S)
        return fail(MITA_ERR_INVALID_ARG, "s=%d must be in [1, min(m=%d, MITA_MAX_S=%d)]", s_route, m, MITA_MAX_S);
    s.s_route = s_route;
    if (!Q || !K || !V || !out || !expert_idx || !route)
        return fail(MITA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out))
        return fail(MITA_ERR_INVALID_ARG, "Q, K, V and out must be 16-byte aligned");
    Plan P;
    if (!make_plan(s, &P, shared, split)) return fail(MITA_ERR_UNSUPPORTED, "problem too large for the launch grids");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* base = nullptr;
    if ((rc = workspace(st, 0, P.total, &base)) != MITA_OK) return rc;
    Work W = carve(P, base);
    return run_forward(P, W, static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
                       static_cast<const __nv_bfloat16*>(V), static_cast<__nv_bfloat16*>(out), expert_idx, route, lq,
                       lv, st);
}

}  // namespace

extern "C" int mita_forward_aux(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h,
                                int grid_w, int m, int k, void* out, int32_t* expert_idx, int32_t* route, float* lq,
                                float* lv, void* stream) {
    return forward_device(Q, K, V, B, H, N, d, grid_h, grid_w, m, k, out, expert_idx, route, lq, lv, stream, true);
}

extern "C" int mita_forward_routed(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h,
                                   int grid_w, int m, int k, void* out, int32_t* expert_idx, int32_t* route,
                                   void* stream) {
    return forward_device(Q, K, V, B, H, N, d, grid_h, grid_w, m, k, out, expert_idx, route, nullptr, nullptr, stream,
                          false);
}

extern "C" int mita_forward_split(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h,
                                  int grid_w, int m, int k, void* out, int32_t* expert_idx, int32_t* route,
                                  void* stream) {
    return forward_device(Q, K, V, B, H, N, d, grid_h, grid_w, m, k, out, expert_idx, route, nullptr, nullptr, stream,
                          true, 1, true);
}

extern "C" int mita_forward_multi(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h,
                                  int grid_w, int m, int k, int s, void* out, int32_t* expert_idx, int32_t* route,
                                  void* stream) {
    return forward_device(Q, K, V, B, H, N, d, grid_h, grid_w, m, k, out, expert_idx, route, nullptr, nullptr, stream,
                          true, s);
}

extern "C" int mita_backward(const void* Q, const void* K, const void* V, const void* dO, int B, int H, int N, int d,
                             int grid_h, int grid_w, int m, int k, const int32_t* expert_idx, const int32_t* route,
                             float* dQ, float* dK, float* dV, void* stream) {
    g_err[0] = 0;
    Shape s;
    bool empty;
    int rc = check_shape(B, H, N, d, grid_h, grid_w, m, k, &s, &empty);
    if (rc != MITA_OK || empty) return rc;
    if (!Q || !K || !V || !dO || !expert_idx || !route || !dQ || !dK || !dV)
        return fail(MITA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dO) || !aligned16(dQ) || !aligned16(dK) ||
        !aligned16(dV))
        return fail(MITA_ERR_INVALID_ARG, "Q, K, V, dO, dQ, dK and dV must be 16-byte aligned");
    Plan P;
    if (!make_plan(s, &P)) return fail(MITA_ERR_UNSUPPORTED, "problem too large for the launch grids");
    // the key-side kernel runs one CTA per 128 keys of every head (the
    // landmark-side grids are no larger)
    if (s.BH * ((s.N + 127) / 128) > 0x7FFFFFFFLL)
        return fail(MITA_ERR_UNSUPPORTED, "problem too large for the backward launch grids");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* base = nullptr;
    if ((rc = workspace(st, 0, P.total, &base)) != MITA_OK) return rc;
    Work W = carve(P, base);
    const BwdLayout L = backward_layout(P);
    void* bbase = nullptr;
    if ((rc = workspace(st, 2, L.total, &bbase)) != MITA_OK) return rc;
    const cudaError_t e =
        launch_backward(P, W, L, bbase, static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
                        static_cast<const __nv_bfloat16*>(V), static_cast<const __nv_bfloat16*>(dO), expert_idx,
                        route, dQ, dK, dV, st);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return MITA_OK;
}

extern "C" int mita_forward(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h,
                            int grid_w, int m, int k, void* out, int32_t* expert_idx, int32_t* route, void* stream) {
    return mita_forward_aux(Q, K, V, B, H, N, d, grid_h, grid_w, m, k, out, expert_idx, route, nullptr, nullptr,
                            stream);
}

namespace {

// Copy streams of the host entry point, one pair per (device, caller stream),
// with their events; created on first use and kept (guarded by g_ws_mu).
struct HostStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t ready[kHostGroups] = {}, done[kHostGroups] = {};
};
std::map<std::pair<int, uintptr_t>, HostStreams> g_hs;

int host_streams(cudaStream_t st, HostStreams** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_ws_mu);
    HostStreams& h = g_hs[{dev, reinterpret_cast<uintptr_t>(st)}];
    if (!h.in) {
        if ((e = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "copy stream creation");
        for (int g = 0; g < kHostGroups; ++g)
            if ((e = cudaEventCreateWithFlags(&h.ready[g], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&h.done[g], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e, "copy event creation");
    }
    *out = &h;
    return MITA_OK;
}

}  // namespace

// Pipelined by groups of heads (the heads are independent problems): group
// g's inputs are copied in on one stream while group g-1 runs on the
// caller's stream and group g-2's results are copied out on a third, so the
// forward pass and the outgoing copies hide under the incoming copies.
extern "C" int mita_forward_host(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int B, int H, int N, int d,
                                 int grid_h, int grid_w, int m, int k, uint16_t* out, int32_t* expert_idx,
                                 int32_t* route, void* stream) {
    g_err[0] = 0;
    Shape s;
    bool empty;
    int rc = check_shape(B, H, N, d, grid_h, grid_w, m, k, &s, &empty);
    if (rc != MITA_OK || empty) return rc;
    if (!Q || !K || !V || !out || !expert_idx || !route)
        return fail(MITA_ERR_INVALID_ARG, "a required pointer is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t head_tok = static_cast<size_t>(s.N) * D * 2;  // bytes of one head's Q (K, V, out)
    const size_t head_e = static_cast<size_t>(s.m) * s.k * sizeof(int32_t);
    const size_t head_r = static_cast<size_t>(s.N) * sizeof(int32_t);
    const size_t tok = static_cast<size_t>(s.BH) * head_tok;
    const size_t eb = static_cast<size_t>(s.BH) * head_e;
    const size_t rb = static_cast<size_t>(s.BH) * head_r;
    size_t off = 0;
    const size_t oq = off; off += align256(tok);
    const size_t ok_ = off; off += align256(tok);
    const size_t ov = off; off += align256(tok);
    const size_t oo = off; off += align256(tok);
    const size_t oe = off; off += align256(eb);
    const size_t orr = off; off += align256(rb);
    void* stage = nullptr;
    if ((rc = workspace(st, 1, off, &stage)) != MITA_OK) return rc;
    char* sb = static_cast<char*>(stage);
    HostStreams* hs = nullptr;
    if ((rc = host_streams(st, &hs)) != MITA_OK) return rc;
    // groups: one per head up to kHostGroups, when the inputs are large
    // enough for the overlap to outweigh the extra launches
    int64_t groups = 3 * tok >= kHostPipelineBytes ? std::min<int64_t>(s.BH, kHostGroups) : 1;
    const int64_t per = cdiv(s.BH, groups);
    groups = cdiv(s.BH, per);
    cudaError_t e = cudaEventRecord(hs->start, st);  // after the caller's earlier work on `stream`
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hs->in, hs->start, 0);
    for (int64_t g = 0; g < groups && e == cudaSuccess && rc == MITA_OK; ++g) {
        const int64_t h0 = g * per, nh = std::min<int64_t>(per, s.BH - h0);
        const size_t t0 = h0 * head_tok, tn = nh * head_tok;
        const uint16_t* src[3] = {Q, K, V};
        const size_t dst[3] = {oq, ok_, ov};
        for (int i = 0; i < 3 && e == cudaSuccess; ++i)
            e = cudaMemcpyAsync(sb + dst[i] + t0, reinterpret_cast<const char*>(src[i]) + t0, tn,
                                cudaMemcpyHostToDevice, hs->in);
        if (e == cudaSuccess) e = cudaEventRecord(hs->ready[g], hs->in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hs->ready[g], 0);
        if (e != cudaSuccess) break;
        rc = mita_forward_aux(sb + oq + t0, sb + ok_ + t0, sb + ov + t0, 1, static_cast<int>(nh), N, d, grid_h,
                              grid_w, m, k, sb + oo + t0, reinterpret_cast<int32_t*>(sb + oe + h0 * head_e),
                              reinterpret_cast<int32_t*>(sb + orr + h0 * head_r), nullptr, nullptr, stream);
        if (rc != MITA_OK) break;
        e = cudaEventRecord(hs->done[g], st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hs->out, hs->done[g], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(reinterpret_cast<char*>(out) + t0, sb + oo + t0, tn, cudaMemcpyDeviceToHost, hs->out);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(reinterpret_cast<char*>(expert_idx) + h0 * head_e, sb + oe + h0 * head_e, nh * head_e,
                                cudaMemcpyDeviceToHost, hs->out);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(reinterpret_cast<char*>(route) + h0 * head_r, sb + orr + h0 * head_r, nh * head_r,
                                cudaMemcpyDeviceToHost, hs->out);
    }
    // every copy touching the caller's host buffers is finished before returning, error or not
    const cudaError_t e_in = cudaStreamSynchronize(hs->in);
    const cudaError_t e_st = cudaStreamSynchronize(st);
    const cudaError_t e_out = cudaStreamSynchronize(hs->out);
    if (rc != MITA_OK) return rc;
    if (e != cudaSuccess) return cuda_fail(e, "host copy pipeline");
    if (e_in != cudaSuccess) return cuda_fail(e_in, "host-to-device copies");
    if (e_st != cudaSuccess) return cuda_fail(e_st, "cudaStreamSynchronize");
    if (e_out != cudaSuccess) return cuda_fail(e_out, "device-to-host copies");
    return MITA_OK;
}

extern "C" size_t mita_workspace_bytes(int B, int H, int N, int d, int grid_h, int grid_w, int m, int k) {
    Shape s;
    bool empty;
    char saved[sizeof g_err];
    memcpy(saved, g_err, sizeof g_err);
    const int rc = check_shape(B, H, N, d, grid_h, grid_w, m, k, &s, &empty);
    memcpy(g_err, saved, sizeof g_err);
    if (rc != MITA_OK || empty) return 0;
    Plan P;
    if (!make_plan(s, &P)) return 0;
    return P.total;
}

extern "C" int mita_plan_info(int B, int H, int N, int d, int grid_h, int grid_w, int m, int k, int64_t* info,
                              int cap) {
    Shape s;
    bool empty;
    char saved[sizeof g_err];
    memcpy(saved, g_err, sizeof g_err);
    const int rc = check_shape(B, H, N, d, grid_h, grid_w, m, k, &s, &empty);
    memcpy(g_err, saved, sizeof g_err);
    if (rc != MITA_OK || empty) return 0;
    Plan P;
    if (!make_plan(s, &P)) return 0;
    int64_t v[3 + 3 * 4];
    int n = 0;
    v[n++] = P.nlev;
    v[n++] = P.dense ? 1 : 0;
    v[n++] = P.spec_j;
    for (int l = 0; l < P.nlev; ++l) {
        v[n++] = P.lev[l].S;
        v[n++] = P.lev[l].stride;
        v[n++] = P.lev[l].dense ? 1 : 0;
    }
    for (int i = 0; i < n && i < cap && info; ++i) info[i] = v[i];
    return n;
}

static int* noalloc_status(int dev);

extern "C" int mita_sync_status(void* stream) {
    g_err[0] = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int status = MITA_OK;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto& kv : g_ws) {
        if (kv.first.first != dev || kv.first.second.second != 0 || !kv.second.ptr) continue;
        if (reinterpret_cast<cudaStream_t>(kv.first.second.first) != st) continue;
        int word = 0;
        if ((e = cudaMemcpy(&word, kv.second.ptr, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
            return cuda_fail(e, "status read");
        if (word != 0) {
            status = word;
            const int zero = 0;
            cudaMemcpy(kv.second.ptr, &zero, sizeof(int), cudaMemcpyHostToDevice);
        }
    }
    // the no-allocation entry point's scratch (shared by every stream of the device)
    if (int* nw = noalloc_status(dev)) {
        int word = 0;
        if ((e = cudaMemcpy(&word, nw, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
            return cuda_fail(e, "status read");
        if (word != 0) {
            if (status == MITA_OK || word == MITA_ERR_TIMEOUT) status = word;
            const int zero = 0;
            cudaMemcpy(nw, &zero, sizeof(int), cudaMemcpyHostToDevice);
        }
    }
    if (status != MITA_OK)
        return fail(status, "%s (status %d)",
                    status == MITA_ERR_TIMEOUT ? "a bounded device-side wait gave up"
                                               : "a device-side check found an index out of range",
                    status);
    return MITA_OK;
}

extern "C" int mita_selftest_wait(int64_t limit_us, void* stream) {
    g_err[0] = 0;
    if (limit_us < 1 || limit_us > 2000000)
        return fail(MITA_ERR_INVALID_ARG, "limit_us=%lld must be in [1, 2000000]", static_cast<long long>(limit_us));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* base = nullptr;
    int rc = workspace(st, 0, 256, &base);  // the status word at offset 0 (any plan's)
    if (rc != MITA_OK) return rc;
    const cudaError_t e = launch_wait_selftest(static_cast<int*>(base), static_cast<uint64_t>(limit_us) * 1000u, st);
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return MITA_OK;
}

extern "C" int mita_profile_enable(int on) {
    t_profile = on != 0;
    return MITA_OK;
}

extern "C" int mita_profile_read(double* stage_ms, int64_t* stage_launches, int max_stages, void* stream) {
    g_err[0] = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    const int n = std::min(max_stages, kStages);
    std::vector<Recorded> keep;
    int rc = MITA_OK;
    for (auto& r : t_records) {
        if (r.stream != st) {
            keep.push_back(r);
            continue;
        }
        for (int i = 0; i < n; ++i) {
            float ms = 0.f;
            // (the select stage on the side stream: its own events; it overlaps routing)
            const bool sel_side = r.side_on && i == 3;
            cudaEvent_t e0 = sel_side ? r.side[0] : r.ev[i], e1 = sel_side ? r.side[1] : r.ev[i + 1];
            if (i >= r.first && rc == MITA_OK && (e = cudaEventElapsedTime(&ms, e0, e1)) != cudaSuccess)
                rc = cuda_fail(e, "cudaEventElapsedTime");
            if (stage_ms) stage_ms[i] += ms;
            if (stage_launches) stage_launches[i] += r.launches[i];
        }
        for (auto& ev : r.ev) t_free_events.push_back(ev);
        for (auto& ev : r.side) t_free_events.push_back(ev);
    }
    t_records.swap(keep);
    return rc == MITA_OK ? kStages : rc;
}

extern "C" const char* mita_stage_name(int i) { return (i >= 0 && i < kStages) ? kStageNames[i] : nullptr; }

extern "C" const char* mita_last_error(void) { return g_err; }

extern "C" void mita_release_workspace(void) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : g_ws) {
        if (!kv.second.ptr) continue;
        cudaSetDevice(kv.first.first);
        cudaDeviceSynchronize();
        // stream-ordered memory: freed on the legacy stream (the caller's may be
        // gone) once the device is idle
        cudaFreeAsync(kv.second.ptr, nullptr);
        cudaDeviceSynchronize();
        kv.second.ptr = nullptr;
        kv.second.bytes = 0;
    }
    g_ws.clear();
    for (auto& kv : g_hs) {
        HostStreams& h = kv.second;
        cudaSetDevice(kv.first.first);
        if (h.in) cudaStreamSynchronize(h.in);
        if (h.out) cudaStreamSynchronize(h.out);
        for (int g = 0; g < kHostGroups; ++g) {
            if (h.ready[g]) cudaEventDestroy(h.ready[g]);
            if (h.done[g]) cudaEventDestroy(h.done[g]);
        }
        if (h.start) cudaEventDestroy(h.start);
        if (h.in) cudaStreamDestroy(h.in);
        if (h.out) cudaStreamDestroy(h.out);
    }
    g_hs.clear();
    for (auto& kv : g_side) {
        SideStream& h = kv.second;
        cudaSetDevice(kv.first.first);
        if (h.s) cudaStreamSynchronize(h.s);
        if (h.fork) cudaEventDestroy(h.fork);
        if (h.join) cudaEventDestroy(h.join);
        if (h.s) cudaStreamDestroy(h.s);
    }
    g_side.clear();
    cudaSetDevice(cur);
}

// ---------------------------------------------------------------------------
// Forward pass without allocation (see mita_forward_noalloc in mita.h).
// Its scratch is this file-scope device array: the CUDA runtime reserves it
// on every device that loads the library's module, until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[MITA_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
std::map<int, void*> g_noalloc_addr;  // device -> device address of g_noalloc_scratch

// Device address of the static scratch on the current device. In host code
// the array's name is only a host-side stand-in, so the address is asked
// from the runtime once per device, with that device current; the same
// set-up clears the array's status word (offset 0 of every plan) on `st`.
int noalloc_scratch(cudaStream_t st, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    auto it = g_noalloc_addr.find(dev);
    if (it == g_noalloc_addr.end()) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return fail(MITA_ERR_CUDA, "cudaGetSymbolAddress of the static scratch on device %d: %s", dev,
                        cudaGetErrorString(e));
        if ((e = cudaMemsetAsync(p, 0, sizeof(int), st)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
        it = g_noalloc_addr.emplace(dev, p).first;
    }
    *out = it->second;
    return MITA_OK;
}

}  // namespace

// The status word of the static scratch of device `dev` (nullptr before the
// first mita_forward_noalloc call there).
static int* noalloc_status(int dev) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    auto it = g_noalloc_addr.find(dev);
    return it == g_noalloc_addr.end() ? nullptr : static_cast<int*>(it->second);
}

namespace {

}  // namespace

extern "C" int mita_forward_noalloc(const void* Q, const void* K, const void* V, int B, int H, int N, int d,
                                    int grid_h, int grid_w, int m, int k, void* out, int32_t* expert_idx,
                                    int32_t* route, void* stream) {
    g_err[0] = 0;
    Shape s;
    bool empty;
    int rc = check_shape(B, H, N, d, grid_h, grid_w, m, k, &s, &empty);
    if (rc != MITA_OK || empty) return rc;
    if (!Q || !K || !V || !out || !expert_idx || !route)
        return fail(MITA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out))
        return fail(MITA_ERR_INVALID_ARG, "Q, K, V and out must be 16-byte aligned");
    Plan P;
    if (!make_plan(s, &P)) return fail(MITA_ERR_UNSUPPORTED, "problem too large for the launch grids");
    if (P.total > static_cast<size_t>(MITA_NOALLOC_SCRATCH_BYTES))
        return fail(MITA_ERR_UNSUPPORTED,
                    "this shape needs %zu bytes of scratch; mita_forward_noalloc has %d (MITA_NOALLOC_SCRATCH_BYTES)",
                    P.total, MITA_NOALLOC_SCRATCH_BYTES);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* base = nullptr;
    if ((rc = noalloc_scratch(st, &base)) != MITA_OK) return rc;
    // The array keeps the previous call's contents: the forward sequence clears
    // what must start at zero (the per-expert counters); the status word keeps
    // a timeout until mita_sync_status reports and clears it.
    Work W = carve(P, base);
    const bool prof = t_profile;  // stage timing would create events: keep it off here
    t_profile = false;
    rc = run_forward(P, W, static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
                     static_cast<const __nv_bfloat16*>(V), static_cast<__nv_bfloat16*>(out), expert_idx, route,
                     nullptr, nullptr, st);
    t_profile = prof;
    return rc;
}
