/*
 * mita.h -- C ABI of libmita.so, a GB300 (sm_103a) implementation of the
 * forward pass of Mixture-of-Top-k Attention (MiTA).
 *
 * The method (described in prose in "NeurIPS 2026 | Mixture-of-Top-k 注意力：
 * 从快权重统一高效注意力…" (shuwu5.cn), section "MiTA：用少量地标查询，同时完成
 * 压缩与专家构造"; the same steps in "NeurIPS'26：注意力也是FFN？…"
 * (pro-axy-igame.com), section "用少量地标查询，同时构造全局概括与细节专家", and in
 * the Figure 3 and Algorithm 1 captions of "And attention is also FFN? …"
 * (en.roboind.com)), per head (b,h), with tau = 1/sqrt(d):
 *   1. landmarks   Lq_i = mean of the query rows in local window i (i < m);
 *   2. scan        s_ij = tau <Lq_i, K_j> over all N keys;
 *                  shared expert value LV_i = sum_j softmax_j(s_i.) V_j;
 *                  routed expert E_i = the k keys with the largest s_ij;
 *   3. routing     e(n) = argmax_i tau <q_n, Lq_i>;
 *   4. attention   out_n = softmax over the m logits tau<q_n, Lq_i> and the k
 *                  logits tau<q_n, K_j> (j in E_e(n)) together, applied to
 *                  the values [LV_1..LV_m ; V_j, j in E_e(n)].
 *
 * Conventions shared by every entry point
 *   Q, K, V, out  bf16, layout [B][H][N][d], contiguous, 16-byte aligned.
 *   d             must be 64 (MITA_ERR_UNSUPPORTED otherwise).
 *   grid_h,grid_w both 0: 1-D landmarks over contiguous windows
 *                 [floor(i N/m), ceil((i+1) N/m)).
 *                 both > 0: 2-D adaptive pooling of a grid_h x grid_w token
 *                 grid (row-major, grid_h*grid_w == N) onto a p x p landmark
 *                 grid, m = p*p (a non-square m is MITA_ERR_UNSUPPORTED);
 *                 landmark (r,c) pools rows [floor(r gh/p), ceil((r+1) gh/p))
 *                 and columns [floor(c gw/p), ceil((c+1) gw/p)).
 *   m, k          1 <= m <= min(N, MITA_MAX_M), 1 <= k <= min(N, MITA_MAX_K).
 *   expert_idx    int32 [B][H][m][k]: E_i in ascending key order. Ties in s
 *                 go to the lower key index.
 *   route         int32 [B][H][N]: e(n) in [0, m). Ties go to the lower
 *                 landmark index.
 *   B*H == 0      is an empty problem: nothing is read or written, MITA_OK.
 *   Ownership     the caller owns every buffer passed in; the library never
 *                 frees or retains them. The library owns a cached scratch
 *                 workspace per (device, stream), grown on demand in stream
 *                 order (cudaMallocAsync / cudaFreeAsync on `stream`, from the
 *                 device's default memory pool) and freed by
 *                 mita_release_workspace().
 *   Streams       device entry points enqueue all work on `stream` (a
 *                 cudaStream_t; NULL = the legacy default stream) and return
 *                 without synchronising the host, also when the workspace
 *                 grows. Calls on different streams use different workspaces.
 *   Errors        a negative MITA_ERR_* code; mita_last_error() gives the
 *                 message. Argument errors are found before anything is
 *                 launched. A fault inside a kernel surfaces, as with any CUDA
 *                 call, at the caller's next synchronisation; waits inside the
 *                 kernels are bounded and report MITA_ERR_TIMEOUT through
 *                 mita_sync_status() instead of hanging. A timeout stays
 *                 recorded in the stream's workspace until mita_sync_status()
 *                 reports and clears it; until then the kernels of later calls
 *                 on that stream give up at their first wait that does not
 *                 complete at once, so their outputs are not valid. Other
 *                 codes in the status word (mita_backward's index check) do
 *                 not affect later calls.
 */
#ifndef MITA_H
#define MITA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MITA_OK 0
#define MITA_ERR_INVALID_ARG (-1) /* null/misaligned pointer, bad size or grid */
#define MITA_ERR_UNSUPPORTED (-2) /* valid for the method, not built here (d != 64, non-square 2-D m, limits) */
#define MITA_ERR_ALLOC (-3)       /* workspace allocation failed */
#define MITA_ERR_CUDA (-4)        /* a CUDA runtime call or launch failed */
#define MITA_ERR_TIMEOUT (-5)     /* a bounded device-side wait gave up */

#define MITA_MAX_M 1024
#define MITA_MAX_K 1024
#define MITA_MAX_S 8 /* routed experts per query (mita_forward_multi) */

/*
 * The MiTA forward pass, stages 1-4 above, on device buffers.
 * Q, K, V: device, bf16 [B][H][N][d] (read only). out: device, bf16
 * [B][H][N][d]. expert_idx: device, int32 [B][H][m][k]. route: device, int32
 * [B][H][N]. Returns MITA_OK or a MITA_ERR_* code; asynchronous on `stream`.
 */
int mita_forward(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h, int grid_w,
                 int m, int k, void* out, int32_t* expert_idx, int32_t* route, void* stream);

/*
 * The routing-only ablation of MiTA ("NeurIPS 2026 | Mixture-of-Top-k 注意力"
 * (shuwu5.cn), results section, and Figure 4 of "And attention is also FFN?
 * …" (en.roboind.com): routed experts alone, without the shared branch).
 * Stages 1-3 as in mita_forward (landmarks, top-k experts, routing); in
 * stage 4 each query attends only to the k pairs (K_j, V_j) of its routed
 * expert, under one softmax over those k logits. The pages compare it with
 * MiTA at k' = m + k routed pairs: pass that k'. Arguments, layouts, errors
 * and asynchrony as for mita_forward.
 */
int mita_forward_routed(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h,
                        int grid_w, int m, int k, void* out, int32_t* expert_idx, int32_t* route, void* stream);

/*
 * mita_forward computed the other way the pages allow: the Algorithm 1
 * caption of "And attention is also FFN? …" (en.roboind.com) combines the
 * shared and routed branches by online softmax, and "NeurIPS 2026 |
 * Mixture-of-Top-k 注意力" (shuwu5.cn), section "MiTA：用少量地标查询，同时完成
 * 压缩与专家构造", reuses the query-to-landmark logits for routing. Here the
 * routing kernel keeps each query's m landmark logits and also forms the
 * shared branch's softmax over them (its log-sum-exp and normalised output);
 * the expert attention then runs over the k routed keys alone, starting its
 * online softmax from that partial. Same results as mita_forward up to
 * rounding (same routes and expert sets; outputs within the same
 * tolerances). Measured slower than mita_forward on GB300, so mita_forward
 * does not use it; shapes where its kernels do not apply (m > 256, large k)
 * run mita_forward's sequence. Arguments, layouts, errors and asynchrony as
 * for mita_forward; the workspace adds 132 bytes per query.
 */
int mita_forward_split(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h,
                       int grid_w, int m, int k, void* out, int32_t* expert_idx, int32_t* route, void* stream);

/*
 * MiTA with s routed experts per query. The pages run what they call the
 * s = 1 configuration ("NeurIPS 2026 | Mixture-of-Top-k 注意力"
 * (shuwu5.cn), end of section "MiTA：用少量地标查询，同时完成压缩与专家构造") and do
 * not describe s > 1; this entry point takes the plain generalisation:
 * stage 3 gives each query the s landmarks with the highest logits
 * tau <q, Lq_i> (highest first, ties to the lower landmark index), and stage
 * 4 attends, under ONE softmax, to the m shared pairs and the union of the s
 * experts' keys (a key held by several of them enters once).
 * route: device, int32 [B][H][N][s], each query's landmarks highest first.
 * 1 <= s <= min(m, MITA_MAX_S). s = 1 is exactly mita_forward. Other
 * arguments, layouts, errors and asynchrony as for mita_forward. The extra
 * workspace is an fp32 state row of 272 bytes per query (s > 1).
 */
int mita_forward_multi(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h,
                       int grid_w, int m, int k, int s, void* out, int32_t* expert_idx, int32_t* route, void* stream);

/*
 * Backward pass: dQ, dK, dV of sum(out * dO) for the MiTA forward pass
 * (mita_forward; one routed expert per query, with the shared pairs), with
 * each landmark's top-k key set and each query's route held fixed -- they
 * are piecewise constant in the inputs, so their derivative is zero almost
 * everywhere. The pages train MiTA models ("NeurIPS 2026 | Mixture-of-Top-k
 * 注意力" (shuwu5.cn), results section: Long Range Arena training times) but
 * do not describe the backward pass; this is the derivative of the forward
 * pass of section "MiTA：用少量地标查询，同时完成压缩与专家构造" through the pooling,
 * the landmark attention (LV) and the query-expert attention.
 * Q, K, V, dO: device, bf16 [B][H][N][d] (read only). expert_idx, route:
 * device, int32, as returned by mita_forward for the same Q, K, V (read only;
 * an entry out of range is left out and makes mita_sync_status report
 * MITA_ERR_INVALID_ARG). dQ, dK, dV: device, float32 [B][H][N][d], overwritten.
 * Returns MITA_OK or a MITA_ERR_* code; asynchronous on `stream`.
 */
int mita_backward(const void* Q, const void* K, const void* V, const void* dO, int B, int H, int N, int d,
                  int grid_h, int grid_w, int m, int k, const int32_t* expert_idx, const int32_t* route, float* dQ,
                  float* dK, float* dV, void* stream);

/*
 * mita_forward with two optional extra device outputs (either may be NULL):
 * lq, float32 [B][H][m][d], the landmark queries of stage 1, and lv,
 * float32 [B][H][m][d], the shared-expert values LV of stage 2.
 */
int mita_forward_aux(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h, int grid_w,
                     int m, int k, void* out, int32_t* expert_idx, int32_t* route, float* lq, float* lv,
                     void* stream);

/*
 * mita_forward on HOST buffers (same shapes and dtypes; bf16 as uint16 bit
 * patterns). Copies the inputs to the device, runs the forward pass on
 * `stream`, copies out, expert_idx and route back, and returns once every
 * copy has finished (also on error: no copy touches the caller's buffers
 * after the call returns). When Q, K and V together reach 256 MiB the heads
 * go in up to 8 groups: one group's inputs are copied in while the previous
 * group runs on `stream` and the one before is copied out, on two copy
 * streams the library creates per (device, stream) and keeps until
 * mita_release_workspace. Host buffers may be pageable; pinned buffers copy
 * faster and overlap. Device staging buffers are part of the cached workspace.
 */
int mita_forward_host(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int B, int H, int N, int d,
                      int grid_h, int grid_w, int m, int k, uint16_t* out, int32_t* expert_idx, int32_t* route,
                      void* stream);

/*
 * mita_forward for callers that cannot allocate device memory. (The paper has
 * no counterpart: this entry point exists for library users, not for the
 * method.) Some callers must not call cudaMalloc: a framework that owns all
 * device memory through its own pool (a direct cudaMalloc would bypass its
 * accounting, and can fail once the pool has reserved the device), or a
 * latency-critical loop that cannot afford the device-wide synchronisation
 * cudaMalloc and cudaFree imply. This variant allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library call. Its scratch is one
 * static device array of MITA_NOALLOC_SCRATCH_BYTES (64 MiB), which every GPU
 * that loads the library holds until the process exits.
 *
 * Same arguments, layouts and results as mita_forward (the caller still
 * provides Q, K, V, out, expert_idx and route). A shape whose scratch
 * (mita_workspace_bytes) exceeds MITA_NOALLOC_SCRATCH_BYTES is rejected with
 * MITA_ERR_UNSUPPORTED before anything is enqueued; the ViT-sized workloads
 * (N up to a few thousand tokens, m and k in the tens) fit.
 *
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress (with that device current) and clears the array's
 * status word on `stream`; make that first call before any stream capture.
 * Every call on a device shares the one array and finds the previous call's
 * contents in it (it clears what must start at zero), so calls whose work
 * overlaps on the GPU -- concurrent streams, or several host threads -- race;
 * order them on one stream. Stage timing is not recorded for these calls. A
 * device-side timeout in them is recorded in the array's status word and
 * reported (and cleared) by mita_sync_status called with any stream of the
 * device; as for the other entry points, the outputs of a call that timed
 * out, and of later calls until the timeout is cleared, are not valid.
 */
#define MITA_NOALLOC_SCRATCH_BYTES (64 << 20)
int mita_forward_noalloc(const void* Q, const void* K, const void* V, int B, int H, int N, int d, int grid_h,
                         int grid_w, int m, int k, void* out, int32_t* expert_idx, int32_t* route, void* stream);

/*
 * Bytes of scratch one mita_forward call of this shape holds in the
 * workspace (device buffers only; excludes mita_forward_host staging).
 * Returns 0 for an invalid or empty shape.
 */
size_t mita_workspace_bytes(int B, int H, int N, int d, int grid_h, int grid_w, int m, int k);

/*
 * The landmark scan's schedule for one shape: how the k best keys of each
 * landmark ("NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
 * "MiTA：用少量地标查询，同时完成压缩与专家构造": each landmark's routed
 * expert) are found. A diagnostic for library users; host only, it needs
 * no GPU and launches nothing. Writes at most cap values to info (int64,
 * caller-owned): the number of scan levels L (the pilot levels on strided
 * key samples, then the main scan over every key); 1 when the main scan
 * writes every logit of its rows and ranks whole rows, else 0; the rank j
 * of the last pilot's speculative threshold key (0: none, the threshold is
 * the k-th best sample key); then for each level its number of keys S, the
 * stride between them, and 1 when the level writes every logit, else 0.
 * Returns the number of values a full answer takes (3 + 3 L; values past
 * cap are not written), or 0 for an invalid or empty shape (info untouched).
 */
int mita_plan_info(int B, int H, int N, int d, int grid_h, int grid_w, int m, int k, int64_t* info, int cap);

/*
 * Waits for `stream`, then reports and clears the device-side status words of
 * the current device that calls on `stream` write (its workspace's, and the
 * no-allocation scratch's): MITA_OK, MITA_ERR_TIMEOUT when a bounded wait
 * inside a kernel gave up since the last check, MITA_ERR_INVALID_ARG when
 * mita_backward found a route or expert index out of range, or MITA_ERR_CUDA
 * when the stream itself failed.
 */
int mita_sync_status(void* stream);

/*
 * Diagnostic (no counterpart in the method): enqueues on `stream` one kernel
 * whose single thread waits, with the same bounded wait the forward kernels
 * use for their handshakes, on a barrier that nothing completes. After
 * limit_us microseconds (1 <= limit_us <= 2000000, else MITA_ERR_INVALID_ARG)
 * the wait gives up, records MITA_ERR_TIMEOUT in the stream's workspace status
 * word and the kernel exits. The next mita_sync_status(stream) then reports
 * MITA_ERR_TIMEOUT and clears it; the call after that reports MITA_OK. It
 * lets a caller check that the timeout path works on its GPU: nothing hangs,
 * traps or faults. Asynchronous; returns MITA_OK or a MITA_ERR_* code.
 */
int mita_selftest_wait(int64_t limit_us, void* stream);

/*
 * Stage timing (off by default). While enabled on a host thread, every
 * forward call made from that thread records CUDA events on its stream around
 * each stage: 0 landmark pooling, 1 pilot scans (top-k thresholds from key
 * samples), 2 landmark scan, 3 expert merge/selection, 4 routing,
 * 5 grouping, 6 expert attention. mita_profile_read() waits for
 * `stream`, adds the elapsed times of all recorded calls on it to stage_ms
 * and the number of kernels each stage launched to stage_launches (arrays of
 * at least max_stages entries, either may be NULL), forgets those records and
 * returns the number of stages (7), or a MITA_ERR_* code.
 */
int mita_profile_enable(int on);
int mita_profile_read(double* stage_ms, int64_t* stage_launches, int max_stages, void* stream);
/* Name of stage i, or NULL. */
const char* mita_stage_name(int i);

/* Message for the last non-zero return on this host thread ("" if none). */
const char* mita_last_error(void);

/*
 * Frees every cached workspace of every device. Synchronises each device that
 * holds one; call it when no mita_* work is in flight.
 */
void mita_release_workspace(void);

#ifdef __cplusplus
}
#endif

#endif /* MITA_H */
