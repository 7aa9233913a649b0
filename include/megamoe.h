/*
 * megamoe.h -- C ABI of the GB300 (sm_103a) fused MoE layer forward, a8w4.
 *
 * One call runs a whole routed-expert MoE layer on one GPU: sigmoid top-k
 * routing, the fused EPLB logical->physical remap with per-expert load
 * recording, MXFP8 activation quantisation, dispatch into expert-sorted
 * tiles, GEMM1 (gate/up) with a SwiGLU + MXFP8 requantisation epilogue,
 * GEMM2 (down) and the top-k weighted combine.  Sources for the operation:
 *   - "sglang PR #47065" (Title/switches, Modifications): quantisation,
 *     dispatch, both expert GEMMs and the combine form one operator, with a
 *     single-kernel small-input path (up to 512 tokens) and a persistent large-input path
 *     (>= 1024 tokens), a per-layer slot (bind_layer) and a three-state
 *     large-input switch;
 *   - "sglang PR #35619" (Summary, EPLB arm settings): fused EPLB remap and
 *     per-expert load recording, enabled for prefill only, and graph-safe
 *     handling of an idle batch;
 *   - "InferenceX PR #3430" (draft-precision notes): routed experts are MXFP4
 *     and the MoE runs a8w4.
 * On one GPU the pages' cross-rank dispatch/combine is a local permute and a
 * local gather.
 *
 * Conventions for every call:
 *   - every function returns an mm_status; nothing throws or aborts;
 *   - a handle is not thread-safe; use it from one host thread and, for
 *     mm_forward, one stream at a time;
 *   - "device pointer" means memory of the handle's device (cudaMalloc or
 *     torch CUDA tensors); "host pointer" means ordinary CPU memory;
 *   - the library never takes ownership of caller memory.
 *
 * Formats:
 *   bf16      IEEE bfloat16, little endian
 *   MXFP4     OCP Microscaling v1.0: e2m1 elements, two per byte, element 2i
 *             in the low nibble of byte i; one e8m0 scale byte per 32
 *             consecutive elements along the reduction (K) axis
 *   MXFP8     e4m3 elements, one e8m0 scale byte per 32 along K
 */
#ifndef MEGAMOE_H
#define MEGAMOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MM_API __attribute__((visibility("default")))
#else
#define MM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mm_ctx *mm_handle;
typedef struct CUstream_st *mm_stream; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    MM_OK = 0,
    MM_ERR_INVALID_ARG = 1, /* null pointer, bad value or misaligned pointer */
    MM_ERR_UNSUPPORTED = 2, /* shape outside the supported set, or no sm_103 GPU */
    MM_ERR_NOT_READY = 3,   /* weights (or, when P > E, the EPLB map) not set */
    MM_ERR_CAPACITY = 4,    /* tokens above mm_reserve, or forced small path above its limit */
    MM_ERR_CUDA = 5,        /* a CUDA runtime call failed (allocation, copy, launch) */
    MM_ERR_TIMEOUT = 6,     /* a device-side wait gave up (latched, see mm_get_status) */
    MM_ERR_DEVICE = 7       /* a device-side check failed (latched, see mm_get_status) */
} mm_status;

typedef enum {
    MM_ROUTE_AUTO = 0,  /* T <= small limit (512): small path; otherwise large path */
    MM_ROUTE_SMALL = 1, /* always the small path; T above its limit -> MM_ERR_CAPACITY */
    MM_ROUTE_LARGE = 2  /* always the large path */
} mm_route;

typedef enum {
    MM_ACT_MXFP8 = 0,   /* a8w4: activations quantised to MXFP8 before each expert GEMM (default) */
    MM_ACT_BF16 = 1     /* a16w4: bf16 activations into both expert GEMMs, h rounded to bf16 */
} mm_act;

#define MM_MAX_LAYERS 256
#define MM_MAX_EXPERTS 512
#define MM_MAX_TOPK 8

/* Create a layer operator.  num_experts E (logical), num_physical P >= E
 * (physical slots; P - E redundant replicas), topk k, hidden H, inter I.
 * Supported: 1 <= k <= min(E, 8), E <= 512, P <= 512, H % 128 == 0,
 * I % 128 == 0, H <= 16384, I <= 8192; otherwise MM_ERR_UNSUPPORTED.
 * Uses the current CUDA device, which must be sm_103.  Allocates the
 * per-layer count table; weights and workspace come later.  The environment
 * variables MM_SMALL_M_MAX (default 512) and MM_LARGE_M_MIN (default 1024)
 * are read here, once. */
MM_API mm_status mm_create(int num_experts, int num_physical, int topk, int hidden, int inter,
                    mm_handle *out);

/* Free everything the handle owns.  Waits for the device.  NULL is a no-op. */
MM_API mm_status mm_destroy(mm_handle h);

/* Expert weights, indexed by physical expert (device pointers, 32-byte
 * aligned):
 *   w1       [P, 2I, H/2]  MXFP4 elements; rows 0..I-1 gate, I..2I-1 up
 *   w1_scale [P, 2I, H/32] e8m0
 *   w2       [P, H, I/2]   MXFP4 elements
 *   w2_scale [P, H, I/32]  e8m0
 * (P + S experts when S fused shared experts are set, see
 * mm_set_shared_experts.)  Copied (scales re-laid out for the tensor cores)
 * into library-owned memory; the caller may free its buffers after return.
 * Synchronous.  Not allowed during stream capture. */
MM_API mm_status mm_set_weights(mm_handle h, const uint8_t *w1, const uint8_t *w1_scale,
                         const uint8_t *w2, const uint8_t *w2_scale);

/* EPLB map (host pointers): phys_of_logical [E, max_replicas] row-major,
 * replica_counts [E].  Entries of row e beyond replica_counts[e] are ignored.
 * Valid iff 1 <= replica_counts[e] <= max_replicas and every physical id
 * 0..P-1 appears exactly once among the used entries; otherwise
 * MM_ERR_INVALID_ARG and the previous map stays.  A (token t, slot j) pair
 * routed to logical e goes to phys_of_logical[e][(t + j) % replica_counts[e]]
 * ("sglang PR #35619", fused EPLB remap).  When P == E the identity map is
 * the default; when P > E, mm_forward returns MM_ERR_NOT_READY until a map is
 * set.  Synchronous; not allowed during stream capture. */
MM_API mm_status mm_set_eplb_map(mm_handle h, const int32_t *phys_of_logical,
                          const int32_t *replica_counts, int max_replicas);

/* Select the count slot that later forwards record into (the pages' per-layer
 * protocol slot, "sglang PR #47065", Modifications).  0 <= layer < 256. */
MM_API mm_status mm_bind_layer(mm_handle h, int layer);

/* Per-logical-expert load recording for later forwards: on != 0 enables it.
 * Off by default; the pages enable it for prefill steps only, which is the
 * caller's choice here ("sglang PR #35619", EPLB arm settings). */
MM_API mm_status mm_set_recording(mm_handle h, int on);

/* Route selection for later forwards (three-state analogue of the pages'
 * set_large_m_enabled, "sglang PR #47065", aiter commit message). */
MM_API mm_status mm_set_route(mm_handle h, mm_route route);

/* Activation format of later forwards.  MM_ACT_MXFP8 is the fused a8w4
 * operator ("sglang PR #47065"; "InferenceX PR #3430", draft-precision notes:
 * the expert-parallel arm runs MegaMoE a8w4 on the MXFP4 experts).
 * MM_ACT_BF16 is the a16w4 variant of the other serving arms (same notes:
 * MXFP4 experts with the default bf16 activations): the hidden rows are
 * dispatched in bf16, GEMM1 runs bf16 x MXFP4 with fp32 accumulation,
 * h = silu(gate) * up is rounded to bf16 and GEMM2 runs bf16 x MXFP4; routing,
 * EPLB remap, recording and combine are unchanged.  The bf16 format runs the
 * multi-launch path only: with it, mm_set_route(MM_ROUTE_SMALL) makes
 * mm_forward return MM_ERR_UNSUPPORTED.  Changing the format drops the
 * workspace (call mm_reserve again before forwarding).  Synchronous; not
 * allowed during stream capture.  An unknown value -> MM_ERR_INVALID_ARG. */
MM_API mm_status mm_set_activation_format(mm_handle h, mm_act act);

/* Fused shared experts ("sglang PR #35619", settings that silently break it:
 * fusion sizes the operator with top-k plus the number of fused shared
 * experts).  With num_shared = S > 0 every token gets S slots after its k
 * routed ones: slot k + s is shared expert s, physical expert P + s, weight 1
 * (its output is added as is), logical id E + s in the idx intermediate, never
 * counted by the recorder.  mm_set_weights then takes P + S experts (the
 * routed physical experts, then the shared ones); the EPLB map still covers the
 * P routed ones.  Changing S drops the weights and the workspace (set them
 * again).  0 <= S, k + S <= MM_MAX_TOPK, P + S <= MM_MAX_EXPERTS, else
 * MM_ERR_INVALID_ARG.  Synchronous; not allowed during stream capture. */
MM_API mm_status mm_set_shared_experts(mm_handle h, int num_shared);

/* Reserve workspace for up to max_tokens tokens per forward (the pages' MTPR
 * capacity).  Allocates; call before any stream capture.  Calling again with
 * a larger value reallocates (synchronous); a smaller value is a no-op. */
MM_API mm_status mm_reserve(mm_handle h, int64_t max_tokens);

/* The layer forward.  Device pointers, 16-byte aligned:
 *   hidden   [T, H] bf16
 *   logits   [T, E] fp32 router logits (finite)
 *   bias     [E]    fp32 selection bias, or NULL for zeros
 *   out      [T, H] bf16, must not overlap any input
 * num_tokens T >= 0.  Enqueued on `stream`; no host synchronisation and no
 * allocation, so the call can be captured into a CUDA graph.  T == 0 returns
 * MM_OK and enqueues nothing (idle batch, "sglang PR #35619", graph-safe idle
 * handling).  T > reserved capacity -> MM_ERR_CAPACITY, nothing enqueued.
 * Device-side failures (a wait that timed out) are latched and reported by
 * mm_get_status and mm_read_counts. */
MM_API mm_status mm_forward(mm_handle h, const void *hidden, const float *logits, const float *bias,
                     void *out, int64_t num_tokens, mm_stream stream);

/* Copy the int64 per-logical-expert counts [E] of slot `layer`, accumulated
 * since creation or the last mm_reset_counts, to host memory out_host.
 * Synchronises the device first (the only device-to-host read on the path).
 * Returns the latched device error, if any, after copying. */
MM_API mm_status mm_read_counts(mm_handle h, int layer, int64_t *out_host);

/* Zero the counts of slot `layer` (-1: every slot).  Synchronous. */
MM_API mm_status mm_reset_counts(mm_handle h, int layer);

/* Synchronise the device, store the latched device status in *device_code
 * (0 = none, else an mm_status value) and clear it.  After a device error it
 * also resets the fused kernel's grid-barrier count (an aborted launch may
 * have left arrivals missing), so call it before the next forward once a
 * forward has failed on the device.  Until it is called, a forward that takes
 * the fused small-input kernel does no work at all (its output is not
 * written) and the error stays latched, so a forward made after an unread
 * failure never passes off stale output as a success. */
MM_API mm_status mm_get_status(mm_handle h, int *device_code);

/* Intermediates of the last forward, for tests.  Synchronous.  `stage`:
 *   0 idx     int32 [T, k]     logical experts in selection order
 *   1 weights fp32  [T, k]     normalised routing weights
 *   2 phys    int32 [T, k]     physical experts
 *   3 pos     int32 [T, k]     dispatch row of each (token, slot) pair
 *   4 offsets int32 [P + 1]    start row of each physical expert's segment
 *                              (segments are padded to 16 rows); [P] = total
 *   5 xq      uint8 [rows, H]  dispatched MXFP8 activation codes
 *             (bf16 format: the dispatched bf16 rows [rows, H])
 *   6 xs      uint8 [rows, H/32] their scale bytes, row-major (bf16: empty)
 *   7 hq      uint8 [rows, I]  GEMM1 output codes (after SwiGLU, requant)
 *             (bf16 format: h in bf16 [rows, I])
 *   8 hs      uint8 [rows, I/32] their scale bytes, row-major (bf16: empty)
 *   9 y       bf16  [rows, H]  GEMM2 output rows
 * where rows = offsets[P].  Copies min(bytes, size of the stage) bytes into
 * dst_host; MM_ERR_INVALID_ARG for an unknown stage. */
MM_API mm_status mm_debug_dump(mm_handle h, int stage, void *dst_host, size_t bytes);

/* Stage 10 of mm_debug_dump: int32 [4] = {route taken by the last forward
 * (1 small, 2 large), number of kernels it launched, site of the last
 * device-side timeout or check (0 none; see WaitSite in the sources), the
 * grouped GEMM kernel of the large path (0 none, 1 one CTA per unit, 2 CTA
 * pairs with 2-SM MMAs, 3 the a16w4 kernel)}.  By default both a8w4 kernels
 * are launched and the tile scan picks one on the device: the pair kernel when
 * the experts' odd tile counts add at most 1/64 to the MMA work (environment
 * MM_GEMM_2SM=0 or 1 fixes the one-CTA or the pair kernel); the entry then
 * names the kernel that ran and the launch count includes the other.
 * Stage 11: uint64 [SMs][8] %globaltimer readings (ns) of each CTA of the last
 * fused small-input launch at its stage boundaries: start, routed, past
 * barrier 1, dispatched, past barrier 2, GEMMs done, past barrier 3, end.
 * Stage 12: int32 [tiles][3] token tiles of the last forward, each {physical
 * expert, first dispatch row, rows}: a segment is cut into tiles of 128 rows
 * (large-input path) or of 64 or 128 rows (fused small-input kernel, which
 * takes 64 unless that adds more than 1/16 to the number of tiles). */

/* Size in bytes of a debug stage for the last forward (0 before any). */
MM_API mm_status mm_debug_size(mm_handle h, int stage, size_t *bytes);

/* EPLB replica planner (host only, no CUDA).  load [E] (host): recorded
 * tokens per logical expert, e.g. from mm_read_counts over a rebalance
 * interval (the pages rebalance every 200 iterations from the recorder's
 * statistics, "sglang PR #35619", EPLB arm settings).  Every logical expert e
 * keeps physical slot e; each redundant slot E..P-1 in turn goes to the
 * expert with the highest load per replica (load[e] / replicas, compared
 * exactly; the lower index on ties) among those below max_replicas.  Writes
 * phys_of_logical [E, max_replicas] (unused entries -1) and replica_counts
 * [E], ready for mm_set_eplb_map.  MM_ERR_INVALID_ARG if P - E slots cannot be
 * placed under max_replicas. */
MM_API mm_status mm_plan_replicas(const int64_t *load, int num_experts, int num_physical, int max_replicas,
                                  int32_t *phys_of_logical, int32_t *replica_counts);

/* Rebalance the handle's replicas from the counts recorded in slot `layer`:
 * plans with mm_plan_replicas, copies each re-assigned physical slot's
 * weights on the device from its logical expert's own slot (slot e must hold
 * logical e), and installs the new map.  Synchronous; not allowed during
 * stream capture.  A no-op when P == E.  Outputs of later forwards are
 * unchanged (replicas are byte copies); only the load spread changes. */
MM_API mm_status mm_rebalance(mm_handle h, int layer, int max_replicas);

/* Per-launch timing of the dominant kernel (the grouped GEMM, or the fused
 * small-input kernel).  mm_profile_begin creates max_launches pairs of CUDA
 * events (allocation: call it outside stream capture); each later mm_forward
 * records one pair on its stream right around that kernel, until
 * max_launches forwards have been recorded.  mm_profile_end synchronises,
 * writes up to max_out durations in milliseconds to ms_out (host), stores
 * how many in *n_out, and stops recording. */
MM_API mm_status mm_profile_begin(mm_handle h, int max_launches);
MM_API mm_status mm_profile_end(mm_handle h, float *ms_out, int max_out, int *n_out);

/* Dispatch plan without allocation.  The pages have no counterpart; this is a
 * convenience for callers that cannot allocate device memory where they need
 * the plan (code running under another framework's memory pool or an
 * allocator-free runtime, or a steady-state serving loop that must not call
 * cudaMalloc, which synchronises the device).
 *
 * Inputs (device pointers): phys [npairs] int32, the physical expert of each
 * (token, slot) pair in pair order; num_physical P (1..512).  Outputs (device
 * pointers): pos [npairs] int32, the dispatch row of each pair, and offsets
 * [P + 1] int32, each expert's segment start -- the same plan mm_forward's
 * permute builds: pairs grouped by expert in pair order, segments padded to
 * multiples of 16 rows, offsets[P] = total rows.  An id outside [0, P) gets
 * pos = -1 and is left out.  npairs <= 131072, else MM_ERR_CAPACITY.
 *
 * Scratch lives in a 256 KB array inside the library, not in allocated
 * memory; every GPU that loads the library holds it until the process exits.
 * The first call on a device, and the first call after that device's context
 * was created anew (cudaDeviceReset), looks up that array's device address:
 * make it before any stream capture.  All calls share the array, so calls whose
 * kernels overlap on the GPU (different streams, or different threads without
 * ordering) race and must not be made; calls in one stream are fine.
 * Asynchronous on `stream`; allocates nothing. */
MM_API mm_status mm_plan_dispatch_static(const int32_t *phys, int64_t npairs, int num_physical, int32_t *pos,
                                         int32_t *offsets, mm_stream stream);

/* ---- Expert parallelism across ranks -------------------------------------
 * The pages run the fused operator expert-parallel over eight GPUs, with
 * all-to-all dispatch and combine buffers ("sglang PR #35619", launch
 * settings; "sglang PR #47065", Title/switches: one kernel covers quantisation,
 * dispatch, both expert GEMMs and the combine across ranks).  Here the P
 * physical experts are split over `world` ranks in contiguous ranges, each
 * rank one handle on its own GPU, and one rank's forward is:
 *
 *   mm_ep_dispatch   its tokens -> send buffer, rows grouped by destination
 *   (caller)         all-to-all: rank d receives its range from every rank
 *   mm_ep_experts    received rows -> y rows, in the order received
 *   (caller)         all-to-all back: y rows return to the sending rank
 *   mm_ep_combine    y rows in send order -> the layer output
 *
 * Row arithmetic is that of mm_forward (same codes, scales, MMAs, epilogue and
 * combine order), so the output equals the single-GPU forward's bit for bit.
 *
 * mm_set_expert_parallel: make this handle rank `rank` of `world`; first
 * (host, [world + 1]) gives each rank's range [first[r], first[r+1]) of
 * physical experts, first[0] = 0, first[world] = P, every range non-empty.
 * Afterwards mm_set_weights takes the weights of the rank's own experts only
 * ([first[rank+1] - first[rank]] experts, the same layouts), the routing and
 * the EPLB map stay global, and mm_forward, mm_rebalance, shared experts and
 * the a16w4 format return MM_ERR_UNSUPPORTED.  Frees the weights and the
 * workspace.  Synchronous; not during capture. */
MM_API mm_status mm_set_expert_parallel(mm_handle h, int rank, int world, const int32_t *first);

/* Workspace for dispatching up to max_tokens of this rank's tokens and for
 * receiving up to max_recv_rows rows (padding rows included).  Allocates;
 * call before capture. */
MM_API mm_status mm_ep_reserve(mm_handle h, int64_t max_tokens, int64_t max_recv_rows);

/* Rows the send buffers need for num_tokens tokens: T k pairs plus the
 * padding of each expert's segment to a multiple of 16 rows. */
MM_API mm_status mm_ep_send_rows(mm_handle h, int64_t num_tokens, int64_t *rows);

/* Step 1, on the source rank.  hidden [T, H] bf16, logits [T, E] fp32 and
 * bias [E] fp32 (or NULL) as in mm_forward.  The send buffers are caller-owned
 * device buffers of send_capacity rows each (16-byte aligned); they need the
 * rows of mm_ep_send_rows(T), else MM_ERR_CAPACITY and nothing is enqueued.
 * Writes, for rows = mm_ep_send_rows(T):
 *   send_xq  [rows, H]     e4m3 codes of each (token, slot) pair
 *   send_xs  [rows, H/32]  their e8m0 scales, row-major
 *   send_eid [rows] int32  the pair's expert index among its destination
 *                          rank's experts; -1 on a padding row
 * Rows bound for rank d are [row_off[d], row_off[d+1]) (row_off: host,
 * [world + 1], written by this call); inside that range the segments of d's
 * experts in expert order, pairs in (token, slot) order, each segment padded
 * to 16 rows.  Records counts as mm_forward does.  Synchronous at its end (it
 * reads the split sizes back for the all-to-all), so not capturable.
 * T > reserved tokens -> MM_ERR_CAPACITY; T == 0 -> all row_off 0. */
MM_API mm_status mm_ep_dispatch(mm_handle h, const void *hidden, const float *logits, const float *bias,
                                int64_t num_tokens, void *send_xq, void *send_xs, int32_t *send_eid,
                                int64_t send_capacity, int64_t *row_off, mm_stream stream);

/* Step 2, on the destination rank.  recv_xq [n, H], recv_xs [n, H/32] and
 * recv_eid [n] are the rows this rank received (in any order of sources;
 * padding rows, eid -1, are skipped).  Writes y_recv [n, H] bf16: row i is
 * GEMM2(SwiGLU(GEMM1(row i))) of expert recv_eid[i], zeros for a padding
 * row.  Asynchronous on `stream`; allocates nothing.  n > reserved receive
 * rows -> MM_ERR_CAPACITY; weights not set -> MM_ERR_NOT_READY. */
MM_API mm_status mm_ep_experts(mm_handle h, const void *recv_xq, const void *recv_xs, const int32_t *recv_eid,
                               int64_t n, void *y_recv, mm_stream stream);

/* Step 3, on the source rank: y_back [rows, H] bf16 holds the y rows returned
 * by the destinations in send-buffer order (rows of the last mm_ep_dispatch);
 * out [T, H] bf16 = sum_j w[t,j] y_back[row of (t, j)] over that dispatch's
 * tokens, fp32 in slot order.  Asynchronous; allocates nothing. */
MM_API mm_status mm_ep_combine(mm_handle h, const void *y_back, void *out, mm_stream stream);

/* Short text for a status code (static storage). */
MM_API const char *mm_status_string(mm_status s);

#ifdef __cplusplus
}
#endif

#endif /* MEGAMOE_H */
