/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE-layer forward megakernel.
 *
 * The operation (what every call below computes) is the forward pass of one
 * Mixture-of-Experts layer, as described in
 *   Weave abstract (arXiv 2609.21483): routing, then dispatch of tokens to
 *     experts, the expert computation, and the combine back to token order,
 *     run as one persistent megakernel whose CTAs are split by a cost model
 *     into data-movement and computation workers once routing is known;
 *   xxqk.cn/news/665650 section 1 (router, top-k expert selection, the
 *     expert matrix products, weighted merge of the expert outputs) and
 *     section 2.1-2.3 (an in-kernel atomic task queue; per-task dependency
 *     counters that release a task when they reach zero; no global barrier);
 *   m.xxqk.cn/news/657744 section 2.1 (scheduling units: an expert's up
 *     projection, then its down projection, large GEMMs split along K) and
 *     section 5.1 (scheduling state lives in device memory passed to the
 *     kernel).
 *
 * Per token t (T tokens, model dim d, E routed experts, top-k, expert FFN
 * dim f, S in {0,1} always-on shared experts):
 *   L[t,e]  = sum_i x[t,i] * Wr[e,i] + b[e]                (fp32 accumulate)
 *   p[t,:]  = softmax(L[t,:]) over all E experts
 *   idx[t,:]= the k experts with the largest p (ties: lower expert index)
 *   w[t,j]  = p[t,idx[t,j]] / sum_j' p[t,idx[t,j']]         (renormalised)
 *   h       = bf16( silu(Wg[e] x_t) * (Wu[e] x_t) ),  silu(z) = z / (1 + e^-z)
 *   y_e     = Wd[e] h
 *   out[t]  = bf16( sum_j w[t,j] * y_{idx[t,j]}  +  y_shared )
 * Tokens are permuted into per-expert rows in the canonical order: experts
 * ascending, tokens ascending inside an expert.
 *
 * Conventions for every entry point:
 *   - bf16 tensors are IEEE bfloat16, row-major, contiguous, 16-byte aligned
 *     device pointers owned by the caller;
 *       x        [T, d]         token activations
 *       router_w [E, d]         router weight (nn.Linear layout)
 *       w_gate   [E+S, f, d]    gate projections, shared expert stored last
 *       w_up     [E+S, f, d]    up projections
 *       w_down   [E+S, d, f]    down projections
 *       out      [T, d]         overwritten (not accumulated)
 *   - a stream argument is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream);
 *   - every int-returning call returns MOE_OK (0) or one of MOE_E_*; the
 *     message of the last failure on the calling thread is moe_last_error();
 *   - a handle serves one stream at a time; calls on one handle are not
 *     thread-safe.
 * Limits: d % 128 == 0, d <= 32768, f % 128 == 0, 1 <= k <= E <= 256,
 * k <= 16, S <= 1, 0 <= T <= T_max given to moe_layer_reserve, T_max <= 32768.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_layer moe_layer_t;

/* status codes */
#define MOE_OK 0
#define MOE_E_INVAL 1   /* bad argument, alignment, size, or T > T_max    */
#define MOE_E_CUDA 2    /* a CUDA call or kernel launch failed             */
#define MOE_E_TIMEOUT 3 /* a device-side wait ran out of its time budget   */
#define MOE_E_DEVICE 4  /* the kernel found an inconsistent scheduler state */
#define MOE_E_NOMEM 5   /* device or pinned host allocation failed         */
#define MOE_E_STATE 6   /* call order: forward before reserve, etc.        */

/* execution modes (option MOE_OPT_MODE) */
#define MOE_MODE_PERSISTENT 0  /* one persistent megakernel, task queue      */
#define MOE_MODE_MULTIKERNEL 1 /* ablation: one kernel per stage, no queue   */
#define MOE_MODE_STATIC 2      /* ablation: one cooperative launch, tasks
                                  assigned round-robin per stage, grid-wide
                                  barriers between stages, no queue          */

/* option keys for moe_layer_set_option */
#define MOE_OPT_MODE 1         /* MOE_MODE_*                                   */
#define MOE_OPT_TIMEOUT_NS 2   /* device wait budget in ns (default 2e9)      */
#define MOE_OPT_MOVER_CTAS 3   /* >0: fixed number of mover workers (a CTA or
                                  a CTA pair each); 0 = the cost model        */
#define MOE_OPT_GRID_CTAS 4    /* >0: CTAs of the persistent (and static)
                                  grid, rounded down to whole workers (at
                                  least one); 0 = one CTA per SM (every SM
                                  pair the device keeps resident, for pairs) */
#define MOE_OPT_SPLIT_K 5      /* down-projection K splits (1,2,4; 0 = auto)  */
#define MOE_OPT_TOKENS_PER_TILE 6 /* max tokens per GEMM tile: 0 = auto, else
                                     16..256 in steps of 16, used rounded up
                                     to a multiple of 32                       */
#define MOE_OPT_FAULT_DROP_TASK 7 /* test only: -1 off; else drop the dependency
                                     notification of the n-th finished GEMM task,
                                     which must end in MOE_E_TIMEOUT            */
#define MOE_OPT_ROUTE_TOKENS 8 /* tokens per router tile: 64 or 128; 0 (default)
                                  = 64 when T <= 1024 and E >= 64, else 128.
                                  A forward with more than 256 router tiles
                                  fails with MOE_E_INVAL                      */
#define MOE_OPT_CLAIM_AHEAD 9  /* claim the next task while running one when at
                                  least this many tasks wait; -1 auto, 0 off  */
#define MOE_OPT_TRACE 10       /* >0: record up to this many task records per
                                  forward (allocates; see moe_layer_get_trace) */
#define MOE_OPT_RELEASE 11     /* when gate/up tiles become ready: 0 = all at
                                  once after the last gather, f-tile major;
                                  1 = per expert after its gathers (default) */
#define MOE_OPT_PREFETCH 12    /* 1 (default): while a GEMM tile finishes, the
                                  TMA producer starts loading the next tile
                                  claimed ahead; 0: off                        */
#define MOE_OPT_BANDS 13       /* 1 (default): the down tiles of the last
                                  quarter of d run at low priority and the
                                  combine is split in two d bands, so the
                                  first band's combine overlaps them; 0: one
                                  band                                         */
#define MOE_OPT_ROUTE_SPLITS 14 /* K splits of a router tile (1..8; 0 = auto:
                                  enough to spread the tiles over the SMs,
                                  8 k blocks per split at least); capped so
                                  that tiles x splits <= the SM count          */
#define MOE_OPT_L2_PREFETCH 15 /* persistent mode: bytes of the first gate/up
                                  weight tiles (experts in index order) to
                                  prefetch into L2 once the plan is published,
                                  while the gathers run; the plan keeps
                                  experts in index order then.
                                  -1 (default) = 96 MiB when S = 0 and the
                                  mean expert load is at most half a GEMM
                                  tile, else off; 0 = off                      */

#define MOE_OPT_PAIR 16        /* CTAs per worker: 2 = GEMM tiles on CTA pairs
                                  (clusters of two SMs sharing one tensor-core
                                  tile, tcgen05 .cta_group::2, M = 256), 1 =
                                  one CTA per tile (M = 128); 0 (default) =
                                  pairs when the mean rows per expert
                                  (T k / E) are at least 128                 */

#define MOE_OPT_FRONT_SPLIT 17 /* persistent mode, once routing is known:
                                  1 = only the cost model's mover workers
                                  prefer the gathers; the GEMM workers run
                                  the GEMM tiles that are ready and take
                                  gathers only when none is; 0 = every worker
                                  prefers gathers while any is left; -1
                                  (default) = 1 without a shared expert, 0
                                  with one                                   */

#define MOE_OPT_FAULT_DROP_TYPE 18 /* test only: 0 off; 2, 3 or 4 = drop every
                                      dependency notification of gather,
                                      gate/up or down tasks, which must end
                                      in MOE_E_TIMEOUT                        */
#define MOE_OPT_FAULT_CORRUPT_COUNT 19 /* test only: 0 off; else the plan adds
                                      this to the first expert's token count;
                                      its check (counts summing to T k) must
                                      end the pass in MOE_E_DEVICE           */
#define MOE_OPT_FAULT_REPUSH 20 /* test only, with MOE_OPT_DEBUG_CLAIMS: -1
                                  off; else the n-th finished gate/up task is
                                  pushed into the queue again, which the
                                  claimed-twice check must end in
                                  MOE_E_DEVICE (without the check the extra
                                  claim can end the queue's count early: the
                                  output is then undefined)                   */
#define MOE_OPT_DEBUG_CLAIMS 21 /* persistent mode: 1 = every task claimed
                                  sets a bit; a task claimed twice (or an id
                                  outside the layer's tasks) sets
                                  MOE_E_DEVICE, never a trap; 0 (default) off */

#define MOE_OPT_FOLD_GATHER 22 /* 1: a routed gate/up tile gathers its token
                                  rows from x itself (warps idle during its
                                  main loop copy them into the stages through
                                  perm, 16 bytes at a time), and the gather
                                  tasks only write perm and pos; 0 (default):
                                  the gather tasks copy the rows into a
                                  permuted buffer that the tiles load by TMA.
                                  Same bits either way; 1 is slower on this
                                  GPU (the copies keep too few bytes in
                                  flight)                                    */

/* statistics keys for moe_layer_get_stat (values of the last forward;
 * moe_layer_status must have been called after it) */
#define MOE_STAT_MOVER_CTAS 1  /* mover workers the cost model chose          */
#define MOE_STAT_TASKS 2       /* tasks executed (all types)                   */
#define MOE_STAT_GRID 3        /* CTAs launched for the persistent kernel
                                  (MOE_STAT_PAIR per worker)                  */
#define MOE_STAT_GEMM_TASKS 4  /* expert GEMM tasks executed                   */
#define MOE_STAT_MOVER_TASKS 5 /* gather + combine tasks executed              */
#define MOE_STAT_STOLEN 6      /* tasks a CTA ran from the other role's queue  */
#define MOE_STAT_AHEAD 7       /* tasks claimed ahead while another one ran    */
#define MOE_STAT_TRACE_RECORDS 8 /* task records the last forward produced     */
#define MOE_STAT_TILE_TOKENS 9 /* max tokens per GEMM tile of the last forward */
#define MOE_STAT_SPLIT_K 10    /* down-projection K splits of the last forward */
#define MOE_STAT_BANDS 11      /* d bands of the last forward (1 or 2)         */
#define MOE_STAT_Y_BYTES 12    /* bytes the combine read per down-projection
                                  output value in the last forward: 2 (bf16
                                  outputs) or 4 * split_k (fp32 partials)     */
#define MOE_STAT_COMBINE_TOKENS 13 /* tokens per combine tile of the last
                                      forward                                  */
#define MOE_STAT_PAIR 14       /* CTAs per worker of the last forward (1 or 2) */

/* Create a layer description.  Pure host call (no CUDA call, no allocation on
 * the device).  Returns NULL on invalid dimensions (see moe_last_error),
 * among them d > 32768: a gather copies whole bf16 token rows through the
 * pipeline's shared memory, which holds a 64 KB row under every tiling. */
moe_layer_t* moe_layer_create(int d, int f, int E, int k, int shared_experts);

/* Allocate the device workspace for up to T_max tokens on the current device
 * (routing arrays, permuted activations, expert intermediates, scheduler
 * state) and cache the device properties.  The only allocating call besides
 * moe_layer_forward_host's first use; call it before any stream capture.
 * May be called again to grow or shrink. */
int moe_layer_reserve(moe_layer_t* h, int T_max, void* stream);

/* Set the per-expert router bias (fp32 [E] device pointer, added to the
 * logits before softmax and top-k); NULL removes it.  The pointer is read at
 * every forward and must stay valid. */
int moe_layer_set_router_bias(moe_layer_t* h, const float* bias);

/* One forward pass of the layer on T tokens (device pointers, see the layout
 * above).  Asynchronous on `stream`; allocates nothing and never synchronises,
 * so it can be captured in a CUDA graph.  Device-side failures (timeouts,
 * inconsistent state) are reported by the next moe_layer_status. T == 0 is a
 * no-op. */
int moe_layer_forward(moe_layer_t* h, int T, const void* x, const void* router_w,
                      const void* w_gate, const void* w_up, const void* w_down, void* out,
                      void* stream);

/* The forward pass with the residual add and the RMSNorm that end the MoE
 * megakernel (xxqk.cn/news/665650 section 1 lists them after the weighted
 * merge) fused into the combine.  Per token t, with layer[t] the value
 * moe_layer_forward rounds to bf16:
 *   out[t]      = bf16( residual[t] + layer[t] )          (fp32 add)
 *   norm_out[t] = bf16( out[t] * rsqrt(mean_c out[t,c]^2 + eps) * gamma )
 * the mean over the d values of out[t] as stored (bf16).  residual [T, d] and
 * gamma [d] are bf16 device pointers, norm_out [T, d] is overwritten; all
 * 16-byte aligned; 0 <= eps <= 1.  Everything else (routing, scheduling,
 * status, asynchrony, no allocation) is that of moe_layer_forward, except
 * that the combine covers whole rows (MOE_OPT_BANDS does not apply): each
 * combine task adds the residual rows, bulk-copied with the expert rows, and
 * then normalises its tile's rows. */
int moe_layer_forward_residual_norm(moe_layer_t* h, int T, const void* x, const void* router_w,
                                    const void* w_gate, const void* w_up, const void* w_down,
                                    const void* residual, const void* gamma, float eps,
                                    void* out, void* norm_out, void* stream);

/* The same forward pass with x and out in host memory: copies x to the
 * device, runs moe_layer_forward, copies out back and synchronises the
 * stream.  Weights are device pointers as above.  Host buffers may be
 * pageable or pinned; the first call allocates a device staging area for
 * T_max tokens.  Returns the device status of the pass as well. */
int moe_layer_forward_host(moe_layer_t* h, int T, const void* x_host, const void* router_w,
                           const void* w_gate, const void* w_up, const void* w_down,
                           void* out_host, void* stream);

/* The same forward pass without any allocation, for callers that cannot call
 * cudaMalloc: processes whose device memory is owned by another allocator (a
 * framework's caching allocator that must account for every byte), and
 * runtimes that forbid allocation after start-up (fixed memory budgets,
 * real-time or certified deployments).  (The pages have no counterpart: this
 * is an interface convenience, not part of the method.)  Needs only
 * moe_layer_create (host memory); no moe_layer_reserve.  Its scratch is a
 * fixed 32 MiB array inside this library's device code, which every GPU that
 * loads the library holds until the process exits.  Layers whose workspace
 * for T tokens exceeds it are rejected with MOE_E_INVAL and a message naming
 * the size needed (the decode-sized layer, T=256 d=4096 E=8 k=2 f=14336,
 * fits).  The first call on a device looks up the scratch array's device
 * address and sets kernel attributes (no allocation); make that first call
 * before any stream capture.  Later calls look the address up again and
 * redo that set-up if it changed (after a device reset).  Every call on a
 * device shares the one array and the array keeps the last call's contents:
 * the scheduler state is cleared at each call, but calls that overlap on the
 * GPU (two streams, two threads, two handles) race on it.  Inputs, outputs,
 * layouts, options and the asynchronous behaviour are those of
 * moe_layer_forward.  When the fp32 K-split partials of the down projection
 * do not fit the scratch, it keeps them in bf16 with one K split, so its
 * results may differ from moe_layer_forward's in the last bits (both stay
 * within the oracle's tolerance).  After a call, moe_layer_status and
 * moe_layer_get_routing on the same handle report this call (read from the
 * shared array: call them before another no-allocation forward runs on the
 * device); moe_layer_get_trace does not cover these calls. */
int moe_layer_forward_noalloc(moe_layer_t* h, int T, const void* x, const void* router_w,
                              const void* w_gate, const void* w_up, const void* w_down, void* out,
                              void* stream);

/* Copy the routing of the last forward into caller device buffers (any may be
 * NULL): idx int32 [T,k], w fp32 [T,k] (renormalised weights, slot order),
 * counts int32 [E], offsets int32 [E+1], perm int32 [T*k] (source token of
 * each permuted row), pos int32 [T,k] (permuted row of each (token, slot)).
 * Asynchronous on `stream`. */
int moe_layer_get_routing(moe_layer_t* h, int32_t* idx, float* w, int32_t* counts,
                          int32_t* offsets, int32_t* perm, int32_t* pos, void* stream);

/* Synchronise `stream`, then return and clear the sticky device status of the
 * last forward (MOE_OK, MOE_E_TIMEOUT or MOE_E_DEVICE), or MOE_E_CUDA when a
 * CUDA error is pending. */
int moe_layer_status(moe_layer_t* h, void* stream);

/* Automatic granularity calibration (the per-workload tuning of task
 * granularity discussed in xxqk.cn/news/665650 section 4.4 and
 * m.xxqk.cn/news/657744 section 5.2): times the forward pass on these inputs
 * for a few candidate settings -- tokens per GEMM tile (auto, 64, 128, 160,
 * 256), down-projection K splits (auto, 1, 2, 4), one or two d bands -- by
 * coordinate descent from the current options, `reps` timed passes each
 * (1..100, after one untimed pass), and keeps the fastest as the handle's
 * options (MOE_OPT_TOKENS_PER_TILE, MOE_OPT_SPLIT_K, MOE_OPT_BANDS).
 * Arguments are those of moe_layer_forward (out is overwritten, 1 <= T);
 * best_us (may be NULL) receives the best mean time in microseconds.  It runs
 * 10-20 forwards and synchronises the stream after each candidate, so call it
 * at set-up, not under stream capture; it allocates nothing (two CUDA events).
 * Candidates that fail (a tile too large, a device timeout) are skipped; the
 * MOE_STAT_TILE_TOKENS / _SPLIT_K / _BANDS statistics of the next forward
 * report the chosen tiling.  The expert selection of every candidate is the
 * same; K splits change the fp32 summation order, so outputs may differ from
 * the uncalibrated pass in their last bits. */
int moe_layer_calibrate(moe_layer_t* h, int T, const void* x, const void* router_w,
                        const void* w_gate, const void* w_up, const void* w_down, void* out,
                        int reps, float* best_us, void* stream);

/* Set an option (MOE_OPT_*).  Takes effect at the next forward. */
int moe_layer_set_option(moe_layer_t* h, int key, long long value);

/* Read a statistic (MOE_STAT_*) of the last forward whose status was read. */
long long moe_layer_get_stat(moe_layer_t* h, int key);

/* Copy the task trace of the last forward (option MOE_OPT_TRACE) into a host
 * buffer of `cap` records; synchronises `stream`.  Each record is four
 * uint64: (CTA index << 32) | task id, then three %globaltimer readings in ns:
 * when the CTA began claiming the task, when it began running it, and when
 * it had published its results.  Task id bits 28-31 hold the type (1 router
 * tile, 2 gather, 3 gate/up GEMM, 4 down GEMM, 5 combine).  Returns the
 * number of records copied, or -1 on error. */
int moe_layer_get_trace(moe_layer_t* h, uint64_t* records, int cap, void* stream);

/* Bytes of device workspace moe_layer_reserve(T_max) allocates (host-only;
 * -1 for a NULL handle or T_max < 0).  Not monotone in T_max: while four
 * fp32 K-split partials of the down-projection outputs of T_max tokens fit
 * in 512 MB the workspace holds them, beyond that only bf16 outputs. */
long long moe_layer_workspace_bytes(const moe_layer_t* h, int T_max);

/* Free the workspace and the handle.  NULL is ignored. */
void moe_layer_destroy(moe_layer_t* h);

/* Message of the last failed call on this thread ("" if none). */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
