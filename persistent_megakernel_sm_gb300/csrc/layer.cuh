// Launch parameters, workspace layout and task encoding of the MoE-layer
// forward megakernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kThreads = 256;       // 8 warps per CTA
constexpr int kBM = 128;            // weight rows per accumulator in one CTA (a pair's MMA M is 256)
constexpr int kPairMinRows = 128;   // mean rows per expert from which GEMM tiles run on CTA pairs
constexpr int kBK = 64;             // K elements per pipeline stage (128 B rows)
constexpr int kABoxBytes = kBM * kBK * 2;   // 16 KB weight box
constexpr int kBBoxRows = 32;       // token rows per activation box
constexpr int kBBoxBytes = kBBoxRows * kBK * 2;  // 4 KB
constexpr int kGatherRowsCta = 32;  // permuted rows per gather task and CTA of the worker ...
constexpr int kGatherRowsCtaBig = 64;  // ... and in layers of at least kGatherBigRows routed rows
constexpr int kGatherBigRows = 16384;
constexpr int kRouteTokens = 128;   // tokens per router tile (one CTA's 128 rows of the MMA M)
constexpr int kRouteTokensSmall = 64;  // router tile of small layers with many experts
constexpr int kSmallRouteT = 1024;
constexpr int kSmallRouteMinE = 64;
constexpr int kMaxRouteKs = 8;      // K splits of a router tile, at most
constexpr int kShards = 8;          // shards of each task queue
constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kMaxD = 32768;        // model dim limit: one bf16 row (64 KB) fits a gather round
constexpr int kTmemCols = 512;
constexpr int kAcc1Col = 256;       // second accumulator's first TMEM column
constexpr int kEpiBytes = 1024;     // GEMM epilogue staging per compute warp (16 x 32 bf16)

// release policies of the gate/up tiles
constexpr int kReleaseAll = 0;
constexpr int kReleaseExpert = 1;

// task types (bits 28-31 of a task id)
enum TaskType : int {
  kTaskRoute = 1,    // router tiles (one per CTA of the worker): logits, softmax, top-k, counts
  kTaskGather = 2,   // mover: copy token rows of x into permuted rows of Xp
  kTaskGateUp = 3,   // GEMM: H = bf16(silu(Xp Wg^T) * (Xp Wu^T)), one f tile (128 rows per CTA)
  kTaskDown = 4,     // GEMM: Y = H Wd^T, one d tile (256 rows per CTA), one K split
  kTaskCombine = 5,  // mover: out = bf16(sum_j w_j Y[pos] + Y_shared)
  kTaskPlan = 6,     // (trace records only) the plan, run inline after the last router tile
};

__host__ __device__ constexpr int task_id(int type, int payload) { return (type << 28) | payload; }
__host__ __device__ constexpr int task_type(int id) { return (id >> 28) & 0xF; }
__host__ __device__ constexpr int task_payload(int id) { return id & 0x0FFFFFFF; }

// One GEMM row group: up to bn_max permuted rows of one expert (or, for the
// shared expert, up to bn_max consecutive tokens).  An expert with more rows
// has several sibling groups [sib0, sib0 + nsib); its gate/up and down tasks
// are released together and interleaved, so the siblings read each weight
// tile at nearly the same time and the second read is served by L2.
struct Group {
  int e;         // expert index (E for the shared expert)
  int row0;      // first row in H / Y
  int nrows;     // rows in this group
  int src_row0;  // first row of the B operand source (Xp for routed, x for shared)
  int sib0;      // first sibling group of the same expert
  int nsib;      // sibling groups of the expert
  int gchunks;   // gather tasks of all siblings
  int pad;       // the expert's first permuted row (offsets[e]); unused for the shared expert
};

// Scheduler state.  Zeroed before every launch.
// A queue shard word packs the shard's claims (low 32 bits) and dynamic
// pushes (high 32 bits), so one load sees both and one CAS claims.
struct Sched {
  unsigned long long mover_q[kShards];
  unsigned long long gemm_q[kShards];
  int status;
  int route_done;
  int plan_done;
  int n_movers;
  int mover_total_dyn;
  int gemm_total_dyn;
  int n_groups;         // shared + routed groups
  int tasks_done;
  int stat_gemm;
  int stat_mover;
  int stat_stolen;
  int fault_seen;
  int repush_seen;
  int err_info;
  int trace_n;
  int stat_ahead;
  int n_gather;         // gather tasks pushed by the plan (mover slots after the router tasks)
  int gathers_done;
  int gemm_lo_total_dyn;  // low-priority GEMM tasks (the last d band's down tiles)
  unsigned long long gemm_lo_q[kShards];
  int bar_count, bar_gen;  // grid barrier of the static mode
  int pad[8];
};

struct Params {
  // problem
  int T, d, f, E, k, S;
  // tiling
  int pair;          // CTAs per worker: 1, or 2 (a cluster whose CTAs share each GEMM tile)
  int gather_cta_rows;  // permuted rows per gather task and CTA
  int bn_max;        // max tokens per GEMM tile (multiple of 32, <= 256)
  int stages;        // pipeline stages
  int stage_bytes;   // 2 * kABoxBytes + ceil(bn_max / pair / 32) * kBBoxBytes
  int n_ftiles;      // ceil(f / (128 pair)): each gate/up task covers 128 f rows per CTA
  int n_dtiles;      // ceil(d / (256 pair)): each down task covers 256 d rows per CTA
  int ks;            // split of the down projection's K (= f)
  int kb_down;       // k blocks (of 64) per down split
  int rt;            // tokens per router tile (kRouteTokens or kRouteTokensSmall)
  int n_route;       // router tiles
  int route_ks;      // K splits of a router tile
  int n_route_tasks; // ceil(n_route / pair) * route_ks (a task covers one tile per CTA)
  int n_workers;     // workers of the persistent grid (the cost model's N)
  int release;       // kReleaseAll or kReleaseExpert
  int prefetch;      // producer starts the next claimed GEMM tile's loads early
  int ct;            // tokens per combine tile
  int n_comb;        // combine tasks: combine tiles x d bands
  int n_bands;       // d bands of the down tiles and the combines (1 or 2)
  int dt_lo0;        // first d tile of the last band, whose down tiles have low priority
  int n_shared_groups;
  int n_static_gemm; // shared-expert gate/up tasks, ready at launch
  int y_f32;         // Y holds fp32 partial sums [ks][rows][d]; else bf16 [rows][d]
  int rows_y;        // rows of one Y partial (T*k + T*S)
  int max_groups;    // capacity of the group arrays
  int mover_seg, gemm_seg;  // ring capacity of one shard
  int fault_drop;    // -1, or the index of the GEMM completion to drop
  int fault_drop_type;   // 0, or a task type whose every dependency notification is dropped
  int fault_corrupt;     // 0, or a count the plan adds to the first expert's token count
  int fault_repush;      // -1, or the index of the gate/up completion whose task is pushed again
  int mover_override;
  int ahead_depth;   // claim the next task early when this many wait (0 = never)
  int index_order;   // the plan keeps experts in index order (not by count)
  int front_split;   // after the plan only mover workers prefer gathers (else every worker)
  int fold_gather;   // routed gate/up tiles gather their token rows from x themselves
  long long l2_pf_bytes;  // gate/up weight bytes prefetched into L2 at launch (0 = none)
  unsigned long long timeout_ns;
  // cost model constants
  float beta_move;   // bytes/s one mover CTA sustains
  float phi_gemm;    // FLOP/s one GEMM CTA sustains
  float hbm_bw;      // bytes/s of the whole device
  // inputs and output
  const __nv_bfloat16* x;
  const __nv_bfloat16* wr;
  const float* bias;
  const __nv_bfloat16* w_gate;  // [E+S, f, d] (the L2 prefetch reads its address)
  const __nv_bfloat16* w_up;
  __nv_bfloat16* out;
  // optional residual add + RMSNorm fused into the combine (all or none):
  // out = bf16(residual + layer), norm_out = bf16(out / rms(out) * gamma)
  const __nv_bfloat16* residual;  // [T, d]
  const __nv_bfloat16* gamma;     // [d]
  __nv_bfloat16* norm_out;        // [T, d]
  float eps;
  // routing workspace
  int* idx;          // [T, k]
  float* wgt;        // [T, k]
  int* rank;         // [T, k] rank of (t, j) among the tile's tokens of its expert
  int* tile_cnt;     // [n_route, E] per-tile counts, then exclusive prefix over tiles
  uint32_t* rmask;   // [n_route, E, 4] router tile: 128-bit mask of the tokens choosing e
  int* counts;       // [E]
  int* offsets;      // [E + 1]
  int* perm;         // [T * k]
  int* pos;          // [T, k]
  // activations
  __nv_bfloat16* Xp; // [T * k, d]
  __nv_bfloat16* H;  // [T * k + T * S, f]
  void* Y;           // bf16 [rows_y, d] or fp32 [ks, rows_y, d]
  // scheduler
  Group* groups;     // [max_groups]
  int* gather_done;  // [max_groups]
  int* gu_done;      // [max_groups]
  int* comb_done;    // [n_comb]
  int* norm_done;    // [n_comb / n_bands] bands of a combine tile written (fused RMSNorm)
  int* ring_mover;   // [kShards][mover_seg] task id + 1, 0 = not yet pushed
  int* ring_gemm;    // [kShards][gemm_seg]  task id + 1, 0 = not yet pushed
  int* ring_gemm_lo; // [kShards][gemm_seg]  the low-priority GEMM queue
  Sched* sched;
  // debug: one bit per task, set when the task is claimed (persistent mode);
  // null when off.  Bits [0, n_route_tasks) router tasks, then
  // claim_gather_off + g*8 + chunk, claim_gateup_off + the gate/up payload,
  // claim_down_off + the down payload, claim_comb_off + the combine payload.
  uint32_t* claimed;
  int claim_gather_off, claim_gateup_off, claim_down_off, claim_comb_off, claim_bits;
  float* rpart;      // [n_route][route_ks][128][E padded to 16] partial router logits
  int* rsplit_done;  // [n_route] router K splits finished
  unsigned long long* trace;  // [trace_cap][4] task trace records (or null)
  int trace_cap;
};

struct Maps {
  CUtensorMap wg;  // [(E+S) f, d], box 64 x 128
  CUtensorMap wu;  // [(E+S) f, d], box 64 x 128
  CUtensorMap wd;  // [(E+S) d, f], box 64 x 128
  CUtensorMap xp;  // [T k, d],      box 64 x 32
  CUtensorMap x;   // [T, d],        box 64 x 32
  CUtensorMap h;   // [T k + T S, f], box 64 x 32
  CUtensorMap xr;  // [T, d],        box 64 x 128 (router A operand)
  CUtensorMap wr;  // [E, d],        box 64 x 32  (router B operand)
};

}  // namespace moe
