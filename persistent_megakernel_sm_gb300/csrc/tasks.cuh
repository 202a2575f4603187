// Device-side tasks of the MoE-layer forward pass and the in-kernel scheduler.
//
// Every task is a __device__ function run by the CTA's kThreads compute
// threads, which synchronise on a named barrier.  The persistent megakernel
// (moe.cu) pulls task ids from three queues through its scheduler warp; the
// static megakernel runs them round-robin between grid barriers, and the
// multi-kernel ablation launches them one kernel per stage.
#pragma once

#include "layer.cuh"
#include "ptx.cuh"

namespace moe {

// Per-CTA control block, placed after the pipeline stages in shared memory.
struct Ctrl {
  uint64_t full_bar[8];   // (leader's are used) stage s loaded in both CTAs
  uint64_t empty_bar[8];  // stage s free again (the leader's MMAs commit to both CTAs')
  uint64_t acc_bar;       // the tile's accumulators are complete (committed to both CTAs')
  uint64_t tmem_empty;    // (leader's is used) the peer finished reading its TMEM, once per GEMM task
  uint64_t bfull_bar[8];  // (leader's are used) gathered token rows of stage s in every CTA
  unsigned long long deadline;
  unsigned long long t_claim, t_start;
  uint32_t tmem_base;
  int task;
  int flag;
  // mailbox between the scheduler warp and the compute warps (persistent
  // kernel): tasks posted to the compute warps (a ring of two: the running
  // task's slot and the next one), finished tasks handed back for their
  // notifications (a ring of two), and the sequence number of the task whose
  // late phase has begun (the scheduler claims the next task then)
  int mb_task[2];
  unsigned long long mb_tclaim[2];
  int mb_posted, mb_taken, mb_late;
  int mb_done_task[2];
  int mb_done, mb_handled;
  int mb_done_peer;       // (leader) tasks the peer CTA has finished
  int ival[8];
  int qbase[kShards];
  unsigned long long plan_t[8];  // plan phase timestamps (trace only)
  int pl_cb[kMaxE], pl_sib[kMaxE], pl_cpg[kMaxE];  // plan: per expert slot
  uint64_t gbar;                 // bulk-copy barrier of the gather
  uint64_t cbar[2];              // bulk-copy barriers of the combine (two buffers)
  alignas(16) float bias_s[kMaxE];
  // Scratch of one task at a time.  The router, plan, gather and combine
  // tasks use the named arrays; a GEMM task's epilogue (which never runs
  // beside them in one CTA) reuses the same bytes to stage its stores.
  union {
    struct {
      int tok[kThreads];      // token ids / combine tiles per row
      int cnt[kMaxE];         // per-expert counts
      int aux[kMaxE];
      int aux2[kMaxE];
      float wsum[kThreads];
      uint32_t mask[kMaxE * 4];  // router: 128-bit token mask per expert
    };
    alignas(16) char epi[kThreads / 32][kEpiBytes];  // one staging block per compute warp
  };
};

// Per-thread state that lives across tasks.
struct CtaState {
  int rank;             // cluster rank: 0 = the worker's leader (issues the MMAs), 1 = a pair's peer
  uint32_t bphase;      // MMA thread: parity bit per stage of the gathered-row barriers
  int worker;           // worker index (blockIdx.x / CTAs per worker)
  uint32_t lead_ctrl;   // the leader's Ctrl in the cluster's shared window (own for one CTA)
  uint32_t pipe_it;     // k blocks issued / consumed so far (producer & MMA thread)
  uint32_t gemm_count;  // GEMM tasks done (all threads)
  uint64_t deadline;    // globaltimer value after which waits give up
  int role_mover;       // 1 if this CTA prefers mover work (after the plan)
  uint32_t gather_phase;  // parity of the gather barrier (thread 0)
  uint32_t comb_phase;    // parities of the two combine barriers (bits 0, 1; all threads)
  int exit_reason;        // why the scheduler warp stopped (trace only): 1 done, 2 abort, 3 deadline
  unsigned polls;         // scheduler warp: claims that found nothing while idle (trace only)
  unsigned claims;        // scheduler warp: tasks claimed so far (rotates the home shard)
  bool plan_seen;         // scheduler warp: the plan's totals below are cached
  int n_gather, mover_total, gemm_total, gemm_lo_total;
  int pf_task, pf_count;  // producer: task whose first k blocks are already loading
  int taken;              // compute thread 0: tasks taken from the mailbox
};

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float* f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
  float fa[8], fb[8];
  bf16x8_to_f32(a, fa);
  bf16x8_to_f32(b, fb);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s = fmaf(fa[i], fb[i], s);
  return s;
}

__device__ __forceinline__ void set_status(const Params& p, int code, int info) {
  if (atomicCAS(&p.sched->status, 0, code) == 0) p.sched->err_info = info;
}

// Barriers of the kThreads compute threads (named barrier 1).  The persistent
// kernel adds a scheduler warp that never joins them, so task code must not
// use __syncthreads.
__device__ __forceinline__ void cta_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

__device__ __forceinline__ int cta_sync_and(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "n"(kThreads)
      : "memory");
  return r;
}

__device__ __forceinline__ int cta_sync_count(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.popc.u32 %0, 1, %2, p;\n\t}"
      : "=r"(r)
      : "r"(pred), "n"(kThreads)
      : "memory");
  return r;
}

// Release this CTA's global writes (generic and, for TMA readers, async
// proxy) before a dependency counter is bumped.  Called by every compute
// thread.
__device__ __forceinline__ void release_writes() {
  fence_proxy_async_global();
  __threadfence();
  cta_sync();
}

// Group descriptor: shared-expert groups [0, n_shared_groups) are known at
// launch and computed here (their tasks may run before the plan exists);
// routed groups are read from the plan's table.
__device__ __forceinline__ Group load_group(const Params& p, int g) {
  if (g < p.n_shared_groups) {
    const int t0 = g * p.bn_max;
    return Group{p.E, p.T * p.k + t0, min(p.bn_max, p.T - t0), t0, 0, p.n_shared_groups, 0, 0};
  }
  const int4 a = __ldcg(reinterpret_cast<const int4*>(p.groups + g));
  const int4 b = __ldcg(reinterpret_cast<const int4*>(p.groups + g) + 1);
  return Group{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
}

// d tiles [dt0, dt1) of d band `band` (down tiles of 256 rows of d each).
__device__ __forceinline__ int band_dt0(const Params& p, int band) { return band ? p.dt_lo0 : 0; }
__device__ __forceinline__ int band_dt1(const Params& p, int band) {
  return (p.n_bands == 2 && band == 0) ? p.dt_lo0 : p.n_dtiles;
}

__device__ __forceinline__ bool group_ok(const Params& p, const Group& G) {
  return G.nrows >= 1 && G.nrows <= p.bn_max && G.e >= 0 && G.e <= p.E && G.row0 >= 0 &&
         G.row0 + G.nrows <= p.rows_y && G.nsib >= 1 && G.sib0 >= 0 &&
         G.sib0 + G.nsib <= p.max_groups;
}

// ------------------------------------------------------------------ queues
// Three task queues (movers: router tiles, gathers, combines; GEMM workers:
// gate/up and down tiles; low priority: the last d band's down tiles), each
// split into kShards shards.  A shard is one
// 64-bit word -- claims so far (low 32 bits) and dynamic pushes (high 32 bits)
// -- plus a ring segment.  Pushes spread their tasks round-robin over the
// shards; a warp claims by loading every shard word of every queue at once
// and CAS-ing the word of one shard with work, starting at its home shard
// (blockIdx mod kShards) -- the per-SM local queues with stealing of
// xxqk.cn/news/665650 section 4.4 (pitfall 3), each shared by a few CTAs.
// A CAS never takes a slot that has not been pushed, so a claimer never
// waits on work that does not exist yet; sharding keeps the number of CTAs
// contending for one word small.  Tasks known at launch (router tiles,
// shared-expert gate/up tiles) are implicit: static index s lives in shard
// s mod kShards at local slot s / kShards.  Ring entries hold task id + 1
// (0 = not yet written), so one zero memset resets a queue.

struct QueueRef {
  unsigned long long* word;  // [kShards]
  int* ring;                 // [kShards][seg]
  int n_static;
  int seg;
};

__device__ __forceinline__ QueueRef mover_queue(const Params& p) {
  return QueueRef{p.sched->mover_q, p.ring_mover, p.n_route_tasks, p.mover_seg};
}

__device__ __forceinline__ QueueRef gemm_queue(const Params& p) {
  return QueueRef{p.sched->gemm_q, p.ring_gemm, p.n_static_gemm, p.gemm_seg};
}

// Low-priority GEMM queue: the down tiles of the last d band, taken when the
// GEMM queue is empty, so the combines of the other bands can start while
// these still run.
__device__ __forceinline__ QueueRef gemm_lo_queue(const Params& p) {
  return QueueRef{p.sched->gemm_lo_q, p.ring_gemm_lo, 0, p.gemm_seg};
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int shard_static(int n_static, int j) {
  return n_static > j ? (n_static - j + kShards - 1) / kShards : 0;
}

// Tasks i in [0, n) of a push go to shard (r0 + i) mod kShards, at local
// index base_j + i / kShards; shard j receives push_count(n, r0, j) of them.
__device__ __forceinline__ int push_count(int n, int r0, int j) {
  const int off = (j - r0 + kShards) % kShards;
  return off < n ? (n - off + kShards - 1) / kShards : 0;
}

__device__ __forceinline__ int push_start(int key) {
  return (int)(((unsigned)key * 2654435761u) >> 16) & (kShards - 1);
}

// Push the n tasks id_of(i).  Called by all 32 lanes of one warp.
template <class F>
__device__ __forceinline__ void push_gen_warp(const Params& p, const QueueRef& q, int n, F id_of) {
  const int lane = threadIdx.x & 31;
  if (n <= 0) return;
  const int r0 = push_start(id_of(0));
  int base = 0;
  if (lane < kShards) {
    const int cnt = push_count(n, r0, lane);
    if (cnt > 0) {
      base = (int)(atomicAdd(q.word + lane, (unsigned long long)cnt << 32) >> 32);
      if (base + cnt > q.seg) set_status(p, MOE_E_DEVICE, 1);
    }
  }
  for (int i0 = 0; i0 < n; i0 += 32) {  // whole-warp rounds: every lane shuffles
    const int i = i0 + lane;
    const int j = (r0 + i) & (kShards - 1);
    const int bj = __shfl_sync(0xffffffffu, base, j);
    if (i < n && bj + i / kShards < q.seg)
      st_release(q.ring + j * q.seg + bj + i / kShards, id_of(i) + 1);
  }
}

// Push by the whole CTA (every thread calls it).
template <class F>
__device__ __forceinline__ void push_gen_block(const Params& p, const QueueRef& q, int n, F id_of,
                                               Ctrl* c) {
  if (n <= 0) return;
  const int r0 = push_start(id_of(0));
  if (threadIdx.x < kShards) {
    const int cnt = push_count(n, r0, threadIdx.x);
    int base = 0;
    if (cnt > 0) {
      base = (int)(atomicAdd(q.word + threadIdx.x, (unsigned long long)cnt << 32) >> 32);
      if (base + cnt > q.seg) set_status(p, MOE_E_DEVICE, 1);
    }
    c->qbase[threadIdx.x] = base;
  }
  cta_sync();
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const int j = (r0 + i) & (kShards - 1);
    const int slot = c->qbase[j] + i / kShards;
    if (slot < q.seg) st_release(q.ring + j * q.seg + slot, id_of(i) + 1);
  }
}

// Task of local slot `h` of shard `j`: implicit static task or ring entry
// (waited for: the slot was reserved, its entry may still be in flight).
// Returns the task id, or -3 on abort.  One lane only.
__device__ int resolve_slot(const Params& p, const QueueRef& q, bool is_mover, int j, int h,
                            uint64_t deadline) {
  const int nst = shard_static(q.n_static, j);
  if (h < nst) {
    const int sidx = h * kShards + j;
    if (is_mover) return task_id(kTaskRoute, sidx);
    const int nsg = p.n_shared_groups;  // shared-expert gate/up tiles, f-tile major
    return task_id(kTaskGateUp, (sidx % nsg) * p.n_ftiles + sidx / nsg);
  }
  const int* e = q.ring + j * q.seg + (h - nst);
  int v;
  while ((v = ld_acquire(e)) == 0) {
    if (ld_relaxed(&p.sched->status) != 0) return -3;
    if (globaltimer() > deadline) {
      set_status(p, MOE_E_TIMEOUT, 2);
      return -3;
    }
  }
  return v - 1;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One scheduling decision, by a whole warp: the preferred queue first, then
// the other ones.  Returns a task id (the same on every lane), -1 if nothing
// is claimable now, -2 if every queue is finished, -3 to abort, -4 to retry
// at once (the CAS kept losing).  `min_depth` > 1 claims ahead: only from the
// first-choice queue and only when it holds at least that many tasks.
__device__ int claim_once(const Params& p, CtaState& st, int min_depth) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  Sched* s = p.sched;
  if (!st.plan_seen) {  // lane 0 reads, every lane takes its values: decisions stay uniform
    int seen = 0, nm = 0, ng = 0, mt = 0, gt = 0, lt = 0;
    if (lane == 0 && ld_acquire(&s->plan_done) != 0) {
      seen = 1;
      nm = ld_relaxed(&s->n_movers);
      ng = ld_relaxed(&s->n_gather);
      mt = ld_relaxed(&s->mover_total_dyn);
      gt = ld_relaxed(&s->gemm_total_dyn);
      lt = ld_relaxed(&s->gemm_lo_total_dyn);
    }
    if (__shfl_sync(full, seen, 0)) {
      st.plan_seen = true;
      st.role_mover = st.worker < __shfl_sync(full, nm, 0);
      st.n_gather = __shfl_sync(full, ng, 0);
      st.mover_total = __shfl_sync(full, mt, 0);
      st.gemm_total = __shfl_sync(full, gt, 0);
      st.gemm_lo_total = __shfl_sync(full, lt, 0);
    }
  }
  // lanes 0-7: the mover queue's shards, 8-15: the GEMM queue's, 16-23: the
  // low-priority GEMM queue's (lanes 24-31 idle)
  const int qi = lane >> 3;
  const bool mine = qi < 3;
  const int j = lane & (kShards - 1);
  const QueueRef q = qi == 0 ? mover_queue(p) : qi == 1 ? gemm_queue(p) : gemm_lo_queue(p);
  unsigned long long w = 0;
  if (mine) w = ld_acquire_u64(q.word + j);
  const int nst = mine ? shard_static(q.n_static, j) : 0;
  const int h = (int)(w & 0xffffffffu);
  const int avail = nst + (int)(w >> 32);
  const int claimed_m = warp_sum_i(qi == 0 ? h : 0);
  const int claimed_g = warp_sum_i(qi == 1 ? h : 0);
  const int claimed_l = warp_sum_i(qi == 2 ? h : 0);
  const int dep = mine ? max(avail - h, 0) : 0;
  const int depth_m = warp_sum_i(qi == 0 ? dep : 0);
  const int depth_g = warp_sum_i(qi == 1 ? dep : 0);
  const int depth_l = warp_sum_i(qi == 2 ? dep : 0);
  const unsigned ball = __ballot_sync(full, mine && h < avail);
  const bool gathers_left = st.plan_seen && claimed_m < p.n_route_tasks + st.n_gather;
  // Before the plan every worker prefers router tiles: they gate all the
  // GEMM work.  After it, a mover worker takes mover, GEMM, low-priority GEMM
  // work in that order, a GEMM worker GEMM, low-priority GEMM, mover work --
  // so with the spatial split of the front (p.front_split) the GEMM workers
  // run the tiles that are ready (the shared expert's, then each expert's as
  // its gathers land) while the mover workers gather, and take gathers only
  // when no GEMM tile is ready.  Without it every worker prefers gathers
  // while any is unclaimed.
  const bool mover_first =
      !st.plan_seen || (gathers_left && !p.front_split) || st.role_mover;
  const int npass = min_depth > 1 ? 1 : 3;
  // Home shard: fixed for the first multiple of kShards workers; the rest
  // (4 of the 76 CTA pairs of a pair layer) move to the next shard after
  // every claim.  Fixed homes alone drained the shards unevenly (10 home
  // workers on some shards, 9 on others), and tasks pushed together -- an
  // expert's sibling row groups, which read the same weight tiles -- drifted
  // apart by far more than a weight tile stays in L2; moving every worker's
  // home scattered each worker's consecutive claims instead.
  const int fixed = p.n_workers & ~(kShards - 1);
  const int home = (st.worker < fixed ? st.worker : st.worker + (int)st.claims) & (kShards - 1);
  for (int pass = 0; pass < npass; ++pass) {
    const int qq = mover_first ? pass : (pass == 2 ? 0 : pass + 1);
    const int depth = qq == 0 ? depth_m : qq == 1 ? depth_g : depth_l;
    if (depth < max(min_depth, 1)) continue;
    const unsigned sm = (ball >> (qq * kShards)) & ((1u << kShards) - 1u);
    if (!sm) continue;
    // first shard with work at or after the home shard
    const unsigned rot = ((sm >> home) | (sm << (kShards - home))) & ((1u << kShards) - 1u);
    const int pick = (home + __ffs(rot) - 1) & (kShards - 1);
    const int plane = qq * kShards + pick;
    int r = -4;
    if (lane == plane) {
      // a lost CAS returns the word's current value: retry on it at once
      // while the shard still holds work (no reload of the other words)
      unsigned long long cur = w;
      for (int attempt = 0; attempt < 8; ++attempt) {
        const unsigned long long seen = atomicCAS(q.word + pick, cur, cur + 1);
        if (seen == cur) {
          r = resolve_slot(p, q, qq == 0, pick, (int)(cur & 0xffffffffu), st.deadline);
          break;
        }
        cur = seen;
        if ((int)(cur & 0xffffffffu) >= nst + (int)(cur >> 32)) break;  // drained
      }
    }
    r = __shfl_sync(full, r, plane);
    if (r >= 0) ++st.claims;
    if (r >= 0 && pass > 0 && st.plan_seen && lane == 0) atomicAdd(&s->stat_stolen, 1);
    return r;  // a task, -3, or -4 (the shard drained under us: retry)
  }
  const QueueRef mq = mover_queue(p), gq = gemm_queue(p);
  const bool fin_m = st.plan_seen && claimed_m >= mq.n_static + st.mover_total;
  const bool fin_g = st.plan_seen && claimed_g >= gq.n_static + st.gemm_total;
  const bool fin_l = st.plan_seen && claimed_l >= st.gemm_lo_total;
  if (npass == 3 && fin_m && fin_g && fin_l) return -2;
  const int bad = lane == 0 ? ld_relaxed(&s->status) : 0;
  if (__shfl_sync(full, bad, 0) != 0) return -3;
  return -1;
}

// ------------------------------------------------------------------ plan
// Block-wide exclusive scan of one int per thread (blockDim = 256).
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, Ctrl* c) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  cta_sync();
  if (lane == 31) c->ival[warp] = x;
  cta_sync();
  int wbase = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int s = c->ival[w];
    if (w < warp) wbase += s;
    tot += s;
  }
  cta_sync();
  *total = tot;
  return wbase + x - v;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Rows of a gate/up task's f tile, a down task's d tile and a gather task,
// over the worker's CTAs.
__device__ __forceinline__ int ftile_rows(const Params& p) { return kBM * p.pair; }
__device__ __forceinline__ int dtile_rows(const Params& p) { return 2 * kBM * p.pair; }
__device__ __forceinline__ int gather_rows(const Params& p) { return p.gather_cta_rows * p.pair; }

// Number of gather tasks of a group.
__device__ __forceinline__ int gather_chunks(const Params& p, int nrows) {
  return ceil_div(nrows, gather_rows(p));
}

// The plan: runs once, on the CTA that finished the last router tile (or as
// its own kernel in the ablation).  Counts and offsets per expert, the
// canonical permutation (experts ascending, tokens ascending), the GEMM row
// groups (experts in order of decreasing count, each split into balanced
// tiles of at most bn_max rows), the cost-model split of CTAs into movers and
// GEMM workers, and (persistent mode) the first pushes: every gather task.
__device__ void plan_task(const Params& p, char* scratch, Ctrl* c, bool push) {
  const int E = p.E, k = p.k, tid = threadIdx.x;
  int* cnt = c->cnt;     // counts per expert
  int* order = c->aux;   // experts by decreasing count
  int* offs = c->aux2;   // offsets per expert

  if (threadIdx.x == 0) c->plan_t[0] = globaltimer();
  // per expert: exclusive prefix of the router tiles' counts (the tile bases)
  // and the total; in shared memory when the [tiles, E] table fits
  const int ntile = p.n_route;
  const bool in_smem = (size_t)ntile * E * 4 <= (size_t)p.stages * p.stage_bytes;
  int* tb = in_smem ? reinterpret_cast<int*>(scratch) : p.tile_cnt;
  if (in_smem) {  // E is a multiple of 4 or the table is small: int4 where aligned
    const int n = ntile * E;
    if ((n & 3) == 0) {
      const int4* src = reinterpret_cast<const int4*>(p.tile_cnt);
      int4* dst = reinterpret_cast<int4*>(tb);
#pragma unroll 8
      for (int i = tid; i < n / 4; i += kThreads) dst[i] = __ldcg(src + i);
    } else {
      for (int i = tid; i < n; i += kThreads) tb[i] = __ldcg(p.tile_cnt + i);
    }
    cta_sync();
  }
  if (tid < E) {
    int run = 0;
    for (int tau = 0; tau < ntile; ++tau) {
      int* q = tb + (size_t)tau * E + tid;
      const int v = in_smem ? *q : __ldcg(q);
      *q = run;
      run += v;
    }
    cnt[tid] = run;
    p.counts[tid] = run;
  }
  if (in_smem) {  // the gathers read the tile bases from global memory
    cta_sync();
    const int n = ntile * E;
    for (int i = tid; i < n; i += kThreads) p.tile_cnt[i] = tb[i];
  }
  // fault injection (host-set): a wrong count, which the check below catches
  if (tid == 0 && p.fault_corrupt != 0) cnt[0] += p.fault_corrupt;
  cta_sync();
  if (threadIdx.x == 0) c->plan_t[1] = globaltimer();
  int total = 0;
  const int off = block_exclusive_scan(tid < E ? cnt[tid] : 0, &total, c);
  // every token chose k experts: the counts must add up to T k
  if (total != p.T * k) {
    if (tid == 0) set_status(p, MOE_E_DEVICE, 9);
    return;
  }
  if (tid < E) {
    p.offsets[tid] = off;
    offs[tid] = off;
  }
  if (tid == 0) p.offsets[E] = total;
  if (threadIdx.x == 0) c->plan_t[2] = globaltimer();
  // experts ordered by (count desc, expert asc), or by index when the first
  // experts' gate/up weights are being prefetched into L2
  if (tid < E && p.index_order) order[tid] = tid;
  if (tid < E && !p.index_order) {
    const int me = cnt[tid];
    int r = 0;
#pragma unroll 8
    for (int e2 = 0; e2 < E; ++e2) {
      const int o = cnt[e2];
      r += (o > me) || (o == me && e2 < tid);
    }
    order[r] = tid;
  }
  cta_sync();
  if (threadIdx.x == 0) c->plan_t[3] = globaltimer();
  // groups: order slot r -> expert order[r]
  int e_r = tid < E ? order[tid] : 0;
  int n_r = tid < E ? cnt[e_r] : 0;
  int nmt = n_r > 0 ? ceil_div(n_r, p.bn_max) : 0;
  int n_routed = 0;
  const int gfirst = block_exclusive_scan(nmt, &n_routed, c);
  // gather-task prefix in group order
  int rows_per = nmt > 0 ? ((ceil_div(n_r, nmt) + 15) / 16) * 16 : 0;
  int my_chunks = 0;
  for (int m = 0; m < nmt; ++m) my_chunks += gather_chunks(p, min(rows_per, n_r - m * rows_per));
  int n_gather = 0;
  const int chunk_base = block_exclusive_scan(my_chunks, &n_gather, c);
  const int off_e = tid < E ? offs[e_r] : 0;
  if (p.n_shared_groups + n_routed > p.max_groups) {
    if (tid == 0) set_status(p, MOE_E_DEVICE, 4);
    return;
  }
  // routed groups follow the shared-expert groups (see load_group)
  const int sib0 = p.n_shared_groups + gfirst;
  for (int m = 0; m < nmt; ++m) {
    const int nrows = min(rows_per, n_r - m * rows_per);
    const int row0 = off_e + m * rows_per;
    p.groups[sib0 + m] = Group{e_r, row0, nrows, row0, sib0, nmt, my_chunks, off_e};
  }
  if (push) {
    // gather i of the layer: the expert slot whose chunk range holds i, then
    // the group (every group of a slot but its last is full) and the chunk;
    // written by all threads, shard i mod kShards, local slot i / kShards
    if (tid < E) {
      c->pl_cb[tid] = chunk_base;
      c->pl_sib[tid] = sib0;
      c->pl_cpg[tid] = rows_per > 0 ? gather_chunks(p, rows_per) : 1;
    }
    cta_sync();
    for (int i = tid; i < n_gather; i += kThreads) {
      int lo = 0, hi = E - 1;  // last slot whose chunk base is <= i
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (c->pl_cb[mid] <= i) lo = mid;
        else hi = mid - 1;
      }
      const int local = i - c->pl_cb[lo];
      const int m = local / c->pl_cpg[lo], q = local - m * c->pl_cpg[lo];
      if ((i / kShards) < p.mover_seg)
        p.ring_mover[(i & (kShards - 1)) * p.mover_seg + i / kShards] =
            task_id(kTaskGather, (c->pl_sib[lo] + m) * 8 + q) + 1;
    }
  }
  cta_sync();
  if (threadIdx.x == 0) c->plan_t[4] = c->plan_t[5] = globaltimer();
  // cost model (spatial split): CTA-seconds of mover work against GEMM work
  const int touched_routed = cta_sync_count(tid < E && cnt[tid] > 0);
  if (tid == 0) {
    const int n_groups = p.n_shared_groups + n_routed;
    const int n_down = p.n_dtiles * p.ks;
    const int n_down_lo = p.n_bands == 2 ? (p.n_dtiles - p.dt_lo0) * p.ks : 0;
    Sched* s = p.sched;
    s->n_groups = n_groups;
    s->gemm_total_dyn = n_routed * p.n_ftiles + n_groups * (n_down - n_down_lo);
    s->gemm_lo_total_dyn = n_groups * n_down_lo;
    s->mover_total_dyn = n_gather + p.n_comb;
    s->n_gather = n_gather;
    int movers;
    const int N = p.n_workers;
    if (p.mover_override > 0) {
      movers = min(p.mover_override, max(N - 1, 1));
    } else {
      const float ybytes = p.y_f32 ? 4.f * p.ks : 2.f;
      const float Tk = (float)p.T * k;
      const float b_move = Tk * p.d * 2.f * 2.f +                     // gather: read + write
                           ((float)p.T * (k + p.S)) * p.d * ybytes +  // combine reads
                           (float)p.T * p.d * 2.f;                    // combine writes
      const int touched = p.S + touched_routed;
      const float flops = 6.f * (Tk + (float)p.T * p.S) * p.d * p.f;
      const float wbytes = (float)touched * 3.f * p.f * p.d * 2.f;
      const float a = b_move / p.beta_move;                            // CTA-seconds
      const float b = fmaxf(flops / p.phi_gemm, (float)N * wbytes / p.hbm_bw);
      movers = __float2int_rn((float)N * a / (a + b));
      movers = max(1, min(movers, max(N - 1, 1)));
    }
    s->n_movers = movers;
  }
  if (threadIdx.x == 0) c->plan_t[6] = globaltimer();
  if (push) {
    release_writes();
    if (tid < kShards) {
      const int cnt = push_count(n_gather, 0, tid);
      if (cnt > p.mover_seg) set_status(p, MOE_E_DEVICE, 8);
      if (cnt > 0) atomicAdd(p.sched->mover_q + tid, (unsigned long long)cnt << 32);
    }
    cta_sync();
    if (tid == 0) {
      __threadfence();
      st_release(&p.sched->plan_done, 1);
    }
  } else {
    cta_sync();
  }
}

// ------------------------------------------------------------------ gather (mover)
// Xp[row, :] = x[perm[row], :] for up to 32 or 64 rows per CTA of the worker of one
// group, of which this CTA takes part `half` of `nhalf` (the CTAs of a pair
// split the rows).
// One thread moves whole rows with bulk copies through shared memory (global
// -> shared on an mbarrier, then shared -> global), as many rows per round as
// the pipeline stages hold, so hundreds of KB are in flight per SM.
__device__ void gather_task(const Params& p, int g, int chunk, int half, int nhalf, char* smem,
                            Ctrl* c, CtaState& st) {
  const Group G = load_group(p, g);
  const int grows = gather_rows(p);
  if (!group_ok(p, G) || chunk * grows >= G.nrows) {
    if (threadIdx.x == 0) set_status(p, MOE_E_DEVICE, 20);
    return;
  }
  const int nr_chunk = min(grows, G.nrows - chunk * grows);
  const int per = ceil_div(nr_chunk, nhalf);
  const int row_lo = min(nr_chunk, half * per);
  const int r0 = G.row0 + chunk * grows + row_lo;
  const int nr = min(nr_chunk, row_lo + per) - row_lo;
  // Permuted row r of expert e is the (r - off_e)-th token of e in router-tile
  // order: the tile tau with base[tau][e] <= r - off_e < base[tau+1][e], and
  // inside it the token of the (r - off_e - base[tau][e])-th set bit of the
  // tile's mask of e.  This writes perm[r] and pos[t, j] for the chunk's rows.
  int* col = c->aux;  // base[tau][e] for all router tiles tau
  for (int tau = threadIdx.x; tau < p.n_route; tau += kThreads)
    col[tau] = __ldcg(p.tile_cnt + (size_t)tau * p.E + G.e);
  cta_sync();
  if (threadIdx.x < nr) {
    const int r = r0 + threadIdx.x;
    const int local = r - G.pad;
    int lo = 0, hi = p.n_route - 1;  // last tile whose base <= local
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (col[mid] <= local) lo = mid;
      else hi = mid - 1;
    }
    int rank = local - col[lo];
    const uint4 mk = __ldcg(reinterpret_cast<const uint4*>(p.rmask) + (size_t)lo * p.E + G.e);
    const uint32_t words[4] = {mk.x, mk.y, mk.z, mk.w};
    int bit = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int pc = __popc(words[q]);
      if (rank >= 0 && rank < pc) {
        uint32_t wv = words[q];
        for (int z = 0; z < rank; ++z) wv &= wv - 1u;  // drop the lowest set bits
        bit = q * 32 + __ffs(wv) - 1;
      }
      rank -= pc;
    }
    const int t = lo * p.rt + bit;
    c->tok[threadIdx.x] = t;
    p.perm[r] = t;
    for (int j = 0; j < p.k; ++j)
      if (__ldcg(p.idx + (size_t)t * p.k + j) == G.e) p.pos[(size_t)t * p.k + j] = r;
  }
  cta_sync();
  // folded gathers: the gate/up tiles read the token rows of x through perm
  if (threadIdx.x == 0 && (nr <= 0 || p.fold_gather)) st_release_cta_shared(&c->mb_late, st.taken);
  if (threadIdx.x == 0 && nr > 0 && !p.fold_gather) {
    const uint32_t row_bytes = (uint32_t)p.d * 2;
    const int cap = max(1, (int)(((size_t)p.stages * p.stage_bytes) / row_bytes));
    fence_proxy_async_shared();
    for (int r = 0; r < nr; r += cap) {
      const int n = min(cap, nr - r);
      if (r + cap >= nr) st_release_cta_shared(&c->mb_late, st.taken);  // last round
      mbar_arrive_expect_tx(&c->gbar, (uint32_t)n * row_bytes);
      for (int i = 0; i < n; ++i)
        bulk_load(smem + (size_t)i * row_bytes, p.x + (size_t)c->tok[r + i] * p.d, row_bytes,
                  &c->gbar);
      if (!mbar_wait(&c->gbar, st.gather_phase, st.deadline)) {
        set_status(p, MOE_E_TIMEOUT, 21);
        break;
      }
      st.gather_phase ^= 1u;
      for (int i = 0; i < n; ++i)
        bulk_store(p.Xp + (size_t)(r0 + r + i) * p.d, smem + (size_t)i * row_bytes, row_bytes);
      bulk_commit();
      bulk_wait_read_all();
    }
    bulk_wait_all();
  }
}

// ------------------------------------------------------------------ combine (mover)
// acc += residual[t, 8v .. 8v+7] (the residual add fused into the combine).
__device__ __forceinline__ void add_residual(const Params& p, int t, int v, float* acc) {
  float r[8];
  bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(p.residual) + (size_t)t * (p.d >> 3) + v), r);
#pragma unroll
  for (int u = 0; u < 8; ++u) acc[u] += r[u];
}

// Combine straight from global memory (rows too large for shared memory):
// columns [c0, c0 + 8 * nvec) of tokens [t0, t0 + nt).
__device__ void combine_direct(const Params& p, int t0, int nt, int c0, int nvec, Ctrl* c) {
  const int k = p.k, nsrc = k + p.S;
  const int dvec = p.d >> 3;
  uint4* out = reinterpret_cast<uint4*>(p.out) + (c0 >> 3);
  const float* Yf = reinterpret_cast<const float*>(p.Y) + c0;
  const uint4* Yb = reinterpret_cast<const uint4*>(p.Y) + (c0 >> 3);
  const size_t part = (size_t)p.rows_y * p.d;
  for (int i = threadIdx.x; i < nt * nvec; i += kThreads) {
    const int t = i / nvec, q = i - t * nvec;
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    for (int j = 0; j < nsrc; ++j) {
      const int row = j < k ? c->tok[t * k + j] : p.T * k + t0 + t;
      const float w = j < k ? c->wsum[t * k + j] : 1.f;
      float y[8];
      if (p.y_f32) {
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] = 0.f;
        for (int s = 0; s < p.ks; ++s) {
          const float4* src =
              reinterpret_cast<const float4*>(Yf + s * part + (size_t)row * p.d + q * 8);
          const float4 a = __ldcg(src), b = __ldcg(src + 1);
          y[0] += a.x; y[1] += a.y; y[2] += a.z; y[3] += a.w;
          y[4] += b.x; y[5] += b.y; y[6] += b.z; y[7] += b.w;
        }
      } else {
        bf16x8_to_f32(__ldcg(Yb + (size_t)row * dvec + q), y);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = fmaf(w, y[u], acc[u]);
    }
    if (p.residual) add_residual(p, t0 + t, (c0 >> 3) + q, acc);
    out[(size_t)(t0 + t) * dvec + q] = f32x8_to_bf16(acc);
  }
}

// out[t, :] = bf16( sum_j w[t,j] * Y[pos[t,j], :] + Y[T k + t, :] (shared) ),
// fp32 sum in slot order, then the shared expert; with fp32 K-split partials
// each source row is the sum of its splits.  One task covers a tile of
// tokens and one d band (the columns of the band's down tiles).  The source
// rows of a few tokens at a time are bulk-copied into one half of the
// pipeline's shared memory while the other half is being summed (double
// buffering).  This CTA takes part `part` of `nparts` of the tile's tokens
// (the two CTAs of a pair split them).
__device__ void combine_band(const Params& p, int ci, int part, int nparts, char* smem, Ctrl* c,
                             CtaState& st) {
  const int ctile = ci / p.n_bands, band = ci - ctile * p.n_bands;
  const int c0 = band_dt0(p, band) * dtile_rows(p);
  const int c1 = min(p.d, band_dt1(p, band) * dtile_rows(p));
  const int tt0 = ctile * p.ct;
  const int nt_tile = min(p.ct, p.T - tt0);
  const int per = ceil_div(nt_tile, nparts);
  const int tok_lo = min(nt_tile, part * per);
  const int t0 = tt0 + tok_lo;
  const int nt = min(nt_tile, tok_lo + per) - tok_lo;
  const int k = p.k;
  if (nt <= 0) {
    if (threadIdx.x == 0) st_release_cta_shared(&c->mb_late, st.taken);
    return;
  }
  for (int i = threadIdx.x; i < nt * k; i += kThreads) {
    c->tok[i] = __ldcg(p.pos + (size_t)t0 * k + i);
    c->wsum[i] = __ldcg(p.wgt + (size_t)t0 * k + i);
  }
  cta_sync();
  const int nsrc = k + p.S;
  const int nsplit = p.y_f32 ? p.ks : 1;
  const int ebytes = p.y_f32 ? 4 : 2;
  const uint32_t row_bytes = (uint32_t)(c1 - c0) * ebytes;  // one source row's band
  // a token's block: its source rows, then (fused residual) its residual row
  const uint32_t res_bytes = p.residual ? (uint32_t)(c1 - c0) * 2 : 0u;
  const size_t src_bytes = (size_t)nsrc * nsplit * row_bytes;
  const size_t per_tok = src_bytes + res_bytes;
  const size_t mem = (size_t)p.stages * p.stage_bytes;
  if (per_tok > mem) {  // one token's rows do not fit: sum straight from global
    if (threadIdx.x == 0) st_release_cta_shared(&c->mb_late, st.taken);
    combine_direct(p, t0, nt, c0, (c1 - c0) >> 3, c);
    return;
  }
  const int nbuf = per_tok * 2 <= mem ? 2 : 1;
  const size_t half = mem / nbuf;          // bytes of one buffer
  const int tpr = (int)(half / per_tok);   // tokens per round
  const int rounds = (nt + tpr - 1) / tpr;
  const size_t part_bytes = (size_t)p.rows_y * p.d * ebytes;
  const size_t y_row = (size_t)p.d * ebytes;
  const char* Yb = reinterpret_cast<const char*>(p.Y) + (size_t)c0 * ebytes;
  auto issue = [&](int r) {  // thread 0: bulk loads of round r into buffer r % nbuf
    const int b = r % nbuf;
    const int ta = r * tpr, n = min(tpr, nt - ta);
    char* buf = smem + b * half;
    mbar_arrive_expect_tx(&c->cbar[b], (uint32_t)(n * per_tok));
    for (int tt = 0; tt < n; ++tt) {
      const int t = ta + tt;
      for (int j = 0; j < nsrc; ++j) {
        const int row = j < k ? c->tok[t * k + j] : p.T * k + t0 + t;
        for (int s = 0; s < nsplit; ++s)
          bulk_load(buf + (size_t)tt * per_tok + (size_t)(j * nsplit + s) * row_bytes,
                    Yb + s * part_bytes + (size_t)row * y_row, row_bytes, &c->cbar[b]);
      }
      if (res_bytes)
        bulk_load(buf + (size_t)tt * per_tok + src_bytes,
                  p.residual + (size_t)(t0 + t) * p.d + c0, res_bytes, &c->cbar[b]);
    }
  };
  if (threadIdx.x == 0) {
    fence_proxy_async_shared();
    issue(0);
    if (nbuf == 2 && rounds > 1) issue(1);
  }
  const int nvec = (c1 - c0) >> 3, dvec = p.d >> 3;
  uint4* out = reinterpret_cast<uint4*>(p.out) + (c0 >> 3);
  for (int r = 0; r < rounds; ++r) {
    const int b = r % nbuf;
    if (threadIdx.x == 0 && r == rounds - 1) st_release_cta_shared(&c->mb_late, st.taken);
    const bool got = mbar_wait(&c->cbar[b], (st.comb_phase >> b) & 1u, st.deadline);
    st.comb_phase ^= 1u << b;
    if (!cta_sync_and(got ? 1 : 0)) {
      if (threadIdx.x == 0) set_status(p, MOE_E_TIMEOUT, 24);
      return;
    }
    const int ta = r * tpr, n = min(tpr, nt - ta);
    const char* buf = smem + b * half;
    for (int i = threadIdx.x; i < n * nvec; i += kThreads) {
      const int tt = i / nvec, q = i - tt * nvec;
      const int t = ta + tt;
      float acc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = 0.f;
      for (int j = 0; j < nsrc; ++j) {
        const float w = j < k ? c->wsum[t * k + j] : 1.f;
        const char* src = buf + (size_t)tt * per_tok + (size_t)j * nsplit * row_bytes;
        float y[8];
        if (p.y_f32) {
#pragma unroll
          for (int u = 0; u < 8; ++u) y[u] = 0.f;
          for (int s = 0; s < nsplit; ++s) {
            const float4* v = reinterpret_cast<const float4*>(src + s * row_bytes) + 2 * q;
            const float4 a = v[0], bb = v[1];
            y[0] += a.x; y[1] += a.y; y[2] += a.z; y[3] += a.w;
            y[4] += bb.x; y[5] += bb.y; y[6] += bb.z; y[7] += bb.w;
          }
        } else {
          bf16x8_to_f32(reinterpret_cast<const uint4*>(src)[q], y);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = fmaf(w, y[u], acc[u]);
      }
      if (res_bytes) {
        float rv[8];
        bf16x8_to_f32(reinterpret_cast<const uint4*>(buf + (size_t)tt * per_tok + src_bytes)[q], rv);
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] += rv[u];
      }
      out[(size_t)(t0 + t) * dvec + q] = f32x8_to_bf16(acc);
    }
    cta_sync();  // buffer b is free again
    if (threadIdx.x == 0 && r + nbuf < rounds) issue(r + nbuf);
  }
}

// The RMSNorm of the combine tile's tokens, once every band of the tile has
// written its columns of out (the residual stream, bf16): per token,
// norm_out = bf16(out * rsqrt(mean(out^2) + eps) * gamma), the mean over the
// d stored values.  One warp per token (lanes stride the row, then a fixed
// butterfly), eight tokens at a time.
__device__ void norm_tile(const Params& p, int ctile) {
  const int t0 = ctile * p.ct, nt = min(p.ct, p.T - t0);
  const int nvec = p.d >> 3, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* o4 = reinterpret_cast<const uint4*>(p.out);
  const uint4* g4 = reinterpret_cast<const uint4*>(p.gamma);
  uint4* n4 = reinterpret_cast<uint4*>(p.norm_out);
  for (int tt = warp; tt < nt; tt += kThreads / 32) {
    const size_t row = (size_t)(t0 + tt) * nvec;
    float ss = 0.f;
#pragma unroll 4
    for (int q = lane; q < nvec; q += 32) {
      float h[8];
      bf16x8_to_f32(__ldcg(o4 + row + q), h);
#pragma unroll
      for (int u = 0; u < 8; ++u) ss = fmaf(h[u], h[u], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss / (float)p.d + p.eps);
#pragma unroll 4
    for (int q = lane; q < nvec; q += 32) {
      float h[8], g[8], v[8];
      bf16x8_to_f32(__ldcg(o4 + row + q), h);
      bf16x8_to_f32(__ldg(g4 + q), g);
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = h[u] * inv * g[u];
      n4[row + q] = f32x8_to_bf16(v);
    }
  }
}

// One combine task: tile ci / n_bands, band ci % n_bands, this CTA's part
// `half` of `nhalf` of its tokens.  With the fused residual + RMSNorm, the CTA
// whose part completes the tile (a counter per tile: every band, every part)
// then runs the norm of the whole tile.
__device__ void combine_task(const Params& p, int ci, int half, int nhalf, char* smem, Ctrl* c,
                             CtaState& st) {
  combine_band(p, ci, half, nhalf, smem, c, st);
  if (!p.norm_out) return;
  const int ctile = ci / p.n_bands;
  release_writes();
  if (threadIdx.x == 0)
    c->flag = atom_add_acq_rel(p.norm_done + ctile, 1) + 1 == p.n_bands * nhalf;
  cta_sync();
  if (!c->flag) return;
  fence_acq_rel_gpu();
  norm_tile(p, ctile);
}

// ------------------------------------------------------------------ GEMM tile (tcgen05)
// Swap-AB tile: the weights are the MMA's M operand, the tokens its N
// operand, so a handful of tokens still fills the tensor core's M dimension.
// A worker is one CTA (P = 1: M = 128) or a CTA pair on two SMs (P = 2,
// .cta_group::2: M = 256, 128 weight rows in each CTA's shared memory, and
// the first N/2 token rows in the leader's shared memory, the rest in the
// peer's, so each CTA stages only half of the token rows).  With
// m = 128 P rows per accumulator:
//   gate/up (g, ft):  acc0 = Wg[e][ft*m .. +m, :] * B^T,  acc1 = Wu[...] * B^T
//   down (g, dt, s):  acc0 = Wd[e][dt*2m .. +m, Ks] * H^T, acc1 = rows +m .. +2m
// CTA r holds rows 128 r .. 128 r + 127 of each accumulator (its TMEM lanes)
// for all N tokens.  B = the group's rows of Xp (or x for the shared
// expert) / of H, K-major.
// Pipeline: in each CTA warp 0 lane 0 issues the TMA loads of its part into
// a ring of `stages` stages and signals the leader's full barrier; the
// leader's warp 1 lane 0 issues tcgen05.mma into the worker's TMEM and commits
// each stage to every CTA's empty barrier; all 8 warps of each CTA run the
// epilogue from their own TMEM.

struct GemmJob {
  const CUtensorMap* a0;
  const CUtensorMap* a1;  // null: one accumulator only
  const CUtensorMap* b;
  int a_row0, a1_row0;    // this CTA's first A rows of the two accumulators
  int b_row0;             // this CTA's first B row
  int b_rows;             // B rows this CTA loads (n_mma / P, in boxes of 32 rows)
  int n_mma;              // MMA N (multiple of 16 P, <= 256)
  int b_off;              // byte offset of the B tile inside a stage (1024-aligned)
  const int* gperm;       // non-null: B rows gathered from x, row r = token gperm[r] ...
  int b_valid;            // ... for r < b_valid (the others are left unwritten)
  int kb0, nkb;           // first k block and number of k blocks
  bool a_stream;          // A is read by this task only (L2 evict-first); else kept (evict-last)
  int task;               // task id (-1: not a queue task)
};

// Returns false on a timeout (status already set).
__device__ bool make_gemm_job(const Params& p, const Maps& maps, int task, int rank, GemmJob& job);

// Tasks posted to this CTA's mailbox by the leader's scheduler warp: in the
// same CTA for the leader (CTA scope), from the other CTA for the peer
// (cluster scope).
__device__ __forceinline__ int mailbox_posted(Ctrl* c, const CtaState& st) {
  return st.rank == 0 ? ld_acquire_cta_shared(&c->mb_posted)
                      : ld_acquire_cluster(smem_u32(&c->mb_posted));
}

// Producer: TMA loads of this CTA's part of k blocks [kb_from, kb_to) of
// `job` into the stages starting at pipeline index it0.  The CTAs of a pair
// load the same number of bytes per stage; the leader's full barrier expects
// the pair's total.  Returns the number of k blocks issued (fewer on a
// timeout).
template <int P>
__device__ int issue_loads(const Params& p, const GemmJob& job, char* smem, Ctrl* c,
                           const CtaState& st, uint32_t it0, int kb_from, int kb_to,
                           uint64_t pol_a, uint64_t pol_b) {
  const int nbox = job.gperm ? 0 : ceil_div(job.b_rows, kBBoxRows);  // gathered B: not by TMA
  const bool two = job.a1 != nullptr;
  const uint32_t bytes = (two ? 2u : 1u) * kABoxBytes + (uint32_t)nbox * kBBoxBytes;
  const uint32_t full0 = st.lead_ctrl + (uint32_t)offsetof(Ctrl, full_bar);
  uint32_t it = it0;
  int kb = kb_from;
  for (; kb < kb_to; ++kb, ++it) {
    const uint32_t s = it % p.stages, ph = (it / p.stages) & 1u;
    if (!mbar_wait(&c->empty_bar[s], ph ^ 1u, st.deadline)) break;
    char* stage = smem + (size_t)s * p.stage_bytes;
    if (st.rank == 0) mbar_arrive_expect_tx(&c->full_bar[s], (uint32_t)P * bytes);
    const int kc = (job.kb0 + kb) * kBK;
    if constexpr (P == 2) {
      const uint32_t fb = full0 + 8u * s;
      tma_load_2d_pair(stage, job.a0, fb, kc, job.a_row0, pol_a);
      if (two) tma_load_2d_pair(stage + kABoxBytes, job.a1, fb, kc, job.a1_row0, pol_a);
      for (int bx = 0; bx < nbox; ++bx)
        tma_load_2d_pair(stage + job.b_off + bx * kBBoxBytes, job.b, fb, kc,
                         job.b_row0 + bx * kBBoxRows, pol_b);
    } else {
      tma_load_2d(stage, job.a0, &c->full_bar[s], kc, job.a_row0, pol_a);
      if (two) tma_load_2d(stage + kABoxBytes, job.a1, &c->full_bar[s], kc, job.a1_row0, pol_a);
      for (int bx = 0; bx < nbox; ++bx)
        tma_load_2d(stage + job.b_off + bx * kBBoxBytes, job.b, &c->full_bar[s], kc,
                    job.b_row0 + bx * kBBoxRows, pol_b);
    }
  }
  return kb - kb_from;
}

// Barrier of the 128 B-gathering threads (warps 2-5): true on every thread
// when any of them passes true.
__device__ __forceinline__ bool bthreads_any(bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred p, 2, 128, p;\n\t"
      "selp.s32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1 : 0)
      : "memory");
  return r != 0;
}

// The gathered B operand of a routed gate/up tile (the gather folded into the
// tile): warps 2-5 -- idle during the main loop -- copy each of this CTA's token
// rows' eight 16-byte chunks of every k block from x straight into the stage,
// at the offsets the 128-byte swizzle gives a TMA box (row r at
// (r / 8) * 1024 + (r % 8) * 128, chunk c at ((c ^ (r % 8)) * 16)).  Thread t
// takes chunk t % 8 of rows t / 8 + 16 j (j < 16: up to 256 rows).  A stage is signalled on the
// leader's barrier bfull[s] (one arrival per CTA) once its copies are
// complete and fenced to the async proxy, up to three stages behind the
// copies in flight.  Returns false on a timeout (status set); the outcome is the same
// on all 128 threads.
template <int P>
__device__ bool gather_b_loads(const Params& p, const GemmJob& job, char* smem, Ctrl* c,
                               const CtaState& st) {
  const int lag = min(3, p.stages - 1);  // stages of copies in flight per thread
  const int bt = (int)threadIdx.x - 64;
  const int chunk = bt & 7, r0 = bt >> 3;
  // rows r0 + 16 j, up to the 256 rows a one-CTA tile holds (128 for a pair)
  int tok[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int r = r0 + 16 * j;
    tok[j] = r < job.b_valid ? __ldcg(job.gperm + r) : -1;
    if (tok[j] >= p.T) tok[j] = -1;  // (never: perm holds token ids)
  }
  const uint32_t bfull0 = st.lead_ctrl + (uint32_t)offsetof(Ctrl, bfull_bar);
  auto signal = [&](uint32_t it) {  // every B thread: its copies of stage `it` landed
    fence_proxy_async_shared();
    bthreads_any(false);
    if (bt == 0) mbar_arrive_cluster(bfull0 + 8u * (it % p.stages));
  };
  uint32_t it = st.pipe_it, sig = st.pipe_it;
  bool ok = true;
  for (int kb = 0; kb < job.nkb; ++kb, ++it) {
    const uint32_t s = it % p.stages, ph = (it / p.stages) & 1u;
    const bool fail = bt == 0 && !mbar_wait(&c->empty_bar[s], ph ^ 1u, st.deadline);
    if (bthreads_any(fail)) {
      ok = false;
      break;
    }
    char* dst0 = smem + (size_t)s * p.stage_bytes + job.b_off;
    const __nv_bfloat16* src0 = p.x + (size_t)(job.kb0 + kb) * kBK + chunk * 8;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int r = r0 + 16 * j;
      if (tok[j] >= 0)
        cp_async16(dst0 + (r >> 3) * 1024 + (r & 7) * 128 + (chunk ^ (r & 7)) * 16,
                   src0 + (size_t)tok[j] * p.d);
    }
    cp_async_commit();
    // signal the oldest stage once `lag` are in flight; lag < stages, so the
    // copies of stage it never wait on a stage that is not yet signalled
    if (it + 1 - sig >= (uint32_t)lag) {
      if (lag >= 3) cp_async_wait<2>();
      else if (lag == 2) cp_async_wait<1>();
      else cp_async_wait<0>();
      signal(sig++);
    }
  }
  cp_async_wait<0>();
  if (!ok) return false;
  while (sig < it) signal(sig++);
  return true;
}

template <int P>
__device__ bool gemm_mainloop(const Params& p, const Maps& maps, const GemmJob& job, char* smem,
                              Ctrl* c, CtaState& st) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool two = job.a1 != nullptr;
  bool ok = true;
  if (warp == 0 && lane == 0) {
    fence_proxy_async_global();
    fence_proxy_async_shared();
    const uint64_t pol_first = policy_evict_first();
    const uint64_t pol_last = policy_evict_last();
    // A (weights) streams through L2 unless a sibling tile re-reads it soon;
    // B (token rows) is re-read by the expert's other tiles: keep it
    const uint64_t pol_a = job.a_stream ? pol_first : pol_last;
    const uint64_t pol_b = pol_last;
    const int kb_first = (job.task >= 0 && st.pf_task == job.task) ? st.pf_count : 0;
    st.pf_task = -1;
    ok = issue_loads<P>(p, job, smem, c, st, st.pipe_it + kb_first, kb_first, job.nkb, pol_a,
                        pol_b) == job.nkb - kb_first;
    if (!ok) set_status(p, MOE_E_TIMEOUT, 10);
    // Cross-task overlap: this gate/up or down tile has issued all its loads,
    // so its late phase begins (the scheduler warp may claim the next task
    // now).  Until this tile's MMAs complete, wait for that task; when it is
    // a GEMM tile too, start its first stages now -- they fill as this tile's
    // last MMAs release the stages.  (Both CTAs of the pair receive the same
    // tasks in the same order, so their producers stay in step.)
    int nxt = -1;
    if (ok && job.task >= 0) {
      st_release_cta_shared(&c->mb_late, st.taken);
      const uint32_t acc_parity = st.gemm_count & 1u;
      while (true) {
        if (mailbox_posted(c, st) > st.taken) {
          nxt = c->mb_task[st.taken & 1];
          break;
        }
        if (mbar_try_wait(&c->acc_bar, acc_parity) || globaltimer() > st.deadline ||
            ld_relaxed(&p.sched->status) != 0)
          break;
        __nanosleep(64);
      }
    }
    if (ok && p.prefetch && job.task >= 0 && nxt >= 0) {
      GemmJob nj;
      if (make_gemm_job(p, maps, nxt, st.rank, nj)) {
        fence_acq_rel_gpu();
        fence_proxy_async_global();
        const int n = min(p.stages, nj.nkb);
        const uint64_t pa = nj.a_stream ? pol_first : pol_last;
        const uint64_t pb = pol_last;
        const int done = issue_loads<P>(p, nj, smem, c, st, st.pipe_it + job.nkb, 0, n, pa, pb);
        if (done == n) {
          st.pf_task = nxt;
          st.pf_count = n;
        } else {
          set_status(p, MOE_E_TIMEOUT, 13);
          ok = false;
        }
      }
    }
  } else if (warp == 1 && lane == 0 && st.rank == 0) {
    // the leader issues the worker's MMAs; a pair's leader once the peer's
    // epilogue of the previous GEMM task has finished reading the peer's TMEM
    if (P == 2 && st.gemm_count > 0) {
      const uint32_t par = (st.gemm_count - 1u) & 1u;
      bool got;
      while (!(got = mbar_try_wait_cluster(&c->tmem_empty, par)))
        if (globaltimer() > st.deadline) break;
      if (!got) {
        set_status(p, MOE_E_TIMEOUT, 14);
        ok = false;
      }
    }
    if (ok) {
      const uint32_t idesc = idesc_bf16(P * kBM, (uint32_t)job.n_mma);
      const uint32_t t0 = c->tmem_base, t1 = c->tmem_base + kAcc1Col;
      uint32_t it = st.pipe_it;
      for (int kb = 0; kb < job.nkb; ++kb, ++it) {
        const uint32_t s = it % p.stages, ph = (it / p.stages) & 1u;
        if (!mbar_wait(&c->full_bar[s], ph, st.deadline)) {
          set_status(p, MOE_E_TIMEOUT, 11);
          ok = false;
          break;
        }
        if (job.gperm) {  // the gathered token rows of this stage, in every CTA
          bool got;
          const uint32_t bpar = (st.bphase >> s) & 1u;
          while (!(got = mbar_try_wait_cluster(&c->bfull_bar[s], bpar)))
            if (globaltimer() > st.deadline) break;
          if (!got) {
            set_status(p, MOE_E_TIMEOUT, 15);
            ok = false;
            break;
          }
          st.bphase ^= 1u << s;
        }
        tc_fence_after();
        const uint32_t base = smem_u32(smem + (size_t)s * p.stage_bytes);
        const uint64_t da0 = sw128_desc(base), da1 = sw128_desc(base + kABoxBytes);
        const uint64_t db = sw128_desc(base + job.b_off);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
          // advancing 16 bf16 (32 B) inside the 128-B swizzle row: +2 in the
          // 16-byte-granular start-address field
          mma_bf16<P>(t0, da0 + 2 * kk, db + 2 * kk, idesc, acc);
          if (two) mma_bf16<P>(t1, da1 + 2 * kk, db + 2 * kk, idesc, acc);
        }
        mma_commit_all<P>(&c->empty_bar[s]);
      }
    }
    // (also after a failure, so that the epilogue warps stop waiting)
    mma_commit_all<P>(&c->acc_bar);
  } else if (job.gperm && warp >= 2 && warp < 6) {
    ok = gather_b_loads<P>(p, job, smem, c, st);
    if (!ok && threadIdx.x == 64) set_status(p, MOE_E_TIMEOUT, 16);
  }
  st.pipe_it += job.nkb;
  // everyone waits for the accumulators (the leader's commit reaches every CTA)
  __syncwarp();
  const int ok_all = cta_sync_and(ok ? 1 : 0);
  if (!ok_all) return false;
  const bool done = mbar_wait(&c->acc_bar, st.gemm_count & 1u, st.deadline);
  if (!done) set_status(p, MOE_E_TIMEOUT, 12);
  if (!cta_sync_and(done ? 1 : 0)) return false;
  tc_fence_after();
  return true;
}

// The end of every GEMM task (router, gate/up, down), in every CTA, whether
// it succeeded or not: this CTA's TMEM reads are complete; a pair's peer tells
// the leader, whose next MMAs overwrite the peer's accumulators.
template <int P>
__device__ __forceinline__ void gemm_task_end(Ctrl* c, CtaState& st) {
  tc_fence_before();
  st.gemm_count++;
  if (P == 2 && st.rank != 0) {
    cta_sync();
    if (threadIdx.x == 0) mbar_arrive_cluster(st.lead_ctrl + (uint32_t)offsetof(Ctrl, tmem_empty));
  }
}

// SiLU with the approximate divide: an IEEE division here cost the gate/up
// epilogue two thirds of its time.  For z < -88 the denominator overflows
// and the result is -0 (the exact value is below 1e-36 in magnitude).
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// A warp's epilogue writes a block of 16 rows x 32 consecutive columns of a
// row-major output (row stride `ld` elements), lane j holding column j of
// every row.  Element-wise stores would put 64 bytes in each warp store; the
// block goes through the warp's 1 KB staging area instead and leaves as
// 16-byte vectors, 4 lanes per 64-byte row segment.  Rows >= nrows are not
// written; `col_ok` false skips the whole block.
__device__ __forceinline__ void warp_store_bf16_16x32(char* stg, const float (&v)[16], int lane,
                                                      __nv_bfloat16* dst, size_t ld, int nrows,
                                                      bool col_ok) {
  __nv_bfloat16* s16 = reinterpret_cast<__nv_bfloat16*>(stg);
#pragma unroll
  for (int i = 0; i < 16; ++i) s16[i * 32 + lane] = __float2bfloat16_rn(v[i]);
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int e = lane + 32 * j, i = e >> 2, cc = e & 3;
    if (col_ok && i < nrows)
      *reinterpret_cast<uint4*>(dst + i * ld + cc * 8) =
          *reinterpret_cast<const uint4*>(stg + i * 64 + cc * 16);
  }
  __syncwarp();
}

// The same for fp32 values, eight rows (1 KB) at a time.
__device__ __forceinline__ void warp_store_f32_16x32(char* stg, const float (&v)[16], int lane,
                                                     float* dst, size_t ld, int nrows,
                                                     bool col_ok) {
  float* sf = reinterpret_cast<float*>(stg);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int i = 0; i < 8; ++i) sf[i * 32 + lane] = v[h * 8 + i];
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int e = lane + 32 * j, i = e >> 3, cc = e & 7, r = h * 8 + i;
      if (col_ok && r < nrows)
        *reinterpret_cast<float4*>(dst + r * ld + cc * 4) =
            *reinterpret_cast<const float4*>(stg + i * 128 + cc * 16);
    }
    __syncwarp();
  }
}

// The GEMM job of a gate/up or down task id for the CTA of rank `rank` in
// its worker (false for other task types or an inconsistent group).
__device__ bool make_gemm_job(const Params& p, const Maps& maps, int task, int rank, GemmJob& job) {
  const int type = task_type(task), pl = task_payload(task);
  if (type == kTaskGateUp) {
    const int g = pl / p.n_ftiles, ft = pl - g * p.n_ftiles;
    const Group G = load_group(p, g);
    if (!group_ok(p, G) || ft < 0 || ft >= p.n_ftiles) return false;
    const int gran = 16 * p.pair;  // each CTA's share of N a multiple of 16 rows
    job.n_mma = ((G.nrows + gran - 1) / gran) * gran;
    job.a0 = &maps.wg;
    job.a1 = &maps.wu;
    job.b = G.e < p.E ? &maps.xp : &maps.x;
    job.a_row0 = G.e * p.f + ft * ftile_rows(p) + rank * kBM;
    job.a1_row0 = job.a_row0;
    job.b_row0 = G.src_row0 + rank * (job.n_mma / p.pair);
    job.b_rows = job.n_mma / p.pair;
    job.b_off = 2 * kABoxBytes;
    // a routed group's token rows, gathered from x through perm (folded
    // gathers); the shared expert's are consecutive rows of x (TMA)
    job.gperm = (p.fold_gather && G.e < p.E) ? p.perm + job.b_row0 : nullptr;
    job.b_valid = max(0, min(job.b_rows, G.nrows - rank * job.b_rows));
    job.kb0 = 0;
    job.nkb = p.d / kBK;
    job.a_stream = G.nsib == 1;
    job.task = task;
    return true;
  }
  if (type == kTaskDown) {
    const int n_down = p.n_dtiles * p.ks;
    const int g = pl / n_down, r = pl - g * n_down;
    const int dt = r / p.ks, ksplit = r - dt * p.ks;
    const Group G = load_group(p, g);
    if (!group_ok(p, G) || dt >= p.n_dtiles) return false;
    const int gran = 16 * p.pair;
    job.n_mma = ((G.nrows + gran - 1) / gran) * gran;
    job.a0 = &maps.wd;
    job.a1 = &maps.wd;
    job.b = &maps.h;
    job.a_row0 = G.e * p.d + dt * dtile_rows(p) + rank * kBM;
    job.a1_row0 = job.a_row0 + ftile_rows(p);
    job.b_row0 = G.row0 + rank * (job.n_mma / p.pair);
    job.b_rows = job.n_mma / p.pair;
    job.b_off = 2 * kABoxBytes;
    job.gperm = nullptr;
    job.b_valid = job.b_rows;
    job.kb0 = ksplit * p.kb_down;
    job.nkb = p.kb_down;
    job.a_stream = G.nsib == 1;
    job.task = task;
    return true;
  }
  return false;
}

template <int P>
__device__ void gateup_task(const Params& p, const Maps& maps, int task, char* smem, Ctrl* c,
                            CtaState& st) {
  const int pl = task_payload(task);
  const int g = pl / p.n_ftiles, ft = pl - g * p.n_ftiles;
  const Group G = load_group(p, g);
  GemmJob job;
  if (!make_gemm_job(p, maps, task, st.rank, job)) {
    if (threadIdx.x == 0) set_status(p, MOE_E_DEVICE, 21);
    gemm_task_end<P>(c, st);
    return;
  }
  const bool ok = gemm_mainloop<P>(p, maps, job, smem, c, st);
  if (ok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, half = warp >> 2;
    // this warp's 32 f rows: rows q*32.. of this CTA's 128 rows of the tile
    // (the TMEM lanes it may read); lane j holds f row f0 + j
    const int f0 = ft * ftile_rows(p) + st.rank * kBM + q * 32;
    const bool in_f = f0 < p.f;  // the last tile of an f that is an odd multiple of 128
    const uint32_t lane_addr = c->tmem_base + ((uint32_t)(q * 32) << 16);
    __nv_bfloat16* hblk = p.H + (size_t)G.row0 * p.f + f0;
    for (int ch = half; ch * 16 < G.nrows; ch += 2) {
      float gv[16], uv[16];
      tmem_ld2x16(lane_addr + ch * 16, lane_addr + kAcc1Col + ch * 16, gv, uv);
#pragma unroll
      for (int i = 0; i < 16; ++i) gv[i] = silu_f(gv[i]) * uv[i];
      warp_store_bf16_16x32(c->epi[warp], gv, lane, hblk + (size_t)ch * 16 * p.f, p.f,
                            G.nrows - ch * 16, in_f);
    }
  }
  gemm_task_end<P>(c, st);
}

template <int P>
__device__ void down_task(const Params& p, const Maps& maps, int task, char* smem, Ctrl* c,
                          CtaState& st) {
  const int n_down = p.n_dtiles * p.ks;
  const int pl = task_payload(task);
  const int g = pl / n_down, r = pl - g * n_down;
  const int dt = r / p.ks, ksplit = r - dt * p.ks;
  const Group G = load_group(p, g);
  GemmJob job;
  if (!make_gemm_job(p, maps, task, st.rank, job)) {
    if (threadIdx.x == 0) set_status(p, MOE_E_DEVICE, 22);
    gemm_task_end<P>(c, st);
    return;
  }
  const bool ok = gemm_mainloop<P>(p, maps, job, smem, c, st);
  if (ok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, half = warp >> 2;
    // this warp's two blocks of 32 d columns: rows q*32.. of this CTA's 128
    // rows of each accumulator; lane j holds columns d0 + j and d1 + j
    const int d0 = dt * dtile_rows(p) + st.rank * kBM + q * 32;
    const int d1 = d0 + ftile_rows(p);
    const uint32_t lane_addr = c->tmem_base + ((uint32_t)(q * 32) << 16);
    const bool has0 = d0 < p.d, has1 = d1 < p.d;
    for (int ch = half; ch * 16 < G.nrows; ch += 2) {
      float a[16], b[16];
      tmem_ld2x16(lane_addr + ch * 16, lane_addr + kAcc1Col + ch * 16, a, b);
      const size_t row = (size_t)G.row0 + ch * 16;
      const int nr = G.nrows - ch * 16;
      if (p.y_f32) {
        float* Y = reinterpret_cast<float*>(p.Y) + (size_t)ksplit * p.rows_y * p.d + row * p.d;
        warp_store_f32_16x32(c->epi[warp], a, lane, Y + d0, p.d, nr, has0);
        warp_store_f32_16x32(c->epi[warp], b, lane, Y + d1, p.d, nr, has1);
      } else {
        __nv_bfloat16* Y = reinterpret_cast<__nv_bfloat16*>(p.Y) + row * p.d;
        warp_store_bf16_16x32(c->epi[warp], a, lane, Y + d0, p.d, nr, has0);
        warp_store_bf16_16x32(c->epi[warp], b, lane, Y + d1, p.d, nr, has1);
      }
    }
  }
  gemm_task_end<P>(c, st);
}


// ------------------------------------------------------------------ router (tcgen05)
// Router tile: tokens [tau*128, tau*128 + nt).  Logits on the tensor core:
// D[token, e] = x[token, :] . Wr[e, :], tokens as the M = 128 operand and the
// E experts (padded to 16) as N; fp32 accumulation in TMEM.  The epilogue
// (below) keeps each token's top-k list in the order logit descending, expert
// ascending on ties -- the softmax is monotone, so this is the order of p.
// Ranks inside the tile come from a 128-bit token mask per expert.

// Row stride (floats) of the router tile's logits in shared memory: epad + 4
// keeps rows 16-byte aligned and puts the float4 reads of 8 consecutive rows
// (one quarter warp) on distinct banks.
__device__ __forceinline__ int route_row_stride(int E) { return ((E + 15) / 16) * 16 + 4; }

// Shared-memory bytes the router epilogue needs (logits + exchange area), for
// either tile size (128 tokens, two threads per token; 64 tokens, four).
__host__ __device__ __forceinline__ size_t route_smem_bytes(int E) {
  // (parts - 1) lists of 2 KL words per token
  const size_t xch128 = (size_t)(1 * 2 * kMaxK) * 128;
  const size_t xch64 = (size_t)(3 * 2 * kMaxK) * 64;
  return (size_t)kRouteTokens * (((E + 15) / 16) * 16 + 4) * 4 +
         (xch128 > xch64 ? xch128 : xch64) * 4;
}

// The top-k order: larger logit first, smaller expert first on equal logits.
// After topk_cx, (av, ae) is the earlier of the two pairs.  Bitwise, not
// short-circuit, logic keeps the exchange a run of predicated selects.
__device__ __forceinline__ void topk_cx(float& av, int& ae, float& bv, int& be) {
  const bool sw = (bv > av) | ((bv == av) & (be < ae));
  const float v = av;
  const int e = ae;
  av = sw ? bv : av;
  ae = sw ? be : ae;
  bv = sw ? v : bv;
  be = sw ? e : be;
}

// Merge the sorted list b (length KL) into the sorted top-KL list t: the
// better of t[i] and b[KL-1-i] is a bitonic sequence holding the KL best of
// both, which log2(KL) half-cleaner stages sort.  Branch-free: every lane of a
// warp runs the same instructions, whatever its data.
template <int KL, int NB>
__device__ __forceinline__ void topk_merge(float (&tv)[KL], int (&te)[KL], float (&bv)[NB],
                                           int (&be)[NB]) {
  constexpr int M = NB < KL ? NB : KL;
#pragma unroll
  for (int i = 0; i < M; ++i) topk_cx(tv[KL - M + i], te[KL - M + i], bv[M - 1 - i], be[M - 1 - i]);
#pragma unroll
  for (int s = KL / 2; s >= 1; s >>= 1) {
#pragma unroll
    for (int i = 0; i < KL; ++i)
      if ((i & s) == 0) topk_cx(tv[i], te[i], tv[i + s], te[i + s]);
  }
}

// Store a token's k per-slot values (k consecutive 32-bit words at dst):
// 16-byte vectors when k is a multiple of 4 (dst is then 16-byte aligned),
// 8-byte ones when k is even, else one word at a time.  A warp's stores then
// cover its 32 tokens' rows in few wide transactions instead of k scattered
// 4-byte stores per lane.
template <int KL>
__device__ __forceinline__ void store_slots(uint32_t* dst, const uint32_t (&v)[KL], int k) {
  if constexpr (KL >= 4) {
    if ((k & 3) == 0) {
#pragma unroll
      for (int s = 0; s < KL; s += 4)
        if (s < k) *reinterpret_cast<uint4*>(dst + s) = make_uint4(v[s], v[s + 1], v[s + 2], v[s + 3]);
      return;
    }
  }
  if ((k & 1) == 0) {
#pragma unroll
    for (int s = 0; s < KL; s += 2)
      if (s < k) *reinterpret_cast<uint2*>(dst + s) = make_uint2(v[s], v[s + 1]);
    return;
  }
#pragma unroll
  for (int s = 0; s < KL; ++s)
    if (s < k) dst[s] = v[s];
}

// Epilogue of one router tile of rt tokens (p.rt: 128 or 64) whose logits
// (without bias) sit in shared memory, token m's row at lg + m * ls.  The
// CTA's threads split each token's experts: thread t takes token t % rt and
// the (t / rt)-th of kThreads / rt equal expert ranges (multiples of four).
// Pass 1 keeps each range's top-KL list, four logits at a time (sorted by a
// 4-input network, then merged); the other parts hand their lists to part 0,
// which merges them in part order, so its list starts with the row maximum.
// The weights follow from the kept logits alone: w_j = exp(L_j - max) over
// the sum of exp(L_s - max) for the kept s (the softmax's denominator over
// all E cancels in the renormalisation).
template <int KL>
__device__ __noinline__ void route_epilogue(const Params& p, Ctrl* c, int tile, int nt,
                                            const float* lg, int ls, float* xch) {
  const int E = p.E, k = p.k, rt = p.rt;
  const int parts = kThreads / rt;
  const int t0 = tile * rt;
  const int m = threadIdx.x % rt, part = threadIdx.x / rt;
  const int span = ((E + 4 * parts - 1) / (4 * parts)) * 4;  // a multiple of 4: float4 aligned
  const int e0 = min(E, part * span), e1 = min(E, e0 + span);
  float tv[KL];
  int te[KL];
#pragma unroll
  for (int s = 0; s < KL; ++s) {
    tv[s] = -INFINITY;
    te[s] = 0x7fffffff;
  }
  const float4* row = reinterpret_cast<const float4*>(lg + (size_t)m * ls);
  const float4* brow = reinterpret_cast<const float4*>(c->bias_s);
#pragma unroll 1
  for (int e4 = e0; e4 < e1; e4 += 4) {
    const float4 v4 = row[e4 >> 2], b4 = brow[e4 >> 2];
    float nv[4] = {v4.x + b4.x, v4.y + b4.y, v4.z + b4.z, v4.w + b4.w};
    int ne[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      ne[j] = e4 + j;
      // a NaN logit ranks as -inf (below every real expert's finite logit,
      // above the empty slots), so the kept k are always real experts
      nv[j] = nv[j] == nv[j] ? nv[j] : -INFINITY;
      if (e4 + j >= e1) {
        nv[j] = -INFINITY;
        ne[j] = 0x7fffffff;
      }
    }
    topk_cx(nv[0], ne[0], nv[1], ne[1]);
    topk_cx(nv[2], ne[2], nv[3], ne[3]);
    topk_cx(nv[0], ne[0], nv[2], ne[2]);
    topk_cx(nv[1], ne[1], nv[3], ne[3]);
    topk_cx(nv[1], ne[1], nv[2], ne[2]);
    topk_merge<KL, 4>(tv, te, nv, ne);
  }
  // exchange area, token-minor (conflict-free): the lists of parts 1.. :
  // values [KL][rt] and experts [KL][rt] each
  float* x_list = xch;
  const size_t list_words = (size_t)2 * KL * rt;
  if (part > 0) {
    float* v = x_list + (size_t)(part - 1) * list_words;
    int* ev = reinterpret_cast<int*>(v + (size_t)KL * rt);
#pragma unroll
    for (int s = 0; s < KL; ++s) {
      v[s * rt + m] = tv[s];
      ev[s * rt + m] = te[s];
    }
  }
  cta_sync();
  if (part == 0) {
    for (int q = 1; q < parts; ++q) {
      const float* v = x_list + (size_t)(q - 1) * list_words;
      const int* ev = reinterpret_cast<const int*>(v + (size_t)KL * rt);
      float bv[KL];
      int be[KL];
#pragma unroll
      for (int s = 0; s < KL; ++s) {
        bv[s] = v[s * rt + m];
        be[s] = ev[s * rt + m];
      }
      topk_merge<KL, KL>(tv, te, bv, be);
    }
  }
  // The renormalised weights need no softmax denominator: p_j = e_j / S over
  // all experts and w_j = p_j / (sum of the kept p) = e_j / (sum of the kept
  // e), with e_j = exp(L_j - max).  tv[0] is the row maximum.
  const bool valid = part == 0 && m < nt;
  float ek[KL];
  float kept = 0.f;
#pragma unroll
  for (int s = 0; s < KL; ++s) {
    ek[s] = s < k ? __expf(tv[s] - tv[0]) : 0.f;
    kept += ek[s];
  }
  const float inv_kept = 1.f / kept;
  if (valid) {
    const size_t o = (size_t)(t0 + m) * k;
    uint32_t iv[KL], wv[KL];
#pragma unroll
    for (int s = 0; s < KL; ++s) {
      iv[s] = (uint32_t)te[s];
      wv[s] = __float_as_uint(ek[s] * inv_kept);
    }
    store_slots<KL>(reinterpret_cast<uint32_t*>(p.idx + o), iv, k);
    store_slots<KL>(reinterpret_cast<uint32_t*>(p.wgt + o), wv, k);
  }
  // the tile's token mask per expert: word m / 32 of every expert is written
  // by the warp of tokens m / 32 * 32 .., and only by it (rt is a multiple of
  // 32, so lane j holds token 32 (m / 32) + j); the lanes that chose the same
  // expert in slot s merge their bits first, so each distinct expert takes
  // one OR instead of one atomic per lane (the lanes of a warp that picked a
  // popular expert all hit the same word)
  if (part == 0 && (m >> 5) * 32 < nt) {
#pragma unroll
    for (int s = 0; s < KL; ++s) {
      if (s < k) {
        const int e = valid ? te[s] : -1;
        const unsigned same = __match_any_sync(0xffffffffu, e);
        if (valid && (threadIdx.x & 31) == __ffs(same) - 1) c->mask[e * 4 + (m >> 5)] |= same;
      }
    }
  }
  cta_sync();
  if (valid) {
    const size_t o = (size_t)(t0 + m) * k;
    const int wd = m >> 5;
    const uint32_t below = (1u << (m & 31)) - 1u;
    uint32_t rv[KL];
#pragma unroll
    for (int s = 0; s < KL; ++s) {
      rv[s] = 0u;
      if (s < k) {
        const uint32_t* mk = c->mask + te[s] * 4;
        int r = __popc(mk[wd] & below);
        for (int q = 0; q < wd; ++q) r += __popc(mk[q]);
        rv[s] = (uint32_t)r;
      }
    }
    store_slots<KL>(reinterpret_cast<uint32_t*>(p.rank + o), rv, k);
  }
  for (int e = threadIdx.x; e < E; e += kThreads) {
    const uint32_t* mk = c->mask + e * 4;
    p.tile_cnt[(size_t)tile * E + e] = __popc(mk[0]) + __popc(mk[1]) + __popc(mk[2]) + __popc(mk[3]);
    reinterpret_cast<uint4*>(p.rmask)[(size_t)tile * E + e] = make_uint4(mk[0], mk[1], mk[2], mk[3]);
  }
}

__device__ __forceinline__ void route_epilogue_k(const Params& p, Ctrl* c, int tile, int nt,
                                                 const float* lg, int ls, float* xch) {
  if (p.k <= 2) route_epilogue<2>(p, c, tile, nt, lg, ls, xch);
  else if (p.k <= 4) route_epilogue<4>(p, c, tile, nt, lg, ls, xch);
  else if (p.k <= 8) route_epilogue<8>(p, c, tile, nt, lg, ls, xch);
  else route_epilogue<16>(p, c, tile, nt, lg, ls, xch);
}

// One router task: router tile P pt + r for the CTA of rank r, K split
// `split` of p.route_ks, as one MMA of the worker: each CTA's 128 A rows are
// its tile's tokens; for a pair the experts (N, padded to 32) are split in
// halves between the two CTAs' B operands, so each CTA's TMEM receives all
// the logits of its own tokens.  With a single split the epilogue reads the
// logits from TMEM.  With several, each split stores its fp32 partial logits;
// the split that finishes last sums all of them in split order (fixed, so the
// result does not depend on timing) and runs the epilogue.  Returns true when
// this call completed this CTA's tile (the peer of an odd last tile has none).
template <int P>
__device__ bool route_task(const Params& p, const Maps& maps, int pt, int split, char* smem,
                           Ctrl* c, CtaState& st) {
  const int rt = p.rt;  // tokens of a router tile: 128, or 64 for small layers
  const int tile = pt * P + st.rank;
  const bool mine = tile < p.n_route;
  const int t0 = tile * rt;
  const int nt = mine ? min(rt, p.T - t0) : 0;
  const int ks = p.route_ks;
  const int nkb = p.d / kBK;
  const int epad = ((p.E + 15) / 16) * 16;   // logit columns read back
  const int nmma = ((p.E + 16 * P - 1) / (16 * P)) * (16 * P);  // MMA N over the worker
  for (int i = threadIdx.x; i < kMaxE * 4; i += kThreads) c->mask[i] = 0u;
  for (int e = threadIdx.x; e < kMaxE; e += kThreads)
    c->bias_s[e] = (p.bias && e < p.E) ? __ldg(p.bias + e) : 0.f;
  GemmJob job;
  job.a0 = &maps.xr;
  job.a1 = nullptr;
  job.b = &maps.wr;
  job.a_row0 = t0;  // past T (the peer of an odd last tile): zero-filled rows
  job.a1_row0 = 0;
  job.b_row0 = st.rank * (nmma / P);
  job.b_rows = nmma / P;
  job.n_mma = nmma;
  job.b_off = kABoxBytes;
  job.gperm = nullptr;
  job.b_valid = job.b_rows;
  job.kb0 = split * nkb / ks;
  job.nkb = (split + 1) * nkb / ks - job.kb0;
  job.a_stream = true;  // x rows: read by this tile only; Wr (B) is shared by all tiles
  job.task = -1;
  const bool ok = gemm_mainloop<P>(p, maps, job, smem, c, st);
  bool tile_done = false;
  if (ok && mine) {
    const int warp = threadIdx.x >> 5;
    const uint32_t lane_addr = c->tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    const int ls = route_row_stride(p.E);
    float* lg = reinterpret_cast<float*>(smem);  // [128][ls] logits
    float* xch = lg + (size_t)rt * ls;
    const int nch = epad / 16;
    if (ks == 1) {
      // TMEM -> shared, the tile's rt rows: warps w and w + 4 share TMEM
      // lanes, each takes half the chunks (the MMA's rows past rt are unused)
      const int m = (warp & 3) * 32 + (threadIdx.x & 31);
      const int c0 = (warp >> 2) * ((nch + 1) / 2), c1 = (warp >> 2) ? nch : (nch + 1) / 2;
      float4* dst = reinterpret_cast<float4*>(lg + (size_t)m * ls);
      for (int ch = c0; (warp & 3) * 32 < rt && ch < c1; ++ch) {
        float v[16];
        tmem_ld16(lane_addr + ch * 16, v);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[ch * 4 + q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      tc_fence_before();
      cta_sync();
      route_epilogue_k(p, c, tile, nt, lg, ls, xch);
      tile_done = true;
    } else {
      // partial logits of this split: [tile][split][rt][epad] fp32
      if (warp < 4 && warp * 32 < rt) {
        const int m = warp * 32 + (threadIdx.x & 31);
        float4* dst = reinterpret_cast<float4*>(
            p.rpart + (((size_t)tile * ks + split) * rt + m) * epad);
        for (int ch = 0; ch < nch; ++ch) {
          float v[16];
          tmem_ld16(lane_addr + ch * 16, v);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[ch * 4 + q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
      tc_fence_before();
      release_writes();
      if (threadIdx.x == 0) c->flag = atom_add_acq_rel(p.rsplit_done + tile, 1) + 1 == ks;
      cta_sync();
      if (c->flag) {
        fence_acq_rel_gpu();
        // sum the splits into the shared logits, in split order: each thread
        // owns up to 16 float4 of the tile per round and loads that slice of
        // every split in turn (16 independent loads in flight per thread)
        const float4* src = reinterpret_cast<const float4*>(p.rpart + (size_t)tile * ks * rt * epad);
        const int r4 = epad / 4, n4 = rt * r4;
        constexpr int kPer = 16;
        for (int base = 0; base < n4; base += kPer * kThreads) {
          float4 acc[kPer];
#pragma unroll
          for (int u = 0; u < kPer; ++u) {
            const int i = base + u * kThreads + threadIdx.x;
            acc[u] = i < n4 ? __ldcg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          for (int s2 = 1; s2 < ks; ++s2) {
            float4 v[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
              const int i = base + u * kThreads + threadIdx.x;
              v[u] = i < n4 ? __ldcg(src + (size_t)s2 * n4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
              acc[u].x += v[u].x; acc[u].y += v[u].y; acc[u].z += v[u].z; acc[u].w += v[u].w;
            }
          }
#pragma unroll
          for (int u = 0; u < kPer; ++u) {
            const int i = base + u * kThreads + threadIdx.x;
            if (i < n4) {
              const int rw = i / r4;
              reinterpret_cast<float4*>(lg + (size_t)rw * ls)[i - rw * r4] = acc[u];
            }
          }
        }
        cta_sync();
        route_epilogue_k(p, c, tile, nt, lg, ls, xch);
        tile_done = true;
      }
    }
  }
  gemm_task_end<P>(c, st);
  return tile_done;
}

// ------------------------------------------------------------------ claimed-twice check
// (debug) Mark a task claimed in the bitmap; a second claim of the same task,
// or an id outside the layer's tasks, sets MOE_E_DEVICE.  One thread.
__device__ __forceinline__ void check_claim(const Params& p, int task) {
  if (!p.claimed) return;
  const int type = task_type(task), pl = task_payload(task);
  int bit = -1;
  if (type == kTaskRoute) bit = pl < p.n_route_tasks ? pl : -1;
  else if (type == kTaskGather) bit = p.claim_gather_off + pl;
  else if (type == kTaskGateUp) bit = p.claim_gateup_off + pl;
  else if (type == kTaskDown) bit = p.claim_down_off + pl;
  else if (type == kTaskCombine) bit = p.claim_comb_off + pl;
  if (bit < 0 || bit >= p.claim_bits) {
    set_status(p, MOE_E_DEVICE, 51);
    return;
  }
  const uint32_t m = 1u << (bit & 31);
  if (atomicOr(p.claimed + (bit >> 5), m) & m) set_status(p, MOE_E_DEVICE, 50);
}

// ------------------------------------------------------------------ notifications
// (persistent mode) Run by the scheduler warp, all 32 lanes, after the
// compute warps handed a finished task over (their writes were released to
// this warp at CTA scope; sched_notify makes them visible at GPU scope
// first).  They bump the dependency counters the task feeds and push the
// tasks that became ready, while the compute warps already run the next task.

__device__ __forceinline__ bool drop_for_fault(const Params& p) {
  if (p.fault_drop < 0) return false;
  return atomicAdd(&p.sched->fault_seen, 1) == p.fault_drop;
}

// Gather finished.  Release policy (temporal scheduling):
//  - kReleaseAll: when the last gather of the layer is done, every routed
//    gate/up tile is pushed at once, f-tile major across all groups, so all
//    experts finish their gate/up work together and the down tiles of every
//    expert become ready in one wide burst;
//  - kReleaseExpert: when the last gather of an expert is done, its tiles are
//    pushed (f-tile major across its sibling groups).
__device__ void notify_gather_done(const Params& p, int g) {
  const int lane = threadIdx.x & 31;
  const Group G = load_group(p, g);
  if (p.release == kReleaseAll) {
    int last = 0, nr = 0;
    if (lane == 0) {
      const int old = atom_add_acq_rel(&p.sched->gathers_done, 1);
      last = (old + 1 == ld_relaxed(&p.sched->n_gather));
      nr = ld_relaxed(&p.sched->n_groups) - p.n_shared_groups;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    nr = __shfl_sync(0xffffffffu, nr, 0);
    if (last) {
      const int nf = p.n_ftiles, ns0 = p.n_shared_groups;
      push_gen_warp(p, gemm_queue(p), nr * nf, [=](int i) {
        return task_id(kTaskGateUp, (ns0 + i % nr) * nf + i / nr);
      });
    }
    return;
  }
  int ready = 0;
  if (lane == 0) {
    const int old = atom_add_acq_rel(p.gather_done + G.sib0, 1);
    ready = (old + 1 == G.gchunks);
  }
  ready = __shfl_sync(0xffffffffu, ready, 0);
  if (ready) {
    const int nf = p.n_ftiles, ns = G.nsib, s0 = G.sib0;
    push_gen_warp(p, gemm_queue(p), ns * nf, [=](int i) {
      return task_id(kTaskGateUp, (s0 + i % ns) * nf + i / ns);
    });
  }
}

// All gate/up tiles of an expert done: release its down tiles, interleaved
// the same way.
__device__ void notify_gateup_done(const Params& p, int g) {
  const int lane = threadIdx.x & 31;
  const Group G = load_group(p, g);
  int ready = 0;
  if (lane == 0 && !drop_for_fault(p)) {
    const int old = atom_add_acq_rel(p.gu_done + G.sib0, 1);
    ready = (old + 1 == G.nsib * p.n_ftiles);
  }
  ready = __shfl_sync(0xffffffffu, ready, 0);
  if (ready) {  // bands before the last: GEMM queue; the last band: low priority
    const int nd = p.n_dtiles * p.ks, ns = G.nsib, s0 = G.sib0;
    const int nd_hi = p.n_bands == 2 ? p.dt_lo0 * p.ks : nd;
    push_gen_warp(p, gemm_queue(p), ns * nd_hi, [=](int i) {
      return task_id(kTaskDown, (s0 + i % ns) * nd + i / ns);
    });
    if (nd > nd_hi)
      push_gen_warp(p, gemm_lo_queue(p), ns * (nd - nd_hi), [=](int i) {
        return task_id(kTaskDown, (s0 + i % ns) * nd + nd_hi + i / ns);
      });
  }
}

// Target of the counter of combine task (ctile, band): every (token, slot)
// and shared row of the tile, once per down task of the band covering it.
__device__ __forceinline__ int comb_target(const Params& p, int ctile, int band) {
  const int nt = min(p.ct, p.T - ctile * p.ct);
  return nt * (p.k + p.S) * (band_dt1(p, band) - band_dt0(p, band)) * p.ks;
}

// A down tile finished: every combine task of its d band whose token tile
// holds some of its rows gains those rows.  The group's tokens ascend, so
// its rows form runs of one combine tile each; every run (cut at 32-row
// chunk boundaries) is one counter add, and the add that reaches the target
// pushes the combine task.
__device__ void notify_down_done(const Params& p, int task) {
  const int lane = threadIdx.x & 31;
  int drop = lane == 0 ? (drop_for_fault(p) ? 1 : 0) : 0;
  if (__shfl_sync(0xffffffffu, drop, 0)) return;
  const int nd = p.n_dtiles * p.ks, pl = task_payload(task);
  const int g = pl / nd, dt = (pl - g * nd) / p.ks;
  const int band = (p.n_bands == 2 && dt >= p.dt_lo0) ? 1 : 0;
  const Group G = load_group(p, g);
  const bool routed = G.e < p.E;
  for (int r0 = 0; r0 < G.nrows; r0 += 32) {
    const int r = r0 + lane;
    const bool in = r < G.nrows;
    int ct = -1;
    if (in) ct = (routed ? __ldcg(p.perm + G.row0 + r) : G.src_row0 + r) / p.ct;
    const int up = __shfl_up_sync(0xffffffffu, ct, 1);
    const bool start = in && (lane == 0 || ct != up);
    const unsigned starts = __ballot_sync(0xffffffffu, start);
    if (start) {
      const unsigned after = lane == 31 ? 0u : (starts >> (lane + 1));
      const int len = after ? __ffs(after) : min(32, G.nrows - r0) - lane;
      const int ci = ct * p.n_bands + band;
      const int old = atom_add_acq_rel(p.comb_done + ci, len);
      if (old + len == comb_target(p, ct, band)) {
        const QueueRef q = mover_queue(p);
        const int j = push_start(ci);
        const int slot = (int)(atomicAdd(q.word + j, 1ull << 32) >> 32);
        if (slot < q.seg) st_release(q.ring + j * q.seg + slot, task_id(kTaskCombine, ci) + 1);
        else set_status(p, MOE_E_DEVICE, 5);
      }
    }
  }
}

// The notification of one finished task (any type; router tiles and combines
// feed no counter here).  Host-set fault injection: every notification of
// one task type dropped (its dependents are never released: the claims run
// out of time), or one finished gate/up task pushed again (claimed twice).
__device__ void sched_notify(const Params& p, int task) {
  const int type = task_type(task), pl = task_payload(task);
  if (type == p.fault_drop_type) return;
  if (type == kTaskGateUp && p.fault_repush >= 0) {
    int again = 0;
    if ((threadIdx.x & 31) == 0) again = atomicAdd(&p.sched->repush_seen, 1) == p.fault_repush;
    if (__shfl_sync(0xffffffffu, again, 0))
      push_gen_warp(p, gemm_queue(p), 1, [=](int) { return task; });
  }
  if (type == kTaskGather) notify_gather_done(p, pl >> 3);
  else if (type == kTaskGateUp) notify_gateup_done(p, pl / p.n_ftiles);
  else if (type == kTaskDown) notify_down_done(p, task);
}

}  // namespace moe
