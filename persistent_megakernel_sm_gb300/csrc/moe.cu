// MoE-layer forward for GB300 (sm_103a): the persistent megakernel, the
// static persistent megakernel and the one-kernel-per-stage ablation, and the
// C ABI declared in include/moe.h.
//
// Persistent mode (Weave abstract, arXiv 2609.21483; xxqk.cn/news/665650
// sections 2.1-2.3; m.xxqk.cn/news/657744 sections 2.2-2.3): one CTA per SM
// stays resident and loops { claim a task; run it; publish its writes; bump
// the dependency counters it feeds; push the tasks that reached zero } until
// every task queue is drained.  Termination is by task count, never by
// seeing an empty queue (m.xxqk.cn/news/657744 section 3.3 describes the
// early-exit race the other rule invites).  Router tiles and shared-expert
// tiles are ready at launch; the CTA that finishes the last router tile runs
// the plan (scan, permutation, row groups, cost model) and pushes the gathers.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstddef>
#include <cstring>
#include <mutex>
#include <string>

#include "layer.cuh"
#include "tasks.cuh"

namespace moe {

__device__ __forceinline__ char* align1024(char* p) {
  return reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// CTA set-up shared by every kernel: barriers, TMEM, per-thread state.  The
// kernels with tensor-core tasks allocate TMEM (`tmem`); built for CTA pairs
// (P = 2) they run as clusters of two CTAs, allocate the TMEM for the pair
// (one warp in each CTA), and pass a cluster barrier that makes both CTAs'
// barriers visible before any traffic between them.
template <int P>
__device__ __forceinline__ void cta_setup(const Params& p, const Maps& maps, char*& smem,
                                          Ctrl*& c, CtaState& st, bool tmem) {
  constexpr bool pair = P == 2;
  extern __shared__ __align__(1024) char smem_raw[];
  smem = align1024(smem_raw);
  c = reinterpret_cast<Ctrl*>(smem + (size_t)p.stages * p.stage_bytes);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&c->full_bar[s], 1);
      mbar_init(&c->empty_bar[s], 1);
    }
    mbar_init(&c->acc_bar, 1);
    mbar_init(&c->tmem_empty, 1);
    for (int s = 0; s < p.stages; ++s) mbar_init(&c->bfull_bar[s], P);
    mbar_init(&c->gbar, 1);
    mbar_init(&c->cbar[0], 1);
    mbar_init(&c->cbar[1], 1);
    fence_mbar_init();
    c->deadline = globaltimer() + p.timeout_ns;
    c->mb_posted = c->mb_taken = c->mb_done = c->mb_handled = c->mb_done_peer = 0;
    c->mb_late = -1;
  }
  if (tmem && warp == 1) {
    tmem_alloc<P>(&c->tmem_base, kTmemCols);
    tmem_relinquish<P>();
  }
  if (threadIdx.x == 32 * 2) {
    prefetch_tmap(&maps.wg);
    prefetch_tmap(&maps.wu);
    prefetch_tmap(&maps.wd);
    prefetch_tmap(&maps.xp);
    prefetch_tmap(&maps.x);
    prefetch_tmap(&maps.h);
    prefetch_tmap(&maps.xr);
    prefetch_tmap(&maps.wr);
  }
  tc_fence_before();
  __syncthreads();
  if (pair) cluster_sync();
  tc_fence_after();
  st.rank = pair ? (int)cluster_rank() : 0;
  st.worker = (int)(blockIdx.x / P);
  st.lead_ctrl = pair ? mapa_shared(smem_u32(c), 0) : smem_u32(c);
  st.pipe_it = 0;
  st.bphase = 0;
  st.gemm_count = 0;
  st.deadline = c->deadline;
  st.role_mover = 0;
  st.gather_phase = 0;
  st.comb_phase = 0;
  st.exit_reason = 0;
  st.polls = 0;
  st.claims = 0;
  st.plan_seen = false;
  st.n_gather = st.mover_total = st.gemm_total = 0;
  st.pf_task = -1;
  st.pf_count = 0;
  st.taken = 0;
}

// Both CTAs of a pair pass a cluster barrier before either exits or frees the
// pair's TMEM: neither may leave while the other can still signal its
// barriers or read its shared memory.
template <int P>
__device__ __forceinline__ void cta_teardown(Ctrl* c, bool tmem) {
  tc_fence_before();
  __syncthreads();
  if (P == 2) cluster_sync();
  if (tmem && (threadIdx.x >> 5) == 1) {
    tc_fence_after();
    tmem_dealloc<P>(c->tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ persistent megakernel
// Nine warps per CTA.  Warps 0-7 (the compute warps) run tasks: the producer
// (warp 0 lane 0) and MMA issuer (warp 1 lane 0) of the GEMM tiles, the
// epilogues, the bulk-copy movers.  Warp 8 (the scheduler warp) never runs
// task code: it claims the next task while the current one runs -- at once
// when the first-choice queue is deep, else when the running task reaches its
// late phase (a GEMM tile's last loads issued, a mover's last round) -- and
// it runs the notifications of finished tasks (GPU-scope release, counter
// bumps, pushes) while the compute warps already run the next task.  The two
// sides talk through the shared-memory mailbox in Ctrl.

__device__ __forceinline__ void trace_record(const Params& p, unsigned long long w0,
                                             unsigned long long a, unsigned long long b,
                                             unsigned long long e) {
  const int i = atomicAdd(&p.sched->trace_n, 1);
  if (i < p.trace_cap) {
    unsigned long long* r = p.trace + (size_t)i * 4;
    r[0] = w0;
    r[1] = a;
    r[2] = b;
    r[3] = e;
  }
}

// Once the plan is published and until the first gate/up tiles start, HBM
// only carries the gathers: pull the gate/up weight tiles the first GEMM wave
// will read into L2 -- tiles (expert, f tile) in index order, the order the
// plan keeps (Params::index_order) -- spread over the workers, up to
// l2_pf_bytes.  One lane of each worker's leader, asynchronous.  (Issued
// earlier, while the plan runs, the prefetch traffic slows the plan's memory
// accesses: measured 2.5 us slower on the fine and decode workloads.)
__device__ void prefetch_first_weights(const Params& p, const CtaState& st) {
  const int fr = ftile_rows(p);
  const size_t tile_bytes = (size_t)fr * p.d * 2;  // one f tile of w_gate or w_up
  const long long n_tiles =
      min((long long)p.E * p.n_ftiles, p.l2_pf_bytes / (long long)(2 * tile_bytes));
  const int workers = (int)gridDim.x / p.pair;
  constexpr uint32_t kChunk = 128u << 10;
  for (long long i = st.worker; i < n_tiles; i += workers) {
    const int e = (int)(i / p.n_ftiles), ft = (int)(i - (long long)e * p.n_ftiles);
    const int rows = min(fr, p.f - ft * fr);
    const size_t row0 = (size_t)e * p.f + (size_t)ft * fr;
    const char* g = reinterpret_cast<const char*>(p.w_gate + row0 * p.d);
    const char* u = reinterpret_cast<const char*>(p.w_up + row0 * p.d);
    const size_t bytes = (size_t)rows * p.d * 2;
    for (size_t o = 0; o < bytes; o += kChunk) {
      const uint32_t n = (uint32_t)min((size_t)kChunk, bytes - o);
      bulk_prefetch_l2(g + o, n);
      bulk_prefetch_l2(u + o, n);
    }
  }
}

// The compute warps of every CTA of a worker: take the tasks the leader's
// scheduler warp posts to this CTA's mailbox (the same tasks, in the same
// order, in both CTAs of a pair), run this CTA's part of each, and report it
// finished: the leader's own to its scheduler warp through its mailbox, a
// pair's peer's to the leader as a count of finished tasks.
template <int P>
__device__ void compute_loop(const Params& p, const Maps& maps, char* smem, Ctrl* c,
                             CtaState& st) {
  int executed = 0, gemm_tasks = 0, mover_tasks = 0, done = 0;
  const bool lead = st.rank == 0;
  while (true) {
    if (threadIdx.x == 0) {  // take the next posted task, or the exit token
      uint32_t backoff = 32;
      int t = -1;
      while (true) {
        if (mailbox_posted(c, st) > st.taken) {
          t = c->mb_task[st.taken & 1];
          c->t_claim = c->mb_tclaim[st.taken & 1];
          ++st.taken;
          if (lead && t >= 0) check_claim(p, t);
          if (lead) st_release_cta_shared(&c->mb_taken, st.taken);
          else st_release_cluster(smem_u32(&c->mb_taken), st.taken);
          break;
        }
        if (ld_relaxed(&p.sched->status) != 0) break;
        if (globaltimer() > st.deadline) {
          set_status(p, MOE_E_TIMEOUT, 30);
          break;
        }
        __nanosleep(backoff);
        if (backoff < 256) backoff <<= 1;
      }
      c->task = t;
      c->t_start = globaltimer();
    }
    cta_sync();
    const int task = c->task;
    if (task < 0) break;
    ++executed;
    const int type = task_type(task), pl = task_payload(task);
    if (type == kTaskRoute) {
      const int pt = pl / p.route_ks, split = pl - pt * p.route_ks;
      if (route_task<P>(p, maps, pt, split, smem, c, st)) {
        release_writes();
        if (threadIdx.x == 0) {
          const int old = atom_add_acq_rel(&p.sched->route_done, 1);
          c->flag = (old + 1 == p.n_route);
        }
        cta_sync();
        if (c->flag) {  // the last router tile: this CTA runs the plan
          fence_acq_rel_gpu();
          const unsigned long long t_plan = globaltimer();
          plan_task(p, smem, c, true);
          if (threadIdx.x == 0 && p.trace) {
            const unsigned long long w0 = (unsigned long long)blockIdx.x << 32;
            trace_record(p, w0 | (unsigned)task_id(kTaskPlan, 0), t_plan, t_plan, globaltimer());
            for (int ph = 0; ph < 7; ++ph)  // phase boundaries of the plan
              trace_record(p, w0 | (unsigned)task_id(kTaskPlan, 1 + ph), c->plan_t[ph],
                           c->plan_t[ph], c->plan_t[ph]);
          }
        }
      }
    } else if (type == kTaskGather) {
      ++mover_tasks;
      gather_task(p, pl >> 3, pl & 7, st.rank, P, smem, c, st);
    } else if (type == kTaskGateUp) {
      ++gemm_tasks;
      gateup_task<P>(p, maps, task, smem, c, st);
    } else if (type == kTaskDown) {
      ++gemm_tasks;
      down_task<P>(p, maps, task, smem, c, st);
    } else if (type == kTaskCombine) {
      ++mover_tasks;
      combine_task(p, pl, st.rank, P, smem, c, st);
    } else {
      if (threadIdx.x == 0) set_status(p, MOE_E_DEVICE, 6);
      break;
    }
    // hand the finished task over: every compute thread's writes (async
    // proxy included) come before thread 0's release
    fence_proxy_async_global();
    cta_sync();
    if (threadIdx.x == 0) {
      ++done;
      if (lead) {
        if (p.trace)
          trace_record(p, ((unsigned long long)blockIdx.x << 32) | (unsigned)task, c->t_claim,
                       c->t_start, globaltimer());
        while (done - 1 - ld_acquire_cta_shared(&c->mb_handled) >= 2) {  // ring of two
          if (ld_relaxed(&p.sched->status) != 0) break;
          if (globaltimer() > st.deadline) {
            set_status(p, MOE_E_TIMEOUT, 31);
            break;
          }
          __nanosleep(64);
        }
        c->mb_done_task[(done - 1) & 1] = task;
        st_release_cta_shared(&c->mb_done, done);
      } else {
        // the peer's writes (ordered before this store by the CTA barrier)
        // reach the leader's scheduler warp, which fences at GPU scope before
        // it notifies
        st_release_cluster(st.lead_ctrl + (uint32_t)offsetof(Ctrl, mb_done_peer), done);
      }
    }
  }
  if (threadIdx.x == 0 && lead) {
    atomicAdd(&p.sched->tasks_done, executed);
    atomicAdd(&p.sched->stat_gemm, gemm_tasks);
    atomicAdd(&p.sched->stat_mover, mover_tasks);
  }
}

// The leader's scheduler warp (a pair's peer's has nothing to do): claims
// each task for the worker, posts it to every CTA's mailbox, and runs a
// finished task's notifications once every CTA has finished it.
template <int P>
__device__ void scheduler_loop(const Params& p, Ctrl* c, CtaState& st) {
  if (st.rank != 0) return;
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  const uint32_t peer = P == 2 ? mapa_shared(smem_u32(c), 1) : 0u;  // the peer's Ctrl
  const uint32_t off_posted = (uint32_t)offsetof(Ctrl, mb_posted);
  const uint32_t off_taken = (uint32_t)offsetof(Ctrl, mb_taken);
  const uint32_t off_task = (uint32_t)offsetof(Ctrl, mb_task);
  int posted = 0, handled = 0, ahead = 0, polled_seq = -1;
  bool exit_posted = false, prefetched = p.l2_pf_bytes <= 0;
  uint32_t backoff = 32;
  auto post = [&](int t) {
    if (lane == 0) {
      c->mb_task[posted & 1] = t;
      c->mb_tclaim[posted & 1] = globaltimer();
      if (P == 2) st_cluster(peer + off_task + 4u * (posted & 1), t);
    }
    ++posted;
    __syncwarp();
    if (lane == 0) {
      st_release_cta_shared(&c->mb_posted, posted);
      if (P == 2) st_release_cluster(peer + off_posted, posted);
    }
  };
  while (true) {
    bool progress = false;
    // notifications of the tasks both CTAs have finished
    int done = 0, taken = 0, late_seq = 0;
    if (lane == 0) {
      done = ld_acquire_cta_shared(&c->mb_done);
      taken = ld_acquire_cta_shared(&c->mb_taken);
      if (P == 2) {
        done = min(done, ld_acquire_cluster(smem_u32(&c->mb_done_peer)));
        taken = min(taken, ld_acquire_cluster(peer + off_taken));
      }
      late_seq = ld_acquire_cta_shared(&c->mb_late);
    }
    done = __shfl_sync(full, done, 0);
    taken = __shfl_sync(full, taken, 0);
    late_seq = __shfl_sync(full, late_seq, 0);
    if (handled < done) {
      fence_acq_rel_gpu();  // the compute warps' writes, acquired above, before our releases
      while (handled < done) {
        sched_notify(p, c->mb_done_task[handled & 1]);
        ++handled;
      }
      __syncwarp();
      if (lane == 0) st_release_cta_shared(&c->mb_handled, handled);
      progress = true;
    }
    if (!prefetched) {  // the L2 weight prefetch, once the plan is published
      const int pd = __shfl_sync(full, lane == 0 ? ld_relaxed(&p.sched->plan_done) : 0, 0);
      if (pd != 0) {
        if (lane == 0) prefetch_first_weights(p, st);
        prefetched = true;
      }
    }
    const int status = __shfl_sync(full, lane == 0 ? ld_relaxed(&p.sched->status) : 0, 0);
    if (status != 0) {
      st.exit_reason = 2;
      break;
    }
    if (exit_posted) {
      if (handled >= posted - 1) break;  // every real task finished and notified
    } else if (posted == taken) {  // nothing waiting in either mailbox
      const bool idle = taken == done;
      const bool late = late_seq == taken;
      int min_depth = 0;
      if (idle || late) {
        min_depth = 1;
      } else if (p.ahead_depth > 0 && polled_seq != taken) {
        min_depth = p.ahead_depth;  // early claim: once per task, deep queue only
        polled_seq = taken;
      }
      if (min_depth > 0) {
        const int r = claim_once(p, st, min_depth);
        if (r >= 0) {
          post(r);
          if (!idle) ++ahead;
          progress = true;
        } else if (r == -4) {
          progress = true;  // lost a CAS: retry at once
        } else if (r == -2 || r == -3) {
          st.exit_reason = r == -2 ? 1 : 2;
          post(-1);
          exit_posted = true;
          progress = true;
        } else if (idle) {
          ++st.polls;
          const int late_t = __shfl_sync(full, lane == 0 ? (globaltimer() > st.deadline) : 0, 0);
          if (late_t) {
            if (lane == 0) set_status(p, MOE_E_TIMEOUT, 3);
            st.exit_reason = 3;
            break;
          }
        }
      }
    }
    if (progress) {
      backoff = 32;
    } else {
      __nanosleep(backoff);
      if (backoff < 512) backoff <<= 1;
    }
  }
  if (lane == 0) {
    atomicAdd(&p.sched->stat_ahead, ahead);
    if (p.trace)  // exit record: reason and polls, the GEMM queue's first word
      trace_record(p, ((unsigned long long)blockIdx.x << 32) | 0x7fffffffu,
                   ((unsigned long long)st.polls << 8) | (unsigned long long)st.exit_reason,
                   *reinterpret_cast<volatile unsigned long long*>(&p.sched->gemm_q[0]),
                   globaltimer());
  }
}

template <int P>
__global__ void __launch_bounds__(kThreads + 32, 1)
    moe_persistent_kernel(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  char* smem;
  Ctrl* c;
  CtaState st;
  cta_setup<P>(p, maps, smem, c, st, true);
  if (threadIdx.x < kThreads) compute_loop<P>(p, maps, smem, c, st);
  else scheduler_loop<P>(p, c, st);
  cta_teardown<P>(c, true);
}

// ------------------------------------------------------------------ static persistent megakernel
// The static fused baseline: one launch, one CTA per SM, every stage's tasks
// assigned round-robin to the workers (task i of a stage to worker i mod
// workers), and a grid-wide barrier between stages -- no queue, no dependency
// counters, no overlap of stages.  Same tiles as the other two modes, so its
// gap to the persistent kernel is what the queue, the counters and the
// cross-stage overlap buy beyond saving launches.  Launched cooperatively, so
// every CTA is resident and the barrier can wait; each wait is bounded by
// the deadline.

// Grid-wide barrier: every CTA arrives on a counter; the last one resets it
// and bumps the generation the others wait for.  False on timeout or abort.
__device__ bool grid_barrier(const Params& p, Ctrl* c, int& gen, const CtaState& st) {
  release_writes();
  if (threadIdx.x == 0) {
    int ok = 1;
    const int old = atom_add_acq_rel(&p.sched->bar_count, 1);
    if (old == (int)gridDim.x - 1) {
      p.sched->bar_count = 0;
      st_release(&p.sched->bar_gen, gen + 1);
    } else {
      uint32_t backoff = 32;
      while (ld_acquire(&p.sched->bar_gen) == gen) {
        if (ld_relaxed(&p.sched->status) != 0) {
          ok = 0;
          break;
        }
        if (globaltimer() > st.deadline) {
          set_status(p, MOE_E_TIMEOUT, 40);
          ok = 0;
          break;
        }
        __nanosleep(backoff);
        if (backoff < 256) backoff <<= 1;
      }
    }
    c->flag = ok;
  }
  cta_sync();
  ++gen;
  fence_acq_rel_gpu();
  return c->flag != 0;
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1)
    moe_static_kernel(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  char* smem;
  Ctrl* c;
  CtaState st;
  cta_setup<P>(p, maps, smem, c, st, true);
  // tasks go round-robin to the workers; every CTA of a worker runs each one
  const int W = (int)gridDim.x / P, w = st.worker;
  int gen = 0;
  for (int i = w; i < p.n_route_tasks; i += W)
    route_task<P>(p, maps, i / p.route_ks, i % p.route_ks, smem, c, st);
  bool ok = grid_barrier(p, c, gen, st);
  if (ok && blockIdx.x == 0) plan_task(p, smem, c, false);
  ok = ok && grid_barrier(p, c, gen, st);
  const int n_groups = ok ? ld_relaxed(&p.sched->n_groups) : 0;
  const int n_routed = n_groups - p.n_shared_groups;
  for (int i = w; ok && i < n_routed * 8; i += W) {  // (routed group, chunk)
    const int g = p.n_shared_groups + (i >> 3), ch = i & 7;
    if (ch * gather_rows(p) < load_group(p, g).nrows) gather_task(p, g, ch, st.rank, P, smem, c, st);
  }
  ok = ok && grid_barrier(p, c, gen, st);
  for (int i = w; ok && i < n_groups * p.n_ftiles; i += W)
    gateup_task<P>(p, maps, task_id(kTaskGateUp, i), smem, c, st);
  ok = ok && grid_barrier(p, c, gen, st);
  const int n_down = p.n_dtiles * p.ks;
  for (int i = w; ok && i < n_groups * n_down; i += W)
    down_task<P>(p, maps, task_id(kTaskDown, i), smem, c, st);
  ok = ok && grid_barrier(p, c, gen, st);
  for (int i = w; ok && i < p.n_comb; i += W) {
    combine_task(p, i, st.rank, P, smem, c, st);
    cta_sync();
  }
  cta_teardown<P>(c, true);
}

// ------------------------------------------------------------------ ablation: one kernel per stage
// The tensor-core stages (router, gate/up, down) launch one worker (a CTA,
// or a cluster of two) per task; the others one CTA per task.

template <int P>
__global__ void __launch_bounds__(kThreads, 1)
    k_route(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  char* smem;
  Ctrl* c;
  CtaState st;
  cta_setup<P>(p, maps, smem, c, st, true);
  const int i = (int)blockIdx.x / P;
  route_task<P>(p, maps, i / p.route_ks, i % p.route_ks, smem, c, st);
  cta_teardown<P>(c, true);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_plan(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  char* smem;
  Ctrl* c;
  CtaState st;
  cta_setup<1>(p, maps, smem, c, st, false);
  plan_task(p, smem, c, false);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_gather(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  const int g = p.n_shared_groups + (int)(blockIdx.x >> 3), ch = blockIdx.x & 7;
  if (g >= p.sched->n_groups) return;
  const Group G = load_group(p, g);
  if (ch * gather_rows(p) >= G.nrows) return;
  char* smem;
  Ctrl* c;
  CtaState st;
  cta_setup<1>(p, maps, smem, c, st, false);
  gather_task(p, g, ch, 0, 1, smem, c, st);
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1)
    k_gateup(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  const int i = (int)blockIdx.x / P;  // the same for both CTAs of a cluster
  const int g = i / p.n_ftiles;
  if (g >= p.sched->n_groups) return;
  char* smem;
  Ctrl* c;
  CtaState st;
  cta_setup<P>(p, maps, smem, c, st, true);
  gateup_task<P>(p, maps, task_id(kTaskGateUp, i), smem, c, st);
  cta_teardown<P>(c, true);
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1)
    k_down(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  const int n_down = p.n_dtiles * p.ks;
  const int i = (int)blockIdx.x / P;  // the same for both CTAs of a cluster
  const int g = i / n_down;
  if (g >= p.sched->n_groups) return;
  char* smem;
  Ctrl* c;
  CtaState st;
  cta_setup<P>(p, maps, smem, c, st, true);
  down_task<P>(p, maps, task_id(kTaskDown, i), smem, c, st);
  cta_teardown<P>(c, true);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_combine(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  char* smem;
  Ctrl* c;
  CtaState st;
  cta_setup<1>(p, maps, smem, c, st, false);
  combine_task(p, blockIdx.x, 0, 1, smem, c, st);
}

}  // namespace moe

// ====================================================================== host side

using namespace moe;

// Scratch of moe_layer_forward_noalloc: a file-scope device array, so that
// entry point needs no allocation call.  Every GPU that loads this library
// holds it until the process exits.
constexpr size_t kNoallocScratchBytes = 32u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorString(e);
  return MOE_E_CUDA;
}

#define CK(call)                                   \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D bf16 tensor [rows, cols] (row-major), box 64 columns x box_rows rows,
// 128-byte swizzle, out-of-range elements read as zero.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int kSmemBudget = 227 * 1024;

// Sizes that bound the workspace for T_max tokens.
struct Bounds {
  int T;
  int n_route;      // router tiles at the smallest tile
  int max_groups;   // shared + routed groups at the smallest token tile (32)
  int n_comb;       // combine tiles at one token per tile
  int mover_cap, gemm_cap;
  size_t y_elems;   // elements of Y storage (fp32 words or 2x bf16)
  // the debug claimed-twice bitmap: router, gather, gate/up, down and combine
  // tasks at their largest counts (one CTA per worker, 4 K splits)
  int claim_gather_off, claim_gateup_off, claim_down_off, claim_comb_off, claim_bits;
};

}  // namespace

struct moe_layer {
  int d, f, E, k, S;
  int T_max = 0;
  int device = -1;
  int num_sms = 0;
  int max_pairs = 0;  // clusters of two CTAs the persistent kernel can keep resident
  // options
  int pair_opt = 0;  // CTAs per worker: 0 = automatic, 1, 2
  int front_split = -1;  // the spatial split also governs the gathers: -1 = auto
  // routed gate/up tiles gather their token rows themselves: off by default
  // -- bit-identical, but the 16-byte copies keep too few bytes in flight
  // beside the weight stream (gate/up tiles 49 -> 99 us on decode, 50 -> 107
  // us on skew; decode 522 -> 800 us, prefill 6260 -> 10340 us on one box)
  int fold_gather = 0;
  int mode = MOE_MODE_PERSISTENT;
  unsigned long long timeout_ns = 2000000000ull;
  int mover_override = 0;
  int grid_override = 0;
  int split_k = 0;
  int bn_opt = 0;
  int fault_drop = -1;
  int fault_drop_type = 0;
  int fault_corrupt = 0;
  int fault_repush = -1;
  int debug_claims = 0;
  int rt_opt = 0;
  int ahead_opt = -1;
  int release = kReleaseExpert;
  int prefetch = 1;
  int bands = 1;
  int route_splits = 0;
  long long l2_pf = -1;  // bytes; -1 = auto
  int trace_cap = 0;
  unsigned long long* trace = nullptr;
  const float* bias = nullptr;
  // workspace
  char* ws = nullptr;
  size_t ws_bytes = 0;
  Bounds B{};
  // offsets into ws
  size_t o_idx, o_wgt, o_rank, o_tile, o_counts, o_offsets, o_perm, o_pos, o_xp, o_h, o_y,
      o_groups, o_rpart, o_rsd, o_rmask, o_zero, o_gd, o_gu, o_cd, o_nd, o_claimed, o_sched, o_zero_end, o_ring, o_ring_m, o_ring_g, o_ring_gl,
      o_ring_end;
  // where the last forward's routing and scheduler state live: the reserved
  // workspace, or the no-allocation entry point's scratch array
  struct View {
    char* ws = nullptr;
    size_t o_idx = 0, o_wgt = 0, o_counts = 0, o_offsets = 0, o_perm = 0, o_pos = 0, o_sched = 0;
  } view;
  // host staging for moe_layer_forward_host
  void* x_dev_stage = nullptr;
  void* out_dev_stage = nullptr;
  // last forward
  Sched last{};
  bool last_valid = false;
  int last_grid = 0;
  int last_bn = 0, last_ks = 0, last_bands = 0;  // tiling of the last forward
  int last_ybytes = 0;  // bytes the combine reads per expert-output value
  int last_ct = 0;      // tokens per combine tile
  int last_pair = 0;    // CTAs per worker
  int last_T = 0;
};

namespace {

Bounds make_bounds(const moe_layer* h, int T) {
  Bounds b{};
  b.T = T;
  const long long Tk = (long long)T * h->k;
  b.n_route = std::max(1, cdiv(T, kRouteTokensSmall));  // at the smallest router tile
  const int shared_groups = h->S ? cdiv(T, 32) : 0;
  b.max_groups = shared_groups + cdiv(Tk, 32) + std::min<long long>(h->E, Tk) + 1;
  b.n_comb = 2 * std::max(T, 1);  // one token per tile, two d bands
  b.mover_cap = cdiv(Tk, 32) + b.max_groups + b.n_comb + 16;
  const int n_ft = h->f / 128, n_dt = cdiv(h->d, 256);
  b.gemm_cap = b.max_groups * (n_ft + n_dt * 4) + 16;
  b.claim_gather_off = b.n_route * kMaxRouteKs;
  b.claim_gateup_off = b.claim_gather_off + b.max_groups * 8;
  b.claim_down_off = b.claim_gateup_off + b.max_groups * n_ft;
  b.claim_comb_off = b.claim_down_off + b.max_groups * n_dt * 4;
  b.claim_bits = b.claim_comb_off + b.n_comb;
  const long long rows = Tk + (long long)T * h->S;
  // fp32 partials for up to 4 K splits when small, else bf16 (half a word each)
  const long long small = rows * h->d * 4;
  b.y_elems = (size_t)(small <= (1ll << 27) ? small : (rows * h->d + 1) / 2);
  return b;
}

void layout(moe_layer* h, const Bounds& b) {
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o = align_up(o + bytes, 256);
    return r;
  };
  const size_t Tk = (size_t)b.T * h->k;
  const size_t rows = Tk + (size_t)b.T * h->S;
  h->o_idx = take(Tk * 4);
  h->o_wgt = take(Tk * 4);
  h->o_rank = take(Tk * 4);
  h->o_tile = take((size_t)b.n_route * h->E * 4);
  h->o_rmask = take((size_t)b.n_route * h->E * 16);
  h->o_counts = take(h->E * 4);
  h->o_offsets = take((h->E + 1) * 4);
  h->o_perm = take(Tk * 4);
  h->o_pos = take(Tk * 4);
  h->o_xp = take((Tk + 64) * h->d * 2);
  h->o_h = take((rows + 64) * h->f * 2);
  h->o_y = take(b.y_elems * 4 + 4096);
  h->o_groups = take((size_t)b.max_groups * sizeof(Group));
  h->o_rpart = take((size_t)std::max(h->num_sms, 1) * kRouteTokens * (((h->E + 15) / 16) * 16) * 4);
  h->o_zero = o;
  h->o_sched = take(sizeof(Sched));
  h->o_rsd = take((size_t)b.n_route * 4);
  h->o_gd = take((size_t)b.max_groups * 4);
  h->o_gu = take((size_t)b.max_groups * 4);
  h->o_cd = take((size_t)b.n_comb * 4);
  h->o_nd = take((size_t)b.n_comb * 4);
  h->o_claimed = take((size_t)(b.claim_bits + 31) / 32 * 4);
  h->o_zero_end = o;
  h->o_ring = o;
  h->o_ring_m = take((size_t)kShards * (b.mover_cap / kShards * 2 + 64) * 4);
  h->o_ring_g = take((size_t)kShards * (b.gemm_cap / kShards * 2 + 64) * 4);
  h->o_ring_gl = take((size_t)kShards * (b.gemm_cap / kShards * 2 + 64) * 4);
  h->o_ring_end = o;
  h->ws_bytes = o;
}

// Tiling of one forward pass.
struct Tiling {
  int pair, bn, stages, stage_bytes, smem, ks, rt, ct, y_f32;
};

// CTAs per worker: a CTA pair sharing each GEMM tile (.cta_group::2) when the
// experts' row groups are large -- a pair stages half the token rows per SM
// and halves the shared-memory operand traffic of a 256-token tile -- and one
// CTA when they are small, where the pair's cross-SM handshakes and the
// halved number of independent mover workers cost more than they save
// (same-box measurements: decode and fine layers faster with one CTA, the
// prefill layers with pairs).
int choose_pair(const moe_layer* h, int T) {
  if (h->pair_opt == 1 || h->pair_opt == 2) return h->pair_opt;
  const long long rows_per_expert = (long long)T * h->k / h->E;
  return rows_per_expert >= kPairMinRows ? 2 : 1;
}

int choose_tiling(const moe_layer* h, int T, bool whole_rows, Tiling* t) {
  const long long Tk = (long long)T * h->k;
  const int P = choose_pair(h, T);
  t->pair = P;
  int bn = h->bn_opt;
  if (bn <= 0) {
    // at least 160 tokens (or twice the mean expert load): the MMA's N is the
    // group's actual rows, so a larger cap wastes nothing and keeps experts
    // whose load varies from being split into sibling groups that re-read
    // the weights (fine workload: 322, 308, 304, 302, 313 us at 64, 96, 128,
    // 160, 256; the decode workload is the same at 128 and 160)
    const long long avg = Tk / h->E;
    long long want = std::max<long long>(160, 2 * avg);
    want = std::min<long long>(want, std::max(T, 1));
    bn = (int)std::min<long long>(256, ((want + 31) / 32) * 32);
  }
  bn = std::max(32, std::min(256, ((bn + 31) / 32) * 32));
  t->bn = bn;
  // a stage holds this CTA's 128 rows of each weight operand and its share of
  // the tile's token rows (all of them, or half for a CTA pair)
  t->stage_bytes = 2 * kABoxBytes + cdiv(bn / P, kBBoxRows) * kBBoxBytes;
  // the router's tile keeps x (16 KB) then this CTA's share of Wr's E rows
  const int e_mma = ((h->E + 16 * P - 1) / (16 * P)) * (16 * P);
  t->stage_bytes =
      std::max(t->stage_bytes, kABoxBytes + cdiv(e_mma / P, kBBoxRows) * kBBoxBytes);
  const int ctrl = (int)align_up(sizeof(Ctrl), 1024);
  t->stages = std::min(8, (kSmemBudget - 1024 - ctrl) / t->stage_bytes);
  if (t->stages < 2) return fail(MOE_E_INVAL, "tile too large for shared memory");
  if ((size_t)t->stages * t->stage_bytes < route_smem_bytes(h->E))
    return fail(MOE_E_INVAL, "router logits do not fit in shared memory");
  t->smem = 1024 + t->stages * t->stage_bytes + ctrl;
  // down-projection K split: fp32 partials when the batch is small
  const int kblocks = h->f / kBK;
  const long long rows = Tk + (long long)T * h->S;
  int ks = h->split_k;
  if (ks <= 0) {
    // the smallest split that gives about 1.5 waves of down tasks over the
    // workers, counting one row group per expert that can be touched
    // (decode, one CTA per worker: 2 -- 518 us against 521 us at 4 and 529 us
    // at 1)
    const long long groups = std::min<long long>(h->E, Tk) + h->S;
    const long long want = 3ll * std::max(h->num_sms / P, 1) / 2;
    ks = 1;
    while (ks < 4 && groups * cdiv(h->d, 2 * kBM * P) * ks < want) ks <<= 1;
  }
  while (ks > 1 && (kblocks % ks != 0 || (size_t)rows * h->d * ks > h->B.y_elems)) ks >>= 1;
  if (ks < 1) ks = 1;
  t->ks = ks;
  t->y_f32 = ks > 1 ? 1 : ((size_t)rows * h->d <= h->B.y_elems ? 1 : 0);
  // router tile: 64 tokens for small layers with many experts (four threads
  // per token share the top-k and softmax over E, and twice the tiles spread
  // over the SMs; with few experts the extra threads have nothing to do and
  // the extra tiles only add tasks), else 128
  const bool small_rt = T <= kSmallRouteT && h->E >= kSmallRouteMinE;
  t->rt = h->rt_opt ? h->rt_opt : (small_rt ? kRouteTokensSmall : kRouteTokens);
  if (cdiv(T, t->rt) > kMaxE) return fail(MOE_E_INVAL, "too many router tiles: use 128-token tiles");
  // combine tile, <= 256 (token, slot) pairs: one per worker when the
  // combine is split in two d bands (each task then covers part of a row),
  // two per worker with one band; a pair's CTAs split a tile's tokens
  const bool two_bands = h->bands && cdiv(h->d, 2 * kBM * P) >= 2 && !whole_rows;
  int ct = cdiv(T, (two_bands ? 1 : 2) * std::max(h->num_sms / P, 1));
  ct = std::max(1, std::min(ct, kThreads / h->k));
  t->ct = ct;
  return MOE_OK;
}

int set_error_from_sched(const Sched& s) {
  if (s.status == MOE_E_TIMEOUT) {
    g_err = "device wait timed out (site " + std::to_string(s.err_info) + ")";
    return MOE_E_TIMEOUT;
  }
  if (s.status != 0) {
    g_err = "device scheduler inconsistency (site " + std::to_string(s.err_info) + ")";
    return MOE_E_DEVICE;
  }
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The dynamic shared-memory limit of every kernel (both widths of worker).
cudaError_t set_kernel_smem(int bytes) {
  void (*kernels[])(Params, Maps) = {moe_persistent_kernel<1>, moe_persistent_kernel<2>,
                                     moe_static_kernel<1>,     moe_static_kernel<2>,
                                     k_route<1>,               k_route<2>,
                                     k_gateup<1>,              k_gateup<2>,
                                     k_down<1>,                k_down<2>,
                                     k_plan,                   k_gather,
                                     k_combine};
  for (auto k : kernels) {
    cudaError_t e = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Launch one of the kernels: `pair` as clusters of two CTAs (the tensor-core
// kernels built for CTA pairs), `coop` cooperatively.
cudaError_t launch_kernel(void (*kern)(Params, Maps), int grid, int threads, int smem,
                          cudaStream_t s, bool pair, bool coop, const Params& p, const Maps& m) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int n = 0;
  if (pair) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = 2;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  if (coop) {
    at[n].id = cudaLaunchAttributeCooperative;
    at[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = (unsigned)n;
  return cudaLaunchKernelEx(&cfg, kern, p, m);
}

// Clusters of two CTAs of the persistent kernel (one CTA per SM at its shared
// memory size) the device keeps resident at once; 0 if the query fails.
int query_max_pairs(int num_sms) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max(2, num_sms / 2 * 2));
  cfg.blockDim = dim3(kThreads + 32);
  cfg.dynamicSmemBytes = kSmemBudget;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = 2;
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void*)moe_persistent_kernel<2>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

extern "C" {

const char* moe_last_error(void) { return g_err.c_str(); }

moe_layer_t* moe_layer_create(int d, int f, int E, int k, int shared_experts) {
  if (d <= 0 || d % 128 != 0) {
    g_err = "d must be a positive multiple of 128";
    return nullptr;
  }
  if (d > kMaxD) {
    // a gather task stages whole bf16 token rows in the pipeline's shared
    // memory (at least ~145 KB under every tiling): rows of up to 64 KB fit
    g_err = "d must be at most 32768";
    return nullptr;
  }
  if (f <= 0 || f % 128 != 0) {
    g_err = "f must be a positive multiple of 128";
    return nullptr;
  }
  if (E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK) {
    g_err = "need 1 <= k <= E <= 256 and k <= 16";
    return nullptr;
  }
  if (shared_experts < 0 || shared_experts > 1) {
    g_err = "shared_experts must be 0 or 1";
    return nullptr;
  }
  moe_layer_t* h = new (std::nothrow) moe_layer();
  if (!h) {
    g_err = "out of host memory";
    return nullptr;
  }
  h->d = d;
  h->f = f;
  h->E = E;
  h->k = k;
  h->S = shared_experts;
  g_err.clear();
  return h;
}

long long moe_layer_workspace_bytes(const moe_layer_t* h, int T_max) {
  if (!h || T_max < 0) return -1;
  moe_layer tmp = *h;
  tmp.ws = nullptr;
  Bounds b = make_bounds(&tmp, std::max(T_max, 1));
  layout(&tmp, b);
  return (long long)tmp.ws_bytes;
}

int moe_layer_reserve(moe_layer_t* h, int T_max, void* stream) {
  if (!h) return fail(MOE_E_INVAL, "null handle");
  if (T_max < 1 || T_max > kMaxE * kRouteTokens)
    return fail(MOE_E_INVAL, "T_max out of range (1..32768)");
  CK(cudaGetDevice(&h->device));
  CK(cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device));
  int cc_major = 0, cc_minor = 0;
  CK(cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, h->device));
  CK(cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, h->device));
  if (cc_major != 10 || cc_minor != 3)
    return fail(MOE_E_INVAL, "this library is built for sm_103a (GB300) only");
  if (!encode_fn()) return fail(MOE_E_CUDA, "cuTensorMapEncodeTiled is not available");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (h->ws) {
    CK(cudaStreamSynchronize(s));
    CK(cudaFree(h->ws));
    h->ws = nullptr;
  }
  Bounds b = make_bounds(h, T_max);
  layout(h, b);
  h->B = b;
  if (cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess) {
    h->ws = nullptr;
    cudaGetLastError();
    return fail(MOE_E_NOMEM, "workspace allocation failed");
  }
  CK(cudaMemsetAsync(h->ws, 0, h->ws_bytes, s));
  if (h->x_dev_stage) {
    cudaFree(h->x_dev_stage);
    cudaFree(h->out_dev_stage);
    h->x_dev_stage = h->out_dev_stage = nullptr;
  }
  h->T_max = T_max;
  CK(set_kernel_smem(kSmemBudget));
  h->max_pairs = query_max_pairs(h->num_sms);
  g_err.clear();
  return MOE_OK;
}

int moe_layer_set_router_bias(moe_layer_t* h, const float* bias) {
  if (!h) return fail(MOE_E_INVAL, "null handle");
  if (bias && !aligned16(bias)) return fail(MOE_E_INVAL, "bias must be 16-byte aligned");
  h->bias = bias;
  return MOE_OK;
}

int moe_layer_set_option(moe_layer_t* h, int key, long long v) {
  if (!h) return fail(MOE_E_INVAL, "null handle");
  switch (key) {
    case MOE_OPT_MODE:
      if (v != MOE_MODE_PERSISTENT && v != MOE_MODE_MULTIKERNEL && v != MOE_MODE_STATIC)
        return fail(MOE_E_INVAL, "bad mode");
      h->mode = (int)v;
      break;
    case MOE_OPT_TIMEOUT_NS:
      if (v < 1000) return fail(MOE_E_INVAL, "timeout below 1 us");
      h->timeout_ns = (unsigned long long)v;
      break;
    case MOE_OPT_MOVER_CTAS:
      if (v < 0) return fail(MOE_E_INVAL, "negative mover count");
      h->mover_override = (int)v;
      break;
    case MOE_OPT_GRID_CTAS:
      if (v < 0 || v > 4096) return fail(MOE_E_INVAL, "grid out of range");
      h->grid_override = (int)v;
      break;
    case MOE_OPT_SPLIT_K:
      if (v != 0 && v != 1 && v != 2 && v != 4) return fail(MOE_E_INVAL, "split_k must be 0,1,2,4");
      h->split_k = (int)v;
      break;
    case MOE_OPT_TOKENS_PER_TILE:
      if (v != 0 && (v < 16 || v > 256 || v % 16)) return fail(MOE_E_INVAL, "tokens per tile must be 16..256, multiple of 16");
      h->bn_opt = (int)v;
      break;
    case MOE_OPT_FAULT_DROP_TASK:
      h->fault_drop = v < 0 ? -1 : (int)v;
      break;
    case MOE_OPT_FAULT_DROP_TYPE:
      if (v != 0 && v != kTaskGather && v != kTaskGateUp && v != kTaskDown)
        return fail(MOE_E_INVAL, "dropped task type must be 0, 2 (gather), 3 (gate/up) or 4 (down)");
      h->fault_drop_type = (int)v;
      break;
    case MOE_OPT_FAULT_CORRUPT_COUNT:
      if (v < -(1 << 20) || v > (1 << 20)) return fail(MOE_E_INVAL, "count corruption out of range");
      h->fault_corrupt = (int)v;
      break;
    case MOE_OPT_FAULT_REPUSH:
      h->fault_repush = v < 0 ? -1 : (int)std::min<long long>(v, 1 << 30);
      break;
    case MOE_OPT_DEBUG_CLAIMS:
      h->debug_claims = v ? 1 : 0;
      break;
    case MOE_OPT_CLAIM_AHEAD:
      if (v < -1) return fail(MOE_E_INVAL, "claim-ahead depth must be -1, 0 or positive");
      h->ahead_opt = (int)v;
      break;
    case MOE_OPT_TRACE: {
      if (v < 0 || v > (1 << 24)) return fail(MOE_E_INVAL, "trace capacity out of range");
      if (h->trace) {
        cudaDeviceSynchronize();
        cudaFree(h->trace);
        h->trace = nullptr;
      }
      h->trace_cap = 0;
      if (v > 0) {
        if (cudaMalloc(&h->trace, (size_t)v * 32) != cudaSuccess) {
          cudaGetLastError();
          h->trace = nullptr;
          return fail(MOE_E_NOMEM, "trace allocation failed");
        }
        h->trace_cap = (int)v;
      }
      break;
    }
    case MOE_OPT_RELEASE:
      if (v != kReleaseAll && v != kReleaseExpert) return fail(MOE_E_INVAL, "release policy must be 0 or 1");
      h->release = (int)v;
      break;
    case MOE_OPT_PREFETCH:
      h->prefetch = v ? 1 : 0;
      break;
    case MOE_OPT_BANDS:
      h->bands = v ? 1 : 0;
      break;
    case MOE_OPT_L2_PREFETCH:
      if (v < -1) return fail(MOE_E_INVAL, "L2 prefetch must be -1 (auto), 0 (off) or a byte count");
      h->l2_pf = v;
      break;
    case MOE_OPT_ROUTE_SPLITS:
      if (v < 0 || v > kMaxRouteKs) return fail(MOE_E_INVAL, "router K splits must be 0..8");
      h->route_splits = (int)v;
      break;
    case MOE_OPT_FOLD_GATHER:
      h->fold_gather = v ? 1 : 0;
      break;
    case MOE_OPT_FRONT_SPLIT:
      if (v < -1 || v > 1) return fail(MOE_E_INVAL, "front split must be -1 (auto), 0 or 1");
      h->front_split = (int)v;
      break;
    case MOE_OPT_PAIR:
      if (v != 0 && v != 1 && v != 2) return fail(MOE_E_INVAL, "CTAs per worker must be 0 (auto), 1 or 2");
      h->pair_opt = (int)v;
      break;
    case MOE_OPT_ROUTE_TOKENS:
      if (v != 0 && v != kRouteTokens && v != kRouteTokensSmall)
        return fail(MOE_E_INVAL, "router tiles are 64 or 128 tokens (0: automatic)");
      h->rt_opt = (int)v;
      break;
    default:
      return fail(MOE_E_INVAL, "unknown option");
  }
  return MOE_OK;
}

namespace {

// The residual add + RMSNorm fused into the combine (or none).
struct Fuse {
  const void* residual;
  const void* gamma;
  float eps;
  void* norm_out;
};

int forward_impl(moe_layer_t* h, int T, const void* x, const void* router_w, const void* w_gate,
                 const void* w_up, const void* w_down, void* out, const Fuse* fz, void* stream) {
  if (!h) return fail(MOE_E_INVAL, "null handle");
  if (!h->ws) return fail(MOE_E_STATE, "moe_layer_reserve was not called");
  if (T < 0 || T > h->T_max) return fail(MOE_E_INVAL, "T out of range (0..T_max)");
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !w_gate || !w_up || !w_down || !out)
    return fail(MOE_E_INVAL, "null tensor pointer");
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(w_gate) || !aligned16(w_up) ||
      !aligned16(w_down) || !aligned16(out))
    return fail(MOE_E_INVAL, "tensors must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Tiling tl;
  int rc = choose_tiling(h, T, fz != nullptr, &tl);
  if (rc) return rc;

  Params p;
  memset(&p, 0, sizeof(p));
  p.T = T;
  p.d = h->d;
  p.f = h->f;
  p.E = h->E;
  p.k = h->k;
  p.S = h->S;
  p.bn_max = tl.bn;
  p.stages = tl.stages;
  p.stage_bytes = tl.stage_bytes;
  const int P = tl.pair;
  p.pair = P;
  // gather tasks of 64 rows per CTA in large layers (prefill layer, one
  // kernel per stage: the gathers move their 1.9 GB in 273 us at 64 rows per
  // CTA; the persistent kernel's 32-row tasks took 370 us of each worker),
  // 32 in small ones, where the gathers are few and on the critical path
  p.gather_cta_rows = (long long)T * h->k >= kGatherBigRows ? kGatherRowsCtaBig : kGatherRowsCta;
  p.n_ftiles = cdiv(h->f, kBM * P);
  p.n_dtiles = cdiv(h->d, 2 * kBM * P);
  p.ks = tl.ks;
  p.kb_down = (h->f / kBK) / tl.ks;
  p.rt = tl.rt;
  p.n_route = cdiv(T, tl.rt);
  {
    // K splits of the router: spread few router tiles over the SMs, with at
    // least 8 k blocks per split (fine workload: 4 splits, 301 us against
    // 303 us at 8) and at most kMaxRouteKs.  The partial logits hold one
    // [128, E] block per SM, so tiles x splits never exceeds the SM count,
    // the option included.
    const int nkb = h->d / kBK;
    const int cap = std::max(1, std::max(h->num_sms, 1) / p.n_route);
    int ks = std::min(kMaxRouteKs, std::min(std::max(1, nkb / 8), cap));
    if (h->route_splits > 0) ks = std::min(std::min(h->route_splits, nkb), cap);
    p.route_ks = std::max(1, ks);
    p.n_route_tasks = cdiv(p.n_route, P) * p.route_ks;
  }
  p.release = h->release;
  p.prefetch = h->prefetch;
  // the front's spatial split: on without a shared expert (skew layer 1047 ->
  // 1039 us on one box), off with one, whose ready tiles would then run
  // before the routed experts' (prefill layer 6468 -> 6986 us)
  p.front_split = h->front_split < 0 ? (h->S == 0 ? 1 : 0) : h->front_split;
  p.fold_gather = h->fold_gather;
  p.ct = tl.ct;
  // d bands: the down tiles of the last quarter of d (at least one tile)
  // have low priority, so the other band's combines overlap them
  // (with the fused residual + RMSNorm a tile's norm waits for its last band,
  // which runs in the tail: one band measured faster there)
  p.n_bands = (h->bands && p.n_dtiles >= 2 && !fz) ? 2 : 1;
  p.dt_lo0 = p.n_bands == 2 ? p.n_dtiles - std::max(1, p.n_dtiles / 4) : p.n_dtiles;
  p.n_comb = cdiv(T, tl.ct) * p.n_bands;
  p.n_shared_groups = h->S ? cdiv(T, tl.bn) : 0;
  p.n_static_gemm = p.n_shared_groups * p.n_ftiles;
  p.y_f32 = tl.y_f32;
  p.rows_y = T * h->k + T * h->S;
  const long long Tk = (long long)T * h->k;
  p.max_groups = p.n_shared_groups + cdiv(Tk, tl.bn) + (int)std::min<long long>(h->E, Tk);
  if (p.max_groups > h->B.max_groups) return fail(MOE_E_INVAL, "group capacity exceeded");
  p.mover_seg = h->B.mover_cap / kShards * 2 + 64;
  p.gemm_seg = h->B.gemm_cap / kShards * 2 + 64;
  p.fault_drop = h->fault_drop;
  p.fault_drop_type = h->fault_drop_type;
  p.fault_corrupt = h->fault_corrupt;
  p.fault_repush = h->fault_repush;
  p.mover_override = h->mover_override;
  p.trace = h->trace;
  p.trace_cap = h->trace_cap;
  p.timeout_ns = h->timeout_ns;
  // cost-model constants per worker (P CTAs): beta for the movers and one
  // SM's share of 1925 TF/s for the GEMMs, per CTA.  beta is calibrated, not
  // a copy rate (a gather CTA moves ~35 GB/s): GEMM workers steal gathers and
  // combines whenever no tile is ready, so the movers only need to keep the
  // mover work going beside the GEMMs, and sweeps of the mover count on the
  // skew and prefill_small layers put the fastest split at about 4 of 76
  // workers -- the split this beta gives them
  p.beta_move = 140e9f * (float)P;
  p.phi_gemm = (1925e12f / 152.f) * (float)P;
  p.hbm_bw = 6.79e12f;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.wr = static_cast<const __nv_bfloat16*>(router_w);
  p.bias = h->bias;
  if (fz) {
    p.residual = static_cast<const __nv_bfloat16*>(fz->residual);
    p.gamma = static_cast<const __nv_bfloat16*>(fz->gamma);
    p.norm_out = static_cast<__nv_bfloat16*>(fz->norm_out);
    p.eps = fz->eps;
  }
  p.w_gate = static_cast<const __nv_bfloat16*>(w_gate);
  p.w_up = static_cast<const __nv_bfloat16*>(w_up);
  p.out = static_cast<__nv_bfloat16*>(out);
  {
    // L2 prefetch of the first gate/up tiles at launch (persistent mode):
    // auto when no shared expert keeps HBM busy at the start and the routing
    // is expected to be balanced (the mean expert load fits half a GEMM
    // tile), so keeping experts in index order costs no load balance
    long long pf = h->l2_pf;
    if (pf < 0) {
      const bool balanced = h->S == 0 && Tk <= (long long)h->E * (tl.bn / 2);
      pf = balanced ? (96ll << 20) : 0;
    }
    if (h->mode != MOE_MODE_PERSISTENT) pf = 0;
    p.l2_pf_bytes = pf;
    p.index_order = pf > 0 ? 1 : 0;
  }
  char* w = h->ws;
  p.idx = reinterpret_cast<int*>(w + h->o_idx);
  p.wgt = reinterpret_cast<float*>(w + h->o_wgt);
  p.rank = reinterpret_cast<int*>(w + h->o_rank);
  p.tile_cnt = reinterpret_cast<int*>(w + h->o_tile);
  p.rmask = reinterpret_cast<uint32_t*>(w + h->o_rmask);
  p.counts = reinterpret_cast<int*>(w + h->o_counts);
  p.offsets = reinterpret_cast<int*>(w + h->o_offsets);
  p.perm = reinterpret_cast<int*>(w + h->o_perm);
  p.pos = reinterpret_cast<int*>(w + h->o_pos);
  p.Xp = reinterpret_cast<__nv_bfloat16*>(w + h->o_xp);
  p.H = reinterpret_cast<__nv_bfloat16*>(w + h->o_h);
  p.Y = w + h->o_y;
  p.groups = reinterpret_cast<Group*>(w + h->o_groups);
  p.gather_done = reinterpret_cast<int*>(w + h->o_gd);
  p.gu_done = reinterpret_cast<int*>(w + h->o_gu);
  p.comb_done = reinterpret_cast<int*>(w + h->o_cd);
  p.norm_done = reinterpret_cast<int*>(w + h->o_nd);
  p.ring_mover = reinterpret_cast<int*>(w + h->o_ring_m);
  p.ring_gemm = reinterpret_cast<int*>(w + h->o_ring_g);
  p.ring_gemm_lo = reinterpret_cast<int*>(w + h->o_ring_gl);
  p.sched = reinterpret_cast<Sched*>(w + h->o_sched);
  p.claimed = h->debug_claims ? reinterpret_cast<uint32_t*>(w + h->o_claimed) : nullptr;
  p.claim_gather_off = h->B.claim_gather_off;
  p.claim_gateup_off = h->B.claim_gateup_off;
  p.claim_down_off = h->B.claim_down_off;
  p.claim_comb_off = h->B.claim_comb_off;
  p.claim_bits = h->B.claim_bits;
  p.rpart = reinterpret_cast<float*>(w + h->o_rpart);
  p.rsplit_done = reinterpret_cast<int*>(w + h->o_rsd);

  Maps m;
  const int nt = h->E + h->S;
  bool ok = encode_2d(&m.wg, w_gate, (uint64_t)nt * h->f, h->d, kBM) &&
            encode_2d(&m.wu, w_up, (uint64_t)nt * h->f, h->d, kBM) &&
            encode_2d(&m.wd, w_down, (uint64_t)nt * h->d, h->f, kBM) &&
            encode_2d(&m.xp, p.Xp, (uint64_t)Tk, h->d, kBBoxRows) &&
            encode_2d(&m.x, x, (uint64_t)T, h->d, kBBoxRows) &&
            encode_2d(&m.h, p.H, (uint64_t)p.rows_y, h->f, kBBoxRows) &&
            encode_2d(&m.xr, x, (uint64_t)T, h->d, kRouteTokens) &&
            encode_2d(&m.wr, router_w, (uint64_t)h->E, h->d, kBBoxRows);
  if (!ok) return fail(MOE_E_INVAL, "tensor map encoding failed");

  // scheduler counters and task rings are contiguous: one memset resets them
  CK(cudaMemsetAsync(w + h->o_zero, 0, h->o_ring_end - h->o_zero, s));
  // workers: every SM (one CTA each), or every SM pair the device keeps
  // resident as a cluster
  const int max_workers = P == 2 ? (h->max_pairs > 0 ? std::min(h->max_pairs, h->num_sms / 2)
                                                     : h->num_sms / 2)
                                 : h->num_sms;
  const int workers = std::max(1, h->grid_override > 0
                                      ? std::min(h->grid_override / P, std::max(max_workers, 1))
                                      : max_workers);
  p.n_workers = workers;
  const bool cl = P == 2;
  auto K = [&](void (*k1)(Params, Maps), void (*k2)(Params, Maps)) { return P == 2 ? k2 : k1; };
  if (h->mode == MOE_MODE_PERSISTENT) {
    h->last_grid = workers * P;
    p.ahead_depth = h->ahead_opt < 0 ? workers : h->ahead_opt;
    CK(launch_kernel(K(moe_persistent_kernel<1>, moe_persistent_kernel<2>), workers * P,
                     kThreads + 32, tl.smem, s, cl, false, p, m));
  } else if (h->mode == MOE_MODE_STATIC) {
    h->last_grid = workers * P;
    // cooperative, so that every CTA is resident for the grid barrier; where a
    // cooperative cluster launch is refused, a plain one (the grid is within
    // the resident-cluster count, and every barrier wait is bounded)
    auto kern = K(moe_static_kernel<1>, moe_static_kernel<2>);
    cudaError_t e = launch_kernel(kern, workers * P, kThreads, tl.smem, s, cl, true, p, m);
    if (e != cudaSuccess && cl) {
      cudaGetLastError();
      e = launch_kernel(kern, workers * P, kThreads, tl.smem, s, cl, false, p, m);
    }
    CK(e);
  } else {
    h->last_grid = 0;
    CK(launch_kernel(K(k_route<1>, k_route<2>), p.n_route_tasks * P, kThreads, tl.smem, s, cl,
                     false, p, m));
    CK(launch_kernel(k_plan, 1, kThreads, tl.smem, s, false, false, p, m));
    const int routed_max = p.max_groups - p.n_shared_groups;
    CK(launch_kernel(k_gather, routed_max * 8, kThreads, tl.smem, s, false, false, p, m));
    CK(launch_kernel(K(k_gateup<1>, k_gateup<2>), p.max_groups * p.n_ftiles * P, kThreads,
                     tl.smem, s, cl, false, p, m));
    CK(launch_kernel(K(k_down<1>, k_down<2>), p.max_groups * p.n_dtiles * p.ks * P, kThreads,
                     tl.smem, s, cl, false, p, m));
    CK(launch_kernel(k_combine, p.n_comb, kThreads, tl.smem, s, false, false, p, m));
  }
  h->view.ws = h->ws;
  h->view.o_idx = h->o_idx;
  h->view.o_wgt = h->o_wgt;
  h->view.o_counts = h->o_counts;
  h->view.o_offsets = h->o_offsets;
  h->view.o_perm = h->o_perm;
  h->view.o_pos = h->o_pos;
  h->view.o_sched = h->o_sched;
  h->last_valid = false;
  h->last_T = T;
  h->last_bn = tl.bn;
  h->last_ks = tl.ks;
  h->last_bands = p.n_bands;
  h->last_ybytes = p.y_f32 ? 4 * p.ks : 2;
  h->last_ct = p.ct;
  h->last_pair = p.pair;
  return MOE_OK;
}

}  // namespace

int moe_layer_forward(moe_layer_t* h, int T, const void* x, const void* router_w,
                      const void* w_gate, const void* w_up, const void* w_down, void* out,
                      void* stream) {
  return forward_impl(h, T, x, router_w, w_gate, w_up, w_down, out, nullptr, stream);
}

int moe_layer_forward_residual_norm(moe_layer_t* h, int T, const void* x, const void* router_w,
                                    const void* w_gate, const void* w_up, const void* w_down,
                                    const void* residual, const void* gamma, float eps,
                                    void* out, void* norm_out, void* stream) {
  if (!residual || !gamma || !norm_out) return fail(MOE_E_INVAL, "null residual/gamma/norm_out");
  if (!aligned16(residual) || !aligned16(gamma) || !aligned16(norm_out))
    return fail(MOE_E_INVAL, "residual, gamma and norm_out must be 16-byte aligned");
  if (!(eps >= 0.f) || eps > 1.f) return fail(MOE_E_INVAL, "eps must be in [0, 1]");
  const Fuse fz{residual, gamma, eps, norm_out};
  return forward_impl(h, T, x, router_w, w_gate, w_up, w_down, out, &fz, stream);
}

int moe_layer_calibrate(moe_layer_t* h, int T, const void* x, const void* router_w,
                        const void* w_gate, const void* w_up, const void* w_down, void* out,
                        int reps, float* best_us, void* stream) {
  if (!h) return fail(MOE_E_INVAL, "null handle");
  if (!h->ws) return fail(MOE_E_STATE, "moe_layer_reserve was not called");
  if (T < 1 || T > h->T_max) return fail(MOE_E_INVAL, "T out of range (1..T_max)");
  if (reps < 1 || reps > 100) return fail(MOE_E_INVAL, "reps must be 1..100");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  CK(cudaEventCreate(&e0));
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return fail(MOE_E_CUDA, "cudaEventCreate");
  }
  // mean time of `reps` forwards after one untimed one; +inf if a forward or
  // its device status fails (the candidate is then never chosen)
  auto time_it = [&](float* ms) -> int {
    *ms = INFINITY;
    int rc = moe_layer_forward(h, T, x, router_w, w_gate, w_up, w_down, out, stream);
    if (rc == MOE_OK) rc = moe_layer_status(h, stream);
    if (rc != MOE_OK) return rc == MOE_E_CUDA ? rc : MOE_OK;
    if (cudaEventRecord(e0, s) != cudaSuccess) return MOE_E_CUDA;
    for (int r = 0; r < reps && rc == MOE_OK; ++r)
      rc = moe_layer_forward(h, T, x, router_w, w_gate, w_up, w_down, out, stream);
    if (cudaEventRecord(e1, s) != cudaSuccess) return MOE_E_CUDA;
    const int st = moe_layer_status(h, stream);
    if (rc != MOE_OK || st != MOE_OK) return (rc == MOE_E_CUDA || st == MOE_E_CUDA) ? MOE_E_CUDA : MOE_OK;
    float el = 0.f;
    if (cudaEventElapsedTime(&el, e0, e1) != cudaSuccess) return MOE_E_CUDA;
    *ms = el / reps;
    return MOE_OK;
  };
  // coordinate descent from the current settings: tile tokens, then the down
  // K split, then one or two d bands
  const int bn_c[] = {0, 64, 128, 160, 256};
  const int ks_c[] = {0, 1, 2, 4};
  const int bd_c[] = {1, 0};
  float best = INFINITY;
  int rc = time_it(&best);
  for (int i = 0; rc == MOE_OK && i < 5; ++i) {
    const int keep = h->bn_opt;
    if (bn_c[i] == keep) continue;
    h->bn_opt = bn_c[i];
    float t;
    rc = time_it(&t);
    if (t < best) best = t;
    else h->bn_opt = keep;
  }
  for (int i = 0; rc == MOE_OK && i < 4; ++i) {
    const int keep = h->split_k;
    if (ks_c[i] == keep) continue;
    h->split_k = ks_c[i];
    float t;
    rc = time_it(&t);
    if (t < best) best = t;
    else h->split_k = keep;
  }
  for (int i = 0; rc == MOE_OK && i < 2; ++i) {
    const int keep = h->bands;
    if (bd_c[i] == keep) continue;
    h->bands = bd_c[i];
    float t;
    rc = time_it(&t);
    if (t < best) best = t;
    else h->bands = keep;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (rc != MOE_OK) return rc;
  if (!(best < INFINITY)) return fail(MOE_E_DEVICE, "no calibration candidate ran cleanly");
  if (best_us) *best_us = best * 1e3f;
  return MOE_OK;
}

int moe_layer_forward_host(moe_layer_t* h, int T, const void* x_host, const void* router_w,
                           const void* w_gate, const void* w_up, const void* w_down,
                           void* out_host, void* stream) {
  if (!h) return fail(MOE_E_INVAL, "null handle");
  if (!h->ws) return fail(MOE_E_STATE, "moe_layer_reserve was not called");
  if (T < 0 || T > h->T_max) return fail(MOE_E_INVAL, "T out of range (0..T_max)");
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host) return fail(MOE_E_INVAL, "null host pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)h->T_max * h->d * 2;
  if (!h->x_dev_stage) {
    if (cudaMalloc(&h->x_dev_stage, bytes) != cudaSuccess ||
        cudaMalloc(&h->out_dev_stage, bytes) != cudaSuccess) {
      cudaGetLastError();
      return fail(MOE_E_NOMEM, "staging allocation failed");
    }
  }
  const size_t n = (size_t)T * h->d * 2;
  CK(cudaMemcpyAsync(h->x_dev_stage, x_host, n, cudaMemcpyHostToDevice, s));
  int rc = moe_layer_forward(h, T, h->x_dev_stage, router_w, w_gate, w_up, w_down,
                             h->out_dev_stage, stream);
  if (rc) return rc;
  CK(cudaMemcpyAsync(out_host, h->out_dev_stage, n, cudaMemcpyDeviceToHost, s));
  return moe_layer_status(h, stream);
}

int moe_layer_get_routing(moe_layer_t* h, int32_t* idx, float* w, int32_t* counts,
                          int32_t* offsets, int32_t* perm, int32_t* pos, void* stream) {
  if (!h || !h->view.ws) return fail(MOE_E_STATE, "no forward has run on this handle");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // sizes of the last forward are not kept on the host; copy T_max-sized
  // regions would overrun small caller buffers, so the caller passes buffers
  // sized for the T of the last forward and we copy exactly that much.
  const int T = h->last_T;
  const size_t Tk = (size_t)T * h->k;
  const auto& v = h->view;
  char* ws = v.ws;
  if (idx) CK(cudaMemcpyAsync(idx, ws + v.o_idx, Tk * 4, cudaMemcpyDeviceToDevice, s));
  if (w) CK(cudaMemcpyAsync(w, ws + v.o_wgt, Tk * 4, cudaMemcpyDeviceToDevice, s));
  if (counts) CK(cudaMemcpyAsync(counts, ws + v.o_counts, h->E * 4, cudaMemcpyDeviceToDevice, s));
  if (offsets)
    CK(cudaMemcpyAsync(offsets, ws + v.o_offsets, (h->E + 1) * 4, cudaMemcpyDeviceToDevice, s));
  if (perm) CK(cudaMemcpyAsync(perm, ws + v.o_perm, Tk * 4, cudaMemcpyDeviceToDevice, s));
  if (pos) CK(cudaMemcpyAsync(pos, ws + v.o_pos, Tk * 4, cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

int moe_layer_status(moe_layer_t* h, void* stream) {
  if (!h) return fail(MOE_E_INVAL, "null handle");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  char* sched = h->view.ws ? h->view.ws + h->view.o_sched : nullptr;
  if (!sched) return MOE_OK;
  CK(cudaMemcpy(&h->last, sched, sizeof(Sched), cudaMemcpyDeviceToHost));
  h->last_valid = true;
  const int rc = set_error_from_sched(h->last);
  if (rc) {
    int zero = 0;
    CK(cudaMemcpy(sched, &zero, sizeof(int), cudaMemcpyHostToDevice));
  }
  return rc;
}

long long moe_layer_get_stat(moe_layer_t* h, int key) {
  if (!h) return -1;
  if (key == MOE_STAT_TILE_TOKENS) return h->last_T ? h->last_bn : -1;
  if (key == MOE_STAT_SPLIT_K) return h->last_T ? h->last_ks : -1;
  if (key == MOE_STAT_BANDS) return h->last_T ? h->last_bands : -1;
  if (key == MOE_STAT_Y_BYTES) return h->last_T ? h->last_ybytes : -1;
  if (key == MOE_STAT_COMBINE_TOKENS) return h->last_T ? h->last_ct : -1;
  if (key == MOE_STAT_PAIR) return h->last_T ? h->last_pair : -1;
  if (!h->last_valid) return -1;
  switch (key) {
    case MOE_STAT_MOVER_CTAS: return h->last.n_movers;
    case MOE_STAT_TASKS: return h->last.tasks_done;
    case MOE_STAT_GRID: return h->last_grid;
    case MOE_STAT_GEMM_TASKS: return h->last.stat_gemm;
    case MOE_STAT_MOVER_TASKS: return h->last.stat_mover;
    case MOE_STAT_STOLEN: return h->last.stat_stolen;
    case MOE_STAT_AHEAD: return h->last.stat_ahead;
    case MOE_STAT_TRACE_RECORDS: return h->last.trace_n;
    default: return -1;
  }
}

int moe_layer_get_trace(moe_layer_t* h, uint64_t* records, int cap, void* stream) {
  if (!h || !h->ws || cap < 0 || (cap > 0 && !records)) {
    g_err = "bad arguments";
    return -1;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    g_err = "cudaStreamSynchronize failed";
    return -1;
  }
  if (!h->trace) return 0;
  int n = 0;
  if (cudaMemcpy(&n, h->ws + h->o_sched + offsetof(Sched, trace_n), sizeof(int),
                 cudaMemcpyDeviceToHost) != cudaSuccess) {
    g_err = "cudaMemcpy failed";
    return -1;
  }
  n = std::min(std::min(n, h->trace_cap), cap);
  if (n > 0 && cudaMemcpy(records, h->trace, (size_t)n * 32, cudaMemcpyDeviceToHost) != cudaSuccess) {
    g_err = "cudaMemcpy failed";
    return -1;
  }
  return n;
}

/* See include/moe.h.  Runs the unchanged moe_layer_forward on a copy of the
 * handle whose workspace is the file-scope scratch array above, then points
 * the caller's handle at that copy's routing and scheduler state, so that
 * moe_layer_status and moe_layer_get_routing report this call. */
int moe_layer_forward_noalloc(moe_layer_t* h, int T, const void* x, const void* router_w,
                              const void* w_gate, const void* w_up, const void* w_down, void* out,
                              void* stream) {
  if (!h) return fail(MOE_E_INVAL, "null handle");
  if (T < 0) return fail(MOE_E_INVAL, "T must be >= 0");
  if (T == 0) return MOE_OK;
  if (T > kMaxE * kRouteTokens) return fail(MOE_E_INVAL, "T out of range (1..32768)");
  // Set-up per device, with that device current: the scratch array's device
  // address (the host-side symbol is only a stand-in), the device's SM count
  // and the kernels' shared-memory limit.  No allocation.  The address is
  // looked up again at every call (a lookup, no allocation); when it differs
  // from the cached one (the device was reset and the module reloaded) the
  // set-up is redone.
  struct DeviceSetup {
    bool done = false;
    void* scratch = nullptr;
    int num_sms = 0;
    int max_pairs = 0;
  };
  static DeviceSetup setups[64];
  static std::mutex setup_mutex;
  int dev = 0;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(MOE_E_INVAL, "device ordinal out of range");
  void* scratch_now = nullptr;
  {
    cudaError_t e = cudaGetSymbolAddress(&scratch_now, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
  }
  DeviceSetup su;
  {
    std::lock_guard<std::mutex> lock(setup_mutex);
    DeviceSetup& s = setups[dev];
    if (!s.done || s.scratch != scratch_now) {
      s.done = false;
      int cc_major = 0, cc_minor = 0;
      CK(cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, dev));
      CK(cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
      if (cc_major != 10 || cc_minor != 3)
        return fail(MOE_E_INVAL, "this library is built for sm_103a (GB300) only");
      if (!encode_fn()) return fail(MOE_E_CUDA, "cuTensorMapEncodeTiled is not available");
      CK(cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev));
      CK(set_kernel_smem(kSmemBudget));
      s.max_pairs = query_max_pairs(s.num_sms);
      s.scratch = scratch_now;
      s.done = true;
    }
    su = s;
  }
  // A workspace laid out for exactly T tokens inside the scratch array; when
  // the fp32 split-K partials do not fit, the down projection keeps Y in bf16
  // (so the tiling, and the last bits of out, may differ from
  // moe_layer_forward's for the same layer: both are within the oracle's
  // tolerance).
  moe_layer tmp = *h;
  tmp.device = dev;
  tmp.num_sms = su.num_sms;
  tmp.max_pairs = su.max_pairs;
  tmp.x_dev_stage = tmp.out_dev_stage = nullptr;
  tmp.trace = nullptr;  // the trace counters live in the caller's own workspace
  tmp.trace_cap = 0;
  Bounds b = make_bounds(&tmp, T);
  layout(&tmp, b);
  if (tmp.ws_bytes > kNoallocScratchBytes) {
    const long long rows = (long long)T * h->k + (long long)T * h->S;
    b.y_elems = (size_t)((rows * h->d + 1) / 2);
    layout(&tmp, b);
  }
  if (tmp.ws_bytes > kNoallocScratchBytes)
    return fail(MOE_E_INVAL, "layer too large for the " + std::to_string(kNoallocScratchBytes >> 20) +
                                 " MiB scratch of moe_layer_forward_noalloc (needs " +
                                 std::to_string(tmp.ws_bytes >> 20) + " MiB); use moe_layer_reserve");
  tmp.B = b;
  tmp.ws = static_cast<char*>(su.scratch);
  tmp.T_max = T;
  const int rc = moe_layer_forward(&tmp, T, x, router_w, w_gate, w_up, w_down, out, stream);
  if (rc == MOE_OK) {
    h->view = tmp.view;
    h->last_valid = false;
    h->last_T = tmp.last_T;
    h->last_grid = tmp.last_grid;
    h->last_bn = tmp.last_bn;
    h->last_ks = tmp.last_ks;
    h->last_bands = tmp.last_bands;
    h->last_ybytes = tmp.last_ybytes;
    h->last_ct = tmp.last_ct;
    h->last_pair = tmp.last_pair;
  }
  return rc;
}

void moe_layer_destroy(moe_layer_t* h) {
  if (!h) return;
  if (h->trace) cudaFree(h->trace);
  if (h->ws) cudaFree(h->ws);
  if (h->x_dev_stage) cudaFree(h->x_dev_stage);
  if (h->out_dev_stage) cudaFree(h->out_dev_stage);
  delete h;
}

}  // extern "C"
