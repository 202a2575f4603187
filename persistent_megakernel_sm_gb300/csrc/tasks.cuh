// Device-side tasks of the MoE-layer forward pass and the in-kernel scheduler.
//
// Every task is a __device__ function run by a whole CTA (256 threads).  The
// persistent megakernel (moe.cu) pulls task ids from two queues; the
// multi-kernel ablation launches the same functions one kernel per stage.
#pragma once

#include "layer.cuh"
#include "ptx.cuh"

namespace moe {

// Per-CTA control block, placed after the pipeline stages in shared memory.
struct Ctrl {
  uint64_t full_bar[8];
  uint64_t empty_bar[8];
  uint64_t acc_bar;
  unsigned long long deadline;
  uint32_t tmem_base;
  int task;
  int flag;
  int ival[8];
  int tok[kThreads];      // scratch: token ids / combine tiles per row
  int cnt[kMaxE];         // scratch: per-expert counts
  int aux[kMaxE];
  int aux2[kMaxE];
  float wsum[kThreads];
};

// Per-thread state that lives across tasks.
struct CtaState {
  uint32_t pipe_it;     // k blocks issued / consumed so far (producer & MMA thread)
  uint32_t gemm_count;  // GEMM tasks done (all threads)
  uint64_t deadline;    // globaltimer value after which waits give up
  int role_mover;       // 1 if this CTA prefers mover work (after the plan)
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

// Release this CTA's global writes (generic and, for TMA readers, async
// proxy) before a dependency counter is bumped.  Called by every thread.
__device__ __forceinline__ void release_writes() {
  fence_proxy_async_global();
  __threadfence();
  __syncthreads();
}

// Group descriptor: shared-expert groups [0, n_shared_groups) are known at
// launch and computed here (their tasks may run before the plan exists);
// routed groups are read from the plan's table.
__device__ __forceinline__ Group load_group(const Params& p, int g) {
  if (g < p.n_shared_groups) {
    const int t0 = g * p.bn_max;
    return Group{p.E, p.T * p.k + t0, min(p.bn_max, p.T - t0), t0};
  }
  Group G;
  G.e = __ldcg(&p.groups[g].e);
  G.row0 = __ldcg(&p.groups[g].row0);
  G.nrows = __ldcg(&p.groups[g].nrows);
  G.src_row0 = __ldcg(&p.groups[g].src_row0);
  return G;
}

__device__ __forceinline__ bool group_ok(const Params& p, const Group& G) {
  return G.nrows >= 1 && G.nrows <= p.bn_max && G.e >= 0 && G.e <= p.E && G.row0 >= 0 &&
         G.row0 + G.nrows <= p.rows_y;
}

// ------------------------------------------------------------------ queues
// Two ticket queues.  Slots [0, n_static) of a queue are implicit tasks known
// at launch (router tiles for the mover queue, shared-expert gate/up tiles
// for the GEMM queue).  Later slots are reserved by pushers with an atomic add
// on `tail` and filled with a release store; ring entries start at -1.

struct QueueRef {
  int* head;
  int* tail;
  int* ring;
  int n_static;
  int cap;
};

__device__ __forceinline__ QueueRef mover_queue(const Params& p) {
  return QueueRef{&p.sched->mover_head, &p.sched->mover_tail, p.ring_mover, p.n_route,
                  p.mover_cap};
}

__device__ __forceinline__ QueueRef gemm_queue(const Params& p) {
  return QueueRef{&p.sched->gemm_head, &p.sched->gemm_tail, p.ring_gemm, p.n_static_gemm,
                  p.gemm_cap};
}

// Push n consecutive tasks id0, id0 + step, ...  Called by all 32 lanes of one warp.
__device__ __forceinline__ void push_tasks_warp(const Params& p, const QueueRef& q, int id0,
                                                int step, int n) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  if (lane == 0) base = atomicAdd(q.tail, n);
  base = __shfl_sync(0xffffffffu, base, 0);
  if (base + n > q.cap) {
    if (lane == 0) set_status(p, MOE_E_DEVICE, 1);
    return;
  }
  for (int i = lane; i < n; i += 32) st_release(q.ring + base + i, id0 + i * step);
}

// Try to claim one task: >= 0 task id, -1 nothing claimable now, -2 this
// queue is finished.  Thread 0 only.
__device__ int try_claim(const Params& p, const QueueRef& q, int total_dyn, bool plan_done,
                         uint64_t deadline) {
  const int h = ld_relaxed(q.head);
  const int avail = q.n_static + ld_acquire(q.tail);
  if (h >= avail) {
    if (plan_done && h >= q.n_static + total_dyn) return -2;
    return -1;
  }
  if (atomicCAS(q.head, h, h + 1) != h) return -1;
  if (h < q.n_static) return -(1000 + h);  // implicit task, decoded by the caller
  int v;
  while ((v = ld_acquire(q.ring + (h - q.n_static))) < 0) {
    if (globaltimer() > deadline) {
      set_status(p, MOE_E_TIMEOUT, 2);
      return -3;
    }
    if (ld_relaxed(&p.sched->status) != 0) return -3;
  }
  return v;
}

// Decide this CTA's next task (thread 0).  Returns a task id or -1 to exit.
__device__ int claim_next(const Params& p, CtaState& st) {
  Sched* s = p.sched;
  uint32_t backoff = 32;
  while (true) {
    if (ld_relaxed(&s->status) != 0) return -1;
    const bool plan_done = ld_acquire(&s->plan_done) != 0;
    int mover_total = 0, gemm_total = 0;
    if (plan_done) {
      mover_total = ld_relaxed(&s->mover_total_dyn);
      gemm_total = ld_relaxed(&s->gemm_total_dyn);
      st.role_mover = (int)blockIdx.x < ld_relaxed(&s->n_movers);
    }
    // Before the plan every CTA prefers router tiles (they gate everything);
    // afterwards each CTA prefers its own role's queue and steals otherwise.
    const bool mover_first = !plan_done || st.role_mover;
    QueueRef qa = mover_first ? mover_queue(p) : gemm_queue(p);
    QueueRef qb = mover_first ? gemm_queue(p) : mover_queue(p);
    const int ta = mover_first ? mover_total : gemm_total;
    const int tb = mover_first ? gemm_total : mover_total;
    int finished = 0;
    for (int pass = 0; pass < 2; ++pass) {
      const QueueRef& q = pass == 0 ? qa : qb;
      int r = try_claim(p, q, pass == 0 ? ta : tb, plan_done, st.deadline);
      if (r == -3) return -1;
      if (r == -2) {
        ++finished;
        continue;
      }
      if (r == -1) continue;
      const bool is_mover_q = (q.ring == p.ring_mover);
      if (r <= -1000) {
        const int slot = -(r + 1000);
        r = is_mover_q ? task_id(kTaskRoute, slot) : task_id(kTaskGateUp, slot);
      }
      if (pass == 1 && plan_done) atomicAdd(&s->stat_stolen, 1);
      return r;
    }
    if (finished == 2) return -1;
    if (globaltimer() > st.deadline) {
      set_status(p, MOE_E_TIMEOUT, 3);
      return -1;
    }
    __nanosleep(backoff);
    if (backoff < 1024) backoff <<= 1;
  }
}

// ------------------------------------------------------------------ router
// Router tile: tokens [tau*rt, tau*rt + nt).  Logits on CUDA cores (fp32
// accumulate of bf16 products), softmax over all E, top-k by (p desc, e asc),
// renormalised weights, and the tile's per-expert counts and ranks.
__device__ void route_task(const Params& p, int tau, char* scratch, Ctrl* c) {
  const int t0 = tau * p.rt;
  const int nt = min(p.rt, p.T - t0);
  const int E = p.E, k = p.k;
  float* logit = reinterpret_cast<float*>(scratch);  // [rt][E]
  int* sidx = reinterpret_cast<int*>(logit + p.rt * E);  // [rt][k]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = p.d >> 3;

  for (int pr = warp; pr < nt * E; pr += kThreads / 32) {
    const int t = pr / E, e = pr - t * E;
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)(t0 + t) * p.d);
    const uint4* wrr = reinterpret_cast<const uint4*>(p.wr + (size_t)e * p.d);
    float acc = 0.f;
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) acc += dot8(__ldg(xr + v), __ldg(wrr + v));
    acc = warp_sum(acc);
    if (lane == 0) logit[t * E + e] = acc + (p.bias ? __ldg(p.bias + e) : 0.f);
  }
  __syncthreads();

  for (int t = warp; t < nt; t += kThreads / 32) {
    float v[kMaxE / 32];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? logit[t * E + e] : -INFINITY;
      mx = fmaxf(mx, v[i]);
    }
    mx = warp_max(mx);
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? __expf(v[i] - mx) : 0.f;
      z += v[i];
    }
    z = warp_sum(z);
    const float invz = 1.f / z;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) v[i] = (lane + 32 * i) < E ? v[i] * invz : -1.f;
    float kept = 0.f, my_p = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
      float bp = -2.f;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i)
        if (v[i] > bp) {
          bp = v[i];
          be = lane + 32 * i;
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float op = __shfl_xor_sync(0xffffffffu, bp, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (op > bp || (op == bp && oe < be)) {
          bp = op;
          be = oe;
        }
      }
      if ((be & 31) == lane) {
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i)
          if (i == (be >> 5)) v[i] = -2.f;
      }
      if (lane == j) {
        my_p = bp;
        my_e = be;
      }
      kept += bp;
    }
    if (lane < k) {
      const size_t o = (size_t)(t0 + t) * k + lane;
      p.idx[o] = my_e;
      p.wgt[o] = my_p / kept;
      sidx[t * k + lane] = my_e;
    }
  }
  for (int e = threadIdx.x; e < E; e += kThreads) c->cnt[e] = 0;
  __syncthreads();
  for (int ent = threadIdx.x; ent < nt * k; ent += kThreads) {
    const int t = ent / k;
    const int e = sidx[ent];
    int r = 0;
    for (int q = 0; q < t * k; ++q) r += (sidx[q] == e);
    p.rank[(size_t)t0 * k + ent] = r;
    atomicAdd(&c->cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) p.tile_cnt[(size_t)tau * E + e] = c->cnt[e];
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
  __syncthreads();
  if (lane == 31) c->ival[warp] = x;
  __syncthreads();
  int wbase = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int s = c->ival[w];
    if (w < warp) wbase += s;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return wbase + x - v;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Number of gather tasks of a group.
__device__ __forceinline__ int gather_chunks(int nrows) { return ceil_div(nrows, kGatherRows); }

// The plan: runs once, on the CTA that finished the last router tile (or as
// its own kernel in the ablation).  Counts and offsets per expert, the
// canonical permutation (experts ascending, tokens ascending), the GEMM row
// groups (experts in order of decreasing count, each split into balanced
// tiles of at most bn_max rows), the cost-model split of CTAs into movers and
// GEMM workers, and (persistent mode) the first pushes: every gather task.
__device__ void plan_task(const Params& p, Ctrl* c, bool push) {
  const int E = p.E, k = p.k, tid = threadIdx.x;
  int* cnt = c->cnt;     // counts per expert
  int* order = c->aux;   // experts by decreasing count
  int* offs = c->aux2;   // offsets per expert

  // per expert: exclusive prefix over router tiles, in place, and the count
  if (tid < E) {
    int run = 0;
    for (int tau = 0; tau < p.n_route; ++tau) {
      int* q = p.tile_cnt + (size_t)tau * E + tid;
      const int v = __ldcg(q);
      *q = run;
      run += v;
    }
    cnt[tid] = run;
    p.counts[tid] = run;
  }
  __syncthreads();
  int total = 0;
  const int off = block_exclusive_scan(tid < E ? cnt[tid] : 0, &total, c);
  if (tid < E) {
    p.offsets[tid] = off;
    offs[tid] = off;
  }
  if (tid == 0) p.offsets[E] = total;
  // experts ordered by (count desc, expert asc)
  if (tid < E) {
    const int me = cnt[tid];
    int r = 0;
    for (int e2 = 0; e2 < E; ++e2) {
      const int o = cnt[e2];
      r += (o > me) || (o == me && e2 < tid);
    }
    order[r] = tid;
  }
  __syncthreads();
  // groups: order slot r -> expert order[r]
  int e_r = tid < E ? order[tid] : 0;
  int n_r = tid < E ? cnt[e_r] : 0;
  int nmt = n_r > 0 ? ceil_div(n_r, p.bn_max) : 0;
  int n_routed = 0;
  const int gfirst = block_exclusive_scan(nmt, &n_routed, c);
  // gather-task prefix in group order
  int rows_per = nmt > 0 ? ((ceil_div(n_r, nmt) + 15) / 16) * 16 : 0;
  int my_chunks = 0;
  for (int m = 0; m < nmt; ++m) my_chunks += gather_chunks(min(rows_per, n_r - m * rows_per));
  int n_gather = 0;
  const int chunk_base = block_exclusive_scan(my_chunks, &n_gather, c);
  const int off_e = tid < E ? offs[e_r] : 0;
  if (p.n_shared_groups + n_routed > p.max_groups) {
    if (tid == 0) set_status(p, MOE_E_DEVICE, 4);
    return;
  }
  // routed groups follow the shared-expert groups (see load_group)
  {
    int cb = chunk_base;
    for (int m = 0; m < nmt; ++m) {
      const int g = p.n_shared_groups + gfirst + m;
      const int nrows = min(rows_per, n_r - m * rows_per);
      const int row0 = off_e + m * rows_per;
      p.groups[g] = Group{e_r, row0, nrows, row0};
      if (push) {
        const int nc = gather_chunks(nrows);
        for (int q = 0; q < nc; ++q) p.ring_mover[cb + q] = task_id(kTaskGather, g * 8 + q);
        cb += nc;
      }
    }
  }
  __syncthreads();
  // the canonical permutation
  for (int ent = tid; ent < p.T * k; ent += kThreads) {
    const int t = ent / k;
    const int e = __ldcg(p.idx + ent);
    const int tau = t / p.rt;
    const int row = offs[e] + __ldcg(p.tile_cnt + (size_t)tau * E + e) + __ldcg(p.rank + ent);
    p.perm[row] = t;
    p.pos[ent] = row;
  }
  // cost model (spatial split): CTA-seconds of mover work against GEMM work
  if (tid == 0) {
    const int n_groups = p.n_shared_groups + n_routed;
    const int n_down = p.n_dtiles * p.ks;
    Sched* s = p.sched;
    s->n_groups = n_groups;
    s->gemm_total_dyn = n_routed * p.n_ftiles + n_groups * n_down;
    s->mover_total_dyn = n_gather + p.n_comb;
    int movers;
    const int N = gridDim.x;
    if (p.mover_override > 0) {
      movers = min(p.mover_override, max(N - 1, 1));
    } else {
      const double ybytes = p.y_f32 ? 4.0 * p.ks : 2.0;
      const double Tk = (double)p.T * k;
      const double b_move = Tk * p.d * 2.0 * 2.0 +                      // gather: read + write
                            ((double)p.T * (k + p.S)) * p.d * ybytes +  // combine reads
                            (double)p.T * p.d * 2.0;                    // combine writes
      int touched = p.S;
      for (int e = 0; e < E; ++e) touched += cnt[e] > 0;
      const double flops = 6.0 * (Tk + (double)p.T * p.S) * p.d * p.f;
      const double wbytes = (double)touched * 3.0 * p.f * p.d * 2.0;
      const double a = b_move / p.beta_move;                              // CTA-seconds
      const double b = fmax(flops / p.phi_gemm, (double)N * wbytes / p.hbm_bw);
      movers = (int)lrint((double)N * a / (a + b));
      movers = max(1, min(movers, max(N - 1, 1)));
    }
    s->n_movers = movers;
  }
  if (push) {
    release_writes();
    if (tid == 0) {
      atomicAdd(&p.sched->mover_tail, n_gather);
      __threadfence();
      st_release(&p.sched->plan_done, 1);
    }
  } else {
    __syncthreads();
  }
}

// ------------------------------------------------------------------ gather (mover)
// Xp[row, :] = x[perm[row], :] for up to 32 rows of one group.
__device__ void gather_task(const Params& p, int g, int chunk, Ctrl* c) {
  const Group G = load_group(p, g);
  if (!group_ok(p, G) || chunk * kGatherRows >= G.nrows) {
    if (threadIdx.x == 0) set_status(p, MOE_E_DEVICE, 20);
    return;
  }
  const int r0 = G.row0 + chunk * kGatherRows;
  const int nr = min(kGatherRows, G.nrows - chunk * kGatherRows);
  if (threadIdx.x < nr) c->tok[threadIdx.x] = __ldcg(p.perm + r0 + threadIdx.x);
  __syncthreads();
  const int nvec = p.d >> 3;
  const int total = nr * nvec;
  const uint4* x = reinterpret_cast<const uint4*>(p.x);
  uint4* xp = reinterpret_cast<uint4*>(p.Xp);
  constexpr int U = 8;
  for (int base = threadIdx.x; base < total; base += kThreads * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kThreads;
      if (i < total) {
        const int r = i / nvec, q = i - r * nvec;
        v[u] = __ldg(x + (size_t)c->tok[r] * nvec + q);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kThreads;
      if (i < total) {
        const int r = i / nvec, q = i - r * nvec;
        xp[(size_t)(r0 + r) * nvec + q] = v[u];
      }
    }
  }
}

// ------------------------------------------------------------------ combine (mover)
// out[t, :] = bf16( sum_j w[t,j] * Y[pos[t,j], :] + Y[T k + t, :] (shared) ),
// fp32 sum in slot order, then the shared expert; K splits summed first.
__device__ void combine_task(const Params& p, int ctile, Ctrl* c) {
  const int t0 = ctile * p.ct;
  const int nt = min(p.ct, p.T - t0);
  const int k = p.k;
  for (int i = threadIdx.x; i < nt * k; i += kThreads) {
    c->tok[i] = __ldcg(p.pos + (size_t)t0 * k + i);
    c->wsum[i] = __ldcg(p.wgt + (size_t)t0 * k + i);
  }
  __syncthreads();
  const int nvec = p.d >> 3;
  const int total = nt * nvec;
  uint4* out = reinterpret_cast<uint4*>(p.out);
  const size_t part = (size_t)p.rows_y * p.d;  // elements per K split
  for (int i = threadIdx.x; i < total; i += kThreads) {
    const int t = i / nvec, q = i - t * nvec;
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    for (int j = 0; j <= k; ++j) {
      int row;
      float w;
      if (j < k) {
        row = c->tok[t * k + j];
        w = c->wsum[t * k + j];
      } else {
        if (!p.S) break;
        row = p.T * k + t0 + t;
        w = 1.f;
      }
      float y[8];
      if (p.y_f32) {
        const float* Y = reinterpret_cast<const float*>(p.Y);
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] = 0.f;
        for (int s = 0; s < p.ks; ++s) {
          const float4* src =
              reinterpret_cast<const float4*>(Y + s * part + (size_t)row * p.d + q * 8);
          const float4 a = __ldcg(src), b = __ldcg(src + 1);
          y[0] += a.x; y[1] += a.y; y[2] += a.z; y[3] += a.w;
          y[4] += b.x; y[5] += b.y; y[6] += b.z; y[7] += b.w;
        }
      } else {
        const uint4* Y = reinterpret_cast<const uint4*>(p.Y);
        bf16x8_to_f32(__ldcg(Y + (size_t)row * nvec + q), y);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = fmaf(w, y[u], acc[u]);
    }
    out[(size_t)(t0 + t) * nvec + q] = f32x8_to_bf16(acc);
  }
}

// ------------------------------------------------------------------ GEMM tile (tcgen05)
// Swap-AB tile: the weights are the M = 128 operand, the tokens the N operand,
// so a handful of tokens still fills the tensor core's M dimension.
//   gate/up (g, ft):  acc0 = Wg[e][ft*128 .. +128, :] * B^T,  acc1 = Wu[...] * B^T
//   down (g, dt, s):  acc0 = Wd[e][dt*256 .. +128, Ks] * H^T, acc1 = rows +128 .. +256
// B = the group's rows of Xp (or x for the shared expert) / of H, K-major.
// Pipeline: warp 0 lane 0 issues TMA loads into a ring of `stages` stages,
// warp 1 lane 0 issues tcgen05.mma into two TMEM accumulators, all 8 warps
// run the epilogue from TMEM.

struct GemmJob {
  const CUtensorMap* a0;
  const CUtensorMap* a1;
  const CUtensorMap* b;
  int a_row0, a1_row0;  // weight rows of the two accumulators
  int b_row0;           // first B row
  int nrows;            // tokens (columns of the accumulators)
  int kb0, nkb;         // first k block and number of k blocks
};

// Returns false on a timeout (status already set).
__device__ bool gemm_mainloop(const Params& p, const GemmJob& job, char* smem, Ctrl* c,
                              CtaState& st) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nbox = ceil_div(job.nrows, kBBoxRows);
  const uint32_t n_mma = (uint32_t)(((job.nrows + 15) / 16) * 16);
  bool ok = true;
  if (warp == 0 && lane == 0) {
    fence_proxy_async_global();
    fence_proxy_async_shared();
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    const uint32_t bytes = 2u * kABoxBytes + (uint32_t)nbox * kBBoxBytes;
    uint32_t it = st.pipe_it;
    for (int kb = 0; kb < job.nkb; ++kb, ++it) {
      const uint32_t s = it % p.stages, ph = (it / p.stages) & 1u;
      if (!mbar_wait(&c->empty_bar[s], ph ^ 1u, st.deadline)) {
        set_status(p, MOE_E_TIMEOUT, 10);
        ok = false;
        break;
      }
      char* stage = smem + (size_t)s * p.stage_bytes;
      mbar_arrive_expect_tx(&c->full_bar[s], bytes);
      const int kc = (job.kb0 + kb) * kBK;
      tma_load_2d(stage, job.a0, &c->full_bar[s], kc, job.a_row0, pol_w);
      tma_load_2d(stage + kABoxBytes, job.a1, &c->full_bar[s], kc, job.a1_row0, pol_w);
      for (int bx = 0; bx < nbox; ++bx)
        tma_load_2d(stage + 2 * kABoxBytes + bx * kBBoxBytes, job.b, &c->full_bar[s], kc,
                    job.b_row0 + bx * kBBoxRows, pol_a);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16(kBM, n_mma);
    const uint32_t t0 = c->tmem_base, t1 = c->tmem_base + kAcc1Col;
    uint32_t it = st.pipe_it;
    for (int kb = 0; kb < job.nkb; ++kb, ++it) {
      const uint32_t s = it % p.stages, ph = (it / p.stages) & 1u;
      if (!mbar_wait(&c->full_bar[s], ph, st.deadline)) {
        set_status(p, MOE_E_TIMEOUT, 11);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t base = smem_u32(smem + (size_t)s * p.stage_bytes);
      const uint64_t da0 = sw128_desc(base), da1 = sw128_desc(base + kABoxBytes);
      const uint64_t db = sw128_desc(base + 2 * kABoxBytes);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
        // advancing 16 bf16 (32 B) inside the 128-B swizzle row: +2 in the
        // 16-byte-granular start-address field
        mma_bf16(t0, da0 + 2 * kk, db + 2 * kk, idesc, acc);
        mma_bf16(t1, da1 + 2 * kk, db + 2 * kk, idesc, acc);
      }
      mma_commit(&c->empty_bar[s]);
    }
    mma_commit(&c->acc_bar);
  }
  st.pipe_it += job.nkb;
  // everyone waits for the accumulators
  __syncwarp();
  const int ok_all = __syncthreads_and(ok ? 1 : 0);
  if (!ok_all) return false;
  const bool done = mbar_wait(&c->acc_bar, st.gemm_count & 1u, st.deadline);
  if (!done) set_status(p, MOE_E_TIMEOUT, 12);
  if (!__syncthreads_and(done ? 1 : 0)) return false;
  tc_fence_after();
  return true;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + __expf(-z)); }

__device__ void gateup_task(const Params& p, const Maps& maps, int g, int ft, char* smem,
                            Ctrl* c, CtaState& st) {
  const Group G = load_group(p, g);
  if (!group_ok(p, G) || ft < 0 || ft >= p.n_ftiles) {
    if (threadIdx.x == 0) set_status(p, MOE_E_DEVICE, 21);
    return;
  }
  GemmJob job;
  job.a0 = &maps.wg;
  job.a1 = &maps.wu;
  job.b = G.e < p.E ? &maps.xp : &maps.x;
  job.a_row0 = G.e * p.f + ft * kBM;
  job.a1_row0 = job.a_row0;
  job.b_row0 = G.src_row0;
  job.nrows = G.nrows;
  job.kb0 = 0;
  job.nkb = p.d / kBK;
  const bool ok = gemm_mainloop(p, job, smem, c, st);
  if (ok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, half = warp >> 2;
    const int m = q * 32 + lane;  // f row inside the tile
    const uint32_t lane_addr = c->tmem_base + ((uint32_t)(q * 32) << 16);
    __nv_bfloat16* hcol = p.H + (size_t)G.row0 * p.f + ft * kBM + m;
    for (int ch = half; ch * 16 < G.nrows; ch += 2) {
      float gv[16], uv[16];
      tmem_ld2x16(lane_addr + ch * 16, lane_addr + kAcc1Col + ch * 16, gv, uv);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int n = ch * 16 + i;
        if (n < G.nrows) hcol[(size_t)n * p.f] = __float2bfloat16_rn(silu_f(gv[i]) * uv[i]);
      }
    }
  }
  tc_fence_before();
  st.gemm_count++;
}

__device__ void down_task(const Params& p, const Maps& maps, int g, int dt, int ksplit,
                          char* smem, Ctrl* c, CtaState& st) {
  const Group G = load_group(p, g);
  if (!group_ok(p, G) || dt < 0 || dt >= p.n_dtiles || ksplit < 0 || ksplit >= p.ks) {
    if (threadIdx.x == 0) set_status(p, MOE_E_DEVICE, 22);
    return;
  }
  GemmJob job;
  job.a0 = &maps.wd;
  job.a1 = &maps.wd;
  job.b = &maps.h;
  job.a_row0 = G.e * p.d + dt * 2 * kBM;
  job.a1_row0 = job.a_row0 + kBM;
  job.b_row0 = G.row0;
  job.nrows = G.nrows;
  job.kb0 = ksplit * p.kb_down;
  job.nkb = p.kb_down;
  const bool ok = gemm_mainloop(p, job, smem, c, st);
  if (ok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, half = warp >> 2;
    const int m = q * 32 + lane;
    const int col0 = dt * 2 * kBM + m, col1 = col0 + kBM;
    const uint32_t lane_addr = c->tmem_base + ((uint32_t)(q * 32) << 16);
    const bool has1 = col1 < p.d;
    for (int ch = half; ch * 16 < G.nrows; ch += 2) {
      float a[16], b[16];
      tmem_ld2x16(lane_addr + ch * 16, lane_addr + kAcc1Col + ch * 16, a, b);
      if (p.y_f32) {
        float* Y = reinterpret_cast<float*>(p.Y) + (size_t)ksplit * p.rows_y * p.d;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = ch * 16 + i;
          if (n < G.nrows) {
            float* yr = Y + (size_t)(G.row0 + n) * p.d;
            yr[col0] = a[i];
            if (has1) yr[col1] = b[i];
          }
        }
      } else {
        __nv_bfloat16* Y = reinterpret_cast<__nv_bfloat16*>(p.Y);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = ch * 16 + i;
          if (n < G.nrows) {
            __nv_bfloat16* yr = Y + (size_t)(G.row0 + n) * p.d;
            yr[col0] = __float2bfloat16_rn(a[i]);
            if (has1) yr[col1] = __float2bfloat16_rn(b[i]);
          }
        }
      }
    }
  }
  tc_fence_before();
  st.gemm_count++;
}

// ------------------------------------------------------------------ notifications
// (persistent mode) Called by all threads after a task; bumps the dependency
// counters the task feeds and pushes the tasks that became ready.

__device__ __forceinline__ bool drop_for_fault(const Params& p) {
  if (p.fault_drop < 0) return false;
  return atomicAdd(&p.sched->fault_seen, 1) == p.fault_drop;
}

__device__ void notify_gather_done(const Params& p, int g) {
  release_writes();
  if (threadIdx.x < 32) {
    int ready = 0;
    if (threadIdx.x == 0) {
      const Group G = load_group(p, g);
      const int old = atom_add_acq_rel(p.gather_done + g, 1);
      ready = (old + 1 == gather_chunks(G.nrows));
    }
    ready = __shfl_sync(0xffffffffu, ready, 0);
    if (ready) push_tasks_warp(p, gemm_queue(p), task_id(kTaskGateUp, g * p.n_ftiles), 1, p.n_ftiles);
  }
}

__device__ void notify_gateup_done(const Params& p, int g) {
  release_writes();
  if (threadIdx.x < 32) {
    int ready = 0;
    if (threadIdx.x == 0 && !drop_for_fault(p)) {
      const int old = atom_add_acq_rel(p.gu_done + g, 1);
      ready = (old + 1 == p.n_ftiles);
    }
    ready = __shfl_sync(0xffffffffu, ready, 0);
    const int n_down = p.n_dtiles * p.ks;
    if (ready) push_tasks_warp(p, gemm_queue(p), task_id(kTaskDown, g * n_down), 1, n_down);
  }
}

// Target of a combine tile's counter: every (token, slot) and shared row of
// the tile, once per down task covering it.
__device__ __forceinline__ int comb_target(const Params& p, int ctile) {
  const int nt = min(p.ct, p.T - ctile * p.ct);
  return nt * (p.k + p.S) * p.n_dtiles * p.ks;
}

__device__ void notify_down_done(const Params& p, int g, Ctrl* c) {
  release_writes();
  if (threadIdx.x == 0) c->flag = drop_for_fault(p) ? 1 : 0;
  const Group G = load_group(p, g);
  // combine tile of every row of the group (tokens ascending inside a group)
  const int tid = threadIdx.x;
  if (tid < G.nrows) {
    const int t = G.e < p.E ? __ldcg(p.perm + G.row0 + tid) : G.src_row0 + tid;
    c->tok[tid] = t / p.ct;
  }
  __syncthreads();
  if (c->flag) return;
  if (tid < G.nrows && (tid == 0 || c->tok[tid] != c->tok[tid - 1])) {
    const int ct = c->tok[tid];
    int len = 1;
    while (tid + len < G.nrows && c->tok[tid + len] == ct) ++len;
    const int old = atom_add_acq_rel(p.comb_done + ct, len);
    if (old + len == comb_target(p, ct)) {
      const QueueRef q = mover_queue(p);
      const int slot = atomicAdd(q.tail, 1);
      if (slot < q.cap) st_release(q.ring + slot, task_id(kTaskCombine, ct));
      else set_status(p, MOE_E_DEVICE, 5);
    }
  }
}

}  // namespace moe
