// backward.cu -- K-B: backward of the fused forward plus one sparse Adagrad
// step (RecIS §3.2 Algorithm 1, backward semantics: each valid contribution
// r carries w_r * G[s(r), :]; Figure 3: local reduce-ID of the touched rows).
//
// Instead of the pages' wave-level merge with global atomics, the
// contributions the forward recorded as (global row, gradient source) pairs
// are radix-sorted by row, so every unique row becomes one contiguous run
// with exactly one writer:
//   1-2. radix_sort_pairs (radix.cuh) -- one read of the keys for the digit
//                       histograms, then one stable chained-scan scatter per
//                       8-bit digit with bounded decoupled look-back;
//   3. k_segreduce   -- lane groups of dim/4 lanes each walk an equal
//                       contiguous range of sorted contributions in order,
//                       gathering scale * G rows with 16-byte loads (several
//                       in flight) and summing each run; a run that begins
//                       and ends in one range is finished at once (fp32
//                       Adagrad on its row); runs cut by range boundaries are
//                       combined in shared memory in range order, runs cut by
//                       CTA boundaries leave partials;
//   4. k_seg_fixup   -- sums the CTA partials of each cut run in CTA order and
//                       finishes it.
// The sum order is fixed by the sort (stable) and the range layout, so a run
// of the same inputs gives bit-identical results.
#include <algorithm>

#include "plan.cuh"
#include "radix.cuh"
#include "update.cuh"

namespace emb {

constexpr int kSegThreads = 128;
constexpr int kSegWarps = kSegThreads / 32;

// ---------------------------------------------------------------------------
// run ranks (debug outputs only): rank[i] = number of run heads before i
// ---------------------------------------------------------------------------
constexpr int kScanBlock = 1024;

__device__ __forceinline__ bool is_head(const uint32_t* keys, int64_t i, uint32_t sentinel) {
  const uint32_t k = keys[i];
  return k != sentinel && (i == 0 || keys[i - 1] != k);
}

__global__ void __launch_bounds__(kScanBlock) k_rank_reduce(const uint32_t* keys, int64_t n, uint32_t sentinel,
                                                            uint32_t* part) {
  const int64_t i = blockIdx.x * (int64_t)kScanBlock + threadIdx.x;
  const int c = __syncthreads_count(i < n && is_head(keys, i, sentinel));
  if (threadIdx.x == 0) part[blockIdx.x] = (uint32_t)c;
}

__global__ void __launch_bounds__(kScanBlock) k_rank_top(uint32_t* part, int nb, int64_t* n_unique) {
  __shared__ uint32_t wsum[32];
  __shared__ uint32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int b0 = 0; b0 < nb; b0 += kScanBlock) {
    const int i = b0 + threadIdx.x;
    const uint32_t v = i < nb ? part[i] : 0u;
    uint32_t x = v;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    uint32_t base = carry;
    for (int w = 0; w < warp; ++w) base += wsum[w];
    uint32_t tot = 0;
    for (int w = 0; w < 32; ++w) tot += wsum[w];
    if (i < nb) part[i] = base + x - v;
    __syncthreads();
    if (threadIdx.x == 0) carry += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0 && n_unique) *n_unique = carry;
}

__global__ void __launch_bounds__(kScanBlock) k_rank_down(const uint32_t* keys, int64_t n, uint32_t sentinel,
                                                          const uint32_t* part, uint32_t* rank_incl,
                                                          uint32_t* head_pos) {
  __shared__ uint32_t wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i = blockIdx.x * (int64_t)kScanBlock + threadIdx.x;
  const uint32_t v = (i < n && is_head(keys, i, sentinel)) ? 1u : 0u;
  uint32_t x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  uint32_t base = part[blockIdx.x];
  for (int w = 0; w < warp; ++w) base += wsum[w];
  if (i < n) {
    rank_incl[i] = base + x;               // heads at or before i
    if (v) head_pos[base + x - 1] = (uint32_t)i;
  }
}

// Debug outputs of each unique row: table, row and number of contributions.
__global__ void k_dbg_runs(const uint32_t* keys, int64_t n, uint32_t sentinel, const uint32_t* head_pos,
                           const int64_t* n_unique, const uint32_t* table_base, int n_tables, int32_t* dbg_table,
                           int64_t* dbg_row, int32_t* dbg_count) {
  const int64_t nu = *n_unique;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < nu; u += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t p = head_pos[u];
    int64_t pn;
    if (u + 1 < nu) {
      pn = head_pos[u + 1];
    } else {  // first sentinel key: lower bound of the sentinel in the sorted keys
      int64_t lo = p, hi = n;
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (keys[mid] < sentinel) lo = mid + 1; else hi = mid;
      }
      pn = lo;
    }
    const uint32_t key = keys[p];
    const int t = table_of_key(table_base, n_tables, key);
    if (dbg_table) dbg_table[u] = t;
    if (dbg_row) dbg_row[u] = (int64_t)(key - table_base[t]);
    if (dbg_count) dbg_count[u] = (int32_t)(pn - p);
  }
}

// ---------------------------------------------------------------------------
// segmented reduce + Adagrad
// ---------------------------------------------------------------------------
struct SegArgs {
  const uint32_t* keys;
  const uint32_t* vals;
  int64_t n;
  uint32_t sentinel;
  const int4* colg;       // per column: out_col, 1 if MEAN, dim/4
  const float* inv_n;
  const uint2* rec_src;   // weighted forwards: (gradient source, weight bits) per record; vals hold records
  const float* grad_out;
  int64_t ldg;
  const float* grad_seq;
  DivMagic32 bdiv;
  int32_t batch;
  const TableMeta* tables;
  const uint32_t* table_base;
  int32_t n_tables;
  float lr, eps;
  float4* partial;      // [n_blocks][2][maxdim4]: head / tail partial of each CTA
  int32_t* part_pos;    // [n_blocks][2]: end of the head run / start of the tail run
  uint8_t* part_thru;   // [n_blocks]: the CTA lies inside one run that continues past it
  int32_t maxdim4;
  int32_t glog;
  int32_t span;           // sorted entries per CTA (a multiple of the lane groups per CTA)
  // debug outputs
  const uint32_t* rank;
  int32_t* dbg_table;
  int64_t* dbg_row;
  int32_t* dbg_count;
  float* dbg_grad;
  int32_t dbg_ld;
};


__device__ __forceinline__ float4 seg_f4zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }

__device__ __forceinline__ void seg_f4add(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}


// The unique writer of a row: Adagrad step with the summed gradient g.  `end`
// is one past the run's last sorted position (debug: its rank).
template <int V>
__device__ void finish_row(const SegArgs& a, uint32_t key, int64_t end, const float4 (&g)[V], int sub) {
  const int t = table_of_key(a.table_base, a.n_tables, key);
  const int64_t row = key - __ldg(a.table_base + t);
  const TableMeta tm = a.tables[t];
  float* W = tm.weight + row * tm.dim;
  float* A = tm.acc + row * tm.dim;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int f4 = sub + v * 32;
    if (f4 < tm.dim4) {
      float4 w = *reinterpret_cast<float4*>(W + f4 * 4);
      float4 ac = *reinterpret_cast<float4*>(A + f4 * 4);
      adagrad1_fast(w.x, ac.x, g[v].x, a.lr, a.eps);
      adagrad1_fast(w.y, ac.y, g[v].y, a.lr, a.eps);
      adagrad1_fast(w.z, ac.z, g[v].z, a.lr, a.eps);
      adagrad1_fast(w.w, ac.w, g[v].w, a.lr, a.eps);
      *reinterpret_cast<float4*>(W + f4 * 4) = w;
      *reinterpret_cast<float4*>(A + f4 * 4) = ac;
    }
  }
  if (a.rank && a.dbg_grad) {
    const uint32_t u = a.rank[end - 1] - 1;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      if (f4 < tm.dim4) *reinterpret_cast<float4*>(a.dbg_grad + (int64_t)u * a.dbg_ld + f4 * 4) = g[v];
    }
  }
}

// The table a key belongs to and its metadata, tracked while keys ascend
// (reloaded only when the key leaves the current table's range).
struct TableCursor {
  int t = -1;
  uint32_t base = 0, next = 0;
  float* weight = nullptr;
  float* acc = nullptr;
  int dim = 0, dim4 = 0;
  __device__ __forceinline__ void seek(const SegArgs& a, uint32_t key) {
    if (t < 0 || key < base || key >= next) {
      t = table_of_key(a.table_base, a.n_tables, key);
      base = __ldg(a.table_base + t);
      next = __ldg(a.table_base + t + 1);
      const TableMeta& tm = a.tables[t];
      weight = tm.weight;
      acc = tm.acc;
      dim = tm.dim;
      dim4 = tm.dim4;
    }
  }
};

// Ask the memory system to stage `bytes` (a multiple of 16, 16-byte aligned)
// starting at p into L2, without waiting and without using registers.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// A finished run whose weight and accumulator loads are in flight; its
// Adagrad step is applied when the lane group finishes its next run (or at
// the end), so the loads overlap the gathers in between.
template <int V>
struct PendingRow {
  bool on = false;
  int64_t end = 0;
  int dim4 = 0;
  float* W = nullptr;
  float* A = nullptr;
  float4 g[V], w[V], acc[V];

  __device__ __forceinline__ void issue(const SegArgs& a, const TableCursor& tc, uint32_t k, int64_t e,
                                        const float4 (&grad)[V], int sub) {
    on = true;
    end = e;
    const int64_t row = k - tc.base;
    dim4 = tc.dim4;
    W = tc.weight + row * tc.dim;
    A = tc.acc + row * tc.dim;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      g[v] = grad[v];
      const int f4 = sub + v * 32;
      if (f4 < dim4) {
        w[v] = *reinterpret_cast<const float4*>(W + f4 * 4);
        acc[v] = *reinterpret_cast<const float4*>(A + f4 * 4);
      }
    }
  }

  __device__ __forceinline__ void retire(const SegArgs& a, int sub) {
    if (!on) return;
    on = false;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      if (f4 < dim4) {
        adagrad1_fast(w[v].x, acc[v].x, g[v].x, a.lr, a.eps);
        adagrad1_fast(w[v].y, acc[v].y, g[v].y, a.lr, a.eps);
        adagrad1_fast(w[v].z, acc[v].z, g[v].z, a.lr, a.eps);
        adagrad1_fast(w[v].w, acc[v].w, g[v].w, a.lr, a.eps);
        *reinterpret_cast<float4*>(W + f4 * 4) = w[v];
        *reinterpret_cast<float4*>(A + f4 * 4) = acc[v];
      }
    }
    if (a.rank && a.dbg_grad) {
      const uint32_t u = a.rank[end - 1] - 1;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < dim4) *reinterpret_cast<float4*>(a.dbg_grad + (int64_t)u * a.dbg_ld + f4 * 4) = g[v];
      }
    }
  }
};

// Sorted entries per CTA: about 64 per lane group (measured best on the
// training and sequence workloads), between 256 and kSegSpanMax.
constexpr int kSegSpanMax = 1024;
constexpr int kSegPerThread = kSegSpanMax / kSegThreads;
constexpr int kSegPerGroup = 64;

inline int seg_span(int glog) {
  const int ng = kSegThreads / 32 * (32 >> glog);
  const int s = kSegPerGroup * ng;
  return s < 256 ? 256 : (s > kSegSpanMax ? kSegSpanMax : s);
}
// Gradient rows in flight per lane group (4 rows of V float4 per lane) and
// resident CTAs per SM.  Measured on the training and sequence workloads:
// 4-deep groups in more warps beat 6- or 8-deep groups in fewer (more warps
// hide the gather latency better), and six 4-warp CTAs over 1024
// contributions beat three 8-warp CTAs over 2048 (a CTA's warps wait at its
// barrier for its slowest lane group; smaller CTAs wait less).  Rows wider
// than 128 floats take fewer CTAs to stay within the registers.
template <int V>
struct SegDepth {
  static constexpr int value = 4;
  static constexpr int ctas = V == 1 ? 6 : 4;
};
constexpr int kSegMaxGroups = kSegWarps * 32;     // dim 4: 32 one-lane groups per warp
constexpr uint32_t kOffPad = 0x80000000u;         // offset refers to grad_seq
constexpr uint32_t kNoKey = 0xFFFFFFFFu;          // above every key and the sentinel

// One decoded contribution: its row key, the float4 offset of its gradient
// row (kOffPad: in grad_seq), the scale (1/n of a mean bag, else 1) and the
// float4 count of the row.
struct __align__(16) SegRec {
  uint32_t key;
  uint32_t off;
  float scale;
  uint32_t d4;
};

struct SegSmem {
  SegRec rec[kSegSpanMax];
  float4 part[2][kSegWarps * 64];       // head / tail partial of each lane group
  int32_t head_end[kSegMaxGroups];      // end of the run cut at the group's start, -1 if none
  uint32_t tail_key[kSegMaxGroups];     // key of the run left open at the group's end
  uint8_t head_thru[kSegMaxGroups];     // that head run covers the whole range and goes on
  uint8_t tail_valid[kSegMaxGroups];
};

// Runs of sorted contributions are reduced by LANE GROUPS of dim/4 lanes
// (one float4 column slice per lane): the CTA's span is cut into equal
// contiguous ranges, one per group, and a group walks its range in order,
// SegDepth<V> gradient rows in flight, adding each row into the open run's sum and
// closing the run where the key changes.  A run closed inside the range that
// also began there is finished at once (Adagrad on its row, deferred by one
// run so the weight/accumulator loads overlap the next gathers); a run cut at
// the range start leaves a head partial and one open at the range end a tail
// partial, combined in group order after a barrier (and across CTAs by
// k_seg_fixup).
template <int V>
__global__ void __launch_bounds__(kSegThreads, SegDepth<V>::ctas) k_segreduce(const SegArgs a) {
  __shared__ SegSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int glog = a.glog;
  const int G = 32 >> glog;
  const int q = lane >> glog, sub = lane & ((1 << glog) - 1);
  const int NG = kSegWarps * G;
  const int grp = warp * G + q;
  const int64_t B0 = (int64_t)blockIdx.x * a.span;
  const int64_t B1 = min(B0 + (int64_t)a.span, a.n);
  const int span = (int)(B1 - B0);
  const int D4 = a.maxdim4;

  // ---- decode the CTA's entries, coalesced, into shared memory; the
  //      weight and accumulator rows of every run that starts here are
  //      prefetched into L2 so that the updates below find them there ----
  uint32_t lkey = a.sentinel;
  int ld4 = 0;
  TableCursor ptc;
#pragma unroll
  for (int k = 0; k < kSegPerThread; ++k) {
    if (k * kSegThreads >= span) break;
    const int e = k * kSegThreads + tid;
    SegRec r;
    r.key = a.sentinel;
    r.off = 0u;
    r.scale = 0.0f;
    r.d4 = 0u;
    if (e < span) {
      const uint32_t key = __ldg(a.keys + B0 + e);
      r.key = key;
      if (key != a.sentinel && (B0 + e == 0 || __ldg(a.keys + B0 + e - 1) != key)) {
        ptc.seek(a, key);
        const int64_t row = key - ptc.base;
        prefetch_l2(ptc.weight + row * ptc.dim, (uint32_t)ptc.dim * 4u);
        prefetch_l2(ptc.acc + row * ptc.dim, (uint32_t)ptc.dim * 4u);
      }
      if (key != a.sentinel) {
        uint32_t val = __ldg(a.vals + B0 + e);
        float wr = 1.0f;   // value weight of a SUM contribution
        if (a.rec_src) {
          const uint2 rs = __ldg(a.rec_src + val);
          val = rs.x;
          wr = __uint_as_float(rs.y);
        }
        if (val & kPadBit) {
          if (key != lkey) {
            lkey = key;
            ld4 = a.tables[table_of_key(a.table_base, a.n_tables, key)].dim4;
          }
          r.d4 = (uint32_t)ld4;
          r.scale = 1.0f;
          r.off = kOffPad | (val & ~kPadBit);
        } else {
          const uint32_t c = div_magic32(val, a.bdiv);
          const uint32_t b = val - c * (uint32_t)a.batch;
          const int4 cg = __ldg(a.colg + c);
          r.scale = cg.y ? __ldg(a.inv_n + val) : wr;
          r.d4 = (uint32_t)cg.z;
          r.off = (uint32_t)(((int64_t)b * a.ldg + cg.x) >> 2);
        }
      }
    }
    sm.rec[e] = r;
  }
  for (int g = tid; g < NG; g += kSegThreads) {
    sm.head_end[g] = -1;
    sm.head_thru[g] = 0;
    sm.tail_valid[g] = 0;
  }
  __syncthreads();

  // ---- per lane group: its contiguous range, in order ----
  const int R = a.span / NG;
  const int r0 = min(grp * R, span), r1 = min(r0 + R, span);
  uint32_t ckey = kNoKey;   // key of the open run
  bool chead = false;       // the open run began before this range
  if (r0 < r1) {
    ckey = sm.rec[r0].key;
    const uint32_t prev = r0 > 0 ? sm.rec[r0 - 1].key : (B0 > 0 ? __ldg(a.keys + B0 - 1) : kNoKey);
    chead = prev == ckey && ckey != a.sentinel;
  }
  float4 acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = seg_f4zero();
  TableCursor tc;
  PendingRow<V> pend;
  constexpr int kSegU = SegDepth<V>::value;
  for (int i0 = r0; i0 < r1; i0 += kSegU) {
    uint32_t key[kSegU];
    float sc[kSegU];
    float4 x[kSegU][V];
#pragma unroll
    for (int u = 0; u < kSegU; ++u) {
      const int e = i0 + u;
      const SegRec r = e < r1 ? sm.rec[e] : SegRec{kNoKey, 0u, 0.0f, 0u};
      key[u] = r.key;
      sc[u] = r.scale;
      const float* src = (r.off & kOffPad) ? a.grad_seq + (int64_t)(r.off & ~kOffPad) * 4
                                           : a.grad_out + (int64_t)r.off * 4;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        x[u][v] = f4 < (int)r.d4 ? __ldg(reinterpret_cast<const float4*>(src + f4 * 4)) : seg_f4zero();
      }
    }
#pragma unroll
    for (int u = 0; u < kSegU; ++u) {
      if (i0 + u < r1 && key[u] != ckey) {   // the open run ends before this entry
        if (ckey != a.sentinel) {
          if (chead) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
              const int f4 = sub + v * 32;
              if (f4 < D4) sm.part[0][grp * D4 + f4] = acc[v];
            }
            if (sub == 0) sm.head_end[grp] = i0 + u;
          } else {
            pend.retire(a, sub);
            tc.seek(a, ckey);
            pend.issue(a, tc, ckey, B0 + i0 + u, acc, sub);
          }
        }
        ckey = key[u];
        chead = false;
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = seg_f4zero();
      }
#pragma unroll
      for (int v = 0; v < V; ++v) {
        acc[v].x = fmaf(x[u][v].x, sc[u], acc[v].x);
        acc[v].y = fmaf(x[u][v].y, sc[u], acc[v].y);
        acc[v].z = fmaf(x[u][v].z, sc[u], acc[v].z);
        acc[v].w = fmaf(x[u][v].w, sc[u], acc[v].w);
      }
    }
  }
  // the run open at the range end: finished here, or left as a partial
  if (r0 < r1 && ckey != a.sentinel) {
    const uint32_t key_after = r1 < span ? sm.rec[r1].key : (B1 < a.n ? __ldg(a.keys + B1) : kNoKey);
    if (key_after != ckey) {
      if (chead) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const int f4 = sub + v * 32;
          if (f4 < D4) sm.part[0][grp * D4 + f4] = acc[v];
        }
        if (sub == 0) sm.head_end[grp] = r1;
      } else {
        pend.retire(a, sub);
        tc.seek(a, ckey);
        pend.issue(a, tc, ckey, B0 + r1, acc, sub);
      }
    } else {
      const int side = chead ? 0 : 1;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < D4) sm.part[side][grp * D4 + f4] = acc[v];
      }
      if (sub == 0) {
        if (chead) {
          sm.head_end[grp] = r1;
          sm.head_thru[grp] = 1;
        } else {
          sm.tail_valid[grp] = 1;
          sm.tail_key[grp] = ckey;
        }
      }
    }
  }
  pend.retire(a, sub);
  __syncthreads();

  // ---- runs cut between groups: the group holding a run's start adds the
  //      head partials of the following groups in order ----
  int32_t* P = a.part_pos + (int64_t)blockIdx.x * 2;
  float4* GP = a.partial + (int64_t)blockIdx.x * 2 * D4;
  if (sm.tail_valid[grp]) {
    float4 s[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      s[v] = f4 < D4 ? sm.part[1][grp * D4 + f4] : seg_f4zero();
    }
    int g2 = grp + 1;
    bool thru = true;
    int end = span;
    while (g2 < NG && thru) {
      if (sm.head_end[g2] < 0) break;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < D4) seg_f4add(s[v], sm.part[0][g2 * D4 + f4]);
      }
      thru = sm.head_thru[g2] != 0;
      end = sm.head_end[g2];
      ++g2;
    }
    if (g2 == NG && thru) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < D4) GP[D4 + f4] = s[v];
      }
    } else {
      finish_row<V>(a, sm.tail_key[grp], B0 + end, s, sub);
    }
  }
  // ---- the run cut at the CTA start: group 0 sums the head partials ----
  if (grp == 0) {
    bool thru = false;
    int end = 0;
    float4 s[V];
#pragma unroll
    for (int v = 0; v < V; ++v) s[v] = seg_f4zero();
    if (sm.head_end[0] >= 0) {
      int g2 = 0;
      thru = true;
      while (g2 < NG && thru) {
        if (sm.head_end[g2] < 0) {
          thru = false;
          break;
        }
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const int f4 = sub + v * 32;
          if (f4 < D4) seg_f4add(s[v], sm.part[0][g2 * D4 + f4]);
        }
        thru = sm.head_thru[g2] != 0;
        end = sm.head_end[g2];
        ++g2;
      }
      if (g2 < NG) thru = false;
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      if (f4 < D4) GP[f4] = s[v];
    }
    if (sub == 0) {
      P[0] = end;
      a.part_thru[blockIdx.x] = thru ? 1 : 0;
    }
  }
}

// Runs cut by CTA boundaries: one lane group per boundary b (between CTA b-1
// and CTA b) that is the first boundary inside its run.
constexpr int kFixLook = 8;
template <int V>
__global__ void __launch_bounds__(kSegThreads) k_seg_fixup(const SegArgs a, int n_blocks, int64_t span) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int glog = a.glog;
  const int G = 32 >> glog;
  const int grp = lane >> glog, sub = lane & ((1 << glog) - 1);
  const int64_t b = 1 + (int64_t)blockIdx.x * kSegWarps * G + warp * G + grp;
  if (b >= n_blocks) return;
  const int64_t pos = b * span;
  if (pos >= a.n) return;
  const uint32_t key = __ldg(a.keys + pos);
  if (key == a.sentinel || __ldg(a.keys + pos - 1) != key) return;
  if (b > 1 && __ldg(a.keys + (b - 1) * span - 1) == key) return;  // an earlier boundary owns it
  const int D4 = a.maxdim4;
  float4 s[V];
  const float4* T = a.partial + (b - 1) * 2 * D4 + D4;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int f4 = sub + v * 32;
    s[v] = f4 < D4 ? T[f4] : seg_f4zero();
  }
  // CTAs c, c+1, ... contribute their head partials while the one before
  // lies wholly inside the run; their flags and partials are loaded
  // kFixLook at a time (independent loads), then added in CTA order
  int64_t c = b, end = pos;
  bool go = true;
  while (go) {
    bool thru[kFixLook];
    int32_t hp[kFixLook];
    float4 h[kFixLook][V];
#pragma unroll
    for (int j = 0; j < kFixLook; ++j) {
      const int64_t cj = c + j;
      const bool in = cj < n_blocks;
      thru[j] = in && a.part_thru[cj];
      hp[j] = in ? a.part_pos[cj * 2] : 0;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        h[j][v] = (in && f4 < D4) ? a.partial[cj * 2 * D4 + f4] : seg_f4zero();
      }
    }
#pragma unroll
    for (int j = 0; j < kFixLook; ++j) {
      if (go) {
#pragma unroll
        for (int v = 0; v < V; ++v)
          if (sub + v * 32 < D4) seg_f4add(s[v], h[j][v]);
        end = (c + j) * span + hp[j];
        go = thru[j] && c + j + 1 < n_blocks;
      }
    }
    c += kFixLook;
  }
  finish_row<V>(a, key, end, s, sub);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
emb_status launch_backward(emb_plan_s* p, const float* grad_out, const float* grad_seq, float lr, float eps,
                           cudaStream_t stream, const emb_backward_debug* dbg) {
  Workspace& w = p->ws;
  const int64_t n = p->last_n;
  const bool want_dbg = dbg && (dbg->uniq_table || dbg->uniq_row || dbg->counts || dbg->agg_grad || dbg->n_unique);
  if (n == 0) {
    if (want_dbg && dbg->n_unique) EMB_CUDA_TRY(cudaMemsetAsync(dbg->n_unique, 0, sizeof(int64_t), stream));
    return EMB_OK;
  }
  int res = 0;
  emb_status st = radix_sort_pairs<uint32_t>(w.keys, w.vals, n, nullptr, n, p->key_bits, w.hist, p->sm_count,
                                             p->status_d, stream, &res);
  if (st != EMB_OK) return st;
  const uint32_t* skeys = w.keys[res];
  const uint32_t* svals = w.vals[res];

  SegArgs a{};
  a.keys = skeys;
  a.vals = svals;
  a.n = n;
  a.sentinel = p->key_total;
  a.colg = p->colg_d;
  a.inv_n = w.inv_n;
  a.rec_src = p->last_weighted ? w.rec_src : nullptr;
  a.grad_out = grad_out;
  a.ldg = p->out_width;
  a.grad_seq = grad_seq;
  a.batch = p->last_batch > 0 ? p->last_batch : 1;
  a.bdiv = make_div_magic32((uint32_t)a.batch);
  a.tables = p->tables_d;
  a.table_base = p->table_base_d;
  a.n_tables = p->n_tables;
  a.lr = lr;
  a.eps = eps;
  a.maxdim4 = p->max_dim / 4;
  int g = a.maxdim4 > 32 ? 32 : a.maxdim4, glog = 0;
  while ((1 << glog) < g) ++glog;
  a.glog = glog;
  const int NG = kSegWarps * (32 >> glog);
  a.span = seg_span(glog);
  const int64_t span = a.span;
  const int64_t n_blocks = (n + span - 1) / span;
  if (n_blocks > w.n_units_max) return EMB_ERR_UNSUPPORTED;
  a.partial = w.partial;
  a.part_pos = w.part_pos;
  a.part_thru = w.part_thru;
  if (want_dbg) {
    const int nb = (int)((n + kScanBlock - 1) / kScanBlock);
    k_rank_reduce<<<nb, kScanBlock, 0, stream>>>(skeys, n, p->key_total, w.scan_part);
    k_rank_top<<<1, kScanBlock, 0, stream>>>(w.scan_part, nb,
                                             dbg->n_unique ? dbg->n_unique : reinterpret_cast<int64_t*>(w.n_runs));
    k_rank_down<<<nb, kScanBlock, 0, stream>>>(skeys, n, p->key_total, w.scan_part, w.run_head, w.head_pos);
    a.rank = w.run_head;
    a.dbg_table = dbg->uniq_table;
    a.dbg_row = dbg->uniq_row;
    a.dbg_count = dbg->counts;
    a.dbg_grad = dbg->agg_grad;
    a.dbg_ld = p->max_dim;
  }
  const unsigned fix_grid = (unsigned)std::max<int64_t>(1, (n_blocks - 1 + NG - 1) / NG);
  if (a.maxdim4 > 32) {
    k_segreduce<2><<<(unsigned)n_blocks, kSegThreads, 0, stream>>>(a);
    if (n_blocks > 1) k_seg_fixup<2><<<fix_grid, kSegThreads, 0, stream>>>(a, (int)n_blocks, span);
  } else {
    k_segreduce<1><<<(unsigned)n_blocks, kSegThreads, 0, stream>>>(a);
    if (n_blocks > 1) k_seg_fixup<1><<<fix_grid, kSegThreads, 0, stream>>>(a, (int)n_blocks, span);
  }
  if (want_dbg && (dbg->uniq_table || dbg->uniq_row || dbg->counts)) {
    const int64_t* nu = dbg->n_unique ? dbg->n_unique : reinterpret_cast<const int64_t*>(w.n_runs);
    k_dbg_runs<<<p->sm_count * 4, 256, 0, stream>>>(skeys, n, p->key_total, w.head_pos, nu, p->table_base_d,
                                                    p->n_tables, dbg->uniq_table, dbg->uniq_row, dbg->counts);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace emb

// ===========================================================================
// emb_sparse_adagrad_noalloc: the sort + run reduction + Adagrad update above,
// for one table, on a fixed scratch area compiled into the library instead of
// memory from cudaMalloc.
// ===========================================================================
namespace emb {
namespace {

constexpr int64_t kNoAllocMaxN = int64_t(1) << 18;   // contributions per call
constexpr int kNoAllocMaxDim = 256;
constexpr int64_t kNoAllocTiles = (kNoAllocMaxN + kSortTile - 1) / kSortTile;
constexpr int64_t kNoAllocBlocks = (kNoAllocMaxN + 255) / 256;   // the smallest span seg_span() returns
// sort_scratch_words for up to 32-bit keys: four passes of 8-bit digits
constexpr size_t kNoAllocSortWords = 4 * 256 + 4 + 4 * kNoAllocTiles * 256;

struct NoAllocScratch {
  uint32_t keys[2][kNoAllocMaxN];
  uint32_t vals[2][kNoAllocMaxN];
  uint32_t sortw[kNoAllocSortWords];   // histograms, tile tickets, look-back words
  float4 partial[kNoAllocBlocks * 2 * (kNoAllocMaxDim / 4)];
  int32_t part_pos[kNoAllocBlocks * 2];
  uint8_t part_thru[kNoAllocBlocks];
  TableMeta table;
  uint32_t table_base[2];
  int4 colg;
};

}  // namespace

// The scratch area: every GPU that loads the library holds one copy until the
// process exits; all calls on a device share it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(NoAllocScratch)];

__global__ void k_noalloc_setup(NoAllocScratch* s, float* weight, float* acc, int64_t num_rows, int32_t dim) {
  if (threadIdx.x == 0) {
    s->table.weight = weight;
    s->table.acc = acc;
    s->table.num_rows = num_rows;
    s->table.dim = dim;
    s->table.dim4 = dim / 4;
    s->table_base[0] = 0u;
    s->table_base[1] = (uint32_t)num_rows;
    s->colg = make_int4(0, 0, dim / 4, 0);
  }
}

// (row, contribution index) pairs; a row outside [0, num_rows) is dropped by
// giving it the sentinel key num_rows, which sorts after every valid row.
__global__ void k_noalloc_pairs(const int64_t* __restrict__ rows, int64_t n, int64_t num_rows,
                                uint32_t* __restrict__ keys, uint32_t* __restrict__ vals) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i < n) {
    const int64_t r = rows[i];
    keys[i] = (r >= 0 && r < num_rows) ? (uint32_t)r : (uint32_t)num_rows;
    vals[i] = (uint32_t)i;
  }
}

namespace {
constexpr int kNoAllocMaxDevices = 64;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};
int g_noalloc_sms[kNoAllocMaxDevices] = {};

// Device address of the scratch area on the current device (and its SM
// count), looked up once per device: the first call on a device does this
// set-up.
emb_status noalloc_scratch(NoAllocScratch** out, int* sms) {
  int dev = 0;
  EMB_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return EMB_ERR_UNSUPPORTED;
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      cudaGetLastError();
      return EMB_ERR_CUDA;
    }
    int count = 0;
    EMB_CUDA_TRY(cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev));
    g_noalloc_sms[dev] = count > 0 ? count : 1;
    g_noalloc_addr[dev] = ptr;
  }
  *out = static_cast<NoAllocScratch*>(g_noalloc_addr[dev]);
  *sms = g_noalloc_sms[dev];
  return EMB_OK;
}
}  // namespace

}  // namespace emb

extern "C" emb_status emb_sparse_adagrad_noalloc(const int64_t* rows, int64_t n, const float* grads,
                                                 float* weight, float* acc, int64_t num_rows, int32_t dim,
                                                 float lr, float eps, void* stream_) {
  using namespace emb;
  if (n < 0 || num_rows < 1 || dim < 4 || dim % 4 != 0) return EMB_ERR_INVALID_ARG;
  if (n > kNoAllocMaxN || dim > kNoAllocMaxDim || num_rows >= (int64_t(1) << 31)) return EMB_ERR_UNSUPPORTED;
  if (!weight || !acc || !aligned16(weight) || !aligned16(acc)) return EMB_ERR_INVALID_ARG;
  if (n > 0 && (!rows || !grads || !aligned16(grads))) return EMB_ERR_INVALID_ARG;
  if (!(lr == lr) || !(eps == eps)) return EMB_ERR_INVALID_ARG;
  NoAllocScratch* s = nullptr;
  int sms = 1;
  emb_status st = noalloc_scratch(&s, &sms);
  if (st != EMB_OK) return st;
  if (n == 0) return EMB_OK;
  cudaStream_t stream = (cudaStream_t)stream_;

  int key_bits = 1;
  while (key_bits < 32 && (uint64_t(1) << key_bits) <= (uint64_t)num_rows) ++key_bits;
  k_noalloc_setup<<<1, 32, 0, stream>>>(s, weight, acc, num_rows, dim);
  k_noalloc_pairs<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(rows, n, num_rows, s->keys[0], s->vals[0]);
  uint32_t* const nk[2] = {s->keys[0], s->keys[1]};
  uint32_t* const nv[2] = {s->vals[0], s->vals[1]};
  int res = 0;
  // the sort clears its part of the area (histograms, tickets, look-back words) itself
  st = radix_sort_pairs<uint32_t>(nk, nv, n, nullptr, n, key_bits, s->sortw, sms, nullptr, stream, &res);
  if (st != EMB_OK) return st;
  SegArgs a{};
  a.keys = s->keys[res];
  a.vals = s->vals[res];
  a.n = n;
  a.sentinel = (uint32_t)num_rows;
  a.colg = &s->colg;
  a.inv_n = nullptr;
  a.grad_out = grads;
  a.ldg = dim;
  a.grad_seq = nullptr;
  a.batch = (int32_t)n;
  a.bdiv = make_div_magic32((uint32_t)n);
  a.tables = &s->table;
  a.table_base = s->table_base;
  a.n_tables = 1;
  a.lr = lr;
  a.eps = eps;
  a.maxdim4 = dim / 4;
  int g = a.maxdim4 > 32 ? 32 : a.maxdim4, glog = 0;
  while ((1 << glog) < g) ++glog;
  a.glog = glog;
  const int NG = kSegWarps * (32 >> glog);
  a.span = seg_span(glog);
  const int64_t span = a.span;
  const int64_t n_blocks = (n + span - 1) / span;
  a.partial = s->partial;
  a.part_pos = s->part_pos;
  a.part_thru = s->part_thru;
  const unsigned fix_grid = (unsigned)std::max<int64_t>(1, (n_blocks - 1 + NG - 1) / NG);
  if (a.maxdim4 > 32) {
    k_segreduce<2><<<(unsigned)n_blocks, kSegThreads, 0, stream>>>(a);
    if (n_blocks > 1) k_seg_fixup<2><<<fix_grid, kSegThreads, 0, stream>>>(a, (int)n_blocks, span);
  } else {
    k_segreduce<1><<<(unsigned)n_blocks, kSegThreads, 0, stream>>>(a);
    if (n_blocks > 1) k_seg_fixup<1><<<fix_grid, kSegThreads, 0, stream>>>(a, (int)n_blocks, span);
  }
  return cuda_status(cudaGetLastError());
}
