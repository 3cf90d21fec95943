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
//                       gathering scale * G rows (several in flight) and
//                       summing each run; a run that begins
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
  const uint32_t* sort_fail;   // the sort's fail word: nonzero = its output has holes, do nothing
  int32_t prefetch;       // stage run heads' weight / accumulator rows into L2 while decoding
  // debug outputs
  const uint32_t* rank;
  int32_t* dbg_table;
  int64_t* dbg_row;
  int32_t* dbg_count;
  float* dbg_grad;
  int32_t dbg_ld;
};


// Lanes of a lane group; lane `sub` of a group holds float4 slices sub,
// sub + lanes, sub + 2 * lanes, ... of a row (consecutive lanes, consecutive
// 16-byte slices: each slice index v is one coalesced access per group).
__device__ __forceinline__ int seg_lanes(const SegArgs& a) { return 1 << a.glog; }

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
    const int f4 = sub + v * seg_lanes(a);
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
      const int f4 = sub + v * seg_lanes(a);
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
      const int f4 = sub + v * seg_lanes(a);
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
      const int f4 = sub + v * seg_lanes(a);
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
        const int f4 = sub + v * seg_lanes(a);
        if (f4 < dim4) *reinterpret_cast<float4*>(a.dbg_grad + (int64_t)u * a.dbg_ld + f4 * 4) = g[v];
      }
    }
  }
};

// Sorted entries per CTA: about 64 per lane group (measured best on the
// training and sequence workloads), between 256 and kSegSpanMax.
constexpr int kSegSpanMax = 1024;
constexpr int kSegPerGroup = 64;
constexpr int kSegDec = 4;   // entries a thread decodes per batch of loads

inline int seg_span(int glog) {
  const int ng = kSegThreads / 32 * (32 >> glog);
  const int s = kSegPerGroup * ng;
  return s < 256 ? 256 : (s > kSegSpanMax ? kSegSpanMax : s);
}

// The plan's span: seg_span, or less for a step with too few contributions
// to give every SM two CTAs -- down to four entries per lane group and at
// least kUnit entries (the plan's partial buffers hold n / kUnit CTAs).  A
// lane group's chain of dependent row loads is then a few runs long.
inline int seg_span_plan(int glog, int64_t n, int sms) {
  const int ng = kSegThreads / 32 * (32 >> glog);
  const int full = seg_span(glog);
  const int64_t want = (n + 2 * (int64_t)sms - 1) / (2 * (int64_t)sms);
  int s = full;
  while (s > want && s / 2 >= kUnit && s / 2 >= ng * 4 && (s / 2) % ng == 0) s /= 2;
  return s;
}
// Resident CTAs per SM (rows wider than 128 floats take fewer to stay within
// the registers), and gradient rows in flight per lane group.  The rows are
// staged in shared memory by per-thread asynchronous copies (cp.async, 16 B
// per lane and row): each lane copies and later reads only its own slice, so
// a ring of kSegRing rows per group needs no barrier, and the rows in
// flight cost shared memory instead of registers.
template <int V>
struct SegDepth {
  static constexpr int ctas = V == 1 ? 6 : 4;
  static constexpr int ring = 8;   // rows in flight per lane group
};
constexpr uint32_t kOffPad = 0x80000000u;
// The decode stages each run head's weight and accumulator rows into L2 for
// the update that follows: for steps of at least kPrefetchMinN entries and
// runs of pooled gradient sources.  A small step's rows are few and the
// instructions are overhead (tiny step 33.2 -> 31.2 us per step in graphs
// without); runs of padded sources gather their gradient rows from HBM,
// which evicts the staged rows before their update reads them (DRAM reads
// of the padded sequence backward's reduction 12.4 GB, its call 2.82 ms,
// against 2.52 ms without), while the pooled workloads keep their gain
// (training 4.20 -> 4.12 ms, mean sequences 2.18 -> 2.11 ms with it).
constexpr int64_t kPrefetchMinN = int64_t(1) << 16;         // offset refers to grad_seq
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

// Dynamic shared memory of one CTA, laid out for its span and row width:
// the decoded records, the head / tail partial of each lane group, the
// gradient-row ring of every lane, and the per-group run bookkeeping.
struct SegLayout {
  int rec, part, ring, head_end, tail_key, head_thru, tail_valid, bytes;
  __host__ __device__ static SegLayout of(int span, int ng, int d4, int v, int ring_depth, int threads = kSegThreads) {
    SegLayout L;
    int o = 0;
    L.rec = o;
    o += span * (int)sizeof(SegRec);
    L.part = o;
    o += 2 * ng * d4 * 16;
    L.ring = o;
    o += ring_depth * threads * v * 16;
    L.head_end = o;
    o += ng * 4;
    L.tail_key = o;
    o += ng * 4;
    L.head_thru = o;
    o += ng;
    L.tail_valid = o;
    o += ng;
    L.bytes = (o + 15) & ~15;
    return L;
  }
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16 bytes global -> shared, asynchronous; bytes < 16 zero-fills the rest
// (0: nothing is read and the slot reads as zeros).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Runs of sorted contributions are reduced by LANE GROUPS (V float4 slices
// of a row per lane, see seg_lanes): the CTA's span is cut into equal
// contiguous ranges, one per group, and a group walks its range in order,
// kSegRing gradient rows in flight, adding each row into the open run's sum
// and closing the run where the key changes.  A run closed inside the range
// that also began there is finished at once (Adagrad on its row, deferred by
// one run so the weight/accumulator loads overlap the next gathers); a run
// cut at the range start leaves a head partial and one open at the range end
// a tail partial, combined in group order after a barrier (and across CTAs
// by k_seg_fixup).
// The work of one CTA of TH threads over the `span` sorted entries starting
// at cta * span; seg_smem: its dynamic shared memory (SegLayout).
template <int V, int TH>
__device__ __forceinline__ void segreduce_body(const SegArgs& a, int64_t cta, unsigned char* seg_smem) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int glog = a.glog;
  const int G = 32 >> glog;
  const int q = lane >> glog, sub = lane & ((1 << glog) - 1);
  const int NG = (TH / 32) * G;
  const int grp = warp * G + q;
  const int64_t B0 = (int64_t)cta * a.span;
  const int64_t B1 = min(B0 + (int64_t)a.span, a.n);
  const int span = (int)(B1 - B0);
  const int D4 = a.maxdim4;
  constexpr int kSegRing = SegDepth<V>::ring;
  const SegLayout L = SegLayout::of(a.span, NG, D4, V, kSegRing, TH);
  SegRec* rec = reinterpret_cast<SegRec*>(seg_smem + L.rec);
  float4* part = reinterpret_cast<float4*>(seg_smem + L.part);   // [2][NG * D4]
  float4* ring = reinterpret_cast<float4*>(seg_smem + L.ring);   // [kSegRing][TH * V]
  int32_t* head_end = reinterpret_cast<int32_t*>(seg_smem + L.head_end);
  uint32_t* tail_key = reinterpret_cast<uint32_t*>(seg_smem + L.tail_key);
  uint8_t* head_thru = seg_smem + L.head_thru;
  uint8_t* tail_valid = seg_smem + L.tail_valid;

  // ---- decode the CTA's entries, coalesced, into shared memory; the
  //      weight and accumulator rows of the runs of pooled sources that
  //      start here are prefetched into L2 (steps of at least kPrefetchMinN
  //      entries) so that the updates below find them there ----
  //      Entries are taken kSegDec per thread at a time and each stage's
  //      loads (key, previous key and source; weight; column; 1/n) are all
  //      issued before any is used, so a thread waits for each stage once
  //      instead of once per entry.
  uint32_t lkey = a.sentinel;
  int ld4 = 0;
  TableCursor ptc;
  for (int e0 = tid; e0 < a.span; e0 += kSegDec * TH) {
    uint32_t kk[kSegDec], kp[kSegDec], vv[kSegDec];
#pragma unroll
    for (int j = 0; j < kSegDec; ++j) {
      const int e = e0 + j * TH;
      kk[j] = a.sentinel;
      kp[j] = kNoKey;
      vv[j] = 0u;
      if (e < span) {
        kk[j] = __ldg(a.keys + B0 + e);
        vv[j] = __ldg(a.vals + B0 + e);
        if (B0 + e > 0) kp[j] = __ldg(a.keys + B0 + e - 1);
      }
    }
    float wr[kSegDec];   // value weight of a SUM contribution
#pragma unroll
    for (int j = 0; j < kSegDec; ++j) {
      wr[j] = 1.0f;
      if (a.rec_src && kk[j] != a.sentinel) {
        const uint2 rs = __ldg(a.rec_src + vv[j]);
        vv[j] = rs.x;
        wr[j] = __uint_as_float(rs.y);
      }
    }
    int4 cg[kSegDec];
#pragma unroll
    for (int j = 0; j < kSegDec; ++j) {
      cg[j] = make_int4(0, 0, 0, 0);
      if (kk[j] != a.sentinel && !(vv[j] & kPadBit)) cg[j] = __ldg(a.colg + div_magic32(vv[j], a.bdiv));
    }
    float sc[kSegDec];
#pragma unroll
    for (int j = 0; j < kSegDec; ++j) sc[j] = cg[j].y ? __ldg(a.inv_n + vv[j]) : wr[j];
#pragma unroll
    for (int j = 0; j < kSegDec; ++j) {
      const int e = e0 + j * TH;
      if (e >= a.span) break;
      SegRec r;
      r.key = a.sentinel;
      r.off = 0u;
      r.scale = 0.0f;
      r.d4 = 0u;
      const uint32_t key = kk[j];
      if (e < span && key != a.sentinel) {
        r.key = key;
        if (a.prefetch && kp[j] != key && !(vv[j] & kPadBit)) {   // a run of pooled sources starts here
          ptc.seek(a, key);
          const int64_t row = key - ptc.base;
          prefetch_l2(ptc.weight + row * ptc.dim, (uint32_t)ptc.dim * 4u);
          prefetch_l2(ptc.acc + row * ptc.dim, (uint32_t)ptc.dim * 4u);
        }
        const uint32_t val = vv[j];
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
          r.scale = sc[j];
          r.d4 = (uint32_t)cg[j].z;
          r.off = (uint32_t)(((int64_t)b * a.ldg + cg[j].x) >> 2);
        }
      }
      rec[e] = r;
    }
  }
  for (int g = tid; g < NG; g += TH) {
    head_end[g] = -1;
    head_thru[g] = 0;
    tail_valid[g] = 0;
  }
  __syncthreads();

  // ---- per lane group: its contiguous range, in order ----
  const int R = a.span / NG;
  const int r0 = min(grp * R, span), r1 = min(r0 + R, span);
  uint32_t ckey = kNoKey;   // key of the open run
  bool chead = false;       // the open run began before this range
  if (r0 < r1) {
    ckey = rec[r0].key;
    const uint32_t prev = r0 > 0 ? rec[r0 - 1].key : (B0 > 0 ? __ldg(a.keys + B0 - 1) : kNoKey);
    chead = prev == ckey && ckey != a.sentinel;
  }
  // this lane's ring slots: slot j holds V float4 at ring[(j * TH + tid) * V + v]
  const uint32_t ring0 = smem_u32(ring + (size_t)tid * V);
  constexpr uint32_t kSlotBytes = (uint32_t)TH * V * 16u;
  auto issue = [&](int e, int slot) {
    if (e < r1) {
      const SegRec r = rec[e];
      const float* src = (r.off & kOffPad) ? a.grad_seq + (int64_t)(r.off & ~kOffPad) * 4
                                           : a.grad_out + (int64_t)r.off * 4;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * seg_lanes(a);
        const bool in = f4 < (int)r.d4;
        // a lane past the row reads nothing (zero fill) from a valid address
        cp_async16(ring0 + (uint32_t)slot * kSlotBytes + v * 16u, in ? (const void*)(src + f4 * 4) : (const void*)a.keys,
                   in ? 16u : 0u);
      }
    }
    cp_async_commit();   // one group per entry, empty past the range
  };
#pragma unroll
  for (int k = 0; k < kSegRing; ++k) issue(r0 + k, k);

  float4 acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = seg_f4zero();
  TableCursor tc;
  PendingRow<V> pend;
  int slot = 0;
  for (int e = r0; e < r1; ++e) {
    cp_async_wait<kSegRing - 1>();   // entry e's row has landed
    const uint32_t key = rec[e].key;
    const float sc = rec[e].scale;
    float4 x[V];
#pragma unroll
    for (int v = 0; v < V; ++v) x[v] = ring[((size_t)slot * TH + tid) * V + v];
    if (key != ckey) {   // the open run ends before this entry
      if (ckey != a.sentinel) {
        if (chead) {
#pragma unroll
          for (int v = 0; v < V; ++v) {
            const int f4 = sub + v * seg_lanes(a);
            if (f4 < D4) part[grp * D4 + f4] = acc[v];
          }
          if (sub == 0) head_end[grp] = e;
        } else {
          pend.retire(a, sub);
          tc.seek(a, ckey);
          pend.issue(a, tc, ckey, B0 + e, acc, sub);
        }
      }
      ckey = key;
      chead = false;
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] = seg_f4zero();
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
      acc[v].x = fmaf(x[v].x, sc, acc[v].x);
      acc[v].y = fmaf(x[v].y, sc, acc[v].y);
      acc[v].z = fmaf(x[v].z, sc, acc[v].z);
      acc[v].w = fmaf(x[v].w, sc, acc[v].w);
    }
    // the slot just read takes the row kSegRing entries ahead
    issue(e + kSegRing, slot);
    slot = slot + 1 == kSegRing ? 0 : slot + 1;
  }
  cp_async_wait<0>();
  // the run open at the range end: finished here, or left as a partial
  if (r0 < r1 && ckey != a.sentinel) {
    const uint32_t key_after = r1 < span ? rec[r1].key : (B1 < a.n ? __ldg(a.keys + B1) : kNoKey);
    if (key_after != ckey) {
      if (chead) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const int f4 = sub + v * seg_lanes(a);
          if (f4 < D4) part[grp * D4 + f4] = acc[v];
        }
        if (sub == 0) head_end[grp] = r1;
      } else {
        pend.retire(a, sub);
        tc.seek(a, ckey);
        pend.issue(a, tc, ckey, B0 + r1, acc, sub);
      }
    } else {
      const int side = chead ? 0 : 1;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * seg_lanes(a);
        if (f4 < D4) part[side * NG * D4 + grp * D4 + f4] = acc[v];
      }
      if (sub == 0) {
        if (chead) {
          head_end[grp] = r1;
          head_thru[grp] = 1;
        } else {
          tail_valid[grp] = 1;
          tail_key[grp] = ckey;
        }
      }
    }
  }
  pend.retire(a, sub);
  __syncthreads();

  // ---- runs cut between groups: the group holding a run's start adds the
  //      head partials of the following groups in order ----
  int32_t* P = a.part_pos + (int64_t)cta * 2;
  float4* GP = a.partial + (int64_t)cta * 2 * D4;
  if (tail_valid[grp]) {
    float4 s[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * seg_lanes(a);
      s[v] = f4 < D4 ? part[NG * D4 + grp * D4 + f4] : seg_f4zero();
    }
    int g2 = grp + 1;
    bool thru = true;
    int end = span;
    while (g2 < NG && thru) {
      if (head_end[g2] < 0) break;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * seg_lanes(a);
        if (f4 < D4) seg_f4add(s[v], part[g2 * D4 + f4]);
      }
      thru = head_thru[g2] != 0;
      end = head_end[g2];
      ++g2;
    }
    if (g2 == NG && thru) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * seg_lanes(a);
        if (f4 < D4) GP[D4 + f4] = s[v];
      }
    } else {
      finish_row<V>(a, tail_key[grp], B0 + end, s, sub);
    }
  }
  // ---- the run cut at the CTA start: group 0 sums the head partials ----
  if (grp == 0) {
    bool thru = false;
    int end = 0;
    float4 s[V];
#pragma unroll
    for (int v = 0; v < V; ++v) s[v] = seg_f4zero();
    if (head_end[0] >= 0) {
      int g2 = 0;
      thru = true;
      while (g2 < NG && thru) {
        if (head_end[g2] < 0) {
          thru = false;
          break;
        }
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const int f4 = sub + v * seg_lanes(a);
          if (f4 < D4) seg_f4add(s[v], part[g2 * D4 + f4]);
        }
        thru = head_thru[g2] != 0;
        end = head_end[g2];
        ++g2;
      }
      if (g2 < NG) thru = false;
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * seg_lanes(a);
      if (f4 < D4) GP[f4] = s[v];
    }
    if (sub == 0) {
      P[0] = end;
      a.part_thru[cta] = thru ? 1 : 0;
    }
  }
}

template <int V>
__global__ void __launch_bounds__(kSegThreads, SegDepth<V>::ctas) k_segreduce(const SegArgs a) {
  extern __shared__ __align__(16) unsigned char seg_smem[];
  pdl_wait();   // the sort has finished
  pdl_trigger();   // the fixup launched after this kernel may be scheduled
  if (*(volatile const uint32_t*)a.sort_fail) return;   // the same for every thread of the CTA
  segreduce_body<V, kSegThreads>(a, blockIdx.x, seg_smem);
}

// Runs cut by CTA boundaries: one lane group per boundary b (between CTA b-1
// and CTA b) that is the first boundary inside its run.
template <int V>
__global__ void __launch_bounds__(kSegThreads) k_seg_fixup(const SegArgs a, int n_blocks, int64_t span) {
  constexpr int kFixLook = 8;   // CTA partials loaded per round trip
  pdl_wait();   // every CTA of the run reduction has finished
  if (*(volatile const uint32_t*)a.sort_fail) return;
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
    const int f4 = sub + v * seg_lanes(a);
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
        const int f4 = sub + v * seg_lanes(a);
        h[j][v] = (in && f4 < D4) ? a.partial[cj * 2 * D4 + f4] : seg_f4zero();
      }
    }
#pragma unroll
    for (int j = 0; j < kFixLook; ++j) {
      if (go) {
#pragma unroll
        for (int v = 0; v < V; ++v)
          if (sub + v * seg_lanes(a) < D4) seg_f4add(s[v], h[j][v]);
        end = (c + j) * span + hp[j];
        go = thru[j] && c + j + 1 < n_blocks;
      }
    }
    c += kFixLook;
  }
  finish_row<V>(a, key, end, s, sub);
}

// Shared memory bytes of a k_segreduce launch, and the launch itself (the
// attribute for more than 48 KB is set on first use).
// Float4 slices per lane of the run reduction: one, with lane groups of
// dim/4 lanes; two for rows wider than 128 floats (groups of 32 lanes).
// Measured on the training workload (backward + Adagrad per step): four
// slices per lane (eight 4-lane groups per warp) 6.13 ms and two 5.92 ms
// against 4.61 ms with one -- with more groups per warp nearly every step
// of the walk has some group closing a run, so the whole warp pays the
// retire path each step.
inline int seg_v(int maxdim4) { return maxdim4 > 32 ? 2 : 1; }

// log2 of the lanes per group for rows of up to maxdim4 float4.
inline int seg_glog(int maxdim4) {
  const int v = seg_v(maxdim4);
  const int need = (maxdim4 + v - 1) / v;
  int glog = 0;
  while ((1 << glog) < need) ++glog;
  return glog;
}

template <int V>
inline emb_status launch_segreduce_v(const SegArgs& a, int64_t n_blocks, cudaStream_t stream) {
  const int NG = kSegWarps * (32 >> a.glog);
  const unsigned fix_grid = (unsigned)std::max<int64_t>(1, (n_blocks - 1 + NG - 1) / NG);
  const int smem = SegLayout::of(a.span, NG, a.maxdim4, V, SegDepth<V>::ring).bytes;
  EMB_CUDA_TRY(cudaFuncSetAttribute(k_segreduce<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  EMB_CUDA_TRY(launch_dependent(k_segreduce<V>, (unsigned)n_blocks, kSegThreads, smem, stream, a));
  if (n_blocks > 1)
    EMB_CUDA_TRY(launch_dependent(k_seg_fixup<V>, fix_grid, kSegThreads, 0, stream, a, (int)n_blocks, a.span));
  return EMB_OK;
}

// The run reduction and the fixup of its cut runs (the shared-memory size
// attribute is set on every launch: it depends on the span and row width).
inline emb_status launch_segreduce(const SegArgs& a, int64_t n_blocks, cudaStream_t stream) {
  return seg_v(a.maxdim4) == 2 ? launch_segreduce_v<2>(a, n_blocks, stream)
                               : launch_segreduce_v<1>(a, n_blocks, stream);
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
  SegArgs a{};
  a.n = n;
  a.sentinel = p->key_total;
  a.colg = p->colg_d;
  a.inv_n = w.inv_n;
  a.rec_src = p->last_weighted ? w.rec_src : nullptr;
  a.prefetch = n >= kPrefetchMinN ? 1 : 0;
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
  a.partial = w.partial;
  a.part_pos = w.part_pos;
  a.part_thru = w.part_thru;
  int64_t* const n_uniq = want_dbg ? (dbg->n_unique ? dbg->n_unique : reinterpret_cast<int64_t*>(w.n_runs)) : nullptr;
  if (want_dbg) {
    a.dbg_table = dbg->uniq_table;
    a.dbg_row = dbg->uniq_row;
    a.dbg_count = dbg->counts;
    a.dbg_grad = dbg->agg_grad;
    a.dbg_ld = p->max_dim;
  }
  int res = 0;
  emb_status st = radix_sort_pairs<uint32_t>(w.keys, w.vals, n, nullptr, n, p->key_bits, w.hist, p->sm_count,
                                             p->status_d, stream, &res);
  if (st != EMB_OK) return st;
  const uint32_t* skeys = w.keys[res];
  const uint32_t* svals = w.vals[res];
  a.keys = skeys;
  a.vals = svals;
  const int glog = seg_glog(a.maxdim4);
  a.glog = glog;
  a.span = seg_span_plan(glog, n, p->sm_count);
  const int64_t span = a.span;
  const int64_t n_blocks = (n + span - 1) / span;
  if (n_blocks > w.n_units_max) return EMB_ERR_UNSUPPORTED;
  a.sort_fail = sort_fail_word<uint32_t>(w.hist, p->key_bits);
  if (want_dbg) {
    const int nb = (int)((n + kScanBlock - 1) / kScanBlock);
    k_rank_reduce<<<nb, kScanBlock, 0, stream>>>(skeys, n, p->key_total, w.scan_part);
    k_rank_top<<<1, kScanBlock, 0, stream>>>(w.scan_part, nb, n_uniq);
    k_rank_down<<<nb, kScanBlock, 0, stream>>>(skeys, n, p->key_total, w.scan_part, w.run_head, w.head_pos);
    a.rank = w.run_head;
  }
  st = launch_segreduce(a, n_blocks, stream);
  if (st != EMB_OK) return st;
  if (want_dbg && (dbg->uniq_table || dbg->uniq_row || dbg->counts)) {
    const int64_t* nu = n_uniq;
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
constexpr int64_t kNoAllocBlocks = (kNoAllocMaxN + kUnit - 1) / kUnit;   // the smallest span seg_span_plan() returns
// sort_scratch_words for up to 32-bit keys: the larger of four passes of
// 8-bit digits and three of 9-bit digits
constexpr size_t kNoAllocSortWords = 3 * 512 + 3 + 1 + 3 * kNoAllocTiles * 512;
static_assert(kNoAllocSortWords >= 4 * 256 + 4 + 1 + 4 * kNoAllocTiles * 256, "no-alloc sort scratch");

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
  uint32_t status;   // first device-side error since the last emb_noalloc_get_device_status
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
    // the status word starts clear on this device
    EMB_CUDA_TRY(cudaMemset(&static_cast<NoAllocScratch*>(ptr)->status, 0, sizeof(uint32_t)));
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
  SegArgs a{};
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
  a.partial = s->partial;
  a.part_pos = s->part_pos;
  a.part_thru = s->part_thru;
  // the plan path's spans: the same sums in the same order
  int res = 0;
  // the sort clears its part of the area (histograms, tickets, look-back words) itself
  st = radix_sort_pairs<uint32_t>(nk, nv, n, nullptr, n, key_bits, s->sortw, sms, &s->status, stream, &res);
  if (st != EMB_OK) return st;
  a.keys = s->keys[res];
  a.vals = s->vals[res];
  const int glog = seg_glog(a.maxdim4);
  a.glog = glog;
  a.span = seg_span_plan(glog, n, sms);
  const int64_t span = a.span;
  const int64_t n_blocks = (n + span - 1) / span;
  a.sort_fail = sort_fail_word<uint32_t>(s->sortw, key_bits);
  st = launch_segreduce(a, n_blocks, stream);
  if (st != EMB_OK) return st;
  return cuda_status(cudaGetLastError());
}

extern "C" emb_status emb_noalloc_get_device_status(void* stream_) {
  using namespace emb;
  NoAllocScratch* s = nullptr;
  int sms = 1;
  emb_status st = noalloc_scratch(&s, &sms);
  if (st != EMB_OK) return st;
  cudaStream_t stream = (cudaStream_t)stream_;
  uint32_t code = 0;
  EMB_CUDA_TRY(cudaMemcpyAsync(&code, &s->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream));
  EMB_CUDA_TRY(cudaMemsetAsync(&s->status, 0, sizeof(uint32_t), stream));
  EMB_CUDA_TRY(cudaStreamSynchronize(stream));
  return (emb_status)code;
}

// ===========================================================================
// emb_selftest_sort_timeout: the bounded wait of the sort's look-back, made
// to run out on purpose (no counterpart on the pages; see include/emb.h).
// ===========================================================================
namespace emb {
namespace {

__global__ void k_selftest_fill(uint32_t* keys, uint32_t* vals, uint32_t* out_keys, uint32_t* out_vals, int64_t n,
                                uint32_t n_rows, float* grads, int dim) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    keys[i] = (uint32_t)(i % n_rows);   // valid rows of the test table
    vals[i] = (uint32_t)i;              // gradient row i exists
    out_keys[i] = n_rows;               // the sentinel: a hole reads as "no row"
    out_vals[i] = 0u;
    for (int d = 0; d < dim; ++d) grads[i * dim + d] = 1.0f;
  }
}

}  // namespace
}  // namespace emb

extern "C" emb_status emb_selftest_sort_timeout(uint32_t* latched, uint32_t* fail_word, int32_t* table_untouched,
                                                float* wait_ms) {
  using namespace emb;
  if (!latched || !fail_word || !table_untouched) return EMB_ERR_INVALID_ARG;
  constexpr uint32_t kRows = 16;
  constexpr int kDim = 4;
  const int64_t n = 2 * (int64_t)kSortTile;   // two tiles of one pass
  const int key_bits = 8;                      // one pass of 8-bit digits
  uint32_t *keys[2] = {nullptr, nullptr}, *vals[2] = {nullptr, nullptr}, *scratch = nullptr, *status = nullptr;
  float *grads = nullptr, *W = nullptr, *A = nullptr;
  float4* partial = nullptr;
  int32_t* part_pos = nullptr;
  uint8_t* part_thru = nullptr;
  TableMeta* tm_d = nullptr;
  uint32_t* base_d = nullptr;
  int4* colg_d = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  const size_t words = sort_scratch_words<uint32_t>(key_bits, n);
  const int64_t n_blocks = (n + 255) / 256;
  cudaError_t e = cudaSuccess;
  auto alloc = [&](auto** p, size_t bytes) {
    if (e == cudaSuccess) e = dev_alloc((void**)p, bytes);
  };
  for (int i = 0; i < 2; ++i) {
    alloc(&keys[i], sizeof(uint32_t) * n);
    alloc(&vals[i], sizeof(uint32_t) * n);
  }
  alloc(&scratch, sizeof(uint32_t) * words);
  alloc(&status, sizeof(uint32_t));
  alloc(&grads, sizeof(float) * n * kDim);
  alloc(&W, sizeof(float) * kRows * kDim);
  alloc(&A, sizeof(float) * kRows * kDim);
  alloc(&partial, sizeof(float4) * n_blocks * 2);
  alloc(&part_pos, sizeof(int32_t) * n_blocks * 2);
  alloc(&part_thru, n_blocks);
  alloc(&tm_d, sizeof(TableMeta));
  alloc(&base_d, sizeof(uint32_t) * 2);
  alloc(&colg_d, sizeof(int4));
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  float w_init[kRows * kDim];
  for (uint32_t i = 0; i < kRows * kDim; ++i) w_init[i] = 0.5f + (float)i;
  if (e == cudaSuccess) e = cudaMemcpy(W, w_init, sizeof(w_init), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(A, 0, sizeof(float) * kRows * kDim);
  if (e == cudaSuccess) e = cudaMemset(scratch, 0, sizeof(uint32_t) * words);
  if (e == cudaSuccess) e = cudaMemset(status, 0, sizeof(uint32_t));
  if (e == cudaSuccess) {
    TableMeta tm{};
    tm.weight = W;
    tm.acc = A;
    tm.num_rows = kRows;
    tm.dim = kDim;
    tm.dim4 = kDim / 4;
    const uint32_t base[2] = {0u, kRows};
    const int4 cg = make_int4(0, 0, kDim / 4, 0);
    e = cudaMemcpy(tm_d, &tm, sizeof(tm), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(base_d, base, sizeof(base), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(colg_d, &cg, sizeof(cg), cudaMemcpyHostToDevice);
  }
  uint32_t* hist = scratch;
  uint32_t* tickets = hist + 256;
  uint32_t* fail = sort_fail_word<uint32_t>(scratch, key_bits);
  uint32_t* lookback = fail + 1;
  const int smem = (int)sizeof(SortSmemT<uint32_t, 8>);
  if (e == cudaSuccess) {
    k_selftest_fill<<<64, 256>>>(keys[0], vals[0], keys[1], vals[1], n, kRows, grads, kDim);
    k_digit_hist_t<uint32_t, 8><<<8, 512>>>(keys[0], n, nullptr, 1, hist);
    // the first ticket is already taken: the one CTA below draws tile 1,
    // whose look-back waits on tile 0, which no CTA will ever publish
    const uint32_t one = 1u;
    e = cudaMemcpy(tickets, &one, sizeof(one), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_onesweep_t<uint32_t, 8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) {
    cudaEventRecord(e0);
    k_onesweep_t<uint32_t, 8, false><<<1, kSortThreads, smem>>>(keys[0], vals[0], keys[1], vals[1], n, nullptr, 0,
                                                                hist, lookback, tickets, status, fail);
    cudaEventRecord(e1);
    // a run reduction over the incomplete output: must see the fail word
    SegArgs a{};
    a.keys = keys[1];
    a.vals = vals[1];
    a.n = n;
    a.sentinel = kRows;
    a.colg = colg_d;
    a.grad_out = grads;
    a.ldg = kDim;
    a.batch = (int32_t)n;
    a.bdiv = make_div_magic32((uint32_t)n);
    a.tables = tm_d;
    a.table_base = base_d;
    a.n_tables = 1;
    a.lr = 0.5f;
    a.eps = 1e-10f;
    a.maxdim4 = kDim / 4;
    a.glog = 0;
    a.span = 256;   // seg_span for one-lane groups
    a.partial = partial;
    a.part_pos = part_pos;
    a.part_thru = part_thru;
    a.sort_fail = fail;
    if (launch_segreduce(a, n_blocks, 0) != EMB_OK) e = cudaErrorInvalidValue;
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) {
    float w_after[kRows * kDim];
    e = cudaMemcpy(w_after, W, sizeof(w_after), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(latched, status, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(fail_word, fail, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    *table_untouched = 1;
    for (uint32_t i = 0; i < kRows * kDim; ++i)
      if (w_after[i] != w_init[i]) *table_untouched = 0;
    if (wait_ms && e == cudaSuccess) e = cudaEventElapsedTime(wait_ms, e0, e1);
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  for (int i = 0; i < 2; ++i) {
    dev_free(keys[i]);
    dev_free(vals[i]);
  }
  dev_free(scratch);
  dev_free(status);
  dev_free(grads);
  dev_free(W);
  dev_free(A);
  dev_free(partial);
  dev_free(part_pos);
  dev_free(part_thru);
  dev_free(tm_d);
  dev_free(base_d);
  dev_free(colg_d);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_status(e);
  }
  return EMB_OK;
}
