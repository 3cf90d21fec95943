// forward.cu -- K-F: the fused multi-column forward (transform, safety check,
// row gather, pooling / padded copy, default fill) in ONE launch.
//
// Work decomposition (element-count tiling, RecIS §3.1 "Thread mapping for
// skewed inputs"): each of the two jagged value streams is cut into tiles of
// E consecutive elements; a CTA owns every (column, bag) segment whose FIRST
// element lies in its tile, so each pooled output row has exactly one writer
// (RecIS §3.2 Algorithm 1, forward: no atomics).
//
// A CTA walks its segments in chunks that stay inside one column (one table,
// one dim, one transform) and hold at most kChunkBags bags and kChunkElems
// values of short bags:
//   A. every thread transforms values of the chunk (coalesced 8-byte loads,
//      SplitMix64 + invariant-divisor modulo, or a binary search over the
//      boundaries), applies the range guard and writes the row to shared
//      memory -- one memory round trip for the whole chunk;
//   B. the chunk's values are split into equal ranges, one per lane group of
//      dim/4 lanes (so every group runs the same trip count); a group gathers
//      its rows with 16-byte loads four deep and sums them per bag; a bag that
//      spans ranges leaves head/tail partials in shared memory which the
//      group holding its first value adds up in range order (deterministic);
//   C. bags longer than kLongBag (or padded bags with pad_len > kLongBag) are
//      pooled / copied by all eight warps together.
// Empty bags and bags whose values were all dropped get the default vector.
#include <algorithm>

#include "plan.cuh"

namespace emb {

constexpr int kChunkBags = 256;    // == kFwdThreads: one bag per thread in setup
constexpr int kChunkElems = 4096;
constexpr int kU = 4;              // row loads in flight per lane (halved when a lane holds two float4)

struct FwdArgs {
  const ColMeta* meta;
  const int32_t* stream_cols;
  const int64_t* ids;
  const float* fvals;
  const int32_t* offs[2];
  int64_t n[2];
  int32_t ncols[2];
  int32_t col_base[2];
  int32_t tiles[2];
  int32_t tile_elems;
  int32_t batch;
  DivMagic32 bdiv;
  int64_t ldo;
  float* out;
  float* seq_out;
  int64_t* rows_dbg;
  int64_t rec_base[2];     // record index of element 0 of each stream
  uint32_t* keys;          // training: global row per contribution (sentinel if none)
  uint32_t* vals;          // training: gradient source per contribution
  float* inv_n;            // training: 1/n_valid per mean bag
  uint32_t key_sentinel;
  uint32_t* status;
};

struct FwdSmem {
  int32_t rows[kChunkElems];
  uint8_t bag[kChunkElems];
  int32_t pos[kChunkBags + 1];     // first slot of each bag's values in rows[]
  int32_t lo[kChunkBags];          // first stream element of each bag
  int32_t hi[kChunkBags];          // one past its last stream element; -1: long bag
  int32_t len[kChunkBags];         // values of the bag held in rows[]
  int32_t longs[kChunkBags];       // bags left for phase C
  int32_t tailbag[kFwdThreads];    // per lane group: bag whose tail partial it holds
  int32_t nvp[kFwdThreads][2];     // per lane group: valid counts of head/tail partials
  float4 part[2][kFwdWarps * 64];  // per lane group: head / tail partial sums
  int32_t warp_sum[kFwdWarps];
  int32_t seg[2];
  int32_t nlong;
  ColMeta cm;                      // metadata of the chunk's column
};

__device__ __forceinline__ float4 f4zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }

__device__ __forceinline__ void f4add(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ int64_t clamp_off(int32_t o, int64_t n, bool& bad) {
  int64_t v = o;
  if (v < 0) { v = 0; bad = true; }
  if (v > n) { v = n; bad = true; }
  return v;
}

// First index s in [0, S) with clamp(offs[s]) >= e, or S.  32-ary search by
// one warp: each round probes the ends of 32 equal chunks.
__device__ int warp_lower_bound(const int32_t* offs, int S, int64_t e, int64_t n) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
  int lo = 0, hi = S;
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) >> 5;
    const int p = lo + (lane + 1) * step - 1;
    const bool less = (p < hi) && (clamp_off(__ldg(offs + p), n, bad) < e);
    const int k = __popc(__ballot_sync(kFull, less));
    const int nlo = min(lo + k * step, hi);
    hi = min(hi, nlo + step - 1);
    lo = nlo;
  }
  const int p = lo + lane;
  const bool less = (p < hi) && (clamp_off(__ldg(offs + p), n, bad) < e);
  return lo + __popc(__ballot_sync(kFull, less));
}

// Transformed, guarded row of element t of a column; -1 when dropped.
__device__ __forceinline__ int32_t col_row(const ColMeta& m, const int64_t* ids, const float* fvals,
                                           int64_t t) {
  if (m.transform == EMB_T_BUCKETIZE) {
    const float x = __ldcs(fvals + t);
    int lo = 0, hi = m.nb;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(m.bnd + mid) <= x) lo = mid + 1; else hi = mid;
    }
    return lo;
  }
  const int64_t v = __ldcs(ids + t);
  if (m.transform == EMB_T_HASH_MOD) return (int32_t)mod_magic(splitmix64((uint64_t)v), m.mod);
  return (v >= 0 && v < m.num_rows) ? (int32_t)v : -1;
}

__device__ __forceinline__ void record(const FwdArgs& a, int st, int64_t t, int32_t row,
                                       const ColMeta& m, uint32_t gsrc) {
  const int64_t r = a.rec_base[st] + t;
  if (a.rows_dbg) a.rows_dbg[r] = row;
  if (a.keys) {
    a.keys[r] = row >= 0 ? m.table_base + (uint32_t)row : a.key_sentinel;
    a.vals[r] = gsrc;
  }
}

// Final value of float4 slot f4 of a pooled bag: mean / sum / default.
__device__ __forceinline__ float4 finish(const ColMeta& m, float4 s, int nv, int f4) {
  if (nv == 0) return m.dflt ? ldg4(m.dflt + f4 * 4) : f4zero();
  if (m.pooling == EMB_POOL_MEAN) {
    const float fn = (float)nv;
    s.x = __fdiv_rn(s.x, fn);
    s.y = __fdiv_rn(s.y, fn);
    s.z = __fdiv_rn(s.z, fn);
    s.w = __fdiv_rn(s.w, fn);
  }
  return s;
}

__device__ __forceinline__ int lanes_log2(int dim4) {
  const int g = dim4 > 32 ? 32 : dim4;
  int l = 0;
  while ((1 << l) < g) ++l;
  return l;
}

// Exclusive block scan of one int per thread (kFwdThreads threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sum[warp] = x;
  __syncthreads();
  int base = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kFwdWarps; ++w) {
    const int s = warp_sum[w];
    if (w < warp) base += s;
    total += s;
  }
  __syncthreads();
  return base + x - v;
}

// ---------------------------------------------------------------------------
// phase B: pooled bags of a chunk, one equal range of values per lane group
// ---------------------------------------------------------------------------
template <int V>
__device__ void pool_chunk(const FwdArgs& a, FwdSmem& sm, const ColMeta& m, int ns, int T, int b0,
                           int glog) {
  constexpr int U = kU / V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = 32 >> glog;
  const int grp = lane >> glog, sub = lane & ((1 << glog) - 1);
  const int q = warp * G + grp;                 // lane group id
  const int NG = kFwdWarps * G;
  const int R = (T + NG - 1) / NG;
  const int k0 = min(q * R, T), k1 = min(k0 + R, T);
  const float* E = m.weight;

  float4 acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = f4zero();
  int nv = 0;
  int curb = k0 < k1 ? (int)sm.bag[k0] : -1;
  bool head = k0 > 0 && k0 < k1 && (int)sm.bag[k0 - 1] == curb;
  if (sub == 0) sm.tailbag[q] = -1;

  auto write_out = [&](int b, const float4 (&s)[V], int cnt) {
    const int bag = b0 + b;
    float* y = a.out + (int64_t)bag * a.ldo + m.out_col;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      if (f4 < m.dim4) *reinterpret_cast<float4*>(y + f4 * 4) = finish(m, s[v], cnt, f4);
    }
    if (a.inv_n && sub == 0 && m.pooling == EMB_POOL_MEAN)
      a.inv_n[(uint32_t)m.col * (uint32_t)a.batch + (uint32_t)bag] = cnt > 0 ? 1.0f / (float)cnt : 0.0f;
  };
  auto flush = [&](bool tail) {
    if (!head && !tail) {
      write_out(curb, acc, nv);
    } else {
      const int side = head ? 0 : 1;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < m.dim4) sm.part[side][q * m.dim4 + f4] = acc[v];
      }
      if (sub == 0) {
        sm.nvp[q][side] = nv;
        if (!head) sm.tailbag[q] = curb;
      }
    }
  };

  for (int j = 0; j < R; j += U) {
    float4 vals[U][V];
    int bg[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = k0 + j + u;
      const bool in = k < k1;
      const int r = in ? sm.rows[k] : -1;
      bg[u] = in ? (int)sm.bag[k] : -1;
      ok[u] = in && r >= 0;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        vals[u][v] = (ok[u] && f4 < m.dim4) ? ldg4(E + (int64_t)r * m.dim + f4 * 4) : f4zero();
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (bg[u] < 0) continue;
      if (bg[u] != curb) {
        flush(false);
        curb = bg[u];
        head = false;
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = f4zero();
        nv = 0;
      }
#pragma unroll
      for (int v = 0; v < V; ++v) f4add(acc[v], vals[u][v]);
      nv += ok[u];
    }
  }
  if (k0 < k1) flush(k1 < T && (int)sm.bag[k1] == curb);
  __syncthreads();

  // the group holding a cut bag's first value adds the partials in order
  const int tb = sm.tailbag[q];
  if (tb >= 0) {
    float4 s[V];
    int cnt = sm.nvp[q][1];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      s[v] = f4 < m.dim4 ? sm.part[1][q * m.dim4 + f4] : f4zero();
    }
    const int last = (sm.pos[tb] + sm.len[tb] - 1) / R;
    for (int q2 = q + 1; q2 <= last; ++q2) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < m.dim4) f4add(s[v], sm.part[0][q2 * m.dim4 + f4]);
      }
      cnt += sm.nvp[q2][0];
    }
    write_out(tb, s, cnt);
  }
  // empty bags: default vector
  for (int i = threadIdx.x; i < ns; i += kFwdThreads) {
    if (sm.len[i] != 0 || sm.hi[i] < 0) continue;
    float* y = a.out + (int64_t)(b0 + i) * a.ldo + m.out_col;
    for (int f4 = 0; f4 < m.dim4; ++f4) *reinterpret_cast<float4*>(y + f4 * 4) = finish(m, f4zero(), 0, f4);
    if (a.inv_n && m.pooling == EMB_POOL_MEAN)
      a.inv_n[(uint32_t)m.col * (uint32_t)a.batch + (uint32_t)(b0 + i)] = 0.0f;
  }
}

// phase B for padded columns: ns bags x pad_len output rows, flat over groups.
template <int V>
__device__ void pad_chunk(const FwdArgs& a, FwdSmem& sm, const ColMeta& m, int ns, int b0, int glog) {
  constexpr int U = kU / V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = 32 >> glog;
  const int grp = lane >> glog, sub = lane & ((1 << glog) - 1);
  const int q = warp * G + grp;
  const int NG = kFwdWarps * G;
  const int P = m.pad_len;
  const int total = ns * P;
  const float* E = m.weight;
  for (int base = 0; base < total; base += NG * U) {
    float4 vals[U][V];
    int o[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      o[u] = base + u * NG + q;
      int r = -1;
      if (o[u] < total) {
        const int i = o[u] / P, p = o[u] - i * P;
        if (sm.hi[i] >= 0 && p < sm.len[i]) r = sm.rows[sm.pos[i] + p];
      }
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        vals[u][v] = (r >= 0 && f4 < m.dim4) ? ldg4(E + (int64_t)r * m.dim + f4 * 4) : f4zero();
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (o[u] >= total) continue;
      const int i = o[u] / P, p = o[u] - i * P;
      if (sm.hi[i] < 0) continue;   // long bag: phase C writes it
      float* dst = a.seq_out + m.seq_unit * a.batch + ((int64_t)(b0 + i) * P + p) * m.dim;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < m.dim4) *reinterpret_cast<float4*>(dst + f4 * 4) = vals[u][v];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// phase C: one long bag, all warps; values transformed on the fly
// ---------------------------------------------------------------------------
template <int V>
__device__ void cta_bag(const FwdArgs& a, FwdSmem& sm, int st, const ColMeta& m, int32_t b, int64_t lo,
                        int64_t hi, int glog) {
  constexpr int U = kU / V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = 32 >> glog;
  const int grp = lane >> glog, sub = lane & ((1 << glog) - 1);
  const float* E = m.weight;
  if (m.pooling == EMB_POOL_NONE_PADDED) {
    const int P = m.pad_len;
    const int64_t len = hi - lo;
    const int64_t seq0 = m.seq_unit * a.batch + (int64_t)b * P * m.dim;
    float* dst = a.seq_out + seq0;
    for (int64_t p0 = (int64_t)warp * 32; p0 < P; p0 += (int64_t)kFwdWarps * 32) {
      const int cnt = (int)(P - p0 < 32 ? P - p0 : 32);
      int32_t row = -1;
      const int64_t p = p0 + lane;
      if (lane < cnt && p < len) {
        row = col_row(m, a.ids, a.fvals, lo + p);
        record(a, st, lo + p, row, m, kPadBit | (uint32_t)((seq0 + p * m.dim) >> 2));
      }
      for (int k = 0; k < cnt; k += U * G) {
        float4 v[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = k + u * G + grp;
          const int r = __shfl_sync(kFull, row, j & 31);
          const bool ok = (j < cnt) && (r >= 0);
#pragma unroll
          for (int q = 0; q < V; ++q) {
            const int f4 = sub + q * 32;
            v[u][q] = (ok && f4 < m.dim4) ? ldg4(E + (int64_t)r * m.dim + f4 * 4) : f4zero();
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = k + u * G + grp;
#pragma unroll
          for (int q = 0; q < V; ++q) {
            const int f4 = sub + q * 32;
            if (j < cnt && f4 < m.dim4) *reinterpret_cast<float4*>(dst + (p0 + j) * m.dim + f4 * 4) = v[u][q];
          }
        }
      }
    }
    if (a.rows_dbg || a.keys)
      for (int64_t t = lo + P + threadIdx.x; t < hi; t += kFwdThreads) {
        const int64_t r = a.rec_base[st] + t;
        if (a.rows_dbg) a.rows_dbg[r] = col_row(m, a.ids, a.fvals, t);
        if (a.keys) {
          a.keys[r] = a.key_sentinel;
          a.vals[r] = 0u;
        }
      }
    return;
  }
  const uint32_t gsrc = (uint32_t)m.col * (uint32_t)a.batch + (uint32_t)b;
  float4 acc[V];
#pragma unroll
  for (int q = 0; q < V; ++q) acc[q] = f4zero();
  int nv = 0;
  for (int64_t base = lo + (int64_t)warp * 32; base < hi; base += (int64_t)kFwdWarps * 32) {
    const int cnt = (int)(hi - base < 32 ? hi - base : 32);
    int32_t row = -1;
    if (lane < cnt) {
      row = col_row(m, a.ids, a.fvals, base + lane);
      record(a, st, base + lane, row, m, gsrc);
    }
    nv += __popc(__ballot_sync(kFull, row >= 0));
    for (int k = 0; k < cnt; k += U * G) {
      float4 v[U][V];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = k + u * G + grp;
        const int r = __shfl_sync(kFull, row, j & 31);
        const bool ok = (j < cnt) && (r >= 0);
#pragma unroll
        for (int q = 0; q < V; ++q) {
          const int f4 = sub + q * 32;
          v[u][q] = (ok && f4 < m.dim4) ? ldg4(E + (int64_t)r * m.dim + f4 * 4) : f4zero();
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int q = 0; q < V; ++q) f4add(acc[q], v[u][q]);
    }
  }
#pragma unroll
  for (int q = 0; q < V; ++q)
    for (int off = 1 << glog; off < 32; off <<= 1) {
      acc[q].x += __shfl_xor_sync(kFull, acc[q].x, off);
      acc[q].y += __shfl_xor_sync(kFull, acc[q].y, off);
      acc[q].z += __shfl_xor_sync(kFull, acc[q].z, off);
      acc[q].w += __shfl_xor_sync(kFull, acc[q].w, off);
    }
  float4* red = sm.part[0];   // [kFwdWarps][64]
  if (grp == 0) {
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const int f4 = sub + q * 32;
      if (f4 < m.dim4) red[warp * 64 + f4] = acc[q];
    }
  }
  if (lane == 0) sm.nvp[warp][0] = nv;
  __syncthreads();
  int tot = 0;
#pragma unroll
  for (int w = 0; w < kFwdWarps; ++w) tot += sm.nvp[w][0];
  for (int f4 = threadIdx.x; f4 < m.dim4; f4 += kFwdThreads) {
    float4 s = red[f4];
#pragma unroll
    for (int w = 1; w < kFwdWarps; ++w) f4add(s, red[w * 64 + f4]);
    *reinterpret_cast<float4*>(a.out + (int64_t)b * a.ldo + m.out_col + f4 * 4) = finish(m, s, tot, f4);
  }
  if (a.inv_n && threadIdx.x == 0 && m.pooling == EMB_POOL_MEAN)
    a.inv_n[gsrc] = tot > 0 ? 1.0f / (float)tot : 0.0f;
  __syncthreads();
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kFwdThreads, 4) k_forward(const FwdArgs a) {
  __shared__ FwdSmem sm;
  int tile = blockIdx.x, st = 0;
  if (tile >= a.tiles[0]) {
    st = 1;
    tile -= a.tiles[0];
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = a.ncols[st] * a.batch;
  const int64_t e0 = (int64_t)tile * a.tile_elems;
  const bool last = tile == a.tiles[st] - 1;
  const int32_t* offs = a.offs[st];
  const int64_t n = a.n[st];
  if (warp == 0) {
    const int r = warp_lower_bound(offs, S, e0, n);
    if (lane == 0) sm.seg[0] = r;
  } else if (warp == 1) {
    const int r = last ? S : warp_lower_bound(offs, S, e0 + a.tile_elems, n);
    if (lane == 0) sm.seg[1] = r;
  }
  __syncthreads();
  const int s_hi = sm.seg[1];
  int cur = sm.seg[0];
  while (cur < s_hi) {
    // ---- chunk setup: one bag per thread, all inside column cl0 ----
    const int cl0 = (int)div_magic32((uint32_t)cur, a.bdiv);
    const int b0 = cur - cl0 * a.batch;
    const int navail = min(kChunkBags, min(s_hi, (cl0 + 1) * a.batch) - cur);
    static_assert(sizeof(ColMeta) % 4 == 0 && sizeof(ColMeta) / 4 <= kFwdThreads, "metadata copy");
    if (tid < (int)(sizeof(ColMeta) / 4))
      reinterpret_cast<int32_t*>(&sm.cm)[tid] =
          __ldg(reinterpret_cast<const int32_t*>(a.meta + __ldg(a.stream_cols + a.col_base[st] + cl0)) + tid);
    __syncthreads();
    const ColMeta& m = sm.cm;
    const bool padded = m.pooling == EMB_POOL_NONE_PADDED;
    int64_t lo = 0, hi = 0;
    int used = 0;
    bool is_long = false;
    if (tid < navail) {
      bool bad = false;
      lo = clamp_off(__ldg(offs + cur + tid), n, bad);
      hi = clamp_off(__ldg(offs + cur + tid + 1), n, bad);
      if (hi < lo) { hi = lo; bad = true; }
      if (bad) latch(a.status, EMB_ERR_BAD_INDEX);
      const int64_t len = hi - lo;
      is_long = (padded ? (int64_t)m.pad_len : len) > kLongBag;
      used = is_long ? 0 : (int)(padded ? (len < m.pad_len ? len : (int64_t)m.pad_len) : len);
    }
    int total = 0;
    const int pos = block_exclusive_scan(used, sm.warp_sum, total);
    const bool fits = tid < navail && pos + used <= kChunkElems;
    const int ns = __syncthreads_count(fits);
    if (tid == 0) sm.nlong = 0;
    __syncthreads();
    if (tid < ns) {
      sm.pos[tid] = pos;
      sm.lo[tid] = (int32_t)lo;
      sm.len[tid] = used;
      sm.hi[tid] = is_long ? -1 : (int32_t)hi;
      if (is_long) sm.longs[atomicAdd(&sm.nlong, 1)] = tid;
      if (tid == ns - 1) sm.pos[ns] = pos + used;
      for (int k = pos; k < pos + used; ++k) sm.bag[k] = (uint8_t)tid;
    }
    __syncthreads();
    const int T = sm.pos[ns];

    // ---- phase A: transform every value of the chunk's short bags ----
    for (int k = tid; k < T; k += kFwdThreads) {
      const int i = sm.bag[k];
      const int64_t t = (int64_t)sm.lo[i] + (k - sm.pos[i]);
      const int32_t row = col_row(m, a.ids, a.fvals, t);
      sm.rows[k] = row;
      if (a.rows_dbg || a.keys) {
        uint32_t gsrc;
        if (padded)
          gsrc = kPadBit | (uint32_t)((m.seq_unit * a.batch +
                                       ((int64_t)(b0 + i) * m.pad_len + (k - sm.pos[i])) * m.dim) >> 2);
        else
          gsrc = (uint32_t)m.col * (uint32_t)a.batch + (uint32_t)(b0 + i);
        record(a, st, t, row, m, gsrc);
      }
    }
    // values past pad_len of short padded bags: no output, no gradient
    if (padded && (a.rows_dbg || a.keys) && tid < ns && sm.hi[tid] >= 0)
      for (int64_t t = (int64_t)sm.lo[tid] + m.pad_len; t < sm.hi[tid]; ++t) {
        const int64_t r = a.rec_base[st] + t;
        if (a.rows_dbg) a.rows_dbg[r] = col_row(m, a.ids, a.fvals, t);
        if (a.keys) {
          a.keys[r] = a.key_sentinel;
          a.vals[r] = 0u;
        }
      }
    __syncthreads();

    // ---- phase B: pool / copy ----
    const int glog = lanes_log2(m.dim4);
    if (padded) {
      if (m.dim4 > 32) pad_chunk<2>(a, sm, m, ns, b0, glog);
      else pad_chunk<1>(a, sm, m, ns, b0, glog);
    } else {
      if (m.dim4 > 32) pool_chunk<2>(a, sm, m, ns, T, b0, glog);
      else pool_chunk<1>(a, sm, m, ns, T, b0, glog);
    }
    __syncthreads();

    // ---- phase C: long bags of the chunk ----
    const int nlong = sm.nlong;
    for (int j = 0; j < nlong; ++j) {
      const int i = sm.longs[j];
      bool bad = false;
      const int64_t blo = clamp_off(__ldg(offs + cur + i), n, bad);
      int64_t bhi = clamp_off(__ldg(offs + cur + i + 1), n, bad);
      if (bhi < blo) bhi = blo;
      if (m.dim4 > 32) cta_bag<2>(a, sm, st, m, b0 + i, blo, bhi, glog);
      else cta_bag<1>(a, sm, st, m, b0 + i, blo, bhi, glog);
    }
    __syncthreads();
    cur += ns;
  }
}

int forward_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_forward, kFwdThreads, 0) != cudaSuccess) {
    cudaGetLastError();
    n = 4;
  }
  return n > 0 ? n : 1;
}

emb_status launch_forward(emb_plan_s* p, int32_t batch, const int64_t* ids, const int32_t* id_offsets,
                          int64_t n_ids, const float* fvals, const int32_t* f_offsets, int64_t n_fvals,
                          float* out, float* seq_out, int64_t* rows_dbg, cudaStream_t stream) {
  if (batch == 0) return EMB_OK;
  FwdArgs a{};
  a.meta = p->meta_d;
  a.stream_cols = p->stream_cols_d;
  a.ids = ids;
  a.fvals = fvals;
  a.offs[0] = id_offsets;
  a.offs[1] = f_offsets;
  a.n[0] = n_ids;
  a.n[1] = n_fvals;
  a.ncols[0] = p->n_stream_cols[0];
  a.ncols[1] = p->n_stream_cols[1];
  a.col_base[0] = 0;
  a.col_base[1] = p->n_stream_cols[0];
  a.batch = batch;
  a.bdiv = make_div_magic32((uint32_t)batch);
  a.ldo = p->out_width;
  a.out = out;
  a.seq_out = seq_out;
  a.rows_dbg = rows_dbg;
  a.rec_base[0] = 0;
  a.rec_base[1] = n_ids;
  if (p->training) {
    a.keys = p->ws.keys[0];
    a.vals = p->ws.vals[0];
    a.inv_n = p->ws.inv_n;
  }
  a.key_sentinel = p->key_total;
  a.status = p->status_d;
  const int64_t total = n_ids + n_fvals;
  const int64_t resident = (int64_t)p->sm_count * p->fwd_ctas_per_sm;
  const int64_t want = total / std::max<int64_t>(1, 8 * resident);
  int64_t E = 512;
  while (E < want && E < kMaxTileElems) E <<= 1;
  a.tile_elems = (int32_t)E;
  a.tiles[0] = a.ncols[0] > 0 ? (int32_t)(n_ids / E + 1) : 0;
  a.tiles[1] = a.ncols[1] > 0 ? (int32_t)(n_fvals / E + 1) : 0;
  const int grid = a.tiles[0] + a.tiles[1];
  if (grid == 0) return EMB_OK;
  k_forward<<<grid, kFwdThreads, 0, stream>>>(a);
  return cuda_status(cudaGetLastError());
}

}  // namespace emb
