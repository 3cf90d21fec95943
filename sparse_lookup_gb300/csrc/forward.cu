// forward.cu -- K-F: the fused multi-column forward (transform, safety check,
// row gather, pooling / padded copy, default fill) in ONE launch.
//
// Work decomposition (element-count tiling, RecIS §3.1 "Thread mapping for
// skewed inputs"): each of the two jagged value streams is cut into tiles of
// E consecutive elements; a CTA owns every (column, bag) segment whose FIRST
// element lies in its tile, so each pooled output row has exactly one writer
// (RecIS §3.2 Algorithm 1, forward: no atomics).  Inside a CTA, warps pull
// short bags from a shared-memory cursor; bags longer than kLongBag elements
// (or padded bags with pad_len > kLongBag) are pooled by all eight warps
// together, each warp taking every eighth 32-element chunk, with a fixed-order
// shared-memory reduction at the end.
//
// Per 32-element chunk a warp loads the values coalesced (one per lane),
// transforms them in parallel (SplitMix64 + invariant-divisor modulo, or a
// binary search over the boundaries), applies the range guard, then gathers
// rows with 16-byte loads: a row of dim floats is read by dim/4 lanes and
// 32/(dim/4) rows are in flight per warp instruction, four instructions deep.
#include <algorithm>

#include "plan.cuh"

namespace emb {

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

// Sum of the rows of chunks chunk0, chunk0 + step, ... of [lo, hi) into the
// caller's per-lane accumulators (lane group `grp`, float4 slot `sub`).
template <int V>
__device__ __forceinline__ void gather_pool(const FwdArgs& a, const ColMeta& m, int st, int64_t lo,
                                            int64_t hi, int chunk0, int step, int glog,
                                            uint32_t gsrc, float4 (&acc)[V], int& nv) {
  const int lane = threadIdx.x & 31;
  const int G = 32 >> glog;
  const int grp = lane >> glog;
  const int sub = lane & ((1 << glog) - 1);
  const float* E = m.weight;
  for (int64_t base = lo + (int64_t)chunk0 * 32; base < hi; base += (int64_t)step * 32) {
    const int cnt = (int)(hi - base < 32 ? hi - base : 32);
    int32_t row = -1;
    if (lane < cnt) {
      row = col_row(m, a.ids, a.fvals, base + lane);
      record(a, st, base + lane, row, m, gsrc);
    }
    nv += __popc(__ballot_sync(kFull, row >= 0));
    for (int k = 0; k < cnt; k += 4 * G) {
      float4 v[4][V];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
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
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int q = 0; q < V; ++q) f4add(acc[q], v[u][q]);
    }
  }
}

template <int V>
__device__ __forceinline__ void group_reduce(float4 (&acc)[V], int glog) {
#pragma unroll
  for (int q = 0; q < V; ++q)
    for (int off = 1 << glog; off < 32; off <<= 1) {
      acc[q].x += __shfl_xor_sync(kFull, acc[q].x, off);
      acc[q].y += __shfl_xor_sync(kFull, acc[q].y, off);
      acc[q].z += __shfl_xor_sync(kFull, acc[q].z, off);
      acc[q].w += __shfl_xor_sync(kFull, acc[q].w, off);
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

// Padded (unpooled) copy of positions chunk0, chunk0 + step, ... of a bag.
template <int V>
__device__ __forceinline__ void padded_copy(const FwdArgs& a, const ColMeta& m, int st, int64_t lo,
                                            int64_t hi, int32_t b, int chunk0, int step, int glog) {
  const int lane = threadIdx.x & 31;
  const int G = 32 >> glog;
  const int grp = lane >> glog;
  const int sub = lane & ((1 << glog) - 1);
  const int P = m.pad_len;
  const int64_t len = hi - lo;
  const int64_t seq0 = m.seq_unit * a.batch + (int64_t)b * P * m.dim;
  float* dst = a.seq_out + seq0;
  const float* E = m.weight;
  for (int64_t p0 = (int64_t)chunk0 * 32; p0 < P; p0 += (int64_t)step * 32) {
    const int cnt = (int)(P - p0 < 32 ? P - p0 : 32);
    int32_t row = -1;
    const int64_t p = p0 + lane;
    if (lane < cnt && p < len) {
      row = col_row(m, a.ids, a.fvals, lo + p);
      record(a, st, lo + p, row, m, kPadBit | (uint32_t)((seq0 + p * m.dim) >> 2));
    }
    for (int k = 0; k < cnt; k += 4 * G) {
      float4 v[4][V];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
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
      for (int u = 0; u < 4; ++u) {
        const int j = k + u * G + grp;
#pragma unroll
        for (int q = 0; q < V; ++q) {
          const int f4 = sub + q * 32;
          if (j < cnt && f4 < m.dim4)
            *reinterpret_cast<float4*>(dst + (p0 + j) * m.dim + f4 * 4) = v[u][q];
        }
      }
    }
  }
  // values past pad_len: no output, no gradient
  if (a.rows_dbg || a.keys)
    for (int64_t t = lo + P + (int64_t)chunk0 * 32 + lane; t < hi; t += (int64_t)step * 32) {
      const int64_t r = a.rec_base[st] + t;
      if (a.rows_dbg) a.rows_dbg[r] = col_row(m, a.ids, a.fvals, t);
      if (a.keys) {
        a.keys[r] = a.key_sentinel;
        a.vals[r] = 0u;
      }
    }
}

struct SegInfo {
  int32_t c;   // plan column
  int32_t b;   // bag
  int64_t lo, hi;
};

__device__ __forceinline__ SegInfo seg_info(const FwdArgs& a, int st, int s) {
  SegInfo si;
  const uint32_t cl = div_magic32((uint32_t)s, a.bdiv);
  si.b = s - (int32_t)cl * a.batch;
  si.c = __ldg(a.stream_cols + a.col_base[st] + cl);
  bool bad = false;
  const int32_t* offs = a.offs[st];
  si.lo = clamp_off(__ldg(offs + s), a.n[st], bad);
  si.hi = clamp_off(__ldg(offs + s + 1), a.n[st], bad);
  if (si.hi < si.lo) { si.hi = si.lo; bad = true; }
  if (bad && (threadIdx.x & 31) == 0) latch(a.status, EMB_ERR_BAD_INDEX);
  return si;
}

// One warp pools (or copies) one whole bag.
template <int V>
__device__ void warp_bag(const FwdArgs& a, int st, const SegInfo& si, const ColMeta& m, int glog) {
  const int lane = threadIdx.x & 31;
  if (m.pooling == EMB_POOL_NONE_PADDED) {
    padded_copy<V>(a, m, st, si.lo, si.hi, si.b, 0, 1, glog);
    return;
  }
  const uint32_t gsrc = (uint32_t)si.c * (uint32_t)a.batch + (uint32_t)si.b;
  float4 acc[V];
#pragma unroll
  for (int q = 0; q < V; ++q) acc[q] = f4zero();
  int nv = 0;
  gather_pool<V>(a, m, st, si.lo, si.hi, 0, 1, glog, gsrc, acc, nv);
  group_reduce<V>(acc, glog);
  if ((lane >> glog) == 0) {
    float* y = a.out + (int64_t)si.b * a.ldo + m.out_col;
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const int f4 = (lane & ((1 << glog) - 1)) + q * 32;
      if (f4 < m.dim4) *reinterpret_cast<float4*>(y + f4 * 4) = finish(m, acc[q], nv, f4);
    }
  }
  if (a.inv_n && lane == 0 && m.pooling == EMB_POOL_MEAN) a.inv_n[gsrc] = nv > 0 ? 1.0f / (float)nv : 0.0f;
}

// All warps of the CTA pool (or copy) one long bag.
template <int V>
__device__ void cta_bag(const FwdArgs& a, int st, const SegInfo& si, const ColMeta& m, int glog,
                        float4 (*s_red)[64], int* s_nv) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (m.pooling == EMB_POOL_NONE_PADDED) {
    padded_copy<V>(a, m, st, si.lo, si.hi, si.b, warp, kFwdWarps, glog);
    return;
  }
  const uint32_t gsrc = (uint32_t)si.c * (uint32_t)a.batch + (uint32_t)si.b;
  float4 acc[V];
#pragma unroll
  for (int q = 0; q < V; ++q) acc[q] = f4zero();
  int nv = 0;
  gather_pool<V>(a, m, st, si.lo, si.hi, warp, kFwdWarps, glog, gsrc, acc, nv);
  group_reduce<V>(acc, glog);
  if ((lane >> glog) == 0) {
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const int f4 = (lane & ((1 << glog) - 1)) + q * 32;
      if (f4 < m.dim4) s_red[warp][f4] = acc[q];
    }
  }
  if (lane == 0) s_nv[warp] = nv;
  __syncthreads();
  int tot = 0;
#pragma unroll
  for (int w = 0; w < kFwdWarps; ++w) tot += s_nv[w];
  for (int f4 = threadIdx.x; f4 < m.dim4; f4 += blockDim.x) {
    float4 s = s_red[0][f4];
#pragma unroll
    for (int w = 1; w < kFwdWarps; ++w) f4add(s, s_red[w][f4]);
    *reinterpret_cast<float4*>(a.out + (int64_t)si.b * a.ldo + m.out_col + f4 * 4) = finish(m, s, tot, f4);
  }
  if (a.inv_n && threadIdx.x == 0 && m.pooling == EMB_POOL_MEAN)
    a.inv_n[gsrc] = tot > 0 ? 1.0f / (float)tot : 0.0f;
  __syncthreads();
}

__device__ __forceinline__ int lanes_log2(int dim4) {
  // lanes per row: next power of two >= min(dim4, 32)
  int g = dim4 > 32 ? 32 : dim4;
  int l = 0;
  while ((1 << l) < g) ++l;
  return l;
}

__global__ void __launch_bounds__(kFwdThreads) k_forward(const FwdArgs a) {
  __shared__ int s_seg[2];
  __shared__ int s_cursor;
  __shared__ int s_nlong;
  __shared__ int s_long[kMaxLongPerTile];
  __shared__ float4 s_red[kFwdWarps][64];
  __shared__ int s_nv[kFwdWarps];

  int tile = blockIdx.x, st = 0;
  if (tile >= a.tiles[0]) {
    st = 1;
    tile -= a.tiles[0];
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = a.ncols[st] * a.batch;
  const int64_t e0 = (int64_t)tile * a.tile_elems;
  const bool last = tile == a.tiles[st] - 1;
  if (warp == 0) {
    const int r = warp_lower_bound(a.offs[st], S, e0, a.n[st]);
    if (lane == 0) s_seg[0] = r;
  } else if (warp == 1) {
    const int r = last ? S : warp_lower_bound(a.offs[st], S, e0 + a.tile_elems, a.n[st]);
    if (lane == 0) s_seg[1] = r;
  }
  if (threadIdx.x == 0) {
    s_cursor = 0;
    s_nlong = 0;
  }
  __syncthreads();
  const int s_lo = s_seg[0], s_hi = s_seg[1];

  // Phase 1: short bags, one warp each, pulled from a shared cursor.
  for (;;) {
    int k = 0;
    if (lane == 0) k = atomicAdd(&s_cursor, 1);
    k = __shfl_sync(kFull, k, 0);
    const int s = s_lo + k;
    if (s >= s_hi) break;
    const SegInfo si = seg_info(a, st, s);
    const ColMeta m = a.meta[si.c];
    const int work = m.pooling == EMB_POOL_NONE_PADDED ? m.pad_len : (int)(si.hi - si.lo);
    if (work > kLongBag) {
      int idx = 0;
      if (lane == 0) idx = atomicAdd(&s_nlong, 1);
      idx = __shfl_sync(kFull, idx, 0);
      if (idx < kMaxLongPerTile) {
        if (lane == 0) s_long[idx] = s;
        continue;
      }
    }
    const int glog = lanes_log2(m.dim4);
    if (m.dim4 > 32) warp_bag<2>(a, st, si, m, glog);
    else warp_bag<1>(a, st, si, m, glog);
  }
  __syncthreads();

  // Phase 2: long bags, all warps together, one after the other.
  const int nlong = min(s_nlong, kMaxLongPerTile);
  for (int i = 0; i < nlong; ++i) {
    const SegInfo si = seg_info(a, st, s_long[i]);
    const ColMeta m = a.meta[si.c];
    const int glog = lanes_log2(m.dim4);
    if (m.dim4 > 32) cta_bag<2>(a, st, si, m, glog, s_red, s_nv);
    else cta_bag<1>(a, st, si, m, glog, s_red, s_nv);
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
  int64_t want = total / std::max<int64_t>(1, 4 * resident);
  int64_t E = 256;
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
