// forward.cu -- K-F: the fused multi-column forward (transform, safety check,
// row gather, pooling / padded copy, default fill) in ONE launch.
//
// Work decomposition (element-count tiling, RecIS §3.1 "Thread mapping for
// skewed inputs"): each of the two jagged value streams is cut into tiles of
// E consecutive elements and every WARP owns one tile: the (column, bag)
// segments whose FIRST element lies in the tile.  A stream of short bags is
// cut into runs of whole 32-bag chunks of about E values instead, which
// need no search for their ends.  Each pooled output row therefore has
// exactly one writer (RecIS §3.2 Algorithm 1, forward: no atomics), and
// warps never wait on each other -- there is no CTA barrier, so a warp
// stalled on memory never holds up another.
//
// A warp walks its segments in chunks that stay inside one column (one table,
// one dim, one transform) and hold at most 32 bags and kWarpElems values of
// short bags:
//   setup  one lane per bag loads the bag's CSR range; a warp scan places the
//          bags' values back to back in shared memory;
//   A.     lanes transform the chunk's values (coalesced 8-byte loads,
//          SplitMix64 + invariant-divisor modulo, or a binary search over the
//          boundaries), apply the range guard and park the rows in shared
//          memory;
//   B.     lane groups of dim/4 lanes take equal ranges of those values (the
//          same trip count for every group), gather rows with 16-byte loads
//          four deep and sum them per bag; a bag that spans ranges leaves
//          head/tail partials which the group holding its first value adds up
//          in range order (deterministic);
//   C.     pooled bags longer than kLongBag are pooled by the whole warp, 32
//          values per step.
// Padded columns with pad_len > kLongBag are copied in pieces of about
// kPadPiece positions, tiles of their own after the value tiles.
// Empty bags and bags whose values were all dropped get the default vector.
#include <algorithm>

#include <cuda_fp16.h>

#include <type_traits>

#include "plan.cuh"

namespace emb {

constexpr int kWarpElems = 512;    // values of short bags one warp chunk holds
constexpr int kU = 4;              // row loads in flight per lane (halved for two float4 per lane)
constexpr int kUA = 4;             // raw values in flight per lane in phase A
constexpr int kUPool = 4;          // row loads in flight per lane when pooling short bags (8 spills)
constexpr int kOneHotBags = 256;   // bags of one value each that one warp chunk copies
constexpr int kMaxTileBags = 1024;  // static schedule: at most this many bags per tile
constexpr int64_t kShortBagMean = 16;   // static schedule: streams with shorter bags tile by bags
constexpr int kPadPiece = 64;      // positions per piece of a long padded bag (about)
constexpr int kFwdWarpsPerCta = kFwdThreads / kWarp;

struct FwdArgs {
  const ColMeta* meta;     // id-stream columns, then f-stream columns
  const int64_t* ids;
  const float* fvals;
  const float* wts[2];     // per-value weights of each stream (SUM columns), or null
  const int32_t* offs[2];
  int64_t n[2];
  int32_t ncols[2];
  int32_t col_base[2];
  int64_t tiles[2];
  int32_t tile_elems;      // value tiles: values per tile
  int32_t tile_bags[2];    // per stream: bags per tile, or 0 for value tiles
  const int32_t* col_order;  // bag tiles: per stream, column positions in work order (null: stream order)
  int32_t tpc[2];          // bag tiles in work order: tiles per column (batch / tile_bags), else 0
  DivMagic32 tpc_div[2];
  int32_t batch;
  DivMagic32 bdiv;
  int64_t ldo;
  float* out;
  float* seq_out;
  int64_t* rows_dbg;
  int64_t rec_base[2];     // record index of element 0 of each stream
  uint32_t* keys;          // training: global row per contribution (sentinel if none)
  uint32_t* vals;          // training: gradient source per contribution (its record, when weighted)
  uint2* rec_src;          // weighted training: (gradient source, weight bits) per record
  float* inv_n;            // training: 1/n_valid per mean bag
  uint32_t key_sentinel;
  uint32_t* status;
  unsigned long long* ticket;   // [0] next tile, [1] warps done; both 0 between launches
  int64_t n_warps;              // warps launched
  int32_t dynamic;              // schedule: 0 static, 1 persistent warps with tickets
  // pieces of long padded bags, the tiles after the value tiles: tile t is
  // piece t mod npc of bag (t / npc) mod batch of long padded column
  // t / (batch * npc)
  int64_t pad_tiles;
  const int32_t* pad_cols;      // meta position of each long padded column
  int32_t pad_npc;              // pieces per bag
  DivMagic32 pad_ndiv;          // division by pad_npc
  DivMagic32 pad_bdiv;          // division by batch * pad_npc
};

struct __align__(16) WarpSmem {
  float4 part[2][64];      // head / tail partial sums, [group * dim/4 + slot]
  int32_t rows[kWarpElems];
  uint8_t bag[kWarpElems];
  int32_t pos[33];         // first slot of each bag's values in rows[]
  int32_t lo[32];          // first stream element of each bag
  int32_t len[32];         // values of the bag held in rows[]
  int32_t tailbag[32];     // per lane group: bag whose tail partial it holds
  int32_t nvp[32][2];      // per lane group: valid counts of head / tail partials
  ColMeta cm;              // metadata of the chunk's column
};

__device__ __forceinline__ float4 f4zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }

__device__ __forceinline__ void f4add(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

__device__ __forceinline__ void f4fma(float4& a, float w, const float4& b) {
  a.x = fmaf(w, b.x, a.x);
  a.y = fmaf(w, b.y, a.y);
  a.z = fmaf(w, b.z, a.z);
  a.w = fmaf(w, b.w, a.w);
}

__device__ __forceinline__ float4 f4scale(float w, const float4& b) {
  return make_float4(w * b.x, w * b.y, w * b.z, w * b.w);
}

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// One lane's share of a row -- elements 4 f4 .. 4 f4 + 3 -- as loaded, for
// rows stored as DT (emb_table_dtype).  A batch of these stays in flight in
// its stored width (two registers for bf16 / fp16) and becomes fp32 only
// where it is used: bf16 and fp16 convert exactly (bf16 is the upper half of
// an fp32), int8 element q reads as scale * q.
template <int DT>
struct RowRaw {
  float4 x;
};
template <>
struct RowRaw<EMB_DT_BF16> {
  uint2 x;
};
template <>
struct RowRaw<EMB_DT_F16> {
  uint2 x;
};
template <>
struct RowRaw<EMB_DT_I8> {
  uint32_t q;
  float s;
};

// Rows in flight per lane in the whole-warp and padded paths scale with the
// registers a raw share takes: two for the low-precision types against four
// for fp32 (measured: 5 % faster on long bf16 bags; in the lane-group paths
// of short bags the deeper batches measured slower and are not used).
template <int DT>
constexpr int kRawScale = DT == EMB_DT_F32 ? 1 : 2;

template <int DT>
__device__ __forceinline__ RowRaw<DT> raw_zero() {
  RowRaw<DT> z;
  if constexpr (DT == EMB_DT_F32) {
    z.x = f4zero();
  } else if constexpr (DT == EMB_DT_I8) {
    z.q = 0u;
    z.s = 0.0f;
  } else {
    z.x = make_uint2(0u, 0u);
  }
  return z;
}

template <int DT>
__device__ __forceinline__ RowRaw<DT> row_raw(const float* E, int dim, const float* qs, int32_t r, int f4) {
  const int64_t e = (int64_t)r * dim + f4 * 4;
  RowRaw<DT> v;
  if constexpr (DT == EMB_DT_F32) {
    v.x = ldg4(E + e);
  } else if constexpr (DT == EMB_DT_I8) {
    v.q = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const int8_t*>(E) + e));
    v.s = __ldg(qs + r);
  } else {
    v.x = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(E) + e));
  }
  return v;
}

template <int DT>
__device__ __forceinline__ float4 raw_f4(const RowRaw<DT>& v) {
  if constexpr (DT == EMB_DT_F32) {
    return v.x;
  } else if constexpr (DT == EMB_DT_I8) {
    const int32_t q = (int32_t)v.q;
    return make_float4(v.s * (float)((q << 24) >> 24), v.s * (float)((q << 16) >> 24),
                       v.s * (float)((q << 8) >> 24), v.s * (float)(q >> 24));
  } else if constexpr (DT == EMB_DT_BF16) {
    return make_float4(__uint_as_float(v.x.x << 16), __uint_as_float(v.x.x & 0xffff0000u),
                       __uint_as_float(v.x.y << 16), __uint_as_float(v.x.y & 0xffff0000u));
  } else {
    const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&v.x.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&v.x.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  }
}

// Calls f with the column's storage type as a compile-time constant: only
// fp32 unless the launch has low-precision tables (LP).
template <bool LP, class F>
__device__ __forceinline__ void with_dtype(int dtype, F&& f) {
  if constexpr (!LP) {
    f(std::integral_constant<int, EMB_DT_F32>{});
  } else {
    switch (dtype) {
      case EMB_DT_BF16: f(std::integral_constant<int, EMB_DT_BF16>{}); break;
      case EMB_DT_F16: f(std::integral_constant<int, EMB_DT_F16>{}); break;
      case EMB_DT_I8: f(std::integral_constant<int, EMB_DT_I8>{}); break;
      default: f(std::integral_constant<int, EMB_DT_F32>{}); break;
    }
  }
}

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

// Both ends of a tile at once: the first s with clamp(offs[s]) >= e_lo and
// the first with clamp(offs[s]) >= e_hi, each searched by half the warp with
// 16-ary rounds (lanes 0-15: e_lo, lanes 16-31: e_hi), so the two searches
// share their round trips.
__device__ int2 warp_lower_bound2(const int32_t* offs, int S, int64_t e_lo, int64_t e_hi, int64_t n) {
  const int lane = threadIdx.x & 31;
  const int h = lane >> 4, sl = lane & 15;
  const unsigned half = h ? 0xffff0000u : 0x0000ffffu;
  const int64_t e = h ? e_hi : e_lo;
  bool bad = false;
  int lo = 0, hi = S;
  if (S > 0) {
    // First round: 16 probes around the segment a uniform spread of the n
    // values over the S segments puts at e, over a window of about twice the
    // square root of its distance to the nearer end (the spread of a sum of
    // that many similar bag lengths).  If the answer lies outside the window
    // the search goes on from there over the rest of [0, S].
    const int g = e >= n ? S : (int)(e * (int64_t)S / (n > 1 ? n : 1));
    const int d = min(g, S - g);
    const int half_w = min(2048, 32 + 2 * (int)sqrtf((float)d));
    const int wlo = max(0, g - half_w), whi = min(S, g + half_w);
    const int wstep = max(1, (whi - wlo) / 15);
    auto probe_at = [&](int j) { return min(wlo + j * wstep, S - 1); };
    const bool less = clamp_off(__ldg(offs + probe_at(sl)), n, bad) < e;
    const int k = __popc(__ballot_sync(kFull, less) & half);
    if (k == 0) {
      hi = probe_at(0);
    } else if (k == 16) {
      lo = probe_at(15) + 1;
    } else {
      lo = probe_at(k - 1) + 1;
      hi = probe_at(k);
    }
  }
  for (;;) {
    const bool more = hi - lo > 16;
    if (!__any_sync(kFull, more)) break;
    const int step = (hi - lo + 15) >> 4;
    const int p = lo + (sl + 1) * step - 1;
    const bool less = more && (p < hi) && (clamp_off(__ldg(offs + p), n, bad) < e);
    const int k = __popc(__ballot_sync(kFull, less) & half);
    if (more) {
      const int nlo = min(lo + k * step, hi);
      hi = min(hi, nlo + step - 1);
      lo = nlo;
    }
  }
  const int p = lo + sl;
  const bool less = (p < hi) && (clamp_off(__ldg(offs + p), n, bad) < e);
  const int r = lo + __popc(__ballot_sync(kFull, less) & half);
  return make_int2(__shfl_sync(kFull, r, 0), __shfl_sync(kFull, r, 16));
}

// Raw value of element t (int64 id, or the fp32 bits of a bucketize value).
__device__ __forceinline__ int64_t col_load(const ColMeta& m, const int64_t* ids, const float* fvals, int64_t t) {
  if (m.transform == EMB_T_BUCKETIZE) return (int64_t)__float_as_int(__ldcs(fvals + t));
  return __ldcs(ids + t);
}

// Transformed, guarded row of a raw value; -1 when dropped.
__device__ __forceinline__ int32_t col_transform(const ColMeta& m, int64_t v) {
  if (m.transform == EMB_T_BUCKETIZE) {
    const float x = __int_as_float((int32_t)v);
    int lo = 0, hi = m.nb;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(m.bnd + mid) <= x) lo = mid + 1; else hi = mid;
    }
    return lo;
  }
  if (m.transform == EMB_T_HASH_MOD) return (int32_t)mod_magic(splitmix64((uint64_t)v), m.mod);
  return (v >= 0 && v < m.num_rows) ? (int32_t)v : -1;
}

// Rows of kUA raw values of one column.  Bucketize: the kUA binary searches
// advance together, so their boundary loads are in flight at the same time
// (row = #{j : bnd[j] <= x}).
__device__ __forceinline__ void transform_batch(const ColMeta& m, const int64_t (&raw)[kUA], int32_t (&rowv)[kUA]) {
  if (m.transform == EMB_T_BUCKETIZE) {
    int blo[kUA], blen[kUA];
    float x[kUA];
#pragma unroll
    for (int u = 0; u < kUA; ++u) {
      blo[u] = 0;
      blen[u] = m.nb;
      x[u] = __int_as_float((int32_t)raw[u]);
    }
    bool more = m.nb > 0;
    while (more) {
      more = false;
#pragma unroll
      for (int u = 0; u < kUA; ++u) {
        if (blen[u] > 0) {
          const int half = blen[u] >> 1;
          const bool go = __ldg(m.bnd + blo[u] + half) <= x[u];
          blo[u] = go ? blo[u] + half + 1 : blo[u];
          blen[u] = go ? blen[u] - half - 1 : half;
          more |= blen[u] > 0;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUA; ++u) rowv[u] = blo[u];
  } else {
#pragma unroll
    for (int u = 0; u < kUA; ++u) rowv[u] = col_transform(m, raw[u]);
  }
}

__device__ __forceinline__ int32_t col_row(const ColMeta& m, const int64_t* ids, const float* fvals,
                                           int64_t t) {
  return col_transform(m, col_load(m, ids, fvals, t));
}

// WT: the launch carries value weights (training then records them)
template <bool WT>
__device__ __forceinline__ void record(const FwdArgs& a, int st, int64_t t, int32_t row,
                                       const ColMeta& m, uint32_t gsrc) {
  const int64_t r = a.rec_base[st] + t;
  if (a.rows_dbg) a.rows_dbg[r] = row;
  if (a.keys) {
    a.keys[r] = row >= 0 ? m.table_base + (uint32_t)row : a.key_sentinel;
    if (WT && a.rec_src) {
      // the sort carries the record; the backward reads source and weight here
      const float w = (m.pooling == EMB_POOL_SUM && a.wts[st]) ? __ldg(a.wts[st] + t) : 1.0f;
      a.rec_src[r] = make_uint2(gsrc, __float_as_uint(w));
      a.vals[r] = (uint32_t)r;
    } else {
      a.vals[r] = gsrc;
    }
  }
}

__device__ __forceinline__ void record_cut(const FwdArgs& a, int st, int64_t t, const ColMeta& m) {
  // a value past pad_len: no output, no gradient
  const int64_t r = a.rec_base[st] + t;
  if (a.rows_dbg) a.rows_dbg[r] = col_row(m, a.ids, a.fvals, t);
  if (a.keys) {
    a.keys[r] = a.key_sentinel;
    a.vals[r] = 0u;
  }
}

// Compensated (Neumaier) accumulation: the error of a long fp32 sum stays
// near one rounding of the result instead of growing with the chain length.
__device__ __forceinline__ void kadd(float& s, float& c, float x) {
  const float t = s + x;
  c += (fabsf(s) >= fabsf(x)) ? ((s - t) + x) : ((x - t) + s);
  s = t;
}

__device__ __forceinline__ void kadd4(float4& s, float4& c, const float4& x) {
  kadd(s.x, c.x, x.x);
  kadd(s.y, c.y, x.y);
  kadd(s.z, c.z, x.z);
  kadd(s.w, c.w, x.w);
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

__device__ __forceinline__ uint32_t pooled_gsrc(const FwdArgs& a, const ColMeta& m, int32_t bag) {
  return (uint32_t)m.col * (uint32_t)a.batch + (uint32_t)bag;
}

__device__ __forceinline__ uint32_t padded_gsrc(const FwdArgs& a, const ColMeta& m, int32_t bag, int64_t p) {
  return kPadBit | (uint32_t)((m.seq_unit * a.batch + ((int64_t)bag * m.pad_len + p) * m.dim) >> 2);
}

// ---------------------------------------------------------------------------
// phase B, pooled: equal value ranges per lane group; WT: a SUM column of a
// weighted stream, each row scaled by its value's weight W[t]
// ---------------------------------------------------------------------------
template <int V, bool WT, int DT>
__device__ void warp_pool_chunk(const FwdArgs& a, WarpSmem& ws, const ColMeta& m, const float* W, int ns, int T,
                                int b0, int glog, unsigned longmask) {
  constexpr int U = kUPool / V;
  const int dim = m.dim, dim4 = m.dim4;
  const int lane = threadIdx.x & 31;
  const int G = 32 >> glog;
  const int q = lane >> glog, sub = lane & ((1 << glog) - 1);
  const int R = (T + G - 1) / G;
  const int k0 = min(q * R, T), k1 = min(k0 + R, T);
  const float* E = m.weight;
  const float* qs = m.qscale;

  float4 acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = f4zero();
  int nv = 0;
  int curb = k0 < k1 ? (int)ws.bag[k0] : -1;
  bool head = k0 > 0 && k0 < k1 && (int)ws.bag[k0 - 1] == curb;
  if (sub == 0) ws.tailbag[q] = -1;

  auto write_out = [&](int b, const float4 (&s)[V], int cnt) {
    const int bag = b0 + b;
    float* y = a.out + (int64_t)bag * a.ldo + m.out_col;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      if (f4 < m.dim4) *reinterpret_cast<float4*>(y + f4 * 4) = finish(m, s[v], cnt, f4);
    }
    if (a.inv_n && sub == 0 && m.pooling == EMB_POOL_MEAN)
      a.inv_n[pooled_gsrc(a, m, bag)] = cnt > 0 ? 1.0f / (float)cnt : 0.0f;
  };
  auto flush = [&](bool tail) {
    if (!head && !tail) {
      write_out(curb, acc, nv);
      return;
    }
    const int side = head ? 0 : 1;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      if (f4 < m.dim4) ws.part[side][q * m.dim4 + f4] = acc[v];
    }
    if (sub == 0) {
      ws.nvp[q][side] = nv;
      if (!head) ws.tailbag[q] = curb;
    }
  };

  for (int j = 0; j < R; j += U) {
    RowRaw<DT> vals[U][V];
    float wu[WT ? U : 1];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = k0 + j + u;
      const int r = k < k1 ? ws.rows[k] : -1;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        vals[u][v] = (r >= 0 && f4 < dim4) ? row_raw<DT>(E, dim, qs, r, f4) : raw_zero<DT>();
      }
      if constexpr (WT) {
        wu[u] = 0.0f;
        if (r >= 0) {
          const int bg = (int)ws.bag[k];
          wu[u] = __ldg(W + (int64_t)ws.lo[bg] + (k - ws.pos[bg]));
        }
      }
    }
    // bag and validity are read again from shared memory rather than held
    // in registers across the loads, which leaves room for more loads in flight
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = k0 + j + u;
      if (k >= k1) break;
      const int bg = (int)ws.bag[k];
      if (bg != curb) {
        flush(false);
        curb = bg;
        head = false;
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = f4zero();
        nv = 0;
      }
#pragma unroll
      for (int v = 0; v < V; ++v) {
        if constexpr (WT) f4fma(acc[v], wu[u], raw_f4<DT>(vals[u][v]));
        else f4add(acc[v], raw_f4<DT>(vals[u][v]));
      }
      nv += ws.rows[k] >= 0;
    }
  }
  if (k0 < k1) flush(k1 < T && (int)ws.bag[k1] == curb);
  __syncwarp();

  // the group holding a cut bag's first value adds the partials in order
  const int tb = ws.tailbag[q];
  if (tb >= 0) {
    float4 s[V];
    int cnt = ws.nvp[q][1];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      s[v] = f4 < m.dim4 ? ws.part[1][q * m.dim4 + f4] : f4zero();
    }
    const int last = (ws.pos[tb] + ws.len[tb] - 1) / R;
    for (int q2 = q + 1; q2 <= last; ++q2) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < m.dim4) f4add(s[v], ws.part[0][q2 * m.dim4 + f4]);
      }
      cnt += ws.nvp[q2][0];
    }
    write_out(tb, s, cnt);
  }
  // empty bags: default vector
  if (lane < ns && ws.len[lane] == 0 && !((longmask >> lane) & 1u)) {
    float* y = a.out + (int64_t)(b0 + lane) * a.ldo + m.out_col;
    for (int f4 = 0; f4 < m.dim4; ++f4) *reinterpret_cast<float4*>(y + f4 * 4) = finish(m, f4zero(), 0, f4);
    if (a.inv_n && m.pooling == EMB_POOL_MEAN) a.inv_n[pooled_gsrc(a, m, b0 + lane)] = 0.0f;
  }
}

// phase B, padded (short pad_len): ns bags x pad_len output rows, flat over groups
template <int V, int DT>
__device__ void warp_pad_chunk(const FwdArgs& a, WarpSmem& ws, const ColMeta& m, int ns, int b0, int glog,
                               unsigned longmask) {
  constexpr int U = kU / V * kRawScale<DT>;
  const int lane = threadIdx.x & 31;
  const int G = 32 >> glog;
  const int q = lane >> glog, sub = lane & ((1 << glog) - 1);
  const int P = m.pad_len;
  const int total = ns * P;
  const float* E = m.weight;
  for (int base = 0; base < total; base += G * U) {
    RowRaw<DT> vals[U][V];
    int o[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      o[u] = base + u * G + q;
      int r = -1;
      if (o[u] < total) {
        const int i = o[u] / P, p = o[u] - i * P;
        if (p < ws.len[i]) r = ws.rows[ws.pos[i] + p];
      }
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        vals[u][v] = (r >= 0 && f4 < m.dim4) ? row_raw<DT>(E, m.dim, m.qscale, r, f4) : raw_zero<DT>();
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (o[u] >= total) continue;
      const int i = o[u] / P, p = o[u] - i * P;
      if ((longmask >> i) & 1u) continue;
      float* dst = a.seq_out + m.seq_unit * a.batch + ((int64_t)(b0 + i) * P + p) * m.dim;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < m.dim4) __stcs(reinterpret_cast<float4*>(dst + f4 * 4), raw_f4<DT>(vals[u][v]));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// padded pieces: positions [p_lo, p_hi) of one padded bag, the whole warp
// ---------------------------------------------------------------------------
// A long padded bag (pad_len > kLongBag) is copied in pieces of positions,
// each a tile of its own, so that no warp copies a whole bag while the rest
// of the launch has finished.  Positions past the bag's values are zeros.
// The output is written once and never read back by the launch: its stores
// are marked evict-first, so they do not push table rows out of L2.
template <int V, bool WT, int DT>
__device__ void warp_pad_piece(const FwdArgs& a, int st, const ColMeta& m, int32_t b, int64_t lo, int64_t hi,
                               int p_lo, int p_hi, int glog) {
  constexpr int U = kU / V * (WT ? 1 : kRawScale<DT>);
  const int lane = threadIdx.x & 31;
  const int G = 32 >> glog;
  const int grp = lane >> glog, sub = lane & ((1 << glog) - 1);
  const float* E = m.weight;
  const int P = m.pad_len;
  const int64_t len = hi - lo;
  float* dst = a.seq_out + m.seq_unit * a.batch + (int64_t)b * P * m.dim;
  for (int p0 = p_lo; p0 < p_hi; p0 += 32) {
    const int cnt = min(32, p_hi - p0);
    if (p0 >= len) {
      // zeros only: the positions' rows are contiguous in the output
      float4* z = reinterpret_cast<float4*>(dst + (int64_t)p0 * m.dim);
      for (int k = lane; k < cnt * m.dim4; k += 32) __stcs(z + k, f4zero());
      continue;
    }
    int32_t row = -1;
    const int p = p0 + lane;
    if (lane < cnt && p < len) {
      row = col_row(m, a.ids, a.fvals, lo + p);
      record<WT>(a, st, lo + p, row, m, padded_gsrc(a, m, b, p));
    }
    for (int k = 0; k < cnt; k += U * G) {
      RowRaw<DT> v[U][V];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = k + u * G + grp;
        const int r = __shfl_sync(kFull, row, j & 31);
        const bool ok = (j < cnt) && (r >= 0);
#pragma unroll
        for (int q = 0; q < V; ++q) {
          const int f4 = sub + q * 32;
          v[u][q] = (ok && f4 < m.dim4) ? row_raw<DT>(E, m.dim, m.qscale, r, f4) : raw_zero<DT>();
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = k + u * G + grp;
#pragma unroll
        for (int q = 0; q < V; ++q) {
          const int f4 = sub + q * 32;
          if (j < cnt && f4 < m.dim4)
            __stcs(reinterpret_cast<float4*>(dst + (int64_t)(p0 + j) * m.dim + f4 * 4), raw_f4<DT>(v[u][q]));
        }
      }
    }
  }
  // values past pad_len: no output, no gradient (recorded by the last piece)
  if (p_hi == P && (a.rows_dbg || a.keys))
    for (int64_t t = lo + P + lane; t < hi; t += 32) record_cut(a, st, t, m);
}

// ---------------------------------------------------------------------------
// phase C: one long pooled bag, the whole warp, values transformed on the fly
// ---------------------------------------------------------------------------
template <int V, bool WT, int DT>
__device__ void warp_long_bag(const FwdArgs& a, int st, const ColMeta& m, const float* W, int32_t b, int64_t lo,
                              int64_t hi, int glog) {
  constexpr int U = kU / V * (WT ? 1 : kRawScale<DT>);
  const int lane = threadIdx.x & 31;
  const int G = 32 >> glog;
  const int grp = lane >> glog, sub = lane & ((1 << glog) - 1);
  const float* E = m.weight;
  const uint32_t gsrc = pooled_gsrc(a, m, b);
  float4 acc[V], cmp[V];
#pragma unroll
  for (int q = 0; q < V; ++q) {
    acc[q] = f4zero();
    cmp[q] = f4zero();
  }
  int nv = 0;
  for (int64_t base = lo; base < hi; base += 32) {
    const int cnt = (int)(hi - base < 32 ? hi - base : 32);
    int32_t row = -1;
    float wl = 1.0f;
    if (lane < cnt) {
      row = col_row(m, a.ids, a.fvals, base + lane);
      record<WT>(a, st, base + lane, row, m, gsrc);
      if (WT && W && row >= 0) wl = __ldg(W + base + lane);
    }
    nv += __popc(__ballot_sync(kFull, row >= 0));
    for (int k = 0; k < cnt; k += U * G) {
      RowRaw<DT> v[U][V];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = k + u * G + grp;
        const int r = __shfl_sync(kFull, row, j & 31);
        const bool ok = (j < cnt) && (r >= 0);
#pragma unroll
        for (int q = 0; q < V; ++q) {
          const int f4 = sub + q * 32;
          v[u][q] = (ok && f4 < m.dim4) ? row_raw<DT>(E, m.dim, m.qscale, r, f4) : raw_zero<DT>();
        }
      }
      float wj[U];
#pragma unroll
      for (int u = 0; u < U; ++u) wj[u] = 1.0f;
      if (WT && W) {
#pragma unroll
        for (int u = 0; u < U; ++u) wj[u] = __shfl_sync(kFull, wl, (k + u * G + grp) & 31);
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int q = 0; q < V; ++q) {
          const float4 x = raw_f4<DT>(v[u][q]);
          kadd4(acc[q], cmp[q], (WT && W) ? f4scale(wj[u], x) : x);
        }
    }
  }
#pragma unroll
  for (int q = 0; q < V; ++q) {
    acc[q].x += cmp[q].x;
    acc[q].y += cmp[q].y;
    acc[q].z += cmp[q].z;
    acc[q].w += cmp[q].w;
  }
#pragma unroll
  for (int q = 0; q < V; ++q)
    for (int off = 1 << glog; off < 32; off <<= 1) {
      acc[q].x += __shfl_xor_sync(kFull, acc[q].x, off);
      acc[q].y += __shfl_xor_sync(kFull, acc[q].y, off);
      acc[q].z += __shfl_xor_sync(kFull, acc[q].z, off);
      acc[q].w += __shfl_xor_sync(kFull, acc[q].w, off);
    }
  if (grp == 0) {
    float* y = a.out + (int64_t)b * a.ldo + m.out_col;
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const int f4 = sub + q * 32;
      if (f4 < m.dim4) *reinterpret_cast<float4*>(y + f4 * 4) = finish(m, acc[q], nv, f4);
    }
  }
  if (a.inv_n && lane == 0 && m.pooling == EMB_POOL_MEAN) a.inv_n[gsrc] = nv > 0 ? 1.0f / (float)nv : 0.0f;
}

// ---------------------------------------------------------------------------
// one-hot chunk: nb pooled bags of exactly one value each, the values
// t0 .. t0 + nb - 1 of the stream.  A bag's result is its one row (times its
// weight, or the default vector when the value is dropped), so the chunk is
// a transform and a row copy: no offsets per bag, no reduction, and up to
// kOneHotBags bags share each round trip.  WT: the launch carries weights
// (records hold them); W: this column's value weights, or null.
// ---------------------------------------------------------------------------
template <int V, bool WT, int DT>
__device__ void warp_onehot_chunk(const FwdArgs& a, WarpSmem& ws, const ColMeta& m, const float* W, int st,
                                  int64_t t0, int nb, int b0, int glog) {
  constexpr int U = kUPool / V;
  const int lane = threadIdx.x & 31;
  for (int k0 = 0; k0 < nb; k0 += 32 * kUA) {
    int64_t raw[kUA];
#pragma unroll
    for (int u = 0; u < kUA; ++u) {
      const int k = k0 + u * 32 + lane;
      raw[u] = k < nb ? col_load(m, a.ids, a.fvals, t0 + k) : 0;
    }
    int32_t rowv[kUA];
    transform_batch(m, raw, rowv);
#pragma unroll
    for (int u = 0; u < kUA; ++u) {
      const int k = k0 + u * 32 + lane;
      if (k < nb) {
        ws.rows[k] = rowv[u];
        if (a.rows_dbg || a.keys) record<WT>(a, st, t0 + k, rowv[u], m, pooled_gsrc(a, m, b0 + k));
      }
    }
  }
  __syncwarp();
  const int G = 32 >> glog;
  const int q = lane >> glog, sub = lane & ((1 << glog) - 1);
  const float* E = m.weight;
  for (int j = q; j < nb; j += G * U) {
    RowRaw<DT> vals[U][V];
    int r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = j + u * G;
      r[u] = k < nb ? ws.rows[k] : -1;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        vals[u][v] = (r[u] >= 0 && f4 < m.dim4) ? row_raw<DT>(E, m.dim, m.qscale, r[u], f4) : raw_zero<DT>();
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = j + u * G;
      if (k >= nb) break;
      const int cnt = r[u] >= 0 ? 1 : 0;
      const bool wt = WT && W != nullptr;
      const float wk = (wt && cnt) ? __ldg(W + t0 + k) : 1.0f;
      float* y = a.out + (int64_t)(b0 + k) * a.ldo + m.out_col;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int f4 = sub + v * 32;
        if (f4 < m.dim4) {
          const float4 e = wt ? f4scale(wk, raw_f4<DT>(vals[u][v])) : raw_f4<DT>(vals[u][v]);
          *reinterpret_cast<float4*>(y + f4 * 4) = finish(m, e, cnt, f4);
        }
      }
      if (a.inv_n && sub == 0 && m.pooling == EMB_POOL_MEAN) a.inv_n[pooled_gsrc(a, m, b0 + k)] = (float)cnt;
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// the kernel: one warp per element tile
// ---------------------------------------------------------------------------
template <bool WT, bool LP>
__device__ __forceinline__ void forward_tile(const FwdArgs& a, WarpSmem& ws, int st, int64_t tile);
template <bool WT, bool LP>
__device__ __forceinline__ void forward_piece(const FwdArgs& a, WarpSmem& ws, int64_t t);

// Two schedules.  Static: one tile per warp, the grid covers all tiles (warps
// of one CTA hold neighbouring tiles, whose offset searches share L1).
// Dynamic, for long bags: persistent warps start on the tile of their own
// index, then take tiles in ticket order from a counter until none is left,
// so a warp that drew short bags takes the next tile at once instead of
// idling beside a sibling that drew long ones; the last warp to finish
// resets the counter for the next launch (CUDA-graph safe: no host state
// changes between launches).
// WT: a launch with value weights, LP: one with tables stored below fp32;
// each gets its own instance, so the plain fp32 one keeps its registers for
// loads in flight.
template <bool WT, bool LP>
__global__ void __launch_bounds__(kFwdThreads, 4) k_forward(const FwdArgs a) {
  __shared__ WarpSmem smem[kFwdWarpsPerCta];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WarpSmem& ws = smem[warp];
  const int64_t n_vt = a.tiles[0] + a.tiles[1];
  const int64_t n_tiles = n_vt + a.pad_tiles;
  // the first tile of every warp is its warp index; tickets count from there
  int64_t tile = (int64_t)blockIdx.x * kFwdWarpsPerCta + warp;
  while (tile < n_tiles) {
    if (tile >= n_vt) {
      forward_piece<WT, LP>(a, ws, tile - n_vt);
    } else {
      const int st = tile < a.tiles[0] ? 0 : 1;
      int64_t lt = st ? tile - a.tiles[0] : tile;
      if (a.tpc[st] > 0) {
        // bag tiles whole columns apart: take the columns in work order
        const int j = (int)div_magic32((uint32_t)lt, a.tpc_div[st]);
        lt = (int64_t)__ldg(a.col_order + a.col_base[st] + j) * a.tpc[st] + (lt - (int64_t)j * a.tpc[st]);
      }
      forward_tile<WT, LP>(a, ws, st, lt);
    }
    if (!a.dynamic) break;   // static: one tile per warp
    unsigned long long tk = 0;
    if (lane == 0) tk = atomicAdd(&a.ticket[0], 1ull);
    tile = a.n_warps + (int64_t)__shfl_sync(kFull, tk, 0);
  }
  if (a.dynamic && lane == 0) {
    __threadfence();   // this warp's last ticket is taken before it counts itself done
    if (atomicAdd(&a.ticket[1], 1ull) == (unsigned long long)(a.n_warps - 1)) {
      __threadfence();
      atomicExch(&a.ticket[0], 0ull);
      atomicExch(&a.ticket[1], 0ull);
    }
  }
}

// One piece of a long padded bag: its column, bag and positions follow from
// the piece index alone.
template <bool WT, bool LP>
__device__ __forceinline__ void forward_piece(const FwdArgs& a, WarpSmem& ws, int64_t t) {
  const int lane = threadIdx.x & 31;
  const uint32_t tt = (uint32_t)t;
  const uint32_t j = div_magic32(tt, a.pad_bdiv);
  const uint32_t r = tt - j * a.pad_bdiv.d;
  const uint32_t b = div_magic32(r, a.pad_ndiv);
  const int q = (int)(r - b * a.pad_ndiv.d);
  const int mi = __ldg(a.pad_cols + j);
  const int st = mi >= a.ncols[0] ? 1 : 0;
  const int64_t seg = (int64_t)(mi - a.col_base[st]) * a.batch + b;
  const int32_t o_lo = __ldg(a.offs[st] + seg), o_hi = __ldg(a.offs[st] + seg + 1);
  __syncwarp();   // the previous tile's reads of ws.cm are done
  if (lane < (int)(sizeof(ColMeta) / 4))
    reinterpret_cast<int32_t*>(&ws.cm)[lane] = __ldg(reinterpret_cast<const int32_t*>(a.meta + mi) + lane);
  __syncwarp();
  const ColMeta& m = ws.cm;
  bool bad = false;
  const int64_t lo = clamp_off(o_lo, a.n[st], bad);
  int64_t hi = clamp_off(o_hi, a.n[st], bad);
  if (hi < lo) {
    hi = lo;
    bad = true;
  }
  if (bad && lane == 0) latch(a.status, EMB_ERR_BAD_INDEX);
  const int P = m.pad_len;
  const int PL = ((P + a.pad_npc - 1) / a.pad_npc + 31) & ~31;   // positions per piece
  const int p_lo = q * PL, p_hi = min(P, p_lo + PL);
  if (p_lo < p_hi) {
    const int glog = lanes_log2(m.dim4);
    with_dtype<LP>(m.dtype, [&](auto dt) {
      constexpr int DT = decltype(dt)::value;
      if (m.dim4 > 32) warp_pad_piece<2, WT, DT>(a, st, m, (int32_t)b, lo, hi, p_lo, p_hi, glog);
      else warp_pad_piece<1, WT, DT>(a, st, m, (int32_t)b, lo, hi, p_lo, p_hi, glog);
    });
  }
  __syncwarp();
}

template <bool WT, bool LP>
__device__ __forceinline__ void forward_tile(const FwdArgs& a, WarpSmem& ws, int st, int64_t tile) {
  const int lane = threadIdx.x & 31;
  const int S = a.ncols[st] * a.batch;
  const int32_t* offs = a.offs[st];
  const int64_t n = a.n[st];
  int cur, s_hi;
  if (a.tile_bags[st] > 0) {
    // a run of tile_bags consecutive bags
    cur = (int)(tile * a.tile_bags[st]);
    s_hi = (int)min((int64_t)S, (int64_t)cur + a.tile_bags[st]);
  } else {
    // a range of tile_elems values: the bags whose first value lies in it
    const int64_t e0 = tile * a.tile_elems;
    const bool last = tile == a.tiles[st] - 1;
    const int2 ends = warp_lower_bound2(offs, S, e0, last ? INT64_MAX : e0 + a.tile_elems, n);
    cur = ends.x;
    s_hi = ends.y;
  }

  while (cur < s_hi) {
    // ---- setup: one lane per bag, all inside column cl0 ----
    const int cl0 = (int)div_magic32((uint32_t)cur, a.bdiv);
    const int b0 = cur - cl0 * a.batch;
    const int navail = min(32, min(s_hi, (cl0 + 1) * a.batch) - cur);
    // the bags' offsets and the column's metadata are loaded side by side
    int32_t o_lo = 0, o_hi = 0;
    if (lane < navail) {
      o_lo = __ldg(offs + cur + lane);
      o_hi = __ldg(offs + cur + lane + 1);
    }
    static_assert(sizeof(ColMeta) % 4 == 0 && sizeof(ColMeta) / 4 <= 32, "metadata copy");
    if (lane < (int)(sizeof(ColMeta) / 4))
      reinterpret_cast<int32_t*>(&ws.cm)[lane] =
          __ldg(reinterpret_cast<const int32_t*>(a.meta + a.col_base[st] + cl0) + lane);
    __syncwarp();
    const ColMeta& m = ws.cm;
    const bool padded = m.pooling == EMB_POOL_NONE_PADDED;
    int64_t lo = 0, hi = 0;
    int used = 0;
    bool is_long = false, one = false;
    if (lane < navail) {
      bool bad = false;
      lo = clamp_off(o_lo, n, bad);
      hi = clamp_off(o_hi, n, bad);
      if (hi < lo) { hi = lo; bad = true; }
      if (bad) latch(a.status, EMB_ERR_BAD_INDEX);
      one = !bad && hi - lo == 1;
      if (m.trunc > 0 && hi - lo > m.trunc) hi = lo + m.trunc;   // sequence truncation (pooled only)
      const int64_t len = hi - lo;
      is_long = (padded ? (int64_t)m.pad_len : len) > kLongBag;
      used = is_long ? 0 : (int)(padded ? (len < m.pad_len ? len : (int64_t)m.pad_len) : len);
    }
    if (!padded && __ballot_sync(kFull, one) == kFull) {
      // ---- 32 bags of one value each: extend the run of one-value bags
      //      (offsets that step by exactly 1) up to kOneHotBags bags ----
      const int64_t lo0 = __shfl_sync(kFull, lo, 0);
      const int lim = min(kOneHotBags, min(s_hi, (cl0 + 1) * a.batch) - cur);
      int stop = lim;   // bags [0, stop) hold one value each
#pragma unroll
      for (int i = 0; i < kOneHotBags / 32 - 1; ++i) {
        const int k = 33 + i * 32 + lane;   // offsets index after the chunk's first 32 bags
        if (k <= lim && ((int64_t)__ldg(offs + cur + k) != lo0 + k || lo0 + k > n)) stop = min(stop, k - 1);
      }
      stop = __reduce_min_sync(kFull, stop);
      const float* W = WT && m.pooling == EMB_POOL_SUM ? a.wts[st] : nullptr;
      const int glog = lanes_log2(m.dim4);
      with_dtype<LP>(m.dtype, [&](auto dt) {
        constexpr int DT = decltype(dt)::value;
        if (m.dim4 > 32) warp_onehot_chunk<2, WT, DT>(a, ws, m, W, st, lo0, stop, b0, glog);
        else warp_onehot_chunk<1, WT, DT>(a, ws, m, W, st, lo0, stop, b0, glog);
      });
      cur += stop;
      continue;
    }
    int incl = used;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    const int pos = incl - used;
    const int ns = __popc(__ballot_sync(kFull, lane < navail && incl <= kWarpElems));
    const unsigned longmask = __ballot_sync(kFull, lane < ns && is_long);
    if (lane < ns) {
      ws.pos[lane] = pos;
      ws.lo[lane] = (int32_t)lo;
      ws.len[lane] = used;
    }
    if (lane == ns - 1) ws.pos[ns] = incl;
    __syncwarp();
    const int T = ws.pos[ns];

    // ---- phase A: transform the chunk's values into shared memory, the raw
    //      values of kUA slots per lane loaded before any is transformed ----
    for (int k0 = 0; k0 < T; k0 += 32 * kUA) {
      int64_t raw[kUA];
      int bi[kUA];
#pragma unroll
      for (int u = 0; u < kUA; ++u) {
        const int k = k0 + u * 32 + lane;
        int i = 0;                           // last bag whose first slot is <= k
        raw[u] = 0;
        if (k < T) {
          for (int step = 16; step > 0; step >>= 1)
            if (i + step < ns && ws.pos[i + step] <= k) i += step;
          raw[u] = col_load(m, a.ids, a.fvals, (int64_t)ws.lo[i] + (k - ws.pos[i]));
        }
        bi[u] = i;
      }
      int32_t rowv[kUA];
      transform_batch(m, raw, rowv);
#pragma unroll
      for (int u = 0; u < kUA; ++u) {
        const int k = k0 + u * 32 + lane;
        if (k < T) {
          const int i = bi[u];
          const int32_t row = rowv[u];
          ws.rows[k] = row;
          ws.bag[k] = (uint8_t)i;
          if (a.rows_dbg || a.keys) {
            const int64_t t = (int64_t)ws.lo[i] + (k - ws.pos[i]);
            record<WT>(a, st, t, row, m, padded ? padded_gsrc(a, m, b0 + i, k - ws.pos[i]) : pooled_gsrc(a, m, b0 + i));
          }
        }
      }
    }
    if (padded && (a.rows_dbg || a.keys) && lane < ns && !is_long)
      for (int64_t t = lo + m.pad_len; t < hi; ++t) record_cut(a, st, t, m);
    if (m.trunc > 0 && (a.rows_dbg || a.keys)) {
      // values past a truncated bag's first trunc: no output, no gradient; the
      // whole warp writes their records, one cut bag at a time
      bool cutb = false;
      if (lane < ns) {
        bool bad = false;
        cutb = clamp_off(__ldg(offs + cur + lane + 1), n, bad) > hi;
      }
      for (unsigned cm = __ballot_sync(kFull, cutb); cm; cm &= cm - 1) {
        const int i = __ffs(cm) - 1;
        const int64_t t0 = __shfl_sync(kFull, hi, i);
        bool bad = false;
        const int64_t t1 = clamp_off(__ldg(offs + cur + i + 1), n, bad);
        for (int64_t t = t0 + lane; t < t1; t += 32) record_cut(a, st, t, m);
      }
    }
    __syncwarp();

    // ---- phase B: pool / copy ----
    const int glog = lanes_log2(m.dim4);
    const float* W = WT && m.pooling == EMB_POOL_SUM ? a.wts[st] : nullptr;   // value weights
    with_dtype<LP>(m.dtype, [&](auto dt) {
      constexpr int DT = decltype(dt)::value;
      if (padded) {
        if (m.dim4 > 32) warp_pad_chunk<2, DT>(a, ws, m, ns, b0, glog, longmask);
        else warp_pad_chunk<1, DT>(a, ws, m, ns, b0, glog, longmask);
      } else if (WT && W) {
        if (m.dim4 > 32) warp_pool_chunk<2, true, DT>(a, ws, m, W, ns, T, b0, glog, longmask);
        else warp_pool_chunk<1, true, DT>(a, ws, m, W, ns, T, b0, glog, longmask);
      } else {
        if (m.dim4 > 32) warp_pool_chunk<2, false, DT>(a, ws, m, W, ns, T, b0, glog, longmask);
        else warp_pool_chunk<1, false, DT>(a, ws, m, W, ns, T, b0, glog, longmask);
      }
    });

    // ---- phase C: long pooled bags of the chunk (long padded bags are
    //      copied by their pieces' tiles) ----
    for (unsigned lm = padded ? 0u : longmask; lm; lm &= lm - 1) {
      const int i = __ffs(lm) - 1;
      const int64_t blo = __shfl_sync(kFull, lo, i);
      const int64_t bhi = __shfl_sync(kFull, hi, i);
      with_dtype<LP>(m.dtype, [&](auto dt) {
        constexpr int DT = decltype(dt)::value;
        if (m.dim4 > 32) warp_long_bag<2, WT, DT>(a, st, m, W, b0 + i, blo, bhi, glog);
        else warp_long_bag<1, WT, DT>(a, st, m, W, b0 + i, blo, bhi, glog);
      });
    }
    __syncwarp();
    cur += ns;
  }
}

int forward_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_forward<false, false>, kFwdThreads, 0) != cudaSuccess) {
    cudaGetLastError();
    n = 4;
  }
  return n > 0 ? n : 1;
}

emb_status launch_forward(emb_plan_s* p, int32_t batch, const int64_t* ids, const int32_t* id_offsets,
                          const float* id_weights, int64_t n_ids, const float* fvals, const int32_t* f_offsets,
                          const float* f_weights, int64_t n_fvals, float* out, float* seq_out, int64_t* rows_dbg,
                          cudaStream_t stream) {
  if (batch == 0) return EMB_OK;
  FwdArgs a{};
  a.meta = p->meta_d;
  a.ids = ids;
  a.fvals = fvals;
  a.wts[0] = id_weights;
  a.wts[1] = f_weights;
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
    if (id_weights || f_weights) a.rec_src = p->ws.rec_src;
  }
  a.key_sentinel = p->key_total;
  a.status = p->status_d;
  // Schedule and tile size by the mean bag length (measured on the pooled,
  // training and sequence workloads): bags of a few values -> static, about
  // 16 tiles per resident warp, at least 256 values; long bags (a warp pools
  // one whole) -> dynamic, about 32 tiles per resident warp, at least 128.
  const int64_t total = n_ids + n_fvals;
  const int64_t warps = (int64_t)p->sm_count * p->fwd_ctas_per_sm * kFwdWarpsPerCta;
  const int64_t segs = (int64_t)batch * (p->n_stream_cols[0] + p->n_stream_cols[1]);
  a.dynamic = total > (int64_t)(kLongBag / 2) * std::max<int64_t>(segs, 1) ? 1 : 0;
  const int64_t want = total / std::max<int64_t>(1, (a.dynamic ? 32 : 16) * warps);
  int64_t E = a.dynamic ? 128 : 256;
  while (E < want && E < kMaxTileElems) E <<= 1;
  // A launch so small that its tiles would occupy under an eighth of the
  // resident warps (a few thousand values) takes smaller value tiles, down
  // to 32 values: each warp's chain of dependent loads is then one or two
  // chunks long instead of several.
  if (!a.dynamic)
    while (E > 32 && total / E < warps / 8) E >>= 1;
  a.tile_elems = (int32_t)E;
  // a stream whose columns are all long padded has no value tiles: its
  // pieces do all its work
  a.tiles[0] = a.ncols[0] > 0 && !p->long_padded_only[0] ? n_ids / E + 1 : 0;
  a.tiles[1] = a.ncols[1] > 0 && !p->long_padded_only[1] ? n_fvals / E + 1 : 0;
  if (p->n_long_padded > 0) {
    // pieces of about kPadPiece positions, as many per bag for every column
    // (at most 2^31 pieces in all)
    const int64_t bags = (int64_t)batch * p->n_long_padded;
    int64_t npc = (p->max_long_pad + kPadPiece - 1) / kPadPiece;
    npc = std::max<int64_t>(1, std::min<int64_t>(npc, INT32_MAX / bags));
    a.pad_tiles = bags * npc;
    a.pad_cols = p->pad_cols_d;
    a.pad_npc = (int32_t)npc;
    a.pad_ndiv = make_div_magic32((uint32_t)npc);
    a.pad_bdiv = make_div_magic32((uint32_t)(batch * npc));
  }
  if (!a.dynamic) {
    // Streams of short bags (mean length <= kShortBagMean): a tile is a run
    // of bags, about E values' worth rounded to whole 32-bag chunks, so its
    // ends need no search -- the search is a large share of the chain of
    // dependent loads such a small tile walks (measured on the inference,
    // one-value and dynamic workloads: 0.184 -> 0.175 ms, 0.224 -> 0.220 ms,
    // 0.220 -> 0.189 ms; 64-bag tiles were slower, 0.203 ms).  Longer bags
    // keep value tiles: there the search is cheap beside the gathers and
    // equal value counts per tile balance the warps (measured 4 % faster on
    // the training workload than tiles of bags).  A launch too small to
    // give every resident warp a tile keeps the smaller value tiles: there
    // the number of warps in flight decides (200 inference columns: 55.7 us
    // with value tiles, 65.3 us with 32-bag tiles).
    const int64_t nv[2] = {n_ids, n_fvals};
    int64_t k[2] = {0, 0}, t[2] = {a.tiles[0], a.tiles[1]};
    for (int st = 0; st < 2; ++st) {
      const int64_t S = (int64_t)batch * a.ncols[st];
      if (S == 0 || a.tiles[st] == 0 || nv[st] > kShortBagMean * S) continue;
      const int64_t kb = nv[st] > 0 ? E * S / nv[st] : kMaxTileBags;
      k[st] = std::min<int64_t>(std::max<int64_t>(kWarp, (kb + kWarp / 2) / kWarp * kWarp), kMaxTileBags);
      t[st] = (S + k[st] - 1) / k[st];
    }
    if ((k[0] || k[1]) && t[0] + t[1] >= warps) {
      for (int st = 0; st < 2; ++st) {
        a.tile_bags[st] = (int32_t)k[st];
        a.tiles[st] = t[st];
        // Tiles that split the batch evenly cover whole columns: deal them
        // column by column, widest stored rows first, so the longest tiles
        // start early and the launch does not end on them (inference
        // 0.175 -> 0.170 ms; a launch in stream order that ends on wide
        // columns leaves SMs idle while their last tiles run).
        if (k[st] > 0 && batch % k[st] == 0 && p->col_order_d) {
          a.col_order = p->col_order_d;
          a.tpc[st] = (int32_t)(batch / k[st]);
          a.tpc_div[st] = make_div_magic32((uint32_t)a.tpc[st]);
        }
      }
    }
  }
  const int64_t tiles = a.tiles[0] + a.tiles[1] + a.pad_tiles;
  if (tiles == 0) return EMB_OK;
  const int64_t resident = (int64_t)p->sm_count * p->fwd_ctas_per_sm;
  int64_t grid = (tiles + kFwdWarpsPerCta - 1) / kFwdWarpsPerCta;
  if (a.dynamic) grid = std::min<int64_t>(grid, resident);
  a.ticket = p->fwd_ticket;
  a.n_warps = grid * kFwdWarpsPerCta;
  const bool wt = a.wts[0] || a.wts[1];
  if (p->low_precision) {
    if (wt) k_forward<true, true><<<(unsigned)grid, kFwdThreads, 0, stream>>>(a);
    else k_forward<false, true><<<(unsigned)grid, kFwdThreads, 0, stream>>>(a);
  } else {
    if (wt) k_forward<true, false><<<(unsigned)grid, kFwdThreads, 0, stream>>>(a);
    else k_forward<false, false><<<(unsigned)grid, kFwdThreads, 0, stream>>>(a);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace emb
