// atomic.cu -- K-B atomic: the backward the RecIS page gives (§3.2,
// Algorithm 1, backward: identical destination rows merged inside a wave, then
// global atomics, no sort), as a second backward beside the sort-based one,
// selected per plan with EMB_PLAN_ATOMIC_BACKWARD.
//
// A dense gradient over every table row does not fit beside large tables
// (weights and accumulators of the 200-column training tables take 97 GB
// each), so the atomics land in a compact gradient with one row per touched
// table row, found through a row -> slot map:
//   1. k_atomic_mark    -- each valid contribution sets its row's bit in a
//                          bitmap over all global rows (read first, set only
//                          when clear);
//   2. k_bits_count / k_rank_top / k_bits_emit
//                       -- the set bits become the ascending list of touched
//                          rows; each row's slot is its rank (slot_of), and
//                          the bitmap is cleared on the way;
//   3. k_atomic_scatter -- warps take 32 contributions at a time, group equal
//                          rows (match.any), lay the groups out contiguously
//                          in shared memory, and lane groups of dim/4 lanes
//                          walk equal ranges summing scale * G rows per row
//                          and adding each sum to the row's compact gradient
//                          with 16-byte vector atomics;
//   4. k_atomic_update  -- one lane group per touched row: read and clear its
//                          compact gradient row, one Adagrad step on W and acc.
// The atomics make the summation order depend on scheduling, so results are
// not bit-identical run to run (they stay within the fp32 summation bound).
#include <algorithm>

#include "plan.cuh"
#include "update.cuh"

namespace emb {

// exclusive scan of per-block counts, defined with the run-rank kernels of
// the sort-based backward
__global__ void k_rank_top(uint32_t* part, int nb, int64_t* n_unique);

namespace {

constexpr int kBitsBlock = 1024;     // bitmap words per counting / emitting block
constexpr int kAtomThreads = 256;
constexpr int kAtomU = 8;            // gradient rows in flight per lane (halved for two float4 per lane)
constexpr uint32_t kNoSlot = 0xffffffffu;
constexpr uint32_t kOffPadA = 0x80000000u;   // compact source offset: into the padded gradient

struct AtomArgs {
  const uint32_t* keys;
  const uint32_t* vals;
  const uint2* rec_src;    // weighted forwards: (gradient source, weight bits) per record
  int64_t n;
  uint32_t sentinel;
  const int4* colg;
  const float* inv_n;
  const float* grad_out;
  int64_t ldg;
  const float* grad_seq;
  DivMagic32 bdiv;
  int32_t batch;
  const TableMeta* tables;
  const uint32_t* table_base;
  int32_t n_tables;
  uint32_t* touched;       // bitmap over global rows
  uint32_t* slot_of;       // global row -> compact slot (valid for touched rows)
  const uint32_t* uniq;    // slot -> global row, ascending
  const int64_t* n_uniq;
  float* cgrad;            // [slots, cld] compact gradient
  int32_t cld;
  uint32_t* ucount;        // contributions per slot, or null
  float lr, eps;
  int32_t glog;
  // debug outputs
  int32_t* dbg_table;
  int64_t* dbg_row;
  int32_t* dbg_count;
  float* dbg_grad;
  int32_t dbg_ld;
};

__global__ void k_atomic_mark(const uint32_t* __restrict__ keys, int64_t n, uint32_t sentinel,
                              uint32_t* touched) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t k = __ldg(keys + i);
    if (k == sentinel) continue;
    const uint32_t bit = 1u << (k & 31);
    uint32_t* wp = touched + (k >> 5);
    if (!(__ldcg(wp) & bit)) atomicOr(wp, bit);
  }
}

__global__ void __launch_bounds__(kBitsBlock) k_bits_count(const uint32_t* touched, int64_t words, uint32_t* part) {
  __shared__ uint32_t wsum[32];
  const int64_t i = blockIdx.x * (int64_t)kBitsBlock + threadIdx.x;
  uint32_t c = i < words ? (uint32_t)__popc(__ldcg(touched + i)) : 0u;
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t t = wsum[threadIdx.x];
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
    if (threadIdx.x == 0) part[blockIdx.x] = t;
  }
}

// Slots in ascending row order: slot = rank of the row among the set bits.
__global__ void __launch_bounds__(kBitsBlock) k_bits_emit(uint32_t* touched, int64_t words, const uint32_t* part,
                                                          uint32_t* uniq, uint32_t* slot_of) {
  __shared__ uint32_t wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i = blockIdx.x * (int64_t)kBitsBlock + threadIdx.x;
  uint32_t bits = i < words ? __ldcg(touched + i) : 0u;
  const uint32_t v = (uint32_t)__popc(bits);
  uint32_t x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  uint32_t slot = part[blockIdx.x] + x - v;
  for (int w = 0; w < warp; ++w) slot += wsum[w];
  if (bits) {
    touched[i] = 0u;
    while (bits) {
      const uint32_t key = (uint32_t)(i << 5) + (uint32_t)(__ffs(bits) - 1);
      uniq[slot] = key;
      slot_of[key] = slot;
      ++slot;
      bits &= bits - 1;
    }
  }
}

struct __align__(16) AtomRec {
  uint32_t slot;    // compact gradient row (kNoSlot: dropped contribution)
  uint32_t off;     // float4 offset of the gradient row (kOffPadA: in the padded gradient)
  float scale;
  uint32_t d4;
};

// Contribution i's gradient row: float4 offset, scale and width (the
// decoding the sort-based backward applies to its sorted entries).
__device__ __forceinline__ void atom_decode(const AtomArgs& a, uint32_t key, uint32_t val, AtomRec& r,
                                            uint32_t& lkey, int& ld4) {
  float wr = 1.0f;
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
    r.off = kOffPadA | (val & ~kPadBit);
  } else {
    const uint32_t c = div_magic32(val, a.bdiv);
    const uint32_t b = val - c * (uint32_t)a.batch;
    const int4 cg = __ldg(a.colg + c);
    r.scale = cg.y ? __ldg(a.inv_n + val) : wr;
    r.d4 = (uint32_t)cg.z;
    r.off = (uint32_t)(((int64_t)b * a.ldg + cg.x) >> 2);
  }
}

template <int V>
__device__ __forceinline__ void atom_flush(const AtomArgs& a, uint32_t slot, uint32_t d4, const float4 (&acc)[V],
                                           int cnt, int sub) {
  float* dst = a.cgrad + (int64_t)slot * a.cld;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int f4 = sub + v * 32;
    if (f4 < (int)d4) atomicAdd(reinterpret_cast<float4*>(dst + f4 * 4), acc[v]);
  }
  if (a.ucount && sub == 0) atomicAdd(a.ucount + slot, (uint32_t)cnt);
}

template <int V>
__global__ void __launch_bounds__(kAtomThreads) k_atomic_scatter(const AtomArgs a) {
  constexpr int U = kAtomU / V;
  __shared__ AtomRec srec[kAtomThreads];
  const int lane = threadIdx.x & 31;
  AtomRec* wr = srec + (threadIdx.x & ~31);
  const int glog = a.glog;
  const int G = 32 >> glog;
  const int q = lane >> glog, sub = lane & ((1 << glog) - 1);
  const int R = 32 / G;   // grouped entries per lane group
  uint32_t lkey = 0xffffffffu;
  int ld4 = 0;
  const int64_t stride = (int64_t)gridDim.x * kAtomThreads;
  for (int64_t base = (int64_t)blockIdx.x * kAtomThreads + (threadIdx.x & ~31); base < a.n; base += stride) {
    const int64_t i = base + lane;
    AtomRec r;
    r.slot = kNoSlot;
    r.off = 0u;
    r.scale = 0.0f;
    r.d4 = 0u;
    uint32_t key = a.sentinel;
    if (i < a.n) {
      key = __ldg(a.keys + i);
      const uint32_t val = __ldg(a.vals + i);
      if (key != a.sentinel) {
        r.slot = __ldg(a.slot_of + key);   // in flight with the decoding loads
        atom_decode(a, key, val, r, lkey, ld4);
      }
    }
    // equal rows of the 32 contributions: groups ordered by their first lane,
    // members by lane
    const unsigned peers = __match_any_sync(kFull, key);
    const int leader = __ffs(peers) - 1;
    const int gsize = leader == lane ? __popc(peers) : 0;
    int incl = gsize;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    const int gstart = __shfl_sync(kFull, incl - gsize, leader);
    wr[gstart + __popc(peers & ((1u << lane) - 1u))] = r;
    __syncwarp();

    // lane group q walks entries [q R, q R + R), U gradient rows in flight;
    // a sum is added to the compact gradient where its row ends or the range does
    float4 acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t cslot = kNoSlot, cd4 = 0;
    int cnt = 0;
    for (int j = 0; j < R; j += U) {
      float4 g[U][V];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const AtomRec e = j + u < R ? wr[q * R + j + u] : AtomRec{kNoSlot, 0u, 0.0f, 0u};
        const bool ok = e.slot != kNoSlot;
        const float* src = (e.off & kOffPadA) ? a.grad_seq + (int64_t)(e.off & ~kOffPadA) * 4
                                              : a.grad_out + (int64_t)e.off * 4;
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const int f4 = sub + v * 32;
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (ok && f4 < (int)e.d4) x = __ldg(reinterpret_cast<const float4*>(src + f4 * 4));
          g[u][v] = make_float4(e.scale * x.x, e.scale * x.y, e.scale * x.z, e.scale * x.w);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (j + u >= R) break;
        const AtomRec& e = wr[q * R + j + u];
        if (e.slot != cslot) {
          if (cslot != kNoSlot) atom_flush<V>(a, cslot, cd4, acc, cnt, sub);
          cslot = e.slot;
          cd4 = e.d4;
          cnt = 0;
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        ++cnt;
#pragma unroll
        for (int v = 0; v < V; ++v) {
          acc[v].x += g[u][v].x;
          acc[v].y += g[u][v].y;
          acc[v].z += g[u][v].z;
          acc[v].w += g[u][v].w;
        }
      }
    }
    if (cslot != kNoSlot) atom_flush<V>(a, cslot, cd4, acc, cnt, sub);
    __syncwarp();
  }
}

// One lane group per touched row (slots ascend with the rows, so a group's
// consecutive slots mostly stay in one table).
template <int V>
__global__ void __launch_bounds__(256) k_atomic_update(const AtomArgs a) {
  const int lane = threadIdx.x & 31;
  const int glog = a.glog;
  const int sub = lane & ((1 << glog) - 1);
  const int64_t groups = (int64_t)gridDim.x * (blockDim.x >> glog);
  const int64_t nu = *a.n_uniq;
  int t = -1;
  uint32_t tbase = 0, tnext = 0;
  TableMeta tm{};
  for (int64_t u = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> glog; u < nu; u += groups) {
    const uint32_t key = __ldg(a.uniq + u);
    if (t < 0 || key < tbase || key >= tnext) {
      t = table_of_key(a.table_base, a.n_tables, key);
      tbase = __ldg(a.table_base + t);
      tnext = __ldg(a.table_base + t + 1);
      tm = a.tables[t];
    }
    const int64_t row = key - tbase;
    float* gsrc = a.cgrad + u * a.cld;
    float* W = tm.weight + row * tm.dim;
    float* A = tm.acc + row * tm.dim;
    float4 g[V], w[V], ac[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      if (f4 < tm.dim4) {
        g[v] = __ldcg(reinterpret_cast<const float4*>(gsrc + f4 * 4));
        w[v] = *reinterpret_cast<const float4*>(W + f4 * 4);
        ac[v] = *reinterpret_cast<const float4*>(A + f4 * 4);
      }
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int f4 = sub + v * 32;
      if (f4 < tm.dim4) {
        adagrad1_fast(w[v].x, ac[v].x, g[v].x, a.lr, a.eps);
        adagrad1_fast(w[v].y, ac[v].y, g[v].y, a.lr, a.eps);
        adagrad1_fast(w[v].z, ac[v].z, g[v].z, a.lr, a.eps);
        adagrad1_fast(w[v].w, ac[v].w, g[v].w, a.lr, a.eps);
        *reinterpret_cast<float4*>(W + f4 * 4) = w[v];
        *reinterpret_cast<float4*>(A + f4 * 4) = ac[v];
        *reinterpret_cast<float4*>(gsrc + f4 * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.dbg_grad) *reinterpret_cast<float4*>(a.dbg_grad + u * a.dbg_ld + f4 * 4) = g[v];
      }
    }
    if (sub == 0) {
      if (a.dbg_table) a.dbg_table[u] = t;
      if (a.dbg_row) a.dbg_row[u] = row;
      if (a.ucount) {
        if (a.dbg_count) a.dbg_count[u] = (int32_t)a.ucount[u];
        a.ucount[u] = 0u;
      }
    }
  }
}

}  // namespace

emb_status launch_backward_atomic(emb_plan_s* p, const float* grad_out, const float* grad_seq, float lr, float eps,
                                  cudaStream_t stream, const emb_backward_debug* dbg) {
  Workspace& w = p->ws;
  const int64_t n = p->last_n;
  if (n == 0) {
    if (dbg && dbg->n_unique) EMB_CUDA_TRY(cudaMemsetAsync(dbg->n_unique, 0, sizeof(int64_t), stream));
    return EMB_OK;
  }
  const int64_t words = ((int64_t)p->key_total + 31) / 32;
  const int nb = (int)((words + kBitsBlock - 1) / kBitsBlock);
  const int sms = p->sm_count;
  k_atomic_mark<<<sms * 8, 256, 0, stream>>>(w.keys[0], n, p->key_total, w.touched);
  k_bits_count<<<nb, kBitsBlock, 0, stream>>>(w.touched, words, w.bit_part);
  k_rank_top<<<1, 1024, 0, stream>>>(w.bit_part, nb, w.n_uniq);
  k_bits_emit<<<nb, kBitsBlock, 0, stream>>>(w.touched, words, w.bit_part, w.uniq, w.slot_of);

  AtomArgs a{};
  a.keys = w.keys[0];
  a.vals = w.vals[0];
  a.rec_src = p->last_weighted ? w.rec_src : nullptr;
  a.n = n;
  a.sentinel = p->key_total;
  a.colg = p->colg_d;
  a.inv_n = w.inv_n;
  a.grad_out = grad_out;
  a.ldg = p->out_width;
  a.grad_seq = grad_seq;
  a.batch = p->last_batch > 0 ? p->last_batch : 1;
  a.bdiv = make_div_magic32((uint32_t)a.batch);
  a.tables = p->tables_d;
  a.table_base = p->table_base_d;
  a.n_tables = p->n_tables;
  a.touched = w.touched;
  a.slot_of = w.slot_of;
  a.uniq = w.uniq;
  a.n_uniq = w.n_uniq;
  a.cgrad = w.cgrad;
  a.cld = p->max_dim;
  const bool want_count = dbg && dbg->counts;
  a.ucount = want_count ? w.ucount : nullptr;
  a.lr = lr;
  a.eps = eps;
  const int maxdim4 = p->max_dim / 4;
  int g = maxdim4 > 32 ? 32 : maxdim4, glog = 0;
  while ((1 << glog) < g) ++glog;
  a.glog = glog;
  if (dbg) {
    a.dbg_table = dbg->uniq_table;
    a.dbg_row = dbg->uniq_row;
    a.dbg_count = dbg->counts;
    a.dbg_grad = dbg->agg_grad;
    a.dbg_ld = p->max_dim;
  }
  const int64_t warps = (n + 31) / 32;
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>((warps + 7) / 8, (int64_t)sms * 64));
  const unsigned ugrid = (unsigned)(sms * 8);
  if (maxdim4 > 32) {
    k_atomic_scatter<2><<<grid, kAtomThreads, 0, stream>>>(a);
    k_atomic_update<2><<<ugrid, 256, 0, stream>>>(a);
  } else {
    k_atomic_scatter<1><<<grid, kAtomThreads, 0, stream>>>(a);
    k_atomic_update<1><<<ugrid, 256, 0, stream>>>(a);
  }
  if (dbg && dbg->n_unique)
    EMB_CUDA_TRY(cudaMemcpyAsync(dbg->n_unique, w.n_uniq, sizeof(int64_t), cudaMemcpyDeviceToDevice, stream));
  return cuda_status(cudaGetLastError());
}

}  // namespace emb
