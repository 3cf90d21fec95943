// radix.cuh -- stable LSD radix sort of (key, u32 value) pairs, 8-bit digits
// (the kernels take the digit width as a parameter; sort_plan picks it): a
// single read of the keys builds the digit histograms of all
// passes, then each pass is one chained-scan scatter kernel in which a CTA
// ranks its tile in shared memory, publishes its per-digit counts and finds
// its global offsets by decoupled look-back over the earlier tiles (Adinets &
// Merrill, "Onesweep: a faster least significant digit radix sort for GPUs",
// 2022).  Tiles are taken in launch order from a ticket counter, so a CTA
// only ever waits on CTAs that are already running; every wait is bounded and
// latches EMB_ERR_TIMEOUT instead of hanging.  A tile whose wait gave up has
// no valid output offsets: it also raises the sort's fail word (in its
// scratch, cleared by each sort), and kernels that consume the sorted pairs
// check that word and do nothing when it is set, since the output then has
// holes holding an earlier call's pairs.
//
// The element count may live in device memory (n_dev != nullptr): grids are
// then sized for the capacity, the count is clamped to it and tiles past the
// count do nothing.
#pragma once

#include <type_traits>

#include "plan.cuh"

namespace emb {

constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagInc = 2u << 30;
constexpr uint32_t kCountMask = (1u << 30) - 1;
constexpr int kSpinLimit = 1 << 22;
constexpr int kLookWin = 8;   // look-back words loaded per round trip
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kMaxSortPasses = 8;

template <class K>
struct SortItems;
template <>
struct SortItems<uint32_t> {
  static constexpr int value = kSortItems;
};
template <>
struct SortItems<uint64_t> {
  static constexpr int value = 8;
};

template <class K>
constexpr int sort_tile() {
  return kSortThreads * SortItems<K>::value;
}

template <class K, int BITS>
struct SortSmemT {
  static constexpr int kR = 1 << BITS;
  static constexpr int kTile = sort_tile<K>();
  // per-warp digit counts, then slots: at most kTile, so 16 bits hold them
  using Count = typename std::conditional<(BITS > 8), uint16_t, uint32_t>::type;
  K keys[kTile];
  uint32_t vals[kTile];
  Count whist[kSortWarps][kR];         // per-warp digit counts, then each warp's first slot
  uint32_t dstart[kR];                 // first slot of each digit inside the tile
  uint32_t goff[kR];                   // output position of shared slot j of a digit, minus j
  uint32_t hscan[kR];                  // exclusive scan of the pass histogram
  uint32_t wsum[kSortWarps];
  uint32_t tile;
};

// Digit width and number of passes for keys of key_bits bits.  8-bit digits:
// measured on 41.75 M training pairs of 30-bit keys, three passes of 10-bit
// digits (1024 bins, 7.5 pairs per bin and tile) took 1.44 ms against 1.21 ms
// for four passes of 8-bit digits -- the per-tile digit work and the shorter
// output runs cost more than the pass saved.  32-bit keys of 25 to 27 bits
// take three passes of 9-bit digits instead of four passes of which the
// last would sort three bits or fewer.
template <class K>
inline void sort_plan(int key_bits, int* bits, int* passes) {
  const int kb = key_bits < 1 ? 1 : key_bits;
  if (sizeof(K) == 4 && kb > 24 && kb <= 27) {
    *bits = 9;
    *passes = 3;
    return;
  }
  *bits = 8;
  *passes = (kb + 7) / 8;
}

// Element count: n, or the count in device memory clamped to the capacity n.
__device__ __forceinline__ int64_t sort_count(int64_t n, const uint32_t* n_dev) {
  if (!n_dev) return n;
  const int64_t c = (int64_t)*((volatile const uint32_t*)n_dev);
  return c < n ? c : n;
}

template <class K, int BITS>
__device__ __forceinline__ uint32_t sort_digit(K k, int shift) {
  return (uint32_t)(k >> shift) & (uint32_t)((1 << BITS) - 1);
}

// Digit histograms of all passes in one read of the keys.
template <class K, int BITS>
__global__ void __launch_bounds__(512) k_digit_hist_t(const K* __restrict__ keys, int64_t n0,
                                                      const uint32_t* n_dev, int passes,
                                                      uint32_t* __restrict__ hist) {
  constexpr int R = 1 << BITS;
  __shared__ uint32_t h[kMaxSortPasses * R];
  const int64_t n = sort_count(n0, n_dev);
  for (int i = threadIdx.x; i < passes * R; i += blockDim.x) h[i] = 0;
  __syncthreads();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const K k = keys[i];
    for (int p = 0; p < passes; ++p) atomicAdd(&h[p * R + sort_digit<K, BITS>(k, p * BITS)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < passes * R; i += blockDim.x)
    if (h[i]) atomicAdd(&hist[i], h[i]);
}

// Lanes of the warp holding the same digit d, found with one ballot per digit
// bit: the mask starts full and each ballot keeps the lanes that agree with
// this lane on that bit.  All lanes must call.
template <int NB>
__device__ __forceinline__ unsigned warp_match_digit(uint32_t d) {
  unsigned peers = kFull;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const unsigned m = __ballot_sync(kFull, (d >> b) & 1u);
    peers &= ((d >> b) & 1u) ? m : ~m;
  }
  return peers;
}

// Exclusive scan of R per-digit values over the CTA: thread t holds the
// values of digits t*PER .. t*PER+PER-1 in v[] (PER = R / kSortThreads, at
// least 1; threads past the last digit hold zeros).  All threads call.
template <int R>
__device__ __forceinline__ void sort_scan_digits(uint32_t (&v)[(R + kSortThreads - 1) / kSortThreads],
                                                 uint32_t* wsum) {
  constexpr int PER = (R + kSortThreads - 1) / kSortThreads;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t tot = 0;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const uint32_t c = v[q];
    v[q] = tot;   // exclusive within the thread
    tot += c;
  }
  uint32_t x = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  uint32_t base = 0;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  __syncthreads();
  base += x - tot;
#pragma unroll
  for (int q = 0; q < PER; ++q) v[q] += base;
}

// One tile of a pass: rank the items by digit within the tile (stable: warp
// order, then item order, then lane order), publish the tile's digit counts,
// place the items in shared memory in digit order, find the tile's global
// digit offsets by look-back, write out.  The lanes holding the same digit
// are found by one ballot per digit bit on a full tile's first pass and by
// one match.any otherwise: match.any takes longer the more distinct values a
// warp holds, and the lowest digit of keys in their input order is close to
// uniform, while the later passes see runs of repeated (Zipf-hot) keys and a
// partial tile's missing items all hold the marker digit R (measured on the
// training, sequence and tiny workloads).  FULL: the tile holds TILE items
// (no per-item bounds).
template <class K, int BITS>
__device__ __forceinline__ void onesweep_tile(SortSmemT<K, BITS>& sm, const K* __restrict__ kin,
                                              const uint32_t* __restrict__ vin, K* __restrict__ kout,
                                              uint32_t* __restrict__ vout, uint32_t n, uint32_t t, int tile_n,
                                              int shift, uint32_t* lookback, uint32_t* status, uint32_t* fail) {
  using Count = typename SortSmemT<K, BITS>::Count;
  constexpr int R = 1 << BITS;
  constexpr int PER = (R + kSortThreads - 1) / kSortThreads;   // digits per thread
  constexpr int ITEMS = SortItems<K>::value;
  constexpr int TILE = sort_tile<K>();
  const bool FULL = tile_n == TILE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int w0 = warp * 32 * ITEMS;            // the warp's first item in the tile
  const K* wk = kin + (size_t)t * TILE + w0;
  const uint32_t* wv = vin + (size_t)t * TILE + w0;

  K k[ITEMS];
  uint32_t v[ITEMS];
  uint32_t r2[(ITEMS + 1) / 2];   // in-warp ranks (< 2^16), two per register
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int o = i * 32 + lane;
    const bool ok = FULL || w0 + o < tile_n;
    k[i] = ok ? wk[o] : (K)0;
    v[i] = ok ? wv[o] : 0u;
  }
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const bool ok = FULL || w0 + i * 32 + lane < tile_n;
    const uint32_t d = ok ? sort_digit<K, BITS>(k[i], shift) : (uint32_t)R;
    const unsigned peers = (FULL && shift == 0) ? warp_match_digit<BITS>(d) : __match_any_sync(kFull, d);
    const int leader = 31 - __clz(peers);
    uint32_t old = 0;
    if (lane == leader && ok) {
      old = sm.whist[warp][d];
      sm.whist[warp][d] = (Count)(old + __popc(peers));
    }
    old = __shfl_sync(kFull, old, leader);
    __syncwarp();   // the counter update is seen by the next item's leader
    const uint32_t rank = old + __popc(peers & lt);
    if (i & 1) r2[i >> 1] |= rank << 16;
    else r2[i >> 1] = rank;
  }
  __syncthreads();

  // per digit: warp offsets, the tile's count (published at once), the
  // digit's first slot in the tile
  const int d0 = tid * PER;
  uint32_t cnt[PER], ds[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int d = d0 + q;
    uint32_t c = 0;
    if (d < R) {
      for (int w = 0; w < kSortWarps; ++w) {
        const uint32_t x = sm.whist[w][d];
        sm.whist[w][d] = (Count)c;
        c += x;
      }
      *(volatile uint32_t*)(lookback + (size_t)t * R + d) = (t == 0 ? kFlagInc : kFlagAgg) | c;
    }
    cnt[q] = c;
    ds[q] = c;
  }
  sort_scan_digits<R>(ds, sm.wsum);
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int d = d0 + q;
    if (d < R) {
      sm.dstart[d] = ds[q];
      for (int w = 0; w < kSortWarps; ++w)   // slot of each warp's first item of the digit
        sm.whist[w][d] = (Count)(sm.whist[w][d] + ds[q]);
    }
  }
  __syncthreads();
  // the tile's items into shared memory in digit order; this frees their
  // registers before the look-back below
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    if (FULL || w0 + i * 32 + lane < tile_n) {
      const uint32_t rank = (i & 1) ? r2[i >> 1] >> 16 : r2[i >> 1] & 0xffffu;
      const uint32_t pos = sm.whist[warp][sort_digit<K, BITS>(k[i], shift)] + rank;
      sm.keys[pos] = k[i];
      sm.vals[pos] = v[i];
    }
  }
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int d = d0 + q;
    if (d >= R) continue;
    uint32_t excl = 0;
    if (t > 0) {
      // Walk back kLookWin predecessors per round trip: their words are
      // loaded together, then taken newest first, summing aggregates up to
      // the first inclusive prefix.  A word not yet published stops the
      // round; the next round starts at it.  Tile 0 always publishes an
      // inclusive prefix, so the walk never passes it.
      int64_t j = (int64_t)t - 1;
      int spins = 0;
      bool done = false;
      while (!done) {
        uint32_t w[kLookWin];
#pragma unroll
        for (int z = 0; z < kLookWin; ++z)
          w[z] = j - z >= 0 ? *(volatile const uint32_t*)(lookback + (j - z) * R + d) : kFlagInc;
        int z = 0;
#pragma unroll
        for (int zz = 0; zz < kLookWin; ++zz) {
          if (z == zz) {
            const uint32_t flag = w[zz] & ~kCountMask;
            if (flag != 0u) {
              excl += w[zz] & kCountMask;
              if (flag == kFlagInc) done = true;
              else ++z;
            }
          }
        }
        if (done) break;
        j -= z;
        if (z < kLookWin) {   // word j is not published yet
          if (++spins > kSpinLimit) {
            latch(status, EMB_ERR_TIMEOUT);
            *(volatile uint32_t*)fail = 1u;
            break;
          }
          __nanosleep(32);
        }
      }
      *(volatile uint32_t*)(lookback + (size_t)t * R + d) = kFlagInc | ((excl + cnt[q]) & kCountMask);
    }
    // output position of shared slot j of this digit: goff + (j - dstart)
    sm.goff[d] = sm.hscan[d] + excl - ds[q];
  }
  __syncthreads();
  for (int j = tid; j < (FULL ? TILE : tile_n); j += kSortThreads) {
    const K key = sm.keys[j];
    const uint32_t o = sm.goff[sort_digit<K, BITS>(key, shift)] + (uint32_t)j;
    if (o < n) {   // always true unless a look-back wait gave up
      kout[o] = key;
      vout[o] = sm.vals[j];
    }
  }
}

// One tile per CTA (PERSIST = false; the grid covers the tiles), or
// persistent CTAs that take tiles in ticket order until none is left
// (PERSIST = true, for counts that live on the device: the grid is sized for
// the capacity, and CTAs past the count cost one ticket each).  Either way a
// tile only ever waits on tiles whose tickets were drawn earlier, by CTAs
// already running.
template <class K, int BITS, bool PERSIST>
__global__ void __launch_bounds__(kSortThreads, 2)
    k_onesweep_t(const K* __restrict__ kin, const uint32_t* __restrict__ vin, K* __restrict__ kout,
                 uint32_t* __restrict__ vout, int64_t n0, const uint32_t* n_dev, int shift,
                 const uint32_t* __restrict__ hist, uint32_t* lookback, uint32_t* tile_ctr, uint32_t* status,
                 uint32_t* fail) {
  constexpr int R = 1 << BITS;
  constexpr int PER = (R + kSortThreads - 1) / kSortThreads;
  constexpr int TILE = sort_tile<K>();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SortSmemT<K, BITS>& sm = *reinterpret_cast<SortSmemT<K, BITS>*>(smem_raw);
  const int tid = threadIdx.x;
  const int64_t n = sort_count(n0, n_dev);
  const int64_t tiles = (n + TILE - 1) / TILE;
  {
    uint32_t hv[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) hv[q] = tid * PER + q < R ? __ldg(hist + tid * PER + q) : 0u;
    sort_scan_digits<R>(hv, sm.wsum);
#pragma unroll
    for (int q = 0; q < PER; ++q)
      if (tid * PER + q < R) sm.hscan[tid * PER + q] = hv[q];
  }
  do {
    if (tid == 0) sm.tile = atomicAdd(tile_ctr, 1u);
    for (int i = tid; i < kSortWarps * R; i += kSortThreads) (&sm.whist[0][0])[i] = 0;
    __syncthreads();
    const uint32_t t = sm.tile;
    if ((int64_t)t >= tiles) return;   // past the data: nobody waits on this ticket
    const int64_t left = n - (int64_t)t * TILE;
    onesweep_tile<K, BITS>(sm, kin, vin, kout, vout, (uint32_t)n, t, left >= TILE ? TILE : (int)left, shift,
                           lookback, status, fail);
    if (PERSIST) __syncthreads();   // the tile's shared memory is free again
  } while (PERSIST);
}

// A sort whose pairs fit one tile, all passes in one CTA (small steps, where
// the separate histogram and pass launches cost more than the work): each
// pass counts its digits in shared memory, scans them and ranks and
// scatters the tile as tile 0, which publishes its counts and never waits.
// At most two passes: each buffer is then read at most once after it was
// written in this kernel (the ranking reads its input through the
// read-only path, which must not see a line cached before the write).
template <class K, int BITS>
__global__ void __launch_bounds__(kSortThreads, 1)
    k_sort_one_tile(K* k0, uint32_t* v0, K* k1, uint32_t* v1, int n, int passes, uint32_t* lookback,
                    uint32_t* status, uint32_t* fail) {
  constexpr int R = 1 << BITS;
  constexpr int PER = (R + kSortThreads - 1) / kSortThreads;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SortSmemT<K, BITS>& sm = *reinterpret_cast<SortSmemT<K, BITS>*>(smem_raw);
  const int tid = threadIdx.x;
  pdl_trigger();   // the run reduction launched after this sort may be scheduled
  if (tid == 0) *(volatile uint32_t*)fail = 0u;   // no wait here can run out
  for (int p = 0; p < passes; ++p) {
    const K* kin = (p & 1) ? k1 : k0;
    const uint32_t* vin = (p & 1) ? v1 : v0;
    K* kout = (p & 1) ? k0 : k1;
    uint32_t* vout = (p & 1) ? v0 : v1;
    for (int i = tid; i < R; i += kSortThreads) sm.hscan[i] = 0u;
    for (int i = tid; i < kSortWarps * R; i += kSortThreads) (&sm.whist[0][0])[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kSortThreads) atomicAdd(&sm.hscan[sort_digit<K, BITS>(kin[i], p * BITS)], 1u);
    __syncthreads();
    uint32_t hv[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) hv[q] = tid * PER + q < R ? sm.hscan[tid * PER + q] : 0u;
    sort_scan_digits<R>(hv, sm.wsum);
#pragma unroll
    for (int q = 0; q < PER; ++q)
      if (tid * PER + q < R) sm.hscan[tid * PER + q] = hv[q];
    __syncthreads();
    onesweep_tile<K, BITS>(sm, kin, vin, kout, vout, (uint32_t)n, 0u, n, p * BITS, lookback, status, fail);
    __syncthreads();   // this pass's output is complete (and visible to the block) before the next reads it
  }
}

// Words of scratch the sort of keys with key_bits bits needs for cap pairs:
// hist [passes][R], tickets [passes], the fail word, look-back words
// [passes][tiles][R].
template <class K>
inline size_t sort_scratch_words(int key_bits, int64_t cap) {
  int bits = 8, passes = 1;
  sort_plan<K>(key_bits, &bits, &passes);
  const size_t R = (size_t)1 << bits;
  const int64_t tiles = (cap + sort_tile<K>() - 1) / sort_tile<K>();
  return (size_t)passes * R + passes + 1 + (size_t)passes * tiles * R;
}

// The fail word inside a sort's scratch: nonzero after a sort in which a
// look-back wait gave up (its output is then incomplete).
template <class K>
inline uint32_t* sort_fail_word(uint32_t* scratch, int key_bits) {
  int bits = 8, passes = 1;
  sort_plan<K>(key_bits, &bits, &passes);
  return scratch + (size_t)passes * ((size_t)1 << bits) + passes;
}

template <class K, int BITS>
inline emb_status radix_sort_passes(K* const keys[2], uint32_t* const vals[2], int64_t n, const uint32_t* n_dev,
                                    int64_t cap, int passes, uint32_t* scratch, int sm_count, uint32_t* status,
                                    cudaStream_t stream) {
  constexpr int R = 1 << BITS;
  const int64_t tiles = (cap + sort_tile<K>() - 1) / sort_tile<K>();
  uint32_t* hist = scratch;
  uint32_t* tickets = hist + (size_t)passes * R;
  uint32_t* fail = tickets + passes;
  uint32_t* lookback = fail + 1;
  const int hgrid = (int)std::min<int64_t>((cap + 511) / 512, (int64_t)sm_count * 4);
  k_digit_hist_t<K, BITS><<<hgrid, 512, 0, stream>>>(keys[0], n, n_dev, passes, hist);
  const bool persist = n_dev != nullptr;
  const int64_t grid = persist ? std::min<int64_t>(tiles, (int64_t)sm_count * 2) : tiles;   // two CTAs fit an SM
  const int smem = (int)sizeof(SortSmemT<K, BITS>);
  EMB_CUDA_TRY(cudaFuncSetAttribute(k_onesweep_t<K, BITS, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    smem));
  EMB_CUDA_TRY(cudaFuncSetAttribute(k_onesweep_t<K, BITS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    smem));
  for (int ps = 0; ps < passes; ++ps) {
    const int in = ps & 1, out = in ^ 1;
    if (persist)
      k_onesweep_t<K, BITS, true><<<(unsigned)grid, kSortThreads, smem, stream>>>(
          keys[in], vals[in], keys[out], vals[out], n, n_dev, ps * BITS, hist + ps * R,
          lookback + (size_t)ps * tiles * R, tickets + ps, status, fail);
    else
      k_onesweep_t<K, BITS, false><<<(unsigned)grid, kSortThreads, smem, stream>>>(
          keys[in], vals[in], keys[out], vals[out], n, n_dev, ps * BITS, hist + ps * R,
          lookback + (size_t)ps * tiles * R, tickets + ps, status, fail);
  }
  return EMB_OK;
}

// Sorts keys[0]/vals[0] (n pairs, or *n_dev of at most cap) by their low
// key_bits bits into keys[p&1], vals[p&1] with p = the number of passes.
// `scratch` holds sort_scratch_words<K>(key_bits, cap) words and is cleared
// here (fail word included: sort_fail_word reads as 0 unless a wait of this
// sort gave up).  Returns the index of the buffer holding the result.
template <class K>
inline emb_status radix_sort_pairs(K* const keys[2], uint32_t* const vals[2], int64_t n, const uint32_t* n_dev,
                                   int64_t cap, int key_bits, uint32_t* scratch, int sm_count, uint32_t* status,
                                   cudaStream_t stream, int* result) {
  *result = 0;
  if (cap <= 0 || key_bits <= 0) return EMB_OK;
  if (cap > (int64_t)kCountMask) return EMB_ERR_UNSUPPORTED;   // look-back words count in 30 bits
  if (n_dev) n = cap;
  int bits = 8, passes = 1;
  sort_plan<K>(key_bits, &bits, &passes);
  if (passes > kMaxSortPasses) return EMB_ERR_UNSUPPORTED;
  if (!n_dev && n <= (int64_t)sort_tile<K>() && passes <= 2) {
    // one tile: every pass in one CTA, no scratch to clear (tile 0 only
    // writes its look-back words and never reads them)
    const int smem = (int)sizeof(SortSmemT<K, 8>);
    EMB_CUDA_TRY(cudaFuncSetAttribute(k_sort_one_tile<K, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    uint32_t* fail = sort_fail_word<K>(scratch, key_bits);
    k_sort_one_tile<K, 8><<<1, kSortThreads, smem, stream>>>(keys[0], vals[0], keys[1], vals[1], (int)n, passes,
                                                             fail + 1, status, fail);
    *result = passes & 1;
    return cuda_status(cudaGetLastError());
  }
  EMB_CUDA_TRY(cudaMemsetAsync(scratch, 0, sort_scratch_words<K>(key_bits, cap) * sizeof(uint32_t), stream));
  emb_status st;
  if constexpr (sizeof(K) == 4) {
    st = bits == 9 ? radix_sort_passes<K, 9>(keys, vals, n, n_dev, cap, passes, scratch, sm_count, status, stream)
                   : radix_sort_passes<K, 8>(keys, vals, n, n_dev, cap, passes, scratch, sm_count, status, stream);
  } else {
    st = radix_sort_passes<K, 8>(keys, vals, n, n_dev, cap, passes, scratch, sm_count, status, stream);
  }
  if (st != EMB_OK) return st;
  *result = passes & 1;
  return cuda_status(cudaGetLastError());
}

}  // namespace emb
