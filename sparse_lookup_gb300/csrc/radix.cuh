// radix.cuh -- stable LSD radix sort of (key, u32 value) pairs, one 8-bit
// digit per pass: a single read of the keys builds the digit histograms of all
// passes, then each pass is one chained-scan scatter kernel in which a CTA
// ranks its tile in shared memory, publishes its per-digit counts and finds
// its global offsets by decoupled look-back over the earlier tiles (Adinets &
// Merrill, "Onesweep: a faster least significant digit radix sort for GPUs",
// 2022).  Tiles are taken in launch order from a ticket counter, so a CTA
// only ever waits on CTAs that are already running; every wait is bounded and
// latches EMB_ERR_TIMEOUT instead of hanging.
//
// The element count may live in device memory (n_dev != nullptr): grids are
// then sized for the capacity, the count is clamped to it and tiles past the
// count do nothing.
#pragma once

#include "plan.cuh"

namespace emb {

constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagInc = 2u << 30;
constexpr uint32_t kCountMask = (1u << 30) - 1;
constexpr int kSpinLimit = 1 << 22;
constexpr int kLookWin = 8;   // look-back words loaded per round trip
constexpr int kSortWarps = kSortThreads / 32;

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
struct SortSmemT {
  static constexpr int kTile = kSortThreads * SortItems<K>::value;
  K keys[kTile];
  uint32_t vals[kTile];
  uint32_t whist[kSortWarps][kRadix];  // per-warp digit counts, then warp offsets
  uint32_t dstart[kRadix];             // first slot of each digit inside the tile
  uint32_t goff[kRadix];               // global position of the tile's first item of each digit
  uint32_t hscan[kRadix];              // exclusive scan of the pass histogram
  uint32_t wsum[kSortWarps];
  uint32_t tile;
};

// Element count: n, or the count in device memory clamped to the capacity n.
__device__ __forceinline__ int64_t sort_count(int64_t n, const uint32_t* n_dev) {
  if (!n_dev) return n;
  const int64_t c = (int64_t)*((volatile const uint32_t*)n_dev);
  return c < n ? c : n;
}

template <class K>
__global__ void __launch_bounds__(512) k_digit_hist_t(const K* __restrict__ keys, int64_t n0,
                                                      const uint32_t* n_dev, int passes,
                                                      uint32_t* __restrict__ hist) {
  __shared__ uint32_t h[8 * kRadix];
  const int64_t n = sort_count(n0, n_dev);
  for (int i = threadIdx.x; i < passes * kRadix; i += blockDim.x) h[i] = 0;
  __syncthreads();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const K k = keys[i];
    for (int p = 0; p < passes; ++p) atomicAdd(&h[p * kRadix + (uint32_t)((k >> (p * kRadixBits)) & (kRadix - 1))], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < passes * kRadix; i += blockDim.x)
    if (h[i]) atomicAdd(&hist[i], h[i]);
}

// Lanes of the warp holding the same digit d, found with one ballot per digit
// bit: the mask starts full and each ballot keeps the lanes that agree with
// this lane on that bit.  BITS = kRadixBits + 1 when some lanes hold the "no
// item" marker kRadix.  All lanes must call.
template <int BITS>
__device__ __forceinline__ unsigned warp_match_digit(uint32_t d) {
  unsigned peers = kFull;
#pragma unroll
  for (int b = 0; b < BITS; ++b) {
    const unsigned m = __ballot_sync(kFull, (d >> b) & 1u);
    peers &= ((d >> b) & 1u) ? m : ~m;
  }
  return peers;
}

// Exclusive scan over the first 256 threads' values (all threads call).
__device__ __forceinline__ uint32_t sort_scan256(uint32_t v, uint32_t* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31 && warp < kRadix / 32) wsum[warp] = x;
  __syncthreads();
  uint32_t base = 0;
  if (warp < kRadix / 32)
    for (int w = 0; w < warp; ++w) base += wsum[w];
  __syncthreads();
  return base + x - v;
}

template <class K>
__device__ __forceinline__ uint32_t sort_digit(K k, int shift) {
  return (uint32_t)(k >> shift) & (uint32_t)(kRadix - 1);
}

// One tile of a pass: rank the items by digit within the tile (stable: warp
// order, then item order, then lane order), publish the tile's digit counts,
// place the items in shared memory in digit order, find the tile's global
// digit offsets by look-back, write out.  FULL: the tile holds TILE items
// (no per-item bounds, one ballot less).
template <class K>
__device__ __forceinline__ void onesweep_tile(SortSmemT<K>& sm, const K* __restrict__ kin,
                                              const uint32_t* __restrict__ vin, K* __restrict__ kout,
                                              uint32_t* __restrict__ vout, uint32_t n, uint32_t t, int tile_n,
                                              int shift, uint32_t* lookback, uint32_t* status) {
  const bool FULL = tile_n == SortSmemT<K>::kTile;
  constexpr int ITEMS = SortItems<K>::value;
  constexpr int TILE = SortSmemT<K>::kTile;
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
    const uint32_t d = ok ? sort_digit(k[i], shift) : (uint32_t)kRadix;
    const unsigned peers = FULL ? warp_match_digit<kRadixBits>(d) : warp_match_digit<kRadixBits + 1>(d);
    const int leader = 31 - __clz(peers);
    uint32_t old = 0;
    if (lane == leader && ok) {
      old = sm.whist[warp][d];
      sm.whist[warp][d] = old + __popc(peers);
    }
    old = __shfl_sync(kFull, old, leader);
    __syncwarp();   // the counter update is seen by the next item's leader
    const uint32_t rank = old + __popc(peers & lt);
    if (i & 1) r2[i >> 1] |= rank << 16;
    else r2[i >> 1] = rank;
  }
  __syncthreads();

  uint32_t cnt = 0;
  if (tid < kRadix) {
    for (int w = 0; w < kSortWarps; ++w) {
      const uint32_t c = sm.whist[w][tid];
      sm.whist[w][tid] = cnt;
      cnt += c;
    }
    *(volatile uint32_t*)(lookback + (size_t)t * kRadix + tid) = (t == 0 ? kFlagInc : kFlagAgg) | cnt;
  }
  const uint32_t ds = sort_scan256(cnt, sm.wsum);
  if (tid < kRadix) {
    sm.dstart[tid] = ds;
    for (int w = 0; w < kSortWarps; ++w) sm.whist[w][tid] += ds;   // slot of each warp's first item of the digit
  }
  __syncthreads();
  // the tile's items into shared memory in digit order; this frees their
  // registers before the look-back below
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    if (FULL || w0 + i * 32 + lane < tile_n) {
      const uint32_t rank = (i & 1) ? r2[i >> 1] >> 16 : r2[i >> 1] & 0xffffu;
      const uint32_t pos = sm.whist[warp][sort_digit(k[i], shift)] + rank;
      sm.keys[pos] = k[i];
      sm.vals[pos] = v[i];
    }
  }
  if (tid < kRadix) {
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
        for (int q = 0; q < kLookWin; ++q)
          w[q] = j - q >= 0 ? *(volatile const uint32_t*)(lookback + (j - q) * kRadix + tid) : kFlagInc;
        int q = 0;
#pragma unroll
        for (int qq = 0; qq < kLookWin; ++qq) {
          if (q == qq) {
            const uint32_t flag = w[qq] & ~kCountMask;
            if (flag != 0u) {
              excl += w[qq] & kCountMask;
              if (flag == kFlagInc) done = true;
              else ++q;
            }
          }
        }
        if (done) break;
        j -= q;
        if (q < kLookWin) {   // word j is not published yet
          if (++spins > kSpinLimit) {
            latch(status, EMB_ERR_TIMEOUT);
            break;
          }
          __nanosleep(32);
        }
      }
      *(volatile uint32_t*)(lookback + (size_t)t * kRadix + tid) = kFlagInc | ((excl + cnt) & kCountMask);
    }
    // output position of shared slot j of this digit: goff + (j - dstart)
    sm.goff[tid] = sm.hscan[tid] + excl - ds;
  }
  __syncthreads();
  for (int j = tid; j < (FULL ? TILE : tile_n); j += kSortThreads) {
    const K key = sm.keys[j];
    const uint32_t o = sm.goff[sort_digit(key, shift)] + (uint32_t)j;
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
template <class K, bool PERSIST>
__global__ void __launch_bounds__(kSortThreads, 2)
    k_onesweep_t(const K* __restrict__ kin, const uint32_t* __restrict__ vin, K* __restrict__ kout,
                 uint32_t* __restrict__ vout, int64_t n0, const uint32_t* n_dev, int shift,
                 const uint32_t* __restrict__ hist, uint32_t* lookback, uint32_t* tile_ctr, uint32_t* status) {
  constexpr int TILE = SortSmemT<K>::kTile;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SortSmemT<K>& sm = *reinterpret_cast<SortSmemT<K>*>(smem_raw);
  const int tid = threadIdx.x;
  const int64_t n = sort_count(n0, n_dev);
  const int64_t tiles = (n + TILE - 1) / TILE;
  const uint32_t hs = sort_scan256(tid < kRadix ? __ldg(hist + tid) : 0u, sm.wsum);
  if (tid < kRadix) sm.hscan[tid] = hs;
  do {
    if (tid == 0) sm.tile = atomicAdd(tile_ctr, 1u);
    for (int i = tid; i < kSortWarps * kRadix; i += kSortThreads) (&sm.whist[0][0])[i] = 0;
    __syncthreads();
    const uint32_t t = sm.tile;
    if ((int64_t)t >= tiles) return;   // past the data: nobody waits on this ticket
    const int64_t left = n - (int64_t)t * TILE;
    onesweep_tile<K>(sm, kin, vin, kout, vout, (uint32_t)n, t, left >= TILE ? TILE : (int)left, shift, lookback,
                     status);
    if (PERSIST) __syncthreads();   // the tile's shared memory is free again
  } while (PERSIST);
}

// Words of scratch the sort needs: hist [passes][256], tickets [passes],
// look-back words [passes][tiles][256].
template <class K>
inline size_t sort_scratch_words(int passes, int64_t cap) {
  const int64_t tiles = (cap + SortSmemT<K>::kTile - 1) / SortSmemT<K>::kTile;
  return (size_t)passes * kRadix + passes + (size_t)passes * tiles * kRadix;
}

// Sorts keys[0]/vals[0] (n pairs, or *n_dev of at most cap) into keys[p&1],
// vals[p&1] with p = passes.  `scratch` holds sort_scratch_words() words and
// is cleared here.  Returns the index of the buffer holding the result.
template <class K>
inline emb_status radix_sort_pairs(K* const keys[2], uint32_t* const vals[2], int64_t n, const uint32_t* n_dev,
                                   int64_t cap, int passes, uint32_t* scratch, int sm_count, uint32_t* status,
                                   cudaStream_t stream, int* result) {
  *result = 0;
  if (cap <= 0 || passes <= 0) return EMB_OK;
  if (cap > (int64_t)kCountMask) return EMB_ERR_UNSUPPORTED;   // look-back words count in 30 bits
  if (n_dev) n = cap;
  const int64_t tiles = (cap + SortSmemT<K>::kTile - 1) / SortSmemT<K>::kTile;
  uint32_t* hist = scratch;
  uint32_t* tickets = hist + (size_t)passes * kRadix;
  uint32_t* lookback = tickets + passes;
  EMB_CUDA_TRY(cudaMemsetAsync(scratch, 0, sort_scratch_words<K>(passes, cap) * sizeof(uint32_t), stream));
  const int hgrid = (int)std::min<int64_t>((cap + 511) / 512, (int64_t)sm_count * 4);
  k_digit_hist_t<K><<<hgrid, 512, 0, stream>>>(keys[0], n, n_dev, passes, hist);
  const bool persist = n_dev != nullptr;
  const int64_t grid = persist ? std::min<int64_t>(tiles, (int64_t)sm_count * 2) : tiles;   // two CTAs fit an SM
  EMB_CUDA_TRY(cudaFuncSetAttribute(k_onesweep_t<K, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)sizeof(SortSmemT<K>)));
  EMB_CUDA_TRY(cudaFuncSetAttribute(k_onesweep_t<K, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)sizeof(SortSmemT<K>)));
  for (int ps = 0; ps < passes; ++ps) {
    const int in = ps & 1, out = in ^ 1;
    if (persist)
      k_onesweep_t<K, true><<<(unsigned)grid, kSortThreads, sizeof(SortSmemT<K>), stream>>>(
          keys[in], vals[in], keys[out], vals[out], n, n_dev, ps * kRadixBits, hist + ps * kRadix,
          lookback + (size_t)ps * tiles * kRadix, tickets + ps, status);
    else
      k_onesweep_t<K, false><<<(unsigned)grid, kSortThreads, sizeof(SortSmemT<K>), stream>>>(
          keys[in], vals[in], keys[out], vals[out], n, n_dev, ps * kRadixBits, hist + ps * kRadix,
          lookback + (size_t)ps * tiles * kRadix, tickets + ps, status);
  }
  *result = passes & 1;
  return cuda_status(cudaGetLastError());
}

}  // namespace emb
