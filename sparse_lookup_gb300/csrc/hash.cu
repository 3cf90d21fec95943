// hash.cu -- K-H: the collision-free dynamic table (Monolith §2.1 "Tabel
// Hash": distinct IDs never share an embedding; an ID enters the table only
// once it has been seen often enough; IDs idle for longer than a set period
// expire).
//
// The page's table is a cuckoo map on a CPU parameter server.  On one GPU the
// same contract -- distinct (table id, key) pairs never share an entry or a
// row -- is kept by an open-addressing table with linear probing in HBM:
//   slot (16 B) = key (tid << 48 | key), state, last_seen
//   state >= 0: the admitted key's row; state < 0: still counting, with
//   count = -1 - state.
// An insert claims a slot with a compare-and-swap only after its probe has
// reached an EMPTY slot (so the key is known to be absent), taking the first
// tombstone or EMPTY slot on its path; threads inserting the same key meet at
// the same slot.  Expired entries become tombstones that probes step over and
// inserts reuse; the expiry sweep also turns tombstone runs that end at an
// EMPTY slot back into EMPTY slots.
//
//   K-H1 k_hash_probe  one thread per occurrence: find or insert the key
//                      (bounded probing), touch last_seen, count; the one
//                      occurrence whose count reaches the threshold lists the
//                      key for admission.
//   K-H2 admission     the listed keys are radix-sorted by (tid, key); the
//                      i-th key takes the i-th free row of the pool (a bitmap
//                      of used rows, scanned per word), which is the same as
//                      "rows released by expiry in ascending order, then rows
//                      never used"; its weights are initialised from its key.
//        k_hash_fix    occurrences of keys admitted in this call get the row.
//   K-H3 expiry       removes entries idle > ttl and releases their rows:
//                      k_hash_evict_lists checks only the slots that the
//                      lookups of the due steps touched first (each lookup
//                      lists those slots); k_hash_evict sweeps every slot
//                      when a touch may have gone unlisted (a second lookup
//                      at one step, more live steps than lists).
#include <algorithm>
#include <new>

#include "plan.cuh"
#include "radix.cuh"

namespace emb {

constexpr unsigned long long kEmptyKey = ~0ull;
constexpr unsigned long long kTombKey = ~0ull - 1ull;
// last_seen of a slot that holds no entry: a value no lookup step may take,
// so the first touch of a new entry always moves last_seen (and is listed)
constexpr uint32_t kNeverSeen = 0xFFFFFFFFu;
// the (state, last_seen) word of a slot that holds no entry
constexpr unsigned long long kFreeWord = ((unsigned long long)kNeverSeen << 32) | 0xFFFFFFFFull;
constexpr int kTidBits = 15;
constexpr int kKeyBits = 48;
constexpr int kHashKeyBits = 63;   // packed (tid << 48 | key) sort keys
// Lists of the slots each lookup call touched first, kept for incremental
// expiry: with one lookup per step and expiry every step, ttl + 2 lists are
// live at a time, so ttl <= kTouchLists - 2 never needs a full sweep.
constexpr int kTouchLists = 16;

struct __align__(16) Slot {
  unsigned long long key;
  int32_t state;        // low half of the second 8-byte word
  uint32_t last_seen;   // high half: (state, last_seen) change together by CAS
};
static_assert(sizeof(Slot) == 16, "slot layout");

}  // namespace emb

struct emb_hash_s {
  int64_t num_slots = 0;
  int64_t cap = 0;
  int64_t max_keys = 0;
  int32_t dim = 0;
  int32_t thr = 0;
  int32_t max_probes = 0;
  uint64_t seed = 0;
  float init_scale = 0.f;
  emb::Slot* slots = nullptr;
  float* W = nullptr;
  float* acc = nullptr;
  uint32_t* used = nullptr;        // bitmap of rows in use, bits past cap set
  int64_t n_words = 0;
  uint32_t* free_scan = nullptr;   // [n_words + 1] exclusive prefix of free rows per word
  uint32_t* scan_part = nullptr;   // per 1024-word block partials
  uint32_t* free_rows = nullptr;   // [max_keys] the lowest free rows, ascending
  uint64_t* nkeys[2] = {nullptr, nullptr};
  uint32_t* nvals[2] = {nullptr, nullptr};
  uint32_t* counters = nullptr;    // [0] listed keys, [1] exported entries, [2] latest imported step
  uint32_t* sort_scratch = nullptr;
  uint32_t* status = nullptr;
  int sm_count = 0;
  // incremental expiry: the slots whose last_seen a lookup call moved to its
  // step, one list per step
  uint32_t* touch = nullptr;            // [kTouchLists][max_keys]
  uint32_t* touch_n = nullptr;          // [kTouchLists] entries per list
  uint32_t list_step[emb::kTouchLists] = {};
  bool list_live[emb::kTouchLists] = {};
  int cur_list = -1;                    // list of the latest lookup's step
  bool lists_valid = true;              // every touch not yet expired is in a live list
  int64_t unrecorded_step = -1;         // latest step whose touches were not all listed
};

namespace emb {

struct HashArgs {
  Slot* slots;
  uint64_t mask;
  int32_t max_probes;
  int32_t thr;
  uint32_t* n_new;
  uint64_t* nkeys;
  uint32_t* nvals;
  int64_t max_keys;
  uint32_t* status;
  uint32_t* touch;     // list for this call's first touches, or nullptr
  uint32_t* touch_n;
};

// One 16-byte read of a whole slot: the key word and the (state, last_seen)
// word together, in one memory transaction.
__device__ __forceinline__ void load_slot(const Slot* p, unsigned long long& key, unsigned long long& sw) {
  asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(key), "=l"(sw) : "l"(p) : "memory");
}

__device__ __forceinline__ uint64_t home_slot(uint64_t fkey, uint64_t mask) {
  return splitmix64(fkey ^ 0x5851F42D4C957F2Dull) & mask;
}

// K-H1, one occurrence: find or insert its key, touch and count; writes its
// row (or -2 - slot for a key listed for admission, -1 otherwise) and
// returns true when this occurrence moved the slot's last_seen to `step`
// (the call's first touch of the entry), with the slot in *slot_out.
__device__ __forceinline__ bool probe_one(const HashArgs& h, const int32_t* __restrict__ tids,
                                          const int64_t* __restrict__ keys, int64_t i, uint32_t step,
                                          int64_t* __restrict__ rows_out, uint32_t* slot_out) {
  const int32_t tid = tids[i];
  const int64_t key = keys[i];
  if (tid < 0 || tid >= (1 << kTidBits) || key < 0 || key >= (int64_t(1) << kKeyBits)) {
    latch(h.status, EMB_ERR_INVALID_ARG);
    rows_out[i] = -1;
    return false;
  }
  const unsigned long long fkey = ((unsigned long long)tid << kKeyBits) | (unsigned long long)key;
  // Probe from the home slot until the key or an EMPTY slot turns up (the
  // EMPTY slot proves the key is absent), remembering the first slot that
  // could take it (a tombstone or that EMPTY slot); claim that slot by CAS on
  // the value seen there.  If another key took it first, keep probing after
  // it.  Within one call slots only change from EMPTY/tombstone to a key, and
  // every thread inserting the same key walks the same path, so they all end
  // at the one slot the first of them claimed.
  uint64_t start = home_slot(fkey, h.mask);
  int64_t found = -1;
  int budget = h.max_probes;
  unsigned long long sw_seen = 0;   // (state, last_seen) word read with the key
  bool have_sw = false;
  while (budget > 0 && found < 0) {
    uint64_t pos = start;
    int64_t avail = -1;
    unsigned long long avail_val = 0;
    bool seen_empty = false;
    while (budget > 0) {
      unsigned long long k, w;
      load_slot(&h.slots[pos], k, w);
      --budget;
      if (k == fkey) {
        found = (int64_t)pos;
        sw_seen = w;
        have_sw = true;
        break;
      }
      if (k == kEmptyKey) {
        if (avail < 0) {
          avail = (int64_t)pos;
          avail_val = kEmptyKey;
        }
        seen_empty = true;
        break;
      }
      if (k == kTombKey && avail < 0) {
        avail = (int64_t)pos;
        avail_val = kTombKey;
      }
      pos = (pos + 1) & h.mask;
    }
    if (found >= 0 || !seen_empty) break;
    const unsigned long long old = atomicCAS(&h.slots[avail].key, avail_val, fkey);
    if (old == avail_val || old == fkey) {
      found = avail;
      break;
    }
    start = ((uint64_t)avail + 1) & h.mask;
  }
  if (found < 0) {
    latch(h.status, EMB_ERR_PROBE_LIMIT);
    rows_out[i] = -1;
    return false;
  }
  Slot* s = &h.slots[found];
  unsigned long long* sw = reinterpret_cast<unsigned long long*>(&s->state);
  if (!have_sw) sw_seen = *(volatile unsigned long long*)sw;   // the slot was just claimed
  // An admitted state does not change within a call (admission runs after
  // the probes), so the word read with the key decides; a counting state
  // read there may be stale, which the atomics below correct.
  int32_t old = (int32_t)(uint32_t)(sw_seen & 0xffffffffull);
  int64_t out;
  bool first = false;   // this occurrence moved last_seen to this step
  if (old >= 0) {
    out = old;
    if ((uint32_t)(sw_seen >> 32) != step) {
      // Lanes of this warp that hold the same slot touch it with one
      // exchange: a hot key's occurrences would otherwise queue thousands of
      // atomics on one address.  The exchange still decides the call's first
      // touch across warps; the other lanes of the group are not first.
      const unsigned act = __activemask();
      const unsigned grp = __match_any_sync(act, (unsigned long long)found);
      if ((int)(threadIdx.x & 31) == __ffs(grp) - 1) first = atomicExch(&s->last_seen, step) != step;
    }
  } else {
    // Count and touch with atomic updates of the whole (state, last_seen)
    // word, so that "first occurrence of this call" and "count reached the
    // threshold" are decided on one order of updates.  Only the occurrences
    // that find last_seen behind the current step race by CAS to set it;
    // once it equals the step it stays there for the rest of the call, and
    // every later occurrence counts with one atomic add (no retry loop, which
    // on hot keys of a cold table would serialise thousands of CAS attempts).
    // Adding 2^64 - 1 takes one off the low half without a borrow into
    // last_seen, since a not-yet-admitted state is negative (count below
    // 2^31 - 1).
    unsigned long long prev = sw_seen;
    bool counted = false;
    while (old < 0 && (uint32_t)(prev >> 32) != step) {
      const unsigned long long nxt = ((unsigned long long)step << 32) | ((uint32_t)old - 1u);
      const unsigned long long cur = atomicCAS(sw, prev, nxt);
      if (cur == prev) {
        counted = true;
        first = true;
        break;
      }
      prev = cur;
      old = (int32_t)(uint32_t)(prev & 0xffffffffull);
    }
    if (old >= 0) {   // admitted meanwhile (not within one call; kept for safety)
      out = old;
    } else {
      if (!counted) {
        prev = atomicAdd(sw, ~0ull);
        old = (int32_t)(uint32_t)(prev & 0xffffffffull);
      }
      const uint32_t old_seen = (uint32_t)(prev >> 32);
      const int32_t count_old = -1 - old, count_new = count_old + 1;
      // the occurrence that reaches the threshold lists the key; a key left
      // without a row by a full pool is listed again by its first occurrence
      if (count_new >= h.thr && (count_old < h.thr || old_seen != step)) {
        const uint32_t idx = atomicAdd(h.n_new, 1u);
        if ((int64_t)idx < h.max_keys) {
          h.nkeys[idx] = fkey;
          h.nvals[idx] = (uint32_t)found;
        }
      }
      out = -2 - found;
    }
  }
  rows_out[i] = out;
  *slot_out = (uint32_t)found;
  return first;
}

// K-H1.  A slot's first touch of the call goes on the call's list (one entry
// per distinct slot, so at most n): the CTA counts its first touches in
// shared memory and takes their places in the list with ONE global atomic
// (a per-warp atomic on the one list counter queued about 128 K returning
// atomics on a single address per call).
__global__ void __launch_bounds__(256) k_hash_probe(const HashArgs h, const int32_t* __restrict__ tids,
                                                    const int64_t* __restrict__ keys, int64_t n, uint32_t step,
                                                    int64_t* __restrict__ rows_out) {
  __shared__ uint32_t s_cnt, s_base;
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  uint32_t slot = 0;
  const bool first = i < n && probe_one(h, tids, keys, i, step, rows_out, &slot);
  if (!h.touch) return;   // the same for the whole grid
  const int lane = threadIdx.x & 31;
  const unsigned fm = __ballot_sync(kFull, first);
  uint32_t wbase = 0;
  if (lane == 0 && fm) wbase = atomicAdd(&s_cnt, (uint32_t)__popc(fm));
  wbase = __shfl_sync(kFull, wbase, 0);
  __syncthreads();
  if (threadIdx.x == 0) s_base = s_cnt ? atomicAdd(h.touch_n, s_cnt) : 0u;
  __syncthreads();
  if (first) {
    const uint32_t idx = s_base + wbase + (uint32_t)__popc(fm & ((1u << lane) - 1u));
    if ((int64_t)idx < h.max_keys) h.touch[idx] = slot;
  }
}

// free rows per word of the used-row bitmap, exclusive prefix over words
constexpr int kScanBlk = 1024;

__global__ void __launch_bounds__(kScanBlk) k_free_reduce(const uint32_t* used, int64_t nw, uint32_t* part) {
  const int64_t w = blockIdx.x * (int64_t)kScanBlk + threadIdx.x;
  const uint32_t f = w < nw ? (uint32_t)__popc(~used[w]) : 0u;
  uint32_t s = f;
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
  __shared__ uint32_t ws[32];
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int j = 0; j < kScanBlk / 32; ++j) t += ws[j];
    part[blockIdx.x] = t;
  }
}

__global__ void __launch_bounds__(kScanBlk) k_scan_parts(uint32_t* part, int nb) {
  __shared__ uint32_t wsum[32];
  __shared__ uint32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int b0 = 0; b0 < nb; b0 += kScanBlk) {
    const int i = b0 + threadIdx.x;
    const uint32_t v = i < nb ? part[i] : 0u;
    uint32_t x = v;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    uint32_t base = carry, tot = 0;
    for (int w = 0; w < 32; ++w) {
      if (w < warp) base += wsum[w];
      tot += wsum[w];
    }
    if (i < nb) part[i] = base + x - v;
    __syncthreads();
    if (threadIdx.x == 0) carry += tot;
    __syncthreads();
  }
}

// ... and the free rows themselves, in ascending order, as far as the keys
// listed for admission need them: free_rows[i] = the i-th free row.
__global__ void __launch_bounds__(kScanBlk) k_free_down(const uint32_t* used, int64_t nw, const uint32_t* part,
                                                        uint32_t* free_scan, const uint32_t* n_new, int64_t max_keys,
                                                        uint32_t* free_rows) {
  __shared__ uint32_t wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t w = blockIdx.x * (int64_t)kScanBlk + threadIdx.x;
  const uint32_t bits = w < nw ? ~used[w] : 0u;
  const uint32_t f = (uint32_t)__popc(bits);
  uint32_t x = f;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  uint32_t base = part[blockIdx.x];
  for (int j = 0; j < warp; ++j) base += wsum[j];
  if (w < nw) free_scan[w] = base + x - f;
  if (w == nw - 1) free_scan[nw] = base + x;
  const int64_t need = ((int64_t)*n_new < max_keys) ? (int64_t)*n_new : max_keys;
  int64_t pos = (int64_t)(base + x - f);
  for (uint32_t b = bits; b && pos < need; b &= b - 1u, ++pos) free_rows[pos] = (uint32_t)(w * 32 + __ffs(b) - 1);
}

__device__ __forceinline__ float init_value(uint64_t fkey, uint64_t seed, int d, float scale) {
  const uint64_t hsh = splitmix64(fkey ^ seed ^ (uint64_t)(uint32_t)d);
  const int32_t v = (int32_t)(hsh >> 40) - 8388608;
  const float f = __fmul_rn((float)v, 1.0f / 8388608.0f);
  return __fmul_rn(f, scale);
}

// K-H2: the i-th listed key (ascending) takes the i-th free row, listed by
// k_free_down; k_hash_mark sets the bits of the rows handed out afterwards.
// Both do nothing when the sort of the listed keys gave up a wait (sort_fail
// set, EMB_ERR_TIMEOUT latched): its output then has holes, and the listed
// keys stay counting.
__global__ void __launch_bounds__(256) k_hash_admit(Slot* slots, const uint64_t* __restrict__ skeys,
                                                    const uint32_t* __restrict__ svals, const uint32_t* n_new,
                                                    int64_t max_keys, const uint32_t* free_scan,
                                                    const uint32_t* __restrict__ free_rows, int64_t nw, float* W,
                                                    float* A, int dim, uint64_t seed, float scale, uint32_t* status,
                                                    const uint32_t* sort_fail) {
  if (*(volatile const uint32_t*)sort_fail) return;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t nn = ((int64_t)*n_new < max_keys) ? (int64_t)*n_new : max_keys;
  const uint32_t total_free = free_scan[nw];
  for (int64_t i = warp; i < nn; i += nwarps) {
    if (i >= (int64_t)total_free) {
      if (lane == 0) latch(status, EMB_ERR_TABLE_FULL);
      continue;
    }
    const int64_t row = free_rows[i];
    const uint64_t fkey = skeys[i];
    if (lane == 0) slots[svals[i]].state = (int32_t)row;
    for (int d = lane; d < dim; d += 32) {
      W[row * dim + d] = init_value(fkey, seed, d, scale);
      A[row * dim + d] = 0.0f;
    }
  }
}

__global__ void __launch_bounds__(256) k_hash_mark(const Slot* slots, const uint32_t* __restrict__ svals,
                                                   const uint32_t* n_new, int64_t max_keys, uint32_t* used,
                                                   const uint32_t* sort_fail) {
  if (*(volatile const uint32_t*)sort_fail) return;
  const int64_t nn = ((int64_t)*n_new < max_keys) ? (int64_t)*n_new : max_keys;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nn; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t st = slots[svals[i]].state;
    if (st >= 0) atomicOr(&used[st >> 5], 1u << (st & 31));
  }
}

__global__ void __launch_bounds__(256) k_hash_fix(const Slot* slots, int64_t n, int64_t* rows_out) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t v = rows_out[i];
  if (v <= -2) {
    const int32_t st = slots[-2 - v].state;
    rows_out[i] = st >= 0 ? st : -1;
  }
}

// K-H3.  Tombstones are cleared where that is safe: a run of tombstones
// directly before an EMPTY slot lies on no live key's probe path (such a path
// would have to cross the EMPTY slot), so the run may become EMPTY again.
// Slots emptied by other threads during the sweep only leave tombstones
// behind, never a broken path.
constexpr int kTombWalk = 4096;

__global__ void __launch_bounds__(256) k_hash_evict(Slot* slots, int64_t ns, uint32_t now, uint32_t ttl,
                                                    uint32_t* used, unsigned long long* n_evicted) {
  unsigned long long cnt = 0;
  const uint64_t mask = (uint64_t)ns - 1;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < ns; i += (int64_t)gridDim.x * blockDim.x) {
    const unsigned long long k = *(volatile unsigned long long*)&slots[i].key;
    if (k == kEmptyKey) {
      uint64_t j = ((uint64_t)i - 1) & mask;
      for (int w = 0; w < kTombWalk; ++w, j = (j - 1) & mask) {
        if (*(volatile unsigned long long*)&slots[j].key != kTombKey) break;
        slots[j].key = kEmptyKey;
      }
      continue;
    }
    if (k == kTombKey) continue;
    const uint32_t ls = slots[i].last_seen;
    if ((int64_t)now - (int64_t)ls > (int64_t)ttl) {
      const int32_t st = slots[i].state;
      if (st >= 0) atomicAnd(&used[st >> 5], ~(1u << (st & 31)));
      *reinterpret_cast<unsigned long long*>(&slots[i].state) = kFreeWord;
      *(volatile unsigned long long*)&slots[i].key = kTombKey;
      ++cnt;
    }
  }
  if (n_evicted) {
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
    if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(n_evicted, cnt);
  }
}

// Incremental expiry: the slots on the lists of steps now - ttl - 1 and
// before, instead of all slots.  An entry is on the list of every step whose
// lookup touched it first, so each entry idle longer than ttl is on one of
// these lists; it is removed when its last_seen still says so (a later touch
// keeps it).  A slot on two lists is removed once (CAS on the key).  After a
// removal the tombstone run ending at this slot becomes EMPTY when the next
// slot is EMPTY (no probe passes an EMPTY slot, so none needs the run).
struct EvictLists {
  const uint32_t* list[kTouchLists];
  const uint32_t* count[kTouchLists];
  int n;
};

__global__ void __launch_bounds__(256) k_hash_evict_lists(Slot* slots, uint64_t mask, const EvictLists L,
                                                          int64_t cap, uint32_t now, uint32_t ttl, uint32_t* used,
                                                          unsigned long long* n_evicted) {
  unsigned long long cnt = 0;
  const int64_t g0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x, gs = (int64_t)gridDim.x * blockDim.x;
  for (int l = 0; l < L.n; ++l) {
    const int64_t nl = min((int64_t)*L.count[l], cap);
    for (int64_t j = g0; j < nl; j += gs) {
      const uint64_t p = L.list[l][j];
      unsigned long long k, w;
      load_slot(&slots[p], k, w);
      if (k == kEmptyKey || k == kTombKey) continue;
      if ((int64_t)now - (int64_t)(uint32_t)(w >> 32) <= (int64_t)ttl) continue;
      if (atomicCAS(&slots[p].key, k, kTombKey) != k) continue;
      const int32_t st = (int32_t)(uint32_t)(w & 0xffffffffull);
      if (st >= 0) atomicAnd(&used[st >> 5], ~(1u << (st & 31)));
      *reinterpret_cast<unsigned long long*>(&slots[p].state) = kFreeWord;
      ++cnt;
      if (*(volatile unsigned long long*)&slots[(p + 1) & mask].key == kEmptyKey) {
        uint64_t q = p;
        for (int t = 0; t < kTombWalk; ++t, q = (q - 1) & mask)
          if (atomicCAS(&slots[q].key, kTombKey, kEmptyKey) != kTombKey) break;
      }
    }
  }
  if (n_evicted) {
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
    if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(n_evicted, cnt);
  }
}

__global__ void k_hash_init(Slot* slots, int64_t ns, uint32_t* used, int64_t nw, int64_t cap) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < ns; i += (int64_t)gridDim.x * blockDim.x) {
    slots[i].key = kEmptyKey;
    slots[i].state = -1;
    slots[i].last_seen = kNeverSeen;
  }
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < nw; w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t first = w * 32;
    uint32_t bits = 0;
    for (int b = 0; b < 32; ++b)
      if (first + b >= cap) bits |= 1u << b;   // rows past the pool are never free
    used[w] = bits;
  }
}

// hash_import: entry i of a snapshot into a cleared table (every slot EMPTY,
// no tombstone): probe from its home slot to the first EMPTY slot and claim
// it; meeting its own key on the way means the snapshot lists it twice.  An
// admitted entry marks its row used; a row marked already is listed twice.
// Bad entries latch EMB_ERR_INVALID_ARG and are left out.
__global__ void __launch_bounds__(256) k_hash_import(Slot* slots, uint64_t mask, int32_t max_probes, int64_t cap,
                                                     uint32_t* used, const int32_t* __restrict__ tids,
                                                     const int64_t* __restrict__ keys,
                                                     const int64_t* __restrict__ rows,
                                                     const int32_t* __restrict__ counts,
                                                     const uint32_t* __restrict__ last_seen, int64_t n,
                                                     uint32_t* status, uint32_t* max_seen) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int32_t tid = tids[i];
  const int64_t key = keys[i];
  const int64_t row = rows[i];
  const int32_t cnt = counts ? counts[i] : 0;
  const uint32_t ls = last_seen[i];
  if (tid < 0 || tid >= (1 << kTidBits) || key < 0 || key >= (int64_t(1) << kKeyBits) || row >= cap ||
      (row < 0 && (row != -1 || cnt < 0 || cnt == 0x7FFFFFFF)) || ls == kNeverSeen) {
    latch(status, EMB_ERR_INVALID_ARG);
    return;
  }
  if (row >= 0) {
    const uint32_t bit = 1u << (row & 31);
    if (atomicOr(&used[row >> 5], bit) & bit) {   // a second entry with this row
      latch(status, EMB_ERR_INVALID_ARG);
      return;
    }
  }
  const unsigned long long fkey = ((unsigned long long)tid << kKeyBits) | (unsigned long long)key;
  uint64_t pos = home_slot(fkey, mask);
  for (int budget = max_probes; budget > 0; --budget, pos = (pos + 1) & mask) {
    const unsigned long long k = *(volatile unsigned long long*)&slots[pos].key;
    if (k == fkey) {   // listed twice
      latch(status, EMB_ERR_INVALID_ARG);
      return;
    }
    if (k != kEmptyKey) continue;
    const unsigned long long old = atomicCAS(&slots[pos].key, kEmptyKey, fkey);
    if (old == fkey) {
      latch(status, EMB_ERR_INVALID_ARG);
      return;
    }
    if (old != kEmptyKey) continue;   // another key took it: go on past it
    const int32_t state = row >= 0 ? (int32_t)row : -1 - cnt;
    *reinterpret_cast<unsigned long long*>(&slots[pos].state) =
        ((unsigned long long)ls << 32) | (unsigned long long)(uint32_t)state;
    atomicMax(max_seen, ls);
    return;
  }
  latch(status, EMB_ERR_PROBE_LIMIT);
}

__global__ void k_hash_export(const Slot* slots, int64_t ns, int32_t* tids, int64_t* keys, int64_t* rows,
                              int32_t* counts, uint32_t* last_seen, int64_t cap, uint32_t* ctr) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < ns; i += (int64_t)gridDim.x * blockDim.x) {
    const unsigned long long k = slots[i].key;
    if (k == kEmptyKey || k == kTombKey) continue;
    const uint32_t idx = atomicAdd(ctr, 1u);
    if ((int64_t)idx >= cap) continue;
    const int32_t st = slots[i].state;
    if (tids) tids[idx] = (int32_t)(k >> kKeyBits);
    if (keys) keys[idx] = (int64_t)(k & ((1ull << kKeyBits) - 1));
    if (rows) rows[idx] = st >= 0 ? st : -1;
    if (counts) counts[idx] = st >= 0 ? -1 : -1 - st;
    if (last_seen) last_seen[idx] = slots[i].last_seen;
  }
}

}  // namespace emb

using namespace emb;

namespace {

void free_hash(emb_hash_s* h) {
  if (!h) return;
  dev_free(h->slots);
  dev_free(h->W);
  dev_free(h->acc);
  dev_free(h->used);
  dev_free(h->free_scan);
  dev_free(h->scan_part);
  dev_free(h->free_rows);
  dev_free(h->nkeys[0]);
  dev_free(h->nkeys[1]);
  dev_free(h->nvals[0]);
  dev_free(h->nvals[1]);
  dev_free(h->counters);
  dev_free(h->sort_scratch);
  dev_free(h->status);
  dev_free(h->touch);
  dev_free(h->touch_n);
  delete h;
}

}  // namespace

extern "C" emb_status hash_create(int64_t num_slots, int64_t row_capacity, int32_t dim, int32_t admit_threshold,
                                  int32_t max_probes, uint64_t init_seed, float init_scale,
                                  int64_t max_keys_per_call, emb_hash* out) {
  if (!out) return EMB_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_slots < 1024 || (num_slots & (num_slots - 1)) != 0) return EMB_ERR_INVALID_ARG;
  if (num_slots > (int64_t(1) << 31)) return EMB_ERR_UNSUPPORTED;
  if (row_capacity < 1 || row_capacity >= (int64_t(1) << 31)) return EMB_ERR_INVALID_ARG;
  if (dim < 4 || dim % 4 != 0 || dim > 256) return EMB_ERR_INVALID_ARG;
  if (admit_threshold < 1 || max_probes < 1) return EMB_ERR_INVALID_ARG;
  if (max_keys_per_call < 1 || max_keys_per_call >= (int64_t(1) << 30)) return EMB_ERR_INVALID_ARG;
  if (!(init_scale == init_scale)) return EMB_ERR_INVALID_ARG;
  emb_hash_s* h = new (std::nothrow) emb_hash_s();
  if (!h) return EMB_ERR_OOM;
  h->num_slots = num_slots;
  h->cap = row_capacity;
  h->max_keys = max_keys_per_call;
  h->dim = dim;
  h->thr = admit_threshold;
  h->max_probes = max_probes;
  h->seed = init_seed;
  h->init_scale = init_scale;
  h->n_words = (row_capacity + 31) / 32;
  cudaError_t e = cudaSuccess;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, dev);
  auto alloc = [&](auto** p, size_t bytes) {
    if (e == cudaSuccess) e = dev_alloc((void**)p, bytes > 0 ? bytes : 1);
  };
  alloc(&h->slots, sizeof(Slot) * (size_t)num_slots);
  alloc(&h->W, sizeof(float) * (size_t)row_capacity * dim);
  alloc(&h->acc, sizeof(float) * (size_t)row_capacity * dim);
  alloc(&h->used, sizeof(uint32_t) * (size_t)h->n_words);
  alloc(&h->free_scan, sizeof(uint32_t) * (size_t)(h->n_words + 1));
  alloc(&h->scan_part, sizeof(uint32_t) * (size_t)((h->n_words + kScanBlk - 1) / kScanBlk + 1));
  alloc(&h->free_rows, sizeof(uint32_t) * (size_t)max_keys_per_call);
  for (int i = 0; i < 2; ++i) {
    alloc(&h->nkeys[i], sizeof(uint64_t) * (size_t)max_keys_per_call);
    alloc(&h->nvals[i], sizeof(uint32_t) * (size_t)max_keys_per_call);
  }
  alloc(&h->counters, sizeof(uint32_t) * 4);
  alloc(&h->sort_scratch, sizeof(uint32_t) * sort_scratch_words<uint64_t>(kHashKeyBits, max_keys_per_call));
  alloc(&h->status, sizeof(uint32_t));
  alloc(&h->touch, sizeof(uint32_t) * (size_t)kTouchLists * (size_t)max_keys_per_call);
  alloc(&h->touch_n, sizeof(uint32_t) * kTouchLists);
  if (e == cudaSuccess) e = cudaMemset(h->W, 0, sizeof(float) * (size_t)row_capacity * dim);
  if (e == cudaSuccess) e = cudaMemset(h->acc, 0, sizeof(float) * (size_t)row_capacity * dim);
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(uint32_t));
  if (e == cudaSuccess) {
    k_hash_init<<<h->sm_count * 8, 256>>>(h->slots, num_slots, h->used, h->n_words, row_capacity);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_hash(h);
    cudaGetLastError();
    return cuda_status(e);
  }
  *out = h;
  return EMB_OK;
}

extern "C" emb_status hash_rows(emb_hash h, float** weight, float** acc) {
  if (!h) return EMB_ERR_INVALID_ARG;
  if (weight) *weight = h->W;
  if (acc) *acc = h->acc;
  return EMB_OK;
}

extern "C" emb_status hash_lookup_or_insert(emb_hash h, const int32_t* table_ids, const int64_t* keys, int64_t n,
                                            uint32_t step, int64_t* rows_out, void* stream_) {
  if (!h || n < 0 || step == kNeverSeen) return EMB_ERR_INVALID_ARG;
  if (n > h->max_keys) return EMB_ERR_UNSUPPORTED;
  if (n == 0) return EMB_OK;
  if (!table_ids || !keys || !rows_out) return EMB_ERR_INVALID_ARG;
  cudaStream_t stream = (cudaStream_t)stream_;
  HashArgs a{};
  a.slots = h->slots;
  a.mask = (uint64_t)h->num_slots - 1;
  a.max_probes = h->max_probes;
  a.thr = h->thr;
  a.n_new = h->counters;
  a.nkeys = h->nkeys[0];
  a.nvals = h->nvals[0];
  a.max_keys = h->max_keys;
  a.status = h->status;
  // the list for this call's first touches: a fresh one per step; a second
  // call at the same step, or no free list, leaves touches unlisted, and
  // expiry then sweeps all slots until those touches have aged out
  a.touch = nullptr;
  a.touch_n = nullptr;
  int fresh = -1;
  if (!(h->cur_list >= 0 && h->list_step[h->cur_list] == step))
    for (int l = 0; l < kTouchLists; ++l)
      if (!h->list_live[l]) {
        fresh = l;
        break;
      }
  if (fresh >= 0) {
    EMB_CUDA_TRY(cudaMemsetAsync(h->touch_n + fresh, 0, sizeof(uint32_t), stream));
    h->list_live[fresh] = true;
    h->list_step[fresh] = step;
    h->cur_list = fresh;
    a.touch = h->touch + (size_t)fresh * (size_t)h->max_keys;
    a.touch_n = h->touch_n + fresh;
  } else {
    h->lists_valid = false;
    if ((int64_t)step > h->unrecorded_step) h->unrecorded_step = step;
  }
  EMB_CUDA_TRY(cudaMemsetAsync(h->counters, 0, sizeof(uint32_t), stream));
  k_hash_probe<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(a, table_ids, keys, n, step, rows_out);
  int res = 0;
  emb_status st = radix_sort_pairs<uint64_t>(h->nkeys, h->nvals, 0, h->counters, n, kHashKeyBits, h->sort_scratch,
                                             h->sm_count, h->status, stream, &res);
  if (st != EMB_OK) return st;
  const int nb = (int)((h->n_words + kScanBlk - 1) / kScanBlk);
  k_free_reduce<<<nb, kScanBlk, 0, stream>>>(h->used, h->n_words, h->scan_part);
  k_scan_parts<<<1, kScanBlk, 0, stream>>>(h->scan_part, nb);
  k_free_down<<<nb, kScanBlk, 0, stream>>>(h->used, h->n_words, h->scan_part, h->free_scan, h->counters,
                                           h->max_keys, h->free_rows);
  k_hash_admit<<<h->sm_count * 4, 256, 0, stream>>>(h->slots, h->nkeys[res], h->nvals[res], h->counters,
                                                     h->max_keys, h->free_scan, h->free_rows, h->n_words, h->W,
                                                     h->acc, h->dim, h->seed, h->init_scale, h->status,
                                                     sort_fail_word<uint64_t>(h->sort_scratch, kHashKeyBits));
  k_hash_mark<<<h->sm_count * 2, 256, 0, stream>>>(h->slots, h->nvals[res], h->counters, h->max_keys, h->used,
                                                   sort_fail_word<uint64_t>(h->sort_scratch, kHashKeyBits));
  k_hash_fix<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(h->slots, n, rows_out);
  return cuda_status(cudaGetLastError());
}

extern "C" emb_status hash_evict_expired(emb_hash h, uint32_t now, uint32_t ttl, void* stream_,
                                         int64_t* n_evicted_dev) {
  if (!h) return EMB_ERR_INVALID_ARG;
  cudaStream_t stream = (cudaStream_t)stream_;
  if (n_evicted_dev) EMB_CUDA_TRY(cudaMemsetAsync(n_evicted_dev, 0, sizeof(int64_t), stream));
  // lists whose step is more than ttl behind `now`: every entry idle longer
  // than ttl is on one of them (while the lists are complete)
  EvictLists L{};
  for (int l = 0; l < kTouchLists; ++l)
    if (h->list_live[l] && (int64_t)now - (int64_t)h->list_step[l] > (int64_t)ttl) {
      L.list[L.n] = h->touch + (size_t)l * (size_t)h->max_keys;
      L.count[L.n] = h->touch_n + l;
      ++L.n;
      h->list_live[l] = false;
      if (h->cur_list == l) h->cur_list = -1;
    }
  if (!h->lists_valid) {
    k_hash_evict<<<h->sm_count * 8, 256, 0, stream>>>(h->slots, h->num_slots, now, ttl, h->used,
                                                       reinterpret_cast<unsigned long long*>(n_evicted_dev));
    // the unlisted touches are all expired once now is past them by more than ttl
    if ((int64_t)now - h->unrecorded_step > (int64_t)ttl) {
      h->lists_valid = true;
      h->unrecorded_step = -1;
    }
  } else if (L.n > 0) {
    k_hash_evict_lists<<<h->sm_count * 4, 256, 0, stream>>>(h->slots, (uint64_t)h->num_slots - 1, L, h->max_keys,
                                                             now, ttl, h->used,
                                                             reinterpret_cast<unsigned long long*>(n_evicted_dev));
  }
  return cuda_status(cudaGetLastError());
}

extern "C" emb_status hash_export(emb_hash h, int32_t* tids, int64_t* keys, int64_t* rows, int32_t* counts,
                                  uint32_t* last_seen, int64_t cap, int64_t* n_out, void* stream_) {
  if (!h || !n_out || cap < 0) return EMB_ERR_INVALID_ARG;
  cudaStream_t stream = (cudaStream_t)stream_;
  EMB_CUDA_TRY(cudaMemsetAsync(h->counters + 1, 0, sizeof(uint32_t), stream));
  k_hash_export<<<h->sm_count * 8, 256, 0, stream>>>(h->slots, h->num_slots, tids, keys, rows, counts, last_seen,
                                                      cap, h->counters + 1);
  EMB_CUDA_TRY(cudaGetLastError());
  uint32_t cnt = 0;
  EMB_CUDA_TRY(cudaMemcpyAsync(&cnt, h->counters + 1, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream));
  EMB_CUDA_TRY(cudaStreamSynchronize(stream));
  *n_out = cnt;
  return EMB_OK;
}

extern "C" emb_status hash_import(emb_hash h, const int32_t* tids, const int64_t* keys, const int64_t* rows,
                                  const int32_t* counts, const uint32_t* last_seen, int64_t n, void* stream_) {
  if (!h || n < 0) return EMB_ERR_INVALID_ARG;
  if (n > h->num_slots) return EMB_ERR_UNSUPPORTED;
  if (n > 0 && (!tids || !keys || !rows || !last_seen)) return EMB_ERR_INVALID_ARG;
  cudaStream_t stream = (cudaStream_t)stream_;
  // clear: every slot EMPTY, every row of the pool free
  k_hash_init<<<h->sm_count * 8, 256, 0, stream>>>(h->slots, h->num_slots, h->used, h->n_words, h->cap);
  EMB_CUDA_TRY(cudaMemsetAsync(h->counters + 2, 0, sizeof(uint32_t), stream));
  if (n > 0)
    k_hash_import<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
        h->slots, (uint64_t)h->num_slots - 1, h->max_probes, h->cap, h->used, tids, keys, rows, counts, last_seen, n,
        h->status, h->counters + 2);
  EMB_CUDA_TRY(cudaGetLastError());
  uint32_t latest = 0;
  EMB_CUDA_TRY(cudaMemcpyAsync(&latest, h->counters + 2, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream));
  EMB_CUDA_TRY(cudaStreamSynchronize(stream));
  // no touch list holds the imported entries: expiries sweep every slot
  // until the latest imported step is more than ttl behind
  for (int l = 0; l < kTouchLists; ++l) h->list_live[l] = false;
  h->cur_list = -1;
  h->lists_valid = n == 0;
  h->unrecorded_step = n == 0 ? -1 : (int64_t)latest;
  return EMB_OK;
}

extern "C" emb_status hash_get_device_status(emb_hash h, void* stream) {
  if (!h) return EMB_ERR_INVALID_ARG;
  uint32_t st = 0;
  EMB_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
  EMB_CUDA_TRY(cudaMemcpy(&st, h->status, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  EMB_CUDA_TRY(cudaMemset(h->status, 0, sizeof(uint32_t)));
  return (emb_status)st;
}

extern "C" emb_status hash_destroy(emb_hash h) {
  if (!h) return EMB_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  free_hash(h);
  return EMB_OK;
}
