// common.cuh -- helpers shared by the kernels and the host side of the
// library: status latching, the hash transform, exact division by a runtime
// invariant, and the per-column / per-table metadata the kernels read.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "emb.h"

#define EMB_HD __host__ __device__ __forceinline__

namespace emb {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Hash transform: one SplitMix64 output with the state set to x
// (Steele, Lea & Flood, OOPSLA 2014; the gamma is added before mixing).
// ---------------------------------------------------------------------------
EMB_HD uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

EMB_HD uint64_t mulhi64(uint64_t a, uint64_t b) {
#ifdef __CUDA_ARCH__
  return __umul64hi(a, b);
#else
  return (uint64_t)(((unsigned __int128)a * (unsigned __int128)b) >> 64);
#endif
}

// ---------------------------------------------------------------------------
// Unsigned 64-bit division by a runtime-invariant divisor d >= 1 with one
// multiply-high, two shifts and an add (Granlund & Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, Figure 4.1 with N=64):
//   l = ceil(log2 d), m = floor(2^64 (2^l - d) / d) + 1,
//   t = mulhi(m, z), q = (t + ((z - t) >> min(l,1))) >> max(l-1,0).
// Exact for every 64-bit z.  The magic is computed once on the host.
// ---------------------------------------------------------------------------
struct DivMagic {
  uint64_t m;
  uint64_t d;
  uint32_t sh1, sh2;
};

inline DivMagic make_div_magic(uint64_t d) {
  DivMagic g{};
  g.d = d;
  uint32_t l = 0;
  while (l < 64 && ((unsigned __int128)1 << l) < (unsigned __int128)d) ++l;
  unsigned __int128 two_l = (unsigned __int128)1 << l;
  unsigned __int128 num = (two_l - d) << 64;
  g.m = (uint64_t)(num / d) + 1;
  g.sh1 = l < 1 ? l : 1;
  g.sh2 = l > 1 ? l - 1 : 0;
  return g;
}

EMB_HD uint64_t div_magic(uint64_t z, const DivMagic& g) {
  uint64_t t = mulhi64(g.m, z);
  return (t + ((z - t) >> g.sh1)) >> g.sh2;
}

EMB_HD uint64_t mod_magic(uint64_t z, const DivMagic& g) { return z - div_magic(z, g) * g.d; }

// 32-bit variant for dividing segment indices by the batch size.
struct DivMagic32 {
  uint32_t m, d, sh1, sh2;
};

inline DivMagic32 make_div_magic32(uint32_t d) {
  DivMagic32 g{};
  g.d = d;
  uint32_t l = 0;
  while (l < 32 && (1ull << l) < (uint64_t)d) ++l;
  uint64_t num = ((1ull << l) - d) << 32;
  g.m = (uint32_t)(num / d) + 1;
  g.sh1 = l < 1 ? l : 1;
  g.sh2 = l > 1 ? l - 1 : 0;
  return g;
}

EMB_HD uint32_t div_magic32(uint32_t z, const DivMagic32& g) {
#ifdef __CUDA_ARCH__
  uint32_t t = __umulhi(g.m, z);
#else
  uint32_t t = (uint32_t)(((uint64_t)g.m * z) >> 32);
#endif
  return (t + ((z - t) >> g.sh1)) >> g.sh2;
}

// ---------------------------------------------------------------------------
// Device-side status word: the first error wins and stays until read.
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
__device__ __forceinline__ void latch(uint32_t* st, uint32_t code) {
  if (st && *((volatile uint32_t*)st) == 0u) atomicCAS(st, 0u, code);
}

// Programmatic dependent launch.  A kernel launched by launch_dependent()
// may be scheduled before the kernel ahead of it in the stream has finished:
// it calls pdl_wait() before its first memory access, which returns once
// that kernel has completed and its writes are visible (and at once for a
// kernel launched the ordinary way).  The kernel ahead calls pdl_trigger()
// to let its dependant's CTAs be scheduled once all of its own CTAs have
// started, so the dependant's launch overlaps its last wave.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif

// Launch `kernel` so that it may start while the previous kernel in the
// stream finishes (it must begin with pdl_wait()).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                                    cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------------------
// Metadata the kernels read.
// ---------------------------------------------------------------------------
struct ColMeta {
  const float* weight;     // table [num_rows, dim] in dtype
  float* acc;              // Adagrad accumulator (training)
  const float* qscale;     // EMB_DT_I8: per-row scale
  const float* dflt;       // default vector or nullptr
  const float* bnd;        // bucketize boundaries
  int64_t num_rows;
  DivMagic mod;            // HASH_MOD: division by num_rows
  int64_t seq_unit;        // padded: float offset of the column's block for batch 1
  int32_t dim;
  int32_t dim4;            // dim / 4
  int32_t nb;
  int32_t transform;
  int32_t pooling;
  int32_t pad_len;
  int32_t trunc;           // pooled: only the first trunc values of a bag (0 = all)
  int32_t table;
  uint32_t table_base;     // first global row of the column's table
  int32_t out_col;         // pooled: float offset inside an output row
  int32_t col;             // plan column index
  int32_t dtype;           // emb_table_dtype of the rows
};

struct TableMeta {
  float* weight;
  float* acc;
  int64_t num_rows;
  int32_t dim;
  int32_t dim4;
};

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace emb

// Handle layouts (library-internal).
struct emb_plan_s;
struct emb_hash_s;
