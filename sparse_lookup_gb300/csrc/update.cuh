// update.cuh -- pieces both backward kinds share: the table a global row
// key belongs to, and the fp32 Adagrad step (library-internal).
#pragma once

#include "common.cuh"

namespace emb {

__device__ __forceinline__ int table_of_key(const uint32_t* base, int nt, uint32_t key) {
  int lo = 0, hi = nt;  // largest t with base[t] <= key
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(base + mid) <= key) lo = mid; else hi = mid;
  }
  return lo;
}

// One Adagrad step on one element (torch.optim.Adagrad with lr_decay =
// weight_decay = 0, eps outside the root): acc += g*g; w -= lr*g/(sqrt(acc)+eps).
// The square root and the reciprocal use the hardware's approximate forms
// (within a couple of ulp): the accumulator is exact, the weight step
// lr*g/(sqrt(acc)+eps) carries a relative error of about 1e-7.
__device__ __forceinline__ void adagrad1_fast(float& w, float& acc, float g, float lr, float eps) {
  const float a = __fadd_rn(acc, __fmul_rn(g, g));
  float r, inv;
  asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(a));
  const float den = __fadd_rn(r, eps);
  asm("rcp.approx.f32 %0, %1;" : "=f"(inv) : "f"(den));
  acc = a;
  w = __fsub_rn(w, __fmul_rn(__fmul_rn(lr, g), inv));
}


}  // namespace emb
