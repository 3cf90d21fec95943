// backward.cu -- K-B: radix sort of (global row, gradient source) pairs,
// per-unique-row gradient reduction and the fused sparse Adagrad update.
#include "plan.cuh"

namespace emb {

emb_status launch_backward(emb_plan_s* p, const float* grad_out, const float* grad_seq, float lr,
                           float eps, cudaStream_t stream, const emb_backward_debug* dbg) {
  (void)p; (void)grad_out; (void)grad_seq; (void)lr; (void)eps; (void)stream; (void)dbg;
  return EMB_ERR_UNSUPPORTED;
}

}  // namespace emb
