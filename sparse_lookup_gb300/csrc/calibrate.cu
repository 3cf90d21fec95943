// calibrate.cu -- measurement support: a gather-only kernel that reads
// random rows of a table with the same access shape as the forward (16-byte
// loads by dim/4-lane groups, eight rows in flight per lane group) and does
// nothing else, so a benchmark can measure the random-row gather rate this
// GPU sustains for a row size.
#include "plan.cuh"

namespace emb {

// Lane group of 2^GLOG lanes per row; a lane loads R float4 of its row (R = 2
// only for rows wider than 128 floats).  All U*R loads of an iteration are
// straight-line and independent, so a warp keeps U rows in flight per group.
template <int GLOG, int R>
__global__ void __launch_bounds__(256) k_gather_only(const float* __restrict__ E, int dim,
                                                     const uint32_t* __restrict__ idx, int64_t n,
                                                     float* __restrict__ sink) {
  constexpr int G = 32 >> GLOG;
  constexpr int U = 8;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> GLOG, sub = lane & ((1 << GLOG) - 1);
  const int dim4 = dim / 4;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t base = warp * G * U; base < n; base += nwarps * G * U) {
    float4 v[U][R];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + u * G + grp;
      const float4* row = i < n ? reinterpret_cast<const float4*>(E + (int64_t)__ldg(idx + i) * dim) : nullptr;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int f4 = sub + 32 * r;
        v[u][r] = (row && f4 < dim4) ? __ldg(row + f4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        acc.x += v[u][r].x;
        acc.y += v[u][r].y;
        acc.z += v[u][r].z;
        acc.w += v[u][r].w;
      }
  }
  if (acc.x == 1.2345e-38f && sink) sink[0] = acc.y + acc.z + acc.w;   // keeps the loads alive
}

}  // namespace emb

extern "C" emb_status emb_calibrate_gather(const float* table, int64_t num_rows, int32_t dim,
                                           const uint32_t* row_idx, int64_t n, float* sink, void* stream) {
  using namespace emb;
  if (!table || !row_idx || n < 0 || num_rows < 1 || dim < 4 || dim % 4 || dim > 256 || !aligned16(table))
    return EMB_ERR_INVALID_ARG;
  int dev = 0, sms = 1;
  EMB_CUDA_TRY(cudaGetDevice(&dev));
  EMB_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int dim4 = dim / 4;
  int glog = 0;
  while ((1 << glog) < (dim4 > 32 ? 32 : dim4)) ++glog;
  const unsigned grid = (unsigned)sms * 8;
  cudaStream_t s = (cudaStream_t)stream;
  switch (glog) {
    case 0: k_gather_only<0, 1><<<grid, 256, 0, s>>>(table, dim, row_idx, n, sink); break;
    case 1: k_gather_only<1, 1><<<grid, 256, 0, s>>>(table, dim, row_idx, n, sink); break;
    case 2: k_gather_only<2, 1><<<grid, 256, 0, s>>>(table, dim, row_idx, n, sink); break;
    case 3: k_gather_only<3, 1><<<grid, 256, 0, s>>>(table, dim, row_idx, n, sink); break;
    case 4: k_gather_only<4, 1><<<grid, 256, 0, s>>>(table, dim, row_idx, n, sink); break;
    default:
      if (dim4 > 32) k_gather_only<5, 2><<<grid, 256, 0, s>>>(table, dim, row_idx, n, sink);
      else k_gather_only<5, 1><<<grid, 256, 0, s>>>(table, dim, row_idx, n, sink);
      break;
  }
  return cuda_status(cudaGetLastError());
}
