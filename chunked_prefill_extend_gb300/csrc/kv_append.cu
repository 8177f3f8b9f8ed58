// The stand-alone KV append kernel (append_row of kv_append_row.cuh, one
// warp per row).
#include "kv_append_row.cuh"

namespace cpe {

namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(KvAppendArgs a) {
  append_row(a, blockIdx.x * kAppendRowsPerBlock + (threadIdx.x >> 5), threadIdx.x & 31);
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendArgs& a, cudaStream_t s) {
  if (a.total_q <= 0) return cudaSuccess;
  const int blocks = (a.total_q + kAppendRowsPerBlock - 1) / kAppendRowsPerBlock;
  kv_append_kernel<<<blocks, kAppendRowsPerBlock * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace cpe
