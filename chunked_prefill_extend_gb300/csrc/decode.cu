// Decode rows (query length 1): the stand-alone split-KV decode kernel (one
// item of decode_item.cuh per CTA) and the merge of a row's splits.
#include <atomic>

#include "decode_item.cuh"

namespace cpe {

namespace {

template <int D>
__global__ void __launch_bounds__(128) decode_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t dsm[];
  decode_item<D>(a, blockIdx.x, blockIdx.y, blockIdx.z, dsm, threadIdx.x, 0);
}

// Combine the splits of each (decode row, head) by the online-softmax rule.
template <int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(DecodeArgs a) {
  const int sidx = blockIdx.x;
  const int head = blockIdx.y;
  const int s = a.seq_begin + sidx;
  const DecodeSeq dq = decode_seq(a, s, false);
  if (!dq.ok) return;
  const int ns = (dq.L + kDecodeSplit - 1) / kDecodeSplit;
  if (ns <= 1) return;
  const int c = threadIdx.x;
  const int64_t base = (static_cast<int64_t>(sidx) * a.h_q + head) * a.max_splits;
  float M = -INFINITY;
  for (int k = 0; k < ns; ++k) M = fmaxf(M, a.part_ml[(base + k) * 2]);
  float num = 0.f, den = 0.f;
  for (int k = 0; k < ns; ++k) {
    const float wt = fast_exp2(a.part_ml[(base + k) * 2] - M) * a.part_ml[(base + k) * 2 + 1];
    num += wt * a.part_o[(base + k) * D + c];
    den += wt;
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  out[(static_cast<int64_t>(dq.row) * a.h_q + head) * D + c] = __float2bfloat16_rn(num / den);
  if (c == 0 && a.lse) a.lse[static_cast<int64_t>(dq.row) * a.h_q + head] = (M + __log2f(den)) * 0.69314718055994531f;
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t s) {
  const int smem = DecCfg<D>::kSmem;
  static std::atomic<int> ready[64];  // the shared-memory opt-in, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !ready[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) ready[dev].store(1, std::memory_order_release);
  }
  dim3 grid(a.max_splits, a.n_seqs, a.h_kv);
  decode_kernel<D><<<grid, 128, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.max_splits <= 1) return e;
  decode_merge_kernel<D><<<dim3(a.n_seqs, a.h_q), D, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t s) {
  if (a.n_seqs <= 0 || a.max_splits <= 1) return cudaSuccess;
  if (a.d == 128)
    decode_merge_kernel<128><<<dim3(a.n_seqs, a.h_q), 128, 0, s>>>(a);
  else
    decode_merge_kernel<64><<<dim3(a.n_seqs, a.h_q), 64, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.n_seqs <= 0) return cudaSuccess;
  return a.d == 128 ? launch_decode_d<128>(a, s) : launch_decode_d<64>(a, s);
}

}  // namespace cpe
