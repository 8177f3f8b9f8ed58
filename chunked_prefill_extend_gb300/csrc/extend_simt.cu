// Extend attention on CUDA cores in fp32 arithmetic: the path for fp32 data
// (exact fp32 inputs, no tensor-core rounding).  One warp per (query row,
// head); each lane holds d/32 dimensions of q, keys are visited one at a time
// with a warp-reduced dot product and a running (m, l, o).
#include "cpe_device.cuh"
#include "kernels.h"

namespace cpe {

namespace {

template <typename T>
__device__ __forceinline__ float ld(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld<float>(const float* p, int64_t i) { return __ldg(p + i); }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st(T* p, int64_t i, float v);
template <>
__device__ __forceinline__ void st<float>(float* p, int64_t i, float v) { p[i] = v; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

template <typename T, int DPL>  // DPL = d / 32 dimensions per lane
__global__ void __launch_bounds__(128) extend_simt_kernel(ExtendSimtArgs a) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int n_rows = a.total_q - a.row_begin;
  if (warp >= n_rows * a.h_q) return;
  const int row = a.row_begin + warp / a.h_q;
  const int h = warp % a.h_q;
  int lo = a.seq_begin, hi = a.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.qo_indptr[mid] <= row) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  const int E = a.qo_indptr[s + 1] - a.qo_indptr[s];
  const int P = a.prefix_len[s];
  if (P + E > a.max_kv_len || (P + E + a.page_size - 1) / a.page_size > a.max_pages) {
    if (lane == 0) record_error(a.status, kStatusDeviceArg, kDetailBadLength);
    return;
  }
  const int i = row - a.qo_indptr[s];
  const int g = h / (a.h_q / a.h_kv);
  const T* q = static_cast<const T*>(a.q);
  const T* kc = static_cast<const T*>(a.k_cache);
  const T* vc = static_cast<const T*>(a.v_cache);
  float qr[DPL], o[DPL];
  const int64_t qoff = (static_cast<int64_t>(row) * a.h_q + h) * a.d;
#pragma unroll
  for (int x = 0; x < DPL; ++x) {
    qr[x] = ld(q, qoff + lane * DPL + x);
    o[x] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int32_t* pt = a.page_table + static_cast<int64_t>(s) * a.max_pages;
  const int last = P + i;
  for (int j = 0; j <= last; ++j) {
    const int pid = pt[j / a.page_size];
    if (pid < 0 || pid >= a.num_pages) {
      if (lane == 0) record_error(a.status, kStatusDeviceArg, kDetailBadPage);
      return;
    }
    const int64_t koff = ((static_cast<int64_t>(pid) * a.page_size + j % a.page_size) * a.h_kv + g) * a.d +
                         lane * DPL;
    float dot = 0.f;
#pragma unroll
    for (int x = 0; x < DPL; ++x) dot = fmaf(qr[x], ld(kc, koff + x), dot);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o2);
    const float sc = dot * a.sm_scale;
    const float m_new = fmaxf(m, sc);
    const float corr = expf(m - m_new);
    const float p = expf(sc - m_new);
    l = l * corr + p;
#pragma unroll
    for (int x = 0; x < DPL; ++x) o[x] = fmaf(o[x], corr, p * ld(vc, koff + x));
    m = m_new;
  }
  T* out = static_cast<T*>(a.out);
  const float inv = 1.f / l;
#pragma unroll
  for (int x = 0; x < DPL; ++x) st(out, qoff + lane * DPL + x, o[x] * inv);
  if (lane == 0 && a.lse != nullptr) a.lse[static_cast<int64_t>(row) * a.h_q + h] = m + logf(l);
}

}  // namespace

cudaError_t launch_extend_simt(const ExtendSimtArgs& a, cudaStream_t s) {
  const int64_t warps = static_cast<int64_t>(a.total_q - a.row_begin) * a.h_q;
  if (warps <= 0) return cudaSuccess;
  const int blocks = static_cast<int>((warps + 3) / 4);
  if (a.f32) {
    if (a.d == 64) extend_simt_kernel<float, 2><<<blocks, 128, 0, s>>>(a);
    else extend_simt_kernel<float, 4><<<blocks, 128, 0, s>>>(a);
  } else {
    if (a.d == 64) extend_simt_kernel<__nv_bfloat16, 2><<<blocks, 128, 0, s>>>(a);
    else extend_simt_kernel<__nv_bfloat16, 4><<<blocks, 128, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace cpe
