// Extend attention on CUDA cores in fp32 arithmetic: the path for fp32 data
// (exact fp32 inputs, no tensor-core rounding).  One warp per (query row,
// head), keys in blocks of 32: each lane scores one key of the block against
// the whole query row, the warp takes the block's max and sum for the running
// (m, l), and each lane accumulates d/32 output dimensions over the block's
// weighted values.
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
  constexpr int D = 32 * DPL;
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
  // every lane holds the whole query row (for its key's dot product) and
  // DPL output dimensions
  float qr[D], o[DPL];
  const int64_t qoff = (static_cast<int64_t>(row) * a.h_q + h) * D;
#pragma unroll
  for (int x = 0; x < D; ++x) qr[x] = ld(q, qoff + x);
#pragma unroll
  for (int x = 0; x < DPL; ++x) o[x] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int32_t* pt = a.page_table + static_cast<int64_t>(s) * a.max_pages;
  const int last = P + i;
  // Keys in blocks of 32, lane j scoring key kb + j: one warp max and sum per
  // block for the running (m, l), then the block's weighted values.
  for (int kb = 0; kb <= last; kb += 32) {
    const int j = kb + lane;
    int64_t krow = 0;
    float sc = -INFINITY;
    if (j <= last) {
      const int pid = pt[j / a.page_size];
      if (pid < 0 || pid >= a.num_pages) {
        record_error(a.status, kStatusDeviceArg, kDetailBadPage);
      } else {
        krow = ((static_cast<int64_t>(pid) * a.page_size + j % a.page_size) * a.h_kv + g) * D;
        float dot[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (sizeof(T) == 4) {  // the key row in 16-byte vectors
          const float4* kr = reinterpret_cast<const float4*>(kc + krow);
#pragma unroll
          for (int x = 0; x < D / 4; ++x) {
            const float4 k4 = __ldg(kr + x);
            dot[0] = fmaf(qr[4 * x], k4.x, dot[0]);
            dot[1] = fmaf(qr[4 * x + 1], k4.y, dot[1]);
            dot[2] = fmaf(qr[4 * x + 2], k4.z, dot[2]);
            dot[3] = fmaf(qr[4 * x + 3], k4.w, dot[3]);
          }
        } else {
#pragma unroll
          for (int x = 0; x < D; ++x) dot[x & 3] = fmaf(qr[x], ld(kc, krow + x), dot[x & 3]);
        }
        sc = ((dot[0] + dot[1]) + (dot[2] + dot[3])) * a.sm_scale;
      }
    }
    float mb = sc;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o2));
    const float m_new = fmaxf(m, mb);
    const float corr = m == -INFINITY ? 0.f : expf(m - m_new);
    const float p = sc == -INFINITY ? 0.f : expf(sc - m_new);
    float ps = p;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o2);
    l = l * corr + ps;
#pragma unroll
    for (int x = 0; x < DPL; ++x) o[x] *= corr;
    const int nk = min(32, last + 1 - kb);
#pragma unroll 8
    for (int jj = 0; jj < 32; ++jj) {  // (keys past the last have p = 0 and row 0: skipped)
      if (jj < nk) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const int64_t vrow = __shfl_sync(0xffffffffu, krow, jj);
#pragma unroll
        for (int x = 0; x < DPL; ++x) o[x] = fmaf(pj, ld(vc, vrow + lane * DPL + x), o[x]);
      }
    }
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
