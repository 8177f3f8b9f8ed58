// KV append: write the round's new K/V rows into their page slots.
// One warp per new row; a row's [H_kv, d] block is contiguous on both sides,
// so the copy is whole 16-byte vectors, coalesced on the read and the write.
// Shared by the stand-alone append kernel and the prep launch of a mixed step
// (append and extend schedule in one launch).
#pragma once

#include "cpe_device.cuh"
#include "kernels.h"

namespace cpe {

namespace {

constexpr int kAppendRowsPerBlock = 8;  // 256-thread blocks, one warp per row

__device__ __forceinline__ int seq_of_row(const int32_t* qo_indptr, int n_seqs, int row) {
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qo_indptr[mid] <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Row `row` of the round's new K/V, copied by one warp (lane 0..31).
__device__ __forceinline__ void append_row(const KvAppendArgs& a, int row, int lane) {
  if (row >= a.total_q) return;
  const int s = seq_of_row(a.qo_indptr, a.n_seqs, row);
  const int pos = a.prefix_len[s] + row - a.qo_indptr[s];
  if (s >= a.staged_from && a.prefix_len[s] % a.page_size == 0) {
    // the extend launch writes this sequence's full new pages from its staged tiles
    const int full = (a.qo_indptr[s + 1] - a.qo_indptr[s]) / a.page_size * a.page_size;
    if (row - a.qo_indptr[s] < full) return;
  }
  const int pidx = pos / a.page_size;
  if (pos < 0 || pidx >= a.max_pages) {
    if (lane == 0) record_error(a.status, kStatusDeviceArg, kDetailBadLength);
    return;
  }
  const int pid = a.page_table[static_cast<int64_t>(s) * a.max_pages + pidx];
  if (pid < 0 || pid >= a.num_pages) {
    if (lane == 0) record_error(a.status, kStatusDeviceArg, kDetailBadPage);
    return;
  }
  const int64_t dst = (static_cast<int64_t>(pid) * a.page_size + pos % a.page_size) * a.row_bytes;
  const int64_t src = static_cast<int64_t>(row) * a.row_bytes;
  const int nvec = a.row_bytes >> 4;
  const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.k_new) + src);
  const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.v_new) + src);
  uint4* kd = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.k_cache) + dst);
  uint4* vd = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.v_cache) + dst);
  for (int x = lane; x < nvec; x += 32) {
    const uint4 kv = __ldg(ks + x);
    const uint4 vv = __ldg(vs + x);
    kd[x] = kv;
    vd[x] = vv;
  }
}

}  // namespace

}  // namespace cpe
