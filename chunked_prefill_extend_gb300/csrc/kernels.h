// Kernel-launch interfaces between the C ABI layer (api.cu) and the kernel
// translation units.  Host-side only; no torch types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cpe {

constexpr int kBlockM = 128;   // query rows (token x head-in-group) per extend tile
constexpr int kBlockN = 128;   // keys per extend K/V tile
constexpr int kPage = 16;      // page size (tokens)
constexpr int kDecodeSplit = 2048;  // keys per decode split

struct TileEntry {  // one extend work unit
  int seq;
  int q_tile;
  int kv_head;
  int pad;
};

struct ScheduleArgs {
  const int32_t* qo_indptr;
  const int32_t* prefix_len;
  int seq_begin, seq_end;   // sequences [seq_begin, seq_end) take part
  int tok;                  // tokens per tile (kBlockM / G)
  int h_kv;
  int max_kv_len;
  int max_pages;
  int capacity;             // entries in `tiles` (the launch's grid size)
  TileEntry* tiles;
  int* status;
};

struct ExtendTcArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  const int32_t* page_table;
  const int32_t* qo_indptr;
  const int32_t* prefix_len;
  const TileEntry* tiles;
  void* out;
  float* lse;
  int* status;
  int64_t num_pages;
  int max_pages;
  int h_q, h_kv, group, tok, d;
  float scale_log2;
  uint64_t wait_ns;
  int n_ctas;
};

struct ExtendSimtArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* page_table;
  const int32_t* qo_indptr;
  const int32_t* prefix_len;
  void* out;
  float* lse;
  int* status;
  int64_t num_pages;
  int max_pages, n_seqs, seq_begin, total_q, row_begin, h_q, h_kv, d, page_size, max_kv_len;
  float sm_scale;
  int f32;  // 1 = fp32 data, 0 = bf16
};

struct KvAppendArgs {
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int32_t* page_table;
  const int32_t* qo_indptr;
  const int32_t* prefix_len;
  int* status;
  int64_t num_pages;
  int max_pages, n_seqs, total_q, row_bytes, page_size;
};

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* page_table;
  const int32_t* qo_indptr;   // nullable: row of sequence s is qo_indptr[s] (else s)
  const int32_t* prefix_len;
  void* out;
  float* lse;
  float* part_o;   // [n_seqs, h_q, max_splits, d] normalised partial outputs
  float* part_ml;  // [n_seqs, h_q, max_splits, 2] (m in log2 units, l)
  int* status;
  int64_t num_pages;
  int max_pages, n_seqs, seq_begin, h_q, h_kv, d, max_kv_len, max_splits;
  float scale_log2;
};

cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t s);
cudaError_t launch_extend_tc(const ExtendTcArgs& a, cudaStream_t s);
cudaError_t launch_extend_simt(const ExtendSimtArgs& a, cudaStream_t s);
cudaError_t launch_kv_append(const KvAppendArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
size_t extend_tc_smem_bytes(int d);

}  // namespace cpe
