// The C ABI of libcpe: argument validation, workspace layout, TMA tensor
// maps, kernel launches and the device status word.  See include/cpe.h for
// the contract of every entry point.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "cpe.h"
#include "cpe_device.cuh"
#include "kernels.h"

// status[0]: first device error code since the last read, status[1]: detail.
__device__ int g_cpe_status[2];

namespace cpe {

namespace {

thread_local std::string t_last_error;
std::atomic<int64_t> g_wait_ns{4000000000LL};
std::atomic<int64_t> g_launches{0};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};

cpe_status fail(cpe_status st, const char* fn, const char* msg) {
  t_last_error = std::string(fn) + ": " + msg;
  return st;
}

cpe_status cuda_fail(const char* fn, cudaError_t e) {
  t_last_error = std::string(fn) + ": " + cudaGetErrorString(e);
  return CPE_ERR_CUDA;
}

// Device address of the status word on the current device.
int* status_ptr(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_cpe_status);
    if (*err != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 3-D bf16 map {d, heads, rows} with row stride heads*d, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int box_heads, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(heads) * d * 2};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// make_map through a small per-thread cache of encoded maps: successive calls
// on the same cache reuse its four maps (only the query map follows the chunk).
bool cached_map(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int box_heads, int box_rows) {
  struct Entry {
    CUtensorMap map;
    const void* base;
    int64_t rows;
    int d, heads, box_heads, box_rows;
  };
  constexpr int kEntries = 16;
  thread_local Entry cache[kEntries] = {};
  thread_local int next = 0;
  for (const Entry& e : cache)
    if (e.base == base && base != nullptr && e.rows == rows && e.d == d && e.heads == heads &&
        e.box_heads == box_heads && e.box_rows == box_rows) {
      *m = e.map;
      return true;
    }
  if (!make_map(m, base, d, heads, rows, box_heads, box_rows)) return false;
  Entry& e = cache[next];
  next = (next + 1) % kEntries;
  e.map = *m;
  e.base = base;
  e.rows = rows;
  e.d = d;
  e.heads = heads;
  e.box_heads = box_heads;
  e.box_rows = box_rows;
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  size_t header_off, units_off, items_off, split_off, partial_off, part_o_off, part_ml_off, total;
  int unit_capacity, max_splits, slots;
};

int group_of(int h_q, int h_kv) { return h_q / h_kv; }

// Workspace: the extend schedule (header, unit list, item table), the
// partial-result slots of units cut into key-range parts, then the decode
// split partials.
Layout workspace_layout(int n_seqs, int total_q, int h_q, int h_kv, int d, int max_kv_len) {
  Layout L{};
  const int G = group_of(h_q, h_kv);
  const int unit_tok = 2 * (kBlockM / G);
  const int64_t cap = static_cast<int64_t>(h_kv) * ((total_q + unit_tok - 1) / unit_tok + n_seqs);
  L.unit_capacity = static_cast<int>(cap);
  L.max_splits = (max_kv_len + kDecodeSplit - 1) / kDecodeSplit;
  L.header_off = 0;
  L.units_off = 256;
  L.items_off = L.units_off + align256(static_cast<size_t>(cap) * sizeof(UnitEntry));
  L.slots = static_cast<int>(cap * kMaxParts < kMaxSlots ? cap * kMaxParts : kMaxSlots);
  L.split_off = L.items_off + align256((static_cast<size_t>(cap) * kMaxParts + kMaxCtas) * sizeof(ItemDesc));
  L.partial_off = L.split_off + align256(static_cast<size_t>(L.slots / 2 + 1) * sizeof(UnitEntry));
  const size_t parts = static_cast<size_t>(n_seqs) * h_q * L.max_splits;
  L.part_o_off = L.partial_off + align256(static_cast<size_t>(L.slots) * partial_slot_bytes(d));
  L.part_ml_off = L.part_o_off + align256(parts * d * sizeof(float));
  L.total = L.part_ml_off + align256(parts * 2 * sizeof(float));
  return L;
}

ExtendSched sched_of(const Layout& L, void* ws) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  ExtendSched s;
  s.header = reinterpret_cast<int*>(b + L.header_off);
  s.units = reinterpret_cast<UnitEntry*>(b + L.units_off);
  s.items = reinterpret_cast<ItemDesc*>(b + L.items_off);
  s.split = reinterpret_cast<UnitEntry*>(b + L.split_off);
  s.partial = b + L.partial_off;
  return s;
}

// Whether the previous extend call on stream `s` used workspace `ws` (an
// unknown stream counts as yes); records `ws` as the stream's latest.  Only
// then can that call's launches still be reading the schedule this call
// writes: a call on another workspace lets the schedule be written as soon
// as it is computed, while the previous call finishes.
bool reuses_workspace(cudaStream_t s, const void* ws) {
  struct Entry {
    cudaStream_t stream;
    const void* ws;
  };
  constexpr int kEntries = 16;
  static std::mutex mu;
  static Entry table[kEntries] = {};
  static int next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (Entry& e : table)
    if (e.ws != nullptr && e.stream == s) {
      const bool same = e.ws == ws;
      e.ws = ws;
      return same;
    }
  table[next] = Entry{s, ws};
  next = (next + 1) % kEntries;
  return true;
}

// SMs of the current device (the persistent extend grid), at most kMaxCtas.
int persistent_ctas(cudaError_t* err) {
  static int cache[kMaxDevices] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev] == 0) {
    int sms = 0;
    *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (*err != cudaSuccess) return 0;
    cache[dev] = sms < kMaxCtas ? sms : kMaxCtas;
  }
  return cache[dev];
}

struct Common {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  int64_t num_pages;
  const int32_t* page_table;
  int32_t max_pages;
  const int32_t* qo_indptr;
  const int32_t* prefix_len;
  int32_t n_seqs, total_q, max_kv_len, h_q, h_kv, d, page_size;
  float sm_scale;
  cpe_dtype dtype;
  void* out;
  float* lse;
  void* workspace;
  size_t ws_bytes;
};

cpe_status validate(const char* fn, const Common& c, bool need_qo) {
  if (!c.q || !c.k_cache || !c.v_cache || !c.page_table || !c.prefix_len || !c.out || (need_qo && !c.qo_indptr))
    return fail(CPE_ERR_INVALID_ARG, fn, "null pointer argument");
  if (c.n_seqs <= 0 || c.total_q < 0 || c.max_kv_len <= 0 || c.max_pages <= 0 || c.num_pages <= 0 ||
      c.h_q <= 0 || c.h_kv <= 0 || c.d <= 0)
    return fail(CPE_ERR_INVALID_ARG, fn, "sizes must be positive (total_q >= 0)");
  if (c.num_pages > (int64_t(INT32_MAX) / kPage))
    return fail(CPE_ERR_INVALID_ARG, fn, "num_pages too large");
  if (!(c.sm_scale > 0.f) || !std::isfinite(c.sm_scale)) return fail(CPE_ERR_INVALID_ARG, fn, "sm_scale must be finite and > 0");
  if (c.h_q % c.h_kv != 0) return fail(CPE_ERR_INVALID_ARG, fn, "h_q must be a multiple of h_kv");
  const int G = c.h_q / c.h_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return fail(CPE_ERR_UNSUPPORTED, fn, "G = h_q/h_kv must be 1, 2, 4, 8 or 16");
  if (c.d != 64 && c.d != 128) return fail(CPE_ERR_UNSUPPORTED, fn, "head_dim must be 64 or 128");
  if (c.page_size != kPage) return fail(CPE_ERR_UNSUPPORTED, fn, "page_size must be 16");
  if (c.dtype != CPE_BF16 && c.dtype != CPE_F32) return fail(CPE_ERR_UNSUPPORTED, fn, "dtype must be CPE_BF16 or CPE_F32");
  if (!aligned(c.q, 16) || !aligned(c.k_cache, 16) || !aligned(c.v_cache, 16) || !aligned(c.out, 16) ||
      !aligned(c.page_table, 4) || !aligned(c.prefix_len, 4) || (c.qo_indptr && !aligned(c.qo_indptr, 4)) ||
      (c.lse && !aligned(c.lse, 4)))
    return fail(CPE_ERR_INVALID_ARG, fn, "misaligned pointer (16 bytes for tensors, 4 for index arrays)");
  const Layout L = workspace_layout(c.n_seqs, c.total_q, c.h_q, c.h_kv, c.d, c.max_kv_len);
  if (c.workspace == nullptr || c.ws_bytes < L.total)
    return fail(CPE_ERR_CAPACITY, fn, "workspace missing or smaller than cpe_workspace_size()");
  if (!aligned(c.workspace, 256)) return fail(CPE_ERR_INVALID_ARG, fn, "workspace must be 256-byte aligned");
  return CPE_OK;
}

// Split-KV decode of sequences [0, n_dec), one query row each.
DecodeArgs decode_args(const Common& c, const Layout& L, int n_dec, bool use_qo, int* status) {
  DecodeArgs a{};
  a.q = c.q; a.k_cache = c.k_cache; a.v_cache = c.v_cache; a.page_table = c.page_table;
  a.qo_indptr = use_qo ? c.qo_indptr : nullptr; a.prefix_len = c.prefix_len; a.out = c.out; a.lse = c.lse;
  a.part_o = reinterpret_cast<float*>(static_cast<uint8_t*>(c.workspace) + L.part_o_off);
  a.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(c.workspace) + L.part_ml_off);
  a.status = status; a.num_pages = c.num_pages; a.max_pages = c.max_pages; a.n_seqs = n_dec; a.seq_begin = 0;
  a.h_q = c.h_q; a.h_kv = c.h_kv; a.d = c.d; a.max_kv_len = c.max_kv_len; a.max_splits = L.max_splits;
  a.scale_log2 = c.sm_scale * 1.4426950408889634f;
  return a;
}

// Extend path over sequences [seq_begin, n_seqs), whose rows are [row_begin, total_q).
// With dec_rows > 0 (a mixed step, bf16) the decode rows [0, dec_rows) run in the
// same persistent launch on the CTAs the extend part leaves free; with `append`
// the round's K/V append shares the schedule's launch.
cpe_status run_extend(const char* fn, const Common& c, int seq_begin, int row_begin, int* status,
                      cudaStream_t stream, int dec_rows = 0, const KvAppendArgs* append = nullptr) {
  if (c.total_q - row_begin <= 0 || seq_begin >= c.n_seqs) return CPE_OK;
  const Layout L = workspace_layout(c.n_seqs, c.total_q, c.h_q, c.h_kv, c.d, c.max_kv_len);
  cudaError_t e;
  if (c.dtype == CPE_F32) {
    ExtendSimtArgs a{};
    a.q = c.q; a.k_cache = c.k_cache; a.v_cache = c.v_cache;
    a.page_table = c.page_table; a.qo_indptr = c.qo_indptr; a.prefix_len = c.prefix_len;
    a.out = c.out; a.lse = c.lse; a.status = status; a.num_pages = c.num_pages;
    a.max_pages = c.max_pages; a.n_seqs = c.n_seqs; a.seq_begin = seq_begin; a.total_q = c.total_q;
    a.row_begin = row_begin; a.h_q = c.h_q; a.h_kv = c.h_kv; a.d = c.d; a.page_size = c.page_size;
    a.max_kv_len = c.max_kv_len; a.sm_scale = c.sm_scale; a.f32 = 1;
    e = launch_extend_simt(a, stream);
    if (e != cudaSuccess) return cuda_fail(fn, e);
    g_launches += 1;
    return CPE_OK;
  }
  const int G = group_of(c.h_q, c.h_kv);
  const int tok = kBlockM / G;
  const ExtendSched sched = sched_of(L, c.workspace);
  const int n_rows = c.total_q - row_begin;
  const int n_seq = c.n_seqs - seq_begin;
  // units of two query tiles (256 rows) of one sequence and KV head
  const int unit_tok = 2 * tok;
  const int cap = c.h_kv * ((n_rows + unit_tok - 1) / unit_tok + n_seq);
  const int n_ctas = persistent_ctas(&e);
  if (n_ctas <= 0) return cuda_fail(fn, e);

  ScheduleArgs sa{};
  sa.qo_indptr = c.qo_indptr; sa.prefix_len = c.prefix_len; sa.seq_begin = seq_begin; sa.seq_end = c.n_seqs;
  sa.tok = tok; sa.h_kv = c.h_kv; sa.max_kv_len = c.max_kv_len; sa.max_pages = c.max_pages;
  sa.capacity = cap; sa.n_ctas = n_ctas; sa.max_slots = L.slots; sa.sched = sched; sa.status = status;
  sa.d = c.d;
  sa.dec_rows = dec_rows;
  sa.sched_wait = reuses_workspace(stream, c.workspace) ? 1 : 0;
  sa.dec_bytes_per_key = static_cast<int64_t>(c.h_kv) * c.d * 2 * 2;
  // dependent launches hide launch latency; worth it only on short launches
  const double flops_bound = 4.0 * c.d * c.h_q * static_cast<double>(n_rows) * c.max_kv_len;
  const bool dependent = flops_bound < kDependentLaunchFlops;
  // With the round's new rows at hand, a long extend launch reads the chunk's
  // keys from them and writes the full new pages of page-aligned sequences
  // into the cache itself; the prep launch appends the rest.  (On short
  // launches, and beside the decode rows of a fused mixed step, the stores'
  // share of the time measured slower than the prep launch's append, so there
  // the prep launch appends every row.)
  const bool staged = append != nullptr && !dependent && dec_rows == 0;
  KvAppendArgs ka{};
  if (append) {
    ka = *append;
    ka.staged_from = staged ? seq_begin : c.n_seqs;
  }
  e = append ? launch_prep(sa, ka, stream, dependent) : launch_schedule(sa, stream, dependent);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  g_launches += 1;

  ExtendTcArgs a;
  std::memset(&a, 0, sizeof a);
  if (!cached_map(&a.tm_q, c.q, c.d, c.h_q, c.total_q, G, tok) ||
      !cached_map(&a.tm_k, c.k_cache, c.d, c.h_kv, c.num_pages * kPage, 1, kPage) ||
      !cached_map(&a.tm_v, c.v_cache, c.d, c.h_kv, c.num_pages * kPage, 1, kPage) ||
      !cached_map(&a.tm_k128, c.k_cache, c.d, c.h_kv, c.num_pages * kPage, 1, kBlockN) ||
      !cached_map(&a.tm_v128, c.v_cache, c.d, c.h_kv, c.num_pages * kPage, 1, kBlockN) ||
      (staged && (!cached_map(&a.tm_kn, append->k_new, c.d, c.h_kv, c.total_q, 1, kPage) ||
                  !cached_map(&a.tm_vn, append->v_new, c.d, c.h_kv, c.total_q, 1, kPage) ||
                  !cached_map(&a.tm_kn128, append->k_new, c.d, c.h_kv, c.total_q, 1, kBlockN) ||
                  !cached_map(&a.tm_vn128, append->v_new, c.d, c.h_kv, c.total_q, 1, kBlockN))))
    return fail(CPE_ERR_CUDA, fn, "cuTensorMapEncodeTiled failed");
  a.page_table = c.page_table; a.qo_indptr = c.qo_indptr; a.prefix_len = c.prefix_len; a.sched = sched;
  a.out = c.out; a.lse = c.lse; a.status = status; a.num_pages = c.num_pages; a.max_pages = c.max_pages;
  a.h_q = c.h_q; a.h_kv = c.h_kv; a.group = G; a.tok = tok; a.d = c.d;
  a.staged = staged ? 1 : 0;
  a.scale_log2 = c.sm_scale * 1.4426950408889634f;
  a.wait_ns = static_cast<uint64_t>(g_wait_ns.load() < 0 ? 0 : g_wait_ns.load());
  a.n_ctas = n_ctas;
  a.max_split = std::max(1, std::min(cap, L.slots / 2));  // cut units: at most one per unit, two slots each
  if (dec_rows > 0) {
    a.dec = decode_args(c, L, dec_rows, true, status);
    a.dec_items = dec_rows * c.h_kv * L.max_splits;
  }
  e = launch_extend_tc(a, stream, dependent);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  g_launches += 2;  // the extend kernel and the merge of key-range parts
  if (dec_rows > 0 && L.max_splits > 1) {
    e = launch_decode_merge(a.dec, stream);
    if (e != cudaSuccess) return cuda_fail(fn, e);
    g_launches += 1;
  }
  return CPE_OK;
}

cpe_status run_decode(const char* fn, const Common& c, int n_dec, bool use_qo, int* status, cudaStream_t stream) {
  if (n_dec <= 0) return CPE_OK;
  const Layout L = workspace_layout(c.n_seqs, c.total_q, c.h_q, c.h_kv, c.d, c.max_kv_len);
  const DecodeArgs a = decode_args(c, L, n_dec, use_qo, status);
  const cudaError_t e = launch_decode(a, stream);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  g_launches += L.max_splits > 1 ? 2 : 1;
  return CPE_OK;
}

}  // namespace

void set_last_error(const std::string& msg) { t_last_error = msg; }

int* device_status_word(cudaError_t* err) { return status_ptr(err); }

void count_launches(int n) { g_launches += n; }

}  // namespace cpe

using namespace cpe;

extern "C" {

const char* cpe_last_error(void) { return t_last_error.c_str(); }

const char* cpe_status_string(cpe_status st) {
  switch (st) {
    case CPE_OK: return "ok";
    case CPE_ERR_INVALID_ARG: return "invalid argument";
    case CPE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case CPE_ERR_CAPACITY: return "buffer too small";
    case CPE_ERR_CUDA: return "CUDA error";
    case CPE_ERR_TIMEOUT: return "device wait timed out";
    case CPE_ERR_DEVICE_ARG: return "bad page id or length in device data";
  }
  return "unknown status";
}

int64_t cpe_set_wait_limit_ns(int64_t ns) { return g_wait_ns.exchange(ns < 0 ? 0 : ns); }

int64_t cpe_launch_count(void) { return g_launches.load(); }

size_t cpe_workspace_size(int32_t n_seqs, int32_t total_q, int32_t h_q, int32_t h_kv, int32_t d, int32_t max_kv_len) {
  if (n_seqs <= 0 || total_q < 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv || d <= 0 || max_kv_len <= 0) return 0;
  return workspace_layout(n_seqs, total_q, h_q, h_kv, d, max_kv_len).total;
}

cpe_status cpe_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, int64_t num_pages,
                         const int32_t* page_table, int32_t max_pages, const int32_t* qo_indptr,
                         const int32_t* prefix_len, int32_t n_seqs, int32_t total_q, int32_t h_kv, int32_t d,
                         int32_t page_size, cpe_dtype dtype, cpe_stream_t stream) {
  const char* fn = "cpe_kv_append";
  if (!k_new || !v_new || !k_cache || !v_cache || !page_table || !qo_indptr || !prefix_len)
    return fail(CPE_ERR_INVALID_ARG, fn, "null pointer argument");
  if (n_seqs <= 0 || total_q < 0 || h_kv <= 0 || d <= 0 || page_size <= 0 || max_pages <= 0 || num_pages <= 0)
    return fail(CPE_ERR_INVALID_ARG, fn, "sizes must be positive (total_q >= 0)");
  if (dtype != CPE_BF16 && dtype != CPE_F32) return fail(CPE_ERR_UNSUPPORTED, fn, "dtype must be CPE_BF16 or CPE_F32");
  const int esize = dtype == CPE_BF16 ? 2 : 4;
  const int64_t row_bytes = int64_t(h_kv) * d * esize;
  if (row_bytes % 16 != 0 || row_bytes > INT32_MAX) return fail(CPE_ERR_UNSUPPORTED, fn, "h_kv*d*elem must be a multiple of 16 bytes");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(CPE_ERR_INVALID_ARG, fn, "misaligned tensor (16 bytes)");
  if (total_q == 0) return CPE_OK;
  cudaError_t e;
  int* status = status_ptr(&e);
  if (!status) return cuda_fail(fn, e);
  KvAppendArgs a{};
  a.k_new = k_new; a.v_new = v_new; a.k_cache = k_cache; a.v_cache = v_cache; a.page_table = page_table;
  a.qo_indptr = qo_indptr; a.prefix_len = prefix_len; a.status = status; a.num_pages = num_pages;
  a.max_pages = max_pages; a.n_seqs = n_seqs; a.total_q = total_q; a.row_bytes = static_cast<int>(row_bytes);
  a.page_size = page_size;
  a.staged_from = n_seqs;  // every row
  e = launch_kv_append(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, e);
  g_launches += 1;
  return CPE_OK;
}

cpe_status cpe_extend_attention(const void* q, const void* k_cache, const void* v_cache, int64_t num_pages,
                                const int32_t* page_table, int32_t max_pages, const int32_t* qo_indptr,
                                const int32_t* prefix_len, int32_t n_seqs, int32_t total_q, int32_t max_kv_len,
                                int32_t h_q, int32_t h_kv, int32_t d, int32_t page_size, float sm_scale,
                                cpe_dtype dtype, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                cpe_stream_t stream) {
  const char* fn = "cpe_extend_attention";
  Common c{q, k_cache, v_cache, num_pages, page_table, max_pages, qo_indptr, prefix_len, n_seqs, total_q,
           max_kv_len, h_q, h_kv, d, page_size, sm_scale, dtype, out, lse, workspace, workspace_bytes};
  cpe_status st = validate(fn, c, true);
  if (st != CPE_OK) return st;
  if (total_q == 0) return CPE_OK;
  cudaError_t e;
  int* status = status_ptr(&e);
  if (!status) return cuda_fail(fn, e);
  return run_extend(fn, c, 0, 0, status, reinterpret_cast<cudaStream_t>(stream));
}

cpe_status cpe_decode_attention(const void* q, const void* k_cache, const void* v_cache, int64_t num_pages,
                                const int32_t* page_table, int32_t max_pages, const int32_t* prefix_len,
                                int32_t n_seqs, int32_t max_kv_len, int32_t h_q, int32_t h_kv, int32_t d,
                                int32_t page_size, float sm_scale, cpe_dtype dtype, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, cpe_stream_t stream) {
  const char* fn = "cpe_decode_attention";
  Common c{q, k_cache, v_cache, num_pages, page_table, max_pages, nullptr, prefix_len, n_seqs, n_seqs,
           max_kv_len, h_q, h_kv, d, page_size, sm_scale, dtype, out, lse, workspace, workspace_bytes};
  cpe_status st = validate(fn, c, false);
  if (st != CPE_OK) return st;
  if (dtype == CPE_F32) return fail(CPE_ERR_UNSUPPORTED, fn, "the split-KV decode path takes bf16; use cpe_extend_attention for fp32");
  cudaError_t e;
  int* status = status_ptr(&e);
  if (!status) return cuda_fail(fn, e);
  return run_decode(fn, c, n_seqs, false, status, reinterpret_cast<cudaStream_t>(stream));
}

cpe_status cpe_mixed_step(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          int64_t num_pages, const int32_t* page_table, int32_t max_pages, const int32_t* qo_indptr,
                          const int32_t* prefix_len, int32_t n_seqs, int32_t n_decode, int32_t total_q,
                          int32_t max_kv_len, int32_t h_q, int32_t h_kv, int32_t d, int32_t page_size,
                          float sm_scale, cpe_dtype dtype, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, cpe_stream_t stream) {
  const char* fn = "cpe_mixed_step";
  Common c{q, k_cache, v_cache, num_pages, page_table, max_pages, qo_indptr, prefix_len, n_seqs, total_q,
           max_kv_len, h_q, h_kv, d, page_size, sm_scale, dtype, out, lse, workspace, workspace_bytes};
  cpe_status st = validate(fn, c, true);
  if (st != CPE_OK) return st;
  if (n_decode < 0 || n_decode > n_seqs || n_decode > total_q)
    return fail(CPE_ERR_INVALID_ARG, fn, "n_decode must be in [0, min(n_seqs, total_q)]");
  if (!k_new || !v_new) return fail(CPE_ERR_INVALID_ARG, fn, "null k_new / v_new");
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return fail(CPE_ERR_INVALID_ARG, fn, "misaligned k_new / v_new");
  if (total_q == 0) return CPE_OK;
  cudaError_t e;
  int* status = status_ptr(&e);
  if (!status) return cuda_fail(fn, e);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // bf16 with prefill rows: the append rides in the extend schedule's launch
  if (dtype == CPE_BF16 && total_q > n_decode && n_decode < n_seqs) {
    KvAppendArgs ka{};
    ka.k_new = k_new; ka.v_new = v_new; ka.k_cache = k_cache; ka.v_cache = v_cache; ka.page_table = page_table;
    ka.qo_indptr = qo_indptr; ka.prefix_len = prefix_len; ka.status = status; ka.num_pages = num_pages;
    ka.max_pages = max_pages; ka.n_seqs = n_seqs; ka.total_q = total_q; ka.row_bytes = h_kv * d * 2;
    ka.page_size = page_size;
    // (nothing may read the cache before the prep launch: no decode rows, or
    // decode rows inside the same fused launch)
    cudaError_t ce;
    if (n_decode == 0) return run_extend(fn, c, 0, 0, status, s, 0, &ka);
    if (persistent_ctas(&ce) >= 16) return run_extend(fn, c, n_decode, n_decode, status, s, n_decode, &ka);
  }
  st = cpe_kv_append(k_new, v_new, k_cache, v_cache, num_pages, page_table, max_pages, qo_indptr, prefix_len, n_seqs,
                     total_q, h_kv, d, page_size, dtype, stream);
  if (st != CPE_OK) return st;
  // fp32 data: the CUDA-core path computes every row, decode rows included
  if (dtype == CPE_F32) return run_extend(fn, c, 0, 0, status, s);
  // decode rows only (or too few SMs to share): decode rows are sequences
  // [0, n_decode), one row each (rows [0, n_decode)), then the extend path
  st = run_decode(fn, c, n_decode, true, status, s);
  if (st != CPE_OK) return st;
  return run_extend(fn, c, n_decode, n_decode, status, s);
}

cpe_status cpe_get_device_status(cpe_stream_t stream, int32_t* detail) {
  const char* fn = "cpe_get_device_status";
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, e);
  int host[2] = {0, 0};
  e = cudaMemcpyFromSymbol(host, g_cpe_status, sizeof host);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  const int zero[2] = {0, 0};
  e = cudaMemcpyToSymbol(g_cpe_status, zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  if (detail) *detail = host[1];
  return static_cast<cpe_status>(host[0]);
}

}  // extern "C"
