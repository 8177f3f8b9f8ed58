// cpe_decode_attention_noalloc: the split-KV decode path with its scratch in
// a fixed device array owned by this library instead of a caller-supplied
// workspace, for callers that cannot allocate device memory.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes.  Every
// GPU that loads the library holds it until the process exits.  Host code may
// not use the array's name as a device address (on the host it is only a
// stand-in symbol), so the first call on each device, with that device
// current, looks up its device address with cudaGetSymbolAddress and keeps it
// for later calls on that device.
#include <cstdint>
#include <mutex>
#include <string>

#include "cpe.h"
#include "cpe_device.cuh"
#include "kernels.h"

namespace cpe {
void set_last_error(const std::string& msg);
int* device_status_word(cudaError_t* err);
void count_launches(int n);
}  // namespace cpe

namespace {

constexpr size_t kNoAllocScratchBytes = CPE_DECODE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDev] = {};

// Device address of the scratch array on the current device (set up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

cpe_status reject(cpe_status st, const char* msg) {
  cpe::set_last_error(std::string("cpe_decode_attention_noalloc: ") + msg);
  return st;
}

bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" cpe_status cpe_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                   int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                                                   const int32_t* prefix_len, int32_t n_seqs, int32_t max_kv_len,
                                                   int32_t h_q, int32_t h_kv, int32_t d, int32_t page_size,
                                                   float sm_scale, cpe_dtype dtype, void* out, float* lse,
                                                   cpe_stream_t stream) {
  using namespace cpe;
  if (!q || !k_cache || !v_cache || !page_table || !prefix_len || !out) return reject(CPE_ERR_INVALID_ARG, "null pointer argument");
  if (n_seqs <= 0 || max_kv_len <= 0 || max_pages <= 0 || num_pages <= 0 || h_q <= 0 || h_kv <= 0)
    return reject(CPE_ERR_INVALID_ARG, "sizes must be positive");
  if (!(sm_scale > 0.f) || sm_scale != sm_scale || sm_scale > 3.0e38f) return reject(CPE_ERR_INVALID_ARG, "sm_scale must be finite and > 0");
  if (h_q % h_kv != 0) return reject(CPE_ERR_INVALID_ARG, "h_q must be a multiple of h_kv");
  const int G = h_q / h_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return reject(CPE_ERR_UNSUPPORTED, "G = h_q/h_kv must be 1, 2, 4, 8 or 16");
  if (d != 64 && d != 128) return reject(CPE_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (page_size != kPage) return reject(CPE_ERR_UNSUPPORTED, "page_size must be 16");
  if (dtype != CPE_BF16) return reject(CPE_ERR_UNSUPPORTED, "the split-KV decode path takes bf16");
  if (num_pages > int64_t(INT32_MAX) / kPage) return reject(CPE_ERR_INVALID_ARG, "num_pages too large");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) || !aligned(page_table, 4) ||
      !aligned(prefix_len, 4) || (lse && !aligned(lse, 4)))
    return reject(CPE_ERR_INVALID_ARG, "misaligned pointer (16 bytes for tensors, 4 for index arrays)");
  const int max_splits = (max_kv_len + kDecodeSplit - 1) / kDecodeSplit;
  const size_t parts = size_t(n_seqs) * h_q * max_splits;
  const size_t o_bytes = align256(parts * d * sizeof(float));
  const size_t need = o_bytes + align256(parts * 2 * sizeof(float));
  if (need > kNoAllocScratchBytes)
    return reject(CPE_ERR_CAPACITY,
                  ("needs " + std::to_string(need) + " bytes of scratch (n_seqs * h_q * ceil(max_kv_len / 2048) * (d + 2) * 4), "
                   "above the fixed " + std::to_string(kNoAllocScratchBytes) + "-byte array; split the batch or use "
                   "cpe_decode_attention with a workspace").c_str());
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return reject(CPE_ERR_CUDA, cudaGetErrorString(e));
  int* status = device_status_word(&e);
  if (!status) return reject(CPE_ERR_CUDA, cudaGetErrorString(e));
  DecodeArgs a{};
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.page_table = page_table; a.qo_indptr = nullptr;
  a.prefix_len = prefix_len; a.out = out; a.lse = lse;
  a.part_o = static_cast<float*>(scratch);
  a.part_ml = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + o_bytes);
  a.status = status; a.num_pages = num_pages; a.max_pages = max_pages; a.n_seqs = n_seqs; a.seq_begin = 0;
  a.h_q = h_q; a.h_kv = h_kv; a.d = d; a.max_kv_len = max_kv_len; a.max_splits = max_splits;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  e = launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return reject(CPE_ERR_CUDA, cudaGetErrorString(e));
  count_launches(max_splits > 1 ? 2 : 1);
  return CPE_OK;
}
