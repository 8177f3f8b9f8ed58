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

constexpr int kMaxCtas = 160;        // upper bound of the persistent extend grid (SMs used)
constexpr int kMaxParts = 8;         // key-range parts a unit may be cut into
// Costs the extend schedule weighs against key-tile times, measured on GB300
// at d = 128 from rounds of 512 queries: an item's fixed cost (its query
// tiles' load, the pipeline's fill and drain, the output's store), and the
// merge of units cut into parts (the partial results' writes and the merge
// launch after the extend launch has drained).
constexpr float kItemCostTiles = 3.0f;
constexpr float kMergeCostTiles = 4.0f;
constexpr int kSizeBuckets = 4;      // item-size classes of the largest-first order
constexpr int kPairBits = 20;        // ItemDesc::head_pair = kv_head << kPairBits | pair
constexpr int kMaxSlots = 2048;      // partial-result slots in the workspace
constexpr int kCutSlots = 1024;      // of which the uniform cut may use (the rest fill the last wave)
constexpr int kUnitRows = 2 * kBlockM;
constexpr int kMergeRowGroups = 8;  // merge work items per cut unit (32 rows each)
constexpr int kMergeThreads = 256;  // merge block: 8 warps, four rows each

struct UnitEntry {  // one extend work unit: two query tiles of one sequence and KV head
  int seq;
  int pair;      // query tiles 2*pair and 2*pair+1 of the sequence
  int kv_head;
  int n_kv;      // key tiles the unit needs
  int parts;     // key-range parts the unit is cut into (1: it writes its output directly)
  int slot;      // partial slot of its part 0 (parts > 1); part p uses slot + p
};

// One entry of the item table: key tiles [kv_lo, kv_hi) of one unit with all a
// CTA needs to start on it (no further lookups): the sequence, its first row,
// query length and prefix, the KV head and pair, and the part's partial slot
// (-1: the unit is not cut; its output goes straight to out / lse).
// kv_lo >= kv_hi: no item.  Two 16-byte loads.
struct alignas(16) ItemDesc {
  int seq;
  int head_pair;
  int q0, E, P;
  int kv_lo, kv_hi;
  int slot;
};

// Device-side schedule kept in the caller's workspace.  Unit u is cut into
// units[u].parts parts; part p covers key tiles [p*len, min((p+1)*len, n_kv))
// with len = ceil(n_kv / parts).  The item table lists the non-empty parts
// (ItemDesc; empty entries have kv_lo >= kv_hi); CTA c takes table entries
// c, c + header[1], ...
struct ExtendSched {
  int* header;          // [0] total key tiles, [1] CTAs used, [2] units, [3] item table length
                        // (a multiple of [1]), [4] target part length, [5] items, [6] next
                        // decode item of a fused mixed step, [7] units cut into parts
  UnitEntry* units;     // [capacity]
  ItemDesc* items;      // [item capacity]
  uint8_t* partial;     // slots of partial_slot_bytes(d): O [256 x d] bf16 (normalised), then m [256]
                        // (log2) and l [256] fp32
  UnitEntry* split;     // the units cut into parts, in unit order (header[7] of them)
};

__host__ __device__ constexpr size_t partial_slot_bytes(int d) {
  return size_t(kUnitRows) * d * 2 + 2 * size_t(kUnitRows) * 4;
}

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

// Rates that size the split of a fused mixed step between extend CTAs and
// decode workers, measured on GB300 at d = 128: one key tile of a two-tile
// unit takes one SM about 1.85 us alone and about 8 % longer beside decode
// rows (they share HBM); decode rows stream K/V at about 55 GB/s per SM, which
// reaches the 6.67 GB/ms the part sustains at about 120 SMs.  (Swept forced
// splits put the best step at 44 extend CTAs for 256 decode rows beside a
// 2048-token chunk at prefix 30720, and at 128 for the scheduled step with 64
// decode rows and four chunks: the rule picks both.)
constexpr float kTileUsPerSm = 1.85f;
constexpr float kFusedExtendSlowdown = 1.08f;
constexpr float kDecodeBytesPerUs = 6.67e6f;
constexpr int kDecodeSatSms = 120;

struct ScheduleArgs {
  const int32_t* qo_indptr;
  const int32_t* prefix_len;
  int seq_begin, seq_end;   // sequences [seq_begin, seq_end) take part
  int tok;                  // tokens per query tile (kBlockM / G)
  int h_kv;
  int max_kv_len;
  int max_pages;
  int capacity;             // unit entries available
  int n_ctas;               // persistent grid size
  int max_slots;            // partial slots available
  ExtendSched sched;
  int* status;
  // fused mixed step: decode rows [0, dec_rows) run on the CTAs the extend
  // part leaves free (0: no decode rows in this launch)
  int dec_rows;
  int64_t dec_bytes_per_key;  // K + V bytes one key of one decode row reads
  int d;
  // 1: the previous call on this stream used the same workspace, so the
  // schedule is written only once the previous launch has completed; 0: it
  // is written as soon as it is computed
  int sched_wait;
};

struct ExtendTcArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  CUtensorMap tm_k128, tm_v128;  // the same caches with 128-token boxes (8 consecutive pages)
  // the round's new K/V rows [total_q, h_kv, d] (16- and 128-row boxes), when
  // the call has them (staged = 1): for a sequence whose prefix ends on a page
  // boundary the extend launch reads its new keys from these rows and writes
  // the full new pages into the cache from the tiles it staged
  CUtensorMap tm_kn, tm_vn, tm_kn128, tm_vn128;
  int staged;
  const int32_t* page_table;
  const int32_t* qo_indptr;
  const int32_t* prefix_len;
  ExtendSched sched;
  void* out;
  float* lse;
  int* status;
  int64_t num_pages;
  int max_pages;
  int h_q, h_kv, group, tok, d;
  float scale_log2;
  uint64_t wait_ns;
  int n_ctas;
  int max_split;  // units that may be cut into parts (the merge kernel's grid / kMergeRowGroups)
  // fused mixed step: CTAs past the extend part run these decode items
  // ((sequence x KV head) x split, split fastest), taken from header[6]
  DecodeArgs dec;
  int dec_items;
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
  // sequences >= staged_from whose prefix ends on a page boundary have their
  // full new pages written by the extend launch: their rows there are skipped
  // (n_seqs: append every row)
  int staged_from;
};


// The extend schedule; `dependent` as for launch_extend_tc (the schedule is
// computed while the previous launch finishes and written after it).
cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t s, bool dependent);
// One launch: the extend schedule (block 0) and the round's K/V append (the other blocks).
cudaError_t launch_prep(const ScheduleArgs& a, const KvAppendArgs& k, cudaStream_t s, bool dependent);
// The extend launch + the merge of split units.  `dependent`: launch both with
// programmatic stream serialisation (each may be scheduled while the kernel
// before it finishes), which hides launch latency on short launches; on long
// ones (measured on the 128k-token request's 1.7 ms rounds) it costs about 1 %, so the caller
// turns it on only below kDependentLaunchFlops of extend work.
cudaError_t launch_extend_tc(const ExtendTcArgs& a, cudaStream_t s, bool dependent);
constexpr double kDependentLaunchFlops = 2e11;
cudaError_t launch_extend_simt(const ExtendSimtArgs& a, cudaStream_t s);
cudaError_t launch_kv_append(const KvAppendArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t s);  // combine the splits of decode rows
size_t extend_tc_smem_bytes(int d);

}  // namespace cpe
