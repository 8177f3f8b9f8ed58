// Extend attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Work unit: two query tiles of 128 rows of one sequence that share a KV head.
// A tile's rows are (128 / G tokens) x (the G query heads of the group), so
// each K/V tile staged in shared memory serves all G heads of both query
// tiles: 256 rows per K/V byte brought on chip.
//
// Key tiles of 128 are walked in order.  Tiles wholly inside the cached prefix
// are the unmasked rectangle (Stage 1 of the SGLang chunked-prefill article);
// tiles that reach the chunk's own keys form the causal triangle (Stage 2),
// where only the tiles crossing the diagonal apply the mask j <= P + i and
// tiles above it are never loaded.  Both stages feed one running (m, l, O)
// per row: the article's online-softmax LSE merge, applied tile by tile.
//
// Persistent, balanced grid: one CTA per SM.  The schedule kernel lists the
// units and cuts each into key-range parts of about one target length, the
// one with the least estimated time (waves of items, each costing its key
// tiles plus a fixed cost, plus the merge); units of equal length get equal
// parts, and a last wave left partly idle is filled by giving some units one
// more, smaller part.  It orders the parts largest first in a few size
// classes, part-major within a class, and deals them to the CTAs in snake
// order.  CTAs running at the same time then stream the same key range of a
// KV head (the K/V tiles are read from HBM once and served to the others from
// L2), and units of unequal length still even out across CTAs.  A unit cut
// into several parts has each part's normalised partial (O, m, l) written to
// a workspace slot, and the merge kernel combines them with the same
// online-softmax LSE rule.
//
// Warp roles (384 threads, three warpgroups):
//   warp 0      TMA producer: both Q tiles of each unit, then the K ring
//   warp 2      TMA producer: the V ring
//               (page boxes of 16 tokens x 64 dims, 128-byte swizzle; eight
//               pages stack into one 128-key tile; when the eight pages are
//               consecutive in the cache one 128-token box per 64-dim half
//               replaces the sixteen page boxes)
//   warp 1      TMEM owner and MMA issuer: S_t = Q_t K_j^T into TMEM, and
//               O_t += P_t V_j with P read from TMEM, for t = 0, 1 in turn, so
//               the tensor pipe works on one tile while the other's softmax runs
//   warps 4-7   softmax of query tile 0, warps 8-11 of query tile 1: one thread
//               per row reads its S row from TMEM, masks, takes the
//               exponentials against the running max (the tile's own max only
//               when a weight would pass 2^16; the running max then rises only
//               if the tile's exceeds it by more than 2^8, rescaling O), writes
//               P as bf16 over its S columns, and at the end normalises and
//               stores O.
// The first warpgroup gives registers up (setmaxnreg) to the two softmax
// warpgroups; the host checks the launch allocation covers the split.
// TMEM columns: [0,128) S0, [128,256) S1, [256,256+D) O0, [256+D,256+2D) O1.
// Ring stages, S/P phases and the Q buffer advance with running counters that
// every role keeps identically across the CTA's work items.
//
// tcgen05.mma instructions from one thread execute in issue order, so S_t for
// the next key tile may be issued right behind the PV that reads P_t from the
// same columns; tcgen05.commit tracks every earlier MMA of the thread, so the
// S barrier also tells the softmax that the previous PV (and thus O_t) is done.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records
// CPE_ERR_TIMEOUT, every role leaves its loop, in-flight copies and MMAs are
// drained, TMEM is freed and the kernel returns.
#include <algorithm>
#include <atomic>

#include "cpe_device.cuh"
#include "decode_item.cuh"
#include "kv_append_row.cuh"
#include "kernels.h"

namespace cpe {

namespace {

constexpr int kThreads = 384;
constexpr int kRefillPolls = 64;     // staged form: slot polls before a producer's suspending wait
constexpr int kLaunchRegs = 168;     // 384 x 168 = 64512 registers at launch
constexpr int kProducerRegs = 96;    // warpgroup 0 after setmaxnreg.dec
constexpr int kSoftmaxRegs = 200;    // warpgroups 1, 2 after setmaxnreg.inc
static_assert(128 * kProducerRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split");
constexpr uint64_t kDrainNs = 2000000000ull;  // fixed bound for the final drain waits

template <int D>
struct TcCfg {
  static constexpr int kHalves = D / 64;              // 128-byte column blocks per row
  static constexpr int kTileBytes = kBlockM * D * 2;  // 128 rows (or keys) x D bf16
  static constexpr int kStagesK = (D == 128) ? 3 : 6;
  static constexpr int kStagesV = (D == 128) ? 2 : 5;
  static constexpr int kHalfBytes = 128 * 128;        // 128 rows x 128 bytes
  static constexpr int kQOff = 0;                     // two Q tiles
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStagesK * kTileBytes;
  static constexpr int kBarOff = kVOff + kStagesV * kTileBytes;
  static constexpr int kSmem = kBarOff + 512 + 1024;  // + barriers + alignment slack
};

template <int NK, int NV>
struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[NK], k_empty[NK];
  uint64_t v_full[NV], v_empty[NV];
  // cache-page stores owed from each slot's current tile (kept by the slot's
  // producer): pages mask, sequence, key tile, KV head
  int k_owed[NK][4], v_owed[NV][4];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: the abort flag of the final drain waits, which must not give up early
};

__device__ __forceinline__ void setmaxnreg_dec_producer() { asm volatile("setmaxnreg.dec.sync.aligned.u32 96;"); }
__device__ __forceinline__ void setmaxnreg_inc_softmax() { asm volatile("setmaxnreg.inc.sync.aligned.u32 200;"); }

// Work item: key tiles [kv_lo, kv_hi) of one unit.
// The two query tiles' fields are kept as separate scalars and picked with a
// select: indexing a two-element array with a runtime tile number would put the
// array in local memory, whose loads share the L1/shared-memory path that the
// tensor core's operand reads keep busy.
struct Item {
  int seq, g, q0, E, P, kv_lo, kv_hi;
  int i0_0, i0_1, kv_end_0, kv_end_1, n_kt_0, n_kt_1;
  bool whole;  // the unit is not cut: its output goes straight to out / lse
  int slot;    // partial slot of this part otherwise
  __device__ __forceinline__ int i0(int t) const { return t ? i0_1 : i0_0; }
  __device__ __forceinline__ int kv_end(int t) const { return t ? kv_end_1 : kv_end_0; }
  __device__ __forceinline__ int n_kt(int t) const { return t ? n_kt_1 : n_kt_0; }
};

// Fills `it` for item-table entry i (one descriptor: two independent 16-byte
// loads); false for an empty entry.
__device__ __forceinline__ bool load_item(const ExtendTcArgs& a, int i, Item& it) {
  const int4* d = reinterpret_cast<const int4*>(a.sched.items + i);
  const int4 x = d[0];
  const int4 y = d[1];
  it.kv_lo = y.y;
  it.kv_hi = y.z;
  if (it.kv_lo >= it.kv_hi) return false;
  it.seq = x.x;
  it.g = x.y >> kPairBits;
  const int pair = x.y & ((1 << kPairBits) - 1);
  it.q0 = x.z;
  it.E = x.w;
  it.P = y.x;
  it.slot = y.w;
  it.whole = it.slot < 0;
  it.i0_0 = 2 * pair * a.tok;
  it.i0_1 = it.i0_0 + a.tok;
  it.kv_end_0 = it.i0_0 < it.E ? it.P + min(it.E, it.i0_0 + a.tok) : 0;
  it.kv_end_1 = it.i0_1 < it.E ? it.P + min(it.E, it.i0_1 + a.tok) : 0;
  it.n_kt_0 = (it.kv_end_0 + kBlockN - 1) / kBlockN;
  it.n_kt_1 = (it.kv_end_1 + kBlockN - 1) / kBlockN;
  return true;
}

// Pages of key tile j (keys kb + 16 pg) that an item of a page-aligned
// sequence writes to the cache from its staged tile: new pages (keys >= P,
// pg >= pnew) that are full pages of the unit's own tokens
// [P + i0_0, P + min(E, i0_0 + 2 tok)).  Each full new page of a sequence and
// KV head belongs to exactly one unit, and its key tile to one part.
__device__ __forceinline__ uint32_t own_pages(const Item& it, int tok, int kb, int pnew, int npg) {
  const int own_lo = it.P + it.i0_0;
  const int own_hi = it.P + min(it.E, it.i0_0 + 2 * tok);
  uint32_t m = 0;
#pragma unroll
  for (int pg = 0; pg < kBlockN / kPage; ++pg) {
    const int pos = kb + pg * kPage;
    if (pg >= pnew && pg < npg && pos >= own_lo && pos + kPage <= own_hi) m |= 1u << pg;
  }
  return m;
}

// Decode rows of a fused mixed step on a CTA the extend part does not use:
// each of the CTA's three warpgroups takes decode items from the shared
// counter and computes them as the stand-alone decode kernel's CTAs do, in its
// own third of shared memory, on its own named barrier.
template <int D>
__device__ void decode_worker(const ExtendTcArgs& a, uint8_t* smem) {
  static_assert(1024 + 3 * DecCfg<D>::kSmem + 64 <= TcCfg<D>::kSmem, "three decode items fit a CTA's shared memory");
  const int wg = threadIdx.x / 128;
  const int tid = threadIdx.x % 128;
  uint8_t* dsm = smem + wg * DecCfg<D>::kSmem;
  volatile int* slot = reinterpret_cast<volatile int*>(smem + 3 * DecCfg<D>::kSmem) + wg;
  const int splits = a.dec.max_splits;
  for (;;) {
    if (tid == 0) *slot = atomicAdd(&a.sched.header[6], 1);
    group_sync(1 + wg);
    const int item = *slot;
    group_sync(1 + wg);  // every thread has its item before the slot is reused
    if (item >= a.dec_items) break;
    const int sp = item % splits;
    const int rest = item / splits;
    decode_item<D>(a.dec, sp, rest / a.h_kv, rest % a.h_kv, dsm, tid, 1 + wg);
  }
}

// S (staged): the launch reads the chunk's keys from the round's new rows and
// writes the full new pages of page-aligned sequences to the cache (long
// launches with new rows at hand).  F (fused): decode rows share the launch
// (a fused mixed step).  Separate instantiations keep the code of every other
// launch free of that work: three forms per head size, plain, staged and
// fused.
template <int D, bool S, bool F>
__global__ void __launch_bounds__(kThreads, 1) extend_tc_kernel(const __grid_constant__ ExtendTcArgs a) {
  using C = TcCfg<D>;
  constexpr int NK = C::kStagesK;
  constexpr int NV = C::kStagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars<NK, NV>* bars = reinterpret_cast<Bars<NK, NV>*>(smem + C::kBarOff);
  static_assert(sizeof(Bars<NK, NV>) <= 512, "barrier area");

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile int* abort = &bars->abort;

  // The tensor-memory allocation touches no global memory: it runs while
  // the launch before this one (the schedule) finishes.
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  grid_dependency_wait();    // the schedule (and the round's K/V append) are complete
  grid_launch_dependents();  // the merge kernel may be scheduled as CTAs finish
  const int nc = a.sched.header[1];
  const int n_items = a.sched.header[3];  // item-table entries; CTA c takes c, c + nc, ...
  const int cta = blockIdx.x;
  if (cta >= nc) {  // CTAs past the extend part: decode workers of a fused mixed step, else idle
    if (warp == 1) tmem_dealloc(tmem, 512);
    if (a.dec_items > 0) decode_worker<D>(a, smem);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < NK; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < NK; ++i) bars->k_owed[i][0] = 0;
    for (int i = 0; i < NV; ++i) bars->v_owed[i][0] = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->o_done[i], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->never = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();

  if (warp < 4) {
    setmaxnreg_dec_producer();
    if ((warp == 0 || warp == 2) && lane == 0) {
      // ---------------------------------------------------------- producers
      const bool is_k = warp == 0;
      const CUtensorMap* tm = is_k ? &a.tm_k : &a.tm_v;
      const CUtensorMap* tm128 = is_k ? &a.tm_k128 : &a.tm_v128;
      const CUtensorMap* tmn = is_k ? &a.tm_kn : &a.tm_vn;        // the round's new rows
      const CUtensorMap* tmn128 = is_k ? &a.tm_kn128 : &a.tm_vn128;
      const int ns = is_k ? NK : NV;
      uint64_t* full = is_k ? bars->k_full : bars->v_full;
      uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
      uint8_t* ring = smem + (is_k ? C::kKOff : C::kVOff);
      prefetch_tmap(tm);
      prefetch_tmap(tm128);
      if constexpr (S) {
        prefetch_tmap(tmn);
        prefetch_tmap(tmn128);
      }
      if (is_k) prefetch_tmap(&a.tm_q);
      const int oob = static_cast<int>(a.num_pages * kPage);  // a row past the cache: zero fill
      int cnt = 0;       // ring loads issued so far
      int items = 0;     // Q loads issued so far
      int (*owed)[4] = is_k ? bars->k_owed : bars->v_owed;
      // The full new pages of a page-aligned sequence's own tokens are written
      // to the cache from the slot they were staged in, when the slot is
      // refilled (its tile has landed and been consumed by then) or, for the
      // last tiles, once they land at the end.
      auto store_owed = [&](int st) {
        const int* o = owed[st];
        const int32_t* opt = a.page_table + static_cast<int64_t>(o[1]) * a.max_pages;
#pragma unroll
        for (int pg = 0; pg < kBlockN / kPage; ++pg) {
          if (!((o[0] >> pg) & 1)) continue;
          const int pid = opt[o[2] * (kBlockN / kPage) + pg];
          if (pid < 0 || pid >= a.num_pages) continue;  // recorded when the tile was loaded
          for (int h = 0; h < C::kHalves; ++h)
            tma_store_3d(tm, ring + st * C::kTileBytes + h * C::kHalfBytes + pg * (kPage * 128), h * 64, o[3],
                         pid * kPage);
        }
        bulk_commit_group();
        owed[st][0] = 0;
      };
      bool ok = true;
      Item it;
      for (int wi = cta; ok && wi < n_items; wi += nc) {
        if (!load_item(a, wi, it)) continue;
        if (is_k) {
          if (items > 0 &&
              !mbar_wait(&bars->q_empty, (items - 1) & 1, abort, a.wait_ns, a.status, kDetailQFull)) break;
          const int n_q = it.n_kt_1 > 0 ? 2 : 1;
          mbar_arrive_expect_tx(&bars->q_full, n_q * C::kTileBytes);
          for (int t = 0; t < n_q; ++t)
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_3d(smem + C::kQOff + t * C::kTileBytes + h * C::kHalfBytes, &a.tm_q, &bars->q_full, h * 64,
                          it.g * a.group, it.q0 + it.i0(t));
          ++items;
        }
        const int kv_max = max(it.kv_end_0, it.kv_end_1);
        const int32_t* pt = a.page_table + static_cast<int64_t>(it.seq) * a.max_pages;
        // A prefix that ends on a page boundary: the chunk's keys are read from
        // the round's new rows, and the full pages of this unit's own tokens
        // (keys P + [2 pair tok, 2 pair tok + 2 tok)) are written to the cache
        // from the staged tile.  Otherwise everything comes from the cache.
        const bool staged = S && it.P % kPage == 0;
        for (int j = it.kv_lo; j < it.kv_hi; ++j, ++cnt) {
          const int st = cnt % ns;
          const int use = cnt / ns;
          const int kb = j * kBlockN;
          const int keys = min(kBlockN, kv_max - kb);
          const int npg = (keys + kPage - 1) / kPage;
          const int pnew = staged ? min(npg, max(0, (it.P - kb) / kPage)) : npg;  // pages [pnew, npg) are new
          int rows[kBlockN / kPage];  // unrolled loops below keep it in registers
          bool contiguous = npg == kBlockN / kPage && pnew == npg;  // eight cached pages back to back
#pragma unroll
          for (int pg = 0; pg < kBlockN / kPage; ++pg) {
            if (pg >= npg) break;
            const int pid = pt[j * (kBlockN / kPage) + pg];
            if (pid < 0 || pid >= a.num_pages) {
              record_error(a.status, kStatusDeviceArg, kDetailBadPage);
              rows[pg] = oob;
              contiguous = false;
            } else {
              rows[pg] = pid * kPage;
              contiguous = contiguous && rows[pg] == rows[0] + pg * kPage;
            }
          }
          // (the staged form polls the slot first: measured faster on its long
          // launches; on fused mixed steps the polls slowed the softmax warps)
          if (use > 0 && !mbar_wait_polled(&empty[st], (use - 1) & 1, S ? kRefillPolls : 0, abort, a.wait_ns,
                                           a.status, is_k ? kDetailKEmpty : kDetailVEmpty)) {
            ok = false;
            break;
          }
          if (S && owed[st][0]) {  // the slot's previous tile owes cache pages: store them, let them read the slot
            store_owed(st);
            bulk_wait_read_all();
          }
          if (S && staged) {
            const uint32_t own = own_pages(it, a.tok, kb, pnew, npg);
            if (own) {
              owed[st][0] = static_cast<int>(own);
              owed[st][1] = it.seq;
              owed[st][2] = j;
              owed[st][3] = it.g;
            }
          }
          uint8_t* dst = ring + st * C::kTileBytes;
          mbar_arrive_expect_tx(&full[st], npg * C::kHalves * (kPage * 128));
          if (contiguous) {
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_3d(dst + h * C::kHalfBytes, tm128, &full[st], h * 64, it.g, rows[0]);
            // Beside decode rows (a fused mixed step) the HBM is saturated and
            // a copy's latency grows: the tile two ahead is prefetched into L2,
            // on the guess that the pages stay consecutive (a wrong guess only
            // wastes the prefetch).  Elsewhere the CTAs that stream a KV
            // head's keys together already serve each other from L2, and the
            // prefetches measured slower.
            if (F && j + 2 < it.kv_hi && rows[0] + 3 * kBlockN <= oob)
              for (int h = 0; h < C::kHalves; ++h) tma_prefetch_3d(tm128, h * 64, it.g, rows[0] + 2 * kBlockN);
          } else if (!S) {
#pragma unroll
            for (int pg = 0; pg < kBlockN / kPage; ++pg) {
              if (pg >= npg) break;
              for (int h = 0; h < C::kHalves; ++h)
                tma_load_3d(dst + h * C::kHalfBytes + pg * (kPage * 128), tm, &full[st], h * 64, it.g, rows[pg]);
            }
          } else if (pnew == 0 && npg == kBlockN / kPage) {  // eight new pages: rows q0 + kb - P onwards
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_3d(dst + h * C::kHalfBytes, tmn128, &full[st], h * 64, it.g, it.q0 + kb - it.P);
          } else {  // cached pages below P, new rows from P on
#pragma unroll
            for (int pg = 0; pg < kBlockN / kPage; ++pg) {
              if (pg >= npg) break;
              const bool nw = pg >= pnew;
              for (int h = 0; h < C::kHalves; ++h)
                tma_load_3d(dst + h * C::kHalfBytes + pg * (kPage * 128), nw ? tmn : tm, &full[st], h * 64, it.g,
                            nw ? it.q0 + kb + pg * kPage - it.P : rows[pg]);
            }
          }
        }
      }
      // Drain: every copy issued must land before the CTA exits.
      if (*abort) {
        volatile int* no_abort = &bars->never;
        if (is_k && items > 0) mbar_wait(&bars->q_full, (items - 1) & 1, no_abort, kDrainNs, a.status, kDetailDrain);
        for (int n = max(0, cnt - ns); n < cnt; ++n)
          mbar_wait(&full[n % ns], (n / ns) & 1, no_abort, kDrainNs, a.status, kDetailDrain);
      } else if (S) {
        // the last tiles' owed pages, once each has landed
        for (int n = max(0, cnt - ns); n < cnt; ++n) {
          if (!owed[n % ns][0]) continue;
          if (!mbar_wait(&full[n % ns], (n / ns) & 1, abort, a.wait_ns, a.status, is_k ? kDetailKFull : kDetailVFull))
            break;
          store_owed(n % ns);
        }
      }
      if constexpr (S) bulk_wait_read_all();  // no store still reads the ring when the CTA leaves
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kBlockN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);
      auto issue_s = [&](int t, int st) {
        const uint64_t qd = smem_desc_sw128(smem_u32(smem + C::kQOff + t * C::kTileBytes), 16, 1024);
        const uint64_t kd = smem_desc_sw128(smem_u32(smem + C::kKOff + st * C::kTileBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk / 4) * C::kHalfBytes + (kk % 4) * 32) >> 4);
          tc_mma_ss(tmem + t * 128, qd + off, kd + off, idesc_qk, kk > 0);
        }
        tc_commit(&bars->s_full[t]);
      };
      int kc = 0, vc = 0, items = 0;
      int pc0 = 0, pc1 = 0;  // P hand-offs consumed per tile
      bool ok = true;
      Item it;
      for (int wi = cta; ok && wi < n_items; wi += nc) {
        if (!load_item(a, wi, it)) continue;
        if (!mbar_wait(&bars->q_full, items & 1, abort, a.wait_ns, a.status, kDetailQFull) ||
            !mbar_wait(&bars->k_full[kc % NK], (kc / NK) & 1, abort, a.wait_ns, a.status, kDetailKFull)) {
          ok = false;
          break;
        }
        ++items;
        tc_fence_after();
        if (it.kv_lo < it.n_kt_0) issue_s(0, kc % NK);
        if (it.kv_lo < it.n_kt_1) issue_s(1, kc % NK);
        tc_commit(&bars->k_empty[kc % NK]);
        ++kc;
        // Q is released once the item's last S is issued (here for a one-tile
        // item, else in the loop at its second-last key tile), so the next
        // item's Q load overlaps the last tile's softmax and P.V.  The staged
        // form releases it after the item: there the producer's refill of the
        // last tiles' slots stores their owed pages, and those stores, moved
        // under the last P.V bursts, measured slower (long rounds -0.7 %).
        if (!S && it.kv_lo + 1 == it.kv_hi) tc_commit(&bars->q_empty);
        for (int j = it.kv_lo; j < it.kv_hi; ++j) {
          // Both operand stages this key tile needs are waited for up front, so
          // the MMA bursts below are separated only by the softmax hand-offs.
          const int sv_st = vc % NV;
          const bool more = j + 1 < it.kv_hi;
          // V_j, K_{j+1} and tile 0's P are usually ready: test all three at
          // once and wait only for what is not.
          const bool need_p0 = j < it.n_kt_0;
          const uint32_t ready =
              mbar_test3(&bars->v_full[sv_st], (vc / NV) & 1, &bars->k_full[kc % NK], (kc / NK) & 1,
                         &bars->p_full[0], pc0 & 1);
          if ((!(ready & 1u) &&
               !mbar_wait(&bars->v_full[sv_st], (vc / NV) & 1, abort, a.wait_ns, a.status, kDetailVFull)) ||
              (more && !(ready & 2u) &&
               !mbar_wait(&bars->k_full[kc % NK], (kc / NK) & 1, abort, a.wait_ns, a.status, kDetailKFull))) {
            ok = false;
            break;
          }
          const bool p0_ready = need_p0 && (ready & 4u);
          const uint64_t vdesc =
              smem_desc_sw128(smem_u32(smem + C::kVOff + sv_st * C::kTileBytes), C::kHalfBytes, 1024);
          // PV of tile t, then the next S of tile t; called with literal tile
          // numbers so every per-tile value resolves at compile time.
          auto tile_step = [&](const int t) -> bool {
            if (j >= it.n_kt(t)) return true;
            int& pct = t ? pc1 : pc0;
            if (!(t == 0 && p0_ready) &&
                !mbar_wait(&bars->p_full[t], pct & 1, abort, a.wait_ns, a.status, kDetailPFull))
              return false;
            ++pct;
            tc_fence_after();
            const uint32_t dcol = tmem + 256 + t * D;
            const uint32_t acol = tmem + t * 128;
            const int keys = min(kBlockN, it.kv_end(t) - j * kBlockN);
            const uint32_t first = j > it.kv_lo ? 1u : 0u;
            if (keys == kBlockN) {
#pragma unroll
              for (int kk = 0; kk < kBlockN / 16; ++kk)
                tc_mma_ts(dcol, acol + kk * 8, vdesc + static_cast<uint64_t>(kk * (16 * 128 / 16)), idesc_pv,
                          (first || kk > 0) ? 1u : 0u);
            } else {
              const int nsteps = (keys + 15) / 16;  // only pages that were loaded
              for (int kk = 0; kk < nsteps; ++kk)
                tc_mma_ts(dcol, acol + kk * 8, vdesc + static_cast<uint64_t>(kk * (16 * 128 / 16)), idesc_pv,
                          (first || kk > 0) ? 1u : 0u);
            }
            if (j + 1 < min(it.kv_hi, it.n_kt(t)))
              issue_s(t, kc % NK);
            else
              tc_commit(&bars->o_done[t]);
            return true;
          };
          if (!tile_step(0) || !tile_step(1)) {
            ok = false;
            break;
          }
          tc_commit(&bars->v_empty[sv_st]);
          ++vc;
          if (more) {
            tc_commit(&bars->k_empty[kc % NK]);
            ++kc;
          }
          // every S of the item issued (the last at key tile kv_hi - 2, for
          // the query tile with the most key tiles): Q may be replaced
          if (!S && j + 2 == it.kv_hi) tc_commit(&bars->q_empty);
        }
        if (S) tc_commit(&bars->q_empty);
      }
      // Drain: wait until every MMA issued above has completed.
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, &bars->never, kDrainNs, a.status, kDetailDrain);
    }
  } else {
    setmaxnreg_inc_softmax();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) / 4;          // query tile of this warpgroup
    const int quad = warp & 3;             // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;        // query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_col = t * 128;
    const uint32_t o_col = 256 + t * D;
    const float sl2 = a.scale_log2;
    int sc = 0, od = 0;
    bool ok = true;
    Item it;
    for (int wi = cta; ok && wi < n_items; wi += nc) {
      if (!load_item(a, wi, it)) continue;
      const int i0t = it.i0(t);
      const int i = i0t + r / a.group;              // token index within the chunk
      const int lim = it.P + min(i, it.E - 1);    // last key this row may see
      const int jhi = min(it.kv_hi, it.n_kt(t));
      const int R = t * kBlockM + r;               // row of the unit
      if (it.kv_lo >= jhi) {
        // no key tile of this portion reaches this query tile: an empty partial
        if (!it.whole) {  // l = 0 tells the merge to skip this part's O
          float* ml = reinterpret_cast<float*>(a.sched.partial + static_cast<size_t>(it.slot) * partial_slot_bytes(D) +
                                               static_cast<size_t>(kUnitRows) * D * 2);
          ml[R] = -INFINITY;
          ml[kUnitRows + R] = 0.f;
        }
        continue;
      }
      float m_run = -INFINITY;
      float l_run = 0.f;
      for (int j = it.kv_lo; j < jhi; ++j) {
        if (!mbar_wait(&bars->s_full[t], sc & 1, abort, a.wait_ns, a.status, kDetailSFull)) { ok = false; break; }
        ++sc;
        tc_fence_after();
        const int kb = j * kBlockN;
        float sv[kBlockN];
        // the whole S row: four loads in flight, one wait; masked where the
        // tile crosses the diagonal or the end
        auto load_s = [&]() {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          const uint32_t sa = tmem + lane_base + s_col;
          tmem_ld32(sa, r0);
          tmem_ld32(sa + 32, r1);
          tmem_ld32(sa + 64, r2);
          tmem_ld32(sa + 96, r3);
          tc_wait_ld_dep(r0);
          reg_dep(r1);
          reg_dep(r2);
          reg_dep(r3);
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            sv[x] = __uint_as_float(r0[x]);
            sv[32 + x] = __uint_as_float(r1[x]);
            sv[64 + x] = __uint_as_float(r2[x]);
            sv[96 + x] = __uint_as_float(r3[x]);
          }
          if (kb + kBlockN - 1 > it.P + i0t) {
#pragma unroll
            for (int c = 0; c < kBlockN; ++c)
              if (kb + c > lim) sv[c] = -INFINITY;
          }
        };
        load_s();
        // p = 2^(s * scale * log2 e - m): scale-and-subtract and the row sum
        // on pairs; P packed to bf16 pairs in pk0 (columns 0-63) and pk1
        uint32_t pk0[32], pk1[32];
        float sum = 0.f;
        auto exps = [&](float mbase) {
          const float2 sl2x2 = make_float2(sl2, sl2);
          const float2 negm = make_float2(-mbase, -mbase);
          float2 acc[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.f, 0.f);
#pragma unroll
          for (int x = 0; x < kBlockN / 2; ++x) {
            const float2 z = __ffma2_rn(make_float2(sv[2 * x], sv[2 * x + 1]), sl2x2, negm);
            const float2 pp = make_float2(fast_exp2(z.x), fast_exp2(z.y));
            acc[x & 3] = __fadd2_rn(acc[x & 3], pp);
            (x < 32 ? pk0 : pk1)[x & 31] = pack_bf16x2(pp.x, pp.y);
          }
          const float2 a01 = __fadd2_rn(acc[0], acc[1]);
          const float2 a23 = __fadd2_rn(acc[2], acc[3]);
          const float2 a03 = __fadd2_rn(a01, a23);
          sum = a03.x + a03.y;
        };
        // Past the item's first tile the exponentials are taken against the
        // running max at once: the tile's own max matters only if a weight
        // would pass 2^16, which the row sum shows (a sum of at most 2^16
        // bounds every weight; a non-finite one, from a row with no key yet,
        // fails too).  Otherwise (and on the first tile) the max is reduced
        // and the running max raised when the tile's exceeds it by more than
        // 8 (log2 units), with O and l rescaled: the lazy rescale.
        float factor = 1.0f;
        bool grow = false;
        bool done = false;
        if (j > it.kv_lo) {
          exps(m_run);
          done = __all_sync(0xffffffffu, sum <= 65536.0f);
          if (!done) load_s();  // the registers were spent; S is still in TMEM
        }
        if (!done) {
          // row max: 16 independent chains of 3-input maxes, then a tree
          float mx[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            mx[q] = fmax3(sv[q], sv[q + 16], sv[q + 32]);
            mx[q] = fmax3(mx[q], sv[q + 48], sv[q + 64]);
            mx[q] = fmax3(mx[q], sv[q + 80], sv[q + 96]);
            mx[q] = fmaxf(mx[q], sv[q + 112]);
          }
#pragma unroll
          for (int q = 0; q < 5; ++q) mx[q] = fmax3(mx[q], mx[q + 5], mx[q + 10]);
          const float m_tile = fmax3(fmax3(mx[0], mx[1], mx[2]), fmaxf(mx[3], mx[4]), mx[15]) * sl2;
          grow = m_tile > m_run + 8.0f;
          const float m_new = grow ? m_tile : m_run;
          factor = grow ? fast_exp2(m_run - m_new) : 1.0f;
          m_run = m_new;
          exps((m_run == -INFINITY) ? 0.f : m_run);
        }
        l_run = l_run * factor + sum;
        tmem_st32(tmem + lane_base + s_col, pk0);
        tmem_st32(tmem + lane_base + s_col + 32, pk1);
        // The S barrier fired after every earlier MMA, so O_t holds the previous
        // PV: rescale it here, before the next PV is issued.
        if (j > it.kv_lo && __any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o0[32], o1[32];
            const uint32_t oa = tmem + lane_base + o_col + c * 64;
            tmem_ld32(oa, o0);
            tmem_ld32(oa + 32, o1);
            tc_wait_ld_dep(o0);
            reg_dep(o1);
#pragma unroll
            for (int x = 0; x < 32; ++x) {
              o0[x] = __float_as_uint(__uint_as_float(o0[x]) * factor);
              o1[x] = __float_as_uint(__uint_as_float(o1[x]) * factor);
            }
            tmem_st32(oa, o0);
            tmem_st32(oa + 32, o1);
          }
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[t]);
      }
      if (!ok) break;
      // epilogue: wait for the last PV of this tile, normalise, store
      if (!mbar_wait(&bars->o_done[t], od & 1, abort, a.wait_ns, a.status, kDetailOFull)) { ok = false; break; }
      ++od;
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      if (it.whole) {
        const bool valid = i < it.E;
        const int head = it.g * a.group + r % a.group;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.out) +
                              (static_cast<int64_t>(it.q0 + i) * a.h_q + head) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t raw[32];
          tmem_ld32(tmem + lane_base + o_col + c * 32, raw);
          tc_wait_ld_dep(raw);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(raw[8 * x + 0]) * inv_l, __uint_as_float(raw[8 * x + 1]) * inv_l);
              v.y = pack_bf16x2(__uint_as_float(raw[8 * x + 2]) * inv_l, __uint_as_float(raw[8 * x + 3]) * inv_l);
              v.z = pack_bf16x2(__uint_as_float(raw[8 * x + 4]) * inv_l, __uint_as_float(raw[8 * x + 5]) * inv_l);
              v.w = pack_bf16x2(__uint_as_float(raw[8 * x + 6]) * inv_l, __uint_as_float(raw[8 * x + 7]) * inv_l);
              dst[x] = v;
            }
          }
        }
        if (valid && a.lse != nullptr)
          a.lse[static_cast<int64_t>(it.q0 + i) * a.h_q + head] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      } else {
        // one part of a unit: the normalised partial goes to the item's slot
        uint8_t* slot = a.sched.partial + static_cast<size_t>(it.slot) * partial_slot_bytes(D);
        uint4* prow = reinterpret_cast<uint4*>(slot + static_cast<size_t>(R) * D * 2);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t raw[32];
          tmem_ld32(tmem + lane_base + o_col + c * 32, raw);
          tc_wait_ld_dep(raw);
#pragma unroll
          for (int x = 0; x < 4; ++x)  // 32 columns = four 16-byte vectors of bf16 pairs
            prow[c * 4 + x] = make_uint4(
                pack_bf16x2(__uint_as_float(raw[8 * x + 0]) * inv_l, __uint_as_float(raw[8 * x + 1]) * inv_l),
                pack_bf16x2(__uint_as_float(raw[8 * x + 2]) * inv_l, __uint_as_float(raw[8 * x + 3]) * inv_l),
                pack_bf16x2(__uint_as_float(raw[8 * x + 4]) * inv_l, __uint_as_float(raw[8 * x + 5]) * inv_l),
                pack_bf16x2(__uint_as_float(raw[8 * x + 6]) * inv_l, __uint_as_float(raw[8 * x + 7]) * inv_l));
        }
        float* ml = reinterpret_cast<float*>(slot + static_cast<size_t>(kUnitRows) * D * 2);
        ml[R] = m_run;
        ml[kUnitRows + R] = l_run;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Work item w of extend_merge_kernel (see there).
template <int D>
__device__ __forceinline__ void merge_rows(const ExtendTcArgs& a, int w) {
  const UnitEntry e = a.sched.split[w / kMergeRowGroups];
  const int len = (e.n_kv + e.parts - 1) / e.parts;
  const int live = (e.n_kv + len - 1) / len;  // parts that hold key tiles
  const int q0 = a.qo_indptr[e.seq];
  const int E = a.qo_indptr[e.seq + 1] - q0;
  constexpr int kW = D / 64;  // 32-bit words (bf16 pairs) per lane and row
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int row0 = (w % kMergeRowGroups) * 32 + warp * 4;
  const uint8_t* slot0 = a.sched.partial + static_cast<size_t>(e.slot) * partial_slot_bytes(D);
#pragma unroll 1
  for (int rr = 0; rr < 4; rr += 2) {
    float m[2][kMaxParts], l[2][kMaxParts];
    uint32_t v[2][kMaxParts][kW];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int R = row0 + rr + h;
#pragma unroll
      for (int p = 0; p < kMaxParts; ++p) {
        if (p < live) {
          const uint8_t* slot = slot0 + static_cast<size_t>(p) * partial_slot_bytes(D);
          const float* ml = reinterpret_cast<const float*>(slot + static_cast<size_t>(kUnitRows) * D * 2);
          m[h][p] = ml[R];
          l[h][p] = ml[kUnitRows + R];
          const uint32_t* row = reinterpret_cast<const uint32_t*>(slot + static_cast<size_t>(R) * D * 2) + lane * kW;
          if constexpr (kW == 2) {
            const uint2 x = *reinterpret_cast<const uint2*>(row);
            v[h][p][0] = x.x;
            v[h][p][kW - 1] = x.y;
          } else {
            v[h][p][0] = row[0];
          }
        } else {
          m[h][p] = -INFINITY;
          l[h][p] = 0.f;
#pragma unroll
          for (int w = 0; w < kW; ++w) v[h][p][w] = 0u;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int R = row0 + rr + h;
      const int t = R / kBlockM;
      const int r = R % kBlockM;
      const int i = (2 * e.pair + t) * a.tok + r / a.group;
      if (i >= E) continue;
      float M = -INFINITY;
#pragma unroll
      for (int p = 0; p < kMaxParts; ++p)
        if (l[h][p] > 0.f) M = fmaxf(M, m[h][p]);
      float wsum = 0.f;
      float o[2 * kW];
#pragma unroll
      for (int c = 0; c < 2 * kW; ++c) o[c] = 0.f;
#pragma unroll
      for (int p = 0; p < kMaxParts; ++p) {
        if (!(l[h][p] > 0.f)) continue;  // this part holds no key of this row
        const float wgt = fast_exp2(m[h][p] - M) * l[h][p];
        wsum += wgt;
#pragma unroll
        for (int w = 0; w < kW; ++w) {  // bf16 -> fp32 is a shift
          o[2 * w] += wgt * __uint_as_float(v[h][p][w] << 16);
          o[2 * w + 1] += wgt * __uint_as_float(v[h][p][w] & 0xffff0000u);
        }
      }
      const float inv = 1.f / wsum;
      const int head = e.kv_head * a.group + r % a.group;
      uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) +
                                                  (static_cast<int64_t>(q0 + i) * a.h_q + head) * D) + lane * kW;
      if constexpr (kW == 2) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv));
      } else {
        dst[0] = pack_bf16x2(o[0] * inv, o[1] * inv);
      }
      if (lane == 0 && a.lse != nullptr)
        a.lse[static_cast<int64_t>(q0 + i) * a.h_q + head] = (M + __log2f(wsum)) * 0.69314718055994531f;
    }
  }
}

// Combine the parts of each cut unit (the online-softmax LSE rule: weights
// 2^(m_p - M) * l_p of the normalised part outputs) and write its rows.  The
// grid is persistent (two blocks per SM, all resident, so the next launch is
// released at once); block b takes work items b, b + gridDim.x, ..., item
// w being rows [32 g, 32 g + 32), g = w mod kMergeRowGroups, of the
// (w / kMergeRowGroups)-th cut unit.  Each of the 8 warps takes four of the
// rows, two at a time, with every part's loads in flight at once; lane l holds
// columns [l D / 32, (l + 1) D / 32), so one part of one row is one coalesced
// read.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) extend_merge_kernel(const __grid_constant__ ExtendTcArgs a) {
  // The next launch may be scheduled now: the next round's schedule does not
  // depend on this one (its own reads of the cache wait for this launch).
  grid_launch_dependents();
  grid_dependency_wait();  // the extend launch's partials are complete
  const int n_work = a.sched.header[7] * kMergeRowGroups;
  for (int w = blockIdx.x; w < n_work; w += gridDim.x) merge_rows<D>(a, w);
}

// Block-wide exclusive prefix sum (blockDim.x a multiple of 32, <= 1024).
__device__ int block_exclusive_scan(int v, int* total, int* warp_sums) {
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    int ws = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += y;
    }
    warp_sums[lane] = ws;
  }
  __syncthreads();
  const int base = w > 0 ? warp_sums[w - 1] : 0;
  *total = warp_sums[nw - 1];
  __syncthreads();
  return base + x - v;
}

// Query tiles of sequence s (0 if its lengths are out of range).
__device__ int seq_tiles(const ScheduleArgs& a, int s, bool record) {
  const int E = a.qo_indptr[s + 1] - a.qo_indptr[s];
  const int P = a.prefix_len[s];
  const bool bad = E < 0 || P < 0 || P + E > a.max_kv_len ||
                   (P + E + kPage - 1) / kPage > a.max_pages;
  if (bad && record) record_error(a.status, kStatusDeviceArg, kDetailBadLength);
  return bad ? 0 : (E + a.tok - 1) / a.tok;
}

// Parts of a unit of n_kv key tiles for target part length T, and the size
// class of a part of `size` tiles (kSizeBuckets - 1 = the largest).
__device__ __forceinline__ int unit_parts(int n_kv, int T) { return min(kMaxParts, max(1, (n_kv + T - 1) / T)); }
__device__ __forceinline__ int size_bucket(int size, int T) {
  return min(kSizeBuckets - 1, size * kSizeBuckets / (T + 1));
}

constexpr int kSchedThreads = 256;
constexpr int kSchedSeqCache = 2048;   // sequences whose pair offsets stay in shared memory
constexpr int kSchedUnitCache = 8192;  // units whose key-tile counts stay in shared memory

// Block-wide exclusive prefix sums of N per-thread counters at once (blockDim.x
// <= 32 * 32): v is replaced by this thread's prefix, totals[] (shared) gets
// the block totals.  Two barriers.
template <int N>
__device__ void block_scan_n(int (&v)[N], int (*scratch)[N], int* totals) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl[N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    int x = v[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    incl[i] = x;
    if (lane == 31) scratch[w][i] = x;
  }
  __syncthreads();
  if (threadIdx.x < N) {  // warp totals -> exclusive warp offsets, in place
    int run = 0;
    for (int k = 0; k < nw; ++k) {
      const int t = scratch[k][threadIdx.x];
      scratch[k][threadIdx.x] = run;
      run += t;
    }
    totals[threadIdx.x] = run;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = scratch[w][i] + incl[i] - v[i];
  __syncthreads();  // scratch and totals may be reused after this
}

// The work list of one extend launch.
// 1. Units: per KV head, each sequence's units last-first (the longest key
//    range first), two query tiles each.
// 2. Parts: candidate target lengths T = ceil(longest unit / S), S = 1..8; a
//    unit of n_kv key tiles is cut into ceil(n_kv / T) parts.  Each candidate
//    is costed as its waves of CTAs times (T + the fixed cost of an item), plus
//    the merge when units are cut, in key-tile times; the cheapest is taken (a
//    larger S must win clearly, by 3 %, and fit the partial slots).  On a
//    launch of one wave that is the longest item, which cutting shortens while
//    idle SMs take the parts; on long launches it is how well the parts fill
//    whole waves.  Units of equal length get the same number of parts;
//    unequal ones get parts of similar length.
// 3. Order: parts in kSizeBuckets size classes, largest first; within a class
//    part-major, then unit order (so CTAs running at the same time stream the
//    same key range of a KV head).  Position k of that order goes to CTA
//    k mod nc in even waves and nc - 1 - k mod nc in odd ones (snake order),
//    which evens out the CTAs' totals.
__device__ __forceinline__ void schedule_body(const ScheduleArgs& a) {
  constexpr int kRuns = kMaxParts * kSizeBuckets;  // (part, size class) counters
  __shared__ int warp_sums[32];
  __shared__ int scratch[32][kRuns];
  __shared__ int totals[kRuns];
  __shared__ int run_start[kRuns];
  __shared__ int s_seq_off[kSchedSeqCache + 1];
  __shared__ int s_nkv[kSchedUnitCache];
  __shared__ int s_T, s_items, s_fill;
  const int tid = threadIdx.x;
  const int n = a.seq_end - a.seq_begin;
  // pair offsets per sequence (exclusive) and their total; the item table is
  // scratch for them when there are too many sequences for shared memory
  const bool seq_cached = n <= kSchedSeqCache;
  // Launched as a dependent of the previous kernel, the schedule reads only
  // the index arrays (which that kernel does not write).  When the previous
  // round used the same workspace (a.sched_wait), that round may still read
  // it: the wait comes before the first workspace write (at once past the
  // shared-memory caches, where the workspace is scratch).
  if (a.sched_wait && !seq_cached) grid_dependency_wait();
  int* seq_off = seq_cached ? s_seq_off : reinterpret_cast<int*>(a.sched.items);
  int carry = 0;
  for (int c0 = 0; c0 < n; c0 += blockDim.x) {
    const int k = c0 + tid;
    const int np = k < n ? (seq_tiles(a, a.seq_begin + k, true) + 1) / 2 : 0;
    int chunk_total = 0;
    const int off = carry + block_exclusive_scan(np, &chunk_total, warp_sums);
    if (k < n) seq_off[k] = off;
    carry += chunk_total;
  }
  const int pairs = carry;  // units per KV head
  if (tid == 0) seq_off[n] = pairs;
  const int n_units = min(pairs * a.h_kv, a.capacity);
  if (pairs * a.h_kv > a.capacity && tid == 0) record_error(a.status, kStatusDeviceArg, kDetailBadLength);
  const bool unit_cached = n_units <= kSchedUnitCache;
  if (a.sched_wait && seq_cached && !unit_cached) grid_dependency_wait();
  __syncthreads();
  // 1. units (each thread a contiguous range, so unit order is thread order)
  const int per = (n_units + blockDim.x - 1) / blockDim.x;
  const int u_lo = min(n_units, tid * per), u_hi = min(n_units, u_lo + per);
  auto n_kv_of = [&](int u) { return unit_cached ? s_nkv[u] : a.sched.units[u].n_kv; };
  // unit u: sequence, pair and KV head (the sequence by binary search over
  // the pair offsets)
  auto unit_of = [&](int u, int& s, int& pair, int& g) {
    g = u / pairs;
    const int r = u - g * pairs;
    int lo = 0, hi = n;  // the sequence k with seq_off[k] <= r < seq_off[k + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) / 2;
      if (seq_off[mid] <= r) lo = mid; else hi = mid;
    }
    s = a.seq_begin + lo;
    const int np = seq_off[lo + 1] - seq_off[lo];
    pair = np - 1 - (r - seq_off[lo]);
  };
  int W_local = 0, max_local = 0;
  for (int u = u_lo; u < u_hi; ++u) {
    int s, pair, g;
    unit_of(u, s, pair, g);
    const int E = a.qo_indptr[s + 1] - a.qo_indptr[s];
    const int P = a.prefix_len[s];
    const int i_last = min(E, (2 * pair + 2) * a.tok);  // tokens [0, i_last) of the unit's rows
    const int n_kv = (P + i_last + kBlockN - 1) / kBlockN;
    if (unit_cached)
      s_nkv[u] = n_kv;  // the unit entry is written once its parts are known
    else
      a.sched.units[u] = UnitEntry{s, pair, g, n_kv, 1, 0};
    W_local += n_kv;
    max_local = max(max_local, n_kv);
  }
  // total key tiles and the longest unit
  {
    const int wsum = __reduce_add_sync(0xffffffffu, W_local);
    const int wmax = __reduce_max_sync(0xffffffffu, max_local);
    if ((tid & 31) == 0) {
      scratch[tid >> 5][0] = wsum;
      scratch[tid >> 5][1] = wmax;
    }
    __syncthreads();
    if (tid == 0) {
      int t = 0, m = 0;
      for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) {
        t += scratch[k][0];
        m = max(m, scratch[k][1]);
      }
      totals[0] = t;
      totals[1] = m;
    }
    __syncthreads();
  }
  const int W = totals[0];
  const int n_max = totals[1];
  __syncthreads();
  // fused mixed step: give the extend part the CTAs that make the two parts
  // end together (decode time falls off below kDecodeSatSms reading SMs)
  __shared__ int s_next;
  if (a.dec_rows > 0) {
    long long keys = 0;
    for (int s = tid; s < a.dec_rows; s += blockDim.x) keys += a.prefix_len[s] + 1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) keys += __shfl_xor_sync(0xffffffffu, keys, o);
    __shared__ long long dec_keys[32];
    if ((tid & 31) == 0) dec_keys[tid >> 5] = keys;
    __syncthreads();
    if (tid == 0) {
      long long tot = 0;
      for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) tot += dec_keys[k];
      const float t_dec = static_cast<float>(tot) * static_cast<float>(a.dec_bytes_per_key) / kDecodeBytesPerUs;
      const float t_tile = kTileUsPerSm * kFusedExtendSlowdown * static_cast<float>(a.d) / 128.f;
      int best_n = max(1, a.n_ctas - 1);
      float best_t = 3.4e38f;
      for (int nx = 4; nx <= a.n_ctas - 4; nx += 4) {
        const float te = static_cast<float>(W) * t_tile / nx;
        const float td = t_dec * fmaxf(1.f, static_cast<float>(kDecodeSatSms) / (a.n_ctas - nx));
        if (fmaxf(te, td) < best_t) {
          best_t = fmaxf(te, td);
          best_n = nx;
        }
      }
      s_next = best_n;
    }
    __syncthreads();
  } else if (tid == 0) {
    s_next = a.n_ctas;
  }
  __syncthreads();
  const int n_ext = s_next;  // CTAs the extend part may use
  // 2. parts: items and partial slots each candidate S would need
  int v16[2 * kMaxParts] = {};
  for (int u = u_lo; u < u_hi; ++u) {
    const int n_kv = n_kv_of(u);
#pragma unroll
    for (int S = 1; S <= kMaxParts; ++S) {
      const int pc = unit_parts(n_kv, max(1, (n_max + S - 1) / S));
      v16[S - 1] += pc;
      v16[kMaxParts + S - 1] += pc > 1 ? pc : 0;
    }
  }
  block_scan_n<2 * kMaxParts>(v16, reinterpret_cast<int (*)[2 * kMaxParts]>(&scratch[0][0]), totals);
  const int* sums16 = totals;
  if (tid == 0) {
    int best_T = max(1, n_max), best_fill = 0;
    float best_t = 3.4e38f;
    for (int S = 1; S <= kMaxParts; ++S) {
      const int T = max(1, (n_max + S - 1) / S);
      const int items = sums16[S - 1];
      const int slots = S > 1 ? sums16[kMaxParts + S - 1] : 0;
      if (slots > min(a.max_slots, kCutSlots)) break;
      const int ncp = max(1, min(n_ext, items));
      const int waves = (items + ncp - 1) / ncp;
      const float t = waves * (T + kItemCostTiles) + (S > 1 ? kMergeCostTiles : 0.f);
      if (t < best_t * 0.97f) {  // more parts only when they are clearly faster
        best_T = T;
        best_t = t;
        // the last wave's idle CTAs: as many units take one more part (up to
        // two more slots each), where that shortens the last wave by clearly
        // more than an item costs (about T / (S + 1) key tiles)
        const bool worth = T >= 4.f * kItemCostTiles * (S + 1);
        best_fill = (waves > 1 && worth) ? min(waves * ncp - items, (a.max_slots - slots) / 2) : 0;
      }
    }
    s_T = best_T;
    s_fill = best_fill;
  }
  __syncthreads();
  const int T = s_T;
  const int fill = s_fill;
  // Filling the last wave: the first `fill` units in unit order that can take
  // one more part do, so that the items number whole waves; their (smaller)
  // parts go one size class down, after the others, so the last waves get the
  // smaller items.  rank0: this thread's count of earlier such units.
  int rank0 = 0;
  if (fill > 0) {  // (uniform: the scan's barriers are met by every thread)
    int elig = 0;
    for (int u = u_lo; u < u_hi; ++u) {
      const int n_kv = n_kv_of(u);
      elig += (unit_parts(n_kv, T) < kMaxParts && n_kv > unit_parts(n_kv, T)) ? 1 : 0;
    }
    int elig_total = 0;
    rank0 = block_exclusive_scan(elig, &elig_total, warp_sums);
  }
  // parts of a unit of n_kv key tiles; extra: it took a filling part (rank:
  // eligible units before it, advanced here)
  auto parts_of = [&](int n_kv, int& rank, bool& extra) {
    const int pc = unit_parts(n_kv, T);
    extra = false;
    if (fill > 0 && pc < kMaxParts && n_kv > pc) extra = rank++ < fill;
    return pc + (extra ? 1 : 0);
  };
  // 3. parts and partial slots per unit (slots in unit order, split units only)
  // (and the cut units' ranks in the list the merge kernel walks)
  int sc2[2] = {0, 0};
  {
    int rank = rank0;
    bool ex;
    for (int u = u_lo; u < u_hi; ++u) {
      const int pc = parts_of(n_kv_of(u), rank, ex);
      sc2[0] += pc > 1 ? pc : 0;
      sc2[1] += pc > 1 ? 1 : 0;
    }
  }
  block_scan_n<2>(sc2, reinterpret_cast<int (*)[2]>(&scratch[0][0]), totals);
  int slot = sc2[0], split_rank = sc2[1];
  const int n_split = totals[1];
  if (a.sched_wait && unit_cached) grid_dependency_wait();  // the workspace writes start here
  int rank = rank0;
  bool ex;
  for (int u = u_lo; u < u_hi; ++u) {
    const int n_kv = n_kv_of(u);
    const int pc = parts_of(n_kv, rank, ex);
    UnitEntry e;
    if (unit_cached) {
      int s, pair, g;
      unit_of(u, s, pair, g);
      e = UnitEntry{s, pair, g, n_kv, pc, pc > 1 ? slot : 0};
    } else {
      e = a.sched.units[u];
      e.parts = pc;
      e.slot = pc > 1 ? slot : 0;
    }
    a.sched.units[u] = e;
    if (pc > 1) a.sched.split[split_rank++] = e;
    slot += pc > 1 ? pc : 0;
  }
  // item counts per (part, size class); this thread's prefix in each run
  int cnt[kRuns] = {};
  rank = rank0;
  for (int u = u_lo; u < u_hi; ++u) {
    const int n_kv = n_kv_of(u);
    const int pc = parts_of(n_kv, rank, ex);
    const int len = (n_kv + pc - 1) / pc;
#pragma unroll
    for (int p = 0; p < kMaxParts; ++p) {
      const int size = min(len, n_kv - p * len);
      const int b = max(0, size_bucket(max(size, 0), T) - (ex ? 1 : 0));
#pragma unroll
      for (int q = 0; q < kSizeBuckets; ++q) cnt[p * kSizeBuckets + q] += (p < pc && size > 0 && b == q) ? 1 : 0;
    }
  }
  block_scan_n<kRuns>(cnt, scratch, totals);
  // start of each (part, class) run in the largest-first order
  if (tid == 0) {
    int pos = 0;
    for (int b = kSizeBuckets - 1; b >= 0; --b)
      for (int p = 0; p < kMaxParts; ++p) {
        run_start[p * kSizeBuckets + b] = pos;
        pos += totals[p * kSizeBuckets + b];
      }
    s_items = pos;
  }
  __syncthreads();
  const int n_items = s_items;
  const int nc = n_items > 0 ? min(n_ext, n_items) : 0;
  const int table_len = nc > 0 ? (n_items + nc - 1) / nc * nc : 0;
  // the last wave's unused entries read as empty: its low CTAs' entries when
  // that wave runs backwards (odd), its high ones otherwise
  if (table_len > n_items) {
    const int last = table_len / nc - 1;
    const int rem = n_items - last * nc;
    const int e0 = last * nc + ((last & 1) ? 0 : rem);
    for (int i = e0 + tid; i < e0 + (nc - rem); i += blockDim.x) a.sched.items[i] = ItemDesc{0, 0, 0, 0, 0, 0, 0, -1};
  }
  rank = rank0;
  for (int u = u_lo; u < u_hi; ++u) {
    const int n_kv = n_kv_of(u);
    const int pc = parts_of(n_kv, rank, ex);
    const int len = (n_kv + pc - 1) / pc;
    const UnitEntry ue = a.sched.units[u];  // written by this thread above
    const int q0 = a.qo_indptr[ue.seq];
    const int E = a.qo_indptr[ue.seq + 1] - q0;
    const int P = a.prefix_len[ue.seq];
#pragma unroll
    for (int p = 0; p < kMaxParts; ++p) {
      const int size = min(len, n_kv - p * len);
      if (p >= pc || size <= 0) continue;
      const int b = max(0, size_bucket(size, T) - (ex ? 1 : 0));
      int k = 0;  // this item's position: its run's start plus the items before it in the run
#pragma unroll
      for (int q = 0; q < kSizeBuckets; ++q)
        if (b == q) k = run_start[p * kSizeBuckets + q] + cnt[p * kSizeBuckets + q]++;
      const int wave = k / nc, pos = k - wave * nc;
      const int cta = (wave & 1) ? nc - 1 - pos : pos;
      a.sched.items[wave * nc + cta] = ItemDesc{ue.seq, (ue.kv_head << kPairBits) | ue.pair, q0, E, P,
                                                p * len, min(p * len + len, n_kv), pc > 1 ? ue.slot + p : -1};
    }
  }
  if (tid == 0) {
    a.sched.header[0] = W;
    a.sched.header[1] = nc;
    a.sched.header[2] = n_units;
    a.sched.header[3] = table_len;
    a.sched.header[4] = T;
    a.sched.header[5] = n_items;
    a.sched.header[6] = 0;
    a.sched.header[7] = n_split;
  }
}

__global__ void __launch_bounds__(kSchedThreads, 1) schedule_kernel(ScheduleArgs a) {
  grid_launch_dependents();  // the extend launch may be scheduled (it waits for this one)
  schedule_body(a);
  grid_dependency_wait();  // this launch completes after the previous one
}

// A mixed step's prep launch: block 0 builds the extend schedule while the
// other blocks append the round's K/V rows (kAppendRowsPerBlock per block); the
// schedule reads only the index arrays, so the two are independent.
static_assert(kSchedThreads == kAppendRowsPerBlock * 32, "one warp per appended row");
__global__ void __launch_bounds__(kSchedThreads) prep_kernel(ScheduleArgs a, KvAppendArgs k) {
  grid_launch_dependents();
  if (blockIdx.x == 0) {
    schedule_body(a);
    grid_dependency_wait();  // this launch completes after the previous one
  } else {
    grid_dependency_wait();  // the previous launch may still read the cache
    append_row(k, (blockIdx.x - 1) * kAppendRowsPerBlock + (threadIdx.x >> 5), threadIdx.x & 31);
  }
}

}  // namespace

size_t extend_tc_smem_bytes(int d) {
  return d == 128 ? TcCfg<128>::kSmem : TcCfg<64>::kSmem;
}


// The softmax warpgroups raise their register limit at run time; that only
// completes if the launch allocated at least kLaunchRegs per thread.
template <int D, bool S, bool F>
cudaError_t check_regs() {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, extend_tc_kernel<D, S, F>);
  if (e != cudaSuccess) return e;
  return fa.numRegs >= kLaunchRegs ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Launch, with programmatic stream serialisation if `dependent`: the kernel may
// then be scheduled while the one before it finishes and waits in
// grid_dependency_wait().
template <typename Kernel, typename Arg>
cudaError_t launch_dependent(Kernel kernel, int grid, int block, int smem, cudaStream_t s, const Arg& arg,
                             bool dependent) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t s, bool dependent) {
  return launch_dependent(schedule_kernel, 1, kSchedThreads, 0, s, a, dependent);
}

cudaError_t launch_prep(const ScheduleArgs& a, const KvAppendArgs& k, cudaStream_t s, bool dependent) {
  const int blocks = 1 + (k.total_q + kAppendRowsPerBlock - 1) / kAppendRowsPerBlock;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kSchedThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prep_kernel, a, k);
}

// Once per device, head size and form: the register check and the
// shared-memory opt-in (both hold for the loaded module).
template <int D, bool S, bool F>
cudaError_t prepare_extend() {
  static std::atomic<int> ready[64];  // 0: not yet, 1: done
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && ready[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = check_regs<D, S, F>();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(extend_tc_kernel<D, S, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) ready[dev].store(1, std::memory_order_release);
  return cudaSuccess;
}

template <int D, bool S, bool F>
cudaError_t launch_extend_form(const ExtendTcArgs& a, cudaStream_t s, bool dependent) {
  cudaError_t e = prepare_extend<D, S, F>();
  if (e != cudaSuccess) return e;
  e = launch_dependent(extend_tc_kernel<D, S, F>, a.n_ctas, kThreads, TcCfg<D>::kSmem, s, a, dependent);
  if (e != cudaSuccess) return e;
  // the merge's persistent grid: two blocks per SM, fewer if there cannot be that much work
  const int merge_grid = std::max(1, std::min(a.max_split * kMergeRowGroups, 2 * a.n_ctas));
  return launch_dependent(extend_merge_kernel<D>, merge_grid, kMergeThreads, 0, s, a, dependent);
}

cudaError_t launch_extend_tc(const ExtendTcArgs& a, cudaStream_t s, bool dependent) {
  if (a.n_ctas <= 0) return cudaSuccess;
  // (the staged form never carries decode rows: the host stages only launches without them)
  if (a.d == 128) {
    if (a.staged) return launch_extend_form<128, true, false>(a, s, dependent);
    return a.dec_items > 0 ? launch_extend_form<128, false, true>(a, s, dependent)
                           : launch_extend_form<128, false, false>(a, s, dependent);
  }
  if (a.staged) return launch_extend_form<64, true, false>(a, s, dependent);
  return a.dec_items > 0 ? launch_extend_form<64, false, true>(a, s, dependent)
                         : launch_extend_form<64, false, false>(a, s, dependent);
}

}  // namespace cpe
