// Extend attention on CTA pairs: the two-SM form of the 5th-generation
// tensor-core MMA (tcgen05.mma.cta_group::2), for head size 128.
//
// Two CTAs on neighbouring SMs form a cluster and share one work unit of four
// query tiles (512 rows) of one sequence and KV head.  CTA c holds the unit's
// tiles c and c + 2 as its local tiles 0 and 1, so the pair's tile t (rows
// [256 t, 256 t + 256) of the unit) is CTA 0's local tile t on top of CTA 1's.
// One MMA instruction, issued by CTA 0, computes an M = 256 product for both:
// each CTA supplies its own 128 rows of A (Q from its shared memory, or P from
// its tensor memory) and half of B, and receives its own 128 rows of D in its
// tensor memory.  For S = Q K^T the halves of B are keys 0-63 (CTA 0) and
// 64-127 (CTA 1) of the key tile; for O += P V they are the head dimension's
// columns 0-63 and 64-127.  Each CTA therefore stages half of every K and V
// tile (32 KB per key tile instead of 64, each byte serving 512 query rows),
// and the shared memory this frees holds a ring of five key tiles.
//
// Everything else follows the one-CTA kernel (extend_tc.cu): key tiles in
// order, the cached-prefix rectangle (Stage 1 of the SGLang chunked-prefill
// article) unmasked, the chunk's causal triangle (Stage 2) masked only where a
// tile crosses the diagonal, one running (m, l, O) per row (the article's
// online-softmax LSE merge applied tile by tile), the same balanced persistent
// schedule (in units of four tiles, one entry per pair) and the same merge of
// key-range parts.
//
// Roles in each CTA (384 threads):
//   warp 0      TMA producer: the CTA's two Q tiles of each unit, then per key
//               tile its half of K (64 keys x 128 dims) and of V (128 keys x
//               64 dims) into one ring stage
//   warp 1      CTA 0: TMEM owner and the pair's MMA issuer; CTA 1: TMEM owner
//               and relay (it forwards "this CTA's Q / stage has landed" to
//               CTA 0's barriers, so every copy completes on its own CTA's
//               barrier and each producer can drain its own copies)
//   warps 4-11  softmax of local tiles 0 and 1 (one thread per row), as in the
//               one-CTA kernel; P hand-offs of CTA 1 arrive on CTA 0's barrier
// MMA completions are signalled to both CTAs at once (commit with a CTA mask).
// TMEM columns: [0,128) S0, [128,256) S1, [256,384) O0, [384,512) O1.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records
// CPE_ERR_TIMEOUT and every role leaves its loop.  The kernel has one exit for
// the pair's extend work: both CTAs meet at a cluster barrier (after CTA 0's
// MMAs have drained and each producer's copies have landed) and free their
// tensor memory together.
#include <atomic>

#include "cpe_device.cuh"
#include "decode_item.cuh"
#include "kernels.h"

namespace cpe {

namespace {

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr uint64_t kDrainNs = 2000000000ull;

// Shared memory of one CTA of a pair (head size 128).
struct PairCfg {
  static constexpr int D = 128;
  static constexpr int kQTileBytes = kBlockM * D * 2;   // 128 rows x 128 dims
  static constexpr int kQHalfBytes = kBlockM * 128;     // one 128-byte column block of a Q tile
  static constexpr int kKBytes = 64 * D * 2;            // this CTA's 64 keys of a key tile, all dims
  static constexpr int kKHalfBytes = 64 * 128;          // one column block of those
  static constexpr int kVBytes = kBlockN * 128;         // all 128 keys, this CTA's 64 dims
  static constexpr int kStageBytes = kKBytes + kVBytes;
  static constexpr int kStages = 5;
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = 2 * kQTileBytes;
  static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
  static constexpr int kSmem = kBarOff + 512 + 1024;   // + barriers + alignment slack
};
static_assert(PairCfg::kSmem <= 227 * 1024, "shared memory of one CTA");
static_assert(1024 + 3 * DecCfg<128>::kSmem + 64 <= PairCfg::kSmem, "three decode items fit a CTA's shared memory");

struct PairBars {
  uint64_t q_full, q_empty, q_peer;
  uint64_t kv_full[PairCfg::kStages], kv_empty[PairCfg::kStages], kv_peer[PairCfg::kStages];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: the abort flag of the final drain waits, which must not give up early
};
static_assert(sizeof(PairBars) <= 512, "barrier area");

// ---- cluster and two-CTA forms -------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory address (cluster window) of the same location in CTA 0 of the cluster.
__device__ __forceinline__ uint32_t in_cta0(const void* p) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_u32(p)));
  return r;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Every thread of both CTAs: arrive, then wait for all (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ bool try_wait_cl(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// mbar_wait with acquire at cluster scope: for barriers the other CTA arrives on.
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort, uint64_t limit_ns,
                                             int* status, int detail) {
  if (try_wait_cl(bar, parity, 0u)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (limit_ns > 0 && try_wait_cl(bar, parity, 100000u)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 >= limit_ns) {
      record_error(status, kStatusTimeout, detail);
      *abort = 1;
      return false;
    }
  }
}

// Three non-blocking phase tests at cluster scope; bit i set when barrier i's
// phase with parity pi completed.
__device__ __forceinline__ uint32_t test3_cl(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1, uint64_t* b2,
                                             uint32_t p2) {
  uint32_t r0, r1, r2;
  asm volatile(
      "{\n\t.reg .pred q0, q1, q2;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q0, [%3], %4;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q1, [%5], %6;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q2, [%7], %8;\n\t"
      "selp.u32 %0, 1, 0, q0;\n\t"
      "selp.u32 %1, 2, 0, q1;\n\t"
      "selp.u32 %2, 4, 0, q2;\n\t}"
      : "=r"(r0), "=r"(r1), "=r"(r2)
      : "r"(smem_u32(b0)), "r"(p0), "r"(smem_u32(b1)), "r"(p1), "r"(smem_u32(b2)), "r"(p2)
      : "memory");
  return r0 | r1 | r2;
}

// Tensor memory of both CTAs: executed by one warp in each CTA of the pair.
__device__ __forceinline__ void tmem_alloc2(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A[smem] * B[smem] over both CTAs (no "memory" clobber, as for the one-CTA form).
__device__ __forceinline__ void mma2_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D (+)= A[tmem] * B[smem] over both CTAs.
__device__ __forceinline__ void mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Arrive on `bar` in both CTAs once every MMA issued so far by this thread completes.
__device__ __forceinline__ void commit_both(uint64_t* bar) {
  const uint16_t mask = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Arrive on `bar` in this CTA only.
__device__ __forceinline__ void commit_own(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void setmaxnreg_dec_producer() { asm volatile("setmaxnreg.dec.sync.aligned.u32 96;"); }
__device__ __forceinline__ void setmaxnreg_inc_softmax() { asm volatile("setmaxnreg.inc.sync.aligned.u32 200;"); }

// Work item of a pair: key tiles [kv_lo, kv_hi) of one four-tile unit.
struct PairItem {
  int seq, g, q0, E, P, kv_lo, kv_hi, slot;
  bool whole;               // the unit is not cut: its output goes straight to out / lse
  int i0_0, i0_1;           // first token of this CTA's local tiles 0 and 1
  int kv_end_0, kv_end_1;   // key limit of the pair's tiles 0 and 1 (the later of their two CTA tiles)
  int n_kt_0, n_kt_1;       // key tiles of the pair's tiles 0 and 1
  int kv_max;               // key limit of the unit (the copies)
  __device__ __forceinline__ int i0(int t) const { return t ? i0_1 : i0_0; }
  __device__ __forceinline__ int kv_end(int t) const { return t ? kv_end_1 : kv_end_0; }
  __device__ __forceinline__ int n_kt(int t) const { return t ? n_kt_1 : n_kt_0; }
};

__device__ __forceinline__ bool load_pair_item(const ExtendTcArgs& a, int i, uint32_t rank, PairItem& it) {
  const int4* d = reinterpret_cast<const int4*>(a.sched.items + i);
  const int4 x = d[0];
  const int4 y = d[1];
  it.kv_lo = y.y;
  it.kv_hi = y.z;
  if (it.kv_lo >= it.kv_hi) return false;
  it.seq = x.x;
  it.g = x.y >> kPairBits;
  const int unit = x.y & ((1 << kPairBits) - 1);
  it.q0 = x.z;
  it.E = x.w;
  it.P = y.x;
  it.slot = y.w;
  it.whole = it.slot < 0;
  const int base = 4 * unit * a.tok;
  auto end_of = [&](int ut) {  // key limit of unit tile ut (0 when past the chunk)
    const int f = base + ut * a.tok;
    return f < it.E ? it.P + min(it.E, f + a.tok) : 0;
  };
  it.kv_end_0 = max(end_of(0), end_of(1));
  it.kv_end_1 = max(end_of(2), end_of(3));
  it.n_kt_0 = (it.kv_end_0 + kBlockN - 1) / kBlockN;
  it.n_kt_1 = (it.kv_end_1 + kBlockN - 1) / kBlockN;
  it.kv_max = max(it.kv_end_0, it.kv_end_1);
  it.i0_0 = base + static_cast<int>(rank) * a.tok;
  it.i0_1 = base + (2 + static_cast<int>(rank)) * a.tok;
  return true;
}

// The fused mixed step's decode rows on a CTA the extend part does not use
// (as in the one-CTA kernel: three decode items at a time, one per warpgroup).
__device__ void pair_decode_worker(const ExtendTcArgs& a, uint8_t* smem) {
  const int wg = threadIdx.x / 128;
  const int tid = threadIdx.x % 128;
  uint8_t* dsm = smem + wg * DecCfg<128>::kSmem;
  volatile int* slot = reinterpret_cast<volatile int*>(smem + 3 * DecCfg<128>::kSmem) + wg;
  const int splits = a.dec.max_splits;
  for (;;) {
    if (tid == 0) *slot = atomicAdd(&a.sched.header[6], 1);
    group_sync(1 + wg);
    const int item = *slot;
    group_sync(1 + wg);
    if (item >= a.dec_items) break;
    const int sp = item % splits;
    const int rest = item / splits;
    decode_item<128>(a.dec, sp, rest / a.h_kv, rest % a.h_kv, dsm, tid, 1 + wg);
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    extend_pair_kernel(const __grid_constant__ ExtendTcArgs a) {
  using C = PairCfg;
  constexpr int NS = C::kStages;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairBars* bars = reinterpret_cast<PairBars*>(smem + C::kBarOff);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x / 2;
  volatile int* abort = &bars->abort;

  // Both CTAs' tensor memory, allocated together before the dependency wait.
  if (warp == 1) {
    tmem_alloc2(&bars->tmem_base, 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  grid_dependency_wait();
  grid_launch_dependents();
  const int nc = a.sched.header[1];       // pairs with extend work
  const int n_items = a.sched.header[3];  // item-table entries; pair p takes p, p + nc, ...
  if (pair >= nc) {  // both CTAs of the pair take this branch
    if (warp == 1) tmem_dealloc2(tmem, 512);
    if (a.dec_items > 0) pair_decode_worker(a, smem);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->q_peer, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
      mbar_init(&bars->kv_peer[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 8);  // four softmax warps in each CTA
      mbar_init(&bars->o_done[i], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->never = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  cluster_sync();  // both CTAs' barriers are initialised before either arrives on the other's

  if (warp < 4) {
    setmaxnreg_dec_producer();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ producer
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_k64);
      prefetch_tmap(&a.tm_v128);
      const int oob = static_cast<int>(a.num_pages * kPage);  // a row past the cache: zero fill
      const int c = static_cast<int>(rank);
      int cnt = 0, items = 0;
      bool ok = true;
      PairItem it;
      for (int wi = pair; ok && wi < n_items; wi += nc) {
        if (!load_pair_item(a, wi, rank, it)) continue;
        if (items > 0 && !mbar_wait(&bars->q_empty, (items - 1) & 1, abort, a.wait_ns, a.status, kDetailQFull)) break;
        mbar_arrive_expect_tx(&bars->q_full, 2 * C::kQTileBytes);
        for (int t = 0; t < 2; ++t)
          for (int h = 0; h < 2; ++h)
            tma_load_3d(smem + C::kQOff + t * C::kQTileBytes + h * C::kQHalfBytes, &a.tm_q, &bars->q_full, h * 64,
                        it.g * a.group, it.q0 + it.i0(t));
        ++items;
        const int32_t* pt = a.page_table + static_cast<int64_t>(it.seq) * a.max_pages;
        for (int j = it.kv_lo; j < it.kv_hi; ++j, ++cnt) {
          const int st = cnt % NS;
          const int use = cnt / NS;
          const int keys = min(kBlockN, it.kv_max - j * kBlockN);
          const int npv = (keys + kPage - 1) / kPage;                  // pages of V (all of the tile's keys)
          const int npk = (max(0, min(64, keys - 64 * c)) + kPage - 1) / kPage;  // pages of this CTA's keys
          int rows[kBlockN / kPage];
          bool contiguous = true;
#pragma unroll
          for (int pg = 0; pg < kBlockN / kPage; ++pg) {
            if (pg >= npv) break;
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
          if (use > 0 &&
              !mbar_wait(&bars->kv_empty[st], (use - 1) & 1, abort, a.wait_ns, a.status, kDetailKEmpty)) {
            ok = false;
            break;
          }
          uint8_t* kdst = smem + C::kStageOff + st * C::kStageBytes;
          uint8_t* vdst = kdst + C::kKBytes;
          mbar_arrive_expect_tx(&bars->kv_full[st], npk * kPage * 256 + npv * kPage * 128);
          // K: this CTA's pages 4c .. 4c + npk - 1, both 64-dim halves (rows
          // picked by a select: a runtime index would put rows[] in local memory)
          if (contiguous && npk == 4) {
            const int r0 = c ? rows[4] : rows[0];
            for (int h = 0; h < 2; ++h)
              tma_load_3d(kdst + h * C::kKHalfBytes, &a.tm_k64, &bars->kv_full[st], h * 64, it.g, r0);
          } else {
#pragma unroll
            for (int pg = 0; pg < 4; ++pg) {
              if (pg >= npk) break;
              const int rp = c ? rows[4 + pg] : rows[pg];
              for (int h = 0; h < 2; ++h)
                tma_load_3d(kdst + h * C::kKHalfBytes + pg * (kPage * 128), &a.tm_k, &bars->kv_full[st], h * 64, it.g,
                            rp);
            }
          }
          // V: every page of the tile, this CTA's 64 dims
          if (contiguous && npv == kBlockN / kPage) {
            tma_load_3d(vdst, &a.tm_v128, &bars->kv_full[st], 64 * c, it.g, rows[0]);
          } else {
#pragma unroll
            for (int pg = 0; pg < kBlockN / kPage; ++pg) {
              if (pg >= npv) break;
              tma_load_3d(vdst + pg * (kPage * 128), &a.tm_v, &bars->kv_full[st], 64 * c, it.g, rows[pg]);
            }
          }
        }
      }
      // Drain: every copy this CTA issued lands before it leaves.
      if (*abort) {
        volatile int* no_abort = &bars->never;
        if (items > 0) mbar_wait(&bars->q_full, (items - 1) & 1, no_abort, kDrainNs, a.status, kDetailDrain);
        for (int n = max(0, cnt - NS); n < cnt; ++n)
          mbar_wait(&bars->kv_full[n % NS], (n / NS) & 1, no_abort, kDrainNs, a.status, kDetailDrain);
      }
    } else if (warp == 1 && lane == 0 && rank == 1) {
      // ------------------------------------------------------------ relay (CTA 1)
      // Forwards the completion of this CTA's Q and stage copies to CTA 0.
      const uint32_t q_peer = in_cta0(&bars->q_peer);
      int cnt = 0, items = 0;
      bool ok = true;
      PairItem it;
      for (int wi = pair; ok && wi < n_items; wi += nc) {
        if (!load_pair_item(a, wi, rank, it)) continue;
        if (!mbar_wait(&bars->q_full, items & 1, abort, a.wait_ns, a.status, kDetailQFull)) break;
        ++items;
        mbar_arrive_cluster(q_peer);
        for (int j = it.kv_lo; j < it.kv_hi; ++j, ++cnt) {
          const int st = cnt % NS;
          if (!mbar_wait(&bars->kv_full[st], (cnt / NS) & 1, abort, a.wait_ns, a.status, kDetailKFull)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(in_cta0(&bars->kv_peer[st]));
        }
      }
    } else if (warp == 1 && lane == 0 && rank == 0) {
      // ------------------------------------------------------------ MMA issuer (CTA 0)
      constexpr uint32_t idesc_qk = idesc_bf16_f32(256, kBlockN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(256, D, 1);
      // S of the pair's tile t against the K half in stage st
      auto issue_s = [&](int t, int st) {
        const uint64_t qd = smem_desc_sw128(smem_u32(smem + C::kQOff + t * C::kQTileBytes), 16, 1024);
        const uint64_t kd = smem_desc_sw128(smem_u32(smem + C::kStageOff + st * C::kStageBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t qo = static_cast<uint64_t>(((kk / 4) * C::kQHalfBytes + (kk % 4) * 32) >> 4);
          const uint64_t ko = static_cast<uint64_t>(((kk / 4) * C::kKHalfBytes + (kk % 4) * 32) >> 4);
          mma2_ss(tmem + t * 128, qd + qo, kd + ko, idesc_qk, kk > 0);
        }
        commit_both(&bars->s_full[t]);
      };
      // both CTAs' copies of stage st (use u) have landed
      auto stage_wait = [&](int st, int u) {
        return mbar_wait(&bars->kv_full[st], u & 1, abort, a.wait_ns, a.status, kDetailKFull) &&
               mbar_wait_cl(&bars->kv_peer[st], u & 1, abort, a.wait_ns, a.status, kDetailKFull);
      };
      int kc = 0, items = 0;
      int pc0 = 0, pc1 = 0;  // P hand-offs consumed per tile
      bool ok = true;
      PairItem it;
      for (int wi = pair; ok && wi < n_items; wi += nc) {
        if (!load_pair_item(a, wi, rank, it)) continue;
        if (!mbar_wait(&bars->q_full, items & 1, abort, a.wait_ns, a.status, kDetailQFull) ||
            !mbar_wait_cl(&bars->q_peer, items & 1, abort, a.wait_ns, a.status, kDetailQFull) ||
            !stage_wait(kc % NS, kc / NS)) {
          ok = false;
          break;
        }
        ++items;
        tc_fence_after();
        if (it.kv_lo < it.n_kt_0) issue_s(0, kc % NS);
        if (it.kv_lo < it.n_kt_1) issue_s(1, kc % NS);
        for (int j = it.kv_lo; j < it.kv_hi; ++j) {
          const int cur = kc % NS;
          const int nxt = (kc + 1) % NS;
          const uint32_t nph = ((kc + 1) / NS) & 1;
          const bool more = j + 1 < it.kv_hi;
          // the next stage (both halves) and tile 0's P are usually ready:
          // test all three at once and wait only for what is not
          const uint32_t ready = test3_cl(&bars->kv_full[nxt], nph, &bars->kv_peer[nxt], nph, &bars->p_full[0],
                                          pc0 & 1);
          if (more && (!(ready & 1u) || !(ready & 2u)) && !stage_wait(nxt, (kc + 1) / NS)) {
            ok = false;
            break;
          }
          const bool p0_ready = (j < it.n_kt_0) && (ready & 4u);
          const uint64_t vdesc =
              smem_desc_sw128(smem_u32(smem + C::kStageOff + cur * C::kStageBytes + C::kKBytes), 1024, 1024);
          auto tile_step = [&](const int t) -> bool {
            if (j >= it.n_kt(t)) return true;
            int& pct = t ? pc1 : pc0;
            if (!(t == 0 && p0_ready) &&
                !mbar_wait_cl(&bars->p_full[t], pct & 1, abort, a.wait_ns, a.status, kDetailPFull))
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
                mma2_ts(dcol, acol + kk * 8, vdesc + static_cast<uint64_t>(kk * (16 * 128 / 16)), idesc_pv,
                        (first || kk > 0) ? 1u : 0u);
            } else {
              const int nsteps = (keys + 15) / 16;  // only pages that were loaded
              for (int kk = 0; kk < nsteps; ++kk)
                mma2_ts(dcol, acol + kk * 8, vdesc + static_cast<uint64_t>(kk * (16 * 128 / 16)), idesc_pv,
                        (first || kk > 0) ? 1u : 0u);
            }
            if (j + 1 < min(it.kv_hi, it.n_kt(t)))
              issue_s(t, nxt);
            else
              commit_both(&bars->o_done[t]);
            return true;
          };
          if (!tile_step(0) || !tile_step(1)) {
            ok = false;
            break;
          }
          commit_both(&bars->kv_empty[cur]);  // K_j and V_j are read by everything issued so far
          ++kc;
        }
        commit_both(&bars->q_empty);  // every S of this item issued: Q may be replaced
      }
      // Drain: every MMA issued above has completed before the pair frees its tensor memory.
      commit_own(&bars->drain);
      mbar_wait(&bars->drain, 0, &bars->never, kDrainNs, a.status, kDetailDrain);
    }
  } else {
    setmaxnreg_inc_softmax();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) / 4;          // local tile of this warpgroup
    const int quad = warp & 3;             // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;        // row of the local tile
    const int ut = 2 * t + static_cast<int>(rank);  // tile of the unit
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_col = t * 128;
    const uint32_t o_col = 256 + t * D;
    const float sl2 = a.scale_log2;
    constexpr size_t slot_bytes = partial_slot_bytes(D, kPairUnitRows);
    int sc = 0, od = 0;
    bool ok = true;
    PairItem it;
    for (int wi = pair; ok && wi < n_items; wi += nc) {
      if (!load_pair_item(a, wi, rank, it)) continue;
      const int i0t = it.i0(t);
      const int i = i0t + r / a.group;              // token index within the chunk
      const int lim = it.P + min(i, it.E - 1);    // last key this row may see
      const int jhi = min(it.kv_hi, it.n_kt(t));
      const int R = ut * kBlockM + r;              // row of the unit
      if (it.kv_lo >= jhi) {
        if (!it.whole) {  // an empty part for this tile: l = 0 tells the merge to skip it
          float* ml = reinterpret_cast<float*>(a.sched.partial + static_cast<size_t>(it.slot) * slot_bytes +
                                               static_cast<size_t>(kPairUnitRows) * D * 2);
          ml[R] = -INFINITY;
          ml[kPairUnitRows + R] = 0.f;
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
            for (int cc = 0; cc < kBlockN; ++cc)
              if (kb + cc > lim) sv[cc] = -INFINITY;
          }
        };
        load_s();
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
        // Exponentials against the running max first; the tile's own max only
        // when a weight could pass 2^16 (the row sum shows it) or on the
        // item's first tile; the running max then rises only by more than 2^8.
        float factor = 1.0f;
        bool grow = false;
        bool done = false;
        if (j > it.kv_lo) {
          exps(m_run);
          done = __all_sync(0xffffffffu, sum <= 65536.0f);
          if (!done) load_s();
        }
        if (!done) {
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
        if (j > it.kv_lo && __any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb) {
            uint32_t o0[32], o1[32];
            const uint32_t oa = tmem + lane_base + o_col + cb * 64;
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
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(&bars->p_full[t]);
          else
            mbar_arrive_cluster(in_cta0(&bars->p_full[t]));
        }
      }
      if (!ok) break;
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
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t raw[32];
          tmem_ld32(tmem + lane_base + o_col + cb * 32, raw);
          tc_wait_ld_dep(raw);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cb * 32);
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
        uint8_t* slot = a.sched.partial + static_cast<size_t>(it.slot) * slot_bytes;
        uint4* prow = reinterpret_cast<uint4*>(slot + static_cast<size_t>(R) * D * 2);
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t raw[32];
          tmem_ld32(tmem + lane_base + o_col + cb * 32, raw);
          tc_wait_ld_dep(raw);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            prow[cb * 4 + x] = make_uint4(
                pack_bf16x2(__uint_as_float(raw[8 * x + 0]) * inv_l, __uint_as_float(raw[8 * x + 1]) * inv_l),
                pack_bf16x2(__uint_as_float(raw[8 * x + 2]) * inv_l, __uint_as_float(raw[8 * x + 3]) * inv_l),
                pack_bf16x2(__uint_as_float(raw[8 * x + 4]) * inv_l, __uint_as_float(raw[8 * x + 5]) * inv_l),
                pack_bf16x2(__uint_as_float(raw[8 * x + 6]) * inv_l, __uint_as_float(raw[8 * x + 7]) * inv_l));
        }
        float* ml = reinterpret_cast<float*>(slot + static_cast<size_t>(kPairUnitRows) * D * 2);
        ml[R] = m_run;
        ml[kPairUnitRows + R] = l_run;
      }
    }
  }

  // One exit for both CTAs: CTA 0's MMAs have drained and each CTA's copies
  // have landed; after the cluster barrier no CTA touches the other's shared
  // memory, and the pair frees its tensor memory together.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem, 512);
  }
}

}  // namespace

// Once per device: the register check (the softmax warpgroups raise their
// limit at run time, which completes only if the launch allocated kLaunchRegs
// per thread), the shared-memory opt-in, and how many pairs stay resident.
int pair_workers(cudaError_t* err) {
  static std::atomic<int> cache[64];  // 0: not yet, -1: failed, else pairs
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int have = cache[dev].load(std::memory_order_acquire);
  if (have > 0) return have;
  cudaFuncAttributes fa;
  *err = cudaFuncGetAttributes(&fa, extend_pair_kernel);
  if (*err != cudaSuccess) return 0;
  if (fa.numRegs < kLaunchRegs) {
    *err = cudaErrorInvalidConfiguration;
    return 0;
  }
  *err = cudaFuncSetAttribute(extend_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::kSmem);
  if (*err != cudaSuccess) return 0;
  int sms = 0;
  *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (*err != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms & ~1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = PairCfg::kSmem;
  int clusters = 0;
  *err = cudaOccupancyMaxActiveClusters(&clusters, extend_pair_kernel, &cfg);
  if (*err != cudaSuccess) return 0;
  const int pairs = std::min(clusters, std::min(sms / 2, kMaxCtas / 2));
  if (pairs <= 0) {
    *err = cudaErrorInvalidConfiguration;
    return 0;
  }
  cache[dev].store(pairs, std::memory_order_release);
  return pairs;
}

cudaError_t launch_extend_pair(const ExtendTcArgs& a, cudaStream_t s, bool dependent) {
  if (a.n_ctas <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * a.n_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = PairCfg::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, extend_pair_kernel, a);
  if (e != cudaSuccess) return e;
  return launch_extend_merge(a, s, dependent);
}

}  // namespace cpe
