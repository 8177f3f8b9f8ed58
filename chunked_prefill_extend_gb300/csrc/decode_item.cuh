// Split-KV decode attention for one (split, decode sequence, KV head) item,
// HBM-bound; shared by the stand-alone decode kernel (one item per CTA) and
// the decode workers of the fused mixed-step launch (one item per warpgroup).
//
// The G query heads that share the KV head form the rows of an m16n8k16 tile
// (rows >= G are zero), so each K/V byte read from HBM serves all G heads.
// The split's pages are dealt round robin to the item's four warps; each warp
// streams its pages through a two-stage cp.async ring (16-byte vectors, one
// page = 16 keys = 16 x d bf16 rows of K and of V, padded rows so ldmatrix is
// bank-conflict free) and keeps its own running (m, l, O).  The four warps are
// merged through shared memory with the online-softmax LSE rule; with one
// split that is the answer, otherwise the split's normalised partial
// (o, m, l) goes to the workspace and a merge kernel combines the splits by
// the same rule.
#pragma once

#include "cpe_device.cuh"
#include "kernels.h"

namespace cpe {

namespace {

// Barrier over the 128 threads (four warps) of one item; id 0 with a
// 128-thread CTA is the CTA barrier.
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

constexpr int kWarps = 4;
constexpr int kStagesDec = 2;

template <int D>
struct DecCfg {
  static constexpr int kRowBytes = D * 2 + 16;          // padded K/V row in shared memory
  static constexpr int kPageBytes = kPage * kRowBytes;  // one page of K (or of V)
  static constexpr int kWarpBytes = kStagesDec * 2 * kPageBytes;
  static constexpr int kSmem = kWarps * kWarpBytes;
  static constexpr int kChunks = D * 2 / 16;            // 16-byte vectors per row
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct DecodeSeq {
  int row;   // query row in q / out
  int L;     // keys [0, L)
  bool ok;
};

__device__ __forceinline__ DecodeSeq decode_seq(const DecodeArgs& a, int s, bool record) {
  DecodeSeq r;
  r.row = a.qo_indptr ? a.qo_indptr[s] : s;
  r.L = a.prefix_len[s] + 1;
  r.ok = true;
  if (a.qo_indptr && a.qo_indptr[s + 1] - r.row != 1) {
    if (record) record_error(a.status, kStatusDeviceArg, kDetailBadDecodeLen);
    r.ok = false;
  } else if (r.L < 1 || r.L > a.max_kv_len || (r.L + kPage - 1) / kPage > a.max_pages) {
    if (record) record_error(a.status, kStatusDeviceArg, kDetailBadLength);
    r.ok = false;
  }
  return r;
}

// One decode item: split sp of decode sequence sidx for KV head g, computed by
// 128 threads (tid 0..127, four whole warps) with C::kSmem bytes of shared
// memory at dsm; `bar` names the 128-thread barrier the item synchronises on.
template <int D>
__device__ __forceinline__ void decode_item(const DecodeArgs& a, int sp, int sidx, int g, uint8_t* dsm, int tid,
                                            int bar) {
  using C = DecCfg<D>;
  const int s = a.seq_begin + sidx;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const DecodeSeq dq = decode_seq(a, s, sp == 0 && g == 0 && tid == 0);
  if (!dq.ok) return;
  const int ns = (dq.L + kDecodeSplit - 1) / kDecodeSplit;
  if (sp >= ns) return;
  const int G = a.h_q / a.h_kv;
  const int kbeg = sp * kDecodeSplit;
  const int kend = min(dq.L, kbeg + kDecodeSplit);
  const int pbeg = kbeg / kPage;
  const int pend = (kend + kPage - 1) / kPage;
  const int grp = lane >> 2;
  const int tq = lane & 3;
  const float sl2 = a.scale_log2;

  // Q fragments: rows = heads g*G .. g*G+G-1 of this query row, zero beyond G.
  uint32_t qa[D / 16][4];
  {
    const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
    const int64_t base = (static_cast<int64_t>(dq.row) * a.h_q + g * G) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int c0 = ks * 16 + 2 * tq;
      qa[ks][0] = grp < G ? q32[(base + grp * D + c0) >> 1] : 0u;
      qa[ks][1] = grp + 8 < G ? q32[(base + (grp + 8) * D + c0) >> 1] : 0u;
      qa[ks][2] = grp < G ? q32[(base + grp * D + c0 + 8) >> 1] : 0u;
      qa[ks][3] = grp + 8 < G ? q32[(base + (grp + 8) * D + c0 + 8) >> 1] : 0u;
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  uint8_t* wsm = dsm + warp * C::kWarpBytes;
  const int32_t* pt = a.page_table + static_cast<int64_t>(s) * a.max_pages;
  const uint8_t* kc = static_cast<const uint8_t*>(a.k_cache);
  const uint8_t* vc = static_cast<const uint8_t*>(a.v_cache);
  const int64_t tok_stride = static_cast<int64_t>(a.h_kv) * D * 2;  // bytes between tokens

  auto load_page = [&](int pi, int stg) {
    int pid = pt[pi];
    if (pid < 0 || pid >= a.num_pages) {
      if (lane == 0) record_error(a.status, kStatusDeviceArg, kDetailBadPage);
      pid = 0;
    }
    const int64_t src = (static_cast<int64_t>(pid) * kPage * a.h_kv + g) * D * 2;
    uint8_t* sk = wsm + stg * 2 * C::kPageBytes;
    uint8_t* sv = sk + C::kPageBytes;
#pragma unroll
    for (int c = lane; c < kPage * C::kChunks; c += 32) {
      const int r = c / C::kChunks;
      const int ch = c % C::kChunks;
      cp_async16(sk + r * C::kRowBytes + ch * 16, kc + src + r * tok_stride + ch * 16);
      cp_async16(sv + r * C::kRowBytes + ch * 16, vc + src + r * tok_stride + ch * 16);
    }
  };

  const int n_my = (pend - pbeg - warp + kWarps - 1) / kWarps;  // pages of this warp
  if (n_my > 0) load_page(pbeg + warp, 0);
  cp_async_commit();
  for (int k = 0; k < n_my; ++k) {
    if (k + 1 < n_my) load_page(pbeg + warp + (k + 1) * kWarps, (k + 1) % kStagesDec);
    cp_async_commit();
    cp_async_wait1();
    __syncwarp();
    const int pi = pbeg + warp + k * kWarps;
    const uint32_t sk = smem_u32(wsm + (k % kStagesDec) * 2 * C::kPageBytes);
    const uint32_t sv = sk + C::kPageBytes;

    // S = Q K^T for the page's 16 keys (two n-tiles of 8 keys)
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, rr = lane & 7;
      const uint32_t rowaddr = sk + ((mi >> 1) * 8 + rr) * C::kRowBytes + (mi & 1) * 16;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(rowaddr + ks * 32, b0, b1, b2, b3);
        mma_bf16(sc[0], qa[ks], b0, b1);
        mma_bf16(sc[1], qa[ks], b2, b3);
      }
    }
    // mask keys past the end, online softmax per row (rows grp and grp+8)
    const int key0 = pi * kPage;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (key0 + nt * 8 + 2 * tq + (e & 1) >= kend) sc[nt][e] = -INFINITY;
    float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0 * sl2);
    const float mn1 = fmaxf(m1, mx1 * sl2);
    const float f0 = fast_exp2(m0 - mn0);
    const float f1 = fast_exp2(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float p[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      p[nt][0] = fast_exp2(fmaf(sc[nt][0], sl2, -mn0));
      p[nt][1] = fast_exp2(fmaf(sc[nt][1], sl2, -mn0));
      p[nt][2] = fast_exp2(fmaf(sc[nt][2], sl2, -mn1));
      p[nt][3] = fast_exp2(fmaf(sc[nt][3], sl2, -mn1));
    }
    l0 = l0 * f0 + p[0][0] + p[0][1] + p[1][0] + p[1][1];
    l1 = l1 * f1 + p[0][2] + p[0][3] + p[1][2] + p[1][3];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= f0;
      o[n][1] *= f0;
      o[n][2] *= f1;
      o[n][3] *= f1;
    }
    const uint32_t pa[4] = {pack_bf16x2(p[0][0], p[0][1]), pack_bf16x2(p[0][2], p[0][3]),
                            pack_bf16x2(p[1][0], p[1][1]), pack_bf16x2(p[1][2], p[1][3])};
    // O += P V: V rows are keys, read transposed
    {
      const int mi = lane >> 3, rr = lane & 7;
      const uint32_t rowaddr = sv + ((mi & 1) * 8 + rr) * C::kRowBytes + (mi >> 1) * 16;
#pragma unroll
      for (int n2 = 0; n2 < D / 16; ++n2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(rowaddr + n2 * 32, b0, b1, b2, b3);
        mma_bf16(o[2 * n2], pa, b0, b1);
        mma_bf16(o[2 * n2 + 1], pa, b2, b3);
      }
    }
    __syncwarp();
  }
  // full row sums (the quad of lanes sharing a row)
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // merge the four warps through shared memory (reusing the page ring)
  asm volatile("cp.async.wait_all;" ::: "memory");
  group_sync(bar);
  float* sm_o = reinterpret_cast<float*>(dsm);          // [warps][16][D]
  float* sm_ml = sm_o + kWarps * 16 * D;                // [warps][16][2]
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int c = n * 8 + 2 * tq;
    sm_o[(warp * 16 + grp) * D + c] = o[n][0];
    sm_o[(warp * 16 + grp) * D + c + 1] = o[n][1];
    sm_o[(warp * 16 + grp + 8) * D + c] = o[n][2];
    sm_o[(warp * 16 + grp + 8) * D + c + 1] = o[n][3];
  }
  if (tq == 0) {
    sm_ml[(warp * 16 + grp) * 2] = m0;
    sm_ml[(warp * 16 + grp) * 2 + 1] = l0;
    sm_ml[(warp * 16 + grp + 8) * 2] = m1;
    sm_ml[(warp * 16 + grp + 8) * 2 + 1] = l1;
  }
  group_sync(bar);
  for (int e = tid; e < G * D; e += 128) {
    const int r = e / D;
    const int c = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_ml[(w * 16 + r) * 2]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = sm_ml[(w * 16 + r) * 2];
      const float wt = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
      num += wt * sm_o[(w * 16 + r) * D + c];
      den += wt * sm_ml[(w * 16 + r) * 2 + 1];
    }
    const int head = g * G + r;
    if (ns == 1) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
      out[(static_cast<int64_t>(dq.row) * a.h_q + head) * D + c] = __float2bfloat16_rn(num / den);
      if (c == 0 && a.lse) a.lse[static_cast<int64_t>(dq.row) * a.h_q + head] = (M + __log2f(den)) * 0.69314718055994531f;
    } else {
      const int64_t pidx = (static_cast<int64_t>(sidx) * a.h_q + head) * a.max_splits + sp;
      a.part_o[pidx * D + c] = num / den;
      if (c == 0) {
        a.part_ml[pidx * 2] = M;
        a.part_ml[pidx * 2 + 1] = den;
      }
    }
  }
}

}  // namespace

}  // namespace cpe
