// FP8 (E4M3) forward: O (bf16) and LSE from Q, K, V given as E4M3 with one
// descale factor per tensor, d_qk = d_v = 128.
//
// The pages define the fused attention in bf16; this is the adjacent
// precision of the same forward (TransformerEngine PR #3516 diagram: O and
// the softmax statistics).  Reading: the scores are the exact products of the
// E4M3 values, accumulated in fp32 and scaled by scale * descale_q *
// descale_k; P enters the P V product as E4M3(256 p) with p = exp(s - m)
// against the row's final maximum m (so p <= 1 and 256 p <= 256 < 448, the
// largest E4M3 value); the normaliser l sums the p before rounding; and
// O = descale_v * sum_j P8_j v_j / (256 l), LSE = m + ln l.
//
// Quantising P against the final maximum takes two passes over the key tiles
// of a query tile, the first for the row maximum only, so no O rescale (and
// no requantisation) ever happens.  Per work item (128 query rows of one
// head):
//
//   pass 1:  S(j) = Q K(j)^T        kind::f8f6f4, both operands K-major in smem
//            m    = max_j S         softmax warpgroup, one query row per thread
//   pass 2:  S(j) = Q K(j)^T
//            P8(j) = E4M3(256 exp2(S - m))   -> shared memory, K-major
//            O   += P8(j) V(j)      B = V(j)^T, K-major: a transposed copy of V
//                                   made once per call by vt_transpose_kernel
//
// Roles: warp 0 TMA producer, warp 1 MMA issuer, warps 4-7 softmax and
// epilogue.  S is double-buffered in tensor memory, so the tensor core works
// on S(j+1) while the softmax warps read S(j).
#include <cmath>

#include "attn_internal.cuh"

namespace attn {
namespace {
using namespace sm103;

constexpr float kLn2f = 0.6931471805599453f;
constexpr float kPScale = 256.f;  // P8 = E4M3(256 p)

struct F8Layout {
  static constexpr int kT = kTile * kTile;  // one 128 x 128 tile of one-byte elements
  static constexpr int kKStages = 3, kVStages = 2, kPStages = 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kT;
  static constexpr int kVOff = kKOff + kKStages * kT;
  static constexpr int kPOff = kVOff + kVStages * kT;
  static constexpr int kBarOff = kPOff + kPStages * kT;
  static constexpr int kBytes = kBarOff + 1024;  // barriers, then the item ring at +256
  static constexpr int kAlloc = kBytes + 1024;   // slack to align the window to 1 KB
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
  // above half of the SM's shared memory, so two CTAs (each taking all of
  // tensor memory) never share an SM
  static_assert(kAlloc > 114 * 1024, "one CTA per SM");
  static constexpr uint32_t kColS = 0;    // S buffers [0,128), [128,256)
  static constexpr uint32_t kColO = 256;  // O [256,384)
};

struct F8Bars {
  uint64_t q_full, q_empty, o_full, o_empty, drain;
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
};

// item = (query tile w = b * n_qt + t, head h), numbered w * Hq + h
struct F8Item {
  int b, t, h, kv_lo, n;
};

__device__ __forceinline__ F8Item f8_item(const KernelArgs& a, int idx) {
  F8Item it;
  const int w = idx / a.Hq;
  it.h = idx - w * a.Hq;
  it.b = w / a.n_qt;
  it.t = w - it.b * a.n_qt;
  const int2 r = a.q_tile_range[w];
  // Keys are the innermost coordinate of the V^T copies, which must start on
  // a 16-byte boundary: the item's key tiles start at the range's first key
  // rounded down to a multiple of 16 (the keys added in front are masked).
  it.kv_lo = r.x & ~15;
  it.n = (r.y > r.x) ? (r.y - it.kv_lo + kTile - 1) / kTile : 0;
  return it;
}

// Four E4M3 codes, rounded to nearest even and saturated to +-448, of four
// floats; the first lands in the lowest byte (the lowest address).
__device__ __forceinline__ uint32_t e4m3x4(float x0, float x1, float x2, float x3) {
  unsigned short lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// The 128 scores of this thread's row (one S buffer) in fp32, raw (before
// the scale): four loads, one wait.
__device__ __forceinline__ void load_row(uint32_t s_tm, uint32_t (&u)[4][32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) tmem_ld32x32b_x32(s_tm + q * 32, u[q]);
  tmem_ld_wait(u);
}

__global__ void __launch_bounds__(256, 1) fwd_fp8_kernel(const __grid_constant__ KernelArgs a) {
  using L = F8Layout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  F8Bars* bars = reinterpret_cast<F8Bars*>(sm + L::kBarOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kBarOff + sizeof(F8Bars));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  ItemRing* ring = reinterpret_cast<ItemRing*>(sm + L::kBarOff + 256);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = a.B * a.n_qt * a.Hq;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 128);
    mbar_init(&bars->drain, 1);
    for (int s = 0; s < L::kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_empty[s], 128);
      mbar_init(&bars->p_full[s], 128);
      mbar_init(&bars->p_empty[s], 1);
    }
    ring_init(ring, 1 + 128);  // MMA issuer + softmax warpgroup
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  grid_dep_wait();  // the metadata pass (the kernel before this one) has finished
  grid_dep_launch();
  const bool general = path_general(a);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Per item: Q once, then K(0..n-1) for the first pass and K(j), V(j)^T
    // for the second.
    if (lane == 0) {
      prefetch_tensormap(&a.tm_q);
      prefetch_tensormap(&a.tm_k);
      prefetch_tensormap(&a.tm_v);
      uint32_t it = 0, kc = 0, vc = 0;
      bool ok = true;
      for (uint32_t rn = 0;; ++rn) {
        int32_t idx;
        if (!ok || *abort_flag ||
            !(ok = ring_push(ring, rn, &a.hdr->next_item[0], n_items, idx, a.q_order, a.Hq)) ||
            idx < 0)
          break;
        const F8Item w = f8_item(a, idx);
        if (w.n == 0) continue;
        if (it > 0 && !(ok = mbar_wait(&bars->q_empty, (it - 1) & 1))) break;
        const int qrow = w.b * a.Sq + w.t * kTile;
        mbar_arrive_expect_tx(&bars->q_full, L::kT);
        if (ATTN_CHECK(a, tma_box_ok(0, kTile, a.d_qk, 1, w.h, a.Hq, qrow, kTile,
                                     (int64_t)a.B * a.Sq, false), 0x7901))
          tma_load_3d(sm + L::kQOff, &a.tm_q, &bars->q_full, 0, w.h, qrow);
        ++it;
        const int g = w.h / (a.Hq / a.Hkv);
        for (int t2 = 0; t2 < 2 * w.n && ok; ++t2) {
          const int j = t2 < w.n ? t2 : t2 - w.n;
          const int k0 = w.kv_lo + j * kTile;
          const int s = kc % L::kKStages;
          if (kc >= (uint32_t)L::kKStages &&
              !(ok = mbar_wait(&bars->k_empty[s], ((kc / L::kKStages) - 1) & 1)))
            break;
          mbar_arrive_expect_tx(&bars->k_full[s], L::kT);
          const int krow = w.b * a.Skv + k0;
          if (ATTN_CHECK(a, tma_box_ok(0, kTile, a.d_qk, 1, g, a.Hkv, krow, kTile,
                                       (int64_t)a.B * a.Skv, false), 0x7902))
            tma_load_3d(sm + L::kKOff + s * L::kT, &a.tm_k, &bars->k_full[s], 0, g, krow);
          ++kc;
          if (t2 >= w.n) {
            const int s2 = vc % L::kVStages;
            if (vc >= (uint32_t)L::kVStages &&
                !(ok = mbar_wait(&bars->v_empty[s2], ((vc / L::kVStages) - 1) & 1)))
              break;
            mbar_arrive_expect_tx(&bars->v_full[s2], L::kT);
            // V^T plane of (row b, KV head g): keys [k0, k0 + 128), every d
            const int plane = w.b * a.Hkv + g;
            if (ATTN_CHECK(a, tma_box_ok(k0, kTile, a.vt_pad, 1, 0, 1, plane, 1,
                                         (int64_t)a.B * a.Hkv, false), 0x7903))
              tma_load_3d(sm + L::kVOff + s2 * L::kT, &a.tm_v, &bars->v_full[s2], k0, 0, plane);
            ++vc;
          }
        }
      }
      if (!ok) {
        report_timeout(a, 0x910);
        *abort_flag = 1;
      }
      if (*abort_flag) {  // let copies in flight land before the CTA exits
        if (it > 0) mbar_wait(&bars->q_full, (it - 1) & 1, 100000000ull);
        for (uint32_t u = (kc > 3u ? kc - 3u : 0u); u < kc; ++u)
          mbar_wait(&bars->k_full[u % L::kKStages], (u / L::kKStages) & 1, 100000000ull);
        for (uint32_t u = (vc > 2u ? vc - 2u : 0u); u < vc; ++u)
          mbar_wait(&bars->v_full[u % L::kVStages], (u / L::kVStages) & 1, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // S of every tile of both passes in order, each into the S buffer its
    // reader freed two tiles earlier; in the second pass P(j) V(j) follows
    // S(j+1), so the tensor core has the next S while P(j) is formed.
    constexpr uint32_t idesc = idesc_f32acc(0 /* E4M3 */, 128, kTile, false, false);
    const uint32_t tm = warp_uniform(tmem);
    const uint64_t q_desc = sdesc_sw128(smem_u32(sm + L::kQOff), 16, 1024);
    const uint64_t k_desc = sdesc_sw128(smem_u32(sm + L::kKOff), 16, 1024);
    const uint64_t v_desc = sdesc_sw128(smem_u32(sm + L::kVOff), 16, 1024);
    const uint64_t p_desc = sdesc_sw128(smem_u32(sm + L::kPOff), 16, 1024);
    uint32_t T = 0, kc = 0, vc = 0, pc = 0, it = 0;
    bool ok = true;
    auto issue_s = [&]() -> bool {
      const int s = kc % L::kKStages, sb = T & 1;
      if (!mbar_wait_warp(&bars->k_full[s], (kc / L::kKStages) & 1)) return false;
      if (T >= 2 && !mbar_wait_warp(&bars->s_empty[sb], ((T >> 1) - 1) & 1)) return false;
      tc_fence_after();
      const uint64_t kd = k_desc + static_cast<uint32_t>((s * L::kT) >> 4);
      mma_f8_ss4_warp(tm + L::kColS + sb * kTile, q_desc, kd, idesc, 0u);
      mma_commit_warp(&bars->s_full[sb]);
      mma_commit_warp(&bars->k_empty[s]);
      ++kc;
      ++T;
      return true;
    };
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) ||
          !(ok = ring_pop_warp1(ring, rn, idx)) || idx < 0)
        break;
      const int n = warp_uniform(f8_item(a, idx).n);
      if (n == 0) continue;
      if (!(ok = mbar_wait_warp(&bars->q_full, it & 1))) break;
      if (!(ok = issue_s())) break;
      for (int t2 = 0; t2 < 2 * n && ok; ++t2) {
        if (t2 + 1 < 2 * n) {
          if (!(ok = issue_s())) break;
        } else {
          mma_commit_warp(&bars->q_empty);  // every S of this item is issued
        }
        if (t2 < n) continue;
        const int j = t2 - n, pb = pc & 1, s2 = vc % L::kVStages;
        if (!(ok = mbar_wait_warp(&bars->p_full[pb], (pc >> 1) & 1))) break;
        if (j == 0 && it > 0 && !(ok = mbar_wait_warp(&bars->o_empty, (it - 1) & 1))) break;
        if (!(ok = mbar_wait_warp(&bars->v_full[s2], (vc / L::kVStages) & 1))) break;
        tc_fence_after();
        const uint64_t pd = p_desc + static_cast<uint32_t>((pb * L::kT) >> 4);
        const uint64_t vd = v_desc + static_cast<uint32_t>((s2 * L::kT) >> 4);
        mma_f8_ss4_warp(tm + L::kColO, pd, vd, idesc, j > 0 ? 1u : 0u);
        mma_commit_warp(&bars->p_empty[pb]);
        mma_commit_warp(&bars->v_empty[s2]);
        ++pc;
        ++vc;
      }
      if (!ok) break;
      mma_commit_warp(&bars->o_full);  // O of this item is complete once these land
      ++it;
    }
    if (!ok && lane == 0) {
      report_timeout(a, 0x920);
      *abort_flag = 1;
    }
    mma_commit_warp(&bars->drain);
    mbar_wait(&bars->drain, 0, 200000000ull);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = tid - 128;  // TMEM lane = query row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t p_addr = smem_u32(sm + L::kPOff);
    uint32_t T = 0, pc = 0, it = 0;
    bool ok = true;
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) || !(ok = ring_pop(ring, rn, idx)) ||
          idx < 0)
        break;
      const F8Item w = f8_item(a, idx);
      const int i = w.t * kTile + r;
      const bool row_ok = i < a.Sq;
      const int64_t grow = (int64_t)w.b * a.Sq + i;
      bf16* orow = a.o + (grow * a.Hq + w.h) * kTile;
      float* lse_out = a.lse + ((int64_t)w.b * a.Hq + w.h) * a.Sq + i;
      if (w.n == 0) {
        if (row_ok && ATTN_CHECK(a, span_ok(orow - a.o, kTile, (int64_t)a.B * a.Sq * a.Hq * kTile) &&
                                        span_ok(lse_out - a.lse, 1, (int64_t)a.B * a.Hq * a.Sq),
                                 0x7904)) {
#pragma unroll
          for (int c = 0; c < kTile; c += 8)
            *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          *lse_out = -INFINITY;
        }
        continue;
      }
      int rlo = 0, rhi = 0, my_id = 0, my_pos = 0;
      if (row_ok) {
        if (!general) {
          const int2 kr = band_keys_of_query(a, i, a.seg_lo[grow], a.seg_hi[grow]);
          rlo = kr.x;
          rhi = kr.y;
        } else {
          my_id = a.q_id[grow];
          my_pos = a.q_pos[grow];
        }
      }
      auto valid = [&](int j, uint64_t (&vb)[2]) {
        kv_valid_bits(a, general, w.b, w.kv_lo + j * kTile, rlo, rhi, my_id, my_pos, vb);
        if (!row_ok) vb[0] = vb[1] = 0ull;
      };
      // pass 1: the row maximum of the raw scores over valid keys (the scale
      // is positive, so the maximum of the scaled scores is the scaled one)
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
      for (int j = 0; j < w.n; ++j) {
        uint64_t vb[2];
        valid(j, vb);
        const int sb = T & 1;
        if (!(ok = mbar_wait_warp(&bars->s_full[sb], (T >> 1) & 1))) break;
        tc_fence_after();
        uint32_t u[4][32];
        load_row(tmem + lane_base + L::kColS + sb * kTile, u);
        tc_fence_before();
        mbar_arrive(&bars->s_empty[sb]);
        ++T;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t m32 = static_cast<uint32_t>(vb[q >> 1] >> ((q & 1) * 32));
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float x0 = (m32 & (1u << e)) ? __uint_as_float(u[q][e]) : -INFINITY;
            const float x1 = (m32 & (2u << e)) ? __uint_as_float(u[q][e + 1]) : -INFINITY;
            mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], x0, x1);
          }
        }
      }
      if (!ok) break;
      const float mraw = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m = mraw * a.fp8_sc2;  // log2 units (-inf: no valid key)
      const float m_use = (m == -INFINITY) ? 0.f : m;
      // pass 2: P8 = E4M3(256 exp2(s - m)) into shared memory, l = sum of p
      float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      for (int j = 0; j < w.n; ++j) {
        uint64_t vb[2];
        valid(j, vb);
        const int sb = T & 1, pb = pc & 1;
        if (!(ok = mbar_wait_warp(&bars->s_full[sb], (T >> 1) & 1))) break;
        tc_fence_after();
        uint32_t u[4][32];
        load_row(tmem + lane_base + L::kColS + sb * kTile, u);
        tc_fence_before();
        mbar_arrive(&bars->s_empty[sb]);
        ++T;
        uint32_t pw[32];  // 128 E4M3 codes, key order
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t m32 = static_cast<uint32_t>(vb[q >> 1] >> ((q & 1) * 32));
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float p[4];
#pragma unroll
            for (int t = 0; t < 4; t += 2) {
              const float2 y = fma_f32x2(
                  make_float2(__uint_as_float(u[q][e + t]), __uint_as_float(u[q][e + t + 1])),
                  make_float2(a.fp8_sc2, a.fp8_sc2), make_float2(-m_use, -m_use));
              p[t] = (m32 & (1u << (e + t))) ? ex2_approx(y.x) : 0.f;
              p[t + 1] = (m32 & (2u << (e + t))) ? ex2_approx(y.y) : 0.f;
              rs[(e >> 2) & 1] = add_f32x2(rs[(e >> 2) & 1], make_float2(p[t], p[t + 1]));
            }
            pw[q * 8 + e / 4] = e4m3x4(p[0] * kPScale, p[1] * kPScale, p[2] * kPScale,
                                       p[3] * kPScale);
          }
        }
        // the stage's previous P (two tiles back) has been read by its P V
        if (pc >= 2 && !(ok = mbar_wait_warp(&bars->p_empty[pb], ((pc >> 1) - 1) & 1))) break;
        // row r of the K-major, 128-byte-swizzled P tile: 16-byte chunk c
        // (keys 16 c .. 16 c + 15) at chunk c ^ (r % 8)
        const uint32_t prow = p_addr + pb * L::kT + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(prow + ((c ^ (r & 7)) << 4), pw[4 * c], pw[4 * c + 1], pw[4 * c + 2],
                       pw[4 * c + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[pb]);
        ++pc;
      }
      if (!ok) break;
      const float l = (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
      // epilogue: O = descale_v * acc / (256 l), LSE = m + log2 l (natural log out)
      if (!(ok = mbar_wait_warp(&bars->o_full, it & 1))) break;
      tc_fence_after();
      const float inv = (l > 0.f) ? a.fp8_dv / (kPScale * l) : 0.f;
      const bool store = row_ok && ATTN_CHECK(a, span_ok(orow - a.o, kTile,
                                                         (int64_t)a.B * a.Sq * a.Hq * kTile),
                                              0x7905);
#pragma unroll
      for (int q = 0; q < kTile / 32; ++q) {
        uint32_t o[32];
        tmem_ld32x32b_x32(tmem + lane_base + L::kColO + q * 32, o);
        tmem_ld_wait(o);
        if (store) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[c + 0]) * inv, __uint_as_float(o[c + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + q * 32 + c) = v;
          }
        }
      }
      if (row_ok && ATTN_CHECK(a, span_ok(lse_out - a.lse, 1, (int64_t)a.B * a.Hq * a.Sq), 0x7906))
        *lse_out = (l > 0.f) ? (m + __log2f(l)) * kLn2f : -INFINITY;
      if (a.max_logit && ATTN_CHECK(a, span_ok((int64_t)w.b * a.Hq + w.h, 1, (int64_t)a.B * a.Hq),
                                    0x7907))
        warp_max_logit(a.max_logit + (int64_t)w.b * a.Hq + w.h, m);
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
      ++it;
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x930 + (warp & 3));
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// V^T for the second pass: plane (b, g) of the workspace holds, for each of
// the 128 value dims d, the keys [0, vt_pad) of batch row b and KV head g
// (zero beyond Skv), so that V(j)^T is a K-major 128 x 128 tile.  One block
// per (128-key tile, plane): 16 KB in, transposed through shared memory, 16 KB out.
__global__ void __launch_bounds__(256) vt_transpose_kernel(const KernelArgs a) {
  __shared__ uint8_t tile[kTile][kTile + 4];
  const int k0 = blockIdx.x * kTile, plane = blockIdx.y;
  const int b = plane / a.Hkv, g = plane - b * a.Hkv;
  for (int v = threadIdx.x; v < kTile * 8; v += blockDim.x) {
    const int kk = v >> 3, c = v & 7;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (k0 + kk < a.Skv)
      x = ld_nc_v4(a.vt_src + ((int64_t)b * a.Skv + k0 + kk) * a.vt_src_stride + (int64_t)g * kTile +
                   c * 16);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 16; ++e) tile[kk][c * 16 + e] = static_cast<uint8_t>(w[e >> 2] >> ((e & 3) * 8));
  }
  __syncthreads();
  for (int v = threadIdx.x; v < kTile * 8; v += blockDim.x) {
    const int d = v >> 3, c = v & 7;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < 16; ++e) w[e >> 2] |= static_cast<uint32_t>(tile[c * 16 + e][d]) << ((e & 3) * 8);
    const int64_t off = ((int64_t)plane * kTile + d) * a.vt_pad + k0 + c * 16;
    if (ATTN_CHECK(a, span_ok(off, 16, (int64_t)a.B * a.Hkv * kTile * a.vt_pad), 0x7908))
      *reinterpret_cast<uint4*>(a.vt + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_vt_transpose(const KernelArgs& a, cudaStream_t st) {
  const dim3 grid(a.vt_pad / kTile, a.B * a.Hkv);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  vt_transpose_kernel<<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const KernelArgs& a, int nsm, cudaStream_t st) {
  using L = F8Layout;
  cudaError_t e =
      cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int items = a.B * a.n_qt * a.Hq;
  const int grid = items < nsm ? items : nsm;
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(fwd_fp8_kernel, dim3(grid), dim3(256), L::kAlloc, st, a);
}

}  // namespace attn
