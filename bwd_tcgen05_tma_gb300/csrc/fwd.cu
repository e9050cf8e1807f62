// Forward pass: O = softmax(scale * Q K^T + bias, masked) V and LSE, per
// 128-row query tile of one (batch row, query head).
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: Q tile once per work item, K/V tiles through a
//               ring of shared-memory stages;
//   warp 1      allocates tensor memory; lane 0 issues the tcgen05 MMAs
//               S = Q K^T (into one of two TMEM S buffers) and O += P V
//               (O accumulates in TMEM);
//   warps 4-7   softmax warpgroup: thread r owns query row r (TMEM lane r):
//               reads S, applies scale/bias/mask, keeps the running max and
//               sum, writes bf16 P to shared memory, and at the end scales O
//               by 1/l and stores O and LSE.
// S(j+1) is issued before P(j) V(j), so the tensor core works on the next
// score tile while the softmax warps exponentiate the current one.  O is only
// rescaled when the running max grows by more than 2^8 (in log2 units); below
// that the stale max is kept for both P and l, which leaves O / l exact.
//
// Outputs and semantics: TransformerEngine PR #3516 diagram (fused-attention
// forward feeding the backward with O and the softmax statistics); rows with
// no valid key get O = 0, LSE = -inf.
#include <cmath>

#include "attn_internal.cuh"

namespace attn {
namespace {
using namespace sm103;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

template <int DQK, int DV>
struct FwdLayout {
  static constexpr int kQBytes = kTile * DQK * 2;
  static constexpr int kKBytes = kTile * DQK * 2;
  static constexpr int kVBytes = kTile * DV * 2;
  static constexpr int kPBytes = kTile * kTile * 2;
  // K and V have separate rings: K(j) is free once S(j) is done, V(j) once P(j) V(j) is.
  static constexpr int kKStages = 2;
  static constexpr int kVStages = (kQBytes + 2 * kKBytes + 2 * kVBytes + kPBytes <= 210 * 1024) ? 2 : 1;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + kKStages * kKBytes;
  // two P buffers where they fit: P(j) is written while P(j-1) V(j-1) runs
  static constexpr int kPStages =
      (kQBytes + kKStages * kKBytes + kVStages * kVBytes + 2 * kPBytes <= 224 * 1024) ? 2 : 1;
  static constexpr int kPOff = kVOff + kVStages * kVBytes;
  static constexpr int kBarOff = kPOff + kPStages * kPBytes;
  static constexpr int kBytes = kBarOff + 512;  // barriers, then the item ring at +256
  // at least ~116 KB so two CTAs never share an SM (each allocates all of TMEM)
  static constexpr int kAlloc = (kBytes + 1024 > 118 * 1024) ? kBytes + 1024 : 118 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // two S buffers: [0,128) and [128,256)
  static constexpr uint32_t kColO = 256;  // O: [256, 256+DV)
};

struct Bars {
  uint64_t q_full, q_empty, pv_done, o_full, o_empty, drain;
  // per P buffer: with two, warps that finish step j+1 early must not count
  // toward step j
  uint64_t p_full[2];
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], s_empty[2];
};

struct FwdItem {
  int b, t, h, kv_lo, kv_hi, n;
};

__device__ __forceinline__ FwdItem fwd_item(const KernelArgs& a, int idx) {
  const int per_t = a.B * a.Hq;
  const int t_rev = idx / per_t, rem = idx - t_rev * per_t;
  FwdItem it;
  it.t = a.n_qt - 1 - t_rev;  // longest causal rows first
  it.b = rem / a.Hq;
  it.h = rem - it.b * a.Hq;
  const int2 r = a.q_tile_range[it.b * a.n_qt + it.t];
  it.kv_lo = r.x;
  it.kv_hi = r.y;
  it.n = (r.y > r.x) ? (r.y - r.x + kTile - 1) / kTile : 0;
  return it;
}

template <class E, int DQK, int DV, bool HAS_BIAS>
__global__ void __launch_bounds__(256, 1) fwd_kernel(const __grid_constant__ KernelArgs a) {
  using L = FwdLayout<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(sm + L::kBarOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kBarOff + sizeof(Bars));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  ItemRing* ring = reinterpret_cast<ItemRing*>(sm + L::kBarOff + 256);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = a.B * a.n_qt * a.Hq;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->p_full[0], 128);
    mbar_init(&bars->p_full[1], 128);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 128);
    mbar_init(&bars->drain, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_empty[s], 128);
    }
    ring_init(ring, 1 + 128);  // MMA issuer + softmax warpgroup
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  grid_dep_wait();  // the previous kernel on the stream has finished
  grid_dep_launch();
  const bool general = path_general(a);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&a.tm_q);
      prefetch_tensormap(&a.tm_k);
      prefetch_tensormap(&a.tm_v);
      uint32_t kt = 0, it = 0, q_loads = 0, k_loads = 0;
      bool ok = true;
      for (uint32_t rn = 0;; ++rn) {
        int32_t idx;
        if (!ok || *abort_flag || !(ok = ring_push(ring, rn, &a.hdr->next_item[0], n_items, idx)) ||
            idx < 0)
          break;
        const FwdItem w = fwd_item(a, idx);
        if (w.n == 0) continue;
        if (it > 0 && !(ok = mbar_wait(&bars->q_empty, (it - 1) & 1))) break;
        ++q_loads;
        mbar_arrive_expect_tx(&bars->q_full, L::kQBytes);
        const int qrow = w.b * a.Sq + w.t * kTile;
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c)
          if (ATTN_CHECK(a, box_ok(a, &a.tm_q, c * 64, w.h, qrow, kTile), 0x7001))
            tma_load_3d(sm + L::kQOff + c * 16384, &a.tm_q, &bars->q_full, c * 64, w.h, qrow);
        const int g = w.h / (a.Hq / a.Hkv);
        for (int j = 0; j < w.n; ++j, ++kt) {
          const int krow = w.b * a.Skv + w.kv_lo + j * kTile;
          const int ks = kt % L::kKStages, vs = kt % L::kVStages;
          if (kt >= (uint32_t)L::kKStages &&
              !(ok = mbar_wait(&bars->k_empty[ks], ((kt / L::kKStages) - 1) & 1)))
            break;
          uint8_t* kst = sm + L::kKOff + ks * L::kKBytes;
          mbar_arrive_expect_tx(&bars->k_full[ks], L::kKBytes);
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c)
            if (ATTN_CHECK(a, box_ok(a, &a.tm_k, c * 64, g, krow, kTile), 0x7002))
              tma_load_3d(kst + c * 16384, &a.tm_k, &bars->k_full[ks], c * 64, g, krow);
          ++k_loads;
          if (kt >= (uint32_t)L::kVStages &&
              !(ok = mbar_wait(&bars->v_empty[vs], ((kt / L::kVStages) - 1) & 1)))
            break;
          uint8_t* vst = sm + L::kVOff + vs * L::kVBytes;
          mbar_arrive_expect_tx(&bars->v_full[vs], L::kVBytes);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            if (ATTN_CHECK(a, box_ok(a, &a.tm_v, c * 64, g, krow, kTile), 0x7003))
              tma_load_3d(vst + c * 16384, &a.tm_v, &bars->v_full[vs], c * 64, g, krow);
        }
        if (!ok) break;
        ++it;
      }
      if (!ok) {
        report_timeout(a, 0x10);
        *abort_flag = 1;
      }
      // let every copy this thread issued land before the CTA can exit
      if (*abort_flag) {
        if (q_loads > 0) mbar_wait(&bars->q_full, (q_loads - 1) & 1, 100000000ull);
        for (uint32_t u = (k_loads > 2u ? k_loads - 2u : 0u); u < k_loads; ++u)
          mbar_wait(&bars->k_full[u % L::kKStages], (u / L::kKStages) & 1, 100000000ull);
        for (uint32_t u = (kt > 2u ? kt - 2u : 0u); u < kt; ++u)
          mbar_wait(&bars->v_full[u % L::kVStages], (u / L::kVStages) & 1, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop on warp-uniform values; one elected lane
    // issues each GEMM's MMAs from a single asm statement.
    constexpr uint32_t idesc_s = idesc_f32acc(E::kMmaFmt, 128, kTile, false, false);
    constexpr uint32_t idesc_o = idesc_f32acc(E::kMmaFmt, 128, DV, false, true);
    const uint32_t tm = warp_uniform(tmem);
    // operand descriptors are built once; each GEMM only adds a stage offset
    const uint64_t q_desc = sdesc_sw128(smem_u32(sm + L::kQOff), 16, 1024);
    const uint64_t p_desc = sdesc_sw128(smem_u32(sm + L::kPOff), 16, 1024);
    const uint64_t k_desc0 = sdesc_sw128(smem_u32(sm + L::kKOff), 16, 1024);
    const uint64_t v_desc0 = sdesc_sw128(smem_u32(sm + L::kVOff), 16384, 1024);
    uint32_t kt = 0, it = 0;
    bool ok = true;
    auto issue_s = [&](uint32_t k) -> bool {
      const int s = k % L::kKStages, sb = k & 1;
      if (!mbar_wait_warp(&bars->k_full[s], (k / L::kKStages) & 1)) return false;
      if (k >= 2 && !mbar_wait_warp(&bars->s_empty[sb], ((k >> 1) - 1) & 1)) return false;
      tc_fence_after();
      const uint64_t kd = k_desc0 + static_cast<uint64_t>((s * L::kKBytes) >> 4);
      mma_ss_warp<DQK / 16, 4, 2, 1018, 2, 1018>(tm + L::kColS + sb * kTile, q_desc, kd, idesc_s,
                                                 0u);
      mma_commit_warp(&bars->s_full[sb]);
      mma_commit_warp(&bars->k_empty[s]);
      return true;
    };
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) ||
          !(ok = ring_pop_warp1(ring, rn, idx)) || idx < 0)
        break;
      const FwdItem w = fwd_item(a, idx);
      const int n = warp_uniform(w.n);
      if (n == 0) continue;
      if (!(ok = mbar_wait_warp(&bars->q_full, it & 1))) break;
      if (!(ok = issue_s(kt))) break;
      for (int j = 0; j < n; ++j) {
        const uint32_t k = kt + j;
        if (j + 1 < n) {
          if (!(ok = issue_s(k + 1))) break;
        } else {
          mma_commit_warp(&bars->q_empty);  // every S MMA of this item has been issued
        }
        if (!(ok = mbar_wait_warp(&bars->p_full[k & 1], (k >> 1) & 1))) break;
        if (j == 0 && it > 0 && !(ok = mbar_wait_warp(&bars->o_empty, (it - 1) & 1))) break;
        const int s = k % L::kVStages;
        if (!(ok = mbar_wait_warp(&bars->v_full[s], (k / L::kVStages) & 1))) break;
        tc_fence_after();
        const uint64_t vd = v_desc0 + static_cast<uint64_t>((s * L::kVBytes) >> 4);
        const uint64_t pd = p_desc + static_cast<uint32_t>(((k % L::kPStages) * L::kPBytes) >> 4);
        // O += P V: A = P (shared memory, K-major), B = V MN-major
        mma_ss_warp<kTile / 16, 4, 2, 1018, 128, 128>(tm + L::kColO, pd, vd, idesc_o,
                                                      j > 0 ? 1u : 0u);
        mma_commit_warp(&bars->pv_done);
        mma_commit_warp(&bars->v_empty[s]);
      }
      if (!ok) break;
      mma_commit_warp(&bars->o_full);  // O of this item complete once these land
      kt += n;
      ++it;
    }
    if (!ok && lane == 0) {
      report_timeout(a, 0x20);
      *abort_flag = 1;
    }
    mma_commit_warp(&bars->drain);
    mbar_wait(&bars->drain, 0, 200000000ull);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int r = tid - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t p_addr = smem_u32(sm + L::kPOff);
    uint32_t kt = 0, it_sm = 0;  // it_sm: items with work, as the MMA issuer counts them
    bool ok = true;
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) || !(ok = ring_pop(ring, rn, idx)) ||
          idx < 0)
        break;
      const FwdItem w = fwd_item(a, idx);
      const int i = w.t * kTile + r;
      const bool row_ok = i < a.Sq;
      const int64_t grow = (int64_t)w.b * a.Sq + i;
      bf16* orow = a.o + (grow * a.Hq + w.h) * DV;
      float* lse_out = a.lse + ((int64_t)w.b * a.Hq + w.h) * a.Sq + i;
      if (w.n == 0) {
        if (row_ok && ATTN_CHECK(a, span_ok(orow - a.o, DV, (int64_t)a.B * a.Sq * a.Hq * DV) &&
                                        span_ok(lse_out - a.lse, 1, (int64_t)a.B * a.Hq * a.Sq),
                                 0x7004)) {
#pragma unroll
          for (int c = 0; c < DV; c += 8)
            *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          *lse_out = a.sink ? a.sink[w.h] : -INFINITY;  // only the sink, if any
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
      const bf16* bias_row = nullptr;
      if (HAS_BIAS && row_ok) {
        const int bb = a.bias_b > 1 ? w.b : 0, bh = a.bias_h > 1 ? w.h : 0;
        bias_row = a.bias + (((int64_t)bb * a.bias_h + bh) * a.Sq + i) * a.Skv;
      }
      float m_ref = -INFINITY, l = 0.f;
      float row_max = -INFINITY;  // exact row max of the scaled logits (log2 units)
      for (int j = 0; j < w.n; ++j) {
        const uint32_t k = kt + j;
        const int sb = k & 1;
        const int k0 = w.kv_lo + j * kTile;
        float x[kTile];
        // the next key tile's bias row segment toward L2 while this one runs
        if (HAS_BIAS && row_ok && j + 1 < w.n)
          prefetch_bias_lines(a, (bias_row - a.bias) + k0 + kTile, min(kTile, a.Skv - k0 - kTile));
        if (!(ok = mbar_wait_warp(&bars->s_full[sb], (k >> 1) & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < kTile / 32; ++q) {
          uint32_t u[32];
          tmem_ld32x32b_x32(tmem + lane_base + L::kColS + sb * kTile + q * 32, u);
          tmem_ld_wait(u);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 y = mul_f32x2(make_float2(__uint_as_float(u[e]), __uint_as_float(u[e + 1])),
                                       make_float2(a.scale_log2, a.scale_log2));
            x[q * 32 + e] = y.x;
            x[q * 32 + e + 1] = y.y;
          }
        }
        tc_fence_before();
        mbar_arrive(&bars->s_empty[sb]);
        if (HAS_BIAS && row_ok) add_bias_row<E>(x, bias_row + k0, min(kTile, a.Skv - k0));
        // mask (branch-free: a validity bitmask per row and tile)
        uint64_t vb[2];
        kv_valid_bits(a, general, w.b, k0, rlo, rhi, my_id, my_pos, vb);
        // 32-column chunks valid for every row of the warp skip the selects
        // (a separate loop per case keeps both free of per-element branches)
#pragma unroll
        for (int q = 0; q < kTile / 32; ++q) {
          const uint32_t m32 = static_cast<uint32_t>(vb[q >> 1] >> ((q & 1) * 32));
          if (!__all_sync(0xffffffffu, m32 == 0xffffffffu)) {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[q * 32 + e] = (m32 & (1u << e)) ? x[q * 32 + e] : -INFINITY;
          }
        }
        float mx8[8];  // independent max chains
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = x[e];
#pragma unroll
        for (int c = 8; c < kTile; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], x[c], x[c + 1]);
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        row_max = fmaxf(row_max, mx);
        const float m_new = fmaxf(m_ref, mx);
        const bool grow_max = m_new > m_ref + kRescaleThreshold;
        const bool rescale = grow_max && j > 0 && m_ref > -INFINITY;
        // P(j-1) V(j-1) must be finished before O is rescaled or, with one P
        // buffer, before P(j) overwrites P(j-1).  (With two buffers P(j-2) V is
        // already done: S(j) was issued after it.)
        if (j > 0 && (L::kPStages == 1 || __any_sync(0xffffffffu, rescale))) {
          if (!(ok = mbar_wait_warp(&bars->pv_done, (k - 1) & 1))) break;
          tc_fence_after();
        }
        // tensor-memory loads/stores are warp-wide: every lane takes part and
        // the rows that keep their max scale by 1
        if (__any_sync(0xffffffffu, rescale)) {
          const float f = rescale ? ex2_approx(m_ref - m_new) : 1.f;
          l *= f;
#pragma unroll
          for (int q = 0; q < DV / 32; ++q) {
            uint32_t u[32];
            const uint32_t ta = tmem + lane_base + L::kColO + q * 32;
            tmem_ld32x32b_x32(ta, u);
            tmem_ld_wait(u);
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * f);
            tmem_st32x32b_x32(ta, u);
          }
          tmem_st_wait();
        }
        if (grow_max) m_ref = m_new;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // two columns per instruction: x - m, and two pairs of running sums
        float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < kTile; c += 2) {
          const float2 y = sub_f32x2(make_float2(x[c], x[c + 1]), make_float2(m_use, m_use));
          x[c] = ex2_approx(y.x);
          x[c + 1] = ex2_approx(y.y);
          rs[(c >> 1) & 1] = add_f32x2(rs[(c >> 1) & 1], make_float2(x[c], x[c + 1]));
        }
        l += (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
        // P row r -> shared memory, K-major with the 128-byte swizzle
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float* p8 = x + cc * 64 + u * 8;
            st_shared_v4(p_addr + (k % L::kPStages) * L::kPBytes + cc * 16384 + r * 128 + ((u ^ (r & 7)) << 4),
                         E::pack(p8[0], p8[1]), E::pack(p8[2], p8[3]),
                         E::pack(p8[4], p8[5]), E::pack(p8[6], p8[7]));
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[k & 1]);
      }
      if (!ok) break;
      // epilogue: O / l and LSE
      if (!(ok = mbar_wait_warp(&bars->o_full, it_sm & 1))) break;
      tc_fence_after();
      // the sink logit, if any, joins the normaliser (it has no value vector)
      float l_fin = l, m_fin = m_ref, o_scale = 1.f;
      if (a.sink) {
        const float s2 = a.sink[w.h] * kLog2e;
        if (s2 > -INFINITY) {
          m_fin = fmaxf(m_ref, s2);
          o_scale = ex2_approx(m_ref - m_fin);  // 0 for a row without valid keys
          l_fin = l * o_scale + ex2_approx(s2 - m_fin);
        }
      }
      const float inv_l = (l_fin > 0.f) ? o_scale / l_fin : 0.f;
#pragma unroll
      for (int q = 0; q < DV / 32; ++q) {
        uint32_t u[32];
        tmem_ld32x32b_x32(tmem + lane_base + L::kColO + q * 32, u);
        tmem_ld_wait(u);
        if (row_ok && ATTN_CHECK(a, span_ok(orow + q * 32 - a.o, 32, (int64_t)a.B * a.Sq * a.Hq * DV),
                                 0x7005)) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 v;
            v.x = E::pack(__uint_as_float(u[c + 0]) * inv_l, __uint_as_float(u[c + 1]) * inv_l);
            v.y = E::pack(__uint_as_float(u[c + 2]) * inv_l, __uint_as_float(u[c + 3]) * inv_l);
            v.z = E::pack(__uint_as_float(u[c + 4]) * inv_l, __uint_as_float(u[c + 5]) * inv_l);
            v.w = E::pack(__uint_as_float(u[c + 6]) * inv_l, __uint_as_float(u[c + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + q * 32 + c) = v;
          }
        }
      }
      if (row_ok && ATTN_CHECK(a, span_ok(lse_out - a.lse, 1, (int64_t)a.B * a.Hq * a.Sq), 0x7006))
        *lse_out = (l_fin > 0.f) ? (m_fin + __log2f(l_fin)) * kLn2 : -INFINITY;
      if (a.max_logit && ATTN_CHECK(a, span_ok((int64_t)w.b * a.Hq + w.h, 1, (int64_t)a.B * a.Hq), 0x7007))
        warp_max_logit(a.max_logit + (int64_t)w.b * a.Hq + w.h, row_max);
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
      kt += w.n;
      ++it_sm;
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x30 + (warp & 3));
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <class E, int DQK, int DV, bool HB>
cudaError_t launch_fwd_t(const KernelArgs& a, int num_sms, cudaStream_t st) {
  using L = FwdLayout<DQK, DV>;
  auto kern = fwd_kernel<E, DQK, DV, HB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_items = a.B * a.n_qt * a.Hq;
  const int grid = n_items < num_sms ? n_items : num_sms;
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(kern, dim3(grid), dim3(256), L::kAlloc, st, a);
}

template <int DQK, int DV>
cudaError_t launch_fwd_b(const KernelArgs& a, int num_sms, cudaStream_t st) {
  if (a.elem_f16)
    return a.bias ? launch_fwd_t<ElemF16, DQK, DV, true>(a, num_sms, st)
                  : launch_fwd_t<ElemF16, DQK, DV, false>(a, num_sms, st);
  return a.bias ? launch_fwd_t<ElemBf16, DQK, DV, true>(a, num_sms, st)
                : launch_fwd_t<ElemBf16, DQK, DV, false>(a, num_sms, st);
}

}  // namespace

cudaError_t launch_fwd(const KernelArgs& a, int num_sms, cudaStream_t st) {
  // query heads in pairs sharing a KV head: two tiles per CTA, one softmax
  // warpgroup each, P in tensor memory
  if ((a.Hq / a.Hkv) % 2 == 0 && a.d_qk <= 128 && a.d_v <= 128) return launch_fwd2t(a, num_sms, st);
  if (a.d_v == 64) {
    if (a.d_qk == 64) return launch_fwd_b<64, 64>(a, num_sms, st);
    if (a.d_qk == 128) return launch_fwd_b<128, 64>(a, num_sms, st);
    if (a.d_qk == 192) return launch_fwd_b<192, 64>(a, num_sms, st);
  } else if (a.d_v == 128) {
    if (a.d_qk == 64) return launch_fwd_b<64, 128>(a, num_sms, st);
    if (a.d_qk == 128) return launch_fwd_b<128, 128>(a, num_sms, st);
    if (a.d_qk == 192) return launch_fwd_b<192, 128>(a, num_sms, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
