// Forward pass over two query tiles at once: the same 128 query rows of two
// query heads of one KV group (GQA groups of even size, d_qk, d_v <= 128).
//
//   S_X(j)  = Q_X K(j)^T     X in {A, B}; A = Q_X from shared memory, TMEM out
//   P_X(j)  = exp2(S - m)    one softmax warpgroup per head, one query row per
//                            thread, P written back over S_X as packed bf16
//   O_X    += P_X(j) V(j)    A = P_X from TMEM, B = V(j) from shared memory
//
// Both heads read the same K / V tiles.  Each head has its own warpgroup, so
// every scheduler runs two softmax warps whose load, arithmetic and exp2
// phases overlap, and the tensor core alternates between the heads: while one
// warpgroup exponentiates S_A(j), S_B(j) and P_B(j-1) V run.  Tensor memory:
// S_A, S_B, O_A, O_B, 128 columns each.  S_X(j+1) overwrites P_X(j) and is
// issued after P_X(j) V by the same thread, so the in-order pipe orders them;
// for the same reason P_X(j-1) V is complete whenever S_X(j) is, which is all
// a rescale of O_X needs.
//
// Outputs and semantics: TransformerEngine PR #3516 diagram (the fused-attention
// forward that feeds the backward with O and the softmax statistics); rows with
// no valid key get O = 0 and LSE = -inf.
#include <cmath>

#include "attn_internal.cuh"

namespace attn {
namespace {
using namespace sm103;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

template <int DQK, int DV>
struct F2Layout {
  static constexpr int kQBytes = kTile * DQK * 2;                  // one head's Q tile
  static constexpr int kKVBytes = kTile * (DQK > DV ? DQK : DV) * 2;  // one K or V stage
  static constexpr int kQStages = 2;   // Q of the next item loads during this one
  static constexpr int kKVStages = 3;  // K(j), V(j), K(j+1) in flight
  static constexpr int kQOff = 0;      // [stage][head]
  static constexpr int kKVOff = kQStages * 2 * kQBytes;
  static constexpr int kBarOff = kKVOff + kKVStages * kKVBytes;
  static constexpr int kBytes = kBarOff + 512;
  static constexpr int kAlloc = kBytes;  // the dynamic window is 1 KB-aligned (checked)
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t kColS = 0;    // S_A [0,128), S_B [128,256)
  static constexpr uint32_t kColO = 256;  // O_A [256,384), O_B [384,512)
};

struct F2Bars {
  uint64_t q_full[2], q_empty[2], kv_full[3], kv_empty[3];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t drain;
};

struct F2Item {
  int b, t, h0, kv_lo, n;
};

// item = (query tile, head pair), longest causal tiles first
__device__ __forceinline__ F2Item f2_item(const KernelArgs& a, int idx) {
  const int hp = a.Hq / 2;
  const int per_t = a.B * hp;
  const int t_rev = idx / per_t, rem = idx - t_rev * per_t;
  F2Item it;
  it.t = a.n_qt - 1 - t_rev;
  it.b = rem / hp;
  it.h0 = 2 * (rem - it.b * hp);
  const int2 r = a.q_tile_range[it.b * a.n_qt + it.t];
  it.kv_lo = r.x;
  it.n = (r.y > r.x) ? (r.y - r.x + kTile - 1) / kTile : 0;
  return it;
}

// One 32-column chunk of a score row in log2 units: bias and, for chunks not
// valid throughout the warp, the key mask (separate instantiations keep the
// per-element code free of branches).
template <bool MASKED, bool HAS_BIAS>
__device__ __forceinline__ void chunk_max2(const uint32_t (&u)[32], uint32_t m32, float scale_log2,
                                           const bf16* bias_row, int kc0, int Skv, bool row_ok,
                                           float (&mx8)[8]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float x[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      x[t] = __uint_as_float(u[e + t]);
      if (HAS_BIAS) {
        x[t] *= scale_log2;
        if (row_ok && kc0 + e + t < Skv) x[t] += __bfloat162float(bias_row[kc0 + e + t]) * kLog2e;
      }
      if (MASKED) x[t] = (m32 & (1u << (e + t))) ? x[t] : -INFINITY;
    }
    mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], x[0], x[1]);
  }
}

template <bool MASKED, bool HAS_BIAS>
__device__ __forceinline__ void chunk_exp2(const uint32_t (&u)[32], uint32_t m32, float scale_log2,
                                           float m_use, const bf16* bias_row, int kc0, int Skv,
                                           bool row_ok, float (&rs4)[4], uint32_t (&pk)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float y[2];
    if (HAS_BIAS) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int c = 2 * e + t;
        y[t] = __uint_as_float(u[c]) * scale_log2;
        if (row_ok && kc0 + c < Skv) y[t] += __bfloat162float(bias_row[kc0 + c]) * kLog2e;
        y[t] -= m_use;
      }
    } else {
      // both lanes of the pair in one instruction: x * scale - m
      const float2 x2 = make_float2(__uint_as_float(u[2 * e]), __uint_as_float(u[2 * e + 1]));
      const float2 y2 =
          fma_f32x2(x2, make_float2(scale_log2, scale_log2), make_float2(-m_use, -m_use));
      y[0] = y2.x;
      y[1] = y2.y;
    }
    float p2[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float pv = ex2_approx(y[t]);
      p2[t] = MASKED ? ((m32 & (1u << (2 * e + t))) ? pv : 0.f) : pv;
    }
    // two running pairs of partial row sums, (rs4[0], rs4[1]) and (rs4[2], rs4[3])
    const int r = (e & 1) * 2;
    const float2 acc = add_f32x2(make_float2(rs4[r], rs4[r + 1]), make_float2(p2[0], p2[1]));
    rs4[r] = acc.x;
    rs4[r + 1] = acc.y;
    pk[e] = pack_bf16x2(p2[0], p2[1]);
  }
}

template <int DQK, int DV, bool HAS_BIAS>
__global__ void __launch_bounds__(384, 1) fwd2t_kernel(const __grid_constant__ KernelArgs a) {
  using L = F2Layout<DQK, DV>;
  constexpr int NKV = L::kKVStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_u32(sm) & 1023u) {  // swizzled tiles need 1 KB alignment; no slack to realign
    if (threadIdx.x == 0) report_timeout(a, 0x6ff);
    return;
  }
  F2Bars* bars = reinterpret_cast<F2Bars*>(sm + L::kBarOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kBarOff + sizeof(F2Bars));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  ItemRing* ring = reinterpret_cast<ItemRing*>(sm + L::kBarOff + 256);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = a.B * a.n_qt * (a.Hq / 2);

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 128);
      mbar_init(&bars->o_full[s], 1);
      mbar_init(&bars->o_empty[s], 128);
    }
    for (int s = 0; s < NKV; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->drain, 1);
    ring_init(ring, 1 + 256);  // MMA issuer, two softmax warpgroups
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
  grid_dep_wait();  // the previous kernel on the stream has finished
  grid_dep_launch();
  const bool general = path_general(a);

  // Registers: 384 threads x 168 at launch = 64,512 per CTA.  Warpgroup 0
  // (producer, MMA issuer, two idle warps) drops to 104 and the two softmax
  // warpgroups rise to 200, room for a whole S row per thread:
  // 128 x 104 + 256 x 200 = 64,512.
  if (warp < 4) {
    regs_lower<104>();  // once for the whole warpgroup
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        prefetch_tensormap(&a.tm_q);
        prefetch_tensormap(&a.tm_k);
        prefetch_tensormap(&a.tm_v);
        uint32_t it = 0, kvc = 0;  // kvc: K / V stage loads issued, in ring order
        bool ok = true;
        auto load_kv = [&](const CUtensorMap* m, int ncols, int g, int krow) -> bool {
          const int s = kvc % NKV;
          if (kvc >= (uint32_t)NKV && !mbar_wait(&bars->kv_empty[s], ((kvc / NKV) - 1) & 1))
            return false;
          uint8_t* dst = sm + L::kKVOff + s * L::kKVBytes;
          mbar_arrive_expect_tx(&bars->kv_full[s], kTile * ncols * 2);
          for (int c = 0; c < ncols / 64; ++c)
            tma_load_3d(dst + c * 16384, m, &bars->kv_full[s], c * 64, g, krow);
          ++kvc;
          return true;
        };
        for (uint32_t rn = 0;; ++rn) {
          int32_t idx;
          if (!ok || *abort_flag ||
              !(ok = ring_push(ring, rn, &a.hdr->next_item[0], n_items, idx)) ||
              idx < 0)
            break;
          const F2Item w = f2_item(a, idx);
          if (w.n == 0) continue;
          const int qs = it & 1;
          if (it >= 2 && !(ok = mbar_wait(&bars->q_empty[qs], ((it >> 1) - 1) & 1))) break;
          const int qrow = w.b * a.Sq + w.t * kTile;
          mbar_arrive_expect_tx(&bars->q_full[qs], 2 * L::kQBytes);
          for (int x = 0; x < 2; ++x) {
            uint8_t* dst = sm + L::kQOff + (qs * 2 + x) * L::kQBytes;
  #pragma unroll
            for (int c = 0; c < DQK / 64; ++c)
              tma_load_3d(dst + c * 16384, &a.tm_q, &bars->q_full[qs], c * 64, w.h0 + x, qrow);
          }
          ++it;
          const int g = w.h0 / (a.Hq / a.Hkv);
          for (int j = 0; j < w.n && ok; ++j) {
            const int krow = w.b * a.Skv + w.kv_lo + j * kTile;
            ok = load_kv(&a.tm_k, DQK, g, krow) && load_kv(&a.tm_v, DV, g, krow);
          }
        }
        if (!ok) {
          report_timeout(a, 0x610);
          *abort_flag = 1;
        }
        if (*abort_flag) {  // let copies in flight land before the CTA exits
          for (uint32_t u = (it > 2u ? it - 2u : 0u); u < it; ++u)
            mbar_wait(&bars->q_full[u & 1], (u >> 1) & 1, 100000000ull);
          for (uint32_t u = (kvc > (uint32_t)NKV ? kvc - NKV : 0u); u < kvc; ++u)
            mbar_wait(&bars->kv_full[u % NKV], (u / NKV) & 1, 100000000ull);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs this loop on warp-uniform values; one elected lane
      // issues each GEMM's MMAs from a single asm statement.
      constexpr uint32_t id_s = idesc_bf16_f32(128, kTile, false, false);
      constexpr uint32_t id_o = idesc_bf16_f32(128, DV, false, true);
      const uint32_t tm = warp_uniform(tmem);
      const uint64_t q_km = sdesc_sw128(smem_u32(sm + L::kQOff), 16, 1024);
      const uint64_t kv_km = sdesc_sw128(smem_u32(sm + L::kKVOff), 16, 1024);
      const uint64_t kv_mn = sdesc_sw128(smem_u32(sm + L::kKVOff), 16384, 1024);
      uint32_t it = 0, kvc = 0, st = 0;  // st: steps (key tiles) so far
      bool ok = true;
      auto stage_off = [&](uint32_t c) -> uint32_t {
        return static_cast<uint32_t>(((c % NKV) * L::kKVBytes) >> 4);
      };
      // S_X(step) = Q_X K^T; K at ring position kc
      auto issue_s = [&](int x, uint32_t qs, uint32_t kc) {
        const uint64_t qd = q_km + static_cast<uint32_t>(((qs * 2 + x) * L::kQBytes) >> 4);
        const uint64_t kd = kv_km + stage_off(kc);
        mma_ss_warp<DQK / 16, 2, 1018, 2, 1018>(tm + L::kColS + x * kTile, qd, kd, id_s, 0u);
        mma_commit_warp(&bars->s_full[x]);
      };
      // O_X += P_X V; V at ring position vc; P_X packed over S_X
      auto issue_pv = [&](int x, uint32_t vc, bool first) {
        const uint64_t vd = kv_mn + stage_off(vc);
        mma_ts_warp<kTile / 16, 8, 8, 128, 128>(tm + L::kColO + x * kTile, tm + L::kColS + x * kTile,
                                                vd, id_o, first ? 0u : 1u);
      };
      for (uint32_t rn = 0;; ++rn) {
        int32_t idx;
        if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) ||
            !(ok = ring_pop_warp1(ring, rn, idx)) || idx < 0)
          break;
        F2Item w = f2_item(a, idx);
        w.n = warp_uniform(w.n);
        if (w.n == 0) continue;
        const uint32_t qs = it & 1;
        if (!(ok = mbar_wait_warp(&bars->q_full[qs], (it >> 1) & 1))) break;
        // K(0): both S of the first step
        if (!(ok = mbar_wait_warp(&bars->kv_full[kvc % NKV], (kvc / NKV) & 1))) break;
        tc_fence_after();
        issue_s(0, qs, kvc);
        issue_s(1, qs, kvc);
        mma_commit_warp(&bars->kv_empty[kvc % NKV]);
        ++kvc;
        for (int j = 0; j < w.n && ok; ++j) {
          const uint32_t k = st + j;
          const uint32_t vc = kvc;  // V(j)
          const bool more = j + 1 < w.n;
          if (!(ok = mbar_wait_warp(&bars->kv_full[vc % NKV], (vc / NKV) & 1))) break;
          for (int x = 0; x < 2 && ok; ++x) {
            if (!(ok = mbar_wait_warp(&bars->p_full[x], k & 1))) break;
            ATTN_TL(30 + x, k);
            if (j == 0 && it > 0 && !(ok = mbar_wait_warp(&bars->o_empty[x], (it - 1) & 1))) break;
            tc_fence_after();
            issue_pv(x, vc, j == 0);
            if (!more) {
              mma_commit_warp(&bars->o_full[x]);
              continue;
            }
            // S_X(j+1) over P_X(j), after P_X(j) V (same issuer, in-order pipe)
            if (x == 0 &&
                !(ok = mbar_wait_warp(&bars->kv_full[(vc + 1) % NKV], ((vc + 1) / NKV) & 1)))
              break;
            tc_fence_after();
            issue_s(x, qs, vc + 1);
            ATTN_TL(32 + x, k + 1);
          }
          if (!ok) break;
          mma_commit_warp(&bars->kv_empty[vc % NKV]);  // V(j) read by both P V
          if (more) mma_commit_warp(&bars->kv_empty[(vc + 1) % NKV]);  // K(j+1) by both S
          kvc += more ? 2 : 1;
        }
        if (!ok) break;
        mma_commit_warp(&bars->q_empty[qs]);  // every S of this item done once these land
        st += w.n;
        ++it;
      }
      if (!ok && lane == 0) {
        report_timeout(a, 0x620);
        *abort_flag = 1;
      }
      mma_commit_warp(&bars->drain);
      mbar_wait(&bars->drain, 0, 200000000ull);
    }  // warps 2 and 3 have no role
  } else {
    regs_raise<200>();
    // ------------------------------------------------------------ softmax + epilogue
    const int x = (warp - 4) >> 2;  // head of the pair
    const int r = (tid - 128) & 127;  // TMEM lane = query row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + L::kColS + x * kTile;
    const uint32_t o_tm = tmem + lane_base + L::kColO + x * kTile;
    uint32_t st = 0, it = 0;
    bool ok = true;
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) || !(ok = ring_pop(ring, rn, idx)) ||
          idx < 0)
        break;
      const F2Item w = f2_item(a, idx);
      const int h = w.h0 + x;
      const int i = w.t * kTile + r;
      const bool row_ok = i < a.Sq;
      const int64_t grow = (int64_t)w.b * a.Sq + i;
      bf16* orow = a.o + (grow * a.Hq + h) * DV;
      float* lse_out = a.lse + ((int64_t)w.b * a.Hq + h) * a.Sq + i;
      if (w.n == 0) {
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < DV; c += 8)
            *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          *lse_out = a.sink ? a.sink[h] : -INFINITY;  // only the sink, if any
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
        const int bb = a.bias_b > 1 ? w.b : 0, bh = a.bias_h > 1 ? h : 0;
        bias_row = a.bias + (((int64_t)bb * a.bias_h + bh) * a.Sq + i) * a.Skv;
      }
      float m_ref = -INFINITY, l = 0.f;
      float row_max = -INFINITY;  // exact row max of the scaled logits (log2 units)
      for (int j = 0; j < w.n; ++j) {
        const uint32_t k = st + j;
        const int k0 = w.kv_lo + j * kTile;
        uint64_t vb[2];
        kv_valid_bits(a, general, w.b, k0, rlo, rhi, my_id, my_pos, vb);
        if (!row_ok) vb[0] = vb[1] = 0ull;
        bool none[4], all[4];
        uint32_t m32s[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          m32s[q] = static_cast<uint32_t>(vb[q >> 1] >> ((q & 1) * 32));
          none[q] = __all_sync(0xffffffffu, m32s[q] == 0u);
          all[q] = __all_sync(0xffffffffu, m32s[q] == 0xffffffffu);
        }
        if (!(ok = mbar_wait_warp(&bars->s_full[x], k & 1))) break;
        if (lane == 0 && (warp & 3) == 0) ATTN_TL(34 + x, k);
        tc_fence_after();
        // the whole S row of this thread in registers: four loads, one wait
        uint32_t u[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32x32b_x32(s_tm + q * 32, u[q]);
        tmem_ld_wait();
        // pass 1: the row max over valid keys (log2 units)
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (none[q]) continue;
          if (all[q])
            chunk_max2<false, HAS_BIAS>(u[q], m32s[q], a.scale_log2, bias_row, k0 + q * 32, a.Skv,
                                        row_ok, mx8);
          else
            chunk_max2<true, HAS_BIAS>(u[q], m32s[q], a.scale_log2, bias_row, k0 + q * 32, a.Skv,
                                       row_ok, mx8);
        }
        float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                         fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        if (!HAS_BIAS) mx *= a.scale_log2;  // scale > 0 keeps the order
        if (lane == 0 && (warp & 3) == 0) ATTN_TL(36 + x, k);
        row_max = fmaxf(row_max, mx);
        const float m_new = fmaxf(m_ref, mx);
        const bool grow_max = m_new > m_ref + kRescaleThreshold;
        const bool rescale = grow_max && j > 0 && m_ref > -INFINITY;
        const float f = rescale ? ex2_approx(m_ref - m_new) : 1.f;
        if (grow_max) m_ref = m_new;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // pass 2: P = exp2(x - m), packed over S_X (chunk q -> columns [16 q, 16 q + 16))
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[16];
          if (none[q]) {
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = 0u;
          } else if (all[q]) {
            chunk_exp2<false, HAS_BIAS>(u[q], m32s[q], a.scale_log2, m_use, bias_row, k0 + q * 32,
                                        a.Skv, row_ok, rs4, pk);
          } else {
            chunk_exp2<true, HAS_BIAS>(u[q], m32s[q], a.scale_log2, m_use, bias_row, k0 + q * 32,
                                       a.Skv, row_ok, rs4, pk);
          }
          tmem_st32x32b_x16(s_tm + q * 16, pk);
        }
        l = l * f + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
        // P_X(j-1) V is complete (S_X(j) was issued after it) and P_X(j) V waits
        // for this warpgroup's arrival below: O_X may be rescaled here.
        // Tensor-memory loads/stores are warp-wide, so every lane takes part.
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int q = 0; q < DV / 32; ++q) {
            uint32_t o[32];
            tmem_ld32x32b_x32(o_tm + q * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32x32b_x32(o_tm + q * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        if (lane == 0 && (warp & 3) == 0) ATTN_TL(38 + x, k);
        mbar_arrive(&bars->p_full[x]);
      }
      if (!ok) break;
      // epilogue: O / l and LSE
      if (!(ok = mbar_wait_warp(&bars->o_full[x], it & 1))) break;
      tc_fence_after();
      // the sink logit, if any, joins the normaliser (it has no value vector)
      float l_fin = l, m_fin = m_ref, o_scale = 1.f;
      if (a.sink) {
        const float s2 = a.sink[h] * kLog2e;
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
        tmem_ld32x32b_x32(o_tm + q * 32, u);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(u[c + 0]) * inv_l, __uint_as_float(u[c + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(u[c + 2]) * inv_l, __uint_as_float(u[c + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(u[c + 4]) * inv_l, __uint_as_float(u[c + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(u[c + 6]) * inv_l, __uint_as_float(u[c + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + q * 32 + c) = v;
          }
        }
      }
      if (row_ok) *lse_out = (l_fin > 0.f) ? (m_fin + __log2f(l_fin)) * kLn2 : -INFINITY;
      if (a.max_logit) warp_max_logit(a.max_logit + (int64_t)w.b * a.Hq + h, row_max);
      tc_fence_before();
      mbar_arrive(&bars->o_empty[x]);
      st += w.n;
      ++it;
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x630 + (warp & 7));
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

template <int DQK, int DV>
cudaError_t go(const KernelArgs& a, int nsm, cudaStream_t st) {
  using L = F2Layout<DQK, DV>;
  auto kern = a.bias ? fwd2t_kernel<DQK, DV, true> : fwd2t_kernel<DQK, DV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int items = a.B * a.n_qt * (a.Hq / 2);
  const int grid = items < nsm ? items : nsm;
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(kern, dim3(grid), dim3(384), L::kAlloc, st, a);
}

}  // namespace

cudaError_t launch_fwd2t(const KernelArgs& a, int nsm, cudaStream_t st) {
  if (a.d_qk == 64 && a.d_v == 64) return go<64, 64>(a, nsm, st);
  if (a.d_qk == 64 && a.d_v == 128) return go<64, 128>(a, nsm, st);
  if (a.d_qk == 128 && a.d_v == 64) return go<128, 64>(a, nsm, st);
  if (a.d_qk == 128 && a.d_v == 128) return go<128, 128>(a, nsm, st);
  return cudaErrorInvalidValue;
}

}  // namespace attn

#ifdef ATTN_TIMELINE
// Debug builds only: timeline of this translation unit's kernels.
extern "C" int attn_debug_timeline_f2(unsigned long long* out, int cap) {
  cudaDeviceSynchronize();
  const int n = cap < attn::kTimelineCap ? cap : attn::kTimelineCap;
  cudaMemcpyFromSymbol(out, attn::g_timeline, sizeof(unsigned long long) * n);
  static unsigned long long zeros[attn::kTimelineCap];
  cudaMemcpyToSymbol(attn::g_timeline, zeros, sizeof(zeros));
  return n;
}
#endif
