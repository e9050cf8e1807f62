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
// Roles: warp 0 TMA producer, warp 1 MMA issuer, warps 4-11 softmax and
// epilogue.  Each query row is shared by two softmax threads, one per key
// half of the tile (64 keys each, warps 4-7 and 8-11), so a thread's chain
// per tile is half a row and a tile's exponentials spread over eight warps;
// with the maximum fixed before the second pass, the two halves meet only
// twice per item (the row maximum after pass 1, the row sum at the end).  S
// is double-buffered in tensor memory, so the tensor core works on S(j+1)
// while the softmax warps read S(j).  Q of the next item loads during this
// one (two stages), and O leaves through shared memory by TMA stores.
#include <cmath>

#include "attn_internal.cuh"

namespace attn {
namespace {
using namespace sm103;

constexpr float kLn2f = 0.6931471805599453f;
constexpr float kPScale = 256.f;  // P8 = E4M3(256 p)

struct F8Layout {
  static constexpr int kT = kTile * kTile;  // one 128 x 128 tile of one-byte elements
  // Q of the next item loads during this one (stage = item parity)
  static constexpr int kQStages = 2, kKStages = 3, kVStages = 2, kPStages = 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQStages * kT;
  static constexpr int kVOff = kKOff + kKStages * kT;
  static constexpr int kPOff = kVOff + kVStages * kT;
  // O in bf16 for the TMA store: two 64-column boxes of 16 KB, 128-byte swizzled
  static constexpr int kOOff = kPOff + kPStages * kT;
  static constexpr int kBarOff = kOOff + 2 * 16384;
  static constexpr int kXchOff = kBarOff + 1024;  // row exchange slots [set][half][row]
  static constexpr int kBytes = kXchOff + 2048;   // barriers, then the item ring at +256
  static constexpr int kAlloc = kBytes + 1024;   // slack to align the window to 1 KB
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
  // above half of the SM's shared memory, so two CTAs (each taking all of
  // tensor memory) never share an SM
  static_assert(kAlloc > 114 * 1024, "one CTA per SM");
  static constexpr uint32_t kColS = 0;    // S buffers [0,128), [128,256)
  static constexpr uint32_t kColO = 256;  // O [256,384)
};

struct F8Bars {
  uint64_t q_full[2], q_empty[2], o_full, o_empty, drain, stg_full, stg_free;
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
};
static_assert(sizeof(F8Bars) + 8 <= 256, "barriers, tensor-memory holder and flag before the ring");

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

// The 64 scores of this thread's half row (one S buffer) in fp32, raw
// (before the scale): two loads, one wait.
__device__ __forceinline__ void load_half_row(uint32_t s_tm, uint32_t (&u)[2][32]) {
#pragma unroll
  for (int q = 0; q < 2; ++q) tmem_ld32x32b_x32(s_tm + q * 32, u[q]);
  tmem_ld_wait(u);
}

// An empty exchange slot: a NaN payload the arithmetic never produces (the
// GPU's own NaN results are all 0x7fffffff).
constexpr uint32_t kXchEmpty = 0x7fa5a5a5u;

// Row exchange between the two threads of one query row: each writes its
// value into its own slot and takes the other's, leaving that slot empty.
// Slots alternate between two sets, so a thread's next write to a set comes
// after its partner has emptied it (the partner's write in between orders
// them).  The wait is bounded like every other wait.
__device__ __forceinline__ void xch_put(uint32_t* slot, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(v) : "memory");
}
__device__ __forceinline__ bool xch_take(uint32_t* slot, uint32_t& v) {
  const uint32_t addr = smem_u32(slot);
  uint64_t t0 = 0;
  for (uint32_t n = 0;; ++n) {
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    if (v != kXchEmpty) break;
    if ((n & 255u) == 255u) {
      const uint64_t t = globaltimer_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > 2000000000ull) return false;
    }
  }
  asm volatile("st.relaxed.cta.shared::cta.b32 [%0], %1;" ::"r"(addr), "r"(kXchEmpty) : "memory");
  return true;
}

__global__ void __launch_bounds__(384, 1) fwd_fp8_kernel(const __grid_constant__ KernelArgs a) {
  using L = F8Layout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  F8Bars* bars = reinterpret_cast<F8Bars*>(sm + L::kBarOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kBarOff + sizeof(F8Bars));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  ItemRing* ring = reinterpret_cast<ItemRing*>(sm + L::kBarOff + 256);
  uint32_t* xch = reinterpret_cast<uint32_t*>(sm + L::kXchOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = a.B * a.n_qt * a.Hq;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 256);
    mbar_init(&bars->stg_full, 256);  // every softmax thread's share of O staged
    mbar_init(&bars->stg_free, 1);    // the previous O store has read the staging
    mbar_init(&bars->drain, 1);
    for (int s = 0; s < L::kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_empty[s], 256);
      mbar_init(&bars->p_full[s], 256);
      mbar_init(&bars->p_empty[s], 1);
    }
    ring_init(ring, 1 + 256);  // MMA issuer + the softmax threads
    *abort_flag = 0;
    mbar_fence_init();
  }
  for (int i = tid; i < 512; i += blockDim.x) xch[i] = kXchEmpty;
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
        const int qs = it & 1;
        if (it >= 2 && !(ok = mbar_wait(&bars->q_empty[qs], ((it >> 1) - 1) & 1))) break;
        const int qrow = w.b * a.Sq + w.t * kTile;
        mbar_arrive_expect_tx(&bars->q_full[qs], L::kT);
        if (ATTN_CHECK(a, tma_box_ok(0, kTile, a.d_qk, 1, w.h, a.Hq, qrow, kTile,
                                     (int64_t)a.B * a.Sq, false), 0x7901))
          tma_load_3d(sm + L::kQOff + qs * L::kT, &a.tm_q, &bars->q_full[qs], 0, w.h, qrow);
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
          ATTN_TL(1, kc);
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
        for (uint32_t u = (it > 2u ? it - 2u : 0u); u < it; ++u)
          mbar_wait(&bars->q_full[u & 1], (u >> 1) & 1, 100000000ull);
        for (uint32_t u = (kc > (uint32_t)L::kKStages ? kc - L::kKStages : 0u); u < kc; ++u)
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
    uint32_t q_off = 0;  // the current item's Q stage, in 16-byte units
    auto issue_s = [&]() -> bool {
      const int s = kc % L::kKStages, sb = T & 1;
      if (!mbar_wait_warp(&bars->k_full[s], (kc / L::kKStages) & 1)) return false;
      if (T >= 2 && !mbar_wait_warp(&bars->s_empty[sb], ((T >> 1) - 1) & 1)) return false;
      tc_fence_after();
      const uint64_t kd = k_desc + static_cast<uint32_t>((s * L::kT) >> 4);
      mma_f8_ss4_warp(tm + L::kColS + sb * kTile, q_desc + q_off, kd, idesc, 0u);
      mma_commit_warp(&bars->s_full[sb]);
      mma_commit_warp(&bars->k_empty[s]);
      ATTN_TL(10, T);
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
      q_off = static_cast<uint32_t>(((it & 1) * L::kT) >> 4);
      if (!(ok = mbar_wait_warp(&bars->q_full[it & 1], (it >> 1) & 1))) break;
      if (!(ok = issue_s())) break;
      for (int t2 = 0; t2 < 2 * n && ok; ++t2) {
        if (t2 + 1 < 2 * n) {
          if (!(ok = issue_s())) break;
        } else {
          mma_commit_warp(&bars->q_empty[it & 1]);  // every S of this item is issued
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
        ATTN_TL(11, pc);
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
    // thread (r, hf): query row r (TMEM lane r), keys [64 hf, 64 hf + 64) of
    // each tile, value dims [64 hf, 64 hf + 64) of O
    const int hf = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t p_addr = smem_u32(sm + L::kPOff);
    uint32_t T = 0, pc = 0, it = 0, xc = 0;
    bool ok = true;
    // swap v with the other half's thread of this row (warp-uniform result)
    auto exchange = [&](float v, float& other) -> bool {
      const uint32_t set = xc & 1;
      ++xc;
      xch_put(xch + (set * 2 + hf) * 128 + r, __float_as_uint(v));
      uint32_t t = 0;
      const bool got = xch_take(xch + (set * 2 + (hf ^ 1)) * 128 + r, t);
      other = __uint_as_float(t);
      return __all_sync(0xffffffffu, got);
    };
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) || !(ok = ring_pop(ring, rn, idx)) ||
          idx < 0)
        break;
      const F8Item w = f8_item(a, idx);
      const int i = w.t * kTile + r;
      const bool row_ok = i < a.Sq;
      const int64_t grow = (int64_t)w.b * a.Sq + i;
      bf16* orow = a.o + (grow * a.Hq + w.h) * kTile + hf * 64;  // this half's 64 dims
      float* lse_out = a.lse + ((int64_t)w.b * a.Hq + w.h) * a.Sq + i;
      if (w.n == 0) {
        if (row_ok && ATTN_CHECK(a, span_ok(orow - a.o, 64, (int64_t)a.B * a.Sq * a.Hq * kTile) &&
                                        span_ok(lse_out - a.lse, 1, (int64_t)a.B * a.Hq * a.Sq),
                                 0x7904)) {
#pragma unroll
          for (int c = 0; c < 64; c += 8)
            *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          if (hf == 0) *lse_out = -INFINITY;
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
      // validity of this thread's 64 keys of tile j
      auto valid = [&](int j) -> uint64_t {
        uint64_t vb[2];
        kv_valid_bits(a, general, w.b, w.kv_lo + j * kTile, rlo, rhi, my_id, my_pos, vb);
        return row_ok ? vb[hf] : 0ull;
      };
      // pass 1: the row maximum of the raw scores over valid keys (the scale
      // is positive, so the maximum of the scaled scores is the scaled one)
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
      for (int j = 0; j < w.n; ++j) {
        const uint64_t vb = valid(j);
        const int sb = T & 1;
        if (!(ok = mbar_wait_warp(&bars->s_full[sb], (T >> 1) & 1))) break;
        if (lane == 0) ATTN_TL(20 + (warp - 4), T);
        tc_fence_after();
        uint32_t u[2][32];
        load_half_row(tmem + lane_base + L::kColS + sb * kTile + hf * 64, u);
        tc_fence_before();
        mbar_arrive(&bars->s_empty[sb]);
        ++T;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t m32 = static_cast<uint32_t>(vb >> (q * 32));
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float x0 = (m32 & (1u << e)) ? __uint_as_float(u[q][e]) : -INFINITY;
            const float x1 = (m32 & (2u << e)) ? __uint_as_float(u[q][e + 1]) : -INFINITY;
            mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], x0, x1);
          }
        }
      }
      if (!ok) break;
      float mraw = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                         fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      float mo;
      if (!(ok = exchange(mraw, mo))) break;
      mraw = fmaxf(mraw, mo);  // the row's maximum, the same value in both halves
      const float m = mraw * a.fp8_sc2;  // log2 units (-inf: no valid key)
      const float m_use = (m == -INFINITY) ? 0.f : m;
      // pass 2: P8 = E4M3(256 exp2(s - m)) into shared memory, l = sum of p
      float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      for (int j = 0; j < w.n; ++j) {
        const uint64_t vb = valid(j);
        const int sb = T & 1, pb = pc & 1;
        if (!(ok = mbar_wait_warp(&bars->s_full[sb], (T >> 1) & 1))) break;
        if (lane == 0) ATTN_TL(20 + (warp - 4), T);
        tc_fence_after();
        uint32_t u[2][32];
        load_half_row(tmem + lane_base + L::kColS + sb * kTile + hf * 64, u);
        tc_fence_before();
        mbar_arrive(&bars->s_empty[sb]);
        ++T;
        uint32_t pw[16];  // this half's 64 E4M3 codes, key order
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t m32 = static_cast<uint32_t>(vb >> (q * 32));
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
        // (keys 16 c .. 16 c + 15) at chunk c ^ (r % 8); this half writes
        // chunks 4 hf .. 4 hf + 3
        const uint32_t prow = p_addr + pb * L::kT + r * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_shared_v4(prow + (((4 * hf + c) ^ (r & 7)) << 4), pw[4 * c], pw[4 * c + 1],
                       pw[4 * c + 2], pw[4 * c + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        if (lane == 0) ATTN_TL(30 + (warp - 4), pc);
        mbar_arrive(&bars->p_full[pb]);
        ++pc;
      }
      if (!ok) break;
      const float lh = (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
      float lo;
      if (!(ok = exchange(lh, lo))) break;
      const float l = hf == 0 ? lh + lo : lo + lh;  // one order in both halves
      // epilogue: O = descale_v * acc / (256 l), LSE = m + log2 l (natural log out)
      if (lane == 0 && warp == 4) ATTN_TL(40, it);
      if (!(ok = mbar_wait_warp(&bars->o_full, it & 1))) break;
      if (lane == 0 && warp == 4) ATTN_TL(41, it);
      tc_fence_after();
      const float inv = (l > 0.f) ? a.fp8_dv / (kPScale * l) : 0.f;
      // the staging is free once the previous item's O store has read it
      // (the thread that issued that store waits for the read, then releases)
      if (it > 0) {
        if (tid == 128) {
          bulk_wait_read_all();
          mbar_arrive(&bars->stg_free);
        }
        if (!(ok = mbar_wait_warp(&bars->stg_free, (it - 1) & 1))) break;
      }
      // this half's 64 dims of O in bf16 into box hf of the staging, laid out
      // as the store map's 128-byte-swizzled boxes: 16-byte chunk c of row r
      // at chunk c ^ (r % 8)
      const uint32_t stg_row = smem_u32(sm + L::kOOff + hf * 16384 + r * 128);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t o[32];
        tmem_ld32x32b_x32(tmem + lane_base + L::kColO + hf * 64 + q * 32, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int e8 = c * 8;
          st_shared_v4(stg_row + (static_cast<uint32_t>((q * 4 + c) ^ (r & 7)) << 4),
                       pack_bf16x2(__uint_as_float(o[e8 + 0]) * inv, __uint_as_float(o[e8 + 1]) * inv),
                       pack_bf16x2(__uint_as_float(o[e8 + 2]) * inv, __uint_as_float(o[e8 + 3]) * inv),
                       pack_bf16x2(__uint_as_float(o[e8 + 4]) * inv, __uint_as_float(o[e8 + 5]) * inv),
                       pack_bf16x2(__uint_as_float(o[e8 + 6]) * inv, __uint_as_float(o[e8 + 7]) * inv));
        }
      }
      // every row of the tile staged: one thread stores both boxes (rows past
      // the batch row's end are clipped by the map)
      fence_proxy_async_smem();
      mbar_arrive(&bars->stg_full);
      bool sok = true;
      if (tid == 128) {
        sok = mbar_wait(&bars->stg_full, it & 1);
        if (sok) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
            if (ATTN_CHECK(a, tma_box_ok(c * 64, 64, a.d_v, 2, w.h, a.Hq, w.t * kTile, kTile, a.Sq,
                                         true) && w.b >= 0 && w.b < a.B, 0x7905))
              tma_store_4d(&a.tm_o, sm + L::kOOff + c * 16384, c * 64, w.h, w.t * kTile, w.b);
          bulk_commit_group();
        }
      }
      if (!(ok = __all_sync(0xffffffffu, sok))) break;
      if (hf == 0) {
        if (row_ok &&
            ATTN_CHECK(a, span_ok(lse_out - a.lse, 1, (int64_t)a.B * a.Hq * a.Sq), 0x7906))
          *lse_out = (l > 0.f) ? (m + __log2f(l)) * kLn2f : -INFINITY;
        if (a.max_logit && ATTN_CHECK(a, span_ok((int64_t)w.b * a.Hq + w.h, 1, (int64_t)a.B * a.Hq),
                                      0x7907))
          warp_max_logit(a.max_logit + (int64_t)w.b * a.Hq + w.h, m);
      }
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
      if (lane == 0 && warp == 4) ATTN_TL(42, it);
      ++it;
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x930 + (warp - 4));
      *abort_flag = 1;
    }
    if (tid == 128) bulk_wait_all();  // the last O store has read shared memory and landed
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
  return launch_pdl(fwd_fp8_kernel, dim3(grid), dim3(384), L::kAlloc, st, a);
}

}  // namespace attn

#ifdef ATTN_TIMELINE
// Debug builds only: timeline of this translation unit's kernels.
extern "C" int attn_debug_timeline_f8(unsigned long long* out, int cap) {
  cudaDeviceSynchronize();
  const int n = cap < attn::kTimelineCap ? cap : attn::kTimelineCap;
  cudaMemcpyFromSymbol(out, attn::g_timeline, sizeof(unsigned long long) * n);
  static unsigned long long zeros[attn::kTimelineCap];
  cudaMemcpyToSymbol(attn::g_timeline, zeros, sizeof(zeros));
  return n;
}
#endif
