// Deterministic dQ pass with every MMA A operand in tensor memory
// (d_qk, d_v <= 128).
//
// One work item is a 128-row query tile of one query head; the CTA walks the
// key tiles that tile can see in a fixed order, so dQ never depends on the
// grid (maxdiffusion PR #485, review: no accumulation across grid iterations;
// Summary: the separate dQ kernel of the unfused backward).  Per key tile j:
//
//   S(j)   = Q K(j)^T          A = Q   from TMEM, B = K(j)  from smem
//   P(j)   = exp2(S scale log2e - LSE2)       softmax warps, kept packed in registers
//   dP(j)  = dO V(j)^T         A = dO  from TMEM, B = V(j)  from smem
//   dS(j)  = P (dP - D)                       written back over dP as packed bf16
//   dQ    += dS(j) K(j)        A = dS  from TMEM, B = K(j)  (MN-major) from smem
//
// Q and dO are copied once per item from shared memory into tensor memory, so
// the only shared-memory operands are the K / V tiles: 96 KB of operand reads
// per step instead of 192 KB, below the tensor core's own 1536 cycles.
#include <cmath>

#include "attn_internal.cuh"

namespace attn {
namespace {
using namespace sm103;

constexpr float kLog2e = 1.4426950408889634f;

template <int DQK, int DV>
struct Dq128Layout {
  static constexpr int kQBytes = kTile * DQK * 2;
  static constexpr int kOBytes = kTile * DV * 2;
  static constexpr int kKBytes = kTile * DQK * 2;
  static constexpr int kVBytes = kTile * DV * 2;
  // K(j) is read by S(j) and by dQ(j), which waits for dS(j); V(j) only by dP(j)
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kQOff = 0;
  static constexpr int kOOff = kQBytes;
  static constexpr int kKOff = kQBytes + kOBytes;
  static constexpr int kVOff = kKOff + kKStages * kKBytes;
  static constexpr int kBarOff = kVOff + kVStages * kVBytes;
  static constexpr int kBytes = kBarOff + 512;
  static constexpr int kAlloc = kBytes;  // the dynamic window is 1 KB-aligned (checked)
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColQ = 384, kColO = 448;
};

struct Dq128Bars {
  uint64_t qo_full, qo_empty, qo_ready, s_full, s_free, dp_full, ds_ready, acc_full, acc_empty,
      drain, drain2;
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
};

// Validity of the 64 keys [kh, kh + 64) of batch row b for one query row.
// Fast path: the row's key range [rlo, rhi).  General path: same nonzero
// segment id and a key position inside the row's band.
__device__ __forceinline__ uint64_t kv_bits64(const KernelArgs& a, bool general, int b, int kh,
                                              int rlo, int rhi, int my_id, int my_pos) {
  if (!general) return range_bits64(rlo - kh, rhi - kh);
  if (my_id == 0 || kh >= a.Skv) return 0ull;
  const int2 kp = band_key_pos(a, my_pos);
  if ((kh % kChunk) == 0) {
    const int nkc = (a.Skv + kChunk - 1) / kChunk;
    uint64_t bits;
    if (chunk_bits(a.kv_chunk[b * nkc + kh / kChunk], my_id, kp, bits)) return bits;
  }
  // every lane of the warp reads the same keys
  const int32_t* kid = a.kv_id + (int64_t)b * a.Skv + kh;
  const int32_t* kps = a.kv_pos + (int64_t)b * a.Skv + kh;
  const int n = min(64, a.Skv - kh);
  uint64_t v = 0ull;
  for (int c = 0; c < n; ++c) {
    const int pk = __ldg(kps + c);
    const bool ok = (__ldg(kid + c) == my_id) & (pk >= kp.x) & (pk <= kp.y);
    v |= static_cast<uint64_t>(ok) << c;
  }
  return v;
}

template <class E, int DQK, int DV, bool HAS_BIAS>
__global__ void __launch_bounds__(512, 1) dq128_kernel(const __grid_constant__ KernelArgs a) {
  using L = Dq128Layout<DQK, DV>;
  constexpr int KS = L::kKStages, VS = L::kVStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_u32(sm) & 1023u) {  // swizzled tiles need 1 KB alignment; no slack to realign
    if (threadIdx.x == 0) report_timeout(a, 0x4ff);
    return;
  }
  Dq128Bars* bars = reinterpret_cast<Dq128Bars*>(sm + L::kBarOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kBarOff + sizeof(Dq128Bars));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  ItemRing* ring = reinterpret_cast<ItemRing*>(sm + L::kBarOff + 256);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = a.B * a.n_qt * a.Hq;

  if (tid == 0) {
    mbar_init(&bars->qo_full, 1);
    mbar_init(&bars->qo_empty, 256);
    mbar_init(&bars->qo_ready, 256);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 256);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->ds_ready, 256);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 128);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->drain2, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    ring_init(ring, 1 + 1 + 256 + 128);  // two MMA issuers, softmax warps, epilogue
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

  // causal work is heaviest in the last query tiles: hand those out first
  // item = (query tile w = b * n_qt + t, head h), numbered w * Hq + h; the
  // producer claims them with the query tiles in the metadata pass's order
  // (longest first)
  auto item_of = [&](int idx, int& b, int& t, int& h, int& kv_lo, int& n) {
    const int w = idx / a.Hq;
    h = idx - w * a.Hq;
    b = w / a.n_qt;
    t = w - b * a.n_qt;
    const int2 r = a.q_tile_range[w];
    kv_lo = r.x;
    n = (r.y > r.x) ? (r.y - r.x + kTile - 1) / kTile : 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&a.tm_q);
      prefetch_tensormap(&a.tm_k);
      prefetch_tensormap(&a.tm_v);
      prefetch_tensormap(&a.tm_do);
      uint32_t kt = 0, it = 0, k_issued = 0, v_issued = 0;
      bool ok = true;
      for (uint32_t rn = 0;; ++rn) {
        int32_t idx;
        if (!ok || *abort_flag || !(ok = ring_push(ring, rn, &a.hdr->next_item[2], n_items, idx, a.q_order, a.Hq)) ||
            idx < 0)
          break;
        int b, t, h, kv_lo, n;
        item_of(idx, b, t, h, kv_lo, n);
        if (n == 0) continue;
        if (it > 0 && !(ok = mbar_wait(&bars->qo_empty, (it - 1) & 1))) break;
        const int qrow = b * a.Sq + t * kTile;
        mbar_arrive_expect_tx(&bars->qo_full, L::kQBytes + L::kOBytes);
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c)
          if (ATTN_CHECK(a, box_ok(a, &a.tm_q, c * 64, h, qrow, kTile), 0x7401))
            tma_load_3d(sm + L::kQOff + c * 16384, &a.tm_q, &bars->qo_full, c * 64, h, qrow);
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          if (ATTN_CHECK(a, box_ok(a, &a.tm_do, c * 64, h, qrow, kTile), 0x7402))
            tma_load_3d(sm + L::kOOff + c * 16384, &a.tm_do, &bars->qo_full, c * 64, h, qrow);
        ++it;
        const int g = h / (a.Hq / a.Hkv);
        for (int j = 0; j < n; ++j, ++kt) {
          const int krow = b * a.Skv + kv_lo + j * kTile;
          const int ks = kt % KS, vs = kt % VS;
          if (kt >= (uint32_t)KS && !(ok = mbar_wait(&bars->k_empty[ks], ((kt / KS) - 1) & 1)))
            break;
          mbar_arrive_expect_tx(&bars->k_full[ks], L::kKBytes);
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c)
            if (ATTN_CHECK(a, box_ok(a, &a.tm_k, c * 64, g, krow, kTile), 0x7403))
              tma_load_3d(sm + L::kKOff + ks * L::kKBytes + c * 16384, &a.tm_k, &bars->k_full[ks],
                          c * 64, g, krow);
          ++k_issued;
          if (kt >= (uint32_t)VS && !(ok = mbar_wait(&bars->v_empty[vs], ((kt / VS) - 1) & 1)))
            break;
          mbar_arrive_expect_tx(&bars->v_full[vs], L::kVBytes);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            if (ATTN_CHECK(a, box_ok(a, &a.tm_v, c * 64, g, krow, kTile), 0x7404))
              tma_load_3d(sm + L::kVOff + vs * L::kVBytes + c * 16384, &a.tm_v, &bars->v_full[vs],
                          c * 64, g, krow);
          ++v_issued;
        }
      }
      if (!ok) {
        report_timeout(a, 0x410);
        *abort_flag = 1;
      }
      if (*abort_flag) {  // let copies in flight land before the CTA exits
        if (it > 0) mbar_wait(&bars->qo_full, (it - 1) & 1, 100000000ull);
        for (uint32_t u = (k_issued > (uint32_t)KS ? k_issued - KS : 0u); u < k_issued; ++u)
          mbar_wait(&bars->k_full[u % KS], (u / KS) & 1, 100000000ull);
        for (uint32_t u = (v_issued > (uint32_t)VS ? v_issued - VS : 0u); u < v_issued; ++u)
          mbar_wait(&bars->v_full[u % VS], (u / VS) & 1, 100000000ull);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Two issuing warps on different schedulers, one per tensor-memory
    // region: warp 1 issues S (S region), warp 2 issues dP and dQ (dP / dS
    // region and the dQ accumulator).  Each region's writer and readers are in
    // one warp, whose MMAs the in-order pipe orders.  Each warp runs its loop
    // on warp-uniform values; one elected lane issues each GEMM's MMAs from a
    // single asm statement.
    const bool s_side = (warp == 1);
    constexpr uint32_t id_s = idesc_f32acc(E::kMmaFmt, 128, kTile, false, false);
    constexpr uint32_t id_dq = idesc_f32acc(E::kMmaFmt, 128, DQK, false, true);
    const uint32_t tm = warp_uniform(tmem);
    const uint64_t k_km = sdesc_sw128(smem_u32(sm + L::kKOff), 16, 1024);
    const uint64_t k_mn = sdesc_sw128(smem_u32(sm + L::kKOff), 16384, 1024);
    const uint64_t v_km = sdesc_sw128(smem_u32(sm + L::kVOff), 16, 1024);
    uint32_t kt = 0, it = 0;
    bool ok = true;
    auto issue_s = [&](uint32_t k) -> bool {  // S = Q K^T, Q from tensor memory
      const int s_ = k % KS;
      if (!mbar_wait_warp(&bars->k_full[s_], (k / KS) & 1)) return false;
      tc_fence_after();
      const uint64_t kd = k_km + static_cast<uint32_t>((s_ * L::kKBytes) >> 4);
      mma_ts_warp<DQK / 16, 4, 8, 8, 2, 1018>(tm + L::kColS, tm + L::kColQ, kd, id_s, 0u);
      mma_commit_warp(&bars->s_full);
      return true;
    };
    auto issue_dp = [&](uint32_t k) -> bool {  // dP = dO V^T, dO from tensor memory
      const int s_ = k % VS;
      if (!mbar_wait_warp(&bars->v_full[s_], (k / VS) & 1)) return false;
      tc_fence_after();
      const uint64_t vd = v_km + static_cast<uint32_t>((s_ * L::kVBytes) >> 4);
      mma_ts_warp<DV / 16, 4, 8, 8, 2, 1018>(tm + L::kColDP, tm + L::kColO, vd, id_s, 0u);
      mma_commit_warp(&bars->dp_full);
      mma_commit_warp(&bars->v_empty[s_]);
      return true;
    };
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) ||
          !(ok = ring_pop_warp1(ring, rn, idx)) || idx < 0)
        break;
      int b, t, h, kv_lo, n;
      item_of(idx, b, t, h, kv_lo, n);
      n = warp_uniform(n);
      if (n == 0) continue;
      // Q / dO of this item in tensor memory (the softmax warps copied them
      // after the previous item's last S / dP had been read)
      if (!(ok = mbar_wait_warp(&bars->qo_ready, it & 1))) break;
      tc_fence_after();
      if (s_side) {
        if (!(ok = issue_s(kt))) break;
        for (int j = 0; j + 1 < n && ok; ++j) {  // S(k+1) over S(k) once P(k) is held
          const uint32_t k = kt + j;
          if (!(ok = mbar_wait_warp(&bars->s_free, k & 1))) break;
          ok = issue_s(k + 1);
        }
      } else {
        if (!(ok = issue_dp(kt))) break;
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t k = kt + j;
          if (!(ok = mbar_wait_warp(&bars->ds_ready, k & 1))) break;
          if (j == 0 && it > 0 && !(ok = mbar_wait_warp(&bars->acc_empty, (it - 1) & 1))) break;
          tc_fence_after();
          {  // dQ += dS K: A = packed dS (key columns [0,64) at dP columns [0,32),
             // [64,128) at [64,96)), B = K(k) MN-major, K = 128 keys
            const uint64_t kd = k_mn + static_cast<uint32_t>(((k % KS) * L::kKBytes) >> 4);
            mma_ts_warp<kTile / 16, 4, 8, 40, 128, 128>(tm + L::kColDQ, tm + L::kColDP, kd, id_dq,
                                                     j > 0 ? 1u : 0u);
            // S(k) was complete before dS(k) existed: K(k) is free after this
            mma_commit_warp(&bars->k_empty[k % KS]);
          }
          // dP(k+1) over dS(k), after dQ(k) that reads it (same issuing warp)
          if (j + 1 < n) ok = issue_dp(k + 1);
        }
        if (ok) mma_commit_warp(&bars->acc_full);
      }
      if (!ok) break;
      kt += n;
      ++it;
    }
    if (!ok && lane == 0) {
      report_timeout(a, s_side ? 0x430 : 0x431);
      *abort_flag = 1;
    }
    uint64_t* dr = s_side ? &bars->drain : &bars->drain2;
    mma_commit_warp(dr);
    mbar_wait(dr, 0, 200000000ull);
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax / dS warps
    // thread (r, half): query row r (TMEM lane r), key columns [64 half, 64 half + 64)
    const int r = (tid - 128) & 127;
    const int half = (tid - 128) >> 7;
    const int c0h = half * 64;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t kt = 0, it = 0;
    bool ok = true;
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) || !(ok = ring_pop(ring, rn, idx)) ||
          idx < 0)
        break;
      int b, t, h, kv_lo, n;
      item_of(idx, b, t, h, kv_lo, n);
      const int i = t * kTile + r;
      const bool row_ok = i < a.Sq;
      const int64_t grow = (int64_t)b * a.Sq + i;
      if (n == 0) {  // no key visible to the tile: dQ rows are exactly zero
        if (half == 0 && row_ok &&
            ATTN_CHECK(a, dq_span_ok(a, grow, (int64_t)h * DQK, DQK,
                                     a.dq + grow * a.dq_stride + (int64_t)h * DQK, 16), 0x7405)) {
          bf16* dq_row = a.dq + grow * a.dq_stride + (int64_t)h * DQK;
#pragma unroll
          for (int c = 0; c < DQK; c += 8)
            *reinterpret_cast<uint4*>(dq_row + c) = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      // Q (half 0) or dO (half 1) row r: swizzled smem tile -> packed TMEM columns
      if (!(ok = mbar_wait_warp(&bars->qo_full, it & 1))) break;
      {
        const uint32_t src = smem_u32(sm + (half == 0 ? L::kQOff : L::kOOff));
        const uint32_t dst = tmem + lane_base + (half == 0 ? L::kColQ : L::kColO);
        const int nchunk = (half == 0 ? DQK : DV) / 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (c < nchunk) {
            uint32_t w[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint32_t ad = src + c * 16384 + r * 128 + ((u ^ (r & 7)) << 4);
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(w[4 * u]), "=r"(w[4 * u + 1]), "=r"(w[4 * u + 2]),
                             "=r"(w[4 * u + 3])
                           : "r"(ad));
            }
            tmem_st32x32b_x32(dst + c * 32, w);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->qo_ready);
      mbar_arrive(&bars->qo_empty);

      int rlo = 0, rhi = 0, my_id = 0, my_pos = 0;
      float lse2 = INFINITY, Di = 0.f;
      if (row_ok) {
        if (!general) {
          const int2 kr = band_keys_of_query(a, i, a.seg_lo[grow], a.seg_hi[grow]);
          rlo = kr.x;
          rhi = kr.y;
        } else {
          my_id = a.q_id[grow];
          my_pos = a.q_pos[grow];
        }
        const int64_t vi = ((int64_t)b * a.Hq + h) * a.Sq + i;
        lse2 = a.lse2[vi];
        Di = a.Dvec[vi];
      }
      const bf16* bias_row = nullptr;
      if (HAS_BIAS && row_ok) {
        const int bb = a.bias_b > 1 ? b : 0, bh = a.bias_h > 1 ? h : 0;
        bias_row = a.bias + (((int64_t)bb * a.bias_h + bh) * a.Sq + i) * a.Skv;
      }
      const uint32_t s_tm = tmem + lane_base + L::kColS + c0h;
      const uint32_t dp_tm = tmem + lane_base + L::kColDP + c0h;
      for (int j = 0; j < n; ++j) {
        const uint32_t k = kt + j;
        const int kh = kv_lo + j * kTile + c0h;  // first key of this thread's columns
        const uint64_t vbits = row_ok ? kv_bits64(a, general, b, kh, rlo, rhi, my_id, my_pos) : 0ull;
        if (!(ok = mbar_wait_warp(&bars->s_full, k & 1))) break;
        tc_fence_after();
        uint32_t pp[32];  // packed P of the 64 columns, kept for dS
        bool none[2];     // warp-uniform: no valid pair in the 32-column chunk
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t m32 = static_cast<uint32_t>(vbits >> (q * 32));
          none[q] = __all_sync(0xffffffffu, m32 == 0u);
          const bool all = __all_sync(0xffffffffu, m32 == 0xffffffffu);
          // P stays in registers, so the S buffer goes back to the MMA warp
          // once the second chunk of S is loaded: S(j+1) does not wait for the
          // exponentials of that chunk
          if (none[q]) {
#pragma unroll
            for (int e = 0; e < 16; ++e) pp[q * 16 + e] = 0u;
            if (q == 1) {
              tc_fence_before();
              mbar_arrive(&bars->s_free);
            }
            continue;
          }
          uint32_t u[32];
          tmem_ld32x32b_x32(s_tm + q * 32, u);
          tmem_ld_wait(u);
          if (q == 1) {
            tc_fence_before();
            mbar_arrive(&bars->s_free);
          }
          float x[32];
          if (HAS_BIAS) {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(u[e]) * a.scale_log2;
            if (row_ok) {
              const int kq = kh + q * 32;
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (kq + e < a.Skv) x[e] += E::ld(bias_row + kq + e) * kLog2e;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = ex2_approx(x[e] - lse2);
          } else {
            // x * scale - lse, two columns per instruction
            const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
            const float2 nl2 = make_float2(-lse2, -lse2);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 y = fma_f32x2(
                  make_float2(__uint_as_float(u[e]), __uint_as_float(u[e + 1])), sc2, nl2);
              x[e] = ex2_approx(y.x);
              x[e + 1] = ex2_approx(y.y);
            }
          }
          if (!all) {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = (m32 & (1u << e)) ? x[e] : 0.f;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) pp[q * 16 + e] = E::pack(x[2 * e], x[2 * e + 1]);
        }
        // dS = P (dP - D), packed bf16 over this thread's own dP columns
        if (!(ok = mbar_wait_warp(&bars->dp_full, k & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t pk[16];
          if (none[q]) {
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = 0u;
          } else {
            uint32_t u[32];
            tmem_ld32x32b_x32(dp_tm + q * 32, u);
            tmem_ld_wait(u);
            // dP - D in fp32, then one packed bf16 product with P (already bf16)
            const float2 d2 = make_float2(Di, Di);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 g = sub_f32x2(
                  make_float2(__uint_as_float(u[2 * e]), __uint_as_float(u[2 * e + 1])), d2);
              pk[e] = E::mul(pp[q * 16 + e], E::pack(g.x, g.y));
            }
          }
          tmem_st32x32b_x16(dp_tm + q * 16, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->ds_ready);
      }
      if (!ok) break;
      kt += n;
      ++it;
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x440 + (warp & 7));
      *abort_flag = 1;
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ epilogue
    const int r = tid - 384;  // TMEM lane = query row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) || !(ok = ring_pop(ring, rn, idx)) ||
          idx < 0)
        break;
      int b, t, h, kv_lo, n;
      item_of(idx, b, t, h, kv_lo, n);
      if (n == 0) continue;
      const int i = t * kTile + r;
      const bool row_ok = i < a.Sq;
      bf16* dq_row = a.dq + ((int64_t)b * a.Sq + i) * a.dq_stride + (int64_t)h * DQK;
      if (!(ok = mbar_wait_warp(&bars->acc_full, it & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < DQK / 32; ++q) {
        uint32_t u[32];
        tmem_ld32x32b_x32(tmem + lane_base + L::kColDQ + q * 32, u);
        tmem_ld_wait(u);
        if (row_ok) {
          const float sc = a.scale;
#pragma unroll
          for (int c = 0; c < 32; c += 16) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = E::pack(__uint_as_float(u[c + 2 * e]) * sc, __uint_as_float(u[c + 2 * e + 1]) * sc);
            if (ATTN_CHECK(a, dq_span_ok(a, (int64_t)b * a.Sq + i, (int64_t)h * DQK + q * 32 + c, 16,
                                         dq_row + q * 32 + c, a.grad_st32 ? 32 : 16), 0x7406))
              store16_elems(dq_row + q * 32 + c, w, a.grad_st32 != 0);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty);
      ++it;
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x450 + (warp & 3));
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

template <class E, int DQK, int DV>
cudaError_t go(const KernelArgs& a, int nsm, cudaStream_t st) {
  using L = Dq128Layout<DQK, DV>;
  auto kern = a.bias ? dq128_kernel<E, DQK, DV, true> : dq128_kernel<E, DQK, DV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int items = a.B * a.n_qt * a.Hq;
  const int grid = items < nsm ? items : nsm;
  kern<<<grid, 512, L::kAlloc, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

template <class E>
cudaError_t launch_bwd_dq128_e(const KernelArgs& a, int nsm, cudaStream_t st) {
  if (a.d_qk == 64 && a.d_v == 64) return go<E, 64, 64>(a, nsm, st);
  if (a.d_qk == 64 && a.d_v == 128) return go<E, 64, 128>(a, nsm, st);
  if (a.d_qk == 128 && a.d_v == 64) return go<E, 128, 64>(a, nsm, st);
  if (a.d_qk == 128 && a.d_v == 128) return go<E, 128, 128>(a, nsm, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dq128(const KernelArgs& a, int nsm, cudaStream_t st) {
  return a.elem_f16 ? launch_bwd_dq128_e<ElemF16>(a, nsm, st)
                    : launch_bwd_dq128_e<ElemBf16>(a, nsm, st);
}

}  // namespace attn
