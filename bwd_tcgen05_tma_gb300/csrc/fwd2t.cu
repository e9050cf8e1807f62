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
  // one head's Q stage; once the item's S MMAs are done it stages that head's
  // O tile for the TMA store, so it holds the larger of the two
  static constexpr int kQStage = kKVBytes;
  static constexpr int kQStages = 2;   // Q of the next item loads during this one
  static constexpr int kKVStages = 3;  // K(j), V(j), K(j+1) in flight
  static constexpr int kQOff = 0;      // [stage][head]
  static constexpr int kKVOff = kQStages * 2 * kQStage;
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
  int b, t, h0;
};

// item = (query tile w = b * n_qt + t, head pair), numbered w * (Hq / 2) + pair
__device__ __forceinline__ F2Item f2_item(const KernelArgs& a, int idx) {
  const int hp = a.Hq / 2;
  const int w = idx / hp;
  F2Item it;
  it.b = w / a.n_qt;
  it.t = w - it.b * a.n_qt;
  it.h0 = 2 * (idx - w * hp);
  return it;
}

// Ring entry of the c-th claim: (item, key tiles, first key, 0), or
// (-1, 0, 0, 0) past the end.  Claims walk the query tiles in the metadata
// pass's order (longest first), the head pairs of a tile one after another.
__device__ __forceinline__ int4 f2_entry(const KernelArgs& a, int c, int n_items) {
  if (c >= n_items) return make_int4(-1, 0, 0, 0);
  const int hp = a.Hq / 2;
  const int rank = c / hp;
  const int w = a.q_order[rank];
  const int2 r = a.q_tile_range[w];
  const int n = (r.y > r.x) ? (r.y - r.x + kTile - 1) / kTile : 0;
  return make_int4(w * hp + (c - rank * hp), n, r.x, 0);
}

// Per-row state of one softmax thread for one item.
struct F2Row {
  int h, i, b, rlo, rhi, my_id, my_pos;
  bool row_ok;
  int64_t grow;
  const bf16* bias_row;
};

// One 32-column chunk of a score row in log2 units: bias and, for chunks not
// valid throughout the warp, the key mask (separate instantiations keep the
// per-element code free of branches).  The mask also writes -inf over the
// masked scores, so the exponential pass needs no mask of its own.
template <class E, bool MASKED, bool HAS_BIAS>
__device__ __forceinline__ void chunk_max2(uint32_t (&u)[32], uint32_t m32, float scale_log2,
                                           const bf16* bias_row, int kc0, int Skv, bool row_ok,
                                           float (&mx8)[8]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float x[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (MASKED) u[e + t] = (m32 & (1u << (e + t))) ? u[e + t] : 0xff800000u;  // -inf
      x[t] = __uint_as_float(u[e + t]);
      if (HAS_BIAS) {
        x[t] *= scale_log2;
        if (row_ok && kc0 + e + t < Skv) x[t] += E::ld(bias_row + kc0 + e + t) * kLog2e;
      }
    }
    mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], x[0], x[1]);
  }
}

template <class E, bool MASKED, bool HAS_BIAS>
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
        if (row_ok && kc0 + c < Skv) y[t] += E::ld(bias_row + kc0 + c) * kLog2e;
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
    pk[e] = E::pack(p2[0], p2[1]);
  }
}

template <class E, int DQK, int DV, bool HAS_BIAS>
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
  ItemRing4* ring = reinterpret_cast<ItemRing4*>(sm + L::kBarOff + 256);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = a.B * a.n_qt * (a.Hq / 2);

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 2);  // the two epilogue stores
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
    ring4_init(ring, 1 + 1 + 256);  // TMA producer, MMA issuer, two softmax warpgroups
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
      // Takes the items from the ring like every other role.  While it streams
      // the K / V tiles of the current item it already takes the next item
      // (once the scheduler has published it) and loads that item's Q tiles
      // as soon as their stage is free, so the next item's first S can follow
      // this item's last one.
      if (lane == 0) {
        prefetch_tensormap(&a.tm_q);
        prefetch_tensormap(&a.tm_k);
        prefetch_tensormap(&a.tm_v);
        uint32_t qi = 0, kvc = 0, rn = 0;  // Q tile pairs, K / V stage loads, ring entries
        bool ok = true;
        auto load_kv = [&](const CUtensorMap* m, int ncols, int g, int krow) -> bool {
          const int s = kvc % NKV;
          if (kvc >= (uint32_t)NKV && !mbar_wait(&bars->kv_empty[s], ((kvc / NKV) - 1) & 1))
            return false;
          uint8_t* dst = sm + L::kKVOff + s * L::kKVBytes;
          mbar_arrive_expect_tx(&bars->kv_full[s], kTile * ncols * 2);
          for (int c = 0; c < ncols / 64; ++c)
            if (ATTN_CHECK(a, box_ok(a, m, c * 64, g, krow, kTile), 0x7101))
              tma_load_3d(dst + c * 16384, m, &bars->kv_full[s], c * 64, g, krow);
          ++kvc;
          return true;
        };
        // both heads' Q tiles of item e into stage qi & 1 (its previous user done)
        auto q_free = [&]() -> bool {
          return qi < 2 || mbar_test_wait(&bars->q_empty[qi & 1], ((qi >> 1) - 1) & 1);
        };
        auto load_q = [&](int4 e) -> bool {
          const int qs = qi & 1;
          if (qi >= 2 && !mbar_wait(&bars->q_empty[qs], ((qi >> 1) - 1) & 1)) return false;
          const F2Item w = f2_item(a, e.x);
          const int qrow = w.b * a.Sq + w.t * kTile;
          mbar_arrive_expect_tx(&bars->q_full[qs], 2 * L::kQBytes);
          ATTN_TL(50, qi);
          for (int x = 0; x < 2; ++x) {
            uint8_t* dst = sm + L::kQOff + (qs * 2 + x) * L::kQStage;
  #pragma unroll
            for (int c = 0; c < DQK / 64; ++c)
              if (ATTN_CHECK(a, box_ok(a, &a.tm_q, c * 64, w.h0 + x, qrow, kTile), 0x7102))
                tma_load_3d(dst + c * 16384, &a.tm_q, &bars->q_full[qs], c * 64, w.h0 + x, qrow);
          }
          ++qi;
          return true;
        };
        // the next item with key tiles (or the end marker), waiting for the
        // scheduler if `wait`; items without key tiles need no loads.  Returns
        // false without a result when not waiting and nothing is published yet.
        auto next_item = [&](bool wait, int4& e) -> bool {
          for (;;) {
            if (!wait && !ring4_ready(ring, rn)) return false;  // e untouched
            int4 t;
            if (!(ok = ring4_pop1(ring, rn, t))) {
              e = make_int4(-1, 0, 0, 0);
              return true;
            }
            ++rn;
            if (t.x < 0 || t.y > 0) {
              e = t;
              return true;
            }
          }
        };
        int4 cur;
        next_item(true, cur);
        bool cur_q = false;  // cur's Q already loaded
        while (ok && cur.x >= 0 && !*abort_flag) {
          if (!cur_q && !(ok = load_q(cur))) break;
          ATTN_TL(49, qi - 1);
          const F2Item w = f2_item(a, cur.x);
          const int g = w.h0 / (a.Hq / a.Hkv);
          int4 held = make_int4(-2, 0, 0, 0);  // -2: next item not taken yet
          bool held_q = false;
          for (int j = 0; j < cur.y && ok; ++j) {
            const int krow = w.b * a.Skv + cur.z + j * kTile;
            if (!(ok = load_kv(&a.tm_k, DQK, g, krow))) break;
            ATTN_TL(55, (kvc - 1) >> 1);
            if (!(ok = load_kv(&a.tm_v, DV, g, krow))) break;
            ATTN_TL(56, (kvc - 1) >> 1);
            if (held.x == -2) next_item(false, held);
            if (!held_q && held.x >= 0 && q_free()) {
              if (!(ok = load_q(held))) break;
              held_q = true;
            }
          }
          if (!ok) break;
          if (held.x == -2) next_item(true, held);
          cur = held;
          cur_q = held_q;
        }
        if (!ok) {
          report_timeout(a, 0x610);
          *abort_flag = 1;
        }
        if (*abort_flag) {  // let copies in flight land before the CTA exits
          for (uint32_t u = (qi > 2u ? qi - 2u : 0u); u < qi; ++u)
            mbar_wait(&bars->q_full[u & 1], (u >> 1) & 1, 100000000ull);
          for (uint32_t u = (kvc > (uint32_t)NKV ? kvc - NKV : 0u); u < kvc; ++u)
            mbar_wait(&bars->kv_full[u % NKV], (u / NKV) & 1, 100000000ull);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs this loop on warp-uniform values; one elected lane
      // issues each GEMM's MMAs from a single asm statement.
      constexpr uint32_t id_s = idesc_f32acc(E::kMmaFmt, 128, kTile, false, false);
      constexpr uint32_t id_o = idesc_f32acc(E::kMmaFmt, 128, DV, false, true);
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
        const uint64_t qd = q_km + static_cast<uint32_t>(((qs * 2 + x) * L::kQStage) >> 4);
        const uint64_t kd = kv_km + stage_off(kc);
        mma_ss_warp<DQK / 16, 4, 2, 1018, 2, 1018>(tm + L::kColS + x * kTile, qd, kd, id_s, 0u);
        mma_commit_warp(&bars->s_full[x]);
      };
      // O_X += P_X V; V at ring position vc; P_X packed over S_X
      auto issue_pv = [&](int x, uint32_t vc, bool first) {
        const uint64_t vd = kv_mn + stage_off(vc);
        mma_ts_warp<kTile / 16, 4, 8, 8, 128, 128>(tm + L::kColO + x * kTile, tm + L::kColS + x * kTile,
                                                vd, id_o, first ? 0u : 1u);
      };
      uint32_t rn = 0;
      // the next item with key tiles (-1: the end); items without any need
      // no MMAs
      auto next_item = [&](int4& e) -> bool {
        do {
          if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
          if (!ring4_pop_warp1(ring, rn++, e)) return false;
        } while (e.x >= 0 && e.y == 0);
        return true;
      };
      int4 cur;
      if (!(ok = next_item(cur))) cur.x = -1;
      if (cur.x >= 0) {  // both S of the first item's first step
        ATTN_TL(42, 0);
        if ((ok = mbar_wait_warp(&bars->q_full[0], 0) &&
                  mbar_wait_warp(&bars->kv_full[0], 0))) {
          tc_fence_after();
          issue_s(0, 0, 0);
          issue_s(1, 0, 0);
          mma_commit_warp(&bars->kv_empty[0]);
          kvc = 1;
        }
      }
      // Each step j: P_X(j) V, then the S that reuses P_X(j)'s columns: S_X(j+1)
      // of this item or, at its last step, S_X(0) of the next item, so that the
      // next item starts the way a step does.
      while (ok && cur.x >= 0) {
        const int n = cur.y;
        const uint32_t qs = it & 1;
        int4 nxt = make_int4(-1, 0, 0, 0);
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t k = st + j;
          const uint32_t vc = kvc;  // V(j); the next S reads K at vc + 1
          const bool more = j + 1 < n;
          if (!more && !(ok = next_item(nxt))) break;
          const bool go_on = more || nxt.x >= 0;  // an S follows this step's P V
          const uint32_t qs_s = more ? qs : ((it + 1) & 1);
          if (!(ok = mbar_wait_warp(&bars->kv_full[vc % NKV], (vc / NKV) & 1))) break;
          ATTN_TL(57, k);
          for (int x = 0; x < 2 && ok; ++x) {
            if (!(ok = mbar_wait_warp(&bars->p_full[x], k & 1))) break;
            ATTN_TL(30 + x, k);
            if (j == 0 && it > 0 && !(ok = mbar_wait_warp(&bars->o_empty[x], (it - 1) & 1))) break;
            tc_fence_after();
            issue_pv(x, vc, j == 0);
            ATTN_TL(40 + x, k);
            if (!more) mma_commit_warp(&bars->o_full[x]);
            // V(j) is read by both P V and by nothing after them: its stage
            // goes back to the producer now, not after the next S as well,
            // so that K(j+2) starts loading one S earlier
            if (x == 1) mma_commit_warp(&bars->kv_empty[vc % NKV]);
            if (!go_on) continue;
            // the next S over P_X(j), after P_X(j) V (same issuer, in-order pipe)
            if (x == 0) {
              if (!more && !(ok = mbar_wait_warp(&bars->q_full[qs_s], ((it + 1) >> 1) & 1))) break;
              if (!(ok = mbar_wait_warp(&bars->kv_full[(vc + 1) % NKV], ((vc + 1) / NKV) & 1)))
                break;
            }
            tc_fence_after();
            issue_s(x, qs_s, vc + 1);
            ATTN_TL(32 + x, k + 1);
          }
          if (!ok) break;
          if (go_on) mma_commit_warp(&bars->kv_empty[(vc + 1) % NKV]);  // the next K by both S
          kvc += go_on ? 2 : 1;
        }
        if (!ok) break;
        // this item's Q stage is released by the epilogue once its O store has read it
        st += n;
        ++it;
        cur = nxt;
      }
      if (!ok && lane == 0) {
        report_timeout(a, 0x620);
        *abort_flag = 1;
      }
      mma_commit_warp(&bars->drain);
      mbar_wait(&bars->drain, 0, 200000000ull);
    } else if (warp == 2) {
      // ------------------------------------------------------------ scheduler
      // Claims work items from the global counter, looks up each one's key
      // range and publishes them in order; every other role takes them from
      // the ring, so the latency of the claim is off their paths.  (The
      // failure-path test knob keeps it from publishing anything: every other
      // role's bounded wait for work then runs out and the CTA unwinds.)
      if (lane == 0 && !a.test_stall) {
        for (uint32_t pub = 0;; ++pub) {
          const int4 e = f2_entry(a, atomicAdd(&a.hdr->next_item[0], 1), n_items);
          if (*abort_flag) break;
          if (!ring4_publish(ring, pub, e)) {
            report_timeout(a, 0x640);
            *abort_flag = 1;
            break;
          }
          if (e.x < 0) break;
        }
      }
    }  // warp 3 has no role
  } else {
    regs_raise<200>();
    // ------------------------------------------------------------ softmax + epilogue
    const int x = (warp - 4) >> 2;  // head of the pair
    const int r = (tid - 128) & 127;  // TMEM lane = query row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + L::kColS + x * kTile;
    const uint32_t o_tm = tmem + lane_base + L::kColO + x * kTile;
    uint32_t st = 0, it = 0, rn = 0;
    int store_stage = -1;  // thread r == 0: Q stage its last O store still reads
    bool ok = true;
    // this thread's row of item e: indices, mask range or metadata, bias row
    // (the loads are issued here and consumed at the item's first step)
    auto row_of = [&](const int4& e) -> F2Row {
      F2Row R;
      R.rlo = R.rhi = R.my_id = R.my_pos = 0;
      R.bias_row = nullptr;
      const F2Item w = f2_item(a, e.x >= 0 ? e.x : 0);
      R.b = w.b;
      R.h = w.h0 + x;
      R.i = w.t * kTile + r;
      R.row_ok = e.x >= 0 && R.i < a.Sq;
      R.grow = (int64_t)w.b * a.Sq + R.i;
      if (R.row_ok && e.y > 0) {
        if (!general) {
          const int2 kr = band_keys_of_query(a, R.i, a.seg_lo[R.grow], a.seg_hi[R.grow]);
          R.rlo = kr.x;
          R.rhi = kr.y;
        } else {
          R.my_id = a.q_id[R.grow];
          R.my_pos = a.q_pos[R.grow];
        }
        if (HAS_BIAS) {
          const int bb = a.bias_b > 1 ? w.b : 0, bh = a.bias_h > 1 ? R.h : 0;
          R.bias_row = a.bias + (((int64_t)bb * a.bias_h + bh) * a.Sq + R.i) * a.Skv;
        }
      }
      return R;
    };
    int4 e = make_int4(-1, 0, 0, 0);
    if (!(ok = ring4_pop(ring, rn++, e))) e.x = -1;
    F2Row R = row_of(e);
    while (ok && e.x >= 0 && !__any_sync(0xffffffffu, *abort_flag != 0)) {
      const int h = R.h;
      const int i = R.i;
      const bool row_ok = R.row_ok;
      bf16* orow = a.o + (R.grow * a.Hq + h) * DV;
      float* lse_out = a.lse + ((int64_t)R.b * a.Hq + h) * a.Sq + i;
      struct { int b, n, kv_lo; } w = {R.b, e.y, e.z};
      if (w.n == 0) {
        if (row_ok && ATTN_CHECK(a, span_ok(orow - a.o, DV, (int64_t)a.B * a.Sq * a.Hq * DV) &&
                                        span_ok(lse_out - a.lse, 1, (int64_t)a.B * a.Hq * a.Sq),
                                 0x7106)) {
#pragma unroll
          for (int c = 0; c < DV; c += 8)
            *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          *lse_out = a.sink ? a.sink[h] : -INFINITY;  // only the sink, if any
        }
        if (!(ok = ring4_pop(ring, rn++, e))) break;
        R = row_of(e);
        continue;
      }
      const int rlo = R.rlo, rhi = R.rhi, my_id = R.my_id, my_pos = R.my_pos;
      const bf16* bias_row = R.bias_row;
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
        if (lane == 0 && x == 0) ATTN_TL(8 + (warp - 4), k);
        if (r == 0 && store_stage >= 0) {  // the previous item's O store has read its stage
          bulk_wait_read_all();
          mbar_arrive(&bars->q_empty[store_stage]);
          store_stage = -1;
        }
        tc_fence_after();
        // the whole S row of this thread in registers: four loads, one wait
        uint32_t u[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32x32b_x32(s_tm + q * 32, u[q]);
        tmem_ld_wait(u);
        // pass 1: the row max over valid keys (log2 units)
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (none[q]) continue;
          if (all[q])
            chunk_max2<E, false, HAS_BIAS>(u[q], m32s[q], a.scale_log2, bias_row, k0 + q * 32, a.Skv,
                                        row_ok, mx8);
          else
            chunk_max2<E, true, HAS_BIAS>(u[q], m32s[q], a.scale_log2, bias_row, k0 + q * 32, a.Skv,
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
          } else {  // masked scores are -inf by now: exp2 gives 0 there
            chunk_exp2<E, false, HAS_BIAS>(u[q], m32s[q], a.scale_log2, m_use, bias_row, k0 + q * 32,
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
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32x32b_x32(o_tm + q * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        if (lane == 0 && (warp & 3) == 0) ATTN_TL(38 + x, k);
        if (lane == 0) ATTN_TL(0 + (warp - 4), k);
        mbar_arrive(&bars->p_full[x]);
      }
      if (!ok) break;
      // the next item, popped now so that its row loads overlap this epilogue
      int4 e_next;
      if (!(ok = ring4_pop(ring, rn++, e_next))) break;
      if (lane == 0 && warp == 4) ATTN_TL(46, it);
      const F2Row R_next = row_of(e_next);
      // epilogue: O / l and LSE
      if (!(ok = mbar_wait_warp(&bars->o_full[x], it & 1))) break;
      if (lane == 0 && warp == 4) ATTN_TL(47, it);
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
      // O / l in bf16 into this head's Q stage of the item (its S MMAs are
      // done, o_full says so), laid out as the store map's 128-byte-swizzled
      // 64-column boxes: 16-byte chunk c of row r at chunk c ^ (r % 8).  One
      // row per thread; each group of 8 rows spreads over all banks.
      uint8_t* stg = sm + L::kQOff + ((it & 1) * 2 + x) * L::kQStage;
#pragma unroll
      for (int q = 0; q < DV / 32; ++q) {
        uint32_t u[32];
        tmem_ld32x32b_x32(o_tm + q * 32, u);
        tmem_ld_wait(u);
        const uint32_t row = smem_u32(stg + (q >> 1) * 16384 + r * 128);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int e8 = c * 8;
          const uint32_t chunk = static_cast<uint32_t>(((q & 1) * 4 + c) ^ (r & 7));
          st_shared_v4(row + chunk * 16,
                       E::pack(__uint_as_float(u[e8 + 0]) * inv_l, __uint_as_float(u[e8 + 1]) * inv_l),
                       E::pack(__uint_as_float(u[e8 + 2]) * inv_l, __uint_as_float(u[e8 + 3]) * inv_l),
                       E::pack(__uint_as_float(u[e8 + 4]) * inv_l, __uint_as_float(u[e8 + 5]) * inv_l),
                       E::pack(__uint_as_float(u[e8 + 6]) * inv_l, __uint_as_float(u[e8 + 7]) * inv_l));
        }
      }
      // every row of the tile is in shared memory: one thread stores it (rows
      // past the batch row's end are clipped by the map); the stage is
      // released once the store has read it (checked at the next item)
      fence_proxy_async_smem();
      named_bar_sync(1 + x, 128);
      if (r == 0) {
        const F2Item wi = f2_item(a, e.x);
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          if (ATTN_CHECK(a, tma_box_ok(c * 64, 64, DV, 2, h, a.Hq, wi.t * kTile, kTile, a.Sq, true) &&
                                wi.b >= 0 && wi.b < a.B, 0x7103))
            tma_store_4d(&a.tm_o, stg + c * 16384, c * 64, h, wi.t * kTile, wi.b);
        bulk_commit_group();
        store_stage = static_cast<int>(it & 1);
      }
      if (row_ok && ATTN_CHECK(a, span_ok(lse_out - a.lse, 1, (int64_t)a.B * a.Hq * a.Sq), 0x7104))
        *lse_out = (l_fin > 0.f) ? (m_fin + __log2f(l_fin)) * kLn2 : -INFINITY;
      if (a.max_logit && ATTN_CHECK(a, span_ok((int64_t)w.b * a.Hq + h, 1, (int64_t)a.B * a.Hq), 0x7105))
        warp_max_logit(a.max_logit + (int64_t)w.b * a.Hq + h, row_max);
      tc_fence_before();
      mbar_arrive(&bars->o_empty[x]);
      if (lane == 0 && warp == 4) ATTN_TL(48, it);
      st += w.n;
      ++it;
      e = e_next;
      R = R_next;
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x630 + (warp & 7));
      *abort_flag = 1;
    }
    if (r == 0) bulk_wait_all();  // the last O store has read shared memory and landed
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
  using L = F2Layout<DQK, DV>;
  auto kern = a.bias ? fwd2t_kernel<E, DQK, DV, true> : fwd2t_kernel<E, DQK, DV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int items = a.B * a.n_qt * (a.Hq / 2);
  const int grid = items < nsm ? items : nsm;
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(kern, dim3(grid), dim3(384), L::kAlloc, st, a);
}

}  // namespace

template <class E>
cudaError_t launch_fwd2t_e(const KernelArgs& a, int nsm, cudaStream_t st) {
  if (a.d_qk == 64 && a.d_v == 64) return go<E, 64, 64>(a, nsm, st);
  if (a.d_qk == 64 && a.d_v == 128) return go<E, 64, 128>(a, nsm, st);
  if (a.d_qk == 128 && a.d_v == 64) return go<E, 128, 64>(a, nsm, st);
  if (a.d_qk == 128 && a.d_v == 128) return go<E, 128, 128>(a, nsm, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd2t(const KernelArgs& a, int nsm, cudaStream_t st) {
  return a.elem_f16 ? launch_fwd2t_e<ElemF16>(a, nsm, st) : launch_fwd2t_e<ElemBf16>(a, nsm, st);
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
