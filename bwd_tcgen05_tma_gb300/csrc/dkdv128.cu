// dK / dV pass with 128-row query tiles, for the deterministic-dQ mode
// (d_qk, d_v <= 128).  dQ is produced by the separate query-tile pass.
//
// Per 128-row KV tile of one KV head (a work item, as in the 64-row pass) the
// CTA loops sequentially over the query heads of the group and every
// 128-row query tile that can see the KV tile (maxdiffusion PR #485, Summary:
// dK/dV held across Q blocks and GQA heads, accumulation order fixed inside
// the CTA).  Per query tile c:
//
//   S^T(c)  = K Q(c)^T                     smem x smem -> TMEM   (M=128, N=128)
//   P^T(c)  = exp2(S^T - LSE)              softmax warps, written back to TMEM
//                                          as packed bf16 over S^T
//   dP^T(c) = V dO(c)^T                    smem x smem -> TMEM
//   dS^T(c) = P^T (dP^T - D)               written back over dP^T, packed bf16
//   dV     += P^T(c) dO(c)                 A from TMEM
//   dK     += dS^T(c) Q(c)                 A from TMEM, issued one step later
//
// Every MMA has N = 128, half of the operand traffic comes from tensor memory,
// and the tensor core issues S(c), dK(c-1), dP(c) while the softmax warps
// exponentiate P(c).  MMAs that overwrite a TMEM region another MMA reads
// (S(c) over P(c-1), dP(c) over dS(c-1)) are issued after the reader by the
// same thread, so the in-order MMA pipeline orders them.
#include <cmath>

#include "attn_internal.cuh"

namespace attn {
namespace {
using namespace sm103;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kQ = 128;  // query tile

template <int DQK, int DV>
struct D128Layout {
  static constexpr int kKBytes = kTile * DQK * 2;
  static constexpr int kVBytes = kTile * DV * 2;
  static constexpr int kQBytes = kQ * DQK * 2;
  static constexpr int kOBytes = kQ * DV * 2;
  // Q(c) is read by S(c) and by dK(c), which is issued one step later, so Q
  // gets one stage more than dO (read by dP(c) and dV(c) within step c).
  static constexpr int kQStages = 3;
  static constexpr int kOStages = 2;
  static constexpr int kVecStages = 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKBytes;
  static constexpr int kQOff = kKBytes + kVBytes;
  static constexpr int kOOff = kQOff + kQStages * kQBytes;
  static constexpr int kVecOff = kOOff + kOStages * kOBytes;  // 1 KB per stage
  static constexpr int kBarOff = kVecOff + kVecStages * 1024;
  static constexpr int kBytes = kBarOff + 512;
  // the dynamic window starts 1 KB-aligned (checked at kernel entry), so no slack
  static constexpr int kAlloc = kBytes;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384;
};

struct D128Bars {
  uint64_t kv_full, kv_empty, s_full, dp_full, p_ready, ds_ready, acc_full, acc_empty, drain;
  uint64_t q_full[3], q_empty[3], o_full[2], o_empty[2], vec_full[2], vec_empty[2];
};

struct Vec128 {  // per query tile: negated log2-LSE and D
  float nlse2[kQ];
  float D[kQ];
};

template <class E, int DQK, int DV, bool HAS_BIAS, int DBIAS>
__global__ void __launch_bounds__(512, 1) dkdv128_kernel(const __grid_constant__ KernelArgs a) {
  using L = D128Layout<DQK, DV>;
  constexpr int NQ = L::kQStages, NO = L::kOStages, NV = L::kVecStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  // 128-byte swizzled operand tiles need 1 KB alignment; the allocation has no
  // slack to realign, so a misaligned window is reported instead of used
  if (smem_u32(sm) & 1023u) {
    if (threadIdx.x == 0) report_timeout(a, 0x3ff);
    return;
  }
  D128Bars* bars = reinterpret_cast<D128Bars*>(sm + L::kBarOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kBarOff + sizeof(D128Bars));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  Vec128* vec = reinterpret_cast<Vec128*>(sm + L::kVecOff);
  ItemRing* ring = reinterpret_cast<ItemRing*>(sm + L::kBarOff + 256);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = dkdv_n_items(a);
  const int G = a.Hq / a.Hkv;

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, 256);
    mbar_init(&bars->ds_ready, 256);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 128);
    mbar_init(&bars->drain, 1);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    for (int s = 0; s < NO; ++s) {
      mbar_init(&bars->o_full[s], 1);
      mbar_init(&bars->o_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&bars->vec_full[s], 64);
      mbar_init(&bars->vec_empty[s], 256);
    }
    ring_init(ring, 1 + 64 + 256 + 128);  // MMA, vector loader, softmax, epilogue
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&a.tm_q);
      prefetch_tensormap(&a.tm_k);
      prefetch_tensormap(&a.tm_v);
      prefetch_tensormap(&a.tm_do);
      uint32_t st = 0, kvc = 0, q_issued = 0, o_issued = 0;
      bool ok = true;
      for (uint32_t rn = 0;; ++rn) {
        int32_t idx;
        if (!ok || *abort_flag || !(ok = ring_push(ring, rn, &a.hdr->next_item[1], n_items, idx)) ||
            idx < 0)
          break;
        const DkdvItem w = dkdv_item(a, idx);
        for (int b = w.b0; b < w.b1 && ok; ++b) {
          for (int g = w.g0; g < w.g1 && ok; ++g) {
            int q_lo;
            const int nq = dkdv_q_tiles<kQ>(a, b, w.t, q_lo);
            if (nq == 0) continue;
            for (int hh = 0; hh < G && ok; ++hh) {
              const int h = g * G + hh;
              for (int s = 0; s < nq; ++s, ++st) {
                const int qrow = b * a.Sq + q_lo + s * kQ;
                const int sq = st % NQ, so = st % NO;
                if (st >= (uint32_t)NQ &&
                    !(ok = mbar_wait(&bars->q_empty[sq], ((st / NQ) - 1) & 1)))
                  break;
                uint8_t* qs = sm + L::kQOff + sq * L::kQBytes;
                mbar_arrive_expect_tx(&bars->q_full[sq], L::kQBytes);
#pragma unroll
                for (int c = 0; c < DQK / 64; ++c)
                  if (ATTN_CHECK(a, box_ok(a, &a.tm_q, c * 64, h, qrow, kQ), 0x7301))
                    tma_load_3d(qs + c * 16384, &a.tm_q, &bars->q_full[sq], c * 64, h, qrow);
                ++q_issued;
                ATTN_TL(1, st);
                if (hh == 0 && s == 0) {
                  // the group's K / V, after its first Q tile so that Q keeps
                  // streaming while the previous group drains
                  if (kvc > 0 && !(ok = mbar_wait(&bars->kv_empty, (kvc - 1) & 1))) break;
                  const int krow = b * a.Skv + w.t * kTile;
                  mbar_arrive_expect_tx(&bars->kv_full, L::kKBytes + L::kVBytes);
#pragma unroll
                  for (int c = 0; c < DQK / 64; ++c)
                    if (ATTN_CHECK(a, box_ok(a, &a.tm_k, c * 64, g, krow, kTile), 0x7302))
                      tma_load_3d(sm + L::kKOff + c * 16384, &a.tm_k, &bars->kv_full, c * 64, g, krow);
#pragma unroll
                  for (int c = 0; c < DV / 64; ++c)
                    if (ATTN_CHECK(a, box_ok(a, &a.tm_v, c * 64, g, krow, kTile), 0x7303))
                      tma_load_3d(sm + L::kVOff + c * 16384, &a.tm_v, &bars->kv_full, c * 64, g, krow);
                  ++kvc;
                }
                if (st >= (uint32_t)NO &&
                    !(ok = mbar_wait(&bars->o_empty[so], ((st / NO) - 1) & 1)))
                  break;
                uint8_t* os = sm + L::kOOff + so * L::kOBytes;
                mbar_arrive_expect_tx(&bars->o_full[so], L::kOBytes);
#pragma unroll
                for (int c = 0; c < DV / 64; ++c)
                  if (ATTN_CHECK(a, box_ok(a, &a.tm_do, c * 64, h, qrow, kQ), 0x7304))
                    tma_load_3d(os + c * 16384, &a.tm_do, &bars->o_full[so], c * 64, h, qrow);
                ++o_issued;
                ATTN_TL(2, st);
              }
            }
          }
        }
      }
      if (!ok) {
        report_timeout(a, 0x310);
        *abort_flag = 1;
      }
      if (*abort_flag) {
        if (kvc > 0) mbar_wait(&bars->kv_full, (kvc - 1) & 1, 100000000ull);
        for (uint32_t u = (q_issued > (uint32_t)NQ ? q_issued - NQ : 0u); u < q_issued; ++u)
          mbar_wait(&bars->q_full[u % NQ], (u / NQ) & 1, 100000000ull);
        for (uint32_t u = (o_issued > (uint32_t)NO ? o_issued - NO : 0u); u < o_issued; ++u)
          mbar_wait(&bars->o_full[u % NO], (u / NO) & 1, 100000000ull);
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ vector loader
    const int t = tid - 64;
    uint32_t st = 0;
    bool ok = true;
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) || !(ok = ring_pop(ring, rn, idx)) ||
          idx < 0)
        break;
      const DkdvItem w = dkdv_item(a, idx);
      for (int b = w.b0; b < w.b1 && ok; ++b) {
        for (int g = w.g0; g < w.g1 && ok; ++g) {
          int q_lo;
          const int nq = dkdv_q_tiles<kQ>(a, b, w.t, q_lo);
          for (int hh = 0; hh < G && ok && nq > 0; ++hh) {
            const int h = g * G + hh;
            for (int s = 0; s < nq; ++s, ++st) {
              const int stage = st % NV;
              float l2[2], dd[2];
#pragma unroll
              for (int r = 0; r < 2; ++r) {  // global loads ahead of the slot wait
                const int i = q_lo + s * kQ + t + 64 * r;
                const bool in = i < a.Sq;
                const int64_t vi = ((int64_t)b * a.Hq + h) * a.Sq + i;
                l2[r] = in ? a.lse2[vi] : INFINITY;
                dd[r] = in ? a.Dvec[vi] : 0.f;
              }
              if (st >= (uint32_t)NV &&
                  !(ok = mbar_wait_warp(&bars->vec_empty[stage], ((st / NV) - 1) & 1)))
                break;
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                vec[stage].nlse2[t + 64 * r] = -l2[r];
                vec[stage].D[t + 64 * r] = dd[r];
              }
              mbar_arrive(&bars->vec_full[stage]);
              if (lane == 0 && warp == 2) ATTN_TL(3, st);
            }
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x320 + warp);
      *abort_flag = 1;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop on warp-uniform values; one elected lane
    // issues each GEMM's MMAs from a single asm statement.
    constexpr uint32_t id_s = idesc_f32acc(E::kMmaFmt, 128, kQ, false, false);   // S^T, N = query
    constexpr uint32_t id_p = idesc_f32acc(E::kMmaFmt, 128, kQ, false, false);   // dP^T
    constexpr uint32_t id_dv = idesc_f32acc(E::kMmaFmt, 128, DV, false, true);   // dV, B = dO (MN)
    constexpr uint32_t id_dk = idesc_f32acc(E::kMmaFmt, 128, DQK, false, true);  // dK, B = Q (MN)
    const uint32_t tm = warp_uniform(tmem);
    const uint64_t k_km = sdesc_sw128(smem_u32(sm + L::kKOff), 16, 1024);
    const uint64_t v_km = sdesc_sw128(smem_u32(sm + L::kVOff), 16, 1024);
    const uint64_t q_km = sdesc_sw128(smem_u32(sm + L::kQOff), 16, 1024);
    const uint64_t q_mn = sdesc_sw128(smem_u32(sm + L::kQOff), 16384, 1024);
    const uint64_t o_km = sdesc_sw128(smem_u32(sm + L::kOOff), 16, 1024);
    const uint64_t o_mn = sdesc_sw128(smem_u32(sm + L::kOOff), 16384, 1024);
    uint32_t st = 0, kvc = 0, gc = 0;
    bool ok = true;
    auto qoff16 = [&](uint32_t x) -> uint32_t {
      return static_cast<uint32_t>(((x % NQ) * L::kQBytes) >> 4);
    };
    auto ooff16 = [&](uint32_t x) -> uint32_t {
      return static_cast<uint32_t>(((x % NO) * L::kOBytes) >> 4);
    };
    // dK += dS^T(x) Q(x): A = packed dS^T (query columns [0,64) at dP^T columns
    // [0,32), [64,128) at [64,96)), B = Q(x) MN-major; K = 128 query rows
    auto issue_dk = [&](uint32_t x, bool first) {
      mma_ts_warp<kQ / 16, 4, 8, 40, 128, 128>(tm + L::kColDK, tm + L::kColDP, q_mn + qoff16(x), id_dk,
                                            first ? 0u : 1u);
      mma_commit_warp(&bars->q_empty[x % NQ]);
    };
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) ||
          !(ok = ring_pop_warp1(ring, rn, idx)) || idx < 0)
        break;
      const DkdvItem w = dkdv_item(a, idx);
      for (int b = w.b0; b < w.b1 && ok; ++b) {
        for (int g = w.g0; g < w.g1 && ok; ++g) {
          int q_lo;
          const int nq = warp_uniform(dkdv_q_tiles<kQ>(a, b, w.t, q_lo));
          if (nq == 0) continue;
          const uint32_t nsteps = (uint32_t)nq * G;
          if (!(ok = mbar_wait_warp(&bars->kv_full, kvc & 1))) break;
          ++kvc;
          for (uint32_t u = 0; u < nsteps; ++u) {
            const uint32_t cur = st + u;
            if (!(ok = mbar_wait_warp(&bars->q_full[cur % NQ], (cur / NQ) & 1))) break;
            tc_fence_after();
            // S^T(cur) = K Q^T  (over P^T(cur-1), read by dV(cur-1) issued earlier)
            mma_ss_warp<DQK / 16, 4, 2, 1018, 2, 1018>(tm + L::kColS, k_km, q_km + qoff16(cur), id_s,
                                                    0u);
            mma_commit_warp(&bars->s_full);
            ATTN_TL(10, cur);
            if (u > 0) {  // dK(cur-1), once its dS^T is in tensor memory
              if (!(ok = mbar_wait_warp(&bars->ds_ready, (cur - 1) & 1))) break;
              tc_fence_after();
              issue_dk(cur - 1, u == 1);
              ATTN_TL(15, cur - 1);
            }
            if (!(ok = mbar_wait_warp(&bars->o_full[cur % NO], (cur / NO) & 1))) break;
            tc_fence_after();
            // dP^T(cur) = V dO^T  (over dS^T(cur-1), read by dK(cur-1) just issued)
            mma_ss_warp<DV / 16, 4, 2, 1018, 2, 1018>(tm + L::kColDP, v_km, o_km + ooff16(cur), id_p,
                                                   0u);
            mma_commit_warp(&bars->dp_full);
            ATTN_TL(11, cur);
            // dV += P^T(cur) dO(cur)
            if (!(ok = mbar_wait_warp(&bars->p_ready, cur & 1))) break;
            ATTN_TL(12, cur);
            if (u == 0 && gc > 0 && !(ok = mbar_wait_warp(&bars->acc_empty, (gc - 1) & 1))) break;
            tc_fence_after();
            mma_ts_warp<kQ / 16, 4, 8, 40, 128, 128>(tm + L::kColDV, tm + L::kColS, o_mn + ooff16(cur),
                                                  id_dv, u > 0 ? 1u : 0u);
            mma_commit_warp(&bars->o_empty[cur % NO]);
            ATTN_TL(13, cur);
          }
          if (!ok) break;
          // the group's last dK
          const uint32_t last = st + nsteps - 1;
          if (!(ok = mbar_wait_warp(&bars->ds_ready, last & 1))) break;
          tc_fence_after();
          issue_dk(last, nsteps == 1);
          mma_commit_warp(&bars->acc_full);
          mma_commit_warp(&bars->kv_empty);
          ++gc;
          st += nsteps;
        }
      }
    }
    if (!ok && lane == 0) {
      report_timeout(a, 0x330);
      *abort_flag = 1;
    }
    mma_commit_warp(&bars->drain);
    mbar_wait(&bars->drain, 0, 200000000ull);
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ P / dS warps
    // two warpgroups: thread (j, half) owns KV row j (TMEM lane j) and query
    // columns [64 half, 64 half + 64) of every step
    const int j = (tid - 128) & 127;
    const int half = (tid - 128) >> 7;
    const int c0h = half * 64;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int nqc = (a.Sq + kChunk - 1) / kChunk;
    uint32_t st = 0;
    bool ok = true;
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) || !(ok = ring_pop(ring, rn, idx)) ||
          idx < 0)
        break;
      const DkdvItem w = dkdv_item(a, idx);
      const int kj = w.t * kTile + j;
      const bool row_ok = kj < a.Skv;
      for (int b = w.b0; b < w.b1 && ok; ++b) {
        for (int g = w.g0; g < w.g1 && ok; ++g) {
          int q_lo;
          const int nq = dkdv_q_tiles<kQ>(a, b, w.t, q_lo);
          if (nq == 0) continue;
          const int64_t gk = (int64_t)b * a.Skv + kj;
          int qlo = 0, qhi = 0, my_id = 0, my_pos = 0;
          int2 my_qp = make_int2(0, -1);  // query positions that keep this key
          if (row_ok) {
            if (!general) {
              const int2 qr = band_queries_of_key(a, kj, a.kv_seg_lo[gk], a.kv_seg_hi[gk]);
              qlo = qr.x;
              qhi = qr.y;
            } else {
              my_id = a.kv_id[gk];
              my_pos = a.kv_pos[gk];
              my_qp = band_query_pos(a, my_pos);
            }
          }
          for (int hh = 0; hh < G && ok; ++hh) {
            const int h = g * G + hh;
            const int bb = a.bias_b > 1 ? b : 0, bh = a.bias_h > 1 ? h : 0;
            const int64_t bias_base = ((int64_t)bb * a.bias_h + bh) * a.Sq;
            for (int s = 0; s < nq; ++s, ++st) {
              const uint32_t cur = st;
              const int stage = cur % NV;
              const int q0 = q_lo + s * kQ;
              const int qh = q0 + c0h;  // first query row of this thread's columns
              if (j == 0 && half == 0) ATTN_TL(20, cur);
              uint64_t vbits;
              if (!general) {
                vbits = row_ok ? range_bits64(qlo - qh, qhi - qh) : 0ull;
              } else {
                vbits = 0ull;
                bool known = false;  // decided by the query chunk's summary
                if (row_ok && my_id != 0 && qh < a.Sq && (qh % kChunk) == 0)
                  known = chunk_bits(a.q_chunk[b * nqc + qh / kChunk], my_id, my_qp, vbits);
                if (!known && row_ok && my_id != 0) {
                  // per-token compare; every lane of the warp reads the same query row
                  const int32_t* qid = a.q_id + (int64_t)b * a.Sq;
                  const int32_t* qps = a.q_pos + (int64_t)b * a.Sq;
                  const int n = min(64, a.Sq - qh);
                  for (int c = 0; c < n; ++c) {
                    const int pq = __ldg(qps + qh + c);
                    const bool v = (__ldg(qid + qh + c) == my_id) & (pq >= my_qp.x) & (pq <= my_qp.y);
                    vbits |= static_cast<uint64_t>(v) << c;
                  }
                }
              }
              if (!(ok = mbar_wait_warp(&bars->vec_full[stage], (cur / NV) & 1))) break;
              const Vec128& V = vec[stage];
              if (!(ok = mbar_wait_warp(&bars->s_full, cur & 1))) break;
              if (j == 0 && half == 0) ATTN_TL(21, cur);
              tc_fence_after();
              const uint32_t s_tm = tmem + lane_base + L::kColS + c0h;
              // P^T in two 32-column chunks; packed bf16 pairs go back over this
              // thread's own S^T columns (chunk q at packed columns [16 q, 16 q + 16))
              uint32_t pp[32];  // packed P of all 64 columns, kept for dS
              bool none[2];     // warp-uniform: no valid pair in the 32-column chunk
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const uint32_t m32 = static_cast<uint32_t>(vbits >> (q * 32));
                none[q] = __all_sync(0xffffffffu, m32 == 0u);
                const bool all = __all_sync(0xffffffffu, m32 == 0xffffffffu);
                uint32_t pk[16];
                if (none[q]) {
#pragma unroll
                  for (int e = 0; e < 16; ++e) pk[e] = 0u;
                } else {
                  uint32_t u[32];
                  tmem_ld32x32b_x32(s_tm + q * 32, u);
                  tmem_ld_wait(u);
                  float x[32];
                  if (HAS_BIAS) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(u[e]) * a.scale_log2;
                    if (row_ok) {
                      const bf16* bp = a.bias + (bias_base + qh + q * 32) * a.Skv + kj;
#pragma unroll
                      for (int c = 0; c < 32; ++c)
                        if (qh + q * 32 + c < a.Sq)
                          x[c] += E::ld(bp + (int64_t)c * a.Skv) * kLog2e;
                    }
                  }
#pragma unroll
                  for (int c = 0; c < 32; c += 4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(&V.nlse2[c0h + q * 32 + c]);
                    if (HAS_BIAS) {
                      const float nl[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                      for (int e = 0; e < 4; ++e) x[c + e] = ex2_approx(x[c + e] + nl[e]);
                    } else {
                      // x * scale - lse, two columns per instruction
                      const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
                      const float2 y0 = fma_f32x2(
                          make_float2(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), sc2,
                          make_float2(l4.x, l4.y));
                      const float2 y1 = fma_f32x2(
                          make_float2(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])), sc2,
                          make_float2(l4.z, l4.w));
                      x[c] = ex2_approx(y0.x);
                      x[c + 1] = ex2_approx(y0.y);
                      x[c + 2] = ex2_approx(y1.x);
                      x[c + 3] = ex2_approx(y1.y);
                    }
                  }
                  if (!all) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = (m32 & (1u << e)) ? x[e] : 0.f;
                  }
#pragma unroll
                  for (int e = 0; e < 16; ++e) pk[e] = E::pack(x[2 * e], x[2 * e + 1]);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) pp[q * 16 + e] = pk[e];
                tmem_st32x32b_x16(s_tm + q * 16, pk);
              }
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive(&bars->p_ready);
              if (j == 0 && half == 0) ATTN_TL(22, cur);
              // dS^T = P^T (dP^T - D), packed bf16 back over this thread's dP^T columns
              if (!(ok = mbar_wait_warp(&bars->dp_full, cur & 1))) break;
              if (j == 0 && half == 0) ATTN_TL(23, cur);
              tc_fence_after();
              const uint32_t dp_tm = tmem + lane_base + L::kColDP + c0h;
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                if (none[q]) {  // P = 0, so dS = 0
                  uint32_t pk[16];
#pragma unroll
                  for (int e = 0; e < 16; ++e) pk[e] = 0u;
                  tmem_st32x32b_x16(dp_tm + q * 16, pk);
                  // a per-slice dBias already holds zeros; a summed one still
                  // needs its first store or last write of these rows
                  if (DBIAS == 2 && row_ok &&
                      ATTN_CHECK(a, dbias_ok(a, bias_base + qh + q * 32, kj) &&
                                        dbias_ok(a, bias_base + min(qh + q * 32 + 31, a.Sq - 1), kj),
                                 0x7309)) {
                    float zero[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) zero[c] = 0.f;
                    dbias_acc_rows<E>(a, bias_base + qh + q * 32, kj, qh + q * 32,
                                      dbias_rows_written_before<kQ>(a, w.b0, b, w.g0, g, hh, w.t, qh + q * 32),
                                      dbias_rows_written_after<kQ>(a, b, w.b1, g, w.g1, hh, G, w.t, qh + q * 32),
                                      zero);
                  }
                  continue;
                }
                uint32_t u[32];
                tmem_ld32x32b_x32(dp_tm + q * 32, u);
                tmem_ld_wait(u);
                uint32_t pk[16];
                if (DBIAS == 0) {
                  // dP - D in fp32, then one packed bf16 product with P (already
                  // bf16): the product's rounding is the one dS gets anyway
#pragma unroll
                  for (int e = 0; e < 32; e += 4) {
                    const float4 d4 = *reinterpret_cast<const float4*>(&V.D[c0h + q * 32 + e]);
                    const float2 g0 = sub_f32x2(
                        make_float2(__uint_as_float(u[e]), __uint_as_float(u[e + 1])),
                        make_float2(d4.x, d4.y));
                    const float2 g1 = sub_f32x2(
                        make_float2(__uint_as_float(u[e + 2]), __uint_as_float(u[e + 3])),
                        make_float2(d4.z, d4.w));
                    pk[e / 2] = E::mul(pp[q * 16 + e / 2], E::pack(g0.x, g0.y));
                    pk[e / 2 + 1] = E::mul(pp[q * 16 + e / 2 + 1], E::pack(g1.x, g1.y));
                  }
                  tmem_st32x32b_x16(dp_tm + q * 16, pk);
                  continue;
                }
                float ds[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                  const float4 d4 = *reinterpret_cast<const float4*>(&V.D[c0h + q * 32 + e]);
                  const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    const uint32_t w2 = pp[q * 16 + (e + k) / 2];
                    const float pv = ((e + k) & 1) ? E::hi(w2) : E::lo(w2);
                    ds[e + k] = pv * (__uint_as_float(u[e + k]) - dd[k]);
                  }
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = E::pack(ds[2 * e], ds[2 * e + 1]);
                tmem_st32x32b_x16(dp_tm + q * 16, pk);
                if (DBIAS != 0 && row_ok &&
                    ATTN_CHECK(a, dbias_ok(a, bias_base + qh + q * 32, kj) &&
                                      dbias_ok(a, bias_base + min(qh + q * 32 + 31, a.Sq - 1), kj),
                               0x7305)) {
                  if (DBIAS == 1) {
                    bf16* dpb = a.dbias + (bias_base + qh + q * 32) * a.Skv + kj;
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                      if (qh + q * 32 + c < a.Sq) E::st(dpb + (int64_t)c * a.Skv, ds[c]);
                  } else {
                    dbias_acc_rows<E>(a, bias_base + qh + q * 32, kj, qh + q * 32,
                                      dbias_rows_written_before<kQ>(a, w.b0, b, w.g0, g, hh, w.t, qh + q * 32),
                                      dbias_rows_written_after<kQ>(a, b, w.b1, g, w.g1, hh, G, w.t, qh + q * 32),
                                      ds);
                  }
                }
              }
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive(&bars->ds_ready);
              if (j == 0 && half == 0) ATTN_TL(24, cur);
              mbar_arrive(&bars->vec_empty[stage]);
            }
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x340 + (warp & 7));
      *abort_flag = 1;
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dK/dV epilogue
    const int j = tid - 384;  // TMEM lane = KV row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t gc = 0;
    bool ok = true;
    for (uint32_t rn = 0;; ++rn) {
      int32_t idx;
      if (!ok || __any_sync(0xffffffffu, *abort_flag != 0) || !(ok = ring_pop(ring, rn, idx)) ||
          idx < 0)
        break;
      const DkdvItem w = dkdv_item(a, idx);
      const int kj = w.t * kTile + j;
      const bool row_ok = kj < a.Skv;
      for (int b = w.b0; b < w.b1 && ok; ++b) {
        for (int g = w.g0; g < w.g1 && ok; ++g) {
          int q_lo;
          const int nq = dkdv_q_tiles<kQ>(a, b, w.t, q_lo);
          bf16* dv_row = a.dv + ((int64_t)b * a.Skv + kj) * a.dv_stride + (int64_t)g * DV;
          bf16* dk_row = a.dk + ((int64_t)b * a.Skv + kj) * a.dk_stride + (int64_t)g * DQK;
          if (nq == 0) {
            if (row_ok && ATTN_CHECK(a, dv_span_ok(a, (int64_t)b * a.Skv + kj, (int64_t)g * DV, DV, dv_row, 16) &&
                                            dk_span_ok(a, (int64_t)b * a.Skv + kj, (int64_t)g * DQK, DQK, dk_row, 16),
                                     0x7306)) {
#pragma unroll
              for (int c = 0; c < DV; c += 8)
                *reinterpret_cast<uint4*>(dv_row + c) = make_uint4(0, 0, 0, 0);
#pragma unroll
              for (int c = 0; c < DQK; c += 8)
                *reinterpret_cast<uint4*>(dk_row + c) = make_uint4(0, 0, 0, 0);
            }
            continue;
          }
          if (!(ok = mbar_wait_warp(&bars->acc_full, gc & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < DV / 32; ++q) {
            uint32_t u[32];
            tmem_ld32x32b_x32(tmem + lane_base + L::kColDV + q * 32, u);
            tmem_ld_wait(u);
            if (row_ok) {
#pragma unroll
              for (int c = 0; c < 32; c += 16) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  w[e] = E::pack(__uint_as_float(u[c + 2 * e]), __uint_as_float(u[c + 2 * e + 1]));
                if (ATTN_CHECK(a, dv_span_ok(a, (int64_t)b * a.Skv + kj, (int64_t)g * DV + q * 32 + c, 16,
                                             dv_row + q * 32 + c, a.grad_st32 ? 32 : 16), 0x7307))
                  store16_elems(dv_row + q * 32 + c, w, a.grad_st32 != 0);
              }
            }
          }
#pragma unroll
          for (int q = 0; q < DQK / 32; ++q) {
            uint32_t u[32];
            tmem_ld32x32b_x32(tmem + lane_base + L::kColDK + q * 32, u);
            tmem_ld_wait(u);
            if (row_ok) {
              const float sc = a.scale;
#pragma unroll
              for (int c = 0; c < 32; c += 16) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  w[e] = E::pack(__uint_as_float(u[c + 2 * e]) * sc, __uint_as_float(u[c + 2 * e + 1]) * sc);
                if (ATTN_CHECK(a, dk_span_ok(a, (int64_t)b * a.Skv + kj, (int64_t)g * DQK + q * 32 + c, 16,
                                             dk_row + q * 32 + c, a.grad_st32 ? 32 : 16), 0x7308))
                  store16_elems(dk_row + q * 32 + c, w, a.grad_st32 != 0);
              }
            }
          }
          tc_fence_before();
          mbar_arrive(&bars->acc_empty);
          ++gc;
        }
      }
    }
    if (!ok) {
      if (lane == 0) report_timeout(a, 0x350 + (warp & 3));
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

template <class E, int DQK, int DV, bool HB, int DB>
cudaError_t go(const KernelArgs& a, int nsm, cudaStream_t st) {
  using L = D128Layout<DQK, DV>;
  auto kern = dkdv128_kernel<E, DQK, DV, HB, DB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int nb = a.dkdv_batch_loop ? 1 : a.B, ng = a.dkdv_head_loop ? 1 : a.Hkv;
  const int items = a.n_kt * nb * ng;
  const int grid = items < nsm ? items : nsm;
  kern<<<grid, 512, L::kAlloc, st>>>(a);
  return cudaGetLastError();
}

template <class E, int DQK, int DV>
cudaError_t go_bias_e(const KernelArgs& a, int nsm, cudaStream_t st) {
  if (!a.bias) return go<E, DQK, DV, false, 0>(a, nsm, st);
  if (a.dbias_mode == 0) return go<E, DQK, DV, true, 0>(a, nsm, st);
  if (a.dbias_mode == 1) return go<E, DQK, DV, true, 1>(a, nsm, st);
  return go<E, DQK, DV, true, 2>(a, nsm, st);
}

template <int DQK, int DV>
cudaError_t go_bias(const KernelArgs& a, int nsm, cudaStream_t st) {
  return a.elem_f16 ? go_bias_e<ElemF16, DQK, DV>(a, nsm, st)
                    : go_bias_e<ElemBf16, DQK, DV>(a, nsm, st);
}

}  // namespace

cudaError_t launch_bwd_dkdv128(const KernelArgs& a, int nsm, cudaStream_t st) {
  if (a.d_qk == 64 && a.d_v == 64) return go_bias<64, 64>(a, nsm, st);
  if (a.d_qk == 64 && a.d_v == 128) return go_bias<64, 128>(a, nsm, st);
  if (a.d_qk == 128 && a.d_v == 64) return go_bias<128, 64>(a, nsm, st);
  if (a.d_qk == 128 && a.d_v == 128) return go_bias<128, 128>(a, nsm, st);
  return cudaErrorInvalidValue;
}

}  // namespace attn

#ifdef ATTN_TIMELINE
// Debug builds only: timeline of this translation unit's kernels.
extern "C" int attn_debug_timeline128(unsigned long long* out, int cap) {
  cudaDeviceSynchronize();
  const int n = cap < attn::kTimelineCap ? cap : attn::kTimelineCap;
  cudaMemcpyFromSymbol(out, attn::g_timeline, sizeof(unsigned long long) * n);
  static unsigned long long zeros[attn::kTimelineCap];
  cudaMemcpyToSymbol(attn::g_timeline, zeros, sizeof(zeros));
  return n;
}
#endif
