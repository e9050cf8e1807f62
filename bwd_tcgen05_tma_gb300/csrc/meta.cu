// Segment-metadata kernels: normalise the caller's sequence description into
// per-token (id, position) arrays, decide between the fast (segment-boundary)
// and general (per-token comparison) masking paths, and derive the tile ranges
// the attention kernels iterate over.
//
// The fast path is taken only when Q and KV describe the same tokens (same ids
// and same positions) and positions restart at 0 and count up inside every
// segment; otherwise, or when forced, the general path compares ids and
// positions token by token (TransformerEngine PR #3516, Changes 3-4: the
// boundary-only fast path assumes matching Q/KV metadata; equal-length
// cross-attention with independent metadata takes the general path).  When
// segment positions are absent they are derived from the ids as the offset
// inside each run of equal ids (PR #2692, Description: from_segment_ids_and_pos).
#include <algorithm>
#include <climits>

#include "attn_internal.cuh"

namespace attn {
namespace {

constexpr int kMetaThreads = 1024;

__device__ __forceinline__ int warp_incl_max(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = max(v, n);
  }
  return v;
}

__device__ __forceinline__ int warp_incl_min_rev(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_down_sync(0xffffffffu, v, o);
    if (lane + o < 32) v = min(v, n);
  }
  return v;
}

// Block-wide inclusive prefix max (forward) over blockDim.x == 1024 values.
__device__ int block_prefix_max(int v, int* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_incl_max(v);
  if (lane == 31) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    int t = sh[lane];
    t = warp_incl_max(t);
    sh[lane] = t;
  }
  __syncthreads();
  if (w > 0) v = max(v, sh[w - 1]);
  __syncthreads();
  return v;
}

// Block-wide inclusive suffix min.
__device__ int block_suffix_min(int v, int* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_incl_min_rev(v);
  if (lane == 0) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    int t = sh[lane];
    t = warp_incl_min_rev(t);
    sh[lane] = t;
  }
  __syncthreads();
  if (w < 31) v = min(v, sh[w + 1]);
  __syncthreads();
  return v;
}

__device__ int token_id(int fmt, const int32_t* ids, const int32_t* cu, int nseg, int b, int S,
                        int t) {
  if (fmt == 2) {  // ragged offsets: segment k holds cu[k] <= t < cu[k+1]
    int lo = 0, hi = nseg;  // find largest k in [0, nseg] with cu[k] <= t
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return (lo < nseg && t < __ldg(cu + lo + 1)) ? lo + 1 : 0;
  }
  if (ids == nullptr) return 1;
  return __ldg(ids + (int64_t)b * S + t);
}

// Token id of batch row b, token t (or INT_MIN before the row start).
__device__ __forceinline__ int id_at(const int32_t* id_row, int t) {
  return t >= 0 ? id_row[t] : INT_MIN;
}

// All passes run in one cooperative kernel of 1024-thread blocks, separated
// by grid-wide barriers; every pass strides over its work units, so the grid
// only has to fit on the GPU at once (which the cooperative launch checks).
//
//   pass 1  per 1024-token block of each row and side: normalised ids, and
//           the block's first and last run boundary (a boundary is a token
//           whose id differs from its predecessor's, or token 0);
//   pass 2  same blocks: run starts / ends from block scans plus the
//           boundaries of the other blocks; positions (given, or derived as
//           the offset inside the run); fast-path segment bounds; flags
//           positions that do not restart at 0 and count up in a segment;
//   pass 3  Q/KV equality per token (Sq == Skv only) and the 64-token chunk
//           summaries of both sides;
//   pass 4  per 128-row tile the token range of the other side it may meet,
//           and the path decision.

// Grid-wide barrier number k (1, 2, ...) over the header's arrival counter,
// which is zero when the kernel starts.  Thread 0 of each block publishes the
// block's writes (the fence after the block barrier is cumulative), arrives,
// and waits with acquire loads until every block has arrived k times.  The
// wait is bounded: after 2 s it records a timeout and every thread of the
// block gets false, so the kernel returns instead of hanging.
__device__ bool grid_barrier(const KernelArgs& a, unsigned k, int* flag_sh) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&a.hdr->meta_barrier, 1u);
    const unsigned target = k * gridDim.x;
    int ok = 1;
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&a.hdr->meta_barrier) : "memory");
    if (v < target) {
      const uint64_t t0 = sm103::globaltimer_ns();
      for (uint32_t it = 1;; ++it) {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&a.hdr->meta_barrier) : "memory");
        if (v >= target) break;
        if ((it & 63u) == 0u && sm103::globaltimer_ns() - t0 > 2000000000ull) {
          report_timeout(a, 0x300 + static_cast<int>(k));
          ok = 0;
          break;
        }
      }
    }
    *flag_sh = ok;
  }
  __syncthreads();
  return *flag_sh != 0;
}

struct MetaIn {
  int fmt;  // 0 dense rows or per-token ids, 1 per-token ids, 2 ragged offsets
  const int32_t* q_ids;
  const int32_t* q_pos;
  const int32_t* kv_ids;
  const int32_t* kv_pos;
  const int32_t* cu_q;
  const int32_t* cu_kv;
  int nseg;
  int force_general;
  int fast_reason;
  int nblk;  // 1024-token blocks of the longer side
};

constexpr int kOrderBins = kMetaThreads;  // tile counts 0 .. kOrderBins - 1 (larger ones clamp)

struct MetaShared {
  int sh[32];
  int shl[32];
  int carry_start, carry_end;
  int flag;
  int bins[kOrderBins];
};

// Pass 1 for one (block, row, side) unit.
__device__ void meta_ids_unit(const KernelArgs& a, const MetaIn& in, int blk, int b, bool kvside,
                              int2* bounds, MetaShared& sm) {
  const int S = kvside ? a.Skv : a.Sq;
  const int c0 = blk * kMetaThreads;
  if (c0 >= S) return;  // uniform over the block
  const int32_t* ids = kvside ? in.kv_ids : in.q_ids;
  const int32_t* cu = kvside ? in.cu_kv : in.cu_q;
  int32_t* id_out = const_cast<int32_t*>(kvside ? a.kv_id : a.q_id) + (int64_t)b * S;
  const int t = c0 + threadIdx.x;
  int first = INT_MAX, last = -1;
  if (t < S) {
    const int id = token_id(in.fmt, ids, cu, in.nseg, b, S, t);
    id_out[t] = id;
    const bool bnd = (t == 0) || (token_id(in.fmt, ids, cu, in.nseg, b, S, t - 1) != id);
    if (bnd) first = last = t;
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) {
    first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
    last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  }
  if (lane == 0) { sm.sh[w] = first; sm.shl[w] = last; }
  __syncthreads();
  if (w == 0) {
    first = sm.sh[lane];
    last = sm.shl[lane];
    for (int o = 16; o > 0; o >>= 1) {
      first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
      last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    }
    if (lane == 0) bounds[((int)kvside * a.B + b) * in.nblk + blk] = make_int2(first, last);
  }
  __syncthreads();  // sm.sh is reused by the next unit
}

// Pass 2 for one (block, row, side) unit.
__device__ void meta_pos_unit(const KernelArgs& a, const MetaIn& in, int blk, int b, bool kvside,
                              const int2* bounds, MetaShared& sm) {
  const int S = kvside ? a.Skv : a.Sq;
  const int c0 = blk * kMetaThreads;
  if (c0 >= S) return;  // uniform over the block
  const int32_t* ids = kvside ? in.kv_ids : in.q_ids;
  const int32_t* pos_in = kvside ? in.kv_pos : in.q_pos;
  const int32_t* id_row = (kvside ? a.kv_id : a.q_id) + (int64_t)b * S;
  int32_t* pos_out = const_cast<int32_t*>(kvside ? a.kv_pos : a.q_pos) + (int64_t)b * S;
  int32_t* lo_out = const_cast<int32_t*>(kvside ? a.kv_seg_lo : a.seg_lo) + (int64_t)b * S;
  int32_t* hi_out = const_cast<int32_t*>(kvside ? a.kv_seg_hi : a.seg_hi) + (int64_t)b * S;
  const int2* bd = bounds + ((int)kvside * a.B + b) * in.nblk;
  if (threadIdx.x == 0) {
    int cs = 0;  // last boundary before this block (token 0 always is one)
    for (int k = blk - 1; k >= 0; --k)
      if (bd[k].y >= 0) { cs = bd[k].y; break; }
    int ce = S;  // first boundary after this block
    const int nb = (S + kMetaThreads - 1) / kMetaThreads;
    for (int k = blk + 1; k < nb; ++k)
      if (bd[k].x != INT_MAX) { ce = bd[k].x; break; }
    sm.carry_start = cs;
    sm.carry_end = ce;
  }
  const int t = c0 + threadIdx.x;
  int id = 0, start_c = -1, end_c = INT_MAX;
  if (t < S) {
    id = id_row[t];
    if (t == 0 || id_at(id_row, t - 1) != id) start_c = t;
    if (t + 1 < S && id_row[t + 1] != id) end_c = t + 1;
  }
  int start = block_prefix_max(start_c, sm.sh);
  int end = block_suffix_min(end_c, sm.sh);
  if (t < S) {
    if (start < 0) start = sm.carry_start;
    if (end == INT_MAX) end = (t + 1 >= S) ? S : sm.carry_end;
  }
  int nonstd = 0;
  if (t < S) {
    int pos;
    if (in.fmt == 2 || pos_in == nullptr) pos = (ids == nullptr && in.fmt != 2) ? t : t - start;
    else pos = __ldg(pos_in + (int64_t)b * S + t);
    pos_out[t] = pos;
    if (id != 0 && pos != t - start) nonstd = 1;
    lo_out[t] = id != 0 ? start : 0;
    hi_out[t] = id != 0 ? end : 0;
  }
  // also orders this unit's reads of carry_start/end before the next unit's
  // thread 0 rewrites them
  if (__syncthreads_or(nonstd) && threadIdx.x == 0) atomicOr(&a.hdr->mismatch, 4);
}

// Summary of one 64-token chunk computed by a warp (two tokens per lane).
__device__ ChunkInfo chunk_info_warp(const int32_t* id, const int32_t* pos, int S, int c0) {
  const int lane = threadIdx.x & 31;
  int mn = INT_MAX, mx = 0, pmn = INT_MAX, pmx = INT_MIN, has0 = 0;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int t = c0 + lane + 32 * k;
    if (t < S) {
      const int i = id[t];
      if (i == 0) {
        has0 = 1;
      } else {
        mn = min(mn, i);
        mx = max(mx, i);
        pmn = min(pmn, pos[t]);
        pmx = max(pmx, pos[t]);
      }
    } else {
      has0 = 1;  // a chunk that runs past the row end is never uniform
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    pmn = min(pmn, __shfl_xor_sync(0xffffffffu, pmn, o));
    pmx = max(pmx, __shfl_xor_sync(0xffffffffu, pmx, o));
    has0 |= __shfl_xor_sync(0xffffffffu, has0, o);
  }
  ChunkInfo ci;
  ci.min_id = mn;
  ci.max_id = mx;
  ci.min_pos = pmn;
  ci.max_pos = pmx;
  ci.uniform = (!has0 && mx != 0 && mn == mx) ? 1 : 0;
  // consecutive positions: token c0 + k at min_pos + k (read only when uniform,
  // so every token exists)
  bool cons = true;
  if (ci.uniform) {
#pragma unroll
    for (int k = 0; k < 2; ++k) cons &= pos[c0 + lane + 32 * k] == pmn + lane + 32 * k;
  }
  ci.consec = (__all_sync(0xffffffffu, cons) && ci.uniform) ? 1 : 0;
  ci.pad[0] = ci.pad[1] = 0;
  return ci;
}

// Pass 3: Q/KV equality per token (grid-stride over tokens) and the chunk
// summaries (one warp per chunk).
__device__ void meta_match_chunks(const KernelArgs& a) {
  if (a.Sq == a.Skv) {
    const int64_t n = (int64_t)a.B * a.Sq;
    int bits = 0;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n;
         t += (int64_t)gridDim.x * blockDim.x) {
      if (a.q_id[t] != a.kv_id[t]) bits |= 1;
      if (a.q_pos[t] != a.kv_pos[t]) bits |= 2;
    }
    bits = __reduce_or_sync(0xffffffffu, bits);
    if ((threadIdx.x & 31) == 0 && bits) atomicOr(&a.hdr->mismatch, bits);
  }
  const int nqc = (a.Sq + kChunk - 1) / kChunk, nkc = (a.Skv + kChunk - 1) / kChunk;
  const int total = a.B * (nqc + nkc);
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int w = wid; w < total; w += nw) {
    ChunkInfo ci;
    if (w < a.B * nqc) {
      const int b = w / nqc, c = w % nqc;
      ci = chunk_info_warp(a.q_id + (int64_t)b * a.Sq, a.q_pos + (int64_t)b * a.Sq, a.Sq,
                           c * kChunk);
      if ((threadIdx.x & 31) == 0) const_cast<ChunkInfo*>(a.q_chunk)[w] = ci;
    } else {
      const int w2 = w - a.B * nqc;
      const int b = w2 / nkc, c = w2 % nkc;
      ci = chunk_info_warp(a.kv_id + (int64_t)b * a.Skv, a.kv_pos + (int64_t)b * a.Skv, a.Skv,
                           c * kChunk);
      if ((threadIdx.x & 31) == 0) const_cast<ChunkInfo*>(a.kv_chunk)[w2] = ci;
    }
  }
}

__device__ __forceinline__ bool ids_meet(const ChunkInfo& x, int lo, int hi) {
  return x.max_id != 0 && x.min_id <= hi && lo <= x.max_id;
}

__device__ __forceinline__ int warp_min(int v) {
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_max(int v) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Pass 4: per 128-row query tile the KV token range it may attend to; per
// 128-row KV tile the query token range that may attend to it.  One warp per
// tile.
__device__ void meta_ranges(const KernelArgs& a, const MetaIn& in) {
  const int mism = *reinterpret_cast<const volatile int32_t*>(&a.hdr->mismatch);
  const bool general = in.force_general || a.Sq != a.Skv || (mism & 7) != 0;
  const int nqc = (a.Sq + kChunk - 1) / kChunk, nkc = (a.Skv + kChunk - 1) / kChunk;
  const int totq = a.B * a.n_qt, totk = a.B * a.n_kt;
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.hdr->path = general ? 1 : 0;
    int reason;
    if (in.force_general) reason = 2;
    else if (a.Sq != a.Skv) reason = 3;
    else if (mism & 1) reason = in.fmt == 2 ? 7 : 4;
    else if (mism & 2) reason = in.fmt == 2 ? 7 : 5;
    else if (mism & 4) reason = 6;
    else reason = in.fast_reason;  // dense rows or matching metadata
    a.hdr->reason = reason;
  }
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int w = wid; w < totq + totk; w += nw) {
    const bool qside = w < totq;
    const int w2 = qside ? w : w - totq;
    const int nt = qside ? a.n_qt : a.n_kt;
    const int b = w2 / nt, t = w2 % nt;
    const int S_own = qside ? a.Sq : a.Skv, S_oth = qside ? a.Skv : a.Sq;
    const int r0 = t * kTile, r1 = min(S_own, r0 + kTile);
    int lo = INT_MAX, hi = 0;
    if (!general) {
      // rows of this tile; Sq == Skv and the two sides' metadata are equal here
      const int32_t* slo = qside ? a.seg_lo : a.kv_seg_lo;
      const int32_t* shi = qside ? a.seg_hi : a.kv_seg_hi;
      for (int i = r0 + lane; i < r1; i += 32) {
        const int64_t g = (int64_t)b * S_own + i;
        const int sl = slo[g], sh = shi[g];
        if (sh <= sl) continue;
        const int2 r = qside ? band_keys_of_query(a, i, sl, sh) : band_queries_of_key(a, i, sl, sh);
        if (r.y <= r.x) continue;
        lo = min(lo, r.x);
        hi = max(hi, r.y);
      }
    } else {
      const ChunkInfo* own = qside ? a.q_chunk : a.kv_chunk;
      const ChunkInfo* oth = qside ? a.kv_chunk : a.q_chunk;
      const int nown = qside ? nqc : nkc, noth = qside ? nkc : nqc;
      int ilo = INT_MAX, ihi = 0, plo = INT_MAX, phi = INT_MIN;
      for (int c = r0 / kChunk + lane; c * kChunk < r1; c += 32) {
        const ChunkInfo ci = own[b * nown + c];
        if (ci.max_id == 0) continue;
        ilo = min(ilo, ci.min_id);
        ihi = max(ihi, ci.max_id);
        plo = min(plo, ci.min_pos);
        phi = max(phi, ci.max_pos);
      }
      ilo = warp_min(ilo);
      ihi = warp_max(ihi);
      plo = warp_min(plo);
      phi = warp_max(phi);
      if (ihi != 0) {
        // positions of the other side that the band admits for this tile's
        // positions [plo, phi] (a chunk outside them has no valid pair here)
        const int2 ox = qside ? band_key_pos(a, plo) : band_query_pos(a, plo);
        const int2 oy = qside ? band_key_pos(a, phi) : band_query_pos(a, phi);
        const int want_lo = ox.x, want_hi = oy.y;
        for (int c = lane; c < noth; c += 32) {
          const ChunkInfo co = oth[b * noth + c];
          if (ids_meet(co, ilo, ihi) && co.max_pos >= want_lo && co.min_pos <= want_hi) {
            lo = min(lo, c * kChunk);
            hi = max(hi, min(S_oth, (c + 1) * kChunk));
          }
        }
      }
    }
    lo = warp_min(lo);
    hi = warp_max(hi);
    if (lane == 0 &&
        ATTN_CHECK(a, span_ok(w2, 1, (int64_t)a.B * (qside ? a.n_qt : a.n_kt)), 0x7801) &&
        ATTN_CHECK(a, hi <= lo || (lo >= 0 && hi <= S_oth), 0x7802)) {
      const int2 r = (hi > lo) ? make_int2(lo, hi) : make_int2(0, 0);
      if (qside) {
        const_cast<int2*>(a.q_tile_range)[w2] = r;
        if (r.y > r.x)
          atomicAdd(reinterpret_cast<unsigned long long*>(&a.hdr->tile_pairs),
                    (unsigned long long)((r.y - r.x + kTile - 1) / kTile));
      } else {
        const_cast<int2*>(a.kv_tile_range)[w2] = r;
      }
    }
  }
}

// Pass 5, run by the last block to finish pass 4: the query tiles in order
// of decreasing KV-tile count (a counting sort; the order among equal counts
// is not fixed and does not matter).  The persistent passes over query tiles
// map their claim counter through it, so the longest items go out first and
// the end of the grid is made of short ones.
__device__ void meta_order(const KernelArgs& a, MetaShared& sm) {
  const int n = a.B * a.n_qt;
  auto key = [&](int w) -> int {
    const int2 r = __ldcg(a.q_tile_range + w);  // written by other blocks: from L2
    const int c = (r.y > r.x) ? (r.y - r.x + kTile - 1) / kTile : 0;
    return min(c, kOrderBins - 1);
  };
  sm.bins[threadIdx.x] = 0;
  __syncthreads();
  for (int w = threadIdx.x; w < n; w += blockDim.x) atomicAdd(&sm.bins[key(w)], 1);
  __syncthreads();
  // start of each count's run: thread i owns count kOrderBins - 1 - i, so an
  // exclusive prefix sum in thread order runs over decreasing counts
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int mine = sm.bins[kOrderBins - 1 - threadIdx.x];
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sm.sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int t = sm.sh[lane];
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += v;
    }
    sm.shl[lane] = ti - t;  // exclusive over warps
  }
  __syncthreads();
  const int start = sm.shl[warp] + incl - mine;
  __syncthreads();
  sm.bins[kOrderBins - 1 - threadIdx.x] = start;
  __syncthreads();
  int32_t* out = const_cast<int32_t*>(a.q_order);
  for (int w = threadIdx.x; w < n; w += blockDim.x) {
    const int pos = atomicAdd(&sm.bins[key(w)], 1);
    if (ATTN_CHECK(a, span_ok(pos, 1, n), 0x7803)) out[pos] = w;
  }
}

__global__ void __launch_bounds__(kMetaThreads) meta_kernel(const KernelArgs a, const MetaIn in) {
  __shared__ MetaShared sm;
  sm103::grid_dep_launch();  // the forward may be scheduled now; it waits for this grid to finish
  if (a.max_logit) {  // the forward folds its row maxima into these
    const int n = a.B * a.Hq;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < n; t += gridDim.x * blockDim.x)
      a.max_logit[t] = -INFINITY;
  }
  int2* bounds = const_cast<int2*>(a.meta_scan);
  const int units = in.nblk * a.B * 2;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int blk = u % in.nblk, rest = u / in.nblk;
    meta_ids_unit(a, in, blk, rest % a.B, rest >= a.B, bounds, sm);
  }
  if (!grid_barrier(a, 1, &sm.flag)) return;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int blk = u % in.nblk, rest = u / in.nblk;
    meta_pos_unit(a, in, blk, rest % a.B, rest >= a.B, bounds, sm);
  }
  if (!grid_barrier(a, 2, &sm.flag)) return;
  meta_match_chunks(a);
  if (!grid_barrier(a, 3, &sm.flag)) return;
  meta_ranges(a, in);
  // the last block past pass 4 sees every tile range and orders the tiles
  __threadfence();  // this thread's ranges reach L2 before the block counts itself done
  __syncthreads();
  if (threadIdx.x == 0)
    sm.flag = (atomicAdd(&a.hdr->meta_done, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (sm.flag) {
    __threadfence();
    meta_order(a, sm);
  }
}

int meta_max_blocks() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int per_sm = 0, nsm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, meta_kernel, kMetaThreads, 0) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  const int n = per_sm * nsm;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

}  // namespace

cudaError_t launch_meta(const KernelArgs& a, int fmt, const int32_t* q_ids, const int32_t* q_pos,
                        const int32_t* kv_ids, const int32_t* kv_pos, const int32_t* cu_q,
                        const int32_t* cu_kv, int num_segments, int force_general,
                        cudaStream_t st) {
  MetaIn in;
  in.fmt = fmt;
  in.q_ids = q_ids;
  in.q_pos = q_pos;
  in.kv_ids = kv_ids;
  in.kv_pos = kv_pos;
  in.cu_q = cu_q;
  in.cu_kv = cu_kv;
  in.nseg = num_segments;
  in.force_general = force_general;
  in.fast_reason = (fmt == 0 && q_ids == nullptr) ? 0 /* dense */ : 1 /* match */;
  const int smax = a.Sq > a.Skv ? a.Sq : a.Skv;
  in.nblk = (smax + kMetaThreads - 1) / kMetaThreads;
  cudaError_t e = cudaMemsetAsync(a.hdr, 0, sizeof(WsHeader), st);
  if (e != cudaSuccess) return e;
  // enough blocks for the widest pass, at most what fits on the GPU at once
  const int64_t units = (int64_t)in.nblk * a.B * 2;
  const int64_t nqc = (a.Sq + kChunk - 1) / kChunk, nkc = (a.Skv + kChunk - 1) / kChunk;
  const int64_t wpb = kMetaThreads / 32;
  const int64_t chunk_blocks = ((int64_t)a.B * (nqc + nkc) + wpb - 1) / wpb;
  const int64_t range_blocks = ((int64_t)a.B * (a.n_qt + a.n_kt) + wpb - 1) / wpb;
  const int cap = meta_max_blocks();
  if (cap <= 0) return cudaErrorInvalidConfiguration;
  const int64_t want = std::max<int64_t>(1, std::max(units, std::max(chunk_blocks, range_blocks)));
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, cap));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMetaThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, meta_kernel, a, in);
}

}  // namespace attn
