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

// Pass 1, grid (chunks, B, 2 sides), one thread per token of a 1024-token
// chunk: normalised ids, plus the chunk's first and last run boundary (a
// boundary is a token whose id differs from its predecessor's, or token 0).
__global__ void __launch_bounds__(kMetaThreads) meta_ids_kernel(
    const KernelArgs a, int fmt, const int32_t* q_ids, const int32_t* kv_ids, const int32_t* cu_q,
    const int32_t* cu_kv, int nseg, int2* bounds, int nblk) {
  __shared__ int sh[32];
  const int blk = blockIdx.x, b = blockIdx.y;
  const bool kvside = blockIdx.z == 1;
  const int S = kvside ? a.Skv : a.Sq;
  const int c0 = blk * kMetaThreads;
  if (c0 >= S) return;
  const int32_t* ids = kvside ? kv_ids : q_ids;
  const int32_t* cu = kvside ? cu_kv : cu_q;
  int32_t* id_out = const_cast<int32_t*>(kvside ? a.kv_id : a.q_id) + (int64_t)b * S;
  const int t = c0 + threadIdx.x;
  int first = INT_MAX, last = -1;
  if (t < S) {
    const int id = token_id(fmt, ids, cu, nseg, b, S, t);
    id_out[t] = id;
    const bool bnd = (t == 0) || (token_id(fmt, ids, cu, nseg, b, S, t - 1) != id);
    if (bnd) first = last = t;
  }
  // block min / max of the boundary positions
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) {
    first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
    last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  }
  __shared__ int shl[32];
  if (lane == 0) { sh[w] = first; shl[w] = last; }
  __syncthreads();
  if (w == 0) {
    first = sh[lane];
    last = shl[lane];
    for (int o = 16; o > 0; o >>= 1) {
      first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
      last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    }
    if (lane == 0) bounds[((int)kvside * a.B + b) * nblk + blk] = make_int2(first, last);
  }
}

// Pass 2, same grid: run starts / ends from block scans plus the boundaries of
// the other chunks; positions (given, or derived as the offset inside the run);
// fast-path segment bounds; flags positions that do not restart at 0 and count
// up inside every segment.
__global__ void __launch_bounds__(kMetaThreads) meta_pos_kernel(
    const KernelArgs a, int fmt, const int32_t* q_ids, const int32_t* q_pos_in,
    const int32_t* kv_ids, const int32_t* kv_pos_in, const int2* bounds, int nblk) {
  __shared__ int sh[32];
  __shared__ int carry_start, carry_end;
  const int blk = blockIdx.x, b = blockIdx.y;
  const bool kvside = blockIdx.z == 1;
  const int S = kvside ? a.Skv : a.Sq;
  const int c0 = blk * kMetaThreads;
  if (c0 >= S) return;
  const int32_t* ids = kvside ? kv_ids : q_ids;
  const int32_t* pos_in = kvside ? kv_pos_in : q_pos_in;
  const int32_t* id_row = (kvside ? a.kv_id : a.q_id) + (int64_t)b * S;
  int32_t* pos_out = const_cast<int32_t*>(kvside ? a.kv_pos : a.q_pos) + (int64_t)b * S;
  int32_t* lo_out = const_cast<int32_t*>(kvside ? a.kv_seg_lo : a.seg_lo) + (int64_t)b * S;
  int32_t* hi_out = const_cast<int32_t*>(kvside ? a.kv_seg_hi : a.seg_hi) + (int64_t)b * S;
  const int2* bd = bounds + ((int)kvside * a.B + b) * nblk;
  if (threadIdx.x == 0) {
    int cs = 0;  // last boundary before this chunk (token 0 always is one)
    for (int k = blk - 1; k >= 0; --k)
      if (bd[k].y >= 0) { cs = bd[k].y; break; }
    int ce = S;  // first boundary after this chunk
    const int nb = (S + kMetaThreads - 1) / kMetaThreads;
    for (int k = blk + 1; k < nb; ++k)
      if (bd[k].x != INT_MAX) { ce = bd[k].x; break; }
    carry_start = cs;
    carry_end = ce;
  }
  const int t = c0 + threadIdx.x;
  int id = 0, start_c = -1, end_c = INT_MAX;
  if (t < S) {
    id = id_row[t];
    if (t == 0 || id_at(id_row, t - 1) != id) start_c = t;
    if (t + 1 < S && id_row[t + 1] != id) end_c = t + 1;
  }
  int start = block_prefix_max(start_c, sh);
  int end = block_suffix_min(end_c, sh);
  if (t < S) {
    if (start < 0) start = carry_start;
    if (end == INT_MAX) end = (t + 1 >= S) ? S : carry_end;
  }
  int nonstd = 0;
  if (t < S) {
    int pos;
    if (fmt == 2 || pos_in == nullptr) pos = (ids == nullptr && fmt != 2) ? t : t - start;
    else pos = __ldg(pos_in + (int64_t)b * S + t);
    pos_out[t] = pos;
    if (id != 0 && pos != t - start) nonstd = 1;
    lo_out[t] = id != 0 ? start : 0;
    hi_out[t] = id != 0 ? end : 0;
  }
  if (__syncthreads_or(nonstd) && threadIdx.x == 0) atomicOr(&a.hdr->mismatch, 4);
}

// Q/KV equality per token (only launched when Sq == Skv).
__global__ void meta_match_kernel(const KernelArgs a) {
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
  ci.pad[0] = ci.pad[1] = ci.pad[2] = 0;
  return ci;
}

__global__ void meta_chunks_kernel(const KernelArgs a) {
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

// Per 128-row query tile: the KV token range it may attend to; per 128-row KV
// tile: the query token range that may attend to it.  One warp per tile.
__global__ void meta_ranges_kernel(const KernelArgs a, int force_general, int fmt_cu,
                                   int fast_reason) {
  const int mism = a.hdr->mismatch;
  const bool general = force_general || a.Sq != a.Skv || (mism & 7) != 0;
  const int nqc = (a.Sq + kChunk - 1) / kChunk, nkc = (a.Skv + kChunk - 1) / kChunk;
  const int totq = a.B * a.n_qt, totk = a.B * a.n_kt;
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.hdr->path = general ? 1 : 0;
    int reason;
    if (force_general) reason = 2;
    else if (a.Sq != a.Skv) reason = 3;
    else if (mism & 1) reason = fmt_cu ? 7 : 4;
    else if (mism & 2) reason = fmt_cu ? 7 : 5;
    else if (mism & 4) reason = 6;
    else reason = fast_reason;  // dense rows or matching metadata
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
        if (qside) {
          lo = min(lo, sl);
          hi = max(hi, a.causal ? min(i + 1, sh) : sh);
        } else {
          lo = min(lo, a.causal ? max(i, sl) : sl);
          hi = max(hi, sh);
        }
      }
    } else {
      const ChunkInfo* own = qside ? a.q_chunk : a.kv_chunk;
      const ChunkInfo* oth = qside ? a.kv_chunk : a.q_chunk;
      const int nown = qside ? nqc : nkc, noth = qside ? nkc : nqc;
      int ilo = INT_MAX, ihi = 0;
      for (int c = r0 / kChunk + lane; c * kChunk < r1; c += 32) {
        const ChunkInfo ci = own[b * nown + c];
        if (ci.max_id == 0) continue;
        ilo = min(ilo, ci.min_id);
        ihi = max(ihi, ci.max_id);
      }
      ilo = warp_min(ilo);
      ihi = warp_max(ihi);
      if (ihi != 0) {
        for (int c = lane; c < noth; c += 32) {
          if (ids_meet(oth[b * noth + c], ilo, ihi)) {
            lo = min(lo, c * kChunk);
            hi = max(hi, min(S_oth, (c + 1) * kChunk));
          }
        }
      }
    }
    lo = warp_min(lo);
    hi = warp_max(hi);
    if (lane == 0) {
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

}  // namespace

cudaError_t launch_meta(const KernelArgs& a, int fmt, const int32_t* q_ids, const int32_t* q_pos,
                        const int32_t* kv_ids, const int32_t* kv_pos, const int32_t* cu_q,
                        const int32_t* cu_kv, int num_segments, int force_general,
                        cudaStream_t st) {
  const int fast_reason = (fmt == 0 && q_ids == nullptr) ? 0 /* dense */ : 1 /* match */;
  cudaError_t e = cudaMemsetAsync(a.hdr, 0, sizeof(WsHeader), st);
  if (e != cudaSuccess) return e;
  const int smax = a.Sq > a.Skv ? a.Sq : a.Skv;
  const int nblk = (smax + kMetaThreads - 1) / kMetaThreads;
  int2* bounds = const_cast<int2*>(a.meta_scan);
  const dim3 grid(nblk, a.B, 2);
  meta_ids_kernel<<<grid, kMetaThreads, 0, st>>>(a, fmt, q_ids, kv_ids, cu_q, cu_kv, num_segments,
                                                 bounds, nblk);
  meta_pos_kernel<<<grid, kMetaThreads, 0, st>>>(a, fmt, q_ids, q_pos, kv_ids, kv_pos, bounds,
                                                 nblk);
  if (a.Sq == a.Skv) {
    const int64_t n = (int64_t)a.B * a.Sq;
    const int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    meta_match_kernel<<<blocks, 256, 0, st>>>(a);
  }
  {
    const int nqc = (a.Sq + kChunk - 1) / kChunk, nkc = (a.Skv + kChunk - 1) / kChunk;
    const int warps = a.B * (nqc + nkc);
    meta_chunks_kernel<<<(warps + 7) / 8, 256, 0, st>>>(a);
  }
  {
    const int warps = a.B * (a.n_qt + a.n_kt);
    meta_ranges_kernel<<<(warps + 7) / 8, 256, 0, st>>>(a, force_general, fmt == 2, fast_reason);
  }
  return cudaGetLastError();
}

}  // namespace attn
