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

// grid (B, 2): blockIdx.y 0 = query side, 1 = key/value side.
__global__ void __launch_bounds__(kMetaThreads) meta_normalize_kernel(
    const KernelArgs a, int fmt, const int32_t* q_ids, const int32_t* q_pos_in,
    const int32_t* kv_ids, const int32_t* kv_pos_in, const int32_t* cu_q, const int32_t* cu_kv,
    int nseg) {
  __shared__ int sh[32];
  __shared__ int carry_s;
  const int b = blockIdx.x;
  const bool kvside = blockIdx.y == 1;
  const int S = kvside ? a.Skv : a.Sq;
  const int32_t* ids = kvside ? kv_ids : q_ids;
  const int32_t* pos_in = kvside ? kv_pos_in : q_pos_in;
  const int32_t* cu = kvside ? cu_kv : cu_q;
  int32_t* id_out = const_cast<int32_t*>(kvside ? a.kv_id : a.q_id) + (int64_t)b * S;
  int32_t* pos_out = const_cast<int32_t*>(kvside ? a.kv_pos : a.q_pos) + (int64_t)b * S;
  int32_t* lo_out = const_cast<int32_t*>(kvside ? a.kv_seg_lo : a.seg_lo) + (int64_t)b * S;
  int32_t* hi_out = const_cast<int32_t*>(kvside ? a.kv_seg_hi : a.seg_hi) + (int64_t)b * S;

  // pass 1: ids and run starts (prefix max of run-start indices)
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < S; base += kMetaThreads) {
    const int t = base + threadIdx.x;
    int id = 0, start = -1;
    if (t < S) {
      id = token_id(fmt, ids, cu, nseg, b, S, t);
      const int prev = (t > 0) ? token_id(fmt, ids, cu, nseg, b, S, t - 1) : INT_MIN;
      start = (t == 0 || prev != id) ? t : -1;
      id_out[t] = id;
    }
    int run = block_prefix_max(start, sh);
    run = max(run, carry_s);
    if (t < S) lo_out[t] = run;  // run start for now
    __syncthreads();
    if (threadIdx.x == kMetaThreads - 1) carry_s = run;
    __syncthreads();
  }
  // pass 2: run ends (suffix min of next run starts), positions, fast-path bounds
  if (threadIdx.x == 0) carry_s = S;
  __syncthreads();
  int nonstd = 0;
  const int nblk = (S + kMetaThreads - 1) / kMetaThreads;
  for (int blk = nblk - 1; blk >= 0; --blk) {
    const int t = blk * kMetaThreads + threadIdx.x;
    int end_cand = INT_MAX;
    int id = 0;
    if (t < S) {
      id = id_out[t];
      const bool last = (t == S - 1) || (id_out[t + 1] != id);
      end_cand = last ? t + 1 : INT_MAX;
    }
    int end = block_suffix_min(end_cand, sh);
    end = min(end, carry_s);
    if (t < S) {
      const int start = lo_out[t];
      int pos;
      if (fmt == 2 || pos_in == nullptr) pos = (ids == nullptr && fmt != 2) ? t : t - start;
      else pos = __ldg(pos_in + (int64_t)b * S + t);
      pos_out[t] = pos;
      if (id != 0 && pos != t - start) nonstd = 1;
      lo_out[t] = id != 0 ? start : 0;
      hi_out[t] = id != 0 ? end : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) carry_s = end;
    __syncthreads();
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

__device__ ChunkInfo chunk_info(const int32_t* id, const int32_t* pos, int S, int c0) {
  ChunkInfo ci;
  ci.min_id = INT_MAX;
  ci.max_id = 0;
  ci.min_pos = INT_MAX;
  ci.max_pos = INT_MIN;
  int first = -1;
  bool uni = (c0 + kChunk <= S);
  for (int t = c0; t < min(S, c0 + kChunk); ++t) {
    const int i = id[t];
    if (i == 0) { uni = false; continue; }
    if (first < 0) first = i;
    else if (i != first) uni = false;
    ci.min_id = min(ci.min_id, i);
    ci.max_id = max(ci.max_id, i);
    ci.min_pos = min(ci.min_pos, pos[t]);
    ci.max_pos = max(ci.max_pos, pos[t]);
  }
  ci.uniform = (uni && first > 0) ? 1 : 0;
  ci.pad[0] = ci.pad[1] = ci.pad[2] = 0;
  return ci;
}

__global__ void meta_chunks_kernel(const KernelArgs a) {
  const int nqc = (a.Sq + kChunk - 1) / kChunk, nkc = (a.Skv + kChunk - 1) / kChunk;
  const int total = a.B * (nqc + nkc);
  for (int w = blockIdx.x * blockDim.x + threadIdx.x; w < total; w += gridDim.x * blockDim.x) {
    if (w < a.B * nqc) {
      const int b = w / nqc, c = w % nqc;
      const_cast<ChunkInfo*>(a.q_chunk)[w] =
          chunk_info(a.q_id + (int64_t)b * a.Sq, a.q_pos + (int64_t)b * a.Sq, a.Sq, c * kChunk);
    } else {
      const int w2 = w - a.B * nqc;
      const int b = w2 / nkc, c = w2 % nkc;
      const_cast<ChunkInfo*>(a.kv_chunk)[w2] = chunk_info(
          a.kv_id + (int64_t)b * a.Skv, a.kv_pos + (int64_t)b * a.Skv, a.Skv, c * kChunk);
    }
  }
}

__device__ __forceinline__ bool ids_meet(const ChunkInfo& x, int lo, int hi) {
  return x.max_id != 0 && x.min_id <= hi && lo <= x.max_id;
}

__global__ void meta_ranges_kernel(const KernelArgs a, int force_general, int fmt_cu,
                                   int fast_reason) {
  const int mism = a.hdr->mismatch;
  const bool general = force_general || a.Sq != a.Skv || (mism & 7) != 0;
  const int nqc = (a.Sq + kChunk - 1) / kChunk, nkc = (a.Skv + kChunk - 1) / kChunk;
  const int totq = a.B * a.n_qt, totk = a.B * a.n_kt;
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
  for (int w = blockIdx.x * blockDim.x + threadIdx.x; w < totq + totk;
       w += gridDim.x * blockDim.x) {
    int lo = INT_MAX, hi = 0;
    if (w < totq) {
      const int b = w / a.n_qt, t = w % a.n_qt;
      const int q0 = t * kTile, q1 = min(a.Sq, q0 + kTile);
      if (!general) {
        for (int i = q0; i < q1; ++i) {
          const int64_t g = (int64_t)b * a.Sq + i;
          const int sl = a.seg_lo[g], sh = a.seg_hi[g];
          if (sh <= sl) continue;
          const int h2 = a.causal ? min(i + 1, sh) : sh;
          lo = min(lo, sl);
          hi = max(hi, h2);
        }
      } else {
        int qlo = INT_MAX, qhi = 0;
        for (int c = q0 / kChunk; c * kChunk < q1; ++c) {
          const ChunkInfo ci = a.q_chunk[b * nqc + c];
          if (ci.max_id == 0) continue;
          qlo = min(qlo, ci.min_id);
          qhi = max(qhi, ci.max_id);
        }
        if (qhi != 0) {
          for (int c = 0; c < nkc; ++c) {
            if (ids_meet(a.kv_chunk[b * nkc + c], qlo, qhi)) {
              lo = min(lo, c * kChunk);
              hi = max(hi, min(a.Skv, (c + 1) * kChunk));
            }
          }
        }
      }
      const int2 r = (hi > lo) ? make_int2(lo, hi) : make_int2(0, 0);
      const_cast<int2*>(a.q_tile_range)[w] = r;
      if (r.y > r.x)
        atomicAdd(reinterpret_cast<unsigned long long*>(&a.hdr->tile_pairs),
                  (unsigned long long)((r.y - r.x + kTile - 1) / kTile));
    } else {
      const int w2 = w - totq;
      const int b = w2 / a.n_kt, t = w2 % a.n_kt;
      const int k0 = t * kTile, k1 = min(a.Skv, k0 + kTile);
      if (!general) {
        for (int j = k0; j < k1; ++j) {
          const int64_t g = (int64_t)b * a.Skv + j;  // Sq == Skv on the fast path
          const int sl = a.seg_lo[g], sh = a.seg_hi[g];
          if (sh <= sl) continue;
          const int l2 = a.causal ? max(j, sl) : sl;
          lo = min(lo, l2);
          hi = max(hi, sh);
        }
      } else {
        int klo = INT_MAX, khi = 0;
        for (int c = k0 / kChunk; c * kChunk < k1; ++c) {
          const ChunkInfo ci = a.kv_chunk[b * nkc + c];
          if (ci.max_id == 0) continue;
          klo = min(klo, ci.min_id);
          khi = max(khi, ci.max_id);
        }
        if (khi != 0) {
          for (int c = 0; c < nqc; ++c) {
            if (ids_meet(a.q_chunk[b * nqc + c], klo, khi)) {
              lo = min(lo, c * kChunk);
              hi = max(hi, min(a.Sq, (c + 1) * kChunk));
            }
          }
        }
      }
      const_cast<int2*>(a.kv_tile_range)[w2] = (hi > lo) ? make_int2(lo, hi) : make_int2(0, 0);
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
  meta_normalize_kernel<<<dim3(a.B, 2), kMetaThreads, 0, st>>>(a, fmt, q_ids, q_pos, kv_ids,
                                                               kv_pos, cu_q, cu_kv, num_segments);
  if (a.Sq == a.Skv) {
    const int64_t n = (int64_t)a.B * a.Sq;
    const int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    meta_match_kernel<<<blocks, 256, 0, st>>>(a);
  }
  {
    const int nqc = (a.Sq + kChunk - 1) / kChunk, nkc = (a.Skv + kChunk - 1) / kChunk;
    const int n = a.B * (nqc + nkc);
    meta_chunks_kernel<<<(n + 127) / 128, 128, 0, st>>>(a);
  }
  {
    const int n = a.B * (a.n_qt + a.n_kt);
    meta_ranges_kernel<<<(n + 127) / 128, 128, 0, st>>>(a, force_general, fmt == 2,
                                                         fast_reason);
  }
  return cudaGetLastError();
}

}  // namespace attn
