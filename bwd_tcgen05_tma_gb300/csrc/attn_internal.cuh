// Internal definitions shared by the attention kernels and the host API.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "chunk_mask.h"
#include "debug_checks.h"
#include "sm103_ptx.cuh"

namespace attn {

using bf16 = __nv_bfloat16;  // storage of every 16-bit element (bf16 or fp16 bits)

// The 16-bit floating-point element of Q/K/V/O/dO/bias and of the gradients,
// and of the MMA operands built from them (P, dS): bf16 or fp16.  Packing and
// products round to nearest even.  Pointers to such elements are typed bf16*
// and hold either format's bits.
struct ElemBf16 {
  static constexpr uint32_t kMmaFmt = 1;  // kind::f16 operand format
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    return sm103::pack_bf16x2(lo, hi);
  }
  static __device__ __forceinline__ uint32_t mul(uint32_t a, uint32_t b) {
    return sm103::mul_bf16x2(a, b);
  }
  static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
  static __device__ __forceinline__ float ld(const bf16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void st(bf16* p, float x) { *p = __float2bfloat16_rn(x); }
};
struct ElemF16 {
  static constexpr uint32_t kMmaFmt = 0;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    return sm103::pack_f16x2(lo, hi);
  }
  static __device__ __forceinline__ uint32_t mul(uint32_t a, uint32_t b) {
    return sm103::mul_f16x2(a, b);
  }
  static __device__ __forceinline__ float lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
  }
  static __device__ __forceinline__ float hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
  }
  static __device__ __forceinline__ float ld(const bf16* p) {
    return __half2float(*reinterpret_cast<const __half*>(p));
  }
  static __device__ __forceinline__ void st(bf16* p, float x) {
    *reinterpret_cast<__half*>(p) = __float2half_rn(x);
  }
};

constexpr int kChunk = 64;   // granularity of the per-chunk metadata summaries
constexpr int kTile = 128;   // query tile (forward, dQ pass) and KV tile (all kernels)
constexpr int kPreTok = 8;   // tokens per block of the backward preprocess
constexpr int kBwdQ = 64;    // query tile of the dK/dV pass

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
  int32_t status;      // device-side attn_status_t (timeouts, failed bounds checks)
  int32_t path;        // 0 fast, 1 general
  int32_t reason;      // attn_path_reason_t
  int32_t dq_mode;     // dQ mode used
  int64_t tile_pairs;  // scheduled (query tile, KV tile) pairs
  int32_t mismatch;    // bit0 ids differ, bit1 pos differ, bit2 nonstandard pos
  int32_t where;       // site of the first device-side error (wait or bounds check)
  int32_t next_item[4];  // work-item counters of the persistent kernels (zeroed per call)
  uint32_t meta_barrier;  // arrivals at the metadata kernel's grid barriers (zeroed per call)
  uint32_t meta_done;     // metadata blocks past their last pass (zeroed per call)
};

// Dynamic work distribution inside a persistent CTA: one thread claims items
// from a global counter and hands them to every role of the CTA, in order,
// through a small ring in shared memory (-1 ends the stream).
constexpr int kItemRing = 4;
struct ItemRing {
  uint64_t full[kItemRing];
  uint64_t empty[kItemRing];
  int32_t item[kItemRing];
};

__device__ __forceinline__ void ring_init(ItemRing* r, uint32_t consumers) {
  for (int i = 0; i < kItemRing; ++i) {
    sm103::mbar_init(&r->full[i], 1);
    sm103::mbar_init(&r->empty[i], consumers);
  }
}

// Producer side: claim the next item (or -1 once exhausted) and publish it as
// the n-th entry of the ring.  With `order`, claim v stands for item
// order[v / per] * per + v % per (items grouped `per` to a tile, the tiles
// handed out in the order given).  Returns false if the wait for a free slot
// timed out.
__device__ __forceinline__ bool ring_push(ItemRing* r, uint32_t n, int32_t* counter, int n_items,
                                          int32_t& item, const int32_t* order = nullptr,
                                          int per = 1) {
  const int s = n % kItemRing;
  if (n >= (uint32_t)kItemRing && !sm103::mbar_wait(&r->empty[s], ((n / kItemRing) - 1) & 1))
    return false;
  const int32_t v = atomicAdd(counter, 1);
  if (v >= n_items) {
    item = -1;
  } else if (order) {
    const int32_t g = v / per;
    item = order[g] * per + (v - g * per);
  } else {
    item = v;
  }
  *reinterpret_cast<volatile int32_t*>(&r->item[s]) = item;
  sm103::mbar_arrive(&r->full[s]);  // release: the item is visible to waiters
  return true;
}

// Consumer side (every consuming thread): read the n-th entry.  Warp-uniform.
__device__ __forceinline__ bool ring_pop(ItemRing* r, uint32_t n, int32_t& item) {
  const int s = n % kItemRing;
  if (!sm103::mbar_wait_warp(&r->full[s], (n / kItemRing) & 1)) return false;
  item = *reinterpret_cast<volatile int32_t*>(&r->item[s]);
  sm103::mbar_arrive(&r->empty[s]);
  return true;
}

// Whole-warp consumer that counts as one arrival (the warp-wide MMA issuers):
// every lane waits, lane 0 reads the entry and releases the slot, and the
// item reaches every lane as a warp-uniform value.
__device__ __forceinline__ bool ring_pop_warp1(ItemRing* r, uint32_t n, int32_t& item) {
  const int s = n % kItemRing;
  if (!sm103::mbar_wait_warp(&r->full[s], (n / kItemRing) & 1)) return false;
  int32_t v = 0;
  if ((threadIdx.x & 31) == 0) {
    v = *reinterpret_cast<volatile int32_t*>(&r->item[s]);
    sm103::mbar_arrive(&r->empty[s]);
  }
  item = sm103::warp_uniform(v);
  return true;
}

// A ring of work items that also carries what the producer looked up once
// per item: entry = (item index or -1 at the end, key tiles, first key, 0).
// The producer claims and publishes items itself (it may claim one ahead of
// what it publishes, see the forward), so consumers need no global loads to
// start an item.
struct ItemRing4 {
  uint64_t full[kItemRing];
  uint64_t empty[kItemRing];
  int4 item[kItemRing];
};

__device__ __forceinline__ void ring4_init(ItemRing4* r, uint32_t consumers) {
  for (int i = 0; i < kItemRing; ++i) {
    sm103::mbar_init(&r->full[i], 1);
    sm103::mbar_init(&r->empty[i], consumers);
  }
}

// Producer: publish entry n once its slot is free (false: the wait timed out).
__device__ __forceinline__ bool ring4_publish(ItemRing4* r, uint32_t n, int4 v) {
  const int s = n % kItemRing;
  if (n >= (uint32_t)kItemRing && !sm103::mbar_wait(&r->empty[s], ((n / kItemRing) - 1) & 1))
    return false;
  r->item[s] = v;
  sm103::mbar_arrive(&r->full[s]);  // release: the entry is visible to waiters
  return true;
}

// Single-thread consumer (the TMA producer); `ready` tests without waiting.
__device__ __forceinline__ bool ring4_ready(ItemRing4* r, uint32_t n) {
  return sm103::mbar_test_wait(&r->full[n % kItemRing], (n / kItemRing) & 1);
}
__device__ __forceinline__ bool ring4_pop1(ItemRing4* r, uint32_t n, int4& v) {
  const int s = n % kItemRing;
  if (!sm103::mbar_wait(&r->full[s], (n / kItemRing) & 1)) return false;
  v = r->item[s];
  sm103::mbar_arrive(&r->empty[s]);
  return true;
}

// Consumer, every thread of the consuming warps (each arrives once).
__device__ __forceinline__ bool ring4_pop(ItemRing4* r, uint32_t n, int4& v) {
  const int s = n % kItemRing;
  if (!sm103::mbar_wait_warp(&r->full[s], (n / kItemRing) & 1)) return false;
  v = r->item[s];
  sm103::mbar_arrive(&r->empty[s]);
  return true;
}

// Consumer warp that counts as one arrival; v is warp-uniform.
__device__ __forceinline__ bool ring4_pop_warp1(ItemRing4* r, uint32_t n, int4& v) {
  const int s = n % kItemRing;
  if (!sm103::mbar_wait_warp(&r->full[s], (n / kItemRing) & 1)) return false;
  int4 t = make_int4(0, 0, 0, 0);
  if ((threadIdx.x & 31) == 0) {
    t = r->item[s];
    sm103::mbar_arrive(&r->empty[s]);
  }
  v.x = sm103::warp_uniform(t.x);
  v.y = sm103::warp_uniform(t.y);
  v.z = sm103::warp_uniform(t.z);
  v.w = sm103::warp_uniform(t.w);
  return true;
}

// Summary of 64 consecutive tokens of one batch row.
struct ChunkInfo {
  int32_t min_id;   // smallest nonzero id (INT32_MAX if none)
  int32_t max_id;   // largest nonzero id (0 if none)
  int32_t min_pos;  // over tokens with nonzero id
  int32_t max_pos;
  int32_t uniform;  // 1: all 64 tokens exist and carry the same nonzero id
  int32_t consec;   // 1: uniform, and token k of the chunk sits at position min_pos + k
  int32_t pad[2];
};

// Everything a kernel needs; passed by value as a __grid_constant__ parameter
// (the tensor maps must live in parameter space for TMA).
struct KernelArgs {
  CUtensorMap tm_q;    // dims {d_qk, Hq, B*Sq},   box {64, 1, 128 or 64}
  CUtensorMap tm_k;    // dims {d_qk, Hkv, B*Skv}, box {64, 1, 128}
  CUtensorMap tm_v;    // dims {d_v, Hkv, B*Skv},  box {64, 1, 128}
  CUtensorMap tm_do;   // dims {d_v, Hq, B*Sq},    box {64, 1, 128 or 64}
  CUtensorMap tm_dqacc;  // fp32 dQ accumulator: dims {d_qk, Hq, B*Sq}, box {32, 1, 64}
  CUtensorMap tm_o;    // forward output O: dims {d_v, Hq, Sq, B}, box {64, 1, 128, 1}

  int B, Sq, Skv, Hq, Hkv, d_qk, d_v;
  // Position mask: a key at position pk is kept for a query at position pq
  // (same nonzero segment id) when -win_left <= pk - (pq + shift) <= win_right,
  // a negative bound leaving that side open.  Causal: win_right = 0.
  int win_left, win_right, shift;
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  int n_qt;          // query tiles of 128 per row
  int n_kt;          // KV tiles of 128 per row
  int n_qt64;        // query tiles of 64 per row

  // normalised metadata (workspace)
  const int32_t* q_id;
  const int32_t* q_pos;
  const int32_t* kv_id;
  const int32_t* kv_pos;
  const int32_t* seg_lo;   // fast path: segment start of each query token (row-local)
  const int32_t* seg_hi;   // fast path: segment end (exclusive); 0/0 for padding
  const int32_t* kv_seg_lo;  // the same for the key/value tokens
  const int32_t* kv_seg_hi;
  const ChunkInfo* q_chunk;
  const ChunkInfo* kv_chunk;
  const int2* meta_scan;      // [2][B][chunks of 1024] first/last run boundary per chunk
  const int2* q_tile_range;   // [B*n_qt]  KV token range of each 128-row query tile
  const int2* kv_tile_range;  // [B*n_kt]  query token range of each 128-row KV tile
  // query tiles (b * n_qt + t) in order of decreasing KV-tile count: the
  // persistent passes over query tiles hand out their longest items first
  const int32_t* q_order;     // [B*n_qt]
  float* max_logit;  // forward only: fp32 [B, Hq] or null
  const float* sink;  // fp32 [Hq] sink logits or null
  float* dsink;       // backward only: fp32 [Hq] or null
  float* sink_part;   // backward workspace: per preprocess block and head, partial dsink
  WsHeader* hdr;

  // bias
  const bf16* bias;
  int bias_b, bias_h;

  // forward outputs
  bf16* o;
  float* lse;

  // backward
  const bf16* o_in;
  const bf16* d_o;
  const float* lse_in;
  float* lse2;     // LSE * log2(e) (+inf for rows without keys)
  float* Dvec;     // D = rowsum(dO * O), [B, Hq, Sq]
  float* dq_acc;   // fp32 [B*Sq, Hq, d_qk]  (atomic dQ)
  bf16* dq;
  int64_t dq_stride;  // token-row stride of dq in elements
  bf16* dk;
  int64_t dk_stride;
  bf16* dv;
  int64_t dv_stride;
  bf16* dbias;
  float* dbias_acc;   // fp32 like the bias (bias broadcast along batch or heads)
  int dbias_mode;     // 0 none, 1 write bf16 directly, 2 accumulate in fp32
  int elem_f16;        // element type: 0 bf16, 1 fp16
  int test_stall;      // testing knob: the forward's scheduler hands out no work
  int grad_st32;       // 1: dQ/dK/dV rows start 32-byte aligned (256-bit stores)
  int dkdv_batch_loop;  // 1: one dK/dV work item loops over every batch row
  int dkdv_head_loop;   // 1: one dK/dV work item loops over every KV head

  // FP8 (E4M3) forward: tm_q / tm_k map the one-byte Q and K, tm_v the
  // transposed V in the workspace (planes of [128 d][vt_pad keys])
  float fp8_sc2;               // scale * descale_q * descale_k * log2(e)
  float fp8_dv;                // descale_v
  const uint8_t* vt_src;       // V (E4M3), its token-row stride in elements
  int64_t vt_src_stride;
  uint8_t* vt;                 // [B * Hkv][128][vt_pad]
  int vt_pad;                  // keys per plane row: Skv rounded up to 128, plus 128
};

// Opt-in timeline for pipeline debugging (-DATTN_TIMELINE builds only): the
// first threads of each role in CTA 0 append (event, step, SM clock) records.
#ifdef ATTN_TIMELINE
// Slot = event * 2048 + step: plain stores, no round trip on the critical path.
constexpr int kTimelineSteps = 2048;
constexpr int kTimelineCap = 64 * kTimelineSteps;
static __device__ unsigned long long g_timeline[kTimelineCap];  // one copy per translation unit
#define ATTN_TL(ev, step)                                                                    \
  do {                                                                                       \
    if (blockIdx.x == 0 && (ev) >= 0 && (ev) < 64 && (step) >= 0 && (step) < kTimelineSteps) \
      g_timeline[(ev) * kTimelineSteps + (step)] = (unsigned long long)clock64();            \
  } while (0)
#else
#define ATTN_TL(ev, step) \
  do {                    \
  } while (0)
#endif

// Eight packed 16-bit pairs (16 consecutive elements) to global memory: one
// 32-byte store when the row is 32-byte aligned (`st32`), else two 16-byte
// stores.  Row-per-thread epilogues touch one line per lane and store, so
// wider stores halve the store transactions that occupy the load/store path.
__device__ __forceinline__ void store16_elems(bf16* dst, const uint32_t (&w)[8], bool st32) {
  if (st32) {
    sm103::st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
  } else {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

using attn_mask::range_bits64;

__device__ __forceinline__ bool path_general(const KernelArgs& a);

// Key positions [x, y] (inclusive) that a query at position pq keeps.
__device__ __forceinline__ int2 band_key_pos(const KernelArgs& a, int pq) {
  const int c = pq + a.shift;
  return make_int2(a.win_left < 0 ? INT_MIN : c - a.win_left,
                   a.win_right < 0 ? INT_MAX : c + a.win_right);
}
// Query positions [x, y] (inclusive) that keep a key at position pk.
__device__ __forceinline__ int2 band_query_pos(const KernelArgs& a, int pk) {
  const int c = pk - a.shift;
  return make_int2(a.win_right < 0 ? INT_MIN : c - a.win_right,
                   a.win_left < 0 ? INT_MAX : c + a.win_left);
}
// Fast path (equal metadata on both sides, positions = offsets inside the
// segment, shift 0, so pk - pq = j - i): the key tokens [x, y) of query token
// i whose segment spans the tokens [sl, sh), and the query tokens of key j.
__device__ __forceinline__ int2 band_keys_of_query(const KernelArgs& a, int i, int sl, int sh) {
  return make_int2(a.win_left >= 0 ? max(sl, i - a.win_left) : sl,
                   a.win_right >= 0 ? min(sh, i + a.win_right + 1) : sh);
}
__device__ __forceinline__ int2 band_queries_of_key(const KernelArgs& a, int j, int sl, int sh) {
  return make_int2(a.win_right >= 0 ? max(sl, j - a.win_right) : sl,
                   a.win_left >= 0 ? min(sh, j + a.win_left + 1) : sh);
}

// Validity of the 128 keys [k0, k0 + 128) of batch row b for one query row, as
// two 64-bit masks.  Fast path: the row's key range [rlo, rhi).  General path:
// same nonzero segment id and a key position inside the row's band.
// Validity bits of the 64 tokens of one chunk for a token of the other side
// with nonzero segment id `id` whose band admits the positions [p.x, p.y],
// from the chunk's summary alone (attn_mask::chunk_decide).  False when the
// summary does not decide it; the caller then compares token by token.
__device__ __forceinline__ bool chunk_bits(const ChunkInfo& c, int id, int2 p, uint64_t& bits) {
  return attn_mask::chunk_decide(c.min_id, c.max_id, c.min_pos, c.max_pos, c.uniform, c.consec,
                                 id, p.x, p.y, &bits);
}

// General path of kv_valid_bits, out of line: the fast path's loops keep
// their registers and code to themselves.
static __device__ __noinline__ ulonglong2 kv_valid_bits_general(const KernelArgs& a, int b, int k0,
                                                         int my_id, int my_pos) {
  uint64_t vb[2] = {0ull, 0ull};
  if (my_id == 0) return make_ulonglong2(0ull, 0ull);
  const int2 kp = band_key_pos(a, my_pos);
  const int nkc = (a.Skv + kChunk - 1) / kChunk;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {  // the tile's two 64-key halves
    const int kh = k0 + hh * 64;
    if (kh >= a.Skv) continue;
    if ((kh % kChunk) == 0 && chunk_bits(a.kv_chunk[b * nkc + kh / kChunk], my_id, kp, vb[hh]))
      continue;
    const int32_t* kid = a.kv_id + (int64_t)b * a.Skv + kh;
    const int32_t* kpos = a.kv_pos + (int64_t)b * a.Skv + kh;
    const int nv = min(64, a.Skv - kh);
    const bool vec = ((reinterpret_cast<uintptr_t>(kid) & 15u) == 0);
    uint64_t v64 = 0ull;
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
      int ids[4], pss[4];
      if (vec && c + 4 <= nv) {
        const int4 t1 = __ldg(reinterpret_cast<const int4*>(kid + c));
        const int4 t2 = __ldg(reinterpret_cast<const int4*>(kpos + c));
        ids[0] = t1.x; ids[1] = t1.y; ids[2] = t1.z; ids[3] = t1.w;
        pss[0] = t2.x; pss[1] = t2.y; pss[2] = t2.z; pss[3] = t2.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ids[e] = (c + e < nv) ? __ldg(kid + c + e) : -1;
          pss[e] = (c + e < nv) ? __ldg(kpos + c + e) : 0;
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool v = (ids[e] == my_id) & (pss[e] >= kp.x) & (pss[e] <= kp.y);
        v64 |= static_cast<uint64_t>(v) << (c + e);
      }
    }
    vb[hh] = v64;
  }
  return make_ulonglong2(vb[0], vb[1]);
}

// Validity of the 128 keys [k0, k0 + 128) of batch row b for one query row,
// as two 64-bit words.  Fast path: the row's key range [rlo, rhi).  General
// path: same nonzero segment id and a key position inside the row's band,
// from the key chunks' summaries where they decide it.
__device__ __forceinline__ void kv_valid_bits(const KernelArgs& a, bool general, int b, int k0,
                                              int rlo, int rhi, int my_id, int my_pos,
                                              uint64_t (&vb)[2]) {
  if (!general) {
    vb[0] = range_bits64(rlo - k0, rhi - k0);
    vb[1] = range_bits64(rlo - k0 - 64, rhi - k0 - 64);
    return;
  }
  const ulonglong2 r = kv_valid_bits_general(a, b, k0, my_id, my_pos);
  vb[0] = r.x;
  vb[1] = r.y;
}

__device__ __forceinline__ bool path_general(const KernelArgs& a) {
  return *reinterpret_cast<const volatile int32_t*>(&a.hdr->path) != 0;
}

// Largest of the value held at p and v, for any fp32 values including -inf
// (non-negative values order like signed integers, negative ones reversed
// like unsigned integers).
__device__ __forceinline__ void atomic_max_f32(float* p, float v) {
  if (v >= 0.f)
    atomicMax(reinterpret_cast<int*>(p), __float_as_int(v));
  else
    atomicMin(reinterpret_cast<unsigned int*>(p), __float_as_uint(v));
}

// Max-logit of one warp's rows (row_max in log2 units of scaled logits,
// -inf for rows without a valid key) folded into out[b * Hq + h].
__device__ __forceinline__ void warp_max_logit(float* out, float row_max_log2) {
  float v = row_max_log2;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0 && v > -INFINITY) atomic_max_f32(out, v * 0.6931471805599453f);
}

// Records a device-side error; the first one (by arrival) keeps its status
// and its site.
__device__ __forceinline__ void report_device_error(const KernelArgs& a, int status, int where) {
  if (atomicCAS(&a.hdr->status, 0, status) == 0) atomicExch(&a.hdr->where, where);
}

// A timed-out wait.
__device__ __forceinline__ void report_timeout(const KernelArgs& a, int where) {
  report_device_error(a, 6 /* ATTN_ERR_DEVICE_TIMEOUT */, where);
}

// Bounds checks of the checking build.  `ATTN_CHECK(a, cond, site)` is true
// when the access it guards may go ahead: with -DATTN_DEBUG it evaluates
// cond and, when cond fails, records ATTN_ERR_DEVICE_BOUNDS at `site` (codes
// 0x7K.., K the kernel as in the wait sites) and the access is skipped;
// otherwise it is the constant true and cond is not evaluated.
#ifdef ATTN_DEBUG
__device__ __forceinline__ bool debug_check(const KernelArgs& a, bool ok, int site) {
  if (!ok) report_device_error(a, 7 /* ATTN_ERR_DEVICE_BOUNDS */, site);
  return ok;
}
#define ATTN_CHECK(a, cond, site) (::attn::debug_check((a), (cond), (site)))
#else
#define ATTN_CHECK(a, cond, site) true
#endif
using attn_dbg::span_ok;
using attn_dbg::tma_box_ok;
using attn_dbg::row_span_ok;

// The box of a tiled copy through one of the argument block's tensor maps
// (16-bit tensors in 64-column boxes, the fp32 dQ accumulator in 32-column
// boxes; `rows` = the box's row count) lies where the copy engine allows it.
__device__ __forceinline__ bool box_ok(const KernelArgs& a, const CUtensorMap* m, int x, int y,
                                       int64_t z, int rows, bool store = false) {
  const int64_t tq = (int64_t)a.B * a.Sq, tkv = (int64_t)a.B * a.Skv;
  if (m == &a.tm_q) return tma_box_ok(x, 64, a.d_qk, 2, y, a.Hq, z, rows, tq, store);
  if (m == &a.tm_k) return tma_box_ok(x, 64, a.d_qk, 2, y, a.Hkv, z, rows, tkv, store);
  if (m == &a.tm_v) return tma_box_ok(x, 64, a.d_v, 2, y, a.Hkv, z, rows, tkv, store);
  if (m == &a.tm_do) return tma_box_ok(x, 64, a.d_v, 2, y, a.Hq, z, rows, tq, store);
  if (m == &a.tm_dqacc) return tma_box_ok(x, 32, a.d_qk, 4, y, a.Hq, z, rows, tq, store);
  return false;
}

// Gradient rows: n elements from column `col` of token row `row` of dQ
// (query tokens, Hq heads of d_qk), dK (key tokens, Hkv heads of d_qk) or dV
// (key tokens, Hkv heads of d_v), written through `p` with `vec`-byte stores.
__device__ __forceinline__ bool dq_span_ok(const KernelArgs& a, int64_t row, int64_t col, int n,
                                           const void* p, int vec) {
  return row_span_ok(row, (int64_t)a.B * a.Sq, col, n, (int64_t)a.Hq * a.d_qk,
                     reinterpret_cast<uint64_t>(p), vec);
}
__device__ __forceinline__ bool dk_span_ok(const KernelArgs& a, int64_t row, int64_t col, int n,
                                           const void* p, int vec) {
  return row_span_ok(row, (int64_t)a.B * a.Skv, col, n, (int64_t)a.Hkv * a.d_qk,
                     reinterpret_cast<uint64_t>(p), vec);
}
__device__ __forceinline__ bool dv_span_ok(const KernelArgs& a, int64_t row, int64_t col, int n,
                                           const void* p, int vec) {
  return row_span_ok(row, (int64_t)a.B * a.Skv, col, n, (int64_t)a.Hkv * a.d_v,
                     reinterpret_cast<uint64_t>(p), vec);
}
// One element (row, key) of the bias gradient dBias [bias_b, bias_h, Sq, Skv]
// (fp32 accumulator or the output itself) at flat row `brow` = (b * bias_h + h)
// * Sq + query.
__device__ __forceinline__ bool dbias_ok(const KernelArgs& a, int64_t brow, int64_t key) {
  return brow >= 0 && brow < (int64_t)a.bias_b * a.bias_h * a.Sq && key >= 0 && key < a.Skv;
}

// ---------------------------------------------------------------- dK/dV work items
// Work item -> (KV tile, batch range, KV-head range).
struct DkdvItem {
  int t, b0, b1, g0, g1;
};

__device__ __forceinline__ int dkdv_n_items(const KernelArgs& a) {
  const int nb = a.dkdv_batch_loop ? 1 : a.B;
  const int ng = a.dkdv_head_loop ? 1 : a.Hkv;
  return a.n_kt * nb * ng;
}

__device__ __forceinline__ DkdvItem dkdv_item(const KernelArgs& a, int idx) {
  const int ng = a.dkdv_head_loop ? 1 : a.Hkv;
  DkdvItem it;
  // (batch row, KV head)-major: CTAs running at the same time work on KV tiles
  // of the same head and re-read the same Q / dO tiles from L2
  const int combo = idx / a.n_kt;
  it.t = idx - combo * a.n_kt;
  const int bi = combo / ng, gi = combo - (combo / ng) * ng;
  it.b0 = a.dkdv_batch_loop ? 0 : bi;
  it.b1 = a.dkdv_batch_loop ? a.B : bi + 1;
  it.g0 = a.dkdv_head_loop ? 0 : gi;
  it.g1 = a.dkdv_head_loop ? a.Hkv : gi + 1;
  return it;
}

// Query range of KV tile t of row b; returns the number of BQ-row query tiles.
template <int BQ = kBwdQ>
__device__ __forceinline__ int dkdv_q_tiles(const KernelArgs& a, int b, int t, int& q_lo) {
  const int2 r = a.kv_tile_range[b * a.n_kt + t];
  q_lo = r.x;
  return (r.y > r.x) ? (r.y - r.x + BQ - 1) / BQ : 0;
}

// Row-per-thread bias of one 128-key tile: adds bias[i, k0 + c] * log2(e) to
// x[c] for c < nvalid (row pointer given), 16 bytes per load where the row
// segment is 16-byte aligned.
template <class E>
__device__ __forceinline__ void add_bias_row(float (&x)[kTile], const bf16* row, int nvalid) {
  constexpr float kL2e = 1.4426950408889634f;
  const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15u) == 0);
#pragma unroll
  for (int c = 0; c < kTile; c += 8) {
    if (vec && c + 8 <= nvalid) {
      const uint4 u = sm103::ld_nc_v4(row + c);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[c + 2 * e] += E::lo(w[e]) * kL2e;
        x[c + 2 * e + 1] += E::hi(w[e]) * kL2e;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (c + e < nvalid) x[c + e] += E::ld(row + c + e) * kL2e;
    }
  }
}

// Starts moving the bias elements [e0, e0 + n) toward L2 (one bulk prefetch:
// no registers and no wait), so that a later add_bias_row of them hits L2.
// The byte range is clipped to the bias tensor and rounded inward to 16 bytes.
__device__ __forceinline__ void prefetch_bias_l2(const KernelArgs& a, int64_t e0, int n) {
  const int64_t total = (int64_t)a.bias_b * a.bias_h * a.Sq * a.Skv;
  int64_t e1 = e0 + n;
  if (e0 < 0) e0 = 0;
  if (e1 > total) e1 = total;
  const uintptr_t lo = (reinterpret_cast<uintptr_t>(a.bias + e0) + 15u) & ~static_cast<uintptr_t>(15);
  const uintptr_t hi = reinterpret_cast<uintptr_t>(a.bias + e1) & ~static_cast<uintptr_t>(15);
  if (hi > lo)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo),
                 "r"(static_cast<uint32_t>(hi - lo))
                 : "memory");
}

// The same through the load/store path, one prefetch.global.L2 per 128-byte
// line (the lines of in-bounds elements only).  In the one-warpgroup forward
// the bulk form measured slower than no prefetch and this form faster.
__device__ __forceinline__ void prefetch_bias_lines(const KernelArgs& a, int64_t e0, int n) {
  const int64_t total = (int64_t)a.bias_b * a.bias_h * a.Sq * a.Skv;
  int64_t e1 = e0 + n;
  if (e0 < 0) e0 = 0;
  if (e1 > total) e1 = total;
  if (e1 <= e0) return;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(a.bias + e0) & ~static_cast<uintptr_t>(127);
  const uintptr_t hi = reinterpret_cast<uintptr_t>(a.bias + e1);
  for (uintptr_t p = lo; p < hi; p += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Broadcast dBias (summed over batch rows and/or heads).  Every (batch row,
// head) that adds into one dBias row of KV tile t runs in the same dK/dV work
// item, in a fixed order, and writes the query rows its BQ-row query tiles
// cover, [q_lo, q_lo + nq * BQ) within [0, Sq).  For each row, the first of
// them stores dS into the fp32 accumulator (or, if it is also the last, the
// finished bf16 value into dBias), the ones in between add to the
// accumulator, and the last adds and writes the finished value to dBias.
// So the accumulator is never cleared and never converted: dBias is cleared
// before the pass, and rows no step writes stay 0.
//
// Rows [i0, i0 + 32) of the current (batch row b, head g * G + hh) step that
// an earlier step of the same work item has written already, as a bit mask.
template <int BQ>
__device__ __forceinline__ uint32_t dbias_rows_written_before(const KernelArgs& a, int b0, int b,
                                                              int g0, int g, int hh, int t, int i0) {
  if (a.bias_h == 1 && (g > g0 || hh > 0)) return ~0u;  // the item's first head wrote them
  uint32_t seen = 0u;
  if (a.bias_b == 1) {
    for (int bp = b0; bp < b; ++bp) {
      int q_lo;
      const int nq = dkdv_q_tiles<BQ>(a, bp, t, q_lo);
      if (nq > 0) seen |= static_cast<uint32_t>(range_bits64(q_lo - i0, q_lo + nq * BQ - i0));
    }
  }
  return seen;
}
// One thread's share of a step: dS of key kj for the 32 query rows [r0, r0 +
// 32) (rows past Sq skipped), accumulator row brow0 + c.  A step must call it
// even where its dS is 0, or a row's first store or last write is lost.  Eight
// loads in flight before their stores (a store between two loads would
// serialise them: the addresses may alias).
template <class E>
__device__ __forceinline__ void dbias_acc_rows(const KernelArgs& a, int64_t brow0, int kj, int r0,
                                               uint32_t seen, uint32_t later, const float (&ds)[32]) {
  float* acc_p = a.dbias_acc + brow0 * a.Skv + kj;
  bf16* out_p = a.dbias + brow0 * a.Skv + kj;
#pragma unroll
  for (int c8 = 0; c8 < 32; c8 += 8) {
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
      acc[c] = (r0 + c8 + c < a.Sq && ((seen >> (c8 + c)) & 1u)) ? acc_p[(int64_t)(c8 + c) * a.Skv]
                                                                   : 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      if (r0 + c8 + c >= a.Sq) continue;
      const int64_t o = (int64_t)(c8 + c) * a.Skv;
      if ((later >> (c8 + c)) & 1u)
        acc_p[o] = acc[c] + ds[c8 + c];
      else
        E::st(out_p + o, acc[c] + ds[c8 + c]);
    }
  }
}

// ... and that a later step of the item (batch rows up to b1, KV heads up to
// g1, G query heads per KV head) will write again.
template <int BQ>
__device__ __forceinline__ uint32_t dbias_rows_written_after(const KernelArgs& a, int b, int b1, int g,
                                                             int g1, int hh, int G, int t, int i0) {
  if (a.bias_h == 1 && (g < g1 - 1 || hh < G - 1)) return ~0u;  // the item's last head will
  uint32_t later = 0u;
  if (a.bias_b == 1) {
    for (int bp = b + 1; bp < b1; ++bp) {
      int q_lo;
      const int nq = dkdv_q_tiles<BQ>(a, bp, t, q_lo);
      if (nq > 0) later |= static_cast<uint32_t>(range_bits64(q_lo - i0, q_lo + nq * BQ - i0));
    }
  }
  return later;
}


// Launches `kern` with programmatic stream serialisation: the grid may be
// scheduled while the kernel before it on the stream still runs, and waits
// in grid_dep_wait() (which every such kernel calls before it touches data
// that kernel writes) until that kernel has completed.
template <typename... P, typename... Act>
inline cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Act&&>(args)...);
}

// Kernel launchers (defined in the kernel translation units).
cudaError_t launch_meta(const KernelArgs& a, int fmt, const int32_t* q_ids, const int32_t* q_pos,
                        const int32_t* kv_ids, const int32_t* kv_pos, const int32_t* cu_q,
                        const int32_t* cu_kv, int num_segments, int force_general,
                        cudaStream_t st);
cudaError_t launch_fwd(const KernelArgs& a, int num_sms, cudaStream_t st);
// Forward over pairs of query heads of one KV group (even group size, d <= 128).
cudaError_t launch_fwd2t(const KernelArgs& a, int num_sms, cudaStream_t st);
// FP8 forward (d_qk = d_v = 128) and the transposed copy of V it reads.
cudaError_t launch_vt_transpose(const KernelArgs& a, cudaStream_t st);
cudaError_t launch_fwd_fp8(const KernelArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_bwd_pre(const KernelArgs& a, int zero_dq_acc, cudaStream_t st);
cudaError_t launch_sink_reduce(const KernelArgs& a, cudaStream_t st);
cudaError_t launch_bwd_dkdv(const KernelArgs& a, bool atomic_dq, int num_sms, cudaStream_t st);
cudaError_t launch_bwd_dq(const KernelArgs& a, int num_sms, cudaStream_t st);
// The same two passes for one element type (bwd_bf16.cu, bwd_f16.cu).
template <class E>
cudaError_t launch_bwd_dkdv_t(const KernelArgs& a, bool atomic_dq, int num_sms, cudaStream_t st);
template <class E>
cudaError_t launch_bwd_dq_t(const KernelArgs& a, int num_sms, cudaStream_t st);
// dK/dV pass with 128-row query tiles (deterministic dQ mode, d_qk and d_v <= 128).
cudaError_t launch_bwd_dkdv128(const KernelArgs& a, int num_sms, cudaStream_t st);
// Deterministic dQ pass with Q, dO and dS as tensor-memory operands (d_qk, d_v <= 128).
cudaError_t launch_bwd_dq128(const KernelArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_dq_convert(const KernelArgs& a, cudaStream_t st);

}  // namespace attn
