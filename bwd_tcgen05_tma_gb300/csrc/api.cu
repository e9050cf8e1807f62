// Host side of the C ABI: argument validation, packed-layout resolution,
// workspace planning, TMA descriptor encoding and kernel launches.
//
// Layout resolution follows TransformerEngine PR #2358 ("[JAX] Make all jax
// attention calls use non-packed common calls"): a packed QKV buffer yields K
// one head-block and V two head-blocks after Q, and the V slice of a packed KV
// buffer starts num_gqa_groups * v_head_dim elements after K (the page's
// review of the KV-packed stride).  With grouped query heads the 3HD token row
// holds Hq query heads, then Hkv key heads, then Hkv value heads.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.cuh"

namespace attn {
namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Plan {
  size_t hdr, q_id, q_pos, seg_lo, seg_hi, kv_id, kv_pos, kv_seg_lo, kv_seg_hi;
  size_t q_chunk, kv_chunk, q_range, kv_range, q_order, meta_scan, vt;
  size_t fwd_total;
  size_t lse2, dvec, dq_acc, dbias_acc, sink_part;
  size_t bwd_total;
};

bool effective_atomic(const attn_params_t* p) {
  return p->dq_mode == ATTN_DQ_ATOMIC && p->d_qk <= 128;
}

// Bytes per element of Q / K / V.
int64_t elem_bytes(const attn_params_t* p) { return p->dtype == ATTN_DTYPE_FP8_E4M3 ? 1 : 2; }

// Keys per row of a transposed-V plane (FP8 forward): Skv rounded up to a
// whole tile, plus one tile, so that a 128-key box starting at any key below
// Skv stays inside the row.
int64_t vt_pad(const attn_params_t* p) { return ((p->Skv + kTile - 1) / kTile) * kTile + kTile; }

bool dbias_needs_acc(const attn_params_t* p) {
  return p->bias != nullptr && ((p->bias_b == 1 && p->B > 1) || (p->bias_h == 1 && p->Hq > 1));
}

Plan make_plan(const attn_params_t* p) {
  Plan pl{};
  const size_t B = p->B, Sq = p->Sq, Skv = p->Skv;
  const size_t nqc = (Sq + kChunk - 1) / kChunk, nkc = (Skv + kChunk - 1) / kChunk;
  const size_t nqt = (Sq + kTile - 1) / kTile, nkt = (Skv + kTile - 1) / kTile;
  size_t o = 0;
  pl.hdr = o; o = up(o + sizeof(WsHeader));
  pl.q_id = o; o = up(o + B * Sq * 4);
  pl.q_pos = o; o = up(o + B * Sq * 4);
  pl.seg_lo = o; o = up(o + B * Sq * 4);
  pl.seg_hi = o; o = up(o + B * Sq * 4);
  pl.kv_id = o; o = up(o + B * Skv * 4);
  pl.kv_pos = o; o = up(o + B * Skv * 4);
  pl.kv_seg_lo = o; o = up(o + B * Skv * 4);
  pl.kv_seg_hi = o; o = up(o + B * Skv * 4);
  pl.q_chunk = o; o = up(o + B * nqc * sizeof(ChunkInfo));
  pl.kv_chunk = o; o = up(o + B * nkc * sizeof(ChunkInfo));
  pl.q_range = o; o = up(o + B * nqt * sizeof(int2));
  pl.kv_range = o; o = up(o + B * nkt * sizeof(int2));
  pl.q_order = o; o = up(o + B * nqt * 4);
  pl.meta_scan = o; o = up(o + 2 * B * ((std::max(Sq, Skv) + 1023) / 1024) * sizeof(int2));
  pl.vt = o;  // FP8 forward only: V^T planes [B * Hkv][d_v][vt_pad], one byte each
  if (p->dtype == ATTN_DTYPE_FP8_E4M3) o = up(o + B * (size_t)p->Hkv * p->d_v * vt_pad(p));
  pl.fwd_total = o;
  pl.lse2 = o; o = up(o + B * p->Hq * Sq * 4);
  pl.dvec = o; o = up(o + B * p->Hq * Sq * 4);
  pl.dq_acc = o;
  if (effective_atomic(p)) o = up(o + B * Sq * p->Hq * (size_t)p->d_qk * 4);
  pl.dbias_acc = o;
  if (dbias_needs_acc(p)) o = up(o + (size_t)p->bias_b * p->bias_h * Sq * Skv * 4);
  pl.sink_part = o;  // per preprocess block and head: partial sink gradient
  if (p->dsink) o = up(o + ((B * Sq + kPreTok - 1) / kPreTok) * (size_t)p->Hq * 4);
  pl.bwd_total = o;
  return pl;
}

attn_status_t validate(const attn_params_t* p) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (p->struct_version != ATTN_PARAMS_VERSION) return ATTN_ERR_INVALID_ARG;
  if (p->fmt < 0 || p->fmt > 2 || p->layout < 0 || p->layout > 2 || p->mask < 0 || p->mask > 3 ||
      p->dq_mode < 0 || p->dq_mode > 1)
    return ATTN_ERR_INVALID_ARG;
  if (p->B <= 0 || p->Sq <= 0 || p->Skv <= 0 || p->Hq <= 0 || p->Hkv <= 0)
    return ATTN_ERR_INVALID_ARG;
  if ((int64_t)p->B * p->Sq >= (1ll << 31) || (int64_t)p->B * p->Skv >= (1ll << 31))
    return ATTN_ERR_UNSUPPORTED;
  if (p->Hq % p->Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (p->Hq > 256) return ATTN_ERR_UNSUPPORTED;
  if (!(p->scale > 0.f) || p->scale != p->scale) return ATTN_ERR_INVALID_ARG;
  if (p->d_qk != 64 && p->d_qk != 128 && p->d_qk != 192) return ATTN_ERR_UNSUPPORTED;
  if (p->d_v != 64 && p->d_v != 128) return ATTN_ERR_UNSUPPORTED;
  // packed-layout rules (PR #2358: the 3HD check q_max_seqlen == kv_max_seqlen and
  // the KV-packed requirement qk_head_dim == v_head_dim)
  if (p->layout == ATTN_LAYOUT_3HD && p->Sq != p->Skv) return ATTN_ERR_SHAPE_MISMATCH;
  if (p->layout == ATTN_LAYOUT_HD_2HD && p->d_qk != p->d_v) return ATTN_ERR_SHAPE_MISMATCH;
  if (!p->q || !aligned16(p->q)) return ATTN_ERR_INVALID_ARG;
  if (p->layout != ATTN_LAYOUT_3HD && (!p->k || !aligned16(p->k))) return ATTN_ERR_INVALID_ARG;
  if (p->layout == ATTN_LAYOUT_HD_HD_HD && (!p->v || !aligned16(p->v))) return ATTN_ERR_INVALID_ARG;
  // sequence description
  if (p->fmt == ATTN_FMT_THD_SEGMENTS && (!p->q_seg_ids || !p->kv_seg_ids))
    return ATTN_ERR_INVALID_ARG;
  if (p->fmt == ATTN_FMT_THD_CU_SEQLENS) {
    if (p->B != 1 || !p->cu_seqlens_q || !p->cu_seqlens_kv || p->num_segments < 0)
      return ATTN_ERR_INVALID_ARG;
  }
  if (p->fmt != ATTN_FMT_THD_CU_SEQLENS) {
    // ids and positions of one side must agree in shape with each other and with [B, S]
    // (PR #2692: segment_pos must carry the same leading dims as segment_ids)
    const bool qi = p->q_seg_ids != nullptr, ki = p->kv_seg_ids != nullptr;
    if (qi != ki) return ATTN_ERR_INVALID_ARG;
    if ((p->q_seg_pos != nullptr) != (p->kv_seg_pos != nullptr)) return ATTN_ERR_INVALID_ARG;
    if ((p->q_seg_pos && !qi)) return ATTN_ERR_INVALID_ARG;
    if (qi) {
      if (p->q_ids_dims[0] != p->B || p->q_ids_dims[1] != p->Sq) return ATTN_ERR_SHAPE_MISMATCH;
      if (p->kv_ids_dims[0] != p->B || p->kv_ids_dims[1] != p->Skv) return ATTN_ERR_SHAPE_MISMATCH;
      if (p->q_seg_pos) {
        if (p->q_pos_dims[0] != p->q_ids_dims[0] || p->q_pos_dims[1] != p->q_ids_dims[1])
          return ATTN_ERR_SHAPE_MISMATCH;
        if (p->kv_pos_dims[0] != p->kv_ids_dims[0] || p->kv_pos_dims[1] != p->kv_ids_dims[1])
          return ATTN_ERR_SHAPE_MISMATCH;
      }
    }
  }
  const bool causal = p->mask == ATTN_MASK_CAUSAL || p->mask == ATTN_MASK_PADDING_CAUSAL;
  if (p->band && causal && p->window_right > 0) return ATTN_ERR_INVALID_ARG;
  if (p->dtype != ATTN_DTYPE_BF16 && p->dtype != ATTN_DTYPE_FP16 && p->dtype != ATTN_DTYPE_FP8_E4M3)
    return ATTN_ERR_INVALID_ARG;
  if (p->dtype == ATTN_DTYPE_FP8_E4M3) {
    const float d[3] = {p->descale_q, p->descale_k, p->descale_v};
    for (float x : d)
      if (!(x > 0.f) || !std::isfinite(x)) return ATTN_ERR_INVALID_ARG;
    if (p->d_qk != 128 || p->d_v != 128 || p->bias || p->sink) return ATTN_ERR_UNSUPPORTED;
  }
  if (p->bias) {
    if (!aligned16(p->bias)) return ATTN_ERR_INVALID_ARG;
    if (!(p->bias_b == 1 || p->bias_b == p->B) || !(p->bias_h == 1 || p->bias_h == p->Hq))
      return ATTN_ERR_SHAPE_MISMATCH;
  }
  return ATTN_OK;
}

attn_status_t resolve(const attn_params_t* p, void* dq, void* dk, void* dv, attn_resolved_t* r) {
  const char* q = static_cast<const char*>(p->q);
  const int64_t Hq = p->Hq, Hkv = p->Hkv, dqk = p->d_qk, dvv = p->d_v;
  const int64_t es = elem_bytes(p);  // byte offsets of the packed slices
  std::memset(r, 0, sizeof(*r));
  switch (p->layout) {
    case ATTN_LAYOUT_3HD: {
      const int64_t W = Hq * dqk + Hkv * dqk + Hkv * dvv;
      r->q = q;
      r->k = q + Hq * dqk * es;
      r->v = q + (Hq * dqk + Hkv * dqk) * es;
      r->q_token_stride = r->k_token_stride = r->v_token_stride = W;
      if (dq) {
        char* d = static_cast<char*>(dq);
        r->dq = d;
        r->dk = d + Hq * dqk * es;
        r->dv = d + (Hq * dqk + Hkv * dqk) * es;
      }
      break;
    }
    case ATTN_LAYOUT_HD_2HD: {
      const char* k = static_cast<const char*>(p->k);
      r->q = q;
      r->k = k;
      r->v = k + Hkv * dvv * es;  // stride from v_head_dim
      r->q_token_stride = Hq * dqk;
      r->k_token_stride = r->v_token_stride = 2 * Hkv * dvv;
      r->dq = dq;
      if (dk) {
        r->dk = dk;
        r->dv = static_cast<char*>(dk) + Hkv * dvv * es;
      }
      break;
    }
    default:
      r->q = q;
      r->k = p->k;
      r->v = p->v;
      r->q_token_stride = Hq * dqk;
      r->k_token_stride = Hkv * dqk;
      r->v_token_stride = Hkv * dvv;
      r->dq = dq;
      r->dk = dk;
      r->dv = dv;
  }
  return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a token-major tensor: dims {D, H, T}, box {64, 1, rows}.
bool make_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, int D, int H, int64_t T,
              int64_t tok_stride, int rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)tok_stride * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, type, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a token-major tensor of one-byte elements (FP8): dims {D, H,
// T}, box {128, 1, rows} (one 128-byte swizzle row per token).
bool make_map8(CUtensorMap* m, const void* base, int D, int H, int64_t T, int64_t tok_stride,
               int rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)tok_stride};
  cuuint32_t box[3] = {128, 1, (cuuint32_t)rows};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the transposed-V planes of the FP8 forward: dims {vt_pad
// keys, d_v, planes}, box {128 keys, 128 dims, 1}.
bool make_map_vt(CUtensorMap* m, const void* base, int64_t pad, int d_v, int64_t planes) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)pad, (cuuint64_t)d_v, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)pad, (cuuint64_t)(pad * d_v)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over a token-major tensor of B rows of S tokens: dims {D, H, S, B},
// box {64, 1, rows, 1}.  Stores through it stop at each batch row's end.
bool make_map_4d(CUtensorMap* m, CUtensorMapDataType type, const void* base, int D, int H,
                 int64_t S, int B, int64_t tok_stride, int rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)tok_stride * 2,
                           (cuuint64_t)(S * tok_stride * 2)};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, type, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the fp32 dQ accumulator [T, H, D]: box {32, 1, 64}, no swizzle.
bool make_map_f32(CUtensorMap* m, const void* base, int D, int H, int64_t T) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4};
  cuuint32_t box[3] = {32, 1, (cuuint32_t)kBwdQ};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cache[64] = {0};
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64) cache[dev] = n;
  return n;
}

// Tensor-map element type of the call's 16-bit tensors.
CUtensorMapDataType map_type(const attn_params_t* p) {
  return p->dtype == ATTN_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

void fill_common(KernelArgs& a, const attn_params_t* p, char* ws, const Plan& pl) {
  a.elem_f16 = p->dtype == ATTN_DTYPE_FP16 ? 1 : 0;
  a.test_stall = p->test_wait_timeout != 0 ? 1 : 0;
  a.B = p->B; a.Sq = p->Sq; a.Skv = p->Skv; a.Hq = p->Hq; a.Hkv = p->Hkv;
  a.d_qk = p->d_qk; a.d_v = p->d_v;
  const bool causal = p->mask == ATTN_MASK_CAUSAL || p->mask == ATTN_MASK_PADDING_CAUSAL;
  a.win_left = (p->band && p->window_left >= 0) ? p->window_left : -1;
  a.win_right = causal ? 0 : ((p->band && p->window_right >= 0) ? p->window_right : -1);
  a.shift = p->bottom_right ? p->Skv - p->Sq : 0;
  a.scale = p->scale;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.n_qt = (p->Sq + kTile - 1) / kTile;
  a.n_kt = (p->Skv + kTile - 1) / kTile;
  a.n_qt64 = (p->Sq + kBwdQ - 1) / kBwdQ;
  a.hdr = reinterpret_cast<WsHeader*>(ws + pl.hdr);
  a.q_id = reinterpret_cast<int32_t*>(ws + pl.q_id);
  a.q_pos = reinterpret_cast<int32_t*>(ws + pl.q_pos);
  a.seg_lo = reinterpret_cast<int32_t*>(ws + pl.seg_lo);
  a.seg_hi = reinterpret_cast<int32_t*>(ws + pl.seg_hi);
  a.kv_id = reinterpret_cast<int32_t*>(ws + pl.kv_id);
  a.kv_pos = reinterpret_cast<int32_t*>(ws + pl.kv_pos);
  a.kv_seg_lo = reinterpret_cast<int32_t*>(ws + pl.kv_seg_lo);
  a.kv_seg_hi = reinterpret_cast<int32_t*>(ws + pl.kv_seg_hi);
  a.q_chunk = reinterpret_cast<ChunkInfo*>(ws + pl.q_chunk);
  a.kv_chunk = reinterpret_cast<ChunkInfo*>(ws + pl.kv_chunk);
  a.meta_scan = reinterpret_cast<int2*>(ws + pl.meta_scan);
  a.q_tile_range = reinterpret_cast<int2*>(ws + pl.q_range);
  a.kv_tile_range = reinterpret_cast<int2*>(ws + pl.kv_range);
  a.q_order = reinterpret_cast<int32_t*>(ws + pl.q_order);
  a.bias = static_cast<const bf16*>(p->bias);
  a.bias_b = p->bias_b;
  a.bias_h = p->bias_h;
}

thread_local cudaEvent_t g_trace[2 * ATTN_TRACE_SLOTS] = {};
thread_local bool g_trace_on = false;

// Records the start (end = false) or end event of a trace slot, if tracing.
void trace(int slot, bool end, cudaStream_t st) {
  if (!g_trace_on) return;
  cudaEvent_t e = g_trace[2 * slot + (end ? 1 : 0)];
  if (e) cudaEventRecord(e, st);
}

// Second stream for the deterministic 128-row dQ pass, one per host thread
// and device, made on first use outside stream capture.  The dQ pass reads
// what the preprocess wrote and nothing the dK/dV pass writes, so the two run
// side by side: the dK/dV grid (the larger work items) stays on the caller's
// stream right behind the preprocess and takes the SMs first, while the dQ
// grid, released by an event, takes each SM that a dK/dV CTA leaves once the
// dK/dV work queue has run dry, instead of waiting for the slowest dK/dV CTA.
// (A dK/dV grid on the second stream, even at a higher priority, loses the
// SMs to a dQ grid queued directly behind the preprocess, and running CTAs
// are not displaced.)  The fork and join events keep the pair capturable into
// a CUDA graph.
struct AuxStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool failed = false;
};
constexpr int kMaxDevices = 64;
thread_local AuxStream g_aux[kMaxDevices];

// The auxiliary stream of this thread on the current device, or nullptr when
// none can be had (then both passes run one after the other on `st`).
AuxStream* aux_stream(cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  AuxStream& x = g_aux[dev];
  if (x.s) return &x;
  if (x.failed) return nullptr;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();  // leave no stale error for the launch checks that follow
    return nullptr;
  }
  if (cs != cudaStreamCaptureStatusNone) return nullptr;  // made by a later uncaptured call
  if (cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    if (x.s) cudaStreamDestroy(x.s);
    if (x.fork) cudaEventDestroy(x.fork);
    x.s = nullptr;
    x.fork = nullptr;
    x.failed = true;
    return nullptr;
  }
  return &x;
}

attn_status_t run_meta(const KernelArgs& a, const attn_params_t* p, cudaStream_t st) {
  const bool seg = p->fmt != ATTN_FMT_THD_CU_SEQLENS && p->q_seg_ids != nullptr;
  trace(ATTN_TRACE_META, false, st);
  const cudaError_t e =
      launch_meta(a, p->fmt == ATTN_FMT_THD_CU_SEQLENS ? 2 : (seg ? 1 : 0),
                  seg ? p->q_seg_ids : nullptr, seg ? p->q_seg_pos : nullptr,
                  seg ? p->kv_seg_ids : nullptr, seg ? p->kv_seg_pos : nullptr,
                  p->cu_seqlens_q, p->cu_seqlens_kv, p->num_segments, p->force_general_path, st);
  trace(ATTN_TRACE_META, true, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

int32_t attn_abi_version(void) { return ATTN_PARAMS_VERSION; }

int32_t attn_build_flags(void) {
#ifdef ATTN_DEBUG
  return ATTN_BUILD_DEVICE_CHECKS;
#else
  return 0;
#endif
}

attn_status_t attn_event_create(void** event) {
  if (!event) return ATTN_ERR_INVALID_ARG;
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return ATTN_ERR_CUDA;
  *event = e;
  return ATTN_OK;
}

attn_status_t attn_event_destroy(void* event) {
  if (!event) return ATTN_ERR_INVALID_ARG;
  return cudaEventDestroy(static_cast<cudaEvent_t>(event)) == cudaSuccess ? ATTN_OK
                                                                           : ATTN_ERR_CUDA;
}

attn_status_t attn_event_elapsed_ms(const void* start, const void* end, float* ms) {
  if (!start || !end || !ms) return ATTN_ERR_INVALID_ARG;
  const cudaError_t e = cudaEventElapsedTime(
      ms, static_cast<cudaEvent_t>(const_cast<void*>(start)),
      static_cast<cudaEvent_t>(const_cast<void*>(end)));
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error state of this query
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

attn_status_t attn_set_trace_events(void* const* events) {
  if (!events) {
    g_trace_on = false;
    for (auto& e : g_trace) e = nullptr;
    return ATTN_OK;
  }
  for (int i = 0; i < 2 * ATTN_TRACE_SLOTS; ++i) g_trace[i] = static_cast<cudaEvent_t>(events[i]);
  g_trace_on = true;
  return ATTN_OK;
}

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_SHAPE_MISMATCH: return "shape mismatch";
    case ATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case ATTN_ERR_DEVICE_BOUNDS: return "device-side bounds check failed (access skipped)";
  }
  return "unknown status";
}

size_t attn_fwd_workspace_size(const attn_params_t* p) {
  if (validate(p) != ATTN_OK) return 0;
  return make_plan(p).fwd_total;
}

size_t attn_bwd_workspace_size(const attn_params_t* p) {
  if (validate(p) != ATTN_OK) return 0;
  return make_plan(p).bwd_total;
}

attn_status_t attn_resolve_layout(const attn_params_t* p, void* dq, void* dk, void* dv,
                                  attn_resolved_t* out) {
  const attn_status_t s = validate(p);
  if (s != ATTN_OK) return s;
  if (!out) return ATTN_ERR_INVALID_ARG;
  return resolve(p, dq, dk, dv, out);
}

attn_status_t attn_fwd(const attn_params_t* p, void* o, float* lse, void* ws, size_t ws_bytes,
                       void* stream) {
  attn_status_t s = validate(p);
  if (s != ATTN_OK) return s;
  if (!o || !lse || !ws || !aligned16(o) || (reinterpret_cast<uintptr_t>(ws) % kAlign))
    return ATTN_ERR_INVALID_ARG;
  if (p->max_logit && (reinterpret_cast<uintptr_t>(p->max_logit) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (p->sink && (reinterpret_cast<uintptr_t>(p->sink) & 3u)) return ATTN_ERR_INVALID_ARG;
  const Plan pl = make_plan(p);
  if (ws_bytes < pl.fwd_total) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  attn_resolved_t r;
  resolve(p, nullptr, nullptr, nullptr, &r);
  if (!aligned16(r.k) || !aligned16(r.v) || (r.q_token_stride % 8) || (r.k_token_stride % 8) ||
      (r.v_token_stride % 8))
    return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  KernelArgs a;
  std::memset(&a, 0, sizeof(a));
  fill_common(a, p, static_cast<char*>(ws), pl);
  if (p->dtype == ATTN_DTYPE_FP8_E4M3) {
    // V^T planes first (they depend on nothing the metadata pass writes),
    // then the metadata, then the two-pass forward
    a.vt = reinterpret_cast<uint8_t*>(static_cast<char*>(ws) + pl.vt);
    a.vt_pad = static_cast<int>(vt_pad(p));
    a.vt_src = static_cast<const uint8_t*>(r.v);
    a.vt_src_stride = r.v_token_stride;
    a.fp8_sc2 = p->scale * p->descale_q * p->descale_k * 1.4426950408889634f;
    a.fp8_dv = p->descale_v;
    if (!make_map8(&a.tm_q, r.q, p->d_qk, p->Hq, (int64_t)p->B * p->Sq, r.q_token_stride, kTile) ||
        !make_map8(&a.tm_k, r.k, p->d_qk, p->Hkv, (int64_t)p->B * p->Skv, r.k_token_stride, kTile) ||
        !make_map_vt(&a.tm_v, a.vt, a.vt_pad, p->d_v, (int64_t)p->B * p->Hkv) ||
        !make_map_4d(&a.tm_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, o, p->d_v, p->Hq, p->Sq, p->B,
                     (int64_t)p->Hq * p->d_v, kTile))
      return ATTN_ERR_CUDA;
    a.o = static_cast<bf16*>(o);
    a.lse = lse;
    a.max_logit = p->max_logit;
    trace(ATTN_TRACE_FWD, false, st);
    if (launch_vt_transpose(a, st) != cudaSuccess) return ATTN_ERR_CUDA;
    if ((s = run_meta(a, p, st)) != ATTN_OK) return s;
    if (launch_fwd_fp8(a, sm_count(), st) != cudaSuccess) return ATTN_ERR_CUDA;
    trace(ATTN_TRACE_FWD, true, st);
    return ATTN_OK;
  }
  const CUtensorMapDataType mt = map_type(p);
  if (!make_map(&a.tm_q, mt, r.q, p->d_qk, p->Hq, (int64_t)p->B * p->Sq, r.q_token_stride, kTile) ||
      !make_map(&a.tm_k, mt, r.k, p->d_qk, p->Hkv, (int64_t)p->B * p->Skv, r.k_token_stride, kTile) ||
      !make_map(&a.tm_v, mt, r.v, p->d_v, p->Hkv, (int64_t)p->B * p->Skv, r.v_token_stride, kTile) ||
      !make_map_4d(&a.tm_o, mt, o, p->d_v, p->Hq, p->Sq, p->B, (int64_t)p->Hq * p->d_v, kTile))
    return ATTN_ERR_CUDA;
  a.o = static_cast<bf16*>(o);
  a.lse = lse;
  a.max_logit = p->max_logit;
  a.sink = p->sink;
  if ((s = run_meta(a, p, st)) != ATTN_OK) return s;
  trace(ATTN_TRACE_FWD, false, st);
  if (launch_fwd(a, sm_count(), st) != cudaSuccess) return ATTN_ERR_CUDA;
  trace(ATTN_TRACE_FWD, true, st);
  return ATTN_OK;
}

attn_status_t attn_bwd(const attn_params_t* p, const void* o, const void* d_o, const float* lse,
                       void* dq, void* dk, void* dv, void* dbias, void* ws, size_t ws_bytes,
                       void* stream) {
  attn_status_t s = validate(p);
  if (s != ATTN_OK) return s;
  if (p->dtype == ATTN_DTYPE_FP8_E4M3) return ATTN_ERR_UNSUPPORTED;  // forward only
  if (!o || !d_o || !lse || !ws || !aligned16(o) || !aligned16(d_o) ||
      (reinterpret_cast<uintptr_t>(ws) % kAlign))
    return ATTN_ERR_INVALID_ARG;
  if (!dq || !aligned16(dq)) return ATTN_ERR_INVALID_ARG;
  if (p->layout != ATTN_LAYOUT_3HD && (!dk || !aligned16(dk))) return ATTN_ERR_INVALID_ARG;
  if (p->layout == ATTN_LAYOUT_HD_HD_HD && (!dv || !aligned16(dv))) return ATTN_ERR_INVALID_ARG;
  if (dbias && !p->bias) return ATTN_ERR_INVALID_ARG;
  if (dbias && !aligned16(dbias)) return ATTN_ERR_INVALID_ARG;
  if (p->dsink && !p->sink) return ATTN_ERR_INVALID_ARG;  // a gradient needs its logits
  if ((p->sink && (reinterpret_cast<uintptr_t>(p->sink) & 3u)) ||
      (p->dsink && (reinterpret_cast<uintptr_t>(p->dsink) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  const Plan pl = make_plan(p);
  if (ws_bytes < pl.bwd_total) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  attn_resolved_t r;
  resolve(p, dq, dk, dv, &r);
  if (!aligned16(r.k) || !aligned16(r.v) || (r.q_token_stride % 8) || (r.k_token_stride % 8) ||
      (r.v_token_stride % 8))
    return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  KernelArgs a;
  std::memset(&a, 0, sizeof(a));
  fill_common(a, p, w, pl);
  const CUtensorMapDataType mt = map_type(p);
  a.o_in = static_cast<const bf16*>(o);
  a.d_o = static_cast<const bf16*>(d_o);
  a.lse_in = lse;
  a.lse2 = reinterpret_cast<float*>(w + pl.lse2);
  a.Dvec = reinterpret_cast<float*>(w + pl.dvec);
  a.sink = p->sink;
  a.dsink = p->dsink;
  a.sink_part = p->dsink ? reinterpret_cast<float*>(w + pl.sink_part) : nullptr;
  const bool atomic = effective_atomic(p);
  a.dq_acc = atomic ? reinterpret_cast<float*>(w + pl.dq_acc) : nullptr;
  a.dq = static_cast<bf16*>(const_cast<void*>(r.dq));
  a.dk = static_cast<bf16*>(const_cast<void*>(r.dk));
  a.dv = static_cast<bf16*>(const_cast<void*>(r.dv));
  a.dq_stride = r.q_token_stride;
  a.dk_stride = r.k_token_stride;
  a.dv_stride = r.v_token_stride;
  {
    // every row start is the base plus a multiple of 64 elements (head dims
    // and token strides are), so the bases decide 32-byte alignment
    const uintptr_t bases = reinterpret_cast<uintptr_t>(r.dq) | reinterpret_cast<uintptr_t>(r.dk) |
                            reinterpret_cast<uintptr_t>(r.dv);
    a.grad_st32 = (bases & 31u) == 0 ? 1 : 0;
  }
  a.dbias = static_cast<bf16*>(dbias);
  a.dbias_mode = dbias ? (dbias_needs_acc(p) ? 2 : 1) : 0;
  a.dbias_acc = (a.dbias_mode == 2) ? reinterpret_cast<float*>(w + pl.dbias_acc) : nullptr;
  a.dkdv_batch_loop = (a.dbias_mode == 2 && p->bias_b == 1 && p->B > 1) ? 1 : 0;
  a.dkdv_head_loop = (a.dbias_mode == 2 && p->bias_h == 1 && p->Hkv > 1) ? 1 : 0;
  // With metadata_from_forward the forward's metadata stays; the preprocess
  // kernel restarts the work counters of the backward passes either way.
  if (!p->metadata_from_forward && (s = run_meta(a, p, st)) != ATTN_OK) return s;
  trace(ATTN_TRACE_BWD_PRE, false, st);
  if (launch_bwd_pre(a, atomic ? 1 : 0, st) != cudaSuccess) return ATTN_ERR_CUDA;
  if (a.dsink && launch_sink_reduce(a, st) != cudaSuccess) return ATTN_ERR_CUDA;
  trace(ATTN_TRACE_BWD_PRE, true, st);
  // dK/dV pass: 128-row query tiles (deterministic dQ mode, head dims <= 128),
  // otherwise 64-row query tiles
  const bool tile128 = !atomic && p->d_qk <= 128 && p->d_v <= 128;
  const int qrows = tile128 ? kTile : kBwdQ;
  if (!make_map(&a.tm_q, mt, r.q, p->d_qk, p->Hq, (int64_t)p->B * p->Sq, r.q_token_stride, qrows) ||
      !make_map(&a.tm_k, mt, r.k, p->d_qk, p->Hkv, (int64_t)p->B * p->Skv, r.k_token_stride, kTile) ||
      !make_map(&a.tm_v, mt, r.v, p->d_v, p->Hkv, (int64_t)p->B * p->Skv, r.v_token_stride, kTile) ||
      !make_map(&a.tm_do, mt, d_o, p->d_v, p->Hq, (int64_t)p->B * p->Sq, (int64_t)p->Hq * p->d_v,
                qrows))
    return ATTN_ERR_CUDA;
  if (atomic && !make_map_f32(&a.tm_dqacc, a.dq_acc, p->d_qk, p->Hq, (int64_t)p->B * p->Sq))
    return ATTN_ERR_CUDA;
  const int nsm = sm_count();
  // 128-row passes: the dQ pass goes on the auxiliary stream, forked here
  // after the preprocess
  AuxStream* ax = tile128 ? aux_stream(st) : nullptr;
  cudaStream_t sq = st;
  if (ax) {
    if (cudaEventRecord(ax->fork, st) != cudaSuccess ||
        cudaStreamWaitEvent(ax->s, ax->fork, 0) != cudaSuccess)
      return ATTN_ERR_CUDA;
    sq = ax->s;
  }
  // From here on the second stream is forked: every outcome, failed or not,
  // leaves through the join below, so `st` always orders whatever reached
  // the second stream and a stream capture never ends with an unjoined fork.
  s = ATTN_OK;
  trace(ATTN_TRACE_DKDV, false, st);
  const cudaError_t ek = tile128 ? launch_bwd_dkdv128(a, nsm, st) : launch_bwd_dkdv(a, atomic, nsm, st);
  if (ek != cudaSuccess) s = ATTN_ERR_CUDA;
  trace(ATTN_TRACE_DKDV, true, st);
  if (s == ATTN_OK) {
    trace(ATTN_TRACE_DQ, false, sq);
    if (atomic) {
      if (launch_dq_convert(a, st) != cudaSuccess) s = ATTN_ERR_CUDA;
    } else {
      if (!tile128 &&
          (!make_map(&a.tm_q, mt, r.q, p->d_qk, p->Hq, (int64_t)p->B * p->Sq, r.q_token_stride,
                     kTile) ||
           !make_map(&a.tm_do, mt, d_o, p->d_v, p->Hq, (int64_t)p->B * p->Sq,
                     (int64_t)p->Hq * p->d_v, kTile)))
        s = ATTN_ERR_CUDA;
      else if ((tile128 ? launch_bwd_dq128(a, nsm, sq) : launch_bwd_dq(a, nsm, st)) != cudaSuccess)
        s = ATTN_ERR_CUDA;
    }
    trace(ATTN_TRACE_DQ, true, sq);
  }
  if (ax) {
    if (cudaEventRecord(ax->join, sq) != cudaSuccess ||
        cudaStreamWaitEvent(st, ax->join, 0) != cudaSuccess)
      s = ATTN_ERR_CUDA;
  }
  return s;
}

attn_status_t attn_read_status(const void* ws, void* stream, attn_stats_t* stats) {
  if (!ws) return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (stats) {
    stats->status = h.status;
    stats->path = h.path;
    stats->reason = h.reason;
    stats->dq_mode = h.dq_mode;
    stats->tile_pairs = h.tile_pairs;
    stats->wait_site = h.status != 0 ? h.where : 0;
    stats->reserved = 0;
  }
  return h.status == 0 ? ATTN_OK : static_cast<attn_status_t>(h.status);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward without a caller-supplied workspace.
//
// Some callers cannot allocate device memory when they run attention: plugin
// hosts that hand a kernel its inputs and outputs but no workspace, runtimes
// that plan all device memory at initialisation and forbid allocation
// afterwards, and latency-critical loops where cudaMalloc's implicit device
// synchronisation is not acceptable.  For them the forward's scratch (the
// normalised segment metadata, chunk summaries and tile ranges) lives in one
// fixed array in device memory that this library owns for the lifetime of the
// process on every GPU that loads it.
namespace attn {
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // = ATTN_FWD_NOALLOC_SCRATCH_BYTES
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the symbol name is only a host-side stand-in, never a device pointer.
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[256] = {};

attn_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return ATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" attn_status_t attn_fwd_noalloc(const attn_params_t* p, void* o, float* lse,
                                          void* stream) {
  attn_status_t s = validate(p);
  if (s != ATTN_OK) return s;
  if (p->dtype == ATTN_DTYPE_FP8_E4M3) return ATTN_ERR_UNSUPPORTED;  // workspace entry points only
  if (!o || !lse || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  const Plan pl = make_plan(p);
  if (pl.fwd_total > kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  if ((s = noalloc_scratch(&ws)) != ATTN_OK) return s;
  // launch_meta zeroes the header (status word, work counters, grid-barrier
  // count) with a cudaMemsetAsync on `stream` before the cooperative metadata
  // kernel, which needs that count at zero when it starts; every other scratch
  // array is fully written before it is read.
  return attn_fwd(p, o, lse, ws, kNoAllocScratchBytes, stream);
}
