// Internal definitions shared by the attention kernels and the host API.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

using bf16 = __nv_bfloat16;

constexpr int kChunk = 64;   // granularity of the per-chunk metadata summaries
constexpr int kTile = 128;   // query tile (forward, dQ pass) and KV tile (all kernels)
constexpr int kBwdQ = 64;    // query tile of the dK/dV pass

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
  int32_t status;      // device-side attn_status_t (timeouts)
  int32_t path;        // 0 fast, 1 general
  int32_t reason;      // attn_path_reason_t
  int32_t dq_mode;     // dQ mode used
  int64_t tile_pairs;  // scheduled (query tile, KV tile) pairs
  int32_t mismatch;    // bit0 ids differ, bit1 pos differ, bit2 nonstandard pos
  int32_t where;       // debug: which wait timed out (role * 16 + barrier)
};

// Summary of 64 consecutive tokens of one batch row.
struct ChunkInfo {
  int32_t min_id;   // smallest nonzero id (INT32_MAX if none)
  int32_t max_id;   // largest nonzero id (0 if none)
  int32_t min_pos;  // over tokens with nonzero id
  int32_t max_pos;
  int32_t uniform;  // 1: all 64 tokens exist and carry the same nonzero id
  int32_t pad[3];
};

// Everything a kernel needs; passed by value as a __grid_constant__ parameter
// (the tensor maps must live in parameter space for TMA).
struct KernelArgs {
  CUtensorMap tm_q;    // dims {d_qk, Hq, B*Sq},   box {64, 1, 128 or 64}
  CUtensorMap tm_k;    // dims {d_qk, Hkv, B*Skv}, box {64, 1, 128}
  CUtensorMap tm_v;    // dims {d_v, Hkv, B*Skv},  box {64, 1, 128}
  CUtensorMap tm_do;   // dims {d_v, Hq, B*Sq},    box {64, 1, 128 or 64}

  int B, Sq, Skv, Hq, Hkv, d_qk, d_v;
  int causal;
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
  const int2* q_tile_range;   // [B*n_qt]  KV token range of each 128-row query tile
  const int2* kv_tile_range;  // [B*n_kt]  query token range of each 128-row KV tile
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
  int dkdv_batch_loop;  // 1: one dK/dV work item loops over every batch row
  int dkdv_head_loop;   // 1: one dK/dV work item loops over every KV head
};

__device__ __forceinline__ bool path_general(const KernelArgs& a) {
  return *reinterpret_cast<const volatile int32_t*>(&a.hdr->path) != 0;
}

__device__ __forceinline__ void report_timeout(const KernelArgs& a, int where) {
  atomicExch(&a.hdr->status, 6 /* ATTN_ERR_DEVICE_TIMEOUT */);
  atomicExch(&a.hdr->where, where);
}

// Kernel launchers (defined in the kernel translation units).
cudaError_t launch_meta(const KernelArgs& a, int fmt, const int32_t* q_ids, const int32_t* q_pos,
                        const int32_t* kv_ids, const int32_t* kv_pos, const int32_t* cu_q,
                        const int32_t* cu_kv, int num_segments, int force_general,
                        cudaStream_t st);
cudaError_t launch_fwd(const KernelArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_bwd_pre(const KernelArgs& a, int zero_dq_acc, cudaStream_t st);
cudaError_t launch_bwd_dkdv(const KernelArgs& a, bool atomic_dq, int num_sms, cudaStream_t st);
cudaError_t launch_bwd_dq(const KernelArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_dq_convert(const KernelArgs& a, cudaStream_t st);
cudaError_t launch_dbias_convert(const KernelArgs& a, cudaStream_t st);

}  // namespace attn
