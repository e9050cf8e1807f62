// Backward pass: dQ, dK, dV (and dBias) from O, dO and the forward's LSE.
//
//   bwd_pre      D = rowsum(dO * O) per (batch row, head, query) and LSE in
//                log2 units; zeroes the fp32 accumulators it is asked to.
//   dkdv, dq     (bwd_passes.cuh, one translation unit per element type)
//   dkdv         one persistent CTA per SM; a work item is one 128-row KV tile
//                of one KV head (and, when a broadcast bias gradient has to be
//                reduced, of every batch row / head sharing that bias slice).
//                The CTA loops *sequentially* over the query heads of the
//                group and every 64-row query tile that can see the KV tile,
//                accumulating dK and dV in tensor memory.  No accumulation
//                depends on the order in which CTAs run, which is the
//                grid-order hazard of the maxdiffusion PR #485 review (dK/dV
//                initialised and written by whichever grid step happens to run
//                first / last); the fused single-pass structure (KV outer,
//                queries and GQA heads inner, dK/dV held across them) follows
//                that page's Summary.
//                Per query tile:  S^T = K Q^T,  P^T = exp2(S^T - LSE),
//                dP^T = V dO^T,  dS^T = P^T (dP^T - D),  dV += P^T dO,
//                dK += dS^T Q,  and in atomic-dQ mode dQ^T = K^T dS^T, added to an
//                fp32 buffer with red.global.add.
//   dq           deterministic dQ: one 128-row query tile per work item, KV
//                tiles visited in a fixed order, dQ accumulated in tensor
//                memory (recomputes S and dP: two more GEMMs than atomic mode).
//   dq_convert   fp32 dQ accumulator -> bf16 / fp16 in the caller's layout.
// A broadcast dBias is summed in an fp32 accumulator and finished (rounded to
// bf16 / fp16) inside the dK/dV pass by the last step that adds to each row.
//
// Gradient formulas: TransformerEngine PR #3516 (fused-attention backward:
// Q/K/V and optional bias gradients from the saved output and dO); dK/dV of a
// KV head sum over the query heads sharing it (maxdiffusion PR #485, Summary);
// the bias gradient is summed over the axes the bias is broadcast along.
#include <cmath>

#include "attn_internal.cuh"

namespace attn {
namespace {
using namespace sm103;

constexpr float kLog2e = 1.4426950408889634f;

// =========================================================== preprocess
// One warp per token: all Hq head rows of a token are Hq * DV * 2 contiguous
// bytes of O and of dO, read front to back.  Eight consecutive tokens per
// block; their D and LSE values go out through shared memory so each head's
// eight values are written as one 32-byte run of the [B, Hq, Sq] arrays.
constexpr int kPreMaxH = 256;

template <class E, int DV>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const KernelArgs a, int dq_mode_used) {
  constexpr int LPR = DV / 8;    // lanes per head row, 16 bytes each
  constexpr int HPI = 32 / LPR;  // head rows per warp-wide load
  __shared__ float dsm[kPreTok][kPreMaxH];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / LPR, l = lane % LPR;
  const int64_t ntok = (int64_t)a.B * a.Sq;
  const int64_t t0 = (int64_t)blockIdx.x * kPreTok;
  grid_dep_wait();  // O and LSE come from the forward
  grid_dep_launch();
  const int64_t tok = t0 + warp;
  if (tok < ntok) {
    const bf16* orow = a.o_in + tok * a.Hq * DV;
    const bf16* drow = a.d_o + tok * a.Hq * DV;
    for (int h0 = 0; h0 < a.Hq; h0 += 2 * HPI) {  // two loads of each array in flight
      uint4 o[2], d[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int h = h0 + u * HPI + sub;
        if (h < a.Hq) {
          o[u] = ld_nc_v4(orow + h * DV + l * 8);
          d[u] = ld_nc_v4(drow + h * DV + l * 8);
        } else {
          o[u] = d[u] = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t ow[4] = {o[u].x, o[u].y, o[u].z, o[u].w};
        const uint32_t dw[4] = {d[u].x, d[u].y, d[u].z, d[u].w};
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = fmaf(E::lo(ow[e]), E::lo(dw[e]), acc);
          acc = fmaf(E::hi(ow[e]), E::hi(dw[e]), acc);
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const int h = h0 + u * HPI + sub;
        if (l == 0 && h < a.Hq) dsm[warp][h] = acc;
      }
    }
  }
  __syncthreads();
  // thread v handles head v / 8 and token v % 8 of this block; the eight
  // tokens of a head are eight consecutive lanes (blockDim is a multiple of 8)
  for (int v0 = 0; v0 < a.Hq * kPreTok; v0 += blockDim.x) {
    const int v = v0 + threadIdx.x;
    const int h = v / kPreTok, j = v - h * kPreTok;
    const int64_t t = t0 + j;
    float part = 0.f;  // this token's share of the sink gradient
    if (v < a.Hq * kPreTok && t < ntok &&
        ATTN_CHECK(a, span_ok(((t / a.Sq) * a.Hq + h) * a.Sq + t % a.Sq, 1, ntok * a.Hq), 0x7201)) {
      const int b = static_cast<int>(t / a.Sq), i = static_cast<int>(t - (int64_t)b * a.Sq);
      const int64_t idx = ((int64_t)b * a.Hq + h) * a.Sq + i;
      const float D = dsm[j][h];
      a.Dvec[idx] = D;
      const float lse = a.lse_in[idx];
      a.lse2[idx] = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
      // dsink_h = -sum_i P_sink,i D_i with P_sink,i = exp(sink_h - LSE_i)
      if (a.dsink && lse > -INFINITY) part = -__expf(a.sink[h] - lse) * D;
    }
    if (a.dsink) {
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      part += __shfl_xor_sync(0xffffffffu, part, 4);
      if (j == 0 && v < a.Hq * kPreTok) a.sink_part[(int64_t)blockIdx.x * a.Hq + h] = part;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.hdr->dq_mode = dq_mode_used;
    // work counters of the dK/dV and dQ passes, which start after this kernel
    a.hdr->next_item[1] = a.hdr->next_item[2] = a.hdr->next_item[3] = 0;
  }
}

// =========================================================== sink gradient
// dsink[h] = sum over the preprocess blocks of their partials, one block per
// head, in a fixed order (strided per thread, then a fixed tree): the result
// does not depend on scheduling.
__global__ void __launch_bounds__(256) sink_reduce_kernel(const KernelArgs a, int nblocks) {
  __shared__ float red[256];
  const int h = blockIdx.x;
  float acc = 0.f;
  for (int k = threadIdx.x; k < nblocks; k += blockDim.x) acc += a.sink_part[(int64_t)k * a.Hq + h];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) a.dsink[h] = red[0];
}

// =========================================================== converts
template <class E>
__global__ void dq_convert_kernel(const KernelArgs a) {
  const int64_t per_tok = (int64_t)a.Hq * a.d_qk / 8;  // groups of 8 elements
  const int64_t n = (int64_t)a.B * a.Sq * per_tok;
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < n;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = v / per_tok;
    const int64_t e = (v - tok * per_tok) * 8;  // h * d_qk + d
    const float4 x0 = *reinterpret_cast<const float4*>(a.dq_acc + tok * a.Hq * a.d_qk + e);
    const float4 x1 = *reinterpret_cast<const float4*>(a.dq_acc + tok * a.Hq * a.d_qk + e + 4);
    uint4 o;
    o.x = E::pack(x0.x, x0.y);
    o.y = E::pack(x0.z, x0.w);
    o.z = E::pack(x1.x, x1.y);
    o.w = E::pack(x1.z, x1.w);
    if (ATTN_CHECK(a, dq_span_ok(a, tok, e, 8, a.dq + tok * a.dq_stride + e, 16), 0x7202))
      *reinterpret_cast<uint4*>(a.dq + tok * a.dq_stride + e) = o;
  }
}

int blocks_for(int64_t n, int per_block) {
  const int64_t b = (n + per_block - 1) / per_block;
  return static_cast<int>(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

}  // namespace
cudaError_t launch_bwd_pre(const KernelArgs& a, int zero_dq_acc, cudaStream_t st) {
  cudaError_t e;
  if (zero_dq_acc) {
    e = cudaMemsetAsync(a.dq_acc, 0, (size_t)a.B * a.Sq * a.Hq * a.d_qk * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  // dBias rows no dK/dV step writes stay 0; the fp32 accumulator of a
  // broadcast dBias is never cleared (see dbias_rows_written_before)
  const size_t nb = (size_t)a.bias_b * a.bias_h * a.Sq * a.Skv;
  if (a.dbias_mode != 0) {
    e = cudaMemsetAsync(a.dbias, 0, nb * sizeof(bf16), st);
    if (e != cudaSuccess) return e;
  }
  const int mode = zero_dq_acc ? 0 : 1;
  if (a.Hq > kPreMaxH) return cudaErrorInvalidValue;  // rejected on the host before launch
  const int64_t ntok = (int64_t)a.B * a.Sq;
  const unsigned blocks = static_cast<unsigned>((ntok + kPreTok - 1) / kPreTok);
  auto kern = a.elem_f16 ? (a.d_v == 64 ? bwd_pre_kernel<ElemF16, 64> : bwd_pre_kernel<ElemF16, 128>)
                         : (a.d_v == 64 ? bwd_pre_kernel<ElemBf16, 64> : bwd_pre_kernel<ElemBf16, 128>);
  return launch_pdl(kern, dim3(blocks), dim3(256), 0, st, a, mode);
}

cudaError_t launch_bwd_dkdv(const KernelArgs& a, bool atomic, int nsm, cudaStream_t st) {
  return a.elem_f16 ? launch_bwd_dkdv_t<ElemF16>(a, atomic, nsm, st)
                    : launch_bwd_dkdv_t<ElemBf16>(a, atomic, nsm, st);
}

cudaError_t launch_bwd_dq(const KernelArgs& a, int nsm, cudaStream_t st) {
  return a.elem_f16 ? launch_bwd_dq_t<ElemF16>(a, nsm, st) : launch_bwd_dq_t<ElemBf16>(a, nsm, st);
}

cudaError_t launch_dq_convert(const KernelArgs& a, cudaStream_t st) {
  const int64_t n = (int64_t)a.B * a.Sq * a.Hq * a.d_qk / 8;
  if (a.elem_f16)
    dq_convert_kernel<ElemF16><<<blocks_for(n, 256), 256, 0, st>>>(a);
  else
    dq_convert_kernel<ElemBf16><<<blocks_for(n, 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sink_reduce(const KernelArgs& a, cudaStream_t st) {
  const int64_t ntok = (int64_t)a.B * a.Sq;
  const int nblocks = static_cast<int>((ntok + kPreTok - 1) / kPreTok);
  sink_reduce_kernel<<<a.Hq, 256, 0, st>>>(a, nblocks);
  return cudaGetLastError();
}


}  // namespace attn

#ifdef ATTN_TIMELINE
// Debug builds only: copies the timeline records out and resets the counter.
extern "C" int attn_debug_timeline(unsigned long long* out, int cap) {
  cudaDeviceSynchronize();
  const int n = cap < attn::kTimelineCap ? cap : attn::kTimelineCap;
  cudaMemcpyFromSymbol(out, attn::g_timeline, sizeof(unsigned long long) * n);
  static unsigned long long zeros[attn::kTimelineCap];
  cudaMemcpyToSymbol(attn::g_timeline, zeros, sizeof(zeros));
  return n;
}
#endif
