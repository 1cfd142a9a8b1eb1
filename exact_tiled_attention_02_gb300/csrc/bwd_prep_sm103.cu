// bwd_prep_sm103.cu -- the element-wise kernels around the attention
// backward's main kernels (bf16, every head dimension), and its workspace.
//
// "Flash attention and efficient attention -- Hinglish notes", "Backward
// Pass: Recomputation": the backward rebuilds P from the forward's logsumexp;
// the per-row quantities it needs besides lse are computed here.  The
// gradient formulas are the derivative of the forward definition (the pages
// print none): D_i = sum_j P_ij dP_ij = sum_k dO_ik O_ik.
//
//   bwd_prep  per (padded) query row: -D_i and the lse term the main kernel
//             uses (-lse_i log2 e for d = 96 / 128; for d = 64, -lse_i / scale
//             and -D_i as three bf16 terms each, the operand rows that kernel's
//             tensor core adds in), and the row of the fp32 dQ accumulator
//             zeroed.  Rows are padded to a multiple of 128: padding rows get
//             D = 0 and a term that makes their P 0.
//   bwd_dq    dQ = bf16(scale * accumulator).
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

__host__ __device__ __forceinline__ int npad128(int n) { return (n + 127) & ~127; }

// Three bf16 terms whose sum is x to fp32 precision (each term takes what the
// previous ones left; the differences are exact in fp32), with five zeros:
// one 16-byte row of a K = 16 operand whose other 8 elements are zero.
__device__ __forceinline__ uint4 bf16_split3_row(float x) {
  const __nv_bfloat16 h1 = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h1);
  const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
  const __nv_bfloat16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
  uint4 v;
  v.x = static_cast<uint32_t>(__bfloat16_as_ushort(h1)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h2)) << 16);
  v.y = static_cast<uint32_t>(__bfloat16_as_ushort(h3));
  v.z = 0u;
  v.w = 0u;
  return v;
}

// One warp per (padded) row; each pass, lane l reads 4 consecutive bf16
// (8 bytes) of O and dO at column 4l.  (Four rows per warp with all loads
// issued first measured 30% slower.)
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ lse, float* __restrict__ lse2,
                                                         float* __restrict__ dsum, float* __restrict__ dq_acc, int BH,
                                                         int N, int d, float inv_scale, int split) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int np = npad128(N);
  const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;  // padded row index
  if (row >= static_cast<long long>(BH) * np) return;
  const long long bh = row / np;
  const int i = static_cast<int>(row % np);
  if (i >= N) {
    if (lane == 0) {
      if (split) {
        // -lse / scale far below any logit: the row's P underflows to 0
        reinterpret_cast<uint4*>(lse2)[row] = bf16_split3_row(-1e30f);
        reinterpret_cast<uint4*>(dsum)[row] = bf16_split3_row(0.f);
      } else {
        lse2[row] = -INFINITY;
        dsum[row] = 0.f;
      }
    }
    return;
  }
  const long long src = (bh * N + i) * d;
  float acc = 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    const uint2 ov = *reinterpret_cast<const uint2*>(o + src + c);
    const uint2 gv = *reinterpret_cast<const uint2*>(dO + src + c);
    const __nv_bfloat162* op = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float2 a = __bfloat1622float2(op[e]);
      const float2 b = __bfloat1622float2(gp[e]);
      acc = fmaf(a.x, b.x, acc);
      acc = fmaf(a.y, b.y, acc);
    }
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) {
    if (split) {
      reinterpret_cast<uint4*>(lse2)[row] = bf16_split3_row(-lse[bh * N + i] * inv_scale);
      reinterpret_cast<uint4*>(dsum)[row] = bf16_split3_row(-acc);
    } else {
      dsum[row] = -acc;
      lse2[row] = -lse[bh * N + i] * 1.4426950408889634f;
    }
  }
  float4* z = reinterpret_cast<float4*>(dq_acc + src);
  for (int c = lane; c < d / 4; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = bf16(scale * acc), 8 elements per thread
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                       long long n8, float scale) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 out;
  out.x = pack_bf16x2(a.x * scale, a.y * scale);
  out.y = pack_bf16x2(a.z * scale, a.w * scale);
  out.z = pack_bf16x2(b.x * scale, b.y * scale);
  out.w = pack_bf16x2(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = out;
}

}  // namespace

size_t bwd_workspace_layout(int BH, int N, int d, size_t* off_lse2, size_t* off_dsum) {
  const size_t rows = static_cast<size_t>(BH) * N;
  const size_t prow = static_cast<size_t>(BH) * npad128(N);
  const size_t acc = (rows * d * sizeof(float) + 255) & ~size_t(255);
  // d = 64 stores each row's value as three bf16 terms in a 16-byte row
  const size_t vec = (prow * (d == 64 ? 16 : sizeof(float)) + 255) & ~size_t(255);
  if (off_lse2) *off_lse2 = acc;
  if (off_dsum) *off_dsum = acc + vec;
  return acc + 2 * vec;
}

cudaError_t launch_bwd_prep(const BwdParams& p, cudaStream_t s) {
  const long long rows = static_cast<long long>(p.BH) * npad128(p.N);
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_bwd_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(p.o), static_cast<const __nv_bfloat16*>(p.dO), p.lse, p.lse2, p.dsum,
      p.dq_acc, p.BH, p.N, p.d, 1.f / p.scale, p.d == 64);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdParams& p, cudaStream_t s) {
  const long long n8 = static_cast<long long>(p.BH) * p.N * p.d / 8;
  if ((n8 + 255) / 256 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_bwd_dq_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, s>>>(
      p.dq_acc, static_cast<__nv_bfloat16*>(p.dq), n8, p.scale);
  return cudaGetLastError();
}

}  // namespace fa
