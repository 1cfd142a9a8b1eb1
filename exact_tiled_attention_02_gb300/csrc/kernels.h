// kernels.h -- internal interface between the C-ABI layer (fa_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Arguments shared by every forward kernel.  Arrays are [B,H,N,d] row-major;
// lse is [B,H,N].  window_r < 0 means unmasked.
struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;  // may be null
  int BH;      // B * H
  int N;
  int d;
  int window_r;
  float scale;       // multiplies raw scores
  float scale_log2;  // scale * log2(e)
  unsigned int* status;
  unsigned long long wait_ns;
};

struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;  // [B,H,N,d] fp32 workspace
  // [B,H,Npad] workspace rows, Npad = N rounded up to 128.  d = 96, 128: fp32
  // -lse_i * log2(e) (-inf in padding rows) and -D_i = -sum_k dO_ik O_ik (0 in
  // padding rows).  d = 64: 16-byte rows of three bf16 terms of -lse_i / scale
  // (-1e30 in padding rows) and of -D_i (0), then five zeros.
  float* lse2;
  float* dsum;
  // Tail split of the bf16 backward without a window: the
  // key tiles [n_full, n_full + n_split) of the (head, key tile) order run as
  // two CTAs each, over the first and the second half of their query tiles,
  // so that a last, partly filled wave of CTAs takes about half as long.
  // Both halves add their fp32 dV and scale * dK rows into kv_part
  // ([n_split][2][128][d], dV first; zeroed by the prep kernel), and the dQ
  // kernel converts those rows to bf16.  n_split = 0: every tile is whole.
  float* kv_part;
  int n_full;
  int n_split;
  int BH;
  int N;
  int d;
  int window_r;
  float scale;
  float scale_log2;
  unsigned int* status;
  unsigned long long wait_ns;
};

// 3-D TMA maps over a [BH, N, d] bf16 array: dims (d, N, BH), box
// (64, rows, 1), 128-byte swizzle, zero fill out of bounds.
struct FwdMaps {
  CUtensorMap q, k, v;
};
struct BwdMaps {
  CUtensorMap q, k, v, dO;
  CUtensorMap dq_acc;  // fp32 [BH, N, d] accumulator: dims (d, N, BH), box (32, 128, 1), 128-byte swizzle
  CUtensorMap dk, dv;  // the bf16 outputs, for TMA stores: as q (box (64, 128, 1), 128-byte swizzle)
};

// Launchers (each returns the launch's cudaError_t).
cudaError_t launch_fwd_f32_simt(const FwdParams& p, cudaStream_t s);
cudaError_t launch_fwd_bf16_tc(const FwdParams& p, const FwdMaps& m, cudaStream_t s);
cudaError_t launch_fwd_bf16_d256(const FwdParams& p, const FwdMaps& m, cudaStream_t s);
// Windowed forward at d = 64, 96, 128 for bands of radius <= 128: one
// 128-row query tile per CTA, two CTAs per SM (fwd_bf16_win_sm103.cu).
cudaError_t launch_fwd_bf16_win(const FwdParams& p, const FwdMaps& m, cudaStream_t s);
// cuTensorMapEncodeTiled's signature (resolved at run time by the C-ABI layer)
typedef CUresult (*EncodeTiledFnPtr)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                     const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// fp32 forward on the tensor cores by the 3xTF32 split (d <= 128): workspace =
// Q hi, Q lo, K hi, K lo as [BH][N][DP] fp32, then V^T hi, V^T lo as
// [BH][DP][Npad] fp32 (DP = 64 for d <= 64, else 128; Npad = N rounded up
// to 64), each 256-byte aligned.  For d > 64 the Q sections are empty (that
// kernel splits Q itself, into tensor memory).  off (may be null) receives
// the six section offsets.
size_t f32_tc_workspace_layout(int BH, int N, int d, size_t off[6]);
cudaError_t launch_fwd_f32_tc(const FwdParams& p, void* workspace, EncodeTiledFnPtr encode, cudaStream_t s);
// 64 < d <= 128 (fwd_f32_tc128_sm103.cu): maps over K hi / lo ([BH][N][128],
// box (32, 64, 1)) and V^T hi / lo ([BH][128][Npad], box (32, 128, 1)), fp32,
// 128-byte swizzle.
struct Tc128Maps {
  CUtensorMap kh, kl, vh, vl;
};
cudaError_t launch_fwd_f32_tc128_main(const FwdParams& p, const Tc128Maps& m, cudaStream_t s);
// Key-major forward (comparison schedule): one launch per key tile, then a
// finishing launch; workspace = fp32 O~ [BH,N,d], then m and l [BH,N], each
// section 256-byte aligned.
cudaError_t launch_fwd_keymajor(const FwdParams& p, const FwdMaps& m, void* workspace, cudaStream_t s);
size_t keymajor_workspace_layout(int BH, int N, int d, size_t* off_m, size_t* off_l);
cudaError_t launch_bwd_bf16_tc(const BwdParams& p, const BwdMaps& m, cudaStream_t s);
// The backward's prep kernel (row terms, dQ accumulator zeroed) and final dQ
// cast (bwd_prep_sm103.cu), shared by every head dimension.
cudaError_t launch_bwd_prep(const BwdParams& p, cudaStream_t s);
cudaError_t launch_bwd_dq(const BwdParams& p, cudaStream_t s);
// The main kernel of the d = 64 backward (one CTA per 128-key tile; grid = key tiles x B*H).
cudaError_t launch_bwd_main_d64(const BwdParams& p, const BwdMaps& m, unsigned grid, cudaStream_t s);
cudaError_t launch_bwd_f32_simt(const BwdParams& p, cudaStream_t s);
// Byte size of the backward workspace and the offsets of its lse2 / dsum
// sections (dq_acc is at offset 0); rows are padded to multiples of 128.
size_t bwd_workspace_layout(int BH, int N, int d, size_t* off_lse2, size_t* off_dsum, size_t* off_part);
cudaError_t launch_selftest_wait(unsigned int* status, unsigned long long limit_ns, cudaStream_t s);
// fa_bwd's host-side argument checks, without those of the workspace
// (fa_api.cu); FA_OK or the status fa_bwd would return.
fa_status check_bwd_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, const void* dq, const void* dk, const void* dv, int B, int H, int N, int d,
                         float scale, int window, fa_dtype dt);

// Row counts of the tiles the TMA boxes use (host needs them for the maps).
constexpr int kFwdBlockRows = 128;  // query rows per CTA tile
constexpr int kFwdBlockCols = 128;  // keys per K/V tile
constexpr int kBwdBlockRows = 128;  // query rows per step of the backward
constexpr int kBwdBlockCols = 128;  // keys per CTA of the backward
constexpr int kMaxSplitTiles = 128;  // bound on BwdParams::n_split (sizes the kv_part workspace)

}  // namespace fa
