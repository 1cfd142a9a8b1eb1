// bwd_bf16_sm103.cu -- exact attention backward by recomputation for GB300
// (sm_103a), bf16 in / fp32 accumulate, d = 128.
//
// "Flash attention and efficient attention -- Hinglish notes", "Backward Pass:
// Recomputation": the N x N matrices S and P are not stored by the forward and
// not read here; they are rebuilt on chip, one tile at a time, from Q, K and
// the forward's logsumexp:  P_ij = exp(scale q_i.k_j - lse_i).  The gradient
// formulas are the derivative of the forward definition (the pages print
// none): dV = P^T dO, dP = dO V^T, dS = P o (dP - D) with
// D_i = sum_j P_ij dP_ij = sum_k dO_ik O_ik, dQ = scale dS K, dK = scale dS^T Q.
//
// Three kernels:
//   bwd_prep     D_i = rowsum(dO o O) and lse_i * log2(e) into the workspace
//                (rows padded to a multiple of 64: D = 0, lse = +inf, so padded
//                query rows get P = 0), and the fp32 dQ accumulator zeroed.
//   bwd_main     one CTA per 128-key tile of one (batch, head): K_j, V_j stay
//                in shared memory; the CTA walks the 64-row query tiles that
//                can see its keys (only in-band tiles when windowed) and, per
//                tile, issues five tcgen05.mma:
//                  S^T  = K_j Q_i^T        (M=128 keys, N=64 queries, K=d)
//                  dP^T = V_j dO_i^T       (M=128, N=64, K=d)
//                  dV  += P^T dO_i         (M=128, N=d, K=64)
//                  dK  += dS^T Q_i         (M=128, N=d, K=64)
//                  dQ^T = K_j^T dS^T       (M=d, N=64, K=128 keys)
//                dV and dK accumulate in tensor memory for the whole loop; the
//                dQ^T tile is added to the fp32 accumulator with coalesced
//                atomic adds (32 consecutive d of one query row per warp op).
//   bwd_dq       dQ = bf16(scale * accumulator).
// Warp roles in bwd_main (320 threads):
//   warps 0-3  P / dS: thread t owns key row t (TMEM lane t)
//   warps 4-7  dQ^T read-out: thread t owns head-dimension index t
//   warp  8    TMA / bulk-copy producer
//   warp  9    TMEM owner + MMA issuer
// Tensor memory columns: S^T [0,64), dP^T [64,128), dQ^T [128,192),
// dV [256,384), dK [384,512).
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int BM = 64;    // query rows per step
constexpr int BN = 128;   // keys per CTA
constexpr int D = 128;    // head dimension
constexpr int STAGES = 2; // Q/dO/lse/D ring depth
constexpr int kThreads = 320;
constexpr int kTmemCols = 512;
constexpr uint32_t TM_S = 0, TM_DP = 64, TM_DQ = 128, TM_DV = 256, TM_DK = 384;

constexpr int K_BYTES = BN * D * 2;     // 32 KB (two 64-column boxes of 128 rows)
constexpr int Q_BYTES = BM * D * 2;     // 16 KB (two boxes of 64 rows)
constexpr int VEC_BYTES = BM * 4;       // 256 B of lse*log2e or of D
constexpr int PT_BYTES = BN * BM * 2;   // 16 KB: P^T (and dS^T) as [128 keys][64 queries] bf16
// one ring stage: Q_i, dO_i, lse_i * log2e, D_i (padded to 1 KB multiples so
// every TMA destination stays 1024-byte aligned)
constexpr int ST_Q = 0, ST_DO = Q_BYTES, ST_LSE = 2 * Q_BYTES, ST_D = 2 * Q_BYTES + VEC_BYTES;
constexpr int STAGE_STRIDE = ((2 * Q_BYTES + 2 * VEC_BYTES + 1023) / 1024) * 1024;
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + K_BYTES;
constexpr int OFF_STAGE = OFF_V + K_BYTES;
constexpr int OFF_PT = OFF_STAGE + STAGES * STAGE_STRIDE;
constexpr int OFF_DST = OFF_PT + PT_BYTES;
constexpr int OFF_BAR = OFF_DST + PT_BYTES;
// kv_full, q_full[S], q_empty[S], then s_full, s_free, dp_full, dp_free, p_full,
// p_free, ds_full, ds_free, dq_full, dq_free, fin, drain
constexpr int NBAR = 1 + 2 * STAGES + 12;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot + abort flag
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(STAGE_STRIDE >= BN * D * 2, "a stage must hold one bf16 [128 x 128] epilogue tile");

struct Bars {
  uint32_t base;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t q_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t q_empty(int s) const { return base + 8 * (1 + STAGES + s); }
  __device__ uint32_t at(int i) const { return base + 8 * (1 + 2 * STAGES + i); }
  __device__ uint32_t s_full() const { return at(0); }
  __device__ uint32_t s_free() const { return at(1); }
  __device__ uint32_t dp_full() const { return at(2); }
  __device__ uint32_t dp_free() const { return at(3); }
  __device__ uint32_t p_full() const { return at(4); }
  __device__ uint32_t p_free() const { return at(5); }
  __device__ uint32_t ds_full() const { return at(6); }
  __device__ uint32_t ds_free() const { return at(7); }
  __device__ uint32_t dq_full() const { return at(8); }
  __device__ uint32_t dq_free() const { return at(9); }
  __device__ uint32_t fin() const { return at(10); }
  __device__ uint32_t drain() const { return at(11); }
};

__device__ __forceinline__ int npad64(int n) { return (n + 63) & ~63; }

// ---------------------------------------------------------------------------
// bwd_prep: one warp per (padded) query row
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ lse, float* __restrict__ lse2,
                                                         float* __restrict__ dsum, float* __restrict__ dq_acc, int BH,
                                                         int N, int d) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int np = npad64(N);
  const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;  // padded row index
  if (row >= static_cast<long long>(BH) * np) return;
  const long long bh = row / np;
  const int i = static_cast<int>(row % np);
  if (i >= N) {
    if (lane == 0) {
      lse2[row] = INFINITY;
      dsum[row] = 0.f;
    }
    return;
  }
  const long long src = (bh * N + i) * d;
  float acc = 0.f;
  // d = 128: each lane reads 4 consecutive bf16 (8 bytes) of O and dO
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
    dsum[row] = acc;
    lse2[row] = lse[bh * N + i] * 1.4426950408889634f;
  }
  float4* z = reinterpret_cast<float4*>(dq_acc + src);
  for (int c = lane; c < d / 4; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------
// bwd_dq: dQ = bf16(scale * acc), 8 elements per thread
// ---------------------------------------------------------------------------
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

// ---------------------------------------------------------------------------
// bwd_main
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_bf16_sm103_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                             const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sK = sb + OFF_K, sV = sb + OFF_V, sStage = sb + OFF_STAGE, sPT = sb + OFF_PT, sDST = sb + OFF_DST;
  Bars bar{sb + OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const WaitCtl wc{p.status, abort_flag, p.wait_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, r = p.window_r;
  const int nkt = (N + BN - 1) / BN;
  const int bh = blockIdx.x / nkt;
  const int k0 = (blockIdx.x % nkt) * BN;
  const int np = npad64(N);

  // query tiles that can see this key tile
  int t_lo = 0, t_hi = (N + BM - 1) / BM;
  if (r >= 0) {
    t_lo = max(0, k0 - r) / BM;
    t_hi = (min(N, k0 + BN + r) + BM - 1) / BM;
  }
  const int nsteps = t_hi - t_lo;

  if (threadIdx.x == 0) {
    mbar_init(bar.kv_full(), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar.q_full(s), 1);
      mbar_init(bar.q_empty(s), 1);
    }
    mbar_init(bar.s_full(), 1);
    mbar_init(bar.s_free(), 4);
    mbar_init(bar.dp_full(), 1);
    mbar_init(bar.dp_free(), 4);
    mbar_init(bar.p_full(), 4);
    mbar_init(bar.p_free(), 1);
    mbar_init(bar.ds_full(), 4);
    mbar_init(bar.ds_free(), 1);
    mbar_init(bar.dq_full(), 1);
    mbar_init(bar.dq_free(), 4);
    mbar_init(bar.fin(), 1);
    mbar_init(bar.drain(), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
  };

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmq);
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      prefetch_tensormap(&tmdo);
      mbar_arrive_expect_tx(bar.kv_full(), 2 * K_BYTES);
      for (int b = 0; b < 2; ++b) {
        tma_load_3d(sK + b * BN * 128, &tmk, bar.kv_full(), b * 64, k0, bh);
        tma_load_3d(sV + b * BN * 128, &tmv, bar.kv_full(), b * 64, k0, bh);
      }
      int issued = 0;
      for (int it = 0; it < nsteps; ++it) {
        const int st = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!mbar_wait(bar.q_empty(st), ph ^ 1, wc)) break;
        const int q0 = (t_lo + it) * BM;
        const uint32_t base = sStage + st * STAGE_STRIDE;
        mbar_arrive_expect_tx(bar.q_full(st), 2 * Q_BYTES + 2 * VEC_BYTES);
        for (int b = 0; b < 2; ++b) {
          tma_load_3d(base + ST_Q + b * BM * 128, &tmq, bar.q_full(st), b * 64, q0, bh);
          tma_load_3d(base + ST_DO + b * BM * 128, &tmdo, bar.q_full(st), b * 64, q0, bh);
        }
        const size_t vrow = static_cast<size_t>(bh) * np + q0;
        bulk_load(base + ST_LSE, p.lse2 + vrow, VEC_BYTES, bar.q_full(st));
        bulk_load(base + ST_D, p.dsum + vrow, VEC_BYTES, bar.q_full(st));
        issued = it + 1;
      }
      if (*abort_flag) {
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.kv_full(), 0, drain);
        for (int it = max(0, issued - STAGES); it < issued; ++it)
          mbar_wait(bar.q_full(it % STAGES), (it / STAGES) & 1, drain);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(BN, BM, 0, 0);   // K_j (K-major) x Q_i (K-major)
      constexpr uint32_t id_dv = idesc_bf16_f32(BN, D, 0, 1);   // P^T (K-major) x dO_i (MN-major)
      constexpr uint32_t id_dq = idesc_bf16_f32(D, BM, 1, 1);   // K_j^T (MN-major) x dS^T (MN-major)
      bool ok = mbar_wait(bar.kv_full(), 0, wc);
      // S^T and dP^T for step it (needs the stage loaded and both TMEM tiles free)
      auto issue_s_dp = [&](int it) -> bool {
        const int st = it % STAGES;
        const uint32_t base = sStage + st * STAGE_STRIDE;
        if (!mbar_wait(bar.q_full(st), (it / STAGES) & 1, wc)) return false;
        if (it > 0 && !mbar_wait(bar.s_free(), (it - 1) & 1, wc)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offk = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t offq = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + TM_S, sdesc_sw128(sK + offk, 16, 1024), sdesc_sw128(base + ST_Q + offq, 16, 1024),
                      id_s, kk > 0);
        }
        mma_commit(bar.s_full());
        if (it > 0 && !mbar_wait(bar.dp_free(), (it - 1) & 1, wc)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offk = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t offq = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + TM_DP, sdesc_sw128(sV + offk, 16, 1024), sdesc_sw128(base + ST_DO + offq, 16, 1024),
                      id_s, kk > 0);
        }
        mma_commit(bar.dp_full());
        return true;
      };
      if (ok) ok = issue_s_dp(0);
      for (int it = 0; ok && it < nsteps; ++it) {
        const int st = it % STAGES;
        const uint32_t base = sStage + st * STAGE_STRIDE;
        if (it + 1 < nsteps && !issue_s_dp(it + 1)) break;
        // dV += P^T dO_i
        if (!mbar_wait(bar.p_full(), it & 1, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_bf16_ss(tmem + TM_DV, sdesc_sw128(sPT + kk * 32, 16, 1024),
                      sdesc_sw128(base + ST_DO + kk * 16 * 128, BM * 128, 1024), id_dv, (it > 0 || kk > 0));
        mma_commit(bar.p_free());
        // dK += dS^T Q_i ; dQ^T = K_j^T dS^T
        if (!mbar_wait(bar.ds_full(), it & 1, wc)) break;
        if (it > 0 && !mbar_wait(bar.dq_free(), (it - 1) & 1, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_bf16_ss(tmem + TM_DK, sdesc_sw128(sDST + kk * 32, 16, 1024),
                      sdesc_sw128(base + ST_Q + kk * 16 * 128, BM * 128, 1024), id_dv, (it > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ss(tmem + TM_DQ, sdesc_sw128(sK + kk * 16 * 128, BN * 128, 1024),
                      sdesc_sw128(sDST + kk * 16 * 128, 8192, 1024), id_dq, kk > 0);
        mma_commit(bar.ds_free());
        mma_commit(bar.dq_full());
        mma_commit(bar.q_empty(st));
      }
      mma_commit(bar.fin());
      mma_commit(bar.drain());
      WaitCtl drain{nullptr, nullptr, wc.limit_ns};
      mbar_wait(bar.drain(), 0, drain);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------ dQ^T read-out
    const int dd = (warp - 4) * 32 + lane;  // head-dimension index == TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp - 4) * 32) << 16);
    float* acc_base = p.dq_acc + static_cast<size_t>(bh) * N * D + dd;
    for (int it = 0; it < nsteps; ++it) {
      if (!warp_wait(bar.dq_full(), it & 1)) break;
      tc_fence_after();
      uint32_t v[BM];
      tmem_ld_32x32b_x32(tl + TM_DQ, &v[0]);
      tmem_ld_32x32b_x32(tl + TM_DQ + 32, &v[32]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.dq_free());
      const int q0 = (t_lo + it) * BM;
      const int cnt = min(BM, N - q0);
#pragma unroll
      for (int c = 0; c < BM; ++c)
        if (c < cnt) red_add_f32(acc_base + static_cast<size_t>(q0 + c) * D, __uint_as_float(v[c]));
    }
  } else {
    // ------------------------------------------------------------- P / dS
    const int row = threadIdx.x;  // key row within the tile == TMEM lane
    const int kj = k0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < nsteps; ++it) {
      const int st = it % STAGES;
      const uint32_t base = sStage + st * STAGE_STRIDE;
      const int q0 = (t_lo + it) * BM;
      if (!warp_wait(bar.s_full(), it & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[BM];
      tmem_ld_32x32b_x32(tl + TM_S, &sv[0]);
      tmem_ld_32x32b_x32(tl + TM_S + 32, &sv[32]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.s_free());
      // P^T row: P_ij = 2^(s * scale * log2e - lse_i * log2e); padded query rows have lse = +inf
      if (!warp_wait(bar.q_full(st), (it / STAGES) & 1)) {
        ok = false;
        break;
      }
      const float* lse2 = reinterpret_cast<const float*>(smem + (base - sb) + ST_LSE);
      const float* dsv = reinterpret_cast<const float*>(smem + (base - sb) + ST_D);
      const bool key_ok = kj < N;
      const bool edge = r >= 0 && !(q0 >= kj - r && q0 + BM - 1 <= kj + r);
      float pr[BM];
#pragma unroll
      for (int c = 0; c < BM; ++c) {
        float pv = ex2_approx(fmaf(__uint_as_float(sv[c]), sl, -lse2[c]));
        if (edge && abs(q0 + c - kj) > r) pv = 0.f;
        pr[c] = key_ok ? pv : 0.f;
      }
      // P^T buffer is free once the previous dV MMA has completed
      if (it > 0 && !warp_wait(bar.p_free(), (it - 1) & 1)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int c16 = 0; c16 < BM / 8; ++c16) {
        const uint32_t addr = sPT + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
        st_shared_v4(addr, pack_bf16x2(pr[8 * c16], pr[8 * c16 + 1]), pack_bf16x2(pr[8 * c16 + 2], pr[8 * c16 + 3]),
                     pack_bf16x2(pr[8 * c16 + 4], pr[8 * c16 + 5]), pack_bf16x2(pr[8 * c16 + 6], pr[8 * c16 + 7]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full());

      // dS^T row = P^T o (dP^T - D)
      if (!warp_wait(bar.dp_full(), it & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dpv[BM];
      tmem_ld_32x32b_x32(tl + TM_DP, &dpv[0]);
      tmem_ld_32x32b_x32(tl + TM_DP + 32, &dpv[32]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.dp_free());
      if (it > 0 && !warp_wait(bar.ds_free(), (it - 1) & 1)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int c16 = 0; c16 < BM / 8; ++c16) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 8 * c16 + 2 * e;
          w[e] = pack_bf16x2(pr[c] * (__uint_as_float(dpv[c]) - dsv[c]),
                             pr[c + 1] * (__uint_as_float(dpv[c + 1]) - dsv[c + 1]));
        }
        st_shared_v4(sDST + row * 128 + (((c16 & 7) ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.ds_full());
    }

    // ------------------------------------------------------------ epilogue
    const bool have = ok && warp_wait(bar.fin(), 0);
    // stage bf16 dV and scale*dK rows in the (idle) Q/dO stage buffers
    const uint32_t stage_dv = sStage, stage_dk = sStage + STAGE_STRIDE;
    if (have) {
      tc_fence_after();
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t tcol = which == 0 ? TM_DV : TM_DK;
        const float mul = which == 0 ? 1.f : p.scale;
        const uint32_t dst = which == 0 ? stage_dv : stage_dk;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tl + tcol + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int c16 = c * 4 + q4;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2 * e]) * mul, __uint_as_float(v[q4 * 8 + 2 * e + 1]) * mul);
            // row-major [128 keys][128 d] bf16 with 16-byte chunks swizzled by row
            st_shared_v4(dst + row * 256 + (((c16 & 15) ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
    tc_fence_before();
    named_bar_sync(1, 128);
    if (have && !*abort_flag) {
      uint8_t* gdv = reinterpret_cast<uint8_t*>(p.dv) + (static_cast<size_t>(bh) * N + k0) * D * 2;
      uint8_t* gdk = reinterpret_cast<uint8_t*>(p.dk) + (static_cast<size_t>(bh) * N + k0) * D * 2;
      for (int idx = row; idx < BN * 16; idx += 128) {
        const int rr = idx >> 4, c16 = idx & 15;
        if (k0 + rr < N) {
          const uint32_t off = rr * 256 + (((c16 & 15) ^ (rr & 7)) << 4);
          st_global_v4(gdv + static_cast<size_t>(rr) * 256 + c16 * 16, ld_shared_v4(stage_dv + off));
          st_global_v4(gdk + static_cast<size_t>(rr) * 256 + c16 * 16, ld_shared_v4(stage_dk + off));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t bwd_workspace_layout(int BH, int N, int d, size_t* off_lse2, size_t* off_dsum) {
  const size_t rows = static_cast<size_t>(BH) * N;
  const size_t prow = static_cast<size_t>(BH) * ((N + 63) & ~63);
  const size_t acc = (rows * d * sizeof(float) + 255) & ~size_t(255);
  const size_t vec = (prow * sizeof(float) + 255) & ~size_t(255);
  if (off_lse2) *off_lse2 = acc;
  if (off_dsum) *off_dsum = acc + vec;
  return acc + 2 * vec;
}

cudaError_t launch_bwd_bf16_tc(const BwdParams& p, const BwdMaps& m, cudaStream_t s) {
  if (p.d != D) return cudaErrorNotSupported;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_bf16_sm103_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long np = (p.N + 63) & ~63;
  const long long prep_rows = static_cast<long long>(p.BH) * np;
  const long long prep_blocks = (prep_rows + 7) / 8;
  const long long nkt = (p.N + BN - 1) / BN;
  const long long grid = nkt * p.BH;
  const long long n8 = static_cast<long long>(p.BH) * p.N * p.d / 8;
  if (prep_blocks > 0x7fffffffLL || grid > 0x7fffffffLL || (n8 + 255) / 256 > 0x7fffffffLL)
    return cudaErrorInvalidConfiguration;
  fa_bwd_prep_kernel<<<static_cast<unsigned>(prep_blocks), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(p.o), static_cast<const __nv_bfloat16*>(p.dO), p.lse, p.lse2, p.dsum,
      p.dq_acc, p.BH, p.N, p.d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_bf16_sm103_kernel<<<static_cast<unsigned>(grid), kThreads, SMEM_BYTES, s>>>(m.q, m.k, m.v, m.dO, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_dq_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, s>>>(
      p.dq_acc, static_cast<__nv_bfloat16*>(p.dq), n8, p.scale);
  return cudaGetLastError();
}

}  // namespace fa
