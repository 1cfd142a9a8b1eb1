// fwd_f32_tc128_sm103.cu -- tiled exact attention forward for float32 inputs
// on the tensor cores by the three-term tf32 split ("3xTF32"), for head
// dimensions 64 < d <= 128 (fwd_f32_tc_sm103.cu covers d <= 64 and holds
// the split kernels and the launcher).
//
// What it computes is the forward of fwd_f32_simt.cu ("Flash attention and
// efficient attention -- Hinglish notes", "The Standard Attention Problem",
// one key/value tile at a time with the running maximum / running sum merge
// of "Derivation: Incremental Softmax", Steps 1-3; the window of "Worked
// example Local Attention Window"), float32 in and out.  Every float32
// operand x is split as hi = tf32(x), lo = tf32(x - hi), and every product is
// taken as hi_a hi_b + hi_a lo_b + lo_a hi_b (the dropped lo_a lo_b term and
// the rounding of lo are below 2^-21 relative).
//
// At d = 128 the fp32 operands are twice the bf16 size, so shared memory
// cannot hold Q's two parts (128 KB) beside the K and V^T tiles.  Q lives in
// tensor memory instead, as the A operand of S = Q K^T: each softmax thread
// reads its own query row once, splits it and stores both parts (256
// columns).  Beside O (128 columns) that leaves two 64-column S buffers, P hi
// written over S; P lo goes to shared memory (two buffers) and enters P V as
// the A operand of the P_lo V_hi products.  The tensor core then runs
// S_0, S_1, P_0 V_0, S_2, P_1 V_1, ...: S_{j+1} runs while the softmax turns
// S_j into P_j.  (With P lo in tensor memory beside a single S buffer, each
// tile ran S_j, the softmax and P_j V_j in sequence, the tensor pipe busy 45%
// of cycles.)  K and V^T each stream through a single slot: K_{j+1} loads
// once S_j has read K_j, V_{j+1} once P_j V_j has read V_j.
//
// CTA: one 128-row query tile of one head, 192 threads: warps 0-3 softmax
// (thread = row = TMEM lane), warp 4 TMEM owner + MMA issuer, warp 5 TMA
// producer.  Tensor memory: Q hi [0,128), Q lo [128,256), O [256,384),
// S / P hi of tiles j = b (mod 2) at [384 + 64b, 448 + 64b).
#include "kernels.h"
#include "sm103.cuh"
#include "sm103_tf32.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int DP = 128;  // padded head dimension of the split operands
constexpr int BR = 128;  // query rows per CTA
constexpr int BC = 64;   // keys per tile
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr uint32_t TM_QH = 0, TM_QL = 128, TM_O = 256, TM_S = 384;  // S buffer b at TM_S + 64 b
constexpr float kRescaleThreshold = 8.0f;  // lazy rescaling, as in the other forward kernels
// shared memory: fp32 boxes of 32 columns (128-byte rows), 128-byte swizzle
constexpr int K_BOX = BC * 128;    // K part [64 keys][32 dims]: 8 KB
constexpr int K_PART = 4 * K_BOX;  // K hi or lo of a tile, [64][128]: 32 KB
constexpr int V_BOX = DP * 128;    // V^T part [128 dims][32 keys]: 16 KB
constexpr int V_PART = 2 * V_BOX;  // V^T hi or lo of a tile, [128][64]: 32 KB
constexpr int PL_BOX = BR * 128;   // P lo [128 rows][32 keys]: 16 KB
constexpr int PL_BUF = 2 * PL_BOX; // P lo of a tile, [128][64]: 32 KB
constexpr int OFF_K = 0;                    // K hi, then K lo
constexpr int OFF_V = OFF_K + 2 * K_PART;   // V^T hi, then V^T lo
constexpr int OFF_PL = OFF_V + 2 * V_PART;  // P lo of tiles j = b (mod 2) at OFF_PL + b PL_BUF
constexpr int OFF_BAR = OFF_PL + 2 * PL_BUF;
// q_ready, k_full, k_empty, v_full, v_empty, s_full[2], p_full[2], o_done, drain
constexpr int NBAR = 11;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Bars {
  uint32_t base;
  __device__ uint32_t q_ready() const { return base; }
  __device__ uint32_t k_full() const { return base + 8; }
  __device__ uint32_t k_empty() const { return base + 16; }
  __device__ uint32_t v_full() const { return base + 24; }
  __device__ uint32_t v_empty() const { return base + 32; }
  __device__ uint32_t s_full(int b) const { return base + 40 + 8 * b; }
  __device__ uint32_t p_full(int b) const { return base + 56 + 8 * b; }
  __device__ uint32_t o_done() const { return base + 72; }
  __device__ uint32_t drain() const { return base + 80; }
};

template <bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_f32_tc128_sm103_kernel(const __grid_constant__ Tc128Maps mp, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + SMEM_USED > static_cast<uint32_t>(SMEM_BYTES)) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const Bars bar{sb + OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const WaitCtl wc{p.status, abort_flag, p.wait_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N;
  const int r = WIN ? p.window_r : -1;
  const int nqt = (N + BR - 1) / BR;
  const int bh = blockIdx.x / nqt;
  const int i0 = (blockIdx.x % nqt) * BR;
  int j_lo = 0, j_hi = (N + BC - 1) / BC;
  if (WIN) {
    j_lo = max(0, i0 - r) / BC;
    j_hi = (min(N, min(N, i0 + BR) + r) + BC - 1) / BC;
  }
  const int ntiles = j_hi - j_lo;

  if (threadIdx.x == 0) {
    mbar_init(bar.q_ready(), 4);  // one arrive per softmax warp, once its Q rows are in tensor memory
    mbar_init(bar.k_full(), 1);
    mbar_init(bar.k_empty(), 1);
    mbar_init(bar.v_full(), 1);
    mbar_init(bar.v_empty(), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.s_full(b), 1);
      mbar_init(bar.p_full(b), 4);
    }
    mbar_init(bar.o_done(), 1);
    mbar_init(bar.drain(), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 5) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      prefetch_tensormap(&mp.kh);
      prefetch_tensormap(&mp.kl);
      prefetch_tensormap(&mp.vh);
      prefetch_tensormap(&mp.vl);
      bool ok = true;
      int kq = 0, vq = 0;  // K / V^T tiles issued
      auto load_k = [&](int j) {  // K hi, lo of key tile j
        if (j > 0 && !mbar_wait_backoff(bar.k_empty(), (j - 1) & 1, wc)) {
          ok = false;
          return;
        }
        const int kv0 = (j_lo + j) * BC;
        mbar_arrive_expect_tx(bar.k_full(), 2 * K_PART);
        for (int b = 0; b < 4; ++b) {
          tma_load_3d(sb + OFF_K + b * K_BOX, &mp.kh, bar.k_full(), 32 * b, kv0, bh);
          tma_load_3d(sb + OFF_K + K_PART + b * K_BOX, &mp.kl, bar.k_full(), 32 * b, kv0, bh);
        }
        kq = j + 1;
      };
      auto load_v = [&](int j) {  // V^T hi, lo of key tile j (128 dims x 64 keys)
        if (j > 0 && !mbar_wait_backoff(bar.v_empty(), (j - 1) & 1, wc)) {
          ok = false;
          return;
        }
        const int kv0 = (j_lo + j) * BC;
        mbar_arrive_expect_tx(bar.v_full(), 2 * V_PART);
        for (int b = 0; b < 2; ++b) {
          tma_load_3d(sb + OFF_V + b * V_BOX, &mp.vh, bar.v_full(), kv0 + 32 * b, 0, bh);
          tma_load_3d(sb + OFF_V + V_PART + b * V_BOX, &mp.vl, bar.v_full(), kv0 + 32 * b, 0, bh);
        }
        vq = j + 1;
      };
      // consumption order S_0, S_1, P_0 V_0, S_2, P_1 V_1, S_3, ...: K_j loads
      // once S_{j-1} has read K_{j-1}, V_j once P_{j-1} V_{j-1} has read V_{j-1}
      if (ntiles > 0) load_k(0);
      if (ok && ntiles > 0) load_v(0);
      if (ok && ntiles > 1) load_k(1);
      for (int j = 1; ok && j < ntiles; ++j) {
        if (j + 1 < ntiles) load_k(j + 1);
        if (ok) load_v(j);
      }
      if (*abort_flag) {
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        if (kq > 0) mbar_wait(bar.k_full(), (kq - 1) & 1, drain);
        if (vq > 0) mbar_wait(bar.v_full(), (vq - 1) & 1, drain);
      }
    }
    __syncwarp();
  } else if (warp == 4) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_tf32_f32(BR, BC);  // S: N = 64 keys
      constexpr uint32_t idesc_o = idesc_tf32_f32(BR, DP);  // P V: N = 128 dims
      // S_m = Q K_m^T into S buffer m % 2 (A = Q from tensor memory; the
      // buffer's previous P hi was read by P_{m-2} V_{m-2}, issued before)
      auto issue_s = [&](int m) -> bool {
        if (!mbar_wait(bar.k_full(), m & 1, wc)) return false;
        tc_fence_after();
        const uint32_t d_s = tmem + TM_S + 64 * (m & 1);
#pragma unroll
        for (int kk = 0; kk < DP / 8; ++kk) {  // 8 dimensions (32 bytes) per step
          const uint32_t ok_ = (kk >> 2) * K_BOX + (kk & 3) * 32;
          const uint64_t kh = sdesc_sw128(sb + OFF_K + ok_, 16, 1024);
          const uint64_t kl = sdesc_sw128(sb + OFF_K + K_PART + ok_, 16, 1024);
          mma_tf32_ts(d_s, tmem + TM_QH + 8 * kk, kh, idesc_s, kk > 0);
          mma_tf32_ts(d_s, tmem + TM_QH + 8 * kk, kl, idesc_s, 1);
          mma_tf32_ts(d_s, tmem + TM_QL + 8 * kk, kh, idesc_s, 1);
        }
        mma_commit(bar.k_empty());
        mma_commit(bar.s_full(m & 1));
        return true;
      };
      bool ok = mbar_wait(bar.q_ready(), 0, wc);
      if (ok && ntiles > 0) ok = issue_s(0);
      if (ok && ntiles > 1) ok = issue_s(1);
      for (int j = 0; ok && j < ntiles; ++j) {
        // O (+)= P_j V_j: P hi from tensor memory, P lo from shared memory
        if (!mbar_wait2(bar.p_full(j & 1), (j >> 1) & 1, bar.v_full(), j & 1, wc)) break;
        tc_fence_after();
        const uint32_t a_hi = tmem + TM_S + 64 * (j & 1);
        const uint32_t pl = sb + OFF_PL + (j & 1) * PL_BUF;
#pragma unroll
        for (int kk = 0; kk < BC / 8; ++kk) {  // 8 keys per step
          const uint32_t ov = (kk >> 2) * V_BOX + (kk & 3) * 32;
          const uint64_t vh = sdesc_sw128(sb + OFF_V + ov, 16, 1024);
          const uint64_t vl = sdesc_sw128(sb + OFF_V + V_PART + ov, 16, 1024);
          const uint64_t al = sdesc_sw128(pl + (kk >> 2) * PL_BOX + (kk & 3) * 32, 16, 1024);
          mma_tf32_ts(tmem + TM_O, a_hi + 8 * kk, vh, idesc_o, (j > 0 || kk > 0));
          mma_tf32_ts(tmem + TM_O, a_hi + 8 * kk, vl, idesc_o, 1);
          mma_tf32_ss(tmem + TM_O, al, vh, idesc_o, 1);
        }
        mma_commit(bar.v_empty());
        mma_commit(bar.o_done());
        if (j + 2 < ntiles && !issue_s(j + 2)) break;
      }
      mma_commit(bar.drain());
      WaitCtl drain{nullptr, nullptr, wc.limit_ns};
      mbar_wait(bar.drain(), 0, drain);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const int row = threadIdx.x;
    const int qi = i0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl = p.scale_log2;
    const int qlo = i0, qhi = i0 + BR - 1;
    const int d = p.d;
    auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
    };
    // this row of Q, split into tf32 hi and lo, into tensor memory (columns
    // past d and rows past N are zero)
    {
      const float* qrow = static_cast<const float*>(p.q) + (static_cast<size_t>(bh) * N + qi) * d;
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t h[32], lo[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = 32 * c + e;
          const float x = (qi < N && col < d) ? qrow[col] : 0.f;
          const float xh = tf32_rna(x);
          h[e] = __float_as_uint(xh);
          lo[e] = __float_as_uint(tf32_rna(x - xh));
        }
        tmem_st_32x32b_x32(tl + TM_QH + 32 * c, h);
        tmem_st_32x32b_x32(tl + TM_QL + 32 * c, lo);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.q_ready());
    }
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      // S_j has completed, and with it P_{j-2} V_{j-2} (issued before it),
      // the last reader of this tile's P lo buffer
      const uint32_t tS = tl + TM_S + 64 * (j & 1);
      if (!warp_wait(bar.s_full(j & 1), (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[BC];
      tmem_ld_32x32b_x32(tS, &sr[0]);
      tmem_ld_32x32b_x32(tS + 32, &sr[32]);
      tmem_wait_ld();
      float sv[BC];
#pragma unroll
      for (int c = 0; c < BC; ++c) sv[c] = __uint_as_float(sr[c]);
      const int kv0 = (j_lo + j) * BC;
      const bool edge = (kv0 + BC > N) || (WIN && !(kv0 >= qhi - r && kv0 + BC - 1 <= qlo + r));
      if (edge) {
        int lo = 0, hi = min(BC, N - kv0);
        if (WIN) {
          lo = max(lo, qi - r - kv0);
          hi = min(hi, qi + r + 1 - kv0);
        }
        const unsigned span = hi > lo ? static_cast<unsigned>(hi - lo) : 0u;
#pragma unroll
        for (int c = 0; c < BC; ++c) sv[c] = (static_cast<unsigned>(c - lo) < span) ? sv[c] : -INFINITY;
      }
      float mx[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) mx[a] = fmaxf(sv[a], sv[a + 4]);
#pragma unroll
      for (int c = 8; c < BC; c += 8)
#pragma unroll
        for (int a = 0; a < 4; ++a) mx[a] = fmax3(mx[a], sv[c + a], sv[c + 4 + a]);
      const float mt = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl;
      float alpha = 1.f;
      if (mt > m_ref + kRescaleThreshold) {
        alpha = ex2_approx(m_ref - mt);
        m_ref = mt;
      }
      const float nref = (m_ref == -INFINITY) ? 0.f : -m_ref;
      float rsum = 0.f;
      // P = 2^(s * scale * log2 e - m_ref) in fp32: hi over S's columns (read
      // above), lo to shared memory as this row of a [128 rows][32 keys]
      // 128-byte-swizzled box per 32 keys (the layout the P_lo V_hi products
      // read, K-major)
      const uint32_t plrow = sb + OFF_PL + (j & 1) * PL_BUF + row * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t ph[32], pl[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float pv = ex2_approx(fmaf(sv[32 * h + c], sl, nref));
          rsum += pv;
          const float hi = tf32_rna(pv);
          ph[c] = __float_as_uint(hi);
          pl[c] = __float_as_uint(tf32_rna(pv - hi));
        }
        tmem_st_32x32b_x32(tS + 32 * h, ph);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          st_shared_v4(plrow + h * PL_BOX + ((c4 ^ (row & 7)) << 4), pl[4 * c4], pl[4 * c4 + 1], pl[4 * c4 + 2],
                       pl[4 * c4 + 3]);
      }
      fence_proxy_async_smem();
      // O may be rescaled once P_{j-1} V_{j-1} has completed
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!warp_wait(bar.o_done(), (j - 1) & 1)) {
          tmem_wait_st();
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DP / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tl + TM_O + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_32x32b_x32(tl + TM_O + 32 * c, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full(j & 1));
      l = l * alpha + rsum;
    }
    // Up to two P V products may still be running here (S_{T-1} was issued
    // before P_{T-2} V_{T-2}), so o_done's parity cannot tell the last one
    // apart; the drain commit, issued after every product, can
    const bool have = ok && ntiles > 0 && warp_wait(bar.drain(), 0);
    if (have && !*abort_flag) {
      // tcgen05.ld is warp-collective: every lane loads, rows past N store nothing
      tc_fence_after();
      const float inv_l = 1.f / l;
      float* orow = static_cast<float*>(p.o) + (static_cast<size_t>(bh) * N + qi) * d;
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tl + TM_O + 32 * c, o);
        tmem_wait_ld();
        if (qi < N) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e < d) orow[32 * c + e] = __uint_as_float(o[e]) * inv_l;
        }
      }
      if (p.lse != nullptr && qi < N) {
        const float mref = (m_ref == -INFINITY) ? 0.f : m_ref;
        p.lse[static_cast<size_t>(bh) * N + qi] = (mref + __log2f(l)) * 0.69314718055994531f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool WIN>
cudaError_t launch_win(const FwdParams& p, const Tc128Maps& m, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_f32_tc128_sm103_kernel<WIN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long grid = static_cast<long long>((p.N + BR - 1) / BR) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_fwd_f32_tc128_sm103_kernel<WIN><<<static_cast<unsigned>(grid), kThreads, SMEM_BYTES, s>>>(m, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32_tc128_main(const FwdParams& p, const Tc128Maps& m, cudaStream_t s) {
  return p.window_r >= 0 ? launch_win<true>(p, m, s) : launch_win<false>(p, m, s);
}

}  // namespace fa
