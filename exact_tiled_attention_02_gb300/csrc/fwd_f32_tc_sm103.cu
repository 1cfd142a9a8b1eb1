// fwd_f32_tc_sm103.cu -- tiled exact attention forward for float32 inputs on
// the tensor cores, by a three-term tf32 split ("3xTF32"): the kernel for
// d <= 64, the split kernels and the launcher for every d <= 128 (64 < d <=
// 128 runs the kernel in fwd_f32_tc128_sm103.cu).
//
// What it computes is the forward of fwd_f32_simt.cu ("Flash attention and
// efficient attention -- Hinglish notes", "The Standard Attention Problem",
// one key/value tile at a time with the running maximum / running sum merge
// of "Derivation: Incremental Softmax", Steps 1-3; the window of "Worked
// example Local Attention Window"), in fp32 input and output.  The tensor
// core multiplies tf32 values (11 significant bits), so every float32
// operand x is split as x = hi + lo with hi = tf32(x) and lo = tf32(x - hi)
// (together 22 significant bits), and every product is taken as
// hi_a hi_b + hi_a lo_b + lo_a hi_b; the dropped lo_a lo_b term and the
// rounding of lo are below 2^-21 relative.  That is done for S = Q K^T (split
// Q, K) and for O += P V (split P, V), so the result stays within a few
// float32 roundings of the exact value.
//
// Kernels:
//   split_rows   Q and K -> hi / lo, [B*H][N][DP] (DP = 64, or 128 for d > 64;
//                columns past d zero)
//   split_vt     V -> V^T hi / lo, [B*H][DP][Npad] (Npad = N rounded up to 64),
//                so that P V reads V K-major (keys contiguous), the layout
//                tcgen05.mma takes for tf32 operands here
//   main         one CTA = one 128-row query tile of one head, 224 threads:
//                warps 0-3 softmax (thread = row = TMEM lane), warp 4 TMEM
//                owner + issuer of the S products, warp 5 TMA producer, warp
//                6 issuer of the P V products.  64-key tiles; K and V^T each
//                stream through their own two-slot ring; S is double-buffered
//                in tensor memory so that S_{j+1} is computed while the
//                softmax turns S_j into P_j.  S_{j+2} goes into the buffer
//                P_j occupied once P_j V_j has completed (pv_done).  Each
//                product is three kind::tf32 MMAs per K-step, 24 instructions
//                of N = 64 per product; one thread issuing both products
//                (an instruction takes about as long to issue as to execute
//                at N = 64) measured ~3900 cycles per key tile.
// Tensor memory (512 columns): buffer b at 128 b: S_b / P_b hi in columns
// [0, 64), P_b lo in [64, 128); O in [256, 320).
#include "kernels.h"
#include "sm103.cuh"
#include "sm103_tf32.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int D = 64;   // padded head dimension of the split operands
constexpr int BR = 128;  // query rows per CTA
constexpr int BC = 64;   // keys per tile
constexpr int kThreads = 224;
constexpr int kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleThreshold = 8.0f;  // lazy rescaling, as in the bf16 kernels
// shared memory: fp32 boxes of 32 columns (128 bytes) per row, 128-byte swizzle
constexpr int Q_BOX = BR * 128;        // [128 rows][32 cols]: 16 KB
constexpr int KV_BOX = 64 * 128;       // [64 rows][32 cols]: 8 KB
constexpr int Q_BYTES = 2 * Q_BOX;     // one of Q hi / Q lo: 32 KB
constexpr int SLOT_BYTES = 4 * KV_BOX; // hi then lo, each two boxes: 32 KB
constexpr int OFF_QH = 0;
constexpr int OFF_QL = OFF_QH + Q_BYTES;
constexpr int OFF_K = OFF_QL + Q_BYTES;       // two K slots
constexpr int OFF_V = OFF_K + 2 * SLOT_BYTES;  // two V^T slots
constexpr int OFF_BAR = OFF_V + 2 * SLOT_BYTES;
// q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], o_done, drain, pv_done[2]
constexpr int NBAR = 1 + 8 + 2 + 2 + 2 + 2;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Bars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (3 + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (5 + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (7 + s); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (9 + b); }
  // P_j of buffer b = j % 2 is in tensor memory.  One barrier per buffer: the
  // softmax may finish P_{j+1} before the MMA warp has waited for P_j, but it
  // cannot finish P_{j+2} (that needs S_{j+2}, issued after P_j V_j)
  __device__ uint32_t p_full(int b) const { return base + 8 * (11 + b); }
  __device__ uint32_t o_done() const { return base + 8 * 13; }
  __device__ uint32_t drain() const { return base + 8 * 14; }
  // P_j V_j (buffer b = j % 2) has completed: S_{j+2} may overwrite the buffer
  __device__ uint32_t pv_done(int b) const { return base + 8 * (15 + b); }
};

// hi / lo rows of DP columns (zero past d): 16-byte chunks, four per thread
// (256 apart, so each pass is one coalesced sweep), every load issued before
// any is used.  The rows of x start on 16-byte boundaries when d % 4 == 0;
// otherwise each element is read alone.
template <int DP>
__global__ void __launch_bounds__(256) fa_split_rows_kernel(const float* __restrict__ x, float* __restrict__ hi,
                                                            float* __restrict__ lo, long long n4, int d) {
  constexpr int C4 = DP / 4;  // chunks per row, a power of two
  const long long b0 = static_cast<long long>(blockIdx.x) * 1024 + threadIdx.x;
  const bool vec = (d & 3) == 0;
  float4 v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const long long i4 = b0 + u * 256;
    v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i4 >= n4) continue;
    const long long r = i4 / C4;
    const int c = static_cast<int>(i4 % C4) * 4;
    const float* src = x + r * d + c;
    if (vec) {
      if (c < d) v[u] = __ldg(reinterpret_cast<const float4*>(src));
    } else {
      if (c < d) v[u].x = __ldg(src);
      if (c + 1 < d) v[u].y = __ldg(src + 1);
      if (c + 2 < d) v[u].z = __ldg(src + 2);
      if (c + 3 < d) v[u].w = __ldg(src + 3);
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const long long i4 = b0 + u * 256;
    if (i4 >= n4) continue;
    const float4 h = make_float4(tf32_rna(v[u].x), tf32_rna(v[u].y), tf32_rna(v[u].z), tf32_rna(v[u].w));
    reinterpret_cast<float4*>(hi)[i4] = h;
    reinterpret_cast<float4*>(lo)[i4] = make_float4(tf32_rna(v[u].x - h.x), tf32_rna(v[u].y - h.y),
                                                    tf32_rna(v[u].z - h.z), tf32_rna(v[u].w - h.w));
  }
}

// V^T hi / lo, [B*H][dp][npad] (zero past d and N), through a shared-memory
// tile of 64 keys x 32 columns: read along the columns of V's rows, written
// along the keys of V^T's rows, both coalesced.  Block (32, 8).
__global__ void __launch_bounds__(256) fa_split_vt_kernel(const float* __restrict__ v, float* __restrict__ hi,
                                                          float* __restrict__ lo, int N, int npad, int d, int dp) {
  __shared__ float tile[64][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int nt = npad / 64, ct = dp / 32;
  const long long blk = blockIdx.x;
  const long long bh = blk / (static_cast<long long>(nt) * ct);
  const int rem = static_cast<int>(blk % (static_cast<long long>(nt) * ct));
  const int c0 = (rem / nt) * 32, n0 = (rem % nt) * 64;
  const int c = c0 + tx;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int n = n0 + ty + 8 * j;
    tile[ty + 8 * j][tx] = (n < N && c < d) ? __ldg(v + (bh * N + n) * d + c) : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int cc = ty + 8 * j, nn = 2 * tx;
    const float x0 = tile[nn][cc], x1 = tile[nn + 1][cc];
    const float h0 = tf32_rna(x0), h1 = tf32_rna(x1);
    const long long o = ((bh * dp + c0 + cc) * npad + n0 + nn) / 2;
    reinterpret_cast<float2*>(hi)[o] = make_float2(h0, h1);
    reinterpret_cast<float2*>(lo)[o] = make_float2(tf32_rna(x0 - h0), tf32_rna(x1 - h1));
  }
}

struct TcMaps {
  CUtensorMap qh, ql, kh, kl, vh, vl;
};

template <bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_f32_tc_sm103_kernel(const __grid_constant__ TcMaps mp, const FwdParams p) {
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
    mbar_init(bar.q_full(), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.k_full(s), 1);
      mbar_init(bar.k_empty(s), 1);
      mbar_init(bar.v_full(s), 1);
      mbar_init(bar.v_empty(s), 1);
      mbar_init(bar.s_full(s), 1);
      mbar_init(bar.p_full(s), 4);
      mbar_init(bar.pv_done(s), 1);
    }
    mbar_init(bar.o_done(), 1);
    mbar_init(bar.drain(), 2);  // both MMA issuers
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
      prefetch_tensormap(&mp.qh);
      prefetch_tensormap(&mp.ql);
      prefetch_tensormap(&mp.kh);
      prefetch_tensormap(&mp.kl);
      prefetch_tensormap(&mp.vh);
      prefetch_tensormap(&mp.vl);
      mbar_arrive_expect_tx(bar.q_full(), 2 * Q_BYTES);
      for (int b = 0; b < 2; ++b) {
        tma_load_3d(sb + OFF_QH + b * Q_BOX, &mp.qh, bar.q_full(), 32 * b, i0, bh);
        tma_load_3d(sb + OFF_QL + b * Q_BOX, &mp.ql, bar.q_full(), 32 * b, i0, bh);
      }
      bool ok = true;
      int kq = 0, vq = 0;  // K / V^T tiles issued
      auto load_k = [&](int j) {  // K hi, lo of key tile j into slot j % 2
        const int s = j & 1;
        if (!mbar_wait_backoff(bar.k_empty(s), ((j >> 1) & 1) ^ 1, wc)) {
          ok = false;
          return;
        }
        const uint32_t dst = sb + OFF_K + s * SLOT_BYTES;
        const int kv0 = (j_lo + j) * BC;
        mbar_arrive_expect_tx(bar.k_full(s), SLOT_BYTES);
        for (int b = 0; b < 2; ++b) {
          tma_load_3d(dst + b * KV_BOX, &mp.kh, bar.k_full(s), 32 * b, kv0, bh);
          tma_load_3d(dst + 2 * KV_BOX + b * KV_BOX, &mp.kl, bar.k_full(s), 32 * b, kv0, bh);
        }
        kq = j + 1;
      };
      auto load_v = [&](int j) {  // V^T hi, lo of key tile j (64 dims x 64 keys) into slot j % 2
        const int s = j & 1;
        if (!mbar_wait_backoff(bar.v_empty(s), ((j >> 1) & 1) ^ 1, wc)) {
          ok = false;
          return;
        }
        const uint32_t dst = sb + OFF_V + s * SLOT_BYTES;
        const int kv0 = (j_lo + j) * BC;
        mbar_arrive_expect_tx(bar.v_full(s), SLOT_BYTES);
        for (int b = 0; b < 2; ++b) {
          tma_load_3d(dst + b * KV_BOX, &mp.vh, bar.v_full(s), kv0 + 32 * b, 0, bh);
          tma_load_3d(dst + 2 * KV_BOX + b * KV_BOX, &mp.vl, bar.v_full(s), kv0 + 32 * b, 0, bh);
        }
        vq = j + 1;
      };
      // consumption order: S_0, S_1, then P_j V_j and S_{j+2}
      for (int j = 0; ok && j < ntiles && j < 2; ++j) load_k(j);
      for (int j = 0; ok && j < ntiles; ++j) {
        load_v(j);
        if (ok && j + 2 < ntiles) load_k(j + 2);
      }
      if (*abort_flag) {
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.q_full(), 0, drain);
        for (int j = max(0, kq - 2); j < kq; ++j) mbar_wait(bar.k_full(j & 1), (j >> 1) & 1, drain);
        for (int j = max(0, vq - 2); j < vq; ++j) mbar_wait(bar.v_full(j & 1), (j >> 1) & 1, drain);
      }
    }
    __syncwarp();
  } else if (warp == 4) {
    // ------------------------------------------------------- S products (MMA)
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_tf32_f32(BR, 64);  // N = 64 keys
      bool ok = mbar_wait(bar.q_full(), 0, wc);
      for (int j = 0; ok && j < ntiles; ++j) {  // S_j = Q K_j^T into buffer j % 2
        const int s = j & 1;
        // K_j resident; for j >= 2, P_{j-2} V_{j-2} has read the buffer
        if (!mbar_wait(bar.k_full(s), (j >> 1) & 1, wc) ||
            (j >= 2 && !mbar_wait(bar.pv_done(s), ((j >> 1) & 1) ^ 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dtm = tmem + 128 * s;
        const uint32_t kb = sb + OFF_K + s * SLOT_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 8; ++kk) {  // 8 dimensions (32 bytes) per step
          const uint32_t oq = (kk >> 2) * Q_BOX + (kk & 3) * 32, ok_ = (kk >> 2) * KV_BOX + (kk & 3) * 32;
          const uint64_t qh = sdesc_sw128(sb + OFF_QH + oq, 16, 1024), ql = sdesc_sw128(sb + OFF_QL + oq, 16, 1024);
          const uint64_t kh = sdesc_sw128(kb + ok_, 16, 1024), kl = sdesc_sw128(kb + 2 * KV_BOX + ok_, 16, 1024);
          mma_tf32_ss(dtm, qh, kh, idesc, kk > 0);
          mma_tf32_ss(dtm, qh, kl, idesc, 1);
          mma_tf32_ss(dtm, ql, kh, idesc, 1);
        }
        mma_commit(bar.k_empty(s));
        mma_commit(bar.s_full(s));
      }
      mma_commit(bar.drain());
      WaitCtl drain{nullptr, nullptr, wc.limit_ns};
      mbar_wait(bar.drain(), 0, drain);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ----------------------------------------------------- P V products (MMA)
    // every P in order, so this thread sees each phase of p_full and
    // completes each phase of pv_done in turn
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_tf32_f32(BR, 64);  // N = 64 dims
      bool ok = true;
      for (int j = 0; ok && j < ntiles; ++j) {  // O (+)= P_j V_j
        const int s = j & 1;
        if (!mbar_wait(bar.p_full(s), (j >> 1) & 1, wc) || !mbar_wait(bar.v_full(s), (j >> 1) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ph = tmem + 128 * s, pl = ph + 64;
        const uint32_t vb = sb + OFF_V + s * SLOT_BYTES;
#pragma unroll
        for (int kk = 0; kk < BC / 8; ++kk) {  // 8 keys per step
          const uint32_t ov = (kk >> 2) * KV_BOX + (kk & 3) * 32;
          const uint64_t vh = sdesc_sw128(vb + ov, 16, 1024), vl = sdesc_sw128(vb + 2 * KV_BOX + ov, 16, 1024);
          mma_tf32_ts(tmem + kTmemO, ph + 8 * kk, vh, idesc, (j > 0 || kk > 0));
          mma_tf32_ts(tmem + kTmemO, ph + 8 * kk, vl, idesc, 1);
          mma_tf32_ts(tmem + kTmemO, pl + 8 * kk, vh, idesc, 1);
        }
        mma_commit(bar.v_empty(s));
        mma_commit(bar.o_done());
        mma_commit(bar.pv_done(s));
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
    const uint32_t tO = tl + kTmemO;
    const float sl = p.scale_log2;
    const int qlo = i0, qhi = i0 + BR - 1;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
    };
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      if (!warp_wait(bar.s_full(s), (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tl + 128 * s;
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
      // P = 2^(s * scale * log2 e - m_ref) in fp32; hi and lo tf32 parts over
      // columns [0, 64) (S, already read) and [64, 128) of the buffer
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
        tmem_st_32x32b_x32(tS + 64 + 32 * h, pl);
      }
      // O may be rescaled only once the previous P V has completed; here
      // P_{j-2} V_{j-2} has completed (S_j was issued after its pv_done) and
      // P_j V_j has not been issued, so o_done is within one phase of the one
      // waited for
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!warp_wait(bar.o_done(), (j - 1) & 1)) {
          tmem_wait_st();
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_32x32b_x32(tO + 32 * c, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full(s));
      l = l * alpha + rsum;
    }
    // every MMA has completed once both issuers' drain commits have (up to two
    // P V may be in flight after the last softmax step)
    const bool have = ok && ntiles > 0 && warp_wait(bar.drain(), 0);
    if (have && !*abort_flag) {
      // tcgen05.ld is warp-collective: every lane loads, rows past N store nothing
      tc_fence_after();
      const float inv_l = 1.f / l;
      const int d = p.d;
      float* orow = static_cast<float*>(p.o) + (static_cast<size_t>(bh) * N + qi) * d;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + 32 * c, o);
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

bool make_map_f32(CUtensorMap* m, EncodeTiledFnPtr fn, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint32_t box0, uint32_t box1) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool WIN>
cudaError_t launch_main(const FwdParams& p, const TcMaps& m, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_f32_tc_sm103_kernel<WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long grid = static_cast<long long>((p.N + BR - 1) / BR) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_fwd_f32_tc_sm103_kernel<WIN><<<static_cast<unsigned>(grid), kThreads, SMEM_BYTES, s>>>(m, p);
  return cudaGetLastError();
}

}  // namespace

size_t f32_tc_workspace_layout(int BH, int N, int d, size_t off[6]) {
  const size_t dp = d <= D ? D : 128;
  const size_t npad = (static_cast<size_t>(N) + 63) & ~size_t(63);
  const size_t rows = (static_cast<size_t>(BH) * N * dp * 4 + 255) & ~size_t(255);
  const size_t vt = (static_cast<size_t>(BH) * dp * npad * 4 + 255) & ~size_t(255);
  size_t o = 0;
  for (int i = 0; i < 4; ++i) {
    if (off) off[i] = o;
    if (i >= 2 || d <= D) o += rows;  // Q hi / lo only for d <= 64
  }
  for (int i = 4; i < 6; ++i, o += vt)
    if (off) off[i] = o;
  return o;
}

cudaError_t launch_fwd_f32_tc(const FwdParams& p, void* workspace, EncodeTiledFnPtr encode, cudaStream_t s) {
  if (p.d > 128 || encode == nullptr) return cudaErrorInvalidValue;
  const int dp = p.d <= D ? D : 128;
  size_t off[6];
  f32_tc_workspace_layout(p.BH, p.N, p.d, off);
  char* ws = static_cast<char*>(workspace);
  float* buf[6];
  for (int i = 0; i < 6; ++i) buf[i] = reinterpret_cast<float*>(ws + off[i]);
  const long long rows = static_cast<long long>(p.BH) * p.N;
  const int npad = (p.N + 63) & ~63;
  const long long n4 = rows * dp / 4, b1 = (n4 + 1023) / 1024;
  const long long b2 = static_cast<long long>(p.BH) * (npad / 64) * (dp / 32);
  if (b1 > 0x7fffffffLL || b2 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const auto split_rows = [&](const void* x, float* h, float* l) {
    if (dp == D)
      fa_split_rows_kernel<D><<<static_cast<unsigned>(b1), 256, 0, s>>>(static_cast<const float*>(x), h, l, n4, p.d);
    else
      fa_split_rows_kernel<128><<<static_cast<unsigned>(b1), 256, 0, s>>>(static_cast<const float*>(x), h, l, n4, p.d);
  };
  if (dp == D) split_rows(p.q, buf[0], buf[1]);
  split_rows(p.k, buf[2], buf[3]);
  fa_split_vt_kernel<<<static_cast<unsigned>(b2), 256, 0, s>>>(static_cast<const float*>(p.v), buf[4], buf[5], p.N,
                                                               npad, p.d, dp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const uint64_t BH = static_cast<uint64_t>(p.BH), Nn = static_cast<uint64_t>(p.N);
  if (dp != D) {
    Tc128Maps m;
    if (!make_map_f32(&m.kh, encode, buf[2], 128, Nn, BH, 32, 64) ||
        !make_map_f32(&m.kl, encode, buf[3], 128, Nn, BH, 32, 64) ||
        !make_map_f32(&m.vh, encode, buf[4], static_cast<uint64_t>(npad), 128, BH, 32, 128) ||
        !make_map_f32(&m.vl, encode, buf[5], static_cast<uint64_t>(npad), 128, BH, 32, 128))
      return cudaErrorInvalidValue;
    return launch_fwd_f32_tc128_main(p, m, s);
  }
  TcMaps m;
  if (!make_map_f32(&m.qh, encode, buf[0], D, Nn, BH, 32, BR) || !make_map_f32(&m.ql, encode, buf[1], D, Nn, BH, 32, BR) ||
      !make_map_f32(&m.kh, encode, buf[2], D, Nn, BH, 32, BC) || !make_map_f32(&m.kl, encode, buf[3], D, Nn, BH, 32, BC) ||
      !make_map_f32(&m.vh, encode, buf[4], static_cast<uint64_t>(npad), D, BH, 32, D) ||
      !make_map_f32(&m.vl, encode, buf[5], static_cast<uint64_t>(npad), D, BH, 32, D))
    return cudaErrorInvalidValue;
  return p.window_r >= 0 ? launch_main<true>(p, m, s) : launch_main<false>(p, m, s);
}

}  // namespace fa
