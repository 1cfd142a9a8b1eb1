// fwd_keymajor_sm103.cu -- the forward pass in the key-major loop order, kept
// as a measured comparison point for the query-major kernels.
//
// "Compute attention one tile at a time" (TensorViz), fidelity note: the
// teaching example loops over query tiles outermost, while the original
// paper's Algorithm 1 loops over key/value tiles outermost.  Here the outer
// loop over key/value tiles j is a sequence of launches on one stream; the
// inner loop's iterations (query tiles i) do not depend on one another, so
// they are the CTAs of each launch.  Every (i, j) merges one tile into the
// running statistics of query tile i exactly as "Flash attention and
// efficient attention -- Hinglish notes", "Derivation: Incremental Softmax",
// Steps 2-3 prescribe: per row, the tile's maximum m~ and P~ = exp(S - m~)
// (taken against the merged maximum), m_new = max(m, m~),
// l_new = e^(m - m_new) l + rowsum(P~), O~_new = e^(m - m_new) O~ + P~ V_j,
// with the unnormalised O~, m and l kept in an fp32 workspace in device
// memory between launches and a single division at the end.  That round
// trip of O~ through device memory on every step is what the query-major
// kernels avoid by keeping O in tensor memory.
//
// Step kernel, one CTA per (query tile i, head) for key tile j, 192 threads:
// warps 0-3 own the 128 query rows (thread = row = TMEM lane), warp 4 issues
// tcgen05.mma and owns tensor memory (S: 128 columns, P V_j: D columns),
// warp 5 loads Q_i, K_j, V_j by TMA.  The tile's P V_j is staged in shared
// memory so that the read-modify-write of O~ is coalesced.
// Finish kernel: O = O~ / l (bf16), lse = ln sum exp.
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int BR = 128;  // query rows per tile
constexpr int BC = 128;  // keys per tile
constexpr int kThreads = 192;
constexpr int kTmemCols = 256;
constexpr uint32_t kTmemS = 0, kTmemO = 128;

template <int D>
struct KmCfg {
  static constexpr int BOXES = D / 64;
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE_BYTES;
  static constexpr int OFF_V = OFF_K + TILE_BYTES;
  static constexpr int STAGE_BYTES = BR * D * 4;  // fp32 P V_j tile, over Q/K/V once they are consumed
  static constexpr int OFF_ALPHA = (3 * TILE_BYTES > STAGE_BYTES) ? 3 * TILE_BYTES : STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_ALPHA + BR * 4;
  static constexpr int NBAR = 6;  // qk_full, v_full, s_full, p_full, o_full, drain
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;
  static_assert(SMEM_BYTES <= 113 * 1024, "two CTAs per SM");
};

// first key tile that any row of query tile i can see (0 unless windowed)
__device__ __forceinline__ int first_key_tile(int i0, int r) { return r < 0 ? 0 : max(0, i0 - r) / BC; }

template <int D>
__global__ void __launch_bounds__(kThreads)
    fa_fwd_keymajor_step_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                                const __grid_constant__ CUtensorMap tmv, const FwdParams p, float* __restrict__ o_acc,
                                float* __restrict__ m_acc, float* __restrict__ l_acc, int j) {
  using C = KmCfg<D>;
  const int N = p.N, r = p.window_r;
  const int nqt = (N + BR - 1) / BR;
  const int bh = blockIdx.x / nqt;
  const int i0 = (blockIdx.x % nqt) * BR;
  const int kv0 = j * BC;
  // no row of this query tile sees a key of tile j: nothing to merge
  if (r >= 0 && (kv0 > min(N, i0 + BR) - 1 + r || kv0 + BC - 1 < i0 - r)) return;
  const bool first = (j == first_key_tile(i0, r));

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + C::SMEM_USED > static_cast<uint32_t>(C::SMEM_BYTES)) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V;
  float* alpha_s = reinterpret_cast<float*>(smem + C::OFF_ALPHA);
  const uint32_t bar = sb + C::OFF_BAR;
  const uint32_t qk_full = bar, v_full = bar + 8, s_full = bar + 16, p_full = bar + 24, o_full = bar + 32,
                 drain_bar = bar + 40;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const WaitCtl wc{p.status, abort_flag, p.wait_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(qk_full, 1);
    mbar_init(v_full, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(o_full, 1);
    mbar_init(drain_bar, 1);
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

  bool ok = true;
  if (warp == 5) {
    if (lane == 0) {
      prefetch_tensormap(&tmq);
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      mbar_arrive_expect_tx(qk_full, 2 * C::TILE_BYTES);
      for (int b = 0; b < C::BOXES; ++b) {
        tma_load_3d(sQ + b * BR * 128, &tmq, qk_full, b * 64, i0, bh);
        tma_load_3d(sK + b * BC * 128, &tmk, qk_full, b * 64, kv0, bh);
      }
      mbar_arrive_expect_tx(v_full, C::TILE_BYTES);
      for (int b = 0; b < C::BOXES; ++b) tma_load_3d(sV + b * BC * 128, &tmv, v_full, b * 64, kv0, bh);
      if (*abort_flag) {
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(qk_full, 0, drain);
        mbar_wait(v_full, 0, drain);
      }
    }
    __syncwarp();
  } else if (warp == 4) {
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BR, BC, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BR, D, 0, 1);
      if (mbar_wait(qk_full, 0, wc)) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (BR * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + kTmemS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), idesc_qk, kk > 0);
        }
        mma_commit(s_full);
        if (mbar_wait(v_full, 0, wc) && mbar_wait(p_full, 0, wc)) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BC / 16; ++kk)
            mma_bf16_ts(tmem + kTmemO, tmem + kTmemS + kk * 8, sdesc_sw128(sV + kk * 16 * 128, BC * 128, 1024),
                        idesc_pv, kk > 0);
          mma_commit(o_full);
        }
      }
      // every MMA issued here must finish before tensor memory is freed
      mma_commit(drain_bar);
      WaitCtl drain{nullptr, nullptr, wc.limit_ns};
      mbar_wait(drain_bar, 0, drain);
    }
    __syncwarp();
  } else {
    const int row = threadIdx.x;  // 0..127
    const int qi = i0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl = p.scale_log2;
    auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
    };
    float alpha = 0.f;  // factor on the old O~ of this row
    ok = warp_wait(s_full, 0);
    if (ok) {
      tc_fence_after();
      uint32_t sr[BC];
#pragma unroll
      for (int c = 0; c < BC / 32; ++c) tmem_ld_32x32b_x32(tl + kTmemS + c * 32, &sr[c * 32]);
      tmem_wait_ld();
      // visible keys of row qi in this tile: one contiguous column range [lo, hi)
      int lo = 0, hi = min(BC, N - kv0);
      if (r >= 0) {
        lo = max(lo, qi - r - kv0);
        hi = min(hi, qi + r + 1 - kv0);
      }
      const unsigned span = hi > lo ? static_cast<unsigned>(hi - lo) : 0u;
      float s[BC];
#pragma unroll
      for (int c = 0; c < BC; ++c) s[c] = (static_cast<unsigned>(c - lo) < span) ? __uint_as_float(sr[c]) : -INFINITY;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BC; ++c) mx = fmaxf(mx, s[c]);
      // Step 3: merged maximum (log2 units of scaled scores) and the old part's factor
      const size_t srow = static_cast<size_t>(bh) * N + qi;
      const bool live = qi < N;
      const float m_old = (first || !live) ? -INFINITY : m_acc[srow];
      const float l_old = (first || !live) ? 0.f : l_acc[srow];
      const float m_new = fmaxf(m_old, mx * sl);
      alpha = (m_old == -INFINITY) ? 0.f : ex2_approx(m_old - m_new);
      const float ref = (m_new == -INFINITY) ? 0.f : m_new;
      float rsum = 0.f;
      uint32_t pk[BC / 2];
#pragma unroll
      for (int c = 0; c < BC / 2; ++c) {
        const float p0 = ex2_approx(fmaf(s[2 * c], sl, -ref));
        const float p1 = ex2_approx(fmaf(s[2 * c + 1], sl, -ref));
        rsum += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) tmem_st_32x32b_x16(tl + kTmemS + 16 * g, &pk[16 * g]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      if (live) {
        m_acc[srow] = m_new;
        l_acc[srow] = alpha * l_old + rsum;
      }
      ok = warp_wait(o_full, 0);
    }
    // stage P V_j (fp32) over Q/K/V, which the finished products no longer read;
    // 16-byte chunks of a row are swizzled by the row so the stores spread over banks
    if (ok) {
      tc_fence_after();
      alpha_s[row] = first ? 0.f : alpha;
      uint8_t* st = smem + static_cast<size_t>(row) * D * 4;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tl + kTmemO + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const int ch = c * 8 + q4;  // 16-byte chunk of the row
          const int sw = (ch & ~7) | ((ch & 7) ^ (row & 7));
          *reinterpret_cast<uint4*>(st + sw * 16) = make_uint4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
        }
      }
    }
    named_bar_sync(1, 128);
    if (ok && !*abort_flag) {
      // O~ = alpha O~ + P V_j, coalesced: consecutive threads take consecutive 16-byte chunks
      constexpr int CH = D / 4;
      float* obase = o_acc + (static_cast<size_t>(bh) * N + i0) * D;
      for (int idx = row; idx < BR * CH; idx += 128) {
        const int rr = idx / CH, ch = idx % CH;
        if (i0 + rr >= N) continue;
        const int sw = (ch & ~7) | ((ch & 7) ^ (rr & 7));
        const float4 pv = *reinterpret_cast<const float4*>(smem + static_cast<size_t>(rr) * D * 4 + sw * 16);
        float4* dst = reinterpret_cast<float4*>(obase + static_cast<size_t>(rr) * D) + ch;
        const float a = alpha_s[rr];
        float4 out = pv;
        if (a != 0.f) {
          const float4 old = *dst;
          out = make_float4(fmaf(a, old.x, pv.x), fmaf(a, old.y, pv.y), fmaf(a, old.z, pv.z), fmaf(a, old.w, pv.w));
        }
        *dst = out;
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

// O = O~ / l as bf16, lse = (m + log2 l) ln 2; one thread per 8 elements
__global__ void __launch_bounds__(256) fa_fwd_keymajor_finish_kernel(const float* __restrict__ o_acc,
                                                                     const float* __restrict__ m_acc,
                                                                     const float* __restrict__ l_acc,
                                                                     __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                                     long long rows, int d) {
  const long long n8 = rows * d / 8;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const long long row = (i * 8) / d;
  const float inv = 1.f / l_acc[row];
  const float4 a = reinterpret_cast<const float4*>(o_acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(o_acc)[2 * i + 1];
  uint4 out;
  out.x = pack_bf16x2(a.x * inv, a.y * inv);
  out.y = pack_bf16x2(a.z * inv, a.w * inv);
  out.z = pack_bf16x2(b.x * inv, b.y * inv);
  out.w = pack_bf16x2(b.z * inv, b.w * inv);
  reinterpret_cast<uint4*>(o)[i] = out;
  if (lse != nullptr && (i * 8) % d == 0) lse[row] = (m_acc[row] + __log2f(l_acc[row])) * 0.69314718055994531f;
}

template <int D>
cudaError_t launch_steps(const FwdParams& p, const FwdMaps& m, float* o_acc, float* m_acc, float* l_acc,
                         cudaStream_t s) {
  using C = KmCfg<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_keymajor_step_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long grid = static_cast<long long>((p.N + BR - 1) / BR) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int nkt = (p.N + BC - 1) / BC;
  for (int j = 0; j < nkt; ++j) {
    fa_fwd_keymajor_step_kernel<D><<<static_cast<unsigned>(grid), kThreads, C::SMEM_BYTES, s>>>(m.q, m.k, m.v, p, o_acc,
                                                                                                 m_acc, l_acc, j);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

size_t keymajor_workspace_layout(int BH, int N, int d, size_t* off_m, size_t* off_l) {
  const size_t rows = static_cast<size_t>(BH) * N;
  const size_t acc = (rows * d * sizeof(float) + 255) & ~size_t(255);
  const size_t vec = (rows * sizeof(float) + 255) & ~size_t(255);
  if (off_m) *off_m = acc;
  if (off_l) *off_l = acc + vec;
  return acc + 2 * vec;
}

cudaError_t launch_fwd_keymajor(const FwdParams& p, const FwdMaps& m, void* workspace, cudaStream_t s) {
  size_t off_m = 0, off_l = 0;
  keymajor_workspace_layout(p.BH, p.N, p.d, &off_m, &off_l);
  float* o_acc = static_cast<float*>(workspace);
  float* m_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + off_m);
  float* l_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + off_l);
  cudaError_t e;
  if (p.d == 128)
    e = launch_steps<128>(p, m, o_acc, m_acc, l_acc, s);
  else if (p.d == 64)
    e = launch_steps<64>(p, m, o_acc, m_acc, l_acc, s);
  else
    return cudaErrorNotSupported;
  if (e != cudaSuccess) return e;
  const long long rows = static_cast<long long>(p.BH) * p.N;
  const long long n8 = rows * p.d / 8;
  if ((n8 + 255) / 256 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_fwd_keymajor_finish_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, s>>>(
      o_acc, m_acc, l_acc, static_cast<__nv_bfloat16*>(p.o), p.lse, rows, p.d);
  return cudaGetLastError();
}

}  // namespace fa
