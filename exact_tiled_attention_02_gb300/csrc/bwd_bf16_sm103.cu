// bwd_bf16_sm103.cu -- exact attention backward by recomputation for GB300
// (sm_103a), bf16 in / fp32 accumulate: the main kernel for head dimension
// d = 96 and 128, and the launcher for every bf16 head dimension (d = 64 has
// its own main kernel, bwd_bf16_d64_sm103.cu, which TMEM room at that size
// lets overlap one query tile's element-wise work with the next tile's
// products; the prep and dq kernels are in bwd_prep_sm103.cu).
//
// "Flash attention and efficient attention -- Hinglish notes", "Backward Pass:
// Recomputation": the N x N matrices S and P are not stored by the forward and
// not read here; they are rebuilt on chip, one tile at a time, from Q, K and
// the forward's logsumexp:  P_ij = exp(scale q_i.k_j - lse_i).  The gradient
// formulas are the derivative of the forward definition (the pages print
// none): dV = P^T dO, dP = dO V^T, dS = P o (dP - D) with
// D_i = sum_j P_ij dP_ij = sum_k dO_ik O_ik, dQ = scale dS K, dK = scale dS^T Q.
//
// Three launches: bwd_prep (-D_i and -lse_i log2 e per query row, the dQ
// accumulator zeroed), then
//   bwd_main     one CTA per 128-key tile of one (batch, head): K_j, V_j stay
//                in shared memory; the CTA walks the 128-row query tiles that
//                can see its keys (only in-band tiles when windowed) and, per
//                query tile i, issues five tcgen05.mma, all M = N = 128:
//                  S^T  = K_j Q_i^T        (A, B from shared memory)
//                  dP^T = V_j dO_i^T       (shared memory)
//                  dV  += P^T dO_i         (P^T from tensor memory)
//                  dK  += dS^T Q_i         (dS^T from tensor memory)
//                  dQ   = dS K_j          (shared memory: dS^T and K_j read
//                                           MN-major; TMEM lanes = queries)
//                dV and dK accumulate in tensor memory for the whole loop; each
//                dQ tile is staged as fp32 [128 queries][d] (d / 32 128-byte-
//                swizzled boxes of 32 columns) in the shared-memory stage its
//                Q / dO tiles just vacated, and added to the fp32 accumulator
//                by TMA reductions (cp.reduce.async.bulk.tensor .add.f32), so
//                the memory system does the adds in whole lines;
// then bwd_dq (dQ = bf16(scale * accumulator)).
// (Measured on GB300: tcgen05.mma with M = 128 and K = 16 takes 64 cycles at
// N = 128 but 48 at N = 64, so 64-row query tiles would waste a third of the
// tensor core on three of the five products.)
//
// Warp roles in bwd_main (384 threads; registers are granted per four-warp
// group, so the two idle warps cost nothing):
//   warps 0-3   compute warpgroup 0: query columns 0-63 of every tile
//   warps 4-7   compute warpgroup 1: query columns 64-127
//               (thread t owns key row t == TMEM lane t; for the dQ
//               read-out it owns query row t)
//   warp  8     TMEM owner + MMA issuer (one elected lane)
//   warp  9     TMA producer (one elected lane): loads Q_i, dO_i, lse_i, D_i into
//               a two-stage ring, issues the dQ^T reduction of tile i from
//               stage i%2 and refills that stage with tile i+2 once the
//               reduction has read it
//   warps 10-11 idle
// Tensor memory columns (128 lanes each):
//   [0,128)   S^T; warpgroup g writes its bf16 P^T over [64g, 64g+32);
//             then dQ of the same tile (written after dV has read P^T)
//   [128,256) dP^T; warpgroup g writes its bf16 dS^T over [128+64g, 128+64g+32)
//   [256,384) dV      [384,512) dK
// tcgen05.mma operations issued by one thread execute in order, so a product
// that overwrites columns another product reads is issued after it.
#include <type_traits>

#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int BM = 128;    // query rows per step
constexpr int BN = 128;    // keys per CTA
constexpr int kThreads = 384;
constexpr int kTmemCols = 512;
constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256;  // dK follows dV
constexpr int BOX_BYTES = 128 * 128;      // 16 KB: one bf16 [128 rows x 64 cols] box
constexpr int VEC_BYTES = BM * 4;         // 512 B of lse*log2e or of D
constexpr int DQ_BOX_BYTES = BM * 32 * 4; // 16 KB: fp32 dQ staging box [128 queries][32 d], 128-byte swizzled
constexpr int DST_BYTES = BN * BM * 2;    // 32 KB: bf16 dS^T [128 keys][128 queries] as two boxes

// D = 96 or 128 (d = 64 has its own main kernel).  Tiles in shared memory
// are DP = 128 columns wide (whole 128-byte swizzle atoms; for D = 96 the
// TMA zero-fills columns 96..127).  S^T and dP^T contract over the D real
// columns; the three products with N = d (dV, dK, dQ) run with N = DP, since a
// 128-byte-swizzled MN-major operand is laid out in 64-column atoms: the zero
// columns only produce zero columns, which are never read.
template <int D>
struct Cfg {
  static_assert(D == 96 || D == 128, "d = 64 runs bwd_bf16_d64_sm103.cu");
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int STAGES = 2;                    // Q/dO/lse/D ring depth
  static constexpr int BOXES = DP / 64;               // 64-column boxes per row of a Q / K / V / dO tile
  static constexpr int TILE_BYTES = 128 * DP * 2;     // a bf16 [128 x DP] tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // Q_i then dO_i; also holds the fp32 [128 x D] dQ staging
  // dQ staging: fp32 boxes of 32 columns; warpgroup 0 stages boxes [0, QBOXES)
  // over the Q half of the stage, warpgroup 1 the rest over the dO half
  static constexpr int DQ_BOXES = D / 32;
  static constexpr int QBOXES = TILE_BYTES / DQ_BOX_BYTES;
  static constexpr int DQ_COLS0 = 32 * QBOXES;       // d columns of warpgroup 0
  static constexpr int DQ_COLS1 = D - DQ_COLS0;      // d columns of warpgroup 1
  static constexpr uint32_t TM_DK = TM_DV + DP;
  // 1024-aligned region: K, V, the stages, dS^T; then the small items
  // (per-stage lse2 / D vectors, barriers, tmem slot, abort flag)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_BYTES;
  static constexpr int OFF_STAGE = OFF_V + TILE_BYTES;
  static constexpr int OFF_DST = OFF_STAGE + STAGES * STAGE_BYTES;
  static constexpr int OFF_VEC = OFF_DST + DST_BYTES;
  static constexpr int OFF_BAR = OFF_VEC + STAGES * 2 * VEC_BYTES;
  // kv_full, qa_full[S] (Q + vectors), qo_full[S] (dO), staged_q[S], staged_o[S] (the two halves of the dQ
  // staging), s_full, dp_full, p_full, ds_full, dq_full, dq_free, fin, drain, dk_done
  static constexpr int NBAR = 1 + 4 * STAGES + 9;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = (SMEM_USED + 1024 <= 227 * 1024) ? SMEM_USED + 1024 : 227 * 1024;
  static constexpr int kMaxPad = SMEM_BYTES - SMEM_USED;  // the kernel checks the alignment pad fits
  static_assert(kMaxPad >= 0, "shared memory budget");
  static_assert(D % 32 == 0 && DQ_COLS1 > 0 && DQ_COLS1 <= TILE_BYTES / (BM * 4), "dQ staging fits the stage");
  static_assert(TM_DK + DP <= kTmemCols, "tensor memory budget");
};

template <int STAGES>
struct Bars {
  uint32_t base;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t qa_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t qo_full(int s) const { return base + 8 * (1 + STAGES + s); }
  __device__ uint32_t staged_q(int s) const { return base + 8 * (1 + 2 * STAGES + s); }
  __device__ uint32_t staged_o(int s) const { return base + 8 * (1 + 3 * STAGES + s); }
  __device__ uint32_t at(int k) const { return base + 8 * (1 + 4 * STAGES + k); }
  __device__ uint32_t s_full() const { return at(0); }
  __device__ uint32_t dp_full() const { return at(1); }
  __device__ uint32_t p_full() const { return at(2); }
  __device__ uint32_t ds_full() const { return at(3); }
  __device__ uint32_t dq_full() const { return at(4); }
  __device__ uint32_t dq_free() const { return at(5); }
  __device__ uint32_t fin() const { return at(6); }
  __device__ uint32_t drain() const { return at(7); }
  __device__ uint32_t dk_done() const { return at(8); }
};

__host__ __device__ __forceinline__ int npad128(int n) { return (n + 127) & ~127; }

// ---------------------------------------------------------------------------
// bwd_main
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_bf16_sm103_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                             const __grid_constant__ CUtensorMap tmdq, const __grid_constant__ CUtensorMap tmdk,
                             const __grid_constant__ CUtensorMap tmdv, const BwdParams p) {
  using C = Cfg<D>;
  constexpr int STAGES = C::STAGES;
  constexpr int TILE_BYTES = C::TILE_BYTES, STAGE_BYTES = C::STAGE_BYTES;
  constexpr uint32_t TM_DK = C::TM_DK;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad > static_cast<uint32_t>(C::kMaxPad)) {
    // cannot happen with a 1024-aligned dynamic shared memory base; refuse rather than overrun
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sK = sb + C::OFF_K, sV = sb + C::OFF_V, sStage = sb + C::OFF_STAGE, sDS = sb + C::OFF_DST, sVec = sb + C::OFF_VEC;
  const Bars<STAGES> bar{sb + C::OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const WaitCtl wc{p.status, abort_flag, p.wait_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N, r = p.window_r;
  const int nkt = (N + BN - 1) / BN;
  // CTAs past n_full take one half of a split key tile's query tiles each
  int tile = static_cast<int>(blockIdx.x), half = -1;
  if (tile >= p.n_full) {
    half = (tile - p.n_full) & 1;
    tile = p.n_full + ((tile - p.n_full) >> 1);
  }
  const int bh = tile / nkt;
  const int k0 = (tile % nkt) * BN;
  const int np = npad128(N);

  // query tiles that can see this key tile
  int t_lo = 0, t_hi = (N + BM - 1) / BM;
  if (r >= 0) {
    t_lo = max(0, k0 - r) / BM;
    t_hi = (min(N, k0 + BN + r) + BM - 1) / BM;
  }
  if (half >= 0) {
    const int mid = t_lo + (t_hi - t_lo) / 2;
    if (half == 0)
      t_hi = mid;
    else
      t_lo = mid;
  }
  const int nsteps = t_hi - t_lo;

  if (threadIdx.x == 0) {
    mbar_init(bar.kv_full(), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar.qa_full(s), 1);
      mbar_init(bar.qo_full(s), 1);
      mbar_init(bar.staged_q(s), 4);  // one arrive per warp of compute warpgroup 0
      mbar_init(bar.staged_o(s), 4);  // ... of compute warpgroup 1
    }
    mbar_init(bar.s_full(), 1);
    mbar_init(bar.dp_full(), 1);
    mbar_init(bar.p_full(), 8);  // one arrive per compute warp
    mbar_init(bar.ds_full(), 8);
    mbar_init(bar.dq_full(), 1);
    mbar_init(bar.dq_free(), 8);
    mbar_init(bar.fin(), 1);
    mbar_init(bar.drain(), 1);
    mbar_init(bar.dk_done(), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 8) {
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

  if (warp >= 10) {
    // idle
  } else if (warp == 9) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmq);
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      prefetch_tensormap(&tmdo);
      prefetch_tensormap(&tmdq);
      mbar_arrive_expect_tx(bar.kv_full(), 2 * TILE_BYTES);
      for (int b = 0; b < C::BOXES; ++b) {
        tma_load_3d(sK + b * BOX_BYTES, &tmk, bar.kv_full(), b * 64, k0, bh);
        tma_load_3d(sV + b * BOX_BYTES, &tmv, bar.kv_full(), b * 64, k0, bh);
      }
      // tile `it` into stage it % STAGES, in two parts: Q_it with the lse / D
      // vectors, and dO_it (each part reuses the stage half that the dQ
      // staging of tile it - STAGES occupied)
      auto load_q = [&](int it) {
        const int st = it % STAGES;
        const int q0 = (t_lo + it) * BM;
        const uint32_t base = sStage + st * STAGE_BYTES;
        const uint32_t vec = sVec + st * 2 * VEC_BYTES;
        mbar_arrive_expect_tx(bar.qa_full(st), TILE_BYTES + 2 * VEC_BYTES);
        for (int b = 0; b < C::BOXES; ++b) tma_load_3d(base + b * BOX_BYTES, &tmq, bar.qa_full(st), b * 64, q0, bh);
        const size_t vrow = static_cast<size_t>(bh) * np + q0;
        bulk_load(vec, p.lse2 + vrow, VEC_BYTES, bar.qa_full(st));
        bulk_load(vec + VEC_BYTES, p.dsum + vrow, VEC_BYTES, bar.qa_full(st));
      };
      auto load_o = [&](int it) {
        const int st = it % STAGES;
        const int q0 = (t_lo + it) * BM;
        const uint32_t base = sStage + st * STAGE_BYTES + TILE_BYTES;
        mbar_arrive_expect_tx(bar.qo_full(st), TILE_BYTES);
        for (int b = 0; b < C::BOXES; ++b) tma_load_3d(base + b * BOX_BYTES, &tmdo, bar.qo_full(st), b * 64, q0, bh);
      };
      int loaded = 0;
      for (; loaded < STAGES && loaded < nsteps; ++loaded) {
        load_q(loaded);
        load_o(loaded);
      }
      for (int it = 0; it < nsteps; ++it) {
        // tile it's dQ is staged in stage it % STAGES: warpgroup 0's columns over
        // the Q half, warpgroup 1's over the dO half.  Reduce the Q half first
        // and reload Q (which the first product of a step needs) as soon as
        // that half has been read, then the dO half.
        const int st = it % STAGES;
        const uint32_t sbase = sStage + st * STAGE_BYTES;
        const int q0 = (t_lo + it) * BM;
        if (!mbar_wait_backoff(bar.staged_q(st), (it / STAGES) & 1, wc)) break;
#pragma unroll
        for (int b = 0; b < C::QBOXES; ++b)
          tma_reduce_add_3d(&tmdq, sbase + b * DQ_BOX_BYTES, 32 * b, q0, bh);
        bulk_commit_group();
        // Q_{it+STAGES} is loaded before the dO half's reduction is issued, so
        // the load does not queue behind that reduction's read of shared memory
        if (loaded < nsteps) {
          bulk_wait_read_all();  // the Q half has been read
          load_q(loaded);
        }
        if (!mbar_wait_backoff(bar.staged_o(st), (it / STAGES) & 1, wc)) break;
#pragma unroll
        for (int b = C::QBOXES; b < C::DQ_BOXES; ++b)
          tma_reduce_add_3d(&tmdq, sbase + b * DQ_BOX_BYTES, 32 * b, q0, bh);
        bulk_commit_group();
        if (loaded < nsteps) {
          bulk_wait_read_all();  // the dO half has been read
          load_o(loaded);
          ++loaded;
        }
      }
      bulk_wait_all();  // reductions complete (and their sources read) before the stages are reused or the CTA exits
      if (*abort_flag) {
        WaitCtl drain{nullptr, nullptr, wc.limit_ns};
        mbar_wait(bar.kv_full(), 0, drain);
        for (int it = max(0, loaded - STAGES); it < loaded; ++it) {
          mbar_wait(bar.qa_full(it % STAGES), (it / STAGES) & 1, drain);
          mbar_wait(bar.qo_full(it % STAGES), (it / STAGES) & 1, drain);
        }
      }
    }
    __syncwarp();
  } else if (warp == 8) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);  // both operands K-major
      constexpr uint32_t id_kb = idesc_bf16_f32(128, C::DP, 0, 1);  // A K-major (TMEM), B MN-major, N = DP
      constexpr uint32_t id_mm = idesc_bf16_f32(128, C::DP, 1, 1);  // both MN-major (dS^T, K), N = DP
      // S^T_i = K Q_i^T (the caller has waited for Q_i), then dP^T_i = V dO_i^T
      // once dO_i is resident (the producer refills that half of the stage last)
      auto issue_s_dp = [&](int i) -> bool {
        const int st = i % STAGES;
        const uint32_t qb = sStage + st * STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
          mma_bf16_ss(tmem + TM_S, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(qb + off, 16, 1024), id_kk, kk > 0);
        }
        mma_commit(bar.s_full());
        if (!mbar_wait(bar.qo_full(st), (i / STAGES) & 1, wc)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
          mma_bf16_ss(tmem + TM_DP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(qb + TILE_BYTES + off, 16, 1024),
                      id_kk, kk > 0);
        }
        mma_commit(bar.dp_full());
        return true;
      };
      bool ok = mbar_wait2(bar.kv_full(), 0, bar.qa_full(0), 0, wc);
      if (ok) {
        tc_fence_after();
        ok = issue_s_dp(0);
      }
      for (int i = 0; ok && i < nsteps; ++i) {
        const int st = i % STAGES;
        const uint32_t ph = i & 1;
        const uint32_t qb = sStage + st * STAGE_BYTES;
        // dV += P^T dO_i   (P^T in TMEM: query columns 16kk.. at column 8kk, or 64 + 8(kk-4))
        if (!mbar_wait(bar.p_full(), ph, wc)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_bf16_ts(tmem + TM_DV, tmem + TM_S + (kk < 4 ? 8 * kk : 64 + 8 * (kk - 4)),
                      sdesc_sw128(qb + TILE_BYTES + kk * 2048, BOX_BYTES, 1024), id_kb, (i > 0 || kk > 0));
        // dQ = dS K first (over the S^T / P^T columns, after dV read P^T), so the
        // warpgroups can read dQ and free those columns while dK += dS^T Q_i runs
        if (!mbar_wait(bar.ds_full(), ph, wc)) break;
        tc_fence_after();
        const uint32_t dsb = sDS;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ss(tmem + TM_S, sdesc_sw128(dsb + kk * 2048, BOX_BYTES, 1024),
                      sdesc_sw128(sK + kk * 2048, BOX_BYTES, 1024), id_mm, kk > 0);
        mma_commit(bar.dq_full());
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_bf16_ts(tmem + TM_DK, tmem + TM_DP + (kk < 4 ? 8 * kk : 64 + 8 * (kk - 4)),
                      sdesc_sw128(qb + kk * 2048, BOX_BYTES, 1024), id_kb, (i > 0 || kk > 0));
        mma_commit(bar.dk_done());  // Q_i's last reader: its stage may take the dQ staging
        // next tile's S^T and dP^T once dQ has been read out of the S^T columns
        // (and Q_{i+1} is resident: one round trip, see mbar_wait2)
        if (i + 1 < nsteps) {
          if (!mbar_wait2(bar.dq_free(), ph, bar.qa_full((i + 1) % STAGES), ((i + 1) / STAGES) & 1, wc)) break;
          tc_fence_after();
          if (!issue_s_dp(i + 1)) break;
        }
      }
      mma_commit(bar.fin());
      mma_commit(bar.drain());
      WaitCtl drain{nullptr, nullptr, wc.limit_ns};
      mbar_wait(bar.drain(), 0, drain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- compute warpgroups
    const int g = warp >> 2;            // query columns [64g, 64g + 64) of every tile
    const int row = threadIdx.x & 127;  // key row within the tile == TMEM lane (== d index for dQ^T)
    const int kj = k0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t tS = tl + TM_S + 64 * g, tDP = tl + TM_DP + 64 * g;
    const uint32_t sDSg = sDS + g * BOX_BYTES;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    // Key rows past N hold zeros (TMA zero fill): their P and dS are finite and
    // meet K = 0 in dQ; their dK / dV rows are never stored.  No mask needed.
    bool ok = true;
    for (int i = 0; i < nsteps; ++i) {
      const uint32_t ph = i & 1;
      const int st = i % STAGES;
      const int q0 = (t_lo + i) * BM + 64 * g;  // first query column of this warpgroup
      // ---- P^T = exp2(S^T * scale * log2e - lse * log2e)
      if (!warp_wait(bar.s_full(), ph) || !warp_wait(bar.qa_full(st), (i / STAGES) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_32x32b_x32(tS, &sv[0]);
      tmem_ld_32x32b_x32(tS + 32, &sv[32]);
      tmem_wait_ld();
      const float4* nlse4 = reinterpret_cast<const float4*>(smem + C::OFF_VEC + st * 2 * VEC_BYTES + 64 * 4 * g);
      const float4* nd4 = reinterpret_cast<const float4*>(smem + C::OFF_VEC + st * 2 * VEC_BYTES + VEC_BYTES + 64 * 4 * g);
      float pr[64];
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 l4 = nlse4[c4];
        const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sv[4 * c4]), __uint_as_float(sv[4 * c4 + 1])), sl2,
                                     make_float2(l4.x, l4.y));
        const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sv[4 * c4 + 2]), __uint_as_float(sv[4 * c4 + 3])), sl2,
                                     make_float2(l4.z, l4.w));
        pr[4 * c4] = ex2_approx(x0.x);
        pr[4 * c4 + 1] = ex2_approx(x0.y);
        pr[4 * c4 + 2] = ex2_approx(x1.x);
        pr[4 * c4 + 3] = ex2_approx(x1.y);
      }
      if (r >= 0 && !(q0 >= kj - r && q0 + 63 <= kj + r)) {
        // window: the queries that see key kj form one contiguous column range [lo, hi)
        const int lo = max(0, kj - r - q0), hi = min(64, kj + r + 1 - q0);
        const unsigned span = hi > lo ? static_cast<unsigned>(hi - lo) : 0u;
#pragma unroll
        for (int c = 0; c < 64; ++c) pr[c] = (static_cast<unsigned>(c - lo) < span) ? pr[c] : 0.f;
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(pr[2 * c], pr[2 * c + 1]);
        tmem_st_32x32b_x32(tS, pk);  // P^T over this warpgroup's first 32 S^T columns
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full());

      // ---- dS^T = P^T o (dP^T - D), to TMEM (for dK) and shared memory (for dQ)
      if (!warp_wait(bar.dp_full(), ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dpv[64];
      tmem_ld_32x32b_x32(tDP, &dpv[0]);
      tmem_ld_32x32b_x32(tDP + 32, &dpv[32]);
      tmem_wait_ld();
      {
        uint32_t dk[32];
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 n4 = nd4[c4];
          const float2 t0 = __fadd2_rn(make_float2(__uint_as_float(dpv[4 * c4]), __uint_as_float(dpv[4 * c4 + 1])),
                                       make_float2(n4.x, n4.y));
          const float2 t1 = __fadd2_rn(make_float2(__uint_as_float(dpv[4 * c4 + 2]), __uint_as_float(dpv[4 * c4 + 3])),
                                       make_float2(n4.z, n4.w));
          const float2 d0 = __fmul2_rn(make_float2(pr[4 * c4], pr[4 * c4 + 1]), t0);
          const float2 d1 = __fmul2_rn(make_float2(pr[4 * c4 + 2], pr[4 * c4 + 3]), t1);
          dk[2 * c4] = pack_bf16x2(d0.x, d0.y);
          dk[2 * c4 + 1] = pack_bf16x2(d1.x, d1.y);
        }
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          st_shared_v4(sDSg + row * 128 + ((c8 ^ (row & 7)) << 4), dk[4 * c8], dk[4 * c8 + 1], dk[4 * c8 + 2],
                       dk[4 * c8 + 3]);
        tmem_st_32x32b_x32(tDP, dk);  // dS^T over this warpgroup's first 32 dP^T columns
      }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.ds_full());

      // ---- dQ read-out (thread = query row; warpgroup 0 takes the d columns
      //      that fill the Q half of the stage, warpgroup 1 the rest), staged as
      //      fp32 in stage i % STAGES as 128-byte-swizzled [128 queries][32 d]
      //      boxes for the producer's TMA reductions (half 0 held Q_i, half 1
      //      held dO_i)
      if (!warp_wait(bar.dq_full(), ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this warpgroup's NC d columns from col0: read out, free the columns, stage
      auto dq_out = [&](auto nc, int col0) -> bool {
        constexpr int NC = decltype(nc)::value;
        uint32_t qv[NC];
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) tmem_ld_32x32b_x32(tl + TM_S + col0 + 32 * c, &qv[32 * c]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.dq_free());
        // warpgroup 0 stages over Q_i, which dK_i (issued after dQ_i) may still be
        // reading; warpgroup 1 stages over dO_i, last read by dV_i (before dQ_i)
        if (col0 == 0 && !warp_wait(bar.dk_done(), ph)) return false;
        const uint32_t stg = sStage + st * STAGE_BYTES + row * 128;
#pragma unroll
        for (int c4 = 0; c4 < NC / 4; ++c4) {  // 16-byte chunk c4 of this row's NC values
          const int col = col0 + 4 * c4;       // first d column of the chunk
          const uint32_t box = col >> 5, chunk = (col & 31) >> 2;
          st_shared_v4(stg + box * DQ_BOX_BYTES + ((chunk ^ (row & 7)) << 4), qv[4 * c4], qv[4 * c4 + 1],
                       qv[4 * c4 + 2], qv[4 * c4 + 3]);
        }
        return true;
      };
      const bool staged = (g == 0) ? dq_out(std::integral_constant<int, C::DQ_COLS0>{}, 0)
                                   : dq_out(std::integral_constant<int, C::DQ_COLS1>{}, C::DQ_COLS0);
      if (!staged) {
        ok = false;
        break;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(g == 0 ? bar.staged_q(st) : bar.staged_o(st));
    }

    // ------------------------------------------------------------ epilogue
    // warpgroup 0 writes dV, warpgroup 1 writes scale * dK, each staged as a
    // bf16 [128 keys][D] tile over K (dV) or V (dK): once every product has
    // completed (fin) nothing reads them any more, so the staging overlaps
    // the producer's last dQ reductions, which read the Q/dO stages (the
    // epilogue used to stage over a stage and wait for them: measured
    // 1.3 us of a 77 us CTA at 4x16x4096x128)
    const bool have = ok && warp_wait(bar.fin(), 0);
    const uint32_t stage_out = g == 0 ? sK : sV;
    if (have && half >= 0) {
      // one half of a split key tile: add this row's fp32 values into the
      // partial rows (both halves add into zeroed memory, so the sum does not
      // depend on their order)
      tc_fence_after();
      const uint32_t tcol = g == 0 ? TM_DV : TM_DK;
      const float mul = g == 0 ? 1.f : p.scale;
      float* dst = p.kv_part + ((static_cast<size_t>(tile - p.n_full) * 2 + g) * BN + row) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tl + tcol + c * 32, v);
        tmem_wait_ld();
        if (k0 + row < N) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            red_add_v4_f32(dst + c * 32 + 4 * e, __uint_as_float(v[4 * e]) * mul, __uint_as_float(v[4 * e + 1]) * mul,
                           __uint_as_float(v[4 * e + 2]) * mul, __uint_as_float(v[4 * e + 3]) * mul);
        }
      }
    } else if (have) {
      // staged in the TMA box layout of the outputs' maps ([128 keys][64
      // columns] boxes, 16-byte chunk c of row r at c ^ (r % 8)), then written
      // by two TMA stores per warpgroup; keys past N are not written (from
      // registers, a thread per row: ≈ 4000 cycles per 128 keys at the
      // window-257 workload)
      tc_fence_after();
      const uint32_t tcol = g == 0 ? TM_DV : TM_DK;
      const float mul = g == 0 ? 1.f : p.scale;
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
          st_shared_v4(stage_out + (c16 >> 3) * BOX_BYTES + row * 128 + (((c16 & 7) ^ (row & 7)) << 4), w[0], w[1],
                       w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    named_bar_sync(1 + g, 128);
    if (have && half < 0 && !*abort_flag && (row & 127) == 0) {
      const CUtensorMap* out = g == 0 ? &tmdv : &tmdk;
      for (int b = 0; b < C::BOXES; ++b) tma_store_3d(out, stage_out + b * BOX_BYTES, 64 * b, k0, bh);
      bulk_commit_group();
      // the stores have read the staging before the CTA's shared memory is
      // released; their global writes complete before the kernel does, so the
      // SM can start its next CTA meanwhile
      bulk_wait_read_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace {

template <int D>
cudaError_t launch_main(const BwdParams& p, const BwdMaps& m, unsigned grid, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_bf16_sm103_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<D>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  fa_bwd_bf16_sm103_kernel<D><<<grid, kThreads, Cfg<D>::SMEM_BYTES, s>>>(m.q, m.k, m.v, m.dO, m.dq_acc, m.dk, m.dv,
                                                                           p);
  return cudaGetLastError();
}

}  // namespace

namespace {

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace

cudaError_t launch_bwd_bf16_tc(const BwdParams& p_in, const BwdMaps& m, cudaStream_t s) {
  if (p_in.d != 128 && p_in.d != 96 && p_in.d != 64) return cudaErrorNotSupported;
  BwdParams p = p_in;
  const long long nkt = (p.N + BN - 1) / BN;
  const long long tiles = nkt * p.BH;
  // One CTA per SM.  When the last wave would hold at most half the SMs, its
  // key tiles are split in two (no window, at least two query tiles): 2w
  // half-length CTAs instead of w full ones.
  long long split = 0;
  if (p.window_r < 0 && p.N > BM) {
    const int sms = device_sm_count();
    const long long w = sms > 0 ? tiles % sms : 0;
    if (w > 0 && 2 * w <= sms && w <= kMaxSplitTiles) split = w;
  }
  p.n_split = static_cast<int>(split);
  p.n_full = static_cast<int>(tiles - split);
  const long long grid = tiles + split;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = launch_bwd_prep(p, s);
  if (e != cudaSuccess) return e;
  e = p.d == 128  ? launch_main<128>(p, m, static_cast<unsigned>(grid), s)
      : p.d == 96 ? launch_main<96>(p, m, static_cast<unsigned>(grid), s)
                  : launch_bwd_main_d64(p, m, static_cast<unsigned>(grid), s);
  if (e != cudaSuccess) return e;
  return launch_bwd_dq(p, s);
}

}  // namespace fa
