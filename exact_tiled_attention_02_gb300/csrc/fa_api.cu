// fa_api.cu -- the C ABI declared in include/fa.h: argument validation, TMA
// descriptor construction, the device status word, and dispatch to the
// kernels.  Nothing here allocates device memory or synchronises, except
// fa_last_device_status().
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kMaxDevices = 64;
constexpr long long kDefaultWaitUs = 1000000;  // 1 s per device-side wait

// Device status word: kernels OR error bits into it (FA_ERR_TIMEOUT); the
// host reads and clears it in fa_last_device_status().
__device__ unsigned int g_status;

std::atomic<long long> g_wait_limit_us{kDefaultWaitUs};

struct DeviceState {
  std::once_flag once;
  unsigned int* status = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceState g_dev[kMaxDevices];

// Resolves, once per device, the device address of the status word.
cudaError_t status_ptr(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st]() {
    void* p = nullptr;
    st.err = cudaGetSymbolAddress(&p, g_status);
    st.status = static_cast<unsigned int*>(p);
  });
  *out = st.status;
  return st.err;
}

typedef EncodeTiledFnPtr EncodeTiledFn;

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library does not link against libcuda directly.
EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over a [BH, N, d] bf16 array: dims (d, N, BH), box (64, rows, 1),
// 128-byte swizzle; rows past N read as zero.
bool make_map_bf16(CUtensorMap* m, const void* base, int BH, int N, int d, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the fp32 [BH, N, d] dQ accumulator for TMA reductions: dims
// (d, N, BH), box (32, rows, 1) with 128-byte swizzle; rows past N are not
// written.
bool make_map_f32_acc(CUtensorMap* m, const void* base, int BH, int N, int d, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side validation shared by forward and backward; runs before any CUDA
// call so invalid requests have no side effect.
fa_status check_common(int B, int H, int N, int d, float scale, int window, fa_dtype dt) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID;
  if (window > 0 && (window % 2) == 0) return FA_ERR_INVALID;
  if (dt != FA_DTYPE_F32 && dt != FA_DTYPE_BF16) return FA_ERR_INVALID;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > 0x7fffffffLL) return FA_ERR_INVALID;
  if (bh * N > (1LL << 40) / (d > 0 ? d : 1)) return FA_ERR_INVALID;
  if (dt == FA_DTYPE_BF16 && d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (dt == FA_DTYPE_F32 && d > 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int radius(int window) { return window > 0 ? (window - 1) / 2 : -1; }

}  // namespace

// Every check fa_bwd makes on its arguments other than the workspace: null
// and misaligned pointers, sizes, scale, window, dtype, and the head
// dimensions the backward does not implement.
fa_status check_bwd_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, const void* dq, const void* dk, const void* dv, int B, int H, int N, int d,
                         float scale, int window, fa_dtype dt) {
  const void* ptrs[] = {q, k, v, o, dO, dq, dk, dv, lse};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID;
  const fa_status c = check_common(B, H, N, d, scale, window, dt);
  if (c != FA_OK) return c;
  if (dt == FA_DTYPE_BF16 && d == 256) return FA_ERR_UNSUPPORTED;  // forward only at d = 256
  return FA_OK;
}

namespace {

unsigned long long wait_ns() { return static_cast<unsigned long long>(g_wait_limit_us.load()) * 1000ull; }

// Device-side self-test of the bounded wait: one thread waits on a barrier
// nothing arrives on until the limit passes, then records the timeout.
__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = sm103::smem_u32(&bar);
  if (threadIdx.x == 0) {
    sm103::mbar_init(b, 1);
    abort_flag = 0;
    sm103::fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    sm103::WaitCtl w{status, &abort_flag, limit_ns};
    sm103::mbar_wait(b, 0, w);  // phase 0 never completes: times out
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned int* status, unsigned long long limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID: return "FA_ERR_INVALID: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported dtype/head dimension for this entry point";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call or kernel launch failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a bounded device-side wait ran out";
  }
  return "unknown fa_status";
}

long long fa_set_wait_limit_us(long long limit_us) {
  if (limit_us <= 0) limit_us = kDefaultWaitUs;
  return g_wait_limit_us.exchange(limit_us);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > 0x7fffffffLL) return 0;
  return bwd_workspace_layout(static_cast<int>(bh), N, d, nullptr, nullptr, nullptr);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int window, fa_dtype dt, void* stream) {
  if (!q || !k || !v || !o) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID;
  const fa_status c = check_common(B, H, N, d, scale, window, dt);
  if (c != FA_OK) return c;

  FwdParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.BH = B * H;
  p.N = N;
  p.d = d;
  p.window_r = radius(window);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = wait_ns();
  if (status_ptr(&p.status) != cudaSuccess) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (dt == FA_DTYPE_F32) return launch_fwd_f32_simt(p, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;

  FwdMaps m;
  if (!make_map_bf16(&m.q, q, p.BH, N, d, kFwdBlockRows) || !make_map_bf16(&m.k, k, p.BH, N, d, kFwdBlockCols) ||
      !make_map_bf16(&m.v, v, p.BH, N, d, kFwdBlockCols))
    return FA_ERR_CUDA;
  return launch_fwd_bf16_tc(p, m, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_fwd_key_major_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > 0x7fffffffLL) return 0;
  return keymajor_workspace_layout(static_cast<int>(bh), N, d, nullptr, nullptr);
}

fa_status fa_fwd_key_major(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                           int d, float scale, int window, fa_dtype dt, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (!q || !k || !v || !o || !workspace) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_INVALID;
  const fa_status c = check_common(B, H, N, d, scale, window, dt);
  if (c != FA_OK) return c;
  if (dt != FA_DTYPE_BF16 || (d != 64 && d != 128)) return FA_ERR_UNSUPPORTED;
  if (workspace_bytes < fa_fwd_key_major_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID;

  FwdParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.BH = B * H;
  p.N = N;
  p.d = d;
  p.window_r = radius(window);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = wait_ns();
  if (status_ptr(&p.status) != cudaSuccess) return FA_ERR_CUDA;
  FwdMaps m;
  if (!make_map_bf16(&m.q, q, p.BH, N, d, 128) || !make_map_bf16(&m.k, k, p.BH, N, d, 128) ||
      !make_map_bf16(&m.v, v, p.BH, N, d, 128))
    return FA_ERR_CUDA;
  return launch_fwd_keymajor(p, m, workspace, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                  : FA_ERR_CUDA;
}

size_t fa_fwd_f32_3xtf32_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > 0x7fffffffLL) return 0;
  return f32_tc_workspace_layout(static_cast<int>(bh), N, d, nullptr);
}

fa_status fa_fwd_f32_3xtf32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int H,
                            int N, int d, float scale, int window, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!q || !k || !v || !o || !workspace) return FA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_INVALID;
  const fa_status c = check_common(B, H, N, d, scale, window, FA_DTYPE_F32);
  if (c != FA_OK) return c;
  if (workspace_bytes < fa_fwd_f32_3xtf32_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID;

  FwdParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.BH = B * H;
  p.N = N;
  p.d = d;
  p.window_r = radius(window);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = wait_ns();
  if (status_ptr(&p.status) != cudaSuccess) return FA_ERR_CUDA;
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return FA_ERR_CUDA;
  return launch_fwd_f32_tc(p, workspace, fn, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                : FA_ERR_CUDA;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int window, fa_dtype dt,
                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return FA_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_INVALID;
  const fa_status c = check_bwd_args(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, window, dt);
  if (c != FA_OK) return c;
  if (workspace_bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID;

  BwdParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.dO = dO;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  size_t off_lse2 = 0, off_dsum = 0, off_part = 0;
  bwd_workspace_layout(B * H, N, d, &off_lse2, &off_dsum, &off_part);
  p.dq_acc = static_cast<float*>(workspace);
  p.lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + off_lse2);
  p.dsum = reinterpret_cast<float*>(static_cast<char*>(workspace) + off_dsum);
  p.kv_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + off_part);
  p.n_full = 0;  // set by the bf16 launcher
  p.n_split = 0;
  p.BH = B * H;
  p.N = N;
  p.d = d;
  p.window_r = radius(window);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = wait_ns();
  if (status_ptr(&p.status) != cudaSuccess) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (dt == FA_DTYPE_F32) return launch_bwd_f32_simt(p, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;

  BwdMaps m;
  if (!make_map_bf16(&m.q, q, p.BH, N, d, kBwdBlockRows) || !make_map_bf16(&m.k, k, p.BH, N, d, kBwdBlockCols) ||
      !make_map_bf16(&m.v, v, p.BH, N, d, kBwdBlockCols) || !make_map_bf16(&m.dO, dO, p.BH, N, d, kBwdBlockRows) ||
      !make_map_f32_acc(&m.dq_acc, p.dq_acc, p.BH, N, d, kBwdBlockRows) ||
      !make_map_bf16(&m.dk, dk, p.BH, N, d, kBwdBlockCols) || !make_map_bf16(&m.dv, dv, p.BH, N, d, kBwdBlockCols))
    return FA_ERR_CUDA;
  const cudaError_t e = launch_bwd_bf16_tc(p, m, s);
  if (e == cudaErrorNotSupported) return FA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_last_device_status(void* stream) {
  unsigned int* sp = nullptr;
  if (status_ptr(&sp) != cudaSuccess) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  if (cudaMemcpyAsync(&host, sp, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemsetAsync(sp, 0, sizeof(unsigned int), s) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  if (host & sm103::kStatusTimeout) return FA_ERR_TIMEOUT;
  if (host & sm103::kStatusLayout) return FA_ERR_CUDA;
  return FA_OK;
}

fa_status fa_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 100000) return FA_ERR_INVALID;
  unsigned int* sp = nullptr;
  if (status_ptr(&sp) != cudaSuccess) return FA_ERR_CUDA;
  return launch_selftest_wait(sp, static_cast<unsigned long long>(limit_us) * 1000ull,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // extern "C"
