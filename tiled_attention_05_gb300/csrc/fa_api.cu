// C ABI of the attention library: argument validation, TMA descriptor
// encoding, the device status word and the workspace query.  The kernels and
// their launchers live in fa_fwd.cu and fa_bwd.cu.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <set>
#include <utility>

#include "fa_internal.h"

namespace {

__device__ int g_fa_status;  // 0, or a kernel's DEV_* code after a bounded wait gave up

thread_local int t_last_launches = 0;

#ifdef FA_TEST_HOOKS
std::atomic<int> g_test_withhold{0};
#endif

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates dims; on success fills *pr.  Null data pointers are only an error
// when the tensor they point to is non-empty.
fa_status check_dims(const fa_dims* dims, fa::Problem* pr) {
  if (!dims) return FA_ERR_INVALID_ARG;
  const fa_dims& z = *dims;
  if (z.B < 0 || z.Hq < 0 || z.Hkv < 0 || z.Tq < 0 || z.Tk < 0 || z.d < 1 || z.dv < 1) return FA_ERR_INVALID_ARG;
  if (z.causal != 0 && z.causal != 1) return FA_ERR_INVALID_ARG;
  if (z.window < 0 || (z.window > 0 && !z.causal)) return FA_ERR_INVALID_ARG;
  if (z.Hq > 0 && (z.Hkv < 1 || z.Hq % z.Hkv != 0)) return FA_ERR_INVALID_ARG;
  if (!(z.scale == z.scale) || std::isinf(z.scale)) return FA_ERR_INVALID_ARG;
  if ((z.d != 64 && z.d != 128) || (z.dv != 64 && z.dv != 128)) return FA_ERR_UNSUPPORTED;
  // TMA coordinates and grid dimensions are 32-bit; keep every index in range.
  if ((long long)z.B * z.Hq > 0x7fffffffLL || (long long)z.B * z.Hkv > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (z.Tq > (1 << 30) || z.Tk > (1 << 30)) return FA_ERR_UNSUPPORTED;
  // Size limits: the forward's pairs of 128-row query tiles per head (kept
  // within 16 bits, which bounds Tq at 65535 * 256) and the backward's linear
  // grid of (batch, kv head, key tile) CTAs.
  const long long q_pairs = ((long long)z.Tq + 255) / 256, kv_tiles = ((long long)z.Tk + 127) / 128;
  if (q_pairs > 65535 || (long long)z.B * z.Hkv * kv_tiles > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  pr->B = z.B;
  pr->Hq = z.Hq;
  pr->Hkv = z.Hkv;
  pr->Tq = z.Tq;
  pr->Tk = z.Tk;
  pr->d = z.d;
  pr->dv = z.dv;
  pr->causal = z.causal;
  // A window of Tk keys or more hides nothing (row i's window starts at or
  // before key i + Tk - Tq - Tk < 0); dropping it keeps kernel indices small.
  pr->window = z.window >= z.Tk ? 0 : z.window;
  pr->scale = z.scale > 0.f ? z.scale : 1.0f / std::sqrt((float)z.d);
  return FA_OK;
}

fa_status check_ptr(const void* p, long long elems) {
  if (elems == 0) return FA_OK;
  if (!p || !aligned16(p)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

}  // namespace

namespace fa {

#ifdef FA_TEST_HOOKS
int test_withhold() { return g_test_withhold.load(); }
#endif

bool encode_rows_bf16(CUtensorMap* map, const void* base, int inner, int rows, long long outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * (cuuint64_t)rows};
  cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_acc_f32(CUtensorMap* map, const void* base, int inner, long long rows, long long outer, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)inner * 4, (cuuint64_t)inner * 4 * (cuuint64_t)rows};
  cuuint32_t box[3] = {32, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int* device_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

cudaError_t allow_dynamic_smem(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

}  // namespace fa

extern "C" {

fa_status fa_forward(const fa_dims* dims, const void* Q, const void* K, const void* V, void* O, float* L,
                     void* stream) {
  t_last_launches = 0;
  fa::Problem pr;
  fa_status s = check_dims(dims, &pr);
  if (s != FA_OK) return s;
  const long long nq = (long long)pr.B * pr.Hq * pr.Tq * pr.d, nqv = (long long)pr.B * pr.Hq * pr.Tq * pr.dv;
  const long long nk = (long long)pr.B * pr.Hkv * pr.Tk * pr.d, nkv = (long long)pr.B * pr.Hkv * pr.Tk * pr.dv;
  if ((s = check_ptr(Q, nq)) || (s = check_ptr(K, nk)) || (s = check_ptr(V, nkv)) || (s = check_ptr(O, nqv)) ||
      (s = check_ptr(L, (long long)pr.B * pr.Hq * pr.Tq)))
    return s;
  if (nq == 0) return FA_OK;
  if (!fa::device_status_word()) return FA_ERR_CUDA;
  int launches = 0;
  cudaError_t e = fa::launch_forward(pr, Q, K, V, O, L, static_cast<cudaStream_t>(stream), &launches);
  t_last_launches = launches;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_backward_workspace_bytes(const fa_dims* dims) {
  fa::Problem pr;
  if (check_dims(dims, &pr) != FA_OK) return 0;
  return fa::backward_workspace_layout(pr).total;
}

size_t fa_backward_workspace_min_bytes(const fa_dims* dims) {
  fa::Problem pr;
  if (check_dims(dims, &pr) != FA_OK) return 0;
  return fa::backward_workspace_layout(pr).total_min;
}

fa_status fa_backward_stages(const fa_dims* dims, const void* Q, const void* K, const void* V, const void* O,
                             const void* dO, const float* L, void* dQ, void* dK, void* dV, void* workspace,
                             size_t workspace_bytes, int stages, void* stream) {
  t_last_launches = 0;
  fa::Problem pr;
  fa_status s = check_dims(dims, &pr);
  if (s != FA_OK) return s;
  if (stages < 0 || stages > FA_BWD_ALL) return FA_ERR_INVALID_ARG;
  const long long nq = (long long)pr.B * pr.Hq * pr.Tq * pr.d, nqv = (long long)pr.B * pr.Hq * pr.Tq * pr.dv;
  const long long nk = (long long)pr.B * pr.Hkv * pr.Tk * pr.d, nkv = (long long)pr.B * pr.Hkv * pr.Tk * pr.dv;
  if ((s = check_ptr(Q, nq)) || (s = check_ptr(K, nk)) || (s = check_ptr(V, nkv)) || (s = check_ptr(O, nqv)) ||
      (s = check_ptr(dO, nqv)) || (s = check_ptr(L, (long long)pr.B * pr.Hq * pr.Tq)) || (s = check_ptr(dQ, nq)) ||
      (s = check_ptr(dK, nk)) || (s = check_ptr(dV, nkv)))
    return s;
  if ((nq == 0 && nk == 0) || stages == 0) return FA_OK;
  const size_t need = fa::backward_workspace_layout(pr).total_min;
  if (nq > 0 && nk > 0) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
      return FA_ERR_INVALID_ARG;
  }
  if (!fa::device_status_word()) return FA_ERR_CUDA;
  int launches = 0;
  cudaError_t e = fa::launch_backward(pr, Q, K, V, O, dO, L, dQ, dK, dV, workspace, workspace_bytes, stages,
                                      static_cast<cudaStream_t>(stream), &launches);
  t_last_launches = launches;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_backward(const fa_dims* dims, const void* Q, const void* K, const void* V, const void* O,
                      const void* dO, const float* L, void* dQ, void* dK, void* dV, void* workspace,
                      size_t workspace_bytes, void* stream) {
  return fa_backward_stages(dims, Q, K, V, O, dO, L, dQ, dK, dV, workspace, workspace_bytes, FA_BWD_ALL, stream);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK:
      return "ok";
    case FA_ERR_INVALID_ARG:
      return "invalid argument (null or misaligned pointer, negative size, Hq not a multiple of Hkv, "
             "bad causal flag, window or scale, or workspace too small)";
    case FA_ERR_UNSUPPORTED:
      return "unsupported shape (d and dv must each be 64 or 128; sizes within the grid limits)";
    case FA_ERR_CUDA:
      return "CUDA error while encoding tensor maps or launching kernels";
    case FA_ERR_TIMEOUT:
      return "a kernel gave up waiting on an on-chip barrier; outputs are undefined";
    case FA_ERR_SCRATCH_TOO_SMALL:
      return "problem needs more scratch than fa_backward_noalloc's fixed array holds; use fa_backward";
  }
  return "unknown status";
}

fa_status fa_last_device_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  int* w = fa::device_status_word();
  if (!w) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyAsync(&v, w, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemsetAsync(w, 0, sizeof(int), st) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  return v == 0 ? FA_OK : FA_ERR_TIMEOUT;
}

int fa_last_launch_count(void) { return t_last_launches; }

#ifdef FA_TEST_HOOKS
// Test build only (not declared in fa.h): 1 makes the forward's producer
// withhold the Q tile, 2 the backward's producer withhold every dO tile, 0
// restores normal loads.  Applies to launches made after the call.
FA_API void fa_test_set_withhold(int what) { g_test_withhold.store(what); }
#endif

}  // extern "C"
