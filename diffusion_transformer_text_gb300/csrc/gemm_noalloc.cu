// qi_gemm_bf16_noalloc: the tensor-core GEMM for callers that may not allocate.
//
// qi_gemm_bf16 needs a qi_dit handle because the GEMM's bounded waits report
// into a device status word, and that word lives in memory the handle
// allocates. Creating a handle calls cudaMalloc (weights, activations). Some
// callers cannot do that: code running inside a host that owns all device
// memory (an inference server with a fixed arena, a plugin that is not allowed
// to touch the CUDA allocator). This entry point keeps the status word in a
// file-scope static device array instead, so it allocates nothing.
//
// The first call on a device does the set-up (the array's device address is
// looked up once, with that device current); make it before any stream
// capture. The address is kept for the life of the process, so the entry point
// must not be used on a device after cudaDeviceReset (or any other teardown of
// the device's primary context) in the same process. All calls on a device
// share the array and the last call's status stays in it: each call clears the
// word first, so calls that overlap on the GPU race on it and must be
// serialised by the caller.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/qidit.h"
#include "internal.h"

namespace {

// Scratch shared by every call on a device: 64 status words (256 bytes). Word 0
// is the GEMM's status (0 = ok, else the code of the wait that ran out). The
// array exists once per device that loads the library and lives until exit.
constexpr int kStatusWords = 64;
static __device__ __align__(256) int g_noalloc_status[kStatusWords];

// Largest shapes accepted: those of the DiT's own GEMMs. Rows: the longer of a
// joint pass (L + N) and the batch-2 image-only guidance pass (2 N); columns: the
// stacked gate/up width; contraction: the SwiGLU inner width.
constexpr int kMaxM = QI_L_MAX + QI_N_MAX > 2 * QI_N_MAX ? QI_L_MAX + QI_N_MAX : 2 * QI_N_MAX;
constexpr int kMaxN = 2 * QI_FFN;
constexpr int kMaxK = QI_FFN;
constexpr int kMaxDevices = 64;

struct DeviceSlot {
  int* status = nullptr;  // device address of g_noalloc_status on this device
  int num_sms = 0;
};
DeviceSlot g_slots[kMaxDevices];
std::mutex g_slots_mu;

qi_status noalloc_fail(qi_status st, const char* fmt, int a = 0, int b = 0, int c = 0, int d = 0, int e = 0,
                       int f = 0) {
  char buf[256];
  snprintf(buf, sizeof(buf), fmt, a, b, c, d, e, f);
  qi::set_last_error(buf);  // read back with qi_last_error()
  return st;
}

// Once per device, with that device current: look up the array's device address.
qi_status device_slot(DeviceSlot** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return noalloc_fail(QI_ERR_CUDA, "qi_gemm_bf16_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(QI_ERR_INVALID_ARG, "qi_gemm_bf16_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_slots_mu);
  DeviceSlot& s = g_slots[dev];
  if (s.status == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_status);
    if (e != cudaSuccess || ptr == nullptr)
      return noalloc_fail(QI_ERR_CUDA, "qi_gemm_bf16_noalloc: cudaGetSymbolAddress failed on device %d", dev);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms <= 0)
      return noalloc_fail(QI_ERR_CUDA, "qi_gemm_bf16_noalloc: SM count query failed on device %d", dev);
    s.num_sms = sms;
    s.status = static_cast<int*>(ptr);
  }
  *out = &s;
  return QI_OK;
}

}  // namespace

extern "C" qi_status qi_gemm_bf16_noalloc(const uint16_t* A, const uint16_t* B, float* D, int M, int N, int K,
                                          int sync_check, qi_stream_t stream) {
  if (!A || !B || !D) return noalloc_fail(QI_ERR_INVALID_ARG, "qi_gemm_bf16_noalloc: NULL argument");
  if (M < 1 || N < qi::kBN || N % qi::kBN != 0 || K < qi::kBK || K % qi::kBK != 0)
    return noalloc_fail(QI_ERR_SHAPE, "qi_gemm_bf16_noalloc: M %d N %d K %d (need N %% 256 == 0, K %% 64 == 0)", M,
                        N, K);
  if (M > kMaxM || N > kMaxN || K > kMaxK)
    return noalloc_fail(QI_ERR_SHAPE, "qi_gemm_bf16_noalloc: M %d N %d K %d above the limits %d x %d x %d", M, N, K,
                        kMaxM, kMaxN, kMaxK);
  if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
      (reinterpret_cast<uintptr_t>(D) & 15))
    return noalloc_fail(QI_ERR_INVALID_ARG, "qi_gemm_bf16_noalloc: A, B and D must be 16-byte aligned");
  DeviceSlot* slot = nullptr;
  qi_status st = device_slot(&slot);
  if (st != QI_OK) return st;
  CUtensorMap ma, mb;
  // the same bf16 maps qi_gemm_bf16 builds, so both entry points run identical launches
  if (!qi::encode_map16(&ma, A, M, K, 128, true) || !qi::encode_map16(&mb, B, N, K, qi::kBoxRowsPair, true))
    return noalloc_fail(QI_ERR_CUDA, "qi_gemm_bf16_noalloc: tensor map encoding failed");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word must start at zero for this call
  cudaError_t e = cudaMemsetAsync(slot->status, 0, sizeof(int), s);
  if (e != cudaSuccess) return noalloc_fail(QI_ERR_CUDA, "qi_gemm_bf16_noalloc: clearing the status word failed");
  qi::GemmParams g{};
  g.M = M;
  g.N = N;
  g.K = K;
  g.d = D;
  g.err = slot->status;
  e = qi::launch_gemm(qi::kEpiF32, ma, mb, g, slot->num_sms, s);
  if (e != cudaSuccess) return noalloc_fail(QI_ERR_CUDA, "qi_gemm_bf16_noalloc: launch failed");
  if (sync_check) {
    int h = 0;
    e = cudaMemcpyAsync(&h, slot->status, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return noalloc_fail(QI_ERR_CUDA, "qi_gemm_bf16_noalloc: status read failed");
    if (h != 0) return noalloc_fail(QI_ERR_DEVICE_TIMEOUT, "qi_gemm_bf16_noalloc: a bounded wait expired (code %d)", h);
  }
  return QI_OK;
}
