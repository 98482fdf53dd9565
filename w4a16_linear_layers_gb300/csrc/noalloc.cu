// noalloc.cu -- qlin_gemm_w8a8_gs128_noalloc: the W8A8 GS128 linear for
// callers that cannot allocate device memory.
//
// The regular GEMM entry points take a caller-provided workspace for their
// split-K partial sums and arrival counters.  Some callers cannot provide one:
// code that runs where cudaMalloc is forbidden or unavailable (inside a
// custom allocator or memory-pool callback, in a plugin whose host framework
// owns every allocation, or in a process that must not grow its device
// footprint after start-up).  This entry point runs the same kernel with that
// scratch memory taken from a fixed array compiled into the library instead.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// (24 MiB).  Every GPU on which the library's module is loaded holds it until
// the process exits.  Host code cannot use the array's name as a device
// address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it; make that
// first call before any stream capture.  Problems whose scratch need exceeds
// the array are rejected with QLIN_ERR_TOO_LARGE (on a 152-SM GB300 this
// covers every shape with M <= 96 and K <= 50,000).
//
// All calls share the one array and it keeps the last call's contents: the
// arrival counters are cleared with cudaMemsetAsync on the call's stream
// before each launch.  Calls that overlap on the GPU (different streams, or
// different host threads without ordering) race on the array.
#include <mutex>

#include "../../include/qlin.h"
#include "qlin_device.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr size_t kNoAllocScratchBytes = 24u << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

void lookup_scratch(int dev) {
  void* ptr = nullptr;
  g_scratch_err[dev] = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (g_scratch_err[dev] != cudaSuccess) {
    cudaGetLastError();
    ptr = nullptr;
  }
  g_scratch_ptr[dev] = ptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace qlin

using namespace qlin;

extern "C" qlin_status_t qlin_gemm_w8a8_gs128_noalloc(const int8_t* q_a, const float* s_a,
                                                      const int32_t* qweight,
                                                      const uint16_t* scales, int64_t M,
                                                      int64_t N, int64_t K, uint16_t* y,
                                                      qlin_stream_t stream) {
  if ((M != 0 && (q_a == nullptr || s_a == nullptr || y == nullptr)) || qweight == nullptr ||
      scales == nullptr)
    return QLIN_ERR_NULL;
  if (M < 0 || M > 2147483647LL || N < 8 || N > 2147483647LL || (N % 8) != 0 || K < kGroup ||
      K > 2147483647LL || (K % kGroup) != 0)
    return QLIN_ERR_SHAPE;
  if (!aligned16(q_a) || !aligned16(s_a) || !aligned16(qweight) || !aligned16(scales) ||
      !aligned16(y))
    return QLIN_ERR_ALIGN;
  const DeviceInfo* d = current_device();
  if (d == nullptr || !d->supported) return QLIN_ERR_DEVICE;
  if (M == 0) return QLIN_OK;
  const GemmPlan plan = plan_gemm(M, N, K, d->sm_count);
  if (plan.workspace_bytes > kNoAllocScratchBytes) return QLIN_ERR_TOO_LARGE;

  std::call_once(g_scratch_once[d->device], lookup_scratch, d->device);
  void* scratch = g_scratch_ptr[d->device];
  if (scratch == nullptr) return QLIN_ERR_CUDA;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, plan.counter_bytes, s) != cudaSuccess) return QLIN_ERR_CUDA;
  GemmArgs a{GemmMode::kW8A8, q_a, s_a, qweight, scales, y, M, N, K, scratch,
             kNoAllocScratchBytes};
  return launch_gemm(a, plan, d->err_word, s) == cudaSuccess ? QLIN_OK : QLIN_ERR_CUDA;
}
