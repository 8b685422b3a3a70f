// quantize_noalloc.cu -- sage_quantize_qkv for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they quantise: a host thread running under a framework that
// owns every device allocation, a real-time loop that must not take the
// driver's allocation locks, or code on a device whose memory is fully
// reserved up front.  sage_quantize_qkv normally takes its small scratch (the
// per-channel |V| maxima, 4 * B * H * 128 bytes) from a stream-ordered pool;
// the entry point here uses a fixed array in device memory instead, so it
// allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds kScratchBytes of it until the process exits.  Host code sees
// only a stand-in for its name, so its device address is looked up once per
// device (cudaGetSymbolAddress, with that device current) and passed to the
// kernels.
#include <climits>
#include <mutex>

#include "sage.h"
#include "sage_internal.cuh"

namespace {

constexpr int kMaxBH = 8192;                                   // B * H limit
constexpr size_t kScratchWords = static_cast<size_t>(kMaxBH) * sage::kHeadDim;

// The scratch: per-(batch*head, channel) |V| maxima as fp32 bit patterns.
static __device__ __align__(256) uint32_t g_vmax_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device

// Looks up (once per device, with that device current) the device address of
// g_vmax_scratch.  Returns nullptr and records the error text on failure.
uint32_t* scratch_for_current_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    sage::set_last_error("cudaGetDevice failed: %s", cudaGetErrorString(e));
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    sage::set_last_error("device index %d exceeds the %d-device table of sage_quantize_qkv_noalloc", dev,
                         kMaxDevices);
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_vmax_scratch);
    if (e != cudaSuccess || !p) {
      sage::set_last_error("cudaGetSymbolAddress of the scratch array failed: %s", cudaGetErrorString(e));
      return nullptr;
    }
    g_scratch_addr[dev] = static_cast<uint32_t*>(p);
  }
  return g_scratch_addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" sage_status sage_quantize_qkv_noalloc(const void* q, const void* k, const void* v, int B,
                                                 int S, int H, int D, int8_t* q_i8, float* q_scale,
                                                 int8_t* k_i8, float* k_scale, uint8_t* vt_fp8,
                                                 float* v_scale, void* stream) {
  if (D != sage::kHeadDim) {
    sage::set_last_error("head dimension %d is not supported: this kernel takes D = 128", D);
    return SAGE_ERR_UNSUPPORTED;
  }
  if (B < 1 || S < 1 || H < 1 || S > (1 << 28)) {
    sage::set_last_error("B, S and H must be >= 1 and S <= 2^28 (got %d, %d, %d)", B, S, H);
    return SAGE_ERR_INVALID_ARG;
  }
  if (static_cast<long long>(B) * H > kMaxBH) {
    sage::set_last_error("B*H = %lld exceeds %d, the size of the built-in scratch of "
                         "sage_quantize_qkv_noalloc (use sage_quantize_qkv)",
                         static_cast<long long>(B) * H, kMaxBH);
    return SAGE_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {q, k, v, q_i8, q_scale, k_i8, k_scale, vt_fp8, v_scale};
  const char* names[] = {"q", "k", "v", "q_i8", "q_scale", "k_i8", "k_scale", "vt_fp8", "v_scale"};
  for (int i = 0; i < 9; ++i) {
    if (!ptrs[i]) {
      sage::set_last_error("%s is NULL", names[i]);
      return SAGE_ERR_INVALID_ARG;
    }
    if (!aligned16(ptrs[i])) {
      sage::set_last_error("%s is not 16-byte aligned", names[i]);
      return SAGE_ERR_MISALIGNED;
    }
  }
  uint32_t* scratch = scratch_for_current_device();
  if (!scratch) return SAGE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  sage::QKQuantArgs<int8_t> qa;
  qa.q = static_cast<const uint16_t*>(q);
  qa.k = static_cast<const uint16_t*>(k);
  qa.q_codes = q_i8;
  qa.k_codes = k_i8;
  qa.q_scale = q_scale;
  qa.k_scale = k_scale;
  qa.BH = B * H;
  qa.H = H;
  qa.set_lengths(S, S);
  // launch_qkv_quantize zeroes the maxima (a kernel, no allocation) before
  // reducing into them, so the previous call's contents never leak.
  cudaError_t e = sage::launch_qkv_quantize<int8_t>(qa, static_cast<const uint16_t*>(v), scratch, vt_fp8, v_scale, st);
  if (e != cudaSuccess) {
    sage::set_last_error("quantisation launch failed: %s", cudaGetErrorString(e));
    return SAGE_ERR_CUDA;
  }
  return SAGE_OK;
}
