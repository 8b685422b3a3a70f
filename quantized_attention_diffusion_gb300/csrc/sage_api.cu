// sage_api.cu -- the extern "C" boundary: argument checks, workspace layout,
// stream-ordered scratch, launch sequences and error mapping.  Declarations
// and their contracts are in include/sage.h.
#include <atomic>
#include <cinttypes>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "sage.h"
#include "sage_internal.cuh"

using namespace sage;

namespace {

thread_local std::string t_last_error;
thread_local cudaEvent_t t_attn_before = nullptr, t_attn_after = nullptr;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

sage_status fail(sage_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

sage_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SAGE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

sage_status check_shape(int B, int S, int H, int D) {
  if (D != kHeadDim)
    return fail(SAGE_ERR_UNSUPPORTED, "head dimension %d is not supported: this kernel takes D = 128", D);
  if (B < 1 || S < 1 || H < 1) return fail(SAGE_ERR_INVALID_ARG, "B, S and H must be >= 1 (got %d, %d, %d)", B, S, H);
  if (static_cast<int64_t>(B) * H > INT_MAX) return fail(SAGE_ERR_INVALID_ARG, "B*H exceeds 2^31-1");
  if (S > (1 << 28)) return fail(SAGE_ERR_INVALID_ARG, "S = %d exceeds 2^28", S);
  return SAGE_OK;
}

sage_status check_scale(float softmax_scale) {
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.0f))
    return fail(SAGE_ERR_INVALID_ARG, "softmax_scale must be finite and > 0 (got %g)", softmax_scale);
  return SAGE_OK;
}

sage_status check_ptrs(std::initializer_list<std::pair<const void*, const char*>> ptrs) {
  for (auto& pr : ptrs) {
    if (!pr.first) return fail(SAGE_ERR_INVALID_ARG, "%s is NULL", pr.second);
    if (!aligned(pr.first, 16)) return fail(SAGE_ERR_MISALIGNED, "%s is not 16-byte aligned", pr.second);
  }
  return SAGE_OK;
}

// The attention kernel writes each output row as 32-byte vectors.
sage_status check_out(const void* out) {
  if (!aligned(out, 32)) return fail(SAGE_ERR_MISALIGNED, "out is not 32-byte aligned");
  return SAGE_OK;
}

// Workspace layout (all offsets 256-byte aligned).
struct WsLayout {
  size_t q16, k16, vt, qs, ks, vs, vamax, ksum, kmean, total;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Sq query rows, Sk key/value rows (equal for self-attention).
WsLayout ws_layout(int B, int Sq, int Sk, int H) {
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t Sqp = padded_len(Sq), Skp = padded_len(Sk), nbq = num_blocks(Sq), nbk = num_blocks(Sk);
  WsLayout w;
  size_t off = 0;
  w.q16 = off; off += align256(BH * Sqp * kHeadDim * sizeof(__half));
  w.k16 = off; off += align256(BH * Skp * kHeadDim * sizeof(__half));
  w.vt = off; off += align256(BH * kHeadDim * Skp);
  w.qs = off; off += align256(BH * nbq * sizeof(float));
  w.ks = off; off += align256(BH * nbk * sizeof(float));
  w.vs = off; off += align256(BH * kHeadDim * sizeof(float));
  w.vamax = off; off += align256(BH * kHeadDim * sizeof(uint32_t));
  w.ksum = off; off += align256(BH * kHeadDim * sizeof(unsigned long long));
  w.kmean = off; off += align256(BH * kHeadDim * sizeof(float));
  w.total = off;
  return w;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}

// Host-only fault injection (a test hook, off by default): when armed for a
// site, the site's skip-th next event reports a failure without doing the
// work (no allocation, no launch), and the hook disarms.  Nothing faults on
// the device.
std::atomic<int> g_fault_site{0};
std::atomic<int> g_fault_skip{0};

bool fault_fires(int site) {
  if (g_fault_site.load(std::memory_order_relaxed) != site) return false;
  if (g_fault_skip.fetch_sub(1, std::memory_order_relaxed) > 0) return false;
  g_fault_site.store(0, std::memory_order_relaxed);
  return true;
}

// One private stream-ordered pool per device; memory is kept by the pool
// (release threshold = max) so steady-state calls do not go to the driver.
// A pool is published in g_pools only once its release threshold is set.
constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

sage_status current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices)
    return fail(SAGE_ERR_CUDA, "device index %d exceeds this library's %d-device table", *dev, kMaxDevices);
  return SAGE_OK;
}

// `bytes` of stream-ordered scratch for `what` on the current device.
sage_status pool_alloc(void** ptr, size_t bytes, cudaStream_t stream, const char* what) {
  if (fault_fires(SAGE_FAULT_POOL_ALLOC))
    return fail(SAGE_ERR_NO_MEMORY, "%s allocation of %zu bytes failed: injected fault", what, bytes);
  int dev = 0;
  sage_status s = current_device(&dev);
  if (s != SAGE_OK) return s;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (!g_pools[dev]) {
      cudaMemPoolProps props;
      std::memset(&props, 0, sizeof props);
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t fresh = nullptr;
      cudaError_t e = cudaMemPoolCreate(&fresh, &props);
      if (e != cudaSuccess) return cuda_fail(e, "memory pool creation");
      uint64_t thr = UINT64_MAX;
      e = cudaMemPoolSetAttribute(fresh, cudaMemPoolAttrReleaseThreshold, &thr);
      if (e != cudaSuccess) {
        (void)cudaMemPoolDestroy(fresh);
        return cuda_fail(e, "memory pool release threshold");
      }
      g_pools[dev] = fresh;
    }
    pool = g_pools[dev];
  }
  cudaError_t e = cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
  if (e != cudaSuccess) {
    // An out-of-memory result is not sticky, but the runtime keeps it as the
    // thread's last error: clear it so that it is not reported by a later
    // call's launch check.
    (void)cudaGetLastError();
    return fail(SAGE_ERR_NO_MEMORY, "%s allocation of %zu bytes failed: %s", what, bytes, cudaGetErrorString(e));
  }
  return SAGE_OK;
}

// Allocate `bytes` of workspace from the pool, run `body(ws)`, release the
// workspace in stream order whatever body returned.
template <typename Body>
sage_status with_pool_workspace(size_t bytes, cudaStream_t st, Body body) {
  void* ws = nullptr;
  sage_status s = pool_alloc(&ws, bytes, st, "workspace");
  if (s != SAGE_OK) return s;
  s = body(ws);
  cudaError_t e = cudaFreeAsync(ws, st);
  if (s != SAGE_OK) return s;
  if (e != cudaSuccess) return cuda_fail(e, "workspace release");
  return SAGE_OK;
}

uint64_t timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

// Arguments of the Q/K quantisation that feeds the attention kernel: integer
// codes stored as fp16 (the MMA operand type), [B, H, S_pad, 128].  With
// k_only, Q is left to the attention kernel; k_mean selects K smoothing.
QKQuantArgs<__half> staging_args(const void* q, const void* k, int B, int Sq, int Sk, int H, __half* q16,
                                 float* q_scale, __half* k16, float* k_scale, bool k_only, const float* k_mean) {
  QKQuantArgs<__half> qa;
  qa.q = static_cast<const uint16_t*>(q);
  qa.k = static_cast<const uint16_t*>(k);
  qa.q_codes = q16;
  qa.k_codes = k16;
  qa.q_scale = q_scale;
  qa.k_scale = k_scale;
  qa.BH = B * H;
  qa.H = H;
  qa.set_lengths(Sq, Sk);
  qa.first = k_only ? 1 : 0;
  qa.k_mean = k_mean;
  return qa;
}

// Arguments of the public INT8 quantisation (sage_quantize_qkv and its
// variants): codes [B, H, S_pad, 128].
QKQuantArgs<int8_t> public_args(const void* q, const void* k, int B, int S, int H, int8_t* q_i8, float* q_scale,
                                int8_t* k_i8, float* k_scale, const float* k_mean) {
  QKQuantArgs<int8_t> qa;
  qa.q = static_cast<const uint16_t*>(q);
  qa.k = static_cast<const uint16_t*>(k);
  qa.q_codes = q_i8;
  qa.k_codes = k_i8;
  qa.q_scale = q_scale;
  qa.k_scale = k_scale;
  qa.BH = B * H;
  qa.H = H;
  qa.set_lengths(S, S);
  qa.k_mean = k_mean;
  return qa;
}

// Quantise Q, K and V, then attend.  With fuse_q, only K and V are quantised
// here and the attention kernel quantises Q itself (q_dump / q_scale_dump
// then receive its codes and scales, if given).
sage_status run_fused(const void* q, const void* k, const void* v, void* out, int B, int Sq, int Sk,
                      int H, float softmax_scale, void* ws, cudaStream_t st, float* lse = nullptr,
                      bool fuse_q = false, int8_t* q_dump = nullptr, float* q_scale_dump = nullptr,
                      bool smooth_k = false) {
  const WsLayout w = ws_layout(B, Sq, Sk, H);
  if (smooth_k) {
    cudaError_t e0 = launch_k_channel_means(static_cast<const uint16_t*>(k), B, Sk, H, at<unsigned long long>(ws, w.ksum),
                                            at<float>(ws, w.kmean), st);
    if (e0 != cudaSuccess) return cuda_fail(e0, "K channel means launch");
  }
  const QKQuantArgs<__half> qa = staging_args(q, k, B, Sq, Sk, H, at<__half>(ws, w.q16), at<float>(ws, w.qs),
                                              at<__half>(ws, w.k16), at<float>(ws, w.ks), fuse_q,
                                              smooth_k ? at<float>(ws, w.kmean) : nullptr);
  if (fault_fires(SAGE_FAULT_QUANT_LAUNCH)) return fail(SAGE_ERR_CUDA, "quantisation launch: injected fault");
  cudaError_t e = launch_qkv_quantize<__half>(qa, static_cast<const uint16_t*>(v), at<uint32_t>(ws, w.vamax),
                                              at<uint8_t>(ws, w.vt), at<float>(ws, w.vs), st);
  if (e != cudaSuccess) return cuda_fail(e, "quantisation launch");
  AttnArgs aa;
  aa.q_bf16 = fuse_q ? static_cast<const uint16_t*>(q) : nullptr;
  aa.q_dump = q_dump;
  aa.q_scale_dump = q_scale_dump;
  aa.q_codes = fuse_q ? nullptr : qa.q_codes;
  aa.k_codes = qa.k_codes;
  aa.vt = at<uint8_t>(ws, w.vt);
  aa.q_scale = fuse_q ? nullptr : qa.q_scale;
  aa.k_scale = qa.k_scale;
  aa.v_scale = at<float>(ws, w.vs);
  aa.out = static_cast<uint16_t*>(out);
  aa.s_dump = nullptr;
  aa.lse = lse;
  aa.B = B;
  aa.Sq = Sq;
  aa.Skv = Sk;
  aa.H = H;
  aa.Sq_pad = padded_len(Sq);
  aa.Skv_pad = padded_len(Sk);
  aa.nbq = num_blocks(Sq);
  aa.nbk = num_blocks(Sk);
  aa.softmax_scale = softmax_scale;
  aa.timeout_ns = timeout_ns();
  if (t_attn_before && (e = cudaEventRecord(t_attn_before, st)) != cudaSuccess)
    return cuda_fail(e, "timing event record");
  if (fault_fires(SAGE_FAULT_ATTN_LAUNCH)) return fail(SAGE_ERR_CUDA, "attention launch: injected fault");
  e = launch_attention(aa, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  if (t_attn_after && (e = cudaEventRecord(t_attn_after, st)) != cudaSuccess)
    return cuda_fail(e, "timing event record");
  return SAGE_OK;
}

sage_status run_quantized(const int8_t* q_i8, const float* q_scale, const int8_t* k_i8,
                          const float* k_scale, const uint8_t* vt, const float* v_scale, void* out,
                          int32_t* s_dump, int B, int S, int H, float softmax_scale, void* ws,
                          cudaStream_t st) {
  const WsLayout w = ws_layout(B, S, S, H);
  const int Sp = padded_len(S);
  const size_t n = static_cast<size_t>(B) * H * Sp * kHeadDim;
  cudaError_t e = launch_widen_codes(q_i8, at<__half>(ws, w.q16), n, st);
  if (e == cudaSuccess) e = launch_widen_codes(k_i8, at<__half>(ws, w.k16), n, st);
  if (e != cudaSuccess) return cuda_fail(e, "code widening launch");
  AttnArgs aa;
  aa.q_bf16 = nullptr;
  aa.q_dump = nullptr;
  aa.q_scale_dump = nullptr;
  aa.q_codes = at<__half>(ws, w.q16);
  aa.k_codes = at<__half>(ws, w.k16);
  aa.vt = vt;
  aa.q_scale = q_scale;
  aa.k_scale = k_scale;
  aa.v_scale = v_scale;
  aa.out = static_cast<uint16_t*>(out);
  aa.s_dump = s_dump;
  aa.lse = nullptr;
  aa.B = B;
  aa.Sq = S;
  aa.Skv = S;
  aa.H = H;
  aa.Sq_pad = Sp;
  aa.Skv_pad = Sp;
  aa.nbq = num_blocks(S);
  aa.nbk = num_blocks(S);
  aa.softmax_scale = softmax_scale;
  aa.timeout_ns = timeout_ns();
  e = launch_attention(aa, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return SAGE_OK;
}

sage_status check_workspace(void* ws, size_t bytes, int B, int S, int H) {
  const size_t need = ws_layout(B, S, S, H).total;
  if (!ws) return fail(SAGE_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(SAGE_ERR_MISALIGNED, "workspace is not 256-byte aligned");
  if (bytes < need)
    return fail(SAGE_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", bytes, need);
  return SAGE_OK;
}

}  // namespace

// The host object behind sage_plan (opaque to callers).
struct sage_plan {
  int device;              // device the graph and workspace belong to
  void* ws;                // cudaMalloc'd workspace the recorded launches use
  cudaGraphExec_t exec;    // the recorded sage_attn_fwd_cross call
};

void sage::set_last_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
}

extern "C" {

int64_t sage_padded_len(int S) { return S < 1 ? 0 : static_cast<int64_t>(padded_len(S)); }

int sage_attn_fwd_launches(int B, int Sq, int Skv, int H, int smooth_k) {
  if (B < 1 || Sq < 1 || Skv < 1 || H < 1) return -1;
  // Zeroing of the V maxima, Q/K quantisation with the V maxima, V encoding,
  // attention; K smoothing adds the channel sums and means.
  return 4 + (smooth_k ? 2 : 0);
}

size_t sage_workspace_bytes(int B, int S, int H, int D) {
  if (D != kHeadDim || B < 1 || S < 1 || H < 1 || static_cast<int64_t>(B) * H > INT_MAX || S > (1 << 28))
    return 0;
  return ws_layout(B, S, S, H).total;
}

sage_status sage_quantize_qkv(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                              int8_t* q_i8, float* q_scale, int8_t* k_i8, float* k_scale,
                              uint8_t* vt_fp8, float* v_scale, void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK)
    s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {q_i8, "q_i8"}, {q_scale, "q_scale"}, {k_i8, "k_i8"},
                    {k_scale, "k_scale"}, {vt_fp8, "vt_fp8"}, {v_scale, "v_scale"}});
  if (s != SAGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  s = pool_alloc(&scratch, static_cast<size_t>(B) * H * kHeadDim * sizeof(uint32_t), st, "V maxima scratch");
  if (s != SAGE_OK) return s;
  const QKQuantArgs<int8_t> qa = public_args(q, k, B, S, H, q_i8, q_scale, k_i8, k_scale, nullptr);
  cudaError_t e = launch_qkv_quantize<int8_t>(qa, static_cast<const uint16_t*>(v), static_cast<uint32_t*>(scratch),
                                              vt_fp8, v_scale, st);
  cudaError_t e2 = cudaFreeAsync(scratch, st);
  if (e != cudaSuccess) return cuda_fail(e, "quantisation launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "scratch release");
  return SAGE_OK;
}

sage_status sage_quantize_qkv_smooth_k(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                                       int8_t* q_i8, float* q_scale, int8_t* k_i8, float* k_scale, uint8_t* vt_fp8,
                                       float* v_scale, float* k_mean, void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK)
    s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {q_i8, "q_i8"}, {q_scale, "q_scale"}, {k_i8, "k_i8"},
                    {k_scale, "k_scale"}, {vt_fp8, "vt_fp8"}, {v_scale, "v_scale"}, {k_mean, "k_mean"}});
  if (s != SAGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t sum_bytes = align256(BH * kHeadDim * sizeof(unsigned long long));
  void* scratch = nullptr;
  s = pool_alloc(&scratch, sum_bytes + BH * kHeadDim * sizeof(uint32_t), st, "K sums and V maxima scratch");
  if (s != SAGE_OK) return s;
  unsigned long long* sums = static_cast<unsigned long long*>(scratch);
  cudaError_t e = launch_k_channel_means(static_cast<const uint16_t*>(k), B, S, H, sums, k_mean, st);
  if (e == cudaSuccess) {
    const QKQuantArgs<int8_t> qa = public_args(q, k, B, S, H, q_i8, q_scale, k_i8, k_scale, k_mean);
    e = launch_qkv_quantize<int8_t>(qa, static_cast<const uint16_t*>(v), at<uint32_t>(scratch, sum_bytes), vt_fp8,
                                    v_scale, st);
  }
  cudaError_t e2 = cudaFreeAsync(scratch, st);
  if (e != cudaSuccess) return cuda_fail(e, "quantisation launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "scratch release");
  return SAGE_OK;
}

sage_status sage_attn_fwd_smooth_k(const void* q, const void* k, const void* v, void* out, int B, int S, int H,
                                   int D, float softmax_scale, void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK) s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s != SAGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return with_pool_workspace(ws_layout(B, S, S, H).total, st, [&](void* ws) {
    return run_fused(q, k, v, out, B, S, S, H, softmax_scale, ws, st, nullptr, false, nullptr, nullptr, true);
  });
}

sage_status sage_attn_fwd_ws(const void* q, const void* k, const void* v, void* out, int B, int S,
                             int H, int D, float softmax_scale, void* workspace,
                             size_t workspace_bytes, void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK) s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s == SAGE_OK) s = check_workspace(workspace, workspace_bytes, B, S, H);
  if (s != SAGE_OK) return s;
  return run_fused(q, k, v, out, B, S, S, H, softmax_scale, workspace, static_cast<cudaStream_t>(stream));
}

sage_status sage_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int S, int H,
                          int D, float softmax_scale, void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK) s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s != SAGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return with_pool_workspace(ws_layout(B, S, S, H).total, st, [&](void* ws) {
    return run_fused(q, k, v, out, B, S, S, H, softmax_scale, ws, st);
  });
}

sage_status sage_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                              int S, int H, int D, float softmax_scale, void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK) s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}, {lse, "lse"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s != SAGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return with_pool_workspace(ws_layout(B, S, S, H).total, st, [&](void* ws) {
    return run_fused(q, k, v, out, B, S, S, H, softmax_scale, ws, st, lse);
  });
}

sage_status sage_attn_fwd_cross(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                                int Sq, int Skv, int H, int D, float softmax_scale, void* stream) {
  sage_status s = check_shape(B, Sq, H, D);
  if (s == SAGE_OK) s = check_shape(B, Skv, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK) s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s == SAGE_OK && lse) s = check_ptrs({{lse, "lse"}});
  if (s != SAGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return with_pool_workspace(ws_layout(B, Sq, Skv, H).total, st, [&](void* ws) {
    return run_fused(q, k, v, out, B, Sq, Skv, H, softmax_scale, ws, st, lse);
  });
}

sage_status sage_plan_create(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Sq,
                             int Skv, int H, int D, float softmax_scale, sage_plan** plan) {
  return sage_plan_create_ex(q, k, v, out, lse, B, Sq, Skv, H, D, softmax_scale, 0u, plan);
}

sage_status sage_plan_create_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Sq,
                                int Skv, int H, int D, float softmax_scale, unsigned flags, sage_plan** plan) {
  if (!plan) return fail(SAGE_ERR_INVALID_ARG, "plan is NULL");
  *plan = nullptr;
  if ((flags & ~(SAGE_PLAN_SMOOTH_K | SAGE_PLAN_FUSED_Q)) != 0u ||
      flags == (SAGE_PLAN_SMOOTH_K | SAGE_PLAN_FUSED_Q))
    return fail(SAGE_ERR_UNSUPPORTED, "plan flags 0x%x: no call offers that combination", flags);
  const bool smooth_k = (flags & SAGE_PLAN_SMOOTH_K) != 0u, fuse_q = (flags & SAGE_PLAN_FUSED_Q) != 0u;
  if (flags != 0u && (Sq != Skv || lse != nullptr))
    return fail(SAGE_ERR_INVALID_ARG, "plan flags 0x%x record a self-attention call without LSE (Sq %d, Skv %d%s)",
                flags, Sq, Skv, lse ? ", lse given" : "");
  sage_status s = check_shape(B, Sq, H, D);
  if (s == SAGE_OK) s = check_shape(B, Skv, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK) s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s == SAGE_OK && lse) s = check_ptrs({{lse, "lse"}});
  int dev = 0;
  if (s == SAGE_OK) s = current_device(&dev);
  if (s != SAGE_OK) return s;

  const size_t bytes = ws_layout(B, Sq, Skv, H).total;
  void* ws = nullptr;
  cudaError_t e = fault_fires(SAGE_FAULT_POOL_ALLOC) ? cudaErrorMemoryAllocation : cudaMalloc(&ws, bytes);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(SAGE_ERR_NO_MEMORY, "plan workspace allocation of %zu bytes failed: %s", bytes, cudaGetErrorString(e));
  }
  cudaStream_t cs = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  e = load_quantize_kernels();                       // no module loading inside the capture
  if (e == cudaSuccess) e = load_attention_kernels();
  if (e != cudaSuccess) {
    cudaFree(ws);
    return cuda_fail(e, "plan kernel loading");
  }
  e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    cudaFree(ws);
    return cuda_fail(e, "plan capture stream");
  }
  // Record the launches of the call; the timing hook stays out of the graph.
  const cudaEvent_t before = t_attn_before, after = t_attn_after;
  t_attn_before = t_attn_after = nullptr;
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    s = run_fused(q, k, v, out, B, Sq, Skv, H, softmax_scale, ws, cs, lse, fuse_q, nullptr, nullptr, smooth_k);
    const cudaError_t e_end = cudaStreamEndCapture(cs, &graph);   // ends the capture whatever happened
    if (s == SAGE_OK && e_end != cudaSuccess) s = cuda_fail(e_end, "plan capture");
  } else {
    s = cuda_fail(e, "plan capture start");
  }
  t_attn_before = before;
  t_attn_after = after;
  if (s == SAGE_OK) {
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) s = cuda_fail(e, "plan graph instantiation");
  }
  if (graph) cudaGraphDestroy(graph);
  cudaStreamDestroy(cs);
  sage_plan* p = nullptr;
  if (s == SAGE_OK) {
    p = new (std::nothrow) sage_plan{dev, ws, exec};
    if (!p) s = fail(SAGE_ERR_NO_MEMORY, "plan object allocation failed");
  }
  if (s != SAGE_OK) {
    if (exec) cudaGraphExecDestroy(exec);
    cudaFree(ws);
    (void)cudaGetLastError();   // a failed capture leaves no error for the next call
    return s;
  }
  *plan = p;
  return SAGE_OK;
}

sage_status sage_plan_launch(sage_plan* plan, void* stream) {
  if (!plan) return fail(SAGE_ERR_INVALID_ARG, "plan is NULL");
  int dev = 0;
  sage_status s = current_device(&dev);
  if (s != SAGE_OK) return s;
  if (dev != plan->device)
    return fail(SAGE_ERR_INVALID_ARG, "plan was created on device %d, current device is %d", plan->device, dev);
  if (fault_fires(SAGE_FAULT_ATTN_LAUNCH)) return fail(SAGE_ERR_CUDA, "plan launch: injected fault");
  const cudaError_t e = cudaGraphLaunch(plan->exec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  return SAGE_OK;
}

sage_status sage_plan_destroy(sage_plan* plan) {
  if (!plan) return SAGE_OK;
  cudaError_t e = cudaGraphExecDestroy(plan->exec);
  const cudaError_t e2 = cudaFree(plan->ws);
  delete plan;
  if (e == cudaSuccess) e = e2;
  if (e != cudaSuccess) return cuda_fail(e, "plan release");
  return SAGE_OK;
}

sage_status sage_attn_fwd_quantized(const int8_t* q_i8, const float* q_scale, const int8_t* k_i8,
                                    const float* k_scale, const uint8_t* vt_fp8,
                                    const float* v_scale, void* out, int B, int S, int H, int D,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK)
    s = check_ptrs({{q_i8, "q_i8"}, {q_scale, "q_scale"}, {k_i8, "k_i8"}, {k_scale, "k_scale"},
                    {vt_fp8, "vt_fp8"}, {v_scale, "v_scale"}, {out, "out"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s == SAGE_OK) s = check_workspace(workspace, workspace_bytes, B, S, H);
  if (s != SAGE_OK) return s;
  return run_quantized(q_i8, q_scale, k_i8, k_scale, vt_fp8, v_scale, out, nullptr, B, S, H, softmax_scale,
                       workspace, static_cast<cudaStream_t>(stream));
}

sage_status sage_debug_qk_int32(const int8_t* q_i8, const float* q_scale, const int8_t* k_i8,
                                const float* k_scale, const uint8_t* vt_fp8, const float* v_scale,
                                void* out, int32_t* s_out, int B, int S, int H, int D,
                                float softmax_scale, void* workspace, size_t workspace_bytes,
                                void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK)
    s = check_ptrs({{q_i8, "q_i8"}, {q_scale, "q_scale"}, {k_i8, "k_i8"}, {k_scale, "k_scale"},
                    {vt_fp8, "vt_fp8"}, {v_scale, "v_scale"}, {out, "out"}, {s_out, "s_out"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s == SAGE_OK) s = check_workspace(workspace, workspace_bytes, B, S, H);
  if (s != SAGE_OK) return s;
  return run_quantized(q_i8, q_scale, k_i8, k_scale, vt_fp8, v_scale, out, s_out, B, S, H, softmax_scale,
                       workspace, static_cast<cudaStream_t>(stream));
}

sage_status sage_attn_fwd_fused_q(const void* q, const void* k, const void* v, void* out, int B, int S,
                                  int H, int D, float softmax_scale, void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK) s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s != SAGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return with_pool_workspace(ws_layout(B, S, S, H).total, st, [&](void* ws) {
    return run_fused(q, k, v, out, B, S, S, H, softmax_scale, ws, st, nullptr, true);
  });
}

sage_status sage_debug_fused_q(const void* q, const void* k, const void* v, void* out, int B, int S, int H,
                               int D, float softmax_scale, int8_t* q_i8, float* q_scale, void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK) s = check_scale(softmax_scale);
  if (s == SAGE_OK)
    s = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}, {q_i8, "q_i8"}, {q_scale, "q_scale"}});
  if (s == SAGE_OK) s = check_out(out);
  if (s != SAGE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return with_pool_workspace(ws_layout(B, S, S, H).total, st, [&](void* ws) {
    return run_fused(q, k, v, out, B, S, S, H, softmax_scale, ws, st, nullptr, true, q_i8, q_scale);
  });
}

sage_status sage_debug_staging_codes(const void* q, const void* k, int B, int S, int H, int D, void* q16,
                                     float* q_scale, void* k16, float* k_scale, void* stream) {
  sage_status s = check_shape(B, S, H, D);
  if (s == SAGE_OK)
    s = check_ptrs({{q, "q"}, {k, "k"}, {q16, "q16"}, {q_scale, "q_scale"}, {k16, "k16"}, {k_scale, "k_scale"}});
  if (s != SAGE_OK) return s;
  const QKQuantArgs<__half> qa = staging_args(q, k, B, S, S, H, static_cast<__half*>(q16), q_scale,
                                              static_cast<__half*>(k16), k_scale, false, nullptr);
  cudaError_t e = launch_qkv_quantize<__half>(qa, nullptr, nullptr, nullptr, nullptr, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "Q/K quantisation launch");
  return SAGE_OK;
}

sage_status sage_debug_inject_fault(int site, int skip) {
  if (site < SAGE_FAULT_NONE || site > SAGE_FAULT_ATTN_LAUNCH || skip < 0)
    return fail(SAGE_ERR_INVALID_ARG, "fault site %d / skip %d out of range", site, skip);
  g_fault_site.store(SAGE_FAULT_NONE, std::memory_order_relaxed);
  g_fault_skip.store(skip, std::memory_order_relaxed);
  g_fault_site.store(site, std::memory_order_relaxed);
  return SAGE_OK;
}

sage_status sage_debug_pool_state(int* created, uint64_t* used_bytes) {
  if (!created || !used_bytes) return fail(SAGE_ERR_INVALID_ARG, "created and used_bytes must not be NULL");
  int dev = 0;
  sage_status s = current_device(&dev);
  if (s != SAGE_OK) return s;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    pool = g_pools[dev];
  }
  *created = pool != nullptr;
  *used_bytes = 0;
  if (pool) {
    cuuint64_t used = 0;
    cudaError_t e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemCurrent, &used);
    if (e != cudaSuccess) return cuda_fail(e, "memory pool query");
    *used_bytes = static_cast<uint64_t>(used);
  }
  return SAGE_OK;
}

sage_status sage_debug_wait_timeout(uint64_t ns, void* stream) {
  if (ns < 1 || ns > 10000000000ull) return fail(SAGE_ERR_INVALID_ARG, "timeout_ns must be in [1, 1e10]");
  cudaError_t e = launch_wait_timeout_probe(ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
  return SAGE_OK;
}

sage_status sage_sync_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
  int code = 0;
  e = read_and_clear_device_error(&code, st);
  if (e != cudaSuccess) return cuda_fail(e, "device error word read");
  if (code == SAGE_DEVERR_TIMEOUT)
    return fail(SAGE_ERR_TIMEOUT, "a device-side wait gave up after its time limit");
  return SAGE_OK;
}

void sage_set_attention_events(void* before, void* after) {
  t_attn_before = static_cast<cudaEvent_t>(before);
  t_attn_after = static_cast<cudaEvent_t>(after);
}

void sage_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : kDefaultTimeoutNs); }

const char* sage_last_error(void) { return t_last_error.c_str(); }

const char* sage_status_string(sage_status s) {
  switch (s) {
    case SAGE_OK: return "SAGE_OK";
    case SAGE_ERR_INVALID_ARG: return "SAGE_ERR_INVALID_ARG";
    case SAGE_ERR_UNSUPPORTED: return "SAGE_ERR_UNSUPPORTED";
    case SAGE_ERR_MISALIGNED: return "SAGE_ERR_MISALIGNED";
    case SAGE_ERR_CUDA: return "SAGE_ERR_CUDA";
    case SAGE_ERR_NO_MEMORY: return "SAGE_ERR_NO_MEMORY";
    case SAGE_ERR_TIMEOUT: return "SAGE_ERR_TIMEOUT";
    case SAGE_ERR_WORKSPACE: return "SAGE_ERR_WORKSPACE";
  }
  return "SAGE_ERR_UNKNOWN";
}

}  // extern "C"
