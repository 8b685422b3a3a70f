// sage_internal.cuh -- declarations shared by the library's translation units
// (kernel launchers and their argument blocks).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace sage {

constexpr int kHeadDim = 128;   // the only head dimension the method takes
constexpr int kQKBlock = 32;    // tokens per Q/K quantisation block
constexpr int kTile = 128;      // query rows per Q tile and keys per KV tile

// Device error word codes (read back by the host after a stream sync).
enum : int { SAGE_DEVERR_NONE = 0, SAGE_DEVERR_TIMEOUT = 1 };

inline int padded_len(int S) { return (S + kTile - 1) / kTile * kTile; }
inline int num_blocks(int S) { return (S + kQKBlock - 1) / kQKBlock; }

template <typename CodeT>
struct QKQuantArgs {
  const uint16_t* q;   // bf16 [B, S, H, 128]
  const uint16_t* k;
  CodeT* q_codes;      // [B, H, S_pad, 128]
  CodeT* k_codes;
  float* q_scale;      // [B, H, nb]
  float* k_scale;
  int BH, H;
  int S[2], S_pad[2], nb[2];   // per tensor: [0] Q, [1] K (cross-attention: they differ)
  int first = 0;               // 1: quantise K only (Q is quantised inside the attention kernel)
  const float* k_mean = nullptr;   // K smoothing: per (b, h, d) means of K over its tokens [B*H*128]
  void set_lengths(int Sq, int Sk) {
    S[0] = Sq; S_pad[0] = padded_len(Sq); nb[0] = num_blocks(Sq);
    S[1] = Sk; S_pad[1] = padded_len(Sk); nb[1] = num_blocks(Sk);
  }
};

// The quantisation of Q, K and V, in three launches: the zeroing of the
// per-channel V maxima (amax_bits [B*H*128] scratch), the Q/K codes together
// with those maxima, then the E4M3 V^T codes and scales (vt [B, H, 128,
// S_pad], v_scale [B, H, 128]).  V has the K length a.S[1].  With
// v == nullptr only the Q/K codes are made (one launch; amax_bits, vt and
// v_scale unused).
template <typename CodeT>
cudaError_t launch_qkv_quantize(const QKQuantArgs<CodeT>& a, const uint16_t* v, uint32_t* amax_bits, uint8_t* vt,
                                float* v_scale, cudaStream_t stream);

// K smoothing: per-channel means of K over its S tokens, mean = fp32(sum / S)
// with the sum exact (64-bit fixed point, 2^-40, for |k| in [2^-33, 2^23)).
// sums: [B*H*128] 64-bit scratch (zeroed here); mean: [B*H*128] floats out.
cudaError_t launch_k_channel_means(const uint16_t* k, int B, int S, int H, unsigned long long* sums, float* mean,
                                   cudaStream_t stream);


cudaError_t launch_widen_codes(const int8_t* src, __half* dst, size_t n, cudaStream_t stream);

struct AttnArgs {
  const uint16_t* q_bf16;   // if set: bf16 Q [B, Sq, H, 128], quantised inside the attention kernel
                            // (q_codes and q_scale are then not read)
  int8_t* q_dump;           // optional (with q_bf16): the kernel's Q codes, int8 [B, H, Sq_pad, 128]
  float* q_scale_dump;      // optional (with q_bf16): its Q block scales [B, H, nbq]
  const __half* q_codes;    // integer-valued fp16 codes [B, H, S_pad, 128]
  const __half* k_codes;
  const uint8_t* vt;        // e4m3 V^T [B, H, 128, S_pad]
  const float* q_scale;     // [B, H, nbq]
  const float* k_scale;     // [B, H, nbk]
  const float* v_scale;     // [B, H, 128]
  uint16_t* out;            // bf16 [B, Sq, H, 128]
  int32_t* s_dump;          // optional int32 Q K^T [B, H, Sq, Skv] (debug entry only)
  float* lse;               // optional fp32 [B, H, Sq]: per-row log-sum-exp
  int B, Sq, Skv, H, Sq_pad, Skv_pad, nbq, nbk;   // Q rows / K,V rows (equal unless cross)
  float softmax_scale;
  uint64_t timeout_ns;
};

// Encodes the three TMA maps and launches the fused attention kernel.
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream);

// Load every kernel a quantise-then-attend call can launch (K smoothing and
// the fused-Q attention kernel included) into the current context, so that a
// stream capture that launches them does not have to load a module.
cudaError_t load_attention_kernels();
cudaError_t load_quantize_kernels();

// Records printf-style text as this thread's sage_last_error() message.
void set_last_error(const char* fmt, ...);

// Device error word helpers (per device; set by bounded waits).
cudaError_t read_and_clear_device_error(int* code, cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(uint64_t timeout_ns, cudaStream_t stream);

// ------------------------------------------------------ device helpers --
// Shared by the quantisation and attention kernels.


}  // namespace sage
