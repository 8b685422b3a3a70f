// quantize.cu -- HBM-bound quantisation kernels (sm_103a).
//
// Q/K: INT8 per 32-token block of one (batch, head), one fp32 scale per block
// (diffusers issue #15014 "gfx1201 (RDNA4) SageAttention attention backend",
// kernel contract: "Q/K are quantized per 32-row block").  scale = amax/127,
// code = clamp(rint(x/scale), -127, 127) with correctly rounded fp32
// divisions, so the codes are bit-identical to a plain CPU statement.
//
// V: FP8 E4M3 per channel of one (batch, head) over all tokens (same passage:
// "V per channel"; diffusers PR #15060 "Add aiter_sage_hub attention backend",
// "What does this PR do?": FP8 PV).  sv = amax/448, code = e4m3_rn_sat(v/sv).
// V is written transposed, [B, H, 128, S_pad], so that the attention kernel's
// PV operand is K-major.
//
// This file is compiled without fast-math and without flush-to-zero: the
// divisions are IEEE round-to-nearest-even (div.rn.f32).
#include <algorithm>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "sage_internal.cuh"
#include "qk_codes.cuh"
#include "sm103_ptx.cuh"

namespace sage {

namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// a * b + c elementwise on the packed FP32 pipe, one rounding per lane.
__device__ __forceinline__ float2 ffma2v(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmov.b64 z, {%6, %7};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

template <typename CodeT>
struct CodeStore;

template <>
struct CodeStore<int8_t> {
  // 8 integer-valued floats -> 8 bytes (two's complement)
  __device__ static void store(int8_t* dst, const float (&c)[8]) {
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = (__float_as_uint(c[i] + kRoundMagic) - 0x4B400000u) & 0xFFu;
    const uint32_t lo = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
    const uint32_t hi = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
  }
};

template <>
struct CodeStore<__half> {
  // 8 integer-valued floats -> 8 halves (exact for |c| <= 127)
  __device__ static void store(__half* dst, const float (&c)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h2 = __floats2half2_rn(c[2 * i], c[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// One warp per (tensor, batch*head, 32-token block), eight blocks per CTA of
// 256 threads.  Lanes 0-15 own the even tokens of the block, lanes 16-31 the
// odd ones, lane%16 owns channels 8*(lane%16) .. +7: a load or store
// instruction of the warp covers two whole 256-byte token rows.  A lane loads
// all its 16 tokens before anything else (256 bytes in flight), and the block
// max is a warp shuffle: no shared memory, no block-wide barrier.  `tensor`
// selects Q (0) or K (1).
template <typename CodeT, bool kSmooth>
__device__ __forceinline__ void qk_warp(const QKQuantArgs<CodeT>& a, int tensor) {
  const uint16_t* __restrict__ x = tensor == 0 ? a.q : a.k;
  CodeT* __restrict__ codes = tensor == 0 ? a.q_codes : a.k_codes;
  float* __restrict__ scale = tensor == 0 ? a.q_scale : a.k_scale;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S[tensor], S_pad = a.S_pad[tensor], nb = a.nb[tensor];
  const int nbp = S_pad / 32;
  const long long gblk = static_cast<long long>(blockIdx.x) * 8 + warp;
  if (gblk >= static_cast<long long>(a.BH) * nbp) return;   // warp-uniform; no block-wide sync below
  const int blk = static_cast<int>(gblk % nbp);
  const int bh = static_cast<int>(gblk / nbp);
  const int b = bh / a.H, h = bh % a.H;
  const int half = lane >> 4;
  const int c8 = (lane & 15) * 8;
  // K smoothing: subtract the channel means before quantising.
  float mu[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const bool smooth = kSmooth && tensor == 1;
  if (smooth) {
    const float4* m4 = reinterpret_cast<const float4*>(a.k_mean + static_cast<size_t>(bh) * kHeadDim + c8);
    const float4 m0 = m4[0], m1 = m4[1];
    mu[0] = m0.x; mu[1] = m0.y; mu[2] = m0.z; mu[3] = m0.w;
    mu[4] = m1.x; mu[5] = m1.y; mu[6] = m1.z; mu[7] = m1.w;
  }
  const int tok0 = blk * 32 + half;   // this lane's tokens: tok0 + 2*it, it = 0..15
  const size_t tok_stride = static_cast<size_t>(a.H) * kHeadDim;
  const uint16_t* src = x + (static_cast<size_t>(b) * S * a.H + h) * kHeadDim + c8;

  uint4 raw[16];
#pragma unroll
  for (int it = 0; it < 16; ++it) {
    const int s = tok0 + 2 * it;
    raw[it] = s < S ? __ldcs(reinterpret_cast<const uint4*>(src + static_cast<size_t>(s) * tok_stride))
                    : make_uint4(0, 0, 0, 0);
  }
  float amax = 0.0f;
#pragma unroll
  for (int it = 0; it < 16; ++it) {
    const uint32_t w[4] = {raw[it].x, raw[it].y, raw[it].z, raw[it].w};
    if (smooth) {
      if (tok0 + 2 * it < S) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          amax = fmax3(amax, fabsf(bf16_lo(w[i]) - mu[2 * i]), fabsf(bf16_hi(w[i]) - mu[2 * i + 1]));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) amax = fmax3(amax, fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i])));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  const float sc = __fdiv_rn(amax, 127.0f);
  const float rcp = __frcp_rn(sc);
  const bool fast_sc = sc >= 0x1p-125f && sc <= 0x1p125f;
  if (lane == 0 && blk < nb) scale[static_cast<size_t>(bh) * nb + blk] = sc;

  CodeT* dst = codes + (static_cast<size_t>(bh) * S_pad + tok0) * kHeadDim + c8;
#pragma unroll
  for (int it = 0; it < 16; ++it) {
    const uint32_t w[4] = {raw[it].x, raw[it].y, raw[it].z, raw[it].w};
    float xs[8], c[8];
    const bool valid = tok0 + 2 * it < S;   // rows past the end stay 0 (no -mean)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xs[2 * i] = smooth && valid ? bf16_lo(w[i]) - mu[2 * i] : bf16_lo(w[i]);
      xs[2 * i + 1] = smooth && valid ? bf16_hi(w[i]) - mu[2 * i + 1] : bf16_hi(w[i]);
    }
    codes8(xs, sc, rcp, fast_sc, c);
    CodeStore<CodeT>::store(dst + static_cast<size_t>(2 * it) * kHeadDim, c);
  }
}

// Per-channel |v| maxima of one 256-token slice of one (batch, head), by a
// whole CTA of 256 threads: thread t owns channels 8*(t%16) .. +7 of every
// 16th token.  Results are merged with atomicMax on the fp32 bit patterns
// (order-preserving for non-negative values) into amax_bits [B*H, 128], which
// must start at 0.
constexpr int kVRowsPerCta = 256;

// Grids over (x blocks per head, heads): the head index spans y and z, y
// below 65535 (the y and z limit), so B*H up to 2^31 - 1 fits; x runs
// fastest, so a head's blocks are adjacent in launch order.
constexpr unsigned kGridYMax = 65535;

// Zeroes n words (the channel maxima the first pass merges with atomicMax).
// Its dependent, the first pass, may start at once: only that pass's V
// maxima role waits for this grid before touching these words.
__global__ void __launch_bounds__(256) zero_words_kernel(uint32_t* __restrict__ p, size_t n) {
  asm volatile("griddepcontrol.launch_dependents;");
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0u;
}

// Launch `kernel` as a programmatic dependent of the grid before it on
// `stream` (programmatic stream serialisation): it may be scheduled once
// every CTA of that grid has triggered or finished, and must itself wait
// (griddepcontrol.wait) before reading anything that grid writes.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, cudaStream_t stream,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}
inline dim3 heads_grid(int x, int heads) {
  const unsigned y = static_cast<unsigned>(heads < static_cast<int>(kGridYMax) ? heads : static_cast<int>(kGridYMax));
  const unsigned z = (static_cast<unsigned>(heads) + kGridYMax - 1) / kGridYMax;
  return dim3(static_cast<unsigned>(x), y, z);
}

__device__ __forceinline__ void v_amax_slice(const uint16_t* __restrict__ v, int S, int H,
                                             uint32_t* __restrict__ amax_bits, int bh, int slice) {
  __shared__ float part[16][kHeadDim];
  const int b = bh / H, h = bh % H;
  const int t = threadIdx.x, c8 = (t & 15) * 8, r = t >> 4;
  const int s0 = slice * kVRowsPerCta;
  const int s1 = min(S, s0 + kVRowsPerCta);
  const size_t tok_stride = static_cast<size_t>(H) * kHeadDim;
  const uint16_t* src = v + (static_cast<size_t>(b) * S * H + h) * kHeadDim + c8;
  float m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  uint4 raw[kVRowsPerCta / 16];            // all of this thread's (at most 16) tokens in flight at once
#pragma unroll
  for (int k = 0; k < kVRowsPerCta / 16; ++k) {
    const int s = s0 + r + 16 * k;
    raw[k] = s < s1 ? __ldcs(reinterpret_cast<const uint4*>(src + static_cast<size_t>(s) * tok_stride))
                    : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int k = 0; k < kVRowsPerCta / 16; ++k) {
    const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m[2 * i] = fmaxf(m[2 * i], fabsf(bf16_lo(w[i])));
      m[2 * i + 1] = fmaxf(m[2 * i + 1], fabsf(bf16_hi(w[i])));
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) part[r][c8 + i] = m[i];
  __syncthreads();
  if (t < kHeadDim) {
    // The words were zeroed by the grid before this one, which this grid may
    // have started ahead of.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float mm = part[0][t];
#pragma unroll
    for (int i = 1; i < 16; ++i) mm = fmaxf(mm, part[i][t]);
    atomicMax(amax_bits + static_cast<size_t>(bh) * kHeadDim + t, __float_as_uint(mm));
  }
}

// First quantisation pass, one launch: Q and K codes (grid.y role 0 and 1,
// qk_warp) and the per-channel V maxima (role 2, one CTA per 256-token slice
// of one (batch, head)).  The roles are CTA-uniform.
struct VMaxArgs {
  const uint16_t* v;      // bf16 [B, S, H, 128]; nullptr: no V maxima
  uint32_t* amax_bits;    // [B*H, 128], zeroed before the launch
  int S, H, BH, nslices;  // nslices = ceil(S / kVRowsPerCta)
};

template <typename CodeT, bool kSmooth>
__global__ void __launch_bounds__(256, 2) qkv_pass1_kernel(QKQuantArgs<CodeT> a, VMaxArgs vm) {
  // The V^T encoder launched after this grid may be scheduled once every CTA
  // here has started (it waits for this grid's completion before reading the
  // channel maxima), so its V loads overlap this grid's last wave.
  asm volatile("griddepcontrol.launch_dependents;");
  const int role = blockIdx.y + a.first;
  if (role == 2) {
    const long long idx = blockIdx.x;
    if (idx >= static_cast<long long>(vm.BH) * vm.nslices) return;   // CTA-uniform
    v_amax_slice(vm.v, vm.S, vm.H, vm.amax_bits, static_cast<int>(idx / vm.nslices),
                 static_cast<int>(idx % vm.nslices));
    return;
  }
  qk_warp<CodeT, kSmooth>(a, role);
}

// A bf16 value times 2^40 as a 64-bit integer: exact for |x| in [2^-33, 2^22)
// (8 significant bits, the lowest at or above 2^-40) and for 0; smaller
// magnitudes are truncated, larger ones saturate.  A channel's sum stays
// exact while its magnitude is below 2^23, and converts to double exactly
// below 2^13 (bf16 activations of a few units sum far below that).
__device__ __forceinline__ long long bf16_fixed40(uint32_t h) {
  const uint32_t e = (h >> 7) & 0xFFu;
  const long long m = static_cast<long long>((h & 0x7Fu) | (e ? 0x80u : 0u));
  const int sh = static_cast<int>(e ? e : 1u) - 127 - 7 + 40;
  long long v = sh >= 0 ? (sh < 55 ? (m << sh) : (255LL << 54)) : (sh > -8 ? (m >> -sh) : 0LL);
  return (h & 0x8000u) ? -v : v;
}

// Per-channel sums of K over one 256-token slice of one (batch, head), in
// 64-bit fixed point (2^-40): integer additions, so the merged result does not
// depend on the order of the slices, and it equals the exact sum for the
// magnitudes bf16_fixed40 keeps exactly.
//
// A thread first adds its 16 tokens of 8 channels in fp32 and keeps a
// channel's sum only where it is provably exact in that grid: every value
// zero or in [2^-33, 2^22) (so a whole number of 2^-40 units, as
// bf16_fixed40 counts it), every addition exact (the TwoSum rounding error
// (a - (s - b')) + (x - b') with b' = s - a is zero) and the partial sum
// below 2^23 (so times 2^40 it is an int64).  Then sum * 2^40 is the integer
// bf16_fixed40 would have accumulated; a channel that fails redoes its 16
// values with bf16_fixed40.
__global__ void __launch_bounds__(256) k_sum_kernel(const uint16_t* __restrict__ k, int S, int H, int BH,
                                                    unsigned long long* __restrict__ sums) {
  __shared__ long long part[16][kHeadDim];
  // grid (slices, heads): the head index spans y and z (y < 65535).
  const int bh = static_cast<int>(blockIdx.z * kGridYMax + blockIdx.y);
  if (bh >= BH) return;                    // CTA-uniform, before any barrier
  const int b = bh / H, h = bh % H;
  const int t = threadIdx.x, c8 = (t & 15) * 8, r = t >> 4;
  const int s0 = static_cast<int>(blockIdx.x) * kVRowsPerCta;
  const int s1 = min(S, s0 + kVRowsPerCta);
  const size_t tok_stride = static_cast<size_t>(H) * kHeadDim;
  const uint16_t* src = k + (static_cast<size_t>(b) * S * H + h) * kHeadDim + c8;
  uint4 buf[kVRowsPerCta / 16];   // all of this thread's tokens in flight (zeros past the slice)
#pragma unroll
  for (int u = 0; u < kVRowsPerCta / 16; ++u) {
    const int s = s0 + r + 16 * u;
    buf[u] = s < s1 ? __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(s) * tok_stride))
                    : make_uint4(0u, 0u, 0u, 0u);
  }
  float f[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  uint32_t inexact = 0;   // bit i: channel c8 + i takes the fixed-point path
#pragma unroll
  for (int u = 0; u < kVRowsPerCta / 16; ++u) {
    const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x = __uint_as_float((i & 1) ? (w[i >> 1] & 0xFFFF0000u) : (w[i >> 1] << 16));
      const float ax = fabsf(x);
      const float a = f[i], sum = a + x, bp = sum - a;
      const bool ok = (((ax >= 0x1p-33f) & (ax < 0x1p22f)) | (ax == 0.0f)) & ((a - (sum - bp)) + (x - bp) == 0.0f);
      inexact |= ok ? 0u : (1u << i);
      f[i] = sum;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (!(fabsf(f[i]) < 0x1p23f)) inexact |= 1u << i;
    part[r][c8 + i] = __float2ll_rz(f[i] * 0x1p40f);
  }
  // The channels whose fp32 sum is not provably exact, again in fixed point.
#pragma unroll 1
  for (int i = 0; i < 8; ++i) {
    if (!(inexact & (1u << i))) continue;
    long long acc = 0;
    for (int s = s0 + r; s < s1; s += 16) acc += bf16_fixed40(src[static_cast<size_t>(s) * tok_stride + i]);
    part[r][c8 + i] = acc;
  }
  __syncthreads();
  if (t < kHeadDim) {
    long long mm = part[0][t];
#pragma unroll
    for (int i = 1; i < 16; ++i) mm += part[i][t];
    atomicAdd(sums + static_cast<size_t>(bh) * kHeadDim + t, static_cast<unsigned long long>(mm));
  }
}

// mean = fp32(sum / S) per (batch, head, channel): the fixed-point sum is
// converted to double (exact below 2^53 units of 2^-40) and divided once.
__global__ void k_mean_kernel(const unsigned long long* __restrict__ sums, int S, int n, float* __restrict__ mean) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const double sum = static_cast<double>(static_cast<long long>(sums[i])) * 0x1p-40;
    mean[i] = static_cast<float>(sum / static_cast<double>(S));
  }
}

// E4M3 code of fl(x / sv) by the division itself (0 for sv = 0, where every
// value of the channel is zero): the path for a scale outside [2^-100, 2^125].
__device__ __forceinline__ uint8_t e4m3_code_div(float x, float sv) {
  return static_cast<uint8_t>(cvt_e4m3x2(sv == 0.0f ? 0.0f : __fdiv_rn(x, sv), 0.0f));
}

// Encode one 128-token tile of one (batch, head) and write it transposed.
// grid = (S_pad / 128, heads) through heads_grid, 256 threads.
//   Load: warp w covers tile tokens 16w .. 16w+15; in load instruction i
//   (0..7) lanes 0-15 read token 16w + i and lanes 16-31 token 16w + 8 + i,
//   lane l channels 8(l%16) .. +7 (16 bytes): two whole 256-byte rows per
//   instruction.  A lane so holds 8 consecutive tokens (token group tg =
//   2w + l/16: tile tokens 8tg .. 8tg+7) of 8 channels.  Meanwhile threads
//   0-127 form the 128 channel scales sv = fl(amax / 448) and nr =
//   -fl(1/sv) once, in shared memory.
//   Codes: the quotient's correction step of Markstein (IBM J. Res. Dev.
//   34(1), 1990: a faithful quotient, its exact residual by one FMA and a
//   second FMA with the correctly rounded reciprocal give the correctly
//   rounded quotient), with the reciprocal negated:
//     z = fl(x nr),  r = fma(z, sv, x),  y = fma(r, nr, z)  =  -fl(x / sv),
//   zeros included (y = -0 for x = +0 and +0 for x = -0), and the E4M3 code
//   of fl(x / sv) is the code of y with its sign bit flipped.  This holds
//   for every bf16 x with |x| <= amax and every bf16 amax whose scale lies
//   in [2^-100, 2^125] (every such pair has been checked against the
//   division); a channel outside that range (an all-zero channel, or one
//   whose values are all below ~2^-91) is re-encoded by the division after
//   the tile is written.  Three packed FP32 operations and one paired
//   conversion per two values, no compare and no branch.
//   Transpose: each lane's 8 tokens x 8 channels of E4M3 codes are
//   transposed in registers and stored, 8 bytes per channel, into a 128 x
//   128-byte tile (channel rows); the 8-byte chunk of token group tg in
//   channel row c sits at chunk tg ^ ((c / 8) % 16 & ~1), so that the 32
//   stores of an instruction fall into distinct bank pairs twice (two
//   wavefronts) and token groups 2m, 2m+1 stay one ordered 16-byte piece.
//   Store: 8 lanes write one channel row's 128 contiguous bytes of V^T.
// Tokens >= S get code 0.
constexpr int kVEncThreads = 256;

__global__ void __launch_bounds__(kVEncThreads, 4) v_encode_kernel(const uint16_t* __restrict__ v, int S, int H,
                                                                   int BH, int S_pad,
                                                                   const uint32_t* __restrict__ amax_bits,
                                                                   uint8_t* __restrict__ vt,
                                                                   float* __restrict__ v_scale) {
  __shared__ __align__(16) uint8_t tile[kHeadDim * 128];
  __shared__ __align__(16) float s_sv[kHeadDim];
  __shared__ __align__(16) float s_nr[kHeadDim];
  __shared__ __align__(16) int s_out[kHeadDim];   // scale outside [2^-100, 2^125]
  // grid (tiles, heads): the head index spans y and z (y < 65535).
  const int bh = static_cast<int>(blockIdx.z * kGridYMax + blockIdx.y);
  if (bh >= BH) return;                    // CTA-uniform, before any barrier
  const int b = bh / H, h = bh % H;
  const int tile_idx = static_cast<int>(blockIdx.x);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane & 15;                 // channels 8g .. 8g+7
  const int tg = 2 * warp + (lane >> 4);   // token group: tile tokens 8tg .. 8tg+7
  const int s0 = tile_idx * 128 + 8 * tg;
  const size_t tok_stride = static_cast<size_t>(H) * kHeadDim;
  const uint16_t* src = v + (static_cast<size_t>(b) * S * H + h) * kHeadDim + 8 * g + static_cast<size_t>(s0) * tok_stride;
  uint4 raw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    raw[i] = s0 + i < S ? __ldcs(reinterpret_cast<const uint4*>(src + i * tok_stride)) : make_uint4(0, 0, 0, 0);
  if (threadIdx.x < kHeadDim) {
    const int c = threadIdx.x;
    // The channel maxima come from the preceding grid: wait for its
    // completion (a no-op when this grid was not launched as its dependent).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float sv = __fdiv_rn(__uint_as_float(amax_bits[static_cast<size_t>(bh) * kHeadDim + c]), 448.0f);
    s_sv[c] = sv;
    s_nr[c] = -__frcp_rn(sv);
    s_out[c] = !(sv >= 0x1p-100f && sv <= 0x1p125f);
    if (tile_idx == 0) v_scale[static_cast<size_t>(bh) * kHeadDim + c] = sv;
  }
  __syncthreads();
  float sv[8], nr[8];
  uint32_t out_of_range = 0;               // bit c: channel 8g + c takes the division
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    sv[c] = s_sv[8 * g + c];
    nr[c] = s_nr[8 * g + c];
    out_of_range |= static_cast<uint32_t>(s_out[8 * g + c] != 0) << c;
  }
  // tw[i][k]: token i's codes of channels 8g+4k .. +3 (channel in byte order)
  uint32_t tw[8][2];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 x0 = make_float2(bf16_lo(w[2 * k]), bf16_hi(w[2 * k]));
      const float2 x1 = make_float2(bf16_lo(w[2 * k + 1]), bf16_hi(w[2 * k + 1]));
      const float2 n0 = make_float2(nr[4 * k], nr[4 * k + 1]), n1 = make_float2(nr[4 * k + 2], nr[4 * k + 3]);
      const float2 z0 = fmul2v(x0, n0), z1 = fmul2v(x1, n1);
      const float2 r0 = ffma2v(z0, make_float2(sv[4 * k], sv[4 * k + 1]), x0);
      const float2 r1 = ffma2v(z1, make_float2(sv[4 * k + 2], sv[4 * k + 3]), x1);
      const float2 y0 = ffma2v(r0, n0, z0), y1 = ffma2v(r1, n1, z1);
      tw[i][k] = cvt_e4m3x4(y0.x, y0.y, y1.x, y1.y) ^ 0x80808080u;
    }
  }
  // 4x4 byte transposes: cw[c][p] = tokens 4p .. 4p+3 of channel 8g + c.
  uint32_t cw[8][2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      const uint32_t w0 = tw[4 * pp][k], w1 = tw[4 * pp + 1][k], w2 = tw[4 * pp + 2][k], w3 = tw[4 * pp + 3][k];
      const uint32_t a01 = __byte_perm(w0, w1, 0x5140), b01 = __byte_perm(w0, w1, 0x7362);
      const uint32_t a23 = __byte_perm(w2, w3, 0x5140), b23 = __byte_perm(w2, w3, 0x7362);
      cw[4 * k + 0][pp] = __byte_perm(a01, a23, 0x5410);
      cw[4 * k + 1][pp] = __byte_perm(a01, a23, 0x7632);
      cw[4 * k + 2][pp] = __byte_perm(b01, b23, 0x5410);
      cw[4 * k + 3][pp] = __byte_perm(b01, b23, 0x7632);
    }
  }
  uint8_t* my_chunk = tile + 8 * g * 128 + ((tg ^ (g & 14)) << 3);   // channel row 8g; + c * 128 for row 8g + c
#pragma unroll
  for (int c = 0; c < 8; ++c)   // channel row 8g + c, swizzle (8g + c) / 8 % 16 & ~1 = g & 14
    *reinterpret_cast<uint2*>(my_chunk + c * 128) = make_uint2(cw[c][0], cw[c][1]);
  if (__builtin_expect(out_of_range != 0u, 0)) {
    // Re-encode this lane's out-of-range channels by the division: it reads
    // its tokens again and overwrites its own bytes of the tile.
    for (int i = 0; i < 8; ++i) {
      const uint4 r = s0 + i < S ? *reinterpret_cast<const uint4*>(src + i * tok_stride) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if ((out_of_range >> c) & 1u)
          my_chunk[c * 128 + i] = e4m3_code_div((c & 1) ? bf16_hi(w[c >> 1]) : bf16_lo(w[c >> 1]), sv[c]);
    }
  }
  __syncthreads();
  const int m = threadIdx.x & 7;           // 16-byte piece m of a row: token groups 2m, 2m+1
#pragma unroll
  for (int it = 0; it < kHeadDim / (kVEncThreads / 8); ++it) {
    const int c = it * (kVEncThreads / 8) + (threadIdx.x >> 3);
    const int gc = (c >> 3) & 15;
    const uint4 x = *reinterpret_cast<const uint4*>(tile + c * 128 + ((m ^ (gc >> 1)) << 4));
    *reinterpret_cast<uint4*>(vt + (static_cast<size_t>(bh) * kHeadDim + c) * S_pad + tile_idx * 128 + 16 * m) = x;
  }
}

// int8 codes -> integer-valued fp16 codes, 16 per thread.
__global__ void __launch_bounds__(256) widen_codes_kernel(const int8_t* __restrict__ src,
                                                          __half* __restrict__ dst, size_t n16) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const int4 q = __ldcs(reinterpret_cast<const int4*>(src) + i);
  const int w[4] = {q.x, q.y, q.z, q.w};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int lo = static_cast<int8_t>((w[k] >> (16 * j)) & 0xFF);
      const int hi = static_cast<int8_t>((w[k] >> (16 * j + 8)) & 0xFF);
      __half2 h2 = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
      o[2 * k + j] = *reinterpret_cast<uint32_t*>(&h2);
    }
  }
  uint4* d = reinterpret_cast<uint4*>(dst) + 2 * i;
  d[0] = make_uint4(o[0], o[1], o[2], o[3]);
  d[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace

template <typename CodeT>
cudaError_t launch_qkv_quantize(const QKQuantArgs<CodeT>& a, const uint16_t* v, uint32_t* amax_bits, uint8_t* vt,
                                float* v_scale, cudaStream_t stream) {
  VMaxArgs vm;
  vm.v = v;
  vm.amax_bits = amax_bits;
  vm.S = a.S[1];
  vm.H = a.H;
  vm.BH = a.BH;
  vm.nslices = (a.S[1] + kVRowsPerCta - 1) / kVRowsPerCta;
  if (v != nullptr) {
    const size_t n = static_cast<size_t>(a.BH) * kHeadDim;
    zero_words_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(amax_bits, n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const long long blocks = static_cast<long long>(a.BH) * (std::max(a.first ? 0 : a.S_pad[0], a.S_pad[1]) / 32);
  long long ctas = (blocks + 7) / 8;
  if (v != nullptr) ctas = std::max(ctas, static_cast<long long>(a.BH) * vm.nslices);
  if (ctas > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(ctas), (v != nullptr ? 3 : 2) - a.first);
  // With V, the first pass is a programmatic dependent of the zeroing kernel
  // just launched (its Q/K roles never read what that kernel writes);
  // without V nothing precedes it that it may overlap.
  cudaError_t e;
  if (v != nullptr) {
    e = a.k_mean != nullptr ? launch_dependent(qkv_pass1_kernel<CodeT, true>, grid, dim3(256), stream, a, vm)
                            : launch_dependent(qkv_pass1_kernel<CodeT, false>, grid, dim3(256), stream, a, vm);
  } else {
    if (a.k_mean != nullptr)
      qkv_pass1_kernel<CodeT, true><<<grid, 256, 0, stream>>>(a, vm);
    else
      qkv_pass1_kernel<CodeT, false><<<grid, 256, 0, stream>>>(a, vm);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || v == nullptr) return e;
  const int S_pad = a.S_pad[1];
  // A programmatic dependent of the first pass (see the kernels).
  return launch_dependent(v_encode_kernel, heads_grid(S_pad / 128, a.BH), dim3(kVEncThreads), stream, v, a.S[1],
                          a.H, a.BH, S_pad, static_cast<const uint32_t*>(amax_bits), vt, v_scale);
}

// Every kernel a quantise-then-attend call launches, K smoothing included.
cudaError_t load_quantize_kernels() {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, zero_words_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, qkv_pass1_kernel<__half, false>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, qkv_pass1_kernel<__half, true>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, v_encode_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k_sum_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k_mean_kernel);
  return e;
}

template cudaError_t launch_qkv_quantize<int8_t>(const QKQuantArgs<int8_t>&, const uint16_t*, uint32_t*, uint8_t*,
                                                 float*, cudaStream_t);
template cudaError_t launch_qkv_quantize<__half>(const QKQuantArgs<__half>&, const uint16_t*, uint32_t*, uint8_t*,
                                                 float*, cudaStream_t);

cudaError_t launch_k_channel_means(const uint16_t* k, int B, int S, int H, unsigned long long* sums, float* mean,
                                   cudaStream_t stream) {
  const int BH = B * H;
  cudaError_t e = cudaMemsetAsync(sums, 0, static_cast<size_t>(BH) * kHeadDim * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  k_sum_kernel<<<heads_grid((S + kVRowsPerCta - 1) / kVRowsPerCta, BH), 256, 0, stream>>>(k, S, H, BH, sums);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n = BH * kHeadDim;
  k_mean_kernel<<<(n + 255) / 256, 256, 0, stream>>>(sums, S, n, mean);
  return cudaGetLastError();
}

cudaError_t launch_widen_codes(const int8_t* src, __half* dst, size_t n, cudaStream_t stream) {
  const size_t n16 = n / 16;
  widen_codes_kernel<<<static_cast<unsigned>((n16 + 255) / 256), 256, 0, stream>>>(src, dst, n16);
  return cudaGetLastError();
}

}  // namespace sage
