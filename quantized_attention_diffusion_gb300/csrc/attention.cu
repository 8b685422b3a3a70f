// attention.cu -- fused SageAttention-style forward for sm_103a.
//
// What it computes (diffusers issue #15014 "gfx1201 (RDNA4) SageAttention
// attention backend", kernel contract: INT8 QK^T and FP8 PV with FP32
// accumulation, Q/K quantized per 32-row block and V per channel inside the
// kernel, BF16 [B, S, H, 128], no mask, non-causal; diffusers PR #15060,
// "What does this PR do?": no LSE).  Per query row, over KV tiles of 96 keys:
//
//   acc_j  = sum_c q[c] k_j[c]                     exact (|acc| < 2^24)
//   x_j    = acc_j * cb_j,  cb_j = (sq * softmax_scale * log2 e) * sk_{j/32}
//   m_t    = max(m_{t-1}, max_{j in tile t} x_j)   running max (base 2)
//   p~_j   = e4m3(2^(acc_j * cb_j - (m_t - log2 448)))   P in FP8, <= 448
//   L, O  <- 2^(m_{t-1} - m_t) * (L, O) + (sum p~_j, sum p~_j v~_j)
//   out    = bf16(O * sv / L)
//
// GB300 mapping.  sm_103a has no INT8 tcgen05 MMA, so QK^T runs as
// tcgen05 kind::f16 on fp16 copies of the INT8 codes: every code, product
// and partial sum is an integer below 2^24, so the FP32 accumulator holds the
// exact INT32 result.  PV runs as kind::f8f6f4 (E4M3 x E4M3 -> FP32) with
// N = 144: V^T's 128 channel rows plus 16 rows of E4M3 ones, so the same MMA
// accumulates L = sum p~ (rescaled with O) in accumulator column 128.
//
// One CTA owns two 128-row Q tiles of one (batch, head) and streams every KV
// tile of that head.  384 threads:
//   warp 0       TMA producer of Q (once) and K (3-stage ring)
//   warp 1       TMEM allocator; issues the QK^T MMAs (one thread)
//   warp 2       issues the PV MMAs (one thread)
//   warp 3       TMA producer of V^T (4-stage ring, 32-byte swizzle)
//   warps 2-3    first write the ones rows of the V stages
//   warps 4-7    softmax + epilogue of Q tile 0, one thread per query row
//   warps 8-11   the same for Q tile 1
// TMEM (512 columns allocated): S0 [0,96)  S1 [96,192)  O0 [192,336)
// O1 [336,480).  KV tiles are 96 keys so that two S tiles and two N=144
// accumulators fit; 96 keys are exactly three K quantisation blocks and
// three K=32 steps of the PV MMA.
//
// P~ goes to shared memory (one 128-row, 128-byte-pitch tile per Q tile, in
// the swizzled layout the MMA descriptors read), not over S.  A softmax
// thread hands its S columns back as soon as it has loaded them, so QK(j+1)
// of a tile runs while the softmax of tile j is still computing, and the two
// issuing threads keep QK and PV apart: QK runs ahead as far as S is free,
// PV follows P~.  Before writing P~(j) or rescaling O, a softmax thread waits
// for PV(j-1) of its tile.
//
// An M=128 MMA from one thread takes about 48-72 SM clocks here, barely more
// than one thread needs to issue it, so the issue loops are kept short:
// descriptors are formed from precomputed lower words, and barrier waits
// inline only their first poll.
#include <cmath>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qk_codes.cuh"
#include "sage_internal.cuh"
#include "sm103_ptx.cuh"

namespace sage {

__device__ int g_sage_error;   // SAGE_DEVERR_* of the last failed wait on this device

namespace {

constexpr int kKV = 96;                                   // keys per KV tile
constexpr int kStages = 3;
constexpr int kThreads = 384;
constexpr uint32_t kQHalf = 128 * 64 * 2;                // 128 rows x 64 fp16
constexpr uint32_t kQTileBytes = 2 * kQHalf;
constexpr uint32_t kKHalf = kKV * 64 * 2;                // 96 rows x 64 fp16
constexpr uint32_t kKTileBytes = 2 * kKHalf;
constexpr int kVStages = 4;                               // V^T ring depth (K ring: kStages)
// A V^T stage holds one KV tile as three 32-key sub-tiles (one per K=32 step
// of the PV MMA), each 144 rows x 32 bytes with 32-byte swizzle: V^T's 128
// channel rows, then 16 rows of E4M3 ones.  Only the 96 keys of the tile
// are loaded, which is what makes room for four stages.
constexpr uint32_t kVSubBytes = 144 * 32;
constexpr uint32_t kVOnesOffset = 128 * 32;              // ones rows within a sub-tile
constexpr uint32_t kVStageBytes = 3 * kVSubBytes;
constexpr uint32_t kVLoadBytes = 3 * 128 * 32;           // bytes TMA writes per stage
constexpr uint32_t kPTileBytes = 128 * 128;              // P~: 128 rows x 128 bytes (96 used)
constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemK = kSmemQ + 2 * kQTileBytes;
constexpr uint32_t kSmemV = kSmemK + kStages * kKTileBytes;
constexpr uint32_t kSmemP = kSmemV + kVStages * kVStageBytes;
constexpr uint32_t kSmemTiles = kSmemP + 2 * kPTileBytes;
constexpr uint32_t kSmemDynamic = kSmemTiles + 1024;     // slack for 1024-byte alignment
// TMEM columns of tile t's scores (96) and accumulator (144; L at +128).
__host__ __device__ constexpr uint32_t col_s(int t) { return static_cast<uint32_t>(t) * kKV; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 2 * kKV + static_cast<uint32_t>(t) * 144; }
constexpr float kLog2P = 8.80735492706298828125f;         // fp32(log2 448): P scale 448
constexpr float kLog2e = 1.44269502162933349609375f;      // fp32(log2 e)
constexpr float kLn2 = 0.693147182464599609375f;          // fp32(ln 2)
constexpr uint32_t kE4M3One = 0x38383838u;                // four E4M3 1.0

static_assert(kSmemDynamic <= 227 * 1024 - 1024, "shared memory budget");
static_assert(kSmemQ % 1024 == 0 && kSmemK % 1024 == 0 && kSmemP % 1024 == 0 && kKTileBytes % 1024 == 0 &&
                  kQHalf % 1024 == 0 && kKHalf % 1024 == 0 && kPTileBytes % 1024 == 0,
              "128-byte swizzle atoms are 1024-byte aligned");
static_assert(kSmemV % 256 == 0 && kVSubBytes % 256 == 0, "32-byte swizzle atoms are 256-byte aligned");

struct Params {
  int fuse_q;             // 1: Q arrives as bf16 and is quantised here (q_scale unused)
  int8_t* q_dump;         // optional with fuse_q: the Q codes, int8 [B, H, Sq_pad, 128]
  float* q_scale_dump;    // optional with fuse_q: the Q block scales [B, H, nbq]
  int Sq_pad;
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  uint16_t* out;
  int32_t* s_dump;
  float* lse;             // optional [B, H, S]
  int Sq, Skv, H, nbq, nbk, n_kv, n_pairs;   // query rows, key/value rows (equal unless cross)
  float c_scale;          // fp32(softmax_scale * fp32(log2 e))
  uint64_t timeout_ns;
};

struct Barriers {
  uint64_t q_full, q_ready;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], o_full[2];
  uint64_t drain_qk, drain_pv;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint64_t timeout_ns) {
  return mbar_wait(bar, parity, abort_flag, &g_sage_error, timeout_ns);
}

// Bounded wait that ignores the abort flag: used to let in-flight copies and
// MMAs land before the CTA releases its shared memory and TMEM.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  int local_abort = 0;
  (void)mbar_wait(bar, parity, &local_abort, &g_sage_error, timeout_ns);
}

// Sixteen floats -> sixteen bf16 (round to nearest even) in one 32-byte
// store; dst must be 32-byte aligned.
__device__ __forceinline__ void store_bf16x16(uint16_t* dst, const float (&v)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// One row's 96 integer scores -> 96 E4M3 probabilities p~ = e4m3(2^(acc *
// cb[block] - bias)), four codes per word, key k in byte k%4 of word k/4.
__device__ __forceinline__ void softmax_p(const float (&a)[kKV], const float (&cb)[3], float bias,
                                          uint32_t (&pk)[kKV / 4]) {
#pragma unroll
  for (int blk = 0; blk < 3; ++blk) {
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int c = blk * 32 + w * 4;
      const float2 x01 = ffma2_bc(a[c], a[c + 1], cb[blk], -bias);
      const float2 x23 = ffma2_bc(a[c + 2], a[c + 3], cb[blk], -bias);
      const float p0 = ex2_approx(x01.x), p1 = ex2_approx(x01.y);
      const float p2 = ex2_approx(x23.x), p3 = ex2_approx(x23.y);
      pk[blk * 8 + w] = cvt_e4m3x4(p0, p1, p2, p3);
    }
  }
}

// 32 TMEM columns (as loaded) times alpha, on the packed FP32 pipe.
__device__ __forceinline__ void scale_cols(uint32_t (&o)[32], float alpha) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 r = fmul2(__uint_as_float(o[i]), __uint_as_float(o[i + 1]), alpha);
    o[i] = __float_as_uint(r.x);
    o[i + 1] = __float_as_uint(r.y);
  }
}

// Row r of a P~ tile in the 128-byte-swizzled K-major layout: 16-byte chunk
// c of row r sits at (r/8)*1024 + (r%8)*128 + (c ^ (r%8))*16.  Chunks 0-5
// hold the 96 codes.
__device__ __forceinline__ void store_p_row(uint8_t* tile, int r, const uint32_t (&pk)[kKV / 4]) {
  uint8_t* base = tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
  for (int c = 0; c < kKV / 16; ++c)
    *reinterpret_cast<uint4*>(base + ((c ^ (r & 7)) << 4)) =
        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
}

// One lane per row: quantise row r (0..127) of a bf16 Q tile in shared
// memory (two 64-column halves, 128-byte swizzled rows) in place to
// integer-valued fp16 codes.  The 32 lanes of the warp are one 32-row block:
// scale = amax / 127 over the block (fp32 RNE division).  Two passes over
// the row (max, then codes) keep few registers live.  Returns the scale.
__device__ __forceinline__ float quantize_q_rows(uint8_t* tile, int r, int bh, int tile_row0, int8_t* q_dump,
                                                 float* q_scale_dump, int Sq_pad, int nbq) {
  const uint32_t roff = static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128);
  float amax = 0.0f;
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int hf = i >> 3, c = i & 7;
    const uint4 ch = *reinterpret_cast<const uint4*>(tile + hf * kQHalf + roff + ((c ^ (r & 7)) << 4));
    const uint32_t w[4] = {ch.x, ch.y, ch.z, ch.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  const float sc = __fdiv_rn(amax, 127.0f);
  const float rcp = __frcp_rn(sc);
  const bool fast_sc = sc >= 0x1p-125f && sc <= 0x1p125f;
  const int grow = tile_row0 + r;
  int8_t* dump = (q_dump != nullptr && grow < Sq_pad)
                     ? q_dump + (static_cast<size_t>(bh) * Sq_pad + grow) * kHeadDim : nullptr;
#pragma unroll 2
  for (int i = 0; i < 16; ++i) {
    const int hf = i >> 3, c = i & 7;
    uint4* cp = reinterpret_cast<uint4*>(tile + hf * kQHalf + roff + ((c ^ (r & 7)) << 4));
    const uint4 ch = *cp;
    const uint32_t w[4] = {ch.x, ch.y, ch.z, ch.w};
    float xs[8], code[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      xs[2 * e] = __uint_as_float(w[e] << 16);
      xs[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
    codes8(xs, sc, rcp, fast_sc, code);   // integer-valued, |code| <= 127: exact in fp16
    uint32_t h2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 hh = __floats2half2_rn(code[2 * e], code[2 * e + 1]);
      h2[e] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    *cp = make_uint4(h2[0], h2[1], h2[2], h2[3]);
    if (dump) {
      uint32_t b8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) b8[e] = (__float_as_uint(code[e] + kRoundMagic) - 0x4B400000u) & 0xFFu;
      *reinterpret_cast<uint2*>(dump + hf * 64 + c * 8) =
          make_uint2(b8[0] | (b8[1] << 8) | (b8[2] << 16) | (b8[3] << 24), b8[4] | (b8[5] << 8) | (b8[6] << 16) | (b8[7] << 24));
    }
  }
  const int blk = (tile_row0 + (r & ~31)) / kQKBlock;
  if (q_scale_dump != nullptr && (r & 31) == 0 && blk < nbq)
    q_scale_dump[static_cast<size_t>(bh) * nbq + blk] = sc;
  return sc;
}

template <bool kDumpS, bool kFuseQ>
__global__ void __launch_bounds__(kThreads, 1)
    sage_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float sv_smem[kHeadDim];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x / p.n_pairs;
  const int q_row0 = (blockIdx.x % p.n_pairs) * 2 * kTile;
  volatile int* abort_v = &abort_flag;
  uint8_t* sQ = smem + kSmemQ;
  uint8_t* sK = smem + kSmemK;
  uint8_t* sV = smem + kSmemV;
  uint8_t* sP = smem + kSmemP;

  if (threadIdx.x == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_ready, 256);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.s_free[t], 128);
      mbar_init(&bars.p_full[t], 128);
      mbar_init(&bars.pv_done[t], 1);
      mbar_init(&bars.o_full[t], 1);
    }
    mbar_init(&bars.drain_qk, 1);
    mbar_init(&bars.drain_pv, 1);
    abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    // This thread is also the Q/K producer: Q and the first K stages go out
    // now, while the rest of the block still sets up (their regions of shared
    // memory are touched by nothing else before the block barrier).
    mbar_arrive_expect_tx(&bars.q_full, 2 * kQTileBytes);
    for (int t = 0; t < 2; ++t) {
      if constexpr (kFuseQ) {   // bf16 [B, S, H, 128]: box of 64 channels x 128 tokens of one (b, h)
        const int b = bh / p.H, h = bh % p.H;
        tma_load_4d(sQ + t * kQTileBytes, &tmQ, &bars.q_full, 0, h, q_row0 + t * kTile, b);
        tma_load_4d(sQ + t * kQTileBytes + kQHalf, &tmQ, &bars.q_full, 64, h, q_row0 + t * kTile, b);
      } else {
        tma_load_3d(sQ + t * kQTileBytes, &tmQ, &bars.q_full, 0, q_row0 + t * kTile, bh);
        tma_load_3d(sQ + t * kQTileBytes + kQHalf, &tmQ, &bars.q_full, 64, q_row0 + t * kTile, bh);
      }
    }
    for (int j = 0; j < kStages && j < p.n_kv; ++j) {
      mbar_arrive_expect_tx(&bars.k_full[j], kKTileBytes);
      tma_load_3d(sK + j * kKTileBytes, &tmK, &bars.k_full[j], 0, j * kKV, bh);
      tma_load_3d(sK + j * kKTileBytes + kKHalf, &tmK, &bars.k_full[j], 64, j * kKV, bh);
    }
  }
  if (threadIdx.x < kHeadDim) sv_smem[threadIdx.x] = p.v_scale[static_cast<size_t>(bh) * kHeadDim + threadIdx.x];
  if (warp == 2 || warp == 3) {
    // Rows 128..143 of every V stage: E4M3 ones (any swizzle of equal bytes is
    // the same), the extra N rows that make PV also sum P.
    constexpr uint32_t kOnesWords = 16 * 32 / 4;   // per sub-tile
    for (uint32_t i = threadIdx.x - 64; i < kVStages * 3 * kOnesWords; i += 64) {
      const uint32_t sub = i / kOnesWords, w = i % kOnesWords;
      reinterpret_cast<uint32_t*>(sV + sub * kVSubBytes + kVOnesOffset)[w] = kE4M3One;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      // Q and the first kStages K stages were issued during set-up.
      int k_issued = min(kStages, p.n_kv);
      for (int j = k_issued; j < p.n_kv; ++j) {
        const int s = j % kStages, r = j / kStages;
        if (r > 0 && !wait_bar(&bars.k_empty[s], (r - 1) & 1, abort_v, p.timeout_ns)) break;
        mbar_arrive_expect_tx(&bars.k_full[s], kKTileBytes);
        tma_load_3d(sK + s * kKTileBytes, &tmK, &bars.k_full[s], 0, j * kKV, bh);
        tma_load_3d(sK + s * kKTileBytes + kKHalf, &tmK, &bars.k_full[s], 64, j * kKV, bh);
        k_issued = j + 1;
      }
      // Let every issued copy land before the CTA can exit.
      drain_bar(&bars.q_full, 0, p.timeout_ns);
      for (int j = k_issued - 1; j >= 0 && j >= k_issued - kStages; --j)
        drain_bar(&bars.k_full[j % kStages], (j / kStages) & 1, p.timeout_ns);
    }
  } else if (warp == 3) {
    // ---------------------------------------------------- V^T producer --
    // Its own thread, so that a V stage still in use never holds up K.
    if (lane == 0) {
      int v_issued = 0;
      for (int j = 0; j < p.n_kv; ++j) {
        const int s = j % kVStages, r = j / kVStages;
        if (r > 0 && !wait_bar(&bars.v_empty[s], (r - 1) & 1, abort_v, p.timeout_ns)) break;
        mbar_arrive_expect_tx(&bars.v_full[s], kVLoadBytes);
#pragma unroll
        for (int k = 0; k < 3; ++k)
          tma_load_3d(sV + s * kVStageBytes + k * kVSubBytes, &tmV, &bars.v_full[s], j * kKV + 32 * k, 0, bh);
        v_issued = j + 1;
      }
      for (int j = v_issued - 1; j >= 0 && j >= v_issued - kVStages; --j)
        drain_bar(&bars.v_full[j % kVStages], (j / kVStages) & 1, p.timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ QK^T issuer --
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f32acc(128, kKV, 0, 0);   // F16 x F16 -> F32
      const uint32_t q_lo = sw128_desc_lo(smem_addr(sQ)), k_lo = sw128_desc_lo(smem_addr(sK));
      // Q codes: straight from TMA, or after the softmax warps quantised them.
      if (wait_bar(kFuseQ ? &bars.q_ready : &bars.q_full, 0, abort_v, p.timeout_ns)) {
        for (int j = 0; j < p.n_kv; ++j) {
          const int s = j % kStages;
          if (!wait_bar(&bars.k_full[s], (j / kStages) & 1, abort_v, p.timeout_ns)) break;
          const uint32_t b0 = k_lo + s * (kKTileBytes >> 4);
          bool ok = true;
#pragma unroll
          for (int t = 0; t < 2; ++t) {   // S_t = Q_t K(j)^T once S_t is free
            if (j > 0 && !wait_bar(&bars.s_free[t], (j - 1) & 1, abort_v, p.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = q_lo + t * (kQTileBytes >> 4);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_f16_ss(tmem + col_s(t), a0 + (((k >> 2) * kQHalf + (k & 3) * 32) >> 4),
                         b0 + (((k >> 2) * kKHalf + (k & 3) * 32) >> 4), idesc, k > 0);
            mma_commit(&bars.s_full[t]);
          }
          if (!ok) break;
          mma_commit(&bars.k_empty[s]);
        }
      }
      // Wait for every issued MMA before TMEM can be released.
      mma_commit(&bars.drain_qk);
      drain_bar(&bars.drain_qk, 0, p.timeout_ns);
    }
  } else if (warp == 2) {
    // -------------------------------------------------------- PV issuer --
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f32acc(128, 144, 0, 0);   // E4M3 x E4M3 -> F32
      const uint32_t p_lo = sw128_desc_lo(smem_addr(sP)), v_lo = sw128_desc_lo(smem_addr(sV));
      for (int j = 0; j < p.n_kv; ++j) {
        const int s = j % kVStages;
        if (!wait_bar(&bars.v_full[s], (j / kVStages) & 1, abort_v, p.timeout_ns)) break;
        const uint32_t b0 = v_lo + s * (kVStageBytes >> 4);
        bool ok = true;
#pragma unroll
        for (int t = 0; t < 2; ++t) {     // O_t[0:144] += P~_t [V^T(j); ones]^T
          if (!wait_bar(&bars.p_full[t], j & 1, abort_v, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = p_lo + t * (kPTileBytes >> 4);
#pragma unroll
          for (int k = 0; k < 3; ++k)
            mma_f8_ss(tmem + col_o(t), a0 + 2 * k, b0 + k * (kVSubBytes >> 4), idesc, (j > 0 || k > 0), kSw32DescHi);
          mma_commit(&bars.pv_done[t]);
        }
        if (!ok) break;
        mma_commit(&bars.v_empty[s]);
      }
      mma_commit(&bars.o_full[0]);
      mma_commit(&bars.o_full[1]);
      mma_commit(&bars.drain_pv);
      drain_bar(&bars.drain_pv, 0, p.timeout_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------- softmax + epilogue (x2) --
    const int t = (warp - 4) >> 2;        // which Q tile
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;  // query row within the tile
    const int qrow = q_row0 + t * kTile + row;
    const bool row_valid = qrow < p.Sq;
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_bits + col_s(t);
    const uint32_t tO = tmem + lane_bits + col_o(t);
    const float* ksc = p.k_scale + static_cast<size_t>(bh) * p.nbk;
    float sq = 0.0f;
    bool ok = true;
    if constexpr (kFuseQ) {
      // Quantise this warp's own 32 rows of Q (one K-block-sized Q block, the
      // rows its softmax serves) in place: bf16 in, integer-valued fp16 out.
      ok = __all_sync(0xFFFFFFFFu, wait_bar(&bars.q_full, 0, abort_v, p.timeout_ns));
      if (ok)
        sq = quantize_q_rows(sQ + t * kQTileBytes, row, bh, q_row0 + t * kTile, p.q_dump, p.q_scale_dump,
                             p.Sq_pad, p.nbq);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // codes visible to the MMA
      mbar_arrive(&bars.q_ready);
    } else {
      sq = row_valid ? p.q_scale[static_cast<size_t>(bh) * p.nbq + qrow / kQKBlock] : 0.0f;
    }
    const float c_row = sq * p.c_scale;

    float m_run = -INFINITY;
    float sk_next[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) sk_next[i] = i < p.nbk ? __ldg(ksc + i) : 0.0f;

    for (int j = 0; j < (ok ? p.n_kv : 0); ++j) {
      float cb[3];
#pragma unroll
      for (int i = 0; i < 3; ++i) cb[i] = c_row * sk_next[i];
      if (j + 1 < p.n_kv) {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const int idx_k = 3 * (j + 1) + i;
          sk_next[i] = idx_k < p.nbk ? __ldg(ksc + idx_k) : 0.0f;
        }
      }
      // Warp-uniform outcome: the tcgen05 loads below are .sync.aligned.
      if (!__all_sync(0xFFFFFFFFu, wait_bar(&bars.s_full[t], j & 1, abort_v, p.timeout_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float a[kKV];
      {
        uint32_t r01[64], r2[32];
        tmem_ld64(tS, r01);
        tmem_ld32(tS + 64, r2);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 64; ++i) a[i] = __uint_as_float(r01[i]);
#pragma unroll
        for (int i = 0; i < 32; ++i) a[64 + i] = __uint_as_float(r2[i]);
      }
      // The scores are in registers: S_t may take the next tile's scores.
      tc_fence_before();
      mbar_arrive(&bars.s_free[t]);
      if constexpr (kDumpS) {
        if (row_valid) {
          int32_t* drow = p.s_dump + (static_cast<size_t>(bh) * p.Sq + qrow) * p.Skv + j * kKV;
          const int lim = min(kKV, p.Skv - j * kKV);
          for (int c = 0; c < lim; ++c) drow[c] = __float2int_rn(a[c]);
        }
      }

      const int valid = p.Skv - j * kKV;  // keys of this tile that exist (>= 1)
      if (valid < kKV) {
#pragma unroll
        for (int c = 0; c < kKV; ++c) a[c] = c < valid ? a[c] : -INFINITY;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < 3; ++i) {       // four independent chains per K block
        const float* ab = a + 32 * i;
        float m0 = ab[0], m1 = ab[1], m2 = ab[2], m3 = ab[3];
#pragma unroll
        for (int c = 4; c < 28; c += 8) {
          m0 = fmax3(m0, ab[c], ab[c + 1]);
          m1 = fmax3(m1, ab[c + 2], ab[c + 3]);
          m2 = fmax3(m2, ab[c + 4], ab[c + 5]);
          m3 = fmax3(m3, ab[c + 6], ab[c + 7]);
        }
        m0 = fmax3(m0, ab[28], ab[29]);
        m1 = fmax3(m1, ab[30], ab[31]);
        const float mx = fmax3(m0, m1, fmaxf(m2, m3));
        mt = fmaxf(mt, mx * cb[i]);       // a block past the end gives -inf or NaN: ignored
      }
      const float m_new = fmaxf(m_run, mt);
      const float bias = m_new - kLog2P;
      uint32_t pk[kKV / 4];
      softmax_p(a, cb, bias, pk);
      if (valid < kKV) {                  // keys past the end: code 0
#pragma unroll
        for (int w = 0; w < kKV / 4; ++w) {
          const int keep = min(max(valid - 4 * w, 0), 4);
          pk[w] &= keep == 4 ? 0xFFFFFFFFu : ((1u << (8 * keep)) - 1u);
        }
      }
      // PV(j-1) of this tile has read the P~ buffer and left O final.
      if (j > 0 && !__all_sync(0xFFFFFFFFu, wait_bar(&bars.pv_done[t], (j - 1) & 1, abort_v, p.timeout_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      store_p_row(sP + t * kPTileBytes, row, pk);
      // Rescale O and L when the running max moved.
      const bool need = (j > 0) && (m_new != m_run);
      if (__any_sync(0xFFFFFFFFu, need)) {
        // Two rounds of loads (64 columns, then 64 + L) so that only two
        // TMEM load latencies are exposed; the score registers are dead here.
        const float alpha = ex2_approx(m_run - m_new);
        uint32_t o0[32], o1[32], o2[32], o3[32], l4[4];
        tmem_ld32(tO, o0);
        tmem_ld32(tO + 32, o1);
        tmem_ld_wait();
        tmem_ld32(tO + 64, o2);
        tmem_ld32(tO + 96, o3);
        tmem_ld4(tO + 128, l4);
        scale_cols(o0, alpha);
        tmem_st32(tO, o0);
        scale_cols(o1, alpha);
        tmem_st32(tO + 32, o1);
        tmem_ld_wait();
        scale_cols(o2, alpha);
        tmem_st32(tO + 64, o2);
        scale_cols(o3, alpha);
        tmem_st32(tO + 96, o3);
        l4[0] = __float_as_uint(__uint_as_float(l4[0]) * alpha);
        tmem_st4(tO + 128, l4);
        tmem_st_wait();
      }
      m_run = m_new;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // P~ visible to the MMA
      tc_fence_before();
      mbar_arrive(&bars.p_full[t]);
    }

    // ----------------------------------------------------------- epilogue --
    if (ok && __all_sync(0xFFFFFFFFu, wait_bar(&bars.o_full[t], 0, abort_v, p.timeout_ns))) {
      tc_fence_after();
      uint32_t l4[4];
      tmem_ld4(tO + 128, l4);
      tmem_ld_wait();
      const float inv_l = 1.0f / __uint_as_float(l4[0]);
      // log sum_j exp(score_j) = ln 2 * (m + log2 L - log2 448): P~ = 448 at the max.
      if (p.lse != nullptr && row_valid)
        p.lse[static_cast<size_t>(bh) * p.Sq + qrow] = (m_run + log2f(__uint_as_float(l4[0])) - kLog2P) * kLn2;
      const int b = bh / p.H, h = bh % p.H;
      uint16_t* orow = p.out + ((static_cast<size_t>(b) * p.Sq + qrow) * p.H + h) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait();
        if (row_valid) {
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            float v16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int d = c * 32 + g * 16 + e;
              v16[e] = __uint_as_float(o[g * 16 + e]) * (sv_smem[d] * inv_l);
            }
            store_bf16x16(orow + c * 32 + g * 16, v16);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 3-D map over [BH][rows][inner] with a box of box_inner x box_rows x 1 and
// 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint32_t esize,
                uint64_t inner, uint64_t rows, uint64_t bh, uint32_t box_inner, uint32_t box_rows,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  std::memset(m, 0, sizeof(*m));
  cuuint64_t dims[3] = {inner, rows, bh};
  cuuint64_t strides[2] = {inner * esize, inner * rows * esize};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over bf16 [B, S, H, 128] with a box of 64 channels x 1 head x 128
// tokens x 1 batch and 128-byte swizzle: one half of a 128-row Q tile of one
// (batch, head).  Tokens past S read as zeros.
bool encode_map_bshd(CUtensorMap* m, const void* base, int B, int S, int H) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  std::memset(m, 0, sizeof(*m));
  const cuuint64_t e = 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {kHeadDim * e, static_cast<cuuint64_t>(H) * kHeadDim * e,
                           static_cast<cuuint64_t>(S) * H * kHeadDim * e};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kTile), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__global__ void wait_timeout_probe_kernel(uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the wait must give up after timeout_ns.
  (void)mbar_wait(&bar, 0, &abort_flag, &g_sage_error, timeout_ns);
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  const uint64_t BH = static_cast<uint64_t>(a.B) * a.H;
  CUtensorMap tmQ, tmK, tmV;
  const bool qmap_ok = a.q_bf16 != nullptr
                           ? encode_map_bshd(&tmQ, a.q_bf16, a.B, a.Sq, a.H)
                           : encode_map(&tmQ, a.q_codes, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, kHeadDim, a.Sq_pad, BH,
                                        64, 128);
  if (!qmap_ok ||
      !encode_map(&tmK, a.k_codes, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, kHeadDim, a.Skv_pad, BH, 64, kKV) ||
      !encode_map(&tmV, a.vt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.Skv_pad, kHeadDim, BH, 32, 128,
                  CU_TENSOR_MAP_SWIZZLE_32B))
    return cudaErrorInvalidValue;
  Params p;
  p.fuse_q = a.q_bf16 != nullptr;
  p.q_dump = a.q_dump;
  p.q_scale_dump = a.q_scale_dump;
  p.Sq_pad = a.Sq_pad;
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.out = a.out;
  p.s_dump = a.s_dump;
  p.lse = a.lse;
  p.Sq = a.Sq;
  p.Skv = a.Skv;
  p.H = a.H;
  p.nbq = a.nbq;
  p.nbk = a.nbk;
  p.n_kv = (a.Skv + kKV - 1) / kKV;
  p.n_pairs = (a.Sq_pad / kTile + 1) / 2;
  p.c_scale = a.softmax_scale * kLog2e;
  p.timeout_ns = a.timeout_ns;
  const uint64_t grid = BH * static_cast<uint64_t>(p.n_pairs);
  if (grid > 0x7FFFFFFFull) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  auto go = [&](auto kernel) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemDynamic);
    if (e == cudaSuccess) kernel<<<static_cast<unsigned>(grid), kThreads, kSmemDynamic, stream>>>(tmQ, tmK, tmV, p);
  };
  if (a.s_dump)
    go(sage_attn_kernel<true, false>);
  else if (p.fuse_q)
    go(sage_attn_kernel<false, true>);
  else
    go(sage_attn_kernel<false, false>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t load_attention_kernels() {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, sage_attn_kernel<false, false>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, sage_attn_kernel<false, true>);
  return e;
}

cudaError_t read_and_clear_device_error(int* code, cudaStream_t stream) {
  int host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_sage_error, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  *code = host;
  if (host != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_sage_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  }
  return e;
}

cudaError_t launch_wait_timeout_probe(uint64_t timeout_ns, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(timeout_ns);
  return cudaGetLastError();
}

}  // namespace sage
