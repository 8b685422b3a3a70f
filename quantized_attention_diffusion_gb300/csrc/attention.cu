// attention.cu -- fused SageAttention-style forward for sm_103a.
//
// What it computes (diffusers issue #15014 "gfx1201 (RDNA4) SageAttention
// attention backend", kernel contract: INT8 QK^T and FP8 PV with FP32
// accumulation, Q/K quantized per 32-row block and V per channel inside the
// kernel, BF16 [B, S, H, 128], no mask, non-causal; diffusers PR #15060,
// "What does this PR do?": no LSE).  Per query row, over KV tiles of 128 keys:
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
// accumulates L = sum p~ (rescaled with O) in columns 128..143.
//
// One CTA owns one 128-row Q tile of one (batch, head) and streams every KV
// tile of that head.  640 threads:
//   warp 0       TMA producer (Q once; K and V^T through 3-stage rings)
//   warp 1       TMEM allocator and the single MMA-issuing thread
//   warps 2-3    fill the ones rows, then idle
//   warps 4-19   softmax + epilogue: four threads per query row, thread
//                group g = (warp-4)/4 owns keys [32g, 32g+32) of every KV
//                tile (exactly one K quantisation block) and output
//                columns [32g, 32g+32)
// TMEM (512 columns): S0 [0,128)  S1 [128,256)  O [256,400).
// S is double-buffered: the MMA queue runs PV(j), QK(j+2), so the scores of
// the next tile are ready while the softmax works on this one.  P~ (E4M3, 4
// per column) overwrites the first 32 columns of its S buffer and is the A
// operand of PV straight from TMEM.  The four threads of a row swap partial
// maxima through shared memory (a named barrier per TMEM lane quarter).
// Quarters are not synchronised with each other, so one may run a tile ahead
// of another: "P ready" alternates between two barriers by tile parity, so
// arrivals for tile j+1 can never complete tile j's phase.  (No thread gets
// two tiles ahead: tile j+2's scores wait for PV(j), which waits for all.)
#include <cmath>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sage_internal.cuh"
#include "sm103_ptx.cuh"

namespace sage {

__device__ int g_sage_error;   // SAGE_DEVERR_* of the last failed wait on this device

namespace {

constexpr int kStages = 3;
constexpr int kThreads = 640;
constexpr uint32_t kHalfBytes = 128 * 64 * 2;            // 128 rows x 64 fp16
constexpr uint32_t kQKTileBytes = 2 * kHalfBytes;        // 128 x 128 fp16
constexpr uint32_t kVTileBytes = 128 * 128;              // 128 x 128 e4m3 (TMA part)
constexpr uint32_t kOnesBytes = 16 * 128;                // 16 rows of E4M3 1.0
constexpr uint32_t kVStageBytes = kVTileBytes + kOnesBytes;
constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemK = kSmemQ + kQKTileBytes;
constexpr uint32_t kSmemV = kSmemK + kStages * kQKTileBytes;
constexpr uint32_t kSmemTiles = kSmemV + kStages * kVStageBytes;
constexpr uint32_t kSmemDynamic = kSmemTiles + 1024;     // slack for 1024-byte alignment
constexpr uint32_t kColO = 256;                          // O accumulator, 144 columns
constexpr uint32_t kColL = kColO + 128;                  // L (16 equal columns)
constexpr float kLog2P = 8.80735492706298828125f;         // fp32(log2 448): P scale 448
constexpr float kLog2e = 1.44269502162933349609375f;      // fp32(log2 e)
constexpr uint32_t kE4M3One = 0x38383838u;                // four E4M3 1.0

struct Params {
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  uint16_t* out;
  int32_t* s_dump;
  int S, H, S_pad, nb, n_kv, n_qt;
  float c_scale;          // fp32(softmax_scale * fp32(log2 e))
  uint64_t timeout_ns;
};

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], pv_done, o_full;
  uint64_t drain;
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

// Named barrier over `count` threads that also ANDs a flag across them, so
// that every participant leaves with the same verdict.
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t count, bool flag) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\tsetp.ne.u32 pin, %1, 0;\n\t"
      "bar.red.and.pred pout, %2, %3, pin;\n\tselp.u32 %0, 1, 0, pout;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(flag)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void store_bf16x8(uint16_t* dst, const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// This thread's 32 integer scores of one row -> 32 E4M3 probabilities
// p~ = e4m3(2^(acc * cb - bias)) in 8 TMEM columns (4 codes per column), the
// A operand of the PV MMA.  kMasked: keys at or beyond `valid` get 0.
template <bool kMasked>
__device__ __forceinline__ void softmax_p32(const float (&a)[32], float cb, float bias, int valid,
                                            uint32_t tP) {
  uint32_t pk[8];
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int c = w * 4;
    const float2 x01 = ffma2_bc(a[c], a[c + 1], cb, -bias);
    const float2 x23 = ffma2_bc(a[c + 2], a[c + 3], cb, -bias);
    float p0 = ex2_approx(x01.x), p1 = ex2_approx(x01.y);
    float p2 = ex2_approx(x23.x), p3 = ex2_approx(x23.y);
    if constexpr (kMasked) {
      p0 = c < valid ? p0 : 0.0f;
      p1 = c + 1 < valid ? p1 : 0.0f;
      p2 = c + 2 < valid ? p2 : 0.0f;
      p3 = c + 3 < valid ? p3 : 0.0f;
    }
    pk[w] = static_cast<uint32_t>(cvt_e4m3x2(p0, p1)) | (static_cast<uint32_t>(cvt_e4m3x2(p2, p3)) << 16);
  }
  tmem_st8(tP, pk);
}

template <bool kDumpS>
__global__ void __launch_bounds__(kThreads, 1)
    sage_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ Barriers bars;
  __shared__ float max_part[2][4][128];   // [tile parity][key group][row]
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float sv_smem[kHeadDim];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x / p.n_qt;
  const int q_row0 = (blockIdx.x % p.n_qt) * kTile;
  volatile int* abort_v = &abort_flag;
  uint8_t* sQ = smem + kSmemQ;
  uint8_t* sK = smem + kSmemK;
  uint8_t* sV = smem + kSmemV;

  if (threadIdx.x == 0) {
    mbar_init(&bars.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.s_full[0], 1);
    mbar_init(&bars.s_full[1], 1);
    mbar_init(&bars.p_full[0], 512);
    mbar_init(&bars.p_full[1], 512);
    mbar_init(&bars.pv_done, 1);
    mbar_init(&bars.o_full, 1);
    mbar_init(&bars.drain, 1);
    abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (threadIdx.x < kHeadDim) sv_smem[threadIdx.x] = p.v_scale[static_cast<size_t>(bh) * kHeadDim + threadIdx.x];
  if (warp == 2 || warp == 3) {
    // rows 128..143 of every V stage: E4M3 ones (any swizzle of equal bytes is
    // the same), the extra N rows that make PV also sum P
    for (uint32_t i = threadIdx.x - 64; i < kStages * kOnesBytes / 4; i += 64) {
      const uint32_t s = i / (kOnesBytes / 4), w = i % (kOnesBytes / 4);
      reinterpret_cast<uint32_t*>(sV + s * kVStageBytes + kVTileBytes)[w] = kE4M3One;
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
      mbar_arrive_expect_tx(&bars.q_full, kQKTileBytes);
      tma_load_3d(sQ, &tmQ, &bars.q_full, 0, q_row0, bh);
      tma_load_3d(sQ + kHalfBytes, &tmQ, &bars.q_full, 64, q_row0, bh);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < p.n_kv; ++j) {
        const int s = j % kStages, r = j / kStages;
        if (r > 0 && !wait_bar(&bars.k_empty[s], (r - 1) & 1, abort_v, p.timeout_ns)) break;
        mbar_arrive_expect_tx(&bars.k_full[s], kQKTileBytes);
        tma_load_3d(sK + s * kQKTileBytes, &tmK, &bars.k_full[s], 0, j * kTile, bh);
        tma_load_3d(sK + s * kQKTileBytes + kHalfBytes, &tmK, &bars.k_full[s], 64, j * kTile, bh);
        k_issued = j + 1;
        if (r > 0 && !wait_bar(&bars.v_empty[s], (r - 1) & 1, abort_v, p.timeout_ns)) break;
        mbar_arrive_expect_tx(&bars.v_full[s], kVTileBytes);
        tma_load_3d(sV + s * kVStageBytes, &tmV, &bars.v_full[s], j * kTile, 0, bh);
        v_issued = j + 1;
      }
      // Let every issued copy land before the CTA can exit.
      drain_bar(&bars.q_full, 0, p.timeout_ns);
      for (int j = k_issued - 1; j >= 0 && j >= k_issued - kStages; --j)
        drain_bar(&bars.k_full[j % kStages], (j / kStages) & 1, p.timeout_ns);
      for (int j = v_issued - 1; j >= 0 && j >= v_issued - kStages; --j)
        drain_bar(&bars.v_full[j % kStages], (j / kStages) & 1, p.timeout_ns);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc_f32acc(128, 128, 0, 0);   // F16 x F16 -> F32
      const uint32_t idesc_pv = make_idesc_f32acc(128, 144, 0, 0);   // E4M3 x E4M3 -> F32
      const uint32_t sq_addr = smem_addr(sQ), sk_addr = smem_addr(sK), sv_addr = smem_addr(sV);
      auto qk = [&](int j) {   // S[j % 2] = Q K(j)^T
        const int s = j % kStages;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
          mma_f16_ss(tmem + (j & 1) * 128, make_sw128_desc(sq_addr + off),
                     make_sw128_desc(sk_addr + s * kQKTileBytes + off), idesc_qk, k > 0);
        }
        mma_commit(&bars.s_full[j & 1]);
        mma_commit(&bars.k_empty[s]);
      };
      bool ok = wait_bar(&bars.q_full, 0, abort_v, p.timeout_ns);
      for (int j = 0; ok && j < 2 && j < p.n_kv; ++j) {
        ok = wait_bar(&bars.k_full[j % kStages], (j / kStages) & 1, abort_v, p.timeout_ns);
        if (ok) {
          tc_fence_after();
          qk(j);
        }
      }
      for (int j = 0; ok && j < p.n_kv; ++j) {
        const int s = j % kStages;
        if (!wait_bar(&bars.v_full[s], (j / kStages) & 1, abort_v, p.timeout_ns)) break;
        if (!wait_bar(&bars.p_full[j & 1], (j >> 1) & 1, abort_v, p.timeout_ns)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)   // O[0:144] += P~(S[j % 2] cols 8k..8k+7) x [V^T; 1] rows
          mma_f8_ts(tmem + kColO, tmem + (j & 1) * 128 + k * 8,
                    make_sw128_desc(sv_addr + s * kVStageBytes + k * 32), idesc_pv, (j > 0 || k > 0));
        mma_commit(&bars.pv_done);
        mma_commit(&bars.v_empty[s]);
        if (j + 2 < p.n_kv) {
          if (!wait_bar(&bars.k_full[(j + 2) % kStages], ((j + 2) / kStages) & 1, abort_v, p.timeout_ns))
            break;
          tc_fence_after();
          qk(j + 2);
        }
      }
      mma_commit(&bars.o_full);
      // Wait for every issued MMA before TMEM can be released.
      mma_commit(&bars.drain);
      drain_bar(&bars.drain, 0, p.timeout_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax + epilogue --
    const int g = (warp - 4) >> 2;        // key group: keys [32g, 32g+32) of each tile
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;  // query row within the tile
    const int qrow = q_row0 + row;
    const bool row_valid = qrow < p.S;
    const uint32_t bar_id = 1 + quarter;  // the 4 warps (128 threads) sharing these rows
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const float* ksc = p.k_scale + static_cast<size_t>(bh) * p.nb;
    const float sq = row_valid ? p.q_scale[static_cast<size_t>(bh) * p.nb + qrow / kQKBlock] : 0.0f;
    const float c_row = sq * p.c_scale;

    float m_run = -INFINITY;
    float sk_next = g < p.nb ? __ldg(ksc + g) : 0.0f;
    bool ok = true;

    for (int j = 0; j < p.n_kv; ++j) {
      const float cb = c_row * sk_next;
      if (j + 1 < p.n_kv) {
        const int idx_k = 4 * (j + 1) + g;
        sk_next = idx_k < p.nb ? __ldg(ksc + idx_k) : 0.0f;
      }
      const uint32_t tS = tmem + lane_bits + (j & 1) * 128;
      const bool got = ok && __all_sync(0xFFFFFFFFu, wait_bar(&bars.s_full[j & 1], (j >> 1) & 1, abort_v,
                                                               p.timeout_ns));
      tc_fence_after();
      float a[32];
      {
        uint32_t r[32];
        tmem_ld32(tS + g * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = __uint_as_float(r[i]);
      }
      if constexpr (kDumpS) {
        if (row_valid && got) {
          int32_t* drow = p.s_dump + (static_cast<size_t>(bh) * p.S + qrow) * p.S + j * kTile + g * 32;
          const int lim = min(32, p.S - j * kTile - g * 32);
          for (int c = 0; c < lim; ++c) drow[c] = __float2int_rn(a[c]);
        }
      }
      const int valid = p.S - j * kTile - g * 32;   // keys of this group that exist (may be <= 0)
      float mt;
      if (valid >= 32) {
        float mx = a[0];
#pragma unroll
        for (int c = 1; c < 31; c += 2) mx = fmax3(mx, a[c], a[c + 1]);
        mx = fmaxf(mx, a[31]);
        mt = mx * cb;
      } else {
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) mx = c < valid ? fmaxf(mx, a[c]) : mx;
        mt = valid > 0 ? mx * cb : -INFINITY;
      }
      // Swap partial maxima with the row's other three threads.  The barrier
      // also orders all four threads' TMEM reads of S before any of them
      // writes P~ over the first 32 columns, and carries the wait verdicts.
      max_part[j & 1][g][row] = mt;
      tc_fence_before();
      if (!bar_and(bar_id, 128, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      mt = fmaxf(fmaxf(max_part[j & 1][0][row], max_part[j & 1][1][row]),
                 fmaxf(max_part[j & 1][2][row], max_part[j & 1][3][row]));

      const float m_new = fmaxf(m_run, mt);
      const float bias = m_new - kLog2P;
      if (valid >= 32)
        softmax_p32<false>(a, cb, bias, valid, tS + g * 8);
      else
        softmax_p32<true>(a, cb, bias, valid, tS + g * 8);
      // Rescale O (and L) when the running max moved.  PV(j-1) must have
      // landed first; it was queued right after P(j-1), so this rarely waits.
      const bool need = (j > 0) && (m_new != m_run);
      if (__any_sync(0xFFFFFFFFu, need)) {
        ok = __all_sync(0xFFFFFFFFu, wait_bar(&bars.pv_done, (j - 1) & 1, abort_v, p.timeout_ns));
        tc_fence_after();
        const float alpha = ex2_approx(m_run - m_new);
        uint32_t o[32];
        tmem_ld32(tmem + lane_bits + kColO + g * 32, o);
        uint32_t l4[4];
        tmem_ld4(tmem + lane_bits + kColL + g * 4, l4);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
#pragma unroll
        for (int i = 0; i < 4; ++i) l4[i] = __float_as_uint(__uint_as_float(l4[i]) * alpha);
        tmem_st32(tmem + lane_bits + kColO + g * 32, o);
        tmem_st4(tmem + lane_bits + kColL + g * 4, l4);
      }
      m_run = m_new;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full[j & 1]);
    }

    // ----------------------------------------------------------- epilogue --
    if (ok && __all_sync(0xFFFFFFFFu, wait_bar(&bars.o_full, 0, abort_v, p.timeout_ns))) {
      tc_fence_after();
      uint32_t o[32];
      uint32_t l4[4];
      tmem_ld32(tmem + lane_bits + kColO + g * 32, o);
      tmem_ld4(tmem + lane_bits + kColL, l4);
      tmem_ld_wait();
      if (row_valid) {
        const float inv_l = 1.0f / __uint_as_float(l4[0]);
        const int b = bh / p.H, h = bh % p.H;
        uint16_t* orow = p.out + ((static_cast<size_t>(b) * p.S + qrow) * p.H + h) * kHeadDim + g * 32;
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          float v8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int d = g * 32 + q8 * 8 + e;
            v8[e] = __uint_as_float(o[q8 * 8 + e]) * (sv_smem[d] * inv_l);
          }
          store_bf16x8(orow + q8 * 8, v8);
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

// 3-D map over [BH][rows][inner] with a box of box_inner x 128 x 1 and
// 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint32_t esize,
                uint64_t inner, uint64_t rows, uint64_t bh, uint32_t box_inner) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  std::memset(m, 0, sizeof(*m));
  cuuint64_t dims[3] = {inner, rows, bh};
  cuuint64_t strides[2] = {inner * esize, inner * rows * esize};
  cuuint32_t box[3] = {box_inner, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
  if (!encode_map(&tmQ, a.q_codes, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, kHeadDim, a.S_pad, BH, 64) ||
      !encode_map(&tmK, a.k_codes, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, kHeadDim, a.S_pad, BH, 64) ||
      !encode_map(&tmV, a.vt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.S_pad, kHeadDim, BH, 128))
    return cudaErrorInvalidValue;
  Params p;
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.out = a.out;
  p.s_dump = a.s_dump;
  p.S = a.S;
  p.H = a.H;
  p.S_pad = a.S_pad;
  p.nb = a.nb;
  p.n_kv = a.S_pad / kTile;
  p.n_qt = a.S_pad / kTile;
  p.c_scale = a.softmax_scale * kLog2e;
  p.timeout_ns = a.timeout_ns;
  const uint64_t grid = BH * static_cast<uint64_t>(p.n_qt);
  if (grid > 0x7FFFFFFFull) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  if (a.s_dump) {
    e = cudaFuncSetAttribute(sage_attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemDynamic);
    if (e != cudaSuccess) return e;
    sage_attn_kernel<true><<<static_cast<unsigned>(grid), kThreads, kSmemDynamic, stream>>>(tmQ, tmK, tmV, p);
  } else {
    e = cudaFuncSetAttribute(sage_attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemDynamic);
    if (e != cudaSuccess) return e;
    sage_attn_kernel<false><<<static_cast<unsigned>(grid), kThreads, kSmemDynamic, stream>>>(tmQ, tmK, tmV, p);
  }
  return cudaGetLastError();
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
