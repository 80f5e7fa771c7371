// gdn_chunked.cu — chunked gated-delta-rule prefill on the tcgen05 tensor cores (sm_103a).
//
// Method (Gated Delta Networks, Yang, Kautz & Hatamizadeh, 2024, in its chunked UT/WY
// form). Per (prompt, value head) unit the state S (d_v x d_k = 128 x 128, fp32) is carried
// through chunks of C = 64 tokens. For a chunk of L <= C tokens with chunk-local inclusive
// log-decay sums G_i and L2-normalised keys/queries:
//     A_ij  = beta_i exp(G_i - G_j) (k_i . k_j)   (j < i)        T = (I + A)^-1
//     W^T   = K^T (T diag(beta e^G))^T            U^T = V^T (T diag(beta))^T
//     D^T   = U^T - S W^T                          (row i of D: what token i writes)
//     O^T   = S (diag(e^G) Q)^T + D^T P^T,         P_tj = exp(G_t - G_j) (q_t . k_j), j <= t
//     S    <- e^{G_L} S + D^T diag(exp(G_L - G)) K
// All exponents are <= 0. Every product runs on the tensor cores in the transposed
// orientation, so the 128-row M side is always d_v or d_k and every MMA is M = 128.
//
// Precision: every tensor-core operand is IEEE fp16 (11-bit significand) with fp32
// accumulation; q and k are normalised in fp32 before their single rounding, v is widened
// exactly from bf16, and the fp32 state is kept in TMEM (the fp16 copy that feeds the MMAs
// is refreshed every chunk). This keeps outputs within 2e-3 relative L2 of an fp64
// evaluation where bf16 operands would not. Operands must stay inside the fp16 range
// (|v| and state entries below 65504).
//
// Per CTA (256 threads, 8 warps): one unit, chunks in order. TMEM (256 columns):
//   [0, 64)    R0: the current product (K K^T | Q K^T, W^T, D^T, O^T), fp32
//   [64, 128)  S16: fp16 copy of S, the A operand of the state products
//   [128, 256) S32: the fp32 state, accumulated in place by the update product
// Shared memory holds the chunk's fp16 tiles in the 128B-swizzled layout (see
// ptx_sm103.cuh), about 90 KB, so two CTAs share an SM and hide each other's latency.
// Every mbarrier wait is bounded; a timeout is reported through the status word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn_internal.h"
#include "ptx_sm103.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk
constexpr int kD = 128;         // head dim
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kStatusTimeout = 5;  // GDN_ERR_DEVICE_TIMEOUT
constexpr int kLd = 65;          // fp32 matrix row stride (bank-conflict padding)

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;                       // [K;Q] 128 rows x 128 fp16: 32 KB
constexpr uint32_t OFF_V = OFF_KQ + 32768;           // V: 64 rows x 128 fp16: 16 KB
constexpr uint32_t OFF_P = OFF_V + 16384;            // P: 64 x 64 fp16: 8 KB
constexpr uint32_t OFF_A = OFF_P + 8192;             // A fp32 [64][65], later T1 | T2 fp16
constexpr uint32_t OFF_T1 = OFF_A;                   //   T diag(beta e^G): 8 KB
constexpr uint32_t OFF_T2 = OFF_A + 8192;            //   T diag(beta): 8 KB
constexpr uint32_t OFF_WD = OFF_A + 17408;           // T fp32 [64][65], then W^T, then D^T
constexpr uint32_t OFF_X = OFF_WD + 17408;           // inverse scratch: 3 x 16 x 16 fp32
constexpr uint32_t OFF_VEC = OFF_X + 3072;           // G, beta, 1/|k|, 1/|q|: 4 x 64 fp32
constexpr uint32_t SMEM_USED = OFF_VEC + 1024;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;    // + alignment slack

constexpr uint32_t TM_R0 = 0, TM_S16 = 64, TM_S32 = 128, TM_COLS = 256;

struct __align__(8) Smem {
  uint64_t bar;
  uint32_t tmem_base;
  int32_t fail;
};

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Sum over the 16 lanes that share a token row.
__device__ __forceinline__ float sum16(float x) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Stores 8 consecutive fp16 values (one 16-byte chunk) of tile row `row`, columns col..col+7.
__device__ __forceinline__ void st_chunk(uint8_t* tile, uint32_t row, uint32_t col,
                                         uint32_t rows_per_region, const float (&x)[8]) {
  uint4 v;
  v.x = pack_half2(x[0], x[1]);
  v.y = pack_half2(x[2], x[3]);
  v.z = pack_half2(x[4], x[5]);
  v.w = pack_half2(x[6], x[7]);
  *reinterpret_cast<uint4*>(tile + sw128_offset(row, col, rows_per_region)) = v;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& w, float (&x)[8]) {
  x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
  x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
}

// Load this thread's 8-element slice of token row `t` (bf16) as fp32; zeros past the chunk.
__device__ __forceinline__ void load_row8(const __nv_bfloat16* base, size_t row_stride, int t,
                                          int L, int c8, float (&x)[8]) {
  if (t < L) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(base + (size_t)t * row_stride + c8));
    unpack_bf16x8(w, x);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.f;
  }
}

// Wait for the MMA barrier, uniformly across the block; returns false on timeout.
__device__ __forceinline__ bool wait_mma(Smem& sm, uint32_t& phase) {
  const bool ok = mbar_wait_bounded(&sm.bar, phase & 1u, kWaitLimit);
  phase ^= 1u;
  tc_fence_after();
  return !__syncthreads_or(!ok);
}

// Makes generic-proxy smem writes and TMEM stores visible to the next MMA issue.
__device__ __forceinline__ void publish_operands() {
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// (I + A)^-1 for a 64 x 64 strictly-lower A (fp32, row stride kLd), by 16 x 16 blocks:
// diagonal blocks by forward substitution, then T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj in
// order of increasing i - j. Writes the lower triangle (with the unit diagonal) of T.
__device__ void invert_unit_lower(const float* A, float* T, float* X, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < 4 && lane < 16) {
    const int b = warp, j = lane, o = 16 * b;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < i; ++k) s += A[(o + i) * kLd + o + k] * x[k];
      x[i] = (i == j) ? 1.f : (i < j ? 0.f : -s);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) T[(o + i) * kLd + o + j] = x[i];
  }
  __syncthreads();
  // distance 1, 2, 3 between block row and block column
  for (int dist = 1; dist <= 3; ++dist) {
    const int nblk = 4 - dist;  // blocks (bi, bj) with bi - bj = dist
    for (int idx = tid; idx < nblk * 256; idx += kThreads) {
      const int bj = idx >> 8, bi = bj + dist, r = (idx >> 4) & 15, c = idx & 15;
      float s = 0.f;
      for (int bk = bj; bk < bi; ++bk) {
        const float* Ar = A + (16 * bi + r) * kLd + 16 * bk;
        const float* Tc = T + (16 * bk) * kLd + 16 * bj + c;
#pragma unroll
        for (int k = 0; k < 16; ++k) s += Ar[k] * Tc[k * kLd];
      }
      X[idx] = s;
    }
    __syncthreads();
    for (int idx = tid; idx < nblk * 256; idx += kThreads) {
      const int bj = idx >> 8, bi = bj + dist, r = (idx >> 4) & 15, c = idx & 15;
      const float* Tr = T + (16 * bi + r) * kLd + 16 * bi;
      const float* Xc = X + (bj << 8) + c;
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) s += (k <= r ? Tr[k] : 0.f) * Xc[k * 16];
      T[(16 * bi + r) * kLd + 16 * bj + c] = -s;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 2) chunked_prefill_kernel(PrefillArgs p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Smem sm;
  uint8_t* sKQ = smem + OFF_KQ;
  uint8_t* sV = smem + OFF_V;
  uint8_t* sP = smem + OFF_P;
  float* sA = reinterpret_cast<float*>(smem + OFF_A);
  uint8_t* sT1 = smem + OFF_T1;
  uint8_t* sT2 = smem + OFF_T2;
  float* sT = reinterpret_cast<float*>(smem + OFF_WD);
  uint8_t* sWD = smem + OFF_WD;
  float* sX = reinterpret_cast<float*>(smem + OFF_X);
  float* sG = reinterpret_cast<float*>(smem + OFF_VEC);
  float* sB = sG + 64;
  float* sRk = sG + 128;
  float* sRq = sG + 192;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GdnUnit u = p.units[blockIdx.x];
  const GdnSeq sd = p.seqs[u.seq];
  const int h = u.head, hk = h / p.group;
  const size_t qk_stride = (size_t)p.hk_heads * kD;  // elements between tokens
  const size_t v_stride = (size_t)p.hv_heads * kD;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) +
                            (size_t)sd.tok_start * qk_stride + (size_t)hk * kD;
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(p.k) +
                            (size_t)sd.tok_start * qk_stride + (size_t)hk * kD;
  const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(p.v) +
                            (size_t)sd.tok_start * v_stride + (size_t)h * kD;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + (size_t)sd.tok_start * v_stride +
                      (size_t)h * kD;
  const float* ag = p.a + (size_t)sd.tok_start * p.hv_heads + h;
  const float* bg = p.beta + (size_t)sd.tok_start * p.hv_heads + h;
  const size_t state_off = ((size_t)u.seq * p.hv_heads + h) * kD * kD;

  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
    sm.fail = 0;
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  // this warp's TMEM lanes (subpartition) and column half
  const uint32_t sub = warp & 3, half = warp >> 2;
  const uint32_t row = 32 * sub + lane;             // TMEM lane = matrix row of this thread
  const uint32_t t_lane = tbase + ((32 * sub) << 16);

  // ---- initial state -> S32 (fp32) and S16 (fp16) -----------------------------------
  {
    const float* src = p.init ? p.init + state_off + (size_t)row * kD + 64 * half : nullptr;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
      uint32_t r[16];
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        float4 v = src ? __ldg(reinterpret_cast<const float4*>(src + c0 + e))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        r[e] = __float_as_uint(v.x); r[e + 1] = __float_as_uint(v.y);
        r[e + 2] = __float_as_uint(v.z); r[e + 3] = __float_as_uint(v.w);
      }
      tmem_st16(t_lane + TM_S32 + 64 * half + c0, r);
      uint32_t h8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        h8[e] = pack_half2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
      tmem_st8(t_lane + TM_S16 + 32 * half + c0 / 2, h8);
    }
    tmem_st_wait();
  }

  uint32_t phase = 0;
  bool ok = true;
  int c_next = sd.ckpt_begin;
  const float scale = p.scale;

  for (int t0 = 0; t0 < sd.len && ok; t0 += kC) {
    const int L = min(kC, sd.len - t0);

    // ---- (1) gates: G = chunk-local inclusive cumsum of a; beta (zero past L) ----------
    if (warp == 0) {
      float a0 = lane < L ? __ldg(ag + (size_t)(t0 + lane) * p.hv_heads) : 0.f;
      float a1 = lane + 32 < L ? __ldg(ag + (size_t)(t0 + lane + 32) * p.hv_heads) : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, a0, off);
        const float y1 = __shfl_up_sync(0xffffffffu, a1, off);
        if (lane >= off) { a0 += y0; a1 += y1; }
      }
      a1 += __shfl_sync(0xffffffffu, a0, 31);
      sG[lane] = a0;
      sG[lane + 32] = a1;
      sB[lane] = lane < L ? __ldg(bg + (size_t)(t0 + lane) * p.hv_heads) : 0.f;
      sB[lane + 32] = lane + 32 < L ? __ldg(bg + (size_t)(t0 + lane + 32) * p.hv_heads) : 0.f;
    }

    // ---- (2) normalised K (rows 0-63) and Q (rows 64-127), V, all fp16 -------------------
    {
      const int rsub = tid >> 4, c8 = (tid & 15) * 8;  // 16 rows per pass, 8 cols/thread
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        const int t = pass * 16 + rsub;
        float xk[8], xq[8], xv[8];
        load_row8(kg + (size_t)t0 * qk_stride, qk_stride, t, L, c8, xk);
        load_row8(qg + (size_t)t0 * qk_stride, qk_stride, t, L, c8, xq);
        load_row8(vg + (size_t)t0 * v_stride, v_stride, t, L, c8, xv);
        float kk = 0.f, qq = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) { kk += xk[e] * xk[e]; qq += xq[e] * xq[e]; }
        kk = sum16(kk);
        qq = sum16(qq);
        const float rk = p.l2norm ? rsqrtf(kk + kL2NormEps) : 1.f;
        const float rq = p.l2norm ? rsqrtf(qq + kL2NormEps) : 1.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) { xk[e] *= rk; xq[e] *= rq; }
        st_chunk(sKQ, t, c8, 128, xk);
        st_chunk(sKQ, 64 + t, c8, 128, xq);
        st_chunk(sV, t, c8, 64, xv);
        if ((tid & 15) == 0) { sRk[t] = rk; sRq[t] = rq; }
      }
    }
    publish_operands();

    // ---- (3) M1: [K; Q] K^T -> R0 (128 x 64) ------------------------------------------
    if (tid == 0) {
      const uint32_t idesc = idesc_f16(128, 64, 0, 0);
      const uint32_t a0 = smem_u32(sKQ);
#pragma unroll
      for (int s = 0; s < kD / 16; ++s) {
        const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
        mma_f16_ss(tbase + TM_R0, smem_desc_sw128(a0 + off, 16, 1024),
                   smem_desc_sw128(a0 + off, 16, 1024), idesc, s > 0);
      }
      mma_commit(&sm.bar);
    }
    __syncwarp();
    if (!(ok = wait_mma(sm, phase))) break;

    // ---- (4) A (rows 0-63) and P (rows 64-127) from R0 ------------------------------------
    {
      uint32_t r[32];
      tmem_ld32(t_lane + TM_R0 + 32 * half, r);
      tmem_ld_wait();
      const int j0 = 32 * half;
      if (row < 64) {
        const int i = row;
        const float gi = sG[i], bi = sB[i];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int j = j0 + e;
          sA[i * kLd + j] = j < i ? bi * __expf(gi - sG[j]) * __uint_as_float(r[e]) : 0.f;
        }
      } else {
        const int t = row - 64;
        const float gt = sG[t];
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float x[8];
#pragma unroll
          for (int f = 0; f < 8; ++f) {
            const int j = j0 + e + f;
            x[f] = j <= t ? __expf(gt - sG[j]) * __uint_as_float(r[e + f]) : 0.f;
          }
          st_chunk(sP, t, j0 + e, 64, x);
        }
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- (5) T = (I + A)^-1; T1 = T diag(beta e^G), T2 = T diag(beta) in fp16 ---------------
    invert_unit_lower(sA, sT, sX, tid);
    {
      const int i = tid >> 2, jb = (tid & 3) * 16;
      float x1[8], x2[8];
#pragma unroll
      for (int h8 = 0; h8 < 16; h8 += 8) {
#pragma unroll
        for (int f = 0; f < 8; ++f) {
          const int j = jb + h8 + f;
          const float tij = j <= i ? sT[i * kLd + j] : 0.f;
          const float bj = sB[j];
          x2[f] = tij * bj;
          x1[f] = x2[f] * __expf(sG[j]);
        }
        st_chunk(sT1, i, jb + h8, 64, x1);
        st_chunk(sT2, i, jb + h8, 64, x2);
      }
    }
    publish_operands();

    // ---- (6) M2: W^T = K^T T1^T -> R0 (128 x 64) -------------------------------------------
    if (tid == 0) {
      const uint32_t idesc = idesc_f16(128, 64, 1, 0);
      const uint32_t a0 = smem_u32(sKQ), b0 = smem_u32(sT1);
#pragma unroll
      for (int s = 0; s < kC / 16; ++s)
        mma_f16_ss(tbase + TM_R0, smem_desc_sw128(a0 + s * 2048, 16384, 1024),
                   smem_desc_sw128(b0 + s * 32, 16, 1024), idesc, s > 0);
      mma_commit(&sm.bar);
    }
    __syncwarp();
    if (!(ok = wait_mma(sm, phase))) break;

    // ---- (7) W^T -> smem (fp16); K~, Q~ over K, Q; S32 *= e^{G_L} ----------------------------
    {
      uint32_t r[32];
      tmem_ld32(t_lane + TM_R0 + 32 * half, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        float x[8];
#pragma unroll
        for (int f = 0; f < 8; ++f) x[f] = __uint_as_float(r[e + f]);
        st_chunk(sWD, row, 32 * half + e, 128, x);  // W^T row d_k, columns = tokens
      }
      const float gL = sG[L - 1];
      const float decay = __expf(gL);
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t s32[32];
        tmem_ld32(t_lane + TM_S32 + 64 * half + c0, s32);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) s32[e] = __float_as_uint(__uint_as_float(s32[e]) * decay);
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) { lo[e] = s32[e]; hi[e] = s32[16 + e]; }
        tmem_st16(t_lane + TM_S32 + 64 * half + c0, lo);
        tmem_st16(t_lane + TM_S32 + 64 * half + c0 + 16, hi);
      }
      const int rsub = tid >> 4, c8 = (tid & 15) * 8;
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        const int t = pass * 16 + rsub;
        float xk[8], xq[8];
        load_row8(kg + (size_t)t0 * qk_stride, qk_stride, t, L, c8, xk);
        load_row8(qg + (size_t)t0 * qk_stride, qk_stride, t, L, c8, xq);
        const float fk = sRk[t] * __expf(gL - sG[t]);
        const float fq = sRq[t] * __expf(sG[t]);
#pragma unroll
        for (int e = 0; e < 8; ++e) { xk[e] *= fk; xq[e] *= fq; }
        st_chunk(sKQ, t, c8, 128, xk);
        st_chunk(sKQ, 64 + t, c8, 128, xq);
      }
      tmem_st_wait();
    }
    publish_operands();

    // ---- (8) M3: D^T = V^T T2^T - S16 W^T -> R0 -------------------------------------------------
    if (tid == 0) {
      const uint32_t id_u = idesc_f16(128, 64, 1, 0);
      const uint32_t id_w = idesc_f16(128, 64, 0, 1, 0, 1);  // B negated
      const uint32_t v0 = smem_u32(sV), t2 = smem_u32(sT2), w0 = smem_u32(sWD);
#pragma unroll
      for (int s = 0; s < kC / 16; ++s)
        mma_f16_ss(tbase + TM_R0, smem_desc_sw128(v0 + s * 2048, 8192, 1024),
                   smem_desc_sw128(t2 + s * 32, 16, 1024), id_u, s > 0);
#pragma unroll
      for (int s = 0; s < kD / 16; ++s)
        mma_f16_ts(tbase + TM_R0, tbase + TM_S16 + s * 8,
                   smem_desc_sw128(w0 + s * 2048, 16384, 1024), id_w, 1);
      mma_commit(&sm.bar);
    }
    __syncwarp();
    if (!(ok = wait_mma(sm, phase))) break;

    // ---- (9) D^T -> smem (fp16, K-major A: rows d_v, columns tokens) ------------------------
    {
      uint32_t r[32];
      tmem_ld32(t_lane + TM_R0 + 32 * half, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        float x[8];
#pragma unroll
        for (int f = 0; f < 8; ++f) x[f] = __uint_as_float(r[e + f]);
        st_chunk(sWD, row, 32 * half + e, 128, x);
      }
    }
    publish_operands();

    // ---- (10) M4/M5: O^T = S16 Q~^T + D^T P^T -> R0; S32 += D^T K~ ----------------------------
    if (tid == 0) {
      const uint32_t id_n64 = idesc_f16(128, 64, 0, 0);
      const uint32_t id_n128 = idesc_f16(128, 128, 0, 1);
      const uint32_t kq = smem_u32(sKQ), d0 = smem_u32(sWD), p0 = smem_u32(sP);
#pragma unroll
      for (int s = 0; s < kD / 16; ++s) {
        const uint32_t off = 8192 + (s >> 2) * 16384 + (s & 3) * 32;  // Q~ rows 64-127
        mma_f16_ts(tbase + TM_R0, tbase + TM_S16 + s * 8, smem_desc_sw128(kq + off, 16, 1024),
                   id_n64, s > 0);
      }
#pragma unroll
      for (int s = 0; s < kC / 16; ++s)
        mma_f16_ss(tbase + TM_R0, smem_desc_sw128(d0 + s * 32, 16, 1024),
                   smem_desc_sw128(p0 + s * 32, 16, 1024), id_n64, 1);
#pragma unroll
      for (int s = 0; s < kC / 16; ++s)
        mma_f16_ss(tbase + TM_S32, smem_desc_sw128(d0 + s * 32, 16, 1024),
                   smem_desc_sw128(kq + s * 2048, 16384, 1024), id_n128, 1);
      mma_commit(&sm.bar);
    }
    __syncwarp();
    if (!(ok = wait_mma(sm, phase))) break;

    // ---- (11) o, S16 refresh, checkpoints ---------------------------------------------------
    {
      uint32_t r[32];
      tmem_ld32(t_lane + TM_R0 + 32 * half, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = 32 * half + e;
        if (t < L)
          og[(size_t)(t0 + t) * v_stride + row] = __float2bfloat16_rn(scale * __uint_as_float(r[e]));
      }
      const int pos = t0 + L;
      const bool emit = c_next < sd.ckpt_end && p.ckpt_pos[c_next] == pos;
      const bool last = pos == sd.len;
      float* ck = emit ? p.ckpt + ((size_t)c_next * p.hv_heads + h) * kD * kD + (size_t)row * kD
                       : nullptr;
      float* fin = last ? p.final_state + state_off + (size_t)row * kD : nullptr;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t s32[32];
        tmem_ld32(t_lane + TM_S32 + 64 * half + c0, s32);
        tmem_ld_wait();
        uint32_t h16[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          h16[e] = pack_half2(__uint_as_float(s32[2 * e]), __uint_as_float(s32[2 * e + 1]));
        tmem_st16(t_lane + TM_S16 + 32 * half + c0 / 2, h16);
        const int col = 64 * half + c0;
        if (ck) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<uint4*>(ck + col + e) =
                make_uint4(s32[e], s32[e + 1], s32[e + 2], s32[e + 3]);
        }
        if (fin) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<uint4*>(fin + col + e) =
                make_uint4(s32[e], s32[e + 1], s32[e + 2], s32[e + 3]);
        }
      }
      if (emit) ++c_next;
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (ok && sd.len == 0) {
    // zero-length prompt: the final state is the initial state
    const float* src = p.init ? p.init + state_off + (size_t)row * kD + 64 * half : nullptr;
    float* dst = p.final_state + state_off + (size_t)row * kD + 64 * half;
    for (int e = 0; e < 64; e += 4)
      *reinterpret_cast<float4*>(dst + e) =
          src ? __ldg(reinterpret_cast<const float4*>(src + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (!ok) {
    if (tid == 0 && p.status) atomicExch(p.status, kStatusTimeout);
    // give an MMA that may still be in flight one more bounded chance to land
    mbar_wait_bounded(&sm.bar, phase & 1u, kWaitLimit);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

int chunked_prefill_smem_bytes() { return (int)SMEM_BYTES; }

int launch_chunked_prefill(const PrefillArgs& a, void* stream) {
  if (a.num_units == 0) return 0;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(chunked_prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return (int)e;
    configured = true;
  }
  chunked_prefill_kernel<<<a.num_units, kThreads, SMEM_BYTES, static_cast<cudaStream_t>(stream)>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace gdn
