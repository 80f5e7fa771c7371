// gdn_chunk_util.cuh — device helpers shared by the two schedules of the chunked prefill
// kernel (gdn_chunked.cu, gdn_chunked_pipe.cu): fp16 packing into 128B-swizzled operand
// tiles, the bf16 -> fp16 widening of q/k/v, the gate loads of a chunk, the per-token gate
// factors (one code path, so that both schedules compute them bit for bit alike) and the
// warp-level f16 tile products of the 64 x 64 triangular inverse.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "gdn_internal.h"
#include "ptx_sm103.cuh"

namespace gdn {
namespace chunk {

constexpr int kC = 64;          // tokens per chunk
constexpr int kD = 128;         // head dim
constexpr int kLd = 68;         // fp32 64x64 matrix row stride (conflict-free float4 rows)
constexpr int kLdX = 36;        // row stride of the 32 x 32 merge scratch (2 kLdX = 8 mod
                                // 32: its f16 B-fragment loads fall on distinct banks)
constexpr int kLdXs = 12;       // row stride of a warp's 16 x 8 merge scratch (likewise:
                                // 2 kLdXs = 24 mod 32 and kLdXs = 12 mod 32)
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kStatusTimeout = 5;  // GDN_ERR_DEVICE_TIMEOUT
constexpr float kLog2e = 1.4426950408889634f;
// Lowest log2-decay of one token in the chunk scan (see gate_scan).
constexpr float kMinLog2Decay = -200.f;

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Eight fp32 values as fp16 into one 16-byte chunk of a 128B-swizzled tile.
__device__ __forceinline__ void st_chunk(uint8_t* tile, uint32_t row, uint32_t col,
                                         uint32_t rows_per_region, const float (&x)[8]) {
  uint4 v;
  v.x = pack_half2(x[0], x[1]);
  v.y = pack_half2(x[2], x[3]);
  v.z = pack_half2(x[4], x[5]);
  v.w = pack_half2(x[6], x[7]);
  *reinterpret_cast<uint4*>(tile + ptx::sw128_offset(row, col, rows_per_region)) = v;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& w, float (&x)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(u[i] << 16);
    x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// bf16 -> fp16 is exact for magnitudes in [2^-17, 65504] (8 significant bits fit in 11).
__device__ __forceinline__ uint4 bf16x8_to_half8(const uint4& w) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 hh = __floats2half2_rn(__uint_as_float(u[i] << 16),
                                         __uint_as_float(u[i] & 0xFFFF0000u));
    o[i] = *reinterpret_cast<const uint32_t*>(&hh);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 pack_half8(const float (&x)[8]) {
  return make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]),
                    pack_half2(x[6], x[7]));
}

// Starts the loads of the log-decays and betas of the chunk at token t0 (one warp, two
// tokens per lane). Token indices are clamped into the prompt so that nothing waits on the
// loads here; gates_of() masks the tokens past the chunk when the values are used.
__device__ __forceinline__ void fetch_gates(const float* ag, const float* bg, size_t stride,
                                            int t0, int len, int lane, float (&g)[4]) {
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const size_t t = (size_t)min(t0 + lane + 32 * hh, len - 1);
    g[hh] = __ldg(ag + t * stride);
    g[2 + hh] = __ldg(bg + t * stride);
  }
}

// Gates of the chunk at t0 from fetch_gates' values: raw inputs are transformed, and
// tokens past the chunk get a = beta = 0.
__device__ __forceinline__ void gates_of(const float (&raw_g)[4], int t0, int len, int lane,
                                         bool raw, float a_log, float dt_bias, float (&g)[4]) {
  const int L = min(kC, len - t0);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float a = raw_g[hh], b = raw_g[2 + hh];
    if (raw) gate_from_raw(a_log, dt_bias, a, b);
    const bool live = lane + 32 * hh < L;
    g[hh] = live ? a : 0.f;
    g[2 + hh] = live ? b : 0.f;
  }
}

// Per-token factors of one chunk: eight 64-float arrays from one base.
struct Factors {
  float* G;    // log2-scaled inclusive cumulative log-decay
  float* B;    // beta
  float* Gq;   // scale e^{G_t} / |q_t|: row factor of Q~
  float* BG;   // beta_j e^{G_j} / |k_j|: column factor of T1
  float* Dec;  // e^{G_L - G_j} / |k_j|: row factor of D'
  float* Gp;   // G_j - log2(1/|k_j|): column exponent of A and P
  float* Rk;   // 1/|k_j|
  float* Rq;   // 1/|q_t|
  __device__ explicit Factors(float* base)
      : G(base), B(base + 64), Gq(base + 128), BG(base + 192), Dec(base + 256),
        Gp(base + 320), Rk(base + 384), Rq(base + 448) {}
};

// Chunk-local inclusive cumulative log-decay (log2 units) of tokens lane and lane + 32 by
// a warp scan (a0, a1); returns the chunk total G_L. Every product and sum is rounded on
// its own (no contraction), so that every caller, in either schedule, gets the same bits.
__device__ __forceinline__ float gate_scan(const float (&g)[4], int lane, float& a0,
                                           float& a1) {
  // A token's log2-decay is held at -200 or above: a = -inf (g = 0, the state restarts at
  // that token) then gives factors 2^-200, which are exactly 0 in fp32, and no inf - inf in
  // the differences of the scan. Decays above -200 (a > -138.6) keep their bits.
  a0 = fmaxf(__fmul_rn(g[0], kLog2e), kMinLog2Decay);
  a1 = fmaxf(__fmul_rn(g[1], kLog2e), kMinLog2Decay);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y0 = __shfl_up_sync(0xffffffffu, a0, off);
    const float y1 = __shfl_up_sync(0xffffffffu, a1, off);
    if (lane >= off) {
      a0 = __fadd_rn(a0, y0);
      a1 = __fadd_rn(a1, y1);
    }
  }
  a1 = __fadd_rn(a1, __shfl_sync(0xffffffffu, a0, 31));
  return __shfl_sync(0xffffffffu, a1, 31);  // padded tokens add nothing
}

// The gate factors of one chunk from its gates (one warp, tokens lane and lane + 32); the
// norms are folded in later. Returns e^{G_L}.
__device__ __forceinline__ float write_gate_factors(const Factors& f, const float (&g)[4],
                                                    float scale, int lane) {
  float a0, a1;
  const float gl = gate_scan(g, lane, a0, a1);
  const float b0 = g[2], b1 = g[3];
  const float e0 = ptx::ex2(a0), e1 = ptx::ex2(a1);
  f.G[lane] = a0;
  f.G[lane + 32] = a1;
  f.B[lane] = b0;
  f.B[lane + 32] = b1;
  f.Gq[lane] = __fmul_rn(scale, e0);
  f.Gq[lane + 32] = __fmul_rn(scale, e1);
  f.BG[lane] = __fmul_rn(b0, e0);
  f.BG[lane + 32] = __fmul_rn(b1, e1);
  f.Dec[lane] = ptx::ex2(__fsub_rn(gl, a0));
  f.Dec[lane + 32] = ptx::ex2(__fsub_rn(gl, a1));
  return ptx::ex2(gl);
}

// q and k of one chunk (K rows 0-63, Q rows 64-127 of a 128B-swizzled tile whose two
// 64-column regions start kRegionBytes apart) to fp16 in place (exact: bf16 values are fp16
// values), with their inverse L2 norms into f.Rk / f.Rq (0 for rows past the chunk's L
// tokens, which are zeroed). The norms are not applied to the tile: they are folded into
// per-token factors. One group of 256 threads (gtid), 16 per row and 8 rows each.
//  * Each row piece is stored as soon as it is converted: the stores need no norm.
//  * The 8 rows' sums of squares are reduced over the 16 threads of a row by a
//    reduce-scatter (each level keeps half of the partial sums), 8 shuffles in all; the
//    thread pair (j, j^1) ends with the sum of row j >> 1, and thread j even writes its norm.
// Both schedules of the chunked kernel call this one function, so that their norms, and
// everything built from them, agree bit for bit.
template <uint32_t kRegionBytes>
__device__ __forceinline__ void convert_kq(uint8_t* sKQ, const Factors& f, int L, bool l2norm,
                                           int gtid) {
  const int j = gtid & 15, rsub = gtid >> 4;  // piece j of the row
  const uint32_t reg = j >> 3, cc = j & 7;
  auto at = [&](uint32_t r) {
    return reinterpret_cast<uint4*>(sKQ + reg * kRegionBytes + (r >> 3) * 1024 + (r & 7) * 128 +
                                    ((cc ^ (r & 7)) << 4));
  };
  uint4 w[8];
#pragma unroll
  for (int pass = 0; pass < 8; ++pass) w[pass] = *at(pass * 16 + rsub);
  float ss[8];
#pragma unroll
  for (int pass = 0; pass < 8; ++pass) {
    const uint32_t r = pass * 16 + rsub;
    float x[8];
    unpack_bf16x8(w[pass], x);
    // sum of squares of the piece: even and odd elements in two lanes of packed FMAs
    float2 a = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float2 xe = make_float2(x[e], x[e + 1]);
      a = ptx::fma2(xe, xe, a);
    }
    ss[pass] = __fadd_rn(a.x, a.y);
    *at(r) = (int)(r & 63) < L ? pack_half8(x) : make_uint4(0u, 0u, 0u, 0u);
  }
  // reduce-scatter: 8 partial sums -> 4 (xor 8) -> 2 (xor 4) -> 1 (xor 2) -> full (xor 1)
  const bool b8 = j & 8, b4 = j & 4, b2 = j & 2;
  float s4[4], s2[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b8 ? ss[i] : ss[4 + i];
    s4[i] = __fadd_rn(b8 ? ss[4 + i] : ss[i], __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b4 ? s4[i] : s4[2 + i];
    s2[i] = __fadd_rn(b4 ? s4[2 + i] : s4[i], __shfl_xor_sync(0xffffffffu, send, 4));
  }
  float s1 = __fadd_rn(b2 ? s2[1] : s2[0],
                       __shfl_xor_sync(0xffffffffu, b2 ? s2[0] : s2[1], 2));
  s1 = __fadd_rn(s1, __shfl_xor_sync(0xffffffffu, s1, 1));
  if (!(j & 1)) {
    const int pass = j >> 1;  // 4 b8 + 2 b4 + b2
    const uint32_t t = (uint32_t)(pass * 16 + rsub) & 63;
    const float rn = (int)t < L ? (l2norm ? rsqrtf(s1 + kL2NormEps) : 1.f) : 0.f;
    (pass < 4 ? f.Rk : f.Rq)[t] = rn;
  }
}

// Chunks whose total log2-decay is at least this take the factored form of the A/P
// epilogue (ap_row): their column factors 2^{-Gp_j} = 2^{-G_j} / |k_j| stay below 2^110,
// since 1/|k_j| <= 1/sqrt(kL2NormEps) < 2^10.
constexpr float kFactoredMinLog2Decay = -100.f;

// Column factor of the factored A/P epilogue for token j: 2^{-Gp_j} = e^{-G_j} / |k_j| (0
// for padded tokens, whose Gp is +inf). Written by the warp that folds the norms into Gp.
__device__ __forceinline__ float col_factor(float gp) { return ptx::ex2(-gp); }

// One thread's 32 columns j0..j0+31 of row `row` of the first product [K;Q]K^T (r: its fp32
// accumulators) scaled into
//   A (rows 0-63):   A_ij = beta_i e^{G_i - G_j} (k_i . k_j) / (|k_i| |k_j|)  for j < i, else 0
//                    (fp32, row stride kLd), or
//   P (rows 64-127): P_tj = scale e^{G_t - G_j} (q_t . k_j) / (|q_t| |k_j|)  for j <= t, else 0
//                    (fp16 128B-swizzled tile).
// The scale factor of an entry is 2^{x_i - Gp_j}, with x_i the row's exponent (G_i plus the
// log2 of its beta, or scale, and inverse norm). With `factored` (the chunk's total log2-decay
// is at least kFactoredMinLog2Decay) it is split as 2^{x_i} 2^{-Gp_j}, and an entry costs two
// multiplies with the column factors cf (col_factor) read from shared memory. Both factors
// are finite; below the diagonal their product is the entry's factor (at most 1 before the
// norms), and above it, where the product may overflow to inf, the entry is masked to 0
// (no NaN: the first product is finite). A row factor below the normal range only scales
// entries far below the fp16 rounding of T. Otherwise every entry takes its own ex2 of the
// difference, which is never above 0 below the diagonal. Both schedules call this one
// function, so that A and P agree bit for bit between them.
template <bool kFactored>
__device__ __forceinline__ void ap_row_form(const uint32_t (&r)[32], uint32_t row, int j0,
                                            const Factors& f, const float* cf, float scale,
                                            float* sA, uint8_t* sP) {
  const float* w_src = kFactored ? cf : f.Gp;  // column factors or column exponents
  if (row < 64) {
    const int i = row;
    const float xi = f.G[i] + __log2f(f.B[i] * f.Rk[i]);
    const float ri = kFactored ? ptx::ex2(xi) : 0.f;
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 w = *reinterpret_cast<const float4*>(w_src + j0 + e);
      const float w4[4] = {w.x, w.y, w.z, w.w};
      float x4[4];
      if (kFactored) {  // (a ri) w per entry, two entries per packed multiply
#pragma unroll
        for (int q = 0; q < 4; q += 2) {
          const float2 t = ptx::mul2(
              make_float2(__uint_as_float(r[e + q]), __uint_as_float(r[e + q + 1])),
              make_float2(ri, ri));
          const float2 y = ptx::mul2(t, make_float2(w4[q], w4[q + 1]));
          x4[q] = y.x;
          x4[q + 1] = y.y;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) x4[q] = __uint_as_float(r[e + q]) * ptx::ex2(xi - w4[q]);
      }
      float4 v;
      float* vv = reinterpret_cast<float*>(&v);
#pragma unroll
      for (int q = 0; q < 4; ++q) vv[q] = j0 + e + q < i ? x4[q] : 0.f;
      *reinterpret_cast<float4*>(sA + i * kLd + j0 + e) = v;
    }
  } else {
    const int t = row - 64;
    const float xt = f.G[t] + __log2f(scale * f.Rq[t]);
    const float rt = kFactored ? ptx::ex2(xt) : 0.f;
#pragma unroll
    for (int e = 0; e < 32; e += 8) {
      const float4 wa = *reinterpret_cast<const float4*>(w_src + j0 + e);
      const float4 wb = *reinterpret_cast<const float4*>(w_src + j0 + e + 4);
      const float w8[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      float x[8];
      float y8[8];
      if (kFactored) {  // (a rt) w per entry, two entries per packed multiply
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
          const float2 u = ptx::mul2(
              make_float2(__uint_as_float(r[e + q]), __uint_as_float(r[e + q + 1])),
              make_float2(rt, rt));
          const float2 y = ptx::mul2(u, make_float2(w8[q], w8[q + 1]));
          y8[q] = y.x;
          y8[q + 1] = y.y;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) y8[q] = __uint_as_float(r[e + q]) * ptx::ex2(xt - w8[q]);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) x[q] = j0 + e + q <= t ? y8[q] : 0.f;
      st_chunk(sP, t, j0 + e, 64, x);
    }
  }
}

__device__ __forceinline__ void ap_row(const uint32_t (&r)[32], uint32_t row, int j0,
                                       const Factors& f, const float* cf, float scale,
                                       bool factored, float* sA, uint8_t* sP) {
  if (factored)
    ap_row_form<true>(r, row, j0, f, cf, scale, sA, sP);
  else
    ap_row_form<false>(r, row, j0, f, cf, scale, sA, sP);
}

// Column j of the inverse of the unit lower-triangular 16 x 16 block I + A[o:o+16, o:o+16]
// (A strictly lower, fp32, row stride kLd) into x: x_i = delta_ij - sum_{k<i} A_ik x_k, by
// forward substitution. Every x_i is the same chain of fused multiply-adds over k in
// ascending order in both forms below, so they give the same bits:
//  * diag_block_column (row by row) reads row i of the block as float4s that every lane
//    handling the block shares (broadcasts): 36 loads instead of one per term;
//  * diag_block_column_rl (column by column: x_k, once final, is taken out of every later
//    row) reads one element per term and holds fewer registers, for the 16-warp schedule,
//    whose register budget the row form overflows.
__device__ __forceinline__ void diag_block_column(const float* A, int o, int j,
                                                  float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float acc = i == j ? 1.f : 0.f;
    const float* ar = A + (o + i) * kLd + o;
#pragma unroll
    for (int k4 = 0; k4 < i; k4 += 4) {
      const float4 a = *reinterpret_cast<const float4*>(ar + k4);
      const float a4[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int f = 0; f < 4; ++f)
        if (k4 + f < i) acc = __fmaf_rn(-a4[f], x[k4 + f], acc);
    }
    x[i] = acc;
  }
}

__device__ __forceinline__ void diag_block_column_rl(const float* A, int o, int j,
                                                     float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = i == j ? 1.f : 0.f;
#pragma unroll
  for (int k = 0; k < 15; ++k) {
    const float xk = x[k];
#pragma unroll
    for (int i = k + 1; i < 16; ++i) x[i] = __fmaf_rn(-A[(o + i) * kLd + o + k], xk, x[i]);
  }
}

// One 16 x 8 output tile D += sum_k Ablk[r0.., k] * Bblk[k.., n0..] over k in [k_lo, k_hi)
// (multiples of 16, at most 32 wide) on one warp, f16 warp MMAs (m16n8k16) with fp32
// accumulation. Both matrices fp32 with row strides lda/ldb, rounded to fp16
// (round to nearest even) as they are loaded: fp16 keeps tf32's 10-bit significand, and
// the inverse's entries stay far inside its range. Each 16-wide k step goes into a zeroed
// tile of its own and the partial tiles are added in a fixed order, so the steps run side
// by side instead of as a chain of dependent warp MMAs.
__device__ __forceinline__ void tile_mm(float (&d)[4], const float* Am, int lda, int r0,
                                        const float* Bm, int ldb, int n0, int k_lo, int k_hi,
                                        int gid, int tig) {
  float p[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
#pragma unroll
    for (int e = 0; e < 4; ++e) p[s][e] = 0.f;
    const int k = k_lo + 16 * s;
    if (k < k_hi) {
      const float* a0 = Am + (r0 + gid) * lda + k + 2 * tig;  // scalar loads: no bank
      const float* a1 = a0 + 8 * lda;                          // conflicts with lda = 68
      const uint32_t a[4] = {ptx::f16x2(a0[0], a0[1]), ptx::f16x2(a1[0], a1[1]),
                             ptx::f16x2(a0[8], a0[9]), ptx::f16x2(a1[8], a1[9])};
      const float* bc = Bm + n0 + gid;
      const uint32_t b[2] = {ptx::f16x2(bc[(k + 2 * tig) * ldb], bc[(k + 2 * tig + 1) * ldb]),
                             ptx::f16x2(bc[(k + 2 * tig + 8) * ldb], bc[(k + 2 * tig + 9) * ldb])};
      ptx::mma_f16_16816(p[s], a, b);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] += p[0][e] + p[1][e];
}

// Stores a 16 x 8 accumulator tile (optionally negated) at (r0, n0) of an fp32 matrix.
__device__ __forceinline__ void tile_store(float* M, int ld, int r0, int n0, const float (&d)[4],
                                           float sign, int gid, int tig) {
  M[(r0 + gid) * ld + n0 + 2 * tig] = sign * d[0];
  M[(r0 + gid) * ld + n0 + 2 * tig + 1] = sign * d[1];
  M[(r0 + gid + 8) * ld + n0 + 2 * tig] = sign * d[2];
  M[(r0 + gid + 8) * ld + n0 + 2 * tig + 1] = sign * d[3];
}

// A negated 16 x 8 accumulator tile of T at (r0, n0) into T1 and T2 (column pairs as half2).
__device__ __forceinline__ void tile_store_t12(uint8_t* T1, uint8_t* T2, int r0, int n0,
                                               const float (&d)[4], const float* c1,
                                               const float* c2, int gid, int tig) {
  const int col = n0 + 2 * tig;
  const float g0 = c1[col], g1 = c1[col + 1], b0 = c2[col], b1 = c2[col + 1];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const uint32_t off = ptx::sw128_offset(r0 + gid + 8 * hh, col, 64);
    const float2 x = make_float2(-d[2 * hh], -d[2 * hh + 1]);
    const float2 y1 = ptx::mul2(x, make_float2(g0, g1)), y2 = ptx::mul2(x, make_float2(b0, b1));
    *reinterpret_cast<uint32_t*>(T1 + off) = pack_half2(y1.x, y1.y);
    *reinterpret_cast<uint32_t*>(T2 + off) = pack_half2(y2.x, y2.y);
  }
}

// The state of unit (prompt, value head) in the init / final arrays ([.][H_v][D][D]): the
// prompt's state slot.
template <int D>
__device__ __forceinline__ size_t state_offset(const PrefillArgs& p, const GdnSeq& sd, int h) {
  return ((size_t)sd.state_slot * p.hv_heads + h) * D * D;
}

// The initial state of the unit, or nullptr for a zero state.
template <int D>
__device__ __forceinline__ const float* initial_state(const PrefillArgs& p, const GdnSeq& sd,
                                                      int h) {
  return p.init && !(sd.flags & kSeqZeroInit) ? p.init + state_offset<D>(p, sd, h) : nullptr;
}

// A unit of a prompt with one token or none, run by a whole block of kThreads threads (128,
// 256 or 512) with the decode step's arithmetic: no chunk phases, no tensor memory (a
// one-token prompt costs only its state traffic). Both chunked schedules call it, so their
// results agree bit for bit. Each state row is owned by 4 threads holding 32 entries each
// as float4 chunks c = sub + 4 m (sub = tid % 4); the block covers kThreads / 4 rows per
// pass. Every pass's state loads are issued first, so that their latency overlaps the q/k
// normalisation. The state comes from the prompt's initial state (zero without one) and
// goes to its final state, and to the prompt's checkpoint when one is requested at
// position 1; an empty prompt copies its initial state. The initial state may alias the
// final state: a thread reads each chunk of its rows before it writes it.
// sk, sq: 128 floats of shared memory each.
template <int kThreads, int D>
__device__ __forceinline__ void short_unit(const PrefillArgs& p, const GdnUnit& u,
                                           const GdnSeq& sd, float* sk, float* sq, int tid) {
  // rows per pass (threads past them idle when the block has more than 4 threads per row)
  constexpr int kRowsPass = kThreads / 4 < D ? kThreads / 4 : D;
  constexpr int kVec = D / 16, kPass = D / kRowsPass;
  static_assert(kPass >= 1 && kPass * kRowsPass == D, "rows per pass");
  const bool has_row = (tid >> 2) < kRowsPass;
  const int h = u.head, hk = h / p.group;
  const int warp = tid >> 5, lane = tid & 31, sub = tid & 3;
  const float* init = initial_state<D>(p, sd, h);
  float* fin = p.final_state + state_offset<D>(p, sd, h);
  if (sd.len == 0) {  // empty prompt: the final state is the initial state
    for (int i = tid; i < D * D / 4; i += kThreads)
      reinterpret_cast<float4*>(fin)[i] =
          init ? reinterpret_cast<const float4*>(init)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const size_t tok = (size_t)sd.tok_start;
  float4 S[kPass][kVec];
  float vi[kPass];
#pragma unroll
  for (int ps = 0; ps < kPass; ++ps) {
    const int row = has_row ? ps * kRowsPass + (tid >> 2) : 0;
    const float4* src = init ? reinterpret_cast<const float4*>(init + (size_t)row * D) : nullptr;
#pragma unroll
    for (int m = 0; m < kVec; ++m)
      S[ps][m] = src ? src[sub + 4 * m] : make_float4(0.f, 0.f, 0.f, 0.f);
    vi[ps] = (sd.flags & kSeqZeroV)
                 ? 0.f
                 : __bfloat162float(
                       static_cast<const __nv_bfloat16*>(p.v)[(tok * p.hv_heads + h) * D + row]);
  }
  float ga = p.a[tok * p.hv_heads + h], bb = p.beta[tok * p.hv_heads + h];
  if (warp == 0) {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q) + (tok * p.hk_heads + hk) * D;
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(p.k) + (tok * p.hk_heads + hk) * D;
    float qv[D / 32], kv[D / 32], qq = 0.f, kk = 0.f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      qv[e] = __bfloat162float(q[lane + 32 * e]);
      kv[e] = __bfloat162float(k[lane + 32 * e]);
      qq += qv[e] * qv[e];
      kk += kv[e] * kv[e];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      qq += __shfl_xor_sync(0xffffffffu, qq, off);
      kk += __shfl_xor_sync(0xffffffffu, kk, off);
    }
    const float qs = p.l2norm ? rsqrtf(qq + kL2NormEps) : 1.f;
    const float ks = p.l2norm ? rsqrtf(kk + kL2NormEps) : 1.f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      sq[lane + 32 * e] = qv[e] * qs;
      sk[lane + 32 * e] = kv[e] * ks;
    }
  }
  if (p.gate_mode == 1) gate_from_raw(p.a_log[h], p.dt_bias[h], ga, bb);
  const float g = __expf(ga);
  __syncthreads();
  const float4* kr = reinterpret_cast<const float4*>(sk);
  const float4* qr = reinterpret_cast<const float4*>(sq);
  const bool ckpt1 = sd.ckpt_end > sd.ckpt_begin && p.ckpt_pos[sd.ckpt_begin] == 1;
  if (!has_row) return;  // (whole warps: the row loop shuffles within a warp)
#pragma unroll
  for (int ps = 0; ps < kPass; ++ps) {
    const int row = ps * kRowsPass + (tid >> 2);
    float dot = 0.f;
#pragma unroll
    for (int m = 0; m < kVec; ++m) {
      const float4 k4 = kr[sub + 4 * m];
      S[ps][m].x *= g; S[ps][m].y *= g; S[ps][m].z *= g; S[ps][m].w *= g;
      dot += S[ps][m].x * k4.x + S[ps][m].y * k4.y + S[ps][m].z * k4.z + S[ps][m].w * k4.w;
    }
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    const float delta = bb * (vi[ps] - dot);
    float4* dst = reinterpret_cast<float4*>(fin + (size_t)row * D);
    float4* ck = ckpt1 ? reinterpret_cast<float4*>(p.ckpt + ((size_t)sd.ckpt_begin * p.hv_heads + h) *
                                                              D * D + (size_t)row * D)
                       : nullptr;
    float outv = 0.f;
#pragma unroll
    for (int m = 0; m < kVec; ++m) {
      const float4 k4 = kr[sub + 4 * m];
      const float4 q4 = qr[sub + 4 * m];
      S[ps][m].x += delta * k4.x; S[ps][m].y += delta * k4.y;
      S[ps][m].z += delta * k4.z; S[ps][m].w += delta * k4.w;
      outv += S[ps][m].x * q4.x + S[ps][m].y * q4.y + S[ps][m].z * q4.z + S[ps][m].w * q4.w;
      dst[sub + 4 * m] = S[ps][m];
      if (ck) ck[sub + 4 * m] = S[ps][m];
    }
    outv += __shfl_xor_sync(0xffffffffu, outv, 1);
    outv += __shfl_xor_sync(0xffffffffu, outv, 2);
    if (sub == 0)
      static_cast<__nv_bfloat16*>(p.o)[(tok * p.hv_heads + h) * D + row] =
          __float2bfloat16_rn(p.scale * outv);
  }
}

}  // namespace chunk
}  // namespace gdn
