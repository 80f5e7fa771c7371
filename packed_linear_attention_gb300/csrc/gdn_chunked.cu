// gdn_chunked.cu — chunked gated-delta-rule prefill on the tcgen05 tensor cores (sm_103a),
// throughput schedule.
//
// Method (Gated Delta Networks, Yang, Kautz & Hatamizadeh, 2024, in its chunked UT/WY
// form). Per (prompt, value head) unit the state S (d_v x d_k = 128 x 128, fp32) is carried
// through chunks of C = 64 tokens. For a chunk of L <= C tokens with chunk-local inclusive
// log-decay sums G_i and L2-normalised keys/queries:
//     A_ij  = beta_i exp(G_i - G_j) (k_i . k_j)   (j < i)        T = (I + A)^-1
//     W^T   = K^T (T diag(beta e^G))^T            U^T = V^T (T diag(beta))^T
//     D^T   = U^T - S W^T                          (row i of D: what token i writes)
//     O^T   = S (diag(e^G) Q)^T + D^T P^T,         P_tj = exp(G_t - G_j) (q_t . k_j), j <= t
//     S    <- e^{G_L} S + (diag(exp(G_L - G)) D)^T K
// All exponents are <= 0. Every tensor-core product runs in the transposed orientation, so
// the 128-row M side is always d_v or d_k and every MMA is M = 128.
//
// Precision: every tcgen05 operand is IEEE fp16 (11-bit significand) with fp32
// accumulation; q and k are normalised in fp32 before their rounding, v is widened exactly
// from bf16, and the fp32 state lives in TMEM for the whole prompt (its fp16 copy feeds
// the MMAs and is refreshed every chunk). The 64x64 triangular inverse is fp32 (diagonal
// blocks by forward substitution, off-diagonal blocks by warp-level f16 products).
// Operands must stay inside the fp16 range (|v| and state entries below 65504).
// Heads of d = 64 run zero-padded to 128: only the first 64-column region of q, k and v is
// copied in (the other stays zero), so every product sees exact zeros past d and the state
// rows and columns past d stay zero; only the d x d state and d output columns are stored.
//
// Throughput schedule: per CTA (256 threads, 8 warps, two CTAs per SM) one unit, the
// phases of each chunk in sequence; the two CTAs of an SM hide each other's latencies.
// The pipelined schedule (gdn_chunked_pipe.cu) computes the same chunk algebra with one
// 16-warp CTA per SM, rounding every value the same way (the code they share is in
// gdn_chunk_util.cuh), so their results are bit-identical; launch_chunked_prefill picks
// between them.
//   TMEM (256 columns): [0,64) R0 = the current product (fp32); [64,128) S16 = fp16 state
//   copy (A operand of the state products); [128,256) S32 = fp32 state, accumulated in
//   place by the update product.
//   Shared memory (128B-swizzled fp16 tiles, see ptx_sm103.cuh): raw bf16 q/k/v arrive by
//   TMA and are converted in place; the next chunk's v is fetched as soon as the current
//   one is consumed, q/k as soon as the last product of the chunk has read them.
// Every mbarrier wait is bounded (a poll count and about one second); a timeout is
// reported through the status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn_internal.h"
#include "gdn_chunk_util.cuh"
#include "ptx_sm103.cuh"

namespace gdn {
namespace {

using namespace ptx;
using namespace chunk;

constexpr int kThreads = 256;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;         // K (rows 0-63) and Q (rows 64-127): 2 regions x 16 KB
constexpr uint32_t OFF_V = 32768;      // V: 2 regions x 8 KB
constexpr uint32_t OFF_P = 49152;      // P: 64 x 64 fp16
constexpr uint32_t OFF_A = 57344;      // A fp32 [64][68] -> T1 (first 8 KB) -> D' -> o staging
constexpr uint32_t OFF_WD = 75776;     // T fp32 [64][68] -> W^T -> D
constexpr uint32_t OFF_XS = OFF_WD + 17408;  // inverse scratch: 32 x kLdX fp32 (5 KB)
constexpr uint32_t OFF_VEC = OFF_XS + 5120;  // per-token gate factors: 8 x 64 fp32
constexpr uint32_t OFF_T2 = OFF_VEC + 2048;  // T2 (fp16 64 x 64), a region of its own
static_assert(OFF_T2 % 1024 == 0, "shared-memory map");
constexpr uint32_t SMEM_USED = OFF_T2 + 8192;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack

constexpr uint32_t TM_R0 = 0, TM_S16 = 64, TM_S32 = 128, TM_COLS = 256;
constexpr uint32_t KQ_BYTES = 32768, V_BYTES = 16384;

struct ChunkedParams {
  PrefillArgs a;
  CUtensorMap tq, tk, tv;  // 2D bf16 maps: (H*128 columns, T rows), 64 x 64 boxes, SW128
  CUtensorMap to;          // o: (H_v*128 columns, T rows), 64-row x 128-column boxes, no swizzle
};

struct __align__(8) Smem {
  uint64_t bar_mma, bar_kq, bar_v;
  uint32_t tmem_base;
  float next_decay;  // e^{G_L} of the next chunk
};
// The warp that owns the gates: idle while thread 0 issues the chunk's last products (warp 1
// folds the norms during the first product). (A second thread issuing the state update
// alongside thread 0 was measured slower.)
constexpr int kGateWarp = 2;

// Waits (every thread, bounded) for the pending phase of an mbarrier, with one answer for
// the whole block (false on a timeout). A phase that a thread saw complete advances its
// `phase` and clears its `pending`; after a timeout both still name the pending phase, for
// the cleanup. (Thread 0 polling alone, the other warps waiting at the block barrier, was
// measured slower: the barrier's wake-up after the phase completes costs more than the
// polls take from the other CTA on the SM.)
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t& phase, bool& pending) {
  const bool ok = mbar_wait_bounded(bar, phase & 1u, kWaitLimit);
  if (ok) {
    phase ^= 1u;
    pending = false;
  }
  tc_fence_after();
  return !__syncthreads_or(!ok);
}

// wait_all for the q/k copy and (when `with_v`) the v copy, with one block barrier.
__device__ __forceinline__ bool wait_copies(uint64_t* bar_kq, uint32_t& ph_kq, bool& kq_pending,
                                            uint64_t* bar_v, uint32_t& ph_v, bool& v_pending,
                                            bool with_v) {
  bool ok = mbar_wait_bounded(bar_kq, ph_kq & 1u, kWaitLimit);
  if (ok) {
    ph_kq ^= 1u;
    kq_pending = false;
  }
  if (ok && with_v) {
    ok = mbar_wait_bounded(bar_v, ph_v & 1u, kWaitLimit);
    if (ok) {
      ph_v ^= 1u;
      v_pending = false;
    }
  }
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

// Issue the TMA loads of one chunk: q and k (one barrier; 2 boxes per 64 columns of d)
// and/or v (1 box per 64 columns). `dh`: the head dim (64 or 128).
__device__ __forceinline__ void issue_kq(const ChunkedParams& P, uint8_t* sKQ, uint64_t* bar,
                                         int hk, int row, int dh) {
  mbar_arrive_expect_tx(bar, KQ_BYTES / (kD / dh));
  for (int r = 0; r < dh / 64; ++r) {
    tma_load_2d(sKQ + r * 16384, &P.tk, hk * dh + 64 * r, row, bar);
    tma_load_2d(sKQ + r * 16384 + 8192, &P.tq, hk * dh + 64 * r, row, bar);
  }
}
__device__ __forceinline__ void issue_v(const ChunkedParams& P, uint8_t* sV, uint64_t* bar,
                                        int h, int row, int dh) {
  mbar_arrive_expect_tx(bar, V_BYTES / (kD / dh));
  for (int r = 0; r < dh / 64; ++r) tma_load_2d(sV + r * 8192, &P.tv, h * dh + 64 * r, row, bar);
}


// Loads the log-decays and betas of the chunk starting at token t0 (one warp); with raw
// gate inputs they are turned into gates here. Tokens past the chunk get a = beta = 0.
__device__ __forceinline__ void load_gates(const float* ag, const float* bg, size_t stride,
                                           int t0, int len, int lane, bool raw,
                                           float a_log, float dt_bias, float (&g)[4]) {
  const int L = min(kC, len - t0);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int t = lane + 32 * hh;
    float a = 0.f, b = 0.f;
    if (t < L) {
      a = __ldg(ag + (size_t)(t0 + t) * stride);
      b = __ldg(bg + (size_t)(t0 + t) * stride);
      if (raw) gate_from_raw(a_log, dt_bias, a, b);
    }
    g[hh] = a;
    g[2 + hh] = b;
  }
}

// (I + A)^-1 for a 64 x 64 strictly-lower A (fp32, row stride kLd) into T (same stride):
//  1. (invert_diag_blocks) the four 16 x 16 diagonal blocks by forward
//     substitution in fp32 (two blocks per warp, one column per lane);
//  2. (invert_merge) recursive doubling: for L = [[L11, 0], [L21, L22]], L^-1 has off-diagonal block
//     -L22^-1 L21 L11^-1; first for the 16 x 16 pairs, then for the two 32 x 32 halves.
// Products run on f16 warp MMAs (m16n8k16, fp32 accumulation): the off-diagonal blocks are
// small next to the unit diagonal, so rounding their factors to fp16 (tf32's 10-bit
// significand) leaves T within about 1e-6 relative, far below the fp16
// rounding of the operands built from T. Only the lower triangle and the unit diagonal of
// T are written; blocks of T above the diagonal are never read.
// Step 1 of the inverse: one warp inverts diagonal blocks 2 pair and 2 pair + 1 (pair 0 or 1;
// lanes 0-15 the first block, 16-31 the second) while the other warps do independent work.
__device__ __forceinline__ void invert_diag_blocks(const float* A, float* T, int pair,
                                                   int lane) {
  const int o = 16 * (2 * pair + (lane >> 4)), j = lane & 15;
  float x[16];
  diag_block_column(A, o, j, x);
#pragma unroll
  for (int i = 0; i < 16; ++i) T[(o + i) * kLd + o + j] = x[i];
}

// Step 2 of the inverse (all warps), after the diagonal blocks are in T; it also writes the
// fp16 operands T1 = T diag(c1) and T2 = T diag(c2) (128B-swizzled 64 x 64 tiles, zero
// above the diagonal). T1 shares its shared memory with rows 0-30 of A, which the 16 -> 32
// level reads for the last time; T2 has a region of its own. So the blocks of T1/T2 that
// are final after that level are written while the products of the 32 -> 64 level run,
// and that level's last product goes straight from its accumulator into T1/T2. Ends
// before the tiles are published to the tensor cores.
__device__ void invert_merge(const float* A, float* T, float* X, uint8_t* T1, uint8_t* T2,
                             const float* c1, const float* c2, int tid) {
  const int warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  // 16 -> 32: T[16b+16.., 16b..] = -T22 (A21 T11) for b = 0, 2; warps 0-3, one 8-column slice
  if (warp < 4) {
    const int b = 2 * (warp >> 1), r0 = 16 * b + 16, n0 = 16 * b + 8 * (warp & 1);
    float* xs = X + warp * 16 * kLdXs;  // 16 x 8 scratch, row stride kLdXs
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mm(d, A, kLd, r0, T, kLd, n0, 16 * b, 16 * b + 16, gid, tig);
    tile_store(xs, kLdXs, 0, 0, d, 1.f, gid, tig);
    __syncwarp();
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mm(y, T + r0 * kLd + r0, kLd, 0, xs, kLdXs, 0, 0, 16, gid, tig);
    tile_store(T, kLd, r0, n0, y, -1.f, gid, tig);
  }
  __syncthreads();
  // 32 -> 64: X = A[32:64, 0:32] T[0:32, 0:32], then T[32:64, 0:32] = -T[32:64, 32:64] X;
  // eight 16 x 8 tiles, one per warp; zero blocks of the triangular factors are skipped
  const int mt = warp >> 2, nt = warp & 3;
  const int r0 = 16 * mt, n0 = 8 * nt;
  {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mm(d, A + 32 * kLd, kLd, r0, T, kLd, n0, nt >= 2 ? 16 : 0, 32, gid, tig);
    // while the warp MMAs run: the two diagonal 32 x 32 blocks of T1/T2, from T, and the
    // zero block above them. A thread takes 8 columns of one row of a diagonal block (warps
    // 0-3 the first, 4-7 the second) and one 16-byte chunk of zeros; the 8 lanes of each
    // quarter warp take 8 consecutive rows at the same columns, so that their float4 reads
    // of T fall on distinct banks and those of the column factors are broadcasts.
    {
      const int bk = warp >> 2, i = 32 * bk + 8 * (warp & 3) + (lane & 7);
      const int j0 = 32 * bk + 8 * (lane >> 3);
      float x1[8], x2[8];
#pragma unroll
      for (int q4 = 0; q4 < 8; q4 += 4) {
        const int j = j0 + q4;
        const float4 tv = *reinterpret_cast<const float4*>(T + i * kLd + j);
        const float4 gv = *reinterpret_cast<const float4*>(c1 + j);
        const float4 bv = *reinterpret_cast<const float4*>(c2 + j);
        const float t4[4] = {tv.x, tv.y, tv.z, tv.w}, g4[4] = {gv.x, gv.y, gv.z, gv.w},
                    b4[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int f = 0; f < 4; f += 2) {
          const float2 tij = make_float2(j + f <= i ? t4[f] : 0.f,  // zero above the diagonal
                                         j + f + 1 <= i ? t4[f + 1] : 0.f);
          const float2 y1 = mul2(tij, make_float2(g4[f], g4[f + 1]));
          const float2 y2 = mul2(tij, make_float2(b4[f], b4[f + 1]));
          x1[q4 + f] = y1.x;
          x1[q4 + f + 1] = y1.y;
          x2[q4 + f] = y2.x;
          x2[q4 + f + 1] = y2.y;
        }
      }
      st_chunk(T1, i, j0, 64, x1);
      st_chunk(T2, i, j0, 64, x2);
      // T1 (warps 0-3) or T2 (warps 4-7), rows 0-31, columns 32-63
      *reinterpret_cast<uint4*>((bk ? T2 : T1) + ptx::sw128_offset(i - 32 * bk, j0 + 32 - 32 * bk, 64)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    tile_store(X, kLdX, r0, n0, d, 1.f, gid, tig);
  }
  __syncthreads();
  {  // T[32:64, 0:32] = -T[32:64, 32:64] X straight into T1/T2
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mm(y, T + 32 * kLd + 32, kLd, r0, X, kLdX, n0, 0, mt == 0 ? 16 : 32, gid, tig);
    tile_store_t12(T1, T2, 32 + r0, n0, y, c1, c2, gid, tig);
  }
}

template <int kDh>  // the head dim d: 128, or 64 (zero-padded to 128)
__global__ void __launch_bounds__(kThreads, 2)
chunked_prefill_kernel(const __grid_constant__ ChunkedParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Smem sm;
  const PrefillArgs& p = P.a;
  uint8_t* sKQ = smem + OFF_KQ;
  uint8_t* sV = smem + OFF_V;
  uint8_t* sP = smem + OFF_P;
  float* sA = reinterpret_cast<float*>(smem + OFF_A);
  uint8_t* sT1 = smem + OFF_A;
  uint8_t* sT2 = smem + OFF_T2;
  uint8_t* sDp = smem + OFF_A;   // D' after the inverse and M3
  uint8_t* sO = smem + OFF_A;    // bf16 output staging [64][128] after M5
  float* sT = reinterpret_cast<float*>(smem + OFF_WD);
  uint8_t* sWD = smem + OFF_WD;
  float* sXs = reinterpret_cast<float*>(smem + OFF_XS);
  float* sG = reinterpret_cast<float*>(smem + OFF_VEC);  // log2-scaled cumulative log-decay
  float* sB = sG + 64;     // beta
  float* sGq = sG + 128;   // scale e^{G_t} / |q_t|: row factor of Q~
  float* sBG = sG + 192;   // beta_j e^{G_j} / |k_j|: column factor of T1
  float* sDec = sG + 256;  // e^{G_L - G_j} / |k_j|: row factor of D'
  float* sGp = sG + 320;   // G_j - log2(1/|k_j|): column exponent of A and P
  float* sRk = sG + 384;   // 1/|k_j|
  float* sRq = sG + 448;   // 1/|q_t|

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GdnUnit u = p.units[blockIdx.x];
  const GdnSeq sd = p.seqs[u.seq];
  constexpr int dh = kDh;
  if (sd.len <= 1) {  // a prompt of one token or none: the decode step's arithmetic
    float* sk = reinterpret_cast<float*>(smem);
    short_unit<kThreads, kDh>(p, u, sd, sk, sk + kD, tid);
    if (p.ckpt_ready) signal_ckpt_ready(p.ckpt_ready, u.seq, 0, kThreads, tid == 0);
    return;
  }
  const int h = u.head, hk = h / p.group;
  const size_t v_stride = (size_t)p.hv_heads * dh;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + (size_t)sd.tok_start * v_stride +
                      (size_t)h * dh;
  const float* ag = p.a + (size_t)sd.tok_start * p.hv_heads + h;
  const float* bg = p.beta + (size_t)sd.tok_start * p.hv_heads + h;
  const size_t state_off = state_offset<kDh>(p, sd, h);
  const float* init = initial_state<kDh>(p, sd, h);
  const int nchunks = (sd.len + kC - 1) / kC;  // >= 1: len >= 2 here

  if (tid == 0) {
    mbar_init(&sm.bar_mma, 1);
    mbar_init(&sm.bar_kq, 1);
    mbar_init(&sm.bar_v, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    if (nchunks > 0) {
      prefetch_tmap(&P.tq);
      prefetch_tmap(&P.tk);
      prefetch_tmap(&P.tv);
      if (!p.test_skip_first_copy) issue_kq(P, sKQ, &sm.bar_kq, hk, sd.tok_start, dh);
      if (!(sd.flags & kSeqZeroV)) issue_v(P, sV, &sm.bar_v, h, sd.tok_start, dh);
    }
  }
  if (dh == 64) {  // the second 64-column regions of q, k and v are never copied: zeros
    for (int i = tid; i < 1024; i += kThreads) {
      *reinterpret_cast<uint4*>(sKQ + 16384 + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
      if (i < 512) *reinterpret_cast<uint4*>(sV + 8192 + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, TM_COLS);
    tmem_relinquish();
  }
  // gate factors of chunk 0; the gate warp keeps the next chunk's gates in registers (every
  // later chunk's factors are written while the previous chunk's last products run)
  float gnext[4] = {0.f, 0.f, 0.f, 0.f};
  const bool raw = p.gate_mode == 1;
  const float a_log = raw ? __ldg(p.a_log + h) : 0.f;
  const float dt_bias = raw ? __ldg(p.dt_bias + h) : 0.f;
  const float scale = p.scale;
  if (warp == kGateWarp && nchunks > 0) {
    load_gates(ag, bg, p.hv_heads, 0, sd.len, lane, raw, a_log, dt_bias, gnext);
    const float d = write_gate_factors(Factors(sG), gnext, scale, lane);
    if (lane == 0) sm.next_decay = d;
    if (nchunks > 1) load_gates(ag, bg, p.hv_heads, kC, sd.len, lane, raw, a_log, dt_bias, gnext);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  const uint32_t sub = warp & 3, half = warp >> 2;
  const uint32_t row = 32 * sub + lane;  // TMEM lane = matrix row of this thread
  const uint32_t t_lane = tbase + ((32 * sub) << 16);

  // ---- initial state -> S32 (scaled by the first chunk's decay) and S16 ----------------
  {
    const float d0 = nchunks > 0 ? sm.next_decay : 1.f;
    // (rows and columns past d are zero)
    const float* src = init && (int)row < dh && 64 * (int)half < dh
                           ? init + (size_t)row * dh + 64 * half
                           : nullptr;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
      uint32_t r[16], h8[8];
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        const float4 v = src ? __ldg(reinterpret_cast<const float4*>(src + c0 + e))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        r[e] = __float_as_uint(v.x * d0); r[e + 1] = __float_as_uint(v.y * d0);
        r[e + 2] = __float_as_uint(v.z * d0); r[e + 3] = __float_as_uint(v.w * d0);
        h8[e / 2] = pack_half2(v.x, v.y);
        h8[e / 2 + 1] = pack_half2(v.z, v.w);
      }
      tmem_st16(t_lane + TM_S32 + 64 * half + c0, r);
      tmem_st8(t_lane + TM_S16 + 32 * half + c0 / 2, h8);
    }
    tmem_st_wait();
  }

  uint32_t ph_mma = 0, ph_kq = 0, ph_v = 0;
  bool ok = true;
  const bool vz = sd.flags & kSeqZeroV;  // v taken as zero: no v copies at all
  // copies and products in flight (meaningful in thread 0, which issues them)
  bool kq_inflight = nchunks > 0 && !p.test_skip_first_copy;
  bool v_inflight = nchunks > 0 && !vz, mma_inflight = false;
  bool store_pending = false;  // a TMA store of output rows still reading the staging tile
  int c_next = sd.ckpt_begin;
  // the next checkpoint's position (-1: none left), read again only after a checkpoint is
  // stored, so that no chunk waits on a global load to decide
  int ck_pos = c_next < sd.ckpt_end ? __ldg(p.ckpt_pos + c_next) : -1;
  bool signaled = false;  // the prompt's ready counter has this block's arrival

  for (int c = 0; c < nchunks && ok; ++c) {
    const int t0 = c * kC;
    const int L = min(kC, sd.len - t0);

    // ---- (2) wait for q, k, v; convert in place to fp16 (q, k normalised); zero past L ----
    if (!(ok = wait_copies(&sm.bar_kq, ph_kq, kq_inflight, &sm.bar_v, ph_v, v_inflight, !vz)))
      break;
    if (tid == 0 && c + 1 < nchunks) {  // warm L2 with the next chunk's q, k, v
      const int nrow = sd.tok_start + t0 + kC;
#pragma unroll
      for (int r = 0; r < dh / 64; ++r) {
        tma_prefetch_l2_2d(&P.tk, hk * dh + 64 * r, nrow);
        tma_prefetch_l2_2d(&P.tq, hk * dh + 64 * r, nrow);
        tma_prefetch_l2_2d(&P.tv, h * dh + 64 * r, nrow);
      }
    }
    convert_kq<16384>(sKQ, Factors(sG), L, p.l2norm != 0, tid);  // with the norms
    publish_operands();

    // ---- (3) M1: [K; Q] K^T -> R0 (128 x 64) ------------------------------------------------
    if (tid == 0) {
      const uint32_t idesc = idesc_f16(128, 64, 0, 0);
      const uint32_t a0 = smem_u32(sKQ);
#pragma unroll
      for (int s = 0; s < kD / 16; ++s) {
        const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
        mma_f16_ss(tbase + TM_R0, smem_desc_sw128(a0 + off, 16, 1024),
                   smem_desc_sw128(a0 + off, 16, 1024), idesc, s > 0);
      }
      mma_commit(&sm.bar_mma);
      mma_inflight = true;
    }
    __syncwarp();
    if (warp == 1) {  // fold the norms into the per-token factors
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = lane + 32 * hh;
        const float rk = sRk[i], rq = sRq[i];
        sGp[i] = sG[i] - __log2f(rk);  // +inf for padded tokens: their column terms vanish
        sXs[i] = col_factor(sGp[i]);    // (the merge scratch is idle until the inverse)
        sBG[i] *= rk;
        sDec[i] *= rk;
        sGq[i] *= rq;
      }
    }
    {  // V rows 0-63 while M1 runs (V is first read by M3)
      const int j = tid & 15, rsub = tid >> 4;
      const uint32_t reg = j >> 3, cc = j & 7;
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      uint4 w[4];
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        const uint32_t r = pass * 16 + rsub;
        w[pass] = *reinterpret_cast<const uint4*>(sV + reg * 8192 + (r >> 3) * 1024 +
                                                  (r & 7) * 128 + ((cc ^ (r & 7)) << 4));
      }
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        const uint32_t r = pass * 16 + rsub;
        *reinterpret_cast<uint4*>(sV + reg * 8192 + (r >> 3) * 1024 + (r & 7) * 128 +
                                  ((cc ^ (r & 7)) << 4)) =
            (int)r < L && !vz ? bf16x8_to_half8(w[pass]) : zero;
      }
    }
    // the previous chunk's output store must have read its staging tile (it shares shared
    // memory with A, written right after this barrier)
    if (tid == 0 && store_pending) {
      bulk_wait_read_all();
      store_pending = false;
    }
    if (!(ok = wait_all(&sm.bar_mma, ph_mma, mma_inflight))) break;

    // ---- (4) A (rows 0-63, fp32) and P (rows 64-127, fp16); Q~ = scale e^G Q / |q| over Q -
    // Warps whose 32 x 32 block lies above the diagonal (rows 0-31 of A or of P, columns
    // 32-63) compute nothing: that block of A is never read, that block of P is zero.
    if (half == 1 && (sub == 0 || sub == 2)) {
      if (sub == 2) {
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 32; e += 8) st_chunk(sP, row - 64, 32 + e, 64, z);
      }
    } else {
      uint32_t r[32];
      tmem_ld32(t_lane + TM_R0 + 32 * half, r);
      tmem_ld_wait();
      ap_row(r, row, 32 * half, Factors(sG), sXs, scale, sG[63] >= kFactoredMinLog2Decay, sA,
             sP);
    }
    tc_fence_before();

    // ---- (5) T = (I + A)^-1; T1 = T diag(beta e^G), T2 = T diag(beta) (fp16) -----------------
    // The diagonal 16 x 16 blocks of A lie in rows that the inverting warps have just written
    // themselves: warp 0 wrote rows 0-31, columns 0-31 (blocks 0 and 1) and warp 5 rows 32-63,
    // columns 32-63 (blocks 2 and 3). They invert them at once, without waiting for the other
    // warps, which scale Q~ meanwhile (M1 has consumed Q).
    if (warp == 0 || warp == 5) {
      __syncwarp();
      invert_diag_blocks(sA, sT, warp == 0 ? 0 : 1, lane);
    } else {
      const int rank = warp < 5 ? warp - 1 : warp - 2;  // 0-5 over warps 1-4, 6, 7
      for (int idx = 32 * rank + lane; idx < 1024; idx += kThreads - 64) {
        const uint32_t t = idx >> 4, j = idx & 15, rr = 64 + t;
        const uint32_t reg = j >> 3, cc = j & 7;
        uint4* ptr = reinterpret_cast<uint4*>(sKQ + reg * 16384 + (rr >> 3) * 1024 +
                                              (rr & 7) * 128 + ((cc ^ (rr & 7)) << 4));
        uint4 w = *ptr;
        const __half2 gm = __float2half2_rn(sGq[t]);
        uint32_t* u = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 y = __hmul2(*reinterpret_cast<const __half2*>(&u[e]), gm);
          u[e] = *reinterpret_cast<const uint32_t*>(&y);
        }
        *ptr = w;
      }
    }
    __syncthreads();
    invert_merge(sA, sT, sXs, sT1, sT2, sBG, sB, tid);
    publish_operands();

    // ---- (6) M2: W^T = K^T T1^T -> R0 (128 x 64) -----------------------------------------------
    if (tid == 0) {
      const uint32_t idesc = idesc_f16(128, 64, 1, 0);
      const uint32_t a0 = smem_u32(sKQ), b0 = smem_u32(sT1);
#pragma unroll
      for (int s = 0; s < kC / 16; ++s)
        mma_f16_ss(tbase + TM_R0, smem_desc_sw128(a0 + s * 2048, 16384, 1024),
                   smem_desc_sw128(b0 + s * 32, 16, 1024), idesc, s > 0);
      mma_commit(&sm.bar_mma);
      mma_inflight = true;
    }
    __syncwarp();
    if (!(ok = wait_all(&sm.bar_mma, ph_mma, mma_inflight))) break;

    // ---- (7) W^T -> smem (fp16, MN-major B: rows d_k, columns tokens) ---------------------------
    // Once every warp has read W^T out of R0, the first half of M3 (V^T T2^T, whose operands
    // were published before M2) starts into R0 while the warps store W^T.
    {
      uint32_t r[32];
      tmem_ld32(t_lane + TM_R0 + 32 * half, r);
      tmem_ld_wait();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
        const uint32_t id_u = idesc_f16(128, 64, 1, 0);
        const uint32_t v0 = smem_u32(sV), t2 = smem_u32(sT2);
#pragma unroll
        for (int s = 0; s < kC / 16; ++s)
          mma_f16_ss(tbase + TM_R0, smem_desc_sw128(v0 + s * 2048, 8192, 1024),
                     smem_desc_sw128(t2 + s * 32, 16, 1024), id_u, s > 0);
      }
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        float x[8];
#pragma unroll
        for (int f = 0; f < 8; ++f) x[f] = __uint_as_float(r[e + f]);
        st_chunk(sWD, row, 32 * half + e, 128, x);
      }
    }
    publish_operands();

    // ---- (8) M3: D^T = V^T T2^T - S16 W^T -> R0 (V^T T2^T already issued) ---------------------
    if (tid == 0) {
      const uint32_t id_w = idesc_f16(128, 64, 0, 1, 0, 1);  // B negated
      const uint32_t w0 = smem_u32(sWD);
#pragma unroll
      for (int s = 0; s < kD / 16; ++s)
        mma_f16_ts(tbase + TM_R0, tbase + TM_S16 + s * 8,
                   smem_desc_sw128(w0 + s * 2048, 16384, 1024), id_w, 1);
      mma_commit(&sm.bar_mma);
      mma_inflight = true;
    }
    __syncwarp();
    if (!(ok = wait_all(&sm.bar_mma, ph_mma, mma_inflight))) break;
    // V and T2 are consumed: fetch the next chunk's v now
    if (tid == 0 && c + 1 < nchunks && !vz) {
      issue_v(P, sV, &sm.bar_v, h, sd.tok_start + t0 + kC, dh);
      v_inflight = true;
    }

    // ---- (9) D^T and D'^T = D^T diag(e^{G_L - G}) -> smem (fp16 K-major A operands) -------------
    // Once every warp has read D^T out of R0, the first half of M4 (S16 Q~^T; Q~ was published
    // before M2) starts into R0 while the warps store D and D'.
    {
      uint32_t r[32];
      tmem_ld32(t_lane + TM_R0 + 32 * half, r);
      tmem_ld_wait();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
        const uint32_t id_n64 = idesc_f16(128, 64, 0, 0);
        const uint32_t kq = smem_u32(sKQ);
#pragma unroll
        for (int s = 0; s < kD / 16; ++s) {
          const uint32_t off = 8192 + (s >> 2) * 16384 + (s & 3) * 32;  // Q~ rows 64-127
          mma_f16_ts(tbase + TM_R0, tbase + TM_S16 + s * 8, smem_desc_sw128(kq + off, 16, 1024),
                     id_n64, s > 0);
        }
      }
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        const float4 da = *reinterpret_cast<const float4*>(sDec + 32 * half + e);
        const float4 db = *reinterpret_cast<const float4*>(sDec + 32 * half + e + 4);
        const float d8[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
        float x[8], y[8];
#pragma unroll
        for (int f = 0; f < 8; f += 2) {
          x[f] = __uint_as_float(r[e + f]);
          x[f + 1] = __uint_as_float(r[e + f + 1]);
          const float2 t = mul2(make_float2(x[f], x[f + 1]), make_float2(d8[f], d8[f + 1]));
          y[f] = t.x;
          y[f + 1] = t.y;
        }
        st_chunk(sWD, row, 32 * half + e, 128, x);
        st_chunk(sDp, row, 32 * half + e, 128, y);
      }
    }
    publish_operands();

    // ---- (10) O^T = S16 Q~^T + D^T P^T -> R0 (S16 Q~^T already issued);  S32 += D'^T K ------
    if (tid == 0) {
      const uint32_t id_n64 = idesc_f16(128, 64, 0, 0);
      const uint32_t kq = smem_u32(sKQ), d0 = smem_u32(sWD), p0 = smem_u32(sP);
#pragma unroll
      for (int s = 0; s < kC / 16; ++s)
        mma_f16_ss(tbase + TM_R0, smem_desc_sw128(d0 + s * 32, 16, 1024),
                   smem_desc_sw128(p0 + s * 32, 16, 1024), id_n64, 1);
      const uint32_t id_n128 = idesc_f16(128, 128, 0, 1);
      const uint32_t dp = smem_u32(sDp);
#pragma unroll
      for (int s = 0; s < kC / 16; ++s)
        mma_f16_ss(tbase + TM_S32, smem_desc_sw128(dp + s * 32, 16, 1024),
                   smem_desc_sw128(kq + s * 2048, 16384, 1024), id_n128, 1);
      mma_commit(&sm.bar_mma);
      mma_inflight = true;
    }
    __syncwarp();
    // while the products run: the next chunk's gate factors (every read of this chunk's
    // factors is behind the barrier above) and its total decay for the state pre-scale;
    // then the gates of the chunk after it
    if (warp == kGateWarp && c + 1 < nchunks) {
      const float d = write_gate_factors(Factors(sG), gnext, scale, lane);
      if (lane == 0) sm.next_decay = d;
      if (c + 2 < nchunks)
        load_gates(ag, bg, p.hv_heads, t0 + 2 * kC, sd.len, lane, raw, a_log, dt_bias, gnext);
    }
    if (!(ok = wait_all(&sm.bar_mma, ph_mma, mma_inflight))) break;
    // q and k are consumed: fetch the next chunk's
    if (tid == 0 && c + 1 < nchunks) {
      issue_kq(P, sKQ, &sm.bar_kq, hk, sd.tok_start + t0 + kC, dh);
      kq_inflight = true;
    }

    // ---- (11) o via smem staging; S16 refresh; checkpoints; pre-scale S32 for the next chunk --
    {
      uint32_t r[32];
      tmem_ld32(t_lane + TM_R0 + 32 * half, r);
      tmem_ld_wait();
      // lanes 2m and 2m+1 hold value rows dv, dv+1: swap so that each lane owns one
      // (dv, dv+1) pair of a token and stores it as one bf16x2 word
      const bool odd = lane & 1;
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const float mine_lo = __uint_as_float(r[e]), mine_hi = __uint_as_float(r[e + 1]);
        const float other = __shfl_xor_sync(0xffffffffu, odd ? mine_lo : mine_hi, 1);
        const int t = 32 * half + e + (odd ? 1 : 0);
        const __nv_bfloat162 pr = odd ? __floats2bfloat162_rn(other, mine_hi)
                                      : __floats2bfloat162_rn(mine_lo, other);
        *reinterpret_cast<__nv_bfloat162*>(sO + t * 256 + (row & ~1u) * 2) = pr;
      }

      const int pos = t0 + L;
      const bool emit = ck_pos == pos;
      const bool last = c + 1 == nchunks;
      const float nd = last ? 1.f : sm.next_decay;
      // (only the d x d state is stored: rows and columns past d are zero)
      const bool store_row = (int)row < dh;
      float* ck = emit && store_row
                      ? p.ckpt + ((size_t)c_next * p.hv_heads + h) * dh * dh + (size_t)row * dh
                      : nullptr;
      float* fin = last && store_row ? p.final_state + state_off + (size_t)row * dh : nullptr;
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
        const bool store_col = col < dh;
        if (ck && store_col) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<uint4*>(ck + col + e) =
                make_uint4(s32[e], s32[e + 1], s32[e + 2], s32[e + 3]);
        }
        if (last) {
          if (fin && store_col) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<uint4*>(fin + col + e) =
                  make_uint4(s32[e], s32[e + 1], s32[e + 2], s32[e + 3]);
          }
        } else {
          uint32_t lo[16], hi[16];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float2 a = mul2(make_float2(__uint_as_float(s32[e]), __uint_as_float(s32[e + 1])),
                                  make_float2(nd, nd));
            const float2 b = mul2(
                make_float2(__uint_as_float(s32[16 + e]), __uint_as_float(s32[17 + e])),
                make_float2(nd, nd));
            lo[e] = __float_as_uint(a.x);
            lo[e + 1] = __float_as_uint(a.y);
            hi[e] = __float_as_uint(b.x);
            hi[e + 1] = __float_as_uint(b.y);
          }
          tmem_st16(t_lane + TM_S32 + 64 * half + c0, lo);
          tmem_st16(t_lane + TM_S32 + 64 * half + c0 + 16, hi);
        }
      }
      if (emit) {
        ++c_next;
        ck_pos = c_next < sd.ckpt_end ? __ldg(p.ckpt_pos + c_next) : -1;
      }
      tmem_st_wait();
      const bool tma_out = L == kC && dh == kD;  // whole d = 128 chunks leave by TMA
      if (tma_out) fence_proxy_async_smem();
      if (p.ckpt_ready && emit && c_next == sd.ckpt_end) {
        // the unit's last checkpoint is stored: its copy may start (the barrier inside also
        // orders the staging writes before the store below)
        signal_ckpt_ready(p.ckpt_ready, u.seq, 0, kThreads, tid == 0);
        signaled = true;
      } else {
        __syncthreads();
      }
      if (tma_out) {
        // a whole chunk lies inside the prompt: one TMA store of the 64 x 128 tile
        if (tid == 0) {
          tma_store_2d(&P.to, sO, h * kD, sd.tok_start + t0);
          bulk_commit();
          store_pending = true;
        }
      } else {
        // the tail chunk (a whole box would reach the next prompt's rows), or d = 64: only
        // its L rows and d columns, by coalesced 16-byte stores
        const int pieces = dh / 8;  // 16-byte pieces of an output row
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int idx = it * kThreads + tid, t = idx / pieces, ch = idx % pieces;
          if (t < L && idx < kC * pieces)
            *reinterpret_cast<uint4*>(og + (size_t)(t0 + t) * v_stride + ch * 8) =
                *reinterpret_cast<const uint4*>(sO + t * 256 + ch * 16);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (!ok) {
    if (tid == 0 && p.status) atomicExch(p.status, kStatusTimeout);
    // let products and copies still in flight land (bounded) before TMEM and shared
    // memory are released: thread 0 knows what it has outstanding and the parity of each
    // pending phase
    if (tid == 0) {
      if (mma_inflight) mbar_wait_bounded(&sm.bar_mma, ph_mma & 1u, kWaitLimit);
      if (kq_inflight) mbar_wait_bounded(&sm.bar_kq, ph_kq & 1u, kWaitLimit);
      if (v_inflight) mbar_wait_bounded(&sm.bar_v, ph_v & 1u, kWaitLimit);
    }
  }
  if (tid == 0 && store_pending) bulk_wait_all();  // output stores done before the CTA exits
  // a unit without checkpoints, or one that gave up before its last, arrives here
  if (p.ckpt_ready && !signaled) signal_ckpt_ready(p.ckpt_ready, u.seq, 0, kThreads, tid == 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

int launch_chunked_throughput(const PrefillArgs& a, int64_t total_tokens, void* stream) {
  if (a.num_units == 0) return 0;
  static std::atomic<int> configured[kMaxDevices];
  const int ce = configure_once(configured, [] {
    for (const void* k : {(const void*)chunked_prefill_kernel<128>,
                          (const void*)chunked_prefill_kernel<64>}) {
      const cudaError_t e =
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
      if (e != cudaSuccess) return (int)e;
    }
    return 0;
  });
  if (ce != 0) return ce;
  ChunkedParams P;
  P.a = a;
  if (!make_qkv_maps(a, total_tokens, a.head_dim, &P.tq, &P.tk, &P.tv) ||
      !make_out_map(&P.to, a.o, (uint64_t)a.hv_heads * a.head_dim,
                    a.head_dim == kD ? (uint64_t)total_tokens : 0))
    return (int)cudaErrorInvalidValue;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (a.head_dim == 64)
    chunked_prefill_kernel<64><<<a.num_units, kThreads, SMEM_BYTES, st>>>(P);
  else
    chunked_prefill_kernel<128><<<a.num_units, kThreads, SMEM_BYTES, st>>>(P);
  return (int)cudaGetLastError();
}

}  // namespace gdn
