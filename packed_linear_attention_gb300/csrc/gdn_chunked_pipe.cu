// gdn_chunked_pipe.cu — chunked gated-delta-rule prefill on the tcgen05 tensor cores
// (sm_103a), pipelined schedule.
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
// Schedule: one CTA of 16 warps per unit, one CTA per SM, two warp groups in a pipeline.
//   * prep group (warps 0-7): everything of chunk c that does not depend on the state:
//     q/k/v to fp16 and the norms, [K;Q]K^T, A and P, the inverse, T1/T2, W^T and U^T.
//   * chain group (warps 8-15): the recurrence of chunk c-1 meanwhile: D^T = U^T - S W^T,
//     D and D', S += D'^T K, O^T = S Q~^T + D^T P^T, the fp16 state refresh, checkpoints
//     and the output rows.
// Operands pass from prep to chain through double-buffered tiles (q/k/w and P in shared
// memory; U^T in TMEM) and one mbarrier per buffer. The chain issues the next chunk's q/k
// copy into a buffer once its last product has read it, which also tells the prep group
// that the buffer's P, W, U and gate factors are free again.
//   TMEM (512 columns): [0,128) S32 fp32 state; [128,192) S16 fp16 copy (A operand);
//   [192,256) the prep group's product; [256,512) two blocks [O^T | U^T], one per buffer:
//   the chain's single product S16 [Q~; -W]^T starts O^T and turns U^T into D^T.
// Results are bit-identical to the throughput schedule's (gdn_chunked.cu): both round every
// value the same way, with the code they share in gdn_chunk_util.cuh.
// Every mbarrier wait is bounded (a poll count and about one second) and gives up early
// once the other group has; a timeout is reported through the status word and every copy
// and product still in flight is waited for (bounded) before TMEM is released.
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

constexpr int kGroup = 256;     // threads per warp group
constexpr int kThreads = 2 * kGroup;
constexpr uint32_t kBarPrep = 1, kBarChain = 2;  // named barriers of the two groups

// shared-memory map (bytes from a 1024-aligned base)
// q/k/w tile, 2 buffers x 48 KB: two 24 KB regions (64 columns of d each) holding rows
// 0-63 K, 64-127 Q (then Q~), 128-191 -W (K-major), so that [Q~; -W] is one 128-row operand
constexpr uint32_t kRegion = 24576, kKQW = 2 * kRegion;
constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t OFF_V = OFF_KQ + 2 * kKQW;  // V: 2 regions x 8 KB
constexpr uint32_t OFF_P = OFF_V + 16384;      // 2 buffers x P (64 x 64 fp16)
constexpr uint32_t OFF_D = OFF_P + 16384;      // D^T (fp16) -> bf16 output staging [64][128]
static_assert(OFF_D == 131072, "shared-memory map");
constexpr uint32_t OFF_DP = 147456;     // D'^T (fp16)
constexpr uint32_t OFF_A = 163840;      // A fp32 [64][68]
constexpr uint32_t OFF_T = OFF_A + 17408;   // T fp32 [64][68]
constexpr uint32_t OFF_XS = OFF_T + 17408;  // inverse scratch: 32 x kLdX fp32 (5 KB)
constexpr uint32_t OFF_VEC = OFF_XS + 5120;  // 2 buffers x per-token factors (8 x 64 fp32)
constexpr uint32_t OFF_T12 = OFF_VEC + 4096;  // T1 | T2 (fp16 64 x 64); blocks above the diagonal stay 0
constexpr uint32_t SMEM_USED = OFF_T12 + 16384;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack

// TMEM columns: S32 fp32 state, S16 its fp16 copy, the prep group's product, and per buffer b
// the block [O^T | U^T -> D^T] at TM_OU + 128 b, filled by one product S16 [Q~; -W]^T
constexpr uint32_t TM_S32 = 0, TM_S16 = 128, TM_M = 192, TM_OU = 256, TM_COLS = 512;
constexpr uint32_t KQ_BYTES = 32768, V_BYTES = 16384;

// mbarriers, by index
// (B_FLUSH_*: each group leader's final commit, which drains every product it issued)
// (B_CONV*, B_VCONV: the chain group has staged a chunk's q, k and gate factors / its v;
// plain arrivals)
enum : int { B_KQ0, B_KQ1, B_V, B_M1, B_M2, B_READY0, B_READY1, B_D, B_S, B_O, B_FLUSH_P,
             B_FLUSH_C, B_CONV0, B_CONV1, B_VCONV, B_COUNT };

struct ChunkedParams {
  PrefillArgs a;
  CUtensorMap tq, tk, tv;  // 2D bf16 maps: (H*128 columns, T rows), 64 x 64 boxes, SW128
  CUtensorMap to;          // o: (H_v*128 columns, T rows), 64-row x 128-column boxes, no swizzle
};

struct __align__(8) Smem {
  uint64_t bar[B_COUNT];
  uint32_t issued[B_COUNT];   // completions requested (copies and commits), per barrier
  uint32_t waited[B_COUNT];   // completions observed, per barrier
  uint32_t tmem_base;
  volatile int abort;         // set by a group that gave up
  float gamma[2];             // e^{G_L} of the chunk staged in factor buffer b
};

// Waits (every thread of a group) for phase `parity` of mbarrier `i`; gives up after the
// poll or time limit or once the other group has given up. The answer is made uniform
// across the group, and one thread records the observed completion.
__device__ __forceinline__ bool group_wait(Smem& sm, int i, uint32_t parity, uint32_t bar_id,
                                           bool leader, bool extra_fail = false) {
  bool ok = false;
  WaitClock clk;
  for (uint32_t n = 0; n < kWaitLimit; ++n) {
    if (mbar_try_wait(&sm.bar[i], parity)) {
      ok = true;
      break;
    }
    if ((n & 63u) == 63u && sm.abort) break;
    if (clk.expired(n)) break;
  }
  tc_fence_after();
  const bool fail = named_any(bar_id, kGroup, !ok || extra_fail);
  if (ok && leader) ++sm.waited[i];
  return !fail;
}

// Single-thread bounded wait (used by a group leader before it issues products).
__device__ __forceinline__ bool leader_wait(Smem& sm, int i, uint32_t parity) {
  WaitClock clk;
  for (uint32_t n = 0; n < kWaitLimit; ++n) {
    if (mbar_try_wait(&sm.bar[i], parity)) {
      tc_fence_after();
      return true;
    }
    if ((n & 63u) == 63u && sm.abort) break;
    if (clk.expired(n)) break;
  }
  return false;
}

// Makes a group's generic-proxy smem writes and TMEM stores visible to its next MMA issue.
__device__ __forceinline__ void publish(uint32_t bar_id) {
  fence_proxy_async_smem();
  tc_fence_before();
  named_sync(bar_id, kGroup);
  tc_fence_after();
}

// TMA loads of one chunk: q and k (4 boxes, one barrier) or v (2 boxes).
// (one region of 64 columns per 64 columns of d: dh = 64 or 128)
__device__ __forceinline__ void issue_kq(const ChunkedParams& P, Smem& sm, uint8_t* sKQ, int b,
                                         int hk, int row, int dh) {
  uint64_t* bar = &sm.bar[B_KQ0 + b];
  ++sm.issued[B_KQ0 + b];
  mbar_arrive_expect_tx(bar, KQ_BYTES / (kD / dh));
  for (int r = 0; r < dh / 64; ++r) {
    tma_load_2d(sKQ + r * kRegion, &P.tk, hk * dh + 64 * r, row, bar);
    tma_load_2d(sKQ + r * kRegion + 8192, &P.tq, hk * dh + 64 * r, row, bar);
  }
}
__device__ __forceinline__ void issue_v(const ChunkedParams& P, Smem& sm, uint8_t* sV, int h,
                                        int row, int dh) {
  uint64_t* bar = &sm.bar[B_V];
  ++sm.issued[B_V];
  mbar_arrive_expect_tx(bar, V_BYTES / (kD / dh));
  for (int r = 0; r < dh / 64; ++r) tma_load_2d(sV + r * 8192, &P.tv, h * dh + 64 * r, row, bar);
}
__device__ __forceinline__ void commit(Smem& sm, int i) {
  ++sm.issued[i];
  mma_commit(&sm.bar[i]);
}


// (I + A)^-1 for a 64 x 64 strictly-lower A (fp32, row stride kLd) into T (same stride):
//  1. (invert_diag_blocks) the four 16 x 16 diagonal blocks by forward
//     substitution in fp32 (two blocks per warp, one column per lane);
//  2. (invert_merge) recursive doubling: for L = [[L11, 0], [L21, L22]], L^-1 has
//     off-diagonal block -L22^-1 L21 L11^-1; first for the 16 x 16 pairs, then for the two
//     32 x 32 halves.
// Products run on f16 warp MMAs (m16n8k16, fp32 accumulation): the off-diagonal blocks are
// small next to the unit diagonal, so rounding their factors to fp16 (tf32's 10-bit
// significand) leaves T within about 1e-6 relative, far below the fp16
// rounding of the operands built from T. Only the lower triangle and the unit diagonal of
// T are written; blocks of T above the diagonal are never read.
// T is also written into the fp16 operands T1 = T diag(c1) and T2 = T diag(c2) (column
// factors c1, c2; 128B-swizzled 64 x 64 tiles whose blocks above the diagonal are zero):
// the two diagonal 32 x 32 blocks by every prep warp once the first level is done, the
// block below them straight from the last product's accumulator.
// Step 1: one prep warp inverts diagonal blocks 2 pair and 2 pair + 1 (pair 0 or 1; lanes
// 0-15 the first block, 16-31 the second) while the other prep warps do independent work.
__device__ __forceinline__ void invert_diag_blocks(const float* A, float* T, int pair,
                                                   int lane) {
  const int o = 16 * (2 * pair + (lane >> 4)), j = lane & 15;
  float x[16];
  diag_block_column_rl(A, o, j, x);
#pragma unroll
  for (int i = 0; i < 16; ++i) T[(o + i) * kLd + o + j] = x[i];
}

// Step 2 (all prep warps), after the diagonal blocks are in T. Ends with T1/T2 published
// to the tensor cores.
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
  named_sync(kBarPrep, kGroup);
  // 32 -> 64: X = A[32:64, 0:32] T[0:32, 0:32], then T[32:64, 0:32] = -T[32:64, 32:64] X;
  // eight 16 x 8 tiles, one per warp; zero blocks of the triangular factors are skipped
  {
    const int mt = warp >> 2, nt = warp & 3;
    const int r0 = 16 * mt, n0 = 8 * nt;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mm(d, A + 32 * kLd, kLd, r0, T, kLd, n0, nt >= 2 ? 16 : 0, 32, gid, tig);
    // while the warp MMAs run: the two diagonal 32 x 32 blocks of T1/T2, final after the
    // first level. A thread takes 8 columns of one row (warps 0-3 the first block, 4-7 the
    // second); the 8 lanes of each quarter warp take 8 consecutive rows at the same
    // columns, so that their float4 reads of T fall on distinct banks.
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
    }
    tile_store(X, kLdX, r0, n0, d, 1.f, gid, tig);
  }
  named_sync(kBarPrep, kGroup);
  {
    const int mt = warp >> 2, nt = warp & 3;
    const int r0 = 16 * mt, n0 = 8 * nt;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mm(y, T + 32 * kLd + 32, kLd, r0, X, kLdX, n0, 0, mt == 0 ? 16 : 32, gid, tig);
    tile_store_t12(T1, T2, 32 + r0, n0, y, c1, c2, gid, tig);
  }
  fence_proxy_async_smem();
  named_sync(kBarPrep, kGroup);
}

// v of one chunk to fp16 in place (exact); rows past the chunk's L tokens are zeroed. One
// warp group (gtid 0-255).
__device__ __forceinline__ void convert_v(uint8_t* sV, int L, int gtid) {
  const int j = gtid & 15, rsub = gtid >> 4;
  const uint32_t reg = j >> 3, cc = j & 7;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 w[4];
#pragma unroll
  for (int pass = 0; pass < 4; ++pass) {
    const uint32_t r = pass * 16 + rsub;
    w[pass] = *reinterpret_cast<const uint4*>(sV + reg * 8192 + (r >> 3) * 1024 + (r & 7) * 128 +
                                              ((cc ^ (r & 7)) << 4));
  }
#pragma unroll
  for (int pass = 0; pass < 4; ++pass) {
    const uint32_t r = pass * 16 + rsub;
    *reinterpret_cast<uint4*>(sV + reg * 8192 + (r >> 3) * 1024 + (r & 7) * 128 +
                              ((cc ^ (r & 7)) << 4)) = (int)r < L ? bf16x8_to_half8(w[pass]) : zero;
  }
}

template <int kDh>  // the head dim d: 128, or 64 (zero-padded to 128)
__global__ void __launch_bounds__(kThreads, 1)
chunked_pipe_kernel(const __grid_constant__ ChunkedParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Smem sm;
  const PrefillArgs& p = P.a;
  uint8_t* sV = smem + OFF_V;
  uint8_t* sD = smem + OFF_D;
  uint8_t* sDp = smem + OFF_DP;
  uint8_t* sO = smem + OFF_D;  // bf16 output staging [64][128] once D is consumed
  float* sA = reinterpret_cast<float*>(smem + OFF_A);
  uint8_t* sT1 = smem + OFF_T12;
  uint8_t* sT2 = smem + OFF_T12 + 8192;
  float* sT = reinterpret_cast<float*>(smem + OFF_T);
  float* sXs = reinterpret_cast<float*>(smem + OFF_XS);

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
  const float* ag = p.a + (size_t)sd.tok_start * p.hv_heads + h;
  const float* bg = p.beta + (size_t)sd.tok_start * p.hv_heads + h;
  const size_t state_off = state_offset<kDh>(p, sd, h);
  const float* init = initial_state<kDh>(p, sd, h);
  const int nchunks = (sd.len + kC - 1) / kC;  // >= 1: len >= 2 here
  const bool raw = p.gate_mode == 1;
  const float a_log = raw ? __ldg(p.a_log + h) : 0.f;
  const float dt_bias = raw ? __ldg(p.dt_bias + h) : 0.f;
  const float scale = p.scale;

  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < B_COUNT; ++i) {
      mbar_init(&sm.bar[i], 1);
      sm.issued[i] = 0;
      sm.waited[i] = 0;
    }
    sm.abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    if (nchunks > 0) {
      prefetch_tmap(&P.tq);
      prefetch_tmap(&P.tk);
      prefetch_tmap(&P.tv);
      if (!p.test_skip_first_copy) issue_kq(P, sm, smem + OFF_KQ, 0, hk, sd.tok_start, dh);
      if (!(sd.flags & kSeqZeroV)) issue_v(P, sm, sV, h, sd.tok_start, dh);
      if (nchunks > 1) issue_kq(P, sm, smem + OFF_KQ + kKQW, 1, hk, sd.tok_start + kC, dh);
    }
  }
  if (dh == 64) {  // the second 64-column regions of q, k (both buffers) and v: zeros
    for (int i = tid; i < 1024; i += kThreads) {
      *reinterpret_cast<uint4*>(smem + OFF_KQ + kRegion + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + OFF_KQ + kKQW + kRegion + 16 * i) =
          make_uint4(0u, 0u, 0u, 0u);
      if (i < 512) *reinterpret_cast<uint4*>(sV + 8192 + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, TM_COLS);
    tmem_relinquish();
  }
  for (int i = tid; i < 1024; i += kThreads)  // T1/T2 above the diagonal are never written
    reinterpret_cast<uint4*>(sT1)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  const uint32_t sub = warp & 3, half = (warp >> 2) & 1;
  const uint32_t row = 32 * sub + lane;  // TMEM lane = matrix row of this thread
  const uint32_t t_lane = tbase + ((32 * sub) << 16);
  // Shared-memory descriptors with start address 0 for the three tile layouts in use
  // (K-major: LBO 16 B; MN-major with q/k/w or 8 KB regions); a tile's descriptor is the
  // base plus its address / 16, which keeps the per-product issue cost to one add.
  const uint64_t dsc_k = smem_desc_sw128(0, 16, 1024);
  const uint64_t dsc_mnr = smem_desc_sw128(0, kRegion, 1024);
  const uint64_t dsc_mn8 = smem_desc_sw128(0, 8192, 1024);

  if (warp < 8) {
    // =================================== prep group ===================================
    const bool leader = tid == 0;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int b = c & 1, t0 = c * kC, L = min(kC, sd.len - t0);
      uint8_t* sKQ = smem + OFF_KQ + b * kKQW;
      uint8_t* sP = smem + OFF_P + b * 8192;
      const Factors f(reinterpret_cast<float*>(smem + OFF_VEC + b * 2048));

      // ---- (1) this chunk's q, k and gate factors, staged by the chain group (which frees
      // buffer b's P, W, U and factors first)
      if (!(ok = group_wait(sm, B_CONV0 + b, (c >> 1) & 1, kBarPrep, leader))) break;
      if (leader && c + 2 < nchunks) {  // warm L2 two chunks ahead
        const int nrow = sd.tok_start + t0 + 2 * kC;
#pragma unroll
        for (int r = 0; r < dh / 64; ++r) {
          tma_prefetch_l2_2d(&P.tk, hk * dh + 64 * r, nrow);
          tma_prefetch_l2_2d(&P.tq, hk * dh + 64 * r, nrow);
          tma_prefetch_l2_2d(&P.tv, h * dh + 64 * r, nrow);
        }
      }

      // ---- (4) M1: [K; Q] K^T -> TM_M (128 x 64) --------------------------------------------
      if (leader) {
        const uint32_t idesc = idesc_f16(128, 64, 0, 0);
        const uint64_t a0 = dsc_k + (smem_u32(sKQ) >> 4);
#pragma unroll
        for (int s = 0; s < kD / 16; ++s) {
          const uint64_t d = a0 + (((s >> 2) * kRegion + (s & 3) * 32) >> 4);
          mma_f16_ss(tbase + TM_M, d, d, idesc, s > 0);
        }
        commit(sm, B_M1);
      }
      __syncwarp();
      if (warp == 1) {  // fold the norms into the per-token factors
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = lane + 32 * hh;
          const float rk = f.Rk[i], rq = f.Rq[i];
          f.Gp[i] = f.G[i] - __log2f(rk);  // +inf for padded tokens: their column terms vanish
          sXs[i] = col_factor(f.Gp[i]);   // (the merge scratch is idle until the inverse)
          f.BG[i] *= rk;
          f.Dec[i] *= rk;
          f.Gq[i] *= rq;
        }
      }
      if (!(ok = group_wait(sm, B_M1, c & 1, kBarPrep, leader))) break;

      // ---- (5) A (rows 0-63, fp32) and P (rows 64-127, fp16) ----------------------------------
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
        tmem_ld32(t_lane + TM_M + 32 * half, r);
        tmem_ld_wait();
        ap_row(r, row, 32 * half, f, sXs, scale, f.G[63] >= kFactoredMinLog2Decay, sA, sP);
      }
      tc_fence_before();

      // ---- (6) T = (I + A)^-1; Q~ = scale e^G Q / |q| over Q meanwhile ------------------------
      // The diagonal 16 x 16 blocks of A lie in rows that the inverting warps have just
      // written themselves (warp 0: rows and columns 0-31, blocks 0 and 1; warp 5: rows and
      // columns 32-63, blocks 2 and 3), so they start without waiting for the other warps.
      if (warp == 0 || warp == 5) {
        __syncwarp();
        invert_diag_blocks(sA, sT, warp == 0 ? 0 : 1, lane);
      } else {  // M1 has consumed Q
        const int rank = warp < 5 ? warp - 1 : warp - 2;  // 0-5 over warps 1-4, 6, 7
        for (int idx = 32 * rank + lane; idx < 1024; idx += kGroup - 64) {
          const uint32_t t = idx >> 4, j = idx & 15, rr = 64 + t;
          const uint32_t reg = j >> 3, cc = j & 7;
          uint4* ptr = reinterpret_cast<uint4*>(sKQ + reg * kRegion + (rr >> 3) * 1024 +
                                                (rr & 7) * 128 + ((cc ^ (rr & 7)) << 4));
          uint4 w = *ptr;
          const __half2 gm = __float2half2_rn(f.Gq[t]);
          uint32_t* uu = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 y = __hmul2(*reinterpret_cast<const __half2*>(&uu[e]), gm);
            uu[e] = *reinterpret_cast<const uint32_t*>(&y);
          }
          *ptr = w;
        }
      }
      named_sync(kBarPrep, kGroup);
      invert_merge(sA, sT, sXs, sT1, sT2, f.BG, f.B, tid);
      tc_fence_after();

      // ---- (7) M2: W^T = K^T T1^T -> TM_M;  U^T = V^T T2^T -> U^T of block b -------------------
      if (!(ok = group_wait(sm, B_VCONV, c & 1, kBarPrep, leader))) break;  // v staged
      if (leader) {
        const uint32_t idesc = idesc_f16(128, 64, 1, 0);
        const uint64_t k0 = dsc_mnr + (smem_u32(sKQ) >> 4), t1 = dsc_k + (smem_u32(sT1) >> 4),
                       v0 = dsc_mn8 + (smem_u32(sV) >> 4), t2 = dsc_k + (smem_u32(sT2) >> 4);
#pragma unroll
        for (int s = 0; s < kC / 16; ++s)
          mma_f16_ss(tbase + TM_M, k0 + s * 128, t1 + s * 2, idesc, s > 0);
#pragma unroll
        for (int s = 0; s < kC / 16; ++s)
          mma_f16_ss(tbase + TM_OU + 128 * b + 64, v0 + s * 128, t2 + s * 2, idesc, s > 0);
        commit(sm, B_M2);
      }
      __syncwarp();
      if (!(ok = group_wait(sm, B_M2, c & 1, kBarPrep, leader))) break;
      // V is consumed: fetch the next chunk's
      if (leader && c + 1 < nchunks && !(sd.flags & kSeqZeroV))
        issue_v(P, sm, sV, h, sd.tok_start + t0 + kC, dh);

      // ---- (8) -W -> rows 128-191 of the q/k/w tile (fp16, K-major: rows tokens); hand over ---
      {
        uint32_t r[32];
        tmem_ld32(t_lane + TM_M + 32 * half, r);
        tmem_ld_wait();
        // lanes 2m and 2m+1 hold d_k rows i0, i0+1: swap so that each lane writes one
        // (i0, i0+1) pair of one token as a half2 word
        const bool odd = lane & 1;
        const uint32_t i0 = row & ~1u;
        uint8_t* base = sKQ + (i0 >> 6) * kRegion;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float lo = __uint_as_float(r[e]), hi = __uint_as_float(r[e + 1]);
          const float other = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
          const uint32_t t = 32 * half + e + (odd ? 1 : 0);
          *reinterpret_cast<uint32_t*>(base + sw128_offset(128 + t, i0 & 63, 192)) =
              odd ? pack_half2(-other, -hi) : pack_half2(-lo, -other);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(kBarPrep, kGroup);
      if (leader) mbar_arrive(&sm.bar[B_READY0 + b]);
    }
    if (!ok) sm.abort = 1;
    if (leader) {
      mma_commit(&sm.bar[B_FLUSH_P]);
      mbar_wait_bounded(&sm.bar[B_FLUSH_P], 0, kWaitLimit);
    }
  } else {
    // =================================== chain group ==================================
    const int ctid = tid - kGroup;
    const bool leader = ctid == 0;
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + (size_t)sd.tok_start * v_stride +
                        (size_t)h * dh;
    constexpr int kGateWarp = 15;  // writes every chunk's gate factors, two chunks ahead
    float gnext[4] = {0.f, 0.f, 0.f, 0.f};  // its raw gate loads of the next chunk to stage
    if (warp == kGateWarp && nchunks > 0) fetch_gates(ag, bg, p.hv_heads, 0, sd.len, lane, gnext);
    bool ok = true, lead_fail = false;
    bool store_pending = false;  // (leader) a TMA store of output rows still reading sO
    bool signaled = false;       // the prompt's ready counter has this block's arrival

    // Gate factors of chunk cc into factor buffer cc & 1 and its total decay into
    // sm.gamma[cc & 1] (gate warp only; published by the next stage_chunk(cc)).
    auto stage_gates = [&](int cc) {
      float g[4];
      gates_of(gnext, cc * kC, sd.len, lane, raw, a_log, dt_bias, g);
      if (cc + 1 < nchunks) fetch_gates(ag, bg, p.hv_heads, (cc + 1) * kC, sd.len, lane, gnext);
      const float gl = write_gate_factors(
          Factors(reinterpret_cast<float*>(smem + OFF_VEC + (cc & 1) * 2048)), g, scale, lane);
      if (lane == 0) sm.gamma[cc & 1] = gl;
    };
    // Stages chunk cc for the prep group in buffer cc & 1: q, k to fp16 with their norms; the
    // arrival also publishes the chunk's gate factors (stage_gates(cc) ran before).
    auto stage_chunk = [&](int cc) -> bool {
      const int bb = cc & 1;
      if (!group_wait(sm, B_KQ0 + bb, (cc >> 1) & 1, kBarChain, leader)) return false;
      const Factors fb(reinterpret_cast<float*>(smem + OFF_VEC + bb * 2048));
      convert_kq<kRegion>(smem + OFF_KQ + bb * kKQW, fb, min(kC, sd.len - cc * kC),
                          p.l2norm != 0, ctid);
      fence_proxy_async_smem();
      named_sync(kBarChain, kGroup);
      if (leader) mbar_arrive(&sm.bar[B_CONV0 + bb]);
      return true;
    };
    // Stages chunk cc's v (copied by the prep group once the previous v was consumed).
    // (v taken as zero: the tile is zeroed once and never copied into)
    auto stage_v = [&](int cc) -> bool {
      if (!(sd.flags & kSeqZeroV)) {
        if (!group_wait(sm, B_V, cc & 1, kBarChain, leader)) return false;
        convert_v(sV, min(kC, sd.len - cc * kC), ctid);
      } else if (cc == 0) {
        for (int i = ctid; i < 1024; i += kGroup)
          reinterpret_cast<uint4*>(sV)[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      named_sync(kBarChain, kGroup);
      if (leader) mbar_arrive(&sm.bar[B_VCONV]);
      return true;
    };
    if (warp == kGateWarp) {
      if (nchunks > 0) stage_gates(0);
      if (nchunks > 1) stage_gates(1);
    }
    if (nchunks > 0) ok = stage_chunk(0) && stage_v(0) && (nchunks < 2 || stage_chunk(1));

    // ---- initial state -> S32 (scaled by the first chunk's decay) and S16 ------------------
    named_sync(kBarChain, kGroup);
    {
      const float d0 = nchunks > 0 ? sm.gamma[0] : 1.f;
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
      const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {  // O^T of both blocks starts from zero
        tmem_st16(t_lane + TM_OU + 128 * bb + 32 * half, z);
        tmem_st16(t_lane + TM_OU + 128 * bb + 32 * half + 16, z);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    named_sync(kBarChain, kGroup);
    tc_fence_after();

    // The state product of chunk c, S16 [Q~; -W]^T (N = 128), into block [O^T | U^T] of
    // buffer c & 1: it starts O^T (zeroed beforehand) and turns U^T into D^T = U^T - S W^T.
    const uint32_t id_ow = idesc_f16(128, 128, 0, 0);
    const uint32_t id_n64 = idesc_f16(128, 64, 0, 0);
    const uint32_t id_n128 = idesc_f16(128, 128, 0, 1);
    auto issue_state = [&](int c) {
      const int b = c & 1;
      const uint64_t qw = dsc_k + ((smem_u32(smem + OFF_KQ + b * kKQW) + 8192) >> 4);
#pragma unroll
      for (int s = 0; s < kD / 16; ++s)
        mma_f16_ts(tbase + TM_OU + 128 * b, tbase + TM_S16 + s * 8,
                   qw + (((s >> 2) * kRegion + (s & 3) * 32) >> 4), id_ow, 1);
      commit(sm, B_D);
    };

    if (leader && nchunks > 0 && ok) {
      if (leader_wait(sm, B_READY0, 0)) {
        issue_state(0);
      } else {
        lead_fail = true;
      }
    }
    __syncwarp();
    int c_next = sd.ckpt_begin;
    // the next checkpoint's position (-1: none left), read again only after a checkpoint is
    // stored, so that no chunk waits on a global load to decide
    int ck_pos = c_next < sd.ckpt_end ? __ldg(p.ckpt_pos + c_next) : -1;

    for (int c = 0; c < nchunks && ok; ++c) {
      const int b = c & 1, t0 = c * kC, L = min(kC, sd.len - t0);
      const bool last = c + 1 == nchunks;
      const Factors f(reinterpret_cast<float*>(smem + OFF_VEC + b * 2048));

      // ---- (C1) D^T = U^T - S16 W^T is ready: D^T and D'^T = D^T diag(dec) -> smem (fp16) ---
      // (the previous chunk's output store must have read sO, which D^T overwrites)
      if (leader && store_pending) {
        bulk_wait_read_all();
        store_pending = false;
      }
      if (!(ok = group_wait(sm, B_D, c & 1, kBarChain, leader, lead_fail))) break;
      {
        uint32_t r[32];
        tmem_ld32(t_lane + TM_OU + 128 * b + 64 + 32 * half, r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          const float4 da = *reinterpret_cast<const float4*>(f.Dec + 32 * half + e);
          const float4 db = *reinterpret_cast<const float4*>(f.Dec + 32 * half + e + 4);
          const float d8[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
          float x[8], y[8];
#pragma unroll
          for (int q = 0; q < 8; q += 2) {
            x[q] = __uint_as_float(r[e + q]);
            x[q + 1] = __uint_as_float(r[e + q + 1]);
            const float2 t = mul2(make_float2(x[q], x[q + 1]), make_float2(d8[q], d8[q + 1]));
            y[q] = t.x;
            y[q + 1] = t.y;
          }
          st_chunk(sD, row, 32 * half + e, 128, x);
          st_chunk(sDp, row, 32 * half + e, 128, y);
        }
      }
      publish(kBarChain);
      // gate factors of chunk c+2 (buffer b's factors were last read just above), while the
      // leader issues this chunk's last products
      if (warp == kGateWarp && c + 2 < nchunks) stage_gates(c + 2);

      // ---- (C2) S32 += D'^T K (-> B_S);  O^T += D^T P^T (-> B_O) -------------------------------
      if (leader) {
        const uint64_t kq = dsc_mnr + (smem_u32(smem + OFF_KQ + b * kKQW) >> 4),
                       d0 = dsc_k + (smem_u32(sD) >> 4), dp = dsc_k + (smem_u32(sDp) >> 4),
                       p0 = dsc_k + (smem_u32(smem + OFF_P + b * 8192) >> 4);
#pragma unroll
        for (int s = 0; s < kC / 16; ++s)
          mma_f16_ss(tbase + TM_S32, dp + s * 2, kq + s * 128, id_n128, 1);
        commit(sm, B_S);
#pragma unroll
        for (int s = 0; s < kC / 16; ++s)
          mma_f16_ss(tbase + TM_OU + 128 * b, d0 + s * 2, p0 + s * 2, id_n64, 1);
        commit(sm, B_O);
      }
      __syncwarp();

      // ---- (C3) S16 refresh, checkpoints, final state; pre-scale S32 by the next decay --------
      if (!(ok = group_wait(sm, B_S, c & 1, kBarChain, leader))) break;
      // K and Q~ of buffer b are consumed (the commit covers every earlier product): fetch
      // chunk c+2's q, k into it
      if (leader && c + 2 < nchunks)
        issue_kq(P, sm, smem + OFF_KQ + b * kKQW, b, hk, sd.tok_start + t0 + 2 * kC, dh);
      bool last_ckpt = false;  // this chunk stores the unit's last checkpoint
      {
        const int pos = t0 + L;
        const bool emit = ck_pos == pos;
        const float nd = last ? 1.f : sm.gamma[b ^ 1];
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
              const float2 a = mul2(
                  make_float2(__uint_as_float(s32[e]), __uint_as_float(s32[e + 1])),
                  make_float2(nd, nd));
              const float2 bq = mul2(
                  make_float2(__uint_as_float(s32[16 + e]), __uint_as_float(s32[17 + e])),
                  make_float2(nd, nd));
              lo[e] = __float_as_uint(a.x);
              lo[e + 1] = __float_as_uint(a.y);
              hi[e] = __float_as_uint(bq.x);
              hi[e + 1] = __float_as_uint(bq.y);
            }
            tmem_st16(t_lane + TM_S32 + 64 * half + c0, lo);
            tmem_st16(t_lane + TM_S32 + 64 * half + c0 + 16, hi);
          }
        }
        if (emit) {
          ++c_next;
          ck_pos = c_next < sd.ckpt_end ? __ldg(p.ckpt_pos + c_next) : -1;
        }
        last_ckpt = emit && c_next == sd.ckpt_end;
        tmem_st_wait();
      }
      tc_fence_before();
      if (p.ckpt_ready && last_ckpt) {  // the copy of the prompt's checkpoints may start
        signal_ckpt_ready(p.ckpt_ready, u.seq, kBarChain, kGroup, leader);
        signaled = true;
      } else {
        named_sync(kBarChain, kGroup);
      }
      tc_fence_after();

      // ---- (C4) next chunk's D^T product now if its operands are ready (else after C5) -------
      bool w_issued = false;
      if (leader && !last && mbar_try_wait(&sm.bar[B_READY0 + (b ^ 1)], ((c + 1) >> 1) & 1)) {
        tc_fence_after();
        issue_state(c + 1);
        w_issued = true;
      }
      __syncwarp();

      // the next chunk's v for the prep group (copied once the prep group's U^T product of this
      // chunk read the previous one)
      if (!last && !(ok = stage_v(c + 1))) break;

      // ---- (C5) output rows of this chunk (bf16) ------------------------------------------------
      if (!(ok = group_wait(sm, B_O, c & 1, kBarChain, leader, lead_fail))) break;
      {
        uint32_t r[32];
        tmem_ld32(t_lane + TM_OU + 128 * b + 32 * half, r);
        tmem_ld_wait();
        const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        tmem_st16(t_lane + TM_OU + 128 * b + 32 * half, z);  // zero O^T for chunk c+2
        tmem_st16(t_lane + TM_OU + 128 * b + 32 * half + 16, z);
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
        tmem_st_wait();
      }
      const bool tma_out = L == kC && dh == kD;  // whole d = 128 chunks leave by TMA
      if (tma_out) fence_proxy_async_smem();
      tc_fence_before();
      named_sync(kBarChain, kGroup);
      if (tma_out) {
        // a whole chunk lies inside the prompt: one TMA store of the 64 x 128 tile
        if (leader) {
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
          const int idx = it * kGroup + ctid, t = idx / pieces, ch = idx % pieces;
          if (t < L && idx < kC * pieces)
            *reinterpret_cast<uint4*>(og + (size_t)(t0 + t) * v_stride + ch * 8) =
                *reinterpret_cast<const uint4*>(sO + t * 256 + ch * 16);
        }
      }

      // ---- (C6) stage chunk c+2 (copied into buffer b since C3) ------------------------------
      // (the group waits also order the staging reads above before the next D^T lands there)
      if (c + 2 < nchunks && !(ok = stage_chunk(c + 2))) break;
      named_sync(kBarChain, kGroup);

      // ---- (C7) the next chunk's state products, if C4 could not issue them ------------------
      if (leader && !last && !w_issued) {
        if (leader_wait(sm, B_READY0 + (b ^ 1), ((c + 1) >> 1) & 1)) {
          issue_state(c + 1);
        } else {
          lead_fail = true;
        }
      }
      __syncwarp();
    }
    if (!ok) sm.abort = 1;
    if (leader) {
      mma_commit(&sm.bar[B_FLUSH_C]);
      mbar_wait_bounded(&sm.bar[B_FLUSH_C], 0, kWaitLimit);
      if (store_pending) bulk_wait_all();  // output stores done before the CTA exits
    }

    // a unit without checkpoints, or one that gave up before its last, arrives here
    if (p.ckpt_ready && !signaled) signal_ckpt_ready(p.ckpt_ready, u.seq, kBarChain, kGroup, leader);
  }

  // ---- both groups done: let every copy and product still in flight land (bounded) --------
  __syncthreads();
  if (tid == 0) {
    if (sm.abort && p.status) atomicExch(p.status, kStatusTimeout);
#pragma unroll 1
    for (int i = 0; i < B_FLUSH_P; ++i)
      if (sm.issued[i] > sm.waited[i])  // at most one completion is ever outstanding
        mbar_wait_bounded(&sm.bar[i], (sm.issued[i] - 1) & 1u, kWaitLimit);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

int launch_chunked_pipelined(const PrefillArgs& a, int64_t total_tokens, void* stream) {
  if (a.num_units == 0) return 0;
  static std::atomic<int> configured[kMaxDevices];
  const int ce = configure_once(configured, [] {
    for (const void* k : {(const void*)chunked_pipe_kernel<128>,
                          (const void*)chunked_pipe_kernel<64>}) {
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
    chunked_pipe_kernel<64><<<a.num_units, kThreads, SMEM_BYTES, st>>>(P);
  else
    chunked_pipe_kernel<128><<<a.num_units, kThreads, SMEM_BYTES, st>>>(P);
  return (int)cudaGetLastError();
}

}  // namespace gdn
