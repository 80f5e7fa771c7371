// gdn_tma.cu — 2D TMA tensor maps over the packed bf16 q, k, v matrices.
//
// The chunked prefill kernels load 64-token x 64-column boxes of q, k and v with
// cp.async.bulk.tensor; this file encodes the maps through the driver's
// cuTensorMapEncodeTiled, fetched once through the runtime's entry-point query.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "gdn_internal.h"

namespace gdn {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

}  // namespace

bool make_bf16_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool make_out_map(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows) {
  if (rows == 0) {
    memset(m, 0, sizeof(CUtensorMap));
    return true;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {128, 64};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_qkv_maps(const PrefillArgs& a, int64_t total_tokens, int head_dim, CUtensorMap* tq,
                   CUtensorMap* tk, CUtensorMap* tv) {
  if (total_tokens <= 0) {
    memset(tq, 0, sizeof(CUtensorMap));
    memset(tk, 0, sizeof(CUtensorMap));
    memset(tv, 0, sizeof(CUtensorMap));
    return true;
  }
  const uint64_t rows = (uint64_t)total_tokens;
  return make_bf16_map(tq, a.q, (uint64_t)a.hk_heads * head_dim, rows) &&
         make_bf16_map(tk, a.k, (uint64_t)a.hk_heads * head_dim, rows) &&
         make_bf16_map(tv, a.v, (uint64_t)a.hv_heads * head_dim, rows);
}

// Estimated times (microseconds) from costs measured on GB300 with uniform packs of 2- to
// 64-chunk units (8 value heads, L2 flushed, the current kernels):
//  * pipelined (one unit per SM): 5.12 per chunk plus 15.7 per unit (the pipeline's fill and
//    drain and the unit's set-up);
//  * throughput, two units per SM: 8.93 per chunk plus 13.2 per unit; a unit alone on its
//    SM: 6.38 per chunk plus 17.3;
//  * a unit of a prompt with one token or none: 8.0 per pipelined slot, 16.6 per
//    throughput slot.
// A pack takes at least its longest unit's chain, at least its total work spread over the
// SMs' slots, and, since a unit never moves between SMs, at least its whole rounds of the
// mean unit: ceil(units / SMs) pipelined rounds; in the throughput schedule one paired
// round per 2 x SMs units, then a last round that is paired when its units outnumber the
// SMs and alone otherwise. Once units outnumber SMs the longest unit runs paired too.
namespace {

void schedule_estimates(const ChunkLoad& load, int32_t num_sms, double* t_pipe, double* t_thr) {
  constexpr double kPipeChunk = 5.12, kPipeUnit = 15.7, kPipeShort = 8.0;
  constexpr double kThrChunk = 8.93, kThrUnit = 13.2, kThrShort = 16.6;
  constexpr double kAloneChunk = 6.38, kAloneUnit = 17.3;
  const double longest = load.longest, total = (double)load.total, sms = num_sms;
  const double shorts = (double)load.short_units, units = (double)load.units;
  const double has = units > 0 ? 1.0 : 0.0;
  const double mean = units > 0 ? total / units : 0.0;
  const double rounds = std::ceil(units / sms);
  *t_pipe = std::max({longest * kPipeChunk + has * kPipeUnit,
                      (total * kPipeChunk + units * kPipeUnit + shorts * kPipeShort) / sms,
                      rounds * (mean * kPipeChunk + kPipeUnit)});
  const double chain = units > sms ? longest * kThrChunk + kThrUnit
                                   : longest * kAloneChunk + has * kAloneUnit;
  const double slots = kThroughputCtasPerSM * sms;
  const double full = std::floor(units / slots), last = units - full * slots;
  const double paired = mean * kThrChunk + kThrUnit, alone = mean * kAloneChunk + kAloneUnit;
  const double thr_rounds = full * paired + (last > sms ? paired : last > 0 ? alone : 0.0);
  *t_thr = std::max({chain, thr_rounds,
                     (total * kThrChunk + units * kThrUnit + shorts * kThrShort) / slots});
}

}  // namespace

int plan_schedule(const ChunkLoad& load, int32_t num_sms) {
  double t_pipe, t_thr;
  schedule_estimates(load, num_sms, &t_pipe, &t_thr);
  return t_thr < t_pipe ? kChunkedThroughput : kChunkedPipelined;
}

double estimate_pass_us(const ChunkLoad& load, int32_t num_sms) {
  double t_pipe, t_thr;
  schedule_estimates(load, num_sms, &t_pipe, &t_thr);
  return std::min(t_pipe, t_thr);
}

int32_t choose_split_segment(const int32_t* cu, int32_t num_seqs, int32_t num_v_heads,
                             int32_t num_sms) {
  // a launch, the map composition and the state gather: small fixed costs per extra pass
  constexpr double kSplitOverheadUs = 12.0;
  int32_t longest = 0;
  for (int32_t n = 0; n < num_seqs; ++n) longest = std::max(longest, cu[n + 1] - cu[n]);
  double best = estimate_pass_us(chunk_load(cu, num_seqs, num_v_heads), num_sms);
  int32_t best_seg = 0;
  for (int32_t parts = 2; parts <= 16; ++parts) {
    int32_t seg = (longest + parts - 1) / parts;
    seg = (seg + 63) / 64 * 64;
    if (seg < 64 || seg >= longest) continue;
    // the virtual packs of the two passes, by length: pass A runs segment 0 of every prompt
    // and two maps per middle segment of a split prompt; pass B the other segments
    ChunkLoad a, b;
    auto add = [](ChunkLoad& l, int32_t len, int32_t units) {
      if (len <= 1) {
        l.short_units += units;
        return;
      }
      const int32_t c = (len + 63) / 64;
      l.total += (int64_t)c * units;
      l.units += units;
      l.longest = std::max(l.longest, c);
    };
    for (int32_t n = 0; n < num_seqs; ++n) {
      const int32_t len = cu[n + 1] - cu[n];
      add(a, std::min(len, seg), num_v_heads);
      if (len <= seg) continue;
      const int32_t np = (len + seg - 1) / seg;
      for (int32_t q = 1; q + 1 < np; ++q) add(a, seg, 2 * num_v_heads);
      for (int32_t q = 1; q < np; ++q) add(b, std::min(seg, len - q * seg), num_v_heads);
    }
    const double t = estimate_pass_us(a, num_sms) + estimate_pass_us(b, num_sms) +
                     kSplitOverheadUs;
    if (t < best) {
      best = t;
      best_seg = seg;
    }
  }
  return best_seg;
}

namespace {

// SM count per device, asked once per device; concurrent first calls may each ask, and all
// store the same value.
std::atomic<int> g_sms[64];

int device_sms(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  int n = dev >= 0 && dev < 64 ? g_sms[dev].load(std::memory_order_relaxed) : 0;
  if (n == 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    if (dev >= 0 && dev < 64) g_sms[dev].store(n, std::memory_order_relaxed);
  }
  *out = n;
  return 0;
}

}  // namespace

int launch_chunked_prefill(const PrefillArgs& a, int64_t total_tokens, int schedule,
                           const ChunkLoad& load, void* stream) {
  if (schedule == kChunkedAuto) {
    int n = 0;
    const int e = device_sms(&n);
    if (e != 0) return e;
    schedule = plan_schedule(load, n);
  }
  // one launch for every unit: the units of prompts with one token or none close the
  // longest-first work list, and the kernels run them with the decode step's arithmetic
  return schedule == kChunkedThroughput ? launch_chunked_throughput(a, total_tokens, stream)
                                        : launch_chunked_pipelined(a, total_tokens, stream);
}

}  // namespace gdn
