// gdn_internal.h — structures shared by the C ABI layer and the CUDA kernels.
//
// The host scheduler turns cu_seqlens and the checkpoint CSR into a work list that is
// uploaded once per call into the caller's workspace:
//   [GdnUnit units[num_units]] [GdnSeq seqs[num_seqs]] [int32 ckpt_pos[num_ckpt]]
// each array starting on a 256-byte boundary. A unit is one independent piece of the
// recurrence: a (prompt, value head, block of state rows) triple. Rows of the state evolve
// independently (row i only needs k, beta, g and row i itself), so a unit may own any row
// block. Units are ordered longest prompt first so the hardware block scheduler, which
// hands out blocks roughly in index order, runs a longest-processing-time-first schedule.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

#include "../../include/gdn.h"

namespace gdn {

struct GdnUnit {
  int32_t seq;    // prompt index in the pack
  int32_t head;   // value head
  int32_t row0;   // first state row (value dim) owned by the unit
  int32_t nrows;  // number of rows
};

struct GdnSeq {
  int32_t tok_start;   // cu_seqlens[n]
  int32_t len;         // tokens in the prompt's segment
  int32_t ckpt_begin;  // CSR range of this prompt's checkpoints
  int32_t ckpt_end;
  int32_t flags;       // kSeqZeroV, kSeqZeroInit
  int32_t state_slot;  // index of the prompt's [H_v][d][d] state in init / final_state: the
                       // prompt's index, or its pool slot (gdn_prefill_packed_pool)
};
constexpr int32_t kSeqZeroV = 1;     // v is taken as zero (sequence splitting's map runs)
constexpr int32_t kSeqZeroInit = 2;  // the prompt starts from a zero state, whatever init holds

// Everything a prefill kernel needs besides the work list.
struct PrefillArgs {
  const void* q;          // [T][Hk][D]
  const void* k;          // [T][Hk][D]
  const void* v;          // [T][Hv][D]
  const float* a;         // [T][Hv]
  const float* beta;      // [T][Hv]
  const float* init;      // [N][Hv][D][D] or nullptr
  void* o;                // [T][Hv][D]
  float* ckpt;            // [C][Hv][D][D]
  float* final_state;     // [N][Hv][D][D]
  const GdnUnit* units;
  const GdnSeq* seqs;
  const int32_t* ckpt_pos;
  int32_t num_units;
  int32_t hk_heads;
  int32_t hv_heads;
  int32_t group;          // Hv / Hk
  int32_t head_dim = 128; // d_k = d_v (64 or 128)
  float scale;
  int32_t l2norm;
  int32_t* status;        // device status word (0 = ok) or nullptr
  int32_t gate_mode;      // 0: a, beta as given; 1: raw projections (see gate_from_raw)
  const float* a_log;     // [Hv] (gate_mode 1)
  const float* dt_bias;   // [Hv] (gate_mode 1)
  // Test hook (gdn_set_test_hook): the chunked kernels leave out every unit's first q/k
  // copy, so that its first bounded wait runs out and the timeout path runs.
  int32_t test_skip_first_copy = 0;
  // Per-prompt counters (indexed like seqs) or nullptr. Every block of the launch adds 1 to
  // its prompt's counter once all of its checkpoint rows are stored and made visible (a
  // block whose prompt has no checkpoint adds it when it ends), also on the timeout path;
  // gdn_prefill_packed_snapshot starts each prompt's checkpoint copy from that count.
  int32_t* ckpt_ready = nullptr;
};

// Marks a block's checkpoints as stored: every thread that stored checkpoint rows makes its
// stores visible at system scope, the storing threads meet at barrier `bar_id` (`nthreads`
// of them, 0 = the block barrier), then `leader` adds 1 to the prompt's counter. Callers
// skip it (uniformly) when ready is nullptr.
#ifdef __CUDACC__
__device__ __forceinline__ void signal_ckpt_ready(int32_t* ready, int32_t seq, uint32_t bar_id,
                                                  uint32_t nthreads, bool leader) {
  __threadfence_system();
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthreads) : "memory");
  if (leader) atomicAdd(ready + seq, 1);
}
#endif

struct DecodeArgs {
  const void* q;          // [B][Hk][D]
  const void* k;
  const void* v;          // [B][Hv][D]
  const float* a;         // [B][Hv]
  const float* beta;
  float* pool;            // [slots][Hv][D][D]
  const int32_t* slot;    // [B]
  void* o;                // [B][Hv][D]
  int32_t batch;
  int32_t hk_heads;
  int32_t hv_heads;
  int32_t group;
  float scale;
  int32_t l2norm;
  int32_t gate_mode;
  const float* a_log;
  const float* dt_bias;
};

constexpr float kL2NormEps = 1e-6f;

// Gates of the Qwen3.5/3.6-style GDN layer from its raw projections: per value head h,
// a = -exp(A_log[h]) * softplus(a_raw + dt_bias[h]) (the log-decay, g = exp(a)) and
// beta = sigmoid(b_raw). softplus switches to the identity above 20, where
// log1p(exp(x)) equals x to fp32 precision.
#ifdef __CUDACC__
__device__ __forceinline__ void gate_from_raw(float a_log, float dt_bias, float& a, float& b) {
  const float x = a + dt_bias;
  const float sp = x > 20.f ? x : log1pf(expf(x));
  a = -expf(a_log) * sp;
  b = 1.f / (1.f + expf(-b));
}
#endif

// Launchers (defined in the .cu files). Return a cudaError_t as int.
int launch_recurrent_prefill(const PrefillArgs& a, int head_dim, bool bf16, void* stream);
int launch_decode(const DecodeArgs& a, int head_dim, bool bf16, void* stream);

// The chunked tensor-core prefill has two schedules over the same work list (one unit per
// prompt and value head):
//  * throughput (gdn_chunked.cu): two 8-warp CTAs per SM, each running its unit's chunk
//    phases in sequence; best when every SM has several units to run;
//  * pipelined (gdn_chunked_pipe.cu): one 16-warp CTA per SM whose two warp groups overlap
//    the state-independent work of the next chunk with the recurrence of the current one;
//    shortest time per unit, so best for packs with few units per SM or very long prompts.
// kChunkedAuto takes the one with the smaller estimated time (plan_schedule).
enum ChunkedSchedule : int { kChunkedAuto = 0, kChunkedPipelined = 2, kChunkedThroughput = 3 };
constexpr int kThroughputCtasPerSM = 2;  // resident throughput CTAs per SM

// Chunk counts of a pack's work list: over all units, and of the longest unit; and the units
// of prompts with at most one token, which close the longest-first work list and which the
// chunked kernels run with the decode step's arithmetic (no chunk phases, no tensor memory).
struct ChunkLoad {
  int64_t total = 0;
  int32_t longest = 0;
  int64_t short_units = 0;
  int64_t units = 0;  // units with at least one chunk
};
// The load of a pack of prompts (cu: host prefix sums) with `units_per_prompt` units each.
inline ChunkLoad chunk_load(const int32_t* cu, int32_t num_seqs, int32_t units_per_prompt) {
  ChunkLoad l;
  for (int32_t n = 0; n < num_seqs; ++n) {
    const int32_t len = cu[n + 1] - cu[n];
    if (len <= 1) {
      l.short_units += units_per_prompt;
      continue;
    }
    const int32_t c = (len + 63) / 64;
    l.total += (int64_t)c * units_per_prompt;
    l.units += units_per_prompt;
    if (c > l.longest) l.longest = c;
  }
  return l;
}
// kChunkedPipelined or kChunkedThroughput for a pack of this load on `num_sms` SMs.
int plan_schedule(const ChunkLoad& load, int32_t num_sms);
// The cost model's estimate (microseconds) of one chunked launch over this load.
double estimate_pass_us(const ChunkLoad& load, int32_t num_sms);
// The segment length (a multiple of 64) that the cost model expects to run a pack fastest
// through sequence splitting, or 0 when splitting is not expected to pay.
int32_t choose_split_segment(const int32_t* cu, int32_t num_seqs, int32_t num_v_heads,
                             int32_t num_sms);
int launch_chunked_throughput(const PrefillArgs& a, int64_t total_tokens, void* stream);
int launch_chunked_pipelined(const PrefillArgs& a, int64_t total_tokens, void* stream);
int launch_chunked_prefill(const PrefillArgs& a, int64_t total_tokens, int schedule,
                           const ChunkLoad& load, void* stream);

// 2D bf16 tensor maps (64 x 64 boxes, 128-byte swizzle, zero fill past the last row) over
// q, k (H_k * d columns) and v (H_v * d columns) with total_tokens rows (gdn_tma.cu).
bool make_qkv_maps(const PrefillArgs& a, int64_t total_tokens, int head_dim, CUtensorMap* tq,
                   CUtensorMap* tk, CUtensorMap* tv);
// 2D bf16 tensor map over the output o ([rows][cols], row-major) with 64-row x 128-column
// boxes and no swizzle, for TMA stores of whole chunks of one head's output rows.
bool make_out_map(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows);

// Sequence splitting (gdn_split.cu). fill_states modes besides "copy the caller's state of
// prompt i" (i >= 0):
constexpr int32_t kSplitZero = -1, kSplitIdentity = -2;
// One split prompt: its segment-0 final state is finals_a[first_final]; B_p and M_p of
// segments p = 1 .. num_segments - 2 are finals_a[first_map + 2 (p - 1)] and the one after;
// the initial state of segment p >= 1 goes to inits_c[first_init + p - 1].
struct SplitCompose {
  int32_t num_segments, first_final, first_map, first_init;
};
int launch_fill_states(float* dst, const float* src, const int32_t* mode, int count, int hv,
                       int d, void* stream);
int launch_compose_maps(const SplitCompose* jobs, int num_jobs, const float* finals_a,
                        float* inits_c, int hv, int d, void* stream);
// dst[n] = index[n] >= 0 ? src_a[index[n]] : src_c[-1 - index[n]] (per prompt, all heads)
int launch_gather_states(float* dst, const float* src_a, const float* src_c,
                         const int32_t* index, int num_seqs, int hv, int d, void* stream);

// Host-side planning shared with the allocation-free entry point (gdn_noalloc.cu):
// the kernel family, the work-list layout and its size for one pack.
struct PrefillPlan {
  int family;            // 1 = token-serial, 2 = chunked tensor-core
  size_t units_off, seqs_off, pos_off, ready_off, bytes;
  int32_t num_units, num_ckpt;
};
gdn_status plan_prefill(const gdn_handle* h, const gdn_config* cfg, int32_t num_seqs,
                        const int32_t* cu, const int32_t* ckpt_cu, const int32_t* ckpt_pos,
                        PrefillPlan* out);
void write_worklist(void* dst, const PrefillPlan& plan, const gdn_config* cfg, int32_t num_seqs,
                    const int32_t* cu, const int32_t* ckpt_cu, const int32_t* ckpt_pos);

// Row block of a unit for each kernel family.
constexpr int kRecurrentRows = 32;
constexpr bool kChunkedReady = true;

// Once-per-device kernel set-up (cudaFuncSetAttribute acts on the current device): runs
// `fn` on the first call for each device and remembers success. Concurrent first calls
// may each run it, so `fn` must be idempotent. Returns fn's error, or a runtime error.
constexpr int kMaxDevices = 64;
template <class F>
int configure_once(std::atomic<int> (&done)[kMaxDevices], F fn) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  if (tracked && done[dev].load(std::memory_order_acquire)) return 0;
  const int r = fn();
  if (r == 0 && tracked) done[dev].store(1, std::memory_order_release);
  return r;
}

}  // namespace gdn
