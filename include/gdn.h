/*
 * gdn.h — C ABI of the packed gated-delta-rule (GDN) prefill library for sm_103a.
 *
 * What the library computes
 * -------------------------
 * The gated delta rule (Gated Delta Networks, Yang, Kautz & Hatamizadeh, 2024) is the
 * linear-attention layer of the Qwen3.5/3.6 hybrid models ("hybrid attention architecture
 * used by Qwen3.5-style models", vLLM-Ascend tutorial "Qwen3.6-35B-A3B", §1 Introduction).
 * For every packed prompt n and value head h, with key head hk = h / (H_v / H_k), the
 * state S (d_v x d_k, fp32) evolves token by token:
 *
 *     q_t, k_t <- q_t / ||q_t||, k_t / ||k_t||          (when qk_l2norm != 0)
 *     g_t = exp(a_t)
 *     S_t = g_t S_{t-1} - beta_t (g_t S_{t-1} k_t - v_t) k_t^T
 *     o_t = scale * S_t q_t
 *
 * Many prompts share one pass ("packed passes", sparkinfer v0.6.28 release notes, intro).
 * Each prompt may start from its own initial state (a prefix-cache hit) and the pass emits
 * state snapshots at requested prompt positions ("prefix-cache checkpoint", same release
 * notes, bullets 2-4). A one-token decode update serves sequences that are decoding
 * ("packed GDN decode", vllm.cpp "vLLM, online serving", lever 2b).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer named *_host is host memory; every other data pointer is device memory
 *    of the current CUDA device, owned by the caller, and must stay valid until the work
 *    queued on `stream` has finished. The library never frees caller memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). All
 *    device work is asynchronous on it.
 *  - All arguments are validated on the host before anything is enqueued; on an error
 *    nothing is launched and the status says why ("reject unsupported combinations before
 *    model loading", pegainfer PR #786, Changes). A failed launch returns GDN_ERR_CUDA.
 *  - No call logs, throws or exits.
 *  - Token-major layouts: q, k are [T][H_k][d_k]; v, o are [T][H_v][d_v]; a and beta are
 *    [T][H_v]; states are [.][H_v][d_v][d_k] fp32 with d_k contiguous (row = value dim).
 *    T = cu_seqlens_host[num_seqs]. Device buffers must be 16-byte aligned.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 1

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARGUMENT = 1,   /* malformed sizes, pointers, offsets or positions  */
  GDN_ERR_UNSUPPORTED = 2,        /* well-formed but outside what the kernels cover   */
  GDN_ERR_WORKSPACE_TOO_SMALL = 3,
  GDN_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed             */
  GDN_ERR_DEVICE_TIMEOUT = 5,     /* a bounded device-side wait gave up               */
  GDN_ERR_POOL_EXHAUSTED = 6,     /* pinned snapshot pool range out of bounds         */
  GDN_ERR_BUSY = 7                /* the handle's prefill stream already has a prefill */
} gdn_status;

typedef enum gdn_dtype {
  GDN_F32 = 0,   /* q, k, v, o in fp32 */
  GDN_BF16 = 1   /* q, k, v, o in bf16; a, beta and all states stay fp32 */
} gdn_dtype;

/* How the `a` and `beta` arrays of a call are read. */
typedef enum gdn_gate_mode {
  GDN_GATES_DIRECT = 0,  /* a = log-decay (g = exp(a)), beta = write strength, as given */
  GDN_GATES_RAW = 1      /* raw projections of the Qwen3.5/3.6-style GDN layer, turned into
                            gates in the kernel: a = -exp(A_log[h]) * softplus(a_raw +
                            dt_bias[h]), beta = sigmoid(b_raw) (fp32 arithmetic) */
} gdn_gate_mode;

/* Layer shape and gate inputs. Supported: head_dim_k == head_dim_v in {64, 128},
 * num_v_heads a positive multiple of num_k_heads, chunk_size == 64. With gate_mode ==
 * GDN_GATES_RAW, a_log and dt_bias must be non-NULL device arrays of H_v floats (unused
 * otherwise). */
typedef struct gdn_config {
  int32_t num_k_heads;   /* H_k */
  int32_t num_v_heads;   /* H_v; value head h reads key head h / (H_v / H_k)       */
  int32_t head_dim_k;    /* d_k */
  int32_t head_dim_v;    /* d_v */
  int32_t chunk_size;    /* C: token block of the chunked scan; checkpoint grid     */
  float scale;           /* output scale, usually 1/sqrt(d_k)                       */
  int32_t qk_l2norm;     /* nonzero: q, k <- x / sqrt(x.x + 1e-6) per token and head */
  int32_t io_dtype;      /* gdn_dtype of q, k, v, o                                 */
  int32_t gate_mode;     /* gdn_gate_mode of a and beta                              */
  const float* a_log;    /* [H_v] device fp32 per-head log decay rate (GATES_RAW)    */
  const float* dt_bias;  /* [H_v] device fp32 per-head bias of a_raw (GATES_RAW)     */
} gdn_config;

typedef struct gdn_handle gdn_handle;

/* Library ABI version (GDN_ABI_VERSION of the build). */
int32_t gdn_abi_version(void);

/* Static, NUL-terminated name of a status code; unknown codes give "unknown status". */
const char* gdn_status_string(int32_t status);

/* Create a handle bound to CUDA device `device`. The handle owns a pinned host snapshot
 * pool of `pinned_pool_bytes` (0 = none), allocated here, once, rather than in the middle
 * of a pass (sparkinfer v0.6.28, bullet on pinned host buffers), a side stream for
 * checkpoint copies, a pinned staging ring for work lists, and events. On success *out
 * receives the handle. Errors: INVALID_ARGUMENT (out NULL, device out of range), CUDA. */
gdn_status gdn_handle_create(int32_t device, size_t pinned_pool_bytes, gdn_handle** out);

/* Drain the handle's side stream and staging ring, then free what the handle owns
 * ("drain the prefill stream on error, cancellation, drop, and shutdown", pegainfer PR
 * #786, Changes). NULL is accepted and ignored. */
gdn_status gdn_handle_destroy(gdn_handle* handle);

/* Host address and size of the handle's pinned snapshot pool. */
gdn_status gdn_pool_info(gdn_handle* handle, void** host_ptr, size_t* bytes);

/* Kernel choice for later prefill calls on this handle:
 *   0 = automatic: the tensor-core chunked kernel where it applies (bf16 io, d = 64 or
 *       128; d = 64 heads run zero-padded to 128, exact), in the schedule
 *       gdn_chunked_schedule names for the pack; otherwise (fp32 io) the token-serial
 *       CUDA-core kernel;
 *   1 = always the token-serial kernel (a cross-check path);
 *   2 = the chunked kernel's pipelined schedule, 3 = its throughput schedule (where the
 *       chunked kernel applies; otherwise the token-serial kernel).
 * The two chunked schedules give bit-identical results, so choices 0, 2 and 3 agree bit
 * for bit, and a prompt's results do not depend on the pack around it even where the
 * automatic choice differs; the token-serial kernel agrees with them to rounding. Errors: INVALID_ARGUMENT. */
gdn_status gdn_set_kernel_preference(gdn_handle* handle, int32_t preference);

/* Test hook for the device-side timeout path (hook 1; 0 = off, the default). While it is
 * set, the chunked tensor-core kernels leave out every unit's first q/k tile copy, so each
 * unit's first copy wait runs out after its time bound (about one second of polling) with
 * no fault: the kernel records GDN_ERR_DEVICE_TIMEOUT in the status word that
 * gdn_read_device_status returns, lets every copy and product it did issue land, frees its
 * tensor memory and returns. The outputs of such a call are undefined; the CUDA context
 * stays usable. The token-serial kernel ignores the hook. Errors: INVALID_ARGUMENT. */
gdn_status gdn_set_test_hook(gdn_handle* handle, int32_t hook);

/* The chunked kernel's schedule that the automatic choice takes for a pack of `num_seqs`
 * prompts (cu_seqlens_host: prefix sums, as for gdn_prefill_packed) with `num_v_heads`
 * value heads on a GPU with `num_sms` SMs: *schedule = 2 (pipelined) or 3 (throughput),
 * the gdn_set_kernel_preference codes. The choice is the smaller of two estimates from
 * costs measured on GB300 (microseconds): 5.12 per chunk plus 15.7 per unit for a
 * pipelined unit on its own SM; 8.93 per chunk plus 13.2 per unit for one of two
 * throughput units sharing an SM, 6.38 plus 17.3 for one alone; 8.0 and 16.6 per unit of a
 * prompt with one token or none (which the same launch runs with the decode step's
 * arithmetic) on a pipelined or throughput slot. Over W = the chunks of the U other
 * (prompt, value head) units, Lmax = the chunks of the longest and S = the short units:
 *   pipelined:  max(5.12 Lmax + 15.7, (5.12 W + 15.7 U + 8.0 S) / num_sms,
 *                   ceil(U / num_sms) (5.12 W / U + 15.7))
 *   throughput: max(Lchain, R, (8.93 W + 13.2 U + 16.6 S) / (2 num_sms)), with
 *               Lchain = 8.93 Lmax + 13.2 when U > num_sms, else 6.38 Lmax + 17.3, and
 *               R = F (8.93 W / U + 13.2) + the last round, F = floor(U / (2 num_sms)):
 *               paired (8.93 W / U + 13.2) if its units outnumber the SMs, else alone
 *               (6.38 W / U + 17.3), else nothing
 * (the 15.7 and 17.3 terms and the rounds only when U > 0): a unit never moves between
 * SMs, so a pack runs in whole rounds, and a throughput pack with more units than SMs
 * has SMs running two units at once.
 * Both schedules give bit-identical results; only the time differs. Host-only arithmetic,
 * no CUDA call. Errors: INVALID_ARGUMENT (num_seqs < 0, cu NULL with num_seqs > 0,
 * cu[0] != 0 or decreasing, num_v_heads < 1, num_sms < 1, schedule NULL). */
gdn_status gdn_chunked_schedule(int32_t num_seqs, const int32_t* cu_seqlens_host,
                                int32_t num_v_heads, int32_t num_sms, int32_t* schedule);

/* Device workspace bytes that gdn_prefill_packed needs for this pack (the chunk/tile work
 * list). Validates the same arguments gdn_prefill_packed validates about the pack.
 * Result is a multiple of 256 and at least 256. */
gdn_status gdn_prefill_workspace_size(const gdn_config* cfg, int32_t num_seqs,
                                      const int32_t* cu_seqlens_host,
                                      const int32_t* ckpt_cu_host, size_t* bytes);

/* Packed variable-length prefill of the gated delta rule.
 *
 *  num_seqs         N >= 1 prompts in the pack.
 *  cu_seqlens_host  [N+1] int32, cu[0] = 0, non-decreasing; prompt n is tokens
 *                   [cu[n], cu[n+1]). Zero-length prompts are allowed: their final state
 *                   is their initial state and they emit no output.
 *  q, k             [T][H_k][d] io_dtype.   v: [T][H_v][d] io_dtype.
 *  a, beta          [T][H_v] fp32: log-decay (g = exp(a), a <= 0) and the write strength.
 *                   a = -inf (g = 0) is allowed: the state restarts at that token.
 *  initial_state    [N][H_v][d][d] fp32, or NULL for all-zero initial states.
 *  ckpt_cu_host     [N+1] int32 CSR over ckpt_pos_host (ckpt_cu[0] = 0), or NULL when no
 *                   prompt asks for a checkpoint.
 *  ckpt_pos_host    prompt-relative positions p: the snapshot is the state after the first
 *                   p tokens of that prompt's segment. Per prompt strictly increasing, in
 *                   [1, len], and each a multiple of chunk_size or equal to len
 *                   (otherwise GDN_ERR_UNSUPPORTED).
 *  o                [T][H_v][d] io_dtype output.
 *  ckpt_states      [ckpt_cu[N]][H_v][d][d] fp32; slot j holds checkpoint j of the CSR.
 *                   May be NULL only when there is no checkpoint.
 *  final_states     [N][H_v][d][d] fp32 state after each prompt's last token. May equal
 *                   initial_state (in-place update); no other overlap is allowed.
 *  workspace        device scratch of at least gdn_prefill_workspace_size() bytes,
 *                   256-byte aligned; it must not be reused by other work before this
 *                   call's work on `stream` has finished.
 * The result does not depend on how prompts are packed: each prompt's outputs, checkpoints
 * and final state are bit-identical whether it runs alone or inside any pack ("the same
 * checkpoints whether prompts are prefilled alone or packed", sparkinfer v0.6.28,
 * pack_ckpt_check). Errors: INVALID_ARGUMENT, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA. */
gdn_status gdn_prefill_packed(gdn_handle* handle, const gdn_config* cfg, int32_t num_seqs,
                              const int32_t* cu_seqlens_host,
                              const void* q, const void* k, const void* v,
                              const float* a, const float* beta,
                              const float* initial_state,
                              const int32_t* ckpt_cu_host, const int32_t* ckpt_pos_host,
                              void* o, float* ckpt_states, float* final_states,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Host image of the work list that gdn_prefill_packed would upload for this pack and
 * handle (handle may be NULL: automatic kernel choice), for inspection and tests. Layout,
 * each array on a 256-byte boundary: int32 status, int32 num_units, then num_units units
 * {int32 seq, head, row0, nrows} ordered longest prompt first, then per-prompt records
 * {int32 tok_start, len, ckpt_begin, ckpt_end, flags, state_slot}, then the checkpoint
 * positions, then one int32 per prompt (zero: the checkpoint counters that
 * gdn_prefill_packed_snapshot's kernels count up).
 * *bytes_needed receives the size; with out == NULL nothing else is written. Errors as
 * gdn_prefill_packed's pack checks, or WORKSPACE_TOO_SMALL when out_bytes is short. */
gdn_status gdn_prefill_worklist_host(gdn_handle* handle, const gdn_config* cfg,
                                     int32_t num_seqs, const int32_t* cu_seqlens_host,
                                     const int32_t* ckpt_cu_host, const int32_t* ckpt_pos_host,
                                     void* out, size_t out_bytes, size_t* bytes_needed);

/* Read the device status word that the last prefill using `workspace` left behind (0 when
 * every bounded device-side wait completed, GDN_ERR_DEVICE_TIMEOUT when one gave up).
 * Synchronises `stream`. Errors: INVALID_ARGUMENT, CUDA. */
gdn_status gdn_read_device_status(const void* workspace, int32_t* status_out, void* stream);

/* Copy `bytes` of device checkpoint states into the handle's pinned pool at byte offset
 * `pool_offset`, on the handle's side stream, after all work already queued on `stream`
 * (so the scan and the copy of the next prompts overlap; sparkinfer v0.6.28, bullet on
 * separate streams for the scan and the checkpoint copy). Returns at once; completion is
 * observed with gdn_checkpoint_copy_query / _wait. Errors: INVALID_ARGUMENT,
 * POOL_EXHAUSTED (range outside the pool), CUDA. */
gdn_status gdn_checkpoint_copy(gdn_handle* handle, const float* ckpt_states_dev, size_t bytes,
                               size_t pool_offset, void* stream);

/* gdn_prefill_packed whose checkpoints are copied into the handle's pinned pool while the
 * scan still runs ("the scan and the checkpoint copy run on separate streams, not one after
 * another", sparkinfer v0.6.28 release notes, bullet 2; the pool itself: bullet on pinned
 * host buffers). Checkpoint slot j lands at byte pool_offset + j * H_v * d * d * 4 of the
 * pool, the same layout as ckpt_states. Every block of the launch counts its prompt's
 * stored checkpoints in a per-prompt counter in the workspace; on the handle's side
 * stream, each copy of a run of prompts (consecutive prompt indices in the work list's
 * longest-first order, up to 8 MiB) first waits on the device until its prompts' counters
 * are complete (cuStreamWaitValue32), so the snapshots of prompts that finish early leave
 * while later prompts are still in the scan. Where the driver offers no stream wait on
 * memory, one copy follows the whole pass. Outputs are bit-identical to gdn_prefill_packed's.
 * Completion: gdn_checkpoint_copy_query / _wait on the host, gdn_checkpoint_copy_event or
 * gdn_checkpoint_copy_join on the device. Arguments and errors as gdn_prefill_packed, plus
 * POOL_EXHAUSTED when the checkpoints do not fit in the pool at pool_offset. The workspace
 * must not be reused before the copies have completed. */
gdn_status gdn_prefill_packed_snapshot(gdn_handle* handle, const gdn_config* cfg,
                                       int32_t num_seqs, const int32_t* cu_seqlens_host,
                                       const void* q, const void* k, const void* v,
                                       const float* a, const float* beta,
                                       const float* initial_state,
                                       const int32_t* ckpt_cu_host, const int32_t* ckpt_pos_host,
                                       void* o, float* ckpt_states, float* final_states,
                                       size_t pool_offset, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* GDN_OK when every checkpoint copy issued so far has completed, otherwise
 * GDN_ERR_DEVICE_TIMEOUT (not finished yet; nothing is wrong). */
gdn_status gdn_checkpoint_copy_query(gdn_handle* handle);

/* Block the calling host thread until every checkpoint copy issued so far has completed. */
gdn_status gdn_checkpoint_copy_wait(gdn_handle* handle);

/* The device-side completion of the checkpoint copies (the scan and the copy on separate
 * streams, sparkinfer v0.6.28 release notes, bullet 2): *event_out receives the handle's
 * cudaEvent_t (as void*), recorded on the side stream after the last copy issued so far
 * by gdn_checkpoint_copy or gdn_prefill_packed_snapshot, so that a consumer stream can
 * order itself after the snapshots without blocking a host thread
 * (cudaStreamWaitEvent). The handle owns the event; every later copy call records it
 * again, so take it after the copies it should cover have been issued. Before any copy it
 * has never been recorded, and a wait on it completes at once. Errors: INVALID_ARGUMENT. */
gdn_status gdn_checkpoint_copy_event(gdn_handle* handle, void** event_out);

/* Make `stream` wait on the device for every checkpoint copy issued so far (the same
 * ordering as a cudaStreamWaitEvent on gdn_checkpoint_copy_event's event); returns at
 * once. Errors: INVALID_ARGUMENT, CUDA. */
gdn_status gdn_checkpoint_copy_join(gdn_handle* handle, void* stream);

/* Prefill on the handle's own stream, so that a prefill pass overlaps decode steps that
 * keep running on the caller's streams ("run at most one in-flight prefill on an owned
 * CUDA stream", pegainfer PR #786, Changes). Arguments as gdn_prefill_packed; the owned
 * stream first waits for the work already queued on `after_stream` (the inputs'
 * producer), then runs the prefill and records a completion event. At most one prefill
 * is in flight per handle: while the previous one runs, the call returns GDN_ERR_BUSY
 * and enqueues nothing. Completion: gdn_prefill_async_query (poll), _wait (block the
 * host) or _join (make another stream wait on the device). gdn_handle_destroy drains the
 * owned stream first. */
gdn_status gdn_prefill_packed_async(gdn_handle* handle, const gdn_config* cfg,
                                    int32_t num_seqs, const int32_t* cu_seqlens_host,
                                    const void* q, const void* k, const void* v,
                                    const float* a, const float* beta,
                                    const float* initial_state,
                                    const int32_t* ckpt_cu_host, const int32_t* ckpt_pos_host,
                                    void* o, float* ckpt_states, float* final_states,
                                    void* workspace, size_t workspace_bytes,
                                    void* after_stream);

/* GDN_OK when no prefill is in flight on the handle's stream (the last one completed),
 * GDN_ERR_DEVICE_TIMEOUT while it is still running ("poll completion events while
 * decode is active", pegainfer PR #786). */
gdn_status gdn_prefill_async_query(gdn_handle* handle);

/* Block the host until the in-flight prefill (if any) has completed ("wait explicitly
 * when the last decoder retires", pegainfer PR #786). */
gdn_status gdn_prefill_async_wait(gdn_handle* handle);

/* Make `stream` wait on the device for the in-flight prefill (if any); returns at once. */
gdn_status gdn_prefill_async_join(gdn_handle* handle, void* stream);

/* One-token decode update for `batch` decoding sequences, each with its own fp32 state in
 * a caller-owned pool, updated in place (vllm.cpp "vLLM, online serving", packed GDN
 * decode lever). For sequence b:
 *     S = state_pool[slot_idx[b]]   ([H_v][d][d] fp32 per slot)
 *     one step of the recurrence with q[b], k[b] ([batch][H_k][d]), v[b] ([batch][H_v][d]),
 *     a[b], beta[b] ([batch][H_v] fp32); o[b] ([batch][H_v][d] io_dtype) = scale * S_new q
 *  slot_idx_dev     [batch] int32 device array of distinct slot indices in [0, num_slots).
 * Distinct slots are the caller's duty (two batch rows naming one slot race).
 * The call checks its arguments on the host and enqueues one kernel on `stream`, with no
 * copy and no allocation, so a serving loop can capture it in a CUDA graph and replay it
 * (the graph then keeps the buffer addresses of the capture; a test replays captured
 * steps and matches direct calls bit for bit).
 * Errors: INVALID_ARGUMENT, UNSUPPORTED, CUDA. */
gdn_status gdn_decode_step(gdn_handle* handle, const gdn_config* cfg, int32_t batch,
                           const void* q, const void* k, const void* v,
                           const float* a, const float* beta,
                           float* state_pool, int32_t num_slots, const int32_t* slot_idx_dev,
                           void* o, void* stream);

/* Bytes of the fixed device scratch behind gdn_prefill_packed_noalloc (per GPU). */
#define GDN_NOALLOC_SCRATCH_BYTES (1u << 20)

/* gdn_prefill_packed for callers that cannot allocate memory when they call in: there is
 * no workspace and no handle argument, and nothing is allocated. The pages describe no
 * such call; it exists for serving engines whose device memory is all handed to their own
 * pool at start-up, and for plugins whose host framework forbids allocation on the request
 * path. Arguments, layouts, results and errors are those of gdn_prefill_packed, except
 * that a device-side timeout is read with gdn_noalloc_read_status (gdn_read_device_status
 * needs a workspace).
 * The work list lives in one file-scope device array of GDN_NOALLOC_SCRATCH_BYTES per GPU
 * (held from library load to process exit); a pack whose work list does not fit returns
 * GDN_ERR_UNSUPPORTED before anything is enqueued. Every call rewrites that array and
 * clears its status word, so calls whose device work may overlap in time (two streams)
 * race and must be serialised by the caller. The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture. That address belongs to the device's primary
 * context: after a cudaDeviceReset in the same process, do not use this entry point. The
 * host copy of the work list is taken from one fixed host buffer under one process-wide
 * lock with a pageable cudaMemcpyAsync, so a call may block the host until work queued
 * earlier on `stream` has drained, and calls on different GPUs run one after another. */
gdn_status gdn_prefill_packed_noalloc(const gdn_config* cfg, int32_t num_seqs,
                                      const int32_t* cu_seqlens_host,
                                      const void* q, const void* k, const void* v,
                                      const float* a, const float* beta,
                                      const float* initial_state,
                                      const int32_t* ckpt_cu_host, const int32_t* ckpt_pos_host,
                                      void* o, float* ckpt_states, float* final_states,
                                      void* stream);

/* Mixed step in one launch, with the states gathered from a pool (sparkinfer v0.6.4 release
 * notes, "What changed": prompt slices under a 1,024-token budget run in the same pass as
 * the decoding requests; vllm.cpp "vLLM, online serving", lever 2b, packed GDN decode).
 * gdn_prefill_packed in which every prompt's state lives in a caller-owned pool and is
 * updated in place: prompt n reads its initial state from state_pool[slot_idx_host[n]]
 * (or starts from a zero state when start_zero_host is non-NULL and start_zero_host[n] !=
 * 0) and writes its final state back to the same slot. Decoding sequences ride the pack as
 * one-token prompts; every (prompt, value head) unit, prompts of one token or none
 * included, runs in one kernel launch (gdn_prefill_launch_count reports it), so a mixed
 * step of prompt slices and decode tokens needs no caller-side state copies and no second
 * launch.
 *  state_pool       [num_slots][H_v][d][d] fp32 device, 16-byte aligned; slots not named by
 *                   slot_idx_host are neither read nor written.
 *  slot_idx_host    [N] int32 host array of distinct slots in [0, num_slots).
 *  start_zero_host  [N] int32 host array or NULL (NULL: every prompt reads its slot).
 * Everything else as gdn_prefill_packed (the workspace size is gdn_prefill_workspace_size's).
 * The pool may not overlap q, k, v, a, beta, o, ckpt_states or the workspace. Errors:
 * INVALID_ARGUMENT (also for a slot out of range or named twice), UNSUPPORTED,
 * WORKSPACE_TOO_SMALL, CUDA. */
gdn_status gdn_prefill_packed_pool(gdn_handle* handle, const gdn_config* cfg, int32_t num_seqs,
                                   const int32_t* cu_seqlens_host,
                                   const void* q, const void* k, const void* v,
                                   const float* a, const float* beta,
                                   float* state_pool, int32_t num_slots,
                                   const int32_t* slot_idx_host, const int32_t* start_zero_host,
                                   const int32_t* ckpt_cu_host, const int32_t* ckpt_pos_host,
                                   void* o, float* ckpt_states,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* Number of kernels that the handle's last prefill call (gdn_prefill_packed and its _pool,
 * _snapshot, _async, _host and _split forms) enqueued: 1 for any pack of
 * gdn_prefill_packed, gdn_prefill_packed_pool or gdn_prefill_packed_snapshot with at least
 * one prompt. Host-side bookkeeping (no CUDA call). Errors: INVALID_ARGUMENT. */
gdn_status gdn_prefill_launch_count(gdn_handle* handle, int32_t* count);

/* The status word that the last gdn_prefill_packed_noalloc call on the current device
 * left (0, or GDN_ERR_DEVICE_TIMEOUT when a bounded device-side wait gave up) into
 * *status_out: a copy from the fixed device array into the caller's int32 on `stream`,
 * which it synchronises. No allocation. The pages have no counterpart. Errors:
 * INVALID_ARGUMENT, UNSUPPORTED (device index beyond 63), CUDA. */
gdn_status gdn_noalloc_read_status(int32_t* status_out, void* stream);

/* Process-wide test hook of gdn_prefill_packed_noalloc for the device-side timeout path,
 * with the meaning of gdn_set_test_hook's hook 1 (0 = off, the default). The pages have no
 * counterpart. Errors: INVALID_ARGUMENT. */
gdn_status gdn_noalloc_set_test_hook(int32_t hook);

/* ---- prefill from host memory ---------------------------------------------------------- */

/* The arrays of one pack, in the layouts of gdn_prefill_packed: inputs q, k, v, a, beta and
 * initial_state (NULL = zeros), outputs o, ckpt_states (NULL when the pack has no
 * checkpoints) and final_states. */
typedef struct {
  void* q;
  void* k;
  void* v;
  float* a;
  float* beta;
  float* initial_state;
  void* o;
  float* ckpt_states;
  float* final_states;
} gdn_prefill_buffers;

/* gdn_prefill_packed for a pack whose inputs and outputs live in host memory. The prompts
 * are processed in groups of up to `group_prompts`: the groups grow 1, 2, 4, ... prompts up
 * to group_prompts at the start and shrink the same way at the end, which keeps short the
 * copy-in that precedes the first prefill and the copy-out that follows the last one. A
 * group's rows of q, k, v, a, beta and its
 * initial states are copied into `device` on the handle's copy-in stream; its prefill runs
 * on `stream` (exactly as gdn_prefill_packed over that group); its o rows, checkpoints and
 * final states are copied back into `host` on the handle's copy-out stream. The copies of
 * neighbouring groups therefore overlap each other and the prefill: about the larger of
 * the two copy volumes over the link rather than their sum. `stream` waits for the last
 * copy out before anything queued after the call. Host buffers should be pinned
 * (cudaHostAlloc) for full copy speed; `device` buffers are the pack-sized device arrays
 * gdn_prefill_packed would take (their inputs are overwritten with the host inputs).
 * Validation is that of gdn_prefill_packed on the whole pack and on `device`. Errors: also
 * INVALID_ARGUMENT for a missing host array or group_prompts < 1, UNSUPPORTED for more than
 * 64 groups. Results equal gdn_prefill_packed's on the whole pack bit for bit (a prompt's
 * results do not depend on its pack, and both chunked schedules agree bit for bit). The
 * workspace holds every group's work list, uploaded in one copy ahead of the bulk copies
 * (gdn_prefill_host_workspace_size). */
/* Device workspace bytes that gdn_prefill_packed_host needs for this pack and group size
 * (the work lists of all groups). A multiple of 256. */
gdn_status gdn_prefill_host_workspace_size(const gdn_config* cfg, int32_t num_seqs,
                                           const int32_t* cu_seqlens_host,
                                           const int32_t* ckpt_cu_host, int32_t group_prompts,
                                           size_t* bytes);

gdn_status gdn_prefill_packed_host(gdn_handle* handle, const gdn_config* cfg,
                                   int32_t num_seqs, const int32_t* cu_seqlens_host,
                                   const int32_t* ckpt_cu_host, const int32_t* ckpt_pos_host,
                                   const gdn_prefill_buffers* host,
                                   const gdn_prefill_buffers* device, int32_t group_prompts,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* ---- sequence splitting ------------------------------------------------------------ */

/* Device workspace bytes that gdn_prefill_packed_split needs for this pack and segment
 * length (work lists of its two passes plus fp32 scratch states: two per segment map and
 * two per split segment). Validates what gdn_prefill_packed_split validates about the
 * pack. Result is a multiple of 256. */
gdn_status gdn_prefill_split_workspace_size(const gdn_config* cfg, int32_t num_seqs,
                                            const int32_t* cu_seqlens_host,
                                            const int32_t* ckpt_cu_host,
                                            const int32_t* ckpt_pos_host, int32_t segment_len,
                                            size_t* bytes);

/* gdn_prefill_packed with prompts longer than `segment_len` tokens cut into segments of
 * `segment_len` (a multiple of 64, >= 64) that run in parallel: more (segment, value head)
 * units for packs with few prompts, such as one very long prompt. The recurrence is affine
 * in a segment's initial state, S_end = S_start M + B; pass 1 computes, for every middle
 * segment, B (from a zero state) and M (from the identity with v taken as zero) next to
 * segment 0 of every prompt; a scan composes the maps in fp32 into each segment's initial
 * state; pass 2 runs segments 1 .. P-1 from those states with their checkpoints. The work
 * is about (2P - 1) / P times that of one pass, in about 2 / P of its sequential chunks.
 * Arguments, layouts and errors are those of gdn_prefill_packed plus `segment_len`
 * (INVALID_ARGUMENT when it is not a positive multiple of 64). Results equal
 * gdn_prefill_packed's to rounding: the composed state carries the maps' fp32 rounding
 * and the fp16 tensor-core operands of each run (the same tolerance applies). Prompts
 * of at most `segment_len` tokens run exactly as in gdn_prefill_packed. `o` is written
 * twice for middle segments (the first write is scratch). */
gdn_status gdn_prefill_packed_split(gdn_handle* handle, const gdn_config* cfg,
                                    int32_t num_seqs, const int32_t* cu_seqlens_host,
                                    const void* q, const void* k, const void* v,
                                    const float* a, const float* beta,
                                    const float* initial_state, const int32_t* ckpt_cu_host,
                                    const int32_t* ckpt_pos_host, void* o, float* ckpt_states,
                                    float* final_states, int32_t segment_len, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* The segment length for gdn_prefill_packed_split that the chunked kernels' cost model
 * (the per-chunk costs of gdn_chunked_schedule) expects to run this pack fastest, or 0 when
 * splitting is not expected to pay (then call gdn_prefill_packed). It compares the whole
 * pack in one launch with P = 2 .. 16 segments of the longest prompt (each a multiple of
 * 64): pass 1 with segment 0 of every prompt plus two map runs per middle segment, pass 2
 * with the later segments, and 12 us for the extra launches. Splitting shortens the longest
 * chain of chunks, so it pays for packs with few (prompt, value head) units per SM and one
 * long prompt, such as one 32K prompt or a ragged pack with one long prompt; the choice
 * depends on the whole pack, so results split this way carry the split path's rounding
 * (gdn_prefill_packed_split) rather than being bit-identical to gdn_prefill_packed's.
 * Host-only, no CUDA call. Errors: INVALID_ARGUMENT (as gdn_chunked_schedule). */
gdn_status gdn_split_segment_auto(int32_t num_seqs, const int32_t* cu_seqlens_host,
                                  int32_t num_v_heads, int32_t num_sms, int32_t* segment_len);

/* ---- host-side scheduling policy (no device work) ---------------------------------- */

/* Prefix-cache checkpoint position of a prompt of `len` tokens on a grid of `block`
 * tokens: the last multiple of `block` that is <= len, moved back one block when it falls
 * within the prompt's last `tail` tokens, so the prompt can stay in the pack (sparkinfer
 * v0.6.28, bullet on checkpoints in the last 16 tokens; there tail = 16). Returns the
 * position, or 0 when no checkpoint remains (len < block after the move). */
int32_t gdn_ckpt_position(int32_t len, int32_t block, int32_t tail);

/* Mixed-step prompt budget (sparkinfer v0.6.4 release notes, "What changed"): walk the
 * waiting prompts oldest first (index order), at most `max_prompts` of them, giving each
 * min(remaining_i, budget_left) tokens until `budget` tokens are used. take_out[i]
 * receives prompt i's share (0 for prompts not served). Returns the number of prompts
 * served, or -1 on invalid arguments. */
int32_t gdn_mixed_budget(int32_t num_waiting, const int32_t* remaining_host, int32_t budget,
                         int32_t max_prompts, int32_t* take_out_host);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
