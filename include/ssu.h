/*
 * ssu.h -- C ABI of the GB300 (sm_103a) Mamba2 selective-state-update decode
 * library (libssu_gb300.so).
 *
 * The operation is the Mamba2 decode step the following pages call
 * selective_state_update:
 *   - "vllm.model_executor.layers.mamba.ops.ssu_dispatch" (vLLM API docs and
 *     ssu_dispatch.py): the unified selective_state_update signature (state,
 *     x, dt, A, B, C, D, dt_bias, z, dt_softplus, state_batch_indices,
 *     dst_state_batch_indices, null_block_id, out, num_accepted_tokens,
 *     cu_seqlens) and the ReplaySSM tracker kernels
 *     _update_replayssm_ring_trackers_kernel /
 *     _commit_replayssm_ring_trackers_kernel with their wrappers
 *     update_/reset_/commit_replayssm_ring_trackers.
 *   - "mate.mamba" (MATE module source): the FlashInfer-shaped contract of
 *     selective_state_update -- supported dtypes and layouts, per-head A/D/
 *     dt_bias (_per_head), one-token route (ssu_one_token, _slot_vector),
 *     packed varlen route (_packed_selective_state_update, _slot_table,
 *     _dense_seq_starts), pad_slot_id and disable_state_update.
 * For every sequence and head, with g = head / (nheads / ngroups):
 *   dt' = dt + dt_bias; dt' = softplus(dt') if dt_softplus; dA = exp(A * dt')
 *   h[p][n] <- h[p][n] * dA + dt' * x[p] * B[g][n]
 *   y[p] = sum_n h[p][n] * C[g][n] + D * x[p];  y *= silu(z[p]) if z given
 * computed in fp32 registers; the state is read once from its slot and the
 * new state (rounded to nearest even in the state dtype) written to the
 * destination slot(s).
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     allocates nothing and never copies device data to the host.  Each
 *     compute or tracker call (ssu_update, ssu_update_varlen,
 *     ssu_replay_update, ssu_ring_update, ssu_ring_commit) issues exactly
 *     one kernel launch on
 *     `stream` (a cudaStream_t; NULL is the legacy default stream), whatever
 *     the batch, and never synchronises, so it can be captured in a CUDA
 *     graph.  The two diagnostic calls (ssu_device_error,
 *     ssu_selftest_bounded_wait) synchronise the device and must not be made
 *     while any stream of the device is being captured.
 *   - Arguments are validated on the host before any launch; a rejected call
 *     launches nothing and changes nothing.  SSU_ERR_INVALID_ARGUMENT mirrors
 *     the pages' ValueError cases, SSU_ERR_UNSUPPORTED their
 *     NotImplementedError cases, SSU_ERR_CUDA a failed launch.
 *     ssu_last_error() gives a message for the calling thread's last failure.
 *   - Slot indices are int32 or int64.  An index equal to pad_slot_id, or
 *     outside [0, slots), is skipped on the device (no read, no write; the
 *     pages' tracker kernels mask the same way); it never faults.
 *   - A call with zero sequences returns SSU_OK without launching.
 *   - Calls that write the same state slot from two sequences race (the
 *     result is undefined), as in the pages' kernels.
 */
#ifndef SSU_GB300_H
#define SSU_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */

typedef enum ssu_status {
  SSU_OK = 0,
  SSU_ERR_INVALID_ARGUMENT = 1, /* shapes, strides, dtypes or values the contract rejects */
  SSU_ERR_UNSUPPORTED = 2,      /* a valid request the library does not implement */
  SSU_ERR_CUDA = 3              /* the kernel launch failed */
} ssu_status;

/*
 * Kernel selection (the pages' SSU entry points carry an `algorithm` choice
 * too: "ssu_dispatch" forwards MambaConfig.ssu_algorithm, "mate.mamba"
 * accepts auto/simple/vertical/horizontal and runs one kernel for all).
 *   SSU_ALGO_AUTO    the library's choice, the faster as measured: BULK for
 *                    ssu_update, DIRECT for ssu_update_varlen and for every
 *                    call with disable_state_update
 *   SSU_ALGO_DIRECT  one CTA per (sequence, run of heads of one group, row
 *                    tile); slot lookups and B / C staged once for the run,
 *                    each head's state tile copied asynchronously into
 *                    shared memory while the previous head computes.  With disable_state_update the steps of
 *                    a chain are taken in closed form (no state is stored,
 *                    so y_t needs only C_t . h, C_t . B_s and products of
 *                    dA); C_t . h on tensor cores (exact 16-bit products,
 *                    fp32 sums) when the state and B / C share a 16-bit type
 *   SSU_ALGO_BULK    persistent CTAs; a producer warp streams each tile into a
 *                    ring of shared-memory stages with one bulk asynchronous
 *                    copy while consumer warps compute
 * For calls that write state both compute the same arithmetic in the same
 * order (bit-identical results); for calls that write none the closed form
 * rounds differently (within the same tolerances).  Calls with stochastic
 * rounding of 16-bit state (rand_seed set) run on the DIRECT kernels
 * whatever the choice: only those carry the generator.
 */
typedef enum ssu_algorithm {
  SSU_ALGO_AUTO = 0,
  SSU_ALGO_DIRECT = 1,
  SSU_ALGO_BULK = 2
} ssu_algorithm;

typedef enum ssu_dtype {
  SSU_F32 = 0,
  SSU_BF16 = 1,
  SSU_F16 = 2,
  SSU_I32 = 3,
  SSU_I64 = 4
} ssu_dtype;

/*
 * Operands of one selective-state-update call (both routes).  Strides are in
 * ELEMENTS.  Rows are packed tokens: the one-token route has one row per
 * sequence, the varlen route `rows` rows split by cu_seqlens.
 *
 * state      [slots, nheads, headdim, dstate], contiguous, 16-byte aligned,
 *            F32 / BF16 / F16 ("mate.mamba": state fp16/bf16/fp32,
 *            contiguous).  Read and written in place.
 * io_dtype   BF16 or F16: the dtype of x, z, B and C.
 * x          [rows, nheads, headdim]: element (r, h, p) at
 *            x[r * x_row_stride + h * x_head_stride + p].
 * z          same layout as x, or NULL (no silu gate).
 * out        y, same layout as x with its own strides; out_dtype is io_dtype
 *            (the contract) or F32 (full-precision output, an extension of
 *            this library).  Written for every row a sequence covers.
 * dt         fp32, element (r, h, p) at
 *            dt[r * dt_row_stride + h * dt_head_stride + p * dt_dim_stride];
 *            dt_dim_stride = 0 is the per-head form [rows, nheads(, 1)].
 * B, C       [rows, ngroups, dstate], io_dtype: element (r, g, n) at
 *            B[r * B_row_stride + g * B_group_stride + n].
 * A, D, dt_bias  fp32, element (h, p) at A[h * A_stride + p * A_dim_stride]
 *            (likewise D, dt_bias): a dim stride of 0 is the per-head (tied)
 *            form, a nonzero one the per-(head, dim) channel form
 *            ("mate.mamba", _per_head).  D and dt_bias may be NULL (0).
 * dt_softplus, disable_state_update: flags (0 / 1).
 * pad_slot_id: slot id that marks a padded entry (vLLM passes its null
 *            block id; "mate.mamba" defaults to -1).
 * algorithm  an ssu_algorithm (0 = auto).
 * rand_seed  NULL: state is stored rounded to nearest even.  Otherwise a
 *            DEVICE pointer to this call's 64-bit random seed ("ssu_dispatch":
 *            rand_seed drawn per call when stochastic rounding is enabled),
 *            8-byte aligned: every value stored into a bf16 / fp16 pool is
 *            rounded stochastically -- away from zero with probability equal
 *            to its fraction between the format's two neighbours, to 16
 *            bits.  Stored element e (its index in the pool) takes the 16 bits
 *            16 (e mod 4) .. 16 (e mod 4) + 15 of word (e / 4) mod 4 of the
 *            Philox4x64 block with counter (e / 16, 0, 0, 0) and key
 *            (seed, 0).  fp32 pools ignore it.
 * philox_rounds  Philox rounds; <= 0 means 10 ("ssu_dispatch":
 *            philox_rounds ... or 10).
 */
typedef struct ssu_params {
  void* state;
  ssu_dtype state_dtype;
  int64_t slots, nheads, headdim, dstate, ngroups;
  ssu_dtype io_dtype;
  const void* x;
  int64_t x_row_stride, x_head_stride;
  const void* z;
  int64_t z_row_stride, z_head_stride;
  void* out;
  ssu_dtype out_dtype;
  int64_t out_row_stride, out_head_stride;
  const float* dt;
  int64_t dt_row_stride, dt_head_stride, dt_dim_stride;
  const void* B;
  int64_t B_row_stride, B_group_stride;
  const void* C;
  int64_t C_row_stride, C_group_stride;
  const float* A;
  int64_t A_stride, A_dim_stride;
  const float* D;
  int64_t D_stride, D_dim_stride;
  const float* dt_bias;
  int64_t dt_bias_stride, dt_bias_dim_stride;
  int dt_softplus;
  int disable_state_update;
  int64_t pad_slot_id;
  int algorithm; /* ssu_algorithm */
  const uint64_t* rand_seed;
  int philox_rounds;
} ssu_params;

/*
 * A slot table of the packed route ("mate.mamba", _slot_table): entry
 * (sequence s, position t) is indices[s * seq_stride + t * step_stride].  A
 * flat [rows] table has strides (1, 1); a [sequences, steps] table
 * (steps, 1).  Positions t >= steps, or entries at or beyond numel, do not
 * exist (treated like a pad entry).  indices == NULL means "no table".
 */
typedef struct ssu_slot_table {
  const void* indices;
  int64_t numel;
  int64_t seq_stride, step_stride;
  int64_t steps;
} ssu_slot_table;

/*
 * One-token decode: sequence b is row b of x/dt/B/C/z/out, b in [0, batch).
 * ("mate.mamba": ssu_one_token route and _slot_vector; "ssu_dispatch":
 * selective_state_update without cu_seqlens.)
 *   state_batch_indices      [batch] read slots, or NULL for slot b
 *                            (then batch must not exceed slots).
 *   dst_state_batch_indices  [batch] write slots, or NULL to write back to
 *                            the read slot (in place).
 *   index_dtype              SSU_I32 or SSU_I64 for both tables.
 * A sequence whose read slot is pad / out of range runs from a zero state and
 * writes no state; y is still produced.  A pad / out-of-range write slot
 * skips only that write.  disable_state_update writes no state at all.
 */
ssu_status ssu_update(const ssu_params* p, int64_t batch,
                      const void* state_batch_indices,
                      const void* dst_state_batch_indices,
                      ssu_dtype index_dtype,
                      struct CUstream_st* stream);

/*
 * Packed variable-length / speculative (MTP) update.  ("mate.mamba":
 * ssu_packed_varlen route, _packed_selective_state_update, dense 4-D
 * folding via _dense_seq_starts; "ssu_dispatch": selective_state_update with
 * cu_seqlens and num_accepted_tokens.)
 *   nseqs, rows          sequences and packed rows of this call.
 *   cu_seqlens           [nseqs + 1] row starts (int, meta_dtype); sequence s
 *                        owns rows [cu[s], cu[s+1]).  NULL: the dense form,
 *                        every sequence owns `dense_steps` consecutive rows
 *                        (rows must equal nseqs * dense_steps).
 *   num_accepted_tokens  [nseqs] (meta_dtype) or NULL.  Sequence s reads its
 *                        state from position num_accepted[s] - 1 of `src`
 *                        (position 0 when NULL).  Requires a src table.
 *   meta_dtype           SSU_I32 / SSU_I64 for cu_seqlens and
 *                        num_accepted_tokens (they share it, as the pages
 *                        require).
 *   src                  read table, or NULL / indices NULL: sequence s reads
 *                        slot s (then nseqs must not exceed slots).
 *   dst                  write table: step t of sequence s writes position t.
 *                        NULL / indices NULL: the read table's position t
 *                        (or slot s when there is no read table either).
 *   index_dtype          SSU_I32 / SSU_I64 for both tables.
 * The chain over a sequence's rows stays in fp32 registers; each step's state
 * is rounded only when it is written to its destination slot.  An empty
 * sequence reads and writes nothing.  A read position outside the table, or a
 * pad / out-of-range read slot, runs from a zero state and writes no state.
 * Row ranges are clamped to [0, rows).
 */
ssu_status ssu_update_varlen(const ssu_params* p, int64_t nseqs, int64_t rows,
                             const void* cu_seqlens, int64_t dense_steps,
                             const void* num_accepted_tokens, ssu_dtype meta_dtype,
                             const ssu_slot_table* src, const ssu_slot_table* dst,
                             ssu_dtype index_dtype,
                             struct CUstream_st* stream);

/*
 * ReplaySSM ring-tracker update or reset ("ssu_dispatch":
 * _update_replayssm_ring_trackers_kernel, update_replayssm_ring_trackers,
 * reset_replayssm_ring_trackers).  Trackers are int32 vectors indexed by
 * slot; num_states is the shortest of the three lengths.  Sequence i's slot
 * is state_batch_indices[i * sbi_stride] (pass the row length of a 2-D
 * table to use its column 0).
 *   reset != 0: zero all three trackers of every valid slot
 *               (logical_window / ring_buffer_len are ignored).
 *   reset == 0: with prev = prev_num_accepted[slot], start = ring_start[slot]:
 *               if prev + 1 > logical_window:
 *                   ring_start = (start + prev) % ring_buffer_len; prev = 1
 *               else prev = prev + 1.   prev_query_len is left unchanged.
 * int32 arithmetic wraps; % truncates toward zero.  ring_buffer_len must be
 * >= 1 when reset == 0.
 */
ssu_status ssu_ring_update(int32_t* ring_start, int64_t ring_start_len,
                           int32_t* prev_num_accepted, int64_t prev_num_accepted_len,
                           int32_t* prev_query_len, int64_t prev_query_len_len,
                           const void* state_batch_indices, int64_t sbi_stride,
                           ssu_dtype index_dtype, int64_t nseqs, int reset,
                           int32_t logical_window, int32_t ring_buffer_len,
                           int64_t pad_slot_id, struct CUstream_st* stream);

/*
 * ReplaySSM ring-tracker commit of the previous speculative window
 * ("ssu_dispatch": _commit_replayssm_ring_trackers_kernel,
 * commit_replayssm_ring_trackers).  Slots as in ssu_ring_update.  For a
 * valid slot of sequence i, with acc = prev_num_accepted[slot],
 * start = ring_start[slot], pql = prev_query_len[slot],
 * a = num_accepted_tokens[i]:
 *   must = pql > 0 && acc + pql > logical_window
 *   ring_start        = must ? (start + acc) % ring_buffer_len : start
 *   prev_num_accepted = pql == 0 ? 0 : (must ? a : acc + a)
 *   prev_query_len    = query_start_loc[i + 1] - query_start_loc[i]
 * num_accepted_tokens [nseqs] and query_start_loc [nseqs + 1] are meta_dtype
 * (I32 / I64); stored values wrap to int32.  ring_buffer_len must be >= 1.
 */
ssu_status ssu_ring_commit(int32_t* ring_start, int64_t ring_start_len,
                           int32_t* prev_num_accepted, int64_t prev_num_accepted_len,
                           int32_t* prev_query_len, int64_t prev_query_len_len,
                           const void* state_batch_indices, int64_t sbi_stride,
                           ssu_dtype index_dtype,
                           const void* num_accepted_tokens, const void* query_start_loc,
                           ssu_dtype meta_dtype, int64_t nseqs,
                           int32_t logical_window, int32_t ring_buffer_len,
                           int64_t pad_slot_id, struct CUstream_st* stream);

/*
 * ReplaySSM ring caches and trackers of a checkpointing update
 * ("ssu_dispatch": selective_state_update_replayssm_flashinfer, the FlashInfer
 * checkpointing_ssu call it wraps; ring semantics of
 * _update_/_commit_replayssm_ring_trackers_kernel).  All device memory owned
 * by the caller, contiguous; R = ring_len positions per slot.
 *   x_cache            [slots, nheads, R, headdim], io_dtype
 *   B_cache            [slots, ngroups, R, dstate], io_dtype
 *   dt_cache           [slots, nheads, R], fp32 (dt as given: before dt_bias
 *                      and softplus)
 *   ring_start, prev_num_accepted   int32 trackers indexed by slot, at least
 *                      num_states entries each (prev_query_len is not used:
 *                      the one-token tracker rule leaves it unchanged)
 *   logical_window     W: a checkpoint is written when k + L > W
 */
typedef struct ssu_replay_cache {
  void* x_cache;
  void* B_cache;
  float* dt_cache;
  int64_t ring_len;
  int32_t* ring_start;
  int32_t* prev_num_accepted;
  int64_t num_states;
  int32_t logical_window;
} ssu_replay_cache;

/*
 * ReplaySSM checkpointing update (one launch).  state[slot] holds a
 * checkpoint; the slot's state is the checkpoint advanced through the
 * k = prev_num_accepted[slot] tokens cached at ring positions
 * (ring_start[slot] + j) mod R, j < k.  For every sequence s (slot
 * state_batch_indices[s], or s when NULL; rows [cu[s], cu[s+1]), or row s
 * when cu_seqlens is NULL -- then rows == nseqs):
 *   1. replay the k cached tokens (the plain recurrence with this call's A,
 *      dt_bias, dt_softplus) from the checkpoint;
 *   2. if k + L > logical_window, round that state to the state dtype and
 *      write it to state[slot] (the new checkpoint);
 *   3. run the L rows as the plain update does (y into out; z gate; D), and
 *      cache row t's x, B and dt at ring position (ring_start + k + t) mod R;
 *   4. with update_trackers, apply ssu_ring_update's one-token rule to the
 *      slot (what the pages' wrapper runs after the kernel), in this launch.
 *      MTP callers pass 0 and call ssu_ring_commit on their next pass.
 * A sequence is skipped (rows from a zero state, nothing written: no
 * checkpoint, ring entry or tracker) when its slot is pad_slot_id or outside
 * [0, min(slots, num_states)), when it has no rows, or when its trackers are
 * out of range (k < 0, k + L > R, ring_start outside [0, R)).  A ring of
 * max(W, longest pass) + longest pass positions holds every pass after a
 * commit.
 *   p                 operands as for ssu_update_varlen; dt must be per head
 *                     (dt_dim_stride 0: the ring caches one dt per head),
 *                     disable_state_update must be 0; p->algorithm is ignored.
 *   meta_dtype        I32 / I64 of cu_seqlens; index_dtype of
 *                     state_batch_indices, whose entry for sequence s is at
 *                     s * sbi_stride (the row length of a 2-D table: its
 *                     column 0, as the pages' wrapper takes).
 *   scratch           with update_trackers: nseqs uint32 arrival counters
 *                     (scratch_bytes >= 4 * nseqs), all ZERO before the first
 *                     call; every completed call leaves them zero.  Unused
 *                     (may be NULL) without update_trackers.  Two calls that
 *                     share counters must not overlap on the device.
 * Errors as for the other calls; rows must be below 2^31 and ring_len in
 * [1, 2^20].
 */
ssu_status ssu_replay_update(const ssu_params* p, const ssu_replay_cache* rc, int64_t nseqs,
                             int64_t rows, const void* cu_seqlens, ssu_dtype meta_dtype,
                             const void* state_batch_indices, int64_t sbi_stride,
                             ssu_dtype index_dtype, int update_trackers, void* scratch,
                             int64_t scratch_bytes, struct CUstream_st* stream);

/*
 * ssu_replay_update without a scratch argument (the pages have no counterpart
 * of this entry point).  ssu_replay_update's tracker update counts the CTAs of
 * each sequence in caller-provided scratch.  Some callers cannot hand the
 * library such a buffer: a plugin host that gives an operation only its own
 * inputs and outputs, or a serving runtime that plans all device memory at
 * start-up and forbids allocations afterwards (a cudaMalloc can synchronise
 * the device and break a pre-planned pool).  This entry point keeps the
 * counters in a fixed array inside the library instead and allocates nothing:
 * no cudaMalloc, cudaFree or allocating library routine.
 *   - Arguments and behaviour as ssu_replay_update, without scratch.
 *   - At most SSU_REPLAY_STATIC_MAX_SEQS sequences per call; more is rejected
 *     (SSU_ERR_INVALID_ARGUMENT) before anything runs.  The array is 256 KB
 *     of device memory on every GPU that loads the library, held until the
 *     process exits.
 *   - The first call on a device looks up the array's device address (once
 *     per device, on the current device); make that first call before any
 *     stream capture on the device.
 *   - Every call on a device shares the one array and it keeps what the last
 *     call left there: with update_trackers, each call clears the counters it
 *     uses (an asynchronous memset on `stream`, which is issued before the
 *     arguments are checked; the counters are the library's own, so a rejected
 *     call still changes nothing the caller holds).  Calls whose work overlaps
 *     on the device -- on different streams, or from different threads --
 *     race on the counters and must not be made.
 */
#define SSU_REPLAY_STATIC_MAX_SEQS 65536
ssu_status ssu_replay_update_static(const ssu_params* p, const ssu_replay_cache* rc,
                                    int64_t nseqs, int64_t rows, const void* cu_seqlens,
                                    ssu_dtype meta_dtype, const void* state_batch_indices,
                                    int64_t sbi_stride, ssu_dtype index_dtype,
                                    int update_trackers, struct CUstream_st* stream);

/*
 * Packed variable-length SSD prefill ("mate.mamba": ssd_combined_fwd_varlen
 * and its five stages cumsum / chunk_state / state_passing / bmm /
 * chunk_scan).  Over the chunks of a packed batch it computes what the
 * one-token update computes token by token -- dt' = clamp(softplus(dt +
 * dt_bias), dt_min, dt_max) -- and returns the states at chunk ends.
 *   x, z, out     [tokens, nheads, headdim], io_dtype (BF16 / F16),
 *                 contiguous, 16-byte aligned; z may be NULL; out written for
 *                 every token a chunk covers
 *   dt            [tokens, nheads] fp32; A, dt_bias [nheads] fp32 (dt_bias
 *                 may be NULL); D [nheads] or, with D_per_dim, [nheads,
 *                 headdim] fp32, or NULL
 *   B, C          [tokens, ngroups, dstate], io_dtype, contiguous
 *   cu_chunk_seqlens [nchunks + 1]: chunk c covers tokens
 *                 [cu[c], cu[c+1]) (at most chunk_size of them); seq_idx
 *                 [nchunks]: the sequence owning chunk c -- a chunk opens a
 *                 sequence when seq_idx changes, and then starts from
 *                 initial_states[seq_idx[c]] (zeros when NULL);
 *                 last_chunk_indices [batch]: sequence b's last chunk.  All
 *                 meta_dtype (I32 / I64).
 *   initial_states [batch, nheads, headdim, dstate] in initial_dtype, or NULL
 *                 (16-byte aligned, like states)
 *   states        return_intermediate_states: [nchunks, nheads, headdim,
 *                 dstate], every chunk's end state; else [batch, ...], the
 *                 end state of each sequence's last chunk (chunk c is
 *                 sequence seq_idx[c]'s last when last_chunk_indices says so).
 *                 In state_dtype (F32 / BF16 / F16), rounded to nearest even.
 *   workspace     device memory of ssd_workspace_bytes(...) bytes, 16-byte
 *                 aligned, owned by the caller (no contents need be kept
 *                 between calls; calls that share it must not overlap).
 * Supported: headdim 64, dstate 64 or 128, chunk_size a multiple of 16 up to
 * 256, nheads up to 65535, fewer than 2^30 chunks.  Three kernel launches on
 * `stream`: chunk states, state passing, and the scan (which forms C . B^T
 * itself, on the tensor cores).  A tensor-core wait that gives up sets
 * SSU_DEVICE_ERR_MMA_TIMEOUT in the device error word (no valid call does).
 */
typedef struct ssd_params {
  const void* x;
  const float* dt;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  int D_per_dim;
  const void* z;
  const float* dt_bias;
  int dt_softplus;
  float dt_min, dt_max;
  void* out;
  ssu_dtype io_dtype;
  int64_t tokens, nheads, headdim, dstate, ngroups, chunk_size;
  int64_t nchunks, batch;
  const void* cu_chunk_seqlens;
  const void* seq_idx;
  const void* last_chunk_indices;
  ssu_dtype meta_dtype;
  const void* initial_states;
  ssu_dtype initial_dtype;
  void* states;
  ssu_dtype state_dtype;
  int return_intermediate_states;
} ssd_params;

/* Workspace bytes ssd_combined_fwd_varlen needs for these sizes (-1 for a
 * negative size): every chunk's local state (fp32) and entering state (two
 * 16-bit parts), and dt' and the running sum of A dt' per token and head. */
int64_t ssd_workspace_bytes(int64_t nchunks, int64_t nheads, int64_t ngroups, int64_t headdim,
                            int64_t dstate, int64_t chunk_size);

ssu_status ssd_combined_fwd_varlen(const ssd_params* p, void* workspace, int64_t workspace_bytes,
                                   struct CUstream_st* stream);

/*
 * Bits of the device-side error word (values, not bit positions).
 */
#define SSU_DEVICE_ERR_COPY_TIMEOUT 1u    /* a state tile copy never landed */
#define SSU_DEVICE_ERR_RELEASE_TIMEOUT 2u /* a shared-memory stage was never released */
#define SSU_DEVICE_ERR_MMA_TIMEOUT 4u     /* a tensor-core MMA or copy of the SSD scan never completed */

/*
 * Device-side error word of the current device: nonzero after a kernel gave
 * up a bounded wait (a mask of the SSU_DEVICE_ERR_* values above).  No valid
 * call sets it; it exists so that a fault in the copy engine ends a kernel
 * instead of hanging it.  There is one word per device, shared by every call
 * and every host thread: a word set by one call stays set until it is reset.
 * This call SYNCHRONISES the current device; reset != 0 clears the word
 * afterwards.
 */
ssu_status ssu_device_error(unsigned int* value, int reset);

/*
 * Self-test of the bounded waits (no counterpart on the pages): launches, on
 * the current device's legacy default stream, one CTA that waits on an
 * mbarrier nothing completes; the wait must give up after limit_ns (0 <
 * limit_ns <= 1e9), set SSU_DEVICE_ERR_COPY_TIMEOUT in the device error word
 * and return, leaving the context usable.  *waited_ns receives the measured
 * wait.  SYNCHRONISES the device.  The measured wait is kept in one fixed
 * device word shared by all calls, and the test sets the same error word as
 * the compute kernels: self-tests that overlap each other, or compute calls
 * in flight, race on those words, so run it alone and reset the error word
 * afterwards (ssu_device_error(&v, 1)).
 */
ssu_status ssu_selftest_bounded_wait(uint64_t limit_ns, uint64_t* waited_ns);

/* Static description of a status code. */
const char* ssu_status_string(ssu_status status);

/* Message of the calling thread's last failed call ("" if none). */
const char* ssu_last_error(void);

/* ABI version of this header (bumped on any incompatible change). */
#define SSU_ABI_VERSION 4
int ssu_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSU_GB300_H */
