// ssu_abi.cu -- the C ABI of include/ssu.h: host-side validation, operand
// normalisation and dispatch to the typed kernels.  Every check here runs
// before any launch; a rejected call launches nothing.
//
// The checks follow the call contract on "mate.mamba" (selective_state_update,
// _per_head, _slot_vector, _slot_table, _packed_selective_state_update) and the
// tracker wrappers on "vllm.model_executor.layers.mamba.ops.ssu_dispatch".
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/ssu.h"
#include "ssu_launch.cuh"

namespace ssu {
constexpr int kMaxDevices = 64;
}

// Error word of the bulk-copy kernels (one per device: module memory).
__device__ unsigned int g_ssu_device_error = 0;
// Duration the last bounded-wait self-test waited (module memory).
__device__ unsigned long long g_ssu_selftest_waited_ns = 0;

namespace ssu {

unsigned* device_error_word() {
  static std::mutex mu;
  static unsigned* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_ssu_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned*>(a);
  }
  return addr[dev];
}

int sm_count() {
  static std::mutex mu;
  static int count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (count[dev] == 0) {
    int c = 0;
    cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    count[dev] = c > 0 ? c : 1;
  }
  return count[dev];
}

}  // namespace ssu

namespace {

thread_local std::string g_last_error;

ssu_status fail(ssu_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

ssu_status ok() {
  g_last_error.clear();
  return SSU_OK;
}

}  // namespace

namespace ssu {
// Record a failure of an entry point defined in another translation unit.
ssu_status record_error(ssu_status code, const char* message) {
  return fail(code, "%s", message);
}
}  // namespace ssu

namespace {

bool is_index(ssu_dtype d) { return d == SSU_I32 || d == SSU_I64; }

const char* dtype_name(ssu_dtype d) {
  switch (d) {
    case SSU_F32: return "f32";
    case SSU_BF16: return "bf16";
    case SSU_F16: return "f16";
    case SSU_I32: return "i32";
    case SSU_I64: return "i64";
  }
  return "unknown";
}

bool supported_dstate(int64_t n) {
  return n == 16 || n == 32 || n == 64 || n == 128 || n == 256;
}

// Validate the operands shared by both routes and fill the kernel parameters.
ssu_status check_params(const ssu_params* p, ssu::KParams* k) {
  if (!p) return fail(SSU_ERR_INVALID_ARGUMENT, "params must not be NULL");
  if (p->state_dtype != SSU_F32 && p->state_dtype != SSU_BF16 && p->state_dtype != SSU_F16)
    return fail(SSU_ERR_UNSUPPORTED, "state dtype must be f32, bf16 or f16, got %s",
                dtype_name(p->state_dtype));
  if (p->io_dtype != SSU_BF16 && p->io_dtype != SSU_F16)
    return fail(SSU_ERR_UNSUPPORTED, "x/z/B/C dtype must be bf16 or f16, got %s",
                dtype_name(p->io_dtype));
  if (p->out_dtype != p->io_dtype && p->out_dtype != SSU_F32)
    return fail(SSU_ERR_INVALID_ARGUMENT, "out must have the x dtype (%s) or f32, got %s",
                dtype_name(p->io_dtype), dtype_name(p->out_dtype));
  if (p->slots < 0 || p->nheads < 1 || p->headdim < 1 || p->dstate < 1 || p->ngroups < 1)
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "state must be [slots, heads, dim, dstate] with positive sizes, got "
                "[%lld, %lld, %lld, %lld], ngroups %lld",
                (long long)p->slots, (long long)p->nheads, (long long)p->headdim,
                (long long)p->dstate, (long long)p->ngroups);
  if (p->nheads > (1 << 20) || p->headdim > (1 << 20))
    return fail(SSU_ERR_UNSUPPORTED, "nheads and headdim must not exceed 2^20");
  if (p->nheads % p->ngroups != 0)
    return fail(SSU_ERR_INVALID_ARGUMENT, "nheads (%lld) must be a multiple of ngroups (%lld)",
                (long long)p->nheads, (long long)p->ngroups);
  if (!supported_dstate(p->dstate))
    return fail(SSU_ERR_UNSUPPORTED, "dstate %lld is not one of 16, 32, 64, 128, 256",
                (long long)p->dstate);
  if (!p->state && p->slots > 0) return fail(SSU_ERR_INVALID_ARGUMENT, "state must not be NULL");
  if (reinterpret_cast<uintptr_t>(p->state) % 16 != 0)
    return fail(SSU_ERR_INVALID_ARGUMENT, "state must be 16-byte aligned");
  if (!p->x || !p->out || !p->dt || !p->B || !p->C || !p->A)
    return fail(SSU_ERR_INVALID_ARGUMENT, "x, out, dt, B, C and A must not be NULL");
  if (p->algorithm != SSU_ALGO_AUTO && p->algorithm != SSU_ALGO_DIRECT &&
      p->algorithm != SSU_ALGO_BULK)
    return fail(SSU_ERR_INVALID_ARGUMENT, "algorithm must be auto, direct or bulk, got %d",
                p->algorithm);

  k->state = p->state;
  k->slots = p->slots;
  k->H = (int)p->nheads;
  k->P = (int)p->headdim;
  k->hr = (int)(p->nheads / p->ngroups);
  k->tiles = 1;
  k->x = p->x;
  k->x_rs = p->x_row_stride;
  k->x_hs = p->x_head_stride;
  k->z = p->z;
  k->z_rs = p->z_row_stride;
  k->z_hs = p->z_head_stride;
  k->out = p->out;
  k->o_rs = p->out_row_stride;
  k->o_hs = p->out_head_stride;
  k->out_f32 = p->out_dtype == SSU_F32;
  k->dt = p->dt;
  k->dt_rs = p->dt_row_stride;
  k->dt_hs = p->dt_head_stride;
  k->dt_ds = p->dt_dim_stride;
  k->B = p->B;
  k->B_rs = p->B_row_stride;
  k->B_gs = p->B_group_stride;
  k->C = p->C;
  k->C_rs = p->C_row_stride;
  k->C_gs = p->C_group_stride;
  {
    // 16-bit B / C: 8 elements per 16 bytes
    auto a16 = [](const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
    k->bc_vec16 = a16(p->B) && a16(p->C) && p->B_row_stride % 8 == 0 &&
                  p->B_group_stride % 8 == 0 && p->C_row_stride % 8 == 0 &&
                  p->C_group_stride % 8 == 0;
    k->xz_vec16 = a16(p->x) && p->x_row_stride % 8 == 0 && p->x_head_stride % 8 == 0 &&
                  (!p->z || (a16(p->z) && p->z_row_stride % 8 == 0 &&
                             p->z_head_stride % 8 == 0)) &&
                  p->headdim % 8 == 0;
  }
  k->A = p->A;
  k->A_s = p->A_stride;
  k->A_ds = p->A_dim_stride;
  k->D = p->D;
  k->D_s = p->D_stride;
  k->D_ds = p->D_dim_stride;
  k->dt_bias = p->dt_bias;
  k->bias_s = p->dt_bias_stride;
  k->bias_ds = p->dt_bias_dim_stride;
  k->softplus = p->dt_softplus != 0;
  k->disable = p->disable_state_update != 0;
  k->pad = p->pad_slot_id;
  if (reinterpret_cast<uintptr_t>(p->rand_seed) % 8 != 0)
    return fail(SSU_ERR_INVALID_ARGUMENT, "rand_seed must be 8-byte aligned");
  if (p->philox_rounds > 64)
    return fail(SSU_ERR_INVALID_ARGUMENT, "philox_rounds must be at most 64, got %d",
                p->philox_rounds);
  k->sr_seed = reinterpret_cast<const unsigned long long*>(p->rand_seed);
  k->sr_rounds = p->philox_rounds > 0 ? p->philox_rounds : 10;
  return SSU_OK;
}

cudaError_t dispatch(const ssu_params* p, bool varlen, const ssu::KParams& k,
                     const ssu::OneTokenArgs* oa, const ssu::VarlenArgs* va, int64_t nitems,
                     cudaStream_t stream) {
  const bool io_bf16 = p->io_dtype == SSU_BF16;
  const int N = (int)p->dstate;
  switch (p->state_dtype) {
    case SSU_F32:
      return ssu::launch_state_f32(N, io_bf16, varlen, k, oa, va, nitems, stream, p->algorithm);
    case SSU_BF16:
      return ssu::launch_state_bf16(N, io_bf16, varlen, k, oa, va, nitems, stream, p->algorithm);
    case SSU_F16:
      return ssu::launch_state_f16(N, io_bf16, varlen, k, oa, va, nitems, stream, p->algorithm);
    default: return cudaErrorInvalidValue;
  }
}

ssu_status check_table(const ssu_slot_table* t, const char* name, ssu::TableArgs* out) {
  *out = ssu::TableArgs{nullptr, 0, 0, 0, 0};
  if (!t || !t->indices) return SSU_OK;
  if (t->numel < 0 || t->steps < 0)
    return fail(SSU_ERR_INVALID_ARGUMENT, "%s: numel and steps must be >= 0", name);
  *out = ssu::TableArgs{t->indices, t->numel, t->seq_stride, t->step_stride, t->steps};
  return SSU_OK;
}

}  // namespace

#pragma GCC visibility push(default)
extern "C" {

ssu_status ssu_update(const ssu_params* p, int64_t batch, const void* state_batch_indices,
                      const void* dst_state_batch_indices, ssu_dtype index_dtype,
                      struct CUstream_st* stream) {
  ssu::KParams k;
  ssu_status st = check_params(p, &k);
  if (st != SSU_OK) return st;
  if (batch < 0) return fail(SSU_ERR_INVALID_ARGUMENT, "batch must be >= 0");
  if ((state_batch_indices || dst_state_batch_indices) && !is_index(index_dtype))
    return fail(SSU_ERR_INVALID_ARGUMENT, "state_batch_indices must be int32 or int64, got %s",
                dtype_name(index_dtype));
  if (!state_batch_indices && batch > p->slots)
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "without state_batch_indices sequence b uses slot b: batch %lld exceeds %lld "
                "slots",
                (long long)batch, (long long)p->slots);
  if (batch == 0) return ok();
  ssu::OneTokenArgs a{state_batch_indices, dst_state_batch_indices, index_dtype == SSU_I64};
  cudaError_t e = dispatch(p, false, k, &a, nullptr, batch, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return ok();
}

ssu_status ssu_update_varlen(const ssu_params* p, int64_t nseqs, int64_t rows,
                             const void* cu_seqlens, int64_t dense_steps,
                             const void* num_accepted_tokens, ssu_dtype meta_dtype,
                             const ssu_slot_table* src, const ssu_slot_table* dst,
                             ssu_dtype index_dtype, struct CUstream_st* stream) {
  ssu::KParams k;
  ssu_status st = check_params(p, &k);
  if (st != SSU_OK) return st;
  if (nseqs < 0 || rows < 0) return fail(SSU_ERR_INVALID_ARGUMENT, "nseqs and rows must be >= 0");
  ssu::TableArgs ts, td;
  if ((st = check_table(src, "state_batch_indices", &ts)) != SSU_OK) return st;
  if ((st = check_table(dst, "dst_state_batch_indices", &td)) != SSU_OK) return st;
  if ((ts.idx || td.idx) && !is_index(index_dtype))
    return fail(SSU_ERR_INVALID_ARGUMENT, "slot tables must be int32 or int64, got %s",
                dtype_name(index_dtype));
  if ((cu_seqlens || num_accepted_tokens) && !is_index(meta_dtype))
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "cu_seqlens / num_accepted_tokens must be int32 or int64, got %s",
                dtype_name(meta_dtype));
  if (num_accepted_tokens && !ts.idx)
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "num_accepted_tokens selects the read slot, so it needs state_batch_indices "
                "to read it from");
  if (!cu_seqlens) {
    if (dense_steps < 1)
      return fail(SSU_ERR_INVALID_ARGUMENT, "without cu_seqlens dense_steps must be >= 1");
    if (nseqs * dense_steps != rows)
      return fail(SSU_ERR_INVALID_ARGUMENT,
                  "without cu_seqlens %lld rows cannot be split into %lld sequences of %lld "
                  "steps",
                  (long long)rows, (long long)nseqs, (long long)dense_steps);
  }
  if (!ts.idx && nseqs > p->slots)
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "without state_batch_indices sequence s uses slot s: %lld sequences exceed %lld "
                "slots",
                (long long)nseqs, (long long)p->slots);
  if (nseqs == 0) return ok();
  ssu::VarlenArgs a{};
  a.rows = rows;
  a.cu = cu_seqlens;
  a.dense_steps = dense_steps;
  a.na = num_accepted_tokens;
  a.meta64 = meta_dtype == SSU_I64;
  a.src = ts;
  a.dst = td;
  a.idx64 = index_dtype == SSU_I64;
  cudaError_t e = dispatch(p, true, k, nullptr, &a, nseqs, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return ok();
}

ssu_status ssu_replay_update(const ssu_params* p, const ssu_replay_cache* rc, int64_t nseqs,
                             int64_t rows, const void* cu_seqlens, ssu_dtype meta_dtype,
                             const void* state_batch_indices, int64_t sbi_stride,
                             ssu_dtype index_dtype, int update_trackers, void* scratch,
                             int64_t scratch_bytes, struct CUstream_st* stream) {
  ssu::KParams k;
  ssu_status st = check_params(p, &k);
  if (st != SSU_OK) return st;
  if (p->disable_state_update)
    return fail(SSU_ERR_UNSUPPORTED,
                "the checkpointing update has no disable_state_update (it always caches)");
  if (p->dt_dim_stride != 0)
    return fail(SSU_ERR_UNSUPPORTED,
                "the checkpointing update caches one dt per head: dt must be per head");
  if (!rc) return fail(SSU_ERR_INVALID_ARGUMENT, "the replay cache must not be NULL");
  if (nseqs < 0 || rows < 0) return fail(SSU_ERR_INVALID_ARGUMENT, "nseqs and rows must be >= 0");
  if (rows > 0x7fffffffLL) return fail(SSU_ERR_UNSUPPORTED, "rows must be below 2^31");
  if (rc->ring_len < 1 || rc->ring_len > (1 << 20))
    return fail(SSU_ERR_INVALID_ARGUMENT, "ring_len must be in [1, 2^20], got %lld",
                (long long)rc->ring_len);
  if (rc->num_states < 0) return fail(SSU_ERR_INVALID_ARGUMENT, "num_states must be >= 0");
  if (nseqs > 0 && (!rc->x_cache || !rc->B_cache || !rc->dt_cache || !rc->ring_start ||
                    !rc->prev_num_accepted))
    return fail(SSU_ERR_INVALID_ARGUMENT, "the ring caches and trackers must not be NULL");
  if (state_batch_indices && !is_index(index_dtype))
    return fail(SSU_ERR_INVALID_ARGUMENT, "state_batch_indices must be int32 or int64, got %s",
                dtype_name(index_dtype));
  if (cu_seqlens && !is_index(meta_dtype))
    return fail(SSU_ERR_INVALID_ARGUMENT, "cu_seqlens must be int32 or int64, got %s",
                dtype_name(meta_dtype));
  if (!cu_seqlens && rows != nseqs)
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "without cu_seqlens every sequence is one row: rows (%lld) must equal nseqs "
                "(%lld)",
                (long long)rows, (long long)nseqs);
  if (!state_batch_indices && nseqs > p->slots)
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "without state_batch_indices sequence s uses slot s: %lld sequences exceed %lld "
                "slots",
                (long long)nseqs, (long long)p->slots);
  if (update_trackers &&
      (!scratch || scratch_bytes < 4 * nseqs || reinterpret_cast<uintptr_t>(scratch) % 4 != 0))
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "update_trackers needs 4-byte aligned scratch of 4 * nseqs = %lld bytes "
                "(zero-filled before the first call), got %lld",
                (long long)(4 * nseqs), (long long)scratch_bytes);
  if (nseqs == 0) return ok();
  ssu::ReplayArgs a{};
  a.sbi = state_batch_indices;
  a.sbi_stride = sbi_stride;
  a.idx64 = index_dtype == SSU_I64;
  a.cu = cu_seqlens;
  a.meta64 = meta_dtype == SSU_I64;
  a.rows = rows;
  a.x_cache = rc->x_cache;
  a.B_cache = rc->B_cache;
  a.dt_cache = rc->dt_cache;
  a.R = (int)rc->ring_len;
  a.G = (int)p->ngroups;
  a.W = rc->logical_window;
  a.ring_start = rc->ring_start;
  a.prev = rc->prev_num_accepted;
  a.limit = rc->num_states < p->slots ? rc->num_states : p->slots;
  a.update_trackers = update_trackers != 0;
  a.arrivals = static_cast<unsigned*>(scratch);
  const bool io_bf16 = p->io_dtype == SSU_BF16;
  const int N = (int)p->dstate;
  cudaError_t e = cudaErrorInvalidValue;
  switch (p->state_dtype) {
    case SSU_F32: e = ssu::replay_state_f32(N, io_bf16, k, a, nseqs, (cudaStream_t)stream); break;
    case SSU_BF16: e = ssu::replay_state_bf16(N, io_bf16, k, a, nseqs, (cudaStream_t)stream); break;
    case SSU_F16: e = ssu::replay_state_f16(N, io_bf16, k, a, nseqs, (cudaStream_t)stream); break;
    default: break;
  }
  if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return ok();
}

static ssu_status check_trackers(int32_t* rs, int64_t n_rs, int32_t* pna, int64_t n_pna,
                                 int32_t* pql, int64_t n_pql, const void* sbi,
                                 ssu_dtype index_dtype, int64_t nseqs, int64_t* num_states) {
  if (nseqs < 0) return fail(SSU_ERR_INVALID_ARGUMENT, "nseqs must be >= 0");
  if (n_rs < 0 || n_pna < 0 || n_pql < 0)
    return fail(SSU_ERR_INVALID_ARGUMENT, "tracker lengths must be >= 0");
  if (nseqs > 0 && (!rs || !pna || !pql || !sbi))
    return fail(SSU_ERR_INVALID_ARGUMENT, "tracker and slot pointers must not be NULL");
  if (!is_index(index_dtype))
    return fail(SSU_ERR_INVALID_ARGUMENT, "state_batch_indices must be int32 or int64, got %s",
                dtype_name(index_dtype));
  int64_t m = n_rs < n_pna ? n_rs : n_pna;
  *num_states = m < n_pql ? m : n_pql;
  return SSU_OK;
}

ssu_status ssu_ring_update(int32_t* ring_start, int64_t ring_start_len,
                           int32_t* prev_num_accepted, int64_t prev_num_accepted_len,
                           int32_t* prev_query_len, int64_t prev_query_len_len,
                           const void* state_batch_indices, int64_t sbi_stride,
                           ssu_dtype index_dtype, int64_t nseqs, int reset,
                           int32_t logical_window, int32_t ring_buffer_len, int64_t pad_slot_id,
                           struct CUstream_st* stream) {
  int64_t num_states = 0;
  ssu_status st = check_trackers(ring_start, ring_start_len, prev_num_accepted,
                                 prev_num_accepted_len, prev_query_len, prev_query_len_len,
                                 state_batch_indices, index_dtype, nseqs, &num_states);
  if (st != SSU_OK) return st;
  if (!reset && ring_buffer_len < 1)
    return fail(SSU_ERR_INVALID_ARGUMENT, "ring_buffer_len must be >= 1, got %d",
                (int)ring_buffer_len);
  if (nseqs == 0) return ok();
  cudaError_t e = ssu::launch_ring_update(
      ring_start, prev_num_accepted, prev_query_len, state_batch_indices, sbi_stride,
      index_dtype == SSU_I64, nseqs, num_states, reset != 0, reset ? 0 : logical_window,
      reset ? 1 : ring_buffer_len, pad_slot_id, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return ok();
}

ssu_status ssu_ring_commit(int32_t* ring_start, int64_t ring_start_len,
                           int32_t* prev_num_accepted, int64_t prev_num_accepted_len,
                           int32_t* prev_query_len, int64_t prev_query_len_len,
                           const void* state_batch_indices, int64_t sbi_stride,
                           ssu_dtype index_dtype, const void* num_accepted_tokens,
                           const void* query_start_loc, ssu_dtype meta_dtype, int64_t nseqs,
                           int32_t logical_window, int32_t ring_buffer_len, int64_t pad_slot_id,
                           struct CUstream_st* stream) {
  int64_t num_states = 0;
  ssu_status st = check_trackers(ring_start, ring_start_len, prev_num_accepted,
                                 prev_num_accepted_len, prev_query_len, prev_query_len_len,
                                 state_batch_indices, index_dtype, nseqs, &num_states);
  if (st != SSU_OK) return st;
  if (nseqs > 0 && (!num_accepted_tokens || !query_start_loc))
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "num_accepted_tokens and query_start_loc must not be NULL");
  if (!is_index(meta_dtype))
    return fail(SSU_ERR_INVALID_ARGUMENT,
                "num_accepted_tokens / query_start_loc must be int32 or int64, got %s",
                dtype_name(meta_dtype));
  if (ring_buffer_len < 1)
    return fail(SSU_ERR_INVALID_ARGUMENT, "ring_buffer_len must be >= 1, got %d",
                (int)ring_buffer_len);
  if (nseqs == 0) return ok();
  cudaError_t e = ssu::launch_ring_commit(
      ring_start, prev_num_accepted, prev_query_len, state_batch_indices, sbi_stride,
      index_dtype == SSU_I64, num_accepted_tokens, query_start_loc, meta_dtype == SSU_I64, nseqs,
      num_states, logical_window, ring_buffer_len, pad_slot_id, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return ok();
}

ssu_status ssu_device_error(unsigned int* value, int reset) {
  if (!value) return fail(SSU_ERR_INVALID_ARGUMENT, "value must not be NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(value, g_ssu_device_error, sizeof(unsigned));
  if (e == cudaSuccess && reset) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_ssu_device_error, &zero, sizeof zero);
  }
  if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "reading the error word failed: %s",
                                    cudaGetErrorString(e));
  return ok();
}

ssu_status ssu_selftest_bounded_wait(uint64_t limit_ns, uint64_t* waited_ns) {
  if (!waited_ns) return fail(SSU_ERR_INVALID_ARGUMENT, "waited_ns must not be NULL");
  if (limit_ns == 0 || limit_ns > 1000000000ull)
    return fail(SSU_ERR_INVALID_ARGUMENT, "limit_ns must be in (0, 1e9]");
  void* w = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&w, g_ssu_selftest_waited_ns);
  if (e == cudaSuccess)
    e = ssu::launch_bounded_wait_probe(limit_ns, static_cast<unsigned long long*>(w), nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  unsigned long long v = 0;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_ssu_selftest_waited_ns, sizeof v);
  if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "bounded-wait self-test failed: %s",
                                    cudaGetErrorString(e));
  *waited_ns = v;
  return ok();
}

const char* ssu_status_string(ssu_status s) {
  switch (s) {
    case SSU_OK: return "ok";
    case SSU_ERR_INVALID_ARGUMENT: return "invalid argument";
    case SSU_ERR_UNSUPPORTED: return "unsupported";
    case SSU_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* ssu_last_error(void) { return g_last_error.c_str(); }

int ssu_abi_version(void) { return SSU_ABI_VERSION; }

}  // extern "C"
#pragma GCC visibility pop
