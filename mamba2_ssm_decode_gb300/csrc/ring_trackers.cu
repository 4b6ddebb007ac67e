// ring_trackers.cu -- ReplaySSM ring-tracker update / reset / commit.
//
// "vllm.model_executor.layers.mamba.ops.ssu_dispatch":
// _update_replayssm_ring_trackers_kernel and
// _commit_replayssm_ring_trackers_kernel.  One thread per sequence; the
// trackers are int32 vectors indexed by slot.  A slot is used only when it is
// not the pad id and lies in [0, num_states).  Arithmetic is int32 with
// two's-complement wrap-around; % truncates toward zero.
#include "ssu_launch.cuh"

namespace ssu {
namespace {

constexpr int kTrackerThreads = 128;

__device__ __forceinline__ int32_t wrap_add(int32_t a, int32_t b) {
  return (int32_t)((uint32_t)a + (uint32_t)b);
}

__device__ __forceinline__ int32_t to_i32(int64_t v) { return (int32_t)(uint32_t)(uint64_t)v; }

__global__ void __launch_bounds__(kTrackerThreads)
    ring_update_kernel(int32_t* __restrict__ ring_start, int32_t* __restrict__ prev_num_accepted,
                       int32_t* __restrict__ prev_query_len, const void* __restrict__ sbi,
                       int64_t sbi_stride, int idx64, int64_t nseqs, int64_t num_states,
                       int reset, int32_t window, int32_t ring_len, int64_t pad) {
  const int64_t i = (int64_t)blockIdx.x * kTrackerThreads + threadIdx.x;
  if (i >= nseqs) return;
  const int64_t slot = load_int(sbi, i * sbi_stride, idx64);
  if (!(slot != pad && slot >= 0 && slot < num_states)) return;
  if (reset) {
    ring_start[slot] = 0;
    prev_num_accepted[slot] = 0;
    prev_query_len[slot] = 0;  // a reset also clears the pending MTP window
    return;
  }
  const int32_t prev = prev_num_accepted[slot];
  const int32_t start = ring_start[slot];
  const bool checkpoint = wrap_add(prev, 1) > window;
  ring_start[slot] = checkpoint ? wrap_add(start, prev) % ring_len : start;
  prev_num_accepted[slot] = checkpoint ? 1 : wrap_add(prev, 1);
}

__global__ void __launch_bounds__(kTrackerThreads)
    ring_commit_kernel(int32_t* __restrict__ ring_start, int32_t* __restrict__ prev_num_accepted,
                       int32_t* __restrict__ prev_query_len, const void* __restrict__ sbi,
                       int64_t sbi_stride, int idx64, const void* __restrict__ num_accepted,
                       const void* __restrict__ qsl, int meta64, int64_t nseqs,
                       int64_t num_states, int32_t window, int32_t ring_len, int64_t pad) {
  const int64_t i = (int64_t)blockIdx.x * kTrackerThreads + threadIdx.x;
  if (i >= nseqs) return;
  const int64_t slot = load_int(sbi, i * sbi_stride, idx64);
  if (!(slot != pad && slot >= 0 && slot < num_states)) return;
  const int32_t acc = prev_num_accepted[slot];  // accepted since the last checkpoint
  const int32_t start = ring_start[slot];
  const int32_t pql = prev_query_len[slot];     // length of the previous MTP query
  const int32_t a = to_i32(load_int(num_accepted, i, meta64));
  const bool checkpoint = pql > 0 && wrap_add(acc, pql) > window;
  const int32_t next_start = checkpoint ? wrap_add(start, acc) % ring_len : start;
  const int32_t next_prev = pql == 0 ? 0 : (checkpoint ? a : wrap_add(acc, a));
  const int32_t qlen = to_i32(load_int(qsl, i + 1, meta64) - load_int(qsl, i, meta64));
  ring_start[slot] = next_start;
  prev_num_accepted[slot] = next_prev;
  prev_query_len[slot] = qlen;
}

}  // namespace

cudaError_t launch_ring_update(int32_t* rs, int32_t* pna, int32_t* pql, const void* sbi,
                               int64_t sbi_stride, int idx64, int64_t nseqs, int64_t num_states,
                               int reset, int32_t window, int32_t ring_len, int64_t pad,
                               cudaStream_t stream) {
  const int64_t blocks = (nseqs + kTrackerThreads - 1) / kTrackerThreads;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ring_update_kernel<<<(unsigned)blocks, kTrackerThreads, 0, stream>>>(
      rs, pna, pql, sbi, sbi_stride, idx64, nseqs, num_states, reset, window, ring_len, pad);
  return cudaGetLastError();
}

cudaError_t launch_ring_commit(int32_t* rs, int32_t* pna, int32_t* pql, const void* sbi,
                               int64_t sbi_stride, int idx64, const void* na, const void* qsl,
                               int meta64, int64_t nseqs, int64_t num_states, int32_t window,
                               int32_t ring_len, int64_t pad, cudaStream_t stream) {
  const int64_t blocks = (nseqs + kTrackerThreads - 1) / kTrackerThreads;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ring_commit_kernel<<<(unsigned)blocks, kTrackerThreads, 0, stream>>>(
      rs, pna, pql, sbi, sbi_stride, idx64, na, qsl, meta64, nseqs, num_states, window, ring_len,
      pad);
  return cudaGetLastError();
}

}  // namespace ssu
