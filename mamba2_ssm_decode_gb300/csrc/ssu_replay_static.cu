// ssu_replay_static.cu -- ssu_replay_update_static: the checkpointing update
// for callers that cannot pass a scratch buffer.
//
// ssu_replay_update's fused tracker update counts the CTAs of each sequence in
// caller-provided scratch (nseqs uint32 counters).  Some callers cannot hand
// the library such a buffer: a plugin host that gives an operation only its
// own input and output tensors, or a serving runtime that plans all device
// memory at start-up and forbids allocations afterwards (cudaMalloc can
// synchronise the device and breaks a pre-planned pool).  This entry point
// keeps the counters in a file-scope device array instead, so it allocates
// nothing and needs nothing beyond the operation's own tensors.
//
// The array is a fixed kMaxStaticSeqs counters (256 KB), held by every GPU
// that loads the library until the process exits.  Host code cannot use the
// array's name as a device address (it names a host-side stand-in), so the
// address is fetched with cudaGetSymbolAddress once per device, with that
// device current, the first time the entry point runs on it.
#include <cstdio>
#include <mutex>

#include "../../include/ssu.h"
#include "ssu_launch.cuh"

namespace ssu {
ssu_status record_error(ssu_status code, const char* message);  // ssu_abi.cu
}

namespace {

constexpr int64_t kMaxStaticSeqs = SSU_REPLAY_STATIC_MAX_SEQS;
constexpr int kMaxDevices = 64;

// The counters of ssu_replay_update_static, shared by every call on a device.
static __device__ __align__(256) unsigned g_replay_static_arrivals[kMaxStaticSeqs];

// Device address of the current device's counters, fetched once per device
// with that device current; nullptr (and the error) on failure.
unsigned* static_arrivals(cudaError_t* err) {
  static std::mutex mu;
  static unsigned* addr[kMaxDevices] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* a = nullptr;
    *err = cudaGetSymbolAddress(&a, g_replay_static_arrivals);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned*>(a);
  }
  return addr[dev];
}

}  // namespace

#pragma GCC visibility push(default)
extern "C" {

ssu_status ssu_replay_update_static(const ssu_params* p, const ssu_replay_cache* rc,
                                    int64_t nseqs, int64_t rows, const void* cu_seqlens,
                                    ssu_dtype meta_dtype, const void* state_batch_indices,
                                    int64_t sbi_stride, ssu_dtype index_dtype,
                                    int update_trackers, struct CUstream_st* stream) {
  if (nseqs > kMaxStaticSeqs) {
    char msg[160];
    snprintf(msg, sizeof msg,
             "ssu_replay_update_static takes at most %lld sequences (its fixed counter array), "
             "got %lld",
             (long long)kMaxStaticSeqs, (long long)nseqs);
    return ssu::record_error(SSU_ERR_INVALID_ARGUMENT, msg);
  }
  unsigned* arrivals = nullptr;
  if (update_trackers && nseqs > 0) {
    cudaError_t e = cudaSuccess;
    arrivals = static_arrivals(&e);
    // the counters must start at zero: a completed call leaves them zero, and
    // the ones this call uses are cleared on its stream all the same (a memset,
    // no allocation)
    if (arrivals)
      e = cudaMemsetAsync(arrivals, 0, (size_t)nseqs * sizeof(unsigned), (cudaStream_t)stream);
    if (!arrivals || e != cudaSuccess) {
      char msg[200];
      snprintf(msg, sizeof msg, "preparing the static counters failed: %s",
               cudaGetErrorString(e));
      return ssu::record_error(SSU_ERR_CUDA, msg);
    }
  }
  return ssu_replay_update(p, rc, nseqs, rows, cu_seqlens, meta_dtype, state_batch_indices,
                           sbi_stride, index_dtype, update_trackers, arrivals,
                           kMaxStaticSeqs * (int64_t)sizeof(unsigned), stream);
}

}  // extern "C"
#pragma GCC visibility pop
