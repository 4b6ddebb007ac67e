// ssu_launch.cuh -- tile configuration and typed launchers of the SSU kernels.
#pragma once

#include "ssu_kernel.cuh"

namespace ssu {

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }

// Launch shape per (state dtype, dstate): 4 warps, enough unrolled rows per
// thread for 64 headdim rows per CTA, at most 64 state values per thread in
// registers, and up to 4 speculative steps staged at a time.
template <class ST, int N>
struct Tune {
  using L = RowLayout<ST, N>;
  static constexpr int WARPS = 4;
  static constexpr int UNR = cmax(1, cmin(64 / (WARPS * L::RPW), cmax(1, 64 / L::EPL)));
  static constexpr int LMAX = 4;
};

template <class ST, class IT, int N>
cudaError_t launch_typed(bool varlen, KParams p, const OneTokenArgs* oa, const VarlenArgs* va,
                         int64_t nitems, cudaStream_t stream) {
  using T = Tune<ST, N>;
  using Cfg = SSUConfig<ST, IT, N, T::WARPS, T::UNR, T::LMAX>;
  p.tiles = (p.P + Cfg::ROWS - 1) / Cfg::ROWS;
  const int64_t grid = nitems * (int64_t)p.H * p.tiles;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (varlen) {
    ssu_varlen_kernel<ST, IT, N, T::WARPS, T::UNR, T::LMAX>
        <<<(unsigned)grid, Cfg::THREADS, 0, stream>>>(p, *va);
  } else {
    ssu_one_token_kernel<ST, IT, N, T::WARPS, T::UNR>
        <<<(unsigned)grid, Cfg::THREADS, 0, stream>>>(p, *oa);
  }
  return cudaGetLastError();
}

template <class ST, class IT>
cudaError_t launch_io(int N, bool varlen, const KParams& p, const OneTokenArgs* oa,
                      const VarlenArgs* va, int64_t nitems, cudaStream_t stream) {
  switch (N) {
    case 16: return launch_typed<ST, IT, 16>(varlen, p, oa, va, nitems, stream);
    case 32: return launch_typed<ST, IT, 32>(varlen, p, oa, va, nitems, stream);
    case 64: return launch_typed<ST, IT, 64>(varlen, p, oa, va, nitems, stream);
    case 128: return launch_typed<ST, IT, 128>(varlen, p, oa, va, nitems, stream);
    case 256: return launch_typed<ST, IT, 256>(varlen, p, oa, va, nitems, stream);
  }
  return cudaErrorInvalidValue;
}

// defined in ssu_state_{f32,bf16,f16}.cu
cudaError_t launch_state_f32(int N, bool io_bf16, bool varlen, const KParams& p,
                             const OneTokenArgs* oa, const VarlenArgs* va, int64_t nitems,
                             cudaStream_t stream);
cudaError_t launch_state_bf16(int N, bool io_bf16, bool varlen, const KParams& p,
                              const OneTokenArgs* oa, const VarlenArgs* va, int64_t nitems,
                              cudaStream_t stream);
cudaError_t launch_state_f16(int N, bool io_bf16, bool varlen, const KParams& p,
                             const OneTokenArgs* oa, const VarlenArgs* va, int64_t nitems,
                             cudaStream_t stream);

// defined in ring_trackers.cu
cudaError_t launch_ring_update(int32_t* rs, int32_t* pna, int32_t* pql, const void* sbi,
                               int64_t sbi_stride, int idx64, int64_t nseqs, int64_t num_states,
                               int reset, int32_t window, int32_t ring_len, int64_t pad,
                               cudaStream_t stream);
cudaError_t launch_ring_commit(int32_t* rs, int32_t* pna, int32_t* pql, const void* sbi,
                               int64_t sbi_stride, int idx64, const void* na, const void* qsl,
                               int meta64, int64_t nseqs, int64_t num_states, int32_t window,
                               int32_t ring_len, int64_t pad, cudaStream_t stream);

}  // namespace ssu
