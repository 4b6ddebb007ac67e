// ssu_launch.cuh -- tile configuration and typed launchers of the SSU kernels.
#pragma once

#include <algorithm>

#include "ssu_bulk.cuh"
#include "ssu_headrun.cuh"
#include "ssu_replay.cuh"

namespace ssu {

// Host helpers defined in ssu_abi.cu.
unsigned* device_error_word();  // this device's error word (device address)
int sm_count();                 // SMs of the current device

inline void set_divisors(KParams& p) {
  p.fd_tiles.init((uint32_t)p.tiles);
  p.fd_H.init((uint32_t)p.H);
  p.fd_hr.init((uint32_t)p.hr);
}

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

// Head-run kernels: state tiles of at most 16 KB, two per CTA.
template <class ST, int N>
struct HeadRunTune {
  using L = RowLayout<ST, N>;
  static constexpr int WARPS = 4;
  static constexpr int UNR = cmax(
      1, cmin(Tune<ST, N>::UNR, 16384 / (WARPS * L::RPW * N * (int)sizeof(ST))));
  static constexpr int ROWS = WARPS * L::RPW * UNR;
};

// Heads per CTA of the head-run kernels: the largest of 8, 4, 2, 1 dividing
// the heads per group that still leaves at least 4096 CTAs (several waves of
// resident CTAs, so the last one is a small share of the launch).
inline int heads_per_cta(int hr, int64_t ctas_one_head_each) {
  for (int kh = 8; kh > 1; kh /= 2)
    if (hr % kh == 0 && ctas_one_head_each / kh >= 4096) return kh;
  return 1;
}

// Bulk-copy pipeline shape: CW consumer warps, each thread owning UNR state
// rows (capped so a tile has at most 64 rows), plus one producer warp; as
// many tile stages S (2..4, with S + 1 operand buffers) as fit the per-CTA
// budget (two CTAs per SM for 32 KB tiles, three for 16 KB and smaller).
template <class ST, int N, int LMAX, int CW, int UNR_>
struct BulkTune {
  using L = RowLayout<ST, N>;
  static constexpr int WARPS = CW;
  static constexpr int UNR = cmax(1, cmin(UNR_, cmax(1, 64 / (CW * L::RPW))));
  static constexpr int ROWS = WARPS * L::RPW * UNR;
  static constexpr int PER_STAGE = ROWS * N * (int)sizeof(ST);
  static constexpr int PER_VEC = LMAX * (2 * N + 4 * ROWS) * 4;
  static constexpr int BUDGET = (PER_STAGE > 16 * 1024 ? 110 : 76) * 1024;
  static constexpr int S = (4 * PER_STAGE + 5 * PER_VEC <= BUDGET)   ? 4
                           : (3 * PER_STAGE + 4 * PER_VEC <= BUDGET) ? 3
                                                                     : 2;
  static constexpr int SV = S + 1;
};

template <class ST, class IT, int N, bool VARLEN, int CW, int UNR_>
cudaError_t launch_bulk_cfg(KParams p, const OneTokenArgs& oa, const VarlenArgs& va,
                            int64_t nitems, cudaStream_t stream) {
  constexpr int LMAX = VARLEN ? Tune<ST, N>::LMAX : 1;
  using BT = BulkTune<ST, N, LMAX, CW, UNR_>;
  using Cfg = BulkConfig<ST, IT, N, BT::WARPS, BT::UNR, BT::S, BT::SV, LMAX>;
  auto kern = ssu_bulk_kernel<ST, IT, N, BT::WARPS, BT::UNR, BT::S, BT::SV, LMAX, VARLEN>;
  p.tiles = (p.P + Cfg::ROWS - 1) / Cfg::ROWS;
  set_divisors(p);
  const int64_t items = nitems * (int64_t)p.H * p.tiles;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
  if (e != cudaSuccess) return e;
  // all of the unified L1 / shared array as shared memory: several CTAs per SM
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::THREADS, Cfg::SMEM);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t grid = std::min<int64_t>(items, (int64_t)sm_count() * per_sm);
  unsigned* err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  kern<<<(unsigned)grid, Cfg::THREADS, Cfg::SMEM, stream>>>(p, oa, va, items, err);
  return cudaGetLastError();
}

// Tile per state dtype (measured): fp32 state streams best in 32-row tiles
// (16 KB, four stages, three CTAs per SM) when it is written back, in 64-row
// tiles when it is only read (half the bytes per unit of compute); 16-bit
// state in 64-row tiles.
// The consumer-staged variant: two operand buffers (one per alternate item)
// instead of a ring, the same stage budget rule.
template <class ST, int N, int LMAX, int CW, int UNR_>
struct BulkCsTune {
  using L = RowLayout<ST, N>;
  static constexpr int WARPS = CW;
  static constexpr int UNR = cmax(1, cmin(UNR_, cmax(1, 64 / (CW * L::RPW))));
  static constexpr int ROWS = WARPS * L::RPW * UNR;
  static constexpr int PER_STAGE = ROWS * N * (int)sizeof(ST);
  static constexpr int FIXED = 2 * LMAX * (2 * N + 4 * ROWS) * 4;
  static constexpr int BUDGET = (PER_STAGE > 16 * 1024 ? 110 : 72) * 1024;
  static constexpr int S = (4 * PER_STAGE + FIXED <= BUDGET)   ? 4
                           : (3 * PER_STAGE + FIXED <= BUDGET) ? 3
                                                               : 2;
};

template <class ST, class IT, int N, bool VARLEN, int CW, int UNR_>
cudaError_t launch_bulk_cs_cfg(KParams p, const OneTokenArgs& oa, const VarlenArgs& va,
                               int64_t nitems, cudaStream_t stream) {
  constexpr int LMAX = VARLEN ? Tune<ST, N>::LMAX : 1;
  using BT = BulkCsTune<ST, N, LMAX, CW, UNR_>;
  using Cfg = BulkCsConfig<ST, IT, N, BT::WARPS, BT::UNR, BT::S, LMAX>;
  auto kern = ssu_bulk_cs_kernel<ST, IT, N, BT::WARPS, BT::UNR, BT::S, LMAX, VARLEN>;
  p.tiles = (p.P + Cfg::ROWS - 1) / Cfg::ROWS;
  set_divisors(p);
  const int64_t items = nitems * (int64_t)p.H * p.tiles;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::THREADS, Cfg::SMEM);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t grid = std::min<int64_t>(items, (int64_t)sm_count() * per_sm);
  unsigned* err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  kern<<<(unsigned)grid, Cfg::THREADS, Cfg::SMEM, stream>>>(p, oa, va, items, err);
  return cudaGetLastError();
}

// Which bulk pipeline and tile (measured): fp32 state that is written back
// streams best with producer-staged operands in 32-row tiles; 16-bit state
// and calls that write no state (more operand work per byte moved) with
// consumer-staged operands in 64-row tiles.
template <class ST, class IT, int N, bool VARLEN>
cudaError_t launch_bulk(KParams p, const OneTokenArgs& oa, const VarlenArgs& va, int64_t nitems,
                        cudaStream_t stream) {
  if constexpr (sizeof(ST) == 4) {
    if (!p.disable) return launch_bulk_cfg<ST, IT, N, VARLEN, 4, 2>(p, oa, va, nitems, stream);
  }
  return launch_bulk_cs_cfg<ST, IT, N, VARLEN, 4, 4>(p, oa, va, nitems, stream);
}

template <class ST, class IT, int N>
cudaError_t launch_typed(bool varlen, KParams p, const OneTokenArgs* oa, const VarlenArgs* va,
                         int64_t nitems, cudaStream_t stream, int algorithm) {
  using T = Tune<ST, N>;
  // auto (the fastest as measured): the bulk-copy pipeline for one-token calls
  // that write state, the head-run kernels for every other call
  const bool auto_bulk = !varlen && !p.disable;
  // stochastic rounding of 16-bit state: the head-run kernels' SR instances,
  // whatever `algorithm` (the other kernels carry no generator)
  const bool sr = sizeof(ST) == 2 && p.sr_seed != nullptr && !p.disable;
  const bool bulk = !sr && (algorithm == 2 /* SSU_ALGO_BULK */ || (algorithm == 0 && auto_bulk));
  if (bulk) {
    const OneTokenArgs o0 = oa ? *oa : OneTokenArgs{};
    const VarlenArgs v0 = va ? *va : VarlenArgs{};
    return varlen ? launch_bulk<ST, IT, N, true>(p, o0, v0, nitems, stream)
                  : launch_bulk<ST, IT, N, false>(p, o0, v0, nitems, stream);
  }
  if (nitems <= 0) return cudaSuccess;
  // head-run kernels: one launch whatever the batch; grid.x = runs of kh
  // heads of one group x row tiles, sequences over grid.y x grid.z (each at
  // most 65535, so z = ceil(nitems / 65535) and y = ceil(nitems / z) leave
  // fewer than z idle CTAs)
  using NT = HeadRunTune<ST, N>;
  p.tiles = (p.P + NT::ROWS - 1) / NT::ROWS;
  set_divisors(p);
  const int kh = heads_per_cta(p.hr, nitems * p.H * (int64_t)p.tiles);
  const int64_t gx = (int64_t)(p.H / kh) * p.tiles;
  const int64_t gz = (nitems + 65534) / 65535;
  const int64_t gy = (nitems + gz - 1) / gz;
  if (gx > 0x7fffffffLL || gz > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)gz);
  // calls that write no state: the no-write kernel on its (tiles, runs,
  // sequences) grid up to 65535 sequences, beyond that the write kernel
  // (which skips its stores) on the flattened grid -- one launch either way
  const bool nowrite = p.disable && nitems <= 65535;
  if (nowrite) grid = dim3((unsigned)p.tiles, (unsigned)(p.H / kh), (unsigned)nitems);
  const OneTokenArgs o0 = oa ? *oa : OneTokenArgs{};
  const VarlenArgs v0 = va ? *va : VarlenArgs{};
  auto kern2 = varlen ? ssu_run_kernel<ST, IT, N, NT::WARPS, NT::UNR, T::LMAX, true>
                      : ssu_run_kernel<ST, IT, N, NT::WARPS, NT::UNR, 1, false>;
  if constexpr (sizeof(ST) == 2) {
    if (sr)
      kern2 = varlen ? ssu_run_kernel<ST, IT, N, NT::WARPS, NT::UNR, T::LMAX, true, true>
                     : ssu_run_kernel<ST, IT, N, NT::WARPS, NT::UNR, 1, false, true>;
  }
  cudaError_t e;
  if (nowrite) {
    auto nk = varlen ? ssu_nowrite_kernel<ST, IT, N, NT::WARPS, NT::UNR, T::LMAX, true>
                     : ssu_nowrite_kernel<ST, IT, N, NT::WARPS, NT::UNR, 1, false>;
    e = cudaFuncSetAttribute(nk, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  } else {
    e = cudaFuncSetAttribute(kern2, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  }
  if (e != cudaSuccess) return e;
  unsigned* err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  if (nowrite) {
    auto nk = varlen ? ssu_nowrite_kernel<ST, IT, N, NT::WARPS, NT::UNR, T::LMAX, true>
                     : ssu_nowrite_kernel<ST, IT, N, NT::WARPS, NT::UNR, 1, false>;
    nk<<<grid, NT::WARPS * 32, 0, stream>>>(p, o0, v0, nitems, kh, err);
    return cudaGetLastError();
  }
  kern2<<<grid, NT::WARPS * 32, 0, stream>>>(p, o0, v0, nitems, kh, err);
  return cudaGetLastError();
}

// ReplaySSM checkpointing update: the head-run decomposition, chains of up to
// 8 steps staged at once (a window of 4 with 4-token passes; longer chains are
// staged 8 steps at a time).
constexpr int kReplayLmax = 8;

template <class ST, class IT, int N>
cudaError_t launch_replay_typed(KParams p, const ReplayArgs& ra, int64_t nseqs,
                                cudaStream_t stream) {
  using NT = HeadRunTune<ST, N>;
  using RC = ReplayCfg<ST, IT, N, NT::WARPS, NT::UNR, kReplayLmax>;
  p.tiles = (p.P + RC::ROWS - 1) / RC::ROWS;
  set_divisors(p);
  const int kh = heads_per_cta(p.hr, nseqs * p.H * (int64_t)p.tiles);
  const int64_t gx = (int64_t)(p.H / kh) * p.tiles;
  const int64_t gz = (nseqs + 65534) / 65535;
  const int64_t gy = (nseqs + gz - 1) / gz;
  if (gx > 0x7fffffffLL || gz > 65535) return cudaErrorInvalidConfiguration;
  auto kern = ssu_replay_kernel<ST, IT, N, NT::WARPS, NT::UNR, kReplayLmax>;
  if constexpr (sizeof(ST) == 2) {
    if (p.sr_seed) kern = ssu_replay_kernel<ST, IT, N, NT::WARPS, NT::UNR, kReplayLmax, true>;
  }
  const int smem = (int)sizeof(typename RC::Smem);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  unsigned* err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  kern<<<dim3((unsigned)gx, (unsigned)gy, (unsigned)gz), RC::THREADS, smem, stream>>>(p, ra, nseqs,
                                                                                     kh, err);
  return cudaGetLastError();
}

template <class ST, class IT>
cudaError_t launch_replay_io(int N, const KParams& p, const ReplayArgs& ra, int64_t nseqs,
                             cudaStream_t stream) {
  switch (N) {
    case 16: return launch_replay_typed<ST, IT, 16>(p, ra, nseqs, stream);
    case 32: return launch_replay_typed<ST, IT, 32>(p, ra, nseqs, stream);
    case 64: return launch_replay_typed<ST, IT, 64>(p, ra, nseqs, stream);
    case 128: return launch_replay_typed<ST, IT, 128>(p, ra, nseqs, stream);
    case 256: return launch_replay_typed<ST, IT, 256>(p, ra, nseqs, stream);
  }
  return cudaErrorInvalidValue;
}

template <class ST, class IT>
cudaError_t launch_io(int N, bool varlen, const KParams& p, const OneTokenArgs* oa,
                      const VarlenArgs* va, int64_t nitems, cudaStream_t stream, int algo) {
  switch (N) {
    case 16: return launch_typed<ST, IT, 16>(varlen, p, oa, va, nitems, stream, algo);
    case 32: return launch_typed<ST, IT, 32>(varlen, p, oa, va, nitems, stream, algo);
    case 64: return launch_typed<ST, IT, 64>(varlen, p, oa, va, nitems, stream, algo);
    case 128: return launch_typed<ST, IT, 128>(varlen, p, oa, va, nitems, stream, algo);
    case 256: return launch_typed<ST, IT, 256>(varlen, p, oa, va, nitems, stream, algo);
  }
  return cudaErrorInvalidValue;
}

// defined in ssu_state_{f32,bf16,f16}.cu
cudaError_t launch_state_f32(int N, bool io_bf16, bool varlen, const KParams& p,
                             const OneTokenArgs* oa, const VarlenArgs* va, int64_t nitems,
                             cudaStream_t stream, int algorithm);
cudaError_t launch_state_bf16(int N, bool io_bf16, bool varlen, const KParams& p,
                              const OneTokenArgs* oa, const VarlenArgs* va, int64_t nitems,
                              cudaStream_t stream, int algorithm);
cudaError_t launch_state_f16(int N, bool io_bf16, bool varlen, const KParams& p,
                             const OneTokenArgs* oa, const VarlenArgs* va, int64_t nitems,
                             cudaStream_t stream, int algorithm);

// defined in ssu_state_{f32,bf16,f16}.cu
cudaError_t replay_state_f32(int N, bool io_bf16, const KParams& p, const ReplayArgs& ra,
                             int64_t nseqs, cudaStream_t stream);
cudaError_t replay_state_bf16(int N, bool io_bf16, const KParams& p, const ReplayArgs& ra,
                              int64_t nseqs, cudaStream_t stream);
cudaError_t replay_state_f16(int N, bool io_bf16, const KParams& p, const ReplayArgs& ra,
                             int64_t nseqs, cudaStream_t stream);

// defined in selftest.cu
cudaError_t launch_bounded_wait_probe(uint64_t limit_ns, unsigned long long* waited_ns,
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
