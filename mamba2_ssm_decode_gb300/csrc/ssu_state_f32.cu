// ssu_state_f32.cu -- SSU kernels for f32 state pools (all dstate / io dtypes).
#include "ssu_launch.cuh"

namespace ssu {

cudaError_t launch_state_f32(int N, bool io_bf16, bool varlen, const KParams& p,
                              const OneTokenArgs* oa, const VarlenArgs* va, int64_t nitems,
                              cudaStream_t stream, int algorithm) {
  return io_bf16 ? launch_io<float, __nv_bfloat16>(N, varlen, p, oa, va, nitems, stream, algorithm)
                 : launch_io<float, __half>(N, varlen, p, oa, va, nitems, stream, algorithm);
}

cudaError_t replay_state_f32(int N, bool io_bf16, const KParams& p, const ReplayArgs& ra,
                              int64_t nseqs, cudaStream_t stream) {
  return io_bf16 ? launch_replay_io<float, __nv_bfloat16>(N, p, ra, nseqs, stream)
                 : launch_replay_io<float, __half>(N, p, ra, nseqs, stream);
}

}  // namespace ssu
