// ssd.cu -- packed variable-length SSD prefill ("mate.mamba",
// ssd_combined_fwd_varlen) on sm_103a.
//
// The call computes, over every sequence of a packed batch, the Mamba2
// recurrence the one-token update computes (dt' = clamp(softplus(dt +
// dt_bias)); h <- h exp(A dt') + dt' x B; y = h C + D x; y *= silu(z)) and
// returns the state at chunk ends.  The pages name its five stages (cumsum,
// chunk_state, state_passing, bmm, chunk_scan); within a chunk of Lc tokens,
// with a_t the running sum of A dt' over the chunk:
//   chunk_state  S      = sum_s exp(a_{L-1} - a_s) dt'_s x_s (outer) B_s
//   passing      h_end  = exp(a_{L-1}) h_enter + S        (sequential over chunks)
//   bmm          CB[t,s] = C_t . B_s
//   chunk_scan   y_t    = sum_{s<=t} CB[t,s] exp(a_t - a_s) dt'_s x_s
//                         + exp(a_t) C_t . h_enter + D x_t     (times silu(z_t))
// Three launches on the caller's stream, the contractions on the fifth-
// generation tensor cores (tcgen05: MMAs issued by one thread, fp32
// accumulators in tensor memory): (1) dt', a_t and S per chunk and pair of
// heads (cumsum + chunk_state); (2) the sequential state passing, which also
// stores each chunk's entering state in the tensor-core operand layout; (3)
// the scan, which forms C . B^T itself (the bmm stage), 128 source tokens at
// a time, and feeds it, decayed and masked, back into the intra-chunk product.  The inputs x, B, C are 16-bit already;
// an operand the kernels compute (w_s x_s, the decayed C . B^T, h_enter) is
// split into a 16-bit high part and a 16-bit remainder and multiplied twice,
// so that it enters the products to about 2^-16 instead of 2^-8 (the outputs
// of these sums often cancel to far below their terms).
#include <cstdarg>
#include <cstdio>

#include "../../include/ssu.h"
#include "ssd_tc.cuh"
#include "ssu_bulk.cuh"
#include "ssu_headrun.cuh"

namespace ssu {
ssu_status record_error(ssu_status code, const char* message);  // ssu_abi.cu
unsigned* device_error_word();                                   // ssu_abi.cu
}

namespace ssd {
using namespace ssu;

constexpr int kMaxChunk = 256;  // largest supported chunk_size
constexpr unsigned kErrMmaTimeout = SSU_DEVICE_ERR_MMA_TIMEOUT;

struct SSDArgs {
  const void* x;
  const float* dt;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  int D_per_dim;
  const void* z;
  const float* dt_bias;
  int softplus;
  float dt_lo, dt_hi;
  void* out;
  int T, H, G, hr, CS, nchunks, batch;
  const void* cu_chunk;
  const void* seq;
  const void* last;
  int meta64;
  const void* init;
  int init_dtype;  // 0 f32, 1 bf16, 2 f16
  void* states;
  int state_dtype;
  int intermediate;
  float* ws_state;      // [nchunks, H, P, N]: chunk-local states S
  uint8_t* ws_henter;   // [nchunks, H]: entering state, high parts then remainders, 16-bit,
                        // in the scan's operand layout (see ssd_chunk_scan_kernel)
  float* ws_dt;         // [nchunks, H, CS]: dt'
  float* ws_acum;       // [nchunks, H, CS]: a_t
  unsigned* err;        // device error word
};

// tokens [t0, t0 + Lc) of chunk c (Lc clamped to [0, CS])
__device__ __forceinline__ void chunk_span(const SSDArgs& a, int c, int64_t* t0, int* Lc) {
  const int64_t b = load_int(a.cu_chunk, c, a.meta64);
  int64_t e = load_int(a.cu_chunk, c + 1, a.meta64);
  if (e > a.T) e = a.T;
  int64_t n = e - b;
  if (n < 0 || b < 0) n = 0;
  if (n > a.CS) n = a.CS;
  *t0 = b;
  *Lc = (int)n;
}

// hi + lo = (a, b) to 16-bit precision each: packed (low = a, high = b) pairs
template <class IT>
__device__ __forceinline__ void split_packed(float a, float b, uint32_t* hi, uint32_t* lo);

template <>
__device__ __forceinline__ void split_packed<__nv_bfloat16>(float a, float b, uint32_t* hi,
                                                            uint32_t* lo) {
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 l2 = __floats2bfloat162_rn(a - __low2float(h2), b - __high2float(h2));
  *hi = *reinterpret_cast<const uint32_t*>(&h2);
  *lo = *reinterpret_cast<const uint32_t*>(&l2);
}

template <>
__device__ __forceinline__ void split_packed<__half>(float a, float b, uint32_t* hi, uint32_t* lo) {
  const __half2 h2 = __floats2half2_rn(a, b);
  const __half2 l2 = __floats2half2_rn(a - __low2float(h2), b - __high2float(h2));
  *hi = *reinterpret_cast<const uint32_t*>(&h2);
  *lo = *reinterpret_cast<const uint32_t*>(&l2);
}

// Spin on an mbarrier phase (the tensor core finishes within microseconds: a
// suspended wait would add its wake-up latency); false after `limit_ns`.
__device__ __forceinline__ bool spin_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 255u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// 1. dt', a_t and the chunk-local state S on the fifth-generation tensor
//    cores: one CTA of 256 threads per chunk and pair of heads of one group
//    (one head when the groups have an odd number of heads).  With
//    w_{k,s} = exp(a_end - a_s) dt'_s for head k,
//      S_k[p][n] = sum_s (w_{k,s} x_{k,s}[p]) B_s[n]
//    is one M = 128 (two heads x 64 p) x N (dstate) MMA chain over the
//    chunk's tokens, 64 at a time (K = tokens).  Both operands are MN-major,
//    so x and B rows keep their global layout: 16-byte pieces (8 p, or 8 n,
//    of one token) sit at (p / 8 or n / 8) 1040 + 16 s (LBO 128, SBO 1040: the
//    16 bytes of padding per 64 tokens spread the eight pieces of one token's
//    row over distinct banks, so the threads can take a token row's pieces
//    side by side -- whole 128-byte lines from global memory).
//    The A operand w x is computed, so it is split into high parts and
//    remainders (two MMAs per step); B rows are copied in by cp.async one
//    slice ahead.
// ---------------------------------------------------------------------------
constexpr int kStSL = 64;     // tokens per slice
constexpr int kStSBO = 1040;  // bytes between 8-row groups of the MN-major operands

template <int N>
struct StateSmem {
  uint8_t as[2][16 * kStSBO];     // w x of the slice: high parts, remainders
  uint8_t bs[2][N / 8 * kStSBO];  // B rows of a slice, two buffers
  float w[2][kMaxChunk];           // per head: a_t, then w_t
  uint64_t bar;
  uint32_t tmem;
};

template <class IT, int P, int N>
__global__ void __launch_bounds__(256) ssd_chunk_state_kernel(const SSDArgs a) {
  static_assert(P == 64 && (N == 64 || N == 128), "headdim 64, dstate 64 or 128");
  constexpr bool kBF16 = std::is_same<IT, __nv_bfloat16>::value;
  constexpr uint32_t kId = tc::idesc_f16(kBF16, 128, N, true, true);
  constexpr uint32_t kCols = N;  // 64 or 128 fp32 columns
  constexpr int NT = 256;
  const int c = blockIdx.x;
  const bool pair = (a.hr % 2) == 0;
  const int h0 = pair ? 2 * blockIdx.y : blockIdx.y, nh = pair ? 2 : 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<StateSmem<N>*>(smem_raw);
  int64_t t0;
  int Lc;
  chunk_span(a, c, &t0, &Lc);
  if (*reinterpret_cast<volatile unsigned*>(a.err) & kErrMmaTimeout) return;  // a wait gave up
  if (Lc == 0) {  // an empty chunk: S = 0
    for (int i = tid; i < nh * P * N / 4; i += NT)
      reinterpret_cast<float4*>(a.ws_state + ((int64_t)c * a.H + h0) * P * N)[i] =
          make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int g = h0 / a.hr;
  const IT* bg = static_cast<const IT*>(a.B);
  const IT* xg = static_cast<const IT*>(a.x);
  const uint32_t s_as[2] = {smem_addr(sm.as[0]), smem_addr(sm.as[1])};
  const uint32_t s_bs[2] = {smem_addr(sm.bs[0]), smem_addr(sm.bs[1])};
  auto load_b = [&](int j) {
#pragma unroll 1
    for (int q = tid; q < kStSL * (N / 8); q += NT) {
      const int ng = q % (N / 8), sl = q / (N / 8), s = j * kStSL + sl;
      const bool ok = s < Lc;
      tc::cp16(s_bs[j & 1] + ng * kStSBO + sl * 16,
               bg + ((t0 + (ok ? s : 0)) * a.G + g) * N + ng * 8, ok ? 16u : 0u);
    }
  };
  load_b(0);
  tc::cp_commit();
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::alloc(smem_addr(&sm.tmem), kCols);
  // dt', a_t (inclusive running sum of A dt') and w_t per head: warp k takes
  // head h0 + k, eight tokens per lane
  if (warp < nh) {
    const int h = h0 + warp;
    const float Ah = a.A[h];
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.0f;
    float d[8], v[8], run = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = lane * 8 + k;
      float x = 0.0f;
      if (i < Lc) {
        x = a.dt[(t0 + i) * a.H + h] + bias;
        if (a.softplus) x = softplus_f(x);
        x = fminf(fmaxf(x, a.dt_lo), a.dt_hi);
      }
      d[k] = x;
      run += Ah * x;
      v[k] = run;
    }
    float incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    const float before = incl - run;
    float* wdt = a.ws_dt + ((int64_t)c * a.H + h) * a.CS;
    float* wac = a.ws_acum + ((int64_t)c * a.H + h) * a.CS;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = lane * 8 + k;
      v[k] += before;
      sm.w[warp][i] = v[k];
      if (i < Lc) {
        wdt[i] = d[k];
        wac[i] = v[k];
      }
    }
    __syncwarp();
    const float a_end = sm.w[warp][Lc - 1];
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = lane * 8 + k;
      sm.w[warp][i] = i < Lc ? expf(a_end - v[k]) * d[k] : 0.0f;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem;
  bool dead = false;
  auto wait = [&](uint32_t parity) {
    if (!dead && !spin_wait(&sm.bar, parity, kWaitLimitNs)) {
      dead = true;
      atomicOr(a.err, kErrMmaTimeout);
    }
  };
  const int J = (Lc + kStSL - 1) / kStSL;
  uint32_t ph = 0;
  static_assert(2 * kStSL * (P / 8) == 4 * NT, "four 16-byte pieces of w x per thread");
  for (int j = 0; j < J; ++j) {
    // this thread's x pieces of the slice (8 p of one token each), fetched
    // before waiting for the previous MMAs so the loads overlap them
    uint4 raw[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int q = tid + r * NT;
      const int pg = q % (P / 8), rest = q / (P / 8);
      const int sl = rest % kStSL, k = rest / kStSL, s = j * kStSL + sl;
      raw[r] = (k < nh && s < Lc)
                   ? __ldg(reinterpret_cast<const uint4*>(xg + ((t0 + s) * a.H + h0 + k) * P + pg * 8))
                   : make_uint4(0u, 0u, 0u, 0u);
    }
    if (j > 0) {  // the previous MMAs are done: the A buffer and B buffer (j + 1) % 2 are free
      wait(ph);
      ph ^= 1;
    }
    if (j + 1 < J) load_b(j + 1);
    tc::cp_commit();
    // w x of the slice, split into high parts and remainders
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int q = tid + r * NT;
      const int pg = q % (P / 8), rest = q / (P / 8);
      const int sl = rest % kStSL, k = rest / kStSL, s = j * kStSL + sl;
      const IT* e = reinterpret_cast<const IT*>(&raw[r]);
      const float ws = (k < nh && s < Lc) ? sm.w[k][s] : 0.0f;
      uint32_t hp[4], lp[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        split_packed<IT>(ws * io_to_float<IT>(e[2 * u]), ws * io_to_float<IT>(e[2 * u + 1]), &hp[u],
                         &lp[u]);
      const int off = (k * 8 + pg) * kStSBO + sl * 16;
      *reinterpret_cast<uint4*>(sm.as[0] + off) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
      *reinterpret_cast<uint4*>(sm.as[1] + off) = make_uint4(lp[0], lp[1], lp[2], lp[3]);
    }
    tc::cp_wait<1>();  // all but the newest group: B_j has landed
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < kStSL / 16; ++kk)
          tc::mma(tmem, tc::sdesc(s_as[part] + kk * 256, 128, kStSBO),
                  tc::sdesc(s_bs[j & 1] + kk * 256, 128, kStSBO), kId, (j | part | kk) != 0);
      tc::commit(smem_addr(&sm.bar));
    }
  }
  wait(ph);  // the last MMAs are done: S is final
  tc::fence_after_sync();
  // row m = 32 (warp % 4) + lane is (head m / 64, p m % 64); warpgroup
  // warp / 4 stores columns [N/2 (warp / 4), N/2 (warp / 4) + N/2)
  const int m = 32 * (warp & 3) + lane, k = m / P, pp = m % P, wg = warp >> 2;
  float* dst = a.ws_state + (((int64_t)c * a.H + h0 + k) * P + pp) * N + wg * (N / 2);
#pragma unroll 1
  for (int c16 = 0; c16 < N / 32; ++c16) {
    float v[16];
    tc::ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + wg * (N / 2) + c16 * 16, v);
    tc::wait_ld();
    if (k < nh) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        reinterpret_cast<float4*>(dst + c16 * 16)[u] =
            make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, kCols);
}

// ---------------------------------------------------------------------------
// 2. state passing: sequential over chunks, eight state values per thread.
//    One CTA covers 1024 values of one head; per block of chunks the CTA first
//    tabulates each chunk's decay exp(a_{L-1}), whether it opens a sequence
//    and where its end state goes, so that the loop itself only multiplies,
//    adds and streams the chunk states (loaded several chunks ahead).  Each
//    chunk's entering state goes to ws_henter as 16-bit high parts and
//    remainders, laid out as the scan's B operand of C . h_enter^T: a K-major
//    [P rows (p)] x [N (n)] tile whose 16-byte core-matrix rows (8 n of one p)
//    sit at (n / 8) * 16 P + 16 p, high parts first, remainders P N 2 bytes on.
// ---------------------------------------------------------------------------
constexpr int kPassBlock = 256;  // chunks tabulated at a time
constexpr int kPassAhead = 4;    // chunk states in flight per thread

// 8 consecutive values at element offset `o` (a multiple of 8) of an fp32,
// bf16 or fp16 array (16-byte aligned), as floats / from floats (RNE)
__device__ __forceinline__ void load8(const void* p, int64_t o, int dtype, float (&v)[8]) {
  if (dtype == 0) {
    const float4 a = reinterpret_cast<const float4*>(static_cast<const float*>(p) + o)[0];
    const float4 b = reinterpret_cast<const float4*>(static_cast<const float*>(p) + o)[1];
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
    return;
  }
  const uint4 q = *reinterpret_cast<const uint4*>(static_cast<const char*>(p) + o * 2);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (dtype == 1) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    } else {
      const __half2 h2 = *reinterpret_cast<const __half2*>(&w[k]);
      v[2 * k] = __low2float(h2);
      v[2 * k + 1] = __high2float(h2);
    }
  }
}

__device__ __forceinline__ void store8(void* p, int64_t o, int dtype, const float (&v)[8]) {
  if (dtype == 0) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(p) + o);
    d[0] = make_float4(v[0], v[1], v[2], v[3]);
    d[1] = make_float4(v[4], v[5], v[6], v[7]);
    return;
  }
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    w[k] = dtype == 1 ? pack_pair<__nv_bfloat16>(v[2 * k], v[2 * k + 1])
                      : pack_pair<__half>(v[2 * k], v[2 * k + 1]);
  *reinterpret_cast<uint4*>(static_cast<char*>(p) + o * 2) = make_uint4(w[0], w[1], w[2], w[3]);
}

// One CTA covers 1024 values of one head: kPassRows = 1024 / N rows p, all N
// columns; thread (pl, ng) owns row p = kPassRows blockIdx.x + pl, columns
// [8 ng, 8 ng + 8), so that the threads of a warp write whole 16-byte core-
// matrix rows of the operand layout next to each other.
template <class IT, int P, int N>
__global__ void __launch_bounds__(128) ssd_state_passing_kernel(const SSDArgs a) {
  constexpr int kRows = 1024 / N;
  static_assert(P % kRows == 0, "whole CTAs per head");
  __shared__ float s_decay[kPassBlock];
  __shared__ int64_t s_seq[kPassBlock];
  __shared__ int64_t s_dst[kPassBlock];  // destination row of the end state, or -1
  const int64_t HPN = (int64_t)a.H * P * N;
  const int h = blockIdx.x / (P / kRows);
  const int pl = threadIdx.x % kRows, ng = threadIdx.x / kRows;
  const int pp = (blockIdx.x % (P / kRows)) * kRows + pl;
  const int64_t e = (int64_t)h * P * N + (int64_t)pp * N + ng * 8;  // first of this thread's 8
  const uint32_t hoff = (uint32_t)(ng * (P * 16) + pp * 16);         // its 16-byte operand row
  float hc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int64_t prev = -1;
  for (int cb = 0; cb < a.nchunks; cb += kPassBlock) {
    const int nb = min(kPassBlock, a.nchunks - cb);
    __syncthreads();  // the previous block's tables are no longer read
    for (int i = threadIdx.x; i < nb; i += 128) {
      const int c = cb + i;
      int64_t t0;
      int Lc;
      chunk_span(a, c, &t0, &Lc);
      s_decay[i] = Lc > 0 ? expf(a.ws_acum[((int64_t)c * a.H + h) * a.CS + Lc - 1]) : 1.0f;
      const int64_t sq = load_int(a.seq, c, a.meta64);
      s_seq[i] = sq;
      int64_t dst = -1;
      if (a.intermediate) dst = c;
      else if (sq >= 0 && sq < a.batch && load_int(a.last, sq, a.meta64) == c) dst = sq;
      s_dst[i] = dst;
    }
    __syncthreads();
    const float4* wsp = reinterpret_cast<const float4*>(a.ws_state + (int64_t)cb * HPN + e);
    float4 buf[kPassAhead][2];  // chunk states in flight, kPassAhead chunks ahead
#pragma unroll
    for (int k = 0; k < kPassAhead; ++k)
      if (k < nb) {
        buf[k][0] = wsp[(int64_t)k * (HPN / 4)];
        buf[k][1] = wsp[(int64_t)k * (HPN / 4) + 1];
      }
    for (int i0 = 0; i0 < nb; i0 += kPassAhead) {
#pragma unroll
      for (int u = 0; u < kPassAhead; ++u) {
        const int i = i0 + u;
        if (i >= nb) break;
        const float S[8] = {buf[u][0].x, buf[u][0].y, buf[u][0].z, buf[u][0].w,
                            buf[u][1].x, buf[u][1].y, buf[u][1].z, buf[u][1].w};
        if (i + kPassAhead < nb) {
          buf[u][0] = wsp[(int64_t)(i + kPassAhead) * (HPN / 4)];
          buf[u][1] = wsp[(int64_t)(i + kPassAhead) * (HPN / 4) + 1];
        }
        const int64_t sq = s_seq[i];
        if (cb + i == 0 || sq != prev) {  // the chunk opens sequence sq
#pragma unroll
          for (int k = 0; k < 8; ++k) hc[k] = 0.0f;
          if (a.init && sq >= 0 && sq < a.batch) load8(a.init, sq * HPN + e, a.init_dtype, hc);
        }
        prev = sq;
        {  // the entering state, for the scan
          uint8_t* blk = a.ws_henter + ((int64_t)(cb + i) * a.H + h) * (P * N * 4);
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) split_packed<IT>(hc[2 * k], hc[2 * k + 1], &hi[k], &lo[k]);
          *reinterpret_cast<uint4*>(blk + hoff) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(blk + P * N * 2 + hoff) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        const float d = s_decay[i];
#pragma unroll
        for (int k = 0; k < 8; ++k) hc[k] = d * hc[k] + S[k];
        const int64_t dst = s_dst[i];
        if (dst >= 0) store8(a.states, dst * HPN + e, a.state_dtype, hc);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 3. the scan on the fifth-generation tensor cores: y of up to 128 query
//    tokens (one t-block) of one chunk and head per CTA of 512 threads (four
//    warpgroups).  Thread i of each warpgroup owns query row t = 128 tb + i,
//    which is also tensor-memory lane i of every M = 128 accumulator:
//      columns [0, 64)    C_t . h_enter             (K = N, h_enter split)
//      columns [64, 128)  sum_s M[t,s] x_s          (K = 32 source tokens per slice)
//      columns [128, 256) CB = C . B^T for 128 source tokens (one half of the chunk)
//    The tensor core forms CB for source tokens [0, 128) up front and, for the
//    second t-block, CB for [128, 256) once the first half has been read (its
//    B rows are copied in during slices 0 to 2).
//    Source slice j (tokens [32 j, 32 j + 32), up to the t-block's last row):
//    each thread reads 8 columns of its row of CB, decays and masks them
//    (M[t,s] = CB[t,s] exp(a_t - a_s) dt'_s for s <= t), splits them into high
//    parts and remainders in shared memory (two buffers), and the tensor core adds
//    M_j x_j while the threads go on to slice j + 1; x rows are copied
//    (cp.async) one slice ahead.  Once the last C . B^T is done, the x and z
//    rows of the t-block are copied into the C and B tiles for the epilogue.
//    Shared-memory operands (no-swizzle canonical layouts, see ssd_tc.cuh):
//      cq  C rows of the t-block, K-major: core-matrix row (r, n / 8) at
//          (n / 8) 2048 + 16 r                       (LBO 2048, SBO 128)
//      hm  h_enter high parts | remainders, K-major [64 p x N]: (p, n / 8) at
//          (n / 8) 1024 + 16 p (LBO 1024, SBO 128), as stored by the passing
//          kernel; once C . h_enter is done, the same bytes hold two buffers
//          of M_j high parts | remainders, K-major [128 t x 32 s]: (t, s / 8)
//          at (t / 8) 512 + (s / 8) 128 + 16 (t % 8)  (LBO 128, SBO 512)
//      bs  B rows of one half (128 source tokens), K-major: (s, n / 8) at
//          (n / 8) 2048 + 16 s                       (LBO 2048, SBO 128)
//      xs  x rows of a slice (two buffers), MN-major [64 p x 32 s]: the 8 p
//          of (p / 8, s) at (p / 8) 528 + 16 s       (LBO 128, SBO 528; the
//          padding spreads one token's 8 pieces over distinct banks, so
//          neighbouring threads copy one token's 128-byte row)
//    After the last C . B^T: cq holds the x rows and bs the z rows of the
//    t-block for the epilogue, 128 bytes per row, the 16-byte piece k of row r
//    at r 128 + 16 (k ^ r % 8).
// ---------------------------------------------------------------------------
constexpr int kTB = 128;               // query rows per CTA (the MMA M)
constexpr int kSL = 32;                // source tokens per slice
constexpr int kHalf = 128;             // source tokens per C . B^T block
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColInter = 0, kColIntra = 64, kColCB = 128;
constexpr int kScanMinSmem = 78 * 1024;  // at most two CTAs per SM: 2 x 256 columns
constexpr int kMBytes = kTB * kSL * 2;   // one part (high or remainder) of M_j
constexpr int kXsSBO = 528;              // bytes between 8-p groups of an x slice

template <int P, int N>
struct ScanSmem {
  uint8_t cq[kTB * N * 2];
  uint8_t hm[(2 * P * N * 2 > 4 * kMBytes) ? 2 * P * N * 2 : 4 * kMBytes];
  uint8_t bs[kHalf * N * 2];
  uint8_t xs[2][P / 8 * kXsSBO];
  float acum[kMaxChunk], dtp[kMaxChunk], q[kMaxChunk], qs[kMaxChunk];
  int tame[kMaxChunk / kSL];
  uint64_t bar_h, bar_cb, bar_intra;
  uint32_t tmem;
};

template <class IT, int P, int N>
__global__ void __launch_bounds__(512, 2) ssd_chunk_scan_kernel(const SSDArgs a) {
  static_assert(P == 64 && (N == 64 || N == 128), "headdim 64, dstate 64 or 128");
  static_assert(kTB * P * 2 <= kTB * N * 2 && kTB * P * 2 <= kHalf * N * 2, "x / z rows fit the C / B tiles");
  constexpr bool kBF16 = std::is_same<IT, __nv_bfloat16>::value;
  constexpr uint32_t kIdInter = tc::idesc_f16(kBF16, kTB, 64, false, false);
  constexpr uint32_t kIdCB = tc::idesc_f16(kBF16, kTB, kHalf, false, false);
  constexpr uint32_t kIdIntra = tc::idesc_f16(kBF16, kTB, 64, false, true);
  constexpr int NT = 512;
  const int c = blockIdx.x >> 1, tb = blockIdx.x & 1, h = blockIdx.y;
  // four warpgroups: each covers the 128 rows (tensor-memory lanes); warpgroup
  // wg takes columns [8 wg, 8 wg + 8) of each source slice and output
  // columns [16 wg, 16 wg + 16)
  const int tid = threadIdx.x, warp = tid >> 5, wg = warp >> 2, lrow = tid & 127;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<ScanSmem<P, N>*>(smem_raw);
  int64_t t0;
  int Lc;
  chunk_span(a, c, &t0, &Lc);
  const int r0 = tb * kTB;  // this CTA's query rows [r0, tmax) of the chunk
  if (r0 >= Lc) return;
  if (*reinterpret_cast<volatile unsigned*>(a.err) & kErrMmaTimeout) return;  // a wait gave up
  const int tmax = min(Lc, r0 + kTB);
  const int J = (tmax - 1) / kSL + 1;  // source slices
  const int g = h / a.hr;
  const float* wdt = a.ws_dt + ((int64_t)c * a.H + h) * a.CS;
  const float* wac = a.ws_acum + ((int64_t)c * a.H + h) * a.CS;
  for (int i = tid; i < J * kSL; i += NT) {
    const bool in = i < Lc;
    sm.dtp[i] = in ? wdt[i] : 0.0f;
    sm.acum[i] = in ? wac[i] : 0.0f;
  }
  const uint32_t s_cq = smem_addr(sm.cq), s_hm = smem_addr(sm.hm), s_bs = smem_addr(sm.bs);
  const uint32_t s_xs[2] = {smem_addr(sm.xs[0]), smem_addr(sm.xs[1])};
  const IT* cg = static_cast<const IT*>(a.C);
  const IT* bg = static_cast<const IT*>(a.B);
  const IT* xg = static_cast<const IT*>(a.x);
  // rows [base, base + 128) of a [tokens, groups, N] tensor (C or B), K-major
  auto load_rows = [&](uint32_t dst, const IT* src, int base) {
#pragma unroll 1
    for (int q = tid; q < 128 * (N / 8); q += NT) {
      const int r = q % 128, kg = q / 128, tk = base + r;
      const bool ok = tk < Lc;
      tc::cp16(dst + kg * 2048 + r * 16, src + ((t0 + (ok ? tk : 0)) * a.G + g) * N + kg * 8,
               ok ? 16u : 0u);
    }
  };
  auto load_x = [&](int j) {  // one 16-byte piece per thread, a token's 8 side by side
    const int pg = tid % (P / 8), sl = tid / (P / 8), s = j * kSL + sl;
    const bool ok = s < Lc;
    tc::cp16(s_xs[j & 1] + pg * kXsSBO + sl * 16,
             xg + ((t0 + (ok ? s : 0)) * a.H + h) * P + pg * 8, ok ? 16u : 0u);
  };
  static_assert(kSL * (P / 8) == NT / 2, "one x piece per thread of the first half");
  load_rows(s_cq, cg, r0);
  load_rows(s_bs, bg, 0);
  if (tid < NT / 2) load_x(0);
  tc::cp_commit();
  if (tid == 0) {
    mbar_init(&sm.bar_h, 1);
    mbar_init(&sm.bar_cb, 1);
    mbar_init(&sm.bar_intra, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the entering state, already in operand layout: one bulk copy
    mbar_arrive_expect_tx(&sm.bar_h, 2 * P * N * 2);
    bulk_load(sm.hm, a.ws_henter + ((int64_t)c * a.H + h) * (P * N * 4), 2 * P * N * 2,
              &sm.bar_h);
  }
  if (warp == 0) tc::alloc(smem_addr(&sm.tmem), kTmemCols);
  __syncthreads();  // acum / dtp written
  // per source token: exp(a_e - a_s) dt'_s and exp(a_b - a_s) dt'_s, a_b and
  // a_e at the first and last token of its slice; per slice: whether a_b -
  // a_e <= 60, so that the second form cannot overflow
  for (int i = tid; i < J * kSL; i += NT) {
    const int b = (i / kSL) * kSL, e = min(b + kSL - 1, Lc - 1);
    sm.q[i] = i < Lc ? expf(sm.acum[e] - sm.acum[i]) * sm.dtp[i] : 0.0f;
    sm.qs[i] = i < Lc ? expf(fminf(sm.acum[b] - sm.acum[i], 60.0f)) * sm.dtp[i] : 0.0f;
  }
  if (tid < J) {
    const int b = tid * kSL, e = min(b + kSL - 1, Lc - 1);
    sm.tame[tid] = b < Lc && sm.acum[b] - sm.acum[e] <= 60.0f;
  }
  tc::cp_wait<0>();  // C, B rows [0, 128), x_0
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem;
  bool dead = false;  // a bounded wait gave up: finish without waiting again
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (!dead && !spin_wait(bar, parity, kWaitLimitNs)) {
      dead = true;
      atomicOr(a.err, kErrMmaTimeout);
    }
  };
  auto issue_cb = [&]() {  // CB of the 128 source tokens in bs
#pragma unroll
    for (int kk = 0; kk < N / 16; ++kk)
      tc::mma(tmem + kColCB, tc::sdesc(s_cq + kk * 4096, 2048, 128),
              tc::sdesc(s_bs + kk * 4096, 2048, 128), kIdCB, kk != 0);
    tc::commit(smem_addr(&sm.bar_cb));
  };
  if (tid == 0) {
    wait(&sm.bar_h, 0);
    // C . h_enter^T, high parts then remainders
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int kk = 0; kk < N / 16; ++kk)
        tc::mma(tmem + kColInter, tc::sdesc(s_cq + kk * 4096, 2048, 128),
                tc::sdesc(s_hm + part * (P * N * 2) + kk * 2048, 1024, 128), kIdInter,
                (part | kk) != 0);
    issue_cb();
  }
  // a_t is non-increasing along the chunk when A <= 0 and dt' >= 0: then for
  // a slice wholly at or before t, exp(a_t - a_s) = exp(a_t - a_e) exp(a_e - a_s)
  // with both factors <= 1 (no overflow), one exponential per slice and row
  const bool monotone = a.A[h] <= 0.0f && a.dt_lo >= 0.0f;
  const int t = r0 + lrow;
  const bool trow = t < Lc;
  const int tt = trow ? t : -1;  // no source token is at or before a row past the chunk
  const float at = trow ? sm.acum[t] : 0.0f;
  const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const int m_row = (lrow >> 3) * 512 + (lrow & 7) * 16 + wg * 128;  // 8-column group kg = wg
  const IT* zg = static_cast<const IT*>(a.z);
  const int64_t row = trow ? ((t0 + t) * a.H + h) * P : 0;
  uint32_t ph_cb = 0, ph_in = 0;
  const bool two_halves = J * kSL > kHalf;
  // this thread's row of CB for the slice in hand; the next slice's row is
  // read while this one is processed (one tensor-memory round trip per slice
  // hidden), except across the two halves of the chunk
  float cb[8], cbn[8];
  for (int j = 0; j < J; ++j) {
    const int s0 = j * kSL;
    if ((s0 % kHalf) == 0) {  // a new C . B^T block: wait for it, read the slice
      wait(&sm.bar_cb, ph_cb);
      ph_cb ^= 1;
      tc::fence_after_sync();
      tc::ld8(lane_base + kColCB + (s0 % kHalf) + 8 * wg, cb);
      if (s0 + kHalf >= J * kSL) {
        // the last MMA reading the C and B rows is done: the epilogue's x rows
        // of the t-block go where the C rows were, its z rows where the B rows
        // were (row r's 16-byte piece k at (k ^ r % 8), so the epilogue's reads
        // of one piece of 32 rows spread over all banks); they join the next x
        // slice's copy group
#pragma unroll
        for (int u = 0; u < (kTB * 8 * 2) / NT; ++u) {
          const int q = tid + u * NT, which = q / (kTB * 8), r = (q / 8) % kTB, k = q % 8;
          const IT* src = which ? zg : xg;
          if (src) {
            const bool ok = r0 + r < Lc;
            tc::cp16((which ? s_bs : s_cq) + r * 128 + ((k ^ (r & 7)) << 4),
                     src + ((t0 + (ok ? r0 + r : 0)) * a.H + h) * P + k * 8, ok ? 16u : 0u);
          }
        }
      }
    }
    tc::wait_ld();
    if (j > 0 && (s0 % kHalf) != 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) cb[k] = cbn[k];
    }
    if (j + 1 < J && ((s0 + kSL) % kHalf) != 0)
      tc::ld8(lane_base + kColCB + ((s0 + kSL) % kHalf) + 8 * wg, cbn);
    // M_j, row t, columns [8 wg, 8 wg + 8) of the slice, into buffer j % 2
    // (free: M_{j-2} x_{j-2} is done)
    const int sb = s0 + 8 * wg;  // first source token of this thread's columns
    // With a_t non-increasing, exp(a_t - a_s) = exp(a_t - a_ref) exp(a_ref - a_s):
    // a slice wholly at or before t takes a_ref = its last token (both factors
    // <= 1); the slice holding t takes a_ref = its first token when the slice
    // decays by at most e^60 (first factor <= 1, second <= e^60); otherwise one
    // exponential per entry.
    const float* tab = sm.q;
    float rf = 0.0f;
    bool per_entry = false;
    if (s0 <= tt) {
      if (monotone && s0 + kSL - 1 <= tt) {
        rf = expf(at - sm.acum[s0 + kSL - 1]);
      } else if (monotone && sm.tame[j]) {
        rf = expf(at - sm.acum[s0]);
        tab = sm.qs;
      } else {
        per_entry = true;
      }
    }
    uint8_t* m_hi = sm.hm + (j & 1) * (2 * kMBytes) + m_row;
    {
      uint32_t hp[4], lp[4];
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int s = sb + k + e;
          float f;
          if (!per_entry) f = s <= tt ? rf * tab[s] : 0.0f;
          else f = s <= tt ? __expf(at - sm.acum[s]) * sm.dtp[s] : 0.0f;
          v[e] = cb[k + e] * f;
        }
        split_packed<IT>(v[0], v[1], &hp[k / 2], &lp[k / 2]);
      }
      *reinterpret_cast<uint4*>(m_hi) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
      *reinterpret_cast<uint4*>(m_hi + kMBytes) = make_uint4(lp[0], lp[1], lp[2], lp[3]);
    }
    if (j > 0) {  // M_{j-1} x_{j-1} done: x buffer (j + 1) % 2 and M buffer (j + 1) % 2 free
      wait(&sm.bar_intra, ph_in);
      ph_in ^= 1;
    }
    if (j + 1 < J && tid < NT / 2) load_x(j + 1);
    tc::cp_commit();
    if (two_halves && j == 0) {
      // the first half's C . B^T has read bs (its barrier was waited for
      // above): B rows [128, 256) go in now, one group behind x_1, and must
      // have landed by slice 2 (the copy groups complete in order)
      load_rows(s_bs, bg, kHalf);
      tc::cp_commit();
    }
    if (two_halves && j < 2) tc::cp_wait<2>();  // x_j has landed (B may still be in flight)
    else tc::cp_wait<1>();                      // all but x_{j+1}: x_j (and B) have landed
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
      // every row of the first half's CB has been read (each thread waited
      // for its last read before the barrier): C . B^T of the second half
      if (two_halves && s0 + kSL == kHalf) issue_cb();
      // sum_s M[t,s] x_s: high parts, then remainders
      const uint32_t s_m = s_hm + (j & 1) * (2 * kMBytes);
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < kSL / 16; ++kk)
          tc::mma(tmem + kColIntra, tc::sdesc(s_m + part * kMBytes + kk * 256, 128, 512),
                  tc::sdesc(s_xs[j & 1] + kk * 256, 128, kXsSBO), kIdIntra, (j | part | kk) != 0);
      tc::commit(smem_addr(&sm.bar_intra));
    }
  }
  wait(&sm.bar_intra, ph_in);  // the last M x done: every accumulator is final
  tc::cp_wait<0>();             // this thread's pieces of the x and z rows
  tc::fence_before_sync();
  __syncthreads();              // ... and every other thread's
  tc::fence_after_sync();
  // y = intra + exp(a_t) C_t . h_enter + D x_t, times silu(z_t): output
  // columns [16 wg, 16 wg + 16) of row t
  IT* og = static_cast<IT*>(a.out);
  const float dec = expf(at);
  const float Dh = (a.D && !a.D_per_dim) ? a.D[h] : 0.0f;
#pragma unroll 1
  for (int c8 = 2 * wg; c8 < 2 * wg + 2; ++c8) {
    float yi[8], yo[8];
    tc::ld8(lane_base + kColInter + c8 * 8, yi);
    tc::ld8(lane_base + kColIntra + c8 * 8, yo);
    uint4 xq = make_uint4(0u, 0u, 0u, 0u), zq = make_uint4(0u, 0u, 0u, 0u);
    if (trow) {
      const int off = lrow * 128 + ((c8 ^ (lrow & 7)) << 4);
      xq = *reinterpret_cast<const uint4*>(sm.cq + off);
      if (zg) zq = *reinterpret_cast<const uint4*>(sm.bs + off);
    }
    tc::wait_ld();
    if (trow) {
      const IT* xv = reinterpret_cast<const IT*>(&xq);
      const IT* zv = reinterpret_cast<const IT*>(&zq);
      uint32_t packed[4];
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int p = c8 * 8 + k + e;
          float y = yo[k + e] + dec * yi[k + e];
          const float x = io_to_float<IT>(xv[k + e]);
          if (a.D) y += (a.D_per_dim ? a.D[h * P + p] : Dh) * x;
          if (zg) {
            const float zz = io_to_float<IT>(zv[k + e]);
            y *= zz * __frcp_rn(1.0f + __expf(-zz));
          }
          v[e] = y;
        }
        packed[k / 2] = pack_pair<IT>(v[0], v[1]);
      }
      reinterpret_cast<uint4*>(og + row)[c8] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, kTmemCols);
}

template <class IT, int P, int N>
cudaError_t launch(const SSDArgs& a, cudaStream_t stream) {
  auto state = ssd_chunk_state_kernel<IT, P, N>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(state, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(StateSmem<N>))) != cudaSuccess)
    return e;
  const unsigned pairs = (a.hr % 2 == 0) ? (unsigned)(a.H / 2) : (unsigned)a.H;
  state<<<dim3(a.nchunks, pairs), 256, sizeof(StateSmem<N>), stream>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  static_assert((P * N) % 1024 == 0, "a state-passing CTA covers 1024 values of one head");
  ssd_state_passing_kernel<IT, P, N>
      <<<(unsigned)((int64_t)a.H * P * N / 1024), 128, 0, stream>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto scan = ssd_chunk_scan_kernel<IT, P, N>;
  const int smem = (int)sizeof(ScanSmem<P, N>) > kScanMinSmem ? (int)sizeof(ScanSmem<P, N>)
                                                                : kScanMinSmem;
  if ((e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  scan<<<dim3((unsigned)a.nchunks * 2, a.H), 512, smem, stream>>>(a);
  return cudaGetLastError();
}

// chunk states (fp32), entering states (16-bit pairs), dt', a_t
int64_t workspace_bytes(int64_t nchunks, int64_t H, int64_t G, int64_t P, int64_t N,
                        int64_t CS) {
  (void)G;
  auto up = [](int64_t b) { return (b + 255) / 256 * 256; };
  return 2 * up(nchunks * H * P * N * 4) + 2 * up(nchunks * H * CS * 4);
}

}  // namespace ssd

namespace {
ssu_status bad(ssu_status code, const char* fmt, ...) {
  char msg[300];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof msg, fmt, ap);
  va_end(ap);
  return ssu::record_error(code, msg);
}
bool is_idx(ssu_dtype d) { return d == SSU_I32 || d == SSU_I64; }
bool is_float(ssu_dtype d) { return d == SSU_F32 || d == SSU_BF16 || d == SSU_F16; }
int code(ssu_dtype d) { return d == SSU_F32 ? 0 : d == SSU_BF16 ? 1 : 2; }
bool a16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }
}  // namespace

#pragma GCC visibility push(default)
extern "C" {

int64_t ssd_workspace_bytes(int64_t nchunks, int64_t nheads, int64_t ngroups, int64_t headdim,
                            int64_t dstate, int64_t chunk_size) {
  if (nchunks < 0 || nheads < 0 || ngroups < 0 || headdim < 0 || dstate < 0 || chunk_size < 0)
    return -1;
  return ssd::workspace_bytes(nchunks, nheads, ngroups, headdim, dstate, chunk_size);
}

ssu_status ssd_combined_fwd_varlen(const ssd_params* p, void* workspace, int64_t workspace_bytes,
                                   struct CUstream_st* stream) {
  if (!p) return bad(SSU_ERR_INVALID_ARGUMENT, "params must not be NULL");
  if (p->io_dtype != SSU_BF16 && p->io_dtype != SSU_F16)
    return bad(SSU_ERR_INVALID_ARGUMENT, "x, B and C must share one of fp16 / bf16");
  if (p->tokens < 0 || p->nheads < 1 || p->ngroups < 1 || p->nheads % p->ngroups != 0)
    return bad(SSU_ERR_INVALID_ARGUMENT, "heads must be a positive multiple of groups");
  if (!((p->headdim == 64) && (p->dstate == 64 || p->dstate == 128)))
    return bad(SSU_ERR_UNSUPPORTED, "headdim 64 with dstate 64 or 128 only, got %lld / %lld",
               (long long)p->headdim, (long long)p->dstate);
  if (p->chunk_size < 16 || p->chunk_size > ssd::kMaxChunk || p->chunk_size % 16 != 0)
    return bad(p->chunk_size <= 0 ? SSU_ERR_INVALID_ARGUMENT : SSU_ERR_UNSUPPORTED,
               "chunk_size must be a multiple of 16 in [16, %d], got %lld", ssd::kMaxChunk,
               (long long)p->chunk_size);
  if (p->nchunks < 1) return bad(SSU_ERR_INVALID_ARGUMENT, "cu_chunk_seqlens must have at least two entries");
  if (p->batch < 0) return bad(SSU_ERR_INVALID_ARGUMENT, "batch must be >= 0");
  if (p->tokens > 0x7fffffffLL || p->nchunks > 0x3fffffffLL || p->nheads > 65535)
    return bad(SSU_ERR_UNSUPPORTED, "tokens below 2^31, chunks below 2^30 and heads up to 65535");
  if (!is_idx(p->meta_dtype))
    return bad(SSU_ERR_INVALID_ARGUMENT, "chunk metadata must be int32 or int64");
  if (!is_float(p->state_dtype)) return bad(SSU_ERR_INVALID_ARGUMENT, "state_dtype must be fp32, bf16 or fp16");
  if (p->initial_states && !is_float(p->initial_dtype))
    return bad(SSU_ERR_INVALID_ARGUMENT, "initial_states must be fp32, bf16 or fp16");
  if (!p->x || !p->dt || !p->A || !p->B || !p->C || !p->out || !p->states ||
      !p->cu_chunk_seqlens || !p->seq_idx || (!p->return_intermediate_states && !p->last_chunk_indices))
    return bad(SSU_ERR_INVALID_ARGUMENT, "x, dt, A, B, C, out, states and the chunk metadata must not be NULL");
  if (!a16(p->x) || !a16(p->B) || !a16(p->C) || !a16(p->out) || (p->z && !a16(p->z)) ||
      !a16(p->states) || (p->initial_states && !a16(p->initial_states)))
    return bad(SSU_ERR_INVALID_ARGUMENT,
               "x, z, out, B, C, states and initial_states must be 16-byte aligned");
  if (!(p->dt_min <= p->dt_max)) return bad(SSU_ERR_INVALID_ARGUMENT, "dt_limit must be (lo, hi) with lo <= hi");
  const int64_t need = ssd::workspace_bytes(p->nchunks, p->nheads, p->ngroups, p->headdim,
                                            p->dstate, p->chunk_size);
  if (!workspace || workspace_bytes < need || !a16(workspace))
    return bad(SSU_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned and hold %lld bytes, got %lld",
               (long long)need, (long long)workspace_bytes);
  ssd::SSDArgs a{};
  a.x = p->x;
  a.dt = p->dt;
  a.A = p->A;
  a.B = p->B;
  a.C = p->C;
  a.D = p->D;
  a.D_per_dim = p->D_per_dim;
  a.z = p->z;
  a.dt_bias = p->dt_bias;
  a.softplus = p->dt_softplus;
  a.dt_lo = p->dt_min;
  a.dt_hi = p->dt_max;
  a.out = p->out;
  a.T = (int)p->tokens;
  a.H = (int)p->nheads;
  a.G = (int)p->ngroups;
  a.hr = (int)(p->nheads / p->ngroups);
  a.CS = (int)p->chunk_size;
  a.nchunks = (int)p->nchunks;
  a.batch = (int)p->batch;
  a.cu_chunk = p->cu_chunk_seqlens;
  a.seq = p->seq_idx;
  a.last = p->last_chunk_indices;
  a.meta64 = p->meta_dtype == SSU_I64;
  a.init = p->initial_states;
  a.init_dtype = code(p->initial_dtype);
  a.states = p->states;
  a.state_dtype = code(p->state_dtype);
  a.intermediate = p->return_intermediate_states != 0;
  char* ws = static_cast<char*>(workspace);
  auto up = [](int64_t b) { return (b + 255) / 256 * 256; };
  a.ws_state = reinterpret_cast<float*>(ws);
  ws += up(p->nchunks * p->nheads * p->headdim * p->dstate * 4);
  a.ws_henter = reinterpret_cast<uint8_t*>(ws);
  ws += up(p->nchunks * p->nheads * p->headdim * p->dstate * 4);
  a.ws_dt = reinterpret_cast<float*>(ws);
  ws += up(p->nchunks * p->nheads * p->chunk_size * 4);
  a.ws_acum = reinterpret_cast<float*>(ws);
  a.err = ssu::device_error_word();
  if (!a.err) return bad(SSU_ERR_CUDA, "device error word unavailable");
  cudaError_t e;
  const cudaStream_t s = (cudaStream_t)stream;
  if (p->io_dtype == SSU_BF16)
    e = p->dstate == 128 ? ssd::launch<__nv_bfloat16, 64, 128>(a, s)
                         : ssd::launch<__nv_bfloat16, 64, 64>(a, s);
  else
    e = p->dstate == 128 ? ssd::launch<__half, 64, 128>(a, s) : ssd::launch<__half, 64, 64>(a, s);
  if (e != cudaSuccess) return bad(SSU_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  ssu::record_error(SSU_OK, "");
  return SSU_OK;
}

}  // extern "C"
#pragma GCC visibility pop
