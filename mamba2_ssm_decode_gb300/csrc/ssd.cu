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
//   bmm          CB[t,s] = C_t . B_s                       (once per group)
//   chunk_scan   y_t    = sum_{s<=t} CB[t,s] exp(a_t - a_s) dt'_s x_s
//                         + exp(a_t) C_t . h_enter + D x_t     (times silu(z_t))
// The dense contractions (S, CB, the intra-chunk product and C . h_enter) run
// on the tensor cores: warp-level m16n8k16 MMAs with fp32 accumulation, fed by
// ldmatrix from padded (bank-conflict-free) shared tiles.  The inputs x, B, C
// are 16-bit already; an operand the kernels compute (w_s x_s, the scaled CB,
// h_enter) is split into a 16-bit high part and a 16-bit remainder and
// multiplied twice, so that it enters the products to about 2^-16 instead of
// 2^-8 (the outputs of these sums often cancel to far below their terms).
// Four launches on the caller's stream, with the chunk states, dt' and a_t
// and CB in a caller-provided workspace.
#include <cstdarg>
#include <cstdio>

#include "../../include/ssu.h"
#include "ssu_headrun.cuh"

namespace ssu {
ssu_status record_error(ssu_status code, const char* message);  // ssu_abi.cu
}

namespace ssd {
using namespace ssu;

constexpr int kMaxChunk = 256;  // largest supported chunk_size
constexpr int kTile = 64;       // tokens per scan / bmm tile

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
  float* ws_state;  // [nchunks, H, P, N]: chunk-local states, then entering states
  float* ws_dt;     // [nchunks, H, CS]: dt'
  float* ws_acum;   // [nchunks, H, CS]: a_t
  float* ws_cb;     // [nchunks, G, CS, CS]: C_t . B_s (s <= t)
};

// v = hi + lo with hi, lo in the io dtype (lo: the rounding remainder of hi)
template <class IT>
__device__ __forceinline__ void split2(float v, IT* hi, IT* lo) {
  *hi = float_to_io<IT>(v);
  *lo = float_to_io<IT>(v - io_to_float<IT>(*hi));
}

// packed (low, high) pairs of the high parts and of the remainders of (a, b)
template <class IT>
__device__ __forceinline__ void split_pair(float a, float b, uint32_t* hi, uint32_t* lo) {
  IT ah, al, bh, bl;
  split2<IT>(a, &ah, &al);
  split2<IT>(b, &bh, &bl);
  *hi = pack_pair<IT>(io_to_float<IT>(ah), io_to_float<IT>(bh));
  *lo = pack_pair<IT>(io_to_float<IT>(al), io_to_float<IT>(bl));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&a)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float load_f(const void* p, int64_t i, int dtype) {
  if (dtype == 0) return static_cast<const float*>(p)[i];
  if (dtype == 1) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return __half2float(static_cast<const __half*>(p)[i]);
}

__device__ __forceinline__ void store_f(void* p, int64_t i, int dtype, float v) {
  if (dtype == 0) static_cast<float*>(p)[i] = v;
  else if (dtype == 1) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else static_cast<__half*>(p)[i] = __float2half_rn(v);
}

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

// 8 consecutive 16-bit values from global memory into shared (16-byte aligned)
template <class IT>
__device__ __forceinline__ void copy8(IT* dst, const IT* src) {
  *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
}

// ---------------------------------------------------------------------------
// 1. dt', a_t and the chunk-local state S (one CTA per chunk and head)
// ---------------------------------------------------------------------------
template <class IT, int P, int N>
__global__ void __launch_bounds__(128) ssd_chunk_state_kernel(const SSDArgs a) {
  constexpr int KB = 32;  // tokens per staged block
  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float s_dtp[kMaxChunk], s_acum[kMaxChunk], s_w[kMaxChunk];
  __shared__ __align__(16) IT Xs[2][KB][P + 8];  // w_s x_s: high parts, remainders
  __shared__ __align__(16) IT Bs[KB][N + 8];
  int64_t t0;
  int Lc;
  chunk_span(a, c, &t0, &Lc);
  const int g = h / a.hr;
  const float Ah = a.A[h];
  const float bias = a.dt_bias ? a.dt_bias[h] : 0.0f;
  for (int i = tid; i < kMaxChunk; i += 128) {
    float d = 0.0f;
    if (i < Lc) {
      d = a.dt[(t0 + i) * a.H + h] + bias;
      if (a.softplus) d = softplus_f(d);
      d = fminf(fmaxf(d, a.dt_lo), a.dt_hi);
    }
    s_dtp[i] = d;
    s_acum[i] = Ah * d;
  }
  __syncthreads();
  // inclusive running sum over the chunk: warp 0, eight values per lane
  if (warp == 0) {
    float v[8], run = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      run += s_acum[lane * 8 + k];
      v[k] = run;
    }
    float incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    const float before = incl - run;
#pragma unroll
    for (int k = 0; k < 8; ++k) s_acum[lane * 8 + k] = v[k] + before;
  }
  __syncthreads();
  const float a_end = Lc > 0 ? s_acum[Lc - 1] : 0.0f;
  float* wdt = a.ws_dt + ((int64_t)c * a.H + h) * a.CS;
  float* wac = a.ws_acum + ((int64_t)c * a.H + h) * a.CS;
  for (int i = tid; i < Lc; i += 128) {
    wdt[i] = s_dtp[i];
    wac[i] = s_acum[i];
    s_w[i] = expf(a_end - s_acum[i]) * s_dtp[i];
  }
  __syncthreads();

  // S[p][n] = sum_s w_s x_s[p] B_s[n]: M = P (p), N = N (n), K = tokens.
  // Warp w owns p rows [16 w, 16 w + 16).
  constexpr int NT = N / 8;
  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
  const IT* xg = static_cast<const IT*>(a.x);
  const IT* bg = static_cast<const IT*>(a.B);
  for (int k0 = 0; k0 < Lc; k0 += KB) {
    // stage w_s x_s (rounded to the io dtype) and B_s, zero past the chunk
    for (int i = tid; i < KB * (P / 8); i += 128) {
      const int r = i / (P / 8), q8 = (i - r * (P / 8)) * 8;
      const int s = k0 + r;
      if (s < Lc) {
        uint4 raw = __ldg(reinterpret_cast<const uint4*>(xg + ((t0 + s) * a.H + h) * P + q8));
        const IT* e = reinterpret_cast<const IT*>(&raw);
        const float w = s_w[s];
        __align__(16) IT hi[8];
        __align__(16) IT lo[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) split2<IT>(w * io_to_float<IT>(e[k]), &hi[k], &lo[k]);
        *reinterpret_cast<uint4*>(&Xs[0][r][q8]) = *reinterpret_cast<const uint4*>(hi);
        *reinterpret_cast<uint4*>(&Xs[1][r][q8]) = *reinterpret_cast<const uint4*>(lo);
      } else {
        *reinterpret_cast<uint4*>(&Xs[0][r][q8]) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(&Xs[1][r][q8]) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    for (int i = tid; i < KB * (N / 8); i += 128) {
      const int r = i / (N / 8), q8 = (i - r * (N / 8)) * 8;
      const int s = k0 + r;
      if (s < Lc) copy8(&Bs[r][q8], bg + ((t0 + s) * a.G + g) * N + q8);
      else *reinterpret_cast<uint4*>(&Bs[r][q8]) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    if (warp * 16 < P) {
#pragma unroll
      for (int ks = 0; ks < KB / 16; ++ks) {
        const int m = lane >> 3, j = lane & 7;
        uint32_t ah[4], al[4];  // A = (w x)^T: rows p, columns s (stored [s][p])
        ldsm_x4_t(ah, saddr(&Xs[0][ks * 16 + j + (m >= 2 ? 8 : 0)][warp * 16 + (m & 1 ? 8 : 0)]));
        ldsm_x4_t(al, saddr(&Xs[1][ks * 16 + j + (m >= 2 ? 8 : 0)][warp * 16 + (m & 1 ? 8 : 0)]));
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          uint32_t bf[4];  // B: rows s, columns n (stored [s][n]: transposed loads)
          ldsm_x4_t(bf, saddr(&Bs[ks * 16 + j + (m & 1 ? 8 : 0)][np * 16 + (m >= 2 ? 8 : 0)]));
          mma_16816<IT>(acc[2 * np], ah, bf[0], bf[1]);
          mma_16816<IT>(acc[2 * np + 1], ah, bf[2], bf[3]);
          mma_16816<IT>(acc[2 * np], al, bf[0], bf[1]);
          mma_16816<IT>(acc[2 * np + 1], al, bf[2], bf[3]);
        }
      }
    }
    __syncthreads();
  }
  if (warp * 16 < P) {
    float* out = a.ws_state + ((int64_t)c * a.H + h) * P * N;
    const int r0 = warp * 16 + (lane >> 2), c0 = 2 * (lane & 3);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      *reinterpret_cast<float2*>(&out[r0 * N + j * 8 + c0]) = make_float2(acc[j][0], acc[j][1]);
      *reinterpret_cast<float2*>(&out[(r0 + 8) * N + j * 8 + c0]) =
          make_float2(acc[j][2], acc[j][3]);
    }
  }
}

// ---------------------------------------------------------------------------
// 2. state passing: sequential over chunks, four state values per thread.
//    One CTA covers 512 values of one head; per block of chunks the CTA first
//    tabulates each chunk's decay exp(a_{L-1}), whether it opens a sequence
//    and where its end state goes, so that the loop itself only multiplies,
//    adds and streams the chunk states (loaded several chunks ahead).
// ---------------------------------------------------------------------------
constexpr int kPassBlock = 256;  // chunks tabulated at a time
constexpr int kPassAhead = 4;    // chunk states in flight per thread

template <int P, int N>
__global__ void __launch_bounds__(128) ssd_state_passing_kernel(const SSDArgs a) {
  __shared__ float s_decay[kPassBlock];
  __shared__ int64_t s_seq[kPassBlock];
  __shared__ int64_t s_dst[kPassBlock];  // destination row of the end state, or -1
  const int64_t HPN = (int64_t)a.H * P * N;
  const int64_t e = ((int64_t)blockIdx.x * 128 + threadIdx.x) * 4;  // < HPN (exact grid)
  const int h = (int)(((int64_t)blockIdx.x * 512) / (P * N));
  float4 hc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
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
    float4 buf[kPassAhead];
#pragma unroll
    for (int k = 0; k < kPassAhead; ++k)
      if (k < nb) buf[k] = wsp[(int64_t)k * (HPN / 4)];
    for (int i = 0; i < nb; ++i) {
      const float4 S = buf[i % kPassAhead];
      if (i + kPassAhead < nb) buf[i % kPassAhead] = wsp[(int64_t)(i + kPassAhead) * (HPN / 4)];
      const int64_t sq = s_seq[i];
      if (cb + i == 0 || sq != prev) {  // the chunk opens sequence sq
        hc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (a.init && sq >= 0 && sq < a.batch) {
          const int64_t o = sq * HPN + e;
          hc = make_float4(load_f(a.init, o, a.init_dtype), load_f(a.init, o + 1, a.init_dtype),
                           load_f(a.init, o + 2, a.init_dtype),
                           load_f(a.init, o + 3, a.init_dtype));
        }
      }
      prev = sq;
      // the entering state, for the scan
      reinterpret_cast<float4*>(a.ws_state + (int64_t)(cb + i) * HPN + e)[0] = hc;
      const float d = s_decay[i];
      hc = make_float4(d * hc.x + S.x, d * hc.y + S.y, d * hc.z + S.z, d * hc.w + S.w);
      const int64_t dst = s_dst[i];
      if (dst >= 0) {
        const int64_t o = dst * HPN + e;
        store_f(a.states, o, a.state_dtype, hc.x);
        store_f(a.states, o + 1, a.state_dtype, hc.y);
        store_f(a.states, o + 2, a.state_dtype, hc.z);
        store_f(a.states, o + 3, a.state_dtype, hc.w);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 3. CB[t][s] = C_t . B_s for s <= t, once per chunk and group (64 x 64 tiles;
//    exact products of 16-bit inputs, fp32 sums)
// ---------------------------------------------------------------------------
template <class IT, int N>
__global__ void __launch_bounds__(128) ssd_bmm_kernel(const SSDArgs a) {
  const int c = blockIdx.x, g = blockIdx.y;
  const int tb = blockIdx.z / (kMaxChunk / kTile), sb = blockIdx.z % (kMaxChunk / kTile);
  if (sb > tb) return;  // above the diagonal: never read
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ __align__(16) IT Cs[kTile][N + 8];
  __shared__ __align__(16) IT Bs[kTile][N + 8];
  int64_t t0;
  int Lc;
  chunk_span(a, c, &t0, &Lc);
  if (tb * kTile >= Lc) return;
  const IT* bg = static_cast<const IT*>(a.B);
  const IT* cg = static_cast<const IT*>(a.C);
  for (int i = tid; i < kTile * (N / 8); i += 128) {
    const int r = i / (N / 8), q8 = (i - r * (N / 8)) * 8;
    const int t = tb * kTile + r, sI = sb * kTile + r;
    if (t < Lc) copy8(&Cs[r][q8], cg + ((t0 + t) * a.G + g) * N + q8);
    else *reinterpret_cast<uint4*>(&Cs[r][q8]) = make_uint4(0u, 0u, 0u, 0u);
    if (sI < Lc) copy8(&Bs[r][q8], bg + ((t0 + sI) * a.G + g) * N + q8);
    else *reinterpret_cast<uint4*>(&Bs[r][q8]) = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  float acc[kTile / 8][4];
#pragma unroll
  for (int j = 0; j < kTile / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
  const int m = lane >> 3, j8 = lane & 7;
#pragma unroll
  for (int ks = 0; ks < N / 16; ++ks) {
    uint32_t af[4];  // A = C: rows t, columns n
    ldsm_x4(af, saddr(&Cs[warp * 16 + j8 + (m & 1 ? 8 : 0)][ks * 16 + (m >= 2 ? 8 : 0)]));
#pragma unroll
    for (int np = 0; np < kTile / 16; ++np) {
      uint32_t bf[4];  // B = B^T: rows n, columns s (stored [s][n])
      ldsm_x4(bf, saddr(&Bs[np * 16 + j8 + (m >= 2 ? 8 : 0)][ks * 16 + (m & 1 ? 8 : 0)]));
      mma_16816<IT>(acc[2 * np], af, bf[0], bf[1]);
      mma_16816<IT>(acc[2 * np + 1], af, bf[2], bf[3]);
    }
  }
  float* cb = a.ws_cb + ((int64_t)c * a.G + g) * a.CS * a.CS;
  const int r0 = tb * kTile + warp * 16 + (lane >> 2), c0 = sb * kTile + 2 * (lane & 3);
#pragma unroll
  for (int j = 0; j < kTile / 8; ++j) {
    if (c0 + j * 8 >= a.CS) break;  // chunk sizes below 64: columns past the chunk
    if (r0 < a.CS)
      *reinterpret_cast<float2*>(&cb[(int64_t)r0 * a.CS + c0 + j * 8]) =
          make_float2(acc[j][0], acc[j][1]);
    if (r0 + 8 < a.CS)
      *reinterpret_cast<float2*>(&cb[(int64_t)(r0 + 8) * a.CS + c0 + j * 8]) =
          make_float2(acc[j][2], acc[j][3]);
  }
}

// ---------------------------------------------------------------------------
// 4. the scan: y of one chunk and head per CTA, 64 query tokens at a time
// ---------------------------------------------------------------------------
template <class IT, int P, int N>
struct ScanSmem {
  float acum[kMaxChunk], dtp[kMaxChunk];
  IT H[2][P][N + 8];  // h_enter: high parts, remainders
  IT Cq[kTile][N + 8];
  IT Xs[kTile][P + 8];
};

template <class IT, int P, int N>
__global__ void __launch_bounds__(128) ssd_chunk_scan_kernel(const SSDArgs a) {
  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<ScanSmem<IT, P, N>*>(smem_raw);
  int64_t t0;
  int Lc;
  chunk_span(a, c, &t0, &Lc);
  if (Lc <= 0) return;
  const int g = h / a.hr;
  const float* wdt = a.ws_dt + ((int64_t)c * a.H + h) * a.CS;
  const float* wac = a.ws_acum + ((int64_t)c * a.H + h) * a.CS;
  for (int i = tid; i < Lc; i += 128) {
    sm.dtp[i] = wdt[i];
    sm.acum[i] = wac[i];
  }
  const float* hin = a.ws_state + ((int64_t)c * a.H + h) * P * N;
  for (int i = tid; i < P * N / 4; i += 128) {
    const int p = (i * 4) / N, n = (i * 4) - p * N;
    const float4 v = *reinterpret_cast<const float4*>(&hin[p * N + n]);
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) split2<IT>(vv[k], &sm.H[0][p][n + k], &sm.H[1][p][n + k]);
  }
  const IT* cg = static_cast<const IT*>(a.C);
  const IT* xg = static_cast<const IT*>(a.x);
  const float* cbg = a.ws_cb + ((int64_t)c * a.G + g) * a.CS * a.CS;
  const IT* zg = static_cast<const IT*>(a.z);
  IT* og = static_cast<IT*>(a.out);
  const int m = lane >> 3, j8 = lane & 7;
  const int rl = warp * 16 + (lane >> 2);  // this thread's rows rl, rl + 8 of a query tile
  const int c0 = 2 * (lane & 3);
  constexpr int PT = P / 8;

  for (int q0 = 0; q0 < Lc; q0 += kTile) {
    __syncthreads();  // the previous query tile's buffers are free
    for (int i = tid; i < kTile * (N / 8); i += 128) {
      const int r = i / (N / 8), q8 = (i - r * (N / 8)) * 8;
      const int t = q0 + r;
      if (t < Lc) copy8(&sm.Cq[r][q8], cg + ((t0 + t) * a.G + g) * N + q8);
      else *reinterpret_cast<uint4*>(&sm.Cq[r][q8]) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    // C_t . h_enter (A = C rows t; B = h^T, stored [p][n]), high parts + remainders
    float yi[PT][4];
#pragma unroll
    for (int jj = 0; jj < PT; ++jj) yi[jj][0] = yi[jj][1] = yi[jj][2] = yi[jj][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < N / 16; ++ks) {
      uint32_t af[4];
      ldsm_x4(af, saddr(&sm.Cq[warp * 16 + j8 + (m & 1 ? 8 : 0)][ks * 16 + (m >= 2 ? 8 : 0)]));
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int np = 0; np < PT / 2; ++np) {
          uint32_t bf[4];
          ldsm_x4(bf, saddr(&sm.H[part][np * 16 + j8 + (m >= 2 ? 8 : 0)]
                                     [ks * 16 + (m & 1 ? 8 : 0)]));
          mma_16816<IT>(yi[2 * np], af, bf[0], bf[1]);
          mma_16816<IT>(yi[2 * np + 1], af, bf[2], bf[3]);
        }
      }
    }
    const int tA = q0 + rl, tB = tA + 8;
    const float aA = tA < Lc ? sm.acum[tA] : 0.0f, aB = tB < Lc ? sm.acum[tB] : 0.0f;
    // sum_{s <= t} (C_t . B_s) exp(a_t - a_s) dt'_s x_s, 64 source tokens at a time
    float yo[PT][4];
#pragma unroll
    for (int jj = 0; jj < PT; ++jj) yo[jj][0] = yo[jj][1] = yo[jj][2] = yo[jj][3] = 0.0f;
    for (int s0 = 0; s0 <= q0; s0 += kTile) {
      // this thread's CB values (rows tA, tB; the accumulator layout), issued
      // before the x tile is staged
      float cb[kTile / 8][4];
#pragma unroll
      for (int jj = 0; jj < kTile / 8; ++jj) {
        const int sI = s0 + jj * 8 + c0;  // even: sI + 1 < CS whenever sI < Lc
        float2 u = make_float2(0.0f, 0.0f), w = make_float2(0.0f, 0.0f);
        if (sI < Lc && tA < Lc) u = *reinterpret_cast<const float2*>(&cbg[(int64_t)tA * a.CS + sI]);
        if (sI < Lc && tB < Lc) w = *reinterpret_cast<const float2*>(&cbg[(int64_t)tB * a.CS + sI]);
        cb[jj][0] = u.x;
        cb[jj][1] = u.y;
        cb[jj][2] = w.x;
        cb[jj][3] = w.y;
      }
      __syncthreads();  // the previous source tile is free
      for (int i = tid; i < kTile * (P / 8); i += 128) {
        const int r = i / (P / 8), q8 = (i - r * (P / 8)) * 8;
        const int sI = s0 + r;
        if (sI < Lc) copy8(&sm.Xs[r][q8], xg + ((t0 + sI) * a.H + h) * P + q8);
        else *reinterpret_cast<uint4*>(&sm.Xs[r][q8]) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
      // scale by exp(a_t - a_s) dt'_s, mask s > t, split into A fragments
      uint32_t ph[kTile / 16][4], pl[kTile / 16][4];
#pragma unroll
      for (int jj = 0; jj < kTile / 8; ++jj) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int sI = s0 + jj * 8 + c0 + e;
          const bool in = sI < Lc;
          const float ws = in ? sm.dtp[sI] : 0.0f, as = in ? sm.acum[sI] : 0.0f;
          v[e] = (in && sI <= tA && tA < Lc) ? cb[jj][e] * expf(aA - as) * ws : 0.0f;
          v[2 + e] = (in && sI <= tB && tB < Lc) ? cb[jj][2 + e] * expf(aB - as) * ws : 0.0f;
        }
        const int kb = jj >> 1, half = jj & 1;
        split_pair<IT>(v[0], v[1], &ph[kb][half * 2], &pl[kb][half * 2]);
        split_pair<IT>(v[2], v[3], &ph[kb][half * 2 + 1], &pl[kb][half * 2 + 1]);
      }
#pragma unroll
      for (int kb = 0; kb < kTile / 16; ++kb) {
#pragma unroll
        for (int np = 0; np < PT / 2; ++np) {
          uint32_t bf[4];  // B = x: rows s, columns p (stored [s][p]: transposed loads)
          ldsm_x4_t(bf, saddr(&sm.Xs[kb * 16 + j8 + (m & 1 ? 8 : 0)][np * 16 + (m >= 2 ? 8 : 0)]));
          mma_16816<IT>(yo[2 * np], ph[kb], bf[0], bf[1]);
          mma_16816<IT>(yo[2 * np + 1], ph[kb], bf[2], bf[3]);
          mma_16816<IT>(yo[2 * np], pl[kb], bf[0], bf[1]);
          mma_16816<IT>(yo[2 * np + 1], pl[kb], bf[2], bf[3]);
        }
      }
    }
    // y = intra + exp(a_t) C_t . h_enter + D x_t, times silu(z_t)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int t = half ? tB : tA;
      if (t >= Lc) continue;
      const float dec = expf(half ? aB : aA);
      const int64_t row = ((t0 + t) * a.H + h) * P;
#pragma unroll
      for (int jj = 0; jj < PT; ++jj) {
        const int p = jj * 8 + c0;
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float y = yo[jj][half * 2 + e] + dec * yi[jj][half * 2 + e];
          const float xv = io_to_float<IT>(xg[row + p + e]);
          if (a.D) y += (a.D_per_dim ? a.D[h * P + p + e] : a.D[h]) * xv;
          if (zg) {
            const float zv = io_to_float<IT>(zg[row + p + e]);
            y *= zv / (1.0f + expf(-zv));
          }
          v[e] = y;
        }
        *reinterpret_cast<uint32_t*>(&og[row + p]) = pack_pair<IT>(v[0], v[1]);
      }
    }
  }
}

template <class IT, int P, int N>
cudaError_t launch(const SSDArgs& a, cudaStream_t stream) {
  ssd_chunk_state_kernel<IT, P, N><<<dim3(a.nchunks, a.H), 128, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  static_assert((P * N) % 512 == 0, "a state-passing CTA covers 512 values of one head");
  ssd_state_passing_kernel<P, N><<<(unsigned)((int64_t)a.H * P * N / 512), 128, 0, stream>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  constexpr int TB = kMaxChunk / kTile;
  ssd_bmm_kernel<IT, N><<<dim3(a.nchunks, a.G, TB * TB), 128, 0, stream>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto scan = ssd_chunk_scan_kernel<IT, P, N>;
  const int smem = (int)sizeof(ScanSmem<IT, P, N>);
  if ((e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  scan<<<dim3(a.nchunks, a.H), 128, smem, stream>>>(a);
  return cudaGetLastError();
}

int64_t workspace_bytes(int64_t nchunks, int64_t H, int64_t G, int64_t P, int64_t N,
                        int64_t CS) {
  auto up = [](int64_t b) { return (b + 255) / 256 * 256; };
  return up(nchunks * H * P * N * 4) + 2 * up(nchunks * H * CS * 4) + up(nchunks * G * CS * CS * 4);
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
  if (p->tokens > 0x7fffffffLL || p->nchunks > 0x7fffffffLL)
    return bad(SSU_ERR_UNSUPPORTED, "tokens and chunks must be below 2^31");
  if (!is_idx(p->meta_dtype))
    return bad(SSU_ERR_INVALID_ARGUMENT, "chunk metadata must be int32 or int64");
  if (!is_float(p->state_dtype)) return bad(SSU_ERR_INVALID_ARGUMENT, "state_dtype must be fp32, bf16 or fp16");
  if (p->initial_states && !is_float(p->initial_dtype))
    return bad(SSU_ERR_INVALID_ARGUMENT, "initial_states must be fp32, bf16 or fp16");
  if (!p->x || !p->dt || !p->A || !p->B || !p->C || !p->out || !p->states ||
      !p->cu_chunk_seqlens || !p->seq_idx || (!p->return_intermediate_states && !p->last_chunk_indices))
    return bad(SSU_ERR_INVALID_ARGUMENT, "x, dt, A, B, C, out, states and the chunk metadata must not be NULL");
  if (!a16(p->x) || !a16(p->B) || !a16(p->C) || !a16(p->out) || (p->z && !a16(p->z)))
    return bad(SSU_ERR_INVALID_ARGUMENT, "x, z, out, B and C must be 16-byte aligned");
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
  a.ws_dt = reinterpret_cast<float*>(ws);
  ws += up(p->nchunks * p->nheads * p->chunk_size * 4);
  a.ws_acum = reinterpret_cast<float*>(ws);
  ws += up(p->nchunks * p->nheads * p->chunk_size * 4);
  a.ws_cb = reinterpret_cast<float*>(ws);
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
