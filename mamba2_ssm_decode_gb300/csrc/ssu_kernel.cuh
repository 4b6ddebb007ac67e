// ssu_kernel.cuh -- sm_103a kernels of the Mamba2 selective state update.
//
// The operation ("vllm.model_executor.layers.mamba.ops.ssu_dispatch":
// selective_state_update; "mate.mamba": ssu_one_token / ssu_packed_varlen):
// for one (sequence, head) the state block h[P][N] is read from its slot,
// advanced through the sequence's rows
//     h[p][n] <- h[p][n] * exp(A dt'_p) + dt'_p x[p] B[n]
//     y[p]     = sum_n h[p][n] C[n] + D x[p]   (times silu(z[p]))
// and written to each row's destination slot.
//
// Design (HBM-bound; about 6 flops per state element per token, far below
// the fp32 ridge, so no tensor cores):
//   * One CTA owns ROWS consecutive rows (headdim positions) of one head of
//     one sequence: grid = sequences x heads x row tiles, the tile index
//     fastest so consecutive CTAs stream one slot's contiguous blocks.
//   * A state row is dstate elements.  LPR lanes share a row and each lane
//     owns CPL 16-byte chunks of it, interleaved (chunk q + c * LPR) so one
//     warp load instruction covers RPW rows x 128 contiguous bytes.  Every
//     thread issues all UNR x CPL 16-byte loads of its rows before it uses
//     any, so each SM keeps tens of KB of state reads in flight.
//   * The per-step vectors (B, C of the group, and per row dA, dt' x, D x,
//     silu(z)) are staged once per CTA in shared memory, in fp32, while the
//     state loads are in flight; up to LMAX steps are staged at a time.
//   * The state stays in fp32 registers for the whole chain of a sequence;
//     y[p] is reduced across the LPR lanes of a row with xor shuffles.
//   * State loads bypass L1 (read once); stores are plain write-back.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace ssu {

// Exact n / d for 0 <= n < 2^31 and 1 <= d < 2^31 by one high multiply, an
// add and a shift (Granlund and Montgomery, "Division by invariant integers
// using multiplication", 1994): with s = ceil(log2 d) and the 33-bit
// multiplier 2^32 + m, m = floor(2^32 (2^s - d) / d) + 1, the quotient is
// (hi32(n m) + n) >> s; n < 2^31 keeps the sum inside 32 bits.  Replaces
// run-time 64-bit divisions (long software sequences) in the work-index
// decomposition.
struct FastDiv {
  uint32_t m, s;
  __host__ void init(uint32_t d) {
    s = 0;
    while ((1ull << s) < d) ++s;
    m = (uint32_t)(((1ull << 32) * ((1ull << s) - d)) / d + 1);
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return (__umulhi(n, m) + n) >> s;
  }
};

// ---------------------------------------------------------------------------
// kernel parameters (normalised on the host from ssu_params)
// ---------------------------------------------------------------------------
struct KParams {
  void* state;
  int64_t slots;
  int H, P, hr;  // heads, headdim, heads per group
  int tiles;     // row tiles per head
  const void* x;
  int64_t x_rs, x_hs;
  const void* z;
  int64_t z_rs, z_hs;
  void* out;
  int64_t o_rs, o_hs;
  int out_f32;
  const float* dt;
  int64_t dt_rs, dt_hs, dt_ds;
  const void* B;
  int64_t B_rs, B_gs;
  const void* C;
  int64_t C_rs, C_gs;
  const float* A;
  int64_t A_s, A_ds;  // head and dim strides (dim stride 0: per head)
  const float* D;
  int64_t D_s, D_ds;
  const float* dt_bias;
  int64_t bias_s, bias_ds;
  int softplus;
  int disable;
  int bc_vec16;  // B and C rows start on 16-byte boundaries (pointer and strides)
  int xz_vec16;  // so do x and z rows, and headdim is a multiple of 8
  int64_t pad;
  FastDiv fd_tiles, fd_H, fd_hr;  // divisions by tiles, H and heads per group
  const unsigned long long* sr_seed;  // stochastic rounding of 16-bit state: the call's seed
  int sr_rounds;                      // Philox rounds (used when sr_seed is set)
};

// (sequence, head, tile) of work index `idx` (< 2^31), tile fastest.
__device__ __forceinline__ void split_index(const KParams& p, uint32_t idx, int64_t* seq, int* h,
                                            int* tile) {
  const uint32_t rest = p.fd_tiles.div(idx);
  *tile = (int)(idx - rest * (uint32_t)p.tiles);
  const uint32_t sq = p.fd_H.div(rest);
  *h = (int)(rest - sq * (uint32_t)p.H);
  *seq = sq;
}

struct TableArgs {
  const void* idx;  // nullptr = no table
  int64_t numel, ss, ts, steps;
};

struct OneTokenArgs {
  const void* sbi;   // nullptr = slot b
  const void* dsbi;  // nullptr = in place
  int idx64;
};

struct VarlenArgs {
  int64_t rows;
  const void* cu;  // nullptr = dense
  int64_t dense_steps;
  const void* na;  // nullptr = position 0
  int meta64;
  TableArgs src, dst;
  int idx64;
};

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
template <class T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int VEC = 4;  // elements per 16-byte chunk
  __device__ static __forceinline__ void unpack2(const uint4& r, float2* f) {
    f[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
    f[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
  }
  __device__ static __forceinline__ uint4 pack2(const float2* f) {
    return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                      __float_as_uint(f[1].y));
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int VEC = 8;
  __device__ static __forceinline__ void unpack2(const uint4& r, float2* f) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)  // element 2i in the low half, 2i+1 in the high half
      f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  }
  __device__ static __forceinline__ uint4 pack2(const float2* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 v = __float22bfloat162_rn(f[i]);  // .x low, .y high, round to nearest even
      w[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Elem<__half> {
  static constexpr int VEC = 8;
  __device__ static __forceinline__ void unpack2(const uint4& r, float2* f) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
  }
  __device__ static __forceinline__ uint4 pack2(const float2* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 v = __float22half2_rn(f[i]);
      w[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <class IT>
__device__ __forceinline__ float io_to_float(IT v);
template <>
__device__ __forceinline__ float io_to_float<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <>
__device__ __forceinline__ float io_to_float<__half>(__half v) {
  return __half2float(v);
}
template <class IT>
__device__ __forceinline__ IT float_to_io(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 float_to_io<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half float_to_io<__half>(float v) {
  return __float2half_rn(v);
}

// ---------------------------------------------------------------------------
// lane layout of one state row
// ---------------------------------------------------------------------------
template <class ST, int N>
struct RowLayout {
  static constexpr int VEC = Elem<ST>::VEC;
  static_assert(N % VEC == 0, "dstate must fill whole 16-byte chunks");
  static constexpr int CHUNKS = N / VEC;                // 16-byte chunks per row
  static constexpr int LPR = CHUNKS >= 8 ? 8 : CHUNKS;  // lanes sharing one row
  static constexpr int CPL = CHUNKS / LPR;              // chunks per lane
  static constexpr int RPW = 32 / LPR;                  // rows per warp instruction
  static constexpr int EPL = CPL * VEC;                 // elements per lane per row
  static_assert(CHUNKS % LPR == 0 && 32 % LPR == 0, "unsupported dstate");
};

// Position of state column k in a staged fp32 row of B or C.  Lane q of a
// row reads its chunk c as VEC/4 float4 groups; group h of that chunk is
// stored at ((c * VEC/4 + h) * LPR + q) * 4, so the 8 lanes of a quarter-warp
// read 128 consecutive bytes (no bank conflicts) for every state dtype.  For
// fp32 state (VEC 4) this is the identity.
template <class ST, int N>
__device__ __forceinline__ int bc_slot(int k) {
  using L = RowLayout<ST, N>;
  constexpr int H4 = L::VEC / 4;
  const int chunk = k / L::VEC;
  const int q = chunk % L::LPR, c = chunk / L::LPR;
  const int h = (k % L::VEC) / 4;
  return ((c * H4 + h) * L::LPR + q) * 4 + (k & 3);
}

// Reduce-scatter of R per-row partial sums over the lanes of a row group:
// at each offset (from LPR/2 down) a lane keeps half of its rows and sends
// the other half to its partner, so after log2(R) exchanges every lane holds
// one row summed over 2, 4, ... lanes; the remaining offsets are a plain
// xor-reduction.  The sum of each row is formed in the same order as a plain
// xor tree (own value + partner's value at each level).  On return the lane
// owns rows [base, base + R_left) with their sums in v[0..R_left), and
// `plain` holds the offsets of the plain levels (lanes with q & plain == 0
// are the rows' unique owners).
template <int R, int OFF>
struct RowScatter {
  __device__ static __forceinline__ void run(float* v, int q, int& base, int& plain) {
    if constexpr (OFF > 0) {
      if constexpr (R > 1) {
        const bool upper = (q & OFF) != 0;
#pragma unroll
        for (int i = 0; i < R / 2; ++i) {
          const float send = upper ? v[i] : v[R / 2 + i];
          const float keep = upper ? v[R / 2 + i] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
        }
        if (upper) base += R / 2;
        RowScatter<R / 2, OFF / 2>::run(v, q, base, plain);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
        plain |= OFF;
        RowScatter<1, OFF / 2>::run(v, q, base, plain);
      }
    }
  }
};

// One step of the recurrence for this thread's UNR state rows (pairs in hs):
//   h <- h dA + (dt' x) B;  y = sum_n h C + D x;  y *= silu(z)
// with the row's B, C, dA, dt' x, D x, silu(z) read from the staged step tt.
// Rows of the tile are jbase + u * RPW (u < UNR); y goes to out row r.  The
// lane's B and C are read one 16-byte chunk at a time (live registers for one
// chunk, not the whole row); every row still sums its pairs in element order.
template <class ST, class IT, int N, int UNR, class StageT>
__device__ __forceinline__ void step_rows(float2 (&hs)[UNR][RowLayout<ST, N>::EPL / 2],
                                          const StageT& stg, int tt, int q, int jbase,
                                          const KParams& p, int h, int p0, int64_t r) {
  using L = RowLayout<ST, N>;
  constexpr int H4 = L::VEC / 4;
  constexpr int C2 = L::VEC / 2;  // element pairs per chunk
  float dA[UNR], dtx[UNR];
  float2 a2[UNR];  // even and odd elements: two partial sums per row
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
    const int j = jbase + u * L::RPW;
    dA[u] = stg.dA[tt][j];
    dtx[u] = stg.dtx[tt][j];
    a2[u] = make_float2(0.0f, 0.0f);
  }
#pragma unroll
  for (int c = 0; c < L::CPL; ++c) {
    float2 bv[C2], cv[C2];
#pragma unroll
    for (int hh = 0; hh < H4; ++hh) {
      const int o = ((c * H4 + hh) * L::LPR + q) * 4;
      const float4 b4 = *reinterpret_cast<const float4*>(&stg.B[tt][o]);
      const float4 c4 = *reinterpret_cast<const float4*>(&stg.C[tt][o]);
      bv[2 * hh] = make_float2(b4.x, b4.y);
      bv[2 * hh + 1] = make_float2(b4.z, b4.w);
      cv[2 * hh] = make_float2(c4.x, c4.y);
      cv[2 * hh + 1] = make_float2(c4.z, c4.w);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const float2 dA2 = make_float2(dA[u], dA[u]);
      const float2 dtx2 = make_float2(dtx[u], dtx[u]);
#pragma unroll
      for (int i = 0; i < C2; ++i) {
        const float2 hv = __ffma2_rn(hs[u][c * C2 + i], dA2, __fmul2_rn(dtx2, bv[i]));
        hs[u][c * C2 + i] = hv;
        a2[u] = __ffma2_rn(hv, cv[i], a2[u]);
      }
    }
  }
  float acc[UNR];
#pragma unroll
  for (int u = 0; u < UNR; ++u) acc[u] = a2[u].x + a2[u].y;
  int base = 0, plain = 0;
  RowScatter<UNR, L::LPR / 2>::run(acc, q, base, plain);
  constexpr int LEFT = UNR > L::LPR ? UNR / L::LPR : 1;  // rows a lane still owns
  if ((q & plain) == 0) {
#pragma unroll
    for (int i = 0; i < LEFT; ++i) {
      const int j = jbase + (base + i) * L::RPW;
      const int prow = p0 + j;
      if (prow < p.P) {
        const float yv = (acc[i] + stg.Dx[tt][j]) * stg.gate[tt][j];
        const int64_t o = r * p.o_rs + (int64_t)h * p.o_hs + prow;
        if (p.out_f32) static_cast<float*>(p.out)[o] = yv;
        else static_cast<IT*>(p.out)[o] = float_to_io<IT>(yv);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ int64_t load_int(const void* p, int64_t i, int is64) {
  return is64 ? static_cast<const int64_t*>(p)[i]
              : static_cast<int64_t>(static_cast<const int32_t*>(p)[i]);
}

// entry (seq, pos) of a slot table; false when the table has no such entry
__device__ __forceinline__ bool table_entry(const TableArgs& t, int64_t seq, int64_t pos,
                                            int is64, int64_t* out) {
  if (pos < 0 || pos >= t.steps) return false;
  const int64_t e = seq * t.ss + pos * t.ts;
  if (e < 0 || e >= t.numel) return false;
  *out = load_int(t.idx, e, is64);
  return true;
}

__device__ __forceinline__ bool slot_ok(int64_t slot, int64_t pad, int64_t slots) {
  return slot != pad && slot >= 0 && slot < slots;
}

__device__ __forceinline__ float softplus_f(float v) {
  // log(1 + e^v) written as max(v, 0) + log1p(e^-|v|): no overflow, no cutoff
  return fmaxf(v, 0.0f) + log1pf(expf(-fabsf(v)));
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));  // L2 only: the state is read once
}

__device__ __forceinline__ void st_state(void* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// ---------------------------------------------------------------------------
// stochastic rounding of 16-bit state
// ---------------------------------------------------------------------------

// Philox4x64 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC'11): per round, words 0 and 2 are multiplied by two fixed
// 64-bit constants; the products' high halves are xored with words 1, 3 and
// the key, low halves become words 1, 3; the key advances by two Weyl
// increments.
__device__ __forceinline__ void philox4x64(uint64_t (&x)[4], uint64_t k0, uint64_t k1,
                                           int rounds) {
  constexpr uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
#pragma unroll 1
  for (int i = 0; i < rounds; ++i) {
    const uint64_t hi0 = __umul64hi(M0, x[0]), lo0 = M0 * x[0];
    const uint64_t hi1 = __umul64hi(M1, x[2]), lo1 = M1 * x[2];
    x[0] = hi1 ^ x[1] ^ k0;
    x[1] = lo1;
    x[2] = hi0 ^ x[3] ^ k1;
    x[3] = lo0;
    k0 += 0x9E3779B97F4A7C15ull;  // golden ratio
    k1 += 0xBB67AE8584CAA73Bull;  // sqrt(3) - 1
  }
}

// The magnitude rounds away from zero when its fraction between the two
// neighbours of the format, to 16 bits, is at least 1 - r / 2^16.  bf16 keeps
// the top 16 bits of an fp32 value: adding r below them and truncating is
// that rule (a carry moves into the exponent, or to infinity); NaN rounds to
// nearest.
__device__ __forceinline__ uint32_t sr_bf16(float v, uint32_t r) {
  const uint32_t u = __float_as_uint(v);
  if ((u & 0x7fffffffu) > 0x7f800000u) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t*>(&b);
  }
  return (u + r) >> 16;
}

// fp16: v = M 2^x exactly (M the fp32 significand); the fp16 spacing at |v| is
// 2^qe, so D = qe - x bits of M lie below it and the stored magnitude is
// floor(M / 2^D + r / 2^16) 2^qe, formed exactly in 64-bit integers.
__device__ __forceinline__ uint32_t sr_f16(float v, uint32_t r) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t mag = u & 0x7fffffffu;
  if (mag >= 0x7f800000u) {  // infinity, NaN
    const __half h = __float2half_rn(v);
    return *reinterpret_cast<const uint16_t*>(&h);
  }
  const int E = (int)(mag >> 23);
  const uint64_t M = E ? ((mag & 0x7fffffu) | 0x800000u) : (mag & 0x7fffffu);
  const int x = E ? E - 150 : -149;
  const int e = E ? E - 127 : -127;
  const int qe = (e > -14 ? e : -14) - 10;
  const int D = qe - x;  // 13 in the normal fp16 range, more below it
  uint64_t t;
  if (D >= 40) t = 0;  // M 2^-D + r 2^-16 < 1
  else if (D >= 16) t = (M + ((uint64_t)r << (D - 16))) >> D;
  else t = ((M << (16 - D)) + r) >> 16;
  const float m = (float)t * __int_as_float((qe + 127) << 23);  // exact: t <= 2^11
  const __half h = __float2half_rn(m);  // exact, or infinity past the largest value
  return *reinterpret_cast<const uint16_t*>(&h) | ((u >> 16) & 0x8000u);
}

// Store 8 (16-bit state) or 4 (fp32) consecutive state values h (pairs) at
// element `off` of the pool: to nearest even, or -- 16-bit state, in the
// kernels instantiated with SR -- stochastically, element e taking the 16
// bits 16 (e mod 4) of word (e / 4) mod 4 of Philox block e / 16 keyed by
// (seed, 0).  The generator lives only in the SR instantiations, so the
// round-to-nearest kernels keep their code size and registers.
template <class ST, bool SR = false>
__device__ __forceinline__ void store_state(ST* state, int64_t off, const float2* h,
                                            const KParams& p) {
  if constexpr (sizeof(ST) == 4 || !SR) {
    st_state(state + off, Elem<ST>::pack2(h));
  } else {
    uint64_t x[4] = {(uint64_t)off >> 4, 0, 0, 0};
    philox4x64(x, __ldg(p.sr_seed), 0, p.sr_rounds);
    const bool upper = ((uint64_t)off >> 3) & 1;  // the chunk is half a block
    const uint64_t w[2] = {upper ? x[2] : x[0], upper ? x[3] : x[1]};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t word = w[i >> 1];
      const uint32_t r0 = (uint32_t)(word >> (32 * (i & 1))) & 0xffffu;
      const uint32_t r1 = (uint32_t)(word >> (32 * (i & 1) + 16)) & 0xffffu;
      uint32_t lo, hi;
      if constexpr (std::is_same<ST, __nv_bfloat16>::value) {
        lo = sr_bf16(h[i].x, r0);
        hi = sr_bf16(h[i].y, r1);
      } else {
        lo = sr_f16(h[i].x, r0);
        hi = sr_f16(h[i].y, r1);
      }
      out[i] = (lo & 0xffffu) | (hi << 16);
    }
    st_state(state + off, make_uint4(out[0], out[1], out[2], out[3]));
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <class ST, class IT, int N, int WARPS, int UNR, int LMAX>
struct SSUConfig {
  using L = RowLayout<ST, N>;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int ROWS = WARPS * L::RPW * UNR;  // headdim rows per CTA
};

// Shared-memory staging of up to LMAX steps for one CTA (read with 16-byte
// vector loads, hence the alignment).
template <int N, int ROWS, int LMAX>
struct __align__(16) Stage {
  float B[LMAX][N];
  float C[LMAX][N];
  float dA[LMAX][ROWS];
  float dtx[LMAX][ROWS];  // dt' * x
  float Dx[LMAX][ROWS];   // D * x
  float gate[LMAX][ROWS]; // silu(z), or 1
};

// Stage steps [t0, t0 + n) of rows [r0 + t0, ...) for head h / group g.
template <class ST, class IT, int N, int ROWS, int LMAX, int THREADS>
__device__ __forceinline__ void stage_steps(Stage<N, ROWS, LMAX>& s, const KParams& p,
                                            int64_t r0, int t0, int n, int h, int g, int p0) {
  const IT* Bp = static_cast<const IT*>(p.B);
  const IT* Cp = static_cast<const IT*>(p.C);
  // B and C rows of the group
  for (int i = threadIdx.x; i < n * N; i += THREADS) {
    const int tt = i / N, k = i - tt * N;
    const int64_t r = r0 + t0 + tt;
    s.B[tt][bc_slot<ST, N>(k)] = io_to_float<IT>(Bp[r * p.B_rs + (int64_t)g * p.B_gs + k]);
    s.C[tt][bc_slot<ST, N>(k)] = io_to_float<IT>(Cp[r * p.C_rs + (int64_t)g * p.C_gs + k]);
  }
  // per-row scalars
  const IT* xp = static_cast<const IT*>(p.x);
  const IT* zp = static_cast<const IT*>(p.z);
  for (int i = threadIdx.x; i < n * ROWS; i += THREADS) {
    const int tt = i / ROWS, j = i - tt * ROWS;
    const int prow = p0 + j;
    float dA = 1.0f, dtx = 0.0f, Dx = 0.0f, gate = 1.0f;
    if (prow < p.P) {
      const int64_t r = r0 + t0 + tt;
      const float A = p.A[(int64_t)h * p.A_s + (int64_t)prow * p.A_ds];
      const float Dh = p.D ? p.D[(int64_t)h * p.D_s + (int64_t)prow * p.D_ds] : 0.0f;
      const float bias =
          p.dt_bias ? p.dt_bias[(int64_t)h * p.bias_s + (int64_t)prow * p.bias_ds] : 0.0f;
      const float xv = io_to_float<IT>(xp[r * p.x_rs + (int64_t)h * p.x_hs + prow]);
      float dtv = p.dt[r * p.dt_rs + (int64_t)h * p.dt_hs + (int64_t)prow * p.dt_ds] + bias;
      if (p.softplus) dtv = softplus_f(dtv);
      dA = expf(A * dtv);
      dtx = dtv * xv;
      Dx = Dh * xv;
      if (zp) {
        const float zv = io_to_float<IT>(zp[r * p.z_rs + (int64_t)h * p.z_hs + prow]);
        gate = zv / (1.0f + expf(-zv));
      }
    }
    s.dA[tt][j] = dA;
    s.dtx[tt][j] = dtx;
    s.Dx[tt][j] = Dx;
    s.gate[tt][j] = gate;
  }
}

// One CTA: rows [p0, p0 + ROWS) of head h, sequence rows [r0, r0 + len),
// state read from `src` (if read_ok), step t written to dst_of(t).
// (with the stage in caller-provided shared memory)
template <class ST, class IT, int N, int WARPS, int UNR, int LMAX, bool SR, class DstFn,
          class StageT>
__device__ __forceinline__ void ssu_block_on(StageT& stg, const KParams& p, int h, int p0,
                                             int64_t r0, int len, int64_t src, bool read_ok,
                                             DstFn dst_of) {
  using Cfg = SSUConfig<ST, IT, N, WARPS, UNR, LMAX>;
  using L = typename Cfg::L;
  constexpr int ROWS = Cfg::ROWS;
  constexpr int THREADS = Cfg::THREADS;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int q = lane % L::LPR;   // chunk lane within the row
  const int rr = lane / L::LPR;  // row within the warp instruction
  const int g = (int)p.fd_hr.div((uint32_t)h);
  const int64_t block_elems = (int64_t)p.P * N;
  ST* state = static_cast<ST*>(p.state);

  // 1. issue every state load of this thread's rows
  uint4 raw[UNR][L::CPL];
  {
    const ST* base = state + (((read_ok ? src : 0) * p.H + h) * block_elems);
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int prow = p0 + (warp * UNR + u) * L::RPW + rr;
      const bool ok = read_ok && prow < p.P;
#pragma unroll
      for (int c = 0; c < L::CPL; ++c) {
        raw[u][c] = ok ? ld_stream(base + (int64_t)prow * N + (q + c * L::LPR) * L::VEC)
                       : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }

  // 2. stage the first steps while the loads are in flight
  int n0 = len < LMAX ? len : LMAX;
  stage_steps<ST, IT, N, ROWS, LMAX, THREADS>(stg, p, r0, 0, n0, h, g, p0);
  __syncthreads();

  // 3. widen the state to fp32 registers
  float2 hs[UNR][L::EPL / 2];
#pragma unroll
  for (int u = 0; u < UNR; ++u)
#pragma unroll
    for (int c = 0; c < L::CPL; ++c) Elem<ST>::unpack2(raw[u][c], &hs[u][c * L::VEC / 2]);
  const int jbase = warp * UNR * L::RPW + rr;

  for (int t0 = 0; t0 < len; t0 += LMAX) {
    const int n = (len - t0) < LMAX ? (len - t0) : LMAX;
    if (t0 > 0) {
      __syncthreads();  // everyone is done with the previous stage
      stage_steps<ST, IT, N, ROWS, LMAX, THREADS>(stg, p, r0, t0, n, h, g, p0);
      __syncthreads();
    }
    // this chunk's write slots, loaded together ahead of the stores
    int64_t dsts[LMAX];
    bool dok[LMAX];
#pragma unroll
    for (int i = 0; i < LMAX; ++i) {
      int64_t v = -1;
      dok[i] = i < n && read_ok && !p.disable && dst_of(t0 + i, &v) && slot_ok(v, p.pad, p.slots);
      dsts[i] = v;
    }
#pragma unroll
    for (int tt = 0; tt < LMAX; ++tt) {
      if (tt >= n) break;
      step_rows<ST, IT, N, UNR>(hs, stg, tt, q, jbase, p, h, p0, r0 + t0 + tt);
      // write this step's state
      if (dok[tt]) {
        ST* base = state + ((dsts[tt] * p.H + h) * block_elems);
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int prow = p0 + (warp * UNR + u) * L::RPW + rr;
          if (prow < p.P) {
#pragma unroll
            for (int c = 0; c < L::CPL; ++c)
              store_state<ST, SR>(state, base - state + (int64_t)prow * N + (q + c * L::LPR) * L::VEC,
                              &hs[u][c * L::VEC / 2], p);
          }
        }
      }
    }
  }
}

// Slots and rows of packed sequence s; false for an empty sequence.
__device__ __forceinline__ bool varlen_item(const KParams& p, const VarlenArgs& a, int64_t s,
                                            int64_t* r0, int* len, int64_t* src, bool* read_ok) {
  int64_t begin, end;
  if (a.cu) {
    begin = load_int(a.cu, s, a.meta64);
    end = load_int(a.cu, s + 1, a.meta64);
  } else {
    begin = s * a.dense_steps;
    end = begin + a.dense_steps;
  }
  if (begin < 0) begin = 0;
  if (end > a.rows) end = a.rows;
  if (end <= begin) return false;
  *r0 = begin;
  *len = (int)(end - begin);
  *src = s;
  bool ok = true;
  if (a.src.idx) {
    const int64_t col = a.na ? load_int(a.na, s, a.meta64) - 1 : 0;
    ok = table_entry(a.src, s, col, a.idx64, src);
  }
  *read_ok = ok && slot_ok(*src, p.pad, p.slots);
  return true;
}

}  // namespace ssu
