// ssu_headrun.cuh -- head-run kernels: one CTA takes a run of heads of one
// group for one sequence (and one row tile), so the slot lookup, the B / C
// staging and the per-head dt' / dA are done once for the run, and the state
// tiles of the next heads (contiguous in the slot) land in shared memory --
// one bulk asynchronous copy per tile, or 16-byte cp.async where the no-write
// kernel's tensor-core dot products want a swizzled tile -- while the current
// head computes.  Two kernels: calls that write
// state (ssu_run_kernel, the step-by-step update of step_rows per head), and
// calls that write no state (ssu_nowrite_kernel).
//
// Calls that write no state: the steps of a staged chunk have a closed form.
// Unrolling h_t = dA_t h_{t-1} + dtx_t B_t from the chunk's initial state h:
//   C_t . h_t = P_t (C_t . h) + sum_{s <= t} E_{s,t} (C_t . B_s),
//   P_t = dA_0 dA_1 ... dA_t,   E_{s,t} = dtx_s dA_{s+1} ... dA_t.
// A state element then costs one FMA per step (the dot products C_t . h)
// instead of three, the products G[t][s] = C_t . B_s are formed once per
// CTA, and the state never has to sit in registers.
//
// With 16-bit state and B / C of the same type, the dot products C_t . h of
// a tile are one small contraction, [rows x dstate] x [dstate x steps], whose
// products are exact in 16-bit x 16-bit -> fp32 tensor-core MMA: each warp
// takes 16 rows with m16n8k16 MMAs (steps padded to 8), the state fragments
// read by ldmatrix from an XOR-swizzled tile, C_t's fragments built once per
// CTA.  Elsewhere paired fp32 FMAs and a reduce-scatter over each row's lanes.
#pragma once

#include <type_traits>

#include "ssu_kernel.cuh"

namespace ssu {

__device__ __forceinline__ void ldsm_x4(uint32_t (&a)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}

// d += a b for one m16n8k16 tile (row-major A, column-major B, fp32 accumulate)
template <class T>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// two values exactly representable in T, packed low / high
template <class T>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi) {
  uint32_t w;
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    w = *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    w = *reinterpret_cast<uint32_t*>(&v);
  }
  return w;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// wait until at most `pending` of this thread's newest copy groups are in flight
template <int pending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(pending) : "memory");
}

// Lane q's values of its chunk c of a staged row (B / C layout of bc_slot), as pairs.
template <class ST, int N>
__device__ __forceinline__ void lane_chunk(const float* row, int q, int c, float2* v) {
  using L = RowLayout<ST, N>;
  constexpr int H4 = L::VEC / 4;
#pragma unroll
  for (int h = 0; h < H4; ++h) {
    const float4 f = *reinterpret_cast<const float4*>(&row[((c * H4 + h) * L::LPR + q) * 4]);
    v[2 * h] = make_float2(f.x, f.y);
    v[2 * h + 1] = make_float2(f.z, f.w);
  }
}

template <int N, int LMAX>
struct __align__(16) StepsBC {
  float B[LMAX][N];
  float C[LMAX][N];
};

template <int ROWS, int LMAX>
struct __align__(16) HeadRows {
  float dA[LMAX][ROWS];
  float dtx[LMAX][ROWS];   // dt' * x
  float Dx[LMAX][ROWS];    // D * x
  float gate[LMAX][ROWS];  // silu(z), or 1
};

// B and C rows of group g for steps [t0, t0 + n), in the bc_slot layout:
// 16-byte loads of 8 elements where the rows allow them (bc_slot keeps
// every aligned run of 4 columns contiguous), element loads otherwise.
template <class ST, class IT, int N, int LMAX, int THREADS, class BC>
__device__ __forceinline__ void stage_bc(BC& s, const KParams& p, int64_t r0, int t0, int n,
                                         int g) {
  const IT* Bp = static_cast<const IT*>(p.B);
  const IT* Cp = static_cast<const IT*>(p.C);
  if (p.bc_vec16) {
    constexpr int V8 = N / 8;  // 16-byte pieces per row
    for (int i = threadIdx.x; i < 2 * n * V8; i += THREADS) {
      const bool isC = i >= n * V8;
      const int ii = isC ? i - n * V8 : i;
      const int tt = ii / V8, k0 = (ii - tt * V8) * 8;
      const int64_t r = r0 + t0 + tt;
      const IT* src = isC ? Cp + r * p.C_rs + (int64_t)g * p.C_gs + k0
                          : Bp + r * p.B_rs + (int64_t)g * p.B_gs + k0;
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
      const IT* e = reinterpret_cast<const IT*>(&w);
      float* row = isC ? s.C[tt] : s.B[tt];
      *reinterpret_cast<float4*>(&row[bc_slot<ST, N>(k0)]) =
          make_float4(io_to_float<IT>(e[0]), io_to_float<IT>(e[1]), io_to_float<IT>(e[2]),
                      io_to_float<IT>(e[3]));
      *reinterpret_cast<float4*>(&row[bc_slot<ST, N>(k0 + 4)]) =
          make_float4(io_to_float<IT>(e[4]), io_to_float<IT>(e[5]), io_to_float<IT>(e[6]),
                      io_to_float<IT>(e[7]));
    }
    return;
  }
  for (int i = threadIdx.x; i < n * N; i += THREADS) {
    const int tt = i / N, k = i - tt * N;
    const int64_t r = r0 + t0 + tt;
    s.B[tt][bc_slot<ST, N>(k)] = io_to_float<IT>(Bp[r * p.B_rs + (int64_t)g * p.B_gs + k]);
    s.C[tt][bc_slot<ST, N>(k)] = io_to_float<IT>(Cp[r * p.C_rs + (int64_t)g * p.C_gs + k]);
  }
}

// dt' = softplus(dt + dt_bias) and dA = exp(A dt') of heads h0 .. h0 + kh - 1
// for steps [0, n), when dt, A and dt_bias are per head (ignored otherwise).
template <int KMAX, int LMAX>
struct HeadSteps {
  float dt[KMAX][LMAX];
  float dA[KMAX][LMAX];
};

// dt, A and dt_bias all per head: dt' and dA do not depend on the row
__device__ __forceinline__ bool per_head_dt(const KParams& p) {
  return p.dt_ds == 0 && p.A_ds == 0 && (!p.dt_bias || p.bias_ds == 0);
}

template <int KMAX, int LMAX>
__device__ __forceinline__ void stage_head_steps(HeadSteps<KMAX, LMAX>& s, const KParams& p,
                                                 int64_t r0, int n, int h0, int kh) {
  const int i = threadIdx.x;
  if (i >= kh * LMAX) return;
  const int k = i / LMAX, t = i % LMAX;
  if (t >= n) return;
  const int h = h0 + k;
  float d = p.dt[(r0 + t) * p.dt_rs + (int64_t)h * p.dt_hs] +
            (p.dt_bias ? p.dt_bias[(int64_t)h * p.bias_s] : 0.0f);
  if (p.softplus) d = softplus_f(d);
  s.dt[k][t] = d;
  s.dA[k][t] = expf(p.A[(int64_t)h * p.A_s] * d);
}

// The per-row scalars of one head in two halves, so that the loads of the
// next head are in flight while the current head computes: load() issues
// this thread's global loads into registers, finish() evaluates and stores
// them.  Vector form (dt, A, D, dt_bias per head, x / z rows 16-byte
// aligned): task i < LMAX ROWS / 8 takes step i / (ROWS / 8) of 8 rows, with
// one 16-byte load of x and one of z.  Otherwise, with T = THREADS / LMAX,
// thread i keeps step i / T of rows i % T + m T, element by element.
template <class IT, int ROWS, int LMAX, int THREADS>
struct RowPrefetch {
  static_assert(THREADS % LMAX == 0 && ROWS % 8 == 0, "row layout");
  static constexpr int NP = (ROWS * LMAX + THREADS - 1) / THREADS;  // rows per thread
  static constexpr int VT = LMAX * (ROWS / 8);                       // vector tasks
  static constexpr int WN = 6 * NP > 9 ? 6 * NP : 9;
  uint32_t w[WN];  // vector: x (8), z (8), D; elementwise: x, z, D, dt, A, dt_bias per row
  int64_t xo[NP], zo[NP];
  int prow[NP];
  int t;
  int64_t r;  // packed row of step t
  bool vec;

  __device__ __forceinline__ void init(const KParams& p, int64_t r0, int n, int p0, bool v) {
    vec = v;
    if (vec) {
      const int i = threadIdx.x;
      t = i / (ROWS / 8);
      const int j = (i - t * (ROWS / 8)) * 8;
      r = r0 + t;
      prow[0] = (i < VT && t < n && p0 + j < p.P) ? p0 + j : -1;
      xo[0] = r * p.x_rs + prow[0];
      zo[0] = r * p.z_rs + prow[0];
      return;
    }
    t = threadIdx.x / (THREADS / LMAX);
    r = r0 + t;
#pragma unroll
    for (int m = 0; m < NP; ++m) {
      const int j = threadIdx.x - t * (THREADS / LMAX) + m * (THREADS / LMAX);
      prow[m] = (t < n && j < ROWS && p0 + j < p.P) ? p0 + j : -1;
      xo[m] = r * p.x_rs + prow[m];
      zo[m] = r * p.z_rs + prow[m];
    }
  }

  __device__ __forceinline__ void load(const KParams& p, int h, bool tied) {
    const IT* xp = static_cast<const IT*>(p.x);
    const IT* zp = static_cast<const IT*>(p.z);
    if (vec) {
      if (prow[0] >= 0) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xp + xo[0] + (int64_t)h * p.x_hs));
        w[0] = xv.x, w[1] = xv.y, w[2] = xv.z, w[3] = xv.w;
        if (zp) {
          const uint4 zv =
              __ldg(reinterpret_cast<const uint4*>(zp + zo[0] + (int64_t)h * p.z_hs));
          w[4] = zv.x, w[5] = zv.y, w[6] = zv.z, w[7] = zv.w;
        }
        w[8] = __float_as_uint(p.D ? p.D[(int64_t)h * p.D_s] : 0.0f);
      }
      return;
    }
#pragma unroll
    for (int m = 0; m < NP; ++m) {
      float x = 0.0f, z = 0.0f, D = 0.0f, dt = 0.0f, A = 0.0f, bias = 0.0f;
      if (prow[m] >= 0) {
        x = io_to_float<IT>(xp[xo[m] + (int64_t)h * p.x_hs]);
        if (zp) z = io_to_float<IT>(zp[zo[m] + (int64_t)h * p.z_hs]);
        if (p.D) D = p.D[(int64_t)h * p.D_s + (int64_t)prow[m] * p.D_ds];
        if (!tied) {
          dt = p.dt[r * p.dt_rs + (int64_t)h * p.dt_hs + (int64_t)prow[m] * p.dt_ds];
          A = p.A[(int64_t)h * p.A_s + (int64_t)prow[m] * p.A_ds];
          if (p.dt_bias)
            bias = p.dt_bias[(int64_t)h * p.bias_s + (int64_t)prow[m] * p.bias_ds];
        }
      }
      w[6 * m + 0] = __float_as_uint(x);
      w[6 * m + 1] = __float_as_uint(z);
      w[6 * m + 2] = __float_as_uint(D);
      w[6 * m + 3] = __float_as_uint(dt);
      w[6 * m + 4] = __float_as_uint(A);
      w[6 * m + 5] = __float_as_uint(bias);
    }
  }

  // silu(z): the fast exp / division intrinsics (FAST) or the exact forms the
  // state-writing kernels share bit for bit
  template <bool FAST>
  __device__ __forceinline__ static float silu(float z) {
    if constexpr (FAST) return __fdividef(z, 1.0f + __expf(-z));
    else return z / (1.0f + expf(-z));
  }

  // hdt / hdA: this head's per-head dt' and dA by step (used when tied)
  template <bool FAST, class HR>
  __device__ __forceinline__ void finish(HR& s, const KParams& p, int n, int p0, bool tied,
                                         const float* hdt, const float* hdA) const {
    if (vec) {
      if (prow[0] < 0) return;
      const int j0 = prow[0] - p0;
      const float dtv = hdt[t], dA = hdA[t], D = __uint_as_float(w[8]);
      const IT* xe = reinterpret_cast<const IT*>(&w[0]);
      const IT* ze = reinterpret_cast<const IT*>(&w[4]);
      float dtx[8], Dx[8], gate[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xv = io_to_float<IT>(xe[e]);
        dtx[e] = dtv * xv;
        Dx[e] = D * xv;
        gate[e] = 1.0f;
        if (p.z) gate[e] = silu<FAST>(io_to_float<IT>(ze[e]));
      }
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        const int o = j0 + 4 * hq;
        *reinterpret_cast<float4*>(&s.dA[t][o]) = make_float4(dA, dA, dA, dA);
        *reinterpret_cast<float4*>(&s.dtx[t][o]) =
            make_float4(dtx[4 * hq], dtx[4 * hq + 1], dtx[4 * hq + 2], dtx[4 * hq + 3]);
        *reinterpret_cast<float4*>(&s.Dx[t][o]) =
            make_float4(Dx[4 * hq], Dx[4 * hq + 1], Dx[4 * hq + 2], Dx[4 * hq + 3]);
        *reinterpret_cast<float4*>(&s.gate[t][o]) =
            make_float4(gate[4 * hq], gate[4 * hq + 1], gate[4 * hq + 2], gate[4 * hq + 3]);
      }
      return;
    }
    if (t >= n) return;
#pragma unroll
    for (int m = 0; m < NP; ++m) {
      const int j = threadIdx.x - t * (THREADS / LMAX) + m * (THREADS / LMAX);
      if (j >= ROWS) break;
      float dAv = 1.0f, dtx = 0.0f, Dx = 0.0f, gate = 1.0f;
      if (prow[m] >= 0) {
        const float x = __uint_as_float(w[6 * m + 0]), z = __uint_as_float(w[6 * m + 1]);
        float dtv;
        if (tied) {
          dtv = hdt[t];
          dAv = hdA[t];
        } else {
          dtv = __uint_as_float(w[6 * m + 3]) + __uint_as_float(w[6 * m + 5]);
          if (p.softplus) dtv = softplus_f(dtv);
          dAv = expf(__uint_as_float(w[6 * m + 4]) * dtv);
        }
        dtx = dtv * x;
        Dx = __uint_as_float(w[6 * m + 2]) * x;
        if (p.z) gate = silu<FAST>(z);
      }
      s.dA[t][j] = dAv;
      s.dtx[t][j] = dtx;
      s.Dx[t][j] = Dx;
      s.gate[t][j] = gate;
    }
  }
};

// G[t][s] = C_t . B_s for s <= t < n; pair k goes to warp k % WARPS.
template <int N, int LMAX, int WARPS, class BC>
__device__ __forceinline__ void stage_G(const BC& bc, float (&G)[LMAX][LMAX], int n, int warp,
                                        int lane) {
  int k = 0;
#pragma unroll
  for (int t = 0; t < LMAX; ++t) {
#pragma unroll
    for (int s = 0; s <= t; ++s, ++k) {
      if (t < n && (k % WARPS) == warp) {
        float v = 0.0f;
        for (int i = lane; i < N; i += 32) v = fmaf(bc.C[t][i], bc.B[s][i], v);
        v = warp_sum(v);
        if (lane == 0) G[t][s] = v;
      }
    }
  }
}

// y of steps t < n (rows r + t) for row j of the tile, from ct[t] = C_t . h.
template <class IT, int LMAX, class HR>
__device__ __forceinline__ void closed_form_y(const KParams& p, const HR& hr,
                                              const float (&G)[LMAX][LMAX], const float* ct,
                                              int n, int j, int h, int prow, int64_t r) {
  float e[LMAX];
  float P = 1.0f;
#pragma unroll
  for (int t = 0; t < LMAX; ++t) {
    if (t >= n) break;
    const float dA = hr.dA[t][j];
    P *= dA;
#pragma unroll
    for (int s = 0; s < t; ++s) e[s] *= dA;
    e[t] = hr.dtx[t][j];
    float v = P * ct[t];
#pragma unroll
    for (int s = 0; s <= t; ++s) v = fmaf(e[s], G[t][s], v);
    const float yv = (v + hr.Dx[t][j]) * hr.gate[t][j];
    const int64_t o = (r + t) * p.o_rs + (int64_t)h * p.o_hs + prow;
    if (p.out_f32) static_cast<float*>(p.out)[o] = yv;
    else static_cast<IT*>(p.out)[o] = float_to_io<IT>(yv);
  }
}

// y of step t (row r + t) for row j, from ct = C_t . h: the sum over s runs
// from t down, so one running product gives E_{s,t} and, at the end, P_t.
template <class IT, int LMAX, class HR>
__device__ __forceinline__ void closed_form_y_step(const KParams& p, const HR& hr,
                                                   const float (&G)[LMAX][LMAX], float ct, int t,
                                                   int j, int h, int prow, int64_t r) {
  float v = 0.0f, prod = 1.0f;
#pragma unroll
  for (int s = LMAX - 1; s >= 0; --s) {
    if (s > t) continue;
    v = fmaf(prod * hr.dtx[s][j], G[t][s], v);
    prod *= hr.dA[s][j];
  }
  const float yv = (fmaf(prod, ct, v) + hr.Dx[t][j]) * hr.gate[t][j];
  const int64_t o = (r + t) * p.o_rs + (int64_t)h * p.o_hs + prow;
  if (p.out_f32) static_cast<float*>(p.out)[o] = yv;
  else static_cast<IT*>(p.out)[o] = float_to_io<IT>(yv);
}

// Register form for chains longer than one staged chunk: the earlier chunks
// run the step-by-step update (the next chunk needs their state), the last
// one the closed form.
template <class ST, class IT, int N, int WARPS, int UNR, int LMAX, class StageT>
__device__ __noinline__ void ssu_block_nowrite_chain(const KParams& p, int h, int p0, int64_t r0,
                                                     int len, int64_t src, bool read_ok,
                                                     StageT& stg, float (&G)[LMAX][LMAX]) {
  using Cfg = SSUConfig<ST, IT, N, WARPS, UNR, LMAX>;
  using L = typename Cfg::L;
  constexpr int ROWS = Cfg::ROWS;
  constexpr int THREADS = Cfg::THREADS;
  constexpr int C2 = L::VEC / 2;                          // element pairs per chunk
  constexpr int LEFT = UNR > L::LPR ? UNR / L::LPR : 1;  // rows a lane owns after the reduce

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int q = lane % L::LPR;
  const int rr = lane / L::LPR;
  const int g = (int)p.fd_hr.div((uint32_t)h);
  const int64_t block_elems = (int64_t)p.P * N;
  const ST* state = static_cast<const ST*>(p.state);

  float2 hs[UNR][L::EPL / 2];
  {
    const ST* base = state + (((read_ok ? src : 0) * p.H + h) * block_elems);
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int prow = p0 + (warp * UNR + u) * L::RPW + rr;
      const bool ok = read_ok && prow < p.P;
#pragma unroll
      for (int c = 0; c < L::CPL; ++c) {
        const uint4 raw = ok ? ld_stream(base + (int64_t)prow * N + (q + c * L::LPR) * L::VEC)
                             : make_uint4(0u, 0u, 0u, 0u);
        Elem<ST>::unpack2(raw, &hs[u][c * L::VEC / 2]);
      }
    }
  }
  const int jbase = warp * UNR * L::RPW + rr;
  for (int t0 = 0; t0 < len; t0 += LMAX) {
    const int n = (len - t0) < LMAX ? (len - t0) : LMAX;
    __syncthreads();  // the stage is free
    stage_steps<ST, IT, N, ROWS, LMAX, THREADS>(stg, p, r0, t0, n, h, g, p0);
    __syncthreads();
    if (t0 + n < len) {
#pragma unroll
      for (int tt = 0; tt < LMAX; ++tt) {
        if (tt >= n) break;
        step_rows<ST, IT, N, UNR>(hs, stg, tt, q, jbase, p, h, p0, r0 + t0 + tt);
      }
      continue;
    }
    stage_G<N, LMAX, WARPS>(stg, G, n, warp, lane);
    float ct[LEFT][LMAX];
    int base = 0, plain = 0;
#pragma unroll
    for (int t = 0; t < LMAX; ++t) {
      if (t >= n) break;
      float2 a2[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u) a2[u] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int c = 0; c < L::CPL; ++c) {
        float2 cv[C2];
        lane_chunk<ST, N>(stg.C[t], q, c, cv);
#pragma unroll
        for (int u = 0; u < UNR; ++u)
#pragma unroll
          for (int i = 0; i < C2; ++i) a2[u] = __ffma2_rn(hs[u][c * C2 + i], cv[i], a2[u]);
      }
      float acc[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u) acc[u] = a2[u].x + a2[u].y;
      base = 0;
      plain = 0;
      RowScatter<UNR, L::LPR / 2>::run(acc, q, base, plain);
#pragma unroll
      for (int i = 0; i < LEFT; ++i) ct[i][t] = acc[i];
    }
    __syncthreads();  // G complete
    if ((q & plain) == 0) {
#pragma unroll
      for (int i = 0; i < LEFT; ++i) {
        const int j = jbase + (base + i) * L::RPW;
        if (p0 + j < p.P) closed_form_y<IT, LMAX>(p, stg, G, ct[i], n, j, h, p0 + j, r0 + t0);
      }
    }
  }
}

// Coordinates of a head-run CTA: grid.x enumerates (run of kh heads, row
// tile) with the tile fastest, grid.y x grid.z the sequences (z-major), so
// consecutive CTAs stay on one slot's contiguous blocks and any batch fits
// one launch.  False for the few CTAs past the last sequence.
__device__ __forceinline__ bool head_run_coords(const KParams& p, int64_t nseqs, int kh,
                                                int rows, int64_t* s, int* h0, int* p0) {
  const uint32_t run = p.fd_tiles.div(blockIdx.x);
  *p0 = (int)(blockIdx.x - run * (uint32_t)p.tiles) * rows;
  *h0 = (int)run * kh;
  *s = (int64_t)blockIdx.z * gridDim.y + blockIdx.y;
  return *s < nseqs;
}

// No-write kernel, one-token and packed routes: grid (row tiles, runs of kh
// heads of one group, sequences), so at most 65535 sequences per call (the
// launcher sends larger batches to the write kernel, which skips its stores
// under disable_state_update).  The flattened head-run grid, with the same
// order of CTAs, measured 0.76 against 0.85 of the HBM roofline here (fp32
// MTP-4, batch 1024).  Sequences longer than LMAX take the register form,
// head by head.
template <class ST, class IT, int N, int WARPS, int UNR, int LMAX, bool VARLEN>
__global__ void __launch_bounds__(WARPS * 32, 5)
    ssu_nowrite_kernel(const KParams p, const OneTokenArgs oa, const VarlenArgs va, int64_t nseqs,
                       int kh, unsigned* err) {
  using Cfg = SSUConfig<ST, IT, N, WARPS, UNR, LMAX>;
  using L = typename Cfg::L;
  constexpr int ROWS = Cfg::ROWS;
  using StageT = Stage<N, ROWS, LMAX>;
  constexpr int THREADS = Cfg::THREADS;
  constexpr int C2 = L::VEC / 2;
  constexpr int LEFT = UNR > L::LPR ? UNR / L::LPR : 1;  // rows a lane owns after a reduce
  constexpr bool JOINT = LMAX * UNR == L::LPR;           // one (step, row) sum per lane
  constexpr int TILE_BYTES = ROWS * N * (int)sizeof(ST);
  // tensor-core dot products: 16-bit state and B / C of one type, 16 rows per
  // warp, rows of 8 or 16 chunks of 16 bytes (swizzled by row % 8)
  constexpr bool MMA = sizeof(ST) == 2 && std::is_same<ST, IT>::value && (N == 64 || N == 128) &&
                       ROWS == 16 * WARPS && LMAX <= 8;
  constexpr int CHR = N * (int)sizeof(ST) / 16;  // 16-byte chunks per tile row
  constexpr int RAW =
      2 * TILE_BYTES > (int)sizeof(StageT) ? 2 * TILE_BYTES : (int)sizeof(StageT);
  __shared__ __align__(128) unsigned char raw[RAW];  // two state tiles, or a chain's stage
  __shared__ StepsBC<N, LMAX> bc;
  __shared__ HeadRows<ROWS, LMAX> hrows[2];
  __shared__ HeadSteps<8, LMAX> hsteps;
  __shared__ float G[LMAX][LMAX];

  const int64_t s = blockIdx.z;
  const int h0 = (int)blockIdx.y * kh;
  const int p0 = (int)blockIdx.x * ROWS;
  int64_t r0, src;
  int len;
  bool read_ok;
  if constexpr (VARLEN) {
    if (!varlen_item(p, va, s, &r0, &len, &src, &read_ok)) return;
  } else {
    r0 = s;
    len = 1;
    src = oa.sbi ? load_int(oa.sbi, s, oa.idx64) : s;
    read_ok = slot_ok(src, p.pad, p.slots);
  }
  if (len > LMAX) {
    StageT& stg = *reinterpret_cast<StageT*>(raw);
    for (int k = 0; k < kh; ++k)
      ssu_block_nowrite_chain<ST, IT, N, WARPS, UNR, LMAX>(p, h0 + k, p0, r0, len, src, read_ok,
                                                           stg, G);
    return;
  }

  // 1. state tiles of the first two heads: with the tensor-core dot products
  //    by 16-byte async copies into the swizzled layout (zero fill past P or
  //    without a read slot), one commit group per head; otherwise each tile
  //    (the head's contiguous rows) by one bulk asynchronous copy on an
  //    mbarrier, and rows past P or without a read slot read as zeros
  const int64_t block_elems = (int64_t)p.P * N;
  const int nrows = p.P - p0 < ROWS ? p.P - p0 : ROWS;
  const int valid = read_ok ? nrows * N * (int)sizeof(ST) / 16 : 0;
  const char* slot_rows = reinterpret_cast<const char*>(
      static_cast<const ST*>(p.state) + (read_ok ? src : 0) * p.H * block_elems +
      (int64_t)p0 * N);
  __shared__ __align__(8) uint64_t tile_bar[2];
  if (!MMA && threadIdx.x == 0) {
    mbar_init(&tile_bar[0], 1);
    mbar_init(&tile_bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  auto issue_tile = [&](int k, int buf) {
    if constexpr (!MMA) {
      if (threadIdx.x == 0 && k < kh && read_ok) {
        const uint32_t bytes = (uint32_t)(nrows * N * (int)sizeof(ST));
        mbar_arrive_expect_tx(&tile_bar[buf], bytes);
        bulk_load(raw + buf * TILE_BYTES, slot_rows + (size_t)(h0 + k) * block_elems * sizeof(ST),
                  bytes, &tile_bar[buf]);
      }
      return;
    }
    if (k < kh) {
      const char* gsrc = slot_rows + (size_t)(h0 + k) * block_elems * sizeof(ST);
      unsigned char* dst = raw + buf * TILE_BYTES;
#pragma unroll 4
      for (int i = threadIdx.x; i < TILE_BYTES / 16; i += THREADS) {
        const bool v = i < valid;
        int o = i * 16;
        if constexpr (MMA) {  // chunk c of row r at chunk c ^ (r % 8): ldmatrix without conflicts
          const int r = i / CHR, c = i - r * CHR;
          o = (r * CHR + (c ^ (r & 7))) * 16;
        }
        cp_async16(dst + o, v ? gsrc + (size_t)i * 16 : static_cast<const char*>(p.state),
                   v ? 16 : 0);
      }
    }
    cp_async_commit();
  };
  issue_tile(0, 0);
  issue_tile(1, 1);

  // 2. the steps' B / C (shared by the run's heads), the first head's rows and G
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool tied = per_head_dt(p);
  RowPrefetch<IT, ROWS, LMAX, THREADS> pre;
  pre.init(p, r0, len, p0, tied && p.xz_vec16 && (!p.D || p.D_ds == 0));
  pre.load(p, h0, tied);
  stage_bc<ST, IT, N, LMAX, THREADS>(bc, p, r0, 0, len, (int)p.fd_hr.div((uint32_t)h0));
  if (tied) stage_head_steps<8, LMAX>(hsteps, p, r0, len, h0, kh);
  __syncthreads();
  pre.finish<true>(hrows[0], p, len, p0, tied, hsteps.dt[0], hsteps.dA[0]);
  if (kh > 1) pre.load(p, h0 + 1, tied);  // a whole head ahead of its use
  stage_G<N, LMAX, WARPS>(bc, G, len, warp, lane);
  // C's MMA fragments (B operand, k x n = dstate x step): lane holds columns
  // k = 16 ks + 8 half + 2 (lane % 4) + {0, 1} of step lane / 4 (zero past len)
  uint32_t bfr[MMA ? N / 16 : 1][2];
  if constexpr (MMA) {
    const int st = lane >> 2, q4 = lane & 3;
#pragma unroll
    for (int ks = 0; ks < N / 16; ++ks)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int kc = 16 * ks + 8 * half + 2 * q4;
        float lo = 0.0f, hi = 0.0f;
        if (st < len) {
          lo = bc.C[st][bc_slot<ST, N>(kc)];
          hi = bc.C[st][bc_slot<ST, N>(kc + 1)];
        }
        bfr[ks][half] = pack_pair<ST>(lo, hi);
      }
  }

  const int q = lane % L::LPR;
  const int rr = lane / L::LPR;
  const int jbase = warp * UNR * L::RPW + rr;
  // a wait that runs out sets the error word; thread 0 then issues no more
  // copies and, before the CTA ends, waits once more (bounded) for the ones
  // still in flight
  bool dead = false;
  int pend = -1;
  for (int k = 0; k < kh; ++k) {
    if constexpr (MMA) {
      cp_async_wait<1>();  // head k's copies (the newest group is head k + 1's)
    } else if (read_ok && !dead && !mbar_wait(&tile_bar[k & 1], (k >> 1) & 1)) {
      dead = true;
      pend = k;
      if (threadIdx.x == 0) atomicOr(err, kErrFullTimeout);
    }
    __syncthreads();  // head k's tile from every copy; hrows[k & 1] and G complete
    const unsigned char* tile = raw + (k & 1) * TILE_BYTES;

    // 3. ct[t] = C_t . h for this thread's rows: one pass over the tile
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // MMA: rows lane / 4 (+ 8), steps 2 (lane % 4) (+ 1)
    if constexpr (MMA) {
      const int arow = warp * 16 + (lane & 15);
      const uint32_t abase =
          static_cast<uint32_t>(__cvta_generic_to_shared(tile)) + arow * (CHR * 16);
#pragma unroll
      for (int ks = 0; ks < N / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, abase + (((2 * ks + (lane >> 4)) ^ (arow & 7)) << 4));
        mma_16816<ST>(d, a, bfr[ks][0], bfr[ks][1]);
      }
    }
    float2 a2[LMAX][UNR];  // even / odd element partial sums
    if constexpr (!JOINT && !MMA) {
#pragma unroll
      for (int t = 0; t < LMAX; ++t)
#pragma unroll
        for (int u = 0; u < UNR; ++u) a2[t][u] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int c = 0; c < (MMA ? 0 : L::CPL); ++c) {
      float2 cv[LMAX][C2];  // chunk c of every step's C, read once for all rows
#pragma unroll
      for (int t = 0; t < LMAX; ++t)
        if (t < len) lane_chunk<ST, N>(bc.C[t], q, c, cv[t]);
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int j = jbase + u * L::RPW;
        float2 hv[C2];
        const uint4 hraw =
            read_ok && j < nrows
                ? *reinterpret_cast<const uint4*>(
                      tile + ((size_t)j * N + (q + c * L::LPR) * L::VEC) * sizeof(ST))
                : make_uint4(0u, 0u, 0u, 0u);
        Elem<ST>::unpack2(hraw, hv);
#pragma unroll
        for (int t = 0; t < LMAX; ++t) {
          if (t >= len) break;
#pragma unroll
          for (int i = 0; i < C2; ++i)
            a2[t][u] = (JOINT && c == 0 && i == 0) ? __fmul2_rn(hv[i], cv[t][i])
                                                   : __ffma2_rn(hv[i], cv[t][i], a2[t][u]);
        }
      }
    }
    // Where the (step, row) sums number exactly the lanes of a row group, one
    // reduce-scatter over all of them (value v = t UNR + u) leaves every lane
    // one y to form; otherwise one reduce-scatter per step over the rows.
    float acc[JOINT ? LMAX * UNR : 1];
    float ct[JOINT ? 1 : LEFT][LMAX];
    int base = 0, plain = 0;
    if constexpr (MMA) {
    } else if constexpr (JOINT) {
#pragma unroll
      for (int t = 0; t < LMAX; ++t)
#pragma unroll
        for (int u = 0; u < UNR; ++u)
          acc[t * UNR + u] = t < len ? a2[t][u].x + a2[t][u].y : 0.0f;
      RowScatter<LMAX * UNR, L::LPR / 2>::run(acc, q, base, plain);
    } else {
#pragma unroll
      for (int t = 0; t < LMAX; ++t) {
        if (t >= len) break;
        float rs[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) rs[u] = a2[t][u].x + a2[t][u].y;
        base = 0;
        plain = 0;
        RowScatter<UNR, L::LPR / 2>::run(rs, q, base, plain);
#pragma unroll
        for (int i = 0; i < LEFT; ++i) ct[i][t] = rs[i];
      }
    }

    // 4. the next head's rows (loaded one iteration ago) and the loads of the
    //    one after; then the tile buffer goes to head k + 2
    if (k + 1 < kh)
      pre.finish<true>(hrows[(k + 1) & 1], p, len, p0, tied, hsteps.dt[k + 1], hsteps.dA[k + 1]);
    if (k + 2 < kh) pre.load(p, h0 + k + 2, tied);
    __syncthreads();  // every thread is done with tile k; hrows[(k + 1) & 1] complete
    if (!dead) issue_tile(k + 2, k & 1);

    // 5. y of head k
    if constexpr (MMA) {
      // lanes with lane % 4 >= 2 hold only padded steps (4..7): they take
      // over row + 8 of lane - 2, so every lane forms two y of one row
      const float u0 = __shfl_up_sync(0xffffffffu, d[2], 2);
      const float u1 = __shfl_up_sync(0xffffffffu, d[3], 2);
      const bool hi = (lane & 2) != 0;
      const int t = 2 * (lane & 1);
      const int j = warp * 16 + (lane >> 2) + (hi ? 8 : 0);
      const float c0 = hi ? u0 : d[0], c1 = hi ? u1 : d[1];
      if (p0 + j < p.P) {
        if (t < len)
          closed_form_y_step<IT, LMAX>(p, hrows[k & 1], G, c0, t, j, h0 + k, p0 + j, r0);
        if (t + 1 < len)
          closed_form_y_step<IT, LMAX>(p, hrows[k & 1], G, c1, t + 1, j, h0 + k, p0 + j, r0);
      }
    } else if constexpr (JOINT) {
      const int t = base / UNR, u = base - t * UNR;
      const int j = jbase + u * L::RPW;
      if (t < len && p0 + j < p.P)
        closed_form_y_step<IT, LMAX>(p, hrows[k & 1], G, acc[0], t, j, h0 + k, p0 + j, r0);
    } else if ((q & plain) == 0) {
#pragma unroll
      for (int i = 0; i < LEFT; ++i) {
        const int j = jbase + (base + i) * L::RPW;
        if (p0 + j < p.P)
          closed_form_y<IT, LMAX>(p, hrows[k & 1], G, ct[i], len, j, h0 + k, p0 + j, r0);
      }
    }
  }
  if constexpr (!MMA) {
    // after a timeout: the copy that did not land and the one issued after it
    if (threadIdx.x == 0 && pend >= 0) {
      mbar_wait(&tile_bar[pend & 1], (pend >> 1) & 1);
      if (pend + 1 < kh) mbar_wait(&tile_bar[(pend + 1) & 1], ((pend + 1) >> 1) & 1);
    }
  }
}

// ---------------------------------------------------------------------------
// the same head runs for packed chains that write state
// ---------------------------------------------------------------------------

// The stage as step_rows reads it, assembled from the run's shared pieces.
template <int N, int ROWS, int LMAX>
struct StageView {
  const float (*B)[N];
  const float (*C)[N];
  const float (*dA)[ROWS];
  const float (*dtx)[ROWS];
  const float (*Dx)[ROWS];
  const float (*gate)[ROWS];
};

// Calls that write state (packed chains, or one token): one CTA per
// (sequence, run of kh heads of one group, row tile), placed by
// head_run_coords.  The slot lookups, the chain's write
// slots, B / C and the per-head dt' / dA table are formed once for the run;
// each head's state tile (its contiguous rows) lands in shared memory by one
// bulk asynchronous copy on an mbarrier, issued one head ahead so it is in
// flight while the previous head computes; each head then
// runs step_rows on the same staged values, with the same stores, as the bulk
// kernels (so the same bits).  Chains longer than LMAX take the per-head block
// (ssu_block_on), head by head.
// 16-bit state: 64-row tiles hold 64 state values per thread, so three CTAs
// per SM (up to 168 registers, no spills) rather than four.
template <class ST, class IT, int N, int WARPS, int UNR, int LMAX, bool VARLEN, bool SR = false>
__global__ void __launch_bounds__(WARPS * 32, sizeof(ST) == 2 ? 3 : 16 / WARPS)
    ssu_run_kernel(const KParams p, const OneTokenArgs oa, const VarlenArgs va, int64_t nseqs,
                   int kh, unsigned* err) {
  using Cfg = SSUConfig<ST, IT, N, WARPS, UNR, LMAX>;
  using L = typename Cfg::L;
  constexpr int ROWS = Cfg::ROWS;
  constexpr int THREADS = Cfg::THREADS;
  using StageT = Stage<N, ROWS, LMAX>;
  constexpr int TILE_BYTES = ROWS * N * (int)sizeof(ST);
  constexpr int RAW =
      2 * TILE_BYTES > (int)sizeof(StageT) ? 2 * TILE_BYTES : (int)sizeof(StageT);
  __shared__ __align__(128) unsigned char raw[RAW];  // two state tiles, or a chain's stage
  __shared__ StepsBC<N, LMAX> bc;
  __shared__ HeadRows<ROWS, LMAX> hrows[2];
  __shared__ HeadSteps<8, LMAX> hsteps;

  int64_t s;
  int h0, p0;
  if (!head_run_coords(p, nseqs, kh, ROWS, &s, &h0, &p0)) return;
  int64_t r0, src;
  int len;
  bool read_ok;
  if constexpr (VARLEN) {
    if (!varlen_item(p, va, s, &r0, &len, &src, &read_ok)) return;
  } else {
    r0 = s;
    len = 1;
    src = oa.sbi ? load_int(oa.sbi, s, oa.idx64) : s;
    read_ok = slot_ok(src, p.pad, p.slots);
  }
  const TableArgs dtab = va.dst.idx ? va.dst : va.src;  // no write table: the read table
  const int idx64 = VARLEN ? va.idx64 : oa.idx64;
  const void* dsbi = oa.dsbi;
  auto dst_of = [dtab, idx64, s, dsbi, src](int t, int64_t* o) -> bool {
    if constexpr (VARLEN) {
      if (dtab.idx) return table_entry(dtab, s, t, idx64, o);
      *o = s;
    } else {
      *o = dsbi ? load_int(dsbi, s, idx64) : src;
    }
    return true;
  };
  if (VARLEN && len > LMAX) {
    StageT& stg = *reinterpret_cast<StageT*>(raw);
    for (int k = 0; k < kh; ++k) {
      ssu_block_on<ST, IT, N, WARPS, UNR, LMAX, SR>(stg, p, h0 + k, p0, r0, len, src, read_ok,
                                                dst_of);
      __syncthreads();  // the stage is free for the next head
    }
    return;
  }

  // the chain's write slots (the same for every head of the run), -1 where a
  // step writes nothing; kept in shared memory, not in registers
  __shared__ int64_t dsts[LMAX];
  if (threadIdx.x < LMAX) {
    const int i = threadIdx.x;
    int64_t v = -1;
    const bool ok = i < len && read_ok && !p.disable && dst_of(i, &v) && slot_ok(v, p.pad, p.slots);
    dsts[i] = ok ? v : -1;
  }

  // 1. the first head's state tile by one bulk asynchronous copy (TMA
  //    engine) on an mbarrier; each head's tile is issued one head ahead
  const int64_t block_elems = (int64_t)p.P * N;
  const int nrows = p.P - p0 < ROWS ? p.P - p0 : ROWS;
  const uint32_t tile_bytes = (uint32_t)(nrows * N * (int)sizeof(ST));
  const char* slot_rows = reinterpret_cast<const char*>(
      static_cast<const ST*>(p.state) + (read_ok ? src : 0) * p.H * block_elems +
      (int64_t)p0 * N);
  __shared__ __align__(8) uint64_t tile_bar[2];
  if (threadIdx.x == 0) {
    mbar_init(&tile_bar[0], 1);
    mbar_init(&tile_bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  auto issue_tile = [&](int k, int buf) {
    if (threadIdx.x == 0 && k < kh && read_ok) {
      mbar_arrive_expect_tx(&tile_bar[buf], tile_bytes);
      bulk_load(raw + buf * TILE_BYTES, slot_rows + (size_t)(h0 + k) * block_elems * sizeof(ST),
                tile_bytes, &tile_bar[buf]);
    }
  };
  issue_tile(0, 0);

  // 2. B / C, the per-head dt' / dA table and the first head's rows
  const bool tied = per_head_dt(p);
  RowPrefetch<IT, ROWS, LMAX, THREADS> pre;
  pre.init(p, r0, len, p0, tied && p.xz_vec16 && (!p.D || p.D_ds == 0));
  pre.load(p, h0, tied);
  stage_bc<ST, IT, N, LMAX, THREADS>(bc, p, r0, 0, len, (int)p.fd_hr.div((uint32_t)h0));
  if (tied) stage_head_steps<8, LMAX>(hsteps, p, r0, len, h0, kh);
  __syncthreads();
  pre.finish<false>(hrows[0], p, len, p0, tied, hsteps.dt[0], hsteps.dA[0]);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int q = lane % L::LPR;
  const int rr = lane / L::LPR;
  const int jbase = warp * UNR * L::RPW + rr;
  ST* state = static_cast<ST*>(p.state);
  // a wait that runs out sets the error word; thread 0 then issues no more
  // copies and, before the CTA ends, waits once more (bounded) for the one
  // that did not land
  bool dead = false;
  int pend = -1;
  for (int k = 0; k < kh; ++k) {
    if (read_ok && !dead && !mbar_wait(&tile_bar[k & 1], (k >> 1) & 1)) {  // head k's tile
      dead = true;
      pend = k;
      if (threadIdx.x == 0) atomicOr(err, kErrFullTimeout);
    }
    __syncthreads();  // hrows[k & 1] complete; buffer (k + 1) & 1 was read (head k - 1)
    if (!dead) issue_tile(k + 1, (k + 1) & 1);  // in flight during head k's steps
    const int h = h0 + k;
    // 3. this thread's state chunks of head k, widened to fp32
    float2 hs[UNR][L::EPL / 2];
    {
      const unsigned char* tile = raw + (k & 1) * TILE_BYTES;
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int j = jbase + u * L::RPW;
#pragma unroll
        for (int c = 0; c < L::CPL; ++c) {
          const uint4 v = read_ok && j < nrows
                              ? *reinterpret_cast<const uint4*>(
                                    tile + ((size_t)j * N + (q + c * L::LPR) * L::VEC) * sizeof(ST))
                              : make_uint4(0u, 0u, 0u, 0u);
          Elem<ST>::unpack2(v, &hs[u][c * L::VEC / 2]);
        }
      }
    }
    // 4. the next head's rows (into the other buffer)
    if (k + 1 < kh) {
      pre.load(p, h + 1, tied);
      pre.finish<false>(hrows[(k + 1) & 1], p, len, p0, tied, hsteps.dt[k + 1],
                        hsteps.dA[k + 1]);
    }
    // 5. the steps of head k, each step's state to its write slot
    const StageView<N, ROWS, LMAX> view{bc.B, bc.C, hrows[k & 1].dA, hrows[k & 1].dtx,
                                        hrows[k & 1].Dx, hrows[k & 1].gate};
#pragma unroll
    for (int tt = 0; tt < LMAX; ++tt) {
      if (tt >= len) break;
      step_rows<ST, IT, N, UNR>(hs, view, tt, q, jbase, p, h, p0, r0 + tt);
      const int64_t dst = dsts[tt];
      if (dst >= 0) {
        ST* base = state + ((dst * p.H + h) * block_elems);
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
  if (threadIdx.x == 0 && pend >= 0) mbar_wait(&tile_bar[pend & 1], (pend >> 1) & 1);
}

}  // namespace ssu
