// ssu_replay.cuh -- the ReplaySSM checkpointing update
// ("vllm.model_executor.layers.mamba.ops.ssu_dispatch":
// selective_state_update_replayssm_flashinfer and the ring-tracker kernels).
//
// A slot's state is its checkpoint state[slot] advanced through the
// k = prev_num_accepted[slot] tokens cached in its ring at positions
// (ring_start + j) mod R.  One call, per sequence: replay those k tokens,
// store the state they reach as the new checkpoint when k + L exceeds the
// logical window, run the sequence's L rows (y as in the plain update) and
// cache each row at position (ring_start + k + t) mod R.  With
// update_trackers the one-token tracker rule is applied to the slot in the
// same launch.
//
// Work decomposition as in the head-run kernels: one CTA per (sequence, run
// of kh heads of one group, row tile).  The chain -- k cached steps, then L
// new ones -- is staged like a packed chain: B (and C for new steps) and the
// per-head dt' and dA once per run, CTA-wide.  After that every warp runs
// its own pipeline, because a warp only ever touches its own contiguous rows
// of a tile: its part of each head's checkpoint tile lands in shared memory
// by one bulk asynchronous copy (TMA engine) on the warp's own mbarrier, two
// heads ahead; its rows' operands are loaded one head ahead; the warp
// synchronises only with itself.  Cached steps only advance the state (no
// y); new steps are the plain step_rows, so the arithmetic of every step is
// that of the plain kernels.  Chains longer than LMAX steps are staged LMAX
// steps at a time, head by head, CTA-wide.  Every mbarrier wait is bounded: a
// wait that runs out sets the device error word, lets the warp's own copies
// land and ends the warp.
//
// The tracker update must wait until every CTA of the sequence has read the
// trackers: each CTA counts itself in arrivals[s] after its read, and the
// last one writes the trackers and puts the counter back to zero (the
// "last block" pattern: a fence before the count makes the read visible as
// done, a fence after it orders the write).
#pragma once

#include "ssu_bulk.cuh"
#include "ssu_headrun.cuh"

namespace ssu {

struct ReplayArgs {
  const void* sbi;  // read / write slot of sequence s at s * sbi_stride, or nullptr (slot s)
  int64_t sbi_stride;
  int idx64;
  const void* cu;  // [nseqs + 1] row starts, or nullptr (row s)
  int meta64;
  int64_t rows;
  void* x_cache;    // [slots, H, R, P], io dtype
  void* B_cache;    // [slots, G, R, N], io dtype
  float* dt_cache;  // [slots, H, R]
  int R, G, W;
  int32_t* ring_start;
  int32_t* prev;
  int64_t limit;  // slots below this have trackers (min of slots and tracker length)
  int update_trackers;
  unsigned* arrivals;  // [nseqs] counters, zero between calls
};

// Shared memory of one CTA (dynamic: more than the 48 KB static limit).
template <int N, int ROWS, int LMAX, int TILE_BYTES, int WARPS>
struct __align__(128) ReplaySmem {
  unsigned char tile[2][TILE_BYTES];
  uint64_t bar[WARPS][2];  // per warp and tile buffer: its part of the tile landed
  StepsBC<N, LMAX> bc;
  HeadRows<ROWS, LMAX> rows[2];
  float raw_dt[8][LMAX];  // per head of the run and step: dt as cached / given
  float dtp[8][LMAX];     // dt' (per-head parameters only)
  float dA[8][LMAX];
  float Dh[8];            // D per head of the run (per-head D; 0 without D)
  int64_t slot, r0;
  int k, start, L, slot_ok, ok, must;
};

// h <- h dA + (dt' x) B for this thread's rows, no y (a cached step).  The
// same operations, in the same order, as the update half of step_rows.
template <class ST, int N, int UNR, class StageT>
__device__ __forceinline__ void advance_rows(float2 (&hs)[UNR][RowLayout<ST, N>::EPL / 2],
                                             const StageT& stg, int tt, int q, int jbase) {
  using L = RowLayout<ST, N>;
  constexpr int H4 = L::VEC / 4;
  constexpr int C2 = L::VEC / 2;
#pragma unroll
  for (int c = 0; c < L::CPL; ++c) {
    float2 bv[C2];
#pragma unroll
    for (int hh = 0; hh < H4; ++hh) {
      const float4 b4 =
          *reinterpret_cast<const float4*>(&stg.B[tt][((c * H4 + hh) * L::LPR + q) * 4]);
      bv[2 * hh] = make_float2(b4.x, b4.y);
      bv[2 * hh + 1] = make_float2(b4.z, b4.w);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int j = jbase + u * L::RPW;
      const float2 dA2 = make_float2(stg.dA[tt][j], stg.dA[tt][j]);
      const float2 dtx2 = make_float2(stg.dtx[tt][j], stg.dtx[tt][j]);
#pragma unroll
      for (int i = 0; i < C2; ++i)
        hs[u][c * C2 + i] = __ffma2_rn(hs[u][c * C2 + i], dA2, __fmul2_rn(dtx2, bv[i]));
    }
  }
}

__device__ __forceinline__ int ring_pos(int start, int j, int R) {
  const int v = start + j;  // start < R and j < R
  return v >= R ? v - R : v;
}

// B of chain steps [c0, c0 + cn) (cached steps from the ring, new steps from
// B), C of the new ones, in the bc_slot layout; `cache_b` also writes the new
// steps' B into the ring (one CTA per group does).
template <class ST, class IT, int N, int LMAX, int THREADS, class SM>
__device__ __forceinline__ void replay_stage_bc(SM& m, const KParams& p, const ReplayArgs& ra,
                                                int g, int c0, int cn, bool cache_b) {
  const IT* Bp = static_cast<const IT*>(p.B);
  const IT* Cp = static_cast<const IT*>(p.C);
  IT* Bc = static_cast<IT*>(ra.B_cache);
  for (int i = threadIdx.x; i < cn * N; i += THREADS) {
    const int tt = i / N, n = i - tt * N;
    const int j = c0 + tt;
    const int pos = ring_pos(m.start, j, ra.R);
    IT* cached = Bc + ((m.slot * ra.G + g) * ra.R + pos) * N + n;
    float b, c = 0.0f;
    if (j < m.k) {
      b = io_to_float<IT>(*cached);
    } else {
      const int64_t r = m.r0 + (j - m.k);
      const IT bv = Bp[r * p.B_rs + (int64_t)g * p.B_gs + n];
      b = io_to_float<IT>(bv);
      c = io_to_float<IT>(Cp[r * p.C_rs + (int64_t)g * p.C_gs + n]);
      if (cache_b) *cached = bv;
    }
    m.bc.B[tt][bc_slot<ST, N>(n)] = b;
    m.bc.C[tt][bc_slot<ST, N>(n)] = c;
  }
}

// Per head of the run (heads h0 .. h0 + nh - 1 at run positions hh0 ..): the
// steps' dt (cached or given; new ones written to the ring by `cache_dt`) and,
// with per-head parameters, dt' and dA.
template <int LMAX, int THREADS, class SM>
__device__ __forceinline__ void replay_stage_heads(SM& m, const KParams& p, const ReplayArgs& ra,
                                                   int h0, int hh0, int nh, int c0, int cn,
                                                   bool tied, bool cache_dt) {
  for (int i = threadIdx.x; i < nh * LMAX; i += THREADS) {
    const int hh = i / LMAX, tt = i - hh * LMAX;
    if (tt >= cn) continue;
    const int h = h0 + hh, j = c0 + tt;
    float* cached = ra.dt_cache + (m.slot * p.H + h) * ra.R + ring_pos(m.start, j, ra.R);
    float d;
    if (j < m.k) {
      d = *cached;
    } else {
      d = p.dt[(m.r0 + (j - m.k)) * p.dt_rs + (int64_t)h * p.dt_hs];
      if (cache_dt) *cached = d;
    }
    m.raw_dt[hh0 + hh][tt] = d;
    if (tt == 0) m.Dh[hh0 + hh] = p.D ? p.D[(int64_t)h * p.D_s] : 0.0f;
    if (tied) {
      float v = d + (p.dt_bias ? p.dt_bias[(int64_t)h * p.bias_s] : 0.0f);
      if (p.softplus) v = softplus_f(v);
      m.dtp[hh0 + hh][tt] = v;
      m.dA[hh0 + hh][tt] = expf(p.A[(int64_t)h * p.A_s] * v);
    }
  }
}

// Per-row operands of head h (run position hh) for chain steps [c0, c0 + cn)
// and the RW rows of one warp (tile rows w0 .. w0 + RW - 1), in two halves so
// that the loads of the next head are in flight while the current head
// computes: load() issues this lane's loads of x (from the ring for cached
// steps) and z into registers; finish() forms dA, dt' x and, for new steps,
// D x and silu(z) -- the plain kernels' expressions -- stores them for the
// steps, and writes the new steps' x into the ring (`cache_x`).
// The sequence's values every staging call needs, kept in registers (the
// shared copies would be reloaded after every barrier).
struct ReplaySeq {
  int64_t slot, r0;
  int k, start;
};

template <class IT, int RW, int LMAX>
struct ReplayRows {
  static constexpr int NT = (LMAX * RW + 31) / 32;  // tasks per lane
  IT xv[NT], zv[NT];

  __device__ __forceinline__ void load(const ReplaySeq& q, const KParams& p, const ReplayArgs& ra,
                                       int h, int p0, int w0, int c0, int cn, int lane) {
    const IT* xp = static_cast<const IT*>(p.x);
    const IT* zp = static_cast<const IT*>(p.z);
    const IT* xc = static_cast<const IT*>(ra.x_cache);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int i = lane + t * 32;
      const int tt = i / RW;
      const int prow = p0 + w0 + (i - tt * RW);
      if (tt < cn && prow < p.P) {
        const int j = c0 + tt;
        if (j < q.k) {
          xv[t] = xc[((q.slot * p.H + h) * ra.R + ring_pos(q.start, j, ra.R)) * p.P + prow];
        } else {
          const int64_t r = q.r0 + (j - q.k);
          xv[t] = xp[r * p.x_rs + (int64_t)h * p.x_hs + prow];
          if (zp) zv[t] = zp[r * p.z_rs + (int64_t)h * p.z_hs + prow];
        }
      }
    }
  }

  // dtp / dA: this head's dt' and dA by step (per-head parameters); Dh its D
  // (per-head D) -- all from shared memory, staged once per run
  template <class HR>
  __device__ __forceinline__ void finish(const ReplaySeq& q, HR& out, const KParams& p,
                                         const ReplayArgs& ra, int h, const float* raw_dt,
                                         const float* dtp, const float* dA_h, float Dh, int p0,
                                         int w0, int c0, int cn, bool tied, bool cache_x,
                                         int lane) const {
    IT* xc = static_cast<IT*>(ra.x_cache);
    const bool D_row = p.D && p.D_ds != 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int i = lane + t * 32;
      const int tt = i / RW;
      if (tt >= cn) break;  // steps past the chain are never read
      const int row = w0 + (i - tt * RW);
      const int prow = p0 + row;
      const int j = c0 + tt;
      const bool fresh = j >= q.k;
      float dA = 1.0f, dtx = 0.0f;
      if (prow < p.P) {
        const float x = io_to_float<IT>(xv[t]);
        float d;
        if (tied) {
          d = dtp[tt];
          dA = dA_h[tt];
        } else {
          d = raw_dt[tt] +
              (p.dt_bias ? p.dt_bias[(int64_t)h * p.bias_s + (int64_t)prow * p.bias_ds] : 0.0f);
          if (p.softplus) d = softplus_f(d);
          dA = expf(p.A[(int64_t)h * p.A_s + (int64_t)prow * p.A_ds] * d);
        }
        dtx = d * x;
        if (fresh) {  // D x and silu(z): new steps only (cached steps give no y)
          const float Dv = D_row ? p.D[(int64_t)h * p.D_s + (int64_t)prow * p.D_ds] : Dh;
          float gate = 1.0f;
          if (p.z) {
            const float z = io_to_float<IT>(zv[t]);
            gate = z / (1.0f + expf(-z));
          }
          out.Dx[tt][row] = Dv * x;
          out.gate[tt][row] = gate;
          if (cache_x)
            xc[((q.slot * p.H + h) * ra.R + ring_pos(q.start, j, ra.R)) * p.P + prow] = xv[t];
        }
      } else if (fresh) {
        out.Dx[tt][row] = 0.0f;
        out.gate[tt][row] = 1.0f;
      }
      out.dA[tt][row] = dA;
      out.dtx[tt][row] = dtx;
    }
  }
};

template <class ST, class IT, int N, int WARPS, int UNR, int LMAX>
struct ReplayCfg {
  using Cfg = SSUConfig<ST, IT, N, WARPS, UNR, LMAX>;
  static constexpr int ROWS = Cfg::ROWS;
  static constexpr int THREADS = Cfg::THREADS;
  static constexpr int TILE_BYTES = ROWS * N * (int)sizeof(ST);
  using Smem = ReplaySmem<N, ROWS, LMAX, TILE_BYTES, WARPS>;
};

template <class ST, class IT, int N, int WARPS, int UNR, int LMAX, bool SR = false>
__global__ void __launch_bounds__(WARPS * 32, sizeof(ST) == 2 ? 3 : 16 / WARPS)
    ssu_replay_kernel(const KParams p, const ReplayArgs ra, int64_t nseqs, int kh,
                      unsigned* err) {
  using RC = ReplayCfg<ST, IT, N, WARPS, UNR, LMAX>;
  using L = RowLayout<ST, N>;
  constexpr int ROWS = RC::ROWS;
  constexpr int THREADS = RC::THREADS;
  constexpr int RW = UNR * L::RPW;                    // rows of one warp
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto& m = *reinterpret_cast<typename RC::Smem*>(smem_raw);

  int64_t s;
  int h0, p0;
  if (!head_run_coords(p, nseqs, kh, ROWS, &s, &h0, &p0)) return;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  // 1. the sequence's rows and slot (and the warps' mbarriers)
  if (threadIdx.x < 2 * WARPS) mbar_init(&m.bar[threadIdx.x / 2][threadIdx.x % 2], 1);
  if (threadIdx.x == 0) {
    int64_t begin = s, end = s + 1;
    if (ra.cu) {
      begin = load_int(ra.cu, s, ra.meta64);
      end = load_int(ra.cu, s + 1, ra.meta64);
    }
    if (begin < 0) begin = 0;
    if (end > ra.rows) end = ra.rows;
    const int64_t len = end > begin ? end - begin : 0;
    const int64_t slot = ra.sbi ? load_int(ra.sbi, s * ra.sbi_stride, ra.idx64) : s;
    const bool valid = len > 0 && slot != p.pad && slot >= 0 && slot < ra.limit;
    m.slot = valid ? slot : 0;
    m.r0 = begin;
    m.L = (int)len;  // rows < 2^31 (checked on the host)
    m.slot_ok = valid;
  }
  __syncthreads();
  const int len = m.L;
  if (len <= 0) return;

  // 2. each warp requests its part of the first two heads' checkpoint tiles
  //    as soon as the slot is known, before the trackers are read
  const int64_t block_elems = (int64_t)p.P * N;
  const int w0 = warp * RW;  // this warp's first row of a tile
  const int wrows = max(0, min(RW, p.P - p0 - w0));
  const uint32_t wbytes = m.slot_ok ? (uint32_t)(wrows * N * (int)sizeof(ST)) : 0u;
  const ST* wsrc = static_cast<const ST*>(p.state) + m.slot * p.H * block_elems +
                   (int64_t)(p0 + w0) * N;
  auto issue = [&](int kk, int buf) {
    if (lane == 0 && kk < kh) {
      uint64_t* bar = &m.bar[warp][buf];
      if (wbytes) {
        mbar_arrive_expect_tx(bar, wbytes);
        bulk_load(m.tile[buf] + w0 * N * (int)sizeof(ST), wsrc + (int64_t)(h0 + kk) * block_elems,
                  wbytes, bar);
      } else {
        mbar_arrive(bar);
      }
    }
  };
  // a wait that runs out: record it, let this warp's copies still in flight
  // (heads kk and kk + 1) land, and end the warp
  auto give_up = [&](int kk) {
    if (lane == 0) {
      atomicOr(err, kErrFullTimeout);
      for (int t = kk; t < kk + 2 && t < kh; ++t) {
        const uint64_t t0 = global_ns();
        while (!mbar_test(&m.bar[warp][t & 1], (uint32_t)(t >> 1) & 1) &&
               global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  };
  issue(0, 0);
  issue(1, 1);

  // 3. the trackers: a sequence whose k + L does not fit the ring (or whose
  //    values are out of range) runs from a zero state and writes nothing
  if (threadIdx.x == 0) {
    int k = 0, start = 0;
    bool ok = m.slot_ok;
    if (ok) {
      k = ra.prev[m.slot];
      start = ra.ring_start[m.slot];
      ok = k >= 0 && start >= 0 && start < ra.R && (int64_t)k + len <= ra.R;
    }
    m.k = ok ? k : 0;
    m.start = ok ? start : 0;
    m.must = ok && (int64_t)k + len > ra.W;
    m.ok = ok;
  }
  __syncthreads();
  const int k = m.k;
  const bool ok = m.ok, must = m.must;
  const ReplaySeq sq{m.slot, m.r0, k, m.start};
  const int n = k + len;  // chain length
  const int g = (int)p.fd_hr.div((uint32_t)h0);
  const bool tied = per_head_dt(p);
  const bool group_writer = ok && p0 == 0 && (h0 % p.hr) == 0;  // caches B of the group
  const bool single = n <= LMAX;

  const int q = lane % L::LPR;
  const int rr = lane / L::LPR;
  const int jbase = warp * UNR * L::RPW + rr;
  ST* state = static_cast<ST*>(p.state);
  ReplayRows<IT, RW, LMAX> pre;

  // 4. the chain's B / C and the heads' dt', dA (CTA-wide, once per run);
  //    the first head's rows of this warp
  if (single) {
    pre.load(sq, p, ra, h0, p0, w0, 0, n, lane);
    replay_stage_bc<ST, IT, N, LMAX, THREADS>(m, p, ra, g, 0, n, group_writer);
    replay_stage_heads<LMAX, THREADS>(m, p, ra, h0, 0, kh, 0, n, tied, ok && p0 == 0);
    __syncthreads();
    pre.finish(sq, m.rows[0], p, ra, h0, m.raw_dt[0], m.dtp[0], m.dA[0], m.Dh[0], p0, w0, 0, n,
               tied, ok, lane);
    if (kh > 1) pre.load(sq, p, ra, h0 + 1, p0, w0, 0, n, lane);  // a whole head ahead
  }

  for (int kk = 0; kk < kh; ++kk) {
    const int h = h0 + kk;
    const int buf = kk & 1;
    // 5. this warp's rows of head kk's checkpoint, widened to fp32
    bool landed = __all_sync(0xffffffffu, mbar_wait(&m.bar[warp][buf], (uint32_t)(kk >> 1) & 1));
    // the CTA-wide path meets at barriers below: all its warps leave together
    if (!single) landed = __syncthreads_and(landed);
    if (!landed) {
      give_up(kk);
      return;
    }
    float2 hs[UNR][L::EPL / 2];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int j = jbase + u * L::RPW;
#pragma unroll
      for (int c = 0; c < L::CPL; ++c)
        Elem<ST>::unpack2(*reinterpret_cast<const uint4*>(
                              m.tile[buf] + ((size_t)j * N + (q + c * L::LPR) * L::VEC) *
                                                sizeof(ST)),
                          &hs[u][c * L::VEC / 2]);
    }
    if (!ok) {  // the trackers ruled the sequence out: a zero state
#pragma unroll
      for (int u = 0; u < UNR; ++u)
#pragma unroll
        for (int e = 0; e < L::EPL / 2; ++e) hs[u][e] = make_float2(0.0f, 0.0f);
    }
    __syncwarp();      // the warp is done with its part of this buffer; rows of
                       // head kk (staged last iteration) are visible
    issue(kk + 2, buf);
    if (single && kk + 1 < kh) {
      pre.finish(sq, m.rows[(kk + 1) & 1], p, ra, h + 1, m.raw_dt[kk + 1], m.dtp[kk + 1],
                 m.dA[kk + 1], m.Dh[kk + 1], p0, w0, 0, n, tied, ok, lane);
      if (kk + 2 < kh) pre.load(sq, p, ra, h + 2, p0, w0, 0, n, lane);
    }
    ST* ckpt = state + (sq.slot * p.H + h) * block_elems;
    for (int c0 = 0; c0 < n; c0 += LMAX) {
      const int cn = n - c0 < LMAX ? n - c0 : LMAX;
      if (!single) {  // this chunk of head kk, CTA-wide: B / C, dt, rows
        __syncthreads();
        replay_stage_bc<ST, IT, N, LMAX, THREADS>(m, p, ra, g, c0, cn, group_writer && kk == 0);
        replay_stage_heads<LMAX, THREADS>(m, p, ra, h, 0, 1, c0, cn, tied, ok && p0 == 0);
        pre.load(sq, p, ra, h, p0, w0, c0, cn, lane);
        __syncthreads();
        pre.finish(sq, m.rows[0], p, ra, h, m.raw_dt[0], m.dtp[0], m.dA[0], m.Dh[0], p0, w0, c0,
                   cn, tied, ok, lane);
        __syncwarp();
      }
      const auto& hr = m.rows[single ? (kk & 1) : 0];
      const StageView<N, ROWS, LMAX> view{m.bc.B, m.bc.C, hr.dA, hr.dtx, hr.Dx, hr.gate};
#pragma unroll 1
      for (int tt = 0; tt < cn; ++tt) {
        const int j = c0 + tt;
        if (j < k) {
          advance_rows<ST, N, UNR>(hs, view, tt, q, jbase);
          if (j == k - 1 && must) {  // the new checkpoint: the state after the cached steps
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
              const int prow = p0 + (warp * UNR + u) * L::RPW + rr;
              if (prow < p.P) {
#pragma unroll
                for (int c = 0; c < L::CPL; ++c)
                  store_state<ST, SR>(state, ckpt - state + (int64_t)prow * N + (q + c * L::LPR) * L::VEC,
                                  &hs[u][c * L::VEC / 2], p);
              }
            }
          }
        } else {
          step_rows<ST, IT, N, UNR>(hs, view, tt, q, jbase, p, h, p0, sq.r0 + (j - k));
        }
      }
    }
  }

  // 6. the tracker update: the last CTA of the sequence to get here (every
  //    other one has read the trackers before it counted itself) applies the
  //    one-token rule and clears the counter for the next call
  if (threadIdx.x == 0 && ok && ra.update_trackers) {
    __threadfence();
    if (atomicAdd(&ra.arrivals[s], 1u) == gridDim.x - 1) {
      __threadfence();
      const bool mt = k + 1 > ra.W;  // the one-token rule of ssu_ring_update
      ra.ring_start[m.slot] = mt ? (m.start + k) % ra.R : m.start;
      ra.prev[m.slot] = mt ? 1 : k + 1;
      ra.arrivals[s] = 0;
    }
  }
}

}  // namespace ssu
