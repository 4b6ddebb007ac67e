// ssu_bulk.cuh -- persistent, warp-specialised SSU kernel: the state block of
// every work item arrives by one bulk asynchronous copy (cp.async.bulk, the
// TMA engine) into a ring of shared-memory stages.
//
// Why: the SSU is HBM-bound, and a kernel whose state loads land in registers
// can only keep as many bytes in flight as its resident threads have free
// registers, and only while each CTA is in its load phase.  Here the loads
// land in shared memory, issued ahead by a producer warp, so S stages of
// 16-32 KB per CTA stay in flight continuously while the consumer warps work.
//
// Work item = (sequence, head, row tile of ROWS headdim rows); a CTA walks the
// items blockIdx.x, blockIdx.x + gridDim.x, ...  For item k on stage s = k % S:
//   producer (one thread): resolve the item's slots (one item ahead, so the
//     index loads are in flight while it waits), wait empty[s] (the consumers
//     released item k - S), publish the slots in the stage's record, arm
//     full[s] with the tile's byte count and issue one bulk copy of its
//     contiguous rows (or just arrive for a pad / invalid read slot);
//   consumer warps: stage the item's per-step vectors (B, C, dA, dt' x, D x,
//     silu z) into one of two shared buffers with one round of loads while the
//     copy lands, wait full[s], read their chunks of the tile into fp32
//     registers, release empty[s] at once, then run the steps exactly as the
//     register kernel does (same lane layout, same arithmetic, same stores).
// Every wait is bounded (2 s of global time); a wait that runs out records an
// error code in *err and the CTA leaves after its own copies have landed.
#pragma once

#include "ssu_kernel.cuh"

namespace ssu {

constexpr unsigned kErrFullTimeout = 1u;
constexpr unsigned kErrEmptyTimeout = 2u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with `parity` to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_test(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// One bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// A resolved work item.
struct Item {
  int64_t seq, r0, src, dst;  // dst: the one-token write slot
  int h, p0, len;
  bool read_ok;
};

template <int ROWS>
__device__ __forceinline__ Item resolve_one_token(const KParams& p, const OneTokenArgs& a,
                                                  int64_t idx) {
  Item it;
  const int tile = (int)(idx % p.tiles);
  const int64_t rest = idx / p.tiles;
  it.h = (int)(rest % p.H);
  it.seq = rest / p.H;
  it.p0 = tile * ROWS;
  it.r0 = it.seq;
  it.len = 1;
  it.src = a.sbi ? load_int(a.sbi, it.seq, a.idx64) : it.seq;
  it.dst = a.dsbi ? load_int(a.dsbi, it.seq, a.idx64) : it.src;
  it.read_ok = slot_ok(it.src, p.pad, p.slots);
  return it;
}

template <int ROWS>
__device__ __forceinline__ Item resolve_varlen(const KParams& p, const VarlenArgs& a,
                                               int64_t idx) {
  Item it;
  const int tile = (int)(idx % p.tiles);
  const int64_t rest = idx / p.tiles;
  it.h = (int)(rest % p.H);
  it.seq = rest / p.H;
  it.p0 = tile * ROWS;
  int64_t begin, end;
  if (a.cu) {
    begin = load_int(a.cu, it.seq, a.meta64);
    end = load_int(a.cu, it.seq + 1, a.meta64);
  } else {
    begin = it.seq * a.dense_steps;
    end = begin + a.dense_steps;
  }
  if (begin < 0) begin = 0;
  if (end > a.rows) end = a.rows;
  it.r0 = begin;
  it.len = end > begin ? (int)(end - begin) : 0;
  it.src = it.seq;
  it.dst = -1;
  bool ok = true;
  if (a.src.idx) {
    const int64_t col = a.na ? load_int(a.na, it.seq, a.meta64) - 1 : 0;
    ok = table_entry(a.src, it.seq, col, a.idx64, &it.src);
  }
  it.read_ok = it.len > 0 && ok && slot_ok(it.src, p.pad, p.slots);
  return it;
}

template <bool VARLEN, int ROWS>
__device__ __forceinline__ Item resolve_item(const KParams& p, const OneTokenArgs& oa,
                                             const VarlenArgs& va, int64_t idx) {
  if constexpr (VARLEN) return resolve_varlen<ROWS>(p, va, idx);
  else return resolve_one_token<ROWS>(p, oa, idx);
}

// Stage steps [t0, t0 + n) of an item with `nthr` threads numbered `tid`.
template <class IT, int N, int ROWS, int LMAX>
__device__ __forceinline__ void stage_vectors(Stage<N, ROWS, LMAX>& s, const KParams& p,
                                              const Item& it, int t0, int n, int tid, int nthr) {
  const int g = it.h / p.hr;
  const IT* Bp = static_cast<const IT*>(p.B);
  const IT* Cp = static_cast<const IT*>(p.C);
  for (int i = tid; i < n * N; i += nthr) {
    const int tt = i / N, k = i - tt * N;
    const int64_t r = it.r0 + t0 + tt;
    s.B[tt][k] = io_to_float<IT>(Bp[r * p.B_rs + (int64_t)g * p.B_gs + k]);
    s.C[tt][k] = io_to_float<IT>(Cp[r * p.C_rs + (int64_t)g * p.C_gs + k]);
  }
  const IT* xp = static_cast<const IT*>(p.x);
  const IT* zp = static_cast<const IT*>(p.z);
  for (int i = tid; i < n * ROWS; i += nthr) {
    const int tt = i / ROWS, j = i - tt * ROWS;
    const int prow = it.p0 + j;
    float dA = 1.0f, dtx = 0.0f, Dx = 0.0f, gate = 1.0f;
    if (prow < p.P) {
      const int64_t r = it.r0 + t0 + tt;
      const float A = p.A[(int64_t)it.h * p.A_s + (int64_t)prow * p.A_ds];
      const float Dh = p.D ? p.D[(int64_t)it.h * p.D_s + (int64_t)prow * p.D_ds] : 0.0f;
      const float bias =
          p.dt_bias ? p.dt_bias[(int64_t)it.h * p.bias_s + (int64_t)prow * p.bias_ds] : 0.0f;
      const float xv = io_to_float<IT>(xp[r * p.x_rs + (int64_t)it.h * p.x_hs + prow]);
      float dtv = p.dt[r * p.dt_rs + (int64_t)it.h * p.dt_hs + (int64_t)prow * p.dt_ds] + bias;
      if (p.softplus) dtv = softplus_f(dtv);
      dA = expf(A * dtv);
      dtx = dtv * xv;
      Dx = Dh * xv;
      if (zp) {
        const float zv = io_to_float<IT>(zp[r * p.z_rs + (int64_t)it.h * p.z_hs + prow]);
        gate = zv / (1.0f + expf(-zv));
      }
    }
    s.dA[tt][j] = dA;
    s.dtx[tt][j] = dtx;
    s.Dx[tt][j] = Dx;
    s.gate[tt][j] = gate;
  }
}

// Slot resolution of one item, written by the producer for the consumers.
struct __align__(16) SlotRec {
  int64_t src, dst;
  int read_ok, pad_;
};

// Slots of item `idx` (the producer's part of resolve_*: everything the copy
// and the consumers need beyond the item's position).
template <bool VARLEN, int ROWS>
__device__ __forceinline__ SlotRec resolve_slots(const KParams& p, const OneTokenArgs& oa,
                                                 const VarlenArgs& va, int64_t idx, int* p0,
                                                 int* h) {
  const Item it = resolve_item<VARLEN, ROWS>(p, oa, va, idx);
  *p0 = it.p0;
  *h = it.h;
  SlotRec r;
  r.src = it.src;
  r.dst = it.dst;
  r.read_ok = it.read_ok;
  r.pad_ = 0;
  return r;
}

template <class ST, class IT, int N, int WARPS, int UNR, int S, int LMAX>
struct BulkConfig {
  using L = RowLayout<ST, N>;
  static constexpr int ROWS = WARPS * L::RPW * UNR;
  static constexpr int CONSUMERS = WARPS * 32;
  static constexpr int THREADS = CONSUMERS + 32;  // + one producer warp
  static constexpr int STAGE_BYTES = ROWS * N * (int)sizeof(ST);
  using Vec = Stage<N, ROWS, LMAX>;
  static constexpr int VEC_OFF = S * STAGE_BYTES;               // two vector buffers
  static constexpr int REC_OFF = VEC_OFF + 2 * (int)sizeof(Vec);  // S slot records
  static constexpr int BAR_OFF = REC_OFF + S * (int)sizeof(SlotRec);
  static constexpr int SMEM = BAR_OFF + 2 * S * 8;
  static_assert(STAGE_BYTES % 16 == 0 && sizeof(Vec) % 16 == 0, "16-byte stage alignment");
};

template <class ST, class IT, int N, int WARPS, int UNR, int S, int LMAX, bool VARLEN>
__global__ void __launch_bounds__(WARPS * 32 + 32)
    ssu_bulk_kernel(const KParams p, const OneTokenArgs oa, const VarlenArgs va, int64_t nitems,
                    unsigned* err) {
  using Cfg = BulkConfig<ST, IT, N, WARPS, UNR, S, LMAX>;
  using L = typename Cfg::L;
  using Vec = typename Cfg::Vec;
  constexpr int ROWS = Cfg::ROWS;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* bufs = smem;
  Vec* vecs = reinterpret_cast<Vec*>(smem + Cfg::VEC_OFF);
  SlotRec* recs = reinterpret_cast<SlotRec*>(smem + Cfg::REC_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  uint64_t* empty = full + S;
  __shared__ int s_abort;
  __shared__ int s_issued[S];  // last round whose copy was issued on each stage (-1: none)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);        // the producer's arrival (with the copy's bytes)
      mbar_init(&empty[s], WARPS);   // one arrival per consumer warp
      s_issued[s] = -1;
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int64_t block_elems = (int64_t)p.P * N;

  if (warp == WARPS) {
    // ---------------- producer: one thread resolves slots and issues copies ----------------
    if (lane != 0) return;
    int64_t idx = blockIdx.x;
    if (idx >= nitems) return;
    int p0, h;
    SlotRec next = resolve_slots<VARLEN, ROWS>(p, oa, va, idx, &p0, &h);
    for (int64_t k = 0; idx < nitems; idx += gridDim.x, ++k) {
      const SlotRec cur = next;
      const int cur_p0 = p0, cur_h = h;
      if (idx + gridDim.x < nitems)  // prefetch the next item's slots
        next = resolve_slots<VARLEN, ROWS>(p, oa, va, idx + gridDim.x, &p0, &h);
      const int s = (int)(k % S);
      const uint32_t round = (uint32_t)(k / S);
      if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1)) {
        atomicOr(err, kErrEmptyTimeout);
        break;
      }
      recs[s] = cur;
      if (cur.read_ok) {
        const int nrows = min(ROWS, p.P - cur_p0);
        const uint32_t bytes = (uint32_t)(nrows * N * (int)sizeof(ST));
        const ST* src = static_cast<const ST*>(p.state) +
                        ((cur.src * p.H + cur_h) * block_elems + (int64_t)cur_p0 * N);
        s_issued[s] = (int)round;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load(bufs + (size_t)s * Cfg::STAGE_BYTES, src, bytes, &full[s]);
      } else {
        mbar_arrive(&full[s]);
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  const int q = lane % L::LPR;
  const int rr = lane / L::LPR;
  ST* state = static_cast<ST*>(p.state);
  IT* out_io = static_cast<IT*>(p.out);
  float* out_f = static_cast<float*>(p.out);
  const int ctid = threadIdx.x;  // 0 .. CONSUMERS-1
  int64_t k = 0;
  for (int64_t idx = blockIdx.x; idx < nitems; idx += gridDim.x, ++k) {
    const int s = (int)(k % S);
    const uint32_t round = (uint32_t)(k / S);
    Vec& stg = vecs[k & 1];
    // the item's position (no slot loads: the producer resolves those)
    Item it;
    {
      const int tile = (int)(idx % p.tiles);
      const int64_t rest = idx / p.tiles;
      it.h = (int)(rest % p.H);
      it.seq = rest / p.H;
      it.p0 = tile * ROWS;
      if constexpr (VARLEN) {
        int64_t begin, end;
        if (va.cu) {
          begin = load_int(va.cu, it.seq, va.meta64);
          end = load_int(va.cu, it.seq + 1, va.meta64);
        } else {
          begin = it.seq * va.dense_steps;
          end = begin + va.dense_steps;
        }
        if (begin < 0) begin = 0;
        if (end > va.rows) end = va.rows;
        it.r0 = begin;
        it.len = end > begin ? (int)(end - begin) : 0;
      } else {
        it.r0 = it.seq;
        it.len = 1;
      }
    }
    // stage this item's first steps (one round of loads) while its copy lands
    if (it.len > 0)
      stage_vectors<IT, N, ROWS, LMAX>(stg, p, it, 0, min(it.len, LMAX), ctid, Cfg::CONSUMERS);
    if (!mbar_wait(&full[s], round & 1)) s_abort = 1;
    named_sync(1, Cfg::CONSUMERS);
    if (s_abort) {
      if (ctid == 0) {
        atomicOr(err, kErrFullTimeout);
        for (int t = 0; t < S; ++t) {  // let this CTA's own copies land before leaving
          const int r = *(volatile int*)&s_issued[t];
          if (r < 0) continue;
          const uint64_t t0 = global_ns();
          while (!mbar_test(&full[t], (uint32_t)r & 1) && global_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
      return;
    }
    const SlotRec rec = recs[s];
    it.src = rec.src;
    it.dst = rec.dst;
    it.read_ok = rec.read_ok != 0;
    // state chunks of this thread's rows, widened to fp32; then release the stage
    float hs[UNR][L::EPL];
    const unsigned char* buf = bufs + (size_t)s * Cfg::STAGE_BYTES;
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int j = (warp * UNR + u) * L::RPW + rr;
      const bool rd = it.read_ok && it.p0 + j < p.P;
#pragma unroll
      for (int c = 0; c < L::CPL; ++c) {
        const uint4 raw =
            rd ? *reinterpret_cast<const uint4*>(buf + ((size_t)j * N + (q + c * L::LPR) * L::VEC) *
                                                           sizeof(ST))
               : make_uint4(0u, 0u, 0u, 0u);
        Elem<ST>::unpack(raw, &hs[u][c * L::VEC]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    for (int t0 = 0; t0 < it.len; t0 += LMAX) {
      const int n = (it.len - t0) < LMAX ? (it.len - t0) : LMAX;
      if (t0 > 0) {
        named_sync(1, Cfg::CONSUMERS);
        stage_vectors<IT, N, ROWS, LMAX>(stg, p, it, t0, n, ctid, Cfg::CONSUMERS);
        named_sync(1, Cfg::CONSUMERS);
      }
      for (int tt = 0; tt < n; ++tt) {
        const int64_t r = it.r0 + t0 + tt;
        float bv[L::EPL], cv[L::EPL];
#pragma unroll
        for (int c = 0; c < L::CPL; ++c) {
          const int k0 = (q + c * L::LPR) * L::VEC;
#pragma unroll
          for (int e = 0; e < L::VEC; e += 4) {
            const float4 b4 = *reinterpret_cast<const float4*>(&stg.B[tt][k0 + e]);
            const float4 c4 = *reinterpret_cast<const float4*>(&stg.C[tt][k0 + e]);
            bv[c * L::VEC + e + 0] = b4.x; bv[c * L::VEC + e + 1] = b4.y;
            bv[c * L::VEC + e + 2] = b4.z; bv[c * L::VEC + e + 3] = b4.w;
            cv[c * L::VEC + e + 0] = c4.x; cv[c * L::VEC + e + 1] = c4.y;
            cv[c * L::VEC + e + 2] = c4.z; cv[c * L::VEC + e + 3] = c4.w;
          }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int j = (warp * UNR + u) * L::RPW + rr;
          const float dA = stg.dA[tt][j];
          const float dtx = stg.dtx[tt][j];
          float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
          for (int e = 0; e < L::EPL; ++e) {
            const float hv = fmaf(hs[u][e], dA, dtx * bv[e]);
            hs[u][e] = hv;
            if (e & 1) acc1 = fmaf(hv, cv[e], acc1);
            else acc0 = fmaf(hv, cv[e], acc0);
          }
          float acc = acc0 + acc1;
#pragma unroll
          for (int off = L::LPR / 2; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
          const int prow = it.p0 + j;
          if (q == 0 && prow < p.P) {
            const float yv = (acc + stg.Dx[tt][j]) * stg.gate[tt][j];
            const int64_t o = r * p.o_rs + (int64_t)it.h * p.o_hs + prow;
            if (p.out_f32) out_f[o] = yv;
            else out_io[o] = float_to_io<IT>(yv);
          }
        }
        // this step's state
        int64_t dst = -1;
        bool have;
        if constexpr (VARLEN) {
          const TableArgs dtab = va.dst.idx ? va.dst : va.src;
          if (dtab.idx) have = table_entry(dtab, it.seq, t0 + tt, va.idx64, &dst);
          else { dst = it.seq; have = true; }
        } else {
          dst = it.dst;
          have = true;
        }
        if (it.read_ok && !p.disable && have && slot_ok(dst, p.pad, p.slots)) {
          ST* base = state + ((dst * p.H + it.h) * block_elems);
#pragma unroll
          for (int u = 0; u < UNR; ++u) {
            const int prow = it.p0 + (warp * UNR + u) * L::RPW + rr;
            if (prow < p.P) {
#pragma unroll
              for (int c = 0; c < L::CPL; ++c)
                st_state(base + (int64_t)prow * N + (q + c * L::LPR) * L::VEC,
                         Elem<ST>::pack(&hs[u][c * L::VEC]));
            }
          }
        }
      }
    }
  }
}

}  // namespace ssu
