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
// items blockIdx.x, blockIdx.x + gridDim.x, ...  For item k on stage s = k % S
// one producer thread resolves the item's slots (one item ahead, so the index
// loads are in flight while it waits), waits until stage s is free, publishes
// the slots, arms full[s] with the tile's byte count and issues one bulk copy
// of the tile's contiguous rows (or just arrives, for a pad / invalid read
// slot).  The consumer warps wait full[s], read their chunks of the tile into
// fp32 registers, release the stage at once, then run the steps of step_rows
// (the lane layout, arithmetic and stores of the head-run kernel).
// Two kernels differ in who stages the item's per-step operands (B, C, dA,
// dt' x, D x, silu z): in ssu_bulk_kernel the producer warp converts them into
// a ring of operand buffers one item ahead; in ssu_bulk_cs_kernel the consumer
// warps load them with one round of loads while the copy lands.
// Every wait is bounded (2 s of global time); a wait that runs out records an
// error code in *err and the CTA leaves after its own copies have landed.
#pragma once

#include "ssu_kernel.cuh"

namespace ssu {

// error word values (SSU_DEVICE_ERR_COPY_TIMEOUT / SSU_DEVICE_ERR_RELEASE_TIMEOUT
// of the C ABI): a tile copy never landed / a stage was never released
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

// try_wait with a suspend-time hint: a thread whose phase is not complete is
// descheduled until it completes or about `hint_ns` pass, instead of spinning
// (spinning warps take issue slots from the warps that compute).
__device__ __forceinline__ bool mbar_test_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

constexpr uint32_t kSuspendHintNs = 100000u;  // 0.1 ms per try; the phase wakes it sooner

// Wait for the phase with `parity` to complete; false after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_test_sleep(bar, parity, kSuspendHintNs)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
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
  int tile;
  split_index(p, (uint32_t)idx, &it.seq, &it.h, &tile);
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
  int tile;
  split_index(p, (uint32_t)idx, &it.seq, &it.h, &tile);
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
template <class ST, class IT, int N, int ROWS, int LMAX>
__device__ __forceinline__ void stage_vectors(Stage<N, ROWS, LMAX>& s, const KParams& p,
                                              const Item& it, int t0, int n, int tid, int nthr) {
  const int g = (int)p.fd_hr.div((uint32_t)it.h);
  const IT* Bp = static_cast<const IT*>(p.B);
  const IT* Cp = static_cast<const IT*>(p.C);
  for (int i = tid; i < n * N; i += nthr) {
    const int tt = i / N, k = i - tt * N;
    const int64_t r = it.r0 + t0 + tt;
    s.B[tt][bc_slot<ST, N>(k)] = io_to_float<IT>(Bp[r * p.B_rs + (int64_t)g * p.B_gs + k]);
    s.C[tt][bc_slot<ST, N>(k)] = io_to_float<IT>(Cp[r * p.C_rs + (int64_t)g * p.C_gs + k]);
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

// The per-step operands of one item, loaded into registers ahead of use:
// thread `tid` of `NTHR` holds B/C values tid, tid + NTHR, ... of the item's
// [n][2N] block and row values tid, tid + NTHR, ... of its [n][ROWS] block.
template <class ST, class IT, int N, int ROWS, int LMAX, int NTHR>
struct VecPrefetch {
  static constexpr int BCPT = (LMAX * 2 * N + NTHR - 1) / NTHR;
  static constexpr int RPT = (LMAX * ROWS + NTHR - 1) / NTHR;
  IT bc[BCPT];
  IT x[RPT], z[RPT];
  float dt[RPT], A[RPT], D[RPT], bias[RPT];
  int n;  // staged steps (0: nothing)

  // Issue the loads of steps [0, n) of item `it` (rows r0 ..).
  __device__ __forceinline__ void issue(const KParams& p, const Item& it, int n_, int tid) {
    n = n_;
    const int g = (int)p.fd_hr.div((uint32_t)it.h);
    const IT* Bp = static_cast<const IT*>(p.B);
    const IT* Cp = static_cast<const IT*>(p.C);
#pragma unroll
    for (int i = 0; i < BCPT; ++i) {
      const int e = tid + i * NTHR;
      if (e < n * 2 * N) {
        const int tt = e / (2 * N), k = e - tt * 2 * N;
        const int64_t r = it.r0 + tt;
        bc[i] = k < N ? Bp[r * p.B_rs + (int64_t)g * p.B_gs + k]
                      : Cp[r * p.C_rs + (int64_t)g * p.C_gs + (k - N)];
      }
    }
    const IT* xp = static_cast<const IT*>(p.x);
    const IT* zp = static_cast<const IT*>(p.z);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int e = tid + i * NTHR;
      const int tt = e / ROWS, j = e - tt * ROWS;
      const int prow = it.p0 + j;
      if (e < n * ROWS && prow < p.P) {
        const int64_t r = it.r0 + tt;
        x[i] = xp[r * p.x_rs + (int64_t)it.h * p.x_hs + prow];
        if (zp) z[i] = zp[r * p.z_rs + (int64_t)it.h * p.z_hs + prow];
        dt[i] = p.dt[r * p.dt_rs + (int64_t)it.h * p.dt_hs + (int64_t)prow * p.dt_ds];
        A[i] = p.A[(int64_t)it.h * p.A_s + (int64_t)prow * p.A_ds];
        D[i] = p.D ? p.D[(int64_t)it.h * p.D_s + (int64_t)prow * p.D_ds] : 0.0f;
        bias[i] = p.dt_bias ? p.dt_bias[(int64_t)it.h * p.bias_s + (int64_t)prow * p.bias_ds]
                            : 0.0f;
      }
    }
  }

  // Convert and write the loaded values into a staging buffer (the same
  // values stage_vectors computes).
  __device__ __forceinline__ void commit(Stage<N, ROWS, LMAX>& s, const KParams& p, int p0,
                                         int tid) const {
#pragma unroll
    for (int i = 0; i < BCPT; ++i) {
      const int e = tid + i * NTHR;
      if (e < n * 2 * N) {
        const int tt = e / (2 * N), k = e - tt * 2 * N;
        if (k < N) s.B[tt][bc_slot<ST, N>(k)] = io_to_float<IT>(bc[i]);
        else s.C[tt][bc_slot<ST, N>(k - N)] = io_to_float<IT>(bc[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int e = tid + i * NTHR;
      if (e < n * ROWS) {
        const int tt = e / ROWS, j = e - tt * ROWS;
        float dA = 1.0f, dtx = 0.0f, Dx = 0.0f, gate = 1.0f;
        if (p0 + j < p.P) {
          const float xv = io_to_float<IT>(x[i]);
          float dtv = dt[i] + bias[i];
          if (p.softplus) dtv = softplus_f(dtv);
          dA = expf(A[i] * dtv);
          dtx = dtv * xv;
          Dx = D[i] * xv;
          if (p.z) {
            const float zv = io_to_float<IT>(z[i]);
            gate = zv / (1.0f + expf(-zv));
          }
        }
        s.dA[tt][j] = dA;
        s.dtx[tt][j] = dtx;
        s.Dx[tt][j] = Dx;
        s.gate[tt][j] = gate;
      }
    }
  }
};

// What the producer publishes with each item (besides the tile and operands).
template <int LMAX>
struct __align__(16) ItemRec {
  int64_t r0;           // first packed row
  int64_t dst[LMAX];    // write slot of staged step t (valid where bit t of wmask is set)
  int32_t h, p0, len;   // head, first tile row, rows of the sequence
  int32_t read_ok;      // the tile holds the read slot's state (else zeros)
  int32_t wmask;        // bit t: step t writes its state
  int32_t pad_[3];
};

template <class ST, class IT, int N, int WARPS, int UNR, int S, int SV, int LMAX>
struct BulkConfig {
  using L = RowLayout<ST, N>;
  static constexpr int ROWS = WARPS * L::RPW * UNR;
  static constexpr int CONSUMERS = WARPS * 32;
  static constexpr int THREADS = CONSUMERS + 32;  // + one producer warp
  static constexpr int STAGE_BYTES = ROWS * N * (int)sizeof(ST);
  using Vec = Stage<N, ROWS, LMAX>;
  using Rec = ItemRec<LMAX>;
  static constexpr int VEC_OFF = S * STAGE_BYTES;                  // SV operand buffers
  static constexpr int REC_OFF = VEC_OFF + SV * (int)sizeof(Vec);  // S item records
  static constexpr int BAR_OFF = REC_OFF + S * (int)sizeof(Rec);
  static constexpr int SMEM = BAR_OFF + (2 * S + SV) * 8;
  static_assert(STAGE_BYTES % 16 == 0 && sizeof(Vec) % 16 == 0, "16-byte stage alignment");
};

// The persistent pipeline.  Producer warp (32 lanes), for item k of this CTA:
//   resolve the item (one item ahead: its index loads are in flight while the
//   warp waits), wait until stage k % S is free, publish the item record and
//   start the tile's bulk copy (first arrival on full[s], with the byte count),
//   wait until operand buffer k % SV is free, convert the operands it loaded one
//   item earlier into it, arrive on full[s] a second time, then issue the loads
//   of the next item's operands.
// Consumer warps: wait full[s], read the record and their rows of the tile,
//   release the tile (empty_tile[s]) at once, run the steps on the buffered
//   operands, release the operand buffer (empty_vec[v]).  They meet only for
//   the rare chains longer than LMAX steps (re-staging the buffer).
template <class ST, class IT, int N, int WARPS, int UNR, int S, int SV, int LMAX, bool VARLEN>
__global__ void __launch_bounds__(WARPS * 32 + 32,
                                  (WARPS * RowLayout<ST, N>::RPW * UNR * N * sizeof(ST) <= 16384)
                                      ? 3
                                      : 2)
    ssu_bulk_kernel(const KParams p, const OneTokenArgs oa, const VarlenArgs va, int64_t nitems,
                    unsigned* err) {
  using Cfg = BulkConfig<ST, IT, N, WARPS, UNR, S, SV, LMAX>;
  using L = typename Cfg::L;
  using Vec = typename Cfg::Vec;
  using Rec = typename Cfg::Rec;
  constexpr int ROWS = Cfg::ROWS;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* bufs = smem;
  Vec* vring = reinterpret_cast<Vec*>(smem + Cfg::VEC_OFF);
  Rec* recs = reinterpret_cast<Rec*>(smem + Cfg::REC_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  uint64_t* empty_tile = full + S;
  uint64_t* empty_vec = full + 2 * S;
  __shared__ int s_issued[S];  // last round whose copy was issued on each stage (-1: none)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 2);          // producer: record + copy armed; operands staged
      mbar_init(&empty_tile[s], WARPS);
      s_issued[s] = -1;
    }
    for (int v = 0; v < SV; ++v) mbar_init(&empty_vec[v], WARPS);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int64_t block_elems = (int64_t)p.P * N;

  if (warp == WARPS) {
    // ---------------------------- producer warp ----------------------------
    int64_t idx = blockIdx.x;
    if (idx >= nitems) return;
    VecPrefetch<ST, IT, N, ROWS, LMAX, 32> pf;
    Item cur = resolve_item<VARLEN, ROWS>(p, oa, va, idx);
    pf.issue(p, cur, min(cur.len, LMAX), lane);
    for (int64_t k = 0; idx < nitems; idx += gridDim.x, ++k) {
      const int64_t nidx = idx + gridDim.x;
      Item next;
      if (nidx < nitems) next = resolve_item<VARLEN, ROWS>(p, oa, va, nidx);
      const int s = (int)(k % S);
      const int v = (int)(k % SV);
      // the item record: write slots of the staged steps
      Rec rec;
      rec.r0 = cur.r0;
      rec.h = cur.h;
      rec.p0 = cur.p0;
      rec.len = cur.len;
      rec.read_ok = cur.read_ok;
      rec.wmask = 0;
#pragma unroll
      for (int t = 0; t < LMAX; ++t) {
        int64_t d = -1;
        bool w = false;
        if (t < cur.len && cur.read_ok && !p.disable) {
          if constexpr (VARLEN) {
            const TableArgs dtab = va.dst.idx ? va.dst : va.src;
            if (dtab.idx) w = table_entry(dtab, cur.seq, t, va.idx64, &d);
            else { d = cur.seq; w = true; }
          } else {
            d = cur.dst;
            w = true;
          }
          w = w && slot_ok(d, p.pad, p.slots);
        }
        rec.dst[t] = d;
        if (w) rec.wmask |= 1 << t;
      }
      if (k >= S && !mbar_wait(&empty_tile[s], (uint32_t)((k / S) - 1) & 1)) {
        if (lane == 0) atomicOr(err, kErrEmptyTimeout);
        break;
      }
      if (lane == 0) {
        recs[s] = rec;
        if (cur.read_ok) {
          const int nrows = min(ROWS, p.P - cur.p0);
          const uint32_t bytes = (uint32_t)(nrows * N * (int)sizeof(ST));
          const ST* src = static_cast<const ST*>(p.state) +
                          ((cur.src * p.H + cur.h) * block_elems + (int64_t)cur.p0 * N);
          s_issued[s] = (int)(k / S);
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_load(bufs + (size_t)s * Cfg::STAGE_BYTES, src, bytes, &full[s]);
        } else {
          mbar_arrive(&full[s]);
        }
      }
      if (k >= SV && !mbar_wait(&empty_vec[v], (uint32_t)((k / SV) - 1) & 1)) {
        if (lane == 0) atomicOr(err, kErrEmptyTimeout);
        break;
      }
      pf.commit(vring[v], p, cur.p0, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
      if (nidx < nitems) {
        pf.issue(p, next, min(next.len, LMAX), lane);
        cur = next;
      }
    }
    // after an abort, let the copies this CTA issued land before it leaves
    if (lane == 0 && (*(volatile unsigned*)err & kErrEmptyTimeout)) {
      for (int t = 0; t < S; ++t) {
        const int r = *(volatile int*)&s_issued[t];
        if (r < 0) continue;
        const uint64_t t0 = global_ns();
        while (!mbar_test(&full[t], (uint32_t)r & 1) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    return;
  }

  // ---------------------------- consumer warps ----------------------------
  const int q = lane % L::LPR;
  const int rr = lane / L::LPR;
  const int jbase = warp * UNR * L::RPW + rr;  // this thread's first row in a tile
  ST* state = static_cast<ST*>(p.state);
  int64_t k = 0;
  for (int64_t idx = blockIdx.x; idx < nitems; idx += gridDim.x, ++k) {
    const int s = (int)(k % S);
    const int v = (int)(k % SV);
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (uint32_t)(k / S) & 1))) {
      if (lane == 0) atomicOr(err, kErrFullTimeout);
      return;
    }
    const Rec& rec = recs[s];
    const int64_t r0 = rec.r0;
    const int h = rec.h, p0 = rec.p0, len = rec.len, wmask = rec.wmask;
    const bool read_ok = rec.read_ok != 0;
    int64_t dsts[LMAX];
#pragma unroll
    for (int t = 0; t < LMAX; ++t) dsts[t] = rec.dst[t];
    // this thread's rows of the tile, widened to fp32; then release the tile
    float2 hs[UNR][L::EPL / 2];
    const unsigned char* buf = bufs + (size_t)s * Cfg::STAGE_BYTES;
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int j = jbase + u * L::RPW;
      const bool rd = read_ok && p0 + j < p.P;
#pragma unroll
      for (int c = 0; c < L::CPL; ++c) {
        const uint4 raw =
            rd ? *reinterpret_cast<const uint4*>(buf + ((size_t)j * N + (q + c * L::LPR) * L::VEC) *
                                                           sizeof(ST))
               : make_uint4(0u, 0u, 0u, 0u);
        Elem<ST>::unpack2(raw, &hs[u][c * L::VEC / 2]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_tile[s]);

    Vec& stg = vring[v];
    for (int t0 = 0; t0 < len; t0 += LMAX) {
      const int n = (len - t0) < LMAX ? (len - t0) : LMAX;
      int wm = wmask;
      if (t0 > 0) {
        // a chain longer than LMAX: the consumers re-stage the buffer together
        Item it;
        it.h = h;
        it.p0 = p0;
        it.r0 = r0;
        it.seq = p.fd_H.div(p.fd_tiles.div((uint32_t)idx));
        named_sync(1, Cfg::CONSUMERS);
        stage_vectors<ST, IT, N, ROWS, LMAX>(stg, p, it, t0, n, threadIdx.x, Cfg::CONSUMERS);
        named_sync(1, Cfg::CONSUMERS);
        wm = 0;
#pragma unroll
        for (int i = 0; i < LMAX; ++i) {
          int64_t d = -1;
          bool w = false;
          if (i < n && read_ok && !p.disable) {
            if constexpr (VARLEN) {
              const TableArgs dtab = va.dst.idx ? va.dst : va.src;
              if (dtab.idx) w = table_entry(dtab, it.seq, t0 + i, va.idx64, &d);
              else { d = it.seq; w = true; }
            }
            w = w && slot_ok(d, p.pad, p.slots);
          }
          dsts[i] = d;
          if (w) wm |= 1 << i;
        }
      }
#pragma unroll
      for (int tt = 0; tt < LMAX; ++tt) {
        if (tt >= n) break;
        step_rows<ST, IT, N, UNR>(hs, stg, tt, q, jbase, p, h, p0, r0 + t0 + tt);
        if ((wm >> tt) & 1) {
          ST* base = state + ((dsts[tt] * p.H + h) * block_elems);
#pragma unroll
          for (int u = 0; u < UNR; ++u) {
            const int prow = p0 + jbase + u * L::RPW;
            if (prow < p.P) {
#pragma unroll
              for (int c = 0; c < L::CPL; ++c)
                store_state<ST>(state, base - state + (int64_t)prow * N + (q + c * L::LPR) * L::VEC,
                                &hs[u][c * L::VEC / 2], p);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_vec[v]);
  }
}

// ---------------------------------------------------------------------------
// Variant with consumer-staged operands: the producer thread only resolves
// slots and issues tile copies; the consumer warps stage each item's per-step
// operands together (one round of loads, prefetched one item ahead, published
// through a per-item named barrier of the consumer warps).  It wins where the
// per-row operand work is large against the tile's bytes (16-bit state, calls
// that write no state); the producer-staged kernel above wins elsewhere.
// ---------------------------------------------------------------------------
template <class ST, class IT, int N, int WARPS, int UNR, int S, int LMAX>
struct BulkCsConfig {
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
    ssu_bulk_cs_kernel(const KParams p, const OneTokenArgs oa, const VarlenArgs va, int64_t nitems,
                    unsigned* err) {
  using Cfg = BulkCsConfig<ST, IT, N, WARPS, UNR, S, LMAX>;
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
  const int ctid = threadIdx.x;  // 0 .. CONSUMERS-1

  // the position of item idx (no slot loads: the producer resolves those);
  // for the packed route `cu0` / `cu1` are the sequence's cu_seqlens entries
  auto position = [&](int64_t idx, int64_t cu0, int64_t cu1) {
    Item it;
    int tile;
    split_index(p, (uint32_t)idx, &it.seq, &it.h, &tile);
    it.p0 = tile * ROWS;
    if constexpr (VARLEN) {
      int64_t begin = cu0, end = cu1;
      if (begin < 0) begin = 0;
      if (end > va.rows) end = va.rows;
      it.r0 = begin;
      it.len = end > begin ? (int)(end - begin) : 0;
    } else {
      it.r0 = it.seq;
      it.len = 1;
    }
    it.src = it.dst = -1;
    it.read_ok = false;
    return it;
  };
  auto seq_bounds = [&](int64_t idx, int64_t* cu0, int64_t* cu1) {
    if constexpr (VARLEN) {
      const int64_t seq = p.fd_H.div(p.fd_tiles.div((uint32_t)idx));
      if (va.cu) {
        *cu0 = load_int(va.cu, seq, va.meta64);
        *cu1 = load_int(va.cu, seq + 1, va.meta64);
      } else {
        *cu0 = seq * va.dense_steps;
        *cu1 = *cu0 + va.dense_steps;
      }
    } else {
      *cu0 = *cu1 = 0;
    }
  };

  VecPrefetch<ST, IT, N, ROWS, LMAX, Cfg::CONSUMERS> pf;
  int64_t idx = blockIdx.x;
  Item it_next;
  if (idx < nitems) {  // prologue: the first item's operands
    int64_t c0, c1;
    seq_bounds(idx, &c0, &c1);
    it_next = position(idx, c0, c1);
    pf.issue(p, it_next, min(it_next.len, LMAX), ctid);
    pf.commit(vecs[0], p, it_next.p0, ctid);
  }
  int64_t k = 0;
  for (; idx < nitems; idx += gridDim.x, ++k) {
    const int s = (int)(k % S);
    const uint32_t round = (uint32_t)(k / S);
    Vec& stg = vecs[k & 1];
    Item it = it_next;
    const int64_t nidx = idx + gridDim.x;
    int64_t nc0 = 0, nc1 = 0;
    if (nidx < nitems) seq_bounds(nidx, &nc0, &nc1);  // in flight during the wait
    if (!mbar_wait(&full[s], round & 1)) s_abort = 1;
    named_sync(1, Cfg::CONSUMERS);  // also publishes stg (committed last iteration)
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
    float2 hs[UNR][L::EPL / 2];
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
        Elem<ST>::unpack2(raw, &hs[u][c * L::VEC / 2]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    // the next item's operands: loads in flight while this item computes
    if (nidx < nitems) {
      it_next = position(nidx, nc0, nc1);
      pf.issue(p, it_next, min(it_next.len, LMAX), ctid);
    }

    for (int t0 = 0; t0 < it.len; t0 += LMAX) {
      const int n = (it.len - t0) < LMAX ? (it.len - t0) : LMAX;
      if (t0 > 0) {
        named_sync(1, Cfg::CONSUMERS);
        stage_vectors<ST, IT, N, ROWS, LMAX>(stg, p, it, t0, n, ctid, Cfg::CONSUMERS);
        named_sync(1, Cfg::CONSUMERS);
      }
      // this chunk's write slots, loaded together ahead of the stores
      int64_t dsts[LMAX];
      bool dok[LMAX];
#pragma unroll
      for (int i = 0; i < LMAX; ++i) {
        dsts[i] = -1;
        dok[i] = false;
        if (i < n) {
          if constexpr (VARLEN) {
            const TableArgs dtab = va.dst.idx ? va.dst : va.src;
            if (dtab.idx) {
              int64_t v = -1;
              dok[i] = table_entry(dtab, it.seq, t0 + i, va.idx64, &v);
              dsts[i] = v;
            } else {
              dsts[i] = it.seq;
              dok[i] = true;
            }
          } else {
            dsts[i] = it.dst;
            dok[i] = true;
          }
          dok[i] = dok[i] && it.read_ok && !p.disable && slot_ok(dsts[i], p.pad, p.slots);
        }
      }
#pragma unroll
      for (int tt = 0; tt < LMAX; ++tt) {
        if (tt >= n) break;
        step_rows<ST, IT, N, UNR>(hs, stg, tt, q, warp * UNR * L::RPW + rr, p, it.h, it.p0,
                                  it.r0 + t0 + tt);
        // this step's state
        if (dok[tt]) {
          ST* base = state + ((dsts[tt] * p.H + it.h) * block_elems);
#pragma unroll
          for (int u = 0; u < UNR; ++u) {
            const int prow = it.p0 + (warp * UNR + u) * L::RPW + rr;
            if (prow < p.P) {
#pragma unroll
              for (int c = 0; c < L::CPL; ++c)
                store_state<ST>(state, base - state + (int64_t)prow * N + (q + c * L::LPR) * L::VEC,
                                &hs[u][c * L::VEC / 2], p);
            }
          }
        }
      }
    }
    // publish the next item's operands (every consumer left vecs[(k + 1) & 1]
    // behind when it passed this item's barrier)
    if (nidx < nitems) pf.commit(vecs[(k + 1) & 1], p, it_next.p0, ctid);
  }
}

}  // namespace ssu
