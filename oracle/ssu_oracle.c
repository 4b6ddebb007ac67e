/*
 * ssu_oracle.c -- plain, slow, fp64 CPU oracle for the Mamba2 selective state
 * update (SSU) decode step and the ReplaySSM ring trackers.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library; both are written against the same pages.
 *
 * Sources (page title and section):
 *   - "vllm.model_executor.layers.mamba.ops.ssu_dispatch" (vLLM API docs and
 *     the raw ssu_dispatch.py listing): the unified selective_state_update
 *     call contract (state, x, dt, A, B, C, D, dt_bias, z, dt_softplus, slot
 *     tables, null_block_id, num_accepted_tokens, cu_seqlens) and the two
 *     ReplaySSM tracker kernels (_update_replayssm_ring_trackers_kernel,
 *     _commit_replayssm_ring_trackers_kernel).
 *   - "mate.mamba" (MATE module source): selective_state_update's
 *     FlashInfer-shaped contract -- state [slots, heads, dim, dstate], packed
 *     x [rows, heads, dim], B/C [rows, groups, dstate], per-head A/D/dt_bias,
 *     pad_slot_id, disable_state_update, the packed varlen route
 *     (_packed_selective_state_update) and slot-table addressing (_slot_table:
 *     entry = seq * seq_stride + pos * step_stride).
 *   - The recurrence itself, which the pages name but never print, is the
 *     standard Mamba2 decode step:
 *         dt' = dt + dt_bias;  dt' = softplus(dt') if dt_softplus
 *         dA  = exp(A[h] * dt')
 *         h[p][n] <- h[p][n] * dA + dt' * x[p] * B[g][n]
 *         y[p] = sum_n h[p][n] * C[g][n] + D[h] * x[p];  y *= silu(z[p])
 *     with g = h / (heads / groups).
 *
 * A, D and dt_bias are per head ([H], "mate.mamba" _per_head's tied form) or,
 * flagged per parameter, per (head, dim) channel ([H, P], _per_head's
 * channel-wise form).
 *
 * Everything is evaluated in IEEE double from the exact stored input values
 * (bf16 / fp16 / fp32 inputs widen exactly).  Stored state is rounded once,
 * round-to-nearest-even, from the double value to the state dtype.  A chained
 * multi-token run keeps the unrounded double state between its steps.
 *
 * Readings where the pages are silent are listed at each function.  The
 * ReplaySSM checkpointing update (oracle_replay_update, at the end) reuses
 * ssu_step for every replayed and every new token.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes used by this file's interface (its own; not shared).  OR_F64 is
 * accepted for the state only: an fp64 pool (rounding is then the identity)
 * lets the pins compare chains that store state with chains that do not, bit
 * for bit. */
enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2, OR_F64 = 3 };

/* ------------------------------------------------------------------------ */
/* exact widening of stored values                                          */
/* ------------------------------------------------------------------------ */

static double bf16_bits_to_double(uint16_t b) {
  /* bf16 is the top half of an IEEE binary32 */
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double f16_bits_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 10) & 0x1f;
  int m = b & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

static double load_value(const void* base, int64_t i, int dtype) {
  switch (dtype) {
    case OR_F32: return (double)((const float*)base)[i];
    case OR_BF16: return bf16_bits_to_double(((const uint16_t*)base)[i]);
    case OR_F16: return f16_bits_to_double(((const uint16_t*)base)[i]);
    case OR_F64: return ((const double*)base)[i];
  }
  return NAN;
}

/* ------------------------------------------------------------------------ */
/* round-to-nearest-even from double to a binary format                     */
/* ------------------------------------------------------------------------ */

/*
 * Round |v| to `prec` significant bits with minimum normal exponent `emin`
 * (below it the quantum stays 2^(emin-prec+1): gradual underflow) and
 * overflow to infinity above `maxfinite`.  nearbyint() rounds in the default
 * mode, round-to-nearest ties-to-even; dividing by a power of two is exact.
 */
static double round_to_precision(double v, int prec, int emin, double maxfinite) {
  if (v == 0.0 || isnan(v) || isinf(v)) return v;
  int e;
  (void)frexp(fabs(v), &e); /* |v| in [2^(e-1), 2^e) */
  int E = e - 1;
  if (E < emin) E = emin;
  double quantum = ldexp(1.0, E - (prec - 1));
  double r = nearbyint(fabs(v) / quantum) * quantum;
  if (r > maxfinite) r = INFINITY;
  return copysign(r, v);
}

/* value of the bf16 (8 significant bits, emin -126) nearest to v */
double oracle_round_bf16(double v) {
  return round_to_precision(v, 8, -126, ldexp(255.0, 120)); /* (2-2^-7)*2^127 */
}

/* value of the fp16 (11 significant bits, emin -14) nearest to v */
double oracle_round_f16(double v) {
  return round_to_precision(v, 11, -14, 65504.0);
}

/* value of the fp32 nearest to v (the C conversion rounds to nearest even) */
double oracle_round_f32(double v) { return (double)(float)v; }

static uint16_t exact_double_to_bf16_bits(double r) {
  /* r is already a bf16 value, hence exact in binary32 */
  float f = (float)r;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

static uint16_t exact_double_to_f16_bits(double r) {
  /* r is already an fp16 value: encode its sign, exponent and significand */
  uint16_t sign = signbit(r) ? 0x8000 : 0;
  double a = fabs(r);
  if (isnan(r)) return 0x7e00;
  if (isinf(a)) return sign | 0x7c00;
  if (a == 0.0) return sign;
  if (a < ldexp(1.0, -14)) { /* subnormal: a = m * 2^-24 */
    return sign | (uint16_t)(a / ldexp(1.0, -24));
  }
  int e;
  double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  int biased = e - 1 + 15;
  uint16_t frac = (uint16_t)((m * 2.0 - 1.0) * 1024.0);
  return sign | (uint16_t)(biased << 10) | frac;
}

static void store_rounded(void* base, int64_t i, int dtype, double v) {
  switch (dtype) {
    case OR_F32: ((float*)base)[i] = (float)v; break;
    case OR_BF16: ((uint16_t*)base)[i] = exact_double_to_bf16_bits(oracle_round_bf16(v)); break;
    case OR_F16: ((uint16_t*)base)[i] = exact_double_to_f16_bits(oracle_round_f16(v)); break;
    case OR_F64: ((double*)base)[i] = v; break;
  }
}

/* ------------------------------------------------------------------------ */
/* stochastic rounding of 16-bit state                                      */
/* ------------------------------------------------------------------------ */

/*
 * Philox4x64 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 * as 1, 2, 3", SC'11): a counter of four 64-bit words and a key of two are
 * mixed by `rounds` rounds; a round multiplies words 0 and 2 by two fixed
 * 64-bit constants, takes the 128-bit products' high and low halves, xors
 * the high halves with the other two words and the key, and permutes; the
 * key advances by two fixed Weyl increments between rounds.  ("ssu_dispatch"
 * names the generator -- philox_rounds, default 10 -- and a random seed drawn
 * per call, not the variant or the counter layout: both are readings.)
 */
static void mul128(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
  /* schoolbook product of 32-bit halves: exact in 64-bit arithmetic */
  const uint64_t a0 = a & 0xffffffffu, a1 = a >> 32, b0 = b & 0xffffffffu, b1 = b >> 32;
  const uint64_t p00 = a0 * b0, p01 = a0 * b1, p10 = a1 * b0, p11 = a1 * b1;
  const uint64_t mid = (p00 >> 32) + (p01 & 0xffffffffu) + (p10 & 0xffffffffu);
  *lo = (mid << 32) | (p00 & 0xffffffffu);
  *hi = p11 + (p01 >> 32) + (p10 >> 32) + (mid >> 32);
}

void oracle_philox4x64(const uint64_t* counter, const uint64_t* key, int rounds,
                       uint64_t* out) {
  uint64_t x0 = counter[0], x1 = counter[1], x2 = counter[2], x3 = counter[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int i = 0; i < rounds; ++i) {
    uint64_t hi0, lo0, hi1, lo1;
    mul128(0xD2E7470EE14C6C93ull, x0, &hi0, &lo0);
    mul128(0xCA5A826395121157ull, x2, &hi1, &lo1);
    const uint64_t n0 = hi1 ^ x1 ^ k0, n1 = lo1, n2 = hi0 ^ x3 ^ k1, n3 = lo0;
    x0 = n0;
    x1 = n1;
    x2 = n2;
    x3 = n3;
    k0 += 0x9E3779B97F4A7C15ull; /* Weyl increments: golden ratio, sqrt(3) - 1 */
    k1 += 0xBB67AE8584CAA73Bull;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* The 16 random bits of stored element e (its index in the state pool) of a
 * call with `seed`: block e / 16 of the stream keyed by (seed, 0), word
 * (e / 4) mod 4 of it, bits 16 (e mod 4) .. 16 (e mod 4) + 15. */
uint32_t oracle_sr_bits(uint64_t seed, int rounds, int64_t e) {
  const uint64_t counter[4] = {(uint64_t)e >> 4, 0, 0, 0}, key[2] = {seed, 0};
  uint64_t out[4];
  oracle_philox4x64(counter, key, rounds, out);
  return (uint32_t)((out[((uint64_t)e >> 2) & 3] >> (16 * ((uint64_t)e & 3))) & 0xffffu);
}

/* Stochastic rounding of v to a binary format of `prec` significant bits and
 * minimum normal exponent `emin`: with q the format's spacing at |v| and
 * a = |v| / q, the result is q floor(a + r / 2^16) -- the upper neighbour
 * exactly when frac(a) >= 1 - r / 2^16, i.e. with probability frac(a) to 16
 * bits.  Representable values are unchanged; beyond the largest finite value
 * the result is infinite, as rounding makes it. */
static double sr_to_precision(double v, int prec, int emin, double maxfinite, uint32_t r) {
  if (v == 0.0 || isnan(v) || isinf(v)) return v;
  int e;
  (void)frexp(fabs(v), &e);
  int E = e - 1;
  if (E < emin) E = emin;
  const double q = ldexp(1.0, E - (prec - 1));
  const double a = fabs(v) / q; /* exact: a power-of-two scaling */
  const double fl = floor(a);
  const double frac = a - fl; /* exact */
  double t = fl + (frac >= 1.0 - ldexp((double)r, -16) ? 1.0 : 0.0);
  double m = t * q;
  if (m > maxfinite) m = INFINITY;
  return copysign(m, v);
}

double oracle_sr_bf16(double v, uint32_t r) {
  return sr_to_precision(v, 8, -126, ldexp(255.0, 120), r);
}

double oracle_sr_f16(double v, uint32_t r) { return sr_to_precision(v, 11, -14, 65504.0, r); }

/* Stochastic rounding of state writes: a call's random seed (NULL: round to
 * nearest even) and Philox rounds; only 16-bit state is affected. */
typedef struct {
  const uint64_t* seed;
  int rounds;
} sr_ctx;

static void store_state(void* base, int64_t i, int dtype, double v, const sr_ctx* sr) {
  if (!sr || !sr->seed || (dtype != OR_BF16 && dtype != OR_F16)) {
    store_rounded(base, i, dtype, v);
    return;
  }
  const uint32_t r = oracle_sr_bits(*sr->seed, sr->rounds, i);
  if (dtype == OR_BF16)
    ((uint16_t*)base)[i] = exact_double_to_bf16_bits(oracle_sr_bf16(v, r));
  else
    ((uint16_t*)base)[i] = exact_double_to_f16_bits(oracle_sr_f16(v, r));
}

/* Round an array of doubles to `dtype` and write the stored encoding. */
void oracle_encode(const double* v, int64_t n, int dtype, void* out) {
  for (int64_t i = 0; i < n; ++i) store_rounded(out, i, dtype, v[i]);
}

/* Widen an array of stored values to double. */
void oracle_decode(const void* in, int64_t n, int dtype, double* v) {
  for (int64_t i = 0; i < n; ++i) v[i] = load_value(in, i, dtype);
}

/* ------------------------------------------------------------------------ */
/* the recurrence                                                           */
/* ------------------------------------------------------------------------ */

static double softplus(double v) { return log1p(exp(v)); }

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* Operands of one call, shared by the one-token and packed routes. */
typedef struct {
  int64_t H, P, N, G;          /* heads, headdim, dstate, groups */
  const void* x; const void* z; int io_dtype;   /* [rows, H, P]; z may be NULL */
  const float* dt; int dt_per_dim;              /* [rows, H] or [rows, H, P] */
  const float* A; const float* D; const float* dt_bias;  /* [H]; D, dt_bias may be NULL */
  const void* B; const void* C;                 /* [rows, G, N], io dtype */
  int dt_softplus;
  int param_per_dim;  /* bit 0: A, bit 1: D, bit 2: dt_bias given per (head, dim) as [H, P] */
} operands;

/*
 * One decode step of head `h` on the state block hb[P][N] (double, updated in
 * place) for packed row `r`; writes y[r, h, :] as double.
 */
static void ssu_step(const operands* o, int64_t r, int64_t h, double* hb, double* y) {
  const int64_t H = o->H, P = o->P, N = o->N;
  const int64_t g = h / (H / o->G); /* heads of one group are contiguous */
  for (int64_t p = 0; p < P; ++p) {
    /* per head, or per (head, dim) channel ("mate.mamba", _per_head) */
    const double A = (o->param_per_dim & 1) ? o->A[h * P + p] : o->A[h];
    const double D = !o->D ? 0.0 : (o->param_per_dim & 2) ? o->D[h * P + p] : o->D[h];
    const double bias = !o->dt_bias ? 0.0
                        : (o->param_per_dim & 4) ? o->dt_bias[h * P + p] : o->dt_bias[h];
    double dt = o->dt_per_dim ? o->dt[(r * H + h) * P + p] : o->dt[r * H + h];
    dt += bias;
    if (o->dt_softplus) dt = softplus(dt);
    const double dA = exp(A * dt);
    const double xp = load_value(o->x, (r * H + h) * P + p, o->io_dtype);
    double acc = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const double Bn = load_value(o->B, (r * o->G + g) * N + n, o->io_dtype);
      const double Cn = load_value(o->C, (r * o->G + g) * N + n, o->io_dtype);
      double* hv = &hb[p * N + n];
      *hv = *hv * dA + dt * xp * Bn;
      acc += *hv * Cn;
    }
    double out = acc + D * xp;
    if (o->z) out *= silu(load_value(o->z, (r * H + h) * P + p, o->io_dtype));
    y[(r * H + h) * P + p] = out;
  }
}

static int slot_ok(int64_t slot, int64_t pad, int64_t slots) {
  return slot != pad && slot >= 0 && slot < slots;
}

/*
 * One-token decode (MATE's ssu_one_token route; vLLM's plain decode call).
 * Sequence b reads slot sbi[b] (b when sbi is NULL) and writes slot dsbi[b]
 * (the read slot when dsbi is NULL).
 * Readings: a read slot that is pad or outside [0, slots) makes the step run
 * from a zero state and write no state at all; a write slot that is pad or
 * outside [0, slots) skips only the write; disable_state_update skips every
 * state write.  y is always produced.
 */
int oracle_ssu_update(void* state, int state_dtype, int64_t slots,
                      int64_t H, int64_t P, int64_t N, int64_t G, int64_t batch,
                      const void* x, const void* z, int io_dtype,
                      const float* dt, int dt_per_dim,
                      const float* A, const float* D, const float* dt_bias,
                      const void* B, const void* C,
                      const int64_t* sbi, const int64_t* dsbi, int64_t pad_slot_id,
                      int dt_softplus, int disable_state_update, int param_per_dim, double* y,
                      const uint64_t* rand_seed, int philox_rounds) {
  if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0) return 1;
  operands o = {H, P, N, G, x, z, io_dtype, dt, dt_per_dim, A, D, dt_bias, B, C, dt_softplus,
                param_per_dim};
  const sr_ctx sr = {rand_seed, philox_rounds};
  const int64_t block = P * N;
  double* hb = (double*)malloc(sizeof(double) * (size_t)block);
  if (!hb) return 2;
  for (int64_t b = 0; b < batch; ++b) {
    const int64_t src = sbi ? sbi[b] : b;
    const int64_t dst = dsbi ? dsbi[b] : src;
    const int read_ok = slot_ok(src, pad_slot_id, slots);
    const int write_ok = read_ok && !disable_state_update && slot_ok(dst, pad_slot_id, slots);
    for (int64_t h = 0; h < H; ++h) {
      const int64_t in_off = (src * H + h) * block;
      for (int64_t i = 0; i < block; ++i)
        hb[i] = read_ok ? load_value(state, in_off + i, state_dtype) : 0.0;
      ssu_step(&o, b, h, hb, y);
      if (write_ok) {
        const int64_t out_off = (dst * H + h) * block;
        for (int64_t i = 0; i < block; ++i) store_state(state, out_off + i, state_dtype, hb[i], &sr);
      }
    }
  }
  free(hb);
  return 0;
}

/* entry `pos` of sequence `seq` in a slot table, or -1 when it has none */
static int64_t table_entry(const int64_t* tab, int64_t numel, int64_t seq_stride,
                           int64_t step_stride, int64_t steps, int64_t seq, int64_t pos,
                           int64_t* out) {
  if (pos < 0 || pos >= steps) return -1;
  int64_t e = seq * seq_stride + pos * step_stride;
  if (e < 0 || e >= numel) return -1;
  *out = tab[e];
  return 0;
}

/*
 * Packed variable-length (MTP) update (MATE's ssu_packed_varlen route and
 * _packed_selective_state_update; the dense [batch, steps, ...] form is the
 * same call with equal lengths).
 *
 * Sequence s owns packed rows [cu[s], cu[s+1]) (cu NULL: rows
 * [s*dense_steps, (s+1)*dense_steps)).  Its read slot is entry
 * (s, num_accepted[s] - 1) of the read table (column 0 without counts; slot s
 * without a table).  Step t writes its state to entry (s, t) of the write
 * table (of the read table when there is no write table; slot s when there is
 * neither).  The chain between steps keeps the unrounded double state.
 * Readings: an acceptance count whose column lies outside the table, or a
 * read slot that is pad or outside [0, slots), runs the sequence from a zero
 * state and writes no state; a step whose write entry is missing, pad or out
 * of range skips that write only; rows outside [0, rows) are not touched.
 */
int oracle_ssu_update_varlen(void* state, int state_dtype, int64_t slots,
                             int64_t H, int64_t P, int64_t N, int64_t G,
                             int64_t nseqs, int64_t rows,
                             const void* x, const void* z, int io_dtype,
                             const float* dt, int dt_per_dim,
                             const float* A, const float* D, const float* dt_bias,
                             const void* B, const void* C,
                             const int64_t* cu_seqlens, int64_t dense_steps,
                             const int64_t* num_accepted,
                             const int64_t* src_tab, int64_t src_numel, int64_t src_ss,
                             int64_t src_ts, int64_t src_steps,
                             const int64_t* dst_tab, int64_t dst_numel, int64_t dst_ss,
                             int64_t dst_ts, int64_t dst_steps,
                             int64_t pad_slot_id, int dt_softplus, int disable_state_update,
                             int param_per_dim, double* y, const uint64_t* rand_seed,
                             int philox_rounds) {
  if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0) return 1;
  operands o = {H, P, N, G, x, z, io_dtype, dt, dt_per_dim, A, D, dt_bias, B, C, dt_softplus,
                param_per_dim};
  const sr_ctx sr = {rand_seed, philox_rounds};
  const int64_t block = P * N;
  double* hb = (double*)malloc(sizeof(double) * (size_t)block);
  if (!hb) return 2;
  for (int64_t s = 0; s < nseqs; ++s) {
    int64_t begin = cu_seqlens ? cu_seqlens[s] : s * dense_steps;
    int64_t end = cu_seqlens ? cu_seqlens[s + 1] : (s + 1) * dense_steps;
    if (begin < 0) begin = 0;
    if (end > rows) end = rows;
    if (end <= begin) continue; /* an empty sequence reads and writes nothing */

    /* read slot */
    int64_t src = s;
    int read_ok = 1;
    if (src_tab) {
      const int64_t col = num_accepted ? num_accepted[s] - 1 : 0;
      if (table_entry(src_tab, src_numel, src_ss, src_ts, src_steps, s, col, &src) != 0)
        read_ok = 0;
    }
    read_ok = read_ok && slot_ok(src, pad_slot_id, slots);

    for (int64_t h = 0; h < H; ++h) {
      const int64_t in_off = (src * H + h) * block;
      for (int64_t i = 0; i < block; ++i)
        hb[i] = read_ok ? load_value(state, in_off + i, state_dtype) : 0.0;
      for (int64_t t = 0; t < end - begin; ++t) {
        ssu_step(&o, begin + t, h, hb, y);
        if (!read_ok || disable_state_update) continue;
        int64_t dst = s;
        int have = 1;
        if (dst_tab)
          have = table_entry(dst_tab, dst_numel, dst_ss, dst_ts, dst_steps, s, t, &dst) == 0;
        else if (src_tab)
          have = table_entry(src_tab, src_numel, src_ss, src_ts, src_steps, s, t, &dst) == 0;
        if (!have || !slot_ok(dst, pad_slot_id, slots)) continue;
        const int64_t out_off = (dst * H + h) * block;
        for (int64_t i = 0; i < block; ++i) store_state(state, out_off + i, state_dtype, hb[i], &sr);
      }
    }
  }
  free(hb);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* ReplaySSM ring trackers                                                  */
/* ------------------------------------------------------------------------ */

/* int32 arithmetic of the tracker kernels: two's-complement wrap-around */
static int32_t add_i32(int32_t a, int32_t b) { return (int32_t)((uint32_t)a + (uint32_t)b); }

static int64_t min3(int64_t a, int64_t b, int64_t c) {
  int64_t m = a < b ? a : b;
  return m < c ? m : c;
}

/*
 * _update_replayssm_ring_trackers_kernel ("ssu_dispatch", ReplaySSM tracker
 * update).  For sequence i the tracker slot is sbi[i * sbi_stride] (column 0
 * of a 2-D table).  A slot is valid when it is not the pad id and lies in
 * [0, num_states), num_states being the shortest of the three arrays.
 * Reset zeroes all three trackers of a valid slot.  Otherwise, with
 * prev = prev_num_accepted[slot] and start = ring_start[slot]: when one more
 * token would exceed the logical window the ring starts a new checkpoint at
 * (start + prev) mod ring_buffer_len and the count restarts at 1; else the
 * count grows by one.  prev_query_len is left alone.  `%` is C's truncating
 * remainder, the int32 sums wrap.
 */
int oracle_ring_update(int32_t* ring_start, int64_t n_ring_start,
                       int32_t* prev_num_accepted, int64_t n_prev_num_accepted,
                       int32_t* prev_query_len, int64_t n_prev_query_len,
                       const int64_t* sbi, int64_t sbi_stride, int64_t nseqs,
                       int reset, int32_t logical_window, int32_t ring_buffer_len,
                       int64_t pad_slot_id) {
  const int64_t num_states = min3(n_ring_start, n_prev_num_accepted, n_prev_query_len);
  if (!reset && ring_buffer_len <= 0) return 1;
  for (int64_t i = 0; i < nseqs; ++i) {
    const int64_t slot = sbi[i * sbi_stride];
    if (!(slot != pad_slot_id && slot >= 0 && slot < num_states)) continue;
    if (reset) {
      ring_start[slot] = 0;
      prev_num_accepted[slot] = 0;
      prev_query_len[slot] = 0;
      continue;
    }
    const int32_t prev = prev_num_accepted[slot];
    const int32_t start = ring_start[slot];
    const int must_checkpoint = add_i32(prev, 1) > logical_window;
    ring_start[slot] = must_checkpoint ? add_i32(start, prev) % ring_buffer_len : start;
    prev_num_accepted[slot] = must_checkpoint ? 1 : add_i32(prev, 1);
  }
  return 0;
}

/*
 * _commit_replayssm_ring_trackers_kernel ("ssu_dispatch", commit of the
 * previous speculative window).  For a valid slot (as above) of sequence i:
 * acc = prev_num_accepted[slot], start = ring_start[slot],
 * pql = prev_query_len[slot], a = num_accepted[i] (per sequence).  A window
 * is committed only when a previous MTP query exists (pql > 0); it
 * checkpoints when acc + pql exceeds the logical window, moving the ring start
 * by acc.  The new count is 0 with no previous query, a after a checkpoint,
 * acc + a otherwise; prev_query_len records this query's length
 * qsl[i+1] - qsl[i].  Values stored into the int32 trackers wrap to 32 bits.
 */
int oracle_ring_commit(int32_t* ring_start, int64_t n_ring_start,
                       int32_t* prev_num_accepted, int64_t n_prev_num_accepted,
                       int32_t* prev_query_len, int64_t n_prev_query_len,
                       const int64_t* sbi, int64_t sbi_stride,
                       const int64_t* num_accepted, const int64_t* query_start_loc,
                       int64_t nseqs, int32_t logical_window, int32_t ring_buffer_len,
                       int64_t pad_slot_id) {
  const int64_t num_states = min3(n_ring_start, n_prev_num_accepted, n_prev_query_len);
  if (ring_buffer_len <= 0) return 1;
  for (int64_t i = 0; i < nseqs; ++i) {
    const int64_t slot = sbi[i * sbi_stride];
    if (!(slot != pad_slot_id && slot >= 0 && slot < num_states)) continue;
    const int32_t acc = prev_num_accepted[slot];
    const int32_t start = ring_start[slot];
    const int32_t pql = prev_query_len[slot];
    const int32_t a = (int32_t)(uint32_t)(uint64_t)num_accepted[i];
    const int must_checkpoint = pql > 0 && add_i32(acc, pql) > logical_window;
    const int32_t next_start = must_checkpoint ? add_i32(start, acc) % ring_buffer_len : start;
    const int32_t next_prev = pql == 0 ? 0 : (must_checkpoint ? a : add_i32(acc, a));
    const int32_t qlen = (int32_t)(uint32_t)(uint64_t)(query_start_loc[i + 1] - query_start_loc[i]);
    ring_start[slot] = next_start;
    prev_num_accepted[slot] = next_prev;
    prev_query_len[slot] = qlen;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* ReplaySSM checkpointing update                                           */
/* ------------------------------------------------------------------------ */

/*
 * ReplaySSM ("ssu_dispatch": selective_state_update_replayssm_flashinfer, the
 * FlashInfer checkpointing_ssu call it wraps, and the ring semantics of the
 * tracker kernels above).  The pages fix the interface -- a checkpoint
 * `state`, per-slot rings x_cache / B_cache / dt_cache of ring_len positions,
 * ring_start and prev_num_accepted per slot, a logical window -- and where the
 * trackers move the ring, not the arithmetic.  Readings:
 *
 *  - the logical state of a slot is its checkpoint state[slot] advanced, in
 *    order, through the k = prev_num_accepted[slot] cached tokens at ring
 *    positions (ring_start[slot] + j) mod ring_len, j < k; a cached token is
 *    x [H, P], B [G, N] and dt [H] as the caller gave them (dt before dt_bias
 *    and softplus), and its step is the plain step of ssu_step with the call's
 *    A, dt_bias and dt_softplus;
 *  - the call's L rows of the sequence continue the chain from the logical
 *    state (y from the unrounded state, as in the plain calls); row t is cached
 *    at position (ring_start + k + t) mod ring_len;
 *  - when k + L exceeds the logical window, the state after the k replayed
 *    tokens -- the state the trackers' new ring start (ring_start + k) names --
 *    is rounded to the state dtype and written to state[slot];
 *  - a sequence is processed when its slot is neither the pad id nor outside
 *    [0, min(slots, num_states)), it has at least one row, and its trackers are
 *    in range (0 <= k, k + L <= ring_len, 0 <= ring_start < ring_len); any
 *    other sequence runs its rows from a zero state and writes nothing;
 *  - update_trackers applies the one-token tracker rule of
 *    oracle_ring_update (what the wrapper runs after the kernel) to the slot of
 *    every processed sequence, after the call.
 *
 * Layouts (contiguous): x_cache, B_cache in the io dtype, [slots, H, R, P] and
 * [slots, G, R, N]; dt_cache fp32 [slots, H, R]; R = ring_len.  dt is per head
 * [rows, H].  Rows of sequence s: [cu[s], cu[s+1]), or the single row s when
 * cu_seqlens is NULL.  Read/write slot of sequence s: sbi[s] (s when NULL).
 */
static void copy_io(void* dst, int64_t di, const void* src, int64_t si, int io_dtype) {
  (void)io_dtype; /* bf16 and fp16 both move as 16-bit patterns */
  ((uint16_t*)dst)[di] = ((const uint16_t*)src)[si];
}

static int replay_ok(int64_t slot, int64_t pad, int64_t limit, int32_t k, int32_t start,
                     int64_t L, int64_t R) {
  return slot != pad && slot >= 0 && slot < limit && L > 0 && k >= 0 && start >= 0 &&
         start < R && (int64_t)k + L <= R;
}

/* Advance hb (head h of `slot`) through the cached token at ring position pos:
 * the token's x, B, dt become a one-row operand set and take one plain step. */
static void replay_token(const operands* o, int64_t h, const void* x_cache, const void* B_cache,
                         const float* dt_cache, int64_t slot, int64_t pos, int64_t R,
                         void* xrow, void* Brow, float* dtrow, double* ydump, double* hb) {
  const int64_t H = o->H, P = o->P, N = o->N, G = o->G;
  const int64_t g = h / (H / G);
  for (int64_t p = 0; p < P; ++p) copy_io(xrow, h * P + p, x_cache, ((slot * H + h) * R + pos) * P + p, o->io_dtype);
  for (int64_t n = 0; n < N; ++n) copy_io(Brow, g * N + n, B_cache, ((slot * G + g) * R + pos) * N + n, o->io_dtype);
  dtrow[h] = dt_cache[(slot * H + h) * R + pos];
  operands t = *o;
  t.x = xrow;
  t.B = Brow;
  t.C = Brow; /* y of a replayed token is not kept */
  t.z = NULL;
  t.dt = dtrow;
  t.dt_per_dim = 0;
  ssu_step(&t, 0, h, hb, ydump);
}

int oracle_replay_update(void* state, int state_dtype, int64_t slots,
                         int64_t H, int64_t P, int64_t N, int64_t G, int64_t nseqs, int64_t rows,
                         const void* x, const void* z, int io_dtype, const float* dt,
                         const float* A, const float* D, const float* dt_bias,
                         const void* B, const void* C,
                         const int64_t* cu_seqlens, const int64_t* sbi, int64_t pad_slot_id,
                         void* x_cache, void* B_cache, float* dt_cache, int64_t ring_len,
                         int32_t* ring_start, int32_t* prev_num_accepted, int64_t num_states,
                         int32_t logical_window, int update_trackers, int dt_softplus,
                         int param_per_dim, double* y, const uint64_t* rand_seed,
                         int philox_rounds) {
  if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0 || ring_len < 1) return 1;
  operands o = {H, P, N, G, x, z, io_dtype, dt, 0, A, D, dt_bias, B, C, dt_softplus,
                param_per_dim};
  const sr_ctx sr = {rand_seed, philox_rounds};
  const int64_t block = P * N;
  const int64_t limit = slots < num_states ? slots : num_states;
  double* hb = (double*)malloc(sizeof(double) * (size_t)block);
  void* xrow = calloc((size_t)(H * P), 2);
  void* Brow = calloc((size_t)(G * N), 2);
  float* dtrow = (float*)calloc((size_t)H, sizeof(float));
  double* ydump = (double*)malloc(sizeof(double) * (size_t)(H * P));
  int32_t* processed = (int32_t*)calloc((size_t)(nseqs > 0 ? nseqs : 1), sizeof(int32_t));
  if (!hb || !xrow || !Brow || !dtrow || !ydump || !processed) return 2;
  for (int64_t s = 0; s < nseqs; ++s) {
    int64_t begin = cu_seqlens ? cu_seqlens[s] : s;
    int64_t end = cu_seqlens ? cu_seqlens[s + 1] : s + 1;
    if (begin < 0) begin = 0;
    if (end > rows) end = rows;
    const int64_t L = end - begin;
    if (L <= 0) continue;
    const int64_t slot = sbi ? sbi[s] : s;
    const int slot_valid = slot != pad_slot_id && slot >= 0 && slot < limit;
    const int32_t k = slot_valid ? prev_num_accepted[slot] : 0;
    const int32_t start = slot_valid ? ring_start[slot] : 0;
    const int ok = replay_ok(slot, pad_slot_id, limit, k, start, L, ring_len);
    const int checkpoint = ok && (int64_t)k + L > logical_window;
    processed[s] = ok;
    for (int64_t h = 0; h < H; ++h) {
      const int64_t off = (slot * H + h) * block;
      for (int64_t i = 0; i < block; ++i) hb[i] = ok ? load_value(state, off + i, state_dtype) : 0.0;
      if (ok) {
        for (int32_t j = 0; j < k; ++j)
          replay_token(&o, h, x_cache, B_cache, dt_cache, slot, ((int64_t)start + j) % ring_len,
                       ring_len, xrow, Brow, dtrow, ydump, hb);
        if (checkpoint)
          for (int64_t i = 0; i < block; ++i) store_state(state, off + i, state_dtype, hb[i], &sr);
      }
      for (int64_t t = 0; t < L; ++t) {
        const int64_t r = begin + t;
        ssu_step(&o, r, h, hb, y);
        if (!ok) continue;
        const int64_t pos = ((int64_t)start + k + t) % ring_len;
        for (int64_t p = 0; p < P; ++p)
          copy_io(x_cache, ((slot * H + h) * ring_len + pos) * P + p, x, (r * H + h) * P + p,
                  io_dtype);
        dt_cache[(slot * H + h) * ring_len + pos] = dt[r * H + h];
        if (h % (H / G) == 0) { /* B of the group, once per group */
          const int64_t g = h / (H / G);
          for (int64_t n = 0; n < N; ++n)
            copy_io(B_cache, ((slot * G + g) * ring_len + pos) * N + n, B, (r * G + g) * N + n,
                    io_dtype);
        }
      }
    }
  }
  int rc = 0;
  if (update_trackers) {
    for (int64_t s = 0; s < nseqs && rc == 0; ++s) {
      if (!processed[s]) continue;
      const int64_t slot = sbi ? sbi[s] : s;
      rc = oracle_ring_update(ring_start, num_states, prev_num_accepted, num_states,
                              prev_num_accepted /* prev_query_len: untouched by the rule */,
                              num_states, &slot, 1, 1, 0, logical_window, (int32_t)ring_len,
                              pad_slot_id);
    }
  }
  free(hb);
  free(xrow);
  free(Brow);
  free(dtrow);
  free(ydump);
  free(processed);
  return rc;
}

/* The logical state of `slot` (its checkpoint advanced through its k ring
 * entries, the first part of oracle_replay_update) as double [H, P, N]; the
 * trackers are read, nothing is written.  Returns nonzero for a slot whose
 * trackers are out of range (then out is left alone). */
int oracle_replay_state(const void* state, int state_dtype, int64_t slots,
                        int64_t H, int64_t P, int64_t N, int64_t G, int io_dtype,
                        const float* A, const float* dt_bias, int dt_softplus, int param_per_dim,
                        int64_t slot, const void* x_cache, const void* B_cache,
                        const float* dt_cache, int64_t ring_len, const int32_t* ring_start,
                        const int32_t* prev_num_accepted, int64_t num_states, double* out) {
  const int64_t limit = slots < num_states ? slots : num_states;
  if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0 || ring_len < 1) return 1;
  if (slot < 0 || slot >= limit) return 1;
  const int32_t k = prev_num_accepted[slot], start = ring_start[slot];
  if (k < 0 || k > ring_len || start < 0 || start >= ring_len) return 1;
  operands o = {H, P, N, G, NULL, NULL, io_dtype, NULL, 0, A, NULL, dt_bias, NULL, NULL,
                dt_softplus, param_per_dim};
  void* xrow = calloc((size_t)(H * P), 2);
  void* Brow = calloc((size_t)(G * N), 2);
  float* dtrow = (float*)calloc((size_t)H, sizeof(float));
  double* ydump = (double*)malloc(sizeof(double) * (size_t)(H * P));
  if (!xrow || !Brow || !dtrow || !ydump) return 2;
  for (int64_t h = 0; h < H; ++h) {
    double* hb = out + h * P * N;
    for (int64_t i = 0; i < P * N; ++i) hb[i] = load_value(state, (slot * H + h) * P * N + i, state_dtype);
    for (int32_t j = 0; j < k; ++j)
      replay_token(&o, h, x_cache, B_cache, dt_cache, slot, ((int64_t)start + j) % ring_len,
                   ring_len, xrow, Brow, dtrow, ydump, hb);
  }
  free(xrow);
  free(Brow);
  free(dtrow);
  free(ydump);
  return 0;
}
