/*
 * CPU oracle for mixed-dtype FSDP communication-buffer packing.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke()
 * and bench.py's cpu_baseline / reference leg load this file's library.  It
 * shares no code, header, table or constant with the CUDA path and is meant to
 * be read against the pages line by line: single-threaded, no blocking, no
 * vectorisation, loops over (bucket | group, rank, parameter, element) exactly
 * as the definitions state them.
 *
 * Sources (web pages, cited by title and section):
 *   [News]   "FSDP2 per-parameter mixed precision" news item (ainewsletter.today,
 *            ?p=1549): paragraphs 1-2 (staging copies grouped by (src, dst) dtype,
 *            one all-gather per fully_shard; reduce-scatter copy-in reads BF16 and
 *            FP32 and casts into the reduction buffer during chunking and padding;
 *            one bucket per effective reduction dtype).
 *   [Unit]   "The unit you wrapped" (kernels.rudrite.com), sections on the
 *            FlatParameter shard slice (row-major flattening, rank r holds slice r)
 *            and on padding to a multiple of the world size (right-hand padding).
 *   [NeMo]   "Mixed-Precision Training" (NVIDIA NeMo AutoModel), table "Storage
 *            Dtype Compared to Compute Dtype" (param_dtype, reduce_dtype, storage
 *            dtype of the resident shard).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - each parameter is chunked as its flattened row-major vector:
 *     c_p = ceil(n_p / W), rank r owns elements [r*c_p, min(n_p, (r+1)*c_p)),
 *     the rest of its chunk is +0 padding in the destination dtype;
 *   - FP32 -> BF16 is IEEE-754 round to nearest, ties to even, no flush of
 *     subnormals, overflow to infinity; a NaN keeps its sign and top payload
 *     bits and gets the quiet bit;
 *   - all-gather input: groups concatenated in first-appearance order of
 *     (shard dtype, param dtype), each group starting on a 16-byte boundary,
 *     gap and tail bytes zero.
 *
 * Parity pins live in tests/test_oracle_pins.py.  A multi-parameter unit is
 * chunked per parameter (FSDP2's rule: every parameter padded and split into
 * W chunks, rank r's row the concatenation of the chunks r), which is a
 * reading: the pages print shard values only for single-parameter units,
 * where it agrees with FSDP1's one flat vector split W ways.  The
 * per-parameter rule is pinned by brute force (pad, reshape, concatenate) on
 * every one- and two-parameter layout up to 13 elements and W = 5, on sampled
 * three-parameter layouts, and by the per-rank counts the pages print.
 *
 * Dtype codes used by this file only: 0 = FP32, 1 = BF16.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

static int64_t dtype_size(int32_t dt) { return dt == ORACLE_F32 ? 4 : 2; }

/* ---------------------------------------------------------------------------
 * Number formats.
 * ------------------------------------------------------------------------ */

/* Real value of a bfloat16 bit pattern (1 sign, 8 exponent, 7 fraction bits,
 * bias 127) decoded from its fields.  An all-ones exponent with zero fraction
 * is returned as 2^128 in magnitude: the value an unbounded exponent range
 * would give, which is what rounding compares against at the top of the range.
 * Not called for NaN patterns. */
static double bf16_field_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xFF;
  int f = h & 0x7F;
  double mag;
  if (e == 0)
    mag = ldexp((double)f, -126 - 7); /* subnormal: 0.f * 2^-126 */
  else
    mag = ldexp(128.0 + (double)f, e - 127 - 7); /* 1.f * 2^(e-127) */
  return sign ? -mag : mag;
}

/* Real value of a binary32 bit pattern, decoded from its fields (finite only). */
static double f32_field_value(uint32_t u) {
  int sign = (u >> 31) & 1;
  int e = (u >> 23) & 0xFF;
  uint32_t f = u & 0x7FFFFF;
  double mag;
  if (e == 0)
    mag = ldexp((double)f, -126 - 23);
  else
    mag = ldexp(8388608.0 + (double)f, e - 127 - 23);
  return sign ? -mag : mag;
}

/* FP32 -> BF16, round to nearest, ties to even.
 * The two BF16 candidates that bracket x are the pattern with the low 16
 * fraction bits dropped (toward zero) and its successor in magnitude (away
 * from zero).  Their distances to x are compared in double precision, which
 * holds every quantity here exactly.  On a tie the candidate whose last kept
 * fraction bit is 0 wins.  A successor with an all-ones exponent is infinity,
 * so overflow rounds to infinity exactly when IEEE-754 says it does. */
uint16_t oracle_f32_to_bf16(uint32_t u) {
  uint32_t e = (u >> 23) & 0xFF;
  uint32_t f = u & 0x7FFFFF;
  if (e == 0xFF && f != 0) /* NaN: keep sign and top payload, force quiet */
    return (uint16_t)((u >> 16) | 0x0040);
  if (e == 0xFF) /* infinity */
    return (uint16_t)(u >> 16);
  uint16_t toward_zero = (uint16_t)(u >> 16);
  if ((u & 0xFFFF) == 0) /* exactly representable (includes +-0) */
    return toward_zero;
  uint16_t away = (uint16_t)(toward_zero + 1); /* next magnitude, same sign */
  double x = fabs(f32_field_value(u));
  double lo = fabs(bf16_field_value(toward_zero));
  double hi = fabs(bf16_field_value(away));
  double d_lo = x - lo, d_hi = hi - x;
  if (d_lo < d_hi) return toward_zero;
  if (d_hi < d_lo) return away;
  return (toward_zero & 1) ? away : toward_zero; /* tie: even last bit */
}

/* BF16 -> FP32 is exact: every BF16 value is an FP32 value.  Finite values
 * and infinities are decoded to their real value and re-encoded as binary32;
 * a NaN keeps its sign and payload bits in the upper half. */
uint32_t oracle_bf16_to_f32(uint16_t h) {
  int e = (h >> 7) & 0xFF;
  int f = h & 0x7F;
  if (e == 0xFF && f != 0) return (uint32_t)h << 16;
  if (e == 0xFF) return (h & 0x8000) ? 0xFF800000u : 0x7F800000u;
  float v = (float)bf16_field_value(h); /* exact */
  uint32_t out;
  memcpy(&out, &v, 4);
  return out;
}

void oracle_f32_to_bf16_array(const uint32_t *in, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}

void oracle_bf16_to_f32_array(const uint16_t *in, uint32_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(in[i]);
}

/* Cast element si of src (dtype sdt) into element di of dst (dtype ddt). */
static void cast_element(const void *src, int32_t sdt, int64_t si, void *dst,
                         int32_t ddt, int64_t di) {
  if (sdt == ORACLE_F32) {
    uint32_t v = ((const uint32_t *)src)[si];
    if (ddt == ORACLE_F32)
      ((uint32_t *)dst)[di] = v;
    else
      ((uint16_t *)dst)[di] = oracle_f32_to_bf16(v);
  } else {
    uint16_t v = ((const uint16_t *)src)[si];
    if (ddt == ORACLE_BF16)
      ((uint16_t *)dst)[di] = v;
    else
      ((uint32_t *)dst)[di] = oracle_bf16_to_f32(v);
  }
}

static void store_zero(void *dst, int32_t ddt, int64_t di) {
  if (ddt == ORACLE_F32)
    ((uint32_t *)dst)[di] = 0u;
  else
    ((uint16_t *)dst)[di] = 0u;
}

/* ---------------------------------------------------------------------------
 * Reduce-scatter copy-in ([News] paragraph 2; [Unit] shard slice and padding).
 *
 * For every bucket b (one per distinct reduce dtype), rank r, parameter p of
 * bucket b in registration order, and i < c_p:
 *   j = r*c_p + i
 *   buf_b[r*S_b + o_p + i] = cast_{g_p -> rho_b}(grad_p[j])  if j < n_p
 *                          = +0                              otherwise
 * ------------------------------------------------------------------------ */
/* One (bucket, rank, parameter) run of the loops below: the c_p slots that
 * parameter p contributes to row r of its bucket buffer. */
void oracle_pack_segment(int32_t r, int64_t numel, int32_t grad_dtype, int64_t chunk,
                         int64_t bucket_off, int32_t rho, int64_t S_b, const void *grad, void *buf) {
  for (int64_t i = 0; i < chunk; ++i) {
    int64_t j = (int64_t)r * chunk + i;
    int64_t d = (int64_t)r * S_b + bucket_off + i;
    if (j < numel)
      cast_element(grad, grad_dtype, j, buf, rho, d);
    else
      store_zero(buf, rho, d);
  }
}

void oracle_pack_reduce_scatter(int32_t W, int32_t n_params, const int64_t *numel,
                                const int32_t *grad_dtype, const int64_t *chunk,
                                const int32_t *bucket_of, const int64_t *bucket_off,
                                int32_t n_buckets, const int32_t *bucket_dtype,
                                const int64_t *bucket_S, const void *const *grads,
                                void *const *bufs) {
  for (int32_t b = 0; b < n_buckets; ++b)
    for (int32_t r = 0; r < W; ++r)
      for (int32_t p = 0; p < n_params; ++p)
        if (bucket_of[p] == b)
          oracle_pack_segment(r, numel[p], grad_dtype[p], chunk[p], bucket_off[p], bucket_dtype[b],
                              bucket_S[b], grads[p], bufs[b]);
}

/* Value of one element of bucket b at flat index idx (in [0, W*S_b)), computed
 * from the same definition by locating the owning (rank, parameter, i).  Used to
 * check sampled outputs of workloads too large to pack whole on the host. */
static void pack_one(int32_t n_params, const int64_t *numel, const int32_t *grad_dtype,
                     const int64_t *chunk, const int32_t *bucket_of,
                     const int64_t *bucket_off, int32_t b, int32_t rho, int64_t S_b,
                     const void *const *grads, int64_t idx, void *out, int64_t oi) {
  int64_t r = idx / S_b;
  int64_t pos = idx - r * S_b;
  for (int32_t p = 0; p < n_params; ++p) {
    if (bucket_of[p] != b) continue;
    if (pos >= bucket_off[p] && pos < bucket_off[p] + chunk[p]) {
      int64_t j = r * chunk[p] + (pos - bucket_off[p]);
      if (j < numel[p])
        cast_element(grads[p], grad_dtype[p], j, out, rho, oi);
      else
        store_zero(out, rho, oi);
      return;
    }
  }
  store_zero(out, rho, oi); /* unreachable for idx inside the bucket */
}

void oracle_pack_samples(int32_t n_params, const int64_t *numel, const int32_t *grad_dtype,
                         const int64_t *chunk, const int32_t *bucket_of,
                         const int64_t *bucket_off, int32_t b, int32_t rho, int64_t S_b,
                         const void *const *grads, const int64_t *idx, int64_t n_idx,
                         void *out) {
  for (int64_t k = 0; k < n_idx; ++k)
    pack_one(n_params, numel, grad_dtype, chunk, bucket_of, bucket_off, b, rho, S_b,
             grads, idx[k], out, k);
}

/* ---------------------------------------------------------------------------
 * All-gather copy-in for one rank ([News] paragraph 1; [NeMo] storage vs
 * compute dtype).  Gap bytes between groups and the tail up to S_ag are zero;
 * then for every group g, parameter p of g, and i < c_p:
 *   ag_in[G_g + (e_p + i)*size(pi_p)] = cast_{sigma_p -> pi_p}(shard_p[i])
 * ------------------------------------------------------------------------ */
/* Parameter p's part of the loops below: its c_p cast elements. */
void oracle_allgather_copy_in_segment(int64_t chunk, int32_t shard_dtype, int32_t param_dtype,
                                      int64_t group_elem_off, int64_t group_byte_off,
                                      const void *shard, uint8_t *ag_in) {
  void *base = ag_in + group_byte_off;
  for (int64_t i = 0; i < chunk; ++i)
    cast_element(shard, shard_dtype, i, base, param_dtype, group_elem_off + i);
}

void oracle_allgather_copy_in(int32_t n_params, const int64_t *chunk,
                              const int32_t *shard_dtype, const int32_t *param_dtype,
                              const int32_t *group_of, const int64_t *group_elem_off,
                              int32_t n_groups, const int64_t *group_byte_off, int64_t S_ag,
                              const void *const *shards, uint8_t *ag_in) {
  memset(ag_in, 0, (size_t)S_ag);
  for (int32_t g = 0; g < n_groups; ++g)
    for (int32_t p = 0; p < n_params; ++p)
      if (group_of[p] == g)
        oracle_allgather_copy_in_segment(chunk[p], shard_dtype[p], param_dtype[p], group_elem_off[p],
                                         group_byte_off[g], shards[p], ag_in);
}

/* ---------------------------------------------------------------------------
 * All-gather copy-out ([Unit] summon_full_params: the gathered unit has its
 * original shape again).  For every parameter p, rank r and i < c_p with
 * j = r*c_p + i < n_p:
 *   full_p[j] = element (e_p + i) of group g(p) in row r of the gathered buffer,
 *               i.e. the bytes at r*S_ag + G_g + (e_p + i)*size(pi_p).
 * No cast: the gathered dtype is param_dtype.  Padding is dropped.
 * ------------------------------------------------------------------------ */
/* One (parameter, rank) run of the loops below. */
void oracle_allgather_copy_out_segment(int32_t r, int64_t numel, int64_t chunk, int32_t param_dtype,
                                       int64_t group_elem_off, int64_t group_byte_off, int64_t S_ag,
                                       const uint8_t *ag_out, void *param) {
  int64_t sz = dtype_size(param_dtype);
  for (int64_t i = 0; i < chunk; ++i) {
    int64_t j = (int64_t)r * chunk + i;
    if (j >= numel) continue;
    const uint8_t *from = ag_out + (int64_t)r * S_ag + group_byte_off + (group_elem_off + i) * sz;
    memcpy((uint8_t *)param + j * sz, from, (size_t)sz);
  }
}

void oracle_allgather_copy_out(int32_t W, int32_t n_params, const int64_t *numel,
                               const int64_t *chunk, const int32_t *param_dtype,
                               const int32_t *group_of, const int64_t *group_elem_off,
                               const int64_t *group_byte_off, int64_t S_ag,
                               const uint8_t *ag_out, void *const *params) {
  for (int32_t p = 0; p < n_params; ++p)
    for (int32_t r = 0; r < W; ++r)
      oracle_allgather_copy_out_segment(r, numel[p], chunk[p], param_dtype[p], group_elem_off[p],
                                        group_byte_off[group_of[p]], S_ag, ag_out, params[p]);
}

/* ---------------------------------------------------------------------------
 * Reduce-scatter copy-out ([Unit] collective-count section: the reduce-scatter
 * leaves every rank only the slice of the gradient that matches the
 * parameters it owns; [NeMo] table: the resident sharded parameter, and so
 * its gradient, is in the storage dtype).  Given this rank's reduced row of
 * every bucket (S_b elements of rho_b), for every parameter p of bucket b and
 * i < c_p:
 *   sharded_grad_p[i] = cast_{rho_b -> sigma_p}(row_b[o_p + i])
 * The c_p slots include the padding slots of the last ranks.
 * ------------------------------------------------------------------------ */
void oracle_reduce_scatter_copy_out(int32_t n_params, const int64_t *chunk, const int32_t *bucket_of,
                                    const int64_t *bucket_off, const int32_t *bucket_dtype,
                                    const int32_t *shard_dtype, const void *const *rows,
                                    void *const *sharded) {
  for (int32_t p = 0; p < n_params; ++p) {
    int32_t b = bucket_of[p];
    for (int64_t i = 0; i < chunk[p]; ++i)
      cast_element(rows[b], bucket_dtype[b], bucket_off[p] + i, sharded[p], shard_dtype[p], i);
  }
}

/* ---------------------------------------------------------------------------
 * Emulated reduce-scatter on one device (a test utility, not a collective).
 * Every rank's packed bucket buffer has the same [W, S_b] shape, and rank r's
 * reduce-scatter output is row r of their elementwise sum ([Unit]
 * collective-count section: the gradient is reduced across ranks and
 * scattered so every rank keeps its own slice).  The sum runs over ranks
 * q = 0, 1, ..., W-1 in that order, each partial sum rounded to the bucket
 * dtype ("Training frameworks" note, "Check the objective before measuring
 * speed": reduction order changes results, so the order is fixed):
 *   FP32: acc = in_0[i]; acc = fl32(acc + in_q[i])
 *   BF16: acc = in_0[i]; acc = rne_bf16(fl32(f32(acc) + f32(in_q[i])))
 * where fl32 is one IEEE-754 binary32 addition rounded to nearest even.  A
 * sum that is NaN (a NaN operand, or infinities of opposite sign) is the
 * canonical quiet NaN 0x7FC00000 (FP32) / 0x7FC0 (BF16): IEEE-754 leaves the
 * payload of such a result open, and fixing it makes the result the same on
 * every machine.  The first rank's value enters unchanged (with one rank
 * there is no addition and the output is the input, bit for bit).
 * ------------------------------------------------------------------------ */
static float f32_of_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint32_t bits_of_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

/* One binary32 addition, a NaN result made canonical. */
static float add_f32(float a, float b) {
  volatile float s = a + b;
  if (s != s) return f32_of_bits(0x7FC00000u);
  return s;
}

void oracle_emulated_reduce_scatter(int64_t n, int32_t dtype, int32_t n_inputs, const void *const *inputs,
                                    void *out) {
  for (int64_t i = 0; i < n; ++i) {
    if (dtype == ORACLE_F32) {
      float acc = f32_of_bits(((const uint32_t *)inputs[0])[i]);
      for (int32_t q = 1; q < n_inputs; ++q) acc = add_f32(acc, f32_of_bits(((const uint32_t *)inputs[q])[i]));
      ((uint32_t *)out)[i] = bits_of_f32(acc);
    } else {
      uint16_t acc = ((const uint16_t *)inputs[0])[i];
      for (int32_t q = 1; q < n_inputs; ++q) {
        float sum = add_f32(f32_of_bits(oracle_bf16_to_f32(acc)),
                            f32_of_bits(oracle_bf16_to_f32(((const uint16_t *)inputs[q])[i])));
        acc = (sum != sum) ? (uint16_t)0x7FC0 : oracle_f32_to_bf16(bits_of_f32(sum));
      }
      ((uint16_t *)out)[i] = acc;
    }
  }
}
