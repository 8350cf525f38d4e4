/*
 * oracle.c — plain, slow, fp64 CPU statement of the paged-KV hot path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library calls, links or
 * loads this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do. It shares no code, header, table or helper with the CUDA path.
 *
 * Pages followed (cited by title and section):
 *   [vLLM-wiki] itwiki.kr "vLLM": "블록 테이블" (physical block pool, per-request
 *     block table, slot arithmetic), "블록 단위 어텐션 계산" (the equation for
 *     A_ij and o_i; equal to ordinary attention), "블록 공유와 쓰기 시 복사"
 *     (refcounted sharing, copy-on-write), "엔진 구조와 주요 기능" (FP8 KV cache).
 *   [MRV2] llm-wiki.hwlabs.dev "vLLM 0.25 Model Runner V2 …": "재설계 1" (persistent
 *     slots and idx_mapping), "재설계 3" (staged (row, start, value) diffs applied
 *     on the device, then a gather by idx_mapping), "재설계 4" (query_start_loc,
 *     seq_lens, slot_mapping).
 * FP8 E4M3 follows the OCP 8-bit floating point specification (OFP8): bias 7,
 * no infinities, S.1111.111 is NaN, largest finite 448, subnormals kept.
 *
 * Every function is a direct transcription of the definition: no online
 * softmax, no splitting, no blocking. Compile with -ffp-contract=off so that
 * results do not depend on the host's FMA contraction.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARGS 1
#define ORACLE_ERR_RANGE 2

enum { ORACLE_BF16 = 0, ORACLE_FP8_E4M3 = 1 };

/* ---------------------------------------------------------------- numbers */

/* bfloat16 bits are the top half of an IEEE binary32: the conversion is exact. */
static float bf16_bits_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* OFP8 E4M3 decode: sign s, exponent field e (4 bits), mantissa field m (3 bits).
 *   e == 15 && m == 7      : NaN
 *   e == 0                 : subnormal, (m / 8) * 2^(1 - 7)
 *   otherwise              : (1 + m / 8) * 2^(e - 7)                          */
double oracle_e4m3_decode(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, 1 - 7);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* OFP8 E4M3 encode of an fp32 value, round to nearest with ties to even and
 * saturation to the largest finite magnitude ("satfinite").
 * The 127 non-negative finite codes 0x00..0x7E decode to strictly increasing
 * values; the code is found by binary search between the two neighbours of
 * |x|; a tie picks the neighbour whose code (= mantissa) LSB is 0.           */
uint8_t oracle_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 0x7E; /* decode(lo) <= a < decode(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (oracle_e4m3_decode((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid;
  }
  double vlo = oracle_e4m3_decode((uint8_t)lo), vhi = oracle_e4m3_decode((uint8_t)hi);
  int code;
  if (a - vlo < vhi - a)
    code = lo;
  else if (a - vlo > vhi - a)
    code = hi;
  else
    code = (lo & 1) ? hi : lo;
  return (uint8_t)(sign | code);
}

/* The FP8 store of a bf16 input: the quotient float(x) / scale is one IEEE
 * fp32 division (correctly rounded), then the encode above. */
uint8_t oracle_fp8_store(uint16_t bf16_bits, float scale) {
  float x = bf16_bits_to_float(bf16_bits);
  float q = x / scale;
  return oracle_e4m3_encode(q);
}

/* Element (blk, h, t, d) of a pool laid out [num_blocks][Hkv][B][D], as fp64.
 * FP8 codes are decoded and multiplied by the per-tensor scale in fp64. */
static double pool_value(const void* pool, int dtype, int64_t index, double scale) {
  if (dtype == ORACLE_BF16) return (double)bf16_bits_to_float(((const uint16_t*)pool)[index]);
  return oracle_e4m3_decode(((const uint8_t*)pool)[index]) * scale;
}

static int64_t pool_index(int64_t blk, int64_t h, int64_t t, int64_t d, int64_t Hkv, int64_t B,
                          int64_t D) {
  return ((blk * Hkv + h) * B + t) * D + d;
}

/* ------------------------------------------------------------- KV write */

/* [vLLM-wiki "블록 테이블"], [MRV2 "재설계 4"]: token t lands in slot s =
 * physical_block * B + offset; a negative slot is padding and is skipped. */
int oracle_write_kv(void* k_pool, void* v_pool, int32_t num_blocks, int32_t B, int32_t Hkv,
                    int32_t D, int32_t dtype, float k_scale, float v_scale,
                    const uint16_t* k_new, const uint16_t* v_new, const int64_t* slots,
                    int32_t T) {
  if (B <= 0 || Hkv <= 0 || D <= 0 || num_blocks < 0 || T < 0) return ORACLE_ERR_ARGS;
  int status = ORACLE_OK;
  for (int32_t t = 0; t < T; ++t) {
    int64_t s = slots[t];
    if (s < 0) continue;
    int64_t blk = s / B, off = s % B;
    if (blk >= num_blocks) {
      status = ORACLE_ERR_RANGE;
      continue;
    }
    for (int32_t h = 0; h < Hkv; ++h) {
      for (int32_t d = 0; d < D; ++d) {
        int64_t src = ((int64_t)t * Hkv + h) * D + d;
        int64_t dst = pool_index(blk, h, off, d, Hkv, B, D);
        if (dtype == ORACLE_BF16) {
          ((uint16_t*)k_pool)[dst] = k_new[src];
          ((uint16_t*)v_pool)[dst] = v_new[src];
        } else {
          ((uint8_t*)k_pool)[dst] = oracle_fp8_store(k_new[src], k_scale);
          ((uint8_t*)v_pool)[dst] = oracle_fp8_store(v_new[src], v_scale);
        }
      }
    }
  }
  return status;
}

/* ------------------------------------------------------- block copy (CoW) */

/* [vLLM-wiki "블록 공유와 쓰기 시 복사"]: the device half of copy-on-write copies a
 * whole physical block (every kv head, every offset, K and V). Pairs are
 * applied in order. */
int oracle_copy_blocks(void* k_pool, void* v_pool, int32_t num_blocks, int32_t B, int32_t Hkv,
                       int32_t D, int32_t dtype, const int32_t* src, const int32_t* dst,
                       int32_t n) {
  int64_t elt = dtype == ORACLE_BF16 ? 2 : 1;
  int64_t block_bytes = (int64_t)Hkv * B * D * elt;
  int status = ORACLE_OK;
  for (int32_t i = 0; i < n; ++i) {
    if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks) {
      status = ORACLE_ERR_RANGE;
      continue;
    }
    memmove((char*)k_pool + dst[i] * block_bytes, (char*)k_pool + src[i] * block_bytes,
            (size_t)block_bytes);
    memmove((char*)v_pool + dst[i] * block_bytes, (char*)v_pool + src[i] * block_bytes,
            (size_t)block_bytes);
  }
  return status;
}

/* ----------------------------------------------- staged block-table diffs */

/* [MRV2 "재설계 3"]: diffs are applied one after another in record order (so a
 * later diff wins on a shared cell); then [MRV2 "재설계 1"]: the rows of this
 * step are gathered by idx_mapping. Diffs or mapping entries that leave the
 * table are skipped and reported. */
int oracle_apply_staged_writes(int32_t* table, int32_t max_reqs, int32_t max_blocks,
                               const int32_t* rows, const int32_t* starts,
                               const int32_t* val_offsets, const int32_t* vals, int32_t W,
                               const int32_t* idx_mapping, int32_t R, int32_t* gathered) {
  int status = ORACLE_OK;
  for (int32_t w = 0; w < W; ++w) {
    int32_t row = rows[w], start = starts[w];
    int32_t len = val_offsets[w + 1] - val_offsets[w];
    if (row < 0 || row >= max_reqs || start < 0 || len < 0 ||
        (int64_t)start + len > max_blocks || val_offsets[w] < 0 ||
        val_offsets[w + 1] > val_offsets[W]) {
      status = ORACLE_ERR_RANGE;
      continue;
    }
    for (int32_t k = 0; k < len; ++k)
      table[(int64_t)row * max_blocks + start + k] = vals[val_offsets[w] + k];
  }
  for (int32_t i = 0; i < R; ++i) {
    int32_t slot = idx_mapping[i];
    if (slot < 0 || slot >= max_reqs) {
      status = ORACLE_ERR_RANGE;
      continue;
    }
    for (int32_t c = 0; c < max_blocks; ++c)
      gathered[(int64_t)i * max_blocks + c] = table[(int64_t)slot * max_blocks + c];
  }
  return status;
}

/* ------------------------------------------------------------- attention */

/* One output row (token t, query head h) of [vLLM-wiki "블록 단위 어텐션 계산"].
 * With p the absolute position of the query, the visible keys are 0..p when
 * causal (every key of every block before and including the query's own), and
 * 0..seq_len-1 otherwise. Key n lives in physical block table[n / B] at offset
 * n % B. The softmax denominator sums exp over every visible key of every
 * block, so the blockwise sum is ordinary softmax attention:
 *     s_n = scale * sum_d q_d k_nd,   a_n = exp(s_n - max) / sum exp(s - max),
 *     o_d = sum_n a_n v_nd.
 * Writes D doubles to `o`. Returns ORACLE_ERR_RANGE on a block id outside
 * the pool.                                                                   */
static int attention_row(const uint16_t* q_row, double* o, const int32_t* table_row, int32_t n_visible,
                         const void* k_pool, const void* v_pool, int32_t num_blocks, int32_t B,
                         int32_t Hkv, int32_t D, int32_t dtype, double k_scale, double v_scale,
                         int32_t kv_head, double scale, double* s /* scratch [n_visible] */) {
  double qd[256];
  for (int32_t d = 0; d < D; ++d) qd[d] = (double)bf16_bits_to_float(q_row[d]);
  double smax = -INFINITY;
  for (int32_t n = 0; n < n_visible; ++n) {
    int32_t blk = table_row[n / B];
    if (blk < 0 || blk >= num_blocks) return ORACLE_ERR_RANGE;
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d)
      dot += qd[d] * pool_value(k_pool, dtype, pool_index(blk, kv_head, n % B, d, Hkv, B, D),
                                k_scale);
    s[n] = scale * dot;
    if (s[n] > smax) smax = s[n];
  }
  double denom = 0.0;
  for (int32_t n = 0; n < n_visible; ++n) {
    s[n] = exp(s[n] - smax);
    denom += s[n];
  }
  for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
  for (int32_t n = 0; n < n_visible; ++n) {
    int32_t blk = table_row[n / B];
    double a = s[n] / denom;
    for (int32_t d = 0; d < D; ++d)
      o[d] += a * pool_value(v_pool, dtype, pool_index(blk, kv_head, n % B, d, Hkv, B, D),
                             v_scale);
  }
  return ORACLE_OK;
}

/* Paged attention over a batch described by query_start_loc and seq_lens
 * ([MRV2 "재설계 4"]). Query j of request r sits at absolute position
 * seq_len[r] - q_len[r] + j. Query head h reads kv head h / (Hq / Hkv).
 *
 * `rows` optionally restricts the work to n_rows output rows, each encoded as
 * token * Hq + head (out is still indexed [T][Hq][D]); rows == NULL computes
 * every row of every request. Rows of tokens outside [0, qsl[R]) are left
 * untouched. nthreads <= 0 uses the OpenMP default.                          */
int oracle_paged_attention(const uint16_t* q, double* out, const int32_t* qsl,
                           const int32_t* seq_lens, const int32_t* block_tables,
                           int32_t max_blocks, int32_t R, int32_t T, int32_t Hq,
                           const void* k_pool, const void* v_pool, int32_t num_blocks,
                           int32_t B, int32_t Hkv, int32_t D, int32_t dtype, double k_scale,
                           double v_scale, double scale, int32_t causal, const int64_t* rows,
                           int64_t n_rows, int32_t nthreads) {
  if (R < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || D > 256 || B <= 0)
    return ORACLE_ERR_ARGS;
  if (qsl[0] != 0 || qsl[R] > T) return ORACLE_ERR_ARGS;
  int32_t max_seq = 0;
  for (int32_t r = 0; r < R; ++r) {
    int32_t q_len = qsl[r + 1] - qsl[r];
    if (q_len < 0 || (q_len > 0 && (q_len > seq_lens[r] ||
                                     seq_lens[r] > (int64_t)max_blocks * B)))
      return ORACLE_ERR_ARGS;
    if (seq_lens[r] > max_seq) max_seq = seq_lens[r];
  }
  int64_t total = rows ? n_rows : (int64_t)qsl[R] * Hq;
  int32_t g = Hq / Hkv;
  int status = ORACLE_OK;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(max : status)
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_seq > 0 ? max_seq : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < total; ++i) {
      int64_t row = rows ? rows[i] : i;
      int64_t t = row / Hq;
      int32_t h = (int32_t)(row % Hq);
      if (t < 0 || t >= qsl[R]) continue;
      /* request r with qsl[r] <= t < qsl[r+1] (binary search) */
      int32_t lo = 0, hi = R - 1;
      while (lo < hi) {
        int32_t mid = (lo + hi + 1) / 2;
        if (qsl[mid] <= t)
          lo = mid;
        else
          hi = mid - 1;
      }
      int32_t r = lo; /* the largest r with qsl[r] <= t; never an empty request */
      int32_t q_len = qsl[r + 1] - qsl[r];
      int32_t j = (int32_t)(t - qsl[r]);
      int32_t p = seq_lens[r] - q_len + j;
      int32_t n_visible = causal ? p + 1 : seq_lens[r];
      int rc = attention_row(q + (t * Hq + h) * (int64_t)D, out + (t * Hq + h) * (int64_t)D,
                             block_tables + (int64_t)r * max_blocks, n_visible, k_pool, v_pool,
                             num_blocks, B, Hkv, D, dtype, k_scale, v_scale, h / g, scale, s);
      if (rc > status) status = rc;
    }
    free(s);
  }
  return status;
}

/* Threads the OpenMP runtime would use by default (reported with timings). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
