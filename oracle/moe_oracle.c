/*
 * CPU oracle for the sparse top-k Mixture-of-Experts FFN layer: the forward,
 * and its gradient (the backward section at the end).
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * definition that the CUDA library is checked against. Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it. The
 * product library never links, loads or calls it, and it shares no code,
 * header or table with the CUDA path.
 *
 * Every stored input (bf16 bit patterns or fp32) is widened exactly to fp64
 * and all arithmetic is done in fp64, one token at a time, in the order the
 * pages state the method. The only fp32 steps are the ones the routing
 * decision is defined on: the router score is rounded to fp32 once, and the
 * selection key is the fp32 sum of that score and the selection bias, so
 * that both sides of a parity test take the top-k decision in the same
 * precision.
 *
 * Sources (page title, then section):
 *  [P1] "Mixture of experts and speculative decoding":
 *       "Following one token through an MoE layer" (steps 1-4),
 *       "Opening the hood: the MoE layer precisely" (the layer equation),
 *       "Keeping the experts busy" (the balance-loss equation),
 *       "A toy MoE layer in PyTorch" (dispatch semantics).
 *  [P2] "Mixture of Experts and Guided Decoding": the gated-sum example with
 *       three experts, the dense and sparse four-expert examples, and the
 *       auxiliary-loss formula with its balanced / collapsed example.
 *  [P3] "MoE inference: the call centre with 256 specialists and 8 taking
 *       each call": "The bare mechanism" (router, top-k, normalised weights,
 *       SwiGLU experts, shared experts, bias-adjusted routing); "The maths
 *       that matters" and "DeepEP, EPLB and Wide-EP" (experts stored and
 *       tokens dispatched in FP8; NVFP4 experts in the GB200 deployment).
 *
 * Readings taken where the pages are silent or garbled:
 *  - The SwiGLU expert is down( SiLU(gate(x)) * up(x) ) without biases; the
 *    page prints the activation around the product, which is garbled.
 *  - The selection bias enters only the key used to choose the top k; gate
 *    weights and the balance statistics use the unbiased router scores.
 *  - Ties in the selection key go to the lower expert index.
 *  - Shared experts always run with weight 1 and are not part of f or P.
 *  - f_i = count_i / (T*k) and P_i = mean over tokens of softmax(r)_i over
 *    all N routed experts, so both sum to one as in the pages' example.
 *  - Capacity overflow is dropped (oracle_capacity_keep), or rerouted in
 *    rounds to the next-best expert with room (oracle_reroute); the page
 *    names both without an order.
 *
 * Parity unpinned: the SwiGLU expert at realistic sizes has no printed value
 * on the pages; it is pinned by reduction to library routines (N=1, k=1 is a
 * plain SwiGLU FFN) and by the dense-with-zeroed-gates brute force, not by a
 * printed number.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Stored element types of the inputs. */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };
/* Gate modes. */
enum { ORACLE_GATE_TOPK_SOFTMAX = 0, ORACLE_GATE_ALL_SOFTMAX_RENORM = 1 };

/* Exact widening of one stored element to fp64. A bf16 value is the upper
 * half of an fp32 bit pattern, so shifting it up gives the fp32 value. */
static double widen(int dtype, const void* base, size_t i) {
  if (dtype == ORACLE_F64) return ((const double*)base)[i];
  if (dtype == ORACLE_F32) return (double)((const float*)base)[i];
  uint32_t u = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------------------- FP8 ----
 * [P3] "The maths that matters" and "DeepEP, EPLB and Wide-EP": deployed
 * experts are stored, and tokens dispatched, in FP8. The 8-bit format is
 * E4M3: sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
 * holds the subnormals m * 2^-9; the largest finite value is 448 (field 15,
 * mantissa 6); field 15 with mantissa 7 is NaN; there is no infinity.
 * Reading (the pages give no scaling rule): each row (a token's activations,
 * or one output channel of a weight matrix) carries one fp32 scale
 * s = fp32(amax / 448) and codes q_i = E4M3(fp32(v_i * inv)) with
 * inv = fp32(448 / amax), rounded to nearest even and saturated at +-448 (a
 * product rather than v_i / s, so that a kernel quantizes at memory speed);
 * a row of zeros has s = 0 and codes 0. The value of a code is
 * decode(q) * s. */
double oracle_e4m3_decode(uint8_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return (c & 0x80) ? -v : v;
}

/* Definition form of the encoder: the finite code nearest to v, ties to the
 * even code (mantissa bit 0 clear), |v| past 448 saturated to 448. Slow
 * (scans the 127 magnitudes); used to pin the direct encoder below. */
uint8_t oracle_e4m3_encode_scan(float v) {
  if (isnan(v)) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0;
  const double a = fabs((double)v);
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    const double d = fabs(a - oracle_e4m3_decode((uint8_t)c));
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return (uint8_t)(sign | best);
}

/* Direct encoder, the same function: split |v| into exponent and mantissa
 * and round the 3-bit mantissa (or the subnormal step count) to nearest
 * even with rint (default rounding mode); a mantissa that rounds up to 8
 * carries into the exponent. */
uint8_t oracle_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0;
  const double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {                 /* subnormal range: steps of 2^-9 */
    const int m = (int)rint(ldexp(a, 9));   /* 0..8; 8 is the smallest normal */
    return (uint8_t)(sign | m);
  }
  int x;
  const double f = frexp(a, &x);            /* a = f * 2^x, f in [0.5, 1) */
  int E = x - 1;                            /* a = (2f) * 2^E, 2f in [1, 2) */
  int m = (int)rint((2.0 * f - 1.0) * 8.0);
  if (m == 8) {
    m = 0;
    ++E;
  }
  if (E + 7 > 15 || (E + 7 == 15 && m == 7)) return sign | 0x7E;
  return (uint8_t)(sign | ((E + 7) << 3) | m);
}

/* Row-wise quantization of a rows x cols matrix of stored values (see the
 * FP8 note above): scale[r] = fp32(amax_r / 448),
 * q = E4M3(fp32(v * fp32(448 / amax_r))). */
void oracle_quantize_rows_e4m3(int rows, int cols, int dtype, const void* src, uint8_t* q,
                               float* scale) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    float amax = 0.0f;
    for (int c = 0; c < cols; ++c) {
      const float v = (float)widen(dtype, src, (size_t)r * cols + c);
      if (fabsf(v) > amax) amax = fabsf(v);
    }
    const float s = amax / 448.0f;
    const float inv = amax > 0.0f ? 448.0f / amax : 0.0f;
    scale[r] = s;
    for (int c = 0; c < cols; ++c) {
      const float v = (float)widen(dtype, src, (size_t)r * cols + c);
      q[(size_t)r * cols + c] = amax == 0.0f ? 0 : oracle_e4m3_encode(v * inv);
    }
  }
}

/* -------------------------------------------------------------- NVFP4 ----
 * [P3] "The maths that matters" and "DeepEP, EPLB and Wide-EP": the GB200
 * deployment keeps its experts in NVFP4. The pages name the format and no
 * more; its definition: 4-bit E2M1 elements (sign, 2 exponent bits with
 * bias 1, 1 mantissa bit; exponent field 0 holds the subnormal 0.5; the
 * magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4 and 6; no infinity, no NaN) in
 * blocks of 16 consecutive elements along the contraction, each block with
 * an unsigned E4M3 scale.
 * Reading (the pages give no scaling rule): as for the FP8 rows, each row
 * also carries one fp32 scale, so that the block scales use E4M3's range.
 * For a row with max |v| = amax > 0:
 *   scale  = fp32(amax / 2688)                        (2688 = 6 * 448)
 *   block  b = E4M3(fp32(bmax * fp32(448 / amax)))    (bmax: the block's max |v|)
 *   code   q = E2M1(fp32(v * fp32(fp32(2688 / amax) / e4m3(b))))
 * both roundings to nearest even and saturating (at 448 and at 6), the sign
 * of v kept also when q rounds to zero; a block whose scale decodes to 0
 * has codes 0, and a row of zeros has scale 0 and all codes 0. The value of
 * an element is e2m1(q) * e4m3(b) * scale. */
double oracle_e2m1_decode(uint8_t c) {
  const int e = (c >> 1) & 3, m = c & 1;
  const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return (c & 8) ? -v : v;
}

/* Definition form: the code whose magnitude is nearest |v|, ties to the even
 * code (mantissa bit clear); from 6 up, saturated to 6. */
uint8_t oracle_e2m1_encode_scan(float v) {
  const uint8_t sign = signbit(v) ? 8 : 0;
  const double a = fabs((double)v);
  if (a >= 6.0) return (uint8_t)(sign | 7);
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    const double d = fabs(a - oracle_e2m1_decode((uint8_t)c));
    if (d < bd || (d == bd && !(c & 1))) {
      bd = d;
      best = c;
    }
  }
  return (uint8_t)(sign | best);
}

/* Direct form, the same function: the spacing of the magnitudes is 0.5
 * below 2 (where the code is the step count itself), 1 from 2 to 4 and 2
 * from 4 to 6; rint rounds the step count to nearest even, and codes past
 * 7 saturate. */
uint8_t oracle_e2m1_encode(float v) {
  const uint8_t sign = signbit(v) ? 8 : 0;
  const double a = fabs((double)v);
  int c;
  if (a < 2.0)
    c = (int)rint(2.0 * a);
  else if (a < 4.0)
    c = 4 + (int)rint(a - 2.0);
  else
    c = a >= 6.0 ? 7 : 6 + (int)rint(0.5 * (a - 4.0));
  return (uint8_t)(sign | c);
}

/* Row-wise NVFP4 quantization of a rows x cols matrix (cols a multiple of
 * 16; see the NVFP4 note): q[r][c] one E2M1 code per element, bs[r][c/16]
 * the E4M3 block scale codes, scale[r] the fp32 row scale. */
void oracle_quantize_rows_nvfp4(int rows, int cols, int dtype, const void* src, uint8_t* q,
                                uint8_t* bs, float* scale) {
  const int nb = cols / 16;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    float amax = 0.0f;
    for (int c = 0; c < cols; ++c) {
      const float v = (float)widen(dtype, src, (size_t)r * cols + c);
      if (fabsf(v) > amax) amax = fabsf(v);
    }
    scale[r] = amax / 2688.0f;
    const float to_block = amax > 0.0f ? 448.0f / amax : 0.0f;
    const float to_code = amax > 0.0f ? 2688.0f / amax : 0.0f;
    for (int b = 0; b < nb; ++b) {
      float bmax = 0.0f;
      for (int i = 0; i < 16; ++i) {
        const float v = (float)widen(dtype, src, (size_t)r * cols + 16 * b + i);
        if (fabsf(v) > bmax) bmax = fabsf(v);
      }
      const uint8_t code = amax > 0.0f ? oracle_e4m3_encode(bmax * to_block) : 0;
      bs[(size_t)r * nb + b] = code;
      const float bv = (float)oracle_e4m3_decode(code);
      const float inv = bv > 0.0f ? to_code / bv : 0.0f;
      for (int i = 0; i < 16; ++i) {
        const float v = (float)widen(dtype, src, (size_t)r * cols + 16 * b + i);
        q[(size_t)r * cols + 16 * b + i] = bv > 0.0f ? oracle_e2m1_encode(v * inv) : 0;
      }
    }
  }
}

/* Value of element (r, c) of an NVFP4 matrix with cols columns. */
static double nvfp4_value(const uint8_t* q, const uint8_t* bs, const float* scale, int cols,
                          size_t r, int c) {
  return oracle_e2m1_decode(q[r * cols + c]) * oracle_e4m3_decode(bs[r * (cols / 16) + c / 16]) *
         (double)scale[r];
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* softmax(r) over n scores, max-subtracted, fp64. [P1] step 3; [P2] dense
 * four-expert example. */
void oracle_softmax(int n, const double* r, double* p) {
  double m = r[0];
  for (int i = 1; i < n; ++i)
    if (r[i] > m) m = r[i];
  double s = 0.0;
  for (int i = 0; i < n; ++i) {
    p[i] = exp(r[i] - m);
    s += p[i];
  }
  for (int i = 0; i < n; ++i) p[i] /= s;
}

/* Indices of the k largest keys, best first. A key only displaces the
 * current best when it is strictly larger, so equal keys go to the lower
 * index. [P1] step 2 and the layer equation's TopK set; [P3] top-k
 * selection. */
void oracle_topk(int n, int k, const float* key, int32_t* idx) {
  char* taken = (char*)calloc((size_t)n, 1);
  for (int s = 0; s < k; ++s) {
    int best = -1;
    for (int i = 0; i < n; ++i) {
      if (taken[i]) continue;
      if (best < 0 || key[i] > key[best]) best = i;
    }
    idx[s] = best;
    taken[best] = 1;
  }
  free(taken);
}

/* Gate weights of the kept experts from the unbiased scores r (fp64).
 *  TOPK_SOFTMAX: softmax over the k kept scores only ([P1] step 3 and the
 *    layer equation; [P2] sparse example).
 *  ALL_SOFTMAX_RENORM: softmax over all n scores, then the kept
 *    probabilities divided by their sum ([P1] step 3's parenthesis; [P3] the
 *    router's affinity softmax and the renormalised top-k weights). */
void oracle_gates(int n, int k, int mode, const double* r, const int32_t* idx,
                  double* g) {
  if (mode == ORACLE_GATE_TOPK_SOFTMAX) {
    double* kept = (double*)malloc(sizeof(double) * (size_t)k);
    for (int s = 0; s < k; ++s) kept[s] = r[idx[s]];
    oracle_softmax(k, kept, g);
    free(kept);
  } else {
    double* p = (double*)malloc(sizeof(double) * (size_t)n);
    oracle_softmax(n, r, p);
    double z = 0.0;
    for (int s = 0; s < k; ++s) z += p[idx[s]];
    for (int s = 0; s < k; ++s) g[s] = p[idx[s]] / z;
    free(p);
  }
}

/* Router scores r[t][e] = sum_j x[t][j] * W_r[e][j] + logit_bias[e], fp64.
 * W_r is stored [N][d] (one row per expert, the linear-layer weight layout
 * of the pages' toy code). Also writes the scores rounded once to fp32 when
 * r32 is given: that is the value routing decisions are taken on.
 * [P1] step 1 and "r = x W_r"; [P3] the router projection. */
void oracle_router_logits(int T, int d, int N, int xdtype, const void* x,
                          int wdtype, const void* w_router,
                          const double* logit_bias, double* r64, float* r32) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < N; ++e) {
      double acc = 0.0;
      for (int j = 0; j < d; ++j)
        acc += widen(xdtype, x, (size_t)t * d + j) *
               widen(wdtype, w_router, (size_t)e * d + j);
      if (logit_bias) acc += logit_bias[e];
      if (r64) r64[(size_t)t * N + e] = acc;
      if (r32) r32[(size_t)t * N + e] = (float)acc;
    }
  }
}

/* Routing of T tokens from fp32 scores r32[T][N].
 *  key = fp32(r + sel_bias) (sel_bias may be NULL); top-k on the key;
 *  gate weights from the unbiased scores; per-expert counts; and
 *  prob_sum[e] = sum_t softmax(r_t)[e] over all N experts.
 * The fp32 sum of two fp32 values is taken as their exact fp64 sum rounded
 * once to fp32, which is the correctly rounded fp32 sum.
 * [P1] steps 1-3; [P3] "The bare mechanism" (bias-adjusted routing keeps the
 * bias out of the weights); [P1] "Keeping the experts busy" for f and P. */
void oracle_route(int T, int N, int k, int gate_mode, const float* r32,
                  const float* sel_bias, int32_t* topk_idx, double* topk_w,
                  int32_t* counts, double* prob_sum) {
  if (counts) memset(counts, 0, sizeof(int32_t) * (size_t)N);
  if (prob_sum) memset(prob_sum, 0, sizeof(double) * (size_t)N);
  float* key = (float*)malloc(sizeof(float) * (size_t)N);
  double* r = (double*)malloc(sizeof(double) * (size_t)N);
  double* p = (double*)malloc(sizeof(double) * (size_t)N);
  for (int t = 0; t < T; ++t) {
    const float* rt = r32 + (size_t)t * N;
    for (int e = 0; e < N; ++e) {
      r[e] = (double)rt[e];
      key[e] = sel_bias ? (float)((double)rt[e] + (double)sel_bias[e]) : rt[e];
    }
    int32_t* it = topk_idx + (size_t)t * k;
    oracle_topk(N, k, key, it);
    oracle_gates(N, k, gate_mode, r, it, topk_w + (size_t)t * k);
    if (counts)
      for (int s = 0; s < k; ++s) counts[it[s]] += 1;
    if (prob_sum) {
      oracle_softmax(N, r, p);
      for (int e = 0; e < N; ++e) prob_sum[e] += p[e];
    }
  }
  free(key);
  free(r);
  free(p);
}

/* Grouping of the T*k (token, slot) pairs by expert: expert-major, and
 * within one expert by ascending pair id t*k+slot (a token never picks the
 * same expert twice, so this is ascending token order). offsets is the
 * exclusive prefix sum of the per-expert counts, sorted_pair[row] is the
 * pair id stored at that row, inv_pos[pair] is the row of that pair.
 * This is the data layout of the toy layer's per-expert dispatch loop
 * ([P1] "A toy MoE layer in PyTorch"; [P2] sparse MoE code): every token
 * that chose expert e, and only those, is processed by e. */
/* Expert capacity. [P1] "Keeping the experts busy": a system may cap the
 * tokens one expert takes from a batch, and the extras are dropped. Reading:
 * with capacity C > 0, expert e keeps the first C of the pairs that chose it
 * in ascending pair order (token, then slot) and drops the rest; C = 0 sets
 * no cap. keep[p] = 1 for a kept pair, 0 for a dropped one. */
void oracle_capacity_keep(int T, int k, int N, const int32_t* topk_idx, int capacity,
                          uint8_t* keep) {
  for (int e = 0; e < N; ++e) {
    int taken = 0;
    for (int t = 0; t < T; ++t)
      for (int s = 0; s < k; ++s)
        if (topk_idx[(size_t)t * k + s] == e) {
          keep[(size_t)t * k + s] = (capacity == 0 || taken < capacity) ? 1 : 0;
          ++taken;
        }
  }
}

/* Rows grouped by expert, kept pairs only (capacity as in
 * oracle_capacity_keep; 0 = none): offsets[e] is the first row of expert e,
 * sorted_pair[row] the pair id t*k+s, inv_pos[pair] its row, or -1 for a
 * dropped pair. An index of -1 marks a pair with no expert (one that
 * rerouting dropped): it has no row either. [P1] "A toy MoE layer in
 * PyTorch": each expert processes the tokens routed to it. */
void oracle_permute(int T, int k, int N, const int32_t* topk_idx, int capacity,
                    int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos) {
  uint8_t* keep = (uint8_t*)malloc((size_t)T * k + 1);
  oracle_capacity_keep(T, k, N, topk_idx, capacity, keep);
  for (size_t p = 0; p < (size_t)T * k; ++p) inv_pos[p] = -1;
  int32_t row = 0;
  for (int e = 0; e < N; ++e) {
    offsets[e] = row;
    for (int t = 0; t < T; ++t)
      for (int s = 0; s < k; ++s)
        if (topk_idx[(size_t)t * k + s] == e) {
          int32_t pair = t * k + s;
          if (keep[pair]) {
            sorted_pair[row] = pair;
            inv_pos[pair] = row;
            ++row;
          } else {
            inv_pos[pair] = -1;
          }
        }
  }
  offsets[N] = row;
  free(keep);
}

/* Capacity overflow rerouted instead of dropped. [P1] "Keeping the experts
 * busy": the pairs over an expert's capacity are dropped or rerouted. The
 * page gives no order; the reading taken here works in rounds:
 *  round 0  the capacity cut of oracle_capacity_keep. A kept pair stays with
 *           its expert; the others are pending. room[e] = C - kept at e.
 *  round r  every pending pair (t, s), in slot order within its token,
 *           proposes the expert with the highest selection key
 *           fp32(r + sel_bias) (ties to the lower index) that has room > 0
 *           at the start of the round, that the token does not hold (its k
 *           routed experts and those it was rerouted to) and that no lower
 *           slot of the token proposed to in this round. A pair with no such
 *           expert is dropped. Each expert then accepts the proposals it got
 *           in ascending pair id, up to its room; the rest stay pending.
 * The rounds end when one has no proposal. A rerouted pair keeps its slot's
 * gate weight. assign[p] is the expert pair p runs on, or -1 if dropped.
 * A NaN key ranks below every number. capacity = 0 sets no cap (assign =
 * topk_idx). Returns the number of rounds after round 0. */
int oracle_reroute(int T, int k, int N, const float* r32, const float* sel_bias,
                   const int32_t* topk_idx, int capacity, int32_t* assign) {
  const size_t P = (size_t)T * k;
  if (capacity == 0) {
    for (size_t p = 0; p < P; ++p) assign[p] = topk_idx[p];
    return 0;
  }
  enum { PENDING = -2 };
  uint8_t* keep = (uint8_t*)malloc(P + 1);
  uint8_t* held = (uint8_t*)calloc((size_t)T * N + 1, 1);
  uint8_t* tried = (uint8_t*)malloc((size_t)N);
  int32_t* prop = (int32_t*)malloc(sizeof(int32_t) * (P + 1));
  int* room = (int*)malloc(sizeof(int) * (size_t)N);
  int* taken = (int*)malloc(sizeof(int) * (size_t)N);
  /* round 0: the capacity cut */
  oracle_capacity_keep(T, k, N, topk_idx, capacity, keep);
  for (int e = 0; e < N; ++e) room[e] = capacity;
  for (size_t p = 0; p < P; ++p) {
    const int e = topk_idx[p];
    held[(p / k) * N + e] = 1;
    if (keep[p]) {
      assign[p] = e;
      room[e] -= 1;
    } else {
      assign[p] = PENDING;
    }
  }
  int rounds = 0;
  for (;;) {
    /* proposals */
    int proposals = 0;
    for (int t = 0; t < T; ++t) {
      memset(tried, 0, (size_t)N);
      for (int s = 0; s < k; ++s) {
        const size_t p = (size_t)t * k + s;
        prop[p] = -1;
        if (assign[p] != PENDING) continue;
        int best = -1;
        float best_key = 0.0f;
        for (int e = 0; e < N; ++e) {
          if (held[(size_t)t * N + e] || room[e] <= 0 || tried[e]) continue;
          const float r = r32[(size_t)t * N + e];
          float key = sel_bias ? (float)((double)r + (double)sel_bias[e]) : r;
          if (isnan(key)) key = -INFINITY;
          if (best < 0 || key > best_key) {
            best = e;
            best_key = key;
          }
        }
        if (best < 0) {
          assign[p] = -1;  /* no expert left for it: dropped */
        } else {
          prop[p] = best;
          tried[best] = 1;
          ++proposals;
        }
      }
    }
    if (proposals == 0) break;
    ++rounds;
    /* each expert accepts in ascending pair id, up to its room */
    memset(taken, 0, sizeof(int) * (size_t)N);
    for (size_t p = 0; p < P; ++p) {
      const int e = prop[p];
      if (e < 0) continue;
      if (taken[e] < room[e]) {
        assign[p] = e;
        held[(p / k) * N + e] = 1;
        taken[e] += 1;
      }
    }
    for (int e = 0; e < N; ++e) room[e] -= taken[e];
  }
  free(keep);
  free(held);
  free(tried);
  free(prop);
  free(room);
  free(taken);
  return rounds;
}

/* SiLU(z) = z / (1 + e^-z). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* fp32 value rounded to bf16 (nearest even), as the GPU stores H. */
static float round_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) != 0x7F800000u) u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* An expert's three weight matrices in E4M3, one scale per output row. */
typedef struct {
  uint8_t *gq, *uq, *dq;
  float *gs, *us, *ds;
} QExpert;

/* One SwiGLU expert on one token row in FP8 (see the FP8 note): x is the
 * token's dequantized row; every weight is dequantized from its code and its
 * row scale; H is rounded to bf16, quantized as one row, and dequantized
 * before the down projection. */
static void expert_swiglu_fp8(int d, int d_ff, const QExpert* q, const double* x, double* out) {
  float* h = (float*)malloc(sizeof(float) * (size_t)d_ff);
  for (int j = 0; j < d_ff; ++j) {
    double a = 0.0, b = 0.0;
    for (int i = 0; i < d; ++i) {
      a += oracle_e4m3_decode(q->gq[(size_t)j * d + i]) * x[i];
      b += oracle_e4m3_decode(q->uq[(size_t)j * d + i]) * x[i];
    }
    a *= (double)q->gs[j];
    b *= (double)q->us[j];
    h[j] = round_bf16((float)(silu(a) * b));
  }
  uint8_t* hq = (uint8_t*)malloc((size_t)d_ff);
  float hs;
  oracle_quantize_rows_e4m3(1, d_ff, ORACLE_F32, h, hq, &hs);
  for (int c = 0; c < d; ++c) {
    double acc = 0.0;
    for (int j = 0; j < d_ff; ++j)
      acc += oracle_e4m3_decode(q->dq[(size_t)c * d_ff + j]) *
             (oracle_e4m3_decode(hq[j]) * (double)hs);
    out[c] = acc * (double)q->ds[c];
  }
  free(hq);
  free(h);
}

/* An expert's three weight matrices in NVFP4: codes, block scales and row
 * scales of each. */
typedef struct {
  uint8_t *gq, *uq, *dq, *gb, *ub, *db;
  float *gs, *us, *ds;
} Q4Expert;

/* One SwiGLU expert on one token row in NVFP4 (see the NVFP4 note): x is
 * the token's dequantized row, every weight is its NVFP4 value, H is rounded
 * to bf16, quantized as one NVFP4 row and taken at its NVFP4 value by the
 * down projection. */
static void expert_swiglu_nvfp4(int d, int d_ff, const Q4Expert* q, const double* x,
                                double* out) {
  float* h = (float*)malloc(sizeof(float) * (size_t)d_ff);
  for (int j = 0; j < d_ff; ++j) {
    double a = 0.0, b = 0.0;
    for (int i = 0; i < d; ++i) {
      a += nvfp4_value(q->gq, q->gb, q->gs, d, (size_t)j, i) * x[i];
      b += nvfp4_value(q->uq, q->ub, q->us, d, (size_t)j, i) * x[i];
    }
    h[j] = round_bf16((float)(silu(a) * b));
  }
  uint8_t* hq = (uint8_t*)malloc((size_t)d_ff);
  uint8_t* hb = (uint8_t*)malloc((size_t)d_ff / 16);
  float hs;
  oracle_quantize_rows_nvfp4(1, d_ff, ORACLE_F32, h, hq, hb, &hs);
  for (int c = 0; c < d; ++c) {
    double acc = 0.0;
    for (int j = 0; j < d_ff; ++j)
      acc += nvfp4_value(q->dq, q->db, q->ds, d_ff, (size_t)c, j) *
             nvfp4_value(hq, hb, &hs, d_ff, 0, j);
    out[c] = acc;
  }
  free(hb);
  free(hq);
  free(h);
}

/* One SwiGLU expert on one token row x[d] (fp64):
 *   out[c] = sum_j Wd[c][j] * SiLU(sum_i Wg[j][i] x[i]) * (sum_i Wu[j][i] x[i])
 * Wg and Wu are stored [d_ff][d], Wd is stored [d][d_ff] (linear-layer
 * layout, output rows). [P3] "The bare mechanism": the dense FFN in SwiGLU
 * form, read as down(SiLU(gate(x)) * up(x)). */
void oracle_expert_swiglu(int d, int d_ff, int wdtype, const void* wg,
                          const void* wu, const void* wd, const double* x,
                          double* out) {
  double* h = (double*)malloc(sizeof(double) * (size_t)d_ff);
  for (int j = 0; j < d_ff; ++j) {
    double a = 0.0, b = 0.0;
    for (int i = 0; i < d; ++i) {
      a += widen(wdtype, wg, (size_t)j * d + i) * x[i];
      b += widen(wdtype, wu, (size_t)j * d + i) * x[i];
    }
    h[j] = silu(a) * b;
  }
  for (int c = 0; c < d; ++c) {
    double acc = 0.0;
    for (int j = 0; j < d_ff; ++j)
      acc += widen(wdtype, wd, (size_t)c * d_ff + j) * h[j];
    out[c] = acc;
  }
  free(h);
}

/* y[c] = sum_i G[i] * E[i][c]: the gate-weighted sum of expert outputs.
 * [P1] step 4 and the layer equation; [P2] the three-expert example. */
void oracle_gated_sum(int n_terms, int dim, const double* G, const double* E,
                      double* y) {
  for (int c = 0; c < dim; ++c) {
    double acc = 0.0;
    for (int i = 0; i < n_terms; ++i) acc += G[i] * E[(size_t)i * dim + c];
    y[c] = acc;
  }
}

/* Layer output for a list of token rows, given the routing:
 *   y_t = sum_{slot} g[t][slot] * E_{idx[t][slot]}(x_t)
 *         + sum_{shared s} E_{N+s}(x_t)
 * Shared experts are stored after the N routed experts and always run with
 * weight one. wg/wu/wd are per-expert pointer tables of length N+n_shared;
 * an entry may be NULL when no listed token uses that expert (it is then
 * never read; a NULL that is needed makes the call return -1).
 * [P1] layer equation; [P2] sparse MoE; [P3] "The bare mechanism" (shared
 * experts always run, the routed ones are gate-weighted). */
int oracle_layer_rows(int T, int d, int d_ff, int N, int k, int n_shared,
                      int xdtype, const void* x, int wdtype,
                      const void* const* wg, const void* const* wu,
                      const void* const* wd, const int32_t* topk_idx,
                      const double* topk_w, const uint8_t* keep, int quant, int n_rows,
                      const int32_t* rows, double* y) {
  int bad = 0;
  for (int r = 0; r < n_rows; ++r) {
    int t = rows[r];
    if (t < 0 || t >= T) return -1;
    for (int s = 0; s < k; ++s) {
      int e = topk_idx[(size_t)t * k + s];
      if (keep && !keep[(size_t)t * k + s]) continue;  /* dropped: not evaluated */
      if (e < 0 || e >= N || !wg[e] || !wu[e] || !wd[e]) bad = 1;
    }
  }
  for (int s = 0; s < n_shared; ++s)
    if (!wg[N + s] || !wu[N + s] || !wd[N + s]) bad = 1;
  if (bad) return -1;

  /* quant = 1 (FP8) or 2 (NVFP4): quantize every supplied expert's weights
   * once, row by row. */
  const int fp8 = quant == 1, fp4 = quant == 2;
  const int E_all = N + n_shared;
  QExpert* qe = NULL;
  Q4Expert* q4 = NULL;
  if (fp4) {
    q4 = (Q4Expert*)calloc((size_t)E_all, sizeof(Q4Expert));
    for (int e = 0; e < E_all; ++e) {
      if (!wg[e] || !wu[e] || !wd[e]) continue;
      const size_t n = (size_t)d_ff * d;
      q4[e].gq = (uint8_t*)malloc(n);
      q4[e].uq = (uint8_t*)malloc(n);
      q4[e].dq = (uint8_t*)malloc(n);
      q4[e].gb = (uint8_t*)malloc(n / 16);
      q4[e].ub = (uint8_t*)malloc(n / 16);
      q4[e].db = (uint8_t*)malloc(n / 16);
      q4[e].gs = (float*)malloc(sizeof(float) * (size_t)d_ff);
      q4[e].us = (float*)malloc(sizeof(float) * (size_t)d_ff);
      q4[e].ds = (float*)malloc(sizeof(float) * (size_t)d);
      oracle_quantize_rows_nvfp4(d_ff, d, wdtype, wg[e], q4[e].gq, q4[e].gb, q4[e].gs);
      oracle_quantize_rows_nvfp4(d_ff, d, wdtype, wu[e], q4[e].uq, q4[e].ub, q4[e].us);
      oracle_quantize_rows_nvfp4(d, d_ff, wdtype, wd[e], q4[e].dq, q4[e].db, q4[e].ds);
    }
  }
  if (fp8) {
    qe = (QExpert*)calloc((size_t)E_all, sizeof(QExpert));
    for (int e = 0; e < E_all; ++e) {
      if (!wg[e] || !wu[e] || !wd[e]) continue;
      qe[e].gq = (uint8_t*)malloc((size_t)d_ff * d);
      qe[e].uq = (uint8_t*)malloc((size_t)d_ff * d);
      qe[e].dq = (uint8_t*)malloc((size_t)d * d_ff);
      qe[e].gs = (float*)malloc(sizeof(float) * (size_t)d_ff);
      qe[e].us = (float*)malloc(sizeof(float) * (size_t)d_ff);
      qe[e].ds = (float*)malloc(sizeof(float) * (size_t)d);
      oracle_quantize_rows_e4m3(d_ff, d, wdtype, wg[e], qe[e].gq, qe[e].gs);
      oracle_quantize_rows_e4m3(d_ff, d, wdtype, wu[e], qe[e].uq, qe[e].us);
      oracle_quantize_rows_e4m3(d, d_ff, wdtype, wd[e], qe[e].dq, qe[e].ds);
    }
  }

  /* Every (row, term) expert evaluation is independent: evaluate them all
   * (in parallel), then form each row's gated sum in term order. */
  const int terms = k + n_shared;
  double* E = (double*)malloc(sizeof(double) * (size_t)n_rows * terms * d);
  double* G = (double*)malloc(sizeof(double) * (size_t)n_rows * terms);
#pragma omp parallel for schedule(dynamic, 1)
  for (long long q = 0; q < (long long)n_rows * terms; ++q) {
    const int r = (int)(q / terms), s = (int)(q % terms);
    const int t = rows[r];
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
    if (fp8) {  /* the token's row, quantized as one row and dequantized */
      uint8_t* xq = (uint8_t*)malloc((size_t)d);
      float xs;
      oracle_quantize_rows_e4m3(1, d, xdtype, (const char*)x + (size_t)t * d * (xdtype == ORACLE_BF16 ? 2 : xdtype == ORACLE_F32 ? 4 : 8), xq, &xs);
      for (int i = 0; i < d; ++i) xt[i] = oracle_e4m3_decode(xq[i]) * (double)xs;
      free(xq);
    } else if (fp4) {  /* the token's row as one NVFP4 row */
      uint8_t* xq = (uint8_t*)malloc((size_t)d);
      uint8_t* xb = (uint8_t*)malloc((size_t)d / 16);
      float xs;
      oracle_quantize_rows_nvfp4(1, d, xdtype, (const char*)x + (size_t)t * d * (xdtype == ORACLE_BF16 ? 2 : xdtype == ORACLE_F32 ? 4 : 8), xq, xb, &xs);
      for (int i = 0; i < d; ++i) xt[i] = nvfp4_value(xq, xb, &xs, d, 0, i);
      free(xb);
      free(xq);
    } else {
      for (int i = 0; i < d; ++i) xt[i] = widen(xdtype, x, (size_t)t * d + i);
    }
    int e;
    if (s < k) {
      e = topk_idx[(size_t)t * k + s];
      G[q] = topk_w[(size_t)t * k + s];
    } else {
      e = N + (s - k);
      G[q] = 1.0;
    }
    if (s < k && keep && !keep[(size_t)t * k + s]) {
      /* a dropped pair contributes nothing ([P1] "Keeping the experts busy") */
      G[q] = 0.0;
      for (int c = 0; c < d; ++c) E[(size_t)q * d + c] = 0.0;
    } else if (fp8) {
      expert_swiglu_fp8(d, d_ff, &qe[e], xt, E + (size_t)q * d);
    } else if (fp4) {
      expert_swiglu_nvfp4(d, d_ff, &q4[e], xt, E + (size_t)q * d);
    } else {
      oracle_expert_swiglu(d, d_ff, wdtype, wg[e], wu[e], wd[e], xt, E + (size_t)q * d);
    }
    free(xt);
  }
  for (int r = 0; r < n_rows; ++r)
    oracle_gated_sum(terms, d, G + (size_t)r * terms, E + (size_t)r * terms * d,
                     y + (size_t)r * d);
  free(E);
  free(G);
  if (qe) {
    for (int e = 0; e < E_all; ++e) {
      free(qe[e].gq); free(qe[e].uq); free(qe[e].dq);
      free(qe[e].gs); free(qe[e].us); free(qe[e].ds);
    }
    free(qe);
  }
  if (q4) {
    for (int e = 0; e < E_all; ++e) {
      free(q4[e].gq); free(q4[e].uq); free(q4[e].dq);
      free(q4[e].gb); free(q4[e].ub); free(q4[e].db);
      free(q4[e].gs); free(q4[e].us); free(q4[e].ds);
    }
    free(q4);
  }
  return 0;
}

/* Load-balance term alpha * N * sum_i f_i * P_i. [P1] "Keeping the experts
 * busy"; [P2] auxiliary-loss formula and its N = 4 example. */
double oracle_balance_loss(int N, const double* f, const double* P,
                           double alpha) {
  double s = 0.0;
  for (int i = 0; i < N; ++i) s += f[i] * P[i];
  return alpha * (double)N * s;
}

/* f_i = counts_i / (T*k), P_i = prob_sum_i / T, and the balance loss built
 * from them. [P1] "Keeping the experts busy" (f = fraction of tokens sent to
 * expert i, P = average router probability); with k > 1 a token is counted
 * once per expert it is sent to, so f sums to one. */
double oracle_balance_stats(int N, int T, int k, const int32_t* counts,
                            const double* prob_sum, double alpha, double* f,
                            double* P) {
  for (int i = 0; i < N; ++i) {
    f[i] = (double)counts[i] / ((double)T * (double)k);
    P[i] = prob_sum[i] / (double)T;
  }
  return oracle_balance_loss(N, f, P, alpha);
}

/* Selection margin of each token: the gap between the k-th and (k+1)-th
 * largest fp64 key r64 + sel_bias (infinity when k = N). Inputs whose margin
 * is at least 1e-3 have a top-k set that no fp32 rounding of the scores can
 * change, so routing can be compared bit for bit. */
void oracle_selection_margin(int T, int N, int k, const double* r64,
                             const float* sel_bias, double* margin) {
  double* key = (double*)malloc(sizeof(double) * (size_t)N);
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < N; ++e)
      key[e] = r64[(size_t)t * N + e] + (sel_bias ? (double)sel_bias[e] : 0.0);
    /* k-th and (k+1)-th largest by partial selection sort */
    for (int s = 0; s <= k && s < N; ++s) {
      int best = s;
      for (int i = s + 1; i < N; ++i)
        if (key[i] > key[best]) best = i;
      double tmp = key[s];
      key[s] = key[best];
      key[best] = tmp;
    }
    margin[t] = (k < N) ? key[k - 1] - key[k] : INFINITY;
  }
  free(key);
}

/* Order margin of each token: the smallest gap between neighbours among the
 * min(k + 1, N) largest fp64 keys, sorted (infinity when N = 1). It bounds
 * both the selection margin and the gaps between kept experts, so inputs
 * whose order margin is at least 1e-3 fix the top-k set and its order
 * (topk_idx is sorted by key) against any fp32 rounding of the scores. */
void oracle_order_margin(int T, int N, int k, const double* r64,
                         const float* sel_bias, double* margin) {
  double* key = (double*)malloc(sizeof(double) * (size_t)N);
  const int m = k < N ? k + 1 : N;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < N; ++e)
      key[e] = r64[(size_t)t * N + e] + (sel_bias ? (double)sel_bias[e] : 0.0);
    for (int s = 0; s < m; ++s) {
      int best = s;
      for (int i = s + 1; i < N; ++i)
        if (key[i] > key[best]) best = i;
      double tmp = key[s];
      key[s] = key[best];
      key[best] = tmp;
    }
    double g = INFINITY;
    for (int s = 0; s + 1 < m; ++s)
      if (key[s] - key[s + 1] < g) g = key[s] - key[s + 1];
    margin[t] = g;
  }
  free(key);
}

/* ------------------------------------------------------------ backward ----
 * Gradient of the scalar
 *     L = sum_t sum_c dy[t][c] * y[t][c] + aux_grad * aux,
 *     aux = alpha * N * sum_i f_i * P_i,
 * with respect to x, W_r, W_g, W_u and W_d, where y is the layer output
 * ([P1] the layer equation) and aux the balance term ([P1] "Keeping the
 * experts busy"; [P2] the auxiliary-loss formula). Readings:
 *  - The top-k choice, the capacity cut and the counts (so f) are hard
 *    decisions and stay fixed; the gradient flows through the gate weights g
 *    and through P ([P2]: f comes from a hard choice and is not
 *    differentiated, the gradient flows through P).
 *  - The fp32 rounding of the score only fixes the routing decision and is
 *    taken as the identity: g and P are differentiated as the functions of
 *    the score r they are defined as, at the forward's values (the score
 *    rounded to fp32, as the forward evaluates them).
 *  - logit_bias and sel_bias are constants.
 * Everything is the chain rule through the forward's steps, in fp64. The
 * weights are the stacked [N+n_shared] arrays (shared experts last). */

static size_t elem_size(int dtype) {
  return dtype == ORACLE_F64 ? 8 : dtype == ORACLE_F32 ? 4 : 2;
}
static const void* elem_ptr(int dtype, const void* base, size_t i) {
  return (const char*)base + i * elem_size(dtype);
}

/* SiLU'(z) = s * (1 + z * (1 - s)) with s = 1 / (1 + e^-z). */
static double silu_grad(double z) {
  const double s = 1.0 / (1.0 + exp(-z));
  return s * (1.0 + z * (1.0 - s));
}

/* One expert term of one token and its backward. With a = Wg x, b = Wu x,
 * h = SiLU(a) * b and o = Wd h (the expert of oracle_expert_swiglu), the term
 * adds G * o to y, so
 *   do = G * dy,  dh = Wd^T do,  da = dh * b * SiLU'(a),  db = dh * SiLU(a),
 *   dx += Wg^T da + Wu^T db,
 * and dL/dG = <dy, o>, which is returned. h, da, db and do are left for the
 * weight gradients (dWg += da x^T, dWu += db x^T, dWd += do h^T). */
static double expert_backward(int d, int d_ff, int wdtype, const void* wg, const void* wu,
                              const void* wd, const double* xt, const double* dyt, double G,
                              double* h, double* da, double* db, double* dout, double* dxt) {
  double* a = (double*)malloc(sizeof(double) * (size_t)d_ff);
  double* b = (double*)malloc(sizeof(double) * (size_t)d_ff);
  for (int j = 0; j < d_ff; ++j) {
    double aj = 0.0, bj = 0.0;
    for (int i = 0; i < d; ++i) {
      aj += widen(wdtype, wg, (size_t)j * d + i) * xt[i];
      bj += widen(wdtype, wu, (size_t)j * d + i) * xt[i];
    }
    a[j] = aj;
    b[j] = bj;
    h[j] = silu(aj) * bj;
  }
  double dG = 0.0;
  for (int c = 0; c < d; ++c) {
    double o = 0.0;
    for (int j = 0; j < d_ff; ++j) o += widen(wdtype, wd, j + (size_t)c * d_ff) * h[j];
    dG += dyt[c] * o;
    dout[c] = G * dyt[c];
  }
  for (int j = 0; j < d_ff; ++j) {
    double dh = 0.0;
    for (int c = 0; c < d; ++c) dh += widen(wdtype, wd, j + (size_t)c * d_ff) * dout[c];
    da[j] = dh * b[j] * silu_grad(a[j]);
    db[j] = dh * silu(a[j]);
  }
  for (int i = 0; i < d; ++i) {
    double acc = 0.0;
    for (int j = 0; j < d_ff; ++j)
      acc += widen(wdtype, wg, (size_t)j * d + i) * da[j] +
             widen(wdtype, wu, (size_t)j * d + i) * db[j];
    dxt[i] = acc;
  }
  free(a);
  free(b);
  return dG;
}

/* Score gradient of one token. r: its scores (fp32 values widened), idx:
 * its k experts, dG[s]: dL/dg_s, f: the balance fractions. Gates, by mode:
 *  TOPK_SOFTMAX: g = softmax of the k kept scores, so
 *    dr[idx_s] += g_s * (dG_s - sum_l g_l dG_l);
 *  ALL_SOFTMAX_RENORM: p = softmax(r) over all N, Z = sum_s p[idx_s],
 *    g_s = p[idx_s] / Z, so dp[idx_s] = (dG_s - sum_l g_l dG_l) / Z and
 *    dr_i += p_i * (dp_i - sum_m p_m dp_m).
 * Balance term: P_i = (1/T) sum_t p_t[i], so
 *    dr_i += aux_grad * alpha * N / T * p_i * (f_i - sum_m p_m f_m). */
static void score_backward(int N, int k, int T, int gate_mode, const double* r,
                           const int32_t* idx, const double* dG, const double* f, double alpha,
                           double aux_grad, double* dr) {
  double* g = (double*)malloc(sizeof(double) * (size_t)k);
  double* p = (double*)malloc(sizeof(double) * (size_t)N);
  double* dp = (double*)calloc((size_t)N, sizeof(double));
  for (int i = 0; i < N; ++i) dr[i] = 0.0;
  oracle_gates(N, k, gate_mode, r, idx, g);
  oracle_softmax(N, r, p);
  double gdG = 0.0;
  for (int s = 0; s < k; ++s) gdG += g[s] * dG[s];
  if (gate_mode == ORACLE_GATE_TOPK_SOFTMAX) {
    for (int s = 0; s < k; ++s) dr[idx[s]] += g[s] * (dG[s] - gdG);
  } else {
    double Z = 0.0;
    for (int s = 0; s < k; ++s) Z += p[idx[s]];
    for (int s = 0; s < k; ++s) dp[idx[s]] = (dG[s] - gdG) / Z;
    double pdp = 0.0;
    for (int m = 0; m < N; ++m) pdp += p[m] * dp[m];
    for (int i = 0; i < N; ++i) dr[i] += p[i] * (dp[i] - pdp);
  }
  double pf = 0.0;
  for (int m = 0; m < N; ++m) pf += p[m] * f[m];
  const double scale = aux_grad * alpha * (double)N / (double)T;
  for (int i = 0; i < N; ++i) dr[i] += scale * p[i] * (f[i] - pf);
  free(g);
  free(p);
  free(dp);
}

/* Forward routing shared by the two backward entry points: fp32 scores,
 * top-k, gates, counts, kept pairs and f. */
typedef struct {
  float* r32;
  int32_t* idx;
  double* g;
  int32_t* counts;
  uint8_t* keep;
  int32_t* run;  /* the expert each pair runs on, -1 if dropped */
  double* f;
} Routing;

static void routing_forward(int T, int d, int N, int k, int gate_mode, int capacity,
                            int reroute, int xdtype, const void* x, int wdtype,
                            const void* w_router, const double* logit_bias,
                            const float* sel_bias, Routing* R) {
  R->r32 = (float*)malloc(sizeof(float) * (size_t)T * N);
  R->idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  R->g = (double*)malloc(sizeof(double) * (size_t)T * k);
  R->counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
  R->keep = (uint8_t*)malloc((size_t)T * k + 1);
  R->run = (int32_t*)malloc(sizeof(int32_t) * ((size_t)T * k + 1));
  R->f = (double*)malloc(sizeof(double) * (size_t)N);
  oracle_router_logits(T, d, N, xdtype, x, wdtype, w_router, logit_bias, NULL, R->r32);
  oracle_route(T, N, k, gate_mode, R->r32, sel_bias, R->idx, R->g, R->counts, NULL);
  oracle_capacity_keep(T, k, N, R->idx, capacity, R->keep);
  if (reroute) {
    oracle_reroute(T, k, N, R->r32, sel_bias, R->idx, capacity, R->run);
  } else {
    for (size_t q = 0; q < (size_t)T * k; ++q) R->run[q] = R->keep[q] ? R->idx[q] : -1;
  }
  for (int i = 0; i < N; ++i) R->f[i] = (double)R->counts[i] / ((double)T * (double)k);
}

static void routing_free(Routing* R) {
  free(R->r32);
  free(R->idx);
  free(R->g);
  free(R->counts);
  free(R->keep);
  free(R->run);
  free(R->f);
}

/* The expert of term s (< k: routed slot, else shared expert N + s - k) of
 * token t, with its gate (0 for a dropped pair: it is not evaluated). A
 * rerouted slot runs on its new expert with the slot's gate. */
static int term_expert(const Routing* R, int N, int k, int t, int s, double* G) {
  if (s < k) {
    const size_t q = (size_t)t * k + s;
    if (R->run[q] < 0) {
      *G = 0.0;
      return -1;
    }
    *G = R->g[q];
    return R->run[q];
  }
  *G = 1.0;
  return N + (s - k);
}

/* Full backward for all tokens: dx [T][d], dw_router [N][d],
 * dwg/dwu [N+s][d_ff][d], dwd [N+s][d][d_ff], all fp64. dy is [T][d] fp64.
 * Weight gradients sum their terms in ascending (token, term) order. */
void oracle_layer_backward(int T, int d, int d_ff, int N, int k, int n_shared, int gate_mode,
                           int capacity, int reroute, int xdtype, const void* x, int wdtype,
                           const void* w_router, const double* logit_bias,
                           const float* sel_bias, const void* wg, const void* wu,
                           const void* wd, const double* dy, double alpha, double aux_grad,
                           double* dx, double* dw_router, double* dwg, double* dwu,
                           double* dwd) {
  const int terms = k + n_shared, E = N + n_shared;
  Routing R;
  routing_forward(T, d, N, k, gate_mode, capacity, reroute, xdtype, x, wdtype, w_router,
                  logit_bias, sel_bias, &R);
  const size_t Q = (size_t)T * terms;
  double* H = (double*)calloc(Q * d_ff, sizeof(double));
  double* DA = (double*)calloc(Q * d_ff, sizeof(double));
  double* DB = (double*)calloc(Q * d_ff, sizeof(double));
  double* DO = (double*)calloc(Q * d, sizeof(double));
  double* DXE = (double*)calloc(Q * d, sizeof(double));
  double* dG = (double*)calloc((size_t)T * k, sizeof(double));
  int* ex = (int*)malloc(sizeof(int) * Q);
#pragma omp parallel for schedule(dynamic, 1)
  for (long long q = 0; q < (long long)Q; ++q) {
    const int t = (int)(q / terms), s = (int)(q % terms);
    double G;
    const int e = term_expert(&R, N, k, t, s, &G);
    ex[q] = e;
    if (e < 0) continue;  /* dropped pair: no term, dL/dg = 0 */
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < d; ++i) xt[i] = widen(xdtype, x, (size_t)t * d + i);
    const double dGq = expert_backward(
        d, d_ff, wdtype, elem_ptr(wdtype, wg, (size_t)e * d_ff * d),
        elem_ptr(wdtype, wu, (size_t)e * d_ff * d), elem_ptr(wdtype, wd, (size_t)e * d * d_ff),
        xt, dy + (size_t)t * d, G, H + q * d_ff, DA + q * d_ff, DB + q * d_ff, DO + q * d,
        DXE + q * d);
    if (s < k) dG[(size_t)t * k + s] = dGq;
    free(xt);
  }
  double* DR = (double*)malloc(sizeof(double) * (size_t)T * N);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double* r = (double*)malloc(sizeof(double) * (size_t)N);
    for (int e = 0; e < N; ++e) r[e] = (double)R.r32[(size_t)t * N + e];
    score_backward(N, k, T, gate_mode, r, R.idx + (size_t)t * k, dG + (size_t)t * k, R.f, alpha,
                   aux_grad, DR + (size_t)t * N);
    for (int i = 0; i < d; ++i) {
      double acc = 0.0;
      for (int s = 0; s < terms; ++s) acc += DXE[((size_t)t * terms + s) * d + i];
      for (int e = 0; e < N; ++e)
        acc += DR[(size_t)t * N + e] * widen(wdtype, w_router, (size_t)e * d + i);
      dx[(size_t)t * d + i] = acc;
    }
    free(r);
  }
#pragma omp parallel for schedule(static)
  for (int e = 0; e < N; ++e)
    for (int i = 0; i < d; ++i) {
      double acc = 0.0;
      for (int t = 0; t < T; ++t)
        acc += DR[(size_t)t * N + e] * widen(xdtype, x, (size_t)t * d + i);
      dw_router[(size_t)e * d + i] = acc;
    }
#pragma omp parallel for schedule(dynamic, 1)
  for (long long ej = 0; ej < (long long)E * d_ff; ++ej) {
    const int e = (int)(ej / d_ff), j = (int)(ej % d_ff);
    double* rg = dwg + (size_t)ej * d;
    double* ru = dwu + (size_t)ej * d;
    for (int i = 0; i < d; ++i) rg[i] = ru[i] = 0.0;
    for (size_t q = 0; q < Q; ++q) {
      if (ex[q] != e) continue;
      const int t = (int)(q / terms);
      for (int i = 0; i < d; ++i) {
        const double xi = widen(xdtype, x, (size_t)t * d + i);
        rg[i] += DA[q * d_ff + j] * xi;
        ru[i] += DB[q * d_ff + j] * xi;
      }
    }
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (long long ec = 0; ec < (long long)E * d; ++ec) {
    const int e = (int)(ec / d), c = (int)(ec % d);
    double* rd = dwd + (size_t)ec * d_ff;
    for (int j = 0; j < d_ff; ++j) rd[j] = 0.0;
    for (size_t q = 0; q < Q; ++q) {
      if (ex[q] != e) continue;
      for (int j = 0; j < d_ff; ++j) rd[j] += DO[q * d + c] * H[q * d_ff + j];
    }
  }
  free(H);
  free(DA);
  free(DB);
  free(DO);
  free(DXE);
  free(dG);
  free(ex);
  free(DR);
  routing_free(&R);
}

/* The same gradients at sampled places, for sizes where the full backward
 * is too slow: dx rows of the listed tokens, and for each listed (e, j) the
 * row j of dWg[e] and dWu[e] (length d) and the column j of dWd[e] (length
 * d). A column j of the weight gradients needs only a_j, b_j and dh_j of
 * every token the expert takes, so each is one pass over those tokens.
 * wg/wu/wd are per-expert pointer tables (length N + n_shared); an expert
 * no listed token or column uses may be NULL. Returns -1 (and computes
 * nothing) when a needed expert is missing. */
int oracle_backward_samples(int T, int d, int d_ff, int N, int k, int n_shared, int gate_mode,
                            int capacity, int reroute, int xdtype, const void* x, int wdtype,
                            const void* w_router, const double* logit_bias,
                            const float* sel_bias, const void* const* wg,
                            const void* const* wu, const void* const* wd, const double* dy,
                            double alpha, double aux_grad, int n_tok, const int32_t* toks,
                            double* dx_rows, int n_w, const int32_t* w_e, const int32_t* w_j,
                            double* dwg_rows, double* dwu_rows, double* dwd_cols) {
  const int terms = k + n_shared;
  Routing R;
  routing_forward(T, d, N, k, gate_mode, capacity, reroute, xdtype, x, wdtype, w_router,
                  logit_bias, sel_bias, &R);
  int bad = 0;
  for (int n = 0; n < n_tok; ++n)
    for (int s = 0; s < terms; ++s) {
      double G;
      const int e = term_expert(&R, N, k, toks[n], s, &G);
      if (e >= 0 && (!wg[e] || !wu[e] || !wd[e])) bad = 1;
    }
  for (int n = 0; n < n_w; ++n)
    if (!wg[w_e[n]] || !wu[w_e[n]] || !wd[w_e[n]]) bad = 1;
  if (bad) {
    routing_free(&R);
    return -1;
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int n = 0; n < n_tok; ++n) {
    const int t = toks[n];
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)d_ff);
    double* da = (double*)malloc(sizeof(double) * (size_t)d_ff);
    double* db = (double*)malloc(sizeof(double) * (size_t)d_ff);
    double* dout = (double*)malloc(sizeof(double) * (size_t)d);
    double* dxe = (double*)malloc(sizeof(double) * (size_t)d);
    double* dG = (double*)calloc((size_t)k, sizeof(double));
    double* r = (double*)malloc(sizeof(double) * (size_t)N);
    double* dr = (double*)malloc(sizeof(double) * (size_t)N);
    double* out = dx_rows + (size_t)n * d;
    for (int i = 0; i < d; ++i) {
      xt[i] = widen(xdtype, x, (size_t)t * d + i);
      out[i] = 0.0;
    }
    for (int s = 0; s < terms; ++s) {
      double G;
      const int e = term_expert(&R, N, k, t, s, &G);
      if (e < 0) continue;
      const double g = expert_backward(d, d_ff, wdtype, wg[e], wu[e], wd[e], xt,
                                       dy + (size_t)t * d, G, h, da, db, dout, dxe);
      if (s < k) dG[s] = g;
      for (int i = 0; i < d; ++i) out[i] += dxe[i];
    }
    for (int e = 0; e < N; ++e) r[e] = (double)R.r32[(size_t)t * N + e];
    score_backward(N, k, T, gate_mode, r, R.idx + (size_t)t * k, dG, R.f, alpha, aux_grad, dr);
    for (int i = 0; i < d; ++i)
      for (int e = 0; e < N; ++e) out[i] += dr[e] * widen(wdtype, w_router, (size_t)e * d + i);
    free(xt); free(h); free(da); free(db); free(dout); free(dxe); free(dG); free(r); free(dr);
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int n = 0; n < n_w; ++n) {
    const int e = w_e[n], j = w_j[n];
    double* rg = dwg_rows + (size_t)n * d;
    double* ru = dwu_rows + (size_t)n * d;
    double* cd = dwd_cols + (size_t)n * d;
    for (int i = 0; i < d; ++i) rg[i] = ru[i] = cd[i] = 0.0;
    for (int t = 0; t < T; ++t)
      for (int s = 0; s < terms; ++s) {
        double G;
        if (term_expert(&R, N, k, t, s, &G) != e) continue;
        double a = 0.0, b = 0.0, dh = 0.0;
        for (int i = 0; i < d; ++i) {
          const double xi = widen(xdtype, x, (size_t)t * d + i);
          a += widen(wdtype, wg[e], (size_t)j * d + i) * xi;
          b += widen(wdtype, wu[e], (size_t)j * d + i) * xi;
        }
        for (int c = 0; c < d; ++c)
          dh += widen(wdtype, wd[e], (size_t)c * d_ff + j) * G * dy[(size_t)t * d + c];
        const double h = silu(a) * b;
        const double da = dh * b * silu_grad(a), db = dh * silu(a);
        for (int i = 0; i < d; ++i) {
          const double xi = widen(xdtype, x, (size_t)t * d + i);
          rg[i] += da * xi;
          ru[i] += db * xi;
        }
        for (int c = 0; c < d; ++c) cd[c] += G * dy[(size_t)t * d + c] * h;
      }
  }
  routing_free(&R);
  return 0;
}

/* The gradient when dy = 0: only the balance term moves the loss, so
 * dx = dr W_r and dW_r = dr^T x with dr the balance part of score_backward
 * (the gates' part is zero). Needs no expert. dx [T][d], dw_router [N][d]. */
void oracle_balance_backward(int T, int d, int N, int k, int gate_mode, int xdtype,
                             const void* x, int wdtype, const void* w_router,
                             const double* logit_bias, const float* sel_bias, double alpha,
                             double aux_grad, double* dx, double* dw_router) {
  Routing R;
  routing_forward(T, d, N, k, gate_mode, 0, 0, xdtype, x, wdtype, w_router, logit_bias,
                  sel_bias, &R);
  double* DR = (double*)malloc(sizeof(double) * (size_t)T * N);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double* r = (double*)malloc(sizeof(double) * (size_t)N);
    double* dG = (double*)calloc((size_t)k, sizeof(double));
    for (int e = 0; e < N; ++e) r[e] = (double)R.r32[(size_t)t * N + e];
    score_backward(N, k, T, gate_mode, r, R.idx + (size_t)t * k, dG, R.f, alpha, aux_grad,
                   DR + (size_t)t * N);
    for (int i = 0; i < d; ++i) {
      double acc = 0.0;
      for (int e = 0; e < N; ++e)
        acc += widen(wdtype, w_router, (size_t)e * d + i) * DR[(size_t)t * N + e];
      dx[(size_t)t * d + i] = acc;
    }
    free(r);
    free(dG);
  }
#pragma omp parallel for schedule(static)
  for (int e = 0; e < N; ++e)
    for (int i = 0; i < d; ++i) {
      double acc = 0.0;
      for (int t = 0; t < T; ++t)
        acc += DR[(size_t)t * N + e] * widen(xdtype, x, (size_t)t * d + i);
      dw_router[(size_t)e * d + i] = acc;
    }
  free(DR);
  routing_free(&R);
}
