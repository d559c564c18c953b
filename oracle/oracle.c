/*
 * CPU ORACLE for the fused GEMM + epilogue path. TEST INFRASTRUCTURE ONLY:
 * the tests, the smoke check and the benchmark's CPU-baseline leg may call it;
 * the product library never does, and the two share no code.
 *
 * Plain, slow, obviously correct. Each function is one step of the method in
 * the order the pages give it; the Python wrapper (oracle/__init__.py)
 * composes them into the epilogs. Compiled with -ffp-contract=off so that a
 * multiply and an add are never fused and x86-64 and aarch64 give equal bits.
 *
 * Sources (web pages on fused matmul epilogs):
 *  [P1] "Fusing Matmul Epilogs with nvmath-python"
 *       - "The problem addressed by fused epilogs": the forward of a linear
 *         layer is the matrix product, plus a bias for each output column,
 *         then ReLU.
 *       - "Forward-pass capabilities in the source": RELU_BIAS does exactly
 *         that in one call; RELU_AUX_BIAS also returns relu_aux, a
 *         bit-encoded ReLU mask meant for the backward epilog.
 *       - "Backward-pass path shown in the example": the plain backward is the
 *         product with the transposed weight, then the mask applied by hand,
 *         then a sum over the batch for the bias gradient; DRELU_BGRAD does
 *         the same from relu_aux and returns the column-wise sum.
 *  [P2] "nvmath-python 封装 cuBLASLt: 为 PyTorch 提供低开销矩阵乘法与偏置融合原语"
 *       - step 1: fp16 operands, bias of shape (m, 1) (one value per row).
 *       - step 2: COMPUTE_32F_FAST_16F, i.e. fp32 accumulation with fp16
 *         inputs and outputs.
 *       - "other epilogs": BIAS, GELU_BIAS.
 *  [P3] "gemm_swiglu_mlp_fusion.py" (cuDNN frontend sample), module docstring:
 *       h = silu(x Wg^T) * (x Wu^T), out = h Wd^T, dSwiGLU as a GEMM epilogue.
 *
 * Readings where the pages leave a step open (each is restated where used):
 *  - relu_aux encoding: column words, aux[i/32][j] bit (i%32) = (z[i][j] > 0),
 *    padding bits 0.
 *  - mask bit is taken on the fp32 pre-activation, strictly z > 0.
 *  - bias gradient sums the fp32 masked product (before rounding), in double,
 *    ascending rows, stored as fp32 by the caller.
 *  - fp32 -> fp16/bf16 rounding is round-to-nearest-even.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F16 0
#define OR_BF16 1

#define OR_B_KN 0 /* B stored [K][N] row-major */
#define OR_B_NK 1 /* B stored [N][K] row-major (B = W^T for W [N][K]) */

#define OR_BIAS_COL 0 /* bias[N], one value per output column [P1] */
#define OR_BIAS_ROW 1 /* bias[M], shape (m,1) [P2 step 1] */

/* ------------------------------------------------------------------ formats */

/* IEEE binary16 -> binary32, exact: every half is a float. */
float oracle_half_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) & 1u;
  uint32_t exp = (uint32_t)(h >> 10) & 0x1Fu;
  uint32_t man = (uint32_t)h & 0x3FFu;
  float mag;
  if (exp == 0) {
    mag = ldexpf((float)man, -24); /* subnormal: man * 2^-24 */
  } else if (exp == 31) {
    mag = man ? NAN : INFINITY;
  } else {
    mag = ldexpf((float)(man | 0x400u), (int)exp - 25); /* 1.man * 2^(exp-15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16 is the top half of a binary32. */
float oracle_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* binary32 -> binary16, round to nearest, ties to even; overflow -> inf. */
uint16_t oracle_f32_to_half(float f) {
  if (isnan(f)) return (uint16_t)(signbit(f) ? 0xFE00u : 0x7E00u);
  uint16_t sign = signbit(f) ? 0x8000u : 0u;
  double a = fabs((double)f); /* exact */
  if (isinf(f)) return (uint16_t)(sign | 0x7C00u);
  if (a == 0.0) return sign;
  /* scale so the kept bits are the integer part: quantum q = 2^(e-10) for
   * normals (a in [2^e, 2^(e+1))), 2^-24 for subnormals */
  int e;
  frexp(a, &e); /* a = m * 2^e, m in [0.5,1) -> a in [2^(e-1), 2^e) */
  int top = e - 1;
  int qexp = top < -14 ? -24 : top - 10;
  double scaled = ldexp(a, -qexp); /* exact: power-of-two scaling */
  double fl = floor(scaled);
  double rem = scaled - fl;
  if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
  double r = ldexp(fl, qexp); /* the rounded magnitude */
  if (r >= 65520.0 || r > 65504.0) return (uint16_t)(sign | 0x7C00u);
  /* encode r */
  if (r < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)ldexp(r, 24));
  int re;
  frexp(r, &re);
  int rtop = re - 1; /* r in [2^rtop, 2^(rtop+1)) */
  uint32_t man = (uint32_t)(ldexp(r, 10 - rtop) - 1024.0);
  return (uint16_t)(sign | (uint16_t)((uint32_t)(rtop + 15) << 10) | (uint16_t)man);
}

/* binary32 -> bfloat16, round to nearest, ties to even. */
uint16_t oracle_f32_to_bf16(float f) {
  if (isnan(f)) return (uint16_t)(signbit(f) ? 0xFFC0u : 0x7FC0u);
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t upper = u >> 16;
  uint32_t lower = u & 0xFFFFu;
  /* the magnitude bits ordered like integers: rounding up the 16-bit
   * truncation is one increment of the upper half */
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

void oracle_decode(const uint16_t* in, int64_t n, int dtype, float* out) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = dtype == OR_F16 ? oracle_half_to_f32(in[i]) : oracle_bf16_to_f32(in[i]);
}

void oracle_round(const float* in, int64_t n, int dtype, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = dtype == OR_F16 ? oracle_f32_to_half(in[i]) : oracle_f32_to_bf16(in[i]);
}

/* --------------------------------------------------------------------- GEMM */

typedef struct {
  const float* A; /* [R][K] */
  const float* B; /* [K][N] or [N][K] */
  int64_t R, K, N;
  int b_layout;
  float* acc;       /* fp32 result [R][N] */
  double* acc64;    /* or fp64 result [R][N] */
  int64_t r0, r1;
} gemm_job;

static void* gemm_rows(void* p) {
  gemm_job* j = (gemm_job*)p;
  const int64_t K = j->K, N = j->N;
  for (int64_t r = j->r0; r < j->r1; ++r) {
    const float* a = j->A + r * K;
    if (j->acc) {
      float* c = j->acc + r * N;
      for (int64_t n = 0; n < N; ++n) c[n] = 0.0f;
      /* acc[r][n] = (((0 + a0 b0n) + a1 b1n) + ...): fp32 multiply, then fp32
       * add, in ascending p for every n ([P2 step 2]: fp32 accumulation). The
       * loop order only follows the storage of B; the sum order is the same. */
      if (j->b_layout == OR_B_KN) {
        for (int64_t p = 0; p < K; ++p) {
          const float ap = a[p];
          const float* b = j->B + p * N;
          for (int64_t n = 0; n < N; ++n) {
            float prod = ap * b[n];
            c[n] = c[n] + prod;
          }
        }
      } else {
        for (int64_t n = 0; n < N; ++n) {
          const float* b = j->B + n * K;
          float s = 0.0f;
          for (int64_t p = 0; p < K; ++p) {
            float prod = a[p] * b[p];
            s = s + prod;
          }
          c[n] = s;
        }
      }
    } else {
      double* c = j->acc64 + r * N;
      for (int64_t n = 0; n < N; ++n) c[n] = 0.0;
      /* fp64: the product of two fp16/bf16 values is exact in double */
      for (int64_t p = 0; p < K; ++p) {
        const double ap = (double)a[p];
        for (int64_t n = 0; n < N; ++n) {
          double b = j->b_layout == OR_B_KN ? (double)j->B[p * N + n] : (double)j->B[n * K + p];
          c[n] += ap * b;
        }
      }
    }
  }
  return NULL;
}

static void run_gemm(const float* A, int64_t R, int64_t K, const float* B, int64_t N, int b_layout,
                     float* acc, double* acc64, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > R) nthreads = R > 0 ? (int)R : 1;
  gemm_job* jobs = (gemm_job*)calloc((size_t)nthreads, sizeof(gemm_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int t = 0; t < nthreads; ++t) {
    gemm_job j = {A, B, R, K, N, b_layout, acc, acc64, R * t / nthreads, R * (t + 1) / nthreads};
    jobs[t] = j;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, gemm_rows, &jobs[t]);
  gemm_rows(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
}

/* acc = A B with fp32 multiply-then-add in ascending k ([P2 step 2]).
 * A: decoded fp32 [R][K]; B: decoded fp32, [K][N] (OR_B_KN) or [N][K] (OR_B_NK). */
void oracle_gemm_f32(const float* A, int64_t R, int64_t K, const float* B, int64_t N, int b_layout,
                     float* acc, int nthreads) {
  run_gemm(A, R, K, B, N, b_layout, acc, NULL, nthreads);
}

/* The same product with exact products summed in double: brute-force check. */
void oracle_gemm_f64(const float* A, int64_t R, int64_t K, const float* B, int64_t N, int b_layout,
                     double* acc, int nthreads) {
  run_gemm(A, R, K, B, N, b_layout, NULL, acc, nthreads);
}

/* ---------------------------------------------------------------- epilogues */

/* z = acc + bias, in fp32 ([P1] "The problem addressed by fused epilogs";
 * [P2] step 1 for the (m,1) bias). COL: bias[j]; ROW: bias[row_ids[r]]
 * (row_ids NULL: r). In place on z. */
void oracle_add_bias(float* z, int64_t R, int64_t N, const float* bias, int axis,
                     const int64_t* row_ids) {
  for (int64_t r = 0; r < R; ++r) {
    int64_t gr = row_ids ? row_ids[r] : r;
    for (int64_t j = 0; j < N; ++j) {
      float b = axis == OR_BIAS_COL ? bias[j] : bias[gr];
      z[r * N + j] = z[r * N + j] + b;
    }
  }
}

/* y = ReLU(z) = z if z > 0 else 0 ([P1] "The problem addressed by fused epilogs") */
void oracle_relu(const float* z, int64_t n, float* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = z[i] > 0.0f ? z[i] : 0.0f;
}

/* ReLU mask bit = (z > 0) on the fp32 pre-activation ([P1] "Forward-pass
 * capabilities": relu_aux records which pre-ReLU values were positive) */
void oracle_relu_bits(const float* z, int64_t n, uint8_t* bits) {
  for (int64_t i = 0; i < n; ++i) bits[i] = z[i] > 0.0f ? 1u : 0u;
}

/* Pack bits[M][N] into column words: words[w][j] bit b = bits[32w+b][j],
 * bits of rows >= M left 0. words: [ceil(M/32)][N]. */
void oracle_pack_mask(const uint8_t* bits, int64_t M, int64_t N, uint32_t* words) {
  int64_t nw = (M + 31) / 32;
  for (int64_t w = 0; w < nw; ++w)
    for (int64_t j = 0; j < N; ++j) {
      uint32_t word = 0;
      for (int64_t b = 0; b < 32; ++b) {
        int64_t i = 32 * w + b;
        if (i < M && bits[i * N + j]) word |= (uint32_t)1u << b;
      }
      words[w * N + j] = word;
    }
}

/* Read back bit (i, j) of the column-word mask. */
int oracle_mask_bit(const uint32_t* words, int64_t N, int64_t i, int64_t j) {
  return (int)((words[(i / 32) * N + j] >> (i % 32)) & 1u);
}

/* dz = g where the forward mask bit is 1, else 0 ([P1] "Backward-pass path":
 * the ReLU mask applied to the multiplication result). Rows row_ids[r]
 * (NULL: r) of the mask. */
void oracle_drelu(const float* g, int64_t R, int64_t N, const int64_t* row_ids,
                  const uint32_t* words, float* dz) {
  for (int64_t r = 0; r < R; ++r) {
    int64_t gr = row_ids ? row_ids[r] : r;
    for (int64_t j = 0; j < N; ++j)
      dz[r * N + j] = oracle_mask_bit(words, N, gr, j) ? g[r * N + j] : 0.0f;
  }
}

/* bgrad[j] = sum over the batch (rows) of dz[i][j] ([P1] "Backward-pass path":
 * the column-wise sum used as the bias gradient). Double, ascending i. */
void oracle_colsum(const float* dz, int64_t M, int64_t N, double* out) {
  for (int64_t j = 0; j < N; ++j) out[j] = 0.0;
  for (int64_t i = 0; i < M; ++i)
    for (int64_t j = 0; j < N; ++j) out[j] += (double)dz[i * N + j];
}

/* ------------------------------------------------------------ GELU epilogs */
/* [P2] "other epilogs": GELU_BIAS = GELU(acc + bias). The tanh form of GELU
 * (Hendrycks & Gimpel, "Gaussian Error Linear Units", 2016, eq. for the tanh
 * approximation): gelu(z) = 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))).
 * Evaluated in double from the fp32 pre-activation. */
#define OR_GELU_K0 0.7978845608028654 /* sqrt(2/pi) */
#define OR_GELU_K1 0.044715

double oracle_gelu_tanh(double z) {
  double u = OR_GELU_K0 * (z + OR_GELU_K1 * z * z * z);
  return 0.5 * z * (1.0 + tanh(u));
}

/* d/dz of the tanh-form GELU:
 * 0.5 (1 + t) + 0.5 z (1 - t^2) sqrt(2/pi) (1 + 3 * 0.044715 z^2), t = tanh(u). */
double oracle_dgelu_tanh(double z) {
  double u = OR_GELU_K0 * (z + OR_GELU_K1 * z * z * z);
  double t = tanh(u);
  return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * OR_GELU_K0 * (1.0 + 3.0 * OR_GELU_K1 * z * z);
}

/* y = (float) gelu(z) elementwise */
void oracle_gelu(const float* z, int64_t n, float* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = (float)oracle_gelu_tanh((double)z[i]);
}

/* dz = (float) (g * gelu'(z)) elementwise: the GELU backward applied to the
 * product with the transposed weight, z being the saved pre-activation. */
void oracle_dgelu(const float* g, const float* z, int64_t n, float* dz) {
  for (int64_t i = 0; i < n; ++i) dz[i] = (float)((double)g[i] * oracle_dgelu_tanh((double)z[i]));
}

/* ------------------------------------------------------------------ SwiGLU */
/* [P3] "gemm_swiglu_mlp_fusion.py", module docstring: the forward fuses
 * silu(x Wg^T) * (x Wu^T) (gate GEMM + up GEMM + SiLU + mul), the down
 * projection is a separate GEMM, and the backward's dSwiGLU is fused as the
 * epilogue of matmul(dout, Wd) -> dh. silu(g) = g * sigmoid(g),
 * sigmoid(g) = 1 / (1 + exp(-g)). Evaluated in double from fp32 inputs. */
double oracle_sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

double oracle_silu(double g) { return g * oracle_sigmoid(g); }

/* h = (float) (silu(g) * u) elementwise */
void oracle_swiglu(const float* g, const float* u, int64_t n, float* h) {
  for (int64_t i = 0; i < n; ++i) h[i] = (float)(oracle_silu((double)g[i]) * (double)u[i]);
}

/* The derivatives of h = silu(g) * u, applied to dh:
 *   d_up   = dh * silu(g)
 *   d_gate = dh * u * sigmoid(g) * (1 + g * (1 - sigmoid(g)))
 * (d silu / dg = sigmoid(g) + g sigmoid(g) (1 - sigmoid(g))). */
void oracle_dswiglu(const float* dh, const float* g, const float* u, int64_t n, float* d_gate,
                    float* d_up) {
  for (int64_t i = 0; i < n; ++i) {
    double s = oracle_sigmoid((double)g[i]);
    d_up[i] = (float)((double)dh[i] * ((double)g[i] * s));
    d_gate[i] = (float)((double)dh[i] * (double)u[i] * s * (1.0 + (double)g[i] * (1.0 - s)));
  }
}
