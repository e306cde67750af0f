/*
 * oracle.c -- plain CPU reference for the W4A16 fused matrix multiply
 *             Y = X . dequant(W)
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it follows (pages on Marlin, cited by title and section):
 *   - "Marlin / GPTQ-Marlin" (brain.gartu.xyz), section "Le problème": each
 *     linear layer computes Y = X_fp16 x W_int4, dequantising the INT4 weights
 *     to FP16 on the fly before the multiply.
 *   - "Marlin" (dingiv.github.io), section "Group size 为什么是 128": one scale (and one
 *     zero point) per group of 128 consecutive weights.
 *   - same page, section "反量化精度权衡": INT4 -> FP16 is exact (FP16 holds
 *     all 16 values), the multiply accumulates in FP32 and the output is FP16.
 *
 * The oracle computes the plain definition, with no blocking or reordering:
 *   1. q[k][n] = nibble (k mod 8) of Qp[k/8][n]                 (GPTQ order)
 *   2. z[j][n] = nibble (n mod 8) of Zp[j][n/8], or 8 when no zeros are given
 *   3. w[k][n] = fp16_rne( (q - z) * s[k/g][n] )   -- one rounding, exact
 *                product taken in double (|q-z| <= 15 times an fp16 value is
 *                exact in binary64)
 *   4. y[m][n] = sum_k x[m][k] * w[k][n], in binary64, k ascending
 * plus the tile layout of the repacked weights (the "reshuffle" of the pages:
 * "Marlin / GPTQ-Marlin", section "Tiled layout et repacking"; "Marlin Project
 * Overview" (vecbase.com), section "Key Techniques", item "Reshuffling for Access Patterns").  The
 * repacked layout is this library's own, the operand order of a 16x16 fp16
 * tensor-core fragment; its index formula is:
 *   codes: word ((nt*(K/64) + kb)*8 + g)*128 + l*4 + j   (nt < N/128, kb < K/64,
 *          g < 8, l < 32, j < 4) holds at bits 4p..4p+3 (p = 0..7) the code
 *          q[k][n] with n = nt*128 + 16g + l/4 + 8*(p & 1),
 *                      k = kb*64 + 16j + 4*(l % 4) + 2*((p >> 1) & 1) + (p >> 2);
 *   scales: fp16 [N/128][K/g][128], scale (gi, n) at ((n/128)*(K/g) + gi)*128 + n%128;
 *   zeros:  bytes [N/128][K/g][64], the 64-byte slice Zp[gi][16*(n/128) .. +15]
 *           at ((n/128)*(K/g) + gi)*64.
 *
 * 2:4 structured sparsity ("Marlin", section "支持 2:4 稀疏加速"; "Marlin /
 * GPTQ-Marlin", section "4. Support de la sparsité 2:4 NVIDIA"): the compressed
 * form of 2:4 codes, its inverse, the product over the kept terms only, and
 * the library's sparse tile layout (section "2:4 structured sparsity" below).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread (no FMA contraction,
 * so every sum rounds after each add, identically on x86-64 and aarch64).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- IEEE-754 binary16 <-> binary64 (own bit-level routines) ----------- */

/* Exact value of a binary16 bit pattern. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 0x1F) {
    v = f ? NAN : INFINITY;
  } else if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
  } else {
    v = ldexp((double)(1024 + f), e - 25); /* (1024+f) * 2^(e-15-10) */
  }
  return sign ? -v : v;
}

/* Round a binary64 value to the nearest binary16, ties to even, with
 * gradual underflow and overflow to infinity.  Every step below is exact in
 * binary64 except rint(), which performs the single round-to-nearest-even. */
uint16_t oracle_double_to_half_rne(double v) {
  if (isnan(v)) return 0x7E00;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  /* 65504 is the largest finite half; 65520 is the midpoint to 2^16 and rounds
   * to the even neighbour 2^16, i.e. overflows. */
  if (a >= 65520.0) return sign | 0x7C00;
  int E;
  frexp(a, &E);            /* a = f * 2^E, f in [0.5, 1) */
  int e = E - 1;           /* a in [2^e, 2^(e+1)) */
  if (e < -14) {           /* subnormal range: quantum 2^-24 */
    double n = rint(ldexp(a, 24));
    return sign | (uint16_t)n; /* n == 1024 is the smallest normal, 0x0400 */
  }
  double n = rint(ldexp(a, 10 - e)); /* in [1024, 2048] */
  if (n >= 2048.0) { n = 1024.0; e += 1; }
  if (e > 15) return sign | 0x7C00;
  return sign | (uint16_t)(((e + 15) << 10) | ((int)n - 1024));
}

/* ---- steps 1-3: unpack and dequantise ---------------------------------- */

static inline int code_at(const int32_t* Qp, int N, int k, int n) {
  uint32_t word = (uint32_t)Qp[(size_t)(k / 8) * N + n];
  return (int)((word >> (4 * (k % 8))) & 0xFu);
}

static inline int zero_at(const int32_t* Zp, int N, int j, int n) {
  if (!Zp) return 8;
  uint32_t word = (uint32_t)Zp[(size_t)j * (N / 8) + n / 8];
  return (int)((word >> (4 * (n % 8))) & 0xFu);
}

/* q[k*N + n] for k < K, n < N. */
int oracle_unpack_codes(const int32_t* Qp, int K, int N, uint8_t* q) {
  if (K % 8 || K <= 0 || N <= 0) return 1;
  for (int k = 0; k < K; ++k)
    for (int n = 0; n < N; ++n) q[(size_t)k * N + n] = (uint8_t)code_at(Qp, N, k, n);
  return 0;
}

/* z[j*N + n] for j < G, n < N (8 everywhere when Zp is NULL). */
int oracle_unpack_zeros(const int32_t* Zp, int G, int N, uint8_t* z) {
  if (G <= 0 || N % 8) return 1;
  for (int j = 0; j < G; ++j)
    for (int n = 0; n < N; ++n) z[(size_t)j * N + n] = (uint8_t)zero_at(Zp, N, j, n);
  return 0;
}

/* w = fp16_rne((q - z) * s) for one weight. */
static inline uint16_t dequant_one(int q, int z, uint16_t s_bits) {
  double prod = (double)(q - z) * oracle_half_to_double(s_bits);
  return oracle_double_to_half_rne(prod);
}

uint16_t oracle_dequant_scalar(int q, int z, uint16_t s_bits) { return dequant_one(q, z, s_bits); }

/* W[k*N + n] (fp16 bits) = dequant of the whole K x N matrix.
 * S is [K/g][N] fp16 bits, Zp is [K/g][N/8] packed zeros or NULL. */
int oracle_dequant(const int32_t* Qp, const uint16_t* S, const int32_t* Zp, int K, int N, int g,
                   uint16_t* W) {
  if (K % 8 || N % 8 || g <= 0 || K % g) return 1;
  for (int k = 0; k < K; ++k) {
    int j = k / g;
    for (int n = 0; n < N; ++n)
      W[(size_t)k * N + n] = dequant_one(code_at(Qp, N, k, n), zero_at(Zp, N, j, n),
                                         S[(size_t)j * N + n]);
  }
  return 0;
}

/* ---- step 4: fp64 matrix multiply --------------------------------------- */

typedef struct {
  const uint16_t* X;
  const uint16_t* W;
  int M, K, N, n0, n1;
  double* Y;
} gemm_job;

static void* gemm_worker(void* arg) {
  gemm_job* j = (gemm_job*)arg;
  int K = j->K, N = j->N;
  double* wcol = (double*)malloc(sizeof(double) * K);
  for (int n = j->n0; n < j->n1; ++n) {
    for (int k = 0; k < K; ++k) wcol[k] = oracle_half_to_double(j->W[(size_t)k * N + n]);
    for (int m = 0; m < j->M; ++m) {
      const uint16_t* x = j->X + (size_t)m * K;
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += oracle_half_to_double(x[k]) * wcol[k];
      j->Y[(size_t)m * N + n] = acc;
    }
  }
  free(wcol);
  return NULL;
}

/* Y[m*N + n] = sum_k X[m][k] * W[k][n] in binary64, k ascending.
 * Threads split the columns; each column's sums are the same whatever the
 * thread count. */
int oracle_gemm(const uint16_t* X, const uint16_t* W, int M, int K, int N, double* Y, int nthreads) {
  if (M < 0 || K <= 0 || N <= 0) return 1;
  if (M == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > N) nthreads = N;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
  gemm_job* jobs = (gemm_job*)malloc(sizeof(gemm_job) * nthreads);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (gemm_job){X, W, M, K, N, (int)((long long)N * t / nthreads),
                         (int)((long long)N * (t + 1) / nthreads), Y};
    pthread_create(&th[t], NULL, gemm_worker, &jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

/* ---- the whole definition, straight from the packed inputs ------------- */

typedef struct {
  const uint16_t* X;
  const int32_t* Qp;
  const uint16_t* S;
  const int32_t* Zp;
  int M, K, N, g;
  const int64_t* idx; /* flat indices m*N + n; NULL = every entry */
  int64_t i0, i1;
  double* out;
} w4a16_job;

/* y[m][n] for one (m, n): dequantise column n (steps 1-3) and sum (step 4). */
static double entry(const w4a16_job* j, int m, int n) {
  const uint16_t* x = j->X + (size_t)m * j->K;
  double acc = 0.0;
  for (int k = 0; k < j->K; ++k) {
    int grp = k / j->g;
    uint16_t w = dequant_one(code_at(j->Qp, j->N, k, n), zero_at(j->Zp, j->N, grp, n),
                             j->S[(size_t)grp * j->N + n]);
    acc += oracle_half_to_double(x[k]) * oracle_half_to_double(w);
  }
  return acc;
}

static void* w4a16_worker(void* arg) {
  w4a16_job* j = (w4a16_job*)arg;
  if (j->idx) {
    for (int64_t i = j->i0; i < j->i1; ++i) {
      int64_t f = j->idx[i];
      j->out[i] = entry(j, (int)(f / j->N), (int)(f % j->N));
    }
  } else {
    /* whole rows of columns: i indexes columns n, all m */
    for (int64_t n = j->i0; n < j->i1; ++n)
      for (int m = 0; m < j->M; ++m) j->out[(size_t)m * j->N + n] = entry(j, m, (int)n);
  }
  return NULL;
}

/* Y (or the listed entries) of Y = X . dequant(W), computed from the packed
 * GPTQ-order inputs.  idx == NULL: out is [M][N]; else out[i] = y at flat
 * index idx[i] = m*N + n. */
int oracle_w4a16(const uint16_t* X, const int32_t* Qp, const uint16_t* S, const int32_t* Zp, int M,
                 int K, int N, int g, const int64_t* idx, int64_t count, double* out, int nthreads) {
  if (M < 0 || K <= 0 || N <= 0 || K % 8 || N % 8 || g <= 0 || K % g) return 1;
  if (M == 0) return 0;
  int64_t total = idx ? count : N;
  if (total <= 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > total) nthreads = (int)total;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
  w4a16_job* jobs = (w4a16_job*)malloc(sizeof(w4a16_job) * nthreads);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (w4a16_job){X, Qp, S, Zp, M, K, N, g, idx, total * t / nthreads,
                          total * (t + 1) / nthreads, out};
    pthread_create(&th[t], NULL, w4a16_worker, &jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

/* ---- repacked tile layout ------------------------------------------------ */

/* Row (within the 128-column tile) and k (within the 64-row block) of nibble p
 * of the word at (g, l, j) of a chunk. */
static inline int frag_row(int g, int l, int p) { return 16 * g + l / 4 + 8 * (p & 1); }
static inline int frag_k(int l, int j, int p) { return 16 * j + 4 * (l % 4) + 2 * ((p >> 1) & 1) + (p >> 2); }

/* Qp [K/8][N] GPTQ order -> P [(N/128)*(K/64)*1024] words, tile layout. */
int oracle_repack(const int32_t* Qp, int K, int N, int32_t* P) {
  if (K <= 0 || N <= 0 || K % 64 || N % 128) return 1;
  int KB = K / 64, NT = N / 128;
  for (int nt = 0; nt < NT; ++nt)
    for (int kb = 0; kb < KB; ++kb)
      for (int g = 0; g < 8; ++g)
        for (int l = 0; l < 32; ++l)
          for (int j = 0; j < 4; ++j) {
            uint32_t word = 0;
            for (int p = 0; p < 8; ++p) {
              int k = kb * 64 + frag_k(l, j, p);
              int n = nt * 128 + frag_row(g, l, p);
              word |= (uint32_t)code_at(Qp, N, k, n) << (4 * p);
            }
            size_t at = ((size_t)(nt * KB + kb) * 8 + g) * 128 + (size_t)l * 4 + j;
            P[at] = (int32_t)word;
          }
  return 0;
}

/* Inverse of oracle_repack: tile layout -> GPTQ order. */
int oracle_unrepack(const int32_t* P, int K, int N, int32_t* Qp) {
  if (K <= 0 || N <= 0 || K % 64 || N % 128) return 1;
  int KB = K / 64, NT = N / 128;
  memset(Qp, 0, sizeof(int32_t) * (size_t)(K / 8) * N);
  for (int nt = 0; nt < NT; ++nt)
    for (int kb = 0; kb < KB; ++kb)
      for (int g = 0; g < 8; ++g)
        for (int l = 0; l < 32; ++l)
          for (int j = 0; j < 4; ++j) {
            size_t at = ((size_t)(nt * KB + kb) * 8 + g) * 128 + (size_t)l * 4 + j;
            uint32_t word = (uint32_t)P[at];
            for (int p = 0; p < 8; ++p) {
              int k = kb * 64 + frag_k(l, j, p);
              int n = nt * 128 + frag_row(g, l, p);
              uint32_t q = (word >> (4 * p)) & 0xFu;
              Qp[(size_t)(k / 8) * N + n] |= (int32_t)(q << (4 * (k % 8)));
            }
          }
  return 0;
}

/* Scales [G][N] fp16 bits -> tile-major [N/128][G][128]. */
int oracle_repack_scales(const uint16_t* S, int G, int N, uint16_t* out) {
  if (G <= 0 || N <= 0 || N % 128) return 1;
  for (int gi = 0; gi < G; ++gi)
    for (int n = 0; n < N; ++n)
      out[((size_t)(n / 128) * G + gi) * 128 + n % 128] = S[(size_t)gi * N + n];
  return 0;
}

/* Packed zeros [G][N/8] int32 -> tile-major bytes [N/128][G][64]. */
int oracle_repack_zeros(const int32_t* Zp, int G, int N, uint8_t* out) {
  if (G <= 0 || N <= 0 || N % 128) return 1;
  for (int gi = 0; gi < G; ++gi)
    for (int n = 0; n < N; ++n) {
      int z = zero_at(Zp, N, gi, n);
      uint8_t* b = out + ((size_t)(n / 128) * G + gi) * 64 + (n % 128) / 2;
      if (n % 2 == 0) *b = (uint8_t)((*b & 0xF0) | z);
      else *b = (uint8_t)((*b & 0x0F) | (z << 4));
    }
  return 0;
}

/* ---- 2:4 structured sparsity ---------------------------------------------
 *
 * "Marlin" (dingiv.github.io), section "支持 2:4 稀疏加速": in every four
 * weights two are zero, at positions fixed ahead of inference; "Marlin /
 * GPTQ-Marlin" (brain.gartu.xyz), section "4. Support de la sparsité 2:4
 * NVIDIA": the zeros are skipped after dequantisation and the sparse tensor
 * core multiplies only the kept half.
 *
 * Readings (the pages fix neither): a dequantised weight is zero exactly when
 * its code equals its zero point z (w = (q - z)*s); the four weights of a group
 * are four consecutive rows k = 4j .. 4j+3 of one column n, i.e. along the
 * reduction, which is the direction the sparse tensor core compresses.
 *
 * Compressed form, for every (j, n): kept positions i0 < i1 in 0..3 are the
 * positions whose code differs from z, in ascending order, completed (when
 * there are fewer than two) with the lowest positions whose code equals z; the
 * kept codes are c_t = q[4j + i_t][n].  Stored as kc[(2j + t)*N + n] = c_t and
 * ki[j*N + n] = i0 | (i1 << 2).  A group with three or four codes that differ
 * from z is not 2:4; it is counted and keeps its first two such positions.
 *
 * The sparse product is the dense one on the expanded codes, since every
 * dropped weight dequantises to exactly zero; oracle_w4a16_sparse sums only
 * the kept terms, j ascending and i0 before i1, i.e. k ascending. */

static inline int zero_for(const int32_t* Zp, int N, int g, int k, int n) {
  return zero_at(Zp, N, k / g, n);
}

int oracle_sparse_compress(const int32_t* Qp, const int32_t* Zp, int K, int N, int g, uint8_t* kc,
                           uint8_t* ki) {
  if (K <= 0 || N <= 0 || K % 8 || N % 8 || g <= 0 || K % g || g % 4) return -1;
  int bad = 0;
  for (int j = 0; j < K / 4; ++j)
    for (int n = 0; n < N; ++n) {
      int z = zero_for(Zp, N, g, 4 * j, n);
      int pos[4], cnt = 0;
      for (int i = 0; i < 4; ++i)
        if (code_at(Qp, N, 4 * j + i, n) != z && cnt < 2) pos[cnt++] = i;
      int nz = 0;
      for (int i = 0; i < 4; ++i) nz += code_at(Qp, N, 4 * j + i, n) != z;
      if (nz > 2) ++bad;
      /* complete with the lowest positions not yet taken */
      for (int i = 0; i < 4 && cnt < 2; ++i) {
        int taken = 0;
        for (int c = 0; c < cnt; ++c) taken |= pos[c] == i;
        if (!taken) pos[cnt++] = i;
      }
      if (pos[0] > pos[1]) { int t = pos[0]; pos[0] = pos[1]; pos[1] = t; }
      kc[(size_t)(2 * j) * N + n] = (uint8_t)code_at(Qp, N, 4 * j + pos[0], n);
      kc[(size_t)(2 * j + 1) * N + n] = (uint8_t)code_at(Qp, N, 4 * j + pos[1], n);
      ki[(size_t)j * N + n] = (uint8_t)(pos[0] | (pos[1] << 2));
    }
  return bad;
}

/* Dense GPTQ-order codes from the compressed form: z at the dropped rows. */
int oracle_sparse_expand(const uint8_t* kc, const uint8_t* ki, const int32_t* Zp, int K, int N, int g,
                         int32_t* Qp) {
  if (K <= 0 || N <= 0 || K % 8 || N % 8 || g <= 0 || K % g || g % 4) return 1;
  memset(Qp, 0, sizeof(int32_t) * (size_t)(K / 8) * N);
  for (int j = 0; j < K / 4; ++j)
    for (int n = 0; n < N; ++n) {
      int i0 = ki[(size_t)j * N + n] & 3, i1 = (ki[(size_t)j * N + n] >> 2) & 3;
      if (i0 >= i1) return 2;
      for (int i = 0; i < 4; ++i) {
        int k = 4 * j + i;
        int q = zero_for(Zp, N, g, k, n);
        if (i == i0) q = kc[(size_t)(2 * j) * N + n];
        if (i == i1) q = kc[(size_t)(2 * j + 1) * N + n];
        Qp[(size_t)(k / 8) * N + n] |= (int32_t)((uint32_t)(q & 0xF) << (4 * (k % 8)));
      }
    }
  return 0;
}

typedef struct {
  const uint16_t* X;
  const uint8_t *kc, *ki;
  const uint16_t* S;
  const int32_t* Zp;
  int M, K, N, g;
  const int64_t* idx;
  int64_t i0, i1;
  double* out;
} sparse_job;

static double sparse_entry(const sparse_job* j, int m, int n) {
  const uint16_t* x = j->X + (size_t)m * j->K;
  double acc = 0.0;
  for (int jj = 0; jj < j->K / 4; ++jj) {
    uint8_t code_idx = j->ki[(size_t)jj * j->N + n];
    for (int t = 0; t < 2; ++t) {
      int k = 4 * jj + ((code_idx >> (2 * t)) & 3);
      int grp = k / j->g;
      uint16_t w = dequant_one(j->kc[(size_t)(2 * jj + t) * j->N + n], zero_at(j->Zp, j->N, grp, n),
                               j->S[(size_t)grp * j->N + n]);
      acc += oracle_half_to_double(x[k]) * oracle_half_to_double(w);
    }
  }
  return acc;
}

static void* sparse_worker(void* arg) {
  sparse_job* j = (sparse_job*)arg;
  if (j->idx) {
    for (int64_t i = j->i0; i < j->i1; ++i) {
      int64_t f = j->idx[i];
      j->out[i] = sparse_entry(j, (int)(f / j->N), (int)(f % j->N));
    }
  } else {
    for (int64_t n = j->i0; n < j->i1; ++n)
      for (int m = 0; m < j->M; ++m) j->out[(size_t)m * j->N + n] = sparse_entry(j, m, (int)n);
  }
  return NULL;
}

/* Y (or the listed entries) of X . dequant(W) for 2:4 weights in compressed
 * form, summing the kept terms only. */
int oracle_w4a16_sparse(const uint16_t* X, const uint8_t* kc, const uint8_t* ki, const uint16_t* S,
                        const int32_t* Zp, int M, int K, int N, int g, const int64_t* idx,
                        int64_t count, double* out, int nthreads) {
  if (M < 0 || K <= 0 || N <= 0 || K % 8 || N % 8 || g <= 0 || K % g || g % 4) return 1;
  if (M == 0) return 0;
  int64_t total = idx ? count : N;
  if (total <= 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > total) nthreads = (int)total;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
  sparse_job* jobs = (sparse_job*)malloc(sizeof(sparse_job) * nthreads);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (sparse_job){X, kc, ki, S, Zp, M, K, N, g, idx, total * t / nthreads,
                           total * (t + 1) / nthreads, out};
    pthread_create(&th[t], NULL, sparse_worker, &jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

/* The library's tile layout of the compressed form (its own: the operand
 * order of the sparse 16x32 fp16 tensor-core fragment).  Per 128-column tile
 * nt and 64-row block kb (16 groups of four rows):
 *   codes: word ((nt*(K/64) + kb)*8 + gq)*64 + l*2 + s  (gq < 8, l < 32, s < 2)
 *          holds at bits 4p..4p+3 (p < 8) the kept code c_t(j, n) with
 *          n = nt*128 + 16gq + l/4 + 8*(p & 1),
 *          j = kb*16 + 8s + l%4 + 4*((p >> 1) & 1),   t = p >> 2;
 *   meta:  word ((nt*(K/64) + kb)*8 + gq)*32 + (r*2 + h)*2 + s  (r < 8, h < 2, s < 2)
 *          holds at bits 4i..4i+3 (i < 8) the index nibble ki(j, n) with
 *          n = nt*128 + 16gq + r + 8*(i >> 2),   j = kb*16 + 8s + 4h + (i & 3). */
static inline int sp_code_n(int nt, int gq, int l, int p) { return nt * 128 + 16 * gq + l / 4 + 8 * (p & 1); }
static inline int sp_code_j(int kb, int l, int s, int p) { return kb * 16 + 8 * s + l % 4 + 4 * ((p >> 1) & 1); }
static inline int sp_meta_n(int nt, int gq, int r, int i) { return nt * 128 + 16 * gq + r + 8 * (i >> 2); }
static inline int sp_meta_j(int kb, int h, int s, int i) { return kb * 16 + 8 * s + 4 * h + (i & 3); }

int oracle_sparse_repack(const uint8_t* kc, const uint8_t* ki, int K, int N, int32_t* Pc, int32_t* Pm) {
  if (K <= 0 || N <= 0 || K % 64 || N % 128) return 1;
  int KB = K / 64, NT = N / 128;
  for (int nt = 0; nt < NT; ++nt)
    for (int kb = 0; kb < KB; ++kb)
      for (int gq = 0; gq < 8; ++gq) {
        size_t blk = (size_t)(nt * KB + kb) * 8 + gq;
        for (int l = 0; l < 32; ++l)
          for (int s = 0; s < 2; ++s) {
            uint32_t word = 0;
            for (int p = 0; p < 8; ++p) {
              int n = sp_code_n(nt, gq, l, p), j = sp_code_j(kb, l, s, p);
              word |= (uint32_t)(kc[(size_t)(2 * j + (p >> 2)) * N + n] & 0xF) << (4 * p);
            }
            Pc[blk * 64 + (size_t)l * 2 + s] = (int32_t)word;
          }
        for (int r = 0; r < 8; ++r)
          for (int h = 0; h < 2; ++h)
            for (int s = 0; s < 2; ++s) {
              uint32_t word = 0;
              for (int i = 0; i < 8; ++i) {
                int n = sp_meta_n(nt, gq, r, i), j = sp_meta_j(kb, h, s, i);
                word |= (uint32_t)(ki[(size_t)j * N + n] & 0xF) << (4 * i);
              }
              Pm[blk * 32 + (size_t)(r * 2 + h) * 2 + s] = (int32_t)word;
            }
      }
  return 0;
}

/* Inverse of oracle_sparse_repack. */
int oracle_sparse_unrepack(const int32_t* Pc, const int32_t* Pm, int K, int N, uint8_t* kc, uint8_t* ki) {
  if (K <= 0 || N <= 0 || K % 64 || N % 128) return 1;
  int KB = K / 64, NT = N / 128;
  for (int nt = 0; nt < NT; ++nt)
    for (int kb = 0; kb < KB; ++kb)
      for (int gq = 0; gq < 8; ++gq) {
        size_t blk = (size_t)(nt * KB + kb) * 8 + gq;
        for (int l = 0; l < 32; ++l)
          for (int s = 0; s < 2; ++s) {
            uint32_t word = (uint32_t)Pc[blk * 64 + (size_t)l * 2 + s];
            for (int p = 0; p < 8; ++p) {
              int n = sp_code_n(nt, gq, l, p), j = sp_code_j(kb, l, s, p);
              kc[(size_t)(2 * j + (p >> 2)) * N + n] = (uint8_t)((word >> (4 * p)) & 0xF);
            }
          }
        for (int r = 0; r < 8; ++r)
          for (int h = 0; h < 2; ++h)
            for (int s = 0; s < 2; ++s) {
              uint32_t word = (uint32_t)Pm[blk * 32 + (size_t)(r * 2 + h) * 2 + s];
              for (int i = 0; i < 8; ++i) {
                int n = sp_meta_n(nt, gq, r, i), j = sp_meta_j(kb, h, s, i);
                ki[(size_t)j * N + n] = (uint8_t)((word >> (4 * i)) & 0xF);
              }
            }
      }
  return 0;
}

/* Element-wise fp16_rne of n binary64 values (bits out). */
void oracle_round_array(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_half_rne(v[i]);
}

/* Element-wise exact value of n binary16 bit patterns. */
void oracle_widen_array(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(h[i]);
}
