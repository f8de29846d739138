/*
 * ORACLE -- test infrastructure, not product code.
 *
 * Plain, slow, fp64 CPU definition of block-sparse attention and of the
 * mask-to-CSR plan.  Only the tests, the smoke check and the bench's CPU
 * baseline leg may load this library; the product path never does.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes (per query row i of head (b, h)):
 *
 *   allowed(j) = mask[b][h][i/128][j/128] != 0  and  (not causal or j <= i)
 *   s_j        = scale * sum_d q[i][d] * k[j][d]      if allowed(j)
 *              = -inf                                  otherwise
 *   m          = max_j s_j
 *   if m == -inf:  O_i = 0,  LSE_i = -inf               (fully masked row)
 *   else:          w_j = exp(s_j - m),  l = sum_j w_j,
 *                  O_i = sum_j w_j v_j / l,  LSE_i = m + ln(l)
 *
 * Sources:
 *  - "Writing Pallas Kernels for JAX: Stepping Outside the XLA Safety Net",
 *    section "Writing the Kernel Logic: Load, Compute, Store": scaled scores
 *    q.k * 1/sqrt(head_dim), masked entries pushed to -inf before the softmax,
 *    softmax over the key axis, then the weighted sum of V.
 *  - same page, "Designing the Block Specification": 128-token query blocks,
 *    and a block mask loaded per (query block, key block) pair.
 *  - "Pallas-Triton kernels and kernel auto-tuning", section "Flash
 *    Attention": the tiled algorithm computes attention exactly, so the
 *    softmax here is taken over ALL live keys of the row at once (the page-2
 *    sketch sums per-block softmaxes, which is only exact for one live block
 *    per row; the exact reading is the one used).
 *  - Fully masked rows (O = 0, LSE = -inf), the causal flag (element-level
 *    j <= i on top of the block mask) and LSE itself are not on the pages;
 *    they are this library's stated definitions.
 *
 * The score row is materialised in full (length S, -inf where not allowed),
 * as the plain definition has it; no tiling, no online softmax, no blocking.
 * Accumulation is sequential in double.  Inputs are bf16 bit patterns
 * (widened exactly) or doubles.
 *
 * oracle_set_mutation() plants a known mistake (test-only switch, default 0)
 * so that the tests can show each pin catches at least one plausible error.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BLOCK 128

static int g_mutation = 0;

void oracle_set_mutation(int m) { g_mutation = m; }
int oracle_get_mutation(void) { return g_mutation; }

/* bf16 bit pattern -> double, exact: the bf16 bits are the top half of a float. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double load(const void* base, int kind, int64_t idx) {
  if (kind == 0) return bf16_bits_to_double(((const uint16_t*)base)[idx]);
  return ((const double*)base)[idx];
}

static int is_allowed(const uint8_t* mask, int64_t bh, int nb, int64_t i, int64_t j, int causal) {
  int64_t qblk = i / ORACLE_BLOCK, kblk = j / ORACLE_BLOCK;
  if (g_mutation == 3) { int64_t t = qblk; qblk = kblk; kblk = t; }   /* transposed mask */
  if (!mask[(bh * nb + qblk) * nb + kblk]) return 0;
  if (causal && g_mutation != 14) {
    if (g_mutation == 4) return j < i;                                 /* strict causal */
    return j <= i;
  }
  return 1;
}

/*
 * Attention for a list of query rows.
 *   in_kind: 0 = q/k/v are uint16 bf16 bit patterns, 1 = doubles.
 *   q, k, v: [B][H][S][D];  mask: uint8 [B][H][S/128][S/128].
 *   rows[r] = (b*H + h)*S + i  (flat row id);  O: [n_rows][D];  LSE: [n_rows].
 * Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 */
int oracle_attn_rows(int in_kind, const void* q, const void* k, const void* v,
                     const uint8_t* mask, int B, int H, int S, int D, double scale,
                     int causal, const int64_t* rows, int64_t n_rows, double* O,
                     double* LSE, int nthreads) {
  if (B <= 0 || H <= 0 || S <= 0 || D <= 0 || (S % ORACLE_BLOCK) != 0) return -1;
  if (!q || !k || !v || !mask || !rows || !O || !LSE || n_rows < 0) return -1;
  const int nb = S / ORACLE_BLOCK;
  const int64_t total_rows = (int64_t)B * H * S;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= total_rows) return -1;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)S);
    double* qi = (double*)malloc(sizeof(double) * (size_t)D);
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    if (!s || !qi || !acc) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t flat = rows[r];
        const int64_t bh = flat / S;
        const int64_t i = flat % S;
        const int64_t head0 = bh * (int64_t)S;          /* first row of this head */
        for (int d = 0; d < D; ++d) qi[d] = load(q, in_kind, (head0 + i) * D + d);

        /* 1. scores, masked to -inf (the full length-S row) */
        for (int64_t j = 0; j < S; ++j) {
          if (!is_allowed(mask, bh, nb, i, j, causal)) { s[j] = -INFINITY; continue; }
          double dot = 0.0;
          const int dlim = (g_mutation == 10) ? D - 1 : D;           /* dropped term */
          for (int d = 0; d < dlim; ++d) {
            const void* kb = (g_mutation == 7) ? q : k;                /* wrong operand */
            dot += qi[d] * load(kb, in_kind, (head0 + j) * D + d);
          }
          s[j] = (g_mutation == 1) ? dot : scale * dot;              /* scale dropped */
        }

        /* 2. row max */
        double m = -INFINITY;
        for (int64_t j = 0; j < S; ++j) if (s[j] > m) m = s[j];

        double* o = O + r * (int64_t)D;
        if (m == -INFINITY && g_mutation != 9) {
          for (int d = 0; d < D; ++d) o[d] = 0.0;
          LSE[r] = -INFINITY;
          continue;
        }

        /* 3. softmax weights and weighted sum of V */
        double l = 0.0;
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        for (int64_t j = 0; j < S; ++j) {
          if (s[j] == -INFINITY && g_mutation != 9) continue;          /* exp(-inf) = 0 */
          const double w = (g_mutation == 2) ? exp(m - s[j]) : exp(s[j] - m);
          l += w;
          const int64_t vrow = (g_mutation == 8) ? i : j;              /* wrong V row */
          for (int d = 0; d < D; ++d) acc[d] += w * load(v, in_kind, (head0 + vrow) * D + d);
        }
        for (int d = 0; d < D; ++d) o[d] = (g_mutation == 6) ? acc[d] : acc[d] / l;
        if (g_mutation == 5) LSE[r] = log(l);
        else if (g_mutation == 11) LSE[r] = m + log2(l);
        else LSE[r] = m + log(l);
      }
    }
    free(s);
    free(qi);
    free(acc);
  }
  return failed ? -2 : 0;
}

/*
 * Plan oracle: per (b, h, query block qb), the ascending list of key blocks
 * kb with mask != 0 (and kb <= qb when causal).  Row index = (b*H + h)*nb + qb.
 * row_ptr has B*H*nb + 1 entries.  col_idx may be NULL (count only).
 * Returns nnz, or -1 on bad arguments.
 */
int64_t oracle_csr(const uint8_t* mask, int B, int H, int nb, int causal,
                   int32_t* row_ptr, int32_t* col_idx) {
  if (!mask || !row_ptr || B <= 0 || H <= 0 || nb <= 0) return -1;
  int64_t nnz = 0;
  const int64_t nrows = (int64_t)B * H * nb;
  for (int64_t row = 0; row < nrows; ++row) {
    row_ptr[row] = (int32_t)nnz;
    const int64_t qb = row % nb;
    for (int64_t kb = 0; kb < nb; ++kb) {
      if (!mask[row * nb + kb]) continue;
      if (causal && kb > qb) continue;
      if (col_idx) col_idx[nnz] = (int32_t)kb;
      ++nnz;
    }
  }
  row_ptr[nrows] = (int32_t)nnz;
  return nnz;
}
