/*
 * tq_oracle.h -- plain, slow, single-threaded CPU oracle for the ternary
 * FWHT-128 linear-layer path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this code; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code with the CUDA library.
 *
 * Pages cited (no page carries a title, so each is named by its address):
 *   [mhpq]  mhpq.cn/news/1159370  -- "Ternary Bonsai 2 27B" seen from TensorSharp
 *   [dpshk] dpshk.com/news/5289456
 *   [xxqk]  xxqk.cn/news/652513
 *   [zwxr]  zwxr.cn/news/303439
 *
 * Conventions: a weight matrix W is row-major [N][K] (out x in), an
 * activation matrix x is row-major [M][K], y is [M][N].  A "group" is 128
 * consecutive K indices of one row; G = K/128.  K must be a multiple of 128.
 */
#ifndef TQ_ORACLE_H
#define TQ_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* H[i][j] = (-1)^popcount(i & j)   ([dpshk] sec. 2.1). Returns +1 or -1. */
int tqo_hadamard_entry(int i, int j);

/* Sylvester construction H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]
 * ([dpshk] sec. 2.1; [mhpq] sec. 2.2), written into h[n*n] (n a power of 2,
 * n <= 128).  Independent of tqo_hadamard_entry; used to cross-check it. */
void tqo_sylvester(int n, int8_t *h);

/* fp32 constant c = RN_fp32(1/sqrt(128)); the bits are returned. */
uint32_t tqo_norm_const_bits(void);

/* 128-point FWHT in fp32, staged butterflies h = 1, 2, 4, ..., 64, each
 * stage mapping (a, b) -> (a + b, a - b) for every pair (i, i + h) with
 * (i & h) == 0, then one multiply of every element by c
 * ([xxqk] sec. 2, butterfly rounds; [mhpq] sec. 2.2).  in and out may alias. */
void tqo_fwht128_f32(const float *in, float *out);

/* Dense 128-point transform in fp64: out[i] = sum_j H[i][j] in[j] / sqrt(128),
 * H from the popcount definition.  Reference-quality rotation for y. */
void tqo_fwht128_f64(const double *in, double *out);

/* binary16 <-> binary32, round-to-nearest-even, written from the IEEE 754
 * formats (no tables, no hardware conversion). */
uint16_t tqo_f32_to_f16(float f);
float tqo_f16_to_f32(uint16_t h);

/* bfloat16 bits -> fp32 (exact widening). */
float tqo_bf16_to_f32(uint16_t b);

/* absmean ternarisation of one rotated group of 128 values ([mhpq] sec. 1.1,
 * 1.3):  sum |w'| by the halving tree (s[i] += s[i + h] for h = 64 .. 1, in
 * fp32), mean = sum * 2^-7, scale = fp16_RN(mean),
 * t = clamp(rint(w' / fp32(scale)), -1, 1) with IEEE fp32 division and
 * round-half-even; t = 0 throughout when scale == 0.  Returns the fp16 scale
 * bits; writes 128 trits. */
uint16_t tqo_quantize_group(const float *wrot, int8_t *t);

/* Whole matrix: for each row and each group, FWHT-128 in fp32, then
 * tqo_quantize_group.  W is fp32 (wt == 0) or bf16 bits (wt == 1), leading
 * dimension ldw elements.  T is [N][K] trits, S is [N][G] fp16 bits. */
void tqo_quantize_matrix(const void *W, int wt, int64_t N, int64_t K, int64_t ldw,
                         int8_t *T, uint16_t *S);

/* Same, for a list of rows only (T and S hold nrows rows). */
void tqo_quantize_rows(const void *W, int wt, int64_t K, int64_t ldw,
                       const int64_t *rows, int64_t nrows, int8_t *T, uint16_t *S);

/* 2-bit packing: code = t + 1 in bits 2*(k % 4) of byte k / 4 of the row;
 * rows ld2 bytes apart (ld2 >= K/4). */
void tqo_pack2(const int8_t *T, int64_t N, int64_t K, uint8_t *codes, int64_t ld2);
void tqo_unpack2(const uint8_t *codes, int64_t ld2, int64_t N, int64_t K, int8_t *T);

/* base-3 packing, five trits per byte: byte j of a row is
 * sum_{i=0..4} (t[5j+i] + 1) * 3^i; trits past K count as t = 0 (digit 1);
 * bytes from ceil(K/5) up to ld3 are 0. */
int64_t tqo_ld3(int64_t K);  /* ceil(K/5) rounded up to a multiple of 16 */
void tqo_pack3(const int8_t *T, int64_t N, int64_t K, uint8_t *codes, int64_t ld3);
void tqo_unpack3(const uint8_t *codes, int64_t ld3, int64_t N, int64_t K, int8_t *T);

/* y[m][n] = sum_g s[n][g] * sum_{k in g} t[n][k] * x'[m][k]  in fp64, where
 * x' is the fp64 dense rotation of the fp32 (bf16-exact) activations x.
 * rows == NULL means all N rows; else y is [M][nrows] for those rows and
 * T, S hold those rows only. */
void tqo_gemv_f64(const int8_t *T, const uint16_t *S, int64_t N, int64_t K,
                  const float *x, int64_t M, const int64_t *rows, int64_t nrows,
                  double *y);

/* Transform and group variants (see tq_oracle.c): n-point FWHT, n in
 * {64, 128, 256}, fp32 staged and fp64 dense; absmean over groups of
 * g in {128, 256}; quantisation under a (block, group, residual) layout and
 * its fp64 GEMV.  T has Keff = K (2K with residual) columns, S has
 * Geff = K/group (twice that with residual). */
uint32_t tqo_norm_const_bits_n(int n);
void tqo_fwht_f32(int n, const float *in, float *out);
void tqo_fwht_f64(int n, const double *in, double *out);
uint16_t tqo_quantize_group_n(int g, const float *wrot, int8_t *t);
void tqo_quantize_layout_rows(const void *W, int wt, int64_t K, int64_t ldw, const int64_t *rows,
                              int64_t nrows, int block, int group, int residual, int8_t *T,
                              uint16_t *S);
void tqo_gemv_layout_f64(const int8_t *T, const uint16_t *S, int64_t K, const float *x, int64_t M,
                         int64_t nrows, int block, int group, int residual, double *y);

/* ---- 2:4-sparse ternary weights ([mhpq] sec. 1.2: structured 2:4
 * sparsity -- two of every four weights kept, at regular positions -- and
 * the kept weights ternarised).
 *
 * Readings where the page leaves a step open (the plainest ones):
 *   - the pattern is chosen on the rotated weights w' (the matrix the
 *     ternary codes multiply), per quad of four consecutive k of a group;
 *   - the kept pair of a quad is its two largest |w'|, a tie going to the
 *     lower index;
 *   - "ternarise the remaining weights" is the absmean rule of [mhpq]
 *     sec. 1.1 applied to the 64 kept weights of the group: the scale is
 *     fp16_RN(mean |w'| over them), their sum taken by the halving tree over
 *     the kept values in k order (s[i] += s[i + h], h = 32 .. 1, fp32), then
 *     t = clamp(rint(w' / scale), -1, 1) as in tqo_quantize_group; a kept
 *     weight may round to 0; a pruned weight is 0.
 *
 * Storage (one tensor holding mask and trits together, as the page
 * describes, 24 bytes per group of 128):  quad j (k = 4j .. 4j + 3) of a
 * group has pattern p (its kept positions i0 < i1 in the order (0,1),
 * (0,2), (0,3), (1,2), (1,3), (2,3)) and code c = 9 p + 3 (t[i0] + 1) +
 * (t[i1] + 1), 0 <= c < 54.  The low four bits of c are nibble (j % 2) of
 * byte j / 2 of the group (bytes 0..15), its two high bits are bits
 * 2 (j % 4) .. of byte 16 + j / 4 (bytes 16..23).  A row holds its groups in
 * order: ld = 24 K / 128 bytes.  1.5 bits per weight plus 0.125 of scale.
 *
 * tqo_quantize_group_24: one rotated group -> dense t[128] (pruned = 0),
 * keep[128] (1 at kept positions), returns the fp16 scale bits.
 * tqo_quantize_rows_24: rows of W (fp32, wt = 0, or bf16 bits, wt = 1),
 * FWHT-128 per group (tqo_fwht128_f32), then the above; T, KEEP [nrows][K],
 * S [nrows][K/128].  tqo_pack24 / tqo_unpack24 convert (T, KEEP) to and
 * from the codes; tqo_unpack24 returns the number of codes >= 54 seen
 * (0 for a valid tensor; such quads decode as all zero). */
uint16_t tqo_quantize_group_24(const float *wrot, int8_t *t, uint8_t *keep);
void tqo_quantize_rows_24(const void *W, int wt, int64_t K, int64_t ldw, const int64_t *rows,
                          int64_t nrows, int8_t *T, uint8_t *KEEP, uint16_t *S);
int64_t tqo_ld24(int64_t K);
void tqo_pack24(const int8_t *T, const uint8_t *KEEP, int64_t N, int64_t K, uint8_t *codes,
                int64_t ld);
int64_t tqo_unpack24(const uint8_t *codes, int64_t ld, int64_t N, int64_t K, int8_t *T,
                     uint8_t *KEEP);

#ifdef __cplusplus
}
#endif
#endif
