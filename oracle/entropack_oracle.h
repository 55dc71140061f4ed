/*
 * Plain CPU oracle for the EntroPack codec.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header or table with the CUDA library.
 *
 * Method passages followed ("EntroPack: Fast and Accurate Entropy-Coded
 * Weight Compression at Arbitrary Bitrates", Abstract):
 *   row-normalised E8 lattice quantisation        -> oracle_row_rms, oracle_e8_nearest
 *   coordinate probability model given the coset  -> oracle_block_symbols
 *   resolution picked from sampled rate estimates -> oracle_estimate_bpp, oracle_select_j
 *   entropy coding in independently decodable tiles -> oracle_rans_*, oracle_encode
 *   fused decode + reconstruction into BF16/FP16/FP8/INT8 -> oracle_decode
 * Lossless tiled ANS ("EntroPack PyTorch Guide", section "Choose a
 * compression contract", TileANSConfig) -> oracle_encode_lossless.
 * Comparators of the evaluation (Abstract: lower relative L2 weight error
 * than NF4 at a 4-bit target, with less storage, and than fixed-width codes
 * of about the same size) -> oracle_q4_roundtrip with oracle_nf4_levels /
 * oracle_int4_levels, oracle_fp8_row_roundtrip.
 * The stream layout and every constant are this repository's readings of
 * those passages (stream format version 1).
 *
 * Parity pins (tests/test_oracle_*.py): brute-force E8 search, the E8
 * second moment 929/12960, rANS round trip and code-length bounds,
 * conversions against torch, the Gaussian rate-distortion closed form,
 * bitwise lossless recovery, NF4 levels through the normal CDF, brute-force
 * 4-bit quantisation, E4M3 decoding against torch, the rate search's chosen
 * resolution index against an exhaustive scan of every admissible index.
 */
#ifndef ENTROPACK_ORACLE_H
#define ENTROPACK_ORACLE_H
#include <stddef.h>
#include <stdint.h>

/* nearest point of E8 to x; writes the integer coordinates a[8] and the coset */
void oracle_e8_nearest(const double x[8], int64_t a[8], int *coset);

double oracle_row_rms(const uint16_t *w_row, int64_t K);
double oracle_delta(int j);
double oracle_rn7(double v);
double oracle_tr7(double v);

/* 12-bit normaliser of 256 counts */
void oracle_normalize(const uint64_t counts[256], uint32_t freq[256]);

/* rANS on one lane: syms/ freqs given; words written in decode order */
int oracle_rans_encode(const uint8_t *syms, const uint8_t *ctx, int64_t n, const uint32_t *freq_by_ctx,
                       uint32_t *state, uint16_t *words, int64_t max_words, int64_t *n_words);
int oracle_rans_decode(const uint16_t *words, int64_t n_words, uint32_t state, const uint8_t *ctx, int64_t n,
                       const uint32_t *freq_by_ctx, uint8_t *syms_out);

/* conversions from the format definitions */
uint16_t oracle_f32_to_bf16(float v);
uint16_t oracle_f32_to_f16(float v);
uint8_t oracle_f32_to_e4m3_satfinite(float v);
int8_t oracle_f32_to_int8(float v);
double oracle_bf16_to_f64(uint16_t b);

/* symbols of one quantised block (returns the escape count, fills bytes/payloads) */
int oracle_block_symbols(const int64_t a[8], int coset, uint8_t u[8], uint8_t ctx[8], int32_t payload[8]);

/* rate estimate (bits per parameter) on sampled rows at index j */
double oracle_estimate_bpp(const uint16_t *w, int64_t M, int64_t K, float sample_frac, int j);
int oracle_select_j(const uint16_t *w, int64_t M, int64_t K, float target_bpp, float sample_frac, int *j_lo_out);

/* full encoders; *blob is malloc'ed, free with oracle_free */
int oracle_encode(const uint16_t *w, int64_t M, int64_t K, float target_bpp, int container, float sample_frac,
                  uint8_t **blob, size_t *bytes);
int oracle_encode_lossless(const uint16_t *w, int64_t M, int64_t K, uint8_t **blob, size_t *bytes);
/* lossy encode at a given resolution index j (no rate search); target_bpp is
   only recorded in the header.  j below the smallest admissible index -> error */
int oracle_encode_at(const uint16_t *w, int64_t M, int64_t K, float target_bpp, int j, int container,
                     float sample_frac, uint8_t **blob, size_t *bytes);
/* smallest resolution index whose row steps keep every row's peak in range */
int oracle_smallest_valid_j(const uint16_t *w, int64_t M, int64_t K);
/* lossless tiled ANS of BF16 (0), FP16 (1), FP8 e4m3 (2) or FP32 (4) elements */
int oracle_encode_lossless_dtype(const void *w, int64_t M, int64_t K, int dtype, uint8_t **blob, size_t *bytes);
void oracle_free(void *p);

/* decode tiles [t_lo, t_hi) into out (M*K elements of the container) and,
 * for FP8/INT8, the output row scales t_r (written for all rows when t_lo == 0) */
int oracle_decode(const uint8_t *blob, size_t bytes, void *out, float *row_scale_out, int64_t t_lo, int64_t t_hi);
/* the symbol byte u coded for every coordinate (M*K bytes, matrix order) */
int oracle_decode_symbols(const uint8_t *blob, size_t bytes, uint8_t *sym_out, int64_t t_lo, int64_t t_hi);

/* the lattice point of every coordinate as k = 2q (M*K int32, matrix order; lossy blobs) */
int oracle_decode_lattice(const uint8_t *blob, size_t bytes, int32_t *k_out, int64_t t_lo, int64_t t_hi);
/* batch conversions used by the conversion pins: kind 0 bf16, 1 fp16, 2 e4m3 satfinite, 3 int8 */
void oracle_convert_f32(int kind, int64_t n, const float *in, void *out);

/* fixed-width comparators: block-absmax 4-bit codebook quantisers (NF4 and
   INT4 levels; codes, FP32 block scales and BF16 reconstructions; returns the
   bits per weight) and a per-row-scaled FP8 E4M3 round trip */
void oracle_nf4_levels(double cb[16]);
void oracle_int4_levels(double cb[16]);
double oracle_q4_roundtrip(const uint16_t *w, int64_t n, int64_t block, const double levels[16],
                           uint8_t *codes, float *scales, uint16_t *recon);
double oracle_e4m3_to_f64(uint8_t b);
double oracle_fp8_row_roundtrip(const uint16_t *w, int64_t M, int64_t K, uint16_t *recon, uint8_t *codes,
                                float *scales);

/* fp64 reference GEMM: y[t, n] = sum_k x[t, k] * w[n, k] for rows t of x */
void oracle_gemm_f64(const double *x, const double *w, double *y, int64_t T, int64_t N, int64_t K);

#endif
