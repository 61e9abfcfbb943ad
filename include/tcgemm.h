/*
 * tcgemm.h -- C ABI of the GB300 (sm_103a) tensor-core GEMM library.
 *
 * Operation (all entry points):
 *
 *     D[i][j] = fma.rn.f32(alpha, sum_k A[i][k] * B[j][k], beta * C[i][j])
 *
 *  - A is row-major M x K and B is stored N x K, so the product is A times B
 *    transposed ("mma.sync" page, section "Operand coordinates and ownership":
 *    B's atom axes are (N, K/2) although the product uses B transposed).
 *  - A and B are both f16 or both bf16; the sum is accumulated in float32
 *    ("mma.sync" page, introduction); C is float32 (same page, operand table).
 *  - alpha and beta are applied after the product at the call site as one
 *    single-rounded fma.rn.f32 ("mma.sync" page, section "Accumulation,
 *    transpose and alpha/beta"; "fma" page, section "Operand specification":
 *    a*b+c is one fused atom, not a rounded multiply and a rounded add).
 *    With C == NULL or beta == 0, C is not read and D = alpha * sum
 *    (mul.rn.f32).  beta * C is formed with mul.rn.f32 before the fma.
 *  - The K recurrence starts from zero ("mma.sync" page, worked example: the
 *    first K issue uses scalar C = 0, later issues read D); C enters in the
 *    epilogue fma above.
 *  - D is float32, bf16 or f16.  The 16-bit outputs are the float32 result
 *    rounded to nearest even (cvt.rn).
 *
 * Layout: every matrix is row-major with an explicit leading dimension
 * (elements between the starts of consecutive rows).  Rows of A, B and the
 * gather table are K contiguous elements; rows of C and D are N contiguous
 * elements.
 *
 * Ownership: every pointer argument is caller-owned device memory (any
 * allocator; typically PyTorch).  The library never frees or retains caller
 * memory beyond the asynchronous execution of the call.  It holds, per
 * device, a small status word in its own device globals and a host-side cache
 * of TMA descriptors; per device and stream, the skinny (M <= 64) path keeps
 * a workspace for split tiles, and the FP4 path buffers for converted weights
 * or re-pitched scales, each allocated once and grown on demand (so calls on
 * different streams never share them).
 *
 * Execution: calls are asynchronous on `stream` (a cudaStream_t; NULL means
 * the legacy default stream) on the current device.  A call may launch more
 * than one kernel on that stream (a large gathered call runs whole waves of
 * clustered CTAs and, beside them, single CTAs on the SMs no cluster fits;
 * FP4 weights with M > 128 are first converted to bf16); work issued later
 * on the stream still starts only after all of them, and every form can be
 * captured into a CUDA graph.
 *
 * Per-device state (the status word's address, the workspaces, the address of
 * the allocation-free entry point's array) is set up by the first call on a
 * device and kept for the life of the process; it does not survive
 * cudaDeviceReset, after which the library must not be called again.
 *
 * Errors:
 *  - Argument, alignment, aliasing and type errors are returned synchronously
 *    before anything is launched, following the descriptor legality rule that
 *    invalid fields are rejected rather than promoted, folded or reinterpreted
 *    ("cp.async.bulk.tensor" page, section "Operands and descriptor fields").
 *  - Launch failures return GEMM_ERR_CUDA.
 *  - Errors found on the device (a pipeline wait that ran out of time, a
 *    gather index outside the table) are recorded in the device status word
 *    and returned by gemm_check_device_status().  No kernel traps.
 */
#ifndef TCGEMM_H
#define TCGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* negative size, NULL required pointer, bad leading dim, bad enum */
    GEMM_ERR_ALIGNMENT = 2,   /* pointer not 16-byte aligned or row pitch not a multiple of 16 bytes */
    GEMM_ERR_UNSUPPORTED = 3, /* a size of 2^31 or more, or a device without tcgen05 (not sm_103) */
    GEMM_ERR_ALIAS = 4,       /* D overlaps A, B, idx, or C other than exactly in place */
    GEMM_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed */
    GEMM_ERR_TIMEOUT = 6,     /* device: a pipeline wait ran out of time; the kernel returned */
    GEMM_ERR_INDEX = 7        /* device: a gather index was outside [0, table_rows) */
} gemm_status;

typedef enum {
    GEMM_OUT_F32 = 0,
    GEMM_OUT_BF16 = 1,
    GEMM_OUT_F16 = 2
} gemm_out_t;

/*
 * D = fma.rn(alpha, A * B^T, beta * C) with f16 operands.
 *
 *  M, N, K     sizes, each in [0, 2^31).  M == 0 or N == 0: nothing is done.
 *              K == 0: D = beta * C (or 0 when C is absent).
 *  A, lda      M x K f16, lda >= K, lda % 8 == 0, 16-byte aligned.
 *              May be NULL only when K == 0.
 *  B, ldb      N x K f16, ldb >= K, ldb % 8 == 0, 16-byte aligned.
 *              May be NULL only when K == 0.
 *  C, ldc      M x N float32 or NULL (absent); ldc >= N, 4-byte aligned.
 *              Not read when beta == 0.
 *  D, ldd      M x N output of type `out`; ldd >= N, aligned to its element
 *              size.  Only columns j < N of each row are written.  D may be C
 *              exactly (same pointer, ldd == ldc, out == GEMM_OUT_F32); any
 *              other overlap of D with A, B or C is GEMM_ERR_ALIAS.
 *              C and D move through TMA boxes when their base is 16-byte
 *              aligned and their row pitch a multiple of 16 bytes; otherwise
 *              (and for the 16-byte chunk that straddles column N when
 *              N * sizeof(out) is not a multiple of 16) the epilogue uses
 *              plain loads and stores, which is slower but exact.
 *  out         a gemm_out_t value.
 *  stream      cudaStream_t to run on.
 */
gemm_status gemm_f16(int64_t M, int64_t N, int64_t K,
                     const void *A, int64_t lda,
                     const void *B, int64_t ldb,
                     const float *C, int64_t ldc,
                     void *D, int64_t ldd,
                     int out, float alpha, float beta, void *stream);

/* As gemm_f16 with bf16 operands. */
gemm_status gemm_bf16(int64_t M, int64_t N, int64_t K,
                      const void *A, int64_t lda,
                      const void *B, int64_t ldb,
                      const float *C, int64_t ldc,
                      void *D, int64_t ldd,
                      int out, float alpha, float beta, void *stream);

/*
 * Row-gathered form: D[i][:] = fma.rn(alpha, table[idx[i]][:] * B^T, beta * C[i][:])
 * for i < M.  The A rows are fetched four at a time with TMA tile::gather4
 * loads ("cp.async.bulk.tensor" page, section "Gather4 and scatter4": four
 * runtime row coordinates per issue, not necessarily consecutive; choosing
 * them is the caller's logic).  Indices may repeat.
 *
 *  dtype_is_bf16  0: table and B are f16; 1: bf16.
 *  table, lda     table_rows x K, lda >= K, lda % 8 == 0, 16-byte aligned.
 *  table_rows     rows in the table, in [1, 2^31).
 *  idx            M int32 row indices in device memory, 4-byte aligned.
 *                 An index outside [0, table_rows) makes that A row zero (so
 *                 D[i][:] = beta * C[i][:]) and records GEMM_ERR_INDEX in the
 *                 device status word.
 *  Other arguments as in gemm_f16.  D must not overlap idx or the table.
 */
gemm_status gemm_gather_rows(int64_t M, int64_t N, int64_t K, int dtype_is_bf16,
                             const void *table, int64_t table_rows, int64_t lda,
                             const int32_t *idx,
                             const void *B, int64_t ldb,
                             const float *C, int64_t ldc,
                             void *D, int64_t ldd,
                             int out, float alpha, float beta, void *stream);

/*
 * Row-scattered form, the dual of the gathered one: for i < M,
 *     D[idx[i]][:] = fma.rn(alpha, A[i][:] * B^T, beta * C[idx[i]][:]).
 * Row i of the product is written to row idx[i] of D with TMA tile::scatter4
 * stores, four rows per issue ("cp.async.bulk.tensor" page, section "Gather4
 * and scatter4": the store form takes the destination first and four runtime
 * row coordinates; choosing them is the caller's logic).  C is read from the
 * same destination row (by tile::gather4), so C == D is an in-place update of
 * the rows named by idx.  Rows of D that idx does not name are not touched.
 *
 *  A, lda      M x K, lda >= K, lda % 8 == 0, 16-byte aligned (as gemm_f16).
 *  idx         M int32 destination rows in device memory, 4-byte aligned.
 *              An index outside [0, d_rows) writes nothing for that row and
 *              records GEMM_ERR_INDEX in the device status word.  Indices may
 *              repeat: every element of a row named more than once then holds
 *              the value that one of those rows computed (which one is not
 *              specified); with C == D such a row is not specified at all.
 *  d_rows      rows of D (and of C), in [1, 2^31).
 *  C, ldc      NULL or d_rows x N float32 (as gemm_f16).
 *  D, ldd      d_rows x N; stores go through TMA for float32 output with a
 *              16-byte aligned base and row pitch, otherwise (and for a last
 *              column chunk narrower than 32) through plain stores.
 *  Other arguments as in gemm_f16.  D must not overlap idx, A or B.
 */
gemm_status gemm_scatter_rows(int64_t M, int64_t N, int64_t K, int dtype_is_bf16,
                              const void *A, int64_t lda,
                              const void *B, int64_t ldb,
                              const int32_t *idx, int64_t d_rows,
                              const float *C, int64_t ldc,
                              void *D, int64_t ldd,
                              int out, float alpha, float beta, void *stream);

/*
 * FP4 weights: D = fma.rn(alpha, A * W^T, beta * C) with bf16 A (M x K) and
 *     W[n][k] = e2m1(code of element k of row n) * 2^(Bs[k / 32][n] - 127).
 * The "cp.async.bulk.tensor" page (section "Interleave and packed FP4") gives
 * float4_e2m1fn as an operand format; the code values and the block scaling
 * are those of the OCP Microscaling definition that name refers to (E2M1: sign,
 * 2 exponent bits with bias 1, 1 mantissa bit, codes 0..7 = 0, 0.5, 1, 1.5, 2,
 * 3, 4, 6; UE8M0 scale s = 2^(s - 127), 255 = NaN; 32 elements per scale).
 * M <= 64 streams the codes and scales with TMA and converts them to bf16 in
 * tensor memory, where the tensor-core MMA reads them (a quarter of the bytes
 * of a bf16 B); 64 < M <= 128 runs that path twice (rows 0-63, then the
 * rest); larger M converts W to bf16 once (a per-stream buffer the library
 * allocates) and runs the bf16 GEMM.  W's values are exact in bf16 for scales
 * up to 252; 253-254 can overflow to infinity.
 *
 *  A, lda      M x K bf16, as in gemm_bf16.
 *  Bq, ldbq    N rows of K/2 bytes, ldbq bytes apart: element k of a row is
 *              the low nibble of byte k/2 when k is even, the high nibble when
 *              odd.  16-byte aligned, ldbq >= K/2 and a multiple of 16.
 *  Bs, ldbs    K/32 rows of N scale bytes, ldbs bytes apart (row b holds the
 *              scales of elements 32b .. 32b+31 of every row of W), ldbs >= N.
 *              With a 16-byte aligned base and a pitch that is a multiple of
 *              16 the kernel reads them in place; otherwise (M <= 128) the
 *              library first copies them to a padded buffer of its own.
 *  K           a multiple of 32 (GEMM_ERR_UNSUPPORTED otherwise).
 *  Other arguments as in gemm_bf16.  D must not overlap A, Bq or Bs.
 */
gemm_status gemm_bf16_e2m1(int64_t M, int64_t N, int64_t K,
                           const void *A, int64_t lda,
                           const uint8_t *Bq, int64_t ldbq,
                           const uint8_t *Bs, int64_t ldbs,
                           const float *C, int64_t ldc,
                           void *D, int64_t ldd,
                           int out, float alpha, float beta, void *stream);

/*
 * Both operands FP4: D = fma.rn(alpha, A * B^T, beta * C) with
 *     A[i][k] = e2m1(code of element k of row i of Aq) * 2^(As[k / 32][i] - 127),
 *     B[j][k] = e2m1(code of element k of row j of Bq) * 2^(Bs[k / 32][j] - 127),
 * computed by the tensor cores' block-scaled MMAs (fp32 accumulation).  The
 * "cp.async.bulk.tensor" page (section "Interleave and packed FP4") gives
 * float4_e2m1fn as an operand format and its 16U4_ALIGN16B load image; code
 * values and scales are those of the OCP Microscaling definition that name
 * refers to (E2M1 codes 0..7 = 0, 0.5, 1, 1.5, 2, 3, 4, 6, bit 3 the sign;
 * UE8M0 scale s = 2^(s - 127), 255 = NaN; one scale per 32 elements along K).
 *
 *  Aq, ldaq    M rows of K/2 bytes, ldaq bytes apart: element k of a row is
 *              the low nibble of byte k/2 when k is even, the high nibble when
 *              odd.  ldaq >= K/2.
 *  As, ldas    K/32 rows of M scale bytes, ldas bytes apart (row b holds the
 *              scales of elements 32b .. 32b+31 of every row of A), ldas >= M.
 *  Bq, ldbq    N rows of K/2 bytes (as Aq), ldbq >= K/2.
 *  Bs, ldbs    K/32 rows of N scale bytes (as As), ldbs >= N.
 *              Scales with a 16-byte aligned base and a pitch that is a
 *              multiple of 16 are read in place; otherwise the library first
 *              copies them to a padded buffer of its own (per device and stream,
 *              allocated once and grown on demand).
 *  K           a multiple of 32 (GEMM_ERR_UNSUPPORTED otherwise).
 *  image       how the codes reach the tensor cores:
 *              GEMM_FP4_PACKED (0): as stored, two per byte (MMA kind::mxf4);
 *                Aq, Bq 16-byte aligned, ldaq, ldbq multiples of 16.
 *              GEMM_FP4_ALIGN16B (1): through the 16U4_ALIGN16B load image,
 *                sixteen codes in the low 8 bytes of each 16-byte shared block
 *                (MMA kind::mxf8f6f4, half the rate of the packed form); the
 *                page's rules apply: K a multiple of 128 (GEMM_ERR_UNSUPPORTED
 *                otherwise), Aq, Bq 32-byte aligned and ldaq, ldbq multiples of
 *                32 (GEMM_ERR_ALIGNMENT otherwise).
 *              The two forms take the same products; they may add them in a
 *              different order (bit-identical wherever every partial sum is
 *              exact in float32).
 *  Kernels: M <= 64 with packed codes runs on the skinny swap-AB kernel (128
 *  rows of B per tile on the MMA's M side, A's rows padded to 16 / 32 / 64 on
 *  its N side, the K blocks of all tiles shared out over the SMs, a tile's
 *  parts added in a fixed order by the last CTA to finish); otherwise the tile
 *  kernel (gemm_query_plan forms 6 / 7).
 *  C, D, out, alpha, beta, stream as in gemm_f16.  D must not overlap Aq, As,
 *  Bq or Bs.  K == 0: D = beta * C.
 */
enum { GEMM_FP4_PACKED = 0, GEMM_FP4_ALIGN16B = 1 };
gemm_status gemm_e2m1(int64_t M, int64_t N, int64_t K,
                      const uint8_t *Aq, int64_t ldaq,
                      const uint8_t *As, int64_t ldas,
                      const uint8_t *Bq, int64_t ldbq,
                      const uint8_t *Bs, int64_t ldbs,
                      const float *C, int64_t ldc,
                      void *D, int64_t ldd,
                      int out, float alpha, float beta, int image, void *stream);

/*
 * Seeded form, the pages' recurrence taken literally: D = C + A * B^T where C
 * is the accumulator's starting value.  The first K issue reads C and every
 * later one reads the running fp32 sum ("mma.sync" page, section
 * "Accumulation, transpose and alpha/beta": only the first K issue reads the
 * start value, later ones read D).  C (M x N float32, required) is written
 * into the tensor-memory accumulator (tcgen05.st) before the first MMA of
 * each tile, and the result is converted to `out` without a further
 * operation (alpha = beta = 1).  The sum is therefore rounded to fp32 after
 * every K step of 16 with C already in it: for |C| much larger than the
 * products the result can differ from gemm_f16/gemm_bf16's
 * fma.rn(1, acc, C) (where C is added once, at the end) by up to one fp32
 * ulp of the running sum per K step.
 *
 *  Arguments as gemm_f16 without alpha and beta; C must not be NULL (when
 *  M, N > 0).  C == D (float32 out, ldc == ldd) is an in-place update.  M <= 64
 *  runs on the tile kernel (or on the warp-level kernel for tiny problems),
 *  not the skinny one.
 */
gemm_status gemm_seeded(int64_t M, int64_t N, int64_t K, int dtype_is_bf16,
                        const void *A, int64_t lda,
                        const void *B, int64_t ldb,
                        const float *C, int64_t ldc,
                        void *D, int64_t ldd,
                        int out, void *stream);

/*
 * Accumulating form: D[i][j] += alpha * sum_k A[i][k] * B[j][k] for float32 D.
 * The result is added into D by TMA reduce-add stores ("cp.async.bulk.tensor"
 * page, section "Stores, reductions, and completion": the reduction form adds
 * the shared image into the global box, whose contents are the starting
 * value, so the caller initialises D).  Rounding: each element receives
 * D + mul.rn(alpha, acc) with one float32 add per part of the K sum; the
 * tile kernel makes one part, so the result is deterministic; where the
 * skinny kernel runs the call (M <= 64, see gemm_query_plan) the K sum of a
 * tile may be split over several CTAs, each adding its part (in an order
 * that is not specified, so the last bits may differ from call to call
 * unless every partial sum is exact).  Unlike fma.rn(alpha, acc, beta * C)
 * this is two roundings (the product, then the add).
 *
 *  A, lda, B, ldb  as in gemm_f16; dtype_is_bf16 as in gemm_gather_rows.
 *  D, ldd          M x N float32, 4-byte aligned; added into through TMA when
 *                  16-byte aligned with a pitch that is a multiple of 16 bytes,
 *                  otherwise (and for the last column chunk when N * 4 is not
 *                  a multiple of 16) with float32 atomic adds.
 *  K == 0          adds nothing (GEMM_OK, no launch).
 *  Errors as gemm_f16; D must not overlap A or B.
 */
gemm_status gemm_accumulate(int64_t M, int64_t N, int64_t K, int dtype_is_bf16,
                            const void *A, int64_t lda,
                            const void *B, int64_t ldb,
                            float *D, int64_t ldd,
                            float alpha, void *stream);

/*
 * Allocation-free variant of the skinny (M <= 64) path.  The source pages have
 * no counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc where they run the GEMM: code whose device memory is owned by
 * another allocator (a framework's caching allocator, or a serving engine that
 * reserves the whole GPU up front) and latency-critical sections where the
 * implicit synchronisation of cudaMalloc/cudaFree is not allowed.
 *
 * It computes what gemm_f16 / gemm_bf16 compute for M <= 64, always with the
 * skinny kernel (those calls take it only for some shapes, the tile kernel
 * for the rest: the two round alike, element by element, but may add the K
 * sum in another order), and its scratch (partial tiles and arrival counters)
 * lives in one fixed device array inside the library: 16 MiB of partials plus 16384
 * counters (16.06 MiB in all), held by every GPU that loads the library until
 * the process exits.  The call itself allocates no device memory; the caller
 * still owns A, B, C and D.
 *
 *  dtype_is_bf16  0: A and B are f16; 1: bf16.  Other arguments as gemm_f16.
 *
 * Returns GEMM_ERR_UNSUPPORTED when M > 64 or K == 0 (other kernels, which this
 * entry point does not run) or when the problem needs more scratch than the
 * array holds (more than 16384 tiles of 128 columns of N, or more than 16 MiB
 * of partial tiles).  All other errors as gemm_f16.
 *
 * The first call on a device looks up the array's device address (and sets up
 * the library's per-device state); make that first call before any stream
 * capture.  Every call on a device shares the one array, which keeps what the
 * last call left there: a call whose tiles are split over several CTAs (the
 * K sum of a 128-column tile of N shared out) first clears, on `stream`, the
 * arrival counters it uses; a call without split tiles uses no scratch and
 * clears nothing.  gemm_check_device_status also clears them after a
 * device-side error.  Calls whose executions overlap on the GPU (different
 * streams, no ordering between them) race on the array and give wrong results.
 */
gemm_status gemm_skinny_noalloc(int64_t M, int64_t N, int64_t K, int dtype_is_bf16,
                                const void *A, int64_t lda,
                                const void *B, int64_t ldb,
                                const float *C, int64_t ldc,
                                void *D, int64_t ldd,
                                int out, float alpha, float beta, void *stream);

/*
 * Synchronises `stream`, then returns and clears the first error the device
 * recorded since the last call on the current device (GEMM_OK if none).
 * Returns GEMM_ERR_CUDA if the synchronisation itself failed.  After a
 * device-side error it also resets the library's scratch state on this
 * device, so later calls start clean.
 */
gemm_status gemm_check_device_status(void *stream);

/* Static, NUL-terminated name of a status code ("GEMM_OK", ...). */
const char *gemm_status_string(int status);

/*
 * The kernel choice the library makes for a problem, without launching
 * anything and without touching the GPU (for diagnostics and tests; a form
 * forced with gemm_debug_force_tile is applied as a call would apply it).
 * form: 0 = plain, 1 = row-gathered (gemm_gather_rows), 2 = row-scattered
 * (gemm_scatter_rows), 3 = seeded (gemm_seeded), 4 = FP4 weights
 * (gemm_bf16_e2m1), 5 = gemm_skinny_noalloc (kernel 0 where it returns
 * GEMM_ERR_UNSUPPORTED for the shape), 6 / 7 = gemm_e2m1 with packed codes /
 * the 16U4_ALIGN16B image; any other value is GEMM_ERR_INVALID_ARG.
 * has_c: C is given and beta != 0.
 *
 * With M <= 64 rows (bf16 / f16 B; not gathered, not seeded) the skinny
 * kernel runs where it measured faster than the tile kernel: M <= 16 with
 * N * K > 2^21; 16 < M <= 64 with K >= 2 N, or with K >= N and
 * N * K > 2^21.  FP4 weights with M <= 128
 * always take it.
 *
 *  kernel   0 = none (empty problem), 1 = tile kernel (128-row tiles, one
 *           CTA each), 2 = skinny swap-AB kernel (M <= 64), 3 = tile kernel
 *           on CTA pairs (256 x 256 tiles, tcgen05 cta_group::2), 4 = tile
 *           kernel on CTA pairs with 256 x 512 tiles (two MMA halves, one
 *           accumulator), 5 = tile kernel on single CTAs (128 x bn tiles) in
 *           clusters of 4 along N that share each A box by TMA multicast,
 *           6 = the same in clusters of 8, 7 = two CTA pairs (a cluster of
 *           4) with 256 x 512 tiles side by side along N, each CTA loading
 *           half of its A rows and multicasting them to the CTA in the same
 *           place of the other pair, 8 = the same with 256 x 256 tiles,
 *           9 = four CTA pairs (a cluster of 8) with 256 x 512 tiles, each
 *           CTA loading a quarter of its A rows for the four, 10 = the
 *           warp-level kernel (mma.sync.m16n8k16, one 16 x 8 block of D per
 *           warp; problems of at most 2^20 multiply-adds), 11 / 12 = the tile
 *           kernel on FP4 operands with block scales (single CTAs, 128 x bn
 *           tiles, bn 128 or 256; MMA kind::mxf4 on packed codes / kind::mxf8f6f4
 *           on the 16U4_ALIGN16B image), 13 / 14 = the same on CTA pairs
 *           with 256 x 256 tiles, 15 = the skinny kernel on packed FP4
 *           operands (M <= 64, K > 0; block-scaled MMA kind::mxf4)
 *  bm, bn   output tile; for the skinny kernel bm is the padded M and bn 128
 *  stages   shared-memory ring depth
 *  tiles    output tiles; splits = K slices per tile (skinny kernel)
 *  grid     CTAs launched for `sm_count` SMs (pairs: at most sm_count / 2
 *           pairs; on a device, at most the pairs that can be resident)
 */
typedef struct {
    int32_t kernel;
    int32_t bm;
    int32_t bn;
    int32_t stages;
    int64_t tiles;
    int32_t splits;
    int32_t grid;
} gemm_plan;

gemm_status gemm_query_plan(int64_t M, int64_t N, int64_t K, int form, int has_c,
                            int sm_count, gemm_plan *plan);

/*
 * Time limit, in nanoseconds, of every bounded pipeline wait in the kernels
 * (default 2e9).  A wait that runs out records GEMM_ERR_TIMEOUT, the kernel
 * stops its pipeline, releases its tensor memory and returns.  ns == 0
 * restores the default.  Applies to launches made after the call.
 */
gemm_status gemm_set_wait_timeout(uint64_t ns);

/*
 * Test hook.  mode 1: the next launches add 16 bytes to the transaction
 * count the first shared-memory stage expects, so that stage never completes
 * and its bounded wait runs out (all copies still land; nothing faults).
 * mode 0 turns it off.
 */
gemm_status gemm_debug_inject(int mode);

/*
 * Test hook.  Force the form of the tile kernel for later calls: kernel 1 =
 * single CTAs with tile width bn in {64, 128, 256}, kernel 3 = CTA pairs with
 * bn = 256, kernel 4 = CTA pairs with bn = 512, kernel 5 = clusters of 4
 * single CTAs sharing A with bn in {64, 256}, kernel 6 = clusters of 8
 * with bn = 256, kernel 7 = two CTA pairs sharing A with bn = 512,
 * kernel 8 = two CTA pairs sharing A with bn = 256, kernel 9 = four CTA pairs
 * sharing A with bn = 512, kernel 10 = the warp-level kernel with bn = 8 (it
 * then runs every problem), kernels 11 / 12 = the FP4 tile width bn in {128,
 * 256} for gemm_e2m1 (only), kernels 13 / 14 = FP4 CTA pairs with bn = 256
 * (gemm_e2m1 only), kernel 15 = the FP4 skinny kernel with bn = 128 (gemm_e2m1
 * with packed codes, M <= 64, K > 0; other calls keep the automatic choice;
 * forcing 11 - 14 keeps gemm_e2m1 on the tile kernel at M <= 64), kernel 2 = the skinny kernel with bn = 0 or 128
 * (problems it can run: M <= 64, K > 0, not gathered or seeded), kernel 0 =
 * automatic choice (the default).  Tile forms apply to every problem the tile
 * kernel runs, M <= 64 ones included; FP4 weights keep their own paths, and
 * problems the forced form cannot run (K == 0 for clusters and pairs) keep
 * the automatic choice.  Returns GEMM_ERR_INVALID_ARG for other values.
 */
gemm_status gemm_debug_force_tile(int kernel, int bn);

#ifdef __cplusplus
}
#endif

#endif /* TCGEMM_H */
