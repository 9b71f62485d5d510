/*
 * nvfp4rac.h -- C ABI of the GB300 (sm_103a) library for the rollout-side NVFP4 W4A4 linear
 * layer with Residual Activation Compensation (RAC).
 *
 * The method is that of "QUADS: Stabilizing NVFP4 Reinforcement Learning for MoE via
 * QUantization-error Alignment across Dual Sides" (arXiv 2607.15810), cited below as QUADS:
 *   - online activation quantization to NVFP4 (§2.2 "FP4", §3.1 Eq. (9));
 *   - residual R = X - DQ(Q(X)), channel score and top-k selection, second-pass quantization
 *     of the residual on the selected channels (§3.3 Eq. (20)-(24));
 *   - the native block-scaled W4A4 GEMM that carries the correction as extra K-columns
 *     (§3.3 "Targeted residual compensation"), grouped over routed MoE experts;
 *   - the trainer-side weight QDQ whose codes and scales equal the rollout quantizer's
 *     (§3.2 Eq. (12), (15)-(16)).
 *
 * Conventions shared by every call
 *   Memory     All pointers are caller-owned DEVICE memory unless a parameter says otherwise.
 *              The library never allocates device memory and keeps no pointer after a call.
 *   Streams    Every call is asynchronous on the given cudaStream_t (passed as void*; NULL is
 *              the legacy default stream).  Scalars stay on the device.
 *   Errors     Every call returns an nvq_status.  Argument and shape checks run on the host
 *              before anything is launched; on failure nothing is launched and
 *              nvq_last_error() (thread-local) describes the problem.  Device-side waits are
 *              bounded: a wait that runs out records NVQ_ERR_TIMEOUT in a device status word
 *              that nvq_device_status() reads (the kernel then returns without hanging).
 *   Inputs     bf16 inputs must be finite; non-finite inputs give unspecified codes.
 *
 * Data formats
 *   Codes      NVFP4 (E2M1) codes, two per byte, element 2i in the LOW nibble; row-major with a
 *              leading dimension in bytes (multiple of 16).  Code = sign<<3 | magnitude index
 *              into {0, 0.5, 1, 1.5, 2, 3, 4, 6}; a negative value that rounds to 0 keeps its
 *              sign (0x8).
 *   Scales     One UE4M3 byte per 16 consecutive elements of a row, stored in the MMA-ready
 *              blocked layout: with sf_cols scale columns (a multiple of 4) and rows padded
 *              to a multiple of 128, the byte of (row r, scale column c) is at
 *                ((r / 128) * (sf_cols / 4) + c / 4) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4
 *              (nvq_sf_offset).  A buffer for R rows holds nvq_sf_bytes(R, sf_cols) bytes.
 *   RAC tail   The k compensation columns of an operand live in columns [K, K + k) of the same
 *              code and scale buffers, so a GEMM sees K_tot = K + k columns.  Scale columns from
 *              (K + k) / 16 up to sf_cols are written as zero by rac_select_quantize (and by
 *              nvfp4_quantize when k is 0), so sf_cols = nvq_sf_cols(K + k).
 *   Tensor scale  nvq_tensor_scale per tensor (or per row group): amax, S_enc = 2688 / amax,
 *              S_dec = 1 / S_enc (both fp32; amax 0 gives 1 and 1) and the score exponent
 *              E = ilogb(amax) + 2.
 *   Row groups Grouped calls take grp_off (int64 [G + 1]) and grp_rows (int64 [G]) in device
 *              memory: group g owns rows [grp_off[g], grp_off[g] + grp_rows[g]) and
 *              grp_rows[g] <= grp_off[g + 1] - grp_off[g].  grp_rows NULL means
 *              grp_rows[g] = grp_off[g + 1] - grp_off[g].  grp_off NULL with G > 1 means
 *              G equal groups of rows / G rows; G = 1 with grp_off NULL is one dense tensor.
 *              For the GEMM every grp_off[g] must be a multiple of 128 (moe_dispatch writes
 *              such offsets).
 */
#ifndef NVFP4RAC_H
#define NVFP4RAC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvq_status {
    NVQ_OK = 0,
    NVQ_ERR_ARG = 1,     /* null pointer or invalid enumerator */
    NVQ_ERR_SHAPE = 2,   /* unsupported or inconsistent sizes */
    NVQ_ERR_ALIGN = 3,   /* pointer or leading dimension not aligned as required */
    NVQ_ERR_CUDA = 4,    /* a CUDA runtime or driver call failed */
    NVQ_ERR_TIMEOUT = 5  /* a bounded device-side wait ran out (reported by nvq_device_status) */
} nvq_status;

typedef struct nvq_tensor_scale {
    float amax;      /* max |x| over the tensor or group */
    float s_enc;     /* fl(2688 / amax), 1 when amax is 0 */
    float s_dec;     /* fl(1 / s_enc) */
    int32_t shift_e; /* ilogb(amax) + 2, 0 when amax is 0 */
} nvq_tensor_scale;

enum nvq_epilogue {
    NVQ_EPI_STORE = 0,      /* out[r, n] = bf16(alpha_g * acc[r, n]),                 out is [rows][N]   */
    NVQ_EPI_SWIGLU = 1,     /* out[r, j] = bf16(silu(g) * u), g = alpha*acc[r, j],
                               u = alpha*acc[r, N/2 + j], silu(g) = g / (1 + exp(-g)), out is [rows][N/2] */
    NVQ_EPI_ROW_SCALE = 2,  /* out[r, n] = bf16(alpha_g * acc[r, n] * row_w[r]),      out is [rows][N]   */
    NVQ_EPI_STORE_F32 = 3   /* out[r, n] = fl(alpha_g * acc[r, n]) as fp32,            out is [rows][N]   */
};

enum nvq_dtype { NVQ_BF16 = 0, NVQ_F32 = 1 };

/* Message describing the last failure on the calling thread ("" after a success). */
const char* nvq_last_error(void);

/* Reads and clears the device status word of the current device (synchronises the stream).
 * *status receives the first error a kernel recorded since the last read: NVQ_OK, or
 * NVQ_ERR_TIMEOUT (a bounded wait ran out), or NVQ_ERR_ARG (a caller-supplied index outside its
 * range); *where identifies the wait or check.  The index checks, made before any access
 * through the index:
 *   41  moe_dispatch: an expert id outside [0, groups) (the pair is left out of the routing);
 *   42  activation tails (rac_select_quantize, rac_residual_tail): a channel of idx outside
 *       [0, K) (channel 0 is read instead);
 *   43  weight tails (rac_weight_tail, w4a4_rac_grouped_gemm with idx): the same;
 *   44  rac_reconstruct: the same (the tail value is added to column 0 instead);
 *   45  nvfp4_gather_rows / fp8_gather_rows: row_src[i] / topk >= src_rows (row i is written as
 *       a padding row).
 * The output of a call that recorded NVQ_ERR_ARG is meaningless; no access leaves its operands. */
nvq_status nvq_device_status(void* stream, int32_t* status, int32_t* where);

/* Sets the bound of every device-side wait, in GPU clock cycles (default 2^32, about 2 s; any
 * value >= 1).  Applies to launches made after the call.  A wait that runs out records
 * NVQ_ERR_TIMEOUT and its CTA unwinds: before it exits, the CTA waits for the asynchronous copies
 * it already issued, with a bound of its own of at least 2^26 cycles, so a very small limit (as
 * tests use to exercise the timeout path) gives errors, never a copy into a finished CTA. */
nvq_status nvq_set_wait_limit(uint64_t cycles);

/* How rac_select_quantize, rac_residual_tail and rac_weight_tail build the tail columns; every
 * path writes the same bytes.  NVQ_TAIL_GATHER loads the selected channels one by one (the
 * least traffic when k is a small share of K); NVQ_TAIL_ROWS reads whole rows with 16-byte
 * loads, expands them in shared memory and gathers from there (fewer instructions per tail
 * element when k is a large share); NVQ_TAIL_AUTO (the default) takes the row path when
 * k >= K / 4, except for a weight tail given the channel-major copy, which always gathers.
 * A process-wide setting for launches made after the call; NVQ_ERR_ARG for an
 * unknown value.  Not part of the paper's method: a choice between two schedules of Eq. (21). */
enum nvq_tail_path { NVQ_TAIL_AUTO = 0, NVQ_TAIL_GATHER = 1, NVQ_TAIL_ROWS = 2 };
nvq_status nvq_set_tail_path(int32_t path);

/* Measured NVFP4 tensor-core rate of the current GPU (a roofline reference; not part of the
 * paper's method): back-to-back tcgen05 M128 N256 K64 mxf4nvf4 MMAs with FP32 accumulation in
 * TMEM on every SM, no memory traffic, mmas_per_sm per SM (16 .. 2^20).  with_cp != 0 adds the
 * three scale-factor copies into TMEM that the GEMM issues per MMA.  Synchronous on `stream`;
 * *tflops receives the achieved TFLOP/s. */
nvq_status nvq_fp4_mma_rate(int32_t mmas_per_sm, int32_t with_cp, float* tflops, void* stream);

/* Self-check of the quantizer's division of a block amax by 6 (not part of the paper's method:
 * the kernels form fl(amax_b / 6) with a multiply and an FMA correction instead of a division).
 * Runs every finite non-negative bf16 value through both that form and the IEEE division
 * __fdiv_rn on the GPU.  result: device uint32 [2] out; result[0] = number of values whose
 * results differ (0 expected), result[1] = the lowest such bf16 bit pattern (0xffffffff if
 * none).  Asynchronous on `stream`. */
nvq_status nvq_check_block_scale_division(uint32_t* result, void* stream);

/* Scale-layout helpers (host functions, no device access). */
int64_t nvq_sf_cols(int64_t ktot);                      /* roundup(ktot / 16, 4) */
int64_t nvq_sf_bytes(int64_t rows, int64_t sf_cols);    /* roundup(rows, 128) * sf_cols */
int64_t nvq_sf_offset(int64_t row, int64_t col, int64_t sf_cols);

/*
 * nvfp4_quantize -- Q_A of QUADS Eq. (9) / Q_W of Eq. (7): NVFP4 quantization of a bf16 matrix
 * (§2.2 "FP4": E2M1 codes, one E4M3 scale per 16 elements along K, one FP32 tensor scale),
 * plus the per-channel residual scores of Eq. (23) when scores is not NULL.
 *
 *   x         bf16 [rows][ldx], ldx >= K, ldx % 8 == 0, x 16-byte aligned.
 *   rows, K   1 <= rows <= 2^24 (at most 2^19 rows per group when scores is not NULL),
 *             16 <= K <= 8192, K % 16 == 0.
 *   grp_off, grp_rows, groups   row groups (see header); each group gets its own tensor scale
 *             and its own scores; rows outside every group are not read or written.
 *   codes     [rows][ld_codes] bytes, columns [0, K) written; ld_codes % 16 == 0, >= K / 2.
 *   sf        blocked scales with sf_cols columns (sf_cols % 4 == 0, >= K / 16); columns
 *             [0, K / 16) written; if zero_pad is non-zero, columns [K / 16, sf_cols) are
 *             zeroed as well (use it when no RAC tail follows).
 *   tscale    [groups] out.  With amax_given non-zero, tscale[g].amax must already hold the
 *             group's max |x| (as w4a4_rac_grouped_gemm's out_tscale leaves it for the tensor
 *             it writes) and the pass that measures it is skipped; the other fields are
 *             written from it.
 *   scores    NULL, or uint64 [groups][K] out: score_j = sum over the group's rows of
 *             rint(|r_j| * 2^(20 - E))^2, r = x - DQ(Q(x)) in fp32 (exact, order independent).
 * Ownership: all buffers caller-owned; nothing retained.  Errors: NVQ_ERR_ARG / SHAPE / ALIGN
 * before launch, NVQ_ERR_CUDA if a launch fails.
 */
nvq_status nvfp4_quantize(const void* x, int64_t rows, int64_t K, int64_t ldx,
                          const int64_t* grp_off, const int64_t* grp_rows, int32_t groups,
                          uint8_t* codes, int64_t ld_codes, uint8_t* sf, int64_t sf_cols,
                          int32_t zero_pad, nvq_tensor_scale* tscale, uint64_t* scores,
                          int32_t amax_given, void* stream);

/*
 * nvfp4_amax -- the statistic of the FP32 tensor scale (QUADS §2.2 "FP4", second scaling
 * level) alone: tscale[g] is zeroed, then tscale[g].amax = max |x| over group g's rows (exact).
 * The other fields stay 0; nvfp4_quantize(..., amax_given = 1) fills them from amax.  With rows
 * of one batch split over processes, each one's amax, combined by a maximum across processes,
 * is the amax of the whole batch, so the quantization is that of the unsplit batch (the
 * token-sharded path).  Arguments as for nvfp4_quantize.
 */
nvq_status nvfp4_amax(const void* x, int64_t rows, int64_t K, int64_t ldx, const int64_t* grp_off,
                      const int64_t* grp_rows, int32_t groups, nvq_tensor_scale* tscale, void* stream);

/*
 * rac_select_quantize -- channel selection of QUADS Eq. (24) and the second-pass quantization
 * of Eq. (21): per group, S = the k channels with the largest score (ties to the lower channel
 * index), written ascending to idx; then the residual R[:, S] = X[:, S] - DQ(Q(X))[:, S], with
 * blocks of 16 consecutive selected channels and the group's own S_enc, is quantized into
 * columns [K, K + k) of codes and scale columns [K / 16, (K + k) / 16) of sf; scale columns
 * [(K + k) / 16, sf_cols) are zeroed.
 *
 *   x, rows, K, ldx, grp_*, groups   as for nvfp4_quantize (the same call's inputs).
 *   tscale    [groups] from nvfp4_quantize.   scores  uint64 [groups][K] from nvfp4_quantize.
 *   k         0 <= k <= K, k % 16 == 0.  k = 0 only zeroes the scale padding.
 *   codes, sf the buffers nvfp4_quantize wrote; ld_codes >= (K + k) / 2; sf_cols >= (K + k) / 16.
 *   idx       int32 [groups][k] out (may be NULL when k == 0).
 */
nvq_status rac_select_quantize(const void* x, int64_t rows, int64_t K, int64_t ldx,
                               const int64_t* grp_off, const int64_t* grp_rows, int32_t groups,
                               const nvq_tensor_scale* tscale, const uint64_t* scores, int32_t k,
                               uint8_t* codes, int64_t ld_codes, uint8_t* sf, int64_t sf_cols,
                               int32_t* idx, void* stream);

/*
 * rac_select -- the selection half of rac_select_quantize (QUADS Eq. (24)): per group, the k
 * channels with the largest score, ties to the lower channel index, ascending in idx.
 *   scores    uint64 [groups][K] from nvfp4_quantize.   idx  int32 [groups][k] out.
 *   16 <= k <= K, k % 16 == 0.
 */
nvq_status rac_select(const uint64_t* scores, int64_t K, int32_t groups, int32_t k, int32_t* idx,
                      void* stream);

/*
 * rac_residual_tail -- the second-pass half of rac_select_quantize (QUADS Eq. (21)): the
 * residual on the channels in idx (from rac_select, or any ascending set per group) quantized
 * into columns [K, K + k) of codes and scale columns [K / 16, (K + k) / 16) of sf, the scale
 * padding beyond zeroed.  Arguments as for rac_select_quantize; idx may be NULL when k == 0.
 * Split from the selection so that work needing only idx (the weight tail) can run beside it.
 */
nvq_status rac_residual_tail(const void* x, int64_t rows, int64_t K, int64_t ldx,
                             const int64_t* grp_off, const int64_t* grp_rows, int32_t groups,
                             const nvq_tensor_scale* tscale, const int32_t* idx, int32_t k,
                             uint8_t* codes, int64_t ld_codes, uint8_t* sf, int64_t sf_cols,
                             void* stream);

/*
 * rac_reconstruct -- the compensated activation X~ of QUADS Eq. (21) read back from an activation
 * operand (codes, sf and tscale as written by nvfp4_quantize + rac_select_quantize): for row r of
 * group g, out[r][j] = fl(DQ_main[r][j] + DQ_tail[r][p]) where j = idx[g * k + p], and
 * out[r][j] = DQ_main[r][j] for channels outside the group's set; DQ(code) = fl(V * fl(sb *
 * S_dec_g)).  An evaluation entry (the activation error ||X~ - X|| of a k), not a step of the
 * layer: two kernel launches on `stream`.
 *   codes     [rows][ld_codes] with the main columns [0, K) and the tail [K, K + k);
 *             8-byte aligned rows.   sf: blocked scales, sf_cols >= (K + k) / 16.
 *   tscale    [groups] (device).   idx: int32 [groups][k], distinct channels per group (NULL when
 *             k == 0).   grp_off / grp_rows: as for rac_select_quantize (NULL: equal groups).
 *   out       fp32 [rows][ldo], ldo >= K, 16-byte aligned rows; rows outside every group's
 *             range are not written.
 *   Errors: NVQ_ERR_ARG (null pointer), NVQ_ERR_SHAPE (K or k not multiples of 16, k > K, short
 *   leading dimensions), NVQ_ERR_ALIGN, NVQ_ERR_CUDA.
 */
nvq_status rac_reconstruct(const uint8_t* codes, int64_t ld_codes, const uint8_t* sf, int64_t sf_cols,
                           const nvq_tensor_scale* tscale, int64_t rows, int64_t K, int32_t k,
                           const int32_t* idx, const int64_t* grp_off, const int64_t* grp_rows,
                           int32_t groups, float* out, int64_t ldo, void* stream);

/*
 * weight_qdq -- the trainer-side QDQ_W of QUADS Eq. (12): for each of G weight tensors
 * W_g = w[g] ([N][K] bf16, tensor g at w + g * N * ldw elements) the same quantizer as
 * nvfp4_quantize with one tensor scale per tensor, so that its codes and scales are the
 * rollout weight codes bit for bit (Eq. (15)-(16)).  Optionally writes W-hat = DQ(Q(W)).
 *
 *   codes     [G * N][ld_codes], sf blocked scales of G * N rows with sf_cols columns
 *             (rows of tensor g start at row g * N; N % 128 == 0).
 *   tscale    [G] out.
 *   w_hat     NULL, or [G * N][K] of w_hat_dtype (NVQ_BF16: nearest-even bf16 of the fp32
 *             dequantized value; NVQ_F32: the fp32 value fl(V * fl(sb * S_dec))).
 */
nvq_status weight_qdq(const void* w, int32_t groups, int64_t N, int64_t K, int64_t ldw,
                      uint8_t* codes, int64_t ld_codes, uint8_t* sf, int64_t sf_cols,
                      nvq_tensor_scale* tscale, void* w_hat, int32_t w_hat_dtype, void* stream);

/*
 * w4a4_rac_grouped_gemm -- the native block-scaled W4A4 GEMM of QUADS §3.3 with the RAC
 * correction as K-columns [K, K + k), over row groups (routed MoE experts) that each have
 * their own weight matrix:  Y_g = alpha_g * [A_g | R_g] [W_g | W'_g]^T,
 * alpha_g = S_dec(A_g) * S_dec(W_g), FP32 accumulation on tcgen05 tensor cores.
 *
 * When idx is not NULL the call first builds each group's weight tail W'_g into columns
 * [K, K + k) of b_codes / b_sf (as rac_weight_tail does); with idx NULL and k > 0 the tail
 * columns are used as they are (built earlier by rac_weight_tail).
 *
 *   groups, grp_off, grp_rows   A row groups (grp_off[g] % 128 == 0); groups = 1 with
 *             grp_off NULL is a dense GEMM over all `rows`.
 *   rows      number of rows of A and out (buffer extent); rows <= 2^24.
 *   a_codes, lda, a_sf, a_sf_cols    A = quantized activations + RAC tail (nvfp4_quantize +
 *             rac_select_quantize; for routed MoE rows, nvfp4_gather_rows output), [rows] rows.
 *             a_tscale  [groups] if a_scale_per_group else [1].
 *   b_codes, ldb, b_sf, b_sf_cols    W_g = rows [g * N, (g + 1) * N) (weight_qdq output);
 *             tail columns rewritten by this call.  b_tscale  [groups].
 *   N, K, k   N % 256 == 0 (NVQ_EPI_SWIGLU: N / 2 % 128 == 0); K % 64 == 0; k as above.
 *   idx       NULL, or int32 [groups][k] if idx_per_group else [k] (rac_select_quantize output).
 *   epilogue  enum nvq_epilogue.   row_w  fp32 [rows] for NVQ_EPI_ROW_SCALE, else NULL.
 *   out, ldo  bf16 (fp32 for NVQ_EPI_STORE_F32) [rows][ldo], ldo in elements, ldo % 8 == 0;
 *             rows outside every group are not written.
 *   out_tscale  NULL, or nvq_tensor_scale [groups] out (bf16 epilogues): zeroed, then
 *             out_tscale[g].amax = max |out| over group g's rows as stored (bf16, exact), the
 *             statistic nvfp4_quantize(..., amax_given = 1) needs to quantize `out` next
 *             without another pass over it.
 */
nvq_status w4a4_rac_grouped_gemm(int32_t groups, const int64_t* grp_off, const int64_t* grp_rows,
                                 int64_t rows, const uint8_t* a_codes, int64_t lda,
                                 const uint8_t* a_sf, int64_t a_sf_cols,
                                 const nvq_tensor_scale* a_tscale, int32_t a_scale_per_group,
                                 uint8_t* b_codes, int64_t ldb, uint8_t* b_sf, int64_t b_sf_cols,
                                 const nvq_tensor_scale* b_tscale, int64_t N, int64_t K, int32_t k,
                                 const int32_t* idx, int32_t idx_per_group, int32_t epilogue,
                                 const float* row_w, void* out, int64_t ldo,
                                 nvq_tensor_scale* out_tscale, void* stream);

/*
 * rac_weight_tail -- the weight columns that multiply the RAC correction (QUADS §3.3, Eq. (21):
 * the correction term is a product with the same layer's weights on the selected channels).
 * Reading of the paper: W'_g = Q(DQ(W_g)[:, S_g]), i.e. the dequantized stored NVFP4 weights on
 * the selected channels, gathered in ascending channel order and re-quantized (blocks of 16
 * gathered channels) with the weight tensor's own S_enc, written into columns [K, K + k) of
 * b_codes and scale columns [K / 16, (K + k) / 16) of b_sf; scale columns beyond are zeroed.
 *   b_codes, ldb, b_sf, b_sf_cols, b_tscale   weight_qdq output for groups x N rows.
 *   idx       int32 [groups][k] if idx_per_group else [k].  16 <= k <= K, k % 16 == 0.
 *   cm_codes, cm_sf   NULL, or the nvfp4_channel_major copy of the same weights (both or
 *             neither; N % 64 == 0).  With the copy the selected channels are read in
 *             coalesced runs (about 1.5 N bytes per selected channel instead of scattered
 *             bytes of every row); the result is identical.
 */
nvq_status rac_weight_tail(int32_t groups, int64_t N, int64_t K, int32_t k, const int32_t* idx,
                           int32_t idx_per_group, uint8_t* b_codes, int64_t ldb, uint8_t* b_sf,
                           int64_t b_sf_cols, const nvq_tensor_scale* b_tscale,
                           const uint8_t* cm_codes, const uint8_t* cm_sf, void* stream);

/*
 * nvfp4_channel_major -- a channel-major copy of quantized weights (layout only; the paper's
 * weights are static at rollout, so the copy is made once per weight update next to
 * weight_qdq).  It serves rac_weight_tail, which gathers whole channels of W.
 *   b_codes, ldb, b_sf, b_sf_cols   groups x N rows of K codes / K/16 blocked scales.
 *   cm_codes  uint8 [groups][K][N / 2] out: byte (g, j, m) = code of row 2m of channel j
 *             (low nibble) | code of row 2m + 1 (high nibble).  16-byte aligned.
 *   cm_sf     uint8 [groups][K / 16][N] out: scale byte of (row n, block c) at (g, c, n).
 *   N % 64 == 0, groups * N <= 2^24, K % 16 == 0, K <= 8192.
 */
nvq_status nvfp4_channel_major(int32_t groups, int64_t N, int64_t K, const uint8_t* b_codes,
                               int64_t ldb, const uint8_t* b_sf, int64_t b_sf_cols,
                               uint8_t* cm_codes, uint8_t* cm_sf, void* stream);

/*
 * moe_dispatch -- routing plumbing of the MoE expert layer (not described by the paper):
 * a stable counting sort of the tokens * topk (token, slot) pairs by expert.
 *
 *   topk_ids  int32 [tokens][topk] expert ids in [0, groups).   topk_w  fp32 [tokens][topk] or NULL.
 *             An id outside [0, groups) is not written out of bounds: its pair is left out of
 *             the routing (row_of = -1, which moe_combine skips) and the device status word
 *             records NVQ_ERR_ARG (nvq_device_status).
 *   grp_off   int64 [groups + 1] out: group g starts at row grp_off[g] (multiple of 128);
 *             grp_rows int64 [groups] out: number of routed rows of group g.
 *   row_src   int32 [capacity] out: routed row -> token * topk + slot (-1 on padding rows);
 *             inside a group rows are in ascending (token, slot) order.
 *   row_of    int64 [tokens * topk] out: routed row of each (token, slot) (-1: left out).
 *   row_w     fp32 [capacity] out (NULL allowed): topk_w of the routed row, 0 on padding.
 *   capacity  >= moe_capacity(tokens, topk, groups).
 *   workspace device bytes >= moe_dispatch_workspace_size(tokens, topk, groups).
 */
int64_t moe_capacity(int64_t tokens, int32_t topk, int32_t groups);
size_t moe_dispatch_workspace_size(int64_t tokens, int32_t topk, int32_t groups);
nvq_status moe_dispatch(const int32_t* topk_ids, const float* topk_w, int64_t tokens, int32_t topk,
                        int32_t groups, int64_t* grp_off, int64_t* grp_rows, int32_t* row_src,
                        int64_t* row_of, float* row_w, int64_t capacity, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * moe_dispatch_static_scratch -- moe_dispatch that allocates nothing.  The paper has no
 * counterpart: this is a library convenience.  Arguments and outputs are those of moe_dispatch,
 * minus the workspace.  The histogram moe_dispatch keeps in its workspace lives here in one
 * file-scope device array of NVQ_DISPATCH_STATIC_SCRATCH_BYTES (1 MiB).
 *
 * Who needs it: callers that cannot allocate device memory, or thread a workspace, at the
 * point of the call.  Examples are a serving engine that hands its whole HBM budget to a
 * KV cache up front, and a fixed-signature plugin or custom-op interface with no workspace
 * argument.  Another is code that must not pay for cudaMalloc/cudaFree, which can synchronize
 * the device.  The call makes no cudaMalloc, cudaFree or other allocating call.
 *
 * Limit: moe_dispatch_workspace_size(tokens, topk, groups) must be <= 1 MiB; otherwise the call
 * returns NVQ_ERR_SHAPE, launches nothing, and nvq_last_error() names the sizes.  At 128
 * experts the limit is 2048 units of 256 (token, slot) pairs: 65536 tokens at top-8.  groups
 * must be in [1, 1024], as for moe_dispatch.
 *
 * First call: on each device, the first call looks up the array's device address with
 * cudaGetSymbolAddress, with that device current, and caches it.  Make that first call before
 * any stream capture.  A failed lookup returns NVQ_ERR_CUDA.  The cached address belongs to the
 * device's primary context at that time: after cudaDeviceReset on a device, this entry must not
 * be called again on that device in the same process.
 *
 * Sharing: all calls on one device share the array.  Nothing in it needs to start at zero,
 * because each call writes every word it later reads.  Calls that may overlap on the device
 * race on the array and corrupt each other's output.  Examples are calls on two streams
 * without an ordering between them, or a replay that overlaps another call.  Calls
 * serialized on one stream are safe.
 */
#define NVQ_DISPATCH_STATIC_SCRATCH_BYTES (1u << 20)
nvq_status moe_dispatch_static_scratch(const int32_t* topk_ids, const float* topk_w,
                                       int64_t tokens, int32_t topk, int32_t groups,
                                       int64_t* grp_off, int64_t* grp_rows, int32_t* row_src,
                                       int64_t* row_of, float* row_w, int64_t capacity,
                                       void* stream);

/*
 * nvfp4_gather_rows -- copies quantized rows (codes of columns [col0, ktot) and the blocked
 * scale atoms covering them) into the routed layout: out row r = source row row_src[r] / topk,
 * padding rows (row_src < 0) get zero codes and zero scales.  out_sf uses the same sf_cols as
 * sf.  With out_codes NULL only the scales are copied.  col0 % 64 == 0 (a scale atom holds 64
 * columns); two calls with [0, K) and [K, K + k) copy the main columns and the RAC tail
 * separately, so the first can run before the tail exists.
 */
nvq_status nvfp4_gather_rows(const uint8_t* codes, int64_t ld_codes, const uint8_t* sf,
                             int64_t sf_cols, int64_t src_rows, const int32_t* row_src,
                             int32_t topk, int64_t capacity, int64_t ktot, int64_t col0,
                             uint8_t* out_codes, int64_t ld_out, uint8_t* out_sf, void* stream);

/*
 * moe_combine -- out[t, :] = bf16( sum over slots s = 0..topk-1, in slot order, in fp32, of
 * y[row_of[t * topk + s], :] ), slots with row_of < 0 left out.  y bf16 [capacity][ldy]; out
 * bf16 [tokens][ldo].
 */
nvq_status moe_combine(const void* y, int64_t ldy, const int64_t* row_of, int64_t tokens,
                       int32_t topk, int64_t hidden, void* out, int64_t ldo, void* stream);

/* ==========================================================================================
 * FP8 W8A8 block-scaled baseline.  The paper's throughput comparison (§4.4.2: plain W4A4 about
 * 1.3x FP8, W4A4 + RAC about 1.16x) is against FP8 W8A8 rollout with fine-grained block scaling
 * (§2.2 "FP8": E4M3 elements, maximum 448, "each tile of values carries its own alpha", as
 * DeepGEMM does).  Readings where the pages are silent: activation tiles are 1 x 128 (one row,
 * 128 consecutive channels), weight tiles 128 x 128; the tile scale is the power of two
 * alpha = 2^e with e the smallest integer such that 448 * 2^e >= amax of the tile, clamped to
 * [-127, 127] (an all-zero tile gets -127), stored as the UE8M0 byte e + 127 and applied by
 * the tensor core (kind::mxf8f6f4, one scale per 32 elements); an element is E4M3 of
 * x * 2^-e, nearest, ties to even, sign kept.
 *
 * Operand layout: codes [rows][ld] E4M3 bytes, K-major; scales in the blocked layout of
 * nvq_sf_offset with sf_cols = nvq_fp8_sf_cols(K) columns of one UE8M0 byte per 32 elements
 * (a tile's byte repeated in its 4 columns and, for weights, its 128 rows); a buffer for R rows
 * holds nvq_sf_bytes(R, sf_cols) bytes.
 * ========================================================================================== */
int64_t nvq_fp8_sf_cols(int64_t K);  /* roundup(K / 32, 4) */

/*
 * fp8_quantize -- x [rows][ldx] bf16 (16-byte aligned rows) to E4M3 codes [rows][ld_codes]
 * (ld_codes % 16 == 0, 16-byte aligned) and UE8M0 tile scales in sf.  tile_rows 1: 1 x 128
 * activation tiles; tile_rows 128: 128 x 128 weight tiles starting at row 0 (for stacked
 * per-expert weights of N rows each, N % 128 == 0 keeps every tile inside one expert).
 * K % 32 == 0, 32 <= K <= 16384.  Scale columns of a partial last tile beyond K / 32 are zeroed
 * within its 4-column word; rows beyond `rows` are not written.  Errors: NVQ_ERR_ARG,
 * NVQ_ERR_SHAPE, NVQ_ERR_ALIGN, NVQ_ERR_CUDA.
 */
nvq_status fp8_quantize(const void* x, int64_t rows, int64_t K, int64_t ldx, int32_t tile_rows, uint8_t* codes,
                        int64_t ld_codes, uint8_t* sf, int64_t sf_cols, void* stream);

/*
 * fp8_blockscaled_grouped_gemm -- Y[r, n] = sum_c V[a_rc] 2^ea(r, c/128) V[b_nc] 2^eb(n/128, c/128)
 * over row groups (routed experts), the FP8 counterpart of w4a4_rac_grouped_gemm (same tcgen05
 * kernel with E4M3 operands and UE8M0 scales; no tensor scale and no RAC columns).  Arguments as
 * for w4a4_rac_grouped_gemm: groups / grp_off / grp_rows / rows, A codes [rows][lda], B codes
 * [groups * N][ldb] (lda, ldb multiples of 16 covering K bytes, 16-byte aligned), scales with
 * sf_cols >= nvq_fp8_sf_cols(K), N % 256 == 0, epilogue NVQ_EPI_STORE / SWIGLU / ROW_SCALE /
 * STORE_F32 with row_w, out [rows][ldo].  K % 32 == 0, 32 <= K <= 16384.  Device waits are bounded
 * (nvq_device_status).  Errors as for w4a4_rac_grouped_gemm.
 */
nvq_status fp8_blockscaled_grouped_gemm(int32_t groups, const int64_t* grp_off, const int64_t* grp_rows, int64_t rows,
                                        const uint8_t* a_codes, int64_t lda, const uint8_t* a_sf, int64_t a_sf_cols,
                                        const uint8_t* b_codes, int64_t ldb, const uint8_t* b_sf, int64_t b_sf_cols,
                                        int64_t N, int64_t K, int32_t epilogue, const float* row_w, void* out,
                                        int64_t ldo, void* stream);

/*
 * fp8_gather_rows -- nvfp4_gather_rows for FP8 operands: row i of the routed layout receives
 * the K code bytes and the scales of token row_src[i] / topk (zeros where row_src[i] < 0).
 * capacity = the routed layout's rows (a multiple of 128); out_sf has capacity rows of sf_cols
 * columns.  Errors: NVQ_ERR_ARG, NVQ_ERR_SHAPE, NVQ_ERR_ALIGN, NVQ_ERR_CUDA.
 */
nvq_status fp8_gather_rows(const uint8_t* codes, int64_t ld_codes, const uint8_t* sf, int64_t sf_cols, int64_t src_rows,
                           const int32_t* row_src, int32_t topk, int64_t capacity, int64_t K, uint8_t* out_codes,
                           int64_t ld_out, uint8_t* out_sf, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4RAC_H */
