/*
 * qgemv.h -- C ABI of the block-quantized weight x quantized activation
 * product on GB300 (sm_103a).  Plain pointers and sizes; no C++ types.
 *
 * What is computed (the decode engine's numerics page, "ActScaling::PerBlock",
 * functions quantize_blocks / dot / exact_sum / scaled_to_f32; the block-scale
 * lane page, functions block_sums / lane):
 *   - an activation row is quantized per weight block to int8 codes under a
 *     scale m*2^e with m in 128..255 (the least such scale with
 *     127*m*2^e >= the block's largest magnitude; codes the nearest integers
 *     of x/scale, ties to even);
 *   - for every weight block of a row, the two integer sums sum(coef*a) and
 *     sum(offs*a) are formed exactly, multiplied by the block's scales and the
 *     activation scale, summed exactly in a wide integer and rounded once to
 *     f32 (to nearest even on the f32 grid, a subnormal result then flushed to
 *     a zero of its sign);
 *   - the rounded block values of a row are added in block order from +0 in
 *     f32 (round to nearest even, subnormal results flushed).
 * F16 weights (numerics page, f32_to_f16 / fdot / tree): the activation is
 * rounded to f16; element i's exact product goes to lane i mod 8 in index
 * order from +0; the 8 lanes fold as ((l0+l1)+(l2+l3))+((l4+l5)+(l6+l7)).
 *
 * Devices and threads: every call works on the device current in the calling
 * thread.  The launchers raise each kernel's dynamic shared-memory limit once
 * per (kernel, device), under a lock, and cache per-device facts (SM count,
 * the fault word's address) atomically, so one process may drive several
 * GPUs and call the library from several host threads at once.
 *
 * Memory: every data pointer is DEVICE memory owned by the caller; the
 * library allocates nothing and keeps no per-call state.  Weight pointers
 * must be 16-byte aligned.  Calls are asynchronous on `stream` (a
 * cudaStream_t passed as void*, NULL = the legacy default stream), except
 * q_check_weights, which synchronizes that stream.  Kernels are launched with
 * programmatic dependent launch: a product kernel may start streaming its
 * weights (kv_scores: its first key tiles) while the previous kernel on the
 * stream finishes, and waits for it before it reads activations or writes
 * outputs.  So weights and the key cache must be complete before that
 * previous kernel signals its dependents: true for any kernel that does not
 * trigger them early, and for kv_cache_rows, which lets its successor start
 * only when it has finished.
 *
 * Errors: 0 on success, else a negative QB_E_* code (argument checks happen
 * on the host before any launch; nothing is launched on error).
 *
 * Layouts (little endian; the pages fix the logical form of a coded row --
 * every weight is a*coef + b*offs of its segment (numerics page, structs
 * CodedRow, Segment, Scale) -- but no bytes, so these are this library's own).
 * A matrix is `rows` row records laid end to end, q_weight_bytes() in all.
 *   QB_Q8_0 (block 32):  int8 codes[K] | f16 d[K/32] | zero pad to 16 B.
 *                        weight = d*q.
 *   QB_Q4K  (block 256): K/256 blocks of 144 B:
 *                        f16 d | f16 dmin | sc: eight 6-bit fields in a 48-bit
 *                        little-endian integer (field s at bits 6s..6s+5) |
 *                        mn: the same | qs: 16 B per 32-element sub-block s,
 *                        byte j = q[32s+j] | q[32s+16+j] << 4.
 *                        weight = d*sc[s]*q - dmin*mn[s], q in 0..15.
 *   QB_Q6K  (block 256): K/256 blocks of 208 B | f16 d[K/256] | pad to 16 B.
 *                        A block: ql (128 B; per 32-element chunk c, byte j =
 *                        low nibbles of q[32c+j] | q[32c+16+j] << 4) |
 *                        qh (64 B; per chunk c, bytes 0..3: byte b holds the
 *                        top 2 bits of q[32c+4k+b] at bits 2k..2k+1, k=0..3;
 *                        bytes 4..7 the same for q[32c+16+4k+b]) |
 *                        sc (16 x int8, one per 16-element unit).
 *                        weight = d*sc[u]*(q-32), q in 0..63.
 *   QB_F16:              f16 W[rows][K], K % 8 == 0.
 * Activations (ncols columns): codes int8 [ncols][K]; scales qb_scale
 * [ncols][K/block]; sums16 int16 [ncols][K/16] (the sum of each 16-element
 * unit's codes -- the activation side's unit sums of the lane page).
 * Outputs f32 out[c*rows + r].
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QB_API __attribute__((visibility("default")))
#else
#define QB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { QB_F16 = 1, QB_Q8_0 = 8, QB_Q4K = 12, QB_Q6K = 14 } qb_fmt;

enum {
    QB_OK = 0,
    QB_E_ARG = -1,        /* null pointer, misaligned weights, K or rows out of range, ncols not in 1..16 */
    QB_E_FORMAT = -2,     /* a format this library does not read (numerics page, reads) */
    QB_E_BLOCK = -3,      /* act->block differs from the format's block */
    QB_E_CUDA = -4,       /* a CUDA call or launch failed */
    QB_E_UNREADABLE = -5, /* q_check_weights found an inf/NaN block scale (numerics page, Unreadable) */
    QB_E_DEVICE = -6,     /* a kernel gave up a bounded wait (q_device_status) */
    QB_E_SCRATCH = -7     /* q_matvec_static: the request needs more than the library's static scratch */
};

/* Size of the library's static scratch array used by q_matvec_static. */
#define QB_STATIC_SCRATCH_BYTES (1 << 20)

/* An activation block's scale m*2^e, m in 128..255 (numerics page, ActScale
 * under PerBlock).  m == 0 marks a block holding an infinity: it has no scale,
 * and every row's dot with it is the engine's NaN 0x7FC00000. */
typedef struct {
    uint8_t m;
    uint8_t _pad;
    int16_t e;
} qb_scale;

/* A quantized activation (numerics page, struct ActRow): `block` elements
 * share one scale; all pointers device memory, laid out as above. */
typedef struct {
    int block;
    const int8_t *codes;
    const qb_scale *scales;
    const int16_t *sums16;
} qb_act;

/* quantize_blocks (numerics page): x f32 [ncols][K] quantized per block of
 * `block` (32 or 256) elements.  absmax reads a denormal as zero and passes
 * NaN over; a denormal or NaN element gets code 0; an all-zero block gets
 * m=128, e=0; a block with an infinity gets m=0.  K % block == 0, K <= 2^24,
 * ncols in 1..16.  Writes codes, scales and sums16. */
QB_API int quantize_act(int block, const float *x, int64_t K, int ncols, int8_t *codes, qb_scale *scales,
                 int16_t *sums16, void *stream);

/* dot under PerBlock (numerics page) for every row of W and every column of
 * act: out[c*rows + r].  fmt in {QB_Q8_0, QB_Q4K, QB_Q6K}; act->block must be
 * the format's block (32, 256, 256); K % block == 0; ncols in 1..16.  A row
 * with an inf/NaN block scale (numerics page, Unreadable) is written as the
 * engine's NaN 0x7FC00000; use q_check_weights to refuse such matrices up
 * front. */
QB_API int q_gemv(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act *act, int ncols, float *out,
           void *stream);

/* An activation whose codes cross the array in two words (lane page, opening
 * description and WordSums; numerics page, Words): each code a 16-bit integer
 * a = 256*hi + lo, hi its signed high byte and lo its unsigned low byte, with
 * one scale m*2^e per `block` elements (m in 1..255; m == 0: no scale).
 * codes int16 [ncols][K] (16-byte aligned), scales as qb_act's. */
typedef struct {
    int block;
    const int16_t *codes;
    const qb_scale *scales;
} qb_act16;

/* dot under PerBlock (numerics page) with two-word activation codes: for
 * every row of W and column of act, each block's sums sum(coef*a) and
 * sum(offs*a) formed exactly over the 16-bit codes (the lane page's per-word
 * sums joined as 256*high + low), times the block's scales and m*2^e, summed
 * exactly, rounded once, the rounded values added in block order from +0;
 * out[c*rows + r].  fmt in {QB_Q8_0, QB_Q4K, QB_Q6K}; act->block the format's
 * block; K % block == 0 and K small enough that a row's block values fit
 * shared memory (K <= 2^18 for Q4K/Q6K, <= 2^15 for Q8_0, else QB_E_ARG);
 * ncols in 1..16.  Unreadable weight scales and activation blocks without a
 * scale give the engine's NaN rows, as in q_gemv.  Asynchronous on stream. */
QB_API int q_gemv_w2(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act16 *act, int ncols,
                     float *out, void *stream);

/* Bytes of the workspace q_matvec needs for a K x ncols activation: its
 * quantized form (codes, scales, unit sums; or the f16 rounding for QB_F16),
 * each part 16-byte aligned.  Negative QB_E_* for bad arguments. */
QB_API int64_t q_matvec_workspace_bytes(qb_fmt fmt, int64_t K, int ncols);

/* The whole product from an f32 activation: quantize_act (or
 * quantize_act_f16) then q_gemv (or q_gemv_f16), out[c*rows + r], bit for bit
 * the same results.  For one column of a Q8_0/Q4_K/Q6_K matrix with
 * K % 256 == 0, for 2..4 columns of a Q4_K/Q6_K matrix at K = 4096 that the
 * multi-column kernels take (Q4_K: every row count at 3..4 columns, and at
 * 2 columns up to 40 or past 64 rows per SM; Q6_K: up to about 22..28 rows
 * per SM, and 33..57 at 3..4 columns), and for F16 with
 * ncols * K * 4 <= 227 KB (rows short enough
 * for the F16 kernel's rings), it is a single launch that quantizes (or
 * rounds) the activation inside the product kernel and needs no workspace
 * (`workspace` may be NULL; a Q4_K matrix with K >= 12288 given a workspace
 * takes the two launches, measured faster there); otherwise
 * `workspace` must be device memory of at least q_matvec_workspace_bytes()
 * bytes, 16-byte aligned, owned by the caller and not used by another call
 * while this one runs.  x must be 16-byte aligned. */
QB_API int q_matvec(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const float *x, int ncols, float *out,
                    void *workspace, size_t workspace_bytes, void *stream);

/* q_matvec for callers that cannot allocate device memory -- for example a
 * serving process whose device memory all belongs to its own pool after
 * start-up, or a latency-critical loop that must not call cudaMalloc (it can
 * synchronize the device).  (The pages have no counterpart: this is a usage
 * variant, not part of the method.)  Same arguments and results as q_matvec
 * without the workspace: the quantized activation always goes through a
 * QB_STATIC_SCRATCH_BYTES (1 MiB) array inside the library, in two launches
 * (quantize, then multiply).  A request whose q_matvec_workspace_bytes()
 * exceeds that returns QB_E_SCRATCH and launches nothing.  Nothing is
 * allocated, by the library or by any routine it calls.
 * - Set-up: the first call on a device (with that device current) looks up
 *   the array's device address (cudaGetSymbolAddress) and caches it; make
 *   that first call before any stream capture.  The cached address belongs
 *   to the device's context as it was then: after cudaDeviceReset (or any
 *   other end of that primary context) the library must not be called again
 *   in the process on that device.
 * - rows == 0 launches nothing; K == 0 writes +0 to every output (as
 *   q_matvec) without touching the array.
 * - Sharing: every call on a device uses the same array.  Its contents are
 *   whatever the last call left; nothing in it needs to start at zero, since
 *   each call writes all of the quantized activation it then reads.  Calls
 *   whose launches may overlap on the GPU (different streams, or different
 *   host threads, without ordering between them) race on the array; order them
 *   on one stream or with events.
 * - The array lives on every GPU that loads the library until the process
 *   exits. */
QB_API int q_matvec_static(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const float *x, int ncols,
                           float *out, void *stream);

/* f32_to_f16 (numerics page) over x f32 [ncols][K]: round to nearest even,
 * subnormals kept, past the top infinite; NaN becomes 0x7E00. */
QB_API int quantize_act_f16(const float *x, int64_t K, int ncols, uint16_t *x16, void *stream);

/* fdot with LANES = 8 and the pairwise tree (numerics page) for F16 weights
 * W [rows][K] against x16 [ncols][K]: out[c*rows + r].  K % 8 == 0; ncols in
 * 1..16; a NaN result is written as 0x7FC00000. */
QB_API int q_gemv_f16(const uint16_t *W, int64_t rows, int64_t K, const uint16_t *x16, int ncols, float *out,
               void *stream);

/* reads (numerics page) / Unreadable: scans every block scale of W for inf or
 * NaN.  Synchronizes `stream`.  Returns QB_OK, QB_E_UNREADABLE, or an error. */
QB_API int q_check_weights(qb_fmt fmt, const void *W, int64_t rows, int64_t K, void *stream);

/* Bytes of a rows x K matrix in `fmt` (row records included), or a negative
 * QB_E_* code for an unread format or a K the format cannot hold. */
QB_API int64_t q_weight_bytes(qb_fmt fmt, int64_t rows, int64_t K);

/* Per-block results for testing the lane (lane page, block_sums / lane): for
 * every column c, row r and weight block b, the block's exact sums C and O
 * (int32, [ncols][rows][K/block]; O is 0 for formats without offsets) and its
 * value rounded once (f32, same layout).  Same kernels' arithmetic as q_gemv,
 * without the row fold.  Any of C, O, v may be NULL. */
QB_API int q_block_values(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act *act, int ncols,
                   int32_t *C, int32_t *O, float *v, void *stream);

/* Reads and clears the library's device fault word (set when a kernel gives
 * up a bounded wait on its own copies).  Synchronizes `stream`.  Returns
 * QB_OK or QB_E_DEVICE. */
QB_API int q_device_status(void *stream);

/* Most matrices one grouped call (q_gemv_many, q_gemv_f16_many,
 * q_matvec_many) takes. */
#define QB_MAX_MATS 4

/* Several matrices that share one activation, in one pass where the shape
 * allows (bankML forward page: mv_many, qkv -- one quantized activation feeds
 * Q, K and V, another gate and up; bankML f16 page: mat_vec_multi_par --
 * several matrices by one column in one pass).  W[i] is a rows[i] x K matrix
 * in `fmt` (all the same format and K), and out[i][c*rows[i] + r] receives
 * exactly what q_gemv(fmt, W[i], rows[i], K, act, ncols, out[i], stream)
 * would write.  W, rows and out are HOST arrays of nmat (1..QB_MAX_MATS)
 * entries, read during the call; the pointers in them follow q_gemv's rules.
 * One launch where the streaming kernels take the shape (K % 256 == 0; the
 * rows of all matrices form one range), else one launch per matrix. */
QB_API int q_gemv_many(qb_fmt fmt, int nmat, const void *const *W, const int64_t *rows, int64_t K,
                       const qb_act *act, int ncols, float *const *out, void *stream);

/* q_gemv_f16 for several F16 matrices sharing x16 (same host-array
 * conventions as q_gemv_many): one launch where the streaming F16 kernel
 * takes the shape, else one per matrix. */
QB_API int q_gemv_f16_many(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t K,
                           const uint16_t *x16, int ncols, float *const *out, void *stream);

/* q_matvec for several matrices sharing the f32 activation x (host arrays as
 * in q_gemv_many): the activation is quantized once; for one column of a
 * Q8_0/Q4_K/Q6_K format with K % 256 == 0 the whole call is one launch (no
 * workspace needed), otherwise quantize_act (or quantize_act_f16) into
 * `workspace` (q_matvec_workspace_bytes(fmt, K, ncols) bytes) and then the
 * grouped product.  Results are those of q_matvec for each matrix. */
QB_API int q_matvec_many(qb_fmt fmt, int nmat, const void *const *W, const int64_t *rows, int64_t K,
                         const float *x, int ncols, float *const *out, void *workspace, size_t workspace_bytes,
                         void *stream);

/* ---- ActScaling::Sub32 (numerics page: block_scale, quantize, ACT_BLOCK,
 * GROUP, exact_sum, dot; block-scale lane page: group).
 *
 * The activation is quantized per 32 elements with a 4-bit scale
 * significand; a row's dot is made of groups of 256 elements, each group's
 * terms (every 32-element sub-block's integer sums times its weight scales
 * and its own activation scale) summed exactly and rounded once to f32 (the
 * same rounding as above), the group values then added in group order from +0
 * (f32, round to nearest even, subnormal results flushed). */

/* quantize (numerics page, ActScaling::Sub32): x f32 [ncols][K] per 32
 * elements under block_scale -- the least m*2^e, m in 8..15, with
 * 127*m*2^e >= the block's largest magnitude (a denormal read as zero, NaN
 * passed over) -- and codes the nearest integers of x/(m*2^e), ties to even
 * (a denormal or NaN element: 0).  An all-zero block gets m=8, e=0; a block
 * with an infinity m=0 (no scale).  Writes codes int8 [ncols][K], scales
 * [ncols][K/32] and sums16 [ncols][K/16] (device memory, caller-owned).
 * K % 256 == 0 (whole groups), K <= 2^24, ncols in 1..16; x and codes 16-byte
 * aligned. */
QB_API int quantize_act_sub32(const float *x, int64_t K, int ncols, int8_t *codes, qb_scale *scales,
                              int16_t *sums16, void *stream);

/* dot under Sub32 for every row of W (fmt QB_Q8_0, QB_Q4K or QB_Q6K, the
 * layouts above) and every column of act: out[c*rows + r].  act->block must
 * be 32 (scales per 32 elements, as quantize_act_sub32 writes them; any m in
 * 1..255 and e give the exact result, m = 0 gives NaN).  K % 256 == 0,
 * K <= 2^18, ncols in 1..16; sums16 needed for Q4K and Q6K; weights, codes,
 * scales and sums16 16-byte aligned.  A group holding an activation block
 * without a scale or an unreadable weight scale makes the row the engine's
 * NaN 0x7FC00000, as does (never for block_scale scales with f16 weight
 * scales) a group whose terms' exponents lie 318 or more places apart. */
QB_API int q_gemv_sub32(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act *act, int ncols,
                        float *out, void *stream);

/* Workspace bytes q_matvec_sub32 needs (codes, scales and unit sums of the
 * quantized activation), or a negative QB_E_* code. */
QB_API int64_t q_matvec_sub32_workspace_bytes(int64_t K, int ncols);

/* quantize_act_sub32 into `workspace` (16-byte aligned, at least
 * q_matvec_sub32_workspace_bytes(K, ncols) bytes), then q_gemv_sub32: two
 * launches on `stream`, bit for bit the same results.  For one column of a
 * matrix whose rows the streaming kernel takes (K % 256 == 0 and K/128
 * threads a row team) it is a single launch that quantizes x inside the
 * product kernel and needs no workspace (`workspace` may be NULL). */
QB_API int q_matvec_sub32(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const float *x, int ncols,
                          float *out, void *workspace, size_t workspace_bytes, void *stream);

/* ---- FP8 E4M3 weights with 128x128 block scales (colizig OPS page, FP8:
 * e4m3ToF32, dequantRow, matmulFp8).
 *
 * W: rows x K bytes, row-major, each an OCP E4M3 number ([s:1][e:4][m:3],
 * bias 7, subnormals m*2^-9, S.1111.111 NaN, no infinity); scales: f32
 * [ceil(rows/128)][ceil(K/128)], one per 128x128 block; a weight is its
 * decoded byte times its block's scale.  x: f32 [ncols][K]; out[c*rows + r]
 * = the row's dot with column c in f32 arithmetic (a float path, as on the
 * page: the order of the additions is this library's, and the result lies
 * within (K + 4) * 2^-24 * sum |x_i * w_i| of the exact dot of the weights
 * dequantized to f32).  A NaN result is written as 0x7FC00000.
 * K % 16 == 0, 16 <= K <= 32768, ncols in 1..16; W and x 16-byte aligned. */
QB_API int q_gemv_fp8(const uint8_t *W, const float *scales, int64_t rows, int64_t K, const float *x, int ncols,
                      float *out, void *stream);

/* ---- The int8 cache's score path (numerics page: cache_row, int8_codes,
 * INV_127, quantize_head, int8_score). */

/* How a query head is scaled (numerics page, ActScaling): per block of 32
 * with a 4-bit significand, or the whole head one block with an 8-bit one. */
#define QB_PERBLOCK 0
#define QB_SUB32 1

/* Codes a quantized query head holds: d rounded up to a whole number of
 * 256-element groups under QB_SUB32, d under QB_PERBLOCK (scales: dp/32 a
 * head, or one); QB_E_ARG unless d % 16 == 0 and 16 <= d <= 1024. */
QB_API int kv_head_codes(int scaling, int d);

/* cache_row (numerics page) for n rows of d f32 elements x [n][d]: each row's
 * f16 scale f32_to_f16(amax * INV_127) (amax = absmax, INV_127 = 1/127
 * rounded to f32, the product an f32 multiply with subnormals flushed),
 * written as binary16 bits to scales[n], and its codes int8_codes under the
 * reciprocal of that scale (the correctly rounded f32 1/s): x*inv to the
 * nearest integer, ties to even, within +-127, NaN products 0, every code 0
 * when the scale rounded to zero.  codes int8 [n][d].  d % 16 == 0,
 * 16 <= d <= 1024; x and codes 16-byte aligned. */
QB_API int kv_cache_rows(const float *x, int64_t n, int d, int8_t *codes, uint16_t *scales, void *stream);

/* quantize_head (numerics page) for nh query heads q f32 [nh][d]:
 * QB_SUB32 -- each head padded with zeros to dp = kv_head_codes(QB_SUB32, d)
 * elements and quantized per 32 as quantize_act_sub32 does (codes [nh][dp],
 * scales [nh][dp/32]); QB_PERBLOCK -- the whole head one block under
 * wide_scale as quantize_act does (codes [nh][d], scales [nh][1]). */
QB_API int kv_quantize_heads(int scaling, const float *q, int nh, int d, int8_t *codes, qb_scale *scales,
                             void *stream);

/* int8_score (numerics page) of nh quantized query heads (as
 * kv_quantize_heads writes them) against L cached key rows of nkv key heads:
 * query head h reads key head h / (nh / nkv); key codes int8 [nkv][lcap][d]
 * and key scales (binary16 bits) [nkv][lcap] as kv_cache_rows writes them,
 * positions 0..L-1 used.  Per query block b, D_b = sum of q_i*k_i; the terms
 * sig(ks)*m_b*D_b at exponent exp(ks)+e_b are summed exactly and rounded once
 * to f32 (as the products above); the score is then multiplied by `scale`
 * (f32, subnormal results flushed).  out f32 [nh][L].  A key row whose scale
 * is infinite or NaN, or a query block without a scale, gives the engine's
 * NaN.  nh % nkv == 0, lcap >= L; codes 16-byte aligned. */
QB_API int kv_scores(int scaling, const int8_t *qcodes, const qb_scale *qscales, int nh, int d,
                     const int8_t *kcodes, const uint16_t *kscales, int64_t L, int64_t lcap, int nkv, float scale,
                     float *out, void *stream);

/* ---- One call from host memory to host memory. */

/* Device workspace q_matvec_host needs: the activation and the outputs on the
 * device plus q_matvec's (QB_PERBLOCK) or q_matvec_sub32's (QB_SUB32) own
 * workspace; a negative QB_E_* code for a bad request. */
QB_API int64_t q_matvec_host_workspace_bytes(int scaling, qb_fmt fmt, int64_t rows, int64_t K, int ncols);

/* q_matvec (scaling QB_PERBLOCK; every format) or q_matvec_sub32 (QB_SUB32)
 * with the activation x_host f32 [ncols][K] and the result out_host f32
 * [ncols][rows] in HOST memory: one call enqueues on `stream` the copy of x
 * to the device workspace, the product and the copy of the result back
 * (cudaMemcpyAsync each way; asynchronous when the host buffers are pinned,
 * so synchronize the stream before reading out_host).  W is device memory as
 * for q_matvec; workspace is device memory of at least
 * q_matvec_host_workspace_bytes(...) bytes, 16-byte aligned.  Results and
 * errors are those of q_matvec / q_matvec_sub32. */
QB_API int q_matvec_host(int scaling, qb_fmt fmt, const void *W, int64_t rows, int64_t K, const float *x_host,
                         int ncols, float *out_host, void *workspace, size_t workspace_bytes, void *stream);

/* A static string for a status code. */
QB_API const char *q_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
