/*
 * lk.h -- C ABI of the GB300 (sm_103a) Q8_0 decode-projection library.
 *
 * The operations are the ones of the lane kernel library "kernels.rs"
 * (logicaffeine_compile codegen_cuda lane), the QWEN38_EXTRA_KERNELS constant
 * and model-as-a-kernel "megakernel.cu"; each entry point below names the
 * passage that defines it.
 *
 * Conventions shared by every call:
 *   - Every pointer argument is a DEVICE pointer owned by the caller (for
 *     example a torch tensor's data_ptr()), except where a parameter says
 *     "host".  The library never allocates, frees or retains device memory; it
 *     keeps only a small per-device cache of device attributes.
 *   - Every call is asynchronous on the given stream (0 = the legacy default
 *     stream) and never synchronizes, except lk_device_error.
 *   - Every call that launches a configurable kernel takes its launch
 *     settings as `const lk_launch_cfg* cfg`, just before the stream (NULL:
 *     the defaults).  Kernel choice and launch form depend only on the
 *     call's arguments and cfg: the library keeps no setting between calls
 *     apart from the two diagnostic options of lk_set_option, which change
 *     neither.
 *   - Arguments are validated before anything is launched; a failed check
 *     returns a negative status and launches nothing.  A launch failure
 *     reported by the CUDA runtime returns LK_ERR_CUDA.
 *   - Layouts are row-major and dense:
 *       wq  int8   [N][K]       weight levels of a Q8_0 matrix
 *       ws  uint16 [N][K/32]    f16 bit patterns, one scale per 32 weights
 *       x   f32    [M][K]       activation rows (M <= LK_MAX_BATCH; per call
 *                               below: most kernels take M <= LK_MAX_M)
 *       xq  int8   [M][K]       high words of the quantized activation
 *       xl  int8   [M][K]       low words (TwoPassInt8 only)
 *       xs  f32    [M][K/32]    one activation scale per 32 values
 *       y   f32    [M][N]       y[t*N + o] = row o dotted with activation t
 *   - K must be a multiple of 32.  wq, x, xq, xl must be 16-byte aligned;
 *     ws 2-byte, xs and y 4-byte, 64-bit buffers 8-byte aligned.
 *   - M == 0 or N == 0 is an empty problem: nothing is launched, LK_OK.
 */
#ifndef LK_H
#define LK_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Numerics modes ("kernels.rs" module doc, Q8MatKind -> mode()):
 *   LK_DEQUANT  f32 activations, the dot summed in f64;
 *   LK_INT8ACT  activations quantized to int8 per 32-group (one word);
 *   LK_TWOPASS  a high and a low int8 word per activation value. */
typedef enum { LK_DEQUANT = 0, LK_INT8ACT = 1, LK_TWOPASS = 2 } lk_mode;

typedef int lk_status;
#define LK_OK                   0
#define LK_ERR_ARG             -1  /* null pointer, unknown mode or option   */
#define LK_ERR_ALIGN           -2  /* pointer misaligned for its element/vec */
#define LK_ERR_SHAPE           -3  /* K % 32 != 0, M or S out of range, ...  */
#define LK_ERR_WORKSPACE       -4  /* caller's workspace too small           */
#define LK_ERR_CUDA            -5  /* the CUDA runtime reported an error     */
#define LK_ERR_DEVICE_TIMEOUT  -6  /* a device-side bounded wait gave up     */

#define LK_MAX_M      8   /* activation rows that share one weight read (every kernel) */
#define LK_MAX_BATCH  64  /* activation rows of the tensor-core GEMV path and of the
                             norm / quantize / SwiGLU / argmax calls */
#define LK_MAX_SPLITK 64  /* split-K chunks */
#define LK_MAX_GROUP  4   /* matrices of one lk_gemv_q8_group call */
#define LK_TRACE_REC  8   /* entries of one launch record of option "trace" 3 */

/*
 * Per-call launch settings (the library's own design, with no counterpart on
 * the pages).  Zero in every field is the default; NULL means all defaults.
 *   pdl        0: an ordinary launch; 1: a programmatic dependent launch of
 *              the kernel before it on the stream (it starts while that kernel
 *              finishes; GEMVs stream weights meanwhile; every kernel reads
 *              its inputs and writes its outputs only after that kernel)
 *   prefill    warps (four-warp groups in the tensor-core kernel's four-warp
 *              layout) of a GEMV block that issue their first weight stages
 *              before the dependency wait (0: half of them)
 *   path       GEMV kernel: 0 the library's choice, 1 the direct-load kernel,
 *              2 the bulk-copy ring kernel, 3 the tensor-core kernel (2 to
 *              LK_MAX_BATCH rows); a forced kernel that does not take the
 *              shape gives LK_ERR_SHAPE
 *   grid_ctas  blocks of a ring or tensor-core launch along the rows
 *              (0: one per SM; a launch that writes argmax keys takes at most
 *              lk_argmax_parts_max(N), else LK_ERR_ARG)
 *   ring_tk    ring kernel: bytes of K per stage for rows longer than that, a
 *              multiple of 1024 up to 8192 (0: whole rows up to 8192, two
 *              equal slices up to 16384 where a half is a multiple of 1024,
 *              else 4096)
 *   mma_min_m  fewest activation rows that take the tensor-core kernel under
 *              path 0 (0: 2; LK_MAX_BATCH + 1: never)
 *   mma_tk     tensor-core kernel: bytes of K per ring stage (0 auto, else a
 *              multiple of 256 up to 8192)
 *   mma_warps  its warps per block (0 auto, else 1..16)
 *   mma_depth  its ring stages per warp (0: 1, else 1..8)
 *   mma_i8     its dots on the int8 tensor path (mma m16n8k32 s8 on the
 *              levels as they are) or the f16 path (f16 MMAs on converted
 *              levels): 0 auto (int8 for Int8Act with 8+ tiles of 16 rows per
 *              SM), 1 int8, 2 f16
 *   mma_group  its warps per 16-row tile: 0 auto, 1 one warp per tile, 4 four
 *              warps per tile (each one partial b mod 4; for launches with few
 *              tiles per SM)
 *   mma_act16  its activation rows held in shared memory as f16 (0 auto:
 *              where that leaves room for 8 warps; 1 whenever they fit; 2
 *              never: int8, converted per use)
 * Errors: LK_ERR_ARG for a field outside its range.  Every setting gives the
 * same bits: only speed depends on them.
 */
typedef struct {
  int pdl;
  int prefill;
  int path;
  int grid_ctas;
  int ring_tk;
  int mma_min_m;
  int mma_tk;
  int mma_warps;
  int mma_depth;
  int mma_i8;
  int mma_group;
  int mma_act16;
} lk_launch_cfg;

/* A static, human-readable name of a status. */
const char* lk_status_string(lk_status s);

/* Library ABI version (major*100 + minor). */
int lk_version(void);

/*
 * RMSNorm of M rows, then the activation quantizer of `mode`.
 * ("kernels.rs" RMSNORM lk_rmsnorm / lk_rmsnorm_row with lk_quant_lane;
 *  its module doc: each value over the root of the mean square plus eps,
 *  times the gain.)
 *   y[t][i] = x[t][i] / sqrt(sum_k x[t][k]^2 / K + eps) * gain[i]
 * The sum of squares is accumulated in f64 under LK_DEQUANT and in f32
 * otherwise, in the fixed order of a block of min(roundup32(K), 1024)
 * threads (strided per-thread fused multiply-adds, then a shuffle-down tree
 * per warp and over the warps), so results are bit-reproducible.
 *   x     f32 [M][K]   input rows           gain f32 [K]
 *   xn    f32 [M][K]   normed rows; required under LK_DEQUANT (the GEMV's
 *                      activation), optional (may be NULL) otherwise
 *   xq,xs              quantized output (LK_INT8ACT, LK_TWOPASS); ignored
 *                      under LK_DEQUANT
 *   xl                 low words, LK_TWOPASS only
 */
lk_status lk_rmsnorm_quant(const float* x, const float* gain, int M, int K, float eps,
                           lk_mode mode, float* xn, int8_t* xq, int8_t* xl, float* xs,
                           const lk_launch_cfg* cfg, cudaStream_t stream);

/*
 * Residual add, then lk_rmsnorm_quant of the sum: the step between a
 * decoder's projection and the next norm ("kernels.rs" RMSNORM lk_rmsnorm_row
 * with ADD and SUM; QWEN38_EXTRA_KERNELS gk_add_rmsnorm_q8_hl).
 *   v[t][i] = x[t][i] + r[t][i]   (one f32 addition)
 *   s = v (optional), then the RMSNorm of v and the quantizer of `mode`,
 *   bit for bit lk_rmsnorm_quant(v, gain, ...).
 *   x, r  f32 [M][K]   the projection output and the residual stream
 *   s     f32 [M][K]   optional (NULL): the new residual stream v; must not
 *                      overlap x or r (LK_ERR_ARG), since every block of a row
 *                      reads the whole row
 *   gain, xn, xq, xl, xs and the errors as lk_rmsnorm_quant.
 */
lk_status lk_add_rmsnorm_quant(const float* x, const float* r, const float* gain, int M, int K, float eps,
                               lk_mode mode, float* s, float* xn, int8_t* xq, int8_t* xl, float* xs,
                               const lk_launch_cfg* cfg, cudaStream_t stream);

/*
 * The gated activation between a decoder's gate/up and down projections,
 * quantized for the down projection ("kernels.rs" GLU lk_gemv_glu with ACT -1;
 * QWEN38_EXTRA_KERNELS gk_silu_had_q8 / gk_silu_had_q8_hl):
 *   h[t][j] = (g / (1 + expf(-g))) * u,  g = gate[t*ld + j], u = up[t*ld + j]
 * each operation rounded to f32 as written (expf is the CUDA math library's,
 * within 2 ulp), then the activation quantizer of `mode` on h per 32 values.
 *   gate, up  f32 rows of F values at a row pitch of ld >= F floats (for a
 *             fused gate/up output [M][2F]: gate = y, up = y + F, ld = 2F)
 *   h         f32 [M][F]: required under LK_DEQUANT (the down projection's
 *             activation), optional otherwise
 *   hq, hl, hs  [M][F], [M][F], [M][F/32] as lk_quantize_act's outputs
 * F must be a multiple of 32 (LK_ERR_SHAPE); 0 <= M <= LK_MAX_M.
 */
lk_status lk_swiglu_quant(const float* gate, const float* up, int M, int F, long ld, lk_mode mode, float* h,
                          int8_t* hq, int8_t* hl, float* hs, const lk_launch_cfg* cfg, cudaStream_t stream);

/*
 * The activation quantizer alone ("kernels.rs" QUANT lk_quant, PRELUDE
 * lk_quant_lane / lk_two_scale / lk_two_words).  Per 32-value group with
 * a = max|v|:
 *   LK_INT8ACT: s = a/127, hi = rn(v/s); a group with a < 127 * 2^-126
 *               (a/127 not a normal float, a = 0 included) gets s = 1 and
 *               hi = 0, so hi always lies in [-127, 127]
 *   LK_TWOPASS: s = max(a, 1e-30)/127; hi = clamp(rn(v/s));
 *               lo = clamp(rn(fma(-hi, s, v) / (s/128)))
 * rn rounds to nearest even; divisions are IEEE.  mode LK_DEQUANT is an
 * argument error (nothing to quantize).
 */
lk_status lk_quantize_act(const float* x, int M, int K, lk_mode mode, int8_t* xq, int8_t* xl,
                          float* xs, const lk_launch_cfg* cfg, cudaStream_t stream);

/*
 * y = W x for M <= 8 activation rows that share each weight read
 * ("kernels.rs" GEMV_Q8 lk_gemv_q8 and lk_q8_rows_dot; PRELUDE lk_q8_term,
 *  lk_q8_sum4).  Quantized modes: each 32-block's int8 dot d (and e of the
 *  low words) is exact; block b's step goes into partial b mod 4 in ascending
 *  b:  Int8Act p = fma(w*s, d, p);  TwoPass p = fma(w, fma(s, d, (s/128)*e), p);
 *  y = (p0 + p2) + (p1 + p3).  Dequant: the products are summed in f32 over
 *  a stretch of the row -- a 32-block in the direct kernel (scaled by the
 *  f16 weight scale in f64), a stage of at most 8192 values in the bulk-copy
 *  ring kernel (each block's part scaled in f32) -- and the stretches are
 *  added in f64; the f64 row sum is rounded to f32 once (within 1e-5 of
 *  sum|W x| of the exact value, not bit-fixed).  For 2..8
 *  rows of Int8Act / TwoPass the dots run on the tensor cores (f16 MMA on
 *  the exact int8 levels, or int8 MMA; accumulators that hold the exact
 *  integer dot); the combine is the same, so every kernel gives the same
 *  bits.
 *   Dequant reads x; Int8Act reads xq, xs; TwoPass reads xq, xl, xs.
 *   argmax_parts  optional u64 [M][*n_parts_out]: the lm-head epilogue
 *                 (model-as-a-kernel "megakernel.cu" amax_key with
 *                 EP_F32_AMAX): each launched block writes the largest key
 *                 of its rows, key = order-preserving bits of the f32 logit
 *                 (with -0 read as +0) in the high half and 0xFFFFFFFF - row
 *                 in the low half.  Reduce with lk_argmax.  Size it with
 *                 lk_argmax_parts_max(N) entries per activation row.
 *   n_parts_out   HOST int*, required when argmax_parts is given: the number
 *                 of partial keys written per activation row.
 */
lk_status lk_gemv_q8(const int8_t* wq, const uint16_t* ws, int N, int K, lk_mode mode,
                     const float* x, const int8_t* xq, const int8_t* xl, const float* xs, int M,
                     float* y, uint64_t* argmax_parts, int* n_parts_out, const lk_launch_cfg* cfg,
                     cudaStream_t stream);

/* One matrix of a grouped GEMV. */
typedef struct {
  const int8_t* wq;        /* [N][K] levels                                         */
  const uint16_t* ws;      /* [N][K/32] f16 scales                                  */
  int N;
  int reserved;
  float* y;                /* [M][N] output                                         */
} lk_gemv_target;

/*
 * Several GEMVs that read the same activation (the q, k and v projections
 * of a decoder layer, "kernels.rs" GEMV_Q8 applied per matrix): the same as
 * calling lk_gemv_q8 for each target in turn, without argmax, and with the
 * same bits.  Where the tensor-core kernel takes every matrix (2..8 rows,
 * lk_gemv_kernel_for == 3) the group is ONE launch whose 16-row tiles of all
 * matrices are dealt over the grid together.  Otherwise two or more matrices
 * that the bulk-copy ring arrangement takes run as ONE launch of the chain
 * kernel without barriers (each matrix's quads dealt on from where the
 * previous matrix's stopped); anything else is one launch per target.
 * The library extends the pages here; they have no grouped call.
 *   targets  HOST array of n (1..LK_MAX_GROUP) matrices with the same K;
 *            read during the call only (a captured graph keeps the values).
 *   other arguments as lk_gemv_q8.
 * Errors: LK_ERR_ARG for n out of range or a null target field, and every
 * error lk_gemv_q8 reports for a target.
 */
lk_status lk_gemv_q8_group(const lk_gemv_target* targets, int n, int K, lk_mode mode, const float* x,
                           const int8_t* xq, const int8_t* xl, const float* xs, int M, const lk_launch_cfg* cfg,
                           cudaStream_t stream);

/*
 * The gated projection pair of a decoder's MLP with the SwiGLU and the
 * down projection's quantizer in its epilogue ("kernels.rs" GLU lk_gemv_glu
 * with ACT -1 and a quantized output; QWEN38_EXTRA_KERNELS gk_silu_had_q8):
 *   g = Wg x, u = Wu x (each exactly lk_gemv_q8's value for its matrix),
 *   h = (g / (1 + expf(-g))) * u as lk_swiglu_quant computes it, and h
 *   quantized per 32 outputs by the quantizer of `mode`.
 *   wg, wsg / wu, wsu  the gate and up matrices, F rows of K each
 *   x, xq, xl, xs, M   the activation, as lk_gemv_q8
 *   gu     f32 [2][M][F]: receives the gate values gu[0][t][o] and the up
 *          values gu[1][t][o] (always written: the epilogue reads them back)
 *   h      f32 [M][F]: required under LK_DEQUANT (the down projection's
 *          activation), optional otherwise
 *   hq, hl, hs  [M][F], [M][F], [M][F/32]: the quantized h (LK_INT8ACT,
 *          LK_TWOPASS), as lk_quantize_act writes them
 *   cnt    int32 [F/32] zeroed by the caller before the first call; every
 *          completed call leaves it zeroed (after LK_ERR_DEVICE_TIMEOUT zero it
 *          again).  Calls that may run at the same time need separate ones.
 *          May be NULL: then the two launches below are used.
 * With one activation row (M = 1), K % 256 == 0 and cnt given, this is ONE
 * launch of the bulk-copy ring kernel over the 2F rows of both matrices
 * (interleaved in 32-row tiles, so most groups of 32 outputs are finished by
 * the block that computed them; a group split between two blocks is finished
 * by the one whose count completes it).  Otherwise the two GEMVs run as
 * lk_gemv_q8_group and the SwiGLU as lk_swiglu_quant.  Same bits either way.
 * F must be a multiple of 32 (LK_ERR_SHAPE).  The library extends the pages
 * here only in fusing the pair's two matrices into one launch.
 */
lk_status lk_gemv_q8_glu(const int8_t* wg, const uint16_t* wsg, const int8_t* wu, const uint16_t* wsu, int F, int K,
                         lk_mode mode, const float* x, const int8_t* xq, const int8_t* xl, const float* xs, int M,
                         float* gu, float* h, int8_t* hq, int8_t* hl, float* hs, int* cnt, const lk_launch_cfg* cfg,
                         cudaStream_t stream);

/*
 * RMSNorm -> quantize -> GEMV in one launch: every block of the bulk-copy
 * ring kernel computes the activation in shared memory from the raw rows x
 * itself (the in-block norm prologue of model-as-a-kernel "megakernel.cu"
 * ph_gemv, with the arithmetic of lk_rmsnorm_quant / lk_quantize_act), then
 * runs lk_gemv_q8's GEMV on it.  The results are bit for bit those of
 * lk_rmsnorm_quant (gain != NULL) or lk_quantize_act (gain == NULL; Dequant
 * then uses x as is) followed by lk_gemv_q8, without the intermediate
 * buffers or launches.
 *   x     f32 [M][K] raw activation rows (4-byte aligned)
 *   gain  f32 [K] RMSNorm gain, or NULL for the quantizer alone
 *   y, argmax_parts, n_parts_out   as lk_gemv_q8
 * Needs the ring kernel: K % 256 == 0 and the activation area fitting in
 * shared memory (lk_gemv_kernel_for(...) == 2); otherwise LK_ERR_SHAPE.  With
 * cfg->pdl set, the launch is a programmatic dependent launch: its weight
 * stream starts while the previous kernel on the stream finishes, and it
 * reads x only after that kernel has completed.  cfg->path must be 0 or 2.
 */
lk_status lk_rmsnorm_quant_gemv_q8(const int8_t* wq, const uint16_t* ws, int N, int K, lk_mode mode,
                                   const float* x, const float* gain, float eps, int M, float* y,
                                   uint64_t* argmax_parts, int* n_parts_out, const lk_launch_cfg* cfg,
                                   cudaStream_t stream);

/*
 * One step of a GEMV chain: RMSNorm (gain != NULL) or the quantizer alone
 * (gain == NULL) of the raw rows x, then y = W x, as lk_rmsnorm_quant_gemv_q8.
 */
typedef struct {
  const int8_t* wq;        /* [N][K] levels, 16-byte aligned                       */
  const uint16_t* ws;      /* [N][K/32] f16 scales, 16-byte aligned                */
  int N, K;                /* K % 256 == 0                                          */
  const float* x;          /* [M][K] raw f32 input rows                             */
  const float* gain;       /* [K] RMSNorm gain, or NULL                             */
  float* y;                /* [M][N] output                                         */
  uint64_t* argmax_parts;  /* optional [M][lk_argmax_parts_max(N)] partial keys     */
  int32_t* argmax_idx;     /* optional [M]: first index of the max of y (needs parts) */
  int wait;                /* nonzero: x reads an earlier step's output (the blocks
                              meet at a grid-wide barrier before this step)          */
  int reserved;
} lk_chain_op;

/* Bytes of the sync buffer lk_gemv_chain needs (zeroed once by the caller). */
size_t lk_chain_sync_bytes(void);

/*
 * A chain of steps in ONE cooperative launch (one block per SM): the form of
 * model-as-a-kernel "megakernel.cu" (phases separated by a grid barrier,
 * the next GEMV's weights streamed during it) for the projection path.  Each
 * step's result is bit for bit lk_rmsnorm_quant_gemv_q8 of that step.  Steps
 * run in order; a step with `wait` set starts after every block finished the
 * steps before it, so its x may be an earlier step's y; a step without it
 * must not read earlier outputs.  An argmax_idx step is followed by a barrier
 * and a final reduce.
 *   ops      HOST array of n_ops steps (validated and sized from it)
 *   ops_dev  DEVICE copy of the same n_ops entries, read by the kernel
 *   sync     DEVICE buffer of lk_chain_sync_bytes() bytes, zero before the
 *            first call and left consistent by every completed call; after
 *            LK_ERR_DEVICE_TIMEOUT zero it again.  Chains that may run at the
 *            same time need separate sync buffers.
 * Every grid-barrier wait is bounded (option "wait_us"); a timeout sets the
 * device error word (lk_device_error).  LK_ERR_SHAPE if a step's K is not a
 * multiple of 256 or the largest activation area does not fit in shared
 * memory next to four weight stages.  cfg: pdl applies to a chain without
 * barriers (a chain with barriers is always a cooperative launch), prefill
 * as for the ring kernel; the other fields do not apply (one block per SM).
 */
lk_status lk_gemv_chain(const lk_chain_op* ops, const lk_chain_op* ops_dev, int n_ops, lk_mode mode, int M,
                        float eps, uint32_t* sync, const lk_launch_cfg* cfg, cudaStream_t stream);

/*
 * Which GEMV kernel a call of this shape would launch with these settings,
 * for 16-byte aligned operands: 1 the direct-load kernel (any K % 32 == 0,
 * M <= LK_MAX_M), 2 the bulk-copy ring kernel (K % 256 == 0 and the
 * activation fits in shared memory), 3 the tensor-core kernel (LK_INT8ACT
 * or LK_TWOPASS, cfg->mma_min_m (default 2) <= M <= LK_MAX_BATCH,
 * K % 256 == 0, no argmax keys, for split-K every chunk non-empty
 * (S <= K / 128), and the activation (a chunk's columns under split-K)
 * fitting in shared memory next to a weight ring), 0 none (invalid shape or
 * settings, or a kernel
 * forced by cfg->path but not applicable).  S = 0 asks about lk_gemv_q8,
 * S >= 1 about lk_gemv_q8_splitk.  cfg may be NULL (the defaults).
 */
int lk_gemv_kernel_for(int N, int K, lk_mode mode, int M, int S, const lk_launch_cfg* cfg);

/*
 * The split-K chunk count this library's measurements favour for a GEMV of
 * this shape (GB300): S > 1 where, at 2..LK_MAX_BATCH activation rows of
 * Int8Act / TwoPass on the tensor-core kernel, holding only a chunk of the
 * activation rows per block (more weight stages in flight, more work units
 * than tiles) outweighs the extra combine launch; 1 elsewhere (one row,
 * Dequant, a shape the tensor-core kernel does not take).  Split-K is the
 * pages' own operation with its own summation order: lk_gemv_q8_splitk +
 * lk_splitk_combine do not give lk_gemv_q8's bits, so a caller chooses it
 * (the library's extension: the pages fix S per projection by hand).
 */
int lk_splitk_chunks_for(int N, int K, lk_mode mode, int M);

/*
 * Bytes of the split-K partial buffer for (mode, S, M, N): S*M*N values,
 * f64 under LK_DEQUANT, f32 otherwise.
 */
size_t lk_splitk_workspace_bytes(lk_mode mode, int S, int M, int N);

/*
 * The split-K partial GEMV (QWEN38_EXTRA_KERNELS "SPLIT-K FOR THE NARROW
 * PROJECTIONS", gk_gemv_hl_sk).  Chunk c in [0, S) owns the 32-blocks
 * [4*floor(c*G/S), 4*floor((c+1)*G/S)) with G = floor(K/128), the last chunk
 * ending at K/32 (the balanced split of "kernels.rs" GEMM_BLK over four-block
 * groups).  A chunk's value is lk_gemv_q8's rule restricted to its blocks
 * (partial index = global block index mod 4); Dequant chunks are f64 sums.
 * Writes part[c][t][o] (layout [S][M][N], f32 or f64 by mode).  1 <= S <= 64.
 * part_bytes must be >= lk_splitk_workspace_bytes(mode, S, M, N).  Up to
 * LK_MAX_M rows on any kernel; 2..LK_MAX_BATCH rows of Int8Act / TwoPass
 * on the tensor-core kernel, each block holding only its chunk's columns of
 * the activation rows (past LK_MAX_M rows the only kernel: LK_ERR_SHAPE
 * where it does not take the shape).
 */
lk_status lk_gemv_q8_splitk(const int8_t* wq, const uint16_t* ws, int N, int K, lk_mode mode,
                            const float* x, const int8_t* xq, const int8_t* xl, const float* xs,
                            int M, int S, void* part, size_t part_bytes, const lk_launch_cfg* cfg,
                            cudaStream_t stream);

/*
 * The split-K combine (QWEN38_EXTRA_KERNELS gk_sk_combine): a separate
 * kernel, never atomics: y[t][o] = (((0 + part[0][t][o]) + part[1][t][o]) +
 * ...) in ascending chunk order, in f32 (f64 then one rounding to f32 under
 * LK_DEQUANT).  Same inputs give the same bits on every run.  0 <= M <=
 * LK_MAX_BATCH.  cfg: pdl (it reads the partials only after the launch
 * before it completes); the other fields do not apply.
 */
lk_status lk_splitk_combine(lk_mode mode, const void* part, int S, int M, int N, float* y,
                            const lk_launch_cfg* cfg, cudaStream_t stream);

/* Upper bound on the argmax partial keys per activation row that lk_gemv_q8
 * writes for an N-row matrix. */
int lk_argmax_parts_max(int N);

/* Entries of the u64 scratch lk_argmax needs per activation row when it
 * reduces logits directly ("kernels.rs" argmax_blocks: clamp(ceil(N/2048),
 * 1, 64) blocks). */
int lk_argmax_scratch_entries(int N);

/*
 * First index of the maximum of each of M rows ("kernels.rs" module doc on
 * the arg-max: the lowest index among equal maxima; "megakernel.cu"
 * ph_argmax_part / ph_argmax_fin).  Two forms:
 *   parts != NULL: reduce the n_parts keys per row that lk_gemv_q8 wrote
 *                  (logits and scratch are ignored);
 *   parts == NULL: reduce logits f32 [M][N] in two kernels through scratch
 *                  (u64, M * lk_argmax_scratch_entries(N) entries).
 * idx int32 [M].  Logits compare as f32 values with -0 == +0; the result for
 * NaN logits is unspecified.  N >= 1.
 */
lk_status lk_argmax(const float* logits, const uint64_t* parts, int n_parts, int M, int N,
                    int32_t* idx, uint64_t* scratch, cudaStream_t stream);

/*
 * lk_argmax's logits form without any caller-provided scratch, for callers
 * that cannot allocate device memory where they call it: code being captured
 * into a CUDA graph (cudaMalloc is not allowed during stream capture), the
 * enqueue path of an inference-engine plugin that must not allocate, or a
 * real-time loop that forbids allocator calls.  The source pages have no
 * counterpart of this entry point; it computes what lk_argmax(logits, NULL,
 * ...) computes.
 *   logits f32 [M][N], idx int32 [M]; 1 <= M <= LK_MAX_M, N >= 1.
 * The partial keys go to a file-scope device array of LK_MAX_M * 64 keys
 * (4 KB) that every GPU which loads the library keeps until the process
 * exits; shapes that would need more return LK_ERR_WORKSPACE (none do within
 * M <= LK_MAX_M).  The first call on each device looks the array's address up
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Host threads may make first calls at the same
 * time (the per-device address cache is atomic).  The address belongs to the
 * device's context: after cudaDeviceReset() of a device it is stale, as are
 * the library's other per-device addresses, so do not call the library on a
 * device after resetting it.  The call allocates and frees nothing.  All
 * calls share the array: calls that can overlap on the GPU (other streams,
 * other threads) race and must be serialized by the caller; the array keeps
 * the last call's keys, which every call overwrites before reading.
 */
lk_status lk_argmax_noalloc(const float* logits, int M, int N, int32_t* idx, cudaStream_t stream);

/*
 * The GGUF block formats other than Q8_0 ("kernels.rs" decoder library: lk_sub
 * decodes a 32-value sub-block of any of them into int8 levels with a scale
 * d and an offset c per half; lk_row_dot / lk_sub_dot run the projection).
 * `format` is the ggml type number the pages use:
 *   2 Q4_0, 3 Q4_1, 6 Q5_0, 7 Q5_1, 20 IQ4_NL, 39 MXFP4 (32 values a block),
 *   10 Q2_K, 11 Q3_K, 12 Q4_K, 13 Q5_K, 14 Q6_K, 23 IQ4_XS (256 values a block),
 * each block in the format's own byte layout (little-endian f16 scales).  A
 * row of K values is lk_format_row_bytes(format, K) bytes (0: an unknown
 * format or K not a whole number of blocks); a matrix is N such rows back
 * to back, 16-byte aligned.
 */
size_t lk_format_row_bytes(int format, int K);

/*
 * y = W x for a block-format matrix w (N rows) and M <= LK_MAX_M activation
 * rows, the activation as lk_gemv_q8's (x f32 under LK_DEQUANT; xq, xs and
 * under LK_TWOPASS xl, from lk_quantize_act).  The weight of value i of a
 * sub-block is RN(RN(d level_i) + c) in f32.  Quantized modes, bit-fixed
 * ("kernels.rs" lk_row_dot with lk_sub_dot): sub-block sb of a row is in
 * lane sb mod 32; with dh0/dh1 the exact int8 dots of the levels with the
 * activation words over values 0..15 / 16..31 and sh0/sh1 the words' sums,
 *   part = ((d0 dh0 + c0 sh0) + d1 dh1) + c1 sh1   (each op rounded to f32;
 *          TwoPass: part + 2^-7 times the same with the low words),
 * the lane's f32 sum gets s[sb] * part in ascending sb, and the lanes meet in
 * the shuffle-down tree (lane l adds lane l + d, d = 16, 8, 4, 2, 1).
 * Dequant: within 1e-5 of sum |w x| per row of the exact sum (the pages sum
 * in f64; here each lane's products are summed in f32 with a compensation
 * term, the lanes in f64).  K % 256 == 0 and a row a multiple of 16 bytes
 * (LK_ERR_SHAPE otherwise; every format at K = 4096); K = 0 writes zeros.
 * cfg: pdl, grid_ctas.  The library's extension of the Q8_0 path to the
 * pages' other formats.
 */
lk_status lk_gemv_blk(int format, const uint8_t* w, int N, int K, lk_mode mode, const float* x, const int8_t* xq,
                      const int8_t* xl, const float* xs, int M, float* y, const lk_launch_cfg* cfg,
                      cudaStream_t stream);

/*
 * Test hook: the decoded weights out[o][k] = RN(RN(d level) + c) of a
 * block-format matrix (f32 [N][K]), by the same decoders lk_gemv_blk uses.
 */
lk_status lk_dequant_blk(int format, const uint8_t* w, int N, int K, float* out, cudaStream_t stream);

/*
 * Test hook: the exact int32 block dots of one activation row, computed by the
 * same lane arrangement the GEMV uses ("kernels.rs" lk_q8_block_dot).
 *   d[o][b] = sum_k wq[o][32b+k] * xq[32b+k];  e likewise with xl (if both xl
 *   and e are non-NULL).  d, e int32 [N][K/32].
 */
lk_status lk_q8_block_dots(const int8_t* wq, int N, int K, const int8_t* xq, const int8_t* xl,
                           int32_t* d, int32_t* e, cudaStream_t stream);

/*
 * The two diagnostic options (process-wide).  Neither changes which kernel a
 * call launches, how it is launched or any result; launch settings are per
 * call (lk_launch_cfg).  Names:
 *   "trace"       1: the ring and chain kernels write block 0's timestamps
 *                 to the trace buffer (lk_trace_read); 2: the chain also
 *                 records every block's and block 0's warps' step ends, and
 *                 when block 0's warps' first stage of each step was there
 *                 and computed (from index 2048);
 *                 3: launch timeline: every ring, chain, tensor-core, norm
 *                 and quantize launch made after the option was set owns a
 *                 record of LK_TRACE_REC entries (in launch order, 512
 *                 records, wrapping):
 *                 [0] block 0 start, [1] block 0 past the wait on the
 *                 previous kernel (fused launches: the prologue's start; it
 *                 waits inside, after requesting the norm gains), [2] block
 *                 0's activation ready, [3] the last block's end, [4] block
 *                 0's end (all %globaltimer ns), [5] kernel (1 ring, 2 chain,
 *                 3 tensor-core, 4 norm, 5 quantize, 6 split-K combine),
 *                 [6] rows (steps, for a chain), [7] block 0's first weight
 *                 stages issued.  Setting the option restarts the record
 *                 count.
 *   "wait_us"     time limit of every device-side wait, microseconds
 *                 (0 = default, 2 s; at most 6 * 10^7)
 * Unknown names or out-of-range values return LK_ERR_ARG; lk_get_option
 * returns -1 for an unknown name.
 */
lk_status lk_set_option(const char* name, long value);
long lk_get_option(const char* name);

/*
 * Synchronizes the current device and reads the device-side error word that
 * bounded waits set when they give up (0 = none).  *code receives the raw
 * word; returns LK_ERR_DEVICE_TIMEOUT if it is non-zero, LK_OK otherwise.
 * reset != 0 clears the word.
 */
lk_status lk_device_error(int reset, int* code);

/*
 * Tracing (cf. the per-phase clock stamps of model-as-a-kernel
 * "megakernel.cu"): with option "trace" set, block 0 of the last ring or
 * chain launch records %globaltimer nanoseconds.  Ring kernel: [0] start,
 * [1] after the dependency wait, [2] activation ready, [3 + w] warp w done.
 * Chain: [0] start, then per step i: [1 + 3i] step start (after its barrier),
 * [2 + 3i] activation ready, [3 + 3i] block 0's rows done; with "trace" 2,
 * from entry 1024 on: [1024 + i*G + b] block b's end of step i (G blocks),
 * and from entry 1024 + n_ops*G: [.. + i*W + w] warp w of block 0 at the end
 * of its step-i rows (W warps), while they fit in the buffer.  Synchronizes the
 * device and copies the first n (<= 4096) entries to host_out.
 */
lk_status lk_trace_read(uint64_t* host_out, int n);

/*
 * Test hook of the failure path: launches one block that waits, with the
 * library's bounded wait, on an mbarrier that nothing completes.  The wait
 * gives up after limit_us microseconds (1 .. 10^7), sets the device error
 * word and returns; lk_device_error then reports LK_ERR_DEVICE_TIMEOUT and the
 * context stays usable.
 */
lk_status lk_selftest_wait_timeout(unsigned limit_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LK_H */
