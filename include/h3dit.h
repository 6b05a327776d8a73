/*
 * h3dit.h - C ABI of the B300 (sm_103a) forward pass of the MiniMax-H3 DiT
 * block and of the 50-block denoiser step.
 *
 * The method is described by web pages about h3.c ("h3-metal"), an Apple
 * inference engine for MiniMax-H3:
 *   [alphalab]  "h3-metal 把 MiniMax-H3 搬上 Apple Silicon：突破與代價（2026）",
 *               model facts (33B dense single-stream Omni Transformer, 50 layers,
 *               full attention) and the author's test table (warm 50-block forward).
 *   [linlog]    linlog.top article 1265 on h3.c; sections "MiniMax H3：原生音频视频
 *               一体化生成" (AdaLN branch precomputed at inference), "h3.c 的核心设计"
 *               (QKV routed head-major), "int8 量化：从 36 秒到 19 秒" (dynamic int8),
 *               "DiT 融合内核：减少全局内存往返" (gated AdaLN fusion, arena aliasing),
 *               "Token 缩减：28% 的去噪时间消减" (horizontal-pair token reduction).
 *   [steinslab] "零 Python 依赖：Redis 作者的 3.5 秒端侧实验", section "极简主控逻辑"
 *               (spatial RoPE over t/h/w).
 *
 * Conventions for every entry point:
 *  - Every pointer argument named as device memory is a device pointer owned
 *    by the caller; the library never frees or keeps it past the call.  Host
 *    pointers (configs, weight tables, grids) are read during the call only.
 *  - BF16 tensors are row-major and token-major unless stated: [N][d] means
 *    row t (a token) is d consecutive bfloat16 values.  Weights are [out][in]
 *    (one row per output channel), the layout of a PyTorch Linear weight.
 *  - Work is enqueued asynchronously on the given cudaStream_t (0 = legacy
 *    default stream); nothing is synchronised except where stated.
 *  - No entry point allocates device memory on the hot path; scratch comes
 *    from the caller's workspace (h3dit_workspace_size).
 *  - Every call returns an h3dit_status.  On failure nothing is enqueued
 *    (argument errors) or the CUDA error is reported (launch errors), and
 *    h3dit_last_error() returns a message for the calling thread.  The
 *    library never prints, exits or aborts.
 *  - Device-side waits are bounded: a kernel whose pipeline wait runs out
 *    sets a device error word and returns; h3dit_check_device_error() reads
 *    it and reports H3DIT_E_TIMEOUT.
 */
#ifndef H3DIT_H
#define H3DIT_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define H3DIT_VERSION 2

typedef enum {
  H3DIT_OK = 0,
  H3DIT_E_INVAL = 1,        /* a null pointer, a negative size, inconsistent shapes */
  H3DIT_E_UNSUPPORTED = 2,  /* a shape this build does not implement (see each call) */
  H3DIT_E_NOMEM = 3,        /* the workspace passed in is smaller than required */
  H3DIT_E_CUDA = 4,         /* a CUDA runtime or driver call failed */
  H3DIT_E_TIMEOUT = 5       /* a kernel's bounded pipeline wait ran out */
} h3dit_status;

/* Which projections run on dynamic int8 ([linlog] "int8 量化：从 36 秒到 19 秒"
 * compares the MLP alone, QKV alone and all four): H3DIT_INT8 = QKV,
 * out-projection, FC1 and FC2; H3DIT_INT8_MLP = FC1 and FC2; H3DIT_INT8_QKV =
 * the QKV projection only.  The other projections run in BF16. */
typedef enum { H3DIT_BF16 = 0, H3DIT_INT8 = 1, H3DIT_INT8_MLP = 2, H3DIT_INT8_QKV = 3 } h3dit_precision;

/* Shape of one block.  The pages give none of these numbers.
 *  d            model width; a multiple of 256, at most 8192
 *  heads        attention heads; heads * head_dim == d
 *  head_dim     64 or 128
 *  ffn          MLP width F; a multiple of 256
 *  eps          LayerNorm epsilon (LayerNorm: biased variance, no affine)
 *  rope_sections head-dim widths of the (t, y, x) RoPE sections; even, sum head_dim
 *  rope_theta   RoPE base; pair i of a section of width s turns by pos * theta^(-2i/s)
 *  precision    an h3dit_precision: which projections are dynamic int8 */
typedef struct {
  int d;
  int heads;
  int head_dim;
  int ffn;
  float eps;
  int rope_sections[3];
  float rope_theta;
  int precision;
} h3dit_config;

/* One block's projection weights, device pointers.  Each projection is BF16
 * or int8 as the config's precision says (the other form of that projection
 * is never read):
 * BF16 projection: a BF16 [out][in] matrix; its scale pointer is unused (may
 *   be NULL).
 * int8 projection: per-output-channel int8 codes [out][in] in operand form --
 *   each code stored as the BF16 value of the same integer (exact), the form
 *   the tensor cores read, made once from int8 codes by h3dit_widen_codes --
 *   and fp32 per-output-channel scales (h3dit_quantize_weight), as in [linlog]
 *   "int8 量化" (per-output-channel weight scales).  sm_103a has no integer
 *   tensor-core MMA; the int8 products are run exactly on the BF16 path (see
 *   h3dit_linear_i8).
 *   w_qkv [3d][d]  rows 0..d-1 give Q (head h = rows h*Dh..), d..2d-1 K, 2d..3d-1 V
 *   w_o   [d][d]   attention output projection
 *   w1    [F][d]   MLP FC1
 *   w2    [d][F]   MLP FC2
 * codes_int8 = 1 keeps the int8 projections' weights as plain int8 codes
 *   (one byte each, 8-byte aligned: half the bytes of the operand form, the
 *   resident-memory saving of [linlog] "int8 量化"); the library widens each
 *   into the workspace just before its projection (h3dit_widen_codes'
 *   rule, so the results equal the operand-form ones bit for bit), at the
 *   cost of one HBM pass over the operand form per projection and block.
 *   0 = the operand form above.  BF16 projections ignore it. */
typedef struct {
  const void* w_qkv;
  const void* w_o;
  const void* w1;
  const void* w2;
  const float* s_qkv;
  const float* s_o;
  const float* s1;
  const float* s2;
  int codes_int8;
} h3dit_block_weights;

/* Target-video tokens: T*Hh*W consecutive rows starting at row `offset`,
 * ordered t-major, then y, then x.  Other rows (text, audio, conditions)
 * are never reduced. */
typedef struct {
  int offset;
  int T;
  int Hh;
  int W;
} h3dit_video_grid;

/* Token-reduction schedule of the step ([linlog] "Token 缩减"): the video
 * is paired after block reduce_after_block (0-based) and restored before
 * block restore_before_block.  pos_reduced: device [N_reduced][3] fp32
 * positions of the reduced sequence, or NULL to use the pair-mean positions
 * (h3dit_reduced_positions). */
typedef struct {
  h3dit_video_grid grid;
  int reduce_after_block;
  int restore_before_block;
  const float* pos_reduced;
} h3dit_reduction;

/* Consecutive token segments with their own AdaLN modulation ([linlog]
 * "音频处理": the reference audio is conditioned at its own timestep, 1.0, so
 * its precomputed AdaLN vectors differ from the video's).  Segment k covers
 * rows start[k] .. start[k+1]-1 (the last runs to the end); 1 <= count <= 4,
 * start[0] = 0, starts increasing.  With a token reduction every boundary
 * must lie outside the paired video grid (both members of a pair share a
 * segment); boundaries after the grid move up with the rows it removes. */
typedef struct {
  int count;
  int start[4];
} h3dit_segments;

/* ---------------------------------------------------------------- housekeeping */

/* Message of the last failed call on this thread ("" if none).  The string
 * stays valid until the next call on this thread. */
const char* h3dit_last_error(void);

/* H3DIT_VERSION of the loaded library. */
int h3dit_version(void);

/* Synchronises `stream`, then reads and clears the device error word set by
 * a kernel whose bounded wait ran out.  H3DIT_OK if clear, H3DIT_E_TIMEOUT
 * if set, H3DIT_E_CUDA if the synchronisation itself failed. */
h3dit_status h3dit_check_device_error(cudaStream_t stream);

/* Launch behaviour.  Calls are asynchronous and stream-ordered.  The block
 * and step kernels are launched with programmatic stream serialisation:
 * each may be scheduled while the kernel before it on the stream retires
 * its CTAs, and waits for that kernel (griddepcontrol.wait) before it
 * touches global memory, so the results are those of plain stream order.
 * Environment switches for A/B measurement only (all give the same bits;
 * read at every call, H3DIT_DISABLE_GATED_ADALN once per process): H3DIT_PDL=0 plain launches; H3DIT_GEMM_SINGLE_CTA=1
 * projections on single CTAs instead of CTA pairs; H3DIT_GEMM_TAIL=0 no
 * half tiles in a short last wave; H3DIT_GEMM_BAND=k raster bands of k
 * N-tiles (default 16); H3DIT_ATTN_PERSIST=0 attention with one CTA per
 * unit instead of persistent CTAs; H3DIT_DISABLE_GATED_ADALN=1 the gated residual and
 * the following AdaLN as two launches.  One switch changes rounding:
 * H3DIT_ATTN_SPLIT=0 runs the attention units of a short last wave whole,
 * instead of as CTA pairs that each take half of the keys and combine their
 * partial results (the same softmax; the combine rounds differently). */

/* ---------------------------------------------------------------- failure testing
 * Not part of the method (the pages have no counterpart); these let a test
 * drive the failure paths without faulting or hanging a GPU.
 *
 * Host-side injection: with the environment variable H3DIT_FAULT set to
 * alloc, arg, shape or launch, h3dit_block_forward(_seg) and
 * h3dit_step_forward(_seg) fail on purpose where that failure would arise
 * and report E_NOMEM (workspace too small), E_INVAL (invalid argument),
 * E_UNSUPPORTED (unsupported shape) or E_CUDA (the first launch failed);
 * nothing is enqueued.  The variable is read at every call.
 *
 * h3dit_test_set_wait_limit: the device-side limit of every pipeline wait
 * on the current device, in nanoseconds (0 restores the default, 2 s).  A
 * kernel whose wait runs out raises the device error word, lets its own
 * copies and tensor-core work in flight finish, frees its tensor memory and
 * returns.  Synchronous (a copy to a device variable).
 *
 * h3dit_test_stall_next_gemm: the next BF16 projection launched by the
 * library (any entry point, any thread) runs with the TMA producer of its
 * first CTA stopping before k-block `kblock` of its first tile; nothing is
 * loaded for that stage, so the tensor-core thread's wait on it runs out
 * after the wait limit and the launch ends with the device error word set
 * (h3dit_check_device_error then reports E_TIMEOUT, and that launch's
 * output is invalid).  -1 cancels a pending request; a kblock past the
 * launch's last k-block is ignored.  E_INVAL for kblock < -1. */
h3dit_status h3dit_test_set_wait_limit(unsigned long long ns);
h3dit_status h3dit_test_stall_next_gemm(int kblock);

/* Per-kernel-class timing with CUDA events recorded on the launch stream
 * around every launch while enabled (off by default).  Classes:
 * 0 row kernels, 1 QKV GEMM, 2 attention, 3 out-projection GEMM, 4 FC1 GEMM,
 * 5 FC2 GEMM, 6 token reduce/restore, 7 quantise.  h3dit_timing_read
 * synchronises the recorded events and returns the total milliseconds and
 * the number of kernel launches of a class since the last reset. */
h3dit_status h3dit_timing_enable(int on);
h3dit_status h3dit_timing_reset(void);
h3dit_status h3dit_timing_read(int kernel_class, double* total_ms, long long* launches);

/* ---------------------------------------------------------------- the block and the step */

/* Bytes of device workspace a block or step at n_tokens needs (tr may be
 * NULL; with a reduction the reduced stream's buffers are included; with an
 * int8 precision, room for the largest int8 weight in operand form, used
 * when the weights are given as int8 bytes). */
h3dit_status h3dit_workspace_size(const h3dit_config* cfg, int n_tokens,
                                  const h3dit_reduction* tr, size_t* bytes);

/* One dense single-stream DiT block, in place on x ([alphalab] model facts;
 * [linlog] "DiT 融合内核"):
 *   h  = LN(x) * (1 + scale1) + shift1
 *   q, k, v = h W_qkv^T, heads split, q and k turned by 3D RoPE at `pos`
 *   o  = softmax(q k^T / sqrt(Dh)) v over all tokens (non-causal, no mask)
 *   x1 = x + gate1 * (o W_o^T)            rounded to BF16 and stored
 *   h2 = LN(x1) * (1 + scale2) + shift2   (fused with the residual)
 *   x  = x1 + gate2 * (GELU_tanh(h2 W1^T) W2^T)
 * mod: device fp32 [6][d] = shift1, scale1, gate1, shift2, scale2, gate2
 *      (the precomputed AdaLN branch, [linlog] "MiniMax H3" section).
 * x:   device BF16 [n_tokens][d], read and overwritten.
 * pos: device fp32 [n_tokens][3] (t, y, x) rotary positions.
 * ws:  device workspace of at least h3dit_workspace_size bytes, 256-byte aligned.
 * With an int8 precision the selected projections run on int8 codes
 * ([linlog] "int8 量化"): their inputs (h, o, h2 per token; u per token and
 * per 1024 channels) are quantised with h3dit_quantize_act's rule on the BF16
 * values, the weights are operand-form codes with per-output-channel scales,
 * and the outputs are dequantised to BF16 as h3dit_linear_i8 states;
 * attention stays BF16.  An int8 FC2 needs ffn <= 1024 or ffn % 1024 == 0.
 * Errors: E_INVAL (nulls, n_tokens < 1), E_UNSUPPORTED (shape outside the
 * limits of h3dit_config), E_NOMEM (ws_bytes too small), E_CUDA. */
h3dit_status h3dit_block_forward(const h3dit_config* cfg, const h3dit_block_weights* w,
                                 const float* mod, void* x, const float* pos, int n_tokens,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

/* The denoiser step: blocks 0..n_blocks-1 in order, block b with w[b] (a host
 * array of n_blocks weight tables) and mods + 6*d*b, in place on x
 * ([alphalab] 50 layers; [linlog] "--layers" trimming is n_blocks).  The
 * gated residual of each block also emits the next block's AdaLN input
 * ([linlog] "DiT 融合内核"), except at token-reduction boundaries.
 * tr: NULL for no reduction, else the schedule above; x keeps the full
 * resolution state while the reduced blocks run on a workspace copy.
 * Errors as h3dit_block_forward; E_INVAL also for a grid outside the rows. */
h3dit_status h3dit_step_forward(const h3dit_config* cfg, const h3dit_block_weights* w,
                                int n_blocks, const float* mods, void* x, const float* pos,
                                int n_tokens, const h3dit_reduction* tr, void* ws,
                                size_t ws_bytes, cudaStream_t stream);

/* h3dit_block_forward with per-segment modulation: mods is device fp32
 * [seg->count][6][d], segment k's shift1, scale1, gate1, shift2, scale2, gate2
 * applying to its rows (AdaLN-1, the gates and AdaLN-2 all take the row's
 * segment vectors).  seg: host pointer, read during the call.  count = 1
 * with mods [1][6][d] is h3dit_block_forward.  E_INVAL for a malformed
 * segment table. */
h3dit_status h3dit_block_forward_seg(const h3dit_config* cfg, const h3dit_block_weights* w,
                                     const float* mods, const h3dit_segments* seg, void* x,
                                     const float* pos, int n_tokens, void* ws, size_t ws_bytes,
                                     cudaStream_t stream);

/* h3dit_step_forward with per-segment modulation: mods is device fp32
 * [n_blocks][seg->count][6][d]; the segment boundaries are given at full
 * resolution and follow the token reduction as h3dit_segments says. */
h3dit_status h3dit_step_forward_seg(const h3dit_config* cfg, const h3dit_block_weights* w,
                                    int n_blocks, const float* mods, const h3dit_segments* seg,
                                    void* x, const float* pos, int n_tokens,
                                    const h3dit_reduction* tr, void* ws, size_t ws_bytes,
                                    cudaStream_t stream);

/* The block of h3dit_block_forward for callers that cannot allocate device
 * memory or hand over a workspace (for instance a host program whose single
 * allocator owns all device memory, or a serving loop that must not call
 * cudaMalloc because it can synchronise the device).  The pages have no
 * counterpart; this is an interface convenience of this library.
 * The scratch is a fixed 64 MiB array inside the library's device image;
 * the caller still passes x (in/out), weights, mod and pos as above.
 *  - The first call on each device looks up that array's device address
 *    (and so loads the library's device code there); make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process: after cudaDeviceReset on a device, do not call this entry
 *    point on that device again.
 *  - Every call on a device uses the same array, which keeps whatever the
 *    last call left in it (nothing has to start at zero).  Calls that can
 *    overlap on the GPU (other streams, other host threads) race on it:
 *    serialise them.
 *  - Arguments are checked as h3dit_block_forward checks them (E_INVAL,
 *    E_UNSUPPORTED) first; then shapes whose workspace
 *    (h3dit_workspace_size) exceeds 64 MiB are refused with H3DIT_E_NOMEM,
 *    before anything is enqueued.
 * Other errors as h3dit_block_forward. */
h3dit_status h3dit_block_forward_noalloc(const h3dit_config* cfg, const h3dit_block_weights* w,
                                         const float* mod, void* x, const float* pos, int n_tokens,
                                         cudaStream_t stream);

/* ---------------------------------------------------------------- the final layer */

/* One output head of the final layer ([linlog] "DiT 融合内核": the audio and
 * video AdaLN kernels are bound directly to residual-stream offsets, and the
 * BF16 final head applies AdaLN while it loads its projection tiles):
 *   out[r][c] = bf16( sum_k bf16(LN(x[row_start + r])_k (1 + scale_k) + shift_k) * w[c][k] )
 * for r < rows, LayerNorm as in the block (biased variance, cfg->eps).
 * shift, scale: device fp32 [d]; w: device BF16 [c_out][d]; out: device BF16
 * [rows][c_out]; c_out a multiple of 16 in 16..256; all 16-byte aligned. */
typedef struct {
  int row_start;
  int rows;
  const float* shift;
  const float* scale;
  const void* w;
  int c_out;
  void* out;
} h3dit_final_head;

/* The final layer over up to 4 heads (e.g. video and audio rows of the
 * residual stream x, device BF16 [n_tokens][d]).  x is only read; no
 * workspace and no normalised copy of the rows is made: each output row
 * first holds its row's LayerNorm statistics (8 bytes), then the result, so
 * an output must not overlap x or another head's output.  heads: host array,
 * read during the call.  Errors: E_INVAL (nulls, rows outside x, more than 4
 * heads), E_UNSUPPORTED (c_out), E_CUDA. */
h3dit_status h3dit_final_layer(const h3dit_config* cfg, const void* x, int n_tokens,
                               const h3dit_final_head* heads, int n_heads, cudaStream_t stream);

/* ---------------------------------------------------------------- core residual reuse */

/* The speed/quality presets of [linlog] (the preset table: "--core-reuse k"
 * refreshes the patch and head every step but runs the block core less
 * often; "--layers" is n_blocks of h3dit_step_forward; the later restore
 * point is restore_before_block of h3dit_reduction).  A caller runs the core
 * (h3dit_step_forward) on a fresh step and keeps its residual; on a reuse
 * step it adds that residual instead of running the blocks.
 * h3dit_core_residual: delta[i] = x_out[i] - x_in[i] in fp32 (exact when the
 *   two BF16 values' exponents are within 16 of each other).
 * h3dit_core_reuse: x[i] = bf16(x[i] + delta[i]), in place.
 * x_in, x_out, x: device BF16; delta: device fp32; count elements, a multiple
 * of 8; all 16-byte aligned. */
h3dit_status h3dit_core_residual(const void* x_in, const void* x_out, size_t count, float* delta,
                                 cudaStream_t stream);
h3dit_status h3dit_core_reuse(void* x, const float* delta, size_t count, cudaStream_t stream);

/* ---------------------------------------------------------------- quantisation */

/* Dynamic symmetric int8 quantisation ([linlog] "int8 量化": activations
 * quantised dynamically; FC2 input with one scale per 1024 channels).
 * For each row and each group of `group` consecutive columns:
 *   s = absmax / 127 (fp32, correctly rounded); q = clamp(rne(x / s), -127, 127)
 * with x / s correctly rounded in fp32 and ties to even; an all-zero group
 * gives s = 0 and q = 0.
 * x_bf16: device BF16 [rows][cols]; q: device int8 [rows][cols];
 * scales: device fp32 [rows][cols / group].  group divides cols; cols % 8 == 0. */
h3dit_status h3dit_quantize_act(const void* x_bf16, int rows, int cols, int group,
                                int8_t* q, float* scales, cudaStream_t stream);

/* Per-output-channel int8 weights ([linlog] "int8 量化"): the rule of
 * h3dit_quantize_act with one group per row of w [out][in]. */
h3dit_status h3dit_quantize_weight(const void* w_bf16, int out, int in, int8_t* q,
                                   float* scales, cudaStream_t stream);

/* The quantiser of h3dit_quantize_act writing each code as the BF16 value of
 * the same integer (the operand form of the int8 projections).  q_bf16 may
 * be x_bf16 itself (in place).  x_bf16, q_bf16: device BF16 [rows][cols],
 * 16-byte aligned; scales: device fp32 [rows][cols / group]. */
h3dit_status h3dit_quantize_codes(const void* x_bf16, int rows, int cols, int group,
                                  void* q_bf16, float* scales, cudaStream_t stream);

/* int8 codes -> operand form: out[i] = (bf16) q[i], exact.  q: device int8,
 * 8-byte aligned; q_bf16: device BF16, 16-byte aligned; count % 8 == 0. */
h3dit_status h3dit_widen_codes(const int8_t* q, size_t count, void* q_bf16,
                               cudaStream_t stream);

/* Int8 projection on operand-form codes ([linlog] "int8 量化": per-token
 * activation scales, per-output-channel weight scales, FC2 input with one
 * scale per 1024 channels and its scaled partial sums combined per group):
 *   group == k:  c[t][o] = bf16(act(acc[t][o] * sa[t] * sb[o])), sa [m]
 *   group <  k:  c[t][o] = bf16(act(sb[o] * sum_g sa[t][g] * acc_g[t][o])),
 *                sa [m][k / group], g ascending, sums in fp32
 * acc / acc_g are the exact integer sums of a_codes[t][j] * b_codes[o][j] over
 * all j, or over j in group g.  The tensor cores accumulate in fp32, which is
 * exact for integers below 2^24; every chunk of at most 1024 k-columns stays
 * below that (127^2 * 1024 < 2^24) and is drained and added in int32.
 * a_codes: device BF16 [m][k]; b_codes: device BF16 [n][k]; sb: device fp32
 * [n], 16-byte aligned; c: device BF16 [m][n].  act 0 none, 1 GELU (tanh).
 * n % 256 == 0, k % 64 == 0, k <= 131072; group < k needs group % 64 == 0,
 * group <= 1024 and group | k.  Codes outside [-127, 127] are the caller's
 * error (the exactness bound assumes them). */
h3dit_status h3dit_linear_i8(const void* a_codes, const float* sa, int group,
                             const void* b_codes, const float* sb, int m, int n, int k,
                             int act, void* c, cudaStream_t stream);

/* The exact int32 accumulators of h3dit_linear_i8 (group == k) without any
 * scaling: acc[t][o] = sum_j a_codes[t][j] * b_codes[o][j].  acc: device int32
 * [m][n], 16-byte aligned.  Shape limits as h3dit_linear_i8. */
h3dit_status h3dit_linear_i8_acc(const void* a_codes, const void* b_codes, int m, int n, int k,
                                 int32_t* acc, cudaStream_t stream);

/* ---------------------------------------------------------------- token reduction */

/* Rows left after pairing: n_tokens - T*Hh*floor(W/2). */
int h3dit_reduced_tokens(int n_tokens, const h3dit_video_grid* grid);

/* Horizontal-pair reduction ([linlog] "Token 缩减"): video columns (2j, 2j+1)
 * of every (t, y) row become their mean (fp32, rounded to BF16); an odd last
 * column and every non-video row are copied.  x_full: device BF16
 * [n_tokens][d]; x_red: device BF16 [h3dit_reduced_tokens][d]; side: device
 * BF16 [n_tokens][d] copy of x_full, or NULL when the caller keeps x_full
 * itself as the side state.  d % 8 == 0. */
h3dit_status h3dit_token_reduce(const void* x_full, int n_tokens, int d,
                                const h3dit_video_grid* grid, void* x_red, void* side,
                                cudaStream_t stream);

/* Restore ([linlog] "Token 缩减": each token returns its original value plus
 * its pair's learned update): a paired token i of pair p becomes
 *   side[i] + (x_red[p] - bf16(mean(side[2j], side[2j+1])))
 * computed in fp32 and rounded to BF16; every other row takes x_red's row.
 * With a zero update this is the identity, bit for bit.  x_full may alias side. */
h3dit_status h3dit_token_restore(const void* x_red, const void* side, int n_tokens, int d,
                                 const h3dit_video_grid* grid, void* x_full,
                                 cudaStream_t stream);

/* Pair-mean positions of the reduced sequence: device fp32 [n_tokens][3] ->
 * [h3dit_reduced_tokens][3]. */
h3dit_status h3dit_reduced_positions(const float* pos, int n_tokens,
                                     const h3dit_video_grid* grid, float* pos_red,
                                     cudaStream_t stream);

/* ---------------------------------------------------------------- the block's steps one by one */

/* AdaLN: h = bf16(LN(x) * (1 + scale) + shift), LayerNorm with biased
 * variance over d, fp32 arithmetic.  x, h: device BF16 [n][d]; shift, scale:
 * device fp32 [d]. */
h3dit_status h3dit_adaln(const h3dit_config* cfg, const void* x, const float* shift,
                         const float* scale, int n_tokens, void* h, cudaStream_t stream);

/* Gated residual fused with the following AdaLN ([linlog] "DiT 融合内核",
 * gated AdaLN fusion):  x = bf16(x + gate * branch) is written exactly and the
 * rounded row is normalised: h = bf16(LN(x) * (1 + scale) + shift).
 * shift/scale NULL: residual only (h unused).  Env H3DIT_DISABLE_GATED_ADALN=1
 * runs the two halves as separate kernels (bit-identical results).
 * x: device BF16 [n][d] in/out; branch: BF16 [n][d]; gate, shift, scale: fp32 [d]. */
h3dit_status h3dit_gate_residual_adaln(const h3dit_config* cfg, void* x, const void* branch,
                                       const float* gate, const float* shift,
                                       const float* scale, int n_tokens, void* h,
                                       cudaStream_t stream);

/* RoPE table: cos/sin of every (token, pair) angle, device fp32
 * [n_tokens][head_dim/2][2] (cos, sin), from device fp32 pos [n_tokens][3]. */
h3dit_status h3dit_rope_table(const h3dit_config* cfg, const float* pos, int n_tokens,
                              float* table, cudaStream_t stream);

/* QKV projection with 3D RoPE in the epilogue and head-major outputs
 * ([linlog] "h3.c 的核心设计": Q/K/V routed head-major for attention):
 *   q[h][t][:] = RoPE(h_t . W_q[h]),  k likewise,  vt[h][c][t] = (h_t . W_v[h])_c
 * h: BF16 [n][d]; w_qkv: BF16 [3d][d]; table: from h3dit_rope_table;
 * q, k: BF16 [heads][n][head_dim]; vt: BF16 [heads][head_dim][vt_ld],
 * vt_ld >= n, vt_ld % 8 == 0.  BF16 precision only. */
h3dit_status h3dit_qkv_project(const h3dit_config* cfg, const void* h, const void* w_qkv,
                               const float* table, int n_tokens, void* q, void* k, void* vt,
                               int vt_ld, cudaStream_t stream);

/* Full non-causal attention per head ([alphalab] full attention):
 *   o[t][h*Dh + c] = sum_j softmax_j(q[h][t] . k[h][j] / sqrt(Dh)) vt[h][c][j]
 * q, k: BF16 [heads][n][Dh]; vt: BF16 [heads][Dh][vt_ld]; o: BF16 [n][d]. */
h3dit_status h3dit_attention(const h3dit_config* cfg, const void* q, const void* k,
                             const void* vt, int vt_ld, int n_tokens, void* o,
                             cudaStream_t stream);

/* AdaLN followed by per-token dynamic int8 quantisation (the int8 path's
 * AdaLN, [linlog] "int8 量化"): hq receives the codes of h3dit_adaln's BF16 h
 * (the rule of h3dit_quantize_act, one group per row) as BF16 values and
 * hs [n] the scales.  x, hq: device BF16 [n][d]; shift, scale: fp32 [d]. */
h3dit_status h3dit_adaln_quant(const h3dit_config* cfg, const void* x, const float* shift,
                               const float* scale, int n_tokens, void* hq, float* hs,
                               cudaStream_t stream);

/* h3dit_gate_residual_adaln with the AdaLN output quantised as in
 * h3dit_adaln_quant (x updated in place as there). */
h3dit_status h3dit_gate_residual_adaln_quant(const h3dit_config* cfg, void* x, const void* branch,
                                             const float* gate, const float* shift,
                                             const float* scale, int n_tokens, void* hq,
                                             float* hs, cudaStream_t stream);

/* h3dit_qkv_project on the int8 path: the projection is h3dit_linear_i8 of
 * the AdaLN codes hq (BF16 [n][d]) with per-token scales hs [n] and the
 * operand-form weight codes w_qkv [3d][d] with scales s_qkv [3d]; RoPE and
 * the head-major outputs as h3dit_qkv_project. */
h3dit_status h3dit_qkv_project_i8(const h3dit_config* cfg, const void* hq, const float* hs,
                                  const void* w_qkv, const float* s_qkv, const float* table,
                                  int n_tokens, void* q, void* k, void* vt, int vt_ld,
                                  cudaStream_t stream);

/* Projection c = act(a b^T): a BF16 [m][k], b BF16 [n][k] (a Linear weight),
 * c BF16 [m][n]; act 0 = none, 1 = GELU tanh form.  n % 256 == 0,
 * k % 64 == 0, any m >= 1. */
h3dit_status h3dit_linear(const void* a, const void* b, int m, int n, int k, int act, void* c,
                          cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* H3DIT_H */
