/*
 * tpmlp.h -- C ABI of libtpmlp.so: the Megatron tensor-parallel MLP block and its
 * sequence-parallel form, with all t shards held on one GB300 (sm_103a).
 *
 * The operation ("024 | Megatron-LM: 按矩阵结构切分 Transformer", section 二, block
 * "前向少通信，反向为何仍要一次归约？"): X is n x d, A is d x m split by columns into t
 * equal shards A_i, B is m x d split by the matching rows into B_i, and
 *     Z_i = X A_i,  Y_i = gelu(Z_i),  O = sum_i Y_i B_i;
 * with G = dl/dO,
 *     D_i = (G B_i^T) * gelu'(Z_i),  dA_i = X^T D_i,  dB_i = Y_i^T G,  dX = sum_i D_i A_i^T.
 * Shard i is the column range [i*m/t, (i+1)*m/t) of A and the row range of B, so
 * the forward all-reduce (f-bar) and the backward all-reduce (f) of the
 * multi-GPU layout become the K-loop of one GEMM that runs over every shard in
 * order 0..t-1 and accumulates in tensor memory.
 *
 * Conventions for every entry point:
 *  - All matrices are dense and row-major, in the pages' math layout (A is d x m,
 *    B is m x d), not torch.nn.Linear's [out, in].
 *  - Device pointers unless stated otherwise. The caller owns every buffer,
 *    workspace included; the library never allocates, frees or synchronises
 *    (except tpmlp_device_status). Every call is asynchronous on `stream`
 *    (a cudaStream_t; NULL means the legacy default stream).
 *  - dtype TPMLP_BF16: X, A, B, G, O, Z, Y, dX are bfloat16; arithmetic is fp32
 *    accumulation on the tcgen05 tensor cores. Row lengths d and m must be
 *    multiples of 8 and pointers 16-byte aligned (tensor-memory-access rules).
 *    dtype TPMLP_F32: the same tensors in fp32, computed with fp32 FMA (no TF32);
 *    any shape, 4-byte alignment.
 *  - dA and dB are always fp32 and are overwritten (Megatron keeps fp32 main_grad
 *    buffers for weight gradients: "Megatron 训练" notes, mixed-precision section).
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns an error status and launches nothing. A launch failure
 *    returns TPMLP_ERR_CUDA. tpmlp_last_error() gives a message for the calling
 *    thread's last non-OK status. No entry point aborts or throws.
 *  - Kernels that wait on in-kernel barriers give every wait a time limit; on
 *    expiry they record TPMLP_ERR_TIMEOUT in a device status word, release what
 *    they hold and return. tpmlp_device_status() reads that word.
 *  - The library keeps a little state per device (the status word's address, the SM
 *    count, the GEMM's pacing counters), set up by the first call on that device and
 *    kept for the life of the process: calls run in the device's primary context, and
 *    a cudaDeviceReset while the library is in use is not supported.
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TPMLP_OK = 0,
  TPMLP_ERR_INVALID = 1,    /* null pointer, bad enum, negative size, p outside [0,1) */
  TPMLP_ERR_SHAPE = 2,      /* m % t != 0, s % t != 0, t < 1 (t < 2 for the SP block), d or m not a multiple of 8 */
  TPMLP_ERR_DTYPE = 3,      /* unsupported dtype */
  TPMLP_ERR_ALIGN = 4,      /* pointer not 16-byte aligned (bf16) or 4-byte aligned (fp32) */
  TPMLP_ERR_CUDA = 5,       /* a CUDA runtime/driver call or launch failed */
  TPMLP_ERR_TIMEOUT = 6,    /* a kernel's bounded in-kernel wait expired (tpmlp_device_status) */
  TPMLP_ERR_WORKSPACE = 7   /* workspace null or smaller than the *_workspace_size query */
} tpmlp_status;

typedef enum { TPMLP_GELU_ERF = 0, TPMLP_GELU_TANH = 1 } tpmlp_gelu;
typedef enum { TPMLP_F32 = 0, TPMLP_BF16 = 1 } tpmlp_dtype;

/* How the sequence-parallel block realises g-bar (reduce-scatter of the t row-GEMM
 * partials back to the [b, s/t, h] shards). */
typedef enum {
  TPMLP_RS_FUSED = 0,   /* one row GEMM whose K-loop sums all shards; its epilogue stores rows in shard layout */
  TPMLP_RS_SPLITK = 1   /* t row GEMMs write fp32 partials P_i; a reduce-scatter kernel sums them in shard order */
} tpmlp_rs_mode;

/*
 * Forward: Z = X A, Y = gelu(Z), O = Y B = sum_i Y_i B_i
 * ("024 | Megatron-LM", section 二; SenseParrots model-parallel note, section 2.1, eqs. (1)(2)).
 *   X [n][d], A [d][m], B [m][d] (inputs, dtype dt)
 *   O [n][d] (output, dt)
 *   Z_save [n][m] (output, dt; may be NULL, then Z is not stored and backward cannot run)
 *   Y_save [n][m] (output, dt; required: the row GEMM reads it)
 *   n >= 0 tokens, d >= 1, m >= 1, 1 <= t with m % t == 0; gelu selects exact-erf or tanh GeLU.
 *   With n == 0 nothing is launched and X, O, Z_save, Y_save may be NULL.
 * gelu is evaluated in fp32 on the fp32 accumulator before Z and Y are rounded to dt.
 */
tpmlp_status tpmlp_forward(const void* X, const void* A, const void* B,
                           void* O, void* Z_save, void* Y_save,
                           int64_t n, int64_t d, int64_t m, int t,
                           tpmlp_gelu gelu, tpmlp_dtype dt, void* stream);

/* Bytes of device workspace tpmlp_backward needs: D = (G B^T) * gelu'(Z), n x m in dt. */
size_t tpmlp_backward_workspace_size(int64_t n, int64_t m, tpmlp_dtype dt);

/*
 * Backward ("024 | Megatron-LM", section 二, D_i / dA_i / dB_i equations and the dX reduction):
 *   D = (G B^T) * gelu'(Z)  (in workspace, dt; gelu' evaluated in fp32 from the stored Z)
 *   dB = Y^T G   [m][d] fp32     dA = X^T D   [d][m] fp32     dX = D A^T   [n][d] dt
 *   X [n][d], A [d][m], B [m][d], G [n][d], Z_save and Y_save [n][m] as written by tpmlp_forward.
 *   workspace: at least tpmlp_backward_workspace_size(n, m, dt) bytes, 256-byte aligned.
 * n == 0 gives dA = dB = 0 (X, G, Z_save, Y_save, dX, workspace may then be NULL).
 */
tpmlp_status tpmlp_backward(const void* X, const void* A, const void* B, const void* G,
                            const void* Z_save, const void* Y_save,
                            void* dX, float* dA, float* dB,
                            int64_t n, int64_t d, int64_t m, int t,
                            tpmlp_gelu gelu, tpmlp_dtype dt,
                            void* workspace, size_t ws_bytes, void* stream);

/*
 * tpmlp_backward without a caller workspace. The source pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory (a host that passes only the
 * step's tensors and owns no device allocator, or code that must not allocate once its steady
 * state has begun). It computes exactly what tpmlp_backward computes, with the same arguments
 * minus the workspace, and keeps D in a static device array of 64 MiB (67,108,864 bytes)
 * inside the library, which every GPU that loads the library holds until the process exits.
 *   - Arguments are checked exactly as tpmlp_backward checks them, with the same statuses;
 *     then n * m * element size above 64 MiB is rejected with TPMLP_ERR_WORKSPACE before
 *     anything runs (bf16: n * m <= 33,554,432, e.g. n = 8192 with m = 4096; fp32: half that).
 *     Use tpmlp_backward with a workspace for larger problems.
 *   - The result is bit-identical to tpmlp_backward's on the same inputs.
 *   - It allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 *   - The first call on a device looks up the array's device address on that device (once);
 *     make that first call before any stream capture. The address is kept for the life of the
 *     process, so a cudaDeviceReset between calls, or a context other than the device's
 *     primary context, is not supported.
 *   - Every call on a device shares the one array: calls that may overlap on the GPU (on
 *     different streams, or from several threads) race on it and must be serialised by the
 *     caller. D is fully rewritten by each call, so no clearing is needed between calls.
 */
tpmlp_status tpmlp_backward_noalloc(const void* X, const void* A, const void* B, const void* G,
                                    const void* Z_save, const void* Y_save,
                                    void* dX, float* dA, float* dB,
                                    int64_t n, int64_t d, int64_t m, int t,
                                    tpmlp_gelu gelu, tpmlp_dtype dt, void* stream);

/*
 * tpmlp_backward with fp32 gradient accumulation for dA and dB: dA += X^T D, dB += Y^T G, added
 * by the weight-gradient GEMMs' epilogues into the caller's fp32 buffers (Megatron keeps fp32
 * main_grad buffers and fuses the accumulation into the wgrad GEMM: "Megatron 训练" notes,
 * gradient_accumulation_fusion and the mixed-precision section). dX is overwritten as in
 * tpmlp_backward; workspace as for tpmlp_backward. n == 0 leaves dA and dB unchanged.
 */
tpmlp_status tpmlp_backward_accumulate(const void* X, const void* A, const void* B, const void* G,
                                       const void* Z_save, const void* Y_save,
                                       void* dX, float* dA, float* dB,
                                       int64_t n, int64_t d, int64_t m, int t,
                                       tpmlp_gelu gelu, tpmlp_dtype dt,
                                       void* workspace, size_t ws_bytes, void* stream);

/*
 * The same block with Megatron's biases ("Megatron 训练" notes: ColumnParallelLinear keeps a
 * bias split like its output columns; RowParallelLinear keeps one full bias, added once after
 * the all-reduce):
 *   Z = X A + bias1, Y = gelu(Z), O = Y B + bias2
 *   bias1 [m], bias2 [d] in dt (16-byte aligned for bf16), both required. Everything else as
 *   for tpmlp_forward; Z_save then holds the biased pre-activation.
 */
tpmlp_status tpmlp_forward_biased(const void* X, const void* A, const void* B,
                                  const void* bias1, const void* bias2,
                                  void* O, void* Z_save, void* Y_save,
                                  int64_t n, int64_t d, int64_t m, int t,
                                  tpmlp_gelu gelu, tpmlp_dtype dt, void* stream);

/* Bytes of device workspace tpmlp_backward_biased needs: D plus the bias-gradient partial sums. */
size_t tpmlp_backward_biased_workspace_size(int64_t n, int64_t d, int64_t m, tpmlp_dtype dt);

/*
 * tpmlp_backward for the biased block, plus the bias gradients (the matmul-gradient rule of the
 * "Megatron 训练" notes: a broadcast bias collects the sum of its rows' gradients):
 *   dbias1 = sum over tokens of D   [m] fp32 (overwritten)
 *   dbias2 = sum over tokens of G   [d] fp32 (overwritten)
 * Z_save and Y_save come from tpmlp_forward_biased. The sums run in a fixed order
 * (deterministic). workspace: at least tpmlp_backward_biased_workspace_size(n, d, m, dt) bytes.
 */
tpmlp_status tpmlp_backward_biased(const void* X, const void* A, const void* B, const void* G,
                                   const void* Z_save, const void* Y_save,
                                   void* dX, float* dA, float* dB, float* dbias1, float* dbias2,
                                   int64_t n, int64_t d, int64_t m, int t,
                                   tpmlp_gelu gelu, tpmlp_dtype dt,
                                   void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace tpmlp_sp_block needs (LN output in token order, Y, row-GEMM output or partials). */
size_t tpmlp_sp_block_workspace_size(int64_t b, int64_t s, int64_t h, int64_t m, int t,
                                     tpmlp_dtype dt, tpmlp_rs_mode rs);

/*
 * Sequence-parallel MLP block ("Megatron-SP 机制", section "通信插在层内什么位置？"):
 *   out = x + dropout(RS(MLP(AG(LayerNorm(x)))))
 *   x_shards, out_shards: [t][b][s/t][h] in dt (shard j holds sequence positions j*s/t .. (j+1)*s/t-1)
 *   gamma, beta: [h] fp32; eps > 0. LayerNorm uses the biased variance and fp32 statistics.
 *   A [h][m], B [m][h] (dt), gelu as for tpmlp_forward.
 *   Dropout: p_drop in [0, 1) is the drop probability, a double, so that the threshold
 *   T = floor(p_drop * 2^64) (product in double) is the one a caller computes from the same
 *   value (p = 0.1 gives T = 0x1999999999999A00). Element k of the logical [b][s][h] tensor
 *   (row-major flat index) is dropped iff splitmix64(seed ^ k) < T; kept elements are scaled
 *   by 1/(1-p_drop), computed in double and applied in fp32; the residual is x.
 *   mask_bits: NULL, or [ceil(b*s*h/32)] uint32 words; bit i of word w is 1 iff element
 *   32*w+i (global flat index) was dropped. Needs h % 32 == 0.
 *   Z_save, Y_save: NULL, or [b*s][m] in dt (token order): FC1's pre- and post-GeLU activations,
 *   kept for tpmlp_sp_block_backward (pass both or neither).
 *   Requires t >= 2 (sequence parallelism needs a tensor-parallel group:
 *   "Megatron-SP 机制", section "工程约束与实测收益是什么？"), s % t == 0, m % t == 0.
 */
tpmlp_status tpmlp_sp_block(const void* x_shards, const float* gamma, const float* beta, float eps,
                            const void* A, const void* B, double p_drop, uint64_t seed,
                            void* out_shards, uint32_t* mask_bits, void* Z_save, void* Y_save,
                            int64_t b, int64_t s, int64_t h, int64_t m, int t,
                            tpmlp_gelu gelu, tpmlp_dtype dt, tpmlp_rs_mode rs,
                            void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace tpmlp_sp_block_backward needs. */
size_t tpmlp_sp_block_backward_workspace_size(int64_t b, int64_t s, int64_t h, int64_t m, int t,
                                              tpmlp_dtype dt);

/*
 * Backward of tpmlp_sp_block (the SP backward chain of the "Efficient Large-Scale ... Megatron-LM"
 * notes, section 3.5.1: local dropout/LayerNorm gradients, all-gather, row-GEMM backward, GeLU
 * backward, column-GEMM backward, reduce-scatter), from dout_shards = dl/d out_shards:
 *   dx_shards = dout + LayerNorm'(x)^T (dl/d LN output)        [t][b][s/t][h] in dt
 *   dgamma, dbeta: [h] fp32 (overwritten)      dA [h][m], dB [m][h]: fp32 (overwritten)
 * Inputs as for tpmlp_sp_block, plus Z_save and Y_save ([b*s][m] in dt, token order) written by
 * the forward call with the same arguments. The dropout mask is read from mask_bits when it is
 * given (the forward's mask_bits output for the same seed and p_drop; needs h % 32 == 0), else
 * recomputed from (seed, p_drop); both give the same result.
 * The LayerNorm output and the gathered tokens are recomputed from x (memory-bound), not saved.
 * Requires h <= 8192 and h % 8 == 0 in addition to tpmlp_sp_block's rules.
 */
tpmlp_status tpmlp_sp_block_backward(const void* x_shards, const float* gamma, const float* beta, float eps,
                                     const void* A, const void* B, double p_drop, uint64_t seed,
                                     const uint32_t* mask_bits,
                                     const void* Z_save, const void* Y_save, const void* dout_shards,
                                     void* dx_shards, float* dgamma, float* dbeta, float* dA, float* dB,
                                     int64_t b, int64_t s, int64_t h, int64_t m, int t,
                                     tpmlp_gelu gelu, tpmlp_dtype dt,
                                     void* workspace, size_t ws_bytes, void* stream);

/*
 * The sequence-parallel block's memory-bound steps as separate calls, same layouts as above.
 *
 * LayerNorm of `rows` rows of width h ("Megatron 训练" notes, section "LayerNorm";
 * torch.nn.LayerNorm semantics): y = (x - mean) / sqrt(var + eps) * gamma + beta.
 */
tpmlp_status tpmlp_sp_layernorm(const void* x, const float* gamma, const float* beta, float eps,
                                void* y, int64_t rows, int64_t h, tpmlp_dtype dt, void* stream);

/*
 * RMSNorm of `rows` rows of width h ("Megatron 训练" notes, section "RMSNorm": LayerNorm with
 * the mean computation removed), for use in front of either block:
 *   y = x / sqrt(mean(x^2) + eps) * gamma      (mean over the h elements of a row; no bias).
 * x, y: [rows][h] in dt (may alias); gamma: [h] fp32 device. Statistics in fp32.
 * Requires h % 8 == 0 and h <= 8192 (bf16) or 4096 (f32), eps > 0, 16-byte aligned pointers.
 * Errors: TPMLP_ERR_SHAPE, TPMLP_ERR_INVALID (null pointer, eps), TPMLP_ERR_ALIGN, TPMLP_ERR_DTYPE.
 */
tpmlp_status tpmlp_rmsnorm(const void* x, const float* gamma, float eps, void* y, int64_t rows, int64_t h,
                           tpmlp_dtype dt, void* stream);

/*
 * Backward of tpmlp_rmsnorm from dy = dl/dy ([rows][h], dt): with r = 1/sqrt(mean(x^2) + eps),
 * x_hat = x r and g = dy gamma,
 *   dx = r * (g - x_hat * mean(g * x_hat))     ([rows][h], dt, overwritten)
 *   dgamma = sum over rows of dy * x_hat       ([h] fp32, overwritten; summed in a fixed order).
 * workspace: device memory of tpmlp_rmsnorm_backward_workspace_size(rows, h) bytes (per-CTA
 * partial sums), 16-byte aligned. Requires h % 8 == 0 and h <= 8192; rows == 0 zeroes dgamma.
 */
size_t tpmlp_rmsnorm_backward_workspace_size(int64_t rows, int64_t h);
tpmlp_status tpmlp_rmsnorm_backward(const void* x, const float* gamma, float eps, const void* dy, void* dx,
                                    float* dgamma, int64_t rows, int64_t h, tpmlp_dtype dt, void* workspace,
                                    size_t ws_bytes, void* stream);

/*
 * LayerNorm backward of `rows` rows of width h, with an optional residual gradient (the SP
 * backward's last step: "Efficient Large-Scale ... Megatron-LM" notes, section 3.5.1; formulas as
 * in the "Megatron 训练" notes, section "LayerNorm", torch.nn.LayerNorm semantics): with
 * x_hat = (x - mean) / sqrt(var + eps) (biased variance over the row) and g = dy * gamma,
 *   dx = dres + (g - mean(g) - x_hat * mean(g * x_hat)) / sqrt(var + eps)   ([rows][h], dt)
 *   dgamma = sum over rows of dy * x_hat,  dbeta = sum over rows of dy      ([h] fp32, overwritten;
 *   summed in a fixed order, so the result is deterministic).
 * x, dy, dres, dx: [rows][h] in dt; dres may be NULL (no residual term); gamma: [h] fp32.
 * workspace: tpmlp_sp_layernorm_backward_workspace_size(rows, h) bytes (per-CTA partial sums),
 * 16-byte aligned. Requires h % 8 == 0, h <= 8192, eps > 0, 16-byte aligned pointers.
 * rows == 0 zeroes dgamma and dbeta.
 */
size_t tpmlp_sp_layernorm_backward_workspace_size(int64_t rows, int64_t h);
tpmlp_status tpmlp_sp_layernorm_backward(const void* x, const float* gamma, float eps, const void* dy,
                                         const void* dres, void* dx, float* dgamma, float* dbeta,
                                         int64_t rows, int64_t h, tpmlp_dtype dt,
                                         void* workspace, size_t ws_bytes, void* stream);

/*
 * Dropout backward fused with the backward of g-bar (whose backward is an all-gather; "Megatron-SP
 * 机制", f/g operator table): dtok [b][s][h] in token order from dout_shards [t][b][s/t][h],
 *   dtok[k] = keep(k) * dout[k] / (1 - p_drop)   (k the global flat index of the logical [b][s][h]
 * tensor). The mask is read from mask_bits when given (the forward's output for the same seed and
 * p_drop, layout as for tpmlp_sp_block; needs h % 32 == 0), else recomputed from (seed, p_drop)
 * exactly as tpmlp_sp_block draws it.
 */
tpmlp_status tpmlp_sp_dropout_grad_gather(const void* dout_shards, void* dtok, const uint32_t* mask_bits,
                                          double p_drop, uint64_t seed,
                                          int64_t b, int64_t s, int64_t h, int t, tpmlp_dtype dt,
                                          void* stream);

/* g forward, all-gather ("Megatron-SP 机制", f/g operator table): [t][b][s/t][h] -> [b][s][h]. */
tpmlp_status tpmlp_sp_gather(const void* x_shards, void* x_full,
                             int64_t b, int64_t s, int64_t h, int t, tpmlp_dtype dt, void* stream);

/* g-bar forward, reduce-scatter ("Megatron-SP 机制", f/g operator table):
 * partials [t][b*s][h] fp32 in token order -> out_shards [t][b][s/t][h] in dt,
 * out = sum_i partials[i], added in order i = 0..t-1 in fp32. */
tpmlp_status tpmlp_sp_reduce_scatter(const float* partials, void* out_shards,
                                     int64_t b, int64_t s, int64_t h, int t, tpmlp_dtype dt, void* stream);

/* Dropout + residual on shards ("Megatron-SP 机制", placement diagram, last step):
 * out = x + keep * y / (1 - p_drop), mask definition and mask_bits as for tpmlp_sp_block.
 * x_shards, y_shards, out_shards: [t][b][s/t][h] in dt. */
tpmlp_status tpmlp_sp_dropout_residual(const void* x_shards, const void* y_shards, void* out_shards,
                                       uint32_t* mask_bits, double p_drop, uint64_t seed,
                                       int64_t b, int64_t s, int64_t h, int t,
                                       tpmlp_dtype dt, void* stream);

/*
 * Tensor-parallel self-attention block (SenseParrots model-parallel note, section 2.1.1, its
 * parallel multi-head attention code; "Megatron 训练" notes, section "Attention 层":
 * S = Q K^T / sqrt(d), A = softmax(S)). bf16 only.
 *   X [b*s][h]; W_qkv [h][3h] with head j's columns [q | k | v] at (3j .. 3j+3) * head_dim
 *   (column-parallel: shard i owns heads i*heads/t .. (i+1)*heads/t - 1); W_o [h][h]
 *   (row-parallel: shard i owns the rows of its heads).
 *   Per head and sequence: P = softmax(Q K^T / sqrt(head_dim)) over the keys (no mask; no
 *   attention dropout), O_head = P V; O [b*s][h] holds the heads side by side; Y = O W_o, the
 *   K-loop over every head being the shard sum.
 *   Saves (caller-owned, for the backward): QKV_save [b*s][3h], P_save [b][heads][s][s],
 *   O_save [b*s][h]. workspace: per-row softmax statistics (the scores go through two GEMM
 *   passes: row max and sum of exp, then P; no score matrix is stored),
 *   tpmlp_attention_forward_workspace_size bytes, 256-byte aligned.
 *   Requires heads % t == 0, h % heads == 0, head_dim and s multiples of 8, s <= 8192. b == 0
 *   is an empty batch: nothing is computed and the token buffers may be NULL.
 */
size_t tpmlp_attention_forward_workspace_size(int64_t b, int64_t s, int64_t h, int heads, tpmlp_dtype dt);
tpmlp_status tpmlp_attention_forward(const void* X, const void* Wqkv, const void* Wo, void* Y,
                                     void* QKV_save, void* P_save, void* O_save,
                                     int64_t b, int64_t s, int64_t h, int heads, int t, tpmlp_dtype dt,
                                     void* workspace, size_t ws_bytes, void* stream);

/*
 * Backward of the attention block from G = dl/dY [b*s][h]: dX [b*s][h] (bf16), dWqkv [h][3h] and
 * dWo [h][h] (fp32, overwritten). dO = G W_o^T, dW_o = O^T G; per head dV = P^T dO,
 * dP = dO V^T, dS = P * (dP - rowsum(P * dP)) / sqrt(head_dim), dQ = dS K, dK = dS^T Q;
 * dX = dQKV W_qkv^T, dW_qkv = X^T dQKV. Saves from tpmlp_attention_forward. rowsum(P * dP) is
 * taken as rowsum(dO * O) per head (equal, since O = P V), so dS comes out of the dP GEMM's
 * epilogue and dP is never stored. workspace: tpmlp_attention_backward_workspace_size bytes
 * (dO, that row sum, dS, dQKV), 256-byte aligned. With b == 0 the weight gradients are zeroed
 * (empty sums) and the token buffers may be NULL.
 */
size_t tpmlp_attention_backward_workspace_size(int64_t b, int64_t s, int64_t h, int heads, tpmlp_dtype dt);
tpmlp_status tpmlp_attention_backward(const void* X, const void* Wqkv, const void* Wo, const void* G,
                                      const void* QKV_save, const void* P_save, const void* O_save,
                                      void* dX, float* dWqkv, float* dWo,
                                      int64_t b, int64_t s, int64_t h, int heads, int t, tpmlp_dtype dt,
                                      void* workspace, size_t ws_bytes, void* stream);

/*
 * Kernel choice for the plain bf16 GEMMs of every later call in this process, for comparing
 * kernels and testing each one; a user of the library never needs it, and nothing else
 * (no environment variable) changes the choice. The defaults, 1, 1, 0, are the fast path:
 *   pair_kernel 1: clusters of two SMs, on 256 x 512 or 256 x 256 tiles per GEMM by a model of
 *                  the launch's waves; 2: clusters of two SMs on 256 x 256 tiles only; 3: on
 *                  256 x 512 tiles only (a last round that would keep at most half the SM pairs
 *                  busy runs as 256 x 256 half-tiles, one per pair); 0: 128 x 256 tiles on one SM.
 *   pair_pacing 1: pairs wait at intervals of 16 k-blocks for the pairs of the same round of
 *                  tiles, which keeps shared operand panels in L2; 0: no pacing.
 *   pair_group  0: the default tile band (16 pair-rows walked along N, for 256 x 256 and
 *                  256 x 512 tiles); g > 0: g pair-rows walked along N; g < 0: -g N-blocks
 *                  walked along M. |g| <= 4096.
 * The choice is read when a GEMM is launched, so a CUDA graph keeps the one it captured.
 * Every variant computes the same contractions with fp32 accumulation. Errors: TPMLP_ERR_INVALID.
 */
tpmlp_status tpmlp_set_gemm_variant(int pair_kernel, int pair_pacing, int pair_group);

/* Message for the calling thread's last non-OK status ("" if none). Never NULL. */
const char* tpmlp_last_error(void);

/*
 * Synchronises `stream`, then reads the current device's status word, which kernels set when a
 * bounded in-kernel wait expires. Returns TPMLP_OK or TPMLP_ERR_TIMEOUT (or TPMLP_ERR_CUDA if
 * the synchronisation itself fails). clear != 0 resets the word.
 */
tpmlp_status tpmlp_device_status(void* stream, int clear);

/*
 * Exercises the failure path above on the GPU: launches a kernel whose one waiting thread waits
 * on a barrier that nothing completes, gives up after limit_ns nanoseconds (1e3..1e9) and
 * records a timeout in the device status word, exactly as a stalled GEMM or staged kernel would.
 * A following tpmlp_device_status then returns TPMLP_ERR_TIMEOUT; the context stays usable.
 * Nothing faults, traps or spins without a limit.
 */
tpmlp_status tpmlp_check_wait_timeout(uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H */
