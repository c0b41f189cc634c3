// Declarations shared by the translation units of libtpmlp.so (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tpmlp {

constexpr int kGeluErf = 0;
constexpr int kGeluTanh = 1;

// Device status word: bit 0 = a bounded in-kernel wait expired; bits 8.. = where.
constexpr unsigned int kStatusTimeoutBit = 1u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

// Epilogue applied to the fp32 accumulator tile of a GEMM C = Aop * Bop (M x N).
enum EpiKind : int {
  kEpiStore = 0,     // out[r][c] = acc (operand dtype); optional sequence-parallel row remap
  kEpiStoreF32 = 1,  // out[r][c] = acc (fp32)
  kEpiGelu = 2,      // out[r][c] = acc (Z, may be null), out2[r][c] = gelu(acc) (Y)
  kEpiDGelu = 3,     // out[r][c] = acc * gelu'(aux[r][c])  (D = (G B^T) * gelu'(Z))
  kEpiDropoutResidual = 4,  // out[R][c] = aux[R][c] + keep(r, c) * acc * scale, R = remap(r); mask bits
  kEpiAccumF32 = 5,  // out[r][c] += acc (fp32): gradient accumulation into an fp32 main_grad
  // Attention softmax in two GEMM passes over the same scores x = alpha * acc (batched only):
  // (statistics in base 2: y = x * log2(e), so exp(x - max x) = 2^(y - max y))
  kEpiRowStats = 6,     // stats[srow][2*nb + half] = (max y, sum 2^(y - max y)) over the warp's columns
  kEpiSoftmax = 7,      // out[r][c] = 2^(y - rowvec[srow].x), .x = M + log2 L  (P, operand dtype)
  kEpiSoftmaxGrad = 8,  // out[r][c] = escale * aux[r][c] * (x - rowvec[srow])  (dS from dP, P and D)
  // out[r][c] = acc (bf16) and, per 128-column head j of the row, rowdot[(bi * heads + j) * s + si]
  // = sum over the head's columns of out[r][c] * aux[r][c], with r = bi * s + si (plain GEMMs;
  // the attention backward's dO GEMM, aux = O: D = rowsum(dO * O) per head and query row)
  kEpiStoreRowDot = 9,
};

// Dropout of the sequence-parallel block applied in a GEMM epilogue: element (r, c) of the
// token-ordered result has global flat index r * ldo + c and is dropped iff
// splitmix64(seed ^ index) < threshold.
struct DropoutParams {
  uint32_t* mask_bits;  // may be null
  uint64_t threshold;
  uint64_t seed;
  float scale;
};

// Row r of a token-ordered [b][s] x h matrix is written to shard-major position
// [j][bi][l] with r = bi*s + j*(s/t) + l (the reduce-scatter's placement).
struct RowRemap {
  int enabled;
  int64_t b, s, s_per_shard;
};

struct EpiParams {
  void* out;
  void* out2;
  const void* aux;
  const void* bias;  // kEpiGelu, kEpiStore: per-column bias added to the accumulator (operand dtype), or null
  int64_t ldo;  // row stride of out/out2/aux, elements
  int gelu;
  RowRemap remap;
  DropoutParams drop;
  // kEpiRowStats: float2 partial row statistics [rows][2 * N-blocks]; kEpiSoftmax: float2 (M + log2 L, 1/L)
  // per row; kEpiSoftmaxGrad: float D per row. Rows of a batched launch are numbered
  // srow = (z2 * nz1 + z1) * M + r.
  void* stats;
  const void* rowvec;
  float escale;
  // kEpiStoreRowDot: output of the row dots, the sequence length s and the number of heads
  float* rowdot;
  int64_t rowdot_s;
  int rowdot_heads;
};

// A stored operand matrix [rows][cols] with row stride `ld` elements.
//   A operand (M x K): K-major means stored [M][K]; MN-major means stored [K][M].
//   B operand (K x N): K-major means stored [N][K]; MN-major means stored [K][N].
struct Operand {
  const void* ptr;
  int64_t rows, cols, ld;
  bool mn_major;
};

// Batched GEMM: batch index z = z2 * nz1 + z1 (e.g. z1 = attention head, z2 = sequence in the
// batch). A batched operand is a stored matrix per batch index, placed at
// ptr + z1 * z1_stride + z2 * z2_stride (elements) with row stride ld.
struct BatchedOperand {
  const void* ptr;
  int64_t rows, cols, ld;
  int64_t z1_stride, z2_stride;
  bool mn_major;
};

struct BatchSpec {
  int64_t nz1, nz2;
  int64_t out_z1, out_z2;  // element offsets of the output block of batch index (z1, z2)
  float alpha;             // scale applied to the accumulator before the epilogue
};

// Per-device context: SM count and the address of the device status word.
struct DeviceCtx {
  int device;
  int num_sms;
  unsigned int* status;
};

cudaError_t get_device_ctx(DeviceCtx* ctx);

// Sets the calling thread's tpmlp_last_error() message; returns `status`.
int report_error(int status, const char* msg);

// tpmlp_backward's checks of dtype, shape and pointers (everything before its workspace check);
// returns a tpmlp_status and sets the last-error message as tpmlp_backward would.
int validate_backward_args(const void* X, const void* A, const void* B, const void* G, const void* Z_save,
                           const void* Y_save, const void* dX, const float* dA, const float* dB, int64_t n, int64_t d,
                           int64_t m, int t, int gelu, int dt);

// Selects the kernel of later plain bf16 GEMMs (validated by tpmlp_set_gemm_variant).
void set_gemm_variant(int pair_kernel, int pair_pacing, int pair_group);

// bf16 tensor-core GEMM (tcgen05 + TMA). C = Aop(M x K) * Bop(K x N), fp32 accumulation.
cudaError_t gemm_bf16_tc(int64_t M, int64_t N, int64_t K, const Operand& a, const Operand& b, EpiKind epi,
                         const EpiParams& ep, cudaStream_t stream, const DeviceCtx& ctx);

// Batched bf16 tensor-core GEMM: C_z = alpha * Aop_z(M x K) * Bop_z(K x N) for every batch index;
// epilogues kEpiStore (bf16) and kEpiStoreF32, written at ep.out + out offsets of z.
cudaError_t gemm_bf16_tc_batched(int64_t M, int64_t N, int64_t K, const BatchedOperand& a, const BatchedOperand& b,
                                 const BatchSpec& bs, EpiKind epi, const EpiParams& ep, cudaStream_t stream,
                                 const DeviceCtx& ctx);

// fp32 FMA GEMM for the fp32 dtype, same semantics and epilogues (outputs in fp32).
cudaError_t gemm_f32_simt(int64_t M, int64_t N, int64_t K, const Operand& a, const Operand& b, EpiKind epi,
                          const EpiParams& ep, cudaStream_t stream);

// Sequence-parallel memory-bound kernels. `bf16` selects the element type (else fp32).
// rms: RMSNorm instead (beta unused; staged widths only, else cudaErrorNotSupported).
// gather_bst: null, or {b, s, t} of shard-major input rows [t][b][s/t]: the output rows are then
// written in token order [b][s] (the all-gather g fused into the LayerNorm).
cudaError_t launch_layernorm(const void* x, const float* gamma, const float* beta, float eps, void* y,
                             int64_t rows, int64_t h, bool bf16, cudaStream_t stream, int num_sms,
                             unsigned int* status, bool rms = false, const int64_t* gather_bst = nullptr);
cudaError_t launch_gather(const void* x_shards, void* x_full, int64_t b, int64_t s, int64_t h, int t, bool bf16,
                          cudaStream_t stream, int num_sms);
cudaError_t launch_reduce_scatter(const float* partials, void* out_shards, int64_t b, int64_t s, int64_t h, int t,
                                  bool bf16, cudaStream_t stream, int num_sms);
cudaError_t launch_dropout_residual(const void* x_shards, const void* y_shards, void* out_shards,
                                    uint32_t* mask_bits, uint64_t threshold, float scale, uint64_t seed, int64_t b,
                                    int64_t s, int64_t h, int t, bool bf16, cudaStream_t stream, int num_sms,
                                    unsigned int* status);

// Column sums of a row-major [rows][cols] matrix into fp32 out[cols], in a fixed order:
// CTAs sum chunks of kColSumRows rows into partials[chunk][cols], then partials are added in
// chunk order. `partials` needs colsum_partials_floats(rows, cols) floats.
constexpr int kColSumRows = 256;
inline size_t colsum_partials_floats(int64_t rows, int64_t cols) {
  return static_cast<size_t>((rows + kColSumRows - 1) / kColSumRows) * static_cast<size_t>(cols);
}
cudaError_t launch_column_sums(const void* M, int64_t rows, int64_t cols, bool bf16, float* partials, float* out,
                               cudaStream_t stream);

// Sequence-parallel backward: dropout backward fused with the gather into token order; LayerNorm
// backward plus the residual with per-CTA dgamma/dbeta partials ([grid][2][h] fp32, at most
// kLnBwdMaxCtas CTAs) summed in CTA order.
constexpr int kLnBwdMaxCtas = 1024;
constexpr int kNormBwdMaxH = 8192;  // widest row the LayerNorm / RMSNorm backward takes
// mask_bits: the forward's drop bits (read instead of recomputing the hash), or null.
cudaError_t launch_dropout_grad_gather(const void* dout_shards, void* dtok, const uint32_t* mask_bits,
                                       uint64_t threshold, float scale, uint64_t seed, int64_t b, int64_t s,
                                       int64_t h, int t, bool bf16, cudaStream_t stream, int num_sms);
// rms: RMSNorm's backward (dbeta may be null); dout may be null (no residual term).
cudaError_t launch_layernorm_backward(const void* x, const void* dxn, const void* dout, const float* gamma, float eps,
                                      void* dx, float* partials, float* dgamma, float* dbeta, int64_t rows, int64_t h,
                                      bool bf16, cudaStream_t stream, int num_sms, bool rms = false,
                                      unsigned int* status = nullptr);

// Attention helpers: combine the kEpiRowStats partials of each row into (M + log2 L, 1/L); and
// D[(bi*heads + j)*s + si] = dot(dO, O) over head j's columns of token row bi*s + si.
cudaError_t launch_softmax_combine(const void* stats, int nparts, void* rowstats, int64_t rows, cudaStream_t stream,
                                   int num_sms);
cudaError_t launch_row_dot(const void* dO, const void* O, float* D, int64_t b, int64_t s, int64_t h, int heads,
                           cudaStream_t stream, int num_sms);

}  // namespace tpmlp
