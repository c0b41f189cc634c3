// C ABI of libtpmlp.so (declared in include/tpmlp.h): argument validation on the host,
// then dispatch to the tensor-core (bf16) or CUDA-core (fp32) kernels. Nothing here
// allocates, frees or synchronises, except tpmlp_device_status.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/tpmlp.h"
#include "device_common.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {

// Device status word, one per device that loads the library (bounded-wait timeouts).
__device__ unsigned int g_device_status;

namespace {

thread_local char g_last_error[512] = "";

tpmlp_status fail(tpmlp_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

tpmlp_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TPMLP_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_ctx_mutex;
DeviceCtx g_ctx[kMaxDevices];
bool g_ctx_ready[kMaxDevices] = {};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elt_size(tpmlp_dtype dt) { return dt == TPMLP_BF16 ? 2 : 4; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

cudaError_t get_device_ctx(DeviceCtx* ctx) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_ctx_mutex);
  if (!g_ctx_ready[dev]) {
    DeviceCtx c;
    c.device = dev;
    e = cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return e;
    c.status = static_cast<unsigned int*>(p);
    g_ctx[dev] = c;
    g_ctx_ready[dev] = true;
  }
  *ctx = g_ctx[dev];
  return cudaSuccess;
}

}  // namespace tpmlp

namespace tpmlp {
// Lets other translation units of the library set the calling thread's last-error message.
int report_error(int status, const char* msg) { return fail(static_cast<tpmlp_status>(status), "%s", msg); }
// The library's failure path on demand: one thread waits on an mbarrier that nothing ever
// completes, gives up after limit_ns like every in-kernel wait, and records the timeout.
__global__ void wait_timeout_check_kernel(unsigned int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait_for(&bar, 0, status, 0xCC, limit_ns);
  }
}

}  // namespace tpmlp

using namespace tpmlp;

namespace {

tpmlp_status check_common(tpmlp_gelu gelu, tpmlp_dtype dt) {
  if (gelu != TPMLP_GELU_ERF && gelu != TPMLP_GELU_TANH) return fail(TPMLP_ERR_INVALID, "unknown gelu variant %d", (int)gelu);
  if (dt != TPMLP_BF16 && dt != TPMLP_F32) return fail(TPMLP_ERR_DTYPE, "unsupported dtype %d", (int)dt);
  return TPMLP_OK;
}

tpmlp_status check_ptrs(tpmlp_dtype dt, std::initializer_list<std::pair<const void*, const char*>> ptrs) {
  const size_t a = dt == TPMLP_BF16 ? 16 : 4;
  for (auto& p : ptrs) {
    if (!p.first) return fail(TPMLP_ERR_INVALID, "%s is NULL", p.second);
    if (!aligned(p.first, a)) return fail(TPMLP_ERR_ALIGN, "%s is not %zu-byte aligned", p.second, a);
  }
  return TPMLP_OK;
}

tpmlp_status check_mlp_shape(int64_t n, int64_t d, int64_t m, int t, tpmlp_dtype dt) {
  if (n < 0 || d < 1 || m < 1) return fail(TPMLP_ERR_SHAPE, "need n >= 0, d >= 1, m >= 1 (n=%lld d=%lld m=%lld)",
                                           (long long)n, (long long)d, (long long)m);
  if (t < 1) return fail(TPMLP_ERR_SHAPE, "t must be >= 1 (t=%d)", t);
  if (m % t != 0) return fail(TPMLP_ERR_SHAPE, "m=%lld is not divisible by t=%d (shards are an equal split)", (long long)m, t);
  if (dt == TPMLP_BF16 && (d % 8 != 0 || m % 8 != 0))
    return fail(TPMLP_ERR_SHAPE, "bf16 path needs d and m to be multiples of 8 (d=%lld m=%lld)", (long long)d, (long long)m);
  if (n > INT32_MAX || d > INT32_MAX || m > INT32_MAX) return fail(TPMLP_ERR_SHAPE, "dimension exceeds 2^31-1");
  return TPMLP_OK;
}

#define TPMLP_TRY(expr)                 \
  do {                                  \
    tpmlp_status _st = (expr);          \
    if (_st != TPMLP_OK) return _st;    \
  } while (0)

#define TPMLP_CUDA(expr, what)                      \
  do {                                              \
    cudaError_t _e = (expr);                        \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

// C = Aop * Bop with the path chosen by dtype.
cudaError_t gemm(tpmlp_dtype dt, int64_t M, int64_t N, int64_t K, const Operand& a, const Operand& b, EpiKind epi,
                 const EpiParams& ep, cudaStream_t s, const DeviceCtx& ctx) {
  if (dt == TPMLP_BF16) return gemm_bf16_tc(M, N, K, a, b, epi, ep, s, ctx);
  return gemm_f32_simt(M, N, K, a, b, epi, ep, s);
}

EpiParams epi(void* out, void* out2, const void* aux, int64_t ldo, tpmlp_gelu g) {
  EpiParams e;
  e.out = out;
  e.out2 = out2;
  e.aux = aux;
  e.bias = nullptr;
  e.ldo = ldo;
  e.gelu = g == TPMLP_GELU_ERF ? kGeluErf : kGeluTanh;
  e.remap.enabled = 0;
  e.remap.b = e.remap.s = e.remap.s_per_shard = 1;
  e.drop.mask_bits = nullptr;
  e.drop.threshold = 0;
  e.drop.seed = 0;
  e.drop.scale = 1.0f;
  return e;
}

// Forward GEMMs shared by tpmlp_forward(_biased) and the sequence-parallel block. bias1 [m] is
// the column-parallel layer's bias (each shard's slice is its column range), added before the
// GeLU; bias2 [d] the row-parallel layer's, added once after the shard sum.
tpmlp_status run_forward(const void* X, const void* A, const void* B, void* O, void* Z, void* Y, int64_t n, int64_t d,
                         int64_t m, tpmlp_gelu g, tpmlp_dtype dt, const RowRemap* remap, cudaStream_t s,
                         const DeviceCtx& ctx, const void* bias1 = nullptr, const void* bias2 = nullptr) {
  // FC1 (column-parallel, all shards at once): Z = X A (+ b1), Y = gelu(Z).
  EpiParams e1 = epi(Z, Y, nullptr, m, g);
  e1.bias = bias1;
  TPMLP_CUDA(gemm(dt, n, m, d, Operand{X, n, d, d, false}, Operand{A, d, m, m, true}, kEpiGelu, e1, s, ctx),
             "FC1 GEMM");
  // FC2 (row-parallel): O = Y B (+ b2); the K-loop runs over every shard, which is the f-bar sum.
  EpiParams e2 = epi(O, nullptr, nullptr, d, g);
  e2.bias = bias2;
  if (remap) e2.remap = *remap;
  TPMLP_CUDA(gemm(dt, n, d, m, Operand{Y, n, m, m, false}, Operand{B, m, d, d, true}, kEpiStore, e2, s, ctx),
             "FC2 GEMM");
  return TPMLP_OK;
}

tpmlp_status forward_impl(const void* X, const void* A, const void* B, const void* bias1, const void* bias2, void* O,
                          void* Z_save, void* Y_save, int64_t n, int64_t d, int64_t m, int t, tpmlp_gelu gelu,
                          tpmlp_dtype dt, void* stream) {
  TPMLP_TRY(check_common(gelu, dt));
  TPMLP_TRY(check_mlp_shape(n, d, m, t, dt));
  TPMLP_TRY(check_ptrs(dt, {{A, "A"}, {B, "B"}}));
  if (bias1 && !aligned(bias1, dt == TPMLP_BF16 ? 16 : 4)) return fail(TPMLP_ERR_ALIGN, "bias1 is misaligned");
  if (bias2 && !aligned(bias2, dt == TPMLP_BF16 ? 16 : 4)) return fail(TPMLP_ERR_ALIGN, "bias2 is misaligned");
  if (n == 0) return TPMLP_OK;  // token-sized buffers may be NULL when there are no tokens
  TPMLP_TRY(check_ptrs(dt, {{X, "X"}, {O, "O"}, {Y_save, "Y_save"}}));
  if (Z_save && !aligned(Z_save, dt == TPMLP_BF16 ? 16 : 4)) return fail(TPMLP_ERR_ALIGN, "Z_save is misaligned");
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  return run_forward(X, A, B, O, Z_save, Y_save, n, d, m, gelu, dt, nullptr, static_cast<cudaStream_t>(stream), ctx,
                     bias1, bias2);
}

size_t d_bytes(int64_t n, int64_t m, tpmlp_dtype dt) {
  if (n <= 0 || m <= 0) return 0;
  return round_up(static_cast<size_t>(n) * static_cast<size_t>(m) * elt_size(dt), 256);
}

size_t colsum_bytes(int64_t n, int64_t d, int64_t m) {
  if (n <= 0) return 0;
  return round_up(colsum_partials_floats(n, m > d ? m : d) * sizeof(float), 256);
}

// The backward's checks of dtype, shape and pointers, which come before its workspace check.
tpmlp_status backward_arg_checks(const void* X, const void* A, const void* B, const void* G, const void* Z_save,
                                 const void* Y_save, const void* dX, const float* dA, const float* dB, int64_t n,
                                 int64_t d, int64_t m, int t, tpmlp_gelu gelu, tpmlp_dtype dt) {
  TPMLP_TRY(check_common(gelu, dt));
  TPMLP_TRY(check_mlp_shape(n, d, m, t, dt));
  TPMLP_TRY(check_ptrs(dt, {{A, "A"}, {B, "B"}}));
  TPMLP_TRY(check_ptrs(dt, {{dA, "dA"}, {dB, "dB"}}));
  if (n > 0)  // token-sized buffers may be NULL when there are no tokens
    TPMLP_TRY(check_ptrs(dt, {{X, "X"}, {G, "G"}, {Z_save, "Z_save"}, {Y_save, "Y_save"}, {dX, "dX"}}));
  return TPMLP_OK;
}

// Backward GEMMs; with dbias1/dbias2 non-null also the bias gradients (column sums of D and G),
// whose partial sums use the workspace after D.
tpmlp_status backward_impl(const void* X, const void* A, const void* B, const void* G, const void* Z_save,
                           const void* Y_save, void* dX, float* dA, float* dB, float* dbias1, float* dbias2, int64_t n,
                           int64_t d, int64_t m, int t, tpmlp_gelu gelu, tpmlp_dtype dt, void* workspace,
                           size_t ws_bytes, void* stream, bool accumulate = false) {
  TPMLP_TRY(backward_arg_checks(X, A, B, G, Z_save, Y_save, dX, dA, dB, n, d, m, t, gelu, dt));
  const bool biases = dbias1 != nullptr || dbias2 != nullptr;
  if (biases && !(dbias1 && dbias2)) return fail(TPMLP_ERR_INVALID, "pass both dbias1 and dbias2");
  if (biases) TPMLP_TRY(check_ptrs(TPMLP_F32, {{dbias1, "dbias1"}, {dbias2, "dbias2"}}));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n > 0) {
    const size_t need = d_bytes(n, m, dt) + (biases ? colsum_bytes(n, d, m) : 0);
    if (!workspace || ws_bytes < need)
      return fail(TPMLP_ERR_WORKSPACE, "backward needs %zu workspace bytes, got %zu", need, workspace ? ws_bytes : 0);
    if (!aligned(workspace, 256)) return fail(TPMLP_ERR_ALIGN, "workspace is not 256-byte aligned");
  }
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  if (n == 0) {
    if (accumulate) return TPMLP_OK;  // nothing to add
    TPMLP_CUDA(cudaMemsetAsync(dA, 0, sizeof(float) * d * m, s), "zero dA");
    TPMLP_CUDA(cudaMemsetAsync(dB, 0, sizeof(float) * m * d, s), "zero dB");
    if (biases) {
      TPMLP_CUDA(cudaMemsetAsync(dbias1, 0, sizeof(float) * m, s), "zero dbias1");
      TPMLP_CUDA(cudaMemsetAsync(dbias2, 0, sizeof(float) * d, s), "zero dbias2");
    }
    return TPMLP_OK;
  }
  void* D = workspace;
  // dgrad-1 with the GeLU' mask: D = (G B^T) * gelu'(Z)   [B read as an [N][K] K-major operand]
  TPMLP_CUDA(gemm(dt, n, m, d, Operand{G, n, d, d, false}, Operand{B, m, d, d, false}, kEpiDGelu,
                  epi(D, nullptr, Z_save, m, gelu), s, ctx),
             "dgrad-1 GEMM");
  // wgrad-2: dB = Y^T G  (both operands MN-major, K = tokens)
  const EpiKind wgrad_epi = accumulate ? kEpiAccumF32 : kEpiStoreF32;
  TPMLP_CUDA(gemm(dt, m, d, n, Operand{Y_save, n, m, m, true}, Operand{G, n, d, d, true}, wgrad_epi,
                  epi(dB, nullptr, nullptr, d, gelu), s, ctx),
             "wgrad-2 GEMM");
  // wgrad-1: dA = X^T D (or dA += X^T D)
  TPMLP_CUDA(gemm(dt, d, m, n, Operand{X, n, d, d, true}, Operand{D, n, m, m, true}, wgrad_epi,
                  epi(dA, nullptr, nullptr, m, gelu), s, ctx),
             "wgrad-1 GEMM");
  // dgrad-2: dX = D A^T; the K-loop over every shard is the f (backward all-reduce) sum.
  TPMLP_CUDA(gemm(dt, n, d, m, Operand{D, n, m, m, false}, Operand{A, d, m, m, false}, kEpiStore,
                  epi(dX, nullptr, nullptr, d, gelu), s, ctx),
             "dgrad-2 GEMM");
  if (biases) {
    // A broadcast bias collects the sum of its rows' gradients: db1 = 1^T D, db2 = 1^T G.
    float* partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + d_bytes(n, m, dt));
    const bool bf16 = dt == TPMLP_BF16;
    TPMLP_CUDA(launch_column_sums(D, n, m, bf16, partials, dbias1, s), "dbias1 column sums");
    TPMLP_CUDA(launch_column_sums(G, n, d, bf16, partials, dbias2, s), "dbias2 column sums");
  }
  return TPMLP_OK;
}

}  // namespace

namespace tpmlp {
int validate_backward_args(const void* X, const void* A, const void* B, const void* G, const void* Z_save,
                           const void* Y_save, const void* dX, const float* dA, const float* dB, int64_t n, int64_t d,
                           int64_t m, int t, int gelu, int dt) {
  return backward_arg_checks(X, A, B, G, Z_save, Y_save, dX, dA, dB, n, d, m, t, static_cast<tpmlp_gelu>(gelu),
                             static_cast<tpmlp_dtype>(dt));
}
}  // namespace tpmlp

extern "C" {

const char* tpmlp_last_error(void) { return g_last_error; }

tpmlp_status tpmlp_forward(const void* X, const void* A, const void* B, void* O, void* Z_save, void* Y_save, int64_t n,
                           int64_t d, int64_t m, int t, tpmlp_gelu gelu, tpmlp_dtype dt, void* stream) {
  return forward_impl(X, A, B, nullptr, nullptr, O, Z_save, Y_save, n, d, m, t, gelu, dt, stream);
}

tpmlp_status tpmlp_forward_biased(const void* X, const void* A, const void* B, const void* bias1, const void* bias2,
                                  void* O, void* Z_save, void* Y_save, int64_t n, int64_t d, int64_t m, int t,
                                  tpmlp_gelu gelu, tpmlp_dtype dt, void* stream) {
  if (!bias1 || !bias2) return fail(TPMLP_ERR_INVALID, "bias1 and bias2 must not be NULL");
  return forward_impl(X, A, B, bias1, bias2, O, Z_save, Y_save, n, d, m, t, gelu, dt, stream);
}

size_t tpmlp_backward_workspace_size(int64_t n, int64_t m, tpmlp_dtype dt) { return d_bytes(n, m, dt); }

tpmlp_status tpmlp_backward(const void* X, const void* A, const void* B, const void* G, const void* Z_save,
                            const void* Y_save, void* dX, float* dA, float* dB, int64_t n, int64_t d, int64_t m, int t,
                            tpmlp_gelu gelu, tpmlp_dtype dt, void* workspace, size_t ws_bytes, void* stream) {
  return backward_impl(X, A, B, G, Z_save, Y_save, dX, dA, dB, nullptr, nullptr, n, d, m, t, gelu, dt, workspace,
                       ws_bytes, stream);
}

tpmlp_status tpmlp_backward_accumulate(const void* X, const void* A, const void* B, const void* G, const void* Z_save,
                                       const void* Y_save, void* dX, float* dA, float* dB, int64_t n, int64_t d,
                                       int64_t m, int t, tpmlp_gelu gelu, tpmlp_dtype dt, void* workspace,
                                       size_t ws_bytes, void* stream) {
  return backward_impl(X, A, B, G, Z_save, Y_save, dX, dA, dB, nullptr, nullptr, n, d, m, t, gelu, dt, workspace,
                       ws_bytes, stream, true);
}

size_t tpmlp_backward_biased_workspace_size(int64_t n, int64_t d, int64_t m, tpmlp_dtype dt) {
  return d_bytes(n, m, dt) + colsum_bytes(n, d, m);
}

tpmlp_status tpmlp_backward_biased(const void* X, const void* A, const void* B, const void* G, const void* Z_save,
                                   const void* Y_save, void* dX, float* dA, float* dB, float* dbias1, float* dbias2,
                                   int64_t n, int64_t d, int64_t m, int t, tpmlp_gelu gelu, tpmlp_dtype dt,
                                   void* workspace, size_t ws_bytes, void* stream) {
  if (!dbias1 || !dbias2) return fail(TPMLP_ERR_INVALID, "dbias1 and dbias2 must not be NULL");
  return backward_impl(X, A, B, G, Z_save, Y_save, dX, dA, dB, dbias1, dbias2, n, d, m, t, gelu, dt, workspace,
                       ws_bytes, stream);
}

namespace {

struct SPLayout {
  size_t xg, y, o, partials, total;
};

SPLayout sp_layout(int64_t b, int64_t s, int64_t h, int64_t m, int t, tpmlp_dtype dt, tpmlp_rs_mode rs) {
  const size_t e = elt_size(dt);
  const size_t tok = static_cast<size_t>(b) * static_cast<size_t>(s);
  SPLayout L;
  size_t off = 0;
  L.xg = off; off += round_up(tok * h * e, 256);
  L.y = off;  off += round_up(tok * m * e, 256);
  L.o = off;  off += round_up(tok * h * e, 256);
  L.partials = off;
  if (rs == TPMLP_RS_SPLITK) off += round_up(static_cast<size_t>(t) * tok * h * sizeof(float), 256);
  L.total = off;
  return L;
}

tpmlp_status check_sp_shape(int64_t b, int64_t s, int64_t h, int t, tpmlp_dtype dt) {
  if (b < 0 || s < 0 || h < 1) return fail(TPMLP_ERR_SHAPE, "need b >= 0, s >= 0, h >= 1");
  if (t < 2) return fail(TPMLP_ERR_SHAPE, "sequence parallelism needs t >= 2 (a tensor-parallel group), got t=%d", t);
  if (s % t != 0) return fail(TPMLP_ERR_SHAPE, "s=%lld is not divisible by t=%d", (long long)s, t);
  if (h % 8 != 0) return fail(TPMLP_ERR_SHAPE, "h=%lld must be a multiple of 8", (long long)h);
  (void)dt;
  return TPMLP_OK;
}

tpmlp_status check_dropout(double p) {
  if (!(p >= 0.0 && p < 1.0)) return fail(TPMLP_ERR_INVALID, "p_drop must lie in [0, 1), got %g", p);
  return TPMLP_OK;
}

// T = floor(p * 2^64) with the product in double; p in [0, 1).
uint64_t drop_threshold(double p) {
  const double v = p * 18446744073709551616.0;
  return static_cast<uint64_t>(v);
}

}  // namespace

size_t tpmlp_sp_block_workspace_size(int64_t b, int64_t s, int64_t h, int64_t m, int t, tpmlp_dtype dt,
                                     tpmlp_rs_mode rs) {
  if (b <= 0 || s <= 0 || h <= 0 || m <= 0 || t <= 0) return 0;
  return sp_layout(b, s, h, m, t, dt, rs).total;
}

tpmlp_status tpmlp_sp_block(const void* x_shards, const float* gamma, const float* beta, float eps, const void* A,
                            const void* B, double p_drop, uint64_t seed, void* out_shards, uint32_t* mask_bits,
                            void* Z_save, void* Y_save, int64_t b, int64_t s, int64_t h, int64_t m, int t,
                            tpmlp_gelu gelu, tpmlp_dtype dt, tpmlp_rs_mode rs, void* workspace, size_t ws_bytes,
                            void* stream) {
  TPMLP_TRY(check_common(gelu, dt));
  TPMLP_TRY(check_sp_shape(b, s, h, t, dt));
  TPMLP_TRY(check_mlp_shape(b * s, h, m, t, dt));
  TPMLP_TRY(check_dropout(p_drop));
  if (rs != TPMLP_RS_FUSED && rs != TPMLP_RS_SPLITK) return fail(TPMLP_ERR_INVALID, "unknown reduce-scatter mode %d", (int)rs);
  if (!(eps > 0.0f)) return fail(TPMLP_ERR_INVALID, "eps must be > 0");
  TPMLP_TRY(check_ptrs(dt, {{A, "A"}, {B, "B"}}));
  TPMLP_TRY(check_ptrs(TPMLP_BF16, {{gamma, "gamma"}, {beta, "beta"}}));
  if (b * s > 0) TPMLP_TRY(check_ptrs(TPMLP_BF16, {{x_shards, "x_shards"}, {out_shards, "out_shards"}}));
  if (mask_bits && (h % 32 != 0 || !aligned(mask_bits, 4)))
    return fail(TPMLP_ERR_SHAPE, "mask_bits needs h %% 32 == 0 and 4-byte alignment");
  if ((Z_save == nullptr) != (Y_save == nullptr)) return fail(TPMLP_ERR_INVALID, "pass both Z_save and Y_save, or neither");
  if (Z_save && b * s > 0) TPMLP_TRY(check_ptrs(dt, {{Z_save, "Z_save"}, {Y_save, "Y_save"}}));
  if (rs == TPMLP_RS_SPLITK && ((m / t) % 8 != 0 && dt == TPMLP_BF16))
    return fail(TPMLP_ERR_SHAPE, "split-K reduce-scatter on bf16 needs m/t to be a multiple of 8");
  const int64_t n = b * s;
  if (n == 0) return TPMLP_OK;
  const SPLayout L = sp_layout(b, s, h, m, t, dt, rs);
  if (!workspace || ws_bytes < L.total)
    return fail(TPMLP_ERR_WORKSPACE, "sp_block needs %zu workspace bytes, got %zu", L.total, workspace ? ws_bytes : 0);
  if (!aligned(workspace, 256)) return fail(TPMLP_ERR_ALIGN, "workspace is not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  char* ws = static_cast<char*>(workspace);
  void* xg = ws + L.xg;
  void* Y = Y_save ? Y_save : static_cast<void*>(ws + L.y);
  void* o = ws + L.o;
  const bool bf16 = dt == TPMLP_BF16;
  // LayerNorm on the shards (SP region) with g, the all-gather into token order, fused into its
  // stores: each normalised row is written at its token-order position.
  const int64_t gather_bst[3] = {b, s, t};
  TPMLP_CUDA(launch_layernorm(x_shards, gamma, beta, eps, xg, n, h, bf16, st, ctx.num_sms, ctx.status, false,
                              gather_bst),
             "layernorm + gather");
  const uint64_t threshold = drop_threshold(p_drop);
  const float scale = static_cast<float>(1.0 / (1.0 - p_drop));
  RowRemap rm;
  rm.enabled = 1;
  rm.b = b;
  rm.s = s;
  rm.s_per_shard = s / t;
  if (rs == TPMLP_RS_FUSED && bf16 && h % 32 == 0) {
    // FC1 + GeLU; then FC2, whose K-loop sums all shards (g-bar's reduction) and whose epilogue
    // writes shard-major rows (g-bar's scatter) after dropout and the residual add.
    TPMLP_CUDA(gemm(dt, n, m, h, Operand{xg, n, h, h, false}, Operand{A, h, m, m, true}, kEpiGelu,
                    epi(Z_save, Y, nullptr, m, gelu), st, ctx),
               "FC1 GEMM");
    EpiParams e2 = epi(out_shards, nullptr, x_shards, h, gelu);
    e2.remap = rm;
    e2.drop.mask_bits = mask_bits;
    e2.drop.threshold = threshold;
    e2.drop.seed = seed;
    e2.drop.scale = scale;
    TPMLP_CUDA(gemm(dt, n, h, m, Operand{Y, n, m, m, false}, Operand{B, m, h, h, true}, kEpiDropoutResidual, e2, st,
                    ctx),
               "FC2 GEMM + dropout + residual");
    return TPMLP_OK;
  }
  if (rs == TPMLP_RS_FUSED) {
    // FC1 + GeLU, then FC2 whose K-loop sums all shards and whose epilogue writes shard-major rows.
    TPMLP_TRY(run_forward(xg, A, B, o, Z_save, Y, n, h, m, gelu, dt, &rm, st, ctx));
  } else {
    TPMLP_CUDA(gemm(dt, n, m, h, Operand{xg, n, h, h, false}, Operand{A, h, m, m, true}, kEpiGelu,
                    epi(Z_save, Y, nullptr, m, gelu), st, ctx),
               "FC1 GEMM");
    // One row GEMM per shard: P_i = Y_i B_i in fp32, then the reduce-scatter kernel.
    const int64_t mt = m / t;
    const size_t e = elt_size(dt);
    float* partials = reinterpret_cast<float*>(ws + L.partials);
    for (int i = 0; i < t; ++i) {
      const void* Yi = static_cast<const char*>(Y) + static_cast<size_t>(i) * mt * e;
      const void* Bi = static_cast<const char*>(B) + static_cast<size_t>(i) * mt * h * e;
      TPMLP_CUDA(gemm(dt, n, h, mt, Operand{Yi, n, mt, m, false}, Operand{Bi, mt, h, h, true}, kEpiStoreF32,
                      epi(partials + static_cast<size_t>(i) * n * h, nullptr, nullptr, h, gelu), st, ctx),
                 "FC2 shard GEMM");
    }
    TPMLP_CUDA(launch_reduce_scatter(partials, o, b, s, h, t, bf16, st, ctx.num_sms), "reduce-scatter");
  }
  // Dropout + residual (SP region).
  TPMLP_CUDA(launch_dropout_residual(x_shards, o, out_shards, mask_bits, threshold, scale, seed, b, s, h, t, bf16, st,
                                     ctx.num_sms, ctx.status),
             "dropout+residual");
  return TPMLP_OK;
}

size_t tpmlp_sp_block_backward_workspace_size(int64_t b, int64_t s, int64_t h, int64_t m, int t, tpmlp_dtype dt) {
  if (b <= 0 || s <= 0 || h <= 0 || m <= 0 || t <= 0) return 0;
  const size_t e = elt_size(dt);
  const size_t tok = static_cast<size_t>(b) * static_cast<size_t>(s);
  return 3 * round_up(tok * h * e, 256) + round_up(tok * m * e, 256) +
         round_up(static_cast<size_t>(kLnBwdMaxCtas) * 2 * h * sizeof(float), 256);
}

tpmlp_status tpmlp_sp_block_backward(const void* x_shards, const float* gamma, const float* beta, float eps,
                                     const void* A, const void* B, double p_drop, uint64_t seed,
                                     const uint32_t* mask_bits, const void* Z_save,
                                     const void* Y_save, const void* dout_shards, void* dx_shards, float* dgamma,
                                     float* dbeta, float* dA, float* dB, int64_t b, int64_t s, int64_t h, int64_t m,
                                     int t, tpmlp_gelu gelu, tpmlp_dtype dt, void* workspace, size_t ws_bytes,
                                     void* stream) {
  TPMLP_TRY(check_common(gelu, dt));
  TPMLP_TRY(check_sp_shape(b, s, h, t, dt));
  TPMLP_TRY(check_mlp_shape(b * s, h, m, t, dt));
  TPMLP_TRY(check_dropout(p_drop));
  if (h > kNormBwdMaxH)
    return fail(TPMLP_ERR_SHAPE, "sp_block_backward supports h <= %d (h=%lld)", kNormBwdMaxH, (long long)h);
  if (mask_bits && (h % 32 != 0 || !aligned(mask_bits, 4)))
    return fail(TPMLP_ERR_SHAPE, "mask_bits needs h %% 32 == 0 and 4-byte alignment");
  if (!(eps > 0.0f)) return fail(TPMLP_ERR_INVALID, "eps must be > 0");
  TPMLP_TRY(check_ptrs(dt, {{A, "A"}, {B, "B"}}));
  TPMLP_TRY(check_ptrs(TPMLP_BF16, {{gamma, "gamma"}, {beta, "beta"}, {dgamma, "dgamma"}, {dbeta, "dbeta"},
                                    {dA, "dA"}, {dB, "dB"}}));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t n = b * s;
  if (n > 0) {
    TPMLP_TRY(check_ptrs(TPMLP_BF16, {{x_shards, "x_shards"}, {dout_shards, "dout_shards"}, {dx_shards, "dx_shards"},
                                      {Z_save, "Z_save"}, {Y_save, "Y_save"}}));
    const size_t need = tpmlp_sp_block_backward_workspace_size(b, s, h, m, t, dt);
    if (!workspace || ws_bytes < need)
      return fail(TPMLP_ERR_WORKSPACE, "sp_block_backward needs %zu workspace bytes, got %zu", need,
                  workspace ? ws_bytes : 0);
    if (!aligned(workspace, 256)) return fail(TPMLP_ERR_ALIGN, "workspace is not 256-byte aligned");
  }
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  if (n == 0) {
    TPMLP_CUDA(cudaMemsetAsync(dA, 0, sizeof(float) * h * m, st), "zero dA");
    TPMLP_CUDA(cudaMemsetAsync(dB, 0, sizeof(float) * m * h, st), "zero dB");
    TPMLP_CUDA(cudaMemsetAsync(dgamma, 0, sizeof(float) * h, st), "zero dgamma");
    TPMLP_CUDA(cudaMemsetAsync(dbeta, 0, sizeof(float) * h, st), "zero dbeta");
    return TPMLP_OK;
  }
  const size_t e = elt_size(dt);
  const size_t tok = static_cast<size_t>(n);
  char* ws = static_cast<char*>(workspace);
  void* xg = ws;
  void* dtok = ws + round_up(tok * h * e, 256);
  void* D = ws + 2 * round_up(tok * h * e, 256);
  void* dxn = static_cast<char*>(D) + round_up(tok * m * e, 256);
  float* partials = reinterpret_cast<float*>(static_cast<char*>(dxn) + round_up(tok * h * e, 256));
  const bool bf16 = dt == TPMLP_BF16;
  // Recompute the LayerNorm output in token order (the forward's g, fused into the LayerNorm's
  // stores), then the local dropout gradient gathered into token order (g-bar's backward).
  const int64_t gather_bst[3] = {b, s, t};
  TPMLP_CUDA(launch_layernorm(x_shards, gamma, beta, eps, xg, n, h, bf16, st, ctx.num_sms, ctx.status, false,
                              gather_bst),
             "layernorm + gather");
  TPMLP_CUDA(launch_dropout_grad_gather(dout_shards, dtok, mask_bits, drop_threshold(p_drop),
                                        static_cast<float>(1.0 / (1.0 - p_drop)), seed, b, s, h,
                                        t, bf16, st, ctx.num_sms),
             "dropout backward + gather");
  // Row-GEMM backward with the GeLU' mask, the two weight gradients, column-GEMM backward.
  TPMLP_CUDA(gemm(dt, n, m, h, Operand{dtok, n, h, h, false}, Operand{B, m, h, h, false}, kEpiDGelu,
                  epi(D, nullptr, Z_save, m, gelu), st, ctx),
             "dgrad-1 GEMM");
  TPMLP_CUDA(gemm(dt, m, h, n, Operand{Y_save, n, m, m, true}, Operand{dtok, n, h, h, true}, kEpiStoreF32,
                  epi(dB, nullptr, nullptr, h, gelu), st, ctx),
             "wgrad-2 GEMM");
  TPMLP_CUDA(gemm(dt, h, m, n, Operand{xg, n, h, h, true}, Operand{D, n, m, m, true}, kEpiStoreF32,
                  epi(dA, nullptr, nullptr, m, gelu), st, ctx),
             "wgrad-1 GEMM");
  // dgrad-2: its K-loop sums every shard's D_i A_i^T and its epilogue writes the rows back in
  // shard layout (g's backward, the reduce-scatter), in the operand dtype like dX.
  EpiParams e5 = epi(dxn, nullptr, nullptr, h, gelu);
  e5.remap.enabled = 1;
  e5.remap.b = b;
  e5.remap.s = s;
  e5.remap.s_per_shard = s / t;
  TPMLP_CUDA(gemm(dt, n, h, m, Operand{D, n, m, m, false}, Operand{A, h, m, m, false}, kEpiStore, e5, st, ctx),
             "dgrad-2 GEMM");
  // LayerNorm backward on the shards plus the residual path.
  TPMLP_CUDA(launch_layernorm_backward(x_shards, dxn, dout_shards, gamma, eps, dx_shards, partials, dgamma, dbeta, n,
                                       h, bf16, st, ctx.num_sms, false, ctx.status),
             "layernorm backward");
  return TPMLP_OK;
}

tpmlp_status tpmlp_sp_layernorm(const void* x, const float* gamma, const float* beta, float eps, void* y, int64_t rows,
                                int64_t h, tpmlp_dtype dt, void* stream) {
  if (dt != TPMLP_BF16 && dt != TPMLP_F32) return fail(TPMLP_ERR_DTYPE, "unsupported dtype %d", (int)dt);
  if (rows < 0 || h < 1) return fail(TPMLP_ERR_SHAPE, "need rows >= 0 and h >= 1");
  if (!(eps > 0.0f)) return fail(TPMLP_ERR_INVALID, "eps must be > 0");
  if (!x || !y || !gamma || !beta) return fail(TPMLP_ERR_INVALID, "null pointer");
  const bool vec = h % 8 == 0;
  if (vec) {
    TPMLP_TRY(check_ptrs(TPMLP_BF16, {{x, "x"}, {y, "y"}}));
    TPMLP_TRY(check_ptrs(TPMLP_BF16, {{gamma, "gamma"}, {beta, "beta"}}));
  }
  if (rows == 0) return TPMLP_OK;
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  TPMLP_CUDA(launch_layernorm(x, gamma, beta, eps, y, rows, h, dt == TPMLP_BF16, static_cast<cudaStream_t>(stream),
                              ctx.num_sms, ctx.status),
             "layernorm");
  return TPMLP_OK;
}

tpmlp_status tpmlp_rmsnorm(const void* x, const float* gamma, float eps, void* y, int64_t rows, int64_t h,
                           tpmlp_dtype dt, void* stream) {
  if (dt != TPMLP_BF16 && dt != TPMLP_F32) return fail(TPMLP_ERR_DTYPE, "unsupported dtype %d", (int)dt);
  if (rows < 0 || h < 1) return fail(TPMLP_ERR_SHAPE, "need rows >= 0 and h >= 1");
  const int64_t h_max = dt == TPMLP_BF16 ? 8192 : 4096;
  if (h % 8 != 0 || h > h_max)
    return fail(TPMLP_ERR_SHAPE, "rmsnorm needs h %% 8 == 0 and h <= %lld (h=%lld)", (long long)h_max, (long long)h);
  if (!(eps > 0.0f)) return fail(TPMLP_ERR_INVALID, "eps must be > 0");
  if (rows > 0 && (!x || !y)) return fail(TPMLP_ERR_INVALID, "null pointer");
  if (!gamma) return fail(TPMLP_ERR_INVALID, "null pointer");
  if (rows > 0) TPMLP_TRY(check_ptrs(TPMLP_BF16, {{x, "x"}, {y, "y"}}));
  TPMLP_TRY(check_ptrs(TPMLP_BF16, {{gamma, "gamma"}}));
  if (rows == 0) return TPMLP_OK;
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  TPMLP_CUDA(launch_layernorm(x, gamma, nullptr, eps, y, rows, h, dt == TPMLP_BF16, static_cast<cudaStream_t>(stream),
                              ctx.num_sms, ctx.status, true),
             "rmsnorm");
  return TPMLP_OK;
}

size_t tpmlp_rmsnorm_backward_workspace_size(int64_t rows, int64_t h) {
  if (rows < 0 || h <= 0) return 0;
  return round_up(static_cast<size_t>(kLnBwdMaxCtas) * 2 * static_cast<size_t>(h) * sizeof(float), 256);
}

tpmlp_status tpmlp_rmsnorm_backward(const void* x, const float* gamma, float eps, const void* dy, void* dx,
                                    float* dgamma, int64_t rows, int64_t h, tpmlp_dtype dt, void* workspace,
                                    size_t ws_bytes, void* stream) {
  if (dt != TPMLP_BF16 && dt != TPMLP_F32) return fail(TPMLP_ERR_DTYPE, "unsupported dtype %d", (int)dt);
  if (rows < 0 || h < 1) return fail(TPMLP_ERR_SHAPE, "need rows >= 0 and h >= 1");
  if (h % 8 != 0 || h > kNormBwdMaxH)
    return fail(TPMLP_ERR_SHAPE, "rmsnorm_backward needs h %% 8 == 0 and h <= %d (h=%lld)", kNormBwdMaxH,
                (long long)h);
  if (!(eps > 0.0f)) return fail(TPMLP_ERR_INVALID, "eps must be > 0");
  if (!gamma || !dgamma) return fail(TPMLP_ERR_INVALID, "null pointer");
  if (rows > 0 && (!x || !dy || !dx)) return fail(TPMLP_ERR_INVALID, "null pointer");
  if (rows > 0) TPMLP_TRY(check_ptrs(TPMLP_BF16, {{x, "x"}, {dy, "dy"}, {dx, "dx"}}));
  TPMLP_TRY(check_ptrs(TPMLP_BF16, {{gamma, "gamma"}, {dgamma, "dgamma"}}));
  const size_t need = tpmlp_rmsnorm_backward_workspace_size(rows, h);
  if (rows > 0 && (!workspace || ws_bytes < need))
    return fail(TPMLP_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
  if (rows > 0) TPMLP_TRY(check_ptrs(TPMLP_BF16, {{workspace, "workspace"}}));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0) {  // no rows: dgamma is an empty sum
    TPMLP_CUDA(cudaMemsetAsync(dgamma, 0, static_cast<size_t>(h) * sizeof(float), st), "zero dgamma");
    return TPMLP_OK;
  }
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  TPMLP_CUDA(launch_layernorm_backward(x, dy, nullptr, gamma, eps, dx, static_cast<float*>(workspace), dgamma, nullptr,
                                       rows, h, dt == TPMLP_BF16, st, ctx.num_sms, true, ctx.status),
             "rmsnorm backward");
  return TPMLP_OK;
}

size_t tpmlp_sp_layernorm_backward_workspace_size(int64_t rows, int64_t h) {
  return tpmlp_rmsnorm_backward_workspace_size(rows, h);
}

tpmlp_status tpmlp_sp_layernorm_backward(const void* x, const float* gamma, float eps, const void* dy,
                                         const void* dres, void* dx, float* dgamma, float* dbeta, int64_t rows,
                                         int64_t h, tpmlp_dtype dt, void* workspace, size_t ws_bytes, void* stream) {
  if (dt != TPMLP_BF16 && dt != TPMLP_F32) return fail(TPMLP_ERR_DTYPE, "unsupported dtype %d", (int)dt);
  if (rows < 0 || h < 1) return fail(TPMLP_ERR_SHAPE, "need rows >= 0 and h >= 1");
  if (h % 8 != 0 || h > kNormBwdMaxH)
    return fail(TPMLP_ERR_SHAPE, "layernorm_backward needs h %% 8 == 0 and h <= %d (h=%lld)", kNormBwdMaxH,
                (long long)h);
  if (!(eps > 0.0f)) return fail(TPMLP_ERR_INVALID, "eps must be > 0");
  if (!gamma || !dgamma || !dbeta) return fail(TPMLP_ERR_INVALID, "null pointer");
  if (rows > 0 && (!x || !dy || !dx)) return fail(TPMLP_ERR_INVALID, "null pointer");
  if (rows > 0) TPMLP_TRY(check_ptrs(TPMLP_BF16, {{x, "x"}, {dy, "dy"}, {dx, "dx"}}));
  if (rows > 0 && dres) TPMLP_TRY(check_ptrs(TPMLP_BF16, {{dres, "dres"}}));
  TPMLP_TRY(check_ptrs(TPMLP_BF16, {{gamma, "gamma"}, {dgamma, "dgamma"}, {dbeta, "dbeta"}}));
  const size_t need = tpmlp_sp_layernorm_backward_workspace_size(rows, h);
  if (rows > 0 && (!workspace || ws_bytes < need))
    return fail(TPMLP_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace ? ws_bytes : 0);
  if (rows > 0) TPMLP_TRY(check_ptrs(TPMLP_BF16, {{workspace, "workspace"}}));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0) {  // empty sums
    TPMLP_CUDA(cudaMemsetAsync(dgamma, 0, static_cast<size_t>(h) * sizeof(float), st), "zero dgamma");
    TPMLP_CUDA(cudaMemsetAsync(dbeta, 0, static_cast<size_t>(h) * sizeof(float), st), "zero dbeta");
    return TPMLP_OK;
  }
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  TPMLP_CUDA(launch_layernorm_backward(x, dy, dres, gamma, eps, dx, static_cast<float*>(workspace), dgamma, dbeta,
                                       rows, h, dt == TPMLP_BF16, st, ctx.num_sms, false, ctx.status),
             "layernorm backward");
  return TPMLP_OK;
}

tpmlp_status tpmlp_sp_dropout_grad_gather(const void* dout_shards, void* dtok, const uint32_t* mask_bits,
                                          double p_drop, uint64_t seed, int64_t b, int64_t s, int64_t h, int t,
                                          tpmlp_dtype dt, void* stream) {
  if (dt != TPMLP_BF16 && dt != TPMLP_F32) return fail(TPMLP_ERR_DTYPE, "unsupported dtype %d", (int)dt);
  TPMLP_TRY(check_sp_shape(b, s, h, t, dt));
  TPMLP_TRY(check_dropout(p_drop));
  if (mask_bits && (h % 32 != 0 || !aligned(mask_bits, 4)))
    return fail(TPMLP_ERR_SHAPE, "mask_bits needs h %% 32 == 0 and 4-byte alignment");
  if (b * s == 0) return TPMLP_OK;
  TPMLP_TRY(check_ptrs(TPMLP_BF16, {{dout_shards, "dout_shards"}, {dtok, "dtok"}}));
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  TPMLP_CUDA(launch_dropout_grad_gather(dout_shards, dtok, mask_bits, drop_threshold(p_drop),
                                        static_cast<float>(1.0 / (1.0 - p_drop)), seed, b, s, h, t,
                                        dt == TPMLP_BF16, static_cast<cudaStream_t>(stream), ctx.num_sms),
             "dropout backward + gather");
  return TPMLP_OK;
}

tpmlp_status tpmlp_sp_gather(const void* x_shards, void* x_full, int64_t b, int64_t s, int64_t h, int t,
                             tpmlp_dtype dt, void* stream) {
  if (dt != TPMLP_BF16 && dt != TPMLP_F32) return fail(TPMLP_ERR_DTYPE, "unsupported dtype %d", (int)dt);
  TPMLP_TRY(check_sp_shape(b, s, h, t, dt));
  if (b * s == 0) return TPMLP_OK;
  TPMLP_TRY(check_ptrs(TPMLP_BF16, {{x_shards, "x_shards"}, {x_full, "x_full"}}));
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  TPMLP_CUDA(launch_gather(x_shards, x_full, b, s, h, t, dt == TPMLP_BF16, static_cast<cudaStream_t>(stream),
                           ctx.num_sms),
             "gather");
  return TPMLP_OK;
}

tpmlp_status tpmlp_sp_reduce_scatter(const float* partials, void* out_shards, int64_t b, int64_t s, int64_t h, int t,
                                     tpmlp_dtype dt, void* stream) {
  if (dt != TPMLP_BF16 && dt != TPMLP_F32) return fail(TPMLP_ERR_DTYPE, "unsupported dtype %d", (int)dt);
  TPMLP_TRY(check_sp_shape(b, s, h, t, dt));
  if (b * s == 0) return TPMLP_OK;
  TPMLP_TRY(check_ptrs(TPMLP_BF16, {{partials, "partials"}, {out_shards, "out_shards"}}));
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  TPMLP_CUDA(launch_reduce_scatter(partials, out_shards, b, s, h, t, dt == TPMLP_BF16,
                                   static_cast<cudaStream_t>(stream), ctx.num_sms),
             "reduce-scatter");
  return TPMLP_OK;
}

tpmlp_status tpmlp_sp_dropout_residual(const void* x_shards, const void* y_shards, void* out_shards,
                                       uint32_t* mask_bits, double p_drop, uint64_t seed, int64_t b, int64_t s,
                                       int64_t h, int t, tpmlp_dtype dt, void* stream) {
  if (dt != TPMLP_BF16 && dt != TPMLP_F32) return fail(TPMLP_ERR_DTYPE, "unsupported dtype %d", (int)dt);
  TPMLP_TRY(check_sp_shape(b, s, h, t, dt));
  TPMLP_TRY(check_dropout(p_drop));
  if (mask_bits && (h % 32 != 0 || !aligned(mask_bits, 4)))
    return fail(TPMLP_ERR_SHAPE, "mask_bits needs h %% 32 == 0 and 4-byte alignment");
  if (b * s == 0) return TPMLP_OK;
  TPMLP_TRY(check_ptrs(TPMLP_BF16, {{x_shards, "x_shards"}, {y_shards, "y_shards"}, {out_shards, "out_shards"}}));
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  TPMLP_CUDA(launch_dropout_residual(x_shards, y_shards, out_shards, mask_bits, drop_threshold(p_drop),
                                     static_cast<float>(1.0 / (1.0 - p_drop)), seed, b, s, h, t,
                                     dt == TPMLP_BF16, static_cast<cudaStream_t>(stream), ctx.num_sms, ctx.status),
             "dropout+residual");
  return TPMLP_OK;
}

tpmlp_status tpmlp_set_gemm_variant(int pair_kernel, int pair_pacing, int pair_group) {
  if (pair_kernel < 0 || pair_kernel > 3 || (pair_pacing != 0 && pair_pacing != 1))
    return fail(TPMLP_ERR_INVALID, "pair_kernel must lie in 0..3 and pair_pacing be 0 or 1 (got %d, %d)", pair_kernel,
                pair_pacing);
  if (pair_group < -4096 || pair_group > 4096)
    return fail(TPMLP_ERR_INVALID, "pair_group must lie in [-4096, 4096], got %d", pair_group);
  set_gemm_variant(pair_kernel, pair_pacing, pair_group);
  return TPMLP_OK;
}

tpmlp_status tpmlp_check_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000ull)
    return fail(TPMLP_ERR_INVALID, "limit_ns must lie in [1e3, 1e9], got %llu", (unsigned long long)limit_ns);
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  wait_timeout_check_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ctx.status, limit_ns);
  TPMLP_CUDA(cudaGetLastError(), "wait-timeout check launch");
  return TPMLP_OK;
}

tpmlp_status tpmlp_device_status(void* stream, int clear) {
  DeviceCtx ctx;
  TPMLP_CUDA(get_device_ctx(&ctx), "device context");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  TPMLP_CUDA(cudaStreamSynchronize(s), "stream synchronize");
  unsigned int word = 0;
  TPMLP_CUDA(cudaMemcpy(&word, ctx.status, sizeof(word), cudaMemcpyDeviceToHost), "read status");
  if (clear) TPMLP_CUDA(cudaMemset(ctx.status, 0, sizeof(word)), "clear status");
  if (word & kStatusTimeoutBit)
    return fail(TPMLP_ERR_TIMEOUT, "a kernel's bounded wait expired (status word 0x%x)", word);
  return TPMLP_OK;
}

}  // extern "C"
