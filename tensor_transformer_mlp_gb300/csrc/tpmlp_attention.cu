// C ABI of the tensor-parallel self-attention block (SenseParrots model-parallel note, section
// 2.1.1; "Megatron 训练" notes, section "Attention 层"): column-parallel QKV projection with the
// heads split across the t shards, per head softmax(Q K^T / sqrt(head_dim)) V in the classic
// Megatron form (P materialised and saved), and a row-parallel
// output projection whose K-loop over every head is the shard sum. All GEMMs run on the tcgen05
// kernel; the per-head GEMMs are batched over (head, sequence) through 4-D tensor maps.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>

#include "../../include/tpmlp.h"
#include "tpmlp_internal.h"

using namespace tpmlp;

namespace {

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tpmlp_status err(tpmlp_status st, const char* msg) { return static_cast<tpmlp_status>(report_error(st, msg)); }

tpmlp_status cuda_err(cudaError_t e, const char* what) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  return err(TPMLP_ERR_CUDA, msg);
}

#define ATT_CUDA(expr, what)                        \
  do {                                              \
    cudaError_t _e = (expr);                        \
    if (_e != cudaSuccess) return cuda_err(_e, what); \
  } while (0)

EpiParams plain_epi(void* out, int64_t ldo) {
  EpiParams e{};
  e.out = out;
  e.ldo = ldo;
  e.gelu = kGeluTanh;
  e.remap.enabled = 0;
  e.remap.b = e.remap.s = e.remap.s_per_shard = 1;
  e.drop.scale = 1.0f;
  return e;
}

tpmlp_status check_shape(int64_t b, int64_t s, int64_t h, int heads, int t, tpmlp_dtype dt) {
  if (dt != TPMLP_BF16) return err(TPMLP_ERR_DTYPE, "the attention block runs on the bf16 tensor-core path only");
  if (b < 0 || s < 1 || h < 1 || heads < 1 || t < 1)
    return err(TPMLP_ERR_SHAPE, "need b >= 0 and s, h, heads, t >= 1");
  if (heads % t != 0) return err(TPMLP_ERR_SHAPE, "heads must split evenly over the t shards");
  if (h % heads != 0) return err(TPMLP_ERR_SHAPE, "h must be a multiple of heads");
  const int64_t dh = h / heads;
  if (dh % 8 != 0 || s % 8 != 0) return err(TPMLP_ERR_SHAPE, "head_dim and s must be multiples of 8");
  if (s > 8192) return err(TPMLP_ERR_SHAPE, "s must be <= 8192 (one softmax row per CTA)");
  if (b * s > INT32_MAX || 3 * h > INT32_MAX) return err(TPMLP_ERR_SHAPE, "dimension exceeds 2^31-1");
  return TPMLP_OK;
}

size_t scores_elems(int64_t b, int64_t s, int heads) {
  return static_cast<size_t>(b) * static_cast<size_t>(heads) * static_cast<size_t>(s) * static_cast<size_t>(s);
}

// Per-head views of the QKV buffer [b*s][3h]: head j's q, k, v are the column blocks
// (3j + c) * dh .. (3j + c + 1) * dh; z1 = head, z2 = sequence.
BatchedOperand qkv_view(const void* QKV, int c, int64_t s, int64_t h, int64_t dh, bool mn_major) {
  const auto* base = static_cast<const __nv_bfloat16*>(QKV) + c * dh;
  return BatchedOperand{base, s, dh, 3 * h, 3 * dh, s * 3 * h, mn_major};
}

// Per-head views of a [b][heads][s][s] buffer.
BatchedOperand scores_view(const void* P, int64_t s, int heads, bool mn_major) {
  return BatchedOperand{P, s, s, s, s * s, heads * s * s, mn_major};
}

// Per-head views of a [b*s][h] buffer whose head j holds columns j*dh .. (j+1)*dh.
BatchedOperand heads_view(const void* O, int64_t s, int64_t h, int64_t dh, bool mn_major) {
  return BatchedOperand{O, s, dh, h, dh, s * h, mn_major};
}

// Partial row statistics of the scores GEMM: two per 256-column N-block of a row.
int64_t stat_parts(int64_t s) { return 2 * ((s + 255) / 256); }

}  // namespace

extern "C" {

size_t tpmlp_attention_forward_workspace_size(int64_t b, int64_t s, int64_t h, int heads, tpmlp_dtype dt) {
  (void)h;
  (void)dt;
  if (b <= 0 || s <= 0 || heads <= 0) return 0;
  const size_t rows = static_cast<size_t>(b) * static_cast<size_t>(heads) * static_cast<size_t>(s);
  return round_up(rows * static_cast<size_t>(stat_parts(s)) * 8, 256) + round_up(rows * 8, 256);
}

tpmlp_status tpmlp_attention_forward(const void* X, const void* Wqkv, const void* Wo, void* Y, void* QKV_save,
                                     void* P_save, void* O_save, int64_t b, int64_t s, int64_t h, int heads, int t,
                                     tpmlp_dtype dt, void* workspace, size_t ws_bytes, void* stream) {
  tpmlp_status st = check_shape(b, s, h, heads, t, dt);
  if (st != TPMLP_OK) return st;
  for (const void* p : {Wqkv, Wo}) {
    if (!p) return err(TPMLP_ERR_INVALID, "null pointer");
    if (!aligned16(p)) return err(TPMLP_ERR_ALIGN, "pointers must be 16-byte aligned");
  }
  if (b == 0) return TPMLP_OK;  // no tokens: nothing to compute
  for (const void* p : {X, static_cast<const void*>(Y), static_cast<const void*>(QKV_save),
                        static_cast<const void*>(P_save), static_cast<const void*>(O_save)}) {
    if (!p) return err(TPMLP_ERR_INVALID, "null pointer");
    if (!aligned16(p)) return err(TPMLP_ERR_ALIGN, "pointers must be 16-byte aligned");
  }
  const size_t need = tpmlp_attention_forward_workspace_size(b, s, h, heads, dt);
  if (!workspace || ws_bytes < need) return err(TPMLP_ERR_WORKSPACE, "attention forward workspace too small");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return err(TPMLP_ERR_ALIGN, "workspace not 256-byte aligned");
  DeviceCtx ctx;
  ATT_CUDA(get_device_ctx(&ctx), "device context");
  cudaStream_t stm = static_cast<cudaStream_t>(stream);
  const int64_t n = b * s, dh = h / heads;
  const int64_t rows = b * heads * s;
  void* stats = workspace;
  void* rowstats = static_cast<char*>(workspace) + round_up(static_cast<size_t>(rows * stat_parts(s)) * 8, 256);
  // QKV = X W_qkv (column-parallel: every shard's heads at once)
  ATT_CUDA(gemm_bf16_tc(n, 3 * h, h, Operand{X, n, h, h, false}, Operand{Wqkv, h, 3 * h, 3 * h, true}, kEpiStore,
                        plain_epi(QKV_save, 3 * h), stm, ctx),
           "QKV GEMM");
  // P = softmax(Q K^T / sqrt(dh)) per (head, sequence) in two passes over the same scores: the
  // first keeps only each row's running max and sum of exp per N-block, the second recomputes
  // the scores (bit-identical accumulators) and writes exp(x - M) / L; no fp32 score matrix.
  BatchSpec bs_s{heads, b, s * s, heads * s * s, static_cast<float>(1.0 / std::sqrt(static_cast<double>(dh)))};
  EpiParams ep_stats = plain_epi(nullptr, s);
  ep_stats.stats = stats;
  ATT_CUDA(gemm_bf16_tc_batched(s, s, dh, qkv_view(QKV_save, 0, s, h, dh, false), qkv_view(QKV_save, 1, s, h, dh, false),
                                bs_s, kEpiRowStats, ep_stats, stm, ctx),
           "scores GEMM (row statistics)");
  ATT_CUDA(launch_softmax_combine(stats, static_cast<int>(stat_parts(s)), rowstats, rows, stm, ctx.num_sms),
           "softmax statistics");
  EpiParams ep_p = plain_epi(P_save, s);
  ep_p.rowvec = rowstats;
  ATT_CUDA(gemm_bf16_tc_batched(s, s, dh, qkv_view(QKV_save, 0, s, h, dh, false), qkv_view(QKV_save, 1, s, h, dh, false),
                                bs_s, kEpiSoftmax, ep_p, stm, ctx),
           "scores GEMM (softmax)");
  // O_head = P V, written into the head's columns of O [b*s][h]
  BatchSpec bs_o{heads, b, dh, s * h, 1.0f};
  ATT_CUDA(gemm_bf16_tc_batched(s, dh, s, scores_view(P_save, s, heads, false), qkv_view(QKV_save, 2, s, h, dh, true),
                                bs_o, kEpiStore, plain_epi(O_save, h), stm, ctx),
           "PV GEMM");
  // Y = O W_o (row-parallel: the K-loop over every head sums the shards' partials)
  ATT_CUDA(gemm_bf16_tc(n, h, h, Operand{O_save, n, h, h, false}, Operand{Wo, h, h, h, true}, kEpiStore,
                        plain_epi(Y, h), stm, ctx),
           "output projection GEMM");
  return TPMLP_OK;
}

size_t tpmlp_attention_backward_workspace_size(int64_t b, int64_t s, int64_t h, int heads, tpmlp_dtype dt) {
  (void)dt;
  if (b <= 0 || s <= 0 || h <= 0 || heads <= 0) return 0;
  const size_t n = static_cast<size_t>(b) * static_cast<size_t>(s);
  const size_t sc = scores_elems(b, s, heads);
  return round_up(n * h * 2, 256) + round_up(n * heads * sizeof(float), 256) + round_up(sc * 2, 256) +
         round_up(n * 3 * h * 2, 256);
}

tpmlp_status tpmlp_attention_backward(const void* X, const void* Wqkv, const void* Wo, const void* G,
                                      const void* QKV_save, const void* P_save, const void* O_save, void* dX,
                                      float* dWqkv, float* dWo, int64_t b, int64_t s, int64_t h, int heads, int t,
                                      tpmlp_dtype dt, void* workspace, size_t ws_bytes, void* stream) {
  tpmlp_status st = check_shape(b, s, h, heads, t, dt);
  if (st != TPMLP_OK) return st;
  for (const void* p : {Wqkv, Wo, static_cast<const void*>(dWqkv), static_cast<const void*>(dWo)}) {
    if (!p) return err(TPMLP_ERR_INVALID, "null pointer");
    if (!aligned16(p)) return err(TPMLP_ERR_ALIGN, "pointers must be 16-byte aligned");
  }
  if (b == 0) {  // no tokens: the weight gradients are empty sums
    cudaStream_t stm = static_cast<cudaStream_t>(stream);
    ATT_CUDA(cudaMemsetAsync(dWqkv, 0, static_cast<size_t>(h) * 3 * h * sizeof(float), stm), "zero dWqkv");
    ATT_CUDA(cudaMemsetAsync(dWo, 0, static_cast<size_t>(h) * h * sizeof(float), stm), "zero dWo");
    return TPMLP_OK;
  }
  for (const void* p : {X, G, QKV_save, P_save, O_save, static_cast<const void*>(dX)}) {
    if (!p) return err(TPMLP_ERR_INVALID, "null pointer");
    if (!aligned16(p)) return err(TPMLP_ERR_ALIGN, "pointers must be 16-byte aligned");
  }
  const size_t need = tpmlp_attention_backward_workspace_size(b, s, h, heads, dt);
  if (!workspace || ws_bytes < need) return err(TPMLP_ERR_WORKSPACE, "attention backward workspace too small");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return err(TPMLP_ERR_ALIGN, "workspace not 256-byte aligned");
  DeviceCtx ctx;
  ATT_CUDA(get_device_ctx(&ctx), "device context");
  cudaStream_t stm = static_cast<cudaStream_t>(stream);
  const int64_t n = b * s, dh = h / heads;
  const size_t sc = scores_elems(b, s, heads);
  char* ws = static_cast<char*>(workspace);
  void* dO = ws;
  float* D = reinterpret_cast<float*>(ws + round_up(static_cast<size_t>(n) * h * 2, 256));
  void* dS = reinterpret_cast<char*>(D) + round_up(static_cast<size_t>(n) * heads * sizeof(float), 256);
  void* dQKV = static_cast<char*>(dS) + round_up(sc * 2, 256);
  // output projection: dO = G W_o^T, dW_o = O^T G. With 128-column heads, the dO GEMM's epilogue
  // also forms D = rowsum(dO * O) per (head, query row) (an epilogue warp holds one head's 128
  // columns of its rows); otherwise a separate kernel does, after the dV GEMM.
  const bool fused_rowdot = dh == 128;
  EpiParams ep_do = plain_epi(dO, h);
  if (fused_rowdot) {
    ep_do.aux = O_save;
    ep_do.rowdot = D;
    ep_do.rowdot_s = s;
    ep_do.rowdot_heads = heads;
  }
  ATT_CUDA(gemm_bf16_tc(n, h, h, Operand{G, n, h, h, false}, Operand{Wo, h, h, h, false},
                        fused_rowdot ? kEpiStoreRowDot : kEpiStore, ep_do, stm, ctx),
           "dO GEMM");
  ATT_CUDA(gemm_bf16_tc(h, h, n, Operand{O_save, n, h, h, true}, Operand{G, n, h, h, true}, kEpiStoreF32,
                        plain_epi(dWo, h), stm, ctx),
           "dWo GEMM");
  // per head: dV = P^T dO, dP = dO V^T, dS = softmax'(dP) / sqrt(dh), dQ = dS K, dK = dS^T Q
  const BatchSpec bs_qkv{heads, b, 3 * dh, s * 3 * h, 1.0f};
  char* dq = static_cast<char*>(dQKV);
  ATT_CUDA(gemm_bf16_tc_batched(s, dh, s, scores_view(P_save, s, heads, true), heads_view(dO, s, h, dh, true), bs_qkv,
                                kEpiStore, plain_epi(dq + 2 * dh * 2, 3 * h), stm, ctx),
           "dV GEMM");
  // dS = P * (dP - D) / sqrt(dh) with dP = dO V^T computed and consumed in the same GEMM's
  // epilogue; D = rowsum(P * dP) = rowsum(dO * O) per (head, query row), from dO and O alone.
  if (!fused_rowdot) ATT_CUDA(launch_row_dot(dO, O_save, D, b, s, h, heads, stm, ctx.num_sms), "rowsum(dO * O)");
  const BatchSpec bs_p{heads, b, s * s, heads * s * s, 1.0f};
  EpiParams ep_ds = plain_epi(dS, s);
  ep_ds.aux = P_save;
  ep_ds.rowvec = D;
  ep_ds.escale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(dh)));
  ATT_CUDA(gemm_bf16_tc_batched(s, s, dh, heads_view(dO, s, h, dh, false), qkv_view(QKV_save, 2, s, h, dh, false),
                                bs_p, kEpiSoftmaxGrad, ep_ds, stm, ctx),
           "dP GEMM (softmax backward)");
  ATT_CUDA(gemm_bf16_tc_batched(s, dh, s, scores_view(dS, s, heads, false), qkv_view(QKV_save, 1, s, h, dh, true),
                                bs_qkv, kEpiStore, plain_epi(dq, 3 * h), stm, ctx),
           "dQ GEMM");
  ATT_CUDA(gemm_bf16_tc_batched(s, dh, s, scores_view(dS, s, heads, true), qkv_view(QKV_save, 0, s, h, dh, true),
                                bs_qkv, kEpiStore, plain_epi(dq + dh * 2, 3 * h), stm, ctx),
           "dK GEMM");
  // QKV projection: dX = dQKV W_qkv^T (K-loop over every shard's heads), dW_qkv = X^T dQKV
  ATT_CUDA(gemm_bf16_tc(n, h, 3 * h, Operand{dQKV, n, 3 * h, 3 * h, false}, Operand{Wqkv, h, 3 * h, 3 * h, false},
                        kEpiStore, plain_epi(dX, h), stm, ctx),
           "dX GEMM");
  ATT_CUDA(gemm_bf16_tc(h, 3 * h, n, Operand{X, n, h, h, true}, Operand{dQKV, n, 3 * h, 3 * h, true}, kEpiStoreF32,
                        plain_epi(dWqkv, 3 * h), stm, ctx),
           "dWqkv GEMM");
  return TPMLP_OK;
}

}  // extern "C"
