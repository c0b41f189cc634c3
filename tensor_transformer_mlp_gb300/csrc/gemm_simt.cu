// fp32 GEMM on the CUDA cores (fp32 FMA, no TF32) for the fp32 dtype of the tensor-parallel
// MLP block: the same six contractions and fused epilogues as the tensor-core path, for
// workloads that must match a float64 reference to ~1e-5 (the two-shard worked example of
// "024 | Megatron-LM: 按矩阵结构切分 Transformer", section 二) and for shapes of any size.
// 64 x 64 output tile per 256-thread CTA, 4 x 4 outputs per thread, K staged 16 at a time.
#include "device_common.cuh"

namespace tpmlp {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

__device__ __forceinline__ int64_t remap_row_f(const RowRemap& rm, int64_t r) {
  if (!rm.enabled) return r;
  const int64_t bi = r / rm.s;
  const int64_t si = r - bi * rm.s;
  const int64_t j = si / rm.s_per_shard;
  const int64_t l = si - j * rm.s_per_shard;
  return (j * rm.b + bi) * rm.s_per_shard + l;
}

template <int EPI>
__device__ __forceinline__ void epilogue_elem(const EpiParams& ep, int64_t r, int64_t c, float acc) {
  float* out = static_cast<float*>(ep.out);
  if constexpr (EPI == kEpiStore || EPI == kEpiGelu) {
    if (ep.bias) acc += static_cast<const float*>(ep.bias)[c];
  }
  if constexpr (EPI == kEpiStore || EPI == kEpiStoreF32) {
    out[remap_row_f(ep.remap, r) * ep.ldo + c] = acc;
  } else if constexpr (EPI == kEpiGelu) {
    if (out) out[r * ep.ldo + c] = acc;
    static_cast<float*>(ep.out2)[r * ep.ldo + c] = gelu_f<true>(acc, ep.gelu);
  } else if constexpr (EPI == kEpiAccumF32) {
    out[r * ep.ldo + c] += acc;
  } else if constexpr (EPI == kEpiDGelu) {
    const float z = static_cast<const float*>(ep.aux)[r * ep.ldo + c];
    out[r * ep.ldo + c] = acc * gelu_grad_f<true>(z, ep.gelu);
  }
}

// C[M][N] = sum_k a(m,k) b(k,n) with a(m,k) = A[m*sam + k*sak], b(k,n) = B[k*sbk + n*sbn].
template <int EPI>
__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, int64_t sam, int64_t sak,
                                                       const float* __restrict__ B, int64_t sbk, int64_t sbn,
                                                       int64_t M, int64_t N, int64_t K, EpiParams ep) {
  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * TN;
  float acc[4][4] = {};
  // Loads run along whichever index is contiguous in memory.
  const bool a_k_fast = (sak == 1);
  const bool b_k_fast = (sbk == 1);
  for (int64_t k0 = 0; k0 < K; k0 += TK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + i * 256;
      const int mm = a_k_fast ? e / TK : e % TM;
      const int kk = a_k_fast ? e % TK : e / TM;
      const int64_t gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < K) ? A[gm * sam + gk * sak] : 0.0f;
      const int nn = b_k_fast ? e / TK : e % TN;
      const int kb = b_k_fast ? e % TK : e / TN;
      const int64_t gn = n0 + nn, gkb = k0 + kb;
      Bs[kb][nn] = (gn < N && gkb < K) ? B[gkb * sbk + gn * sbn] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = m0 + ty + 16 * i;
    if (r >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t c = n0 + tx + 16 * j;
      if (c < N) epilogue_elem<EPI>(ep, r, c, acc[i][j]);
    }
  }
}

template <int EPI>
cudaError_t launch_f32(const float* A, int64_t sam, int64_t sak, const float* B, int64_t sbk, int64_t sbn,
                       int64_t M, int64_t N, int64_t K, const EpiParams& ep, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>((N + TN - 1) / TN), static_cast<unsigned>((M + TM - 1) / TM));
  gemm_f32_kernel<EPI><<<grid, 256, 0, stream>>>(A, sam, sak, B, sbk, sbn, M, N, K, ep);
  return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_f32_simt(int64_t M, int64_t N, int64_t K, const Operand& a, const Operand& b, EpiKind epi,
                          const EpiParams& ep, cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaErrorInvalidValue;
  if ((M + TM - 1) / TM > 65535) return cudaErrorInvalidValue;
  const float* A = static_cast<const float*>(a.ptr);
  const float* B = static_cast<const float*>(b.ptr);
  const int64_t sam = a.mn_major ? 1 : a.ld, sak = a.mn_major ? a.ld : 1;
  const int64_t sbk = b.mn_major ? b.ld : 1, sbn = b.mn_major ? 1 : b.ld;
  switch (epi) {
    case kEpiStore: return launch_f32<kEpiStore>(A, sam, sak, B, sbk, sbn, M, N, K, ep, stream);
    case kEpiStoreF32: return launch_f32<kEpiStoreF32>(A, sam, sak, B, sbk, sbn, M, N, K, ep, stream);
    case kEpiGelu: return launch_f32<kEpiGelu>(A, sam, sak, B, sbk, sbn, M, N, K, ep, stream);
    case kEpiDGelu: return launch_f32<kEpiDGelu>(A, sam, sak, B, sbk, sbn, M, N, K, ep, stream);
    case kEpiAccumF32: return launch_f32<kEpiAccumF32>(A, sam, sak, B, sbk, sbn, M, N, K, ep, stream);
  }
  return cudaErrorNotSupported;
}

}  // namespace tpmlp
