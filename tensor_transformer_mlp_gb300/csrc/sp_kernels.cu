// Memory-bound kernels of the sequence-parallel MLP block ("Megatron-SP 机制", section
// "通信插在层内什么位置？"): LayerNorm on [b, s/t, h] shards, the all-gather g that turns
// shard-major rows into token order, the reduce-scatter g-bar that sums t fp32 partials
// and writes shard-major rows, and dropout + residual add with a counter-hash mask.
// All shards live in one HBM buffer [t][b][s/t][h], so g and g-bar are row permutations
// (plus the t-way sum for g-bar). Every kernel moves 16-byte vectors, one row per CTA
// iteration, with the shard <-> token mapping computed once per row.
#include "device_common.cuh"

namespace tpmlp {
namespace {

// Token row r = bi*s + j*sl + l  <->  shard-major row R = (j*b + bi)*sl + l.
__device__ __forceinline__ int64_t shard_row_to_token(int64_t R, int64_t b, int64_t s, int64_t sl) {
  const int64_t jb = R / sl;
  const int64_t l = R - jb * sl;
  const int64_t j = jb / b;
  const int64_t bi = jb - j * b;
  return bi * s + j * sl + l;
}

template <typename T>
struct Vec8;  // 8 elements of T

template <>
struct Vec8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void store(__nv_bfloat16* p) const { *reinterpret_cast<uint4*>(p) = u; }
  __device__ __forceinline__ void to_float(float (&f)[8]) const {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = unpack_bf16x2(w[i]);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
  __device__ __forceinline__ void from_float(const float (&f)[8]) {
    u = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                   pack_bf16x2(f[6], f[7]));
  }
};

template <>
struct Vec8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  __device__ __forceinline__ void store(float* p) const {
    reinterpret_cast<float4*>(p)[0] = a;
    reinterpret_cast<float4*>(p)[1] = b;
  }
  __device__ __forceinline__ void to_float(float (&f)[8]) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
  __device__ __forceinline__ void from_float(const float (&f)[8]) {
    a = make_float4(f[0], f[1], f[2], f[3]);
    b = make_float4(f[4], f[5], f[6], f[7]);
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ LayerNorm
// One warp per row; the row stays in registers (MAXV vectors of 8 per lane), so it is
// read from HBM once. Statistics in fp32: mean, then the biased variance of the
// deviations (two passes over registers).
template <typename T, int MAXV>
__global__ void __launch_bounds__(256) layernorm_kernel(const T* __restrict__ x, const float* __restrict__ gamma,
                                                        const float* __restrict__ beta, float eps, T* __restrict__ y,
                                                        int64_t rows, int h) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const float inv_h = 1.0f / static_cast<float>(h);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const T* xr = x + r * h;
    float v[MAXV][8];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int c = (lane + 32 * i) * 8;
      if (c < h) {
        Vec8<T> in;
        in.load(xr + c);
        in.to_float(v[i]);
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += v[i][e];
      }
    }
    const float mean = warp_sum(sum) * inv_h;
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      if ((lane + 32 * i) * 8 < h) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dlt = v[i][e] - mean;
          sq = fmaf(dlt, dlt, sq);
        }
      }
    }
    const float rstd = rsqrtf(warp_sum(sq) * inv_h + eps);
    T* yr = y + r * h;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int c = (lane + 32 * i) * 8;
      if (c < h) {
        const float4 g0 = reinterpret_cast<const float4*>(gamma + c)[0], g1 = reinterpret_cast<const float4*>(gamma + c)[1];
        const float4 b0 = reinterpret_cast<const float4*>(beta + c)[0], b1 = reinterpret_cast<const float4*>(beta + c)[1];
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = fmaf((v[i][e] - mean) * rstd, g[e], bb[e]);
        Vec8<T> out;
        out.from_float(o);
        out.store(yr + c);
      }
    }
  }
}

// Any width: one CTA per row, three passes over the row (it stays in L1/L2).
template <typename T>
__global__ void __launch_bounds__(256) layernorm_generic_kernel(const T* __restrict__ x,
                                                                const float* __restrict__ gamma,
                                                                const float* __restrict__ beta, float eps,
                                                                T* __restrict__ y, int64_t rows, int64_t h) {
  __shared__ float red[8];
  __shared__ float stat;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* xr = x + r * h;
    float acc = 0.f;
    for (int64_t c = threadIdx.x; c < h; c += blockDim.x) acc += static_cast<float>(xr[c]);
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
      for (int w = 0; w < (blockDim.x >> 5); ++w) s += red[w];
      stat = s / static_cast<float>(h);
    }
    __syncthreads();
    const float mean = stat;
    __syncthreads();
    acc = 0.f;
    for (int64_t c = threadIdx.x; c < h; c += blockDim.x) {
      const float dlt = static_cast<float>(xr[c]) - mean;
      acc = fmaf(dlt, dlt, acc);
    }
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
      for (int w = 0; w < (blockDim.x >> 5); ++w) s += red[w];
      stat = rsqrtf(s / static_cast<float>(h) + eps);
    }
    __syncthreads();
    const float rstd = stat;
    for (int64_t c = threadIdx.x; c < h; c += blockDim.x)
      y[r * h + c] = static_cast<T>(fmaf((static_cast<float>(xr[c]) - mean) * rstd, gamma[c], beta[c]));
    __syncthreads();
  }
}

// ------------------------------------------------------------------ gather (g forward)
// Destination row r (token order) <- source shard-major row; rows are copied as 16-byte vectors.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                     int64_t rows, int64_t b, int64_t s, int64_t sl, int row_vecs) {
  for (int64_t R = blockIdx.x; R < rows; R += gridDim.x) {
    const int64_t r = shard_row_to_token(R, b, s, sl);
    const uint4* sr = src + R * row_vecs;
    uint4* dr = dst + r * row_vecs;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) dr[c] = sr[c];
  }
}

// ------------------------------------------------------------------ reduce-scatter (g-bar forward)
// Shard-major output row R <- sum over i = 0..t-1 (in order) of partials[i][token row].
template <typename T>
__global__ void __launch_bounds__(256) reduce_scatter_kernel(const float* __restrict__ partials, T* __restrict__ out,
                                                             int64_t rows, int64_t b, int64_t s, int64_t sl, int h,
                                                             int t) {
  const int64_t plane = rows * static_cast<int64_t>(h);
  const int nvec = h >> 3;
  for (int64_t R = blockIdx.x; R < rows; R += gridDim.x) {
    const int64_t r = shard_row_to_token(R, b, s, sl);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const int c = v * 8;
      float acc[8];
      Vec8<float> p;
      p.load(partials + r * h + c);
      p.to_float(acc);
      for (int i = 1; i < t; ++i) {
        float f[8];
        p.load(partials + i * plane + r * h + c);
        p.to_float(f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += f[e];
      }
      Vec8<T> o;
      o.from_float(acc);
      o.store(out + R * h + c);
    }
  }
}

// ------------------------------------------------------------------ dropout + residual
// SplitMix64 (Steele, Lea, Flood 2014; the splitmix64.c step published by Vigna):
// golden-gamma increment, then the variant-13 mixer.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// out = x + keep * y * scale for shard-major rows; element k of the logical token-order
// tensor is dropped iff splitmix64(seed ^ k) < threshold. Each thread handles 8 consecutive
// elements; 4 neighbouring lanes OR their bits into one 32-bit mask word.
template <typename T>
__global__ void __launch_bounds__(256) dropout_residual_kernel(const T* __restrict__ x, const T* __restrict__ y,
                                                               T* __restrict__ out, uint32_t* __restrict__ mask_bits,
                                                               uint64_t threshold, float scale, uint64_t seed,
                                                               int64_t rows, int64_t b, int64_t s, int64_t sl,
                                                               int h) {
  const int nvec = h >> 3;
  for (int64_t R = blockIdx.x; R < rows; R += gridDim.x) {
    const int64_t r = shard_row_to_token(R, b, s, sl);
    const uint64_t flat_row = static_cast<uint64_t>(r) * static_cast<uint64_t>(h);
    for (int v0 = 0; v0 < nvec; v0 += blockDim.x) {  // uniform trip count across the CTA
      const int v = v0 + threadIdx.x;
      uint32_t bits = 0;
      if (v < nvec) {
        const int c = v * 8;
        Vec8<T> xv, yv;
        xv.load(x + R * h + c);
        yv.load(y + R * h + c);
        float xf[8], yf[8], o[8];
        xv.to_float(xf);
        yv.to_float(yf);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const bool drop = splitmix64(seed ^ (flat_row + static_cast<uint64_t>(c + e))) < threshold;
          bits |= (drop ? 1u : 0u) << e;
          o[e] = drop ? xf[e] : fmaf(yf[e], scale, xf[e]);
        }
        Vec8<T> ov;
        ov.from_float(o);
        ov.store(out + R * h + c);
      }
      if (mask_bits != nullptr) {
        bits <<= 8 * (threadIdx.x & 3);
        bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
        bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
        if (v < nvec && (threadIdx.x & 3) == 0) mask_bits[(flat_row + static_cast<uint64_t>(v) * 8) >> 5] = bits;
      }
    }
  }
}

int rows_grid(int64_t rows, int num_sms, int per_sm) {
  const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
  return static_cast<int>(rows < cap ? (rows > 0 ? rows : 1) : cap);
}

}  // namespace

cudaError_t launch_layernorm(const void* x, const float* gamma, const float* beta, float eps, void* y, int64_t rows,
                             int64_t h, bool bf16, cudaStream_t stream, int num_sms) {
  if (rows <= 0) return cudaSuccess;
  const bool vec_ok = (h % 8 == 0) && (h <= 32 * 8 * 16);
  if (vec_ok) {
    const int warps_per_cta = 8;
    const int64_t ctas = (rows + warps_per_cta - 1) / warps_per_cta;
    const int grid = static_cast<int>(ctas < static_cast<int64_t>(num_sms) * 8 ? ctas : static_cast<int64_t>(num_sms) * 8);
    const int maxv = static_cast<int>((h / 8 + 31) / 32);
    if (bf16) {
      auto xp = static_cast<const __nv_bfloat16*>(x);
      auto yp = static_cast<__nv_bfloat16*>(y);
      if (maxv <= 4) layernorm_kernel<__nv_bfloat16, 4><<<grid, 256, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else if (maxv <= 8) layernorm_kernel<__nv_bfloat16, 8><<<grid, 256, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else layernorm_kernel<__nv_bfloat16, 16><<<grid, 256, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
    } else {
      auto xp = static_cast<const float*>(x);
      auto yp = static_cast<float*>(y);
      if (maxv <= 4) layernorm_kernel<float, 4><<<grid, 256, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else if (maxv <= 8) layernorm_kernel<float, 8><<<grid, 256, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
      else layernorm_kernel<float, 16><<<grid, 256, 0, stream>>>(xp, gamma, beta, eps, yp, rows, (int)h);
    }
  } else {
    const int grid = rows_grid(rows, num_sms, 8);
    if (bf16)
      layernorm_generic_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x), gamma, beta, eps, static_cast<__nv_bfloat16*>(y), rows, h);
    else
      layernorm_generic_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(x), gamma, beta, eps,
                                                                 static_cast<float*>(y), rows, h);
  }
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* x_shards, void* x_full, int64_t b, int64_t s, int64_t h, int t, bool bf16,
                          cudaStream_t stream, int num_sms) {
  const int64_t rows = b * s;
  if (rows <= 0) return cudaSuccess;
  const int64_t row_bytes = h * (bf16 ? 2 : 4);
  if (row_bytes % 16 != 0) return cudaErrorInvalidValue;
  gather_kernel<<<rows_grid(rows, num_sms, 8), 256, 0, stream>>>(static_cast<const uint4*>(x_shards),
                                                                   static_cast<uint4*>(x_full), rows, b, s, s / t,
                                                                   static_cast<int>(row_bytes / 16));
  return cudaGetLastError();
}

cudaError_t launch_reduce_scatter(const float* partials, void* out_shards, int64_t b, int64_t s, int64_t h, int t,
                                  bool bf16, cudaStream_t stream, int num_sms) {
  const int64_t rows = b * s;
  if (rows <= 0) return cudaSuccess;
  if (h % 8 != 0) return cudaErrorInvalidValue;
  const int grid = rows_grid(rows, num_sms, 8);
  if (bf16)
    reduce_scatter_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(partials, static_cast<__nv_bfloat16*>(out_shards),
                                                                    rows, b, s, s / t, static_cast<int>(h), t);
  else
    reduce_scatter_kernel<float><<<grid, 256, 0, stream>>>(partials, static_cast<float*>(out_shards), rows, b, s,
                                                            s / t, static_cast<int>(h), t);
  return cudaGetLastError();
}

cudaError_t launch_dropout_residual(const void* x_shards, const void* y_shards, void* out_shards,
                                    uint32_t* mask_bits, uint64_t threshold, float scale, uint64_t seed, int64_t b,
                                    int64_t s, int64_t h, int t, bool bf16, cudaStream_t stream, int num_sms) {
  const int64_t rows = b * s;
  if (rows <= 0) return cudaSuccess;
  if (h % 8 != 0 || (mask_bits && h % 32 != 0)) return cudaErrorInvalidValue;
  const int grid = rows_grid(rows, num_sms, 8);
  if (bf16)
    dropout_residual_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(x_shards), static_cast<const __nv_bfloat16*>(y_shards),
        static_cast<__nv_bfloat16*>(out_shards), mask_bits, threshold, scale, seed, rows, b, s, s / t,
        static_cast<int>(h));
  else
    dropout_residual_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(x_shards),
                                                              static_cast<const float*>(y_shards),
                                                              static_cast<float*>(out_shards), mask_bits, threshold,
                                                              scale, seed, rows, b, s, s / t, static_cast<int>(h));
  return cudaGetLastError();
}

}  // namespace tpmlp
